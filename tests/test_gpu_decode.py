"""GPU parity of decode (q_len = 1) paged attention against the fp64 oracle,
through the C ABI, run as the whole step (staged diffs + gather, KV write,
forward): bf16 output within max |err| <= 2e-2 and mean |err| <= 2e-3; FP8 runs
against the oracle fed the same E4M3 codes (decoded and scaled in fp64)."""
import numpy as np
import pytest
import torch

import workloads
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import DeviceStep, assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu


def run_and_check(w, dev, max_splits=32, what=""):
    step = DeviceStep(w, dev, max_splits=max_splits)
    out = step.run()
    assert pa.get_error() == pa.PA_OK
    ref, _, _, gathered = oracle_step(w)
    np.testing.assert_array_equal(step.gathered.cpu().numpy(), gathered)
    return assert_attention_close(out, ref, what=what or w.name), out, step


@pytest.mark.parametrize("q_mult", [1.0, 4.0])
def test_tiny_decode_config(cuda_device, q_mult):
    run_and_check(workloads.make(1, device=cuda_device, q_mult=q_mult), cuda_device)


@pytest.mark.parametrize("q_mult", [1.0, 4.0])
def test_decode_7b_config_full(cuda_device, q_mult):
    """The full 256-request decode batch, every output row compared."""
    w = workloads.make(2, device=cuda_device, q_mult=q_mult)
    run_and_check(w, cuda_device)


def test_prefix_shared_fp8_config_full(cuda_device):
    w = workloads.make(4, device=cuda_device)
    assert w.kv_dtype == "fp8"
    run_and_check(w, cuda_device)


CASES = [
    # seq_lens, Hq, Hkv, D, B, dtype
    ([1, 15, 16, 17, 31, 33, 100, 257], 4, 4, 64, 16, "bf16"),
    ([1, 2, 47, 64, 65, 200, 1000], 8, 4, 128, 32, "bf16"),
    ([5, 64, 129, 700], 16, 4, 128, 64, "fp8"),
    ([3, 300, 999, 4000], 32, 4, 128, 16, "fp8"),       # g = 8: two CTAs per kv head
    ([7, 513, 2048], 32, 2, 128, 16, "bf16"),           # g = 16
    ([9, 130, 77], 8, 8, 64, 64, "fp8"),
    ([17, 1111], 4, 1, 64, 32, "bf16"),                 # g = 4, D = 64
    ([3, 47, 1500], 32, 2, 128, 16, "fp8"),             # g = 16: hi and mid in two products
    ([11, 260, 33], 8, 4, 64, 32, "fp8"),               # g = 2, D = 64
    ([31, 32, 33, 777], 16, 8, 128, 32, "fp8"),         # g = 2, B = 32: two chunks per block
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
@pytest.mark.parametrize("max_splits", [0, 3, 64])
def test_decode_shapes(cuda_device, case, max_splits):
    seq, Hq, Hkv, D, B, dt = case
    w = workloads.build(seq, [1] * len(seq), Hq, Hkv, D, B, kv_dtype=dt, seed=sum(seq) + Hq,
                        device=cuda_device, pool_blocks=None)
    run_and_check(w, cuda_device, max_splits=max_splits)


@pytest.mark.parametrize("g", [4, 16])
def test_decode_fp8_query_magnitudes_per_head(cuda_device, g):
    """E4M3 pools: every query head gets its own power-of-two scale before it
    is split into E4M3 parts, so heads of very different size, and an
    all-zero head, keep their accuracy."""
    Hkv = 2
    w = workloads.build([5, 333, 1200], [1, 1, 1], Hq=g * Hkv, Hkv=Hkv, D=128, B=16,
                        kv_dtype="fp8", seed=77, device=cuda_device)
    mult = torch.tensor([0.0, 1e-3, 1.0, 7.5] * (g * Hkv // 4), device=w.q.device)
    w.q.mul_(mult.view(1, -1, 1).to(w.q.dtype))
    run_and_check(w, cuda_device)


def test_decode_long_context_requests(cuda_device):
    """32768-token decodes with B = 64 and 8 query heads per kv head."""
    w = workloads.build([32768, 32768, 20000], [1, 1, 1], Hq=64, Hkv=8, D=128, B=64,
                        seed=55, device=cuda_device)
    run_and_check(w, cuda_device)


def test_decode_output_invariant_under_block_placement(cuda_device):
    """Relocating physical blocks (and the tables with them) leaves the output
    bit-identical: splits are fixed by logical position."""
    w = workloads.build([100, 2000, 517, 33], [1, 1, 1, 1], Hq=8, Hkv=2, D=128, B=16,
                        seed=12, device=cuda_device, pool_blocks=300)
    step = DeviceStep(w, cuda_device)
    base = step.run().clone()
    perm = torch.from_numpy(np.random.default_rng(1).permutation(w.num_blocks)).to(cuda_device)
    k2 = torch.empty_like(step.pool.k)
    v2 = torch.empty_like(step.pool.v)
    k2[perm] = step.pool.k
    v2[perm] = step.pool.v
    pool2 = pa.KVPool(k2, v2, w.k_scale, w.v_scale)
    g = step.gathered
    tables2 = torch.where(g >= 0, perm[g.clamp(min=0).long()].int(), g)
    out2 = torch.empty_like(base)
    pa.forward(step.q, out2, step.qsl, step.seq, w.qsl, w.seq_lens, tables2, pool2, w.scale,
               w.causal, workspace=step.ws)
    assert pa.get_error() == pa.PA_OK
    assert torch.equal(out2.view(torch.int16), base.view(torch.int16))


def test_decode_shared_prefix_equals_private_copies(cuda_device):
    """Requests that share prefix blocks give bit-identical outputs to the same
    requests holding private copies of those blocks."""
    members = list(range(6))
    w = workloads.build([80, 65, 99, 64 + 1, 150, 70], [1] * 6, Hq=8, Hkv=2, D=128, B=16,
                        kv_dtype="fp8", seed=4, device=cuda_device, groups=[(members, 64)],
                        pool_blocks=60)
    step = DeviceStep(w, cuda_device)
    base = step.run().clone()
    g = step.gathered.clone()
    used = set(g[g >= 0].cpu().tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    src, dst = [], []
    for r in range(1, 6):
        for i in range(4):  # the 4 shared blocks
            src.append(int(g[r, i]))
            dst.append(free.pop())
            g[r, i] = dst[-1]
    pa.copy_blocks(step.pool, torch.tensor(src, dtype=torch.int32, device=cuda_device),
                   torch.tensor(dst, dtype=torch.int32, device=cuda_device))
    out2 = torch.empty_like(base)
    pa.forward(step.q, out2, step.qsl, step.seq, w.qsl, w.seq_lens, g, step.pool, w.scale,
               w.causal, workspace=step.ws)
    assert pa.get_error() == pa.PA_OK
    assert torch.equal(out2.view(torch.int16), base.view(torch.int16))


def test_decode_is_deterministic(cuda_device):
    w = workloads.make(2, device=cuda_device, num_requests=64)
    step = DeviceStep(w, cuda_device)
    a = step.run().clone()
    b = step.run().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_empty_requests_rows_untouched(cuda_device):
    w = workloads.build([40, 10, 70], [1, 0, 1], Hq=4, Hkv=2, D=64, B=16, seed=2,
                        device=cuda_device)
    step = DeviceStep(w, cuda_device, out_fill=7.0)
    out = step.run()
    assert pa.get_error() == pa.PA_OK
    ref, *_ = oracle_step(w)
    assert_attention_close(out, ref)
    empty = workloads.build([], [], Hq=4, Hkv=2, D=64, B=16, seed=2, device=cuda_device)
    assert empty.R == 0


def test_forward_flags_bad_block_ids_without_faulting(cuda_device):
    w = workloads.build([50, 20], [1, 1], Hq=2, Hkv=2, D=64, B=16, seed=6, device=cuda_device)
    step = DeviceStep(w, cuda_device)
    step.run()
    assert pa.get_error() == pa.PA_OK
    bad = step.gathered.clone()
    bad[0, 1] = w.num_blocks + 1000
    pa.forward(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens, bad, step.pool,
               w.scale, w.causal)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS


def test_forward_host_checks(cuda_device):
    w = workloads.build([50, 20], [1, 1], Hq=2, Hkv=2, D=64, B=16, seed=6, device=cuda_device)
    step = DeviceStep(w, cuda_device)
    with pytest.raises(pa.PaError) as e:   # seq_len beyond the table
        pa.forward(step.q, step.out, step.qsl, step.seq, w.qsl, np.array([5000, 20]),
                   step.gathered, step.pool, w.scale, 1)
    assert e.value.status == pa.PA_ERR_INVALID
    with pytest.raises(pa.PaError) as e:   # qsl does not end at T
        pa.forward(step.q, step.out, step.qsl, step.seq, np.array([0, 1, 1]), w.seq_lens,
                   step.gathered, step.pool, w.scale, 1)
    assert e.value.status == pa.PA_ERR_INVALID
    with pytest.raises(pa.PaError) as e:   # 3 query heads over 2 kv heads
        pa.forward(step.q[:, :1].contiguous().expand(-1, 3, -1).contiguous(),
                   torch.empty((2, 3, 64), dtype=torch.bfloat16, device=cuda_device),
                   step.qsl, step.seq, w.qsl, w.seq_lens, step.gathered, step.pool, w.scale, 1)
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
    empty = pa.KVPool(step.pool.k[:0], step.pool.v[:0])  # a pool of no blocks
    with pytest.raises(pa.PaError) as e:
        pa.forward(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens, step.gathered,
                   empty, w.scale, 1)
    assert e.value.status == pa.PA_ERR_INVALID
