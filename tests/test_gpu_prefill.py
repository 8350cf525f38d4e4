"""GPU parity of prefill-chunk (q_len > 1) paged attention on tcgen05/TMEM and
of mixed decode + prefill batches against the fp64 oracle, through the C ABI
(whole step: staged diffs + gather, KV write, forward)."""
import numpy as np
import pytest
import torch

import workloads
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import DeviceStep, assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu


def check(w, dev, rows=None, max_splits=32):
    step = DeviceStep(w, dev, max_splits=max_splits)
    out = step.run()
    assert pa.get_error() == pa.PA_OK
    ref, _, _, _ = oracle_step(w, rows=rows)
    return assert_attention_close(out, ref, rows=rows, what=w.name), out, step


CASES = [
    # seq_lens, q_lens, Hq, Hkv, D, B, causal
    ([200], [200], 4, 4, 128, 16, 1),                 # g 1, 2 q tiles, ragged kv tail
    ([129], [129], 1, 1, 128, 16, 1),                 # one row past a tile
    ([300, 77], [45, 77], 8, 2, 128, 32, 1),          # g 4, cached prefix
    ([1000], [333], 16, 2, 128, 64, 1),               # g 8
    ([520, 2], [260, 2], 32, 2, 128, 16, 1),          # g 16, tiny chunk
    ([400], [150], 8, 4, 64, 16, 1),                  # D 64, g 2
    ([250, 64], [250, 64], 4, 2, 128, 16, 0),         # non-causal
    ([33, 1000, 17, 2048], [2, 1, 17, 600], 8, 2, 128, 16, 1),  # mixed with decodes
    ([4096 + 7], [130], 8, 8, 128, 32, 1),            # long prefix, q tile boundary
]


@pytest.mark.parametrize("case", CASES, ids=[f"c{i}" for i in range(len(CASES))])
def test_prefill_shapes(cuda_device, case):
    seq, ql, Hq, Hkv, D, B, causal = case
    w = workloads.build(seq, ql, Hq, Hkv, D, B, causal=causal, seed=sum(seq) + Hq + causal,
                        device=cuda_device)
    check(w, cuda_device)


@pytest.mark.parametrize("q_mult", [1.0, 4.0])
def test_prefill_stress_peaky_softmax(cuda_device, q_mult):
    w = workloads.build([700, 900], [700, 300], Hq=8, Hkv=2, D=128, B=16, seed=91,
                        device=cuda_device, q_mult=q_mult)
    check(w, cuda_device)


def _tile_rows(w, kv_heads=None):
    """Every decode row, plus whole query tiles of every prefill chunk: the
    kernel's tile is 128 // g consecutive tokens x the g query heads of one kv
    head; the tiles at the chunk's start, at the middle of its causal
    diagonal and at its end, for every kv head (or the kv heads that
    kv_heads(r, tile) names). Rows are token * Hq + head."""
    g = w.Hq // w.Hkv
    tpt = 128 // g
    rows = []
    for r in range(w.R):
        a, b = int(w.qsl[r]), int(w.qsl[r + 1])
        ql = b - a
        if ql == 1:
            rows.extend(a * w.Hq + h for h in range(w.Hq))
        elif ql > 1:
            n_tiles = (ql + tpt - 1) // tpt
            for t in sorted({0, (ql // 2) // tpt, n_tiles - 1}):
                kvs = range(w.Hkv) if kv_heads is None else kv_heads(r, t)
                for tok in range(a + t * tpt, min(b, a + (t + 1) * tpt)):
                    for kv in kvs:
                        rows.extend(tok * w.Hq + kv * g + j for j in range(g))
    return np.unique(np.array(rows, np.int64))


def test_mixed_chunked_prefill_config_full_size(cuda_device):
    """The mixed 4096-token step: 64 decodes + chunks 1024/1024/1920 after
    prefixes 0/2048/8192; every decode row and whole query tiles (start,
    diagonal middle, end) of every chunk for every kv head."""
    w = workloads.make(3, device=cuda_device)
    check(w, cuda_device, rows=_tile_rows(w))


def test_mixed_chunked_prefill_reduced_full_compare(cuda_device):
    """Same structure at reduced size, every output row compared."""
    w = workloads.build([1500, 2100, 300, 1200, 2300], [1, 1, 300, 256, 260], Hq=32, Hkv=8,
                        D=128, B=16, seed=33, device=cuda_device)
    check(w, cuda_device)


@pytest.mark.parametrize("n_req,q_len", [(103, 160), (260, 64), (300, 12)],
                         ids=["ordered", "batch-order", "listed-many-requests"])
def test_prefill_launch_orders_past_the_unit_list(cuda_device, n_req, q_len):
    """The launch orders around the unit list's capacity (1024 units): g 16
    gives 8-token tiles, so 103 chunks of 160 tokens are 1030 units (the grid
    with requests ordered by work), 260 chunks of 64 are 1040 units for more
    requests than the order holds (the grid in batch order), and 300 chunks
    of 12 are 300 one-pair units on the list (more requests than the order
    holds, so listed request ids go past 255). Prefixes vary so the
    requests' work differs; every row compared."""
    rng = np.random.default_rng(n_req)
    prefix = rng.integers(0, 300, n_req)
    w = workloads.build([int(p) + q_len for p in prefix], [q_len] * n_req, Hq=16, Hkv=1,
                        D=64, B=16, seed=n_req, device=cuda_device)
    check(w, cuda_device)


def _two_kv_heads(w):
    """Two kv heads per tile, rotating with the chunk and the tile, so every
    kv head is covered across the chunks (keeps the fp64 oracle's work on the
    32768-token contexts to a few tens of seconds)."""
    return lambda r, t: sorted({(r + t) % w.Hkv, (r + t + w.Hkv // 2) % w.Hkv})


@pytest.mark.slow
def test_long_context_bf16_config_full_size(cuda_device):
    """32 requests x 32768 tokens, B 64, 64/8 heads: 8 chunks of 2048 at the
    end of the context plus 24 decodes; every decode row and whole query
    tiles (start, diagonal middle, end) of every chunk for two kv heads."""
    w = workloads.make(5, device=cuda_device, kv_dtype="bf16")
    check(w, cuda_device, rows=_tile_rows(w, _two_kv_heads(w)))


def test_prefill_invariant_under_block_placement(cuda_device):
    w = workloads.build([600, 333], [200, 333], Hq=8, Hkv=2, D=128, B=16, seed=8,
                        device=cuda_device, pool_blocks=90)
    step = DeviceStep(w, cuda_device)
    base = step.run().clone()
    perm = torch.from_numpy(np.random.default_rng(2).permutation(w.num_blocks)).to(cuda_device)
    k2 = torch.empty_like(step.pool.k)
    v2 = torch.empty_like(step.pool.v)
    k2[perm] = step.pool.k
    v2[perm] = step.pool.v
    pool2 = pa.KVPool(k2, v2)
    g = step.gathered
    tables2 = torch.where(g >= 0, perm[g.clamp(min=0).long()].int(), g)
    out2 = torch.empty_like(base)
    pa.forward(step.q, out2, step.qsl, step.seq, w.qsl, w.seq_lens, tables2, pool2, w.scale,
               w.causal, workspace=step.ws)
    assert pa.get_error() == pa.PA_OK
    assert torch.equal(out2.view(torch.int16), base.view(torch.int16))


def test_prefill_is_deterministic(cuda_device):
    w = workloads.build([900, 500], [400, 100], Hq=16, Hkv=4, D=128, B=32, seed=10,
                        device=cuda_device)
    step = DeviceStep(w, cuda_device)
    a = step.run().clone()
    b = step.run().clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


FP8_CASES = [
    # seq_lens, q_lens, Hq, Hkv, D, B, causal
    ([200], [200], 4, 4, 128, 16, 1),
    ([300, 77], [45, 77], 8, 2, 128, 32, 1),
    ([1000], [333], 16, 2, 128, 64, 1),
    ([400], [150], 8, 4, 64, 16, 1),
    ([250, 64], [250, 64], 4, 2, 128, 16, 0),
    ([33, 1000, 17, 2048], [2, 1, 17, 600], 8, 2, 128, 16, 1),
]


@pytest.mark.parametrize("case", FP8_CASES, ids=[f"f{i}" for i in range(len(FP8_CASES))])
def test_prefill_fp8_shapes(cuda_device, case):
    """E4M3 pools: the oracle is fed the same codes (decoded, times the scales)."""
    seq, ql, Hq, Hkv, D, B, causal = case
    w = workloads.build(seq, ql, Hq, Hkv, D, B, kv_dtype="fp8", causal=causal,
                        seed=sum(seq) + 7 * Hq + causal, device=cuda_device)
    check(w, cuda_device)


@pytest.mark.parametrize("q_mult", [0.001, 4.0, 300.0])
def test_prefill_fp8_query_magnitudes(cuda_device, q_mult):
    """The f16 operand path pre-scales each query row by a power of two: tiny
    and large query magnitudes give the same accuracy."""
    w = workloads.build([700, 900], [700, 300], Hq=8, Hkv=2, D=128, B=16, kv_dtype="fp8",
                        seed=92, device=cuda_device, q_mult=q_mult)
    check(w, cuda_device)


@pytest.mark.slow
def test_long_context_fp8_config_full_size(cuda_device):
    w = workloads.make(5, device=cuda_device, kv_dtype="fp8")
    check(w, cuda_device, rows=_tile_rows(w, _two_kv_heads(w)))
