"""GPU parity of pa_forward_shared_prefix (each group's shared prefix read once
for every 64 of its (member, head) rows by warps sharing a ring of K/V
stages, private tails by one warp per task, parts merged by log-sum-exp)
against the fp64 oracle, which knows nothing of groups: it gathers every
request's blocks through its own table row."""
import numpy as np
import pytest
import torch

import workloads
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import DeviceStep, assert_attention_close, group_arrays, oracle_step

pytestmark = pytest.mark.gpu


def check(w, dev, max_splits=32, rows=None):
    step = DeviceStep(w, dev, max_splits=max_splits)
    out = step.run(cascade=True)
    assert pa.get_error() == pa.PA_OK
    ref, _, _, _ = oracle_step(w, rows=rows)
    assert_attention_close(out, ref, rows=rows, what=w.name + " (shared prefix)")
    return out, ref, step


@pytest.mark.parametrize("kv_dtype", ["fp8", "bf16"])
def test_prefix_shared_sampling_config_full(cuda_device, kv_dtype):
    """8 groups x 16 samples sharing a 2048-token prompt, private tails of
    0..512 tokens, 32/8 heads: every output row."""
    w = workloads.make(4, device=cuda_device, kv_dtype=kv_dtype)
    check(w, cuda_device)


def test_cascade_agrees_with_plain_forward(cuda_device):
    w = workloads.make(4, device=cuda_device)
    step = DeviceStep(w, cuda_device)
    a = step.run(cascade=True).clone()
    b = step.run(cascade=False).clone()
    ref, _, _, _ = oracle_step(w)
    assert_attention_close(a, ref, what="cascade")
    assert_attention_close(b, ref, what="plain")
    assert (a.float() - b.float()).abs().max().item() <= 2e-2


CASES = [
    # name, Hq, Hkv, D, B, kv_dtype, batch spec: list of ("g", prefix, tails) / ("d", seq)
    # / ("p", seq, q_len)
    ("g1_mixed", 4, 4, 128, 16, "bf16",
     [("g", 48, [1, 17, 200]), ("d", 300), ("g", 208, [5, 1, 64, 129, 33, 2]), ("p", 400, 150)]),
    ("g8_long_prefix", 16, 2, 128, 32, "bf16",
     [("g", 4096, list(range(1, 400, 10)))]),        # 40 members: 3 q tiles, several pieces
    ("g16_d64", 32, 2, 64, 64, "bf16",
     [("d", 70), ("g", 640, [1, 63, 64, 65, 300] * 4)]),
    ("g2_d64_fp8", 4, 2, 64, 16, "fp8",
     [("g", 16, [1]), ("g", 32, [3, 4]), ("d", 5), ("g", 1024, [700, 1, 2])]),
    ("g4_fp8_mixed", 32, 8, 128, 16, "fp8",
     [("p", 900, 300), ("g", 512, [7, 100, 513, 1] * 3), ("d", 1500), ("g", 2048, [9] * 17)]),
    # 40 members x 4 heads = 160 rows: three 64-row blocks per prefix piece;
    # a 1040-key prefix: pieces of 512, 512 and 16 keys
    ("g4_fp8_wide_groups", 32, 8, 128, 16, "fp8",
     [("g", 256, [3, 40, 1, 77] * 10), ("g", 1040, [1, 2, 700]), ("d", 33)]),
    ("g8_fp8_b32", 16, 2, 128, 32, "fp8",
     [("g", 3072, [1, 31, 32, 33, 600]), ("d", 4000)]),
]


def _build(case, dev, seed):
    name, Hq, Hkv, D, B, kv_dtype, spec = case
    seq, ql, groups = [], [], []
    for item in spec:
        if item[0] == "g":
            _, prefix, tails = item
            groups.append((list(range(len(seq), len(seq) + len(tails))), prefix))
            seq.extend(prefix + t for t in tails)
            ql.extend([1] * len(tails))
        elif item[0] == "d":
            seq.append(item[1])
            ql.append(1)
        else:
            seq.append(item[1])
            ql.append(item[2])
    return workloads.build(seq, ql, Hq, Hkv, D, B, kv_dtype=kv_dtype, seed=seed, device=dev,
                           groups=groups, name=name)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
@pytest.mark.parametrize("max_splits", [32, 2])
def test_shared_prefix_shapes(cuda_device, case, max_splits):
    """Groups next to ungrouped decodes and prefill chunks; tails from one key
    up; prefixes that are not a multiple of the 128-key tile; workspaces from
    roomy to the minimum of two slots per request."""
    w = _build(case, cuda_device, seed=1000 + len(case[0]) + max_splits)
    check(w, cuda_device, max_splits=max_splits)


def test_shared_prefix_without_groups_is_pa_forward(cuda_device):
    w = _build(CASES[0], cuda_device, seed=5)
    step = DeviceStep(w, cuda_device)
    a = step.run().clone()
    pa.forward_shared_prefix(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens,
                             step.gathered, step.pool, w.scale, [], [], [], causal=w.causal,
                             workspace=step.ws)
    assert pa.get_error() == pa.PA_OK
    assert torch.equal(step.out.view(torch.int16), a.view(torch.int16))


def test_shared_prefix_is_deterministic(cuda_device):
    w = _build(CASES[4], cuda_device, seed=6)
    step = DeviceStep(w, cuda_device)
    a = step.run(cascade=True).clone()
    b = step.run(cascade=True).clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_shared_prefix_flags_bad_prefix_block_without_faulting(cuda_device):
    """A prefix block id outside the pool in the first member's row sets
    PA_ERR_DEVICE_BOUNDS; the call returns and the context stays usable."""
    w = _build(CASES[0], cuda_device, seed=7)
    step = DeviceStep(w, cuda_device)
    step.run(cascade=True)
    assert pa.get_error() == pa.PA_OK
    tables = step.gathered.clone()
    tables[0, 1] = w.num_blocks + 5
    first, size, prefix_blocks = group_arrays(w)
    pa.forward_shared_prefix(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens, tables,
                             step.pool, w.scale, first, size, prefix_blocks, causal=w.causal,
                             workspace=step.ws)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert pa.get_error() == pa.PA_OK  # reading the error clears it
    step.run(cascade=True)
    assert pa.get_error() == pa.PA_OK
