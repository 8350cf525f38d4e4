"""GPU parity for GQA group widths g = Hq / Hkv outside the powers of two
(and above 16) against the fp64 oracle, through the C ABI: decode (rows of
the 16-row MMA tile past g are padding; g > 16 takes several CTAs per kv
head), prefill chunks (a 128-row tile holds 128 // g whole tokens of g
heads) and shared-prefix groups. The oracle maps query head h to kv head
h // g for any g."""
import pytest

import workloads
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import DeviceStep, assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu


def check(w, dev, max_splits=32, cascade=False):
    step = DeviceStep(w, dev, max_splits=max_splits)
    out = step.run(cascade=cascade)
    assert pa.get_error() == pa.PA_OK
    ref, _, _, _ = oracle_step(w)
    return assert_attention_close(out, ref, what=w.name)


DECODE = [
    # seq_lens, Hq, Hkv, D, B, dtype
    ([300, 1000, 45, 2000], 6, 2, 128, 16, "bf16"),   # g 3
    ([300, 1000, 45], 12, 2, 128, 16, "fp8"),         # g 6
    ([17, 1000, 2500], 10, 2, 64, 32, "fp8"),         # g 5, D 64
    ([300, 1000, 45], 24, 2, 128, 32, "bf16"),        # g 12
    ([300, 1000, 45], 64, 2, 128, 16, "fp8"),         # g 32: two CTAs of 16 heads
    ([300, 777], 48, 1, 64, 16, "bf16"),              # g 48 (one kv head): three CTAs
    ([129, 4000], 40, 2, 128, 64, "bf16"),            # g 20: 16 + 4 heads
]


@pytest.mark.parametrize("case", DECODE, ids=[f"g{c[1] // c[2]}_{c[5]}" for c in DECODE])
@pytest.mark.parametrize("max_splits", [0, 8])
def test_decode_gqa_widths(cuda_device, case, max_splits):
    seq, Hq, Hkv, D, B, dt = case
    w = workloads.build(seq, [1] * len(seq), Hq, Hkv, D, B, kv_dtype=dt,
                        seed=sum(seq) + Hq + max_splits, device=cuda_device)
    check(w, cuda_device, max_splits=max_splits)


PREFILL = [
    # seq_lens, q_lens, Hq, Hkv, D, B, dtype, causal
    ([500, 300], [200, 1], 6, 2, 128, 16, "bf16", 1),     # g 3: 42 tokens per tile
    ([500, 300], [200, 1], 6, 2, 128, 16, "fp8", 1),
    ([700], [333], 24, 2, 128, 64, "bf16", 1),            # g 12: 10 tokens per tile
    ([700], [333], 24, 2, 128, 64, "fp8", 1),
    ([400, 90], [150, 1], 20, 4, 64, 16, "bf16", 1),      # g 5, D 64
    ([400, 90], [150, 1], 20, 4, 64, 16, "fp8", 1),
    ([600, 100], [130, 1], 64, 2, 128, 16, "bf16", 1),    # g 32: 4 tokens per tile
    ([600], [130], 96, 1, 128, 32, "fp8", 1),             # g 96: 1 token per tile
    ([250, 64], [250, 64], 6, 2, 128, 16, "bf16", 0),     # g 3, non-causal
    ([2100, 77], [1000, 77], 36, 4, 128, 16, "bf16", 1),  # g 9: 14 tokens per tile
]


@pytest.mark.parametrize("case", PREFILL,
                         ids=[f"g{c[2] // c[3]}_d{c[4]}_{c[6]}_c{c[7]}" for c in PREFILL])
def test_prefill_gqa_widths(cuda_device, case):
    seq, ql, Hq, Hkv, D, B, dt, causal = case
    w = workloads.build(seq, ql, Hq, Hkv, D, B, kv_dtype=dt, causal=causal,
                        seed=sum(seq) + 3 * Hq + causal, device=cuda_device)
    check(w, cuda_device)


SHARED = [
    # Hq, Hkv, D, B, dtype, prefix, tails
    (6, 2, 128, 16, "fp8", 512, [1, 40, 300, 7, 129]),              # g 3
    (12, 2, 128, 32, "bf16", 1024, [3, 1, 77] * 4),                 # g 6
    (24, 2, 64, 16, "fp8", 256, [9, 100, 1, 250, 64]),              # g 12, D 64
    (64, 2, 128, 16, "bf16", 2048, [5, 33, 129, 1]),                # g 32
]


@pytest.mark.parametrize("case", SHARED, ids=[f"g{c[0] // c[1]}_{c[4]}" for c in SHARED])
def test_shared_prefix_gqa_widths(cuda_device, case):
    Hq, Hkv, D, B, dt, prefix, tails = case
    n = len(tails)
    w = workloads.build([900] + [prefix + t for t in tails], [1] * (n + 1), Hq, Hkv, D, B,
                        kv_dtype=dt, seed=prefix + Hq, device=cuda_device,
                        groups=[(list(range(1, n + 1)), prefix)])
    check(w, cuda_device, cascade=True)
