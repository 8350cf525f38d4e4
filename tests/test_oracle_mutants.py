"""Sensitivity of the oracle's pins: each test compiles a copy of the oracle
source with one plausible mistake planted in it (on the CPU, in a temporary
directory) and checks that at least one pin fails against the mutant."""
import os
import subprocess

import pytest

from oracle import build as oracle_build
from oracle import oracle as O
from tests import test_oracle_attention as A
from tests import test_oracle_storage as S

MUTANTS = {
    # name: (original text, planted mistake, pins expected to catch it)
    "causal-mask-off-by-one": (
        "int32_t n_visible = causal ? p + 1 : seq_lens[r];",
        "int32_t n_visible = causal ? p : seq_lens[r];",
        [lambda: A.test_oracle_matches_dense_attention(A.CASES[1])]),
    "gqa-head-map": (
        "v_scale, h / g, scale, s);",
        "v_scale, h % Hkv, scale, s);",
        [lambda: A.test_oracle_matches_dense_attention(A.CASES[1])]),
    "dropped-scale": (
        "s[n] = scale * dot;",
        "s[n] = dot;",
        [lambda: A.test_oracle_matches_dense_attention(A.CASES[0])]),
    "transposed-pool-layout": (
        "return ((blk * Hkv + h) * B + t) * D + d;",
        "return ((blk * B + t) * Hkv + h) * D + d;",
        [S.test_write_kv_hand_example]),
    "ties-to-odd": (
        "code = (lo & 1) ? hi : lo;",
        "code = (lo & 1) ? lo : hi;",
        [S.test_e4m3_encode_hand_worked_ties]),
    "diffs-in-reverse-order": (
        "for (int32_t w = 0; w < W; ++w) {",
        "for (int32_t w = W - 1; w >= 0; --w) {",
        [S.test_staged_writes_hand_example_last_writer_wins]),
    "subnormal-exponent": (
        "v = ldexp((double)m / 8.0, 1 - 7);",
        "v = ldexp((double)m / 8.0, -7);",
        [S.test_e4m3_decode_matches_torch_float8_for_all_codes]),
    "softmax-over-one-block": (
        "double denom = 0.0;\n  for (int32_t n = 0; n < n_visible; ++n) {",
        "double denom = 0.0;\n  for (int32_t n = (n_visible - 1) / B * B; n < n_visible; ++n) {",
        [lambda: A.test_oracle_matches_dense_attention(A.CASES[0])]),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_planted_mistake_is_caught(name, tmp_path):
    orig, planted, pins = MUTANTS[name]
    src = open(oracle_build.SRC).read()
    assert src.count(orig) == 1, f"mutation site for {name} not found"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(orig, planted))
    lib = str(tmp_path / "libmutant.so")
    subprocess.run(["gcc", "-O1", "-std=c11", "-fPIC", "-shared", "-fopenmp",
                    "-ffp-contract=off", "-o", lib, str(path), "-lm"], check=True)
    caught = 0
    with O.use_library(lib):
        for pin in pins:
            try:
                pin()
            except (AssertionError, O.OracleError):
                caught += 1
    assert caught > 0, f"no pin caught the planted mistake {name}"
