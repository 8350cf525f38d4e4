"""Pins of the oracle's storage side: FP8 E4M3 codec, KV write, staged
block-table diffs, block copy, and the bytes formula used for rooflines."""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from paged_kv_cache_143_gb300 import accounting
from tests.helpers import bits, oracle_pool

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ------------------------------------------------------------------ FP8 codec

def test_e4m3_decode_matches_torch_float8_for_all_codes():
    """torch's float8_e4m3fn is an independent implementation of the OFP8 E4M3
    format: every one of the 256 codes must decode to the same value."""
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = O.e4m3_table()
    nan = np.isnan(ref)
    assert list(np.nonzero(nan)[0]) == [0x7F, 0xFF]
    assert np.isnan(got[nan]).all()
    np.testing.assert_array_equal(got[~nan], ref[~nan])


def test_e4m3_decode_spec_constants():
    assert O.e4m3_decode(0x7E) == 448.0
    assert O.e4m3_decode(0xFE) == -448.0
    assert O.e4m3_decode(0x01) == 2.0 ** -9
    assert O.e4m3_decode(0x07) == 7 * 2.0 ** -9
    assert O.e4m3_decode(0x08) == 2.0 ** -6
    assert O.e4m3_decode(0x00) == 0.0 and np.signbit(O.e4m3_decode(0x80))
    assert np.isnan(O.e4m3_decode(0x7F)) and np.isnan(O.e4m3_decode(0xFF))
    vals = O.e4m3_table()[:0x7F]
    assert np.all(np.diff(vals) > 0)  # non-negative finite codes are monotone


def test_e4m3_encode_hand_worked_ties():
    with open(os.path.join(GOLDEN, "e4m3_ties.json")) as f:
        cases = json.load(f)["cases"]
    for c in cases:
        assert O.e4m3_encode(c["x"]) == c["code"], c


def test_e4m3_encode_special_values():
    assert O.e4m3_encode(float("nan")) == 0x7F
    assert O.e4m3_encode(float("inf")) == 0x7E
    assert O.e4m3_encode(float("-inf")) == 0xFE


ALL_BF16 = np.arange(65536, dtype=np.uint32).astype(np.uint16)


@pytest.mark.parametrize("scale", [1.0, 0.37, 0.011858259])
def test_fp8_store_all_bf16_inputs_match_torch(scale):
    """The store of every bf16 bit pattern: where the fp32 quotient is within
    the E4M3 range, torch's RNE float8 conversion of the same fp32 quotient is
    an independent reference; beyond it the oracle saturates; NaN -> 0x7F."""
    got = O.fp8_store_array(ALL_BF16, scale)
    x = torch.from_numpy(ALL_BF16.view(np.int16)).view(torch.bfloat16).float()
    qv = x / torch.tensor(np.float32(scale))
    finite = torch.isfinite(qv)
    inrange = finite & (qv.abs() <= 448.0)
    ref = qv[inrange].to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    np.testing.assert_array_equal(got[inrange.numpy()], ref)
    over = (~inrange & ~torch.isnan(qv)).numpy()
    neg = (qv < 0).numpy()
    assert np.all(got[over & neg] == 0xFE) and np.all(got[over & ~neg] == 0x7E)
    assert np.all(got[torch.isnan(qv).numpy()] == 0x7F)


# ------------------------------------------------------------------ KV write

def _tiny_pool(dtype=O.BF16, nb=3, Hkv=2, B=2, D=2):
    dt = np.uint16 if dtype == O.BF16 else np.uint8
    fill = 0x7FC0 if dtype == O.BF16 else 0x7F
    return O.Pool(np.full((nb, Hkv, B, D), fill, dt), np.full((nb, Hkv, B, D), fill, dt), B,
                  dtype, 0.5, 0.25)


def test_write_kv_hand_example():
    """Slot s = block * B + offset ([vLLM-wiki "블록 테이블"]); layout
    [num_blocks][Hkv][B][D]; negative slots skipped; other cells untouched."""
    p = _tiny_pool()
    T, Hkv, D = 3, 2, 2
    k = np.arange(1, T * Hkv * D + 1, dtype=np.uint16).reshape(T, Hkv, D)
    v = k + 100
    before = p.copy()
    O.write_kv(p, k, v, np.array([5, -1, 0], np.int64))
    # token 0 -> slot 5 = block 2, offset 1; token 2 -> slot 0 = block 0, offset 0
    expect_k = before.k.copy()
    expect_v = before.v.copy()
    for h in range(Hkv):
        expect_k[2, h, 1, :] = k[0, h]
        expect_v[2, h, 1, :] = v[0, h]
        expect_k[0, h, 0, :] = k[2, h]
        expect_v[0, h, 0, :] = v[2, h]
    np.testing.assert_array_equal(p.k, expect_k)
    np.testing.assert_array_equal(p.v, expect_v)


def test_write_kv_fp8_uses_per_tensor_scales():
    p = _tiny_pool(O.FP8_E4M3)
    k = torch.tensor([[[1.0, -3.0]], [[0.1, 1000.0]]]).repeat(1, 2, 1).to(torch.bfloat16)
    v = -k
    O.write_kv(p, bits(k), bits(v), np.array([1, 4], np.int64))
    kb = bits(k)
    for t, s in enumerate([1, 4]):
        blk, off = divmod(s, 2)
        for h in range(2):
            for d in range(2):
                assert p.k[blk, h, off, d] == O.fp8_store(kb[t, h, d], 0.5)
                assert p.v[blk, h, off, d] == O.fp8_store(bits(v)[t, h, d], 0.25)
    assert p.k[2, 0, 0, 1] == 0x7E  # 1000 / 0.5 saturates to 448


def test_write_kv_rejects_out_of_range_slot():
    p = _tiny_pool()
    k = np.zeros((1, 2, 2), np.uint16)
    with pytest.raises(O.OracleError):
        O.write_kv(p, k, k, np.array([6], np.int64))


def test_workload_cache_holds_every_token_at_its_position():
    w = workloads.build([20, 35], [3, 1], Hq=2, Hkv=2, D=8, B=16, seed=2, pool_blocks=9)
    p = oracle_pool(w)
    for r in range(w.R):
        for n in range(int(w.seq_lens[r])):
            blk = w.tables[r, n // w.B]
            sel = np.nonzero((w.ctx_req == r) & (w.ctx_pos == n))[0]
            if sel.size:
                want = bits(w.ctx_k[sel[0]])
            else:
                t = int(w.qsl[r]) + n - (int(w.seq_lens[r]) - int(w.qsl[r + 1] - w.qsl[r]))
                want = bits(w.new_k[t])
            np.testing.assert_array_equal(p.k[blk, :, n % w.B, :], want)
    used = np.zeros(p.k.shape[:1] + p.k.shape[2:3], bool)
    for r in range(w.R):
        for n in range(int(w.seq_lens[r])):
            used[w.tables[r, n // w.B], n % w.B] = True
    assert np.all(p.k.transpose(0, 2, 1, 3)[~used] == 0x7FC0)


# ------------------------------------------------------------ staged writes

def test_staged_writes_hand_example_last_writer_wins():
    """[MRV2 "재설계 3"]: (row, start, values) diffs applied in record order."""
    table = np.arange(15, dtype=np.int32).reshape(3, 5)
    rows = [1, 1, 0]
    starts = [0, 2, 4]
    offs = [0, 3, 5, 6]
    vals = [70, 80, 90, 40, 50, 11]
    g = O.apply_staged_writes(table, rows, starts, offs, vals, [1, 0, 1])
    want = np.array([[0, 1, 2, 3, 11], [70, 80, 40, 50, 9], [10, 11, 12, 13, 14]], np.int32)
    np.testing.assert_array_equal(table, want)
    np.testing.assert_array_equal(g, want[[1, 0, 1]])


def test_staged_writes_match_cell_dictionary_model():
    rng = np.random.default_rng(7)
    for trial in range(20):
        mr, mb = int(rng.integers(1, 9)), int(rng.integers(1, 12))
        table = rng.integers(-5, 100, size=(mr, mb)).astype(np.int32)
        cells = {(i, j): int(table[i, j]) for i in range(mr) for j in range(mb)}
        W = int(rng.integers(0, 10))
        rows, starts, offs, vals = [], [], [0], []
        for _ in range(W):
            r = int(rng.integers(0, mr))
            s = int(rng.integers(0, mb))
            n = int(rng.integers(0, mb - s + 1))
            vv = [int(x) for x in rng.integers(0, 1000, size=n)]
            rows.append(r)
            starts.append(s)
            vals.extend(vv)
            offs.append(len(vals))
            for k, x in enumerate(vv):
                cells[(r, s + k)] = x
        idx = [int(x) for x in rng.integers(0, mr, size=int(rng.integers(0, 6)))]
        g = O.apply_staged_writes(table, rows, starts, offs, vals, idx)
        want = np.array([[cells[(i, j)] for j in range(mb)] for i in range(mr)], np.int32)
        np.testing.assert_array_equal(table, want)
        np.testing.assert_array_equal(g.reshape(len(idx), mb), want[idx].reshape(len(idx), mb))


@pytest.mark.parametrize("cfg", [1, 3, 4])
def test_staged_writes_rebuild_the_workload_tables(cfg):
    w = workloads.make(cfg, num_requests=None if cfg == 1 else 16)
    table = w.table_before.copy()
    g = O.apply_staged_writes(table, w.diff_rows, w.diff_starts, w.diff_val_offsets,
                              w.diff_vals, w.idx_mapping)
    np.testing.assert_array_equal(g, w.tables)


def test_staged_writes_reject_out_of_range():
    table = np.zeros((2, 3), np.int32)
    with pytest.raises(O.OracleError):
        O.apply_staged_writes(table, [0], [2], [0, 2], [1, 2], [])
    with pytest.raises(O.OracleError):
        O.apply_staged_writes(table, [], [], [0], [], [2])


# ---------------------------------------------------------------- block copy

def test_copy_blocks_copies_every_head_and_offset():
    p = _tiny_pool(nb=4)
    p.k[:] = np.arange(p.k.size, dtype=np.uint16).reshape(p.k.shape)
    p.v[:] = p.k + 1000
    before = p.copy()
    O.copy_blocks(p, [1, 0], [3, 2])
    np.testing.assert_array_equal(p.k[3], before.k[1])
    np.testing.assert_array_equal(p.k[2], before.k[0])
    np.testing.assert_array_equal(p.v[3], before.v[1])
    np.testing.assert_array_equal(p.k[:2], before.k[:2])


# ------------------------------------------------------------- accounting

def test_kv_bytes_formula_reproduces_opt13b_example():
    with open(os.path.join(GOLDEN, "opt13b_kv_bytes.json")) as f:
        g = json.load(f)
    # hidden width 5120 = 40 heads x 128; MHA so kv heads = heads
    per_token = accounting.kv_bytes_per_token(40, 128, g["bytes_per_element"], g["layers"])
    assert per_token == g["kv_bytes_per_token"] == g["kv_bytes_per_token_kib"] * 1024
    assert abs(per_token * g["tokens"] / 1e9 - g["request_bytes_gb_approx"]) < 0.1


def test_causal_pairs_closed_form():
    for q_len, seq in [(1, 1), (1, 100), (4, 4), (1024, 1024), (1920, 10112), (5, 9)]:
        brute = sum(seq - q_len + j + 1 for j in range(q_len))
        assert accounting.causal_pairs(q_len, seq) == brute
    # the prefill chunks of the mixed config
    assert (accounting.causal_pairs(1024, 1024) + accounting.causal_pairs(1024, 3072)
            + accounting.causal_pairs(1920, 10112)) == 524800 + 2621952 + 17572800


def test_unique_bytes_count_shared_blocks_once():
    tables = np.array([[0, 1, 2], [0, 1, 3]], np.int32)
    b = accounting.unique_kv_bytes(tables, [40, 33], 16, 1, 1, 1)
    # blocks 0,1 full (32 slots), block 2 holds 8, block 3 holds 1
    assert b == 2 * (32 + 8 + 1)
