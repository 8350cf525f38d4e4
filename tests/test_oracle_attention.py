"""Pins of the oracle's attention against things other than itself.

- an independent dense restatement (numpy einsum + masked softmax over the
  generated token values in logical order, FP8 via torch's own float8 type);
- a literal per-block transcription of the blockwise equation of
  [vLLM-wiki "블록 단위 어텐션 계산"] on tiny inputs (block sizes 1, 2, 16);
- closed forms (constant V, zero query, a single key, a dominant key,
  non-causal first query);
- invariance under physical block placement and under sharing vs copying
  prefix blocks ([vLLM-wiki "블록 테이블", "블록 공유와 쓰기 시 복사"]).
"""
import math

import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from tests.helpers import bits, dense_attention, oracle_pool


def run_oracle(w, pool=None, rows=None, tables=None):
    pool = oracle_pool(w) if pool is None else pool
    return O.paged_attention(bits(w.q), w.qsl, w.seq_lens,
                             w.tables if tables is None else tables, pool, w.scale, w.causal,
                             rows=rows)


CASES = [
    # seq_lens, q_lens, Hq, Hkv, D, B, dtype, causal
    ([17, 33, 64, 100], [1, 1, 1, 1], 4, 4, 64, 16, "bf16", 1),
    ([5, 40, 23], [5, 7, 1], 4, 2, 16, 4, "bf16", 1),
    ([5, 40, 23], [5, 7, 1], 4, 2, 16, 4, "bf16", 0),
    ([31, 9, 64, 1], [1, 9, 16, 1], 8, 2, 32, 16, "fp8", 1),
    ([70, 70], [35, 0], 6, 3, 64, 32, "bf16", 1),
]


@pytest.mark.parametrize("case", CASES)
def test_oracle_matches_dense_attention(case):
    seq, ql, Hq, Hkv, D, B, dt, causal = case
    w = workloads.build(seq, ql, Hq, Hkv, D, B, kv_dtype=dt, causal=causal, seed=11,
                        pool_blocks=None)
    got = run_oracle(w)
    want = dense_attention(w)
    rows = np.repeat(np.diff(w.qsl) > 0, np.diff(w.qsl))
    assert np.isfinite(got).all() and np.isfinite(want).all()
    assert rows.sum() == w.T
    np.testing.assert_allclose(got, want, rtol=0, atol=1e-12)


def literal_blockwise(q, K, V, B, scale, p):
    """Direct transcription of the blockwise equation for one query at 0-based
    position p (keys 0..p visible): block j holds keys jB..jB+B-1; the
    numerator of A_ij is exp(scale q.K_j) over the visible keys of block j, the
    denominator sums exp over every visible key of every block up to the
    query's own; o = sum_j V_j A_ij^T. No max subtraction (tiny inputs)."""
    nblocks = p // B + 1
    denom = 0.0
    for t in range(nblocks):
        for k in range(t * B, min((t + 1) * B, p + 1)):
            denom += math.exp(scale * sum(q[d] * K[k][d] for d in range(len(q))))
    o = [0.0] * len(q)
    for j in range(nblocks):
        for k in range(j * B, min((j + 1) * B, p + 1)):
            a = math.exp(scale * sum(q[d] * K[k][d] for d in range(len(q)))) / denom
            for d in range(len(q)):
                o[d] += V[k][d] * a
    return o


@pytest.mark.parametrize("B", [1, 2, 16])
def test_oracle_matches_literal_blockwise_equation(B):
    rng = np.random.default_rng(B)
    seq = [int(x) for x in rng.integers(1, 40, size=3)]
    ql = [min(s, int(x)) for s, x in zip(seq, rng.integers(1, 6, size=3))]
    w = workloads.build(seq, ql, Hq=2, Hkv=1, D=8, B=B, seed=100 + B, pool_blocks=None)
    got = run_oracle(w)
    from tests.helpers import dense_kv
    q = w.q.double().numpy()
    for r in range(w.R):
        K, V = dense_kv(w, r)
        P = seq[r] - ql[r]
        for j in range(ql[r]):
            t = int(w.qsl[r]) + j
            for h in range(2):
                want = literal_blockwise(list(q[t, h]), K[:, 0].tolist(), V[:, 0].tolist(), B,
                                         w.scale, P + j)
                np.testing.assert_allclose(got[t, h], want, rtol=1e-12, atol=1e-14)


def _single_request(seq_len, q_len, D=16, B=16, causal=1, seed=5, Hq=1):
    return workloads.build([seq_len], [q_len], Hq=Hq, Hkv=1, D=D, B=B, causal=causal,
                           seed=seed)


def _set_bf16(t, values):
    t.copy_(torch.as_tensor(values, dtype=torch.float32).to(torch.bfloat16))


def test_closed_form_constant_v():
    w = _single_request(50, 3)
    c = torch.linspace(-2, 2, w.D)
    _set_bf16(w.ctx_v, c.expand_as(w.ctx_v))
    _set_bf16(w.new_v, c.expand_as(w.new_v))
    got = run_oracle(w)
    want = c.to(torch.bfloat16).double().numpy()
    np.testing.assert_allclose(got[:, 0], np.broadcast_to(want, got[:, 0].shape), atol=1e-13)


def test_closed_form_zero_query_is_mean_of_visible_v():
    w = _single_request(37, 4, B=4)
    w.q.zero_()
    got = run_oracle(w)
    from tests.helpers import dense_kv
    _, V = dense_kv(w, 0)
    for j in range(4):
        p = 33 + j
        np.testing.assert_allclose(got[j, 0], V[:p + 1, 0].mean(axis=0), atol=1e-13)


def test_closed_form_single_key():
    w = _single_request(1, 1)
    got = run_oracle(w)
    want = w.new_v[0, 0].double().numpy()
    np.testing.assert_array_equal(got[0, 0], want)


def test_closed_form_dominant_key():
    w = _single_request(64, 1, D=16)
    qv = w.q[0, 0].float()
    # key 20 aligned with q and 100x larger: its weight is ~1
    idx = int(np.nonzero(w.ctx_pos == 20)[0][0])
    _set_bf16(w.ctx_k[idx, 0], 100.0 * qv / qv.norm())
    got = run_oracle(w)
    want = w.ctx_v[idx, 0].double().numpy()
    np.testing.assert_allclose(got[0, 0], want, atol=1e-6)


def test_closed_form_noncausal_first_query_sees_all_keys():
    w = _single_request(24, 24, causal=0, B=8)
    w.q.zero_()
    got = run_oracle(w)
    V = w.new_v[:, 0].double().numpy()
    np.testing.assert_allclose(got[0, 0], V.mean(axis=0), atol=1e-13)
    w.causal = 1
    got_c = run_oracle(w)
    np.testing.assert_array_equal(got_c[0, 0], V[0])  # causal: key 0 only


@pytest.mark.parametrize("dt", ["bf16", "fp8"])
def test_oracle_invariant_under_block_permutation(dt):
    w = workloads.build([45, 16, 100, 3], [1, 16, 5, 3], Hq=4, Hkv=2, D=32, B=16,
                        kv_dtype=dt, seed=21, pool_blocks=20)
    base = run_oracle(w)
    pool = oracle_pool(w)
    rng = np.random.default_rng(3)
    perm = rng.permutation(w.num_blocks)  # block b moves to perm[b]
    moved = pool.copy()
    moved.k[perm] = pool.k
    moved.v[perm] = pool.v
    tables = np.where(w.tables >= 0, perm[np.maximum(w.tables, 0)], -1).astype(np.int32)
    got = run_oracle(w, pool=moved, tables=tables)
    np.testing.assert_array_equal(got, base)


def test_oracle_sharing_equals_duplication():
    """Prefix blocks referenced by several requests give the same result as
    private copies of the same values."""
    members = list(range(4))
    w = workloads.build([40, 33, 34, 47], [1, 1, 1, 1], Hq=4, Hkv=2, D=16, B=16,
                        kv_dtype="fp8", seed=9, groups=[(members, 32)])
    shared = run_oracle(w)
    pool = oracle_pool(w)
    # duplicate the 2 shared blocks for requests 1..3 into fresh blocks
    nb = w.num_blocks + 3 * 2
    k = np.concatenate([pool.k, np.zeros((6,) + pool.k.shape[1:], pool.k.dtype)])
    v = np.concatenate([pool.v, np.zeros((6,) + pool.v.shape[1:], pool.v.dtype)])
    tables = w.tables.copy()
    nxt = w.num_blocks
    for r in (1, 2, 3):
        for i in range(2):
            b = tables[r, i]
            k[nxt], v[nxt] = pool.k[b], pool.v[b]
            tables[r, i] = nxt
            nxt += 1
    assert nxt == nb
    dup = O.Pool(k, v, w.B, pool.dtype, pool.k_scale, pool.v_scale)
    assert len(set(tables[:, :2].ravel())) == 8
    got = run_oracle(w, pool=dup, tables=tables)
    np.testing.assert_array_equal(got, shared)


def test_oracle_rows_subset_matches_full():
    w = workloads.build([100, 20], [10, 1], Hq=4, Hkv=2, D=16, B=16, seed=4)
    full = run_oracle(w)
    rows = np.array([0, 5, 17, 39, 43], np.int64)
    part = run_oracle(w, rows=rows)
    flat_full = full.reshape(-1, w.D)
    flat_part = part.reshape(-1, w.D)
    np.testing.assert_array_equal(flat_part[rows], flat_full[rows])
    others = np.setdiff1d(np.arange(flat_part.shape[0]), rows)
    assert np.isnan(flat_part[others]).all()


def test_oracle_rejects_bad_inputs():
    w = workloads.build([20], [1], Hq=2, Hkv=1, D=16, B=16, seed=1)
    bad = w.tables.copy()
    bad[0, 1] = w.num_blocks + 5
    with pytest.raises(O.OracleError):
        run_oracle(w, tables=bad)
    with pytest.raises(O.OracleError):
        O.paged_attention(bits(w.q), np.array([0, 1], np.int32), np.array([40], np.int32),
                          w.tables, oracle_pool(w), w.scale, 1)


def test_config1_poison_never_read():
    """Config 1 leaves NaN in unused cells; a finite output shows none was read."""
    w = workloads.make(1)
    got = run_oracle(w)
    assert np.isfinite(got).all()
    np.testing.assert_allclose(got, dense_attention(w), atol=1e-12)
