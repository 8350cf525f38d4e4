"""Shared test plumbing: moving workload inputs into the oracle's numpy form and
an independent dense (contiguous) restatement used to pin the oracle."""
import numpy as np
import torch

from oracle import oracle as O


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 (uint16) or uint8 tensor as a numpy array."""
    t = t.detach().contiguous().cpu()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.uint8:
        return t.numpy()
    raise TypeError(t.dtype)


def empty_oracle_pool(w) -> "O.Pool":
    dt = np.uint16 if w.kv_dtype == "bf16" else np.uint8
    fill = w.pool_nan_fill()
    k = np.full(w.pool_shape(), fill, dt)
    v = np.full(w.pool_shape(), fill, dt)
    return O.Pool(k, v, w.B, O.BF16 if w.kv_dtype == "bf16" else O.FP8_E4M3, w.k_scale,
                  w.v_scale)


def oracle_pool(w, include_new=True) -> "O.Pool":
    """The pool as the oracle stores it: context tokens, then the step's tokens."""
    p = empty_oracle_pool(w)
    O.write_kv(p, bits(w.ctx_k), bits(w.ctx_v), w.ctx_slots.cpu().numpy())
    if include_new:
        O.write_kv(p, bits(w.new_k), bits(w.new_v), w.slot_mapping.cpu().numpy())
    return p


def _as_f64(t: torch.Tensor, kv_dtype: str, scale: float) -> np.ndarray:
    """Token values as the cache represents them, computed WITHOUT the oracle:
    bf16 widened exactly; FP8 through torch's own float8_e4m3fn conversion of
    the fp32 quotient (valid because |x / scale| <= 448 by construction of the
    per-tensor scales), times the scale in fp64."""
    x = t.detach().cpu().float()
    if kv_dtype == "bf16":
        return x.double().numpy()
    s = np.float32(scale)
    qv = (x / torch.tensor(s)).to(torch.float8_e4m3fn).to(torch.float64)
    return qv.numpy() * float(s)


def dense_kv(w, r):
    """(K, V) of request r as fp64 [seq_len][Hkv][D] in logical order, assembled
    from the generated token values (not from any pool)."""
    seq = int(w.seq_lens[r])
    ql = int(w.qsl[r + 1] - w.qsl[r])
    P = seq - ql
    K = np.full((seq, w.Hkv, w.D), np.nan)
    V = np.full((seq, w.Hkv, w.D), np.nan)
    sel = np.nonzero(w.ctx_req == r)[0]
    for members in w.groups:
        if r in members and r != min(members):
            first = min(members)
            shared = np.nonzero(w.ctx_req == first)[0]
            own_start = int(w.ctx_pos[sel].min()) if sel.size else P
            shared = shared[w.ctx_pos[shared] < own_start]
            sel = np.concatenate([shared, sel])
    if sel.size:
        idx = torch.from_numpy(sel).to(w.ctx_k.device)
        K[w.ctx_pos[sel]] = _as_f64(w.ctx_k.index_select(0, idx), w.kv_dtype, w.k_scale)
        V[w.ctx_pos[sel]] = _as_f64(w.ctx_v.index_select(0, idx), w.kv_dtype, w.v_scale)
    a, b = int(w.qsl[r]), int(w.qsl[r + 1])
    K[P:seq] = _as_f64(w.new_k[a:b], w.kv_dtype, w.k_scale)
    V[P:seq] = _as_f64(w.new_v[a:b], w.kv_dtype, w.v_scale)
    return K, V


def dense_attention(w, causal=None):
    """fp64 ordinary attention on contiguous per-request K/V (numpy only)."""
    causal = w.causal if causal is None else causal
    q = w.q.detach().cpu().double().numpy()
    out = np.full(q.shape, np.nan)
    g = w.Hq // w.Hkv
    for r in range(w.R):
        a, b = int(w.qsl[r]), int(w.qsl[r + 1])
        if b == a:
            continue
        K, V = dense_kv(w, r)
        seq = K.shape[0]
        P = seq - (b - a)
        Kh = np.repeat(K, g, axis=1)  # [seq][Hq][D]
        Vh = np.repeat(V, g, axis=1)
        s = w.scale * np.einsum("thd,nhd->thn", q[a:b], Kh)
        pos = P + np.arange(b - a)
        if causal:
            mask = np.arange(seq)[None, :] > pos[:, None]
            s = np.where(mask[:, None, :], -np.inf, s)
        s = s - s.max(axis=-1, keepdims=True)
        e = np.exp(s)
        out[a:b] = np.einsum("thn,nhd->thd", e / e.sum(axis=-1, keepdims=True), Vh)
    return out
