"""numpy front end of the C oracle (``oracle.c``).

TEST INFRASTRUCTURE ONLY: used by the tests, the smoke check and the CPU
baseline of the benchmark. It never touches the GPU and never imports the
product package. Arrays are numpy; bf16 values travel as their uint16 bit
patterns, FP8 values as uint8 E4M3 codes.
"""
import contextlib
import ctypes

import numpy as np

from . import build as _build

BF16 = 0
FP8_E4M3 = 1

_lib = None


def _bind(L):
    P, I32, I64, F32, F64 = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64,
                             ctypes.c_float, ctypes.c_double)
    L.oracle_e4m3_decode.restype = F64
    L.oracle_e4m3_decode.argtypes = [ctypes.c_uint8]
    L.oracle_e4m3_encode.restype = ctypes.c_uint8
    L.oracle_e4m3_encode.argtypes = [F32]
    L.oracle_fp8_store.restype = ctypes.c_uint8
    L.oracle_fp8_store.argtypes = [ctypes.c_uint16, F32]
    L.oracle_write_kv.restype = ctypes.c_int
    L.oracle_write_kv.argtypes = [P, P, I32, I32, I32, I32, I32, F32, F32, P, P, P, I32]
    L.oracle_copy_blocks.restype = ctypes.c_int
    L.oracle_copy_blocks.argtypes = [P, P, I32, I32, I32, I32, I32, P, P, I32]
    L.oracle_apply_staged_writes.restype = ctypes.c_int
    L.oracle_apply_staged_writes.argtypes = [P, I32, I32, P, P, P, P, I32, P, I32, P]
    L.oracle_paged_attention.restype = ctypes.c_int
    L.oracle_paged_attention.argtypes = [P, P, P, P, P, I32, I32, I32, I32, P, P, I32, I32,
                                         I32, I32, I32, F64, F64, F64, I32, P, I64, I32]
    L.oracle_max_threads.restype = ctypes.c_int
    L.oracle_max_threads.argtypes = []
    return L


def lib():
    global _lib
    if _lib is None:
        _lib = _bind(ctypes.CDLL(_build.build()))
    return _lib


@contextlib.contextmanager
def use_library(path):
    """Temporarily route every call to another build of the oracle source
    (the tests use it to check that planted mistakes are caught)."""
    global _lib
    old = _lib
    _lib = _bind(ctypes.CDLL(path))
    try:
        yield
    finally:
        _lib = old


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


class OracleError(RuntimeError):
    pass


def _check(rc, what):
    if rc == 1:
        raise OracleError(f"{what}: invalid arguments")
    if rc == 2:
        raise OracleError(f"{what}: index out of range")


# ------------------------------------------------------------------ numbers

def e4m3_decode(code: int) -> float:
    return lib().oracle_e4m3_decode(int(code) & 0xFF)


def e4m3_encode(x: float) -> int:
    return int(lib().oracle_e4m3_encode(float(np.float32(x))))


def fp8_store(bf16_bits: int, scale: float) -> int:
    return int(lib().oracle_fp8_store(int(bf16_bits) & 0xFFFF, float(np.float32(scale))))


def fp8_store_array(bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    """Element-wise FP8 store of an array of bf16 bit patterns (via a 1-token write)."""
    bits = _c(bf16_bits, np.uint16).reshape(-1)
    n = bits.size
    out_k = np.zeros(n, np.uint8)
    out_v = np.zeros(n, np.uint8)
    slots = np.zeros(1, np.int64)
    # one token, one head, D = n, B = 1, one block
    rc = lib().oracle_write_kv(_ptr(out_k), _ptr(out_v), 1, 1, 1, n, FP8_E4M3,
                               float(np.float32(scale)), float(np.float32(scale)),
                               _ptr(bits), _ptr(bits), _ptr(slots), 1)
    _check(rc, "fp8_store_array")
    return out_k


# ------------------------------------------------------------------ pool ops

class Pool:
    """Host copy of a KV pool laid out [num_blocks][Hkv][B][D] (K and V)."""

    def __init__(self, k, v, block_size, dtype, k_scale=1.0, v_scale=1.0):
        self.k = np.ascontiguousarray(k)
        self.v = np.ascontiguousarray(v)
        self.num_blocks, self.Hkv, self.B, self.D = self.k.shape
        assert self.B == block_size and self.v.shape == self.k.shape
        self.dtype = dtype
        want = np.uint16 if dtype == BF16 else np.uint8
        assert self.k.dtype == want and self.v.dtype == want
        self.k_scale = float(np.float32(k_scale))
        self.v_scale = float(np.float32(v_scale))

    def copy(self):
        return Pool(self.k.copy(), self.v.copy(), self.B, self.dtype, self.k_scale, self.v_scale)


def write_kv(pool: Pool, k_new, v_new, slot_mapping):
    k_new = _c(k_new, np.uint16)
    v_new = _c(v_new, np.uint16)
    slots = _c(slot_mapping, np.int64)
    T = slots.size
    assert k_new.size == T * pool.Hkv * pool.D and v_new.size == k_new.size
    rc = lib().oracle_write_kv(_ptr(pool.k), _ptr(pool.v), pool.num_blocks, pool.B, pool.Hkv,
                               pool.D, pool.dtype, pool.k_scale, pool.v_scale, _ptr(k_new),
                               _ptr(v_new), _ptr(slots), T)
    _check(rc, "write_kv")


def copy_blocks(pool: Pool, src, dst):
    src = _c(src, np.int32)
    dst = _c(dst, np.int32)
    rc = lib().oracle_copy_blocks(_ptr(pool.k), _ptr(pool.v), pool.num_blocks, pool.B, pool.Hkv,
                                  pool.D, pool.dtype, _ptr(src), _ptr(dst), src.size)
    _check(rc, "copy_blocks")


def apply_staged_writes(table, rows, starts, val_offsets, vals, idx_mapping):
    """Applies the diffs to ``table`` in place and returns the gathered rows."""
    assert table.dtype == np.int32 and table.flags.c_contiguous
    max_reqs, max_blocks = table.shape
    rows = _c(rows, np.int32)
    starts = _c(starts, np.int32)
    val_offsets = _c(val_offsets, np.int32)
    vals = _c(vals, np.int32) if len(vals) else np.zeros(1, np.int32)
    idx = _c(idx_mapping, np.int32)
    W, R = rows.size, idx.size
    assert val_offsets.size == W + 1
    gathered = np.zeros((R, max_blocks), np.int32)
    rc = lib().oracle_apply_staged_writes(_ptr(table), max_reqs, max_blocks, _ptr(rows),
                                          _ptr(starts), _ptr(val_offsets), _ptr(vals), W,
                                          _ptr(idx), R, _ptr(gathered))
    _check(rc, "apply_staged_writes")
    return gathered


def paged_attention(q, qsl, seq_lens, block_tables, pool: Pool, scale, causal, rows=None,
                    nthreads=0):
    """fp64 attention output [T][Hq][D] (rows not computed are NaN).

    q: uint16 bf16 bits [T][Hq][D]; block_tables int32 [R][max_blocks].
    rows: optional int64 array of token * Hq + head to compute.
    """
    q = _c(q, np.uint16)
    T, Hq, D = q.shape
    assert D == pool.D
    qsl = _c(qsl, np.int32)
    seq_lens = _c(seq_lens, np.int32)
    bt = _c(block_tables, np.int32)
    R = seq_lens.size
    assert qsl.size == R + 1
    max_blocks = bt.shape[1] if bt.ndim == 2 else 0
    out = np.full((T, Hq, D), np.nan, np.float64)
    rows_a = None if rows is None else _c(rows, np.int64)
    n_rows = 0 if rows_a is None else rows_a.size
    rc = lib().oracle_paged_attention(
        _ptr(q), _ptr(out), _ptr(qsl), _ptr(seq_lens), _ptr(bt), max_blocks, R, T, Hq,
        _ptr(pool.k), _ptr(pool.v), pool.num_blocks, pool.B, pool.Hkv, pool.D, pool.dtype,
        pool.k_scale, pool.v_scale, float(scale), int(causal), _ptr(rows_a), n_rows,
        int(nthreads))
    _check(rc, "paged_attention")
    return out


def max_threads() -> int:
    return int(lib().oracle_max_threads())


def bf16_bits_to_f64(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns (the top half of a binary32)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_table() -> np.ndarray:
    """The 256 decoded E4M3 values (NaN for the two NaN codes)."""
    return np.array([e4m3_decode(c) for c in range(256)], np.float64)


def dequantised(pool: Pool):
    """(K, V) as fp64 arrays [num_blocks][Hkv][B][D]: exact for bf16, decode*scale for FP8."""
    if pool.dtype == BF16:
        return bf16_bits_to_f64(pool.k), bf16_bits_to_f64(pool.v)
    t = e4m3_table()
    return t[pool.k] * pool.k_scale, t[pool.v] * pool.v_scale


__all__ = ["BF16", "FP8_E4M3", "Pool", "write_kv", "copy_blocks", "apply_staged_writes",
           "paged_attention", "e4m3_decode", "e4m3_encode", "fp8_store", "fp8_store_array",
           "max_threads", "bf16_bits_to_f64", "e4m3_table", "dequantised", "OracleError"]
