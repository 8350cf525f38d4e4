"""Thin ctypes binding of libpa (C ABI in include/pa.h).

Argument marshalling only: torch tensors are passed as raw device pointers,
the stream as ``torch.cuda.current_stream().cuda_stream`` unless given, and
every status other than PA_OK raises ``PaError``. All computation happens in
the library's CUDA kernels; there is no fallback of any kind. The library is
loaded from this package directory on first use (built with nvcc if it is
absent) and a failure to load it raises immediately.
"""
import ctypes
import os
from typing import Optional

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libpa.so")

PA_OK, PA_ERR_INVALID, PA_ERR_UNSUPPORTED, PA_ERR_CUDA, PA_ERR_DEVICE_BOUNDS, PA_ERR_TIMEOUT = \
    range(6)
PA_KV_BF16, PA_KV_FP8_E4M3 = 0, 1

# every function declared in include/pa.h
EXPORTS = ("pa_write_kv", "pa_forward_workspace_size", "pa_forward", "pa_apply_staged_writes",
           "pa_copy_blocks", "pa_gather_rows", "pa_get_error", "pa_status_string",
           "pa_kernel_launches",
           "pa_forward_noalloc", "pa_selftest_wait_timeout", "pa_forward_shared_prefix",
           "pa_prepare_inputs", "pa_decode_graph_create", "pa_decode_graph_launch",
           "pa_decode_graph_destroy", "pa_decode_graph_kernels",
           # include/pa_sched.h
           "pa_sched_create", "pa_sched_destroy", "pa_sched_add_request", "pa_sched_fork",
           "pa_sched_abort", "pa_sched_step", "pa_sched_commit", "pa_sched_get_stats",
           "pa_sched_block_table")


class PaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


class _Pool(ctypes.Structure):
    _fields_ = [("k_pool", ctypes.c_void_p), ("v_pool", ctypes.c_void_p),
                ("num_blocks", ctypes.c_int32), ("block_size", ctypes.c_int32),
                ("num_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("dtype", ctypes.c_int32), ("k_scale", ctypes.c_float),
                ("v_scale", ctypes.c_float)]


class _DecodeGraphDesc(ctypes.Structure):
    _fields_ = [("pool", ctypes.POINTER(_Pool)), ("scale", ctypes.c_float),
                ("num_q_heads", ctypes.c_int32), ("num_reqs", ctypes.c_int32),
                ("num_steps", ctypes.c_int32), ("num_computed", ctypes.c_void_p),
                ("max_reqs", ctypes.c_int32), ("table", ctypes.c_void_p),
                ("max_blocks", ctypes.c_int32), ("idx_mapping", ctypes.c_void_p),
                ("block_tables", ctypes.c_void_p), ("seq_len_bound_host", ctypes.c_void_p),
                ("q", ctypes.c_void_p), ("k_new", ctypes.c_void_p), ("v_new", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("query_start_loc", ctypes.c_void_p),
                ("seq_lens", ctypes.c_void_p), ("positions", ctypes.c_void_p),
                ("slot_mapping", ctypes.c_void_p), ("workspace", ctypes.c_void_p),
                ("workspace_bytes", ctypes.c_size_t)]


I32P, I64P = ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)


class _SchedConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("num_blocks", "block_size", "max_reqs",
                                                "max_blocks_per_req", "token_budget",
                                                "chunk_cap", "prefix_caching")]


class _SchedBatch(ctypes.Structure):
    _fields_ = [("num_reqs", ctypes.c_int32), ("num_tokens", ctypes.c_int32),
                ("num_decode", ctypes.c_int32), ("req_ids", I64P), ("idx_mapping", I32P),
                ("num_scheduled", I32P), ("query_start_loc", I32P), ("seq_lens", I32P),
                ("positions", I32P), ("token_ids", I32P), ("slot_mapping", I64P),
                ("num_diffs", ctypes.c_int32), ("diff_rows", I32P), ("diff_starts", I32P),
                ("diff_val_offsets", I32P), ("diff_vals", I32P), ("num_copies", ctypes.c_int32),
                ("copy_src", I32P), ("copy_dst", I32P)]


class _SchedStats(ctypes.Structure):
    _fields_ = [("steps", ctypes.c_int64), ("scheduled_tokens", ctypes.c_int64),
                ("preemptions", ctypes.c_int64), ("prefix_hit_tokens", ctypes.c_int64),
                ("finished", ctypes.c_int64), ("running", ctypes.c_int32),
                ("waiting", ctypes.c_int32), ("free_blocks", ctypes.c_int32),
                ("cached_free_blocks", ctypes.c_int32), ("used_blocks", ctypes.c_int32),
                ("stored_tokens", ctypes.c_int64), ("wasted_slots", ctypes.c_int64)]


_lib = None


def lib():
    """The loaded libpa (ctypes.CDLL). Raises if it cannot be built or loaded."""
    global _lib
    if _lib is None:
        from . import build as _build
        if not _build.up_to_date():
            _build.build()
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F32, SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                ctypes.c_size_t)
        PP = ctypes.POINTER(_Pool)
        L.pa_write_kv.restype = ctypes.c_int
        L.pa_write_kv.argtypes = [PP, P, P, P, I32, P]
        L.pa_forward_workspace_size.restype = SZ
        L.pa_forward_workspace_size.argtypes = [I32, I32, I32, I32]
        L.pa_forward.restype = ctypes.c_int
        L.pa_forward.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, PP, F32, I32, P, SZ, P]
        L.pa_apply_staged_writes.restype = ctypes.c_int
        L.pa_apply_staged_writes.argtypes = [P, I32, I32, P, P, P, P, I32, P, I32, P, P]
        L.pa_copy_blocks.restype = ctypes.c_int
        L.pa_copy_blocks.argtypes = [PP, P, P, I32, P]
        L.pa_gather_rows.restype = ctypes.c_int
        L.pa_gather_rows.argtypes = [P, I64, I64, P, I32, P, P]
        L.pa_get_error.restype = ctypes.c_int
        L.pa_get_error.argtypes = [P]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_status_string.argtypes = [ctypes.c_int]
        L.pa_forward_noalloc.restype = ctypes.c_int
        L.pa_forward_noalloc.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, PP, F32, I32,
                                         I32, P]
        L.pa_forward_shared_prefix.restype = ctypes.c_int
        L.pa_forward_shared_prefix.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, PP, F32,
                                               I32, I32, P, P, P, P, SZ, P]
        L.pa_prepare_inputs.restype = ctypes.c_int
        L.pa_prepare_inputs.argtypes = [P, I32, P, I32, I32, I32, P, P, I32, I32, P, P, P, P, P]
        L.pa_decode_graph_create.restype = ctypes.c_int
        L.pa_decode_graph_create.argtypes = [ctypes.POINTER(_DecodeGraphDesc),
                                             ctypes.POINTER(ctypes.c_void_p)]
        L.pa_decode_graph_launch.restype = ctypes.c_int
        L.pa_decode_graph_launch.argtypes = [P, P]
        L.pa_decode_graph_destroy.restype = None
        L.pa_decode_graph_destroy.argtypes = [P]
        L.pa_decode_graph_kernels.restype = ctypes.c_uint32
        L.pa_decode_graph_kernels.argtypes = [P]
        SP = ctypes.c_void_p
        L.pa_sched_create.restype = ctypes.c_int
        L.pa_sched_create.argtypes = [ctypes.POINTER(_SchedConfig), ctypes.POINTER(SP)]
        L.pa_sched_destroy.restype = None
        L.pa_sched_destroy.argtypes = [SP]
        L.pa_sched_add_request.restype = ctypes.c_int
        L.pa_sched_add_request.argtypes = [SP, I64, P, I32, I32, ctypes.c_uint64]
        L.pa_sched_fork.restype = ctypes.c_int
        L.pa_sched_fork.argtypes = [SP, I64, I64, I32]
        L.pa_sched_abort.restype = ctypes.c_int
        L.pa_sched_abort.argtypes = [SP, I64]
        L.pa_sched_step.restype = ctypes.c_int
        L.pa_sched_step.argtypes = [SP, ctypes.POINTER(_SchedBatch)]
        L.pa_sched_commit.restype = ctypes.c_int
        L.pa_sched_commit.argtypes = [SP, P, I32, P, I32, ctypes.POINTER(ctypes.c_int32)]
        L.pa_sched_get_stats.restype = ctypes.c_int
        L.pa_sched_get_stats.argtypes = [SP, ctypes.POINTER(_SchedStats)]
        L.pa_sched_block_table.restype = ctypes.c_int
        L.pa_sched_block_table.argtypes = [SP, I64, P, I32, ctypes.POINTER(ctypes.c_int32)]
        L.pa_selftest_wait_timeout.restype = ctypes.c_int
        L.pa_selftest_wait_timeout.argtypes = [P]
        L.pa_kernel_launches.restype = ctypes.c_uint64
        L.pa_kernel_launches.argtypes = []
        _lib = L
    return _lib


def status_string(status: int) -> str:
    return lib().pa_status_string(int(status)).decode()


def _check(status: int, what: str) -> None:
    if status != PA_OK:
        raise PaError(status, what)


def _stream(stream) -> Optional[int]:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, torch.cuda.Stream):
        return stream.cuda_stream
    return int(stream)


def _dptr(t: Optional[torch.Tensor], dtype=None) -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"expected {dtype}, got {t.dtype}")
    return t.data_ptr() if t.numel() else None


def _np_addr(a: np.ndarray) -> int:
    """Address of a contiguous numpy array's data (cheaper than .ctypes)."""
    return a.__array_interface__["data"][0]


def _host_i32(a) -> np.ndarray:
    if isinstance(a, torch.Tensor):
        a = a.detach().cpu().numpy()
    return np.ascontiguousarray(a, dtype=np.int32)


class KVPool:
    """Caller-owned K and V pools, each [num_blocks][Hkv][B][D] (bf16 or uint8
    E4M3 codes), with per-tensor scales for FP8."""

    def __init__(self, k: torch.Tensor, v: torch.Tensor, k_scale: float = 1.0,
                 v_scale: float = 1.0):
        if k.shape != v.shape or k.dim() != 4 or k.dtype != v.dtype:
            raise ValueError("k and v pools must be [num_blocks][Hkv][B][D] of one dtype")
        if k.dtype == torch.bfloat16:
            self.dtype = PA_KV_BF16
        elif k.dtype == torch.uint8:
            self.dtype = PA_KV_FP8_E4M3
        else:
            raise TypeError("pool dtype must be bfloat16 or uint8 (E4M3 codes)")
        self.k, self.v = k, v
        self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim = k.shape
        self.k_scale, self.v_scale = float(k_scale), float(v_scale)

    def struct(self) -> _Pool:
        return _Pool(_dptr(self.k), _dptr(self.v), self.num_blocks, self.block_size,
                     self.num_kv_heads, self.head_dim, self.dtype, self.k_scale, self.v_scale)

    def ref(self):
        """ctypes reference to the pool's C struct, built once and rebuilt
        after any attribute is reassigned or either tensor's storage moved
        (set_, resize_ or .data = ... keep the attribute but change the
        device pointer)."""
        c = self.__dict__.get("_c")
        k, v = self.__dict__["k"], self.__dict__["v"]
        if c is None or c[2] != k.data_ptr() or c[3] != v.data_ptr():
            st = self.struct()
            c = (st, ctypes.byref(st), k.data_ptr(), v.data_ptr())
            self.__dict__["_c"] = c
        return c[1]

    def __setattr__(self, name, value):
        self.__dict__.pop("_c", None)
        object.__setattr__(self, name, value)


def write_kv(pool: KVPool, k_new: torch.Tensor, v_new: torch.Tensor,
             slot_mapping: torch.Tensor, stream=None) -> None:
    T = slot_mapping.numel()
    st = lib().pa_write_kv(pool.ref(), _dptr(k_new, torch.bfloat16),
                           _dptr(v_new, torch.bfloat16), _dptr(slot_mapping, torch.int64), T,
                           _stream(stream))
    _check(st, "pa_write_kv")


def forward_workspace_size(num_reqs: int, num_q_heads: int, head_dim: int,
                           max_splits: int) -> int:
    return int(lib().pa_forward_workspace_size(num_reqs, num_q_heads, head_dim, max_splits))


def forward(q: torch.Tensor, out: torch.Tensor, query_start_loc: torch.Tensor,
            seq_lens: torch.Tensor, qsl_host, seq_lens_host, block_tables: torch.Tensor,
            pool: KVPool, scale: float, causal: int = 1,
            workspace: Optional[torch.Tensor] = None, stream=None) -> None:
    qh = _host_i32(qsl_host)
    sh = _host_i32(seq_lens_host)
    R = sh.size
    if qh.size != R + 1:
        raise ValueError("qsl_host must have num_reqs + 1 entries")
    T, Hq, D = q.shape
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    ws_ptr = _dptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    st = lib().pa_forward(
        _dptr(q, torch.bfloat16), _dptr(out, torch.bfloat16), _dptr(query_start_loc, torch.int32),
        _dptr(seq_lens, torch.int32), _np_addr(qh),
        _np_addr(sh), _dptr(block_tables, torch.int32), max_blocks, R, T,
        Hq, pool.ref(), float(scale), int(causal), ws_ptr, ws_bytes,
        _stream(stream))
    _check(st, "pa_forward")


MAX_PREFIX_GROUPS = 64  # groups accepted by pa_forward_shared_prefix


def forward_shared_prefix(q: torch.Tensor, out: torch.Tensor, query_start_loc: torch.Tensor,
                          seq_lens: torch.Tensor, qsl_host, seq_lens_host,
                          block_tables: torch.Tensor, pool: KVPool, scale: float,
                          group_first_host, group_size_host, prefix_blocks_host,
                          causal: int = 1, workspace: Optional[torch.Tensor] = None,
                          stream=None) -> None:
    """pa_forward where group k, the group_size_host[k] consecutive decode
    requests from group_first_host[k], shares the first prefix_blocks_host[k]
    block-table entries. The workspace is required (room for at least two
    splits per request)."""
    qh = _host_i32(qsl_host)
    sh = _host_i32(seq_lens_host)
    gf = _host_i32(group_first_host)
    gn = _host_i32(group_size_host)
    pb = _host_i32(prefix_blocks_host)
    R = sh.size
    if qh.size != R + 1:
        raise ValueError("qsl_host must have num_reqs + 1 entries")
    G = pb.size
    if gf.size != G or gn.size != G:
        raise ValueError("group arrays must have num_groups entries each")
    T, Hq, D = q.shape
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    ws_ptr = _dptr(workspace) if workspace is not None else None
    ws_bytes = workspace.numel() * workspace.element_size() if workspace is not None else 0
    host = lambda a: _np_addr(a) if G > 0 else None
    st = lib().pa_forward_shared_prefix(
        _dptr(q, torch.bfloat16), _dptr(out, torch.bfloat16), _dptr(query_start_loc, torch.int32),
        _dptr(seq_lens, torch.int32), _np_addr(qh),
        _np_addr(sh), _dptr(block_tables, torch.int32), max_blocks, R, T,
        Hq, pool.ref(), float(scale), int(causal), G, host(gf), host(gn),
        host(pb), ws_ptr, ws_bytes, _stream(stream))
    _check(st, "pa_forward_shared_prefix")


NOALLOC_SCRATCH_BYTES = 16 << 20  # PA_NOALLOC_SCRATCH_BYTES in include/pa.h


def forward_noalloc(q: torch.Tensor, out: torch.Tensor, query_start_loc: torch.Tensor,
                    seq_lens: torch.Tensor, qsl_host, seq_lens_host,
                    block_tables: torch.Tensor, pool: KVPool, scale: float, causal: int = 1,
                    max_splits: int = 32, stream=None) -> None:
    """pa_forward for callers that cannot allocate device memory: the split-KV
    scratch comes from the library's own fixed device array (16 MiB per GPU),
    so no workspace is passed. Calls that may overlap on the GPU share that
    array and must be serialised by the caller."""
    qh = _host_i32(qsl_host)
    sh = _host_i32(seq_lens_host)
    R = sh.size
    if qh.size != R + 1:
        raise ValueError("qsl_host must have num_reqs + 1 entries")
    T, Hq, D = q.shape
    max_blocks = block_tables.shape[1] if block_tables.dim() == 2 else 0
    st = lib().pa_forward_noalloc(
        _dptr(q, torch.bfloat16), _dptr(out, torch.bfloat16), _dptr(query_start_loc, torch.int32),
        _dptr(seq_lens, torch.int32), _np_addr(qh),
        _np_addr(sh), _dptr(block_tables, torch.int32), max_blocks, R, T,
        Hq, pool.ref(), float(scale), int(causal), int(max_splits),
        _stream(stream))
    _check(st, "pa_forward_noalloc")


def prepare_inputs(num_computed: torch.Tensor, table: torch.Tensor, block_size: int,
                   num_blocks: int, idx_mapping: torch.Tensor, num_scheduled: torch.Tensor,
                   query_start_loc: torch.Tensor, seq_lens: torch.Tensor,
                   positions: torch.Tensor, slot_mapping: torch.Tensor, stream=None) -> None:
    """Device-side step inputs from per-slot state (pa_prepare_inputs); the
    outputs are written into the given device tensors."""
    max_reqs, max_blocks = table.shape
    R = idx_mapping.numel()
    st = lib().pa_prepare_inputs(
        _dptr(num_computed, torch.int32), max_reqs, _dptr(table, torch.int32), max_blocks,
        int(block_size), int(num_blocks), _dptr(idx_mapping, torch.int32),
        _dptr(num_scheduled, torch.int32), R, positions.numel(),
        _dptr(query_start_loc, torch.int32), _dptr(seq_lens, torch.int32),
        _dptr(positions, torch.int32), _dptr(slot_mapping, torch.int64), _stream(stream))
    _check(st, "pa_prepare_inputs")


class DecodeGraph:
    """pa_decode_graph_*: `num_steps` decode steps of the same requests
    captured once into a CUDA graph (prepare inputs, write K/V, attention per
    step) and replayed by launch(). Every tensor passed here must stay alive
    and in place while the graph exists; this object keeps references to
    them. The plan is fixed from seq_len_bound (host, per request)."""

    def __init__(self, pool: KVPool, scale: float, num_computed: torch.Tensor,
                 table: torch.Tensor, idx_mapping: torch.Tensor, block_tables: torch.Tensor,
                 seq_len_bound, q: torch.Tensor, k_new: torch.Tensor, v_new: torch.Tensor,
                 out: torch.Tensor, workspace: Optional[torch.Tensor] = None):
        N, R, Hq, D = q.shape
        self._bound = _host_i32(seq_len_bound)
        dev = q.device
        self.query_start_loc = torch.empty(R + 1, dtype=torch.int32, device=dev)
        self.seq_lens = torch.empty(R, dtype=torch.int32, device=dev)
        self.positions = torch.empty(R, dtype=torch.int32, device=dev)
        self.slot_mapping = torch.empty(R, dtype=torch.int64, device=dev)
        self._pool_struct = pool.struct()
        self._keep = (pool, num_computed, table, idx_mapping, block_tables, q, k_new, v_new, out,
                      workspace)
        d = _DecodeGraphDesc()
        d.pool = ctypes.pointer(self._pool_struct)
        d.scale = float(scale)
        d.num_q_heads, d.num_reqs, d.num_steps = Hq, R, N
        d.num_computed = _dptr(num_computed, torch.int32)
        d.max_reqs = table.shape[0]
        d.table = _dptr(table, torch.int32)
        d.max_blocks = table.shape[1]
        d.idx_mapping = _dptr(idx_mapping, torch.int32)
        d.block_tables = _dptr(block_tables, torch.int32)
        d.seq_len_bound_host = self._bound.ctypes.data_as(ctypes.c_void_p)
        d.q = _dptr(q, torch.bfloat16)
        d.k_new = _dptr(k_new, torch.bfloat16)
        d.v_new = _dptr(v_new, torch.bfloat16)
        d.out = _dptr(out, torch.bfloat16)
        d.query_start_loc = _dptr(self.query_start_loc)
        d.seq_lens = _dptr(self.seq_lens)
        d.positions = _dptr(self.positions)
        d.slot_mapping = _dptr(self.slot_mapping)
        d.workspace = _dptr(workspace) if workspace is not None else None
        d.workspace_bytes = workspace.numel() if workspace is not None else 0
        self._desc = d
        h = ctypes.c_void_p()
        _check(lib().pa_decode_graph_create(ctypes.byref(d), ctypes.byref(h)),
               "pa_decode_graph_create")
        self._h = h

    @property
    def kernels(self) -> int:
        return int(lib().pa_decode_graph_kernels(self._h))

    def launch(self, stream=None) -> None:
        _check(lib().pa_decode_graph_launch(self._h, _stream(stream)), "pa_decode_graph_launch")

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().pa_decode_graph_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class SchedBatch:
    """One scheduled step (numpy copies of the scheduler's arrays)."""
    FIELDS = ("req_ids", "idx_mapping", "num_scheduled", "query_start_loc", "seq_lens",
              "positions", "token_ids", "slot_mapping", "diff_rows", "diff_starts",
              "diff_val_offsets", "diff_vals", "copy_src", "copy_dst")
    _INT64 = frozenset(("req_ids", "slot_mapping"))

    def __init__(self, b: "_SchedBatch"):
        R, T, W, C = b.num_reqs, b.num_tokens, b.num_diffs, b.num_copies
        n_vals = b.diff_val_offsets[W] if W >= 0 else 0
        sizes = (R, R, R, R + 1, R, T, T, T, W, W, W + 1, n_vals, C, C)
        # one memcpy per field (string_at) into a writable buffer: the
        # per-call cost of np.ctypeslib.as_array dominated a serving step's
        # host time
        for name, n in zip(self.FIELDS, sizes):
            dt = np.int64 if name in self._INT64 else np.int32
            if n > 0:
                addr = ctypes.cast(getattr(b, name), ctypes.c_void_p).value
                nbytes = n * (8 if dt is np.int64 else 4)
                arr = np.frombuffer(bytearray(ctypes.string_at(addr, nbytes)), dt)
            else:
                arr = np.zeros(0, dt)
            setattr(self, name, arr)
        self.num_decode = b.num_decode

    @property
    def num_reqs(self) -> int:
        return int(self.req_ids.size)

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])


class Scheduler:
    """pa_sched_*: the native host scheduler and block manager."""

    def __init__(self, num_blocks: int, block_size: int, max_reqs: int,
                 max_blocks_per_req: int, token_budget: int, chunk_cap: int = 1024,
                 prefix_caching: bool = False):
        cfg = _SchedConfig(num_blocks, block_size, max_reqs, max_blocks_per_req, token_budget,
                           chunk_cap, 1 if prefix_caching else 0)
        h = ctypes.c_void_p()
        _check(lib().pa_sched_create(ctypes.byref(cfg), ctypes.byref(h)), "pa_sched_create")
        self._h = h
        self.block_size = block_size

    def add_request(self, req_id: int, prompt, max_new: int, salt: int = 0) -> None:
        p = np.ascontiguousarray(prompt, dtype=np.int32)
        _check(lib().pa_sched_add_request(self._h, int(req_id), _np_addr(p),
                                          p.size, int(max_new), int(salt) & (2**64 - 1)),
               "pa_sched_add_request")

    def fork(self, parent: int, child: int, max_new: int) -> None:
        _check(lib().pa_sched_fork(self._h, int(parent), int(child), int(max_new)),
               "pa_sched_fork")

    def abort(self, req_id: int) -> None:
        _check(lib().pa_sched_abort(self._h, int(req_id)), "pa_sched_abort")

    def step(self) -> SchedBatch:
        b = _SchedBatch()
        _check(lib().pa_sched_step(self._h, ctypes.byref(b)), "pa_sched_step")
        return SchedBatch(b)

    def commit(self, sampled):
        s = np.ascontiguousarray(sampled, dtype=np.int32)
        ids = np.zeros(max(s.size, 1), np.int64)
        n = ctypes.c_int32()
        _check(lib().pa_sched_commit(self._h, _np_addr(s), s.size, _np_addr(ids), ids.size,
                                     ctypes.byref(n)), "pa_sched_commit")
        return ids[:n.value].tolist()

    def stats(self) -> dict:
        st = _SchedStats()
        _check(lib().pa_sched_get_stats(self._h, ctypes.byref(st)), "pa_sched_get_stats")
        return {name: getattr(st, name) for name, _ in _SchedStats._fields_}

    def table(self, req_id: int):
        n = ctypes.c_int32()
        _check(lib().pa_sched_block_table(self._h, int(req_id), None, 0, ctypes.byref(n)),
               "pa_sched_block_table")
        out = np.zeros(max(n.value, 1), np.int32)
        _check(lib().pa_sched_block_table(self._h, int(req_id),
                                          out.ctypes.data_as(ctypes.c_void_p), out.size,
                                          ctypes.byref(n)), "pa_sched_block_table")
        return out[:n.value].tolist()

    def close(self) -> None:
        if getattr(self, "_h", None):
            lib().pa_sched_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def apply_staged_writes(table: torch.Tensor, rows: torch.Tensor, starts: torch.Tensor,
                        val_offsets: torch.Tensor, vals: torch.Tensor,
                        idx_mapping: torch.Tensor, gathered: torch.Tensor, stream=None) -> None:
    max_reqs, max_blocks = table.shape
    W = rows.numel()
    R = idx_mapping.numel()
    st = lib().pa_apply_staged_writes(
        _dptr(table, torch.int32), max_reqs, max_blocks, _dptr(rows, torch.int32),
        _dptr(starts, torch.int32), _dptr(val_offsets, torch.int32), _dptr(vals, torch.int32),
        W, _dptr(idx_mapping, torch.int32), R, _dptr(gathered, torch.int32), _stream(stream))
    _check(st, "pa_apply_staged_writes")


def copy_blocks(pool: KVPool, src: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    st = lib().pa_copy_blocks(pool.ref(), _dptr(src, torch.int32),
                              _dptr(dst, torch.int32), src.numel(), _stream(stream))
    _check(st, "pa_copy_blocks")


def gather_rows(src: torch.Tensor, rows: torch.Tensor, dst: torch.Tensor, stream=None) -> None:
    """dst[i] = src[rows[i]] (rows of src's first dimension) on the device."""
    n = rows.numel()
    if dst.shape[0] < n or dst.shape[1:] != src.shape[1:] or dst.dtype != src.dtype:
        raise ValueError("dst must hold len(rows) rows shaped like src's")
    if not (src.is_contiguous() and dst.is_contiguous()):
        raise ValueError("src and dst must be contiguous")
    row_bytes = src[0].numel() * src.element_size() if src.shape[0] else 16
    _check(lib().pa_gather_rows(_dptr(src), src.shape[0], row_bytes, _dptr(rows, torch.int32), n,
                                _dptr(dst), _stream(stream)), "pa_gather_rows")


def selftest_wait_timeout(stream=None) -> None:
    """Runs the library's bounded device wait on a barrier nothing completes
    (about 2 s); pa_get_error() afterwards reports PA_ERR_TIMEOUT."""
    _check(lib().pa_selftest_wait_timeout(_stream(stream)), "pa_selftest_wait_timeout")


def get_error(stream=None) -> int:
    """Synchronises the stream and returns (and clears) the device error status."""
    return int(lib().pa_get_error(_stream(stream)))


def kernel_launches() -> int:
    """Kernels launched by libpa so far in this process."""
    return int(lib().pa_kernel_launches())
