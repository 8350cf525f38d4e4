"""GPU-side plumbing for the parity tests: run the hot path through the C ABI
on a workload, and the matching oracle computation on the same inputs."""
import numpy as np
import torch

from oracle import oracle as O
from paged_kv_cache_143_gb300 import pa
from tests.helpers import bits, oracle_pool
from workloads.generate import NAN_BF16, NAN_E4M3

MAX_ABS = 2e-2   # bf16 output vs fp64 oracle: max |error|
MEAN_ABS = 2e-3  # and mean |error|


def new_gpu_pool(w, dev) -> pa.KVPool:
    shape = w.pool_shape()
    if w.kv_dtype == "bf16":
        k = torch.full(shape, NAN_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
        v = torch.full(shape, NAN_BF16, dtype=torch.int16, device=dev).view(torch.bfloat16)
    else:
        k = torch.full(shape, NAN_E4M3, dtype=torch.uint8, device=dev)
        v = torch.full(shape, NAN_E4M3, dtype=torch.uint8, device=dev)
    return pa.KVPool(k, v, w.k_scale, w.v_scale)


def gpu_cache(w, dev) -> pa.KVPool:
    """A pool holding the workload's context (the cache before the step)."""
    pool = new_gpu_pool(w, dev)
    if w.ctx_slots.numel():
        pa.write_kv(pool, w.ctx_k.to(dev).contiguous(), w.ctx_v.to(dev).contiguous(),
                    w.ctx_slots.to(dev))
    return pool


class DeviceStep:
    """Device copies of one step's inputs and the call sequence of the hot
    path: staged table diffs + gather, KV write, attention."""

    def __init__(self, w, dev, pool=None, max_splits=32, out_fill=None):
        self.w = w
        self.dev = dev
        self.pool = gpu_cache(w, dev) if pool is None else pool
        i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
        self.table = i32(w.table_before)
        self.rows, self.starts = i32(w.diff_rows), i32(w.diff_starts)
        self.offs, self.vals = i32(w.diff_val_offsets), i32(w.diff_vals)
        self.idx = i32(w.idx_mapping)
        self.gathered = torch.full((w.R, w.max_blocks), -7, dtype=torch.int32, device=dev)
        self.qsl, self.seq = i32(w.qsl), i32(w.seq_lens)
        self.q = w.q.to(dev).contiguous()
        self.new_k = w.new_k.to(dev).contiguous()
        self.new_v = w.new_v.to(dev).contiguous()
        self.slots = w.slot_mapping.to(dev)
        self.out = torch.empty_like(self.q)
        if out_fill is not None:
            self.out.fill_(out_fill)
        nbytes = pa.forward_workspace_size(w.R, w.Hq, w.D, max_splits) if max_splits else 0
        self.ws = torch.empty(max(nbytes, 1), dtype=torch.uint8, device=dev) if nbytes else None

    def run(self, tables=None, cascade=False):
        """cascade: attention through pa_forward_shared_prefix with the
        workload's groups (consecutive requests) and their prefix blocks."""
        w = self.w
        pa.apply_staged_writes(self.table, self.rows, self.starts, self.offs, self.vals,
                               self.idx, self.gathered)
        pa.write_kv(self.pool, self.new_k, self.new_v, self.slots)
        tab = self.gathered if tables is None else tables
        if cascade:
            first, size, prefix_blocks = group_arrays(w)
            pa.forward_shared_prefix(self.q, self.out, self.qsl, self.seq, w.qsl, w.seq_lens,
                                     tab, self.pool, w.scale, first, size, prefix_blocks,
                                     causal=w.causal, workspace=self.ws)
        else:
            pa.forward(self.q, self.out, self.qsl, self.seq, w.qsl, w.seq_lens, tab, self.pool,
                       w.scale, w.causal, workspace=self.ws)
        return self.out


def group_arrays(w):
    """(first [G], size [G], prefix_blocks [G]) of a workload whose groups
    are runs of consecutive requests, sorted by their first member."""
    rows = []
    for members, pt in zip(w.groups, w.group_prefix):
        m = sorted(members)
        assert m == list(range(m[0], m[0] + len(m))), "group members must be consecutive"
        rows.append((m[0], len(m), pt // w.B))
    rows.sort()
    a = np.array(rows, np.int32).reshape(-1, 3)
    return a[:, 0].copy(), a[:, 1].copy(), a[:, 2].copy()


def oracle_step(w, rows=None):
    """The oracle on the same inputs: pool (context + step tokens), the staged
    diffs applied to the persistent table, attention through the gathered rows."""
    pool = oracle_pool(w)
    table = w.table_before.copy()
    gathered = O.apply_staged_writes(table, w.diff_rows, w.diff_starts, w.diff_val_offsets,
                                     w.diff_vals, w.idx_mapping)
    out = O.paged_attention(bits(w.q), w.qsl, w.seq_lens, gathered, pool, w.scale, w.causal,
                            rows=rows)
    return out, pool, table, gathered


def pool_bits(p: pa.KVPool):
    return bits(p.k), bits(p.v)


def assert_attention_close(gpu_out: torch.Tensor, ref: np.ndarray, rows=None, what=""):
    g = gpu_out.detach().float().cpu().double().numpy().reshape(-1, ref.shape[-1])
    r = ref.reshape(-1, ref.shape[-1])
    if rows is not None:
        g, r = g[rows], r[rows]
    assert np.isfinite(g).all(), f"{what}: non-finite GPU output"
    assert np.isfinite(r).all(), f"{what}: oracle rows missing"
    err = np.abs(g - r)
    assert err.max() <= MAX_ABS, f"{what}: max abs error {err.max():.3e}"
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs error {err.mean():.3e}"
    return float(err.max()), float(err.mean())
