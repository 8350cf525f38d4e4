"""Multi-step serving loop over the native scheduler and the device calls.

Each step: the native scheduler (pa_sched_step) decides the batch; the host
packs what the device needs into one pinned buffer and sends it with one
copy; then, on the stream,
  pa_apply_staged_writes  on the per-slot stored-token counts (slots whose
                          count the device does not hold: admissions,
                          resumed or forked requests) and on the block table
                          (the step's diffs, then the gather by idx_mapping),
  pa_copy_blocks          the step's copy-on-write pairs,
  pa_prepare_inputs       query_start_loc, seq_lens, positions, slot mapping,
  pa_write_kv             the step's new K/V,
  pa_forward              attention for every entry,
  pa_gather_rows          the output row of each entry's last token,
and those rows are read back into one of two pinned host buffers.

[MRV2 "재설계 1"] persistent slots and idx_mapping; [MRV2 "재설계 2"] the
host never modifies a buffer the device may still be reading: two pinned
staging buffers alternate, each reused only after the copy that read it has
completed; [MRV2 "재설계 3"] only diffs go to the device table; [MRV2
"재설계 4"] the inputs are prepared on the device.

There is no model: the caller provides the step's Q/K/V rows (token t of the
batch is row t) and the sampled tokens.
"""
from typing import Optional

import numpy as np
import torch

from . import pa


class Engine:
    def __init__(self, sched: "pa.Scheduler", pool: "pa.KVPool", num_q_heads: int, max_reqs: int,
                 max_blocks: int, max_tokens: int, scale: float, max_splits: int = 32,
                 device=None):
        self.sched, self.pool = sched, pool
        self.B, self.Hq, self.D = pool.block_size, num_q_heads, pool.head_dim
        self.max_reqs, self.max_blocks, self.max_tokens = max_reqs, max_blocks, max_tokens
        self.scale = scale
        dev = torch.device("cuda") if device is None else torch.device(device)
        self.dev = dev
        i32 = dict(dtype=torch.int32, device=dev)
        self.table = torch.full((max_reqs, max_blocks), -1, **i32)
        self.gathered = torch.full((max_reqs, max_blocks), -1, **i32)
        self.num_computed = torch.zeros((max_reqs, 1), **i32)
        self.qsl = torch.zeros(max_reqs + 1, **i32)
        self.seq = torch.zeros(max_reqs, **i32)
        self.pos = torch.zeros(max_tokens, **i32)
        self.slots = torch.zeros(max_tokens, dtype=torch.int64, device=dev)
        # staging: the largest step payload (ints)
        self.cap = 6 * max_reqs + 2 * max_reqs * max_blocks + 4 * max_reqs + 16
        self.host = [torch.zeros(self.cap, dtype=torch.int32).pin_memory() for _ in range(2)]
        self.host_np = [h.numpy() for h in self.host]
        self.done = [torch.cuda.Event(), torch.cuda.Event()]
        self.used = [False, False]
        self.dstage = torch.zeros(self.cap, **i32)
        n = pa.forward_workspace_size(max_reqs, num_q_heads, self.D, max_splits)
        self.ws = torch.empty(n, dtype=torch.uint8, device=dev) if n else None
        self.mirror = np.full(max_reqs, -1, np.int64)  # stored-token count the device holds
        # each entry's last output row: gathered on the device, read back into
        # one of two pinned buffers (a step's rows stay valid through the next step)
        self.last_dev = torch.empty((max_reqs, num_q_heads, self.D), dtype=torch.bfloat16,
                                    device=dev)
        self.last_host = [torch.empty((max_reqs, num_q_heads, self.D),
                                      dtype=torch.bfloat16).pin_memory() for _ in range(2)]
        self.last_turn = 0
        self.last_out = None
        self.turn = 0
        self.steps = 0
        self.h2d_bytes = 0
        self.d2h_bytes = 0

    def step(self, q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
             stream=None) -> "pa.SchedBatch":
        """Runs one step; q/k/v/out hold at least the step's tokens as rows.
        Returns the scheduled batch; the output rows of each entry's last
        token are in `last_out` (host, pinned) once the step's stream has
        reached the end of the step (the next `step` or `sync` waits); they
        stay valid through the next step (two buffers alternate)."""
        b = self.sched.step()
        R, T = b.num_reqs, b.num_tokens
        if T > self.max_tokens or R > self.max_reqs:
            raise ValueError("batch larger than the engine's buffers")
        s = torch.cuda.current_stream() if stream is None else stream
        # slots whose stored-token count the device does not hold
        start = (b.seq_lens - b.num_scheduled).astype(np.int64)
        stale = np.nonzero(self.mirror[b.idx_mapping] != start)[0]
        W, C, S = b.diff_rows.size, b.copy_src.size, stale.size
        NV = int(b.diff_val_offsets[-1])
        parts = [b.idx_mapping, b.num_scheduled, b.diff_rows, b.diff_starts, b.diff_val_offsets,
                 b.diff_vals, b.idx_mapping[stale], np.zeros(S, np.int32),
                 np.arange(S + 1, dtype=np.int32), start[stale].astype(np.int32), b.copy_src,
                 b.copy_dst, (b.query_start_loc[1:] - 1).astype(np.int32)]
        total = sum(p.size for p in parts)
        if total > self.cap:
            raise ValueError("step payload larger than the staging buffer")
        i = self.turn
        if self.used[i]:
            self.done[i].synchronize()  # the copy that last read this buffer is over
        h = self.host_np[i]
        offs = [0]
        for p in parts:
            h[offs[-1]:offs[-1] + p.size] = p
            offs.append(offs[-1] + p.size)
        with torch.cuda.stream(s):
            self.dstage[:total].copy_(self.host[i][:total], non_blocking=True)
            self.done[i].record(s)
            self.used[i] = True
            self.turn ^= 1
            d = [self.dstage[offs[j]:offs[j + 1]] for j in range(len(parts))]
            idx, cnt = d[0], d[1]
            if S:
                pa.apply_staged_writes(self.num_computed, d[6], d[7], d[8], d[9],
                                       idx[:0], self.gathered[:0], stream=s)
            pa.apply_staged_writes(self.table, d[2], d[3], d[4], d[5], idx,
                                   self.gathered[:R], stream=s)
            if C:
                pa.copy_blocks(self.pool, d[10], d[11], stream=s)
            pa.prepare_inputs(self.num_computed, self.table, self.B, self.pool.num_blocks, idx,
                              cnt, self.qsl[:R + 1], self.seq[:R], self.pos[:T],
                              self.slots[:T], stream=s)
            pa.write_kv(self.pool, k[:T], v[:T], self.slots[:T], stream=s)
            pa.forward(q[:T], out[:T], self.qsl[:R + 1], self.seq[:R], b.query_start_loc,
                       b.seq_lens, self.gathered[:R], self.pool, self.scale, 1,
                       workspace=self.ws, stream=s)
            host = self.last_host[self.last_turn][:R]
            if R:
                pa.gather_rows(out, d[12], self.last_dev[:R], stream=s)
                host.copy_(self.last_dev[:R], non_blocking=True)
            self.last_out = host
            self.last_turn ^= 1
        self.mirror[b.idx_mapping] = b.seq_lens
        self.h2d_bytes += 4 * total
        self.d2h_bytes += host.numel() * host.element_size()
        self.steps += 1
        self.stream = s
        return b

    def sync(self) -> None:
        self.stream.synchronize()
