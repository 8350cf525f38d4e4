"""Builders for the synthetic workloads (inputs only; see the package docstring)."""
import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence, Tuple

import numpy as np
import torch

CONFIG_NAMES = {
    1: "tiny-decode",
    2: "decode-7b-like",
    3: "mixed-chunked-prefill",
    4: "prefix-shared-sampling-fp8",
    5: "long-context",
}

NAN_BF16 = 0x7FC0
NAN_E4M3 = 0x7F


def config_seed(cfg: int, sub: int = 0) -> int:
    """Seed of config ``cfg`` (sub-runs use (143000 + cfg) * 10 + sub)."""
    return 143000 + cfg if sub == 0 else (143000 + cfg) * 10 + sub


@dataclass
class Workload:
    name: str
    Hq: int
    Hkv: int
    D: int
    B: int
    kv_dtype: str  # "bf16" or "fp8"
    scale: float
    causal: int
    seq_lens: np.ndarray  # int32 [R]
    qsl: np.ndarray  # int32 [R+1]
    num_blocks: int
    tables: np.ndarray  # int32 [R][max_blocks]; -1 past the request's blocks
    q: torch.Tensor  # bf16 [T][Hq][D]
    ctx_k: torch.Tensor  # bf16 [Nctx][Hkv][D]  cached before the step
    ctx_v: torch.Tensor
    ctx_slots: torch.Tensor  # int64 [Nctx]
    ctx_req: np.ndarray  # int32 [Nctx]: request that first stored the token
    ctx_pos: np.ndarray  # int32 [Nctx]: its position in that request
    new_k: torch.Tensor  # bf16 [T][Hkv][D]  written by the step
    new_v: torch.Tensor
    slot_mapping: torch.Tensor  # int64 [T]
    k_scale: float
    v_scale: float
    max_reqs: int
    table_before: np.ndarray  # int32 [max_reqs][max_blocks] before the step's diffs
    idx_mapping: np.ndarray  # int32 [R]: persistent slot of batch entry i
    diff_rows: np.ndarray  # int32 [W]
    diff_starts: np.ndarray  # int32 [W]
    diff_val_offsets: np.ndarray  # int32 [W+1]
    diff_vals: np.ndarray  # int32 [N]
    groups: List[List[int]] = field(default_factory=list)
    group_prefix: List[int] = field(default_factory=list)  # shared prefix tokens per group
    seed: int = 0

    @property
    def R(self) -> int:
        return int(self.seq_lens.size)

    @property
    def T(self) -> int:
        return int(self.qsl[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.tables.shape[1])

    @property
    def q_lens(self) -> np.ndarray:
        return np.diff(self.qsl).astype(np.int32)

    @property
    def elt_bytes(self) -> int:
        return 2 if self.kv_dtype == "bf16" else 1

    def pool_shape(self) -> Tuple[int, int, int, int]:
        return (self.num_blocks, self.Hkv, self.B, self.D)

    def pool_nan_fill(self) -> int:
        return NAN_BF16 if self.kv_dtype == "bf16" else NAN_E4M3


def staged_diffs_from_tables(tables: np.ndarray, first_new_block: np.ndarray,
                             nblocks: np.ndarray, idx_mapping: np.ndarray, max_reqs: int,
                             ) -> Tuple[np.ndarray, ...]:
    """Splits per-request tables into a persistent table (blocks that existed
    before the step) and the step's (row, start, values) diffs (blocks first
    used by the step's tokens)."""
    R, max_blocks = tables.shape
    before = np.full((max_reqs, max_blocks), -1, np.int32)
    rows, starts, offs, vals = [], [], [0], []
    for r in range(R):
        f, n = int(first_new_block[r]), int(nblocks[r])
        before[idx_mapping[r], :f] = tables[r, :f]
        if n > f:
            rows.append(int(idx_mapping[r]))
            starts.append(f)
            vals.extend(int(x) for x in tables[r, f:n])
            offs.append(len(vals))
    return (before, np.array(rows, np.int32), np.array(starts, np.int32),
            np.array(offs, np.int32), np.array(vals, np.int32))


def _randn_bf16(gen: torch.Generator, shape, device, mult: float = 1.0) -> torch.Tensor:
    x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    return x.to(torch.bfloat16)


def build(seq_lens: Sequence[int], q_lens: Sequence[int], Hq: int, Hkv: int, D: int, B: int,
          kv_dtype: str = "bf16", scale: Optional[float] = None, causal: int = 1,
          seed: int = 0, device="cpu", pool_blocks: Optional[int] = None,
          groups: Optional[List[Tuple[List[int], int]]] = None,
          max_reqs: Optional[int] = None, max_blocks: Optional[int] = None,
          q_mult: float = 1.0, name: str = "custom") -> Workload:
    """General builder.

    groups: list of (member request ids, shared prefix tokens); the prefix
    (a whole number of blocks) is stored once in physical blocks shared by
    every member.
    """
    seq = np.asarray(seq_lens, np.int64)
    ql = np.asarray(q_lens, np.int64)
    R = seq.size
    assert ql.size == R and np.all(ql >= 0) and np.all(ql <= seq)
    assert kv_dtype in ("bf16", "fp8")
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    rng = np.random.Generator(np.random.PCG64(seed))
    nblk = -(-seq // B)
    mb = int(max(nblk.max() if R else 1, 1)) if max_blocks is None else max_blocks
    assert mb >= (nblk.max() if R else 0)

    # ---- physical placement: shared prefix blocks once per group, then private
    group_of = {}
    shared_blocks = []
    for gi, (members, prefix) in enumerate(groups or []):
        assert prefix % B == 0
        for r in members:
            assert prefix <= seq[r] - ql[r]
            group_of[int(r)] = gi
        shared_blocks.append(prefix // B)
    total = int(nblk.sum()) - sum((len(m) - 1) * sb for (m, _), sb in
                                  zip(groups or [], shared_blocks))
    nb = total if pool_blocks is None else int(pool_blocks)
    assert nb >= total
    ids = rng.permutation(nb)[:total].astype(np.int32)
    cursor = 0
    group_ids = []
    for sb in shared_blocks:
        group_ids.append(ids[cursor:cursor + sb])
        cursor += sb
    tables = np.full((R, mb), -1, np.int32)
    for r in range(R):
        k = 0
        if r in group_of:
            gids = group_ids[group_of[r]]
            tables[r, :gids.size] = gids
            k = gids.size
        n = int(nblk[r]) - k
        tables[r, k:k + n] = ids[cursor:cursor + n]
        cursor += n
    assert cursor == total

    # ---- tokens: cached context (written before the step) and the step's tokens
    first_writer = {}
    for gi, (members, _) in enumerate(groups or []):
        first_writer[gi] = min(members)
    ctx_slot_list = []
    ctx_req_list, ctx_pos_list = [], []
    new_slot_list = []
    for r in range(R):
        P = int(seq[r] - ql[r])
        start = 0
        if r in group_of and r != first_writer[group_of[r]]:
            start = (groups[group_of[r]][1])  # shared prefix already stored
        pos = np.arange(start, P, dtype=np.int64)
        ctx_slot_list.append(tables[r, pos // B].astype(np.int64) * B + pos % B)
        ctx_req_list.append(np.full(pos.size, r, np.int32))
        ctx_pos_list.append(pos.astype(np.int32))
        pos = np.arange(P, int(seq[r]), dtype=np.int64)
        new_slot_list.append(tables[r, pos // B].astype(np.int64) * B + pos % B)
    ctx_slots = np.concatenate(ctx_slot_list) if R else np.zeros(0, np.int64)
    ctx_req = np.concatenate(ctx_req_list) if R else np.zeros(0, np.int32)
    ctx_pos = np.concatenate(ctx_pos_list) if R else np.zeros(0, np.int32)
    new_slots = np.concatenate(new_slot_list) if R else np.zeros(0, np.int64)
    qsl = np.zeros(R + 1, np.int32)
    qsl[1:] = np.cumsum(ql)
    T = int(qsl[-1])

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))
    Nctx = int(ctx_slots.size)
    ctx_k = _randn_bf16(gen, (Nctx, Hkv, D), device)
    ctx_v = _randn_bf16(gen, (Nctx, Hkv, D), device)
    new_k = _randn_bf16(gen, (T, Hkv, D), device)
    new_v = _randn_bf16(gen, (T, Hkv, D), device)
    q = _randn_bf16(gen, (T, Hq, D), device, q_mult)

    k_scale = v_scale = 1.0
    if kv_dtype == "fp8":
        def amax(a, b):
            m = 0.0
            for x in (a, b):
                if x.numel():
                    m = max(m, float(x.abs().max().float()))
            return m
        # per-tensor scales: amax / 448 in fp32
        k_scale = float(np.float32(np.float32(amax(ctx_k, new_k)) / np.float32(448.0)))
        v_scale = float(np.float32(np.float32(amax(ctx_v, new_v)) / np.float32(448.0)))
        k_scale = k_scale or 1.0
        v_scale = v_scale or 1.0

    # ---- persistent table and the step's staged diffs
    mr = max(1024, R) if max_reqs is None else max_reqs
    assert mr >= R
    idx_mapping = rng.choice(mr, size=R, replace=False).astype(np.int32)
    P = seq - ql
    first_new = -(-P // B)
    before, rows, starts, offs, vals = staged_diffs_from_tables(tables, first_new, nblk,
                                                                idx_mapping, mr)
    return Workload(
        name=name, Hq=Hq, Hkv=Hkv, D=D, B=B, kv_dtype=kv_dtype, scale=float(scale),
        causal=int(causal), seq_lens=seq.astype(np.int32), qsl=qsl, num_blocks=nb,
        tables=tables, q=q, ctx_k=ctx_k, ctx_v=ctx_v,
        ctx_slots=torch.from_numpy(ctx_slots).to(device), ctx_req=ctx_req, ctx_pos=ctx_pos,
        new_k=new_k, new_v=new_v, slot_mapping=torch.from_numpy(new_slots).to(device),
        k_scale=k_scale, v_scale=v_scale, max_reqs=mr, table_before=before,
        idx_mapping=idx_mapping, diff_rows=rows, diff_starts=starts, diff_val_offsets=offs,
        diff_vals=vals, groups=[list(m) for m, _ in (groups or [])],
        group_prefix=[int(p) for _, p in (groups or [])], seed=int(seed))


def make(cfg: int, device="cpu", kv_dtype: Optional[str] = None, sub: int = 0,
         num_requests: Optional[int] = None, q_mult: float = 1.0) -> Workload:
    """Workload ``cfg`` (1..5). ``num_requests`` draws a smaller sample with the
    same per-request distribution (configs 2 and 3 decodes); ``kv_dtype``
    selects config 5's bf16 or FP8 run."""
    seed = config_seed(cfg, sub)
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    name = CONFIG_NAMES[cfg]
    if cfg == 1:
        return build([17, 33, 64, 100], [1, 1, 1, 1], Hq=4, Hkv=4, D=64, B=16,
                     scale=1.0 / 8.0, seed=seed, device=device, pool_blocks=64, q_mult=q_mult,
                     name=name)
    if cfg == 2:
        R = 256 if num_requests is None else num_requests
        seq = rng.integers(128, 2048, size=R, endpoint=True)
        return build(seq, np.ones(R, np.int64), Hq=32, Hkv=32, D=128, B=16, seed=seed,
                     device=device, q_mult=q_mult, name=name)
    if cfg == 3:
        nd = 64 if num_requests is None else num_requests
        dec = rng.integers(1024, 4096, size=nd, endpoint=True)
        chunks = [(1024, 0), (1024, 2048), (1920, 8192)]
        seq = list(dec) + [c + p for c, p in chunks]
        ql = [1] * nd + [c for c, _ in chunks]
        return build(seq, ql, Hq=32, Hkv=8, D=128, B=16, seed=seed, device=device,
                     q_mult=q_mult, name=name)
    if cfg == 4:
        groups, seq = [], []
        n_groups = 8 if num_requests is None else max(1, num_requests // 16)
        for gi in range(n_groups):
            members = list(range(gi * 16, gi * 16 + 16))
            groups.append((members, 2048))
            seq.extend(2048 + int(t) + 1 for t in rng.integers(0, 512, size=16, endpoint=True))
        return build(seq, [1] * len(seq), Hq=32, Hkv=8, D=128, B=16,
                     kv_dtype=kv_dtype or "fp8", seed=seed, device=device, groups=groups,
                     q_mult=q_mult, name=name)
    if cfg == 5:
        R = 32 if num_requests is None else num_requests
        seq = [32768] * R
        ql = [2048 if r % 4 == 0 else 1 for r in range(R)]
        return build(seq, ql, Hq=64, Hkv=8, D=128, B=64, kv_dtype=kv_dtype or "bf16",
                     seed=seed, device=device, q_mult=q_mult,
                     name=f"{name}-{kv_dtype or 'bf16'}")
    raise ValueError(f"unknown config {cfg}")
