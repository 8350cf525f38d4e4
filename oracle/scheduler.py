"""Reference model of the host scheduler and block manager (plain Python).

TEST INFRASTRUCTURE ONLY: the native scheduler is checked against it step by
step. It never touches the GPU and never imports the product package.

The rules, from the pages:
  [V1-blog "고정 예산 기반 청크 분할 알고리즘"]  every step has a token budget;
      each running decode gets its one token first, and the rest of the budget
      goes to prefill chunks of min(remaining prompt, remaining budget, cap)
      tokens (the sketch uses a cap of 1024).
  [vLLM-wiki "블록 테이블"]  a request's blocks map logical to physical blocks;
      a physical block is taken only when a token lands past the last one.
  [vLLM-wiki "블록 공유와 쓰기 시 복사"]  blocks carry reference counts; a
      request that writes into a shared block first copies it.
  [vLLM-wiki "스케줄링과 선점"]  requests are served first come, first served;
      when blocks run out the latest-arrived request is preempted, all of its
      blocks at once, and later recomputed from scratch.
  [vLLM-wiki "엔진 구조와 주요 기능", automatic prefix caching]  a full block is
      keyed by (previous block's key, its tokens, extra ids such as a salt);
      a new request reuses the computed blocks of a matching prefix; only full
      blocks are cached, and blocks no longer referenced are evicted in LRU
      order.
  [MRV2 "재설계 1"]  a live request keeps a fixed persistent slot; a preempted
      request is registered again like a new one when it resumes.
  [MRV2 "재설계 3"]  the device block table receives only (row, start, values)
      diffs.

Where the pages leave a choice open, this model fixes one (the native
scheduler makes the same one): free blocks are a stack whose lowest id comes
out first, a request's blocks are released from its last block to its first,
the LRU evicts the block released longest ago, a free slot is the lowest free
id, a request preempted in a step is not admitted again in that step, the
whole prompt is never served from the cache (its last token is computed), and
the block written first in a step is copied before new blocks are taken.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple


class SchedError(RuntimeError):
    pass


@dataclass
class Request:
    rid: int
    tokens: List[int]
    prompt_len: int
    max_new: int
    salt: int
    arrival: int
    slot: int = -1
    blocks: List[int] = field(default_factory=list)
    num_computed: int = 0
    generated: int = 0
    caught_up: bool = False   # its last step computed all of its tokens
    dirty_from: int = 0       # first table entry the device row lacks
    keys: List[tuple] = field(default_factory=list)  # keys of its full blocks
    state: str = "waiting"


@dataclass
class Batch:
    req_ids: List[int]
    idx_mapping: List[int]
    num_scheduled: List[int]
    query_start_loc: List[int]
    seq_lens: List[int]
    positions: List[int]
    token_ids: List[int]
    slot_mapping: List[int]
    num_decode: int
    diff_rows: List[int]
    diff_starts: List[int]
    diff_val_offsets: List[int]
    diff_vals: List[int]
    copy_src: List[int]
    copy_dst: List[int]


class Scheduler:
    def __init__(self, num_blocks: int, block_size: int, max_reqs: int, max_blocks_per_req: int,
                 token_budget: int, chunk_cap: int = 1024, prefix_caching: bool = False):
        if min(num_blocks, block_size, max_reqs, max_blocks_per_req, token_budget,
               chunk_cap) <= 0:
            raise SchedError("bad configuration")
        self.B = block_size
        self.max_blocks = max_blocks_per_req
        self.budget = token_budget
        self.cap = chunk_cap
        self.caching = prefix_caching
        self.ref = [0] * num_blocks
        self.free = list(range(num_blocks - 1, -1, -1))  # pop() gives the lowest id first
        self.lru: List[int] = []                          # cached, unreferenced; [0] = oldest
        self.cache: Dict[tuple, int] = {}                 # key -> block
        self.block_key: Dict[int, tuple] = {}             # cached block -> key
        self.free_slots = list(range(max_reqs))
        self.reqs: Dict[int, Request] = {}
        self.waiting: List[Request] = []                  # by arrival
        self.running: List[Request] = []                  # by admission
        self.arrivals = 0
        self.last: Optional[List[Request]] = None         # entries of the last step
        self.stats = dict(steps=0, preemptions=0, prefix_hit_tokens=0, finished=0,
                          scheduled_tokens=0)
        self.finished: List[int] = []

    # ------------------------------------------------------------ allocator
    def _available(self) -> int:
        return len(self.free) + len(self.lru)

    def _take(self) -> int:
        if self.free:
            b = self.free.pop()
        elif self.lru:
            b = self.lru.pop(0)
            del self.cache[self.block_key.pop(b)]
        else:
            raise SchedError("out of blocks")
        assert self.ref[b] == 0
        self.ref[b] = 1
        return b

    def _incref(self, b: int) -> None:
        if self.ref[b] == 0:
            self.lru.remove(b)
        self.ref[b] += 1

    def _release(self, b: int) -> None:
        if self.ref[b] <= 0:
            raise SchedError(f"refcount underflow on block {b}")
        self.ref[b] -= 1
        if self.ref[b] == 0:
            if b in self.block_key:
                self.lru.append(b)
            else:
                self.free.append(b)

    def _release_all(self, r: Request) -> None:
        for b in reversed(r.blocks):
            self._release(b)
        r.blocks = []

    # -------------------------------------------------------------- requests
    def add_request(self, rid: int, prompt: List[int], max_new: int, salt: int = 0) -> None:
        if rid in self.reqs or not prompt or max_new < 1:
            raise SchedError("bad request")
        if len(prompt) + max_new > self.max_blocks * self.B:
            raise SchedError("request longer than a table row")
        r = Request(rid, list(prompt), len(prompt), max_new, salt, self.arrivals)
        self.arrivals += 1
        self.reqs[rid] = r
        self.waiting.append(r)

    def fork(self, parent: int, child: int, max_new: int) -> None:
        """The child shares every block of the running parent (parallel
        sampling); it gets a slot of its own."""
        p = self.reqs.get(parent)
        if p is None or p.state != "running" or child in self.reqs or not self.free_slots:
            raise SchedError("bad fork")
        c = Request(child, list(p.tokens), p.prompt_len, max_new, p.salt, self.arrivals)
        self.arrivals += 1
        c.blocks = list(p.blocks)
        for b in c.blocks:
            self._incref(b)
        c.num_computed, c.generated, c.caught_up = p.num_computed, p.generated, p.caught_up
        c.keys = list(p.keys)
        c.slot = self.free_slots.pop(0)
        c.state = "running"
        self.reqs[child] = c
        self.running.append(c)

    def abort(self, rid: int) -> None:
        r = self.reqs.pop(rid)
        if r.state == "running":
            self.running.remove(r)
            self._release_all(r)
            self._free_slot(r)
        elif r.state == "waiting":
            self.waiting.remove(r)
        r.state = "aborted"

    def _free_slot(self, r: Request) -> None:
        self.free_slots.append(r.slot)
        self.free_slots.sort()
        r.slot = -1

    def _preempt(self, r: Request) -> None:
        self.running.remove(r)
        self._release_all(r)
        self._free_slot(r)
        r.num_computed, r.caught_up, r.keys, r.dirty_from = 0, False, [], 0
        r.state = "waiting"
        i = 0
        while i < len(self.waiting) and self.waiting[i].arrival < r.arrival:
            i += 1
        self.waiting.insert(i, r)
        self.stats["preemptions"] += 1

    # ----------------------------------------------------------- step parts
    def _needed(self, r: Request, q: int) -> Tuple[int, bool]:
        nc = r.num_computed
        new = max(0, -(-(nc + q) // self.B) - len(r.blocks))
        cow = nc % self.B != 0 and nc // self.B < len(r.blocks) and \
            self.ref[r.blocks[nc // self.B]] > 1
        return new + (1 if cow else 0), cow

    def _fit(self, r: Request, q: int) -> int:
        """Largest q' <= q whose blocks can be had without preempting."""
        _, cow = self._needed(r, q)
        avail = self._available() - (1 if cow else 0)
        if avail < 0:
            return 0
        most = (len(r.blocks) + avail) * self.B - r.num_computed
        return max(0, min(q, most))

    def _ensure(self, r: Request, q: int, copies: List[Tuple[int, int]]) -> None:
        need, cow = self._needed(r, q)
        assert need <= self._available()
        if cow:
            i = r.num_computed // self.B
            old = r.blocks[i]
            new = self._take()
            self._release(old)
            r.blocks[i] = new
            copies.append((old, new))
            r.dirty_from = min(r.dirty_from, i)
        while len(r.blocks) * self.B < r.num_computed + q:
            r.blocks.append(self._take())

    def _key(self, r: Request, i: int) -> tuple:
        prev = r.keys[i - 1] if i > 0 else None
        return (prev, tuple(r.tokens[i * self.B:(i + 1) * self.B]), r.salt)

    # ------------------------------------------------------------------ step
    def step(self) -> Batch:
        if self.last is not None:
            raise SchedError("commit the previous step first")
        budget = self.budget
        entries: List[Tuple[Request, int]] = []
        scheduled = set()
        preempted_now = set()
        copies: List[Tuple[int, int]] = []
        # 1. one token for every running decode, first
        for r in list(self.running):
            if r.state != "running" or not (r.caught_up and len(r.tokens) - r.num_computed == 1):
                continue
            if budget < 1:
                break
            while self._needed(r, 1)[0] > self._available():
                cand = [x for x in self.running if x.rid not in scheduled]
                victim = max(cand, key=lambda x: x.arrival)
                self._preempt(victim)
                preempted_now.add(victim.rid)
                if victim is r:
                    break
            if r.state != "running":
                continue
            self._ensure(r, 1, copies)
            entries.append((r, 1))
            scheduled.add(r.rid)
            budget -= 1
        num_decode = len(entries)
        # 2. prefill chunks: requests already running, then admissions (FCFS)
        for r in list(self.running):
            if budget <= 0:
                break
            if r.rid in scheduled or r.caught_up:
                continue
            q = self._fit(r, min(len(r.tokens) - r.num_computed, budget, self.cap))
            if q <= 0:
                continue
            self._ensure(r, q, copies)
            entries.append((r, q))
            scheduled.add(r.rid)
            budget -= q
        while self.waiting and budget > 0 and self.free_slots:
            r = self.waiting[0]
            if r.rid in preempted_now:
                break
            hits: List[int] = []
            keys: List[tuple] = []
            if self.caching:
                for i in range((len(r.tokens) - 1) // self.B):
                    key = (keys[-1] if keys else None,
                           tuple(r.tokens[i * self.B:(i + 1) * self.B]), r.salt)
                    b = self.cache.get(key)
                    if b is None:
                        break
                    hits.append(b)
                    keys.append(key)
            for b in hits:
                self._incref(b)
            r.blocks, r.keys, r.num_computed = hits, keys, len(hits) * self.B
            q = self._fit(r, min(len(r.tokens) - r.num_computed, budget, self.cap))
            if q <= 0:
                self._release_all(r)
                r.keys, r.num_computed = [], 0
                break
            self.waiting.pop(0)
            r.slot = self.free_slots.pop(0)
            r.state = "running"
            r.dirty_from = 0
            self.running.append(r)
            self.stats["prefix_hit_tokens"] += r.num_computed
            self._ensure(r, q, copies)
            entries.append((r, q))
            scheduled.add(r.rid)
            budget -= q
        # 3. the batch
        b = Batch([], [], [], [0], [], [], [], [], num_decode, [], [], [0], [], [], [])
        for r, q in entries:
            nc = r.num_computed
            b.req_ids.append(r.rid)
            b.idx_mapping.append(r.slot)
            b.num_scheduled.append(q)
            b.query_start_loc.append(b.query_start_loc[-1] + q)
            b.seq_lens.append(nc + q)
            for p in range(nc, nc + q):
                b.positions.append(p)
                b.token_ids.append(r.tokens[p])
                b.slot_mapping.append(r.blocks[p // self.B] * self.B + p % self.B)
            r.num_computed = nc + q
            r.caught_up = r.num_computed == len(r.tokens)
            if self.caching:
                for i in range(len(r.keys), r.num_computed // self.B):
                    key = self._key(r, i)
                    r.keys.append(key)
                    blk = r.blocks[i]
                    if key not in self.cache and blk not in self.block_key:
                        self.cache[key] = blk
                        self.block_key[blk] = key
            if r.dirty_from < len(r.blocks):
                b.diff_rows.append(r.slot)
                b.diff_starts.append(r.dirty_from)
                b.diff_vals.extend(r.blocks[r.dirty_from:])
                b.diff_val_offsets.append(len(b.diff_vals))
                r.dirty_from = len(r.blocks)
        b.copy_src = [s for s, _ in copies]
        b.copy_dst = [d for _, d in copies]
        self.last = [r for r, _ in entries]
        self.stats["steps"] += 1
        self.stats["scheduled_tokens"] += b.query_start_loc[-1]
        return b

    def commit(self, sampled: List[int]) -> List[int]:
        """Appends the sampled token of every entry that computed all of its
        tokens; returns the requests that finished."""
        if self.last is None or len(sampled) != len(self.last):
            raise SchedError("commit does not match the last step")
        done = []
        for r, t in zip(self.last, sampled):
            if r.state != "running" or not r.caught_up:
                continue
            r.tokens.append(int(t))
            r.generated += 1
            if r.generated >= r.max_new:
                self.running.remove(r)
                self._release_all(r)
                self._free_slot(r)
                r.state = "finished"
                del self.reqs[r.rid]
                done.append(r.rid)
        self.last = None
        self.stats["finished"] += len(done)
        self.finished.extend(done)
        return done

    # ------------------------------------------------------------ inspection
    def table(self, rid: int) -> List[int]:
        return list(self.reqs[rid].blocks)

    def block_usage(self) -> Tuple[int, int]:
        """(blocks referenced, token slots holding stored K/V in them)."""
        fill: Dict[int, int] = {}
        for r in self.running:
            for i, blk in enumerate(r.blocks):
                n = max(0, min(self.B, r.num_computed - i * self.B))
                fill[blk] = max(fill.get(blk, 0), n)
        return len(fill), sum(fill.values())

    def check(self) -> None:
        counts = [0] * len(self.ref)
        for r in self.running:
            if len(r.blocks) != -(-r.num_computed // self.B):
                raise SchedError(f"request {r.rid} holds {len(r.blocks)} blocks for "
                                 f"{r.num_computed} tokens")
            for blk in r.blocks:
                counts[blk] += 1
        if counts != self.ref:
            raise SchedError("refcount differs from the number of table references")
        free, lru = set(self.free), set(self.lru)
        used = {i for i, c in enumerate(counts) if c}
        if len(free) != len(self.free) or len(lru) != len(self.lru) or free & lru or \
                (free | lru) & used or free | lru | used != set(range(len(self.ref))):
            raise SchedError("free, cached and used blocks do not partition the pool")
        if set(self.block_key) != set(self.cache.values()) or lru - set(self.block_key):
            raise SchedError("cache map and cached blocks disagree")
        slots = [r.slot for r in self.running]
        if len(set(slots)) != len(slots) or set(slots) & set(self.free_slots):
            raise SchedError("a persistent slot is used twice")
