"""Reference model of the paged KV block allocator (host side).

TEST INFRASTRUCTURE ONLY. It states the allocation rules plainly so that the
tests can (a) check refcount / copy-on-write invariants and (b) derive the
block copies that the device must perform for a copy-on-write.

Rules followed:
  [vLLM-wiki "블록 테이블"]  memory is one pool of equal-size physical blocks; a
      request's block table maps logical block i to a physical block; a new
      physical block is taken only when the request's last block is full, so a
      request wastes at most the free tail of its last block.
  [vLLM-wiki "블록 공유와 쓰기 시 복사"]  every physical block carries a reference
      count; parallel samples point at the same prompt blocks; a shared block
      is copied only when a sequence must write a new token into it.
  [MRV2 "도입 체크리스트" / "2단계: 출력 계약"]  aborting or finishing a request
      must return its blocks.
"""
from dataclasses import dataclass, field
from typing import Dict, List, Optional, Tuple


class AllocatorError(RuntimeError):
    pass


@dataclass
class Sequence:
    blocks: List[int] = field(default_factory=list)
    length: int = 0  # tokens stored


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks < 0 or block_size <= 0:
            raise AllocatorError("bad pool geometry")
        self.num_blocks = num_blocks
        self.B = block_size
        self.refcount = [0] * num_blocks
        # lowest id first keeps the model deterministic
        self.free: List[int] = list(range(num_blocks - 1, -1, -1))
        self.seqs: Dict[int, Sequence] = {}

    # ----------------------------------------------------------- primitives
    def _take(self) -> int:
        if not self.free:
            raise AllocatorError("out of blocks")
        b = self.free.pop()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        if self.refcount[b] <= 0:
            raise AllocatorError(f"refcount underflow on block {b}")
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.append(b)

    # ------------------------------------------------------------ interface
    def add(self, seq_id: int, num_tokens: int) -> None:
        """Registers a sequence holding ``num_tokens`` tokens (its prompt)."""
        if seq_id in self.seqs:
            raise AllocatorError(f"sequence {seq_id} already live")
        s = Sequence()
        self.seqs[seq_id] = s
        for _ in range(num_tokens):
            self.append_slot(seq_id)

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (parallel sampling)."""
        if child in self.seqs:
            raise AllocatorError(f"sequence {child} already live")
        p = self.seqs[parent]
        for b in p.blocks:
            self.refcount[b] += 1
        self.seqs[child] = Sequence(list(p.blocks), p.length)

    def append_slot(self, seq_id: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserves the slot of the next token of ``seq_id``.

        Returns (slot, copy) where slot = block * B + offset and copy is
        (src, dst) when the write landed in a shared block that had to be
        copied first (copy-on-write), else None.
        """
        s = self.seqs[seq_id]
        off = s.length % self.B
        copy = None
        if off == 0:
            s.blocks.append(self._take())  # the last block is full (or none yet)
        else:
            last = s.blocks[-1]
            if self.refcount[last] > 1:  # shared: copy before writing into it
                fresh = self._take()
                self._release(last)
                s.blocks[-1] = fresh
                copy = (last, fresh)
        s.length += 1
        return s.blocks[-1] * self.B + off, copy

    def free_seq(self, seq_id: int) -> None:
        s = self.seqs.pop(seq_id)
        for b in s.blocks:
            self._release(b)

    # ----------------------------------------------------------- invariants
    def check(self) -> None:
        counts = [0] * self.num_blocks
        for s in self.seqs.values():
            if len(s.blocks) != -(-s.length // self.B):
                raise AllocatorError("a sequence holds more or fewer blocks than it needs")
            for b in s.blocks:
                counts[b] += 1
        if counts != self.refcount:
            raise AllocatorError("refcount differs from the number of table references")
        free = set(self.free)
        if len(free) != len(self.free):
            raise AllocatorError("a block is on the free list twice")
        used = {b for b in range(self.num_blocks) if counts[b] > 0}
        if free & used:
            raise AllocatorError("a referenced block is on the free list")
        if free | used != set(range(self.num_blocks)):
            raise AllocatorError("a block is neither free nor referenced")

    def table(self, seq_id: int) -> List[int]:
        return list(self.seqs[seq_id].blocks)

    def wasted_slots(self) -> int:
        """Free token slots inside allocated blocks (at most B-1 per sequence
        for unshared tails)."""
        used = {}
        for s in self.seqs.values():
            for i, b in enumerate(s.blocks):
                n = min(self.B, s.length - i * self.B)
                used[b] = max(used.get(b, 0), n)
        return sum(self.B - n for n in used.values())
