"""Reference of the device-side step-input preparation (host side, plain Python).

TEST INFRASTRUCTURE ONLY: used by the tests to check the CUDA input-prep
kernel. It never touches the GPU and never imports the product package.

[MRV2 "재설계 1"]: a live request keeps a fixed persistent slot; the step's
order is given by idx_mapping (entry i of the batch is slot idx_mapping[i]).
[MRV2 "재설계 4"]: query_start_loc is the running sum of the per-request token
counts, and positions, seq_lens and the slot mapping are built from the
per-slot state (the GPU does it there).
[vLLM-wiki "블록 테이블"]: token position p of a request lives in logical block
p // B at offset p % B; its slot in the pool is physical_block * B + offset.
"""
from typing import List, Sequence, Tuple


class PrepError(RuntimeError):
    pass


def prepare_inputs(num_computed: Sequence[int], table: Sequence[Sequence[int]], block_size: int,
                   num_blocks: int, idx_mapping: Sequence[int], num_scheduled: Sequence[int]
                   ) -> Tuple[List[int], List[int], List[int], List[int], List[int]]:
    """One step's inputs.

    num_computed[s]  tokens of slot s whose K/V are already stored
    table[s][i]      physical block of logical block i of slot s
    idx_mapping[i]   slot of batch entry i; num_scheduled[i] its token count

    Returns (query_start_loc [R+1], seq_lens [R], positions [T], slot_mapping [T],
    num_computed after the step). Raises PrepError on an entry that points
    outside the slots, a negative count, or a position whose block is missing
    or outside the pool.
    """
    B = block_size
    R = len(idx_mapping)
    if len(num_scheduled) != R:
        raise PrepError("idx_mapping and num_scheduled differ in length")
    nc = list(num_computed)
    qsl = [0]
    seq_lens, positions, slots = [], [], []
    seen = set()
    for i in range(R):
        s, q = idx_mapping[i], num_scheduled[i]
        if not 0 <= s < len(nc) or q < 0 or s in seen:
            raise PrepError(f"entry {i}: slot {s}, count {q}")
        seen.add(s)
        start = nc[s]
        for j in range(q):
            pos = start + j
            lb = pos // B
            if lb >= len(table[s]):
                raise PrepError(f"entry {i}: position {pos} past the table row")
            blk = table[s][lb]
            if not 0 <= blk < num_blocks:
                raise PrepError(f"entry {i}: block {blk} outside the pool")
            positions.append(pos)
            slots.append(blk * B + pos % B)
        seq_lens.append(start + q)
        nc[s] = start + q
        qsl.append(qsl[-1] + q)
    return qsl, seq_lens, positions, slots, nc
