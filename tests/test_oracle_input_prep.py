"""The input-prep reference against an independent source of slots: the
oracle allocator hands out the slot of every token it stores
([vLLM-wiki "블록 테이블"]), so a simulated schedule of prefill chunks and
decode tokens fixes what positions, seq_lens and the slot mapping must be."""
import numpy as np
import pytest

from oracle.block_manager import BlockManager
from oracle.input_prep import PrepError, prepare_inputs


def _simulate(seed, steps=12, max_reqs=16, B=16):
    rng = np.random.default_rng(seed)
    bm = BlockManager(4096, B)
    prompts = {}
    nc = [0] * max_reqs
    live = {}
    for s in rng.choice(max_reqs, size=6, replace=False):
        prompts[int(s)] = int(rng.integers(1, 300))
        bm.add(int(s), 0)
        live[int(s)] = 0
    for _ in range(steps):
        order = [s for s in live if rng.random() < 0.8]
        rng.shuffle(order)
        idx, q, expect_slots = [], [], []
        for s in order:
            remaining = prompts[s] - live[s]
            n = int(min(remaining, rng.integers(1, 130))) if remaining > 0 else 1
            for _ in range(n):
                slot, _ = bm.append_slot(s)
                expect_slots.append(slot)
            idx.append(s)
            q.append(n)
            live[s] += n
        table = [bm.table(s) if s in live else [] for s in range(max_reqs)]
        table = [row + [-1] * (64 - len(row)) for row in table]
        qsl, seq, pos, slots, nc2 = prepare_inputs(nc, table, B, 4096, idx, q)
        yield idx, q, qsl, seq, pos, slots, nc, nc2, expect_slots, live


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_slots_match_the_allocator(seed):
    for idx, q, qsl, seq, pos, slots, nc, nc2, expect, live in _simulate(seed):
        assert slots == expect
        assert qsl == [0] + list(np.cumsum(q))
        assert seq == [live[s] for s in idx]
        assert pos == [p for s, n in zip(idx, q) for p in range(live[s] - n, live[s])]
        for s in idx:
            assert nc2[s] == live[s]
        nc[:] = nc2


def test_errors():
    table = [[3, 5, -1, -1], [7, -1, -1, -1]]
    with pytest.raises(PrepError):
        prepare_inputs([0, 0], table, 16, 8, [2], [1])         # slot outside
    with pytest.raises(PrepError):
        prepare_inputs([0, 0], table, 16, 8, [0, 0], [1, 1])   # same slot twice
    with pytest.raises(PrepError):
        prepare_inputs([30, 0], table, 16, 8, [0], [3])         # block -1
    with pytest.raises(PrepError):
        prepare_inputs([0, 0], [[9, -1, -1, -1]], 16, 8, [0], [1])  # block past pool
    qsl, seq, pos, slots, nc = prepare_inputs([0, 17], table, 16, 8, [1, 0], [0, 2])
    assert qsl == [0, 0, 2] and seq == [17, 2] and pos == [0, 1] and slots == [48, 49]
