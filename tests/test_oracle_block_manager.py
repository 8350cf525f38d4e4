"""Refcount and copy-on-write invariants of the allocator model
([vLLM-wiki "블록 테이블", "블록 공유와 쓰기 시 복사"]), and the end-to-end CoW
data check through the oracle's pool operations."""
import numpy as np
import pytest

from oracle import oracle as O
from oracle.block_manager import AllocatorError, BlockManager


def test_allocation_on_demand_wastes_at_most_one_partial_block():
    bm = BlockManager(64, 16)
    bm.add(0, 1)
    assert len(bm.table(0)) == 1
    for _ in range(15):
        bm.append_slot(0)
    assert len(bm.table(0)) == 1  # 16 tokens fill one block
    bm.append_slot(0)
    assert len(bm.table(0)) == 2  # the 17th takes a new block
    bm.add(1, 100)
    assert bm.wasted_slots() == (16 - 17 % 16) + (16 - 100 % 16)
    bm.check()


def test_fork_shares_blocks_and_cow_copies_only_the_partial_block():
    bm = BlockManager(32, 16)
    bm.add(0, 40)  # 2 full blocks + 8 tokens
    for c in range(1, 4):
        bm.fork(0, c)
    shared = bm.table(0)
    assert all(bm.refcount[b] == 4 for b in shared)
    slot, copy = bm.append_slot(2)
    assert copy is not None and copy[0] == shared[-1]
    assert bm.table(2)[:2] == shared[:2] and bm.table(2)[2] == copy[1]
    assert slot == copy[1] * 16 + 8
    assert bm.refcount[shared[-1]] == 3 and bm.refcount[copy[1]] == 1
    bm.check()
    # a second write by the same sequence no longer copies
    _, copy2 = bm.append_slot(2)
    assert copy2 is None
    bm.check()


def test_aligned_prefix_never_copies():
    """A prompt that ends on a block boundary leaves nothing to copy: the next
    token opens a fresh private block (the prefix-shared decode workload)."""
    bm = BlockManager(512, 16)
    bm.add(0, 2048)
    for c in range(1, 16):
        bm.fork(0, c)
    for c in range(16):
        _, copy = bm.append_slot(c)
        assert copy is None
    assert all(bm.refcount[b] == 16 for b in bm.table(0)[:128])
    bm.check()


def test_free_returns_every_block_and_underflow_is_caught():
    bm = BlockManager(16, 4)
    bm.add(0, 9)
    bm.fork(0, 1)
    bm.append_slot(1)
    bm.free_seq(0)
    bm.free_seq(1)
    bm.check()
    assert sorted(bm.free) == list(range(16))
    with pytest.raises(AllocatorError):
        bm._release(3)
    with pytest.raises(AllocatorError):
        BlockManager(2, 4).add(0, 9)


def test_cow_data_other_sharers_unchanged():
    """After copy-on-write the writer sees the old tokens plus its new one; the
    other sharers see their data unchanged."""
    B, Hkv, D = 4, 2, 8
    bm = BlockManager(8, B)
    pool = O.Pool(np.full((8, Hkv, B, D), 0x7FC0, np.uint16),
                  np.full((8, Hkv, B, D), 0x7FC0, np.uint16), B, O.BF16)
    rng = np.random.default_rng(0)
    bm.add(0, 0)
    toks = []
    for _ in range(6):  # 1 full block + 2 tokens
        s, c = bm.append_slot(0)
        assert c is None
        kv = rng.integers(0, 0x3F00, size=(1, Hkv, D)).astype(np.uint16)
        toks.append(kv)
        O.write_kv(pool, kv, kv, np.array([s], np.int64))
    bm.fork(0, 1)
    parent_before = pool.k[bm.table(0)].copy()
    s, c = bm.append_slot(1)
    O.copy_blocks(pool, [c[0]], [c[1]])
    new = rng.integers(0, 0x3F00, size=(1, Hkv, D)).astype(np.uint16)
    O.write_kv(pool, new, new, np.array([s], np.int64))
    np.testing.assert_array_equal(pool.k[bm.table(0)], parent_before)
    child = pool.k[bm.table(1)]
    np.testing.assert_array_equal(child[0], parent_before[0])
    np.testing.assert_array_equal(child[1][:, :2], parent_before[1][:, :2])
    np.testing.assert_array_equal(child[1][:, 2], new[0])
    bm.check()


hyp = pytest.importorskip("hypothesis")
st = hyp.strategies


@hyp.settings(max_examples=60, deadline=None)
@hyp.given(st.lists(st.tuples(st.sampled_from(["add", "fork", "append", "free"]),
                              st.integers(0, 7), st.integers(0, 7), st.integers(0, 40)),
                    max_size=60),
           st.sampled_from([1, 2, 4, 16]))
def test_random_operation_sequences_keep_invariants(ops, B):
    bm = BlockManager(48, B)
    for op, a, b, n in ops:
        try:
            if op == "add" and a not in bm.seqs:
                bm.add(a, n)
            elif op == "fork" and a in bm.seqs and b not in bm.seqs:
                bm.fork(a, b)
            elif op == "append" and a in bm.seqs:
                bm.append_slot(a)
            elif op == "free" and a in bm.seqs:
                bm.free_seq(a)
        except AllocatorError as e:
            # running out of blocks leaves every table consistent (the failed
            # token is simply not stored)
            assert "out of blocks" in str(e)
        bm.check()
    for s in list(bm.seqs):
        bm.free_seq(s)
    bm.check()
    assert len(bm.free) == 48
