"""The reference scheduler against the pages' rules: decode-first token
budget with capped prefill chunks, FCFS admission, preemption of the latest
arrival with recompute, copy-on-write after a fork, prefix reuse of full
blocks with LRU eviction, and diffs / slots that rebuild the tables and agree
with the (separately pinned) input-prep reference."""
import numpy as np
import pytest

from oracle import oracle as O
from oracle.input_prep import prepare_inputs
from oracle.scheduler import SchedError, Scheduler


def _prompt(rng, n, vocab=50000):
    return rng.integers(0, vocab, size=n).tolist()


def _run_to_decode(s, steps=50):
    """Steps until every admitted request is decoding; returns the batches."""
    out = []
    for _ in range(steps):
        b = s.step()
        out.append(b)
        s.commit([7] * len(b.req_ids))
        if not s.waiting and all(r.caught_up for r in s.running):
            break
    return out


def test_budget_gives_decodes_first_then_capped_chunks():
    rng = np.random.default_rng(0)
    s = Scheduler(num_blocks=4096, block_size=16, max_reqs=256, max_blocks_per_req=512,
                  token_budget=4096, chunk_cap=1024)
    for i in range(64):
        s.add_request(i, _prompt(rng, 100), 50)
    _run_to_decode(s)
    assert len(s.running) == 64 and all(r.caught_up for r in s.running)
    for i, n in enumerate([1024, 1024, 5000, 3000]):
        s.add_request(100 + i, _prompt(rng, n), 10)
    b = s.step()
    assert b.num_decode == 64 and b.num_scheduled[:64] == [1] * 64
    # chunks: min(remaining prompt, remaining budget, 1024), in arrival order
    assert b.num_scheduled[64:] == [1024, 1024, 1024, 4096 - 64 - 3 * 1024]
    assert b.query_start_loc[-1] == 4096
    s.check()


def test_mixed_step_of_the_chunked_prefill_config():
    """64 decodes + chunks of 1024, 1024 and 1920 tokens fit a 4096 budget
    with a 2048 cap: 4032 tokens."""
    rng = np.random.default_rng(1)
    s = Scheduler(8192, 16, 256, 1024, 4096, chunk_cap=2048)
    for i in range(64):
        s.add_request(i, _prompt(rng, 30), 20)
    _run_to_decode(s)
    for i, n in enumerate([1024, 1024, 1920]):
        s.add_request(100 + i, _prompt(rng, n), 5)
    b = s.step()
    assert b.num_scheduled == [1] * 64 + [1024, 1024, 1920]
    assert b.query_start_loc[-1] == 4032


def test_decodes_alone_can_exhaust_the_budget():
    """With a budget of 10, ten decoding requests take the whole step: the
    prompts behind them wait (decode first, never delayed)."""
    rng = np.random.default_rng(2)
    s = Scheduler(1024, 16, 64, 64, token_budget=10)
    for i in range(12):
        s.add_request(i, _prompt(rng, 5), 900)
    for _ in range(30):
        b = s.step()
        s.commit([7] * len(b.req_ids))
    assert [r.rid for r in s.running] == list(range(10))
    assert [r.rid for r in s.waiting] == [10, 11]
    b = s.step()
    assert b.num_decode == 10 and b.req_ids == list(range(10))


def test_admissions_follow_arrival_order():
    """First come, first served: every admission takes the earliest-arrived
    waiting request (preempted requests keep their arrival and go back in
    front of later ones)."""
    rng = np.random.default_rng(3)
    s = Scheduler(num_blocks=60, block_size=16, max_reqs=6, max_blocks_per_req=40,
                  token_budget=96, chunk_cap=64)
    rid = 0
    for step in range(300):
        if rng.random() < 0.5:
            s.add_request(rid, _prompt(rng, int(rng.integers(1, 200))), int(rng.integers(1, 80)))
            rid += 1
        waiting_before = [(r.arrival, r.rid) for r in s.waiting]
        running_before = {r.rid for r in s.running}
        b = s.step()
        admitted = [r for r in b.req_ids if r not in running_before]
        preempted = running_before - {r.rid for r in s.running}
        order = [x for x in sorted(waiting_before) if x[1] not in preempted]
        assert [x[1] for x in order[:len(admitted)]] == admitted
        s.commit([3] * len(b.req_ids))
        s.check()


def test_preemption_takes_the_latest_arrival_and_recomputes():
    rng = np.random.default_rng(4)
    s = Scheduler(num_blocks=12, block_size=16, max_reqs=8, max_blocks_per_req=12,
                  token_budget=256)
    prompts = {i: _prompt(rng, 60) for i in range(3)}
    for i in range(3):
        s.add_request(i, prompts[i], 40)      # 3 x 4 blocks after the prompt
    seen_preempt = False
    tokens = {i: [] for i in range(3)}
    for step in range(200):
        if not s.reqs:
            break
        before = {r.rid for r in s.running}
        b = s.step()
        after = {r.rid for r in s.running}
        if before - after:
            seen_preempt = True
            assert max(before - after) == max(before)  # the latest arrival goes first
        sampled = [1000 + step] * len(b.req_ids)
        s.commit(sampled)
        s.check()
    assert seen_preempt and not s.reqs and s.stats["finished"] == 3


def test_fork_shares_blocks_and_copies_the_partial_block_on_write():
    rng = np.random.default_rng(5)
    s = Scheduler(64, 16, 8, 16, 512)
    s.add_request(0, _prompt(rng, 40), 5)     # 2 full blocks + 8 tokens
    b = s.step()
    s.commit([11])
    parent_blocks = s.table(0)
    s.fork(0, 1, 5)
    s.fork(0, 2, 5)
    assert all(s.ref[blk] == 3 for blk in parent_blocks)
    b = s.step()                               # three decodes write position 40
    assert b.num_decode == 3
    # the first two writers copy the shared partial block; the last one keeps it
    assert b.copy_src == [parent_blocks[2]] * 2 and len(set(b.copy_dst)) == 2
    assert s.table(0)[:2] == s.table(1)[:2] == s.table(2)[:2] == parent_blocks[:2]
    assert s.table(2)[2] == parent_blocks[2]
    s.check()


def test_prefix_reuse_of_full_blocks_and_lru_eviction():
    rng = np.random.default_rng(6)
    B = 16
    s = Scheduler(num_blocks=40, block_size=B, max_reqs=8, max_blocks_per_req=40,
                  token_budget=2048, prefix_caching=True)
    shared = _prompt(rng, 100)                 # 6 full blocks + 4 tokens
    s.add_request(0, shared, 1)
    b = s.step()
    s.commit([5])                              # finishes: blocks go to the LRU, cached
    assert s.stats["finished"] == 1 and len(s.lru) == 6
    s.add_request(1, shared + [1, 2, 3], 1)
    b = s.step()
    assert s.stats["prefix_hit_tokens"] == 6 * B
    assert b.positions[0] == 6 * B and b.num_scheduled == [103 - 96]
    s.commit([5])
    # another salt shares nothing
    s.add_request(2, shared, 1, salt=9)
    s.step()
    s.commit([5])
    assert s.stats["prefix_hit_tokens"] == 6 * B
    # a prompt of exactly 6 full blocks reuses at most 5 (its last token is computed)
    s.add_request(3, shared[:96], 1)
    s.step()
    assert s.stats["prefix_hit_tokens"] == 6 * B + 5 * B
    s.commit([5])
    s.check()
    # exhaust the pool: cached unreferenced blocks are evicted oldest first
    lru_before = list(s.lru)
    s.add_request(4, _prompt(rng, 39 * B), 1)
    s.step()
    evicted = [blk for blk in lru_before if blk not in s.lru]
    assert evicted == lru_before[:len(evicted)] and evicted
    s.check()


def test_diffs_rebuild_tables_and_slots_agree_with_input_prep():
    rng = np.random.default_rng(7)
    B, max_reqs, mb = 16, 32, 64
    s = Scheduler(num_blocks=300, block_size=B, max_reqs=max_reqs, max_blocks_per_req=mb,
                  token_budget=300, chunk_cap=128, prefix_caching=True)
    mirror = np.full((max_reqs, mb), -1, np.int32)
    nc = [0] * max_reqs
    rid = 0
    common = _prompt(rng, 70)
    for step in range(120):
        if rng.random() < 0.3:
            p = common + _prompt(rng, int(rng.integers(1, 200))) if rng.random() < 0.5 \
                else _prompt(rng, int(rng.integers(1, 300)))
            s.add_request(rid, p, int(rng.integers(1, 60)))
            rid += 1
        if rng.random() < 0.1 and s.running:
            par = s.running[int(rng.integers(0, len(s.running)))]
            if par.caught_up and s.free_slots:
                s.fork(par.rid, rid, int(rng.integers(1, 30)))
                rid += 1
        b = s.step()
        table_before = mirror.copy()
        gathered = O.apply_staged_writes(mirror, np.array(b.diff_rows, np.int32),
                                         np.array(b.diff_starts, np.int32),
                                         np.array(b.diff_val_offsets, np.int32),
                                         np.array(b.diff_vals, np.int32),
                                         np.array(b.idx_mapping, np.int32))
        for i, r in enumerate(b.req_ids):
            n = len(s.table(r))
            assert mirror[b.idx_mapping[i], :n].tolist() == s.table(r)
            assert gathered[i, :n].tolist() == s.table(r)
        # slots of the batch = input prep over the rebuilt table and the slot state
        for i, r in enumerate(b.req_ids):
            nc[b.idx_mapping[i]] = b.seq_lens[i] - b.num_scheduled[i]
        qsl, seq, pos, slots, _ = prepare_inputs(nc, mirror.tolist(), B, 300, b.idx_mapping,
                                                 b.num_scheduled)
        assert qsl == b.query_start_loc and seq == b.seq_lens
        assert pos == b.positions and slots == b.slot_mapping
        s.commit(rng.integers(0, 50000, size=len(b.req_ids)).tolist())
        s.check()
        used, stored = s.block_usage()
        assert used * B - stored <= (B - 1) * len(s.running)  # only last blocks have gaps
        del table_before


def test_bad_calls():
    s = Scheduler(16, 16, 2, 4, 64)
    with pytest.raises(SchedError):
        s.add_request(0, [], 1)
    with pytest.raises(SchedError):
        s.add_request(0, [1] * 60, 5)              # longer than a 4-block row
    s.add_request(0, [1, 2], 1)
    with pytest.raises(SchedError):
        s.add_request(0, [1], 1)
    s.step()
    with pytest.raises(SchedError):
        s.step()                                   # commit first
    with pytest.raises(SchedError):
        s.commit([1, 2])
