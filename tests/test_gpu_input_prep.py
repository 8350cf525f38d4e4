"""GPU parity of pa_prepare_inputs against the input-prep reference (integer
work: bit-exact), over multi-step schedules whose slots come from the
reference allocator, batches of more than one scan chunk, and bad input."""
import numpy as np
import pytest
import torch

from oracle.block_manager import BlockManager
from oracle.input_prep import prepare_inputs as ref_prepare
from paged_kv_cache_143_gb300 import pa

pytestmark = pytest.mark.gpu

MAX_REQS, MAX_BLOCKS, B, NUM_BLOCKS = 1024, 128, 16, 65536


def _dev(a, dtype=torch.int32):
    return torch.from_numpy(np.ascontiguousarray(a)).to(dtype).cuda()


def _run(nc_dev, table_dev, idx, q, cap):
    R = len(idx)
    qsl = torch.full((R + 1,), -9, dtype=torch.int32, device="cuda")
    seq = torch.full((max(R, 1),), -9, dtype=torch.int32, device="cuda")[:R]
    pos = torch.full((cap + 64,), -9, dtype=torch.int32, device="cuda")
    slots = torch.full((cap + 64,), -9, dtype=torch.int64, device="cuda")
    pa.prepare_inputs(nc_dev, table_dev, B, NUM_BLOCKS, _dev(np.array(idx, np.int32)),
                      _dev(np.array(q, np.int32)), qsl, seq, pos[:cap], slots[:cap])
    return qsl, seq, pos, slots


@pytest.mark.parametrize("seed", [0, 1])
def test_multi_step_schedule_bit_exact(cuda_device, seed):
    rng = np.random.default_rng(seed)
    bm = BlockManager(NUM_BLOCKS, B)
    prompt = {}
    for s in rng.choice(MAX_REQS, size=200, replace=False):
        prompt[int(s)] = int(rng.integers(1, 1500))
        bm.add(int(s), 0)
    nc = np.zeros(MAX_REQS, np.int32)
    nc_dev = _dev(nc)
    stored = {s: 0 for s in prompt}
    for step in range(6):
        order = [s for s in prompt if rng.random() < 0.7]
        rng.shuffle(order)
        idx, q = [], []
        for s in order:
            rem = prompt[s] - stored[s]
            n = int(min(rem, rng.integers(1, 600))) if rem > 0 else 1
            if step == 3 and rng.random() < 0.1:
                n = 0  # an entry with nothing this step
            for _ in range(n):
                bm.append_slot(s)
            stored[s] += n
            idx.append(s)
            q.append(n)
        table = np.full((MAX_REQS, MAX_BLOCKS), -1, np.int32)
        for s in prompt:
            row = bm.table(s)
            table[s, :len(row)] = row
        ref = ref_prepare(nc, table.tolist(), B, NUM_BLOCKS, idx, q)
        T = ref[0][-1]
        qsl, seq, pos, slots = _run(nc_dev, _dev(table), idx, q, T)
        assert pa.get_error() == pa.PA_OK
        assert qsl.cpu().tolist() == ref[0]
        assert seq.cpu().tolist() == ref[1]
        assert pos[:T].cpu().tolist() == ref[2]
        assert slots[:T].cpu().tolist() == ref[3]
        assert (pos[T:] == -9).all() and (slots[T:] == -9).all()
        nc = np.array(ref[4], np.int32)
        assert nc_dev.cpu().numpy().tolist() == nc.tolist()


def test_many_entries_span_scan_chunks(cuda_device):
    """3000 decode entries (three 1024-entry scan chunks) plus a long chunk."""
    rng = np.random.default_rng(7)
    max_reqs = 4096
    nc = rng.integers(0, 1000, size=max_reqs).astype(np.int32)
    table = rng.integers(0, NUM_BLOCKS, size=(max_reqs, MAX_BLOCKS)).astype(np.int32)
    idx = rng.permutation(max_reqs)[:3001].astype(np.int32)
    q = np.ones(3001, np.int32)
    q[1500] = 700
    ref = ref_prepare(nc.tolist(), table.tolist(), B, NUM_BLOCKS, idx.tolist(), q.tolist())
    nc_dev = _dev(nc)
    T = ref[0][-1]
    qsl, seq, pos, slots = _run(nc_dev, _dev(table), idx.tolist(), q.tolist(), T)
    assert pa.get_error() == pa.PA_OK
    assert qsl.cpu().tolist() == ref[0]
    assert seq.cpu().tolist() == ref[1]
    assert pos[:T].cpu().tolist() == ref[2] and slots[:T].cpu().tolist() == ref[3]
    assert nc_dev.cpu().tolist() == ref[4]


def test_bad_input_is_flagged_and_bounded(cuda_device):
    table = np.full((MAX_REQS, MAX_BLOCKS), -1, np.int32)
    table[3, :2] = [10, 11]
    nc_dev = _dev(np.zeros(MAX_REQS, np.int32))
    # a position whose block is missing: slot -1, flagged
    qsl, seq, pos, slots = _run(nc_dev, _dev(table), [3], [40], 40)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    s = slots[:40].cpu().tolist()
    assert s[:32] == [10 * 16 + i for i in range(16)] + [11 * 16 + i for i in range(16)]
    assert s[32:] == [-1] * 8
    # a slot outside the table: flagged, nothing written for it
    nc_dev = _dev(np.zeros(MAX_REQS, np.int32))
    qsl, seq, pos, slots = _run(nc_dev, _dev(table), [MAX_REQS + 3], [5], 5)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert (slots == -9).all() and qsl.cpu().tolist() == [0, 0]
    # more tokens than the output holds: flagged, writes stop at the capacity
    nc_dev = _dev(np.zeros(MAX_REQS, np.int32))
    qsl, seq, pos, slots = _run(nc_dev, _dev(table), [3], [20], 8)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert (slots[8:] == -9).all() and slots[:8].cpu().tolist() == [160 + i for i in range(8)]
