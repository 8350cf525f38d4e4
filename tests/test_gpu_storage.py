"""GPU parity of the integer / byte side of the hot path against the oracle,
through the C ABI: KV write (bf16 copy, FP8 store), staged block-table diffs
and gather, block copy. All bit-exact."""
import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import gpu_cache, new_gpu_pool, pool_bits
from tests.helpers import bits, oracle_pool

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cfg,kw", [
    (1, {}),
    (4, {"num_requests": 32}),
    (3, {"num_requests": 8}),
    (5, {"num_requests": 4, "kv_dtype": "fp8"}),
])
def test_write_kv_pool_bit_exact(cuda_device, cfg, kw):
    w = workloads.make(cfg, device=cuda_device, **kw)
    pool = gpu_cache(w, cuda_device)
    pa.write_kv(pool, w.new_k, w.new_v, w.slot_mapping)
    assert pa.get_error() == pa.PA_OK
    ref = oracle_pool(w)
    gk, gv = pool_bits(pool)
    np.testing.assert_array_equal(gk, ref.k)
    np.testing.assert_array_equal(gv, ref.v)


def test_write_kv_decode_config_bit_exact(cuda_device):
    w = workloads.make(2, device=cuda_device, num_requests=24)
    pool = gpu_cache(w, cuda_device)
    pa.write_kv(pool, w.new_k, w.new_v, w.slot_mapping)
    ref = oracle_pool(w)
    gk, gv = pool_bits(pool)
    np.testing.assert_array_equal(gk, ref.k)
    np.testing.assert_array_equal(gv, ref.v)


@pytest.mark.parametrize("scale", [1.0, 0.37, 0.011858259])
def test_fp8_store_all_bf16_patterns(cuda_device, scale):
    """Every one of the 65,536 bf16 bit patterns stored as E4M3 at three
    scales equals the oracle's encode (RNE, satfinite, NaN -> 0x7F)."""
    patterns = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    D, Hkv = 128, 1
    T = patterns.size // D
    x = torch.from_numpy(patterns.view(np.int16).reshape(T, Hkv, D)).view(torch.bfloat16)
    # B = 16 blocks: token t -> block t // 16, offset t % 16
    k = torch.zeros((T // 16, 1, 16, D), dtype=torch.uint8, device=cuda_device)
    v = torch.zeros_like(k)
    pool = pa.KVPool(k, v, scale, scale)
    xd = x.to(cuda_device)
    pa.write_kv(pool, xd, xd, torch.arange(T, dtype=torch.int64, device=cuda_device))
    assert pa.get_error() == pa.PA_OK
    got = k.cpu().numpy().reshape(-1)
    want = O.fp8_store_array(patterns, scale)
    np.testing.assert_array_equal(got, want)
    np.testing.assert_array_equal(v.cpu().numpy().reshape(-1), want)


def test_write_kv_skips_padding_and_flags_out_of_range(cuda_device):
    w = workloads.build([20, 5], [4, 5], Hq=2, Hkv=2, D=64, B=16, seed=3, device=cuda_device,
                        pool_blocks=4)
    pool = new_gpu_pool(w, cuda_device)
    before = pool_bits(pool)
    slots = w.slot_mapping.clone()
    slots[1] = -1                               # padding token: skipped
    slots[2] = w.num_blocks * w.B + 3            # outside the pool: skipped + flagged
    pa.write_kv(pool, w.new_k, w.new_v, slots)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert pa.get_error() == pa.PA_OK  # the error word was cleared
    ref = O.Pool(before[0].copy(), before[1].copy(), w.B, O.BF16)
    keep = np.ones(w.T, bool)
    keep[[1, 2]] = False
    O.write_kv(ref, bits(w.new_k)[keep], bits(w.new_v)[keep], slots.cpu().numpy()[keep])
    gk, gv = pool_bits(pool)
    np.testing.assert_array_equal(gk, ref.k)
    np.testing.assert_array_equal(gv, ref.v)


def _rand_diffs(rng, mr, mb, W, overlap=True):
    rows, starts, offs, vals = [], [], [0], []
    for _ in range(W):
        r = int(rng.integers(0, mr if overlap else mr))
        s = int(rng.integers(0, mb))
        n = int(rng.integers(0, mb - s + 1))
        rows.append(r)
        starts.append(s)
        vals.extend(int(x) for x in rng.integers(0, 1 << 20, size=n))
        offs.append(len(vals))
    return (np.array(rows, np.int32), np.array(starts, np.int32), np.array(offs, np.int32),
            np.array(vals, np.int32))


def _gpu_staged(dev, table, rows, starts, offs, vals, idx):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a, np.int32)).to(dev)
    tab = t(table)
    R, mb = len(idx), table.shape[1]
    gathered = torch.full((R, mb), -9, dtype=torch.int32, device=dev)
    pa.apply_staged_writes(tab, t(rows), t(starts), t(offs), t(vals if len(vals) else [0]),
                           t(idx), gathered)
    return tab.cpu().numpy(), gathered.cpu().numpy()


@pytest.mark.parametrize("trial", range(6))
def test_staged_writes_random_overlapping_diffs(cuda_device, trial):
    rng = np.random.default_rng(100 + trial)
    mr, mb = [(7, 5), (1024, 128), (64, 632), (3, 1), (1024, 512), (40, 40)][trial]
    W = int(rng.integers(0, 300))
    table = rng.integers(-1, 1 << 20, size=(mr, mb)).astype(np.int32)
    rows, starts, offs, vals = _rand_diffs(rng, mr, mb, W)
    idx = rng.integers(0, mr, size=int(rng.integers(0, 300))).astype(np.int32)
    g_tab, g_gat = _gpu_staged(cuda_device, table, rows, starts, offs, vals, idx)
    o_tab = table.copy()
    o_gat = O.apply_staged_writes(o_tab, rows, starts, offs, vals, idx)
    assert pa.get_error() == pa.PA_OK
    np.testing.assert_array_equal(g_tab, o_tab)
    np.testing.assert_array_equal(g_gat, o_gat)


def test_staged_writes_many_diffs_on_one_row(cuda_device):
    """More diffs on one row than the gather keeps in shared memory."""
    rng = np.random.default_rng(5)
    mr, mb = 4, 64
    table = np.zeros((mr, mb), np.int32)
    W = 1500
    rows = np.full(W, 2, np.int32)
    starts = rng.integers(0, mb, size=W).astype(np.int32)
    lens = np.minimum(rng.integers(0, 4, size=W), mb - starts)
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    vals = rng.integers(0, 1 << 20, size=int(offs[-1])).astype(np.int32)
    idx = np.array([2, 0, 2], np.int32)
    g_tab, g_gat = _gpu_staged(cuda_device, table, rows, starts, offs, vals, idx)
    o_tab = table.copy()
    o_gat = O.apply_staged_writes(o_tab, rows, starts, offs, vals, idx)
    np.testing.assert_array_equal(g_tab, o_tab)
    np.testing.assert_array_equal(g_gat, o_gat)


def test_staged_writes_admission_burst(cuda_device):
    """An admission burst: 1,024 new rows written whole in one call (1,024
    diffs of up to 512 values), then 1,024 shorter diffs that overwrite parts
    of random rows; table and gathered rows bit-exact against the oracle."""
    rng = np.random.default_rng(6)
    mr, mb = 1024, 512
    table = rng.integers(-1, 1 << 20, size=(mr, mb)).astype(np.int32)
    rows = list(range(mr))
    starts = [0] * mr
    lens = list(rng.integers(1, mb + 1, size=mr))
    for _ in range(1024):
        r, s = int(rng.integers(0, mr)), int(rng.integers(0, mb))
        rows.append(r)
        starts.append(s)
        lens.append(int(rng.integers(0, min(64, mb - s) + 1)))
    offs = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    vals = rng.integers(0, 1 << 20, size=int(offs[-1])).astype(np.int32)
    rows, starts = np.array(rows, np.int32), np.array(starts, np.int32)
    idx = rng.permutation(mr).astype(np.int32)
    g_tab, g_gat = _gpu_staged(cuda_device, table, rows, starts, offs, vals, idx)
    assert pa.get_error() == pa.PA_OK
    o_tab = table.copy()
    o_gat = O.apply_staged_writes(o_tab, rows, starts, offs, vals, idx)
    np.testing.assert_array_equal(g_tab, o_tab)
    np.testing.assert_array_equal(g_gat, o_gat)


def test_staged_writes_out_of_range_are_skipped_and_flagged(cuda_device):
    table = np.arange(12, dtype=np.int32).reshape(3, 4)
    rows = np.array([1, 5, 0], np.int32)       # row 5 is outside the table
    starts = np.array([0, 0, 3], np.int32)
    offs = np.array([0, 2, 3, 5], np.int32)    # the last diff runs past column 3
    vals = np.array([40, 41, 42, 43, 44], np.int32)
    idx = np.array([1, 7, 0], np.int32)        # slot 7 is outside the table
    g_tab, g_gat = _gpu_staged(cuda_device, table, rows, starts, offs, vals, idx)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    want = table.copy()
    want[1, :2] = [40, 41]
    np.testing.assert_array_equal(g_tab, want)
    np.testing.assert_array_equal(g_gat[0], want[1])
    np.testing.assert_array_equal(g_gat[1], [-9] * 4)  # untouched
    np.testing.assert_array_equal(g_gat[2], want[0])


@pytest.mark.parametrize("cfg", [2, 3, 5])
def test_staged_writes_rebuild_workload_tables(cuda_device, cfg):
    w = workloads.make(cfg, device=cuda_device, num_requests=8)
    g_tab, g_gat = _gpu_staged(cuda_device, w.table_before, w.diff_rows, w.diff_starts,
                               w.diff_val_offsets, w.diff_vals, w.idx_mapping)
    o_tab = w.table_before.copy()
    o_gat = O.apply_staged_writes(o_tab, w.diff_rows, w.diff_starts, w.diff_val_offsets,
                                  w.diff_vals, w.idx_mapping)
    np.testing.assert_array_equal(g_tab, o_tab)
    np.testing.assert_array_equal(g_gat, o_gat)
    np.testing.assert_array_equal(g_gat, w.tables)


def test_staged_writes_empty_cases(cuda_device):
    table = np.arange(6, dtype=np.int32).reshape(2, 3)
    g_tab, g_gat = _gpu_staged(cuda_device, table, np.zeros(0), np.zeros(0), [0], [], [1, 0])
    np.testing.assert_array_equal(g_tab, table)
    np.testing.assert_array_equal(g_gat, table[[1, 0]])
    g_tab, g_gat = _gpu_staged(cuda_device, table, [0], [1], [0, 2], [9, 8], [])
    np.testing.assert_array_equal(g_tab[0], [0, 9, 8])


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_copy_blocks_bit_exact(cuda_device, dtype):
    w = workloads.build([64, 40, 17], [1, 1, 1], Hq=8, Hkv=4, D=128, B=32, kv_dtype=dtype,
                        seed=8, device=cuda_device, pool_blocks=12)
    pool = gpu_cache(w, cuda_device)
    ref = oracle_pool(w, include_new=False)
    src = np.array([int(w.tables[0, 0]), int(w.tables[1, 1]), 99], np.int32)
    used = set(w.tables[w.tables >= 0].tolist())
    free = [b for b in range(w.num_blocks) if b not in used]
    dst = np.array([free[0], free[1], free[2]], np.int32)
    pa.copy_blocks(pool, torch.from_numpy(src).to(cuda_device),
                   torch.from_numpy(dst).to(cuda_device))
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS  # the pair (99, .) is skipped
    O.copy_blocks(ref, src[:2], dst[:2])
    gk, gv = pool_bits(pool)
    np.testing.assert_array_equal(gk, ref.k)
    np.testing.assert_array_equal(gv, ref.v)


def test_gather_rows_bit_exact_and_flags_bad_rows(cuda_device):
    """pa_gather_rows: dst[i] = src[rows[i]] bit for bit (repeated and
    unordered rows), against a numpy gather of the same bytes; a row index
    outside src sets PA_ERR_DEVICE_BOUNDS and leaves that dst row as it was."""
    g = torch.Generator().manual_seed(31)
    src = torch.randn((300, 32, 128), generator=g).bfloat16()
    rows = torch.tensor([5, 299, 0, 5, 17, 123, 298, 1], dtype=torch.int32)
    dst = torch.full((8, 32, 128), 7.0, dtype=torch.bfloat16, device=cuda_device)
    pa.gather_rows(src.to(cuda_device), rows.to(cuda_device), dst)
    assert pa.get_error() == pa.PA_OK
    want = src.view(torch.int16).numpy()[rows.numpy()]
    np.testing.assert_array_equal(dst.cpu().view(torch.int16).numpy(), want)
    bad = torch.tensor([2, 300, -1, 4], dtype=torch.int32, device=cuda_device)
    dst2 = torch.full((4, 32, 128), 7.0, dtype=torch.bfloat16, device=cuda_device)
    pa.gather_rows(src.to(cuda_device), bad, dst2)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    got = dst2.cpu().view(torch.int16).numpy()
    np.testing.assert_array_equal(got[0], src.view(torch.int16).numpy()[2])
    np.testing.assert_array_equal(got[3], src.view(torch.int16).numpy()[4])
    assert (dst2[1:3].float() == 7.0).all()
