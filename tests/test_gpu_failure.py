"""Failure detection on the GPU without faulting it: device range errors and
bounded waits are reported through the error word and leave the context
usable (the next call still computes correct results)."""
import time

import numpy as np
import pytest
import torch

import workloads
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import DeviceStep, assert_attention_close, oracle_step

pytestmark = pytest.mark.gpu


def test_bounded_wait_reports_timeout_and_context_survives(cuda_device):
    assert pa.get_error() == pa.PA_OK
    t0 = time.time()
    pa.selftest_wait_timeout()
    assert pa.get_error() == pa.PA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    assert pa.get_error() == pa.PA_OK  # cleared
    # the context is intact: a normal step still matches the oracle
    w = workloads.build([70, 300], [1, 40], Hq=8, Hkv=2, D=128, B=16, seed=1,
                        device=cuda_device)
    step = DeviceStep(w, cuda_device)
    out = step.run()
    assert pa.get_error() == pa.PA_OK
    ref, *_ = oracle_step(w)
    assert_attention_close(out, ref)


def test_prefill_flags_bad_block_ids_without_faulting(cuda_device):
    w = workloads.build([300], [100], Hq=8, Hkv=2, D=128, B=16, seed=2, device=cuda_device)
    step = DeviceStep(w, cuda_device)
    step.run()
    assert pa.get_error() == pa.PA_OK
    bad = step.gathered.clone()
    bad[0, 3] = -5
    pa.forward(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens, bad, step.pool,
               w.scale, w.causal)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    step.run()
    assert pa.get_error() == pa.PA_OK


def test_device_seq_lens_disagreeing_with_host_mirror_are_flagged(cuda_device):
    """The planner sizes grids from the host mirrors; a device seq_len that
    needs more splits than were planned is refused on the device."""
    w = workloads.build([4000, 100], [1, 1], Hq=4, Hkv=4, D=128, B=16, seed=3,
                        device=cuda_device)
    step = DeviceStep(w, cuda_device, max_splits=16)
    step.run()
    assert pa.get_error() == pa.PA_OK
    host_seq = np.array([100, 100], np.int32)  # the host claims short contexts
    pa.forward(step.q, step.out, step.qsl, step.seq, w.qsl, host_seq, step.gathered,
               step.pool, w.scale, w.causal, workspace=step.ws)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS


def _sentinel_out(q, T, extra=8):
    """An output buffer of T + extra rows filled with a sentinel bit pattern;
    the library is given its first T rows."""
    big = torch.empty((T + extra,) + tuple(q.shape[1:]), dtype=torch.bfloat16, device=q.device)
    big.view(torch.int16).fill_(0x1234)
    return big, big[:T]


def test_device_qsl_past_the_batch_is_flagged_and_never_written(cuda_device):
    """A device query_start_loc that disagrees with its host mirror and points
    past the T rows of q / out: the decode, merge and prefill kernels raise
    PA_ERR_DEVICE_BOUNDS and write nothing beyond row T."""
    # decodes: request 1 claims token row T + 2 (one token there)
    w = workloads.build([300, 500, 40], [1, 1, 1], Hq=8, Hkv=2, D=128, B=16, seed=4,
                        device=cuda_device)
    step = DeviceStep(w, cuda_device, max_splits=8)
    step.run()
    assert pa.get_error() == pa.PA_OK
    big, out = _sentinel_out(step.q, w.T)
    bad = torch.tensor([0, w.T + 2, w.T + 3, w.T], dtype=torch.int32, device=cuda_device)
    pa.forward(step.q, out, bad, step.seq, w.qsl, w.seq_lens, step.gathered, step.pool,
               w.scale, w.causal, workspace=step.ws)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert (big[w.T:].view(torch.int16) == 0x1234).all()

    # prefill chunks: the last chunk's end moved past T, and the first chunk
    # made longer than the query tiles the grid was planned for
    w = workloads.build([300, 200], [100, 50], Hq=8, Hkv=2, D=128, B=16, seed=5,
                        device=cuda_device)
    step = DeviceStep(w, cuda_device)
    step.run()
    assert pa.get_error() == pa.PA_OK
    big, out = _sentinel_out(step.q, w.T)
    for qsl in ([0, 100, w.T + 6], [0, 140, w.T]):
        bad = torch.tensor(qsl, dtype=torch.int32, device=cuda_device)
        pa.forward(step.q, out, bad, step.seq, w.qsl, w.seq_lens, step.gathered, step.pool,
                   w.scale, w.causal, workspace=step.ws)
        assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS, qsl
        assert (big[w.T:].view(torch.int16) == 0x1234).all(), qsl
    # the context is intact
    step.run()
    assert pa.get_error() == pa.PA_OK


def test_error_raised_on_another_stream_is_never_lost(cuda_device):
    """pa_get_error reads and clears the error word in one atomic exchange:
    while a kernel on a second stream is about to raise a bit, repeated reads
    on the first stream see that bit exactly once, never clearing it unseen."""
    assert pa.get_error() == pa.PA_OK
    s2 = torch.cuda.Stream()
    pa.selftest_wait_timeout(stream=s2)  # raises PA_ERR_TIMEOUT after about 2 s
    seen = []
    t0 = time.time()
    while not s2.query() and time.time() - t0 < 30:
        seen.append(pa.get_error())
    s2.synchronize()
    seen.append(pa.get_error())
    assert seen.count(pa.PA_ERR_TIMEOUT) == 1, sorted(set(seen))
    assert all(x in (pa.PA_OK, pa.PA_ERR_TIMEOUT) for x in seen)
    assert pa.get_error() == pa.PA_OK


def test_shared_prefix_device_mirror_errors_are_flagged_and_never_written(cuda_device):
    """pa_forward_shared_prefix with device arrays that disagree with their
    host mirrors: a group member whose device query_start_loc points past
    the T rows, and a member whose device seq_len no longer reaches past the
    shared prefix, raise PA_ERR_DEVICE_BOUNDS; nothing is written beyond row
    T, and the next call is clean."""
    from tests.gpu_helpers import group_arrays
    w = workloads.build([64 + 5, 64 + 30, 64 + 1, 64 + 200, 90], [1] * 5, Hq=8, Hkv=2, D=128,
                        B=16, seed=8, device=cuda_device, groups=[([0, 1, 2, 3], 64)])
    step = DeviceStep(w, cuda_device, max_splits=8)
    step.run(cascade=True)
    assert pa.get_error() == pa.PA_OK
    first, size, prefix_blocks = group_arrays(w)
    big, out = _sentinel_out(step.q, w.T)

    def call(qsl, seq):
        pa.forward_shared_prefix(step.q, out, qsl, seq, w.qsl, w.seq_lens, step.gathered,
                                 step.pool, w.scale, first, size, prefix_blocks,
                                 causal=w.causal, workspace=step.ws)

    bad_qsl = torch.tensor([0, 1, 2, w.T + 2, w.T + 3, w.T], dtype=torch.int32,
                           device=cuda_device)
    call(bad_qsl, step.seq)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert (big[w.T:].view(torch.int16) == 0x1234).all()
    short = step.seq.clone()
    short[1] = 64  # member 1: no key after the 64-token prefix
    call(step.qsl, short)
    assert pa.get_error() == pa.PA_ERR_DEVICE_BOUNDS
    assert (big[w.T:].view(torch.int16) == 0x1234).all()
    step.run(cascade=True)
    assert pa.get_error() == pa.PA_OK
