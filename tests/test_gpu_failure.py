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
