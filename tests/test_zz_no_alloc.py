"""pa_forward_noalloc: the attention entry point for callers that cannot
allocate device memory (a plugin whose host runtime owns all device memory,
or a serving loop that forbids cudaMalloc after start-up). Its split-KV scratch
is the library's own fixed device array instead of a caller workspace.

This file is collected last on purpose: the call shares one library-wide
array, and the test must pass both alone in a fresh process and after every
other test has run."""
import numpy as np
import pytest
import torch

import workloads
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import MAX_ABS, MEAN_ABS, DeviceStep

pytestmark = pytest.mark.gpu


def _close(a, b):
    err = (a.float() - b.float()).abs().double()
    return float(err.max()), float(err.mean())


def test_noalloc_forward_matches_workspace_forward_twice(cuda_device):
    # long decodes so that the planner splits the keys and uses the scratch
    w = workloads.build([8000, 5000, 3000, 7777, 129], [1] * 5, Hq=16, Hkv=4, D=128, B=16,
                        seed=77, device=cuda_device)
    step = DeviceStep(w, cuda_device, max_splits=32)
    ref = step.run().clone()
    assert pa.get_error() == pa.PA_OK
    need = pa.forward_workspace_size(w.R, w.Hq, w.D, 32)
    assert 0 < need <= pa.NOALLOC_SCRATCH_BYTES
    for _ in range(2):  # two calls in a row share (and reuse) the array
        out = torch.full_like(ref, float("nan"))
        pa.forward_noalloc(step.q, out, step.qsl, step.seq, w.qsl, w.seq_lens, step.gathered,
                           step.pool, w.scale, w.causal, max_splits=32)
        assert pa.get_error() == pa.PA_OK
        mx, mean = _close(out, ref)
        assert mx <= MAX_ABS and mean <= MEAN_ABS, (mx, mean)


def test_noalloc_rejects_scratch_beyond_its_maximum(cuda_device):
    w = workloads.build([100, 40], [1, 1], Hq=8, Hkv=8, D=128, B=16, seed=3, device=cuda_device)
    step = DeviceStep(w, cuda_device, max_splits=0)
    # the scratch grows by one split row per split: one more split than the
    # array holds rows for is always beyond it
    row = pa.forward_workspace_size(w.R, w.Hq, w.D, 2) - pa.forward_workspace_size(w.R, w.Hq, w.D, 1)
    too_many = pa.NOALLOC_SCRATCH_BYTES // row + 1
    with pytest.raises(pa.PaError) as e:
        pa.forward_noalloc(step.q, step.out, step.qsl, step.seq, w.qsl, w.seq_lens,
                           step.table[:w.R], step.pool, w.scale, 1, max_splits=int(too_many))
    assert e.value.status == pa.PA_ERR_UNSUPPORTED
