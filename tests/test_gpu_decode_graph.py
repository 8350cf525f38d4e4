"""Multi-step decode replayed from a CUDA graph (pa_decode_graph_*): every step
against the fp64 oracle, bit-identical to the same eager calls, launch
accounting, and a sequence bound that the steps outgrow."""
import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from paged_kv_cache_143_gb300 import pa
from tests.gpu_helpers import DeviceStep, assert_attention_close
from tests.helpers import bits, oracle_pool

pytestmark = pytest.mark.gpu


def _setup(dev, ctx, N, Hq=8, Hkv=2, D=128, B=16, kv="bf16", seed=0, max_splits=16):
    """Requests with `ctx` cached tokens and N decode steps ahead: the pool
    holds the context, the persistent table already holds the blocks of the
    N new tokens, and the step inputs are split per step."""
    R = len(ctx)
    w = workloads.build([c + N for c in ctx], [N] * R, Hq, Hkv, D, B, kv_dtype=kv, seed=seed,
                        device=dev)
    step = DeviceStep(w, dev, max_splits=max_splits)
    pa.apply_staged_writes(step.table, step.rows, step.starts, step.offs, step.vals, step.idx,
                           step.gathered)
    nc = torch.zeros(w.max_reqs, dtype=torch.int32, device=dev)
    nc[step.idx.long()] = torch.tensor(ctx, dtype=torch.int32, device=dev)
    # token s of request r is row r * N + s of the workload's step tensors
    per_step = lambda t: t.view(R, N, *t.shape[1:]).transpose(0, 1).contiguous()
    return w, step, nc, per_step(w.q.to(dev)), per_step(w.new_k.to(dev)), per_step(w.new_v.to(dev))


def _oracle_steps(w, ctx, N):
    """Step s of request r: its token s against keys [0, ctx_r + s + 1) of the
    final pool (every step's K/V written)."""
    pool = oracle_pool(w)
    R = len(ctx)
    qb = bits(w.q).reshape(R, N, w.Hq, w.D)
    qsl = np.arange(R + 1, dtype=np.int32)
    outs = []
    for s in range(N):
        seq = np.array([c + s + 1 for c in ctx], np.int32)
        outs.append(O.paged_attention(np.ascontiguousarray(qb[:, s]), qsl, seq, w.tables, pool,
                                      w.scale, 1))
    return outs


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_graph_steps_match_oracle_and_eager(cuda_device, kv):
    ctx, N = [17, 300, 1025, 64, 2000, 5], 6
    R = len(ctx)
    w, step, nc, q, k, v = _setup(cuda_device, ctx, N, kv=kv, seed=3)
    bound = [c + N for c in ctx]
    out = torch.empty_like(q)
    g = pa.DecodeGraph(step.pool, w.scale, nc, step.table, step.idx, step.gathered, bound, q, k,
                       v, out, workspace=step.ws)
    before = pa.kernel_launches()
    g.launch()
    launched = pa.kernel_launches() - before  # pa_get_error launches a kernel of its own
    assert pa.get_error() == pa.PA_OK
    assert launched == g.kernels >= 3 * N
    assert nc[step.idx.long()].cpu().tolist() == bound
    ref = _oracle_steps(w, ctx, N)
    for s in range(N):
        assert_attention_close(out[s], ref[s], what=f"graph step {s}")

    # the same calls made eagerly (same plan bound) give identical bits
    w2, step2, nc2, q2, k2, v2 = _setup(cuda_device, ctx, N, kv=kv, seed=3)
    out2 = torch.empty_like(q2)
    qsl = torch.empty(R + 1, dtype=torch.int32, device=cuda_device)
    seq = torch.empty(R, dtype=torch.int32, device=cuda_device)
    pos = torch.empty(R, dtype=torch.int32, device=cuda_device)
    slots = torch.empty(R, dtype=torch.int64, device=cuda_device)
    for s in range(N):
        pa.lib().pa_prepare_inputs(
            nc2.data_ptr(), nc2.numel(), step2.table.data_ptr(), step2.table.shape[1], w2.B,
            w2.num_blocks, step2.idx.data_ptr(), None, R, R, qsl.data_ptr(), seq.data_ptr(),
            pos.data_ptr(), slots.data_ptr(), torch.cuda.current_stream().cuda_stream)
        pa.write_kv(step2.pool, k2[s], v2[s], slots)
        pa.forward(q2[s], out2[s], qsl, seq, np.arange(R + 1), bound, step2.gathered, step2.pool,
                   w2.scale, 1, workspace=step2.ws)
    assert pa.get_error() == pa.PA_OK
    assert torch.equal(out.view(torch.int16), out2.view(torch.int16))
    g.close()


def test_graph_replays_further_steps(cuda_device):
    """A second launch continues from the advanced slot state: it reproduces
    steps N..2N-1 of an eager run (K/V of the second launch are the same
    per-step buffers, so the oracle is the eager sequence)."""
    ctx, N = [40, 700, 129], 4
    w, step, nc, q, k, v = _setup(cuda_device, ctx, 2 * N, seed=5)
    q1, k1, v1 = q[:N].contiguous(), k[:N].contiguous(), v[:N].contiguous()
    bound = [c + 2 * N for c in ctx]
    out = torch.empty_like(q1)
    g = pa.DecodeGraph(step.pool, w.scale, nc, step.table, step.idx, step.gathered, bound, q1,
                       k1, v1, out, workspace=step.ws)
    g.launch()
    first = out.clone()
    q1.copy_(q[N:])
    k1.copy_(k[N:])
    v1.copy_(v[N:])
    g.launch()
    assert pa.get_error() == pa.PA_OK
    ref = _oracle_steps(w, ctx, 2 * N)
    for s in range(N):
        assert_attention_close(first[s], ref[s], what=f"launch 1 step {s}")
        assert_attention_close(out[s], ref[N + s], what=f"launch 2 step {s}")
    g.close()


@pytest.mark.parametrize("Hq,max_splits", [(8, 8), (2, 8), (8, 0)])
def test_graph_sequences_past_the_bound_are_flagged_or_exact(cuda_device, Hq, max_splits):
    """A bound far below the real lengths: the plan made from it either
    still covers the real lengths (the persistent GQA decode cuts the
    device-side lengths into its CTA ranges at every launch), and the outputs
    match the oracle, or the kernels refuse them with PA_ERR_DEVICE_BOUNDS;
    never a read out of range. The grid decode (g = 1, or no workspace)
    plans one split per request from the bound and must refuse."""
    ctx, N = [3000, 20], 2
    w, step, nc, q, k, v = _setup(cuda_device, ctx, N, seed=9, Hq=Hq, max_splits=max_splits)
    out = torch.zeros_like(q)
    g = pa.DecodeGraph(step.pool, w.scale, nc, step.table, step.idx, step.gathered, [2, 2], q, k,
                       v, out, workspace=step.ws)
    g.launch()
    st = pa.get_error()
    g.close()
    if Hq // 2 == 1 or max_splits == 0:  # g = 1 or no workspace: the grid decode
        assert st == pa.PA_ERR_DEVICE_BOUNDS
    else:
        assert st in (pa.PA_OK, pa.PA_ERR_DEVICE_BOUNDS)
    if st == pa.PA_OK:
        ref = _oracle_steps(w, ctx, N)
        for s in range(N):
            assert_attention_close(out[s], ref[s], what=f"step {s} past the bound")
    assert pa.get_error() == pa.PA_OK
