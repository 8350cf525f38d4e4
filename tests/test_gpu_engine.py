"""The multi-step serving loop (native scheduler + device calls) against an
oracle replay of the same steps: device tables, slot mappings and the pool
bit-exact, every step's attention within the bounds."""
import numpy as np
import pytest
import torch

from oracle import oracle as O
from paged_kv_cache_143_gb300 import pa
from paged_kv_cache_143_gb300.engine import Engine
from tests.gpu_helpers import assert_attention_close
from tests.helpers import bits

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_engine_steps_match_oracle_replay(cuda_device, kv):
    Hq, Hkv, D, B, NB = 8, 2, 128, 16, 192
    max_reqs, max_blocks, max_tokens = 16, 40, 320
    rng = np.random.default_rng(11)
    gen = torch.Generator(device=cuda_device)
    gen.manual_seed(11)
    if kv == "bf16":
        nan, dt, tdt, scales = 0x7FC0, np.uint16, torch.int16, (1.0, 1.0)
    else:
        nan, dt, tdt, scales = 0x7F, np.uint8, torch.uint8, (0.01, 0.0125)
    k_pool = torch.full((NB, Hkv, B, D), nan, dtype=tdt, device=cuda_device)
    v_pool = torch.full((NB, Hkv, B, D), nan, dtype=tdt, device=cuda_device)
    if kv == "bf16":
        k_pool, v_pool = k_pool.view(torch.bfloat16), v_pool.view(torch.bfloat16)
    pool = pa.KVPool(k_pool, v_pool, *scales)
    opool = O.Pool(np.full((NB, Hkv, B, D), nan, dt), np.full((NB, Hkv, B, D), nan, dt), B,
                   O.BF16 if kv == "bf16" else O.FP8_E4M3, *scales)
    sched = pa.Scheduler(NB, B, max_reqs, max_blocks, token_budget=256, chunk_cap=96,
                         prefix_caching=True)
    eng = Engine(sched, pool, Hq, max_reqs, max_blocks, max_tokens, scale=D ** -0.5)
    common = rng.integers(0, 1000, size=3 * B + 5).tolist()
    rid = 0
    forked = set()
    for step in range(40):
        if step < 12 and rng.random() < 0.6:
            p = (common if rng.random() < 0.5 else []) + rng.integers(
                0, 1000, size=int(rng.integers(1, 150))).tolist()
            sched.add_request(rid, p, int(rng.integers(2, 25)))
            rid += 1
        q = torch.randn((max_tokens, Hq, D), generator=gen, device=cuda_device).bfloat16()
        k = torch.randn((max_tokens, Hkv, D), generator=gen, device=cuda_device).bfloat16()
        v = torch.randn((max_tokens, Hkv, D), generator=gen, device=cuda_device).bfloat16()
        out = torch.empty_like(q)
        b = eng.step(q, k, v, out)
        eng.sync()
        assert pa.get_error() == pa.PA_OK
        R, T = b.num_reqs, b.num_tokens
        if R == 0:
            sched.commit([])
            continue
        # device inputs equal the host's view of the step
        assert eng.slots[:T].cpu().numpy().tolist() == b.slot_mapping.tolist()
        assert eng.qsl[:R + 1].cpu().numpy().tolist() == b.query_start_loc.tolist()
        assert eng.seq[:R].cpu().numpy().tolist() == b.seq_lens.tolist()
        tables = np.full((R, max_blocks), -1, np.int32)
        for i, r in enumerate(b.req_ids):
            t = sched.table(int(r))
            tables[i, :len(t)] = t
            assert eng.gathered[i, :len(t)].cpu().numpy().tolist() == t
        # oracle replay: copy-on-write, KV write, attention
        O.copy_blocks(opool, b.copy_src, b.copy_dst)
        O.write_kv(opool, bits(k[:T]), bits(v[:T]), b.slot_mapping)
        ref = O.paged_attention(bits(q[:T]), b.query_start_loc, b.seq_lens, tables, opool,
                                D ** -0.5, 1)
        assert_attention_close(out[:T], ref, what=f"engine step {step} ({kv})")
        # the last-token rows that were read back
        last = b.query_start_loc[1:] - 1
        assert torch.equal(eng.last_out.view(torch.int16), out[last].cpu().view(torch.int16))
        sampled = rng.integers(0, 1000, size=R).tolist()
        sched.commit(sampled)
        # forks of running requests (copy-on-write on their next writes)
        if step in (10, 18):
            for r in b.req_ids[b.num_decode:][:1].tolist() + b.req_ids[:1].tolist():
                if int(r) not in forked and sched.stats()["running"] < max_reqs:
                    try:
                        sched.fork(int(r), 1000 + rid, 6)
                        forked.add(int(r))
                        rid += 1
                    except pa.PaError:
                        pass
    # the pools agree bit for bit
    assert np.array_equal(bits(k_pool), opool.k) and np.array_equal(bits(v_pool), opool.v)
    st = sched.stats()
    assert st["steps"] == 40 and st["prefix_hit_tokens"] > 0
