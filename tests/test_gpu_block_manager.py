"""The native block manager driving the device hot path (parallel sampling, beam search).

One prompt, forked into four samples or four beams; every decode step the manager
hands out slots and copy-on-write pairs, the GPU runs copy_blocks -> reshape_and_cache
-> paged decode, the oracle runs the same operations on host pools, and the outputs
(within tolerance) and the pools (byte for byte) must agree. Beams are re-forked from
chosen parents and the old ones freed after every step.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import binding, inputs
from paged_kv_cache_87_gb300.session import host_tensor, poisoned_cache, to_numpy_storage
from tests.helpers import TOL

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("dt,kv", [("bf16", "bf16"), ("bf16", "e4m3"), ("f32", "f32")])
def test_parallel_sampling_steps(dt, kv):
    rng = np.random.default_rng(31)
    B, NB, Hq, Hkv, d = 16, 96, 8, 2, 128
    kv_scale = 2.0 ** -5 if kv == "e4m3" else 1.0
    scale = 1 / math.sqrt(d)
    m = binding.BlockManager(NB, B, free_order=rng.permutation(NB))
    common = dict(num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=NB)
    hk, hv = inputs.poison_array((NB, Hkv, B, d), kv), inputs.poison_array((NB, Hkv, B, d), kv)
    dk, dv = poisoned_cache((NB, Hkv, B, d), kv, "cuda"), poisoned_cache((NB, Hkv, B, d), kv,
                                                                           "cuda")

    def write(slots, n):
        key = inputs.draw_normal(rng, (n, Hkv, d), dt)
        val = inputs.draw_normal(rng, (n, Hkv, d), dt)
        oracle.reshape_and_cache(key, val, hk, hv, slots, src_dtype=dt, kv_dtype=kv,
                                 kv_scale=kv_scale, **common)
        binding.pkv_reshape_and_cache(host_tensor(key, dt).cuda(), host_tensor(val, dt).cuda(),
                                      dk, dv, torch.from_numpy(slots).cuda(), kv_scale=kv_scale)

    prompt = 40
    m.add_sequence(0, prompt)
    table, _ = m.sequence(0)
    write(np.array([table[t // B] * B + t % B for t in range(prompt)], np.int64), prompt)
    for c in (1, 2, 3):
        m.fork(0, c)
    seqs = [0, 1, 2, 3]
    max_blocks = 12
    ws = None
    for step in range(30):
        slots, pairs, tables, ctx = m.prepare_step(seqs, max_blocks)
        if len(pairs):
            oracle.copy_blocks(hk, hv, pairs, kv_dtype=kv, **common)
            binding.pkv_copy_blocks(dk, dv, pairs)
        write(slots, len(seqs))
        q = inputs.draw_normal(rng, (len(seqs), Hq, d), dt)
        ref = oracle.paged_decode_attention(q, hk, hv, tables, ctx, num_q_heads=Hq,
                                            num_kv_heads=Hkv, head_dim=d, block_size=B,
                                            num_blocks=NB, scale=scale, q_dtype=dt,
                                            kv_dtype=kv, kv_scale=kv_scale)
        out = binding.pkv_paged_decode_attention(
            host_tensor(q, dt).cuda(), dk, dv, torch.from_numpy(tables).cuda(),
            torch.from_numpy(ctx).cuda(), int(ctx.max()), scale, kv_scale=kv_scale,
            workspace=ws)
        err = np.abs(out.double().cpu().numpy() - ref).max()
        assert err <= TOL[kv if kv == "e4m3" else dt], (step, err)
    assert binding.pkv_get_device_status() == 0
    assert to_numpy_storage(dk, kv).view(np.uint8).tobytes() == hk.view(np.uint8).tobytes()
    assert to_numpy_storage(dv, kv).view(np.uint8).tobytes() == hv.view(np.uint8).tobytes()
    # 40 + 30 tokens each: every sample got its own copy of the shared partial block
    for s in seqs:
        assert m.sequence(s)[1] == prompt + 30
    assert m.refcount(m.sequence(0)[0][0]) == 4 and m.refcount(m.sequence(0)[0][1]) == 4


@pytest.mark.parametrize("dt,kv", [("bf16", "bf16"), ("f16", "e4m3")])
def test_beam_search_steps(dt, kv):
    """Beam search ("...Mathematical Foundations" §5 Beam Search) through the engine:
    each step the live beams append a token (copy_blocks for the shared blocks they
    write, reshape_and_cache, paged decode), then K survivors are forked from parents
    drawn from the live beams and the old beams are freed. The outputs follow the oracle
    on host pools, and the pools agree byte for byte."""
    rng = np.random.default_rng(41)
    B, NB, Hq, Hkv, d, K = 8, 160, 8, 2, 128, 4
    kv_scale = 2.0 ** -5 if kv == "e4m3" else 1.0
    scale = 1 / math.sqrt(d)
    m = binding.BlockManager(NB, B, free_order=rng.permutation(NB))
    common = dict(num_kv_heads=Hkv, head_dim=d, block_size=B, num_blocks=NB)
    hk, hv = inputs.poison_array((NB, Hkv, B, d), kv), inputs.poison_array((NB, Hkv, B, d), kv)
    dk, dv = poisoned_cache((NB, Hkv, B, d), kv, "cuda"), poisoned_cache((NB, Hkv, B, d), kv,
                                                                           "cuda")

    def write(slots, n):
        key = inputs.draw_normal(rng, (n, Hkv, d), dt)
        val = inputs.draw_normal(rng, (n, Hkv, d), dt)
        oracle.reshape_and_cache(key, val, hk, hv, slots, src_dtype=dt, kv_dtype=kv,
                                 kv_scale=kv_scale, **common)
        binding.pkv_reshape_and_cache(host_tensor(key, dt).cuda(), host_tensor(val, dt).cuda(),
                                      dk, dv, torch.from_numpy(slots).cuda(), kv_scale=kv_scale)

    prompt = 21
    m.add_sequence(0, prompt)
    table, _ = m.sequence(0)
    write(np.array([table[t // B] * B + t % B for t in range(prompt)], np.int64), prompt)
    live = [0]
    for c in range(1, K):
        m.fork(0, c)
        live.append(c)
    next_id, copies, max_blocks = K, 0, 12
    for step in range(24):
        slots, pairs, tables, ctx = m.prepare_step(live, max_blocks)
        if len(pairs):
            copies += len(pairs)
            oracle.copy_blocks(hk, hv, pairs, kv_dtype=kv, **common)
            binding.pkv_copy_blocks(dk, dv, pairs)
        write(slots, len(live))
        q = inputs.draw_normal(rng, (len(live), Hq, d), dt)
        ref = oracle.paged_decode_attention(q, hk, hv, tables, ctx, num_q_heads=Hq,
                                            num_kv_heads=Hkv, head_dim=d, block_size=B,
                                            num_blocks=NB, scale=scale, q_dtype=dt,
                                            kv_dtype=kv, kv_scale=kv_scale)
        out = binding.pkv_paged_decode_attention(
            host_tensor(q, dt).cuda(), dk, dv, torch.from_numpy(tables).cuda(),
            torch.from_numpy(ctx).cuda(), int(ctx.max()), scale, kv_scale=kv_scale)
        err = np.abs(out.double().cpu().numpy() - ref).max()
        assert err <= TOL[kv if kv == "e4m3" else dt], (step, err)
        parents = rng.choice(live, size=K, replace=True)
        new = []
        for par in parents:
            m.fork(int(par), next_id)
            new.append(next_id)
            next_id += 1
        for s in live:
            m.free_sequence(s)
        live = new
    assert copies > 0
    assert binding.pkv_get_device_status() == 0
    assert to_numpy_storage(dk, kv).view(np.uint8).tobytes() == hk.view(np.uint8).tobytes()
    assert to_numpy_storage(dv, kv).view(np.uint8).tobytes() == hv.view(np.uint8).tobytes()
