"""GPU parity of paged decode attention against the fp64 oracle.

Small workloads are compared element by element; the five workloads at full
size are compared on sampled (sequence, head) outputs in the same launch
configuration the benchmark times.  Tolerances: max abs error 1e-4 (fp32),
5e-3 (fp16), 1.6e-2 (bf16), 1.6e-2 (FP8 KV against the oracle's decode of the
same bytes).
"""
import math
import zlib

import numpy as np
import pytest
import torch

from paged_kv_cache_87_gb300 import binding, inputs
from tests.helpers import (gpu_state, logical_kv_f64, oracle_caches, oracle_decode,
                           relabel_blocks, tolerance, to_f64)

pytestmark = pytest.mark.gpu


def _check(w, got, ref, sel=None):
    err = np.abs(got - ref)
    assert np.isfinite(got).all()
    assert err.max() <= tolerance(w), (err.max(), tolerance(w), np.unravel_index(err.argmax(),
                                                                                  err.shape))


def _full_parity(w):
    st = gpu_state(w)
    kc, vc = oracle_caches(w)
    ref = oracle_decode(w, kc, vc, nthreads=8)
    _check(w, st.out_f64(), ref)
    return st, ref


# ------------------------------------------------ the five workloads, small --

@pytest.mark.parametrize("cid,kw", [
    (0, {}),                                    # full size: 4 seqs, ctx {1,17,100,256}
    (1, dict(num_seqs=6)),                      # ctx U[512,2048]: multi-chunk merge
    (2, dict(num_seqs=24)),                     # lognormal lengths, GQA 4
    (3, dict(num_seqs=2, ctx_cap=6000)),        # GQA 8, B32, long-ish
    (4, dict(num_seqs=8, ctx_cap=1500)),        # FP8 + shared prefix + CoW step
])
def test_config_small_elementwise(cid, kw):
    _full_parity(inputs.make_config(cid, **kw))


# ---------------------------------------------- the workloads at full size --

def _sample_pairs(w, n, seed):
    rng = np.random.default_rng(seed)
    longest = int(np.argmax(w.context_lens))
    shortest = int(np.argmin(w.context_lens))
    seqs = np.concatenate([[longest, shortest], rng.integers(0, w.num_seqs, n - 2)])
    heads = rng.integers(0, w.num_q_heads, n)
    heads[:2] = [0, w.num_q_heads - 1]
    return np.stack([seqs, heads], 1).astype(np.int32)


@pytest.mark.parametrize("cid", [1, 2, 3, 4])
def test_config_full_size_sampled(cid):
    w = inputs.make_config(cid)
    st = gpu_state(w, steps=2)          # steps are idempotent; run the bench's step twice
    sel = _sample_pairs(w, 24, cid)
    kc, vc = oracle_caches(w)
    ref = oracle_decode(w, kc, vc, sel=sel, nthreads=8)
    out = st.out_f64()
    got = out[sel[:, 0], sel[:, 1]]
    _check(w, got, ref)
    # every output is finite; zero-context sequences are zero
    assert np.isfinite(out).all()


# --------------------------------------------------------------- sweeps ----

SWEEP = []
for d in (64, 128):
    for B in (8, 16, 32):
        for (Hq, Hkv) in ((4, 4), (4, 2), (6, 2), (8, 2), (10, 2), (16, 2)):
            SWEEP.append((d, B, Hq, Hkv))


# every (q type, KV type) pair the library accepts: K/V of the query's type, or e4m3
DTYPE_PAIRS = [("f32", "f32"), ("f32", "e4m3"), ("f16", "f16"), ("f16", "e4m3"),
               ("bf16", "bf16"), ("bf16", "e4m3")]


@pytest.mark.parametrize("d,B,Hq,Hkv", SWEEP)
@pytest.mark.parametrize("qdt,kvdt", DTYPE_PAIRS)
def test_sweep_shapes_and_types(d, B, Hq, Hkv, qdt, kvdt):
    """Every shipped decode variant (q type, KV type, head_dim, block size, and
    heads per kv head 1, 2, 3, 4, 5 and 8) against the oracle, elementwise."""
    rng = np.random.default_rng(zlib.crc32(repr((d, B, Hq, Hkv, qdt, kvdt)).encode()))
    ctx = np.array([1, B - 1, B, B + 1, 511, 512, 513, 1100, 0, 3000])
    w = inputs.make_independent("sweep", rng, ctx, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
                                block_size=B, q_dtype=qdt, kv_dtype=kvdt,
                                scale=1.0 / math.sqrt(d),
                                kv_scale=2.0 ** -5 if kvdt == "e4m3" else 1.0)
    st, _ = _full_parity(w)
    assert (st.out_f64()[8] == 0).all()          # context 0 -> zeros


# ------------------------------------------------------------ properties --

def _tiny(seed, ctx, **kw):
    rng = np.random.default_rng(seed)
    a = dict(num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16, q_dtype="f32",
             kv_dtype="f32", scale=1 / math.sqrt(128))
    a.update(kw)
    if a["kv_dtype"] == "e4m3":
        a.setdefault("kv_scale", 2.0 ** -5)
    return inputs.make_independent("tiny", rng, np.array(ctx), **a)


@pytest.mark.parametrize("dt", ["f32", "f16", "bf16"])
def test_context_one_returns_v1_bit_exact(dt):
    w = _tiny(1, [1] * 5, q_dtype=dt, kv_dtype=dt)
    st = gpu_state(w)
    out = st.out.cpu()
    G = w.num_q_heads // w.num_kv_heads
    for s in range(5):
        v = torch.from_numpy(np.ascontiguousarray(w.value[w.seq_tokens[s][0]]))
        if dt == "bf16":
            v = v.view(torch.int16).view(torch.bfloat16)
        assert torch.equal(out[s], v.repeat_interleave(G, 0))


def test_constant_values_give_the_constant():
    w = _tiny(2, [5, 100, 700, 2500], values="constant_v")
    st = gpu_state(w)
    v = to_f64(w.value[0], "f32")
    np.testing.assert_allclose(st.out_f64(), np.repeat(v, 4, 0)[None].repeat(4, 0), atol=2e-6)


def test_physical_block_permutation_is_bit_identical():
    w = _tiny(3, [7, 300, 1200, 2049], q_dtype="bf16", kv_dtype="bf16")
    a = gpu_state(w).out.clone()
    perm = np.random.default_rng(9).permutation(w.num_blocks)
    b = gpu_state(relabel_blocks(w, perm)).out.clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_repeated_decode_is_bit_identical():
    w = _tiny(4, [3000, 4100, 90, 513], q_dtype="f16", kv_dtype="f16")
    st = gpu_state(w)
    first = st.out.clone()
    for _ in range(3):
        st.decode()
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), st.out.view(torch.int16))


def test_nan_poison_outside_context_is_never_read():
    """The pool starts as NaN everywhere; only rows below context_len are written."""
    w = _tiny(5, [1, 15, 17, 33, 1000], q_dtype="bf16", kv_dtype="e4m3")
    st = gpu_state(w)
    assert torch.isfinite(st.out.float()).all()


def test_shared_prefix_cow_step_moves_no_data():
    """The step's copy-on-write repoint changes block ids, not data: the outputs agree.

    (Not bit for bit: the decode groups sequences by the physical blocks their
    tables share, so the repoint changes how much of the prompt is read once
    for the whole group, and with it the summation order.)"""
    w = inputs.make_config(4, num_seqs=16, ctx_cap=2000)
    st = gpu_state(w)
    with_cow = st.out_f64()
    tables = w.block_tables.copy()
    for src, dst in w.step_pairs:
        tables[tables == dst] = src
    st.block_tables.copy_(torch.from_numpy(tables))
    st.decode()
    torch.cuda.synchronize()
    assert np.abs(st.out_f64() - with_cow).max() <= tolerance(w)


def test_matches_dense_attention_on_logical_kv():
    """Independent of both caches: dense fp64 attention on the generator's logical rows."""
    w = _tiny(6, [40, 600, 1500], q_dtype="f32", kv_dtype="f32", num_q_heads=4,
              num_kv_heads=4)
    st = gpu_state(w)
    q = to_f64(w.query, "f32")
    for s in range(3):
        K, V = logical_kv_f64(w, s)
        for h in range(4):
            z = w.scale * K[:, h] @ q[s, h]
            p = np.exp(z - z.max())
            ref = p @ V[:, h] / p.sum()
            assert np.abs(st.out_f64()[s, h] - ref).max() <= 1e-4


# ------------------------------------------------------- device contract --

def test_bad_block_id_is_flagged_not_faulted():
    w = _tiny(7, [40, 40])
    st = gpu_state(w)
    bad = st.block_tables.clone()
    bad[1, 1] = w.num_blocks + 1000
    st.block_tables.copy_(bad)
    st.decode()
    assert binding.pkv_get_device_status() & binding.DEV_BAD_BLOCK_ID


@pytest.mark.parametrize("qdt,kvdt,prefix", [("bf16", "bf16", False), ("bf16", "bf16", True),
                                           ("f16", "e4m3", False), ("f16", "e4m3", True)])
def test_bad_block_id_is_flagged_on_the_tensor_core_paths(qdt, kvdt, prefix):
    """Table entries past the pool or negative, in split units of the tensor-core decode
    and of the prefix-aware launch: the producer flags them and loads block 0 instead."""
    w = _tiny(9, [40, 700, 1300, 1300], q_dtype=qdt, kv_dtype=kvdt)
    st = gpu_state(w, prefix=prefix)
    binding.pkv_get_device_status()          # clear
    bad = st.block_tables.clone()
    bad[1, 3] = w.num_blocks + 1000
    bad[2, 0] = -5
    st.block_tables.copy_(bad)
    st.decode()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_status() & binding.DEV_BAD_BLOCK_ID
    assert np.isfinite(st.out_f64()[0]).all()


def test_context_above_max_context_len_is_clamped_and_flagged():
    w = _tiny(8, [40, 100])
    st = gpu_state(w)
    binding.pkv_paged_decode_attention(st.query, st.k_cache, st.v_cache, st.block_tables,
                                       st.context_lens, 64, w.scale, workspace=st.workspace,
                                       out=st.out)
    assert binding.pkv_get_device_status() & binding.DEV_BAD_CONTEXT
    kc, vc = oracle_caches(w)
    ref = oracle_decode(w, kc, vc, context_lens=np.minimum(w.context_lens, 64))
    _check(w, st.out_f64(), ref)


@pytest.mark.parametrize("d,B,Hq,Hkv", [(64, 16, 8, 8), (128, 8, 8, 2), (64, 32, 12, 4),
                                        (128, 16, 16, 2)])
@pytest.mark.parametrize("qdt,kvdt", [("f32", "f32"), ("f32", "e4m3"), ("bf16", "e4m3")])
def test_single_launch_small_contexts(d, B, Hq, Hkv, qdt, kvdt):
    """Every context within one 512-token chunk: the CUDA-core path launches only the
    decode kernel, which takes its work items from the sequence index; empty
    sequences get zeros."""
    rng = np.random.default_rng(zlib.crc32(repr(("small", d, B, Hq, Hkv, qdt, kvdt)).encode()))
    ctx = np.array([0, 1, B - 1, B, B + 1, 100, 511, 512, 0, 300])
    w = inputs.make_independent("small", rng, ctx, num_q_heads=Hq, num_kv_heads=Hkv,
                                head_dim=d, block_size=B, q_dtype=qdt, kv_dtype=kvdt,
                                scale=1.0 / math.sqrt(d),
                                kv_scale=2.0 ** -5 if kvdt == "e4m3" else 1.0)
    assert w.max_context_len <= 512
    st, _ = _full_parity(w)
    out = st.out_f64()
    assert (out[0] == 0).all() and (out[8] == 0).all()


@pytest.mark.parametrize("qdt,kvdt,B", [("bf16", "bf16", 16), ("f16", "e4m3", 8)])
def test_many_short_units_over_every_cta(qdt, kvdt, B):
    """320 sequences of one or two chunks (about 10 tiles per CTA of the balanced split):
    many units straddle two CTAs' ranges.  Elementwise parity, then three more decodes
    must be bit-identical (every segment's partial state has a fixed slot and the
    merge runs in segment order)."""
    rng = np.random.default_rng(zlib.crc32(repr(("tail", qdt, kvdt, B)).encode()))
    ctx = rng.integers(1, 1100, size=320)
    ctx[:7] = [1, 63, 64, 65, 512, 513, 1099]
    w = inputs.make_independent("many short", rng, ctx, num_q_heads=32, num_kv_heads=8,
                                head_dim=128, block_size=B, q_dtype=qdt, kv_dtype=kvdt,
                                scale=1.0 / math.sqrt(128),
                                kv_scale=2.0 ** -5 if kvdt == "e4m3" else 1.0)
    st, _ = _full_parity(w)
    first = st.out.clone()
    for _ in range(3):
        st.decode()
        torch.cuda.synchronize()
        assert torch.equal(first.view(torch.int16), st.out.view(torch.int16))


@pytest.mark.parametrize("cid,kw,prefix", [(1, dict(num_seqs=8), False),
                                           (2, dict(num_seqs=32), False),
                                           (4, dict(num_seqs=16, ctx_cap=1500), True)])
def test_step_replays_in_a_cuda_graph(cid, kw, prefix):
    """The hot-path step (copy-on-write, cache write, decode: planner, decode kernel and
    for the prefix-aware entry the shared-prefix detection and the merge) captured in a
    CUDA graph after one eager step: every replay reproduces the eager output bit for
    bit (the step is idempotent)."""
    w = inputs.make_config(cid, **kw)
    st = gpu_state(w, prefix=prefix)
    eager = st.out.clone()
    stream = torch.cuda.Stream()
    pre, dec = st.prepare(stream)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        for c in pre:
            c()
        dec()
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            for c in pre:
                c()
            dec()
        for _ in range(2):
            st.out.zero_()
            graph.replay()
            stream.synchronize()
            assert torch.equal(eager.view(torch.int16), st.out.view(torch.int16))
    assert binding.pkv_get_device_status() == 0


@pytest.mark.parametrize("Hq,Hkv", [(32, 2), (64, 2), (128, 1)])
@pytest.mark.parametrize("qdt,kvdt", [("bf16", "bf16"), ("f16", "e4m3"), ("f32", "f32")])
@pytest.mark.parametrize("prefix", [False, True])
def test_wide_head_groups(Hq, Hkv, qdt, kvdt, prefix):
    """16 to 128 query heads per kv head: the tensor-core kernel serves a kv head's group
    in subgroups of 8 heads (each a work unit of its own), the CUDA-core kernel in items
    of up to 4; contexts over several chunks are split and merged. The prefix-aware
    entry point cannot group sequences here (more than 8 heads per kv head), so it runs
    the same units through its own planner and merge."""
    rng = np.random.default_rng(zlib.crc32(repr(("wide", Hq, Hkv, qdt, kvdt, prefix)).encode()))
    ctx = np.array([1, 100, 700, 1500, 0, 33])
    w = inputs.make_independent("wide", rng, ctx, num_q_heads=Hq, num_kv_heads=Hkv,
                                head_dim=128, block_size=16, q_dtype=qdt, kv_dtype=kvdt,
                                scale=1.0 / math.sqrt(128),
                                kv_scale=2.0 ** -5 if kvdt == "e4m3" else 1.0)
    st = gpu_state(w, prefix=prefix)
    kc, vc = oracle_caches(w)
    ref = oracle_decode(w, kc, vc, nthreads=8)
    _check(w, st.out_f64(), ref)
    assert binding.pkv_get_device_status() == 0
