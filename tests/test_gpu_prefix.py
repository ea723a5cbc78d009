"""Prefix-aware decode: sequences whose tables share leading blocks are grouped and the
shared blocks are streamed once for every member ("PagedAttention: Mathematical
Foundations ..." §5 Parallel Sampling, System Prompt Prefix Sharing).  Results must
match the oracle, which knows nothing about sharing."""
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_87_gb300 import binding, inputs
from tests.helpers import gpu_state, oracle_caches, oracle_decode, tolerance

pytestmark = pytest.mark.gpu


def _check(w, prefix=True):
    st = gpu_state(w, prefix=prefix)
    kc, vc = oracle_caches(w)
    ref = oracle_decode(w, kc, vc, nthreads=8)
    err = np.abs(st.out_f64() - ref).max()
    assert np.isfinite(st.out_f64()).all() and err <= tolerance(w), err
    return st


@pytest.mark.parametrize("samples,Hq,Hkv", [(2, 8, 8), (4, 32, 8), (5, 32, 8), (3, 16, 2),
                                            (2, 16, 2), (17, 4, 4), (3, 6, 2)])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_shared_prefix_groups_bf16(samples, Hq, Hkv, B):
    rng = np.random.default_rng(samples * 100 + Hq + B)
    w = inputs.make_shared_prefix("prefix", rng, num_groups=3, samples=samples, prefix_lo=40,
                                  prefix_hi=700, tail_lo=1, tail_hi=150, num_q_heads=Hq,
                                  num_kv_heads=Hkv, head_dim=128, block_size=B, q_dtype="bf16",
                                  kv_dtype="bf16", kv_scale=1.0, scale=1 / math.sqrt(128))
    _check(w)


@pytest.mark.parametrize("dt,kv,d", [("f16", "f16", 64), ("f16", "f16", 128),
                                     ("bf16", "bf16", 64), ("bf16", "e4m3", 128),
                                     ("f16", "e4m3", 128), ("f32", "f32", 64),
                                     ("f32", "e4m3", 128), ("bf16", "e4m3", 64)])
def test_shared_prefix_groups_types(dt, kv, d):
    rng = np.random.default_rng(7)
    w = inputs.make_shared_prefix("prefix", rng, num_groups=4, samples=4, prefix_lo=64,
                                  prefix_hi=2000, tail_lo=1, tail_hi=300, num_q_heads=32,
                                  num_kv_heads=8, head_dim=d, block_size=16, q_dtype=dt,
                                  kv_dtype=kv, kv_scale=2.0 ** -5 if kv == "e4m3" else 1.0,
                                  scale=1 / math.sqrt(d))
    _check(w)


def test_whole_context_shared_and_mixed_batch():
    """Members with identical tables and lengths (nothing private) next to ungrouped ones."""
    rng = np.random.default_rng(11)
    base = inputs.make_independent("x", rng, np.array([256, 77, 512, 300, 1000]),
                                   num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                                   q_dtype="bf16", kv_dtype="bf16", scale=1 / math.sqrt(128))
    # sequences 0,1,2 become copies of sequence 0's table and length (256 = 4 whole tiles):
    # one group whose members have no private tokens
    t = base.block_tables.copy()
    ctx = base.context_lens.copy()
    order = [0, 0, 0, 1, 2, 3, 4]
    w = inputs.Workload(
        name="shared", num_seqs=len(order), num_q_heads=16, num_kv_heads=4, head_dim=128,
        block_size=16, num_blocks=base.num_blocks, q_dtype="bf16", src_dtype="bf16",
        kv_dtype="bf16", kv_scale=1.0, scale=base.scale,
        query=inputs.draw_normal(rng, (len(order), 16, 128), "bf16"), key=base.key,
        value=base.value, setup=base.setup, step_pairs=base.step_pairs,
        new_vec=base.new_vec[order], new_slots=base.new_slots[order],
        block_tables=np.ascontiguousarray(t[order]), context_lens=np.ascontiguousarray(ctx[order]),
        seq_tokens=[base.seq_tokens[i] for i in order])
    st = _check(w)
    _check(w, prefix=False)
    # the three identical sequences differ only in their queries
    assert not torch.equal(st.out[0], st.out[1])


def test_plain_decode_on_shared_prompts():
    """The plain entry point on the same shared-prompt batch (no grouping)."""
    rng = np.random.default_rng(8)
    w = inputs.make_shared_prefix("prefix", rng, num_groups=3, samples=4, prefix_lo=64,
                                  prefix_hi=900, tail_lo=1, tail_hi=100, num_q_heads=16,
                                  num_kv_heads=4, head_dim=128, block_size=16, q_dtype="bf16",
                                  kv_dtype="bf16", kv_scale=1.0, scale=1 / math.sqrt(128))
    _check(w, prefix=False)


def test_grouping_is_invariant_under_block_relabeling():
    from tests.helpers import relabel_blocks
    w = inputs.make_config(4, num_seqs=16, ctx_cap=1500)
    a = gpu_state(w, prefix=True).out.clone()
    perm = np.random.default_rng(3).permutation(w.num_blocks)
    b = gpu_state(relabel_blocks(w, perm), prefix=True).out.clone()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("prefix", [True, False])
def test_batches_above_one_planner_tile(prefix):
    """More than 1024 sequences: the planner walks several tiles of sequences."""
    rng = np.random.default_rng(21)
    w = inputs.make_shared_prefix("many", rng, num_groups=300, samples=4, prefix_lo=64,
                                  prefix_hi=160, tail_lo=1, tail_hi=40, num_q_heads=8,
                                  num_kv_heads=2, head_dim=128, block_size=16, q_dtype="bf16",
                                  kv_dtype="bf16", kv_scale=1.0, scale=1 / math.sqrt(128))
    assert w.num_seqs == 1200
    _check(w, prefix=prefix)


def test_plain_batch_above_one_planner_tile():
    rng = np.random.default_rng(22)
    ctx = rng.integers(0, 300, size=1300)
    w = inputs.make_independent("many", rng, ctx, num_q_heads=16, num_kv_heads=4, head_dim=64,
                                block_size=8, q_dtype="f16", kv_dtype="f16",
                                scale=1 / math.sqrt(64))
    st = _check(w, prefix=False)
    assert (st.out_f64()[ctx == 0] == 0).all()


def _prefix_workload(seed, B=16, groups=3, lo=600, hi=900):
    rng = np.random.default_rng(seed)
    return inputs.make_shared_prefix("prefix", rng, num_groups=groups, samples=4, prefix_lo=lo,
                                     prefix_hi=hi, tail_lo=1, tail_hi=60, num_q_heads=16,
                                     num_kv_heads=4, head_dim=128, block_size=B, q_dtype="bf16",
                                     kv_dtype="bf16", kv_scale=1.0, scale=1 / math.sqrt(128))


@pytest.mark.parametrize("pad", [0, 1, 2, 3])
def test_table_width_of_every_alignment(pad):
    """Tables whose rows start at every 4-byte offset modulo 16 (padded widths)."""
    import dataclasses
    w = _prefix_workload(31)
    width = (w.max_blocks + 3) // 4 * 4 + pad
    t = np.full((w.num_seqs, width), -1, np.int32)
    t[:, :w.max_blocks] = w.block_tables
    _check(dataclasses.replace(w, block_tables=t))


@pytest.mark.parametrize("pad", [0, 1])
def test_member_rows_that_diverge_inside_the_prefix(pad):
    """Members whose rows leave the leader's at entries 5, 100 and 140 (the planner
    compares rows in spans of 128 entries): only the entries before the first
    difference are shared."""
    import dataclasses
    w = _prefix_workload(32, lo=2500, hi=3000)
    width = (w.max_blocks + 3) // 4 * 4 + pad
    t = np.full((w.num_seqs, width), -1, np.int32)
    t[:, :w.max_blocks] = w.block_tables
    donor = int(t[8, 1])                     # a full block of another group's prompt
    for seq, j in ((1, 5), (2, 100), (3, 140)):
        assert t[seq, j] != donor and j * 16 + 16 <= w.context_lens[seq] - 64
        t[seq, j] = donor
    _check(dataclasses.replace(w, block_tables=t))


@pytest.mark.parametrize("kv", ["bf16", "e4m3"])
def test_many_groups_split_over_every_cta(kv):
    """48 groups of 4 samples: shared and private units cut across many CTAs' ranges,
    merged per member; a repeated decode is bit-identical."""
    rng = np.random.default_rng(41 if kv == "bf16" else 42)
    w = inputs.make_shared_prefix("many groups", rng, num_groups=48, samples=4, prefix_lo=600,
                                  prefix_hi=2500, tail_lo=1, tail_hi=200, num_q_heads=32,
                                  num_kv_heads=8, head_dim=128, block_size=16, q_dtype="bf16",
                                  kv_dtype=kv, kv_scale=2.0 ** -5 if kv == "e4m3" else 1.0,
                                  scale=1 / math.sqrt(128))
    st = _check(w)
    first = st.out.clone()
    st.decode()
    torch.cuda.synchronize()
    assert torch.equal(first.view(torch.int16), st.out.view(torch.int16))


@pytest.mark.parametrize("prefix", [True, False])
def test_more_records_than_the_planner_keeps_in_shared_memory(prefix):
    """1,500 groups of 3 samples: 1,500 group records and 4,500 private ones, beyond the
    4,096 record offsets the planner keeps in shared memory, so the workers find their
    first record in the global copy."""
    rng = np.random.default_rng(23)
    w = inputs.make_shared_prefix("records", rng, num_groups=1500, samples=3, prefix_lo=32,
                                  prefix_hi=96, tail_lo=1, tail_hi=30, num_q_heads=8,
                                  num_kv_heads=2, head_dim=128, block_size=16, q_dtype="bf16",
                                  kv_dtype="bf16", kv_scale=1.0, scale=1 / math.sqrt(128))
    assert w.num_seqs == 4500
    _check(w, prefix=prefix)


def test_plain_batch_beyond_the_planner_record_cache():
    """5,000 independent sequences: one record each, beyond the planner's 4,096 cached
    record offsets."""
    rng = np.random.default_rng(24)
    ctx = rng.integers(0, 200, size=5000)
    w = inputs.make_independent("records", rng, ctx, num_q_heads=8, num_kv_heads=2,
                                head_dim=128, block_size=16, q_dtype="bf16", kv_dtype="bf16",
                                scale=1 / math.sqrt(128))
    st = _check(w, prefix=False)
    assert (st.out_f64()[ctx == 0] == 0).all()
