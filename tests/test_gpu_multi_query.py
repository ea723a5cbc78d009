"""Multi-query (causal) paged attention on the GPU against the oracle.

Query row i of a sequence with n queries and ctx cached tokens attends to tokens
0 .. ctx - n + i ("PagedAttention: Mathematical Foundations ..." §1 prefill,
§3 attention through the block table).  The kernel runs Q K^T and P V on the
tcgen05 tensor cores; P is rounded to the operand type, so the comparison is by
the dtype's tolerance.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import binding, inputs
from paged_kv_cache_87_gb300.session import MultiQueryState
from tests.helpers import TOL

pytestmark = pytest.mark.gpu


def _oracle_pool(w):
    kc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    vc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slots, num_kv_heads=w.num_kv_heads,
                             head_dim=w.head_dim, block_size=w.block_size,
                             num_blocks=w.num_blocks, src_dtype=w.kv_dtype,
                             kv_dtype=w.kv_dtype)
    return kc, vc


def _oracle(w, sel=None):
    kc, vc = _oracle_pool(w)
    return oracle.paged_prefill_attention(
        w.query, kc, vc, w.block_tables, w.context_lens, w.query_start,
        num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale, q_dtype=w.q_dtype,
        kv_dtype=w.kv_dtype, sel=sel, nthreads=8)


def _gpu(w):
    st = MultiQueryState(w)
    st.run_setup()
    binding.pkv_get_device_status()          # clear
    st.step()
    torch.cuda.synchronize()
    return st


def _check(w):
    st = _gpu(w)
    got = st.out_f64()
    ref = _oracle(w)
    assert binding.pkv_get_device_status() == 0
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= TOL[w.q_dtype], err
    return st


def test_mixed_query_counts_bf16():
    _check(inputs.make_multi_query_config(0))


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("Hq,Hkv", [(2, 2), (8, 2), (16, 2), (16, 1)])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_groups_dtypes_block_sizes(dt, Hq, Hkv, B):
    rng = np.random.default_rng(Hq * 1000 + Hkv * 100 + B)
    w = inputs.make_multi_query("mq", rng, [0, 70, 250], [1, 40, 150], num_q_heads=Hq,
                                num_kv_heads=Hkv, head_dim=128, block_size=B, dtype=dt)
    _check(w)


def test_prompts_without_prior_context_ragged_tiles():
    rng = np.random.default_rng(21)
    w = inputs.make_multi_query("prefill", rng, [0, 0, 0], [129, 300, 1], num_q_heads=4,
                                num_kv_heads=4, head_dim=128, block_size=16, dtype="bf16")
    _check(w)


@pytest.mark.parametrize("Hq,Hkv", [(64, 1), (128, 1), (128, 2)])
@pytest.mark.parametrize("tree", [False, True])
def test_widest_head_groups(Hq, Hkv, tree):
    """64 and 128 query heads per kv head: a row tile holds two or one query tokens of
    every head of the group (the Q box is 64 elements x G heads x 128 / G tokens)."""
    rng = np.random.default_rng(25 + Hq + Hkv)
    prior, n = [0, 130, 1000, 5], [9, 40, 3, 64]
    if tree:
        w = inputs.make_tree_verify("wide-tree", rng, prior, n, num_q_heads=Hq, num_kv_heads=Hkv,
                                    head_dim=128, block_size=16, dtype="bf16")
        _check_tree(w)
    else:
        w = inputs.make_multi_query("wide", rng, prior, n, num_q_heads=Hq, num_kv_heads=Hkv,
                                    head_dim=128, block_size=16, dtype="bf16")
        _check(w)


@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (16, 4), (32, 1)])
def test_prompts_of_many_lengths(Hq, Hkv):
    """Prompts without prior context: ties, a prompt of zero tokens, prompts shorter than
    one row pair and prompts of many pairs, against the oracle."""
    rng = np.random.default_rng(23 + Hq)
    n = [700, 700, 0, 1, 255, 1300, 64, 513, 256, 900]
    w = inputs.make_multi_query("prompts", rng, [0] * len(n), n, num_q_heads=Hq,
                                num_kv_heads=Hkv, head_dim=128, block_size=16, dtype="bf16")
    _check(w)


def test_prompt_order_leaves_every_prompt_bit_identical():
    """Each prompt's items are computed the same way wherever the planner puts them:
    permuting the prompts permutes the output rows, bit for bit, and a prompt run alone
    gives the same bits."""
    rng = np.random.default_rng(24)
    n = [300, 1025, 17, 600, 600, 90]
    w = inputs.make_multi_query("prompts", rng, [0] * len(n), n, num_q_heads=8, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="f16")
    a = _gpu(w).out.clone()
    perm = np.array([4, 1, 5, 0, 3, 2])
    qs = w.query_start
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in perm])
    nn = np.diff(qs)[perm]
    w2 = inputs.MultiQueryWorkload(**{**w.__dict__, "query": w.query[rows],
                                      "block_tables": w.block_tables[perm],
                                      "context_lens": w.context_lens[perm],
                                      "query_start": np.concatenate([[0], np.cumsum(nn)]).astype(np.int32),
                                      "seq_tokens": [w.seq_tokens[s] for s in perm]})
    b = _gpu(w2).out
    assert binding.pkv_get_device_status() == 0
    assert torch.equal(a[torch.from_numpy(rows).to(a.device)], b)
    one = inputs.MultiQueryWorkload(**{**w.__dict__, "num_seqs": 1, "query": w.query[qs[1]:qs[2]],
                                       "block_tables": w.block_tables[1:2],
                                       "context_lens": w.context_lens[1:2],
                                       "query_start": np.array([0, n[1]], np.int32),
                                       "seq_tokens": [w.seq_tokens[1]]})
    c = _gpu(one).out
    assert torch.equal(a[int(qs[1]):int(qs[2])], c)


def test_long_prior_context_many_kv_tiles():
    rng = np.random.default_rng(22)
    w = inputs.make_multi_query("long", rng, [3000, 1700], [200, 70], num_q_heads=8,
                                num_kv_heads=2, head_dim=128, block_size=16, dtype="bf16")
    _check(w)


def test_scaled_logits_move_the_running_max():
    """Large logits (scale 0.35 instead of 1/sqrt(128)) make later tiles exceed the
    running max by more than the rescale headroom, exercising the O rescale in
    tensor memory."""
    rng = np.random.default_rng(23)
    w = inputs.make_multi_query("big logits", rng, [900], [100], num_q_heads=4, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="bf16", scale=0.35)
    _check(w)


def test_physical_block_relabelling_is_bit_invariant():
    rng = np.random.default_rng(24)
    w = inputs.make_multi_query("relabel", rng, [100, 333], [60, 90], num_q_heads=8,
                                num_kv_heads=2, head_dim=128, block_size=16, dtype="bf16")
    a = _gpu(w).out.clone()
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    w2 = inputs.MultiQueryWorkload(**{**w.__dict__, "slots": perm[w.slots // w.block_size] *
                                      w.block_size + w.slots % w.block_size,
                                      "block_tables": np.where(w.block_tables >= 0,
                                                               perm[np.maximum(w.block_tables, 0)],
                                                               -1).astype(np.int32)})
    b = _gpu(w2).out
    assert torch.equal(a, b)


def test_one_query_per_sequence_equals_the_decode_kernel():
    rng = np.random.default_rng(25)
    w = inputs.make_multi_query("one", rng, [10, 500, 2047, 64], [1, 1, 1, 1], num_q_heads=16,
                                num_kv_heads=4, head_dim=128, block_size=16, dtype="bf16")
    st = _gpu(w)
    dec = binding.pkv_paged_decode_attention(st.query, st.k_cache, st.v_cache, st.block_tables,
                                             st.context_lens, w.max_context_len, w.scale)
    torch.cuda.synchronize()
    err = (st.out.double() - dec.double()).abs().max().item()
    assert err <= TOL["bf16"], err
    ref = _oracle(w)
    assert np.abs(st.out_f64() - ref).max() <= TOL["bf16"]


def test_sequence_with_more_queries_than_context_is_flagged_and_skipped():
    rng = np.random.default_rng(26)
    w = inputs.make_multi_query("bad", rng, [20, 40], [10, 10], num_q_heads=4, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="bf16")
    st = MultiQueryState(w)
    st.run_setup()
    st.append_step()
    st.context_lens[0] = 5                   # 10 queries over 5 tokens: a contract violation
    st.out.fill_(7.0)
    binding.pkv_get_device_status()
    st.attend()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_status() & binding.DEV_BAD_CONTEXT
    assert torch.all(st.out[:10] == 7.0)     # the bad sequence's rows are untouched
    ref = _oracle(w)
    assert np.abs(st.out_f64()[10:] - ref[10:]).max() <= TOL["bf16"]


@pytest.mark.parametrize("tree", [False, True])
def test_bad_block_id_is_flagged_not_faulted(tree):
    """A table entry past the pool: the TMA producer flags it and loads block 0 instead."""
    rng = np.random.default_rng(32)
    make = inputs.make_tree_verify if tree else inputs.make_multi_query
    w = make("bad", rng, [300, 40], [20, 64], num_q_heads=8, num_kv_heads=2, head_dim=128,
             block_size=16, dtype="bf16")
    st = MultiQueryState(w)
    st.run_setup()
    st.append_step()
    binding.pkv_get_device_status()          # clear
    bad = st.block_tables.clone()
    bad[0, 2] = w.num_blocks + 77
    st.block_tables.copy_(bad)
    st.attend()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_status() & binding.DEV_BAD_BLOCK_ID
    assert np.isfinite(st.out_f64()[w.query_start[1]:]).all()   # the other sequence


def test_unsupported_shapes_and_types_are_refused():
    rng = np.random.default_rng(27)
    w = inputs.make_multi_query("f32", rng, [5], [3], num_q_heads=2, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="f32")
    st = MultiQueryState(w)
    with pytest.raises(binding.PagedKVError) as e:
        st.attend()
    assert e.value.status == binding.PKV_ERR_UNSUPPORTED
    w = inputs.make_multi_query("d64", rng, [5], [3], num_q_heads=2, num_kv_heads=2,
                                head_dim=64, block_size=16, dtype="bf16")
    st = MultiQueryState(w)
    with pytest.raises(binding.PagedKVError) as e:
        st.attend()
    assert e.value.status == binding.PKV_ERR_UNSUPPORTED
    w = inputs.make_multi_query("g3", rng, [5], [3], num_q_heads=6, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="bf16")
    st = MultiQueryState(w)
    with pytest.raises(binding.PagedKVError) as e:
        st.attend()
    assert e.value.status == binding.PKV_ERR_UNSUPPORTED


def test_no_queries_is_a_no_op():
    rng = np.random.default_rng(28)
    w = inputs.make_multi_query("empty", rng, [5, 9], [0, 0], num_q_heads=2, num_kv_heads=2,
                                head_dim=128, block_size=16, dtype="bf16")
    st = MultiQueryState(w)
    st.attend()
    torch.cuda.synchronize()


def test_chunked_prefill_workload_sampled():
    """The benchmark's workload at full size: sampled rows of every sequence."""
    w = inputs.make_multi_query_config(1)
    st = _gpu(w)
    assert binding.pkv_get_device_status() == 0
    got = st.out_f64()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(0)
    rows = []
    for s in range(w.num_seqs):
        q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
        rows += [q0, q1 - 1] + list(rng.integers(q0, q1, size=2))
    sel = np.array([(r, int(h)) for r in rows for h in rng.integers(0, w.num_q_heads, size=2)],
                   dtype=np.int32)
    ref = _oracle(w, sel=sel)
    err = np.abs(got[sel[:, 0], sel[:, 1]] - ref).max()
    assert err <= TOL["bf16"], err


def test_more_sequences_than_the_planner_ranks():
    """Above 1024 sequences the planner launches them in index order instead of by
    context length; results must not depend on it."""
    rng = np.random.default_rng(29)
    S = 1100
    w = inputs.make_multi_query("many", rng, rng.integers(0, 41, size=S), rng.integers(1, 4, size=S),
                                num_q_heads=4, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype="bf16")
    _check(w)


def test_launch_order_leaves_every_sequence_bit_identical():
    """The CTAs of each sequence compute the same values whatever position the planner
    gives the sequence: permuting the sequences permutes the output rows, bit for bit."""
    rng = np.random.default_rng(30)
    w = inputs.make_multi_query("order", rng, [700, 3, 260, 1500, 90, 1100], [40, 9, 130, 3, 77, 256],
                                num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype="bf16")
    a = _gpu(w).out.clone()
    perm = np.array([3, 0, 5, 2, 4, 1])
    qs = w.query_start
    rows = np.concatenate([np.arange(qs[s], qs[s + 1]) for s in perm])
    n = np.diff(qs)[perm]
    w2 = inputs.MultiQueryWorkload(**{**w.__dict__, "query": w.query[rows],
                                      "block_tables": w.block_tables[perm],
                                      "context_lens": w.context_lens[perm],
                                      "query_start": np.concatenate([[0], np.cumsum(n)]).astype(np.int32),
                                      "seq_tokens": [w.seq_tokens[s] for s in perm]})
    b = _gpu(w2).out
    assert binding.pkv_get_device_status() == 0
    assert torch.equal(a[torch.from_numpy(rows).to(a.device)], b)


def _offset_out(like: torch.Tensor) -> torch.Tensor:
    """An output tensor shaped like `like` whose data starts 16 bytes past a 32-byte
    boundary (the kernel then writes 16-byte pieces instead of 32-byte ones)."""
    buf = torch.empty(like.numel() + 64, dtype=like.dtype, device=like.device)
    base = buf.data_ptr()
    skip = ((-base) % 32 + 16) // like.element_size()
    out = buf[skip:skip + like.numel()].view(like.shape)
    assert out.data_ptr() % 32 == 16
    return out


@pytest.mark.parametrize("tree", [False, True])
def test_output_16_byte_aligned_only_is_bit_identical(tree):
    """The 32-byte-store and 16-byte-store epilogues write the same bits."""
    rng = np.random.default_rng(31)
    prior, n = [300, 0, 1000, 77], [64, 33 if tree else 200, 40, 9]
    if tree:
        w = inputs.make_tree_verify("tree-align", rng, prior, n, num_q_heads=8, num_kv_heads=2,
                                    head_dim=128, block_size=16, dtype="bf16")
        st = _check_tree(w)
    else:
        w = inputs.make_multi_query("align", rng, prior, n, num_q_heads=8, num_kv_heads=2,
                                    head_dim=128, block_size=16, dtype="bf16")
        st = _check(w)
    assert st.out.data_ptr() % 32 == 0
    out16 = _offset_out(st.out)
    out16.fill_(float("nan"))
    st.attend(out=out16)
    torch.cuda.synchronize()
    assert binding.pkv_get_device_status() == 0
    assert torch.equal(out16, st.out)


# ------------------------------------------------------------ draft trees --

def _oracle_tree(w, sel=None):
    kc, vc = _oracle_pool(w)
    return oracle.paged_tree_attention(
        w.query, kc, vc, w.block_tables, w.context_lens, w.query_start, w.tree,
        num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale, q_dtype=w.q_dtype,
        kv_dtype=w.kv_dtype, sel=sel, nthreads=8)


def _check_tree(w):
    st = _gpu(w)
    got = st.out_f64()
    ref = _oracle_tree(w)
    assert binding.pkv_get_device_status() == 0
    assert np.isfinite(got).all()
    err = np.abs(got - ref).max()
    assert err <= TOL[w.q_dtype], err
    return st


@pytest.mark.parametrize("dt", ["bf16", "f16"])
@pytest.mark.parametrize("Hq,Hkv", [(8, 8), (8, 2), (32, 8), (16, 1)])
@pytest.mark.parametrize("B", [8, 16, 32])
def test_draft_trees_groups_dtypes_block_sizes(dt, Hq, Hkv, B):
    rng = np.random.default_rng(Hq * 100 + Hkv * 10 + B)
    w = inputs.make_tree_verify("trees", rng, [0, 130, 700, 64], [17, 64, 33, 1],
                                kinds=["random", "random", "star", "chain"], num_q_heads=Hq,
                                num_kv_heads=Hkv, head_dim=128, block_size=B, dtype=dt)
    _check_tree(w)


def test_draft_trees_straddling_kv_tiles():
    """Trees whose tokens cross a 128-token K/V tile boundary (prior context 100, 200)."""
    rng = np.random.default_rng(41)
    w = inputs.make_tree_verify("straddle", rng, [100, 200, 1000], [64, 50, 40],
                                num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype="bf16")
    _check_tree(w)


def test_chain_tree_equals_the_causal_kernel_bit_for_bit():
    rng = np.random.default_rng(42)
    w = inputs.make_tree_verify("chain", rng, [300, 5, 2000], [40, 9, 64],
                                kinds=["chain"] * 3, num_q_heads=16, num_kv_heads=4,
                                head_dim=128, block_size=16, dtype="bf16")
    a = _gpu(w).out.clone()
    b = _gpu(inputs.MultiQueryWorkload(**{**w.__dict__, "tree": None})).out
    assert torch.equal(a, b)


def test_tree_of_more_than_64_tokens_is_flagged_and_skipped():
    rng = np.random.default_rng(43)
    w = inputs.make_multi_query("big tree", rng, [50, 80], [65, 20], num_q_heads=4,
                                num_kv_heads=2, head_dim=128, block_size=16, dtype="bf16")
    w.tree = np.concatenate([np.zeros(65, np.uint64),
                             inputs.tree_ancestors(inputs.random_tree_parents(rng, 20))])
    st = MultiQueryState(w)
    st.run_setup()
    st.append_step()
    st.out.fill_(7.0)
    binding.pkv_get_device_status()
    st.attend()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_status() & binding.DEV_BAD_CONTEXT
    assert torch.all(st.out[:65] == 7.0)
    ref = oracle.paged_tree_attention(
        w.query[65:], *_oracle_pool(w), w.block_tables[1:], w.context_lens[1:],
        w.query_start[1:] - 65, w.tree[65:], num_q_heads=4, num_kv_heads=2, head_dim=128,
        block_size=16, num_blocks=w.num_blocks, scale=w.scale, q_dtype="bf16", kv_dtype="bf16")
    assert np.abs(st.out_f64()[65:] - ref).max() <= TOL["bf16"]


def test_tree_verification_workload_sampled():
    """The benchmark's draft-tree workload at full size: sampled rows of every sequence."""
    w = inputs.make_multi_query_config(3)
    st = _gpu(w)
    assert binding.pkv_get_device_status() == 0
    got = st.out_f64()
    assert np.isfinite(got).all()
    rng = np.random.default_rng(1)
    rows = []
    for s in range(w.num_seqs):
        q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
        rows += [q0, q1 - 1] + list(rng.integers(q0, q1, size=2))
    sel = np.array([(r, int(h)) for r in rows for h in rng.integers(0, w.num_q_heads, size=2)],
                   dtype=np.int32)
    ref = _oracle_tree(w, sel=sel)
    err = np.abs(got[sel[:, 0], sel[:, 1]] - ref).max()
    assert err <= TOL["bf16"], err
