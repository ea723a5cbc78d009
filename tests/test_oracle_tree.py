"""Pins of the oracle's draft-tree verification (CPU, no GPU).

The last n tokens of a sequence are a tree of draft tokens laid out parents first;
query i sees the prior context, itself and its ancestors (a reading of the
speculative decoding trees of "PagedAttention: Mathematical Foundations ..." §9,
with the attention of §3).  The pins do not use the oracle's arithmetic: torch's
scaled_dot_product_attention in fp64 with a mask built by walking the parent
pointers, a two-token closed form, and the causal oracle (pinned on its own).
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import inputs


def _pool(w):
    kc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    vc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slots, num_kv_heads=w.num_kv_heads,
                             head_dim=w.head_dim, block_size=w.block_size,
                             num_blocks=w.num_blocks, src_dtype=w.kv_dtype,
                             kv_dtype=w.kv_dtype)
    return kc, vc


def _args(w):
    return dict(num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
                block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale,
                q_dtype=w.q_dtype, kv_dtype=w.kv_dtype)


def _tree(w, kc, vc, tree=None):
    return oracle.paged_tree_attention(w.query, kc, vc, w.block_tables, w.context_lens,
                                       w.query_start, w.tree if tree is None else tree, **_args(w))


def _workload(prior, n, parents, *, hq=4, hkv=2, d=16, b=4, seed=7):
    w = inputs.make_multi_query("tree pin", np.random.default_rng(seed), prior, n,
                                num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=b,
                                dtype="f32")
    w.tree = np.concatenate([inputs.tree_ancestors(p) for p in parents])
    return w


def _sdpa_tree(w, s, parent):
    """torch SDPA (fp64) for sequence s: query i sees the prior context and the tree
    tokens on its path to the root (found by following parent pointers)."""
    f64 = lambda a: np.asarray(a, dtype=np.float64)
    G = w.num_q_heads // w.num_kv_heads
    rows = w.seq_tokens[s]
    K = torch.from_numpy(f64(w.key[rows])).permute(1, 0, 2).repeat_interleave(G, 0)
    V = torch.from_numpy(f64(w.value[rows])).permute(1, 0, 2).repeat_interleave(G, 0)
    q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
    Q = torch.from_numpy(f64(w.query[q0:q1])).permute(1, 0, 2)
    n, ctx = q1 - q0, int(w.context_lens[s])
    mask = torch.zeros(n, ctx, dtype=torch.bool)
    mask[:, :ctx - n] = True
    for i in range(n):
        j = i
        while j >= 0:                      # the token itself, then each ancestor
            mask[i, ctx - n + j] = True
            j = int(parent[j])
    o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask, scale=w.scale)
    return o.permute(1, 0, 2).numpy()


def test_random_trees_match_sdpa_with_parent_walk_mask():
    rng = np.random.default_rng(11)
    n = [5, 9, 1, 13]
    parents = [inputs.random_tree_parents(rng, k) for k in n]
    w = _workload([0, 6, 3, 21], n, parents)
    kc, vc = _pool(w)
    got = _tree(w, kc, vc)
    for s in range(w.num_seqs):
        q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
        np.testing.assert_allclose(got[q0:q1], _sdpa_tree(w, s, parents[s]), rtol=0, atol=1e-12)


def test_chain_tree_and_all_ones_mask_equal_causal_attention():
    n = [4, 7, 1]
    parents = [inputs.random_tree_parents(None, k, "chain") for k in n]
    w = _workload([0, 5, 2], n, parents, seed=8)
    kc, vc = _pool(w)
    causal = oracle.paged_prefill_attention(w.query, kc, vc, w.block_tables, w.context_lens,
                                            w.query_start, **_args(w))
    np.testing.assert_allclose(_tree(w, kc, vc), causal, rtol=0, atol=1e-12)
    # bits j >= i are ignored: every bit set is the causal attention too
    ones = np.full(w.total_q, np.iinfo(np.uint64).max, dtype=np.uint64)
    np.testing.assert_allclose(_tree(w, kc, vc, ones), causal, rtol=0, atol=1e-12)


def test_star_tree_without_prior_context_is_a_two_token_softmax():
    n = 6
    w = _workload([0], [n], [inputs.random_tree_parents(None, n, "star")], hq=2, hkv=2, seed=9)
    kc, vc = _pool(w)
    got = _tree(w, kc, vc)
    K = np.asarray(w.key, np.float64)
    V = np.asarray(w.value, np.float64)
    Q = np.asarray(w.query, np.float64)
    for h in range(w.num_q_heads):
        np.testing.assert_allclose(got[0, h], V[0, h], rtol=0, atol=1e-12)   # the root: itself
        for i in range(1, n):
            z = w.scale * np.array([Q[i, h] @ K[0, h], Q[i, h] @ K[i, h]])
            a = np.exp(z - z.max())
            want = (a[0] * V[0, h] + a[1] * V[i, h]) / a.sum()
            np.testing.assert_allclose(got[i, h], want, rtol=0, atol=1e-12)


def test_tree_ancestor_masks_of_a_known_tree():
    #        0
    #      /   \
    #     1     4
    #    / \
    #   2   3
    anc = inputs.tree_ancestors([-1, 0, 1, 1, 0])
    assert anc.tolist() == [0, 0b1, 0b11, 0b11, 0b1]
    with pytest.raises(ValueError):
        inputs.tree_ancestors([-1, 2, 0])              # a parent after its child
    with pytest.raises(ValueError):
        inputs.tree_ancestors(np.full(65, 0))


def test_trees_of_more_than_64_tokens_are_rejected():
    n = 65
    w = inputs.make_multi_query("big", np.random.default_rng(1), [0], [n], num_q_heads=2,
                                num_kv_heads=2, head_dim=16, block_size=4, dtype="f32")
    kc, vc = _pool(w)
    with pytest.raises(ValueError):
        _tree(w, kc, vc, np.zeros(n, np.uint64))


def test_chain_tree_flops_equal_causal_flops():
    w = _workload([3, 10], [5, 8], [inputs.random_tree_parents(None, k, "chain") for k in (5, 8)])
    causal = inputs.MultiQueryWorkload(**{**w.__dict__, "tree": None})
    assert w.flops == causal.flops
