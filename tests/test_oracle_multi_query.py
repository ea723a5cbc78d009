"""Pins of the oracle's multi-query (causal) paged attention (CPU, no GPU).

Query row i of a sequence with n queries and ctx cached tokens is the token at
position ctx - n + i and attends to tokens 0 .. ctx - n + i ("PagedAttention:
Mathematical Foundations ..." §1, the prefill phase; §3, the attention
formula through the block table).  The pins here do not use the oracle's own
arithmetic: torch's scaled_dot_product_attention in fp64 on the table-free
logical K/V (with an explicit position mask, and with its own is_causal flag
for prompts without prior context), closed forms, and the decode oracle's
result for the last row, which is pinned separately.
"""
import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import inputs


def _pool(w):
    """The oracle's own reshape_and_cache fills a NaN-poisoned pool with every row."""
    kc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    vc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    oracle.reshape_and_cache(w.key, w.value, kc, vc, w.slots, num_kv_heads=w.num_kv_heads,
                             head_dim=w.head_dim, block_size=w.block_size,
                             num_blocks=w.num_blocks, src_dtype=w.kv_dtype,
                             kv_dtype=w.kv_dtype)
    return kc, vc


def _oracle_mq(w, kc, vc, sel=None):
    return oracle.paged_prefill_attention(
        w.query, kc, vc, w.block_tables, w.context_lens, w.query_start,
        num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale, q_dtype=w.q_dtype,
        kv_dtype=w.kv_dtype, sel=sel)


def _f64(a):
    return np.asarray(a, dtype=np.float64)


def _small(prior, n, *, hq=4, hkv=2, d=16, b=4, seed=3):
    return inputs.make_multi_query("pin", np.random.default_rng(seed), prior, n, num_q_heads=hq,
                                   num_kv_heads=hkv, head_dim=d, block_size=b, dtype="f32")


def _sdpa_reference(w, s, causal_flag=False):
    """torch SDPA (fp64) for sequence s on its logical K/V, GQA heads repeated."""
    G = w.num_q_heads // w.num_kv_heads
    rows = w.seq_tokens[s]
    K = torch.from_numpy(_f64(w.key[rows])).permute(1, 0, 2).repeat_interleave(G, 0)
    V = torch.from_numpy(_f64(w.value[rows])).permute(1, 0, 2).repeat_interleave(G, 0)
    q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
    Q = torch.from_numpy(_f64(w.query[q0:q1])).permute(1, 0, 2)       # [Hq, n, d]
    n, ctx = q1 - q0, int(w.context_lens[s])
    if causal_flag:
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, is_causal=True,
                                                             scale=w.scale)
    else:
        pos = torch.arange(n)[:, None] + (ctx - n)
        mask = torch.arange(ctx)[None, :] <= pos                       # [n, ctx]
        o = torch.nn.functional.scaled_dot_product_attention(Q, K, V, attn_mask=mask,
                                                             scale=w.scale)
    return o.permute(1, 0, 2).numpy()                                 # [n, Hq, d]


def test_multi_query_matches_masked_sdpa_on_logical_kv():
    w = _small([0, 5, 9, 17], [3, 4, 1, 6])
    kc, vc = _pool(w)
    got = _oracle_mq(w, kc, vc)
    for s in range(w.num_seqs):
        q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
        np.testing.assert_allclose(got[q0:q1], _sdpa_reference(w, s), rtol=0, atol=1e-12)


def test_prompt_without_prior_context_matches_sdpa_is_causal():
    w = _small([0, 0], [7, 12], hq=2, hkv=2, seed=5)
    kc, vc = _pool(w)
    got = _oracle_mq(w, kc, vc)
    for s in range(w.num_seqs):
        q0, q1 = int(w.query_start[s]), int(w.query_start[s + 1])
        np.testing.assert_allclose(got[q0:q1], _sdpa_reference(w, s, causal_flag=True),
                                   rtol=0, atol=1e-12)


def test_single_token_prompt_returns_its_value_exactly():
    w = _small([0], [1], hq=4, hkv=1, seed=7)
    kc, vc = _pool(w)
    got = _oracle_mq(w, kc, vc)
    v0 = _f64(w.value[0, 0])
    for h in range(w.num_q_heads):
        assert np.array_equal(got[0, h], v0)


def test_first_query_of_a_prompt_sees_only_its_own_token():
    """Row 0 of a prompt with no prior context attends to token 0 alone: out = v_0."""
    w = _small([0, 0], [5, 9], seed=11)
    kc, vc = _pool(w)
    got = _oracle_mq(w, kc, vc)
    G = w.num_q_heads // w.num_kv_heads
    for s in range(w.num_seqs):
        row = int(w.query_start[s])
        first = w.seq_tokens[s][0]
        for h in range(w.num_q_heads):
            assert np.array_equal(got[row, h], _f64(w.value[first, h // G]))


def test_last_query_row_equals_decode_over_the_whole_context():
    w = _small([3, 11], [4, 2], seed=13)
    kc, vc = _pool(w)
    got = _oracle_mq(w, kc, vc)
    for s in range(w.num_seqs):
        row = int(w.query_start[s + 1]) - 1
        # a one-sequence decode of that row over the sequence's full context
        dec = oracle.paged_decode_attention(
            np.ascontiguousarray(w.query[row:row + 1]), kc, vc,
            np.ascontiguousarray(w.block_tables[s:s + 1]), w.context_lens[s:s + 1],
            num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
            block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale,
            q_dtype=w.q_dtype, kv_dtype=w.kv_dtype)
        np.testing.assert_allclose(got[row], dec[0], rtol=0, atol=1e-13)


def test_more_queries_than_context_is_rejected():
    w = _small([0], [4])
    kc, vc = _pool(w)
    bad = w.context_lens.copy()
    bad[0] = 3
    with pytest.raises(ValueError):
        oracle.paged_prefill_attention(
            w.query, kc, vc, w.block_tables, bad, w.query_start, num_q_heads=w.num_q_heads,
            num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
            num_blocks=w.num_blocks, scale=w.scale, q_dtype="f32", kv_dtype="f32")


def test_multi_query_configs_generate_with_documented_shapes():
    w = inputs.make_multi_query_config(0)
    assert (w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim) == (5, 8, 2, 128)
    assert list(np.diff(w.query_start)) == [1, 64, 200, 130, 33]
    assert list(w.context_lens - np.diff(w.query_start)) == [0, 37, 300, 5, 129]
    assert w.flops == 4 * 128 * 8 * sum(p * n + n * (n + 1) // 2 for p, n in
                                        zip([0, 37, 300, 5, 129], [1, 64, 200, 130, 33]))
