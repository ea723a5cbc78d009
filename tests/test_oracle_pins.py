"""Pins of the fp64 oracle to things other than itself (CPU only).

Each test checks the oracle against a value the pages print, a closed form, an
invariant, a special case with a known answer, or a library routine (numpy,
torch's float8/bfloat16 casts, torch's scaled_dot_product_attention).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import inputs
from tests.helpers import (ints, logical_kv_f64, oracle_caches, oracle_decode, read_golden,
                           to_f64)


# ------------------------------------------------------------ closed form --

def test_kv_bytes_per_token_opt13b():
    """"...Mathematical Foundations" §1: M_token = 4 L d_model = 819,200 B for OPT-13B."""
    g = read_golden("kv_footprint.txt")
    got = oracle.kv_bytes_per_token(int(g["num_layers"]), int(g["d_model"]), int(g["elem_bytes"]))
    assert got == int(g["bytes_per_token"]) == 819200
    # 4 L d_model for 2-byte elements, for any L and d_model
    for L, dm in [(1, 1), (12, 768), (80, 8192)]:
        assert oracle.kv_bytes_per_token(L, dm, 2) == 4 * L * dm


# ----------------------------------------------------------------- codecs --

def test_f16_decode_all_codes_match_numpy():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = codes.view(np.float16).astype(np.float64)
    got = np.array([oracle.f16_to_double(c) for c in codes])
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all()
    assert (np.signbit(got) == np.signbit(ref)).all()


def test_bf16_decode_all_codes_match_torch():
    codes = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(codes.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    got = np.array([oracle.bf16_to_double(c) for c in codes])
    assert ((got == ref) | (np.isnan(got) & np.isnan(ref))).all()


def test_e4m3_decode_all_codes_match_torch():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([oracle.e4m3_to_double(c) for c in codes])
    assert ((got == ref) | (np.isnan(got) & np.isnan(ref))).all()
    assert np.isnan(got[[0x7F, 0xFF]]).all() and np.isfinite(np.delete(got, [0x7F, 0xFF])).all()


def test_e4m3_decode_hand_points():
    with open(inputs.__file__.replace("paged_kv_cache_87_gb300/inputs.py",
                                      "tests/golden/e4m3_points.txt")) as f:
        rows = [ln.split() for ln in f if ln.strip() and not ln.startswith("#")]
    assert len(rows) >= 16
    for code, val in rows:
        got = oracle.e4m3_to_double(int(code, 16))
        if val == "nan":
            assert math.isnan(got)
        else:
            assert got == float(val) and math.copysign(1, got) == math.copysign(1, float(val))


def _e4m3_brute(x: float) -> int:
    """Nearest finite E4M3 value by exhaustive search; ties to the even code; saturating."""
    vals = [(c, oracle.e4m3_to_double(c)) for c in range(0x7F)]  # +0 .. 448
    a = abs(x)
    sign = 0x80 if math.copysign(1.0, x) < 0 else 0
    if a >= 448:
        return sign | 0x7E
    best = min(vals, key=lambda cv: (abs(cv[1] - a), cv[0] & 1))
    return sign | best[0]


def test_e4m3_encode_roundtrip_all_codes():
    for c in range(256):
        if c in (0x7F, 0xFF):
            assert oracle.e4m3_from_float(float("nan")) == 0x7F
            continue
        assert oracle.e4m3_from_float(oracle.e4m3_to_double(c)) == c


def test_e4m3_encode_midpoints_and_neighbours():
    """RNE at every midpoint between adjacent codes, and one fp32 ulp either side."""
    pos = [oracle.e4m3_to_double(c) for c in range(0x7F)]
    for lo_c in range(0x7E):
        lo, hi = pos[lo_c], pos[lo_c + 1]
        mid = np.float32((lo + hi) / 2)                # exact in fp32
        assert float(mid) == (lo + hi) / 2
        even = lo_c if lo_c % 2 == 0 else lo_c + 1
        for sgn in (1.0, -1.0):
            s = 0x80 if sgn < 0 else 0
            assert oracle.e4m3_from_float(sgn * mid) == s | even
            below = np.nextafter(mid, np.float32(0))
            above = np.nextafter(mid, np.float32(np.inf))
            assert oracle.e4m3_from_float(sgn * below) == s | lo_c
            assert oracle.e4m3_from_float(sgn * above) == s | (lo_c + 1)


def test_e4m3_encode_matches_torch_and_brute_force():
    rng = np.random.default_rng(1)
    x = np.concatenate([rng.standard_normal(4000) * s for s in (2.0 ** -8, 0.1, 1, 30, 150)])
    x = np.concatenate([x, [0.0, -0.0, 2.0 ** -10, 3 * 2.0 ** -10, 447.9, 448, 463.9, 464, 465,
                            1e6, -1e6, np.inf, -np.inf]]).astype(np.float32)
    got = np.array([oracle.e4m3_from_float(v) for v in x], dtype=np.uint8)
    # torch's cast is round-to-nearest-even but does not saturate (NaN above 464)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    inrange = np.abs(x) < 464
    assert (got[inrange] == ref[inrange]).all()
    big = ~inrange
    assert (got[big] == np.where(x[big] < 0, 0xFE, 0x7E)).all()
    for v, g in zip(x[::37], got[::37]):
        assert g == _e4m3_brute(float(v))


# ------------------------------------------------------------ fixtures --

def test_block_table_worked_example_slot():
    """§4 example: token 9 of the 10-token sequence lands in slot 19*4+1 = 77."""
    g = read_golden("block_table_example.txt")
    B = int(g["block_size"])
    bm = inputs.BlockManager(32, B, rng=None, guards=False)
    bm.free = ints(g["table"]) + [b for b in bm.free if b not in ints(g["table"])]
    table = bm.allocate(int(g["num_tokens"]))
    assert table == ints(g["table"])
    assert bm.slot(table, 9) == int(g["slot_of_token_9"])
    n = int(g["num_tokens"])
    filled = [min(B, n - j * B) for j in range(len(table))]
    assert filled == ints(g["filled"])
    assert len(table) * B - n == int(g["free_slots_in_last_block"])
    # the oracle scatter puts token 9 in physical block 19, row 1 of the layout
    key = np.arange(1 * 1 * 2, dtype=np.float32).reshape(1, 1, 2) + 5
    kc = inputs.poison_array((32, 1, B, 2), "f32")
    vc = inputs.poison_array((32, 1, B, 2), "f32")
    oracle.reshape_and_cache(key, key.copy(), kc, vc, np.array([77]), num_kv_heads=1, head_dim=2,
                             block_size=B, num_blocks=32, src_dtype="f32", kv_dtype="f32")
    assert (kc[19, 0, 1] == [5, 6]).all()
    assert np.isnan(np.delete(kc.reshape(-1, 2), 19 * B + 1, axis=0)).all()


def test_cow_worked_example():
    """§5 Parallel Sampling: prompt [7, 1] ref 2 -> sample 1 gets a copy in 3."""
    g = read_golden("cow_example.txt")
    bm = inputs.BlockManager(16, int(g["block_size"]), rng=None, guards=False)
    bm.free = [7, 1, 3] + [b for b in bm.free if b not in (7, 1, 3)]
    s1 = bm.allocate(int(g["prompt_tokens"]))
    assert s1 == ints(g["prompt_table"])
    s2 = bm.fork(s1)
    assert [bm.refcount[b] for b in s1] == ints(g["refcount_after_fork"])
    pair = bm.copy_on_write(s1, 1)
    assert list(pair) == ints(g["cow_pair"])
    assert s1 == ints(g["sample1_table"]) and s2 == ints(g["sample2_table"])
    for b in (7, 1, 3):
        assert bm.refcount[b] == int(g[f"refcount_{b}"])
    assert bm.copy_on_write(s2, 1) is None        # no longer shared


def test_logical_to_physical_example():
    g = read_golden("logical_physical_example.txt")
    B = int(g["block_size"])
    bm = inputs.BlockManager(16, B, rng=None, guards=False)
    bm.free = ints(g["table"]) + [b for b in bm.free if b not in ints(g["table"])]
    assert bm.allocate(int(g["num_tokens"])) == ints(g["table"])


@pytest.mark.parametrize("cid", [0, 1, 2, 3, 4])
def test_waste_confined_to_last_block(cid):
    """§4: internal fragmentation only in the last block: 0 <= ceil(n/B) B - n <= B - 1."""
    w = inputs.make_config(cid, num_seqs=16 if cid in (1, 2, 4) else None,
                           ctx_cap=600 if cid in (3, 4) else None)
    B = w.block_size
    used = (w.block_tables >= 0).sum(1)
    waste = used * B - w.context_lens
    assert (waste >= 0).all() and (waste <= B - 1).all()
    assert ((w.block_tables >= 0) & (w.block_tables < w.num_blocks)).sum() == used.sum()


def test_cache_layout_tiny_golden():
    g = read_golden("cache_layout_tiny.txt")
    NB, H, B, d = (int(g[k]) for k in ("num_blocks", "num_kv_heads", "block_size", "head_dim"))
    key = np.array([[[100 * t + 10 * h + i for i in range(d)] for h in range(H)]
                    for t in range(3)], dtype=np.float32)
    kc = np.full((NB, H, B, d), -1, np.float32)
    vc = np.full((NB, H, B, d), -1, np.float32)
    oracle.reshape_and_cache(key, key.copy(), kc, vc, np.array(ints(g["slots"])), num_kv_heads=H,
                             head_dim=d, block_size=B, num_blocks=NB, src_dtype="f32",
                             kv_dtype="f32")
    assert kc.reshape(-1).tolist() == [float(x) for x in g["k_cache"].split()]
    assert (vc == kc).all()


def test_reshape_skips_negative_slots_and_rejects_out_of_pool():
    key = np.ones((2, 1, 4), np.float32)
    kc = np.zeros((2, 1, 2, 4), np.float32)
    vc = np.zeros_like(kc)
    oracle.reshape_and_cache(key, key, kc, vc, np.array([-1, 3]), num_kv_heads=1, head_dim=4,
                             block_size=2, num_blocks=2, src_dtype="f32", kv_dtype="f32")
    assert kc.sum() == 4 and (kc[1, 0, 1] == 1).all()
    with pytest.raises(ValueError):
        oracle.reshape_and_cache(key, key, kc, vc, np.array([0, 4]), num_kv_heads=1, head_dim=4,
                                 block_size=2, num_blocks=2, src_dtype="f32", kv_dtype="f32")


def test_reshape_e4m3_matches_torch_cast():
    """FP8 write: e4m3(x / kv_scale), x / kv_scale in fp32 (torch cast, in range)."""
    rng = np.random.default_rng(3)
    T, H, d, B, NB = 24, 2, 16, 8, 5
    x = rng.standard_normal((T, H, d)).astype(np.float32)
    xb = inputs.to_storage(x, "bf16").reshape(T, H, d)
    slots = rng.permutation(NB * B)[:T]
    kc = inputs.poison_array((NB, H, B, d), "e4m3")
    vc = inputs.poison_array((NB, H, B, d), "e4m3")
    scale = np.float32(0.05)   # not a power of two: exercises the division
    oracle.reshape_and_cache(xb, xb, kc, vc, slots, num_kv_heads=H, head_dim=d, block_size=B,
                             num_blocks=NB, src_dtype="bf16", kv_dtype="e4m3", kv_scale=scale)
    xf = torch.from_numpy(xb.view(np.int16)).view(torch.bfloat16).float()
    q = (xf / torch.tensor(scale)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for t in range(T):
        blk, off = divmod(int(slots[t]), B)
        assert (kc[blk, :, off, :] == q[t]).all()


def test_copy_blocks_moves_only_dst_blocks():
    rng = np.random.default_rng(4)
    NB, H, B, d = 9, 2, 4, 8
    kc = rng.integers(0, 255, (NB, H, B, d), dtype=np.uint8)
    vc = rng.integers(0, 255, (NB, H, B, d), dtype=np.uint8)
    k0, v0 = kc.copy(), vc.copy()
    pairs = np.array([[1, 5], [7, 2], [1, 8]], np.int32)
    oracle.copy_blocks(kc, vc, pairs, num_kv_heads=H, head_dim=d, block_size=B, num_blocks=NB,
                       kv_dtype="e4m3")
    for s, t in pairs:
        assert (kc[t] == k0[s]).all() and (vc[t] == v0[s]).all()
    untouched = [b for b in range(NB) if b not in pairs[:, 1]]
    assert (kc[untouched] == k0[untouched]).all() and (vc[untouched] == v0[untouched]).all()
    for bad in ([[0, 9]], [[1, 2], [3, 2]], [[1, 2], [2, 3]], [[-1, 0]]):
        with pytest.raises(ValueError):
            oracle.copy_blocks(kc, vc, np.array(bad, np.int32), num_kv_heads=H, head_dim=d,
                               block_size=B, num_blocks=NB, kv_dtype="e4m3")


# -------------------------------------------------------- attention core --

def _tiny(seed, ctx, *, d=64, B=16, Hq=4, Hkv=4, dt="f32", kv=None, values="normal"):
    rng = np.random.default_rng(seed)
    kv = kv or dt
    return inputs.make_independent("tiny", rng, np.array(ctx), num_q_heads=Hq, num_kv_heads=Hkv,
                                   head_dim=d, block_size=B, q_dtype=dt, kv_dtype=kv,
                                   scale=1.0 / math.sqrt(d),
                                   kv_scale=2.0 ** -5 if kv == "e4m3" else 1.0, values=values)


def _sdpa_reference(w, kv_deq=None):
    """torch scaled_dot_product_attention (fp64, CPU) on the table-free logical K/V."""
    G = w.num_q_heads // w.num_kv_heads
    q = to_f64(w.query, w.q_dtype)
    outs = []
    for s in range(w.num_seqs):
        if w.context_lens[s] == 0:
            outs.append(np.zeros((w.num_q_heads, w.head_dim)))
            continue
        K, V = logical_kv_f64(w, s) if kv_deq is None else kv_deq(s)
        Kt = torch.from_numpy(K).transpose(0, 1).repeat_interleave(G, 0)   # [Hq, T, d]
        Vt = torch.from_numpy(V).transpose(0, 1).repeat_interleave(G, 0)
        qs = torch.from_numpy(q[s]).unsqueeze(1)                           # [Hq, 1, d]
        o = torch.nn.functional.scaled_dot_product_attention(qs, Kt, Vt, scale=w.scale)
        outs.append(o[:, 0].numpy())
    return np.stack(outs)


@pytest.mark.parametrize("case", [
    dict(ctx=[1, 15, 16, 17, 40], d=64, B=16, Hq=4, Hkv=4, dt="f32"),
    dict(ctx=[7, 8, 9, 33], d=128, B=8, Hq=8, Hkv=2, dt="f16"),
    dict(ctx=[31, 32, 33, 100], d=128, B=32, Hq=8, Hkv=1, dt="bf16"),
    dict(ctx=[3, 64, 65], d=64, B=16, Hq=6, Hkv=3, dt="bf16"),
])
def test_decode_matches_sdpa_on_logical_kv(case):
    w = _tiny(11, **case)
    kc, vc = oracle_caches(w)
    got = oracle_decode(w, kc, vc)
    ref = _sdpa_reference(w)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-12)


def test_decode_fp8_matches_sdpa_on_dequantised_kv():
    w = _tiny(12, [5, 16, 47], d=128, B=16, Hq=8, Hkv=2, dt="bf16", kv="e4m3")
    kc, vc = oracle_caches(w)
    scale = np.float32(w.kv_scale)

    def deq(s):
        out = []
        for a in (w.key, w.value):
            xf = torch.from_numpy(np.ascontiguousarray(a[w.seq_tokens[s]]).view(np.int16))
            xf = xf.view(torch.bfloat16).float() / torch.tensor(scale)
            out.append(xf.to(torch.float8_e4m3fn).to(torch.float64).numpy() * float(scale))
        return out

    np.testing.assert_allclose(oracle_decode(w, kc, vc), _sdpa_reference(w, deq),
                               rtol=1e-12, atol=1e-12)


def test_fp8_path_equals_f32_path_on_dequantised_values():
    """Dequantise-on-load: an e4m3 pool with scale s == an f32 pool holding code*s."""
    w = _tiny(13, [9, 40], d=64, B=8, Hq=4, Hkv=2, dt="f32", kv="e4m3")
    kc, vc = oracle_caches(w)
    kf = (to_f64(kc, "e4m3") * w.kv_scale).astype(np.float32)
    vf = (to_f64(vc, "e4m3") * w.kv_scale).astype(np.float32)
    a = oracle_decode(w, kc, vc)
    b = oracle.paged_decode_attention(w.query, kf, vf, w.block_tables, w.context_lens,
                                      num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=8,
                                      num_blocks=w.num_blocks, scale=w.scale, q_dtype="f32",
                                      kv_dtype="f32")
    assert (a == b).all()


def test_context_len_one_returns_v1_exactly():
    w = _tiny(14, [1, 1, 1], d=64, B=16, Hq=4, Hkv=4, dt="f32")
    kc, vc = oracle_caches(w)
    got = oracle_decode(w, kc, vc)
    for s in range(3):
        _, V = logical_kv_f64(w, s)
        assert (got[s] == V[0]).all()


def test_constant_v_returns_the_constant():
    w = _tiny(15, [1, 5, 16, 77], d=64, B=16, Hq=4, Hkv=2, dt="f32", values="constant_v")
    kc, vc = oracle_caches(w)
    got = oracle_decode(w, kc, vc)
    v = to_f64(w.value[0], "f32")                     # [Hkv, d]
    np.testing.assert_allclose(got, np.repeat(v, 2, axis=0)[None].repeat(4, 0), rtol=1e-13,
                               atol=1e-14)


def test_zero_query_gives_mean_of_values():
    w = _tiny(16, [3, 20, 50], d=64, B=8, Hq=2, Hkv=2, dt="f16", values="zero_q")
    kc, vc = oracle_caches(w)
    got = oracle_decode(w, kc, vc)
    for s in range(3):
        _, V = logical_kv_f64(w, s)
        np.testing.assert_allclose(got[s], V.mean(0), rtol=1e-12, atol=1e-13)


def test_context_len_zero_gives_zeros():
    w = _tiny(17, [0, 5], d=64, B=16, Hq=2, Hkv=2)
    kc, vc = oracle_caches(w)
    got = oracle_decode(w, kc, vc)
    assert (got[0] == 0).all() and np.isfinite(got[1]).all() and np.abs(got[1]).sum() > 0


def _online_pseudocode(w, kc, vc, s, h):
    """The decode loop of "...Mathematical Foundations" §7, in plain Python fp64:
    per block, running max / rescale / running sum / rescaled accumulator."""
    G = w.num_q_heads // w.num_kv_heads
    g, B = h // G, w.block_size
    q = to_f64(w.query[s, h], w.q_dtype)
    acc = np.zeros(w.head_dim)
    run_max, run_sum = -math.inf, 0.0
    n = int(w.context_lens[s])
    for j in range(-(-n // B)):
        blk = int(w.block_tables[s, j])
        rows = min(B, n - j * B)                        # the last block may be partial
        pk = to_f64(kc[blk, g, :rows], w.kv_dtype)
        pv = to_f64(vc[blk, g, :rows], w.kv_dtype)
        scores = [w.scale * float(np.dot(q, pk[r])) for r in range(rows)]
        new_max = max(run_max, max(scores))
        rescale = math.exp(run_max - new_max)
        ex = [math.exp(x - new_max) for x in scores]
        run_sum = run_sum * rescale + sum(ex)
        acc = acc * rescale + sum(e * pv[r] for r, e in enumerate(ex))
        run_max = new_max
    return acc / run_sum


def test_online_pseudocode_equals_two_pass_oracle():
    w = _tiny(18, [1, 16, 23, 70], d=64, B=16, Hq=4, Hkv=2, dt="bf16")
    kc, vc = oracle_caches(w)
    got = oracle_decode(w, kc, vc)
    for s in range(w.num_seqs):
        for h in range(w.num_q_heads):
            np.testing.assert_allclose(got[s, h], _online_pseudocode(w, kc, vc, s, h),
                                       rtol=1e-12, atol=1e-13)


def test_split_merge_equals_unsplit():
    w = _tiny(19, [200, 37], d=64, B=8, Hq=4, Hkv=2, dt="f32")
    kc, vc = oracle_caches(w)
    full = oracle_decode(w, kc, vc)
    rng = np.random.default_rng(0)
    common = dict(num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=8,
                  num_blocks=w.num_blocks, scale=w.scale, q_dtype="f32", kv_dtype="f32")
    for s in range(2):
        n = int(w.context_lens[s])
        for h in range(4):
            for nsplit in (1, 2, 5):
                cuts = np.sort(np.concatenate([[0, n], rng.integers(0, n + 1, nsplit - 1)]))
                parts = [oracle.attention_partial(w.query, kc, vc, w.block_tables, seq=s,
                                                  q_head=h, t0=int(a), t1=int(b), **common)
                         for a, b in zip(cuts[:-1], cuts[1:])]
                ms, ls, accs = zip(*parts)
                merged = oracle.merge_partials(ms, ls, np.stack(accs))
                np.testing.assert_allclose(merged, full[s, h], rtol=1e-12, atol=1e-13)
    # a single partial normalises to acc / l; all-empty merges to zeros
    assert (oracle.merge_partials([-math.inf], [0.0], np.zeros((1, 4))) == 0).all()


def test_physical_block_permutation_is_bit_invariant():
    """§3: K_j, V_j are fetched independently per block, so physical placement is free."""
    w = _tiny(20, [5, 33, 64, 90], d=64, B=16, Hq=4, Hkv=2, dt="f16")
    kc, vc = oracle_caches(w)
    base = oracle_decode(w, kc, vc)
    perm = np.random.default_rng(5).permutation(w.num_blocks)
    kp, vp = np.empty_like(kc), np.empty_like(vc)
    kp[perm], vp[perm] = kc, vc
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    got = oracle_decode(w, kp, vp, block_tables=tables.astype(np.int32))
    assert (got.view(np.uint64) == base.view(np.uint64)).all()


def test_gqa_equals_mha_with_repeated_kv_heads():
    w = _tiny(21, [12, 50], d=64, B=16, Hq=8, Hkv=2, dt="f32")
    kc, vc = oracle_caches(w)
    gqa = oracle_decode(w, kc, vc)
    kr, vr = np.repeat(kc, 4, axis=1), np.repeat(vc, 4, axis=1)
    mha = oracle.paged_decode_attention(w.query, np.ascontiguousarray(kr), np.ascontiguousarray(vr),
                                        w.block_tables, w.context_lens, num_q_heads=8,
                                        num_kv_heads=8, head_dim=64, block_size=16,
                                        num_blocks=w.num_blocks, scale=w.scale, q_dtype="f32",
                                        kv_dtype="f32")
    assert (gqa == mha).all()


def test_poison_in_unused_slots_is_never_read():
    w = _tiny(22, [3, 17, 31], d=64, B=16, Hq=2, Hkv=2, dt="bf16")
    kc, vc = oracle_caches(w, poison=True)
    kz, vz = oracle_caches(w, poison=False)
    a, b = oracle_decode(w, kc, vc), oracle_decode(w, kz, vz)
    assert np.isfinite(a).all() and (a == b).all()


def test_shared_prefix_step_copy_keeps_outputs_bit_identical():
    """The step's copy-on-write repoint moves no data: outputs equal the unshared tables."""
    w = inputs.make_config(4, num_seqs=8, ctx_cap=100)
    kc, vc = oracle_caches(w)
    base = oracle_decode(w, kc, vc)
    tables = w.block_tables.copy()
    for src, dst in w.step_pairs:
        tables[tables == dst] = src
    got = oracle_decode(w, kc, vc, block_tables=tables)
    assert (got == base).all()


def test_full_size_configs_generate_with_documented_shapes():
    """Configs at full size: sizes match the workload recipe (no oracle run)."""
    w = inputs.make_config(0)
    assert w.kv_read_bytes == 1531904 and w.num_blocks == 64
    assert (w.block_tables >= 0).sum() == 26
