"""Seeded synthetic inputs for the paged decode hot path.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests.  It holds none of the method's arithmetic: it draws random numbers,
hands out physical block ids from a free list (the host block manager of
"PagedAttention: Mathematical Foundations ..." §4 Allocation Lifecycle and §5
Parallel Sampling), and records which token row goes to which slot.  Writing
rows into the pool, copying blocks, gathering and attention are done by each
side itself (the CUDA library, or the oracle) from what is recorded here.

Every workload is described by:

* ``key`` / ``value``: distinct token vectors [T_vec, Hkv, d] in ``src_dtype``
  (numpy; bf16 as uint16 bit patterns),
* ``setup``: a list of operations that fill the pool before the first step:
  ``("reshape", vec_idx, slots)`` writes rows ``key[vec_idx]`` to ``slots``;
  ``("copy", pairs)`` copies physical blocks (copy-on-write at a fork),
* the step: ``step_pairs`` (copy-on-write pairs, possibly empty), then the new
  token of every sequence (``new_vec`` rows to ``new_slots``), then decode over
  ``context_lens`` tokens through ``block_tables``,
* ``seq_tokens[s]``: the vector index of every logical position of sequence s,
  used only by table-free brute-force checks.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np

DTYPE_BYTES = {"f32": 4, "f16": 2, "bf16": 2, "e4m3": 1}
# numpy container for each element type (raw bits for bf16 / e4m3)
NP_CONTAINER = {"f32": np.float32, "f16": np.float16, "bf16": np.uint16, "e4m3": np.uint8}
# byte pattern that poisons unused cache slots: NaN in every floating format
POISON_BYTE = {"f32": None, "f16": None, "bf16": None, "e4m3": 0x7F}


def poison_array(shape, dtype: str) -> np.ndarray:
    """Host cache buffer whose every element is a NaN of ``dtype``."""
    a = np.empty(shape, dtype=NP_CONTAINER[dtype])
    if dtype == "f32":
        a.fill(np.nan)
    elif dtype == "f16":
        a.fill(np.float16(np.nan))
    elif dtype == "bf16":
        a.fill(0x7FC0)
    else:
        a.fill(0x7F)
    return a


def draw_normal(rng: np.random.Generator, shape, dtype: str, chunk: int = 1 << 26) -> np.ndarray:
    """N(0,1) draws rounded (nearest-even) into ``dtype`` storage.

    The bulk draws come from a torch CPU generator seeded from ``rng`` (about
    twice numpy's normal throughput), so a workload is a function of its seed.
    """
    import torch
    n = int(np.prod(shape))
    gen = torch.Generator().manual_seed(int(rng.integers(0, 2 ** 62)))
    out = np.empty(n, dtype=NP_CONTAINER[dtype])
    for i in range(0, n, chunk):
        x = torch.randn(min(chunk, n - i), generator=gen, dtype=torch.float32)
        out[i:i + x.numel()] = to_storage(x, dtype)
    return out.reshape(shape)


def to_storage(x, dtype: str) -> np.ndarray:
    """Round fp32 values (numpy or torch) into the storage of a 32/16-bit float type."""
    import torch
    t = x if isinstance(x, torch.Tensor) else torch.from_numpy(np.ascontiguousarray(x, np.float32))
    t = t.to(torch.float32)
    if dtype == "f32":
        return t.numpy()
    if dtype == "f16":
        return t.to(torch.float16).numpy()
    if dtype == "bf16":
        return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    raise ValueError(f"no storage rounding for {dtype}")


# ------------------------------------------------------- block manager --

class BlockManager:
    """Host-side free list + reference counts ("...Mathematical Foundations" §4, §5).

    Physical ids come from a seeded random permutation of the pool, so tables
    are scattered like a long-running server's.  The first and last blocks are
    guard blocks and are never handed out.
    """

    def __init__(self, num_blocks: int, block_size: int, rng: np.random.Generator | None = None,
                 guards: bool = True):
        self.num_blocks = num_blocks
        self.block_size = block_size
        lo, hi = (1, num_blocks - 1) if guards else (0, num_blocks)
        ids = np.arange(lo, hi)
        if rng is not None:
            ids = rng.permutation(ids)
        self.free = [int(i) for i in ids]
        self.refcount = np.zeros(num_blocks, dtype=np.int64)

    def take(self) -> int:
        if not self.free:
            raise MemoryError("pool exhausted")
        b = self.free.pop(0)
        self.refcount[b] = 1
        return b

    def allocate(self, num_tokens: int) -> list[int]:
        """Prefill: ceil(num_tokens / B) fresh blocks."""
        return [self.take() for _ in range(-(-num_tokens // self.block_size))]

    def slot(self, table: list[int], pos: int) -> int:
        """Slot id of logical position ``pos`` = physical block * B + offset."""
        return table[pos // self.block_size] * self.block_size + pos % self.block_size

    def append_slot(self, table: list[int], num_filled: int) -> int:
        """Slot for the token at position ``num_filled``; grows the table on overflow."""
        if num_filled // self.block_size >= len(table):
            table.append(self.take())
        return self.slot(table, num_filled)

    def fork(self, table: list[int]) -> list[int]:
        """New sequence sharing every block of ``table`` (reference count + 1)."""
        for b in table:
            self.refcount[b] += 1
        return list(table)

    def copy_on_write(self, table: list[int], logical: int) -> tuple[int, int] | None:
        """Before writing into a shared block: give ``table`` a private copy.

        Returns the (src, dst) pair the copy kernel must execute, or None when
        the block is not shared.
        """
        src = table[logical]
        if self.refcount[src] <= 1:
            return None
        dst = self.take()
        self.refcount[src] -= 1
        table[logical] = dst
        return (src, dst)

    def free_table(self, table: list[int]) -> None:
        for b in table:
            self.refcount[b] -= 1
            if self.refcount[b] == 0:
                self.free.append(b)


# ------------------------------------------------------------ workloads --

@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_dtype: str
    src_dtype: str
    kv_dtype: str
    kv_scale: float
    scale: float
    query: np.ndarray
    key: np.ndarray
    value: np.ndarray
    setup: list
    step_pairs: np.ndarray
    new_vec: np.ndarray
    new_slots: np.ndarray
    block_tables: np.ndarray
    context_lens: np.ndarray
    seq_tokens: list = field(repr=False)
    group_of_seq: np.ndarray | None = None

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def cache_shape(self) -> tuple:
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    @property
    def kv_read_bytes(self) -> int:
        """Bytes of K and V the decode must read: sum_s ctx_s * Hkv * d * e * 2."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * DTYPE_BYTES[self.kv_dtype] * 2

    @property
    def unique_kv_bytes(self) -> int:
        """Bytes of distinct physical K/V rows behind the tables (shared prefixes once)."""
        B = self.block_size
        rows = []
        for s in range(self.num_seqs):
            pos = np.arange(int(self.context_lens[s]), dtype=np.int64)
            rows.append(self.block_tables[s, pos // B].astype(np.int64) * B + pos % B)
        n = np.unique(np.concatenate(rows)).size if rows else 0
        return int(n) * self.num_kv_heads * self.head_dim * DTYPE_BYTES[self.kv_dtype] * 2


def _pack_tables(tables: list[list[int]], pad: int = -1) -> np.ndarray:
    width = max(1, max(len(t) for t in tables))
    out = np.full((len(tables), width), pad, dtype=np.int32)
    for i, t in enumerate(tables):
        out[i, :len(t)] = t
    return out


def make_independent(name: str, rng: np.random.Generator, ctx: np.ndarray, *, num_q_heads: int,
                     num_kv_heads: int, head_dim: int, block_size: int, q_dtype: str,
                     kv_dtype: str, scale: float, src_dtype: str | None = None,
                     kv_scale: float = 1.0, num_blocks: int | None = None, slack: float = 0.10,
                     values: str = "normal") -> Workload:
    """Sequences with private blocks: prefill ctx_s - 1 tokens, the step adds one.

    ``values``: "normal" (N(0,1) q, K, V), "constant_v" (every V row equal),
    "zero_q" (q = 0).
    """
    ctx = np.asarray(ctx, dtype=np.int64)
    S = int(ctx.shape[0])
    src_dtype = src_dtype or (q_dtype if kv_dtype == "e4m3" else kv_dtype)
    nblk = [-(-int(c) // block_size) for c in ctx]
    if num_blocks is None:
        num_blocks = max(4, math.ceil(sum(nblk) * (1.0 + slack)) + 2)
    bm = BlockManager(num_blocks, block_size, rng)
    tables = [bm.allocate(int(c)) for c in ctx]
    T = int(ctx.sum())
    offsets = np.concatenate([[0], np.cumsum(ctx)])
    slots = np.empty(T, dtype=np.int64)
    for s in range(S):
        for p in range(int(ctx[s])):
            slots[offsets[s] + p] = bm.slot(tables[s], p)
    query = draw_normal(rng, (S, num_q_heads, head_dim), q_dtype)
    key = draw_normal(rng, (T, num_kv_heads, head_dim), src_dtype)
    if values == "constant_v":
        row = draw_normal(rng, (1, num_kv_heads, head_dim), src_dtype)
        value = np.ascontiguousarray(np.broadcast_to(row, (T, num_kv_heads, head_dim)))
    else:
        value = draw_normal(rng, (T, num_kv_heads, head_dim), src_dtype)
    if values == "zero_q":
        query = np.zeros_like(query)
    new_vec = np.array([offsets[s] + ctx[s] - 1 if ctx[s] > 0 else -1 for s in range(S)],
                       dtype=np.int64)
    pre = np.ones(T, dtype=bool)
    pre[new_vec[new_vec >= 0]] = False
    pre_idx = np.nonzero(pre)[0]
    new_slots = np.array([slots[v] if v >= 0 else -1 for v in new_vec], dtype=np.int64)
    return Workload(
        name=name, num_seqs=S, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks, q_dtype=q_dtype,
        src_dtype=src_dtype, kv_dtype=kv_dtype, kv_scale=kv_scale, scale=scale, query=query,
        key=key, value=value, setup=[("reshape", pre_idx, slots[pre_idx])],
        step_pairs=np.zeros((0, 2), dtype=np.int32), new_vec=np.maximum(new_vec, 0),
        new_slots=new_slots, block_tables=_pack_tables(tables),
        context_lens=ctx.astype(np.int32),
        seq_tokens=[np.arange(offsets[s], offsets[s + 1]) for s in range(S)])


def make_shared_prefix(name: str, rng: np.random.Generator, *, num_groups: int,
                       samples: int, prefix_lo: int, prefix_hi: int, tail_lo: int, tail_hi: int,
                       num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                       q_dtype: str, kv_dtype: str, kv_scale: float, scale: float,
                       slack: float = 0.10) -> Workload:
    """Parallel sampling: every group's prompt blocks are shared by ``samples`` sequences.

    Setup, in order ("...Mathematical Foundations" §5 Parallel Sampling):
    the prompt is written once; at the fork every sample but the last gets a
    copy of the partially filled last prompt block (copy-on-write); then each
    sample's own tail tokens are written.  The step copies each group's last
    full shared prompt block into a fresh block and repoints sample 0 at it
    (the data is unchanged), writes each sample's newest token, and decodes.
    """
    B = block_size
    S = num_groups * samples
    prefix = rng.integers(prefix_lo, prefix_hi + 1, size=num_groups)
    tails = rng.integers(tail_lo, tail_hi + 1, size=S)
    ctx = np.array([prefix[s // samples] + tails[s] for s in range(S)], dtype=np.int64)
    need = sum(-(-int(p) // B) for p in prefix) + \
        sum(-(-int(ctx[s]) // B) - int(prefix[s // samples]) // B for s in range(S)) + num_groups
    num_blocks = math.ceil(need * (1.0 + slack)) + 2
    bm = BlockManager(num_blocks, B, rng)
    src_dtype = q_dtype
    T = int(prefix.sum() + tails.sum())
    key = draw_normal(rng, (T, num_kv_heads, head_dim), src_dtype)
    value = draw_normal(rng, (T, num_kv_heads, head_dim), src_dtype)
    query = draw_normal(rng, (S, num_q_heads, head_dim), q_dtype)
    vec = 0
    tables, seq_tokens = [], []
    pre_idx, pre_slots, fork_pairs, tail_idx, tail_slots = [], [], [], [], []
    step_pairs, new_vec, new_slots = [], [], []
    group_of_seq = np.repeat(np.arange(num_groups), samples)
    for g in range(num_groups):
        P = int(prefix[g])
        ptab = bm.allocate(P)
        pvec = np.arange(vec, vec + P)
        vec += P
        pre_idx.append(pvec)
        pre_slots.append(np.array([bm.slot(ptab, p) for p in range(P)], dtype=np.int64))
        gtabs = [ptab] + [bm.fork(ptab) for _ in range(samples - 1)]
        for b in ptab:                      # allocate() set 1, each fork added 1
            assert bm.refcount[b] == samples
        for i in range(samples):
            s = g * samples + i
            tab = gtabs[i]
            if P % B and i < samples - 1:   # first write into the shared partial block
                fork_pairs.append(bm.copy_on_write(tab, P // B))
            n_tail = int(tails[s])
            tvec = np.arange(vec, vec + n_tail)
            vec += n_tail
            slots = [bm.append_slot(tab, P + k) for k in range(n_tail)]
            tail_idx.append(tvec[:-1])
            tail_slots.append(np.array(slots[:-1], dtype=np.int64))
            new_vec.append(int(tvec[-1]))
            new_slots.append(int(slots[-1]))
            tables.append(tab)
            seq_tokens.append(np.concatenate([pvec, tvec]))
        # step copy-on-write: the last full prompt block of the group -> fresh block,
        # repointed in sample 0's table
        last_full = P // B - 1
        assert last_full >= 0, "prompt shorter than one block"
        step_pairs.append(bm.copy_on_write(tables[g * samples], last_full))
    assert vec == T
    setup = [("reshape", np.concatenate(pre_idx), np.concatenate(pre_slots))]
    if fork_pairs:
        setup.append(("copy", np.array(fork_pairs, dtype=np.int32)))
    setup.append(("reshape", np.concatenate(tail_idx), np.concatenate(tail_slots)))
    # the step's copy must precede any read of the repointed table: run it once in setup too
    setup.append(("copy", np.array(step_pairs, dtype=np.int32)))
    return Workload(
        name=name, num_seqs=S, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=B, num_blocks=num_blocks, q_dtype=q_dtype,
        src_dtype=src_dtype, kv_dtype=kv_dtype, kv_scale=kv_scale, scale=scale, query=query,
        key=key, value=value, setup=setup, step_pairs=np.array(step_pairs, dtype=np.int32),
        new_vec=np.array(new_vec, dtype=np.int64), new_slots=np.array(new_slots, dtype=np.int64),
        block_tables=_pack_tables(tables), context_lens=ctx.astype(np.int32),
        seq_tokens=seq_tokens, group_of_seq=group_of_seq)


# The five workloads, in order: tiny MHA fp32; OPT-13B-shaped layer (fp16);
# GQA bf16 with lognormal lengths; long-context bf16 (split-KV); FP8 KV with a
# shared prefix.  ``num_seqs`` / ``ctx_cap`` shrink a workload for quick tests
# with the same recipe.
CONFIG_NAMES = [
    "tiny MHA decode: 4 seqs, 8 heads, d64, B16, ctx {1,17,100,256}, fp32",
    "OPT-13B-shaped layer decode: 64 seqs, 40 heads MHA, d128, fp16, B16, ctx U[512,2048]",
    "GQA decode: 256 seqs, 32q/8kv heads, d128, bf16, B16, ctx lognormal(1024, 1) in [1,8192]",
    "long-context split-KV: 8 seqs, 64q/8kv heads, d128, bf16, B32, ctx U[32768,131072]",
    "FP8 KV + shared prefix: 32 prompts x 4 samples, 32q/8kv, d128, e4m3 (scale 2^-5), "
    "prefix U[1024,8192], tails U[1,256]",
]


def make_config(cid: int, *, num_seqs: int | None = None, ctx_cap: int | None = None,
                seed: int | None = None) -> Workload:
    rng = np.random.default_rng(8700 + cid if seed is None else seed)
    name = CONFIG_NAMES[cid]
    if cid == 0:
        ctx = np.array([1, 17, 100, 256])
        if ctx_cap:
            ctx = np.minimum(ctx, ctx_cap)
        return make_independent(name, rng, ctx[:num_seqs], num_q_heads=8, num_kv_heads=8,
                                head_dim=64, block_size=16, q_dtype="f32", kv_dtype="f32",
                                scale=1.0 / 8.0, num_blocks=64)
    if cid == 1:
        S = num_seqs or 64
        ctx = rng.integers(512, 2048 + 1, size=64)[:S]
    elif cid == 2:
        S = num_seqs or 256
        ctx = np.clip(np.rint(rng.lognormal(math.log(1024), 1.0, size=256)), 1, 8192)[:S]
    elif cid == 3:
        S = num_seqs or 8
        ctx = rng.integers(32768, 131072 + 1, size=8)[:S]
    elif cid == 4:
        groups = max(1, (num_seqs or 128) // 4)
        lo, hi = (1024, 8192) if not ctx_cap else (min(1024, ctx_cap), ctx_cap)
        return make_shared_prefix(name, rng, num_groups=groups, samples=4, prefix_lo=lo,
                                  prefix_hi=hi, tail_lo=1, tail_hi=256, num_q_heads=32,
                                  num_kv_heads=8, head_dim=128, block_size=16, q_dtype="bf16",
                                  kv_dtype="e4m3", kv_scale=2.0 ** -5,
                                  scale=1.0 / math.sqrt(128))
    else:
        raise ValueError(cid)
    if ctx_cap:
        ctx = np.minimum(ctx, ctx_cap)
    ctx = ctx.astype(np.int64)
    spec = {1: (40, 40, 16, "f16"), 2: (32, 8, 16, "bf16"), 3: (64, 8, 32, "bf16")}[cid]
    Hq, Hkv, B, dt = spec
    return make_independent(name, rng, ctx, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=128,
                            block_size=B, q_dtype=dt, kv_dtype=dt,
                            scale=1.0 / math.sqrt(128))


# ----------------------------------------------------- multi-query inputs --

@dataclass
class MultiQueryWorkload:
    """Several query tokens per sequence over a paged cache (prefill / chunked prefill).

    Sequence s has prior[s] tokens cached before the step and n[s] new tokens;
    the step writes the new tokens' K/V (rows ``new_idx`` at ``slots[new_idx]``)
    and attends causally with their n[s] queries over ctx = prior + n tokens.
    """
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    q_dtype: str
    kv_dtype: str
    scale: float
    query: np.ndarray          # [total_q, Hq, d] storage
    key: np.ndarray            # [T, Hkv, d] storage: every cached token's key
    value: np.ndarray
    slots: np.ndarray          # [T] int64 slot of each row
    prior_idx: np.ndarray      # rows cached before the step
    new_idx: np.ndarray        # rows the step writes (the queries' own tokens)
    block_tables: np.ndarray   # int32 [S, max_blocks], -1 padded
    context_lens: np.ndarray   # int32 [S] = prior + n
    query_start: np.ndarray    # int32 [S + 1]
    seq_tokens: list           # per sequence: its rows in position order
    # draft-token trees: uint64 [total_q], bit j of row query_start[s] + i set when query
    # i of sequence s sees tree token j < i (its ancestors); None for causal attention
    tree: np.ndarray | None = None

    src_dtype = property(lambda self: self.kv_dtype)
    kv_scale = property(lambda self: 1.0)

    @property
    def total_q(self) -> int:
        return int(self.query_start[-1])

    @property
    def max_blocks(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def cache_shape(self) -> tuple:
        return (self.num_blocks, self.num_kv_heads, self.block_size, self.head_dim)

    @property
    def num_new(self) -> np.ndarray:
        return np.diff(self.query_start.astype(np.int64))

    @property
    def flops(self) -> int:
        """Attention FLOPs: 4 d Hq per (query, visible key) pair (Q K^T and P V)."""
        n = self.num_new
        prior = self.context_lens.astype(np.int64) - n
        if self.tree is None:
            pairs = int((n * prior + n * (n + 1) // 2).sum())
        else:
            # prior context + the token itself + its ancestors
            anc = int(sum(bin(int(x)).count("1") for x in self.tree))
            pairs = int((n * prior + n).sum()) + anc
        return 4 * self.head_dim * self.num_q_heads * pairs

    @property
    def kv_bytes(self) -> int:
        """K and V bytes of every cached token (each read at least once)."""
        return int(self.context_lens.astype(np.int64).sum()) * self.num_kv_heads * \
            self.head_dim * DTYPE_BYTES[self.kv_dtype] * 2


def make_multi_query(name: str, rng: np.random.Generator, prior, n, *, num_q_heads: int,
                     num_kv_heads: int, head_dim: int = 128, block_size: int = 16,
                     dtype: str = "bf16", scale: float | None = None,
                     slack: float = 0.10) -> MultiQueryWorkload:
    """Private blocks per sequence from a seeded permutation of the pool; q/K/V ~ N(0,1)."""
    prior = np.asarray(prior, dtype=np.int64)
    n = np.asarray(n, dtype=np.int64)
    S = int(prior.shape[0])
    ctx = prior + n
    nblk = [-(-int(c) // block_size) for c in ctx]
    num_blocks = max(4, math.ceil(sum(nblk) * (1.0 + slack)) + 2)
    bm = BlockManager(num_blocks, block_size, rng)
    tables = [bm.allocate(int(c)) for c in ctx]
    T = int(ctx.sum())
    offsets = np.concatenate([[0], np.cumsum(ctx)])
    slots = np.empty(T, dtype=np.int64)
    is_new = np.zeros(T, dtype=bool)
    for s in range(S):
        for p in range(int(ctx[s])):
            slots[offsets[s] + p] = bm.slot(tables[s], p)
        is_new[offsets[s] + prior[s]: offsets[s + 1]] = True
    query_start = np.concatenate([[0], np.cumsum(n)]).astype(np.int32)
    query = draw_normal(rng, (int(query_start[-1]), num_q_heads, head_dim), dtype)
    key = draw_normal(rng, (T, num_kv_heads, head_dim), dtype)
    value = draw_normal(rng, (T, num_kv_heads, head_dim), dtype)
    return MultiQueryWorkload(
        name=name, num_seqs=S, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
        head_dim=head_dim, block_size=block_size, num_blocks=num_blocks, q_dtype=dtype,
        kv_dtype=dtype, scale=scale if scale is not None else 1.0 / math.sqrt(head_dim),
        query=query, key=key, value=value, slots=slots,
        prior_idx=np.nonzero(~is_new)[0], new_idx=np.nonzero(is_new)[0],
        block_tables=_pack_tables(tables), context_lens=ctx.astype(np.int32),
        query_start=query_start,
        seq_tokens=[np.arange(offsets[s], offsets[s + 1]) for s in range(S)])


def tree_ancestors(parent) -> np.ndarray:
    """uint64 ancestor masks of a tree given by parent indices (parent[0] = -1 for the
    root, parent[i] < i otherwise): bit j of entry i set when j is an ancestor of i."""
    parent = np.asarray(parent, dtype=np.int64)
    n = parent.shape[0]
    if n > 64:
        raise ValueError("a tree of at most 64 tokens")
    anc = np.zeros(n, dtype=np.uint64)
    for i in range(1, n):
        p = int(parent[i])
        if not 0 <= p < i:
            raise ValueError("parents precede their children")
        anc[i] = anc[p] | np.uint64(1 << p)
    return anc


def random_tree_parents(rng: np.random.Generator, n: int, kind: str = "random") -> np.ndarray:
    """Parent indices of an n-token draft tree laid out parents first: "chain" (each
    token the child of the previous one), "star" (every token a child of the root) or
    "random" (each token the child of one of the 4 tokens before it, so that branches
    and depth both occur)."""
    parent = np.full(n, -1, dtype=np.int64)
    for i in range(1, n):
        if kind == "chain":
            parent[i] = i - 1
        elif kind == "star":
            parent[i] = 0
        else:
            parent[i] = int(rng.integers(max(0, i - 4), i))
    return parent


def make_tree_verify(name: str, rng: np.random.Generator, prior, n, *, kinds=None,
                     **kw) -> MultiQueryWorkload:
    """A multi-query workload whose queries are draft-token trees (n[s] <= 64 tokens each,
    the tree of kind kinds[s], "random" by default) over prior[s] cached tokens."""
    w = make_multi_query(name, rng, prior, n, **kw)
    trees = []
    for s in range(w.num_seqs):
        kind = kinds[s] if kinds is not None else "random"
        trees.append(tree_ancestors(random_tree_parents(rng, int(w.num_new[s]), kind)))
    w.tree = np.concatenate(trees) if trees else np.zeros(0, np.uint64)
    return w


MQ_CONFIG_NAMES = {
    0: "multi-query mix: 5 seqs, 8q/2kv heads, d128, bf16, B16, prior {0..300} + 1..200 queries",
    1: "chunked prefill: 16 seqs, 32q/8kv heads, d128, bf16, B16, prior U[0,8192] + 512 queries",
    2: "prefill MHA: 4 seqs, 16 heads, d128, fp16, B16, prompts U[1024,4096], no prior context",
    3: "draft-tree verification: 64 seqs, 32q/8kv heads, d128, bf16, B16, prior U[1024,8192] + trees of 64 tokens",
}


def make_multi_query_config(cid: int, *, seed: int | None = None) -> MultiQueryWorkload:
    """The seeded multi-query workloads (seed 8790 + id)."""
    rng = np.random.default_rng(8790 + cid if seed is None else seed)
    name = MQ_CONFIG_NAMES[cid]
    if cid == 0:
        return make_multi_query(name, rng, [0, 37, 300, 5, 129], [1, 64, 200, 130, 33],
                                num_q_heads=8, num_kv_heads=2)
    if cid == 1:
        prior = rng.integers(0, 8192 + 1, size=16)
        return make_multi_query(name, rng, prior, np.full(16, 512), num_q_heads=32,
                                num_kv_heads=8)
    if cid == 2:
        n = rng.integers(1024, 4096 + 1, size=4)
        return make_multi_query(name, rng, np.zeros(4, np.int64), n, num_q_heads=16,
                                num_kv_heads=16, dtype="f16")
    if cid == 3:
        prior = rng.integers(1024, 8192 + 1, size=64)
        return make_tree_verify(name, rng, prior, np.full(64, 64), num_q_heads=32, num_kv_heads=8)
    raise ValueError(f"no multi-query workload {cid}")


def seeded_rng(seed: int) -> np.random.Generator:
    return np.random.default_rng(seed)
