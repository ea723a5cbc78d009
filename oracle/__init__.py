"""Plain fp64 CPU oracle for the paged-KV-cache hot path (ctypes wrapper).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` import this package; the product path never does.
It shares no code with the CUDA library.  The arithmetic lives in
``oracle.c`` (plain C, fp64, one loop per step of the definitions in
"PagedAttention: Mathematical Foundations ..." §3/§4/§7 and "Pytorch
implementation of paper ..." §2); this file only builds that C file and
marshals numpy arrays into it.

Element-type codes: F32=0, F16=1, BF16=2, E4M3=3.  Arrays are passed as numpy
arrays whose raw bytes hold the elements (bf16 and e4m3 as uint16 / uint8).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

F32, F16, BF16, E4M3 = 0, 1, 2, 3
DTYPE_CODES = {"f32": F32, "f16": F16, "bf16": BF16, "e4m3": E4M3}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


_CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           "-fno-fast-math"]


def _digest() -> str:
    """SHA-256 of oracle.c, the gcc flags and `gcc --version`: the build is redone
    whenever any of them changes."""
    import hashlib
    h = hashlib.sha256()
    with open(_SRC, "rb") as f:
        h.update(f.read())
    h.update(("\x1f".join(_CFLAGS)).encode())
    h.update(subprocess.run(["gcc", "--version"], capture_output=True, text=True).stdout.encode())
    return h.hexdigest()


def build(force: bool = False) -> str:
    """Compile oracle.c with gcc (IEEE arithmetic: no fast-math, no FMA contraction)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    stamp = _LIB_PATH + ".sha256"
    want = _digest()
    if not force and os.path.exists(_LIB_PATH) and os.path.exists(stamp):
        with open(stamp) as f:
            if f.read().strip() == want:
                return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *_CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    with open(stamp + f".tmp{os.getpid()}", "w") as f:
        f.write(want + "\n")
    os.replace(stamp + f".tmp{os.getpid()}", stamp)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32, f64 = ctypes.c_int, ctypes.c_int64, ctypes.c_float, ctypes.c_double
        lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_f16_to_double.restype = f64
        lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
        lib.oracle_bf16_to_double.restype = f64
        lib.oracle_e4m3_to_double.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_to_double.restype = f64
        lib.oracle_e4m3_from_float.argtypes = [f32]
        lib.oracle_e4m3_from_float.restype = ctypes.c_uint8
        lib.oracle_kv_bytes_per_token.argtypes = [i64, i64, i64]
        lib.oracle_kv_bytes_per_token.restype = i64
        lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32,
                                                 i32, f32]
        lib.oracle_reshape_and_cache.restype = i32
        lib.oracle_copy_blocks.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32]
        lib.oracle_copy_blocks.restype = i32
        lib.oracle_paged_decode_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32,
                                                      i32, f64, i32, i32, f64, P, i32, P, i32]
        lib.oracle_paged_decode_attention.restype = i32
        lib.oracle_attention_partial.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, i32, f64,
                                                 i32, i32, f64, i32, i32, i32, i32, P, P, P]
        lib.oracle_attention_partial.restype = i32
        lib.oracle_merge_partials.argtypes = [i32, P, P, P, i32, P]
        lib.oracle_merge_partials.restype = None
        lib.oracle_paged_prefill_attention.argtypes = [P, P, P, P, P, P, i32, i32, i32, i32,
                                                       i32, i32, i32, f64, i32, i32, f64, P,
                                                       i32, P, i32]
        lib.oracle_paged_prefill_attention.restype = i32
        lib.oracle_paged_tree_attention.argtypes = [P, P, P, P, P, P, P, i32, i32, i32, i32,
                                                    i32, i32, i32, f64, i32, i32, f64, P,
                                                    i32, P, i32]
        lib.oracle_paged_tree_attention.restype = i32
        lib.oracle_max_threads.argtypes = []
        lib.oracle_max_threads.restype = i32
        _lib = lib
        return lib


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return ctypes.c_void_p(a.ctypes.data)


def _code(t) -> int:
    return DTYPE_CODES[t] if isinstance(t, str) else int(t)


# ----------------------------------------------------------------- codecs --

def f16_to_double(bits: int) -> float:
    return _load().oracle_f16_to_double(int(bits))


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(int(bits))


def e4m3_to_double(code: int) -> float:
    return _load().oracle_e4m3_to_double(int(code))


def e4m3_from_float(x: float) -> int:
    return int(_load().oracle_e4m3_from_float(float(np.float32(x))))


def kv_bytes_per_token(num_layers: int, d_model: int, elem_size: int) -> int:
    return int(_load().oracle_kv_bytes_per_token(num_layers, d_model, elem_size))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


# ------------------------------------------------------------ cache ops --

def reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, *, num_kv_heads, head_dim,
                      block_size, num_blocks, src_dtype, kv_dtype, kv_scale=1.0) -> None:
    """In-place scatter of key/value [T, Hkv, d] into the host caches (numpy)."""
    slot_mapping = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    rc = _load().oracle_reshape_and_cache(
        _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache), _ptr(slot_mapping),
        int(slot_mapping.shape[0]), num_kv_heads, head_dim, block_size, num_blocks,
        _code(src_dtype), _code(kv_dtype), float(kv_scale))
    if rc != 0:
        raise ValueError("oracle reshape_and_cache: bad argument or slot outside the pool")


def copy_blocks(k_cache, v_cache, pairs, *, num_kv_heads, head_dim, block_size, num_blocks,
                kv_dtype) -> None:
    pairs = np.ascontiguousarray(pairs, dtype=np.int32).reshape(-1, 2)
    rc = _load().oracle_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(pairs),
                                    int(pairs.shape[0]), num_kv_heads, head_dim, block_size,
                                    num_blocks, _code(kv_dtype))
    if rc != 0:
        raise ValueError("oracle copy_blocks: id out of range, repeated dst, or dst is a src")


# ------------------------------------------------------ decode attention --

def paged_decode_attention(query, k_cache, v_cache, block_tables, context_lens, *, num_q_heads,
                           num_kv_heads, head_dim, block_size, num_blocks, scale, q_dtype,
                           kv_dtype, kv_scale=1.0, sel=None, nthreads=1) -> np.ndarray:
    """fp64 outputs for the (seq, q head) pairs in ``sel`` (all pairs if None).

    Returns an array [len(sel), head_dim] (or [S, Hq, d] when ``sel`` is None).
    """
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    S = context_lens.shape[0]
    full = sel is None
    if full:
        sel = np.stack(np.meshgrid(np.arange(S), np.arange(num_q_heads), indexing="ij"),
                       -1).reshape(-1, 2)
    sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
    out = np.zeros((sel.shape[0], head_dim), dtype=np.float64)
    rc = _load().oracle_paged_decode_attention(
        _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
        int(block_tables.shape[1]), float(scale), _code(q_dtype), _code(kv_dtype),
        float(kv_scale), _ptr(sel), int(sel.shape[0]), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle paged_decode_attention: bad argument or block id out of range")
    return out.reshape(S, num_q_heads, head_dim) if full else out


def attention_partial(query, k_cache, v_cache, block_tables, *, num_q_heads, num_kv_heads,
                      head_dim, block_size, num_blocks, scale, q_dtype, kv_dtype, kv_scale=1.0,
                      seq, q_head, t0, t1):
    """(m, l, acc) of one (seq, q head) over logical tokens [t0, t1)."""
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    m = np.zeros(1, np.float64)
    l = np.zeros(1, np.float64)
    acc = np.zeros(head_dim, np.float64)
    rc = _load().oracle_attention_partial(
        _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), num_q_heads,
        num_kv_heads, head_dim, block_size, num_blocks, int(block_tables.shape[1]),
        float(scale), _code(q_dtype), _code(kv_dtype), float(kv_scale), seq, q_head, t0, t1,
        _ptr(m), _ptr(l), _ptr(acc))
    if rc != 0:
        raise ValueError("oracle attention_partial: block id out of range")
    return float(m[0]), float(l[0]), acc


def paged_prefill_attention(query, k_cache, v_cache, block_tables, context_lens, query_start,
                            *, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                            scale, q_dtype, kv_dtype, kv_scale=1.0, sel=None,
                            nthreads=1) -> np.ndarray:
    """fp64 causal multi-query outputs for the (query row, q head) pairs in ``sel``.

    Query row r of sequence s (query_start[s] <= r < query_start[s+1]) sits at
    position context_lens[s] - n_s + (r - query_start[s]) and attends to every
    token up to and including it.  Returns [len(sel), head_dim], or
    [total_q, Hq, d] when ``sel`` is None.
    """
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    query_start = np.ascontiguousarray(query_start, dtype=np.int32)
    S = context_lens.shape[0]
    total_q = int(query_start[-1])
    full = sel is None
    if full:
        sel = np.stack(np.meshgrid(np.arange(total_q), np.arange(num_q_heads), indexing="ij"),
                       -1).reshape(-1, 2)
    sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
    out = np.zeros((sel.shape[0], head_dim), dtype=np.float64)
    rc = _load().oracle_paged_prefill_attention(
        _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start), S, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
        int(block_tables.shape[1]), float(scale), _code(q_dtype), _code(kv_dtype),
        float(kv_scale), _ptr(sel), int(sel.shape[0]), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle paged_prefill_attention: bad argument, more queries than "
                         "context, or block id out of range")
    return out.reshape(total_q, num_q_heads, head_dim) if full else out


def paged_tree_attention(query, k_cache, v_cache, block_tables, context_lens, query_start, tree,
                         *, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                         scale, q_dtype, kv_dtype, kv_scale=1.0, sel=None,
                         nthreads=1) -> np.ndarray:
    """fp64 outputs of the verification of draft-token trees for the (query row, q head)
    pairs in ``sel``.

    The last n_s <= 64 tokens of sequence s are its tree, each after its ancestors;
    query i sees the prior context, itself, and each earlier tree token j whose bit j
    is set in tree[query_start[s] + i] (uint64).  Returns [len(sel), head_dim], or
    [total_q, Hq, d] when ``sel`` is None.
    """
    block_tables = np.ascontiguousarray(block_tables, dtype=np.int32)
    context_lens = np.ascontiguousarray(context_lens, dtype=np.int32)
    query_start = np.ascontiguousarray(query_start, dtype=np.int32)
    tree = np.ascontiguousarray(tree, dtype=np.uint64)
    S = context_lens.shape[0]
    total_q = int(query_start[-1])
    if tree.shape != (total_q,):
        raise ValueError("tree: one uint64 per query row")
    full = sel is None
    if full:
        sel = np.stack(np.meshgrid(np.arange(total_q), np.arange(num_q_heads), indexing="ij"),
                       -1).reshape(-1, 2)
    sel = np.ascontiguousarray(sel, dtype=np.int32).reshape(-1, 2)
    out = np.zeros((sel.shape[0], head_dim), dtype=np.float64)
    rc = _load().oracle_paged_tree_attention(
        _ptr(query), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), _ptr(context_lens),
        _ptr(query_start), _ptr(tree), S, num_q_heads, num_kv_heads, head_dim, block_size,
        num_blocks, int(block_tables.shape[1]), float(scale), _code(q_dtype), _code(kv_dtype),
        float(kv_scale), _ptr(sel), int(sel.shape[0]), _ptr(out), int(nthreads))
    if rc != 0:
        raise ValueError("oracle paged_tree_attention: bad argument, a tree of more than 64 "
                         "tokens, more queries than context, or block id out of range")
    return out.reshape(total_q, num_q_heads, head_dim) if full else out


def merge_partials(ms, ls, accs) -> np.ndarray:
    ms = np.ascontiguousarray(ms, np.float64)
    ls = np.ascontiguousarray(ls, np.float64)
    accs = np.ascontiguousarray(accs, np.float64)
    n, d = accs.shape
    out = np.zeros(d, np.float64)
    _load().oracle_merge_partials(n, _ptr(ms), _ptr(ls), _ptr(accs), d, _ptr(out))
    return out
