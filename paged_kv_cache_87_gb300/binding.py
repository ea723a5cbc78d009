"""ctypes binding of libpagedkv.so (C ABI: include/pagedkv.h).

Argument marshalling only: shapes, dtypes and the stream are read off torch
tensors and passed as plain pointers and sizes; every step of the hot path
runs in the library's CUDA kernels.  There is no CPU fallback: if the library
cannot be loaded the calls raise.

Functions carry the C names:
  pkv_decode_workspace_bytes, pkv_paged_decode_attention,
  pkv_paged_decode_attention_prefix, pkv_paged_decode_attention_noalloc, pkv_reshape_and_cache, pkv_copy_blocks,
  pkv_get_device_status, pkv_status_string, pkv_version,
and the host block manager pkv_bm_* (wrapped by ``BlockManager``).
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libpagedkv.so")

PKV_F32, PKV_F16, PKV_BF16, PKV_FP8_E4M3 = 0, 1, 2, 3
(PKV_OK, PKV_ERR_INVALID_ARG, PKV_ERR_UNSUPPORTED, PKV_ERR_WORKSPACE, PKV_ERR_CUDA,
 PKV_ERR_OUT_OF_BLOCKS) = range(6)
DEV_BAD_BLOCK_ID, DEV_BAD_CONTEXT, DEV_BAD_SLOT, DEV_BAD_PAIR, DEV_WAIT_TIMEOUT = (
    0x1, 0x2, 0x4, 0x8, 0x10)

# ctypes signatures of every exported symbol
_SIGNATURES = {
    "pkv_decode_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int] * 6 + [ctypes.c_int]),
    "pkv_paged_decode_attention": (
        ctypes.c_int,
        [ctypes.c_void_p] * 5 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_float, ctypes.c_void_p,
                                                     ctypes.c_size_t, ctypes.c_void_p,
                                                     ctypes.c_void_p]),
    "pkv_paged_decode_attention_prefix": (
        ctypes.c_int,
        [ctypes.c_void_p] * 5 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_float, ctypes.c_void_p,
                                                     ctypes.c_size_t, ctypes.c_void_p,
                                                     ctypes.c_void_p]),
    "pkv_multi_query_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int]),
    "pkv_paged_multi_query_attention": (
        ctypes.c_int,
        [ctypes.c_void_p] * 6 + [ctypes.c_int] * 9 + [ctypes.c_float, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_float,
                                                      ctypes.c_void_p, ctypes.c_size_t,
                                                      ctypes.c_void_p, ctypes.c_void_p]),
    "pkv_paged_tree_attention": (
        ctypes.c_int,
        [ctypes.c_void_p] * 7 + [ctypes.c_int] * 9 + [ctypes.c_float, ctypes.c_int,
                                                      ctypes.c_int, ctypes.c_float,
                                                      ctypes.c_void_p, ctypes.c_size_t,
                                                      ctypes.c_void_p, ctypes.c_void_p]),
    "pkv_paged_decode_attention_noalloc": (
        ctypes.c_int,
        [ctypes.c_void_p] * 5 + [ctypes.c_int] * 8 + [ctypes.c_float, ctypes.c_int, ctypes.c_int,
                                                     ctypes.c_float, ctypes.c_void_p,
                                                     ctypes.c_void_p]),
    "pkv_reshape_and_cache": (
        ctypes.c_int,
        [ctypes.c_void_p] * 5 + [ctypes.c_int] * 5 + [ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                                     ctypes.c_void_p]),
    "pkv_copy_blocks": (
        ctypes.c_int,
        [ctypes.c_void_p] * 3 + [ctypes.c_int] * 5 + [ctypes.c_int, ctypes.c_void_p]),
    "pkv_get_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_uint)]),
    "pkv_selftest_wait_bound": (ctypes.c_int, [ctypes.c_void_p]),
    "pkv_swap_blocks": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                       ctypes.c_void_p, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_void_p]),
    "pkv_bm_create": (ctypes.c_void_p, [ctypes.c_int, ctypes.c_int, ctypes.c_void_p,
                                        ctypes.c_int]),
    "pkv_bm_destroy": (None, [ctypes.c_void_p]),
    "pkv_bm_num_free": (ctypes.c_int, [ctypes.c_void_p]),
    "pkv_bm_refcount": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int32]),
    "pkv_bm_add_sequence": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]),
    "pkv_bm_fork": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64]),
    "pkv_bm_append_slot": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64,
                                          ctypes.POINTER(ctypes.c_int64),
                                          ctypes.POINTER(ctypes.c_int32),
                                          ctypes.POINTER(ctypes.c_int32)]),
    "pkv_bm_free_sequence": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64]),
    "pkv_bm_sequence": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_void_p,
                                       ctypes.c_int, ctypes.POINTER(ctypes.c_int),
                                       ctypes.POINTER(ctypes.c_int64)]),
    "pkv_bm_prepare_step": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int,
                                           ctypes.c_void_p, ctypes.c_void_p,
                                           ctypes.POINTER(ctypes.c_int), ctypes.c_void_p,
                                           ctypes.c_int, ctypes.c_void_p]),
    "pkv_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pkv_version": (ctypes.c_int, []),
}

_lock = threading.Lock()
_lib = None


class PagedKVError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        super().__init__(f"{fn} failed: {status_text(status)} (status {status})")


def load(path: str = LIB_PATH):
    """Load the CUDA library (build it first with ``paged_kv_cache_87_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(path):
                raise RuntimeError(f"{path} is missing: build it with "
                                   "`python -m paged_kv_cache_87_gb300.build` (needs nvcc)")
            lib = ctypes.CDLL(path)
            for name, (res, args) in _SIGNATURES.items():
                f = getattr(lib, name)
                f.restype, f.argtypes = res, args
            _lib = lib
        return _lib


def status_text(status: int) -> str:
    return load().pkv_status_string(int(status)).decode()


def _check(fn: str, status: int) -> None:
    if status != PKV_OK:
        raise PagedKVError(fn, status)


_TORCH_CODES = {torch.float32: PKV_F32, torch.float16: PKV_F16, torch.bfloat16: PKV_BF16,
                torch.float8_e4m3fn: PKV_FP8_E4M3, torch.uint8: PKV_FP8_E4M3}
_NAME_CODES = {"f32": PKV_F32, "f16": PKV_F16, "bf16": PKV_BF16, "e4m3": PKV_FP8_E4M3}


def dtype_code(x) -> int:
    if isinstance(x, torch.Tensor):
        return _TORCH_CODES[x.dtype]
    if isinstance(x, torch.dtype):
        return _TORCH_CODES[x]
    if isinstance(x, str):
        return _NAME_CODES[x]
    return int(x)


def _stream_ptr(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _cuda(t: torch.Tensor, name: str) -> torch.Tensor:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")
    return t


# ------------------------------------------------------------------ calls --

def pkv_decode_workspace_bytes(num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                               block_size: int, max_context_len: int, kv_dtype) -> int:
    return int(load().pkv_decode_workspace_bytes(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                 block_size, max_context_len,
                                                 dtype_code(kv_dtype)))


def _decode_args(query, k_cache, v_cache, block_tables, context_lens, max_context_len, scale,
                 kv_scale, workspace, out, stream, prefix):
    """Checks and marshals a decode call: (C function name, argument tuple, out, workspace)."""
    S, Hq, d = query.shape
    NB, Hkv, B, d2 = k_cache.shape
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes must be [num_blocks, num_kv_heads, block_size, head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    for t, n in ((query, "query"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens")):
        _cuda(t, n)
    qc, kc = dtype_code(query), dtype_code(k_cache)
    need = pkv_decode_workspace_bytes(S, Hq, Hkv, d, B, max_context_len, kc)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=query.device)
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    _cuda(workspace, "workspace")
    fn = "pkv_paged_decode_attention_prefix" if prefix else "pkv_paged_decode_attention"
    args = (query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), S, Hq, Hkv, d, B, NB, block_tables.shape[1],
            int(max_context_len), float(scale), qc, kc, float(kv_scale), workspace.data_ptr(),
            workspace.numel() * workspace.element_size(), out.data_ptr(), _stream_ptr(stream))
    return fn, args, out, workspace


def pkv_paged_decode_attention(query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                               block_tables: torch.Tensor, context_lens: torch.Tensor,
                               max_context_len: int, scale: float, kv_scale: float = 1.0,
                               workspace: torch.Tensor | None = None,
                               out: torch.Tensor | None = None, stream=None,
                               prefix: bool = False) -> torch.Tensor:
    """out[s, h] = softmax(scale * q[s, h] . K_s^T) V_s over context_lens[s] tokens.

    query [S, Hq, d]; k_cache / v_cache [NB, Hkv, B, d] (float8_e4m3fn or uint8
    for FP8); block_tables int32 [S, max_blocks]; context_lens int32 [S].
    ``workspace`` (uint8, >= pkv_decode_workspace_bytes) is allocated if None.
    ``prefix=True`` calls pkv_paged_decode_attention_prefix (shared prompts
    read once per group of sequences).
    """
    fn, args, out, _ = _decode_args(query, k_cache, v_cache, block_tables, context_lens,
                                    max_context_len, scale, kv_scale, workspace, out, stream,
                                    prefix)
    _check(fn, getattr(load(), fn)(*args))
    return out


class PreparedCall:
    """One C-ABI call whose arguments (pointers, sizes, stream) were checked and
    marshalled once; calling it issues the same call again.

    For a serving loop that runs the same step on the same buffers every
    iteration: the per-call Python cost drops to one ctypes call.  The tensors
    behind the pointers are kept referenced here and must not be reallocated."""

    def __init__(self, name: str, args: tuple, keep: tuple = ()):
        self.name = name
        self._fn = getattr(load(), name)
        self._args = tuple(args)
        self._keep = keep

    def __call__(self) -> None:
        st = self._fn(*self._args)
        if st != PKV_OK:
            raise PagedKVError(self.name, st)


def prepare_paged_decode_attention(query, k_cache, v_cache, block_tables, context_lens,
                                   max_context_len, scale, kv_scale=1.0, workspace=None,
                                   out=None, stream=None, prefix=False) -> PreparedCall:
    """pkv_paged_decode_attention (or the prefix-aware entry) as a PreparedCall."""
    fn, args, out, workspace = _decode_args(query, k_cache, v_cache, block_tables,
                                            context_lens, max_context_len, scale, kv_scale,
                                            workspace, out, stream, prefix)
    return PreparedCall(fn, args, (query, k_cache, v_cache, block_tables, context_lens,
                                   workspace, out))


def pkv_multi_query_workspace_bytes(num_seqs: int) -> int:
    return int(load().pkv_multi_query_workspace_bytes(int(num_seqs)))


def pkv_paged_multi_query_attention(query: torch.Tensor, k_cache: torch.Tensor,
                                    v_cache: torch.Tensor, block_tables: torch.Tensor,
                                    context_lens: torch.Tensor, query_start: torch.Tensor,
                                    max_context_len: int, scale: float, kv_scale: float = 1.0,
                                    workspace: torch.Tensor | None = None,
                                    out: torch.Tensor | None = None,
                                    stream=None) -> torch.Tensor:
    """Causal attention of several query tokens per sequence over the paged cache.

    query [total_q, Hq, d]; query_start int32 [S + 1] (rows of sequence s are
    query_start[s] .. query_start[s+1]-1; query_start[S] = total_q);
    context_lens int32 [S] counts the cached tokens including the queries'
    own (the last n_s).  Row i of sequence s attends to tokens
    0 .. context_lens[s] - n_s + i.
    """
    return _multi_query("pkv_paged_multi_query_attention", query, k_cache, v_cache,
                        block_tables, context_lens, query_start, None, max_context_len, scale,
                        kv_scale, workspace, out, stream)


def pkv_paged_tree_attention(query: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                             block_tables: torch.Tensor, context_lens: torch.Tensor,
                             query_start: torch.Tensor, tree_mask: torch.Tensor,
                             max_context_len: int, scale: float, kv_scale: float = 1.0,
                             workspace: torch.Tensor | None = None,
                             out: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """Verification of draft-token trees: as pkv_paged_multi_query_attention, but the
    n_s <= 64 queries of sequence s are a tree laid out parents first, and query i sees
    the prior context, itself and each tree token j < i whose bit j is set in
    tree_mask[query_start[s] + i] (int64 / uint64 bits, [total_q])."""
    if tree_mask.dtype not in (torch.int64, torch.uint64) or tree_mask.dim() != 1 or \
            int(tree_mask.shape[0]) != int(query.shape[0]):
        raise ValueError("tree_mask must be 64-bit [total_q]")
    _cuda(tree_mask, "tree_mask")
    return _multi_query("pkv_paged_tree_attention", query, k_cache, v_cache, block_tables,
                        context_lens, query_start, tree_mask, max_context_len, scale, kv_scale,
                        workspace, out, stream)


def _multi_query(name, query, k_cache, v_cache, block_tables, context_lens, query_start,
                 tree_mask, max_context_len, scale, kv_scale, workspace, out, stream):
    total_q, Hq, d = query.shape
    NB, Hkv, B, d2 = k_cache.shape
    S = int(context_lens.shape[0])
    if d2 != d or tuple(v_cache.shape) != tuple(k_cache.shape):
        raise ValueError("cache shapes must be [num_blocks, num_kv_heads, block_size, head_dim]")
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32 or \
            query_start.dtype != torch.int32:
        raise ValueError("block_tables, context_lens and query_start must be int32")
    if int(query_start.shape[0]) != S + 1:
        raise ValueError("query_start must have num_seqs + 1 entries")
    for t, n in ((query, "query"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens"),
                 (query_start, "query_start")):
        _cuda(t, n)
    need = pkv_multi_query_workspace_bytes(S)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=query.device)
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    _cuda(workspace, "workspace")
    head = [query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
            context_lens.data_ptr(), query_start.data_ptr()]
    if tree_mask is not None:
        head.append(tree_mask.data_ptr())
    st = getattr(load(), name)(
        *head, S, total_q, Hq, Hkv, d, B, NB,
        block_tables.shape[1], int(max_context_len), float(scale), dtype_code(query),
        dtype_code(k_cache), float(kv_scale), workspace.data_ptr(),
        workspace.numel() * workspace.element_size(), out.data_ptr(), _stream_ptr(stream))
    _check(name, st)
    return out


NOALLOC_SCRATCH_BYTES = 16 << 20   # PKV_NOALLOC_SCRATCH_BYTES


def pkv_paged_decode_attention_noalloc(query: torch.Tensor, k_cache: torch.Tensor,
                                       v_cache: torch.Tensor, block_tables: torch.Tensor,
                                       context_lens: torch.Tensor, max_context_len: int,
                                       scale: float, kv_scale: float = 1.0,
                                       out: torch.Tensor | None = None,
                                       stream=None) -> torch.Tensor:
    """Decode with the library's static device scratch instead of a workspace.

    For callers that cannot allocate device memory while they decode.  Fails
    with PKV_ERR_WORKSPACE when the sizes need more than 16 MiB of scratch.
    Calls that overlap on the GPU race on the shared scratch: keep them on
    one stream.  (``out`` is allocated here only when not given.)
    """
    S, Hq, d = query.shape
    NB, Hkv, B, _ = k_cache.shape
    for t, n in ((query, "query"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (block_tables, "block_tables"), (context_lens, "context_lens")):
        _cuda(t, n)
    if out is None:
        out = torch.empty_like(query)
    _cuda(out, "out")
    st = load().pkv_paged_decode_attention_noalloc(
        query.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), block_tables.data_ptr(),
        context_lens.data_ptr(), S, Hq, Hkv, d, B, NB, block_tables.shape[1],
        int(max_context_len), float(scale), dtype_code(query), dtype_code(k_cache),
        float(kv_scale), out.data_ptr(), _stream_ptr(stream))
    _check("pkv_paged_decode_attention_noalloc", st)
    return out


def _reshape_args(key, value, k_cache, v_cache, slot_mapping, kv_scale, stream):
    T, Hkv, d = key.shape
    NB, Hkv2, B, d2 = k_cache.shape
    if (Hkv2, d2) != (Hkv, d) or tuple(value.shape) != tuple(key.shape):
        raise ValueError("key/value [T, Hkv, d] do not match the cache [NB, Hkv, B, d]")
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    for t, n in ((key, "key"), (value, "value"), (k_cache, "k_cache"), (v_cache, "v_cache"),
                 (slot_mapping, "slot_mapping")):
        _cuda(t, n)
    return (key.data_ptr(), value.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
            slot_mapping.data_ptr(), T, Hkv, d, B, NB, dtype_code(key), dtype_code(k_cache),
            float(kv_scale), _stream_ptr(stream))


def pkv_reshape_and_cache(key: torch.Tensor, value: torch.Tensor, k_cache: torch.Tensor,
                          v_cache: torch.Tensor, slot_mapping: torch.Tensor,
                          kv_scale: float = 1.0, stream=None) -> None:
    """k_cache[slot // B, h, slot % B] = key[t, h] (e4m3(x / kv_scale) for FP8 caches)."""
    args = _reshape_args(key, value, k_cache, v_cache, slot_mapping, kv_scale, stream)
    _check("pkv_reshape_and_cache", load().pkv_reshape_and_cache(*args))


def prepare_reshape_and_cache(key, value, k_cache, v_cache, slot_mapping, kv_scale=1.0,
                              stream=None) -> PreparedCall:
    """pkv_reshape_and_cache as a PreparedCall."""
    return PreparedCall("pkv_reshape_and_cache",
                        _reshape_args(key, value, k_cache, v_cache, slot_mapping, kv_scale,
                                      stream), (key, value, k_cache, v_cache, slot_mapping))


def validate_pairs(pairs: np.ndarray, num_blocks: int) -> None:
    """Host check of the copy_blocks contract: ids in the pool, distinct dsts, no dst is a src."""
    pairs = np.asarray(pairs).reshape(-1, 2)
    if pairs.size and (pairs.min() < 0 or pairs.max() >= num_blocks):
        raise ValueError("copy_blocks: block id outside the pool")
    dst = pairs[:, 1]
    if len(set(dst.tolist())) != len(dst):
        raise ValueError("copy_blocks: a destination block repeats")
    if set(dst.tolist()) & set(pairs[:, 0].tolist()):
        raise ValueError("copy_blocks: a destination block is also a source")


def _copy_args(k_cache, v_cache, src_dst_pairs, stream):
    NB, Hkv, B, d = k_cache.shape
    _cuda(k_cache, "k_cache")
    _cuda(v_cache, "v_cache")
    if isinstance(src_dst_pairs, torch.Tensor) and src_dst_pairs.is_cuda:
        pairs = src_dst_pairs
    else:
        host = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int32).reshape(-1, 2))
        validate_pairs(host, NB)
        pairs = torch.from_numpy(host).to(k_cache.device)
    if pairs.dtype != torch.int32:
        raise ValueError("src_dst_pairs must be int32")
    n = pairs.numel() // 2
    return (k_cache.data_ptr(), v_cache.data_ptr(), pairs.data_ptr() if n else None, n, Hkv, d,
            B, NB, dtype_code(k_cache), _stream_ptr(stream)), pairs


def pkv_copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor, src_dst_pairs,
                    stream=None) -> None:
    """Copy physical blocks src -> dst of both caches for every (src, dst) pair.

    ``src_dst_pairs``: int32 [n, 2].  A host array/tensor is validated and
    copied to the device; a CUDA tensor is used as is (the caller has
    validated it).
    """
    args, _ = _copy_args(k_cache, v_cache, src_dst_pairs, stream)
    _check("pkv_copy_blocks", load().pkv_copy_blocks(*args))


def prepare_copy_blocks(k_cache, v_cache, src_dst_pairs, stream=None) -> PreparedCall:
    """pkv_copy_blocks as a PreparedCall (device pairs are used as they are then)."""
    args, pairs = _copy_args(k_cache, v_cache, src_dst_pairs, stream)
    return PreparedCall("pkv_copy_blocks", args, (k_cache, v_cache, pairs))


def pkv_swap_blocks(src_k: torch.Tensor, src_v: torch.Tensor, dst_k: torch.Tensor,
                    dst_v: torch.Tensor, src_dst_pairs, stream=None) -> None:
    """Copy blocks between two pools (device or pinned host): dst[p[1]] = src[p[0]].

    Pools are [blocks, kv heads, B, d]; a host pool must be pinned
    (``tensor.pin_memory()``).  Host pairs are validated and staged in a pinned
    buffer; a CUDA or pinned tensor is used as is.
    """
    NBs, Hkv, B, d = src_k.shape
    NBd = dst_k.shape[0]
    if tuple(dst_k.shape[1:]) != (Hkv, B, d) or src_v.shape != src_k.shape or \
            dst_v.shape != dst_k.shape:
        raise ValueError("pools must be [blocks, kv heads, B, d] with matching rows")
    for t, n in ((src_k, "src_k"), (src_v, "src_v"), (dst_k, "dst_k"), (dst_v, "dst_v")):
        if not t.is_contiguous() or not (t.is_cuda or t.is_pinned()):
            raise ValueError(f"{n} must be a contiguous CUDA or pinned host tensor")
    if isinstance(src_dst_pairs, torch.Tensor) and (src_dst_pairs.is_cuda or
                                                    src_dst_pairs.is_pinned()):
        pairs = src_dst_pairs
    else:
        host = np.ascontiguousarray(np.asarray(src_dst_pairs, dtype=np.int32).reshape(-1, 2))
        if host.size and (host[:, 0].min() < 0 or host[:, 0].max() >= NBs or
                          host[:, 1].min() < 0 or host[:, 1].max() >= NBd):
            raise ValueError("swap_blocks: block id outside its pool")
        if len(set(host[:, 1].tolist())) != len(host):
            raise ValueError("swap_blocks: a destination block repeats")
        pairs = torch.from_numpy(host).pin_memory()
    n = pairs.numel() // 2
    st = load().pkv_swap_blocks(src_k.data_ptr(), src_v.data_ptr(), NBs, dst_k.data_ptr(),
                                dst_v.data_ptr(), NBd, pairs.data_ptr() if n else None, n, Hkv,
                                d, B, dtype_code(src_k), _stream_ptr(stream))
    _check("pkv_swap_blocks", st)
    if not (isinstance(src_dst_pairs, torch.Tensor)) and n:
        # the launch reads the staged pairs asynchronously: keep them alive until it ran
        (stream or torch.cuda.current_stream()).synchronize()


def pkv_get_device_status() -> int:
    """Read and clear the current device's status word (PKV_DEV_* bits). Synchronous."""
    v = ctypes.c_uint(0)
    _check("pkv_get_device_status", load().pkv_get_device_status(ctypes.byref(v)))
    return int(v.value)


def pkv_selftest_wait_bound(stream=None) -> None:
    """Launch the wait self-test: a kernel whose pipeline wait never completes gives up
    after the waits' bound (2 s) and sets DEV_WAIT_TIMEOUT in the device status word."""
    _check("pkv_selftest_wait_bound", load().pkv_selftest_wait_bound(_stream_ptr(stream)))


def pkv_status_string(status: int) -> str:
    return status_text(status)


def pkv_version() -> int:
    return int(load().pkv_version())


# ----------------------------------------------------------- block manager --

class BlockManager:
    """The library's host block manager (C ABI pkv_bm_*): free list, reference
    counts, block tables, slots and copy-on-write pairs for the device kernels."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        lib = load()
        self.block_size = block_size
        self.num_blocks = num_blocks
        if free_order is None:
            h = lib.pkv_bm_create(num_blocks, block_size, None, 0)
        else:
            order = np.ascontiguousarray(free_order, dtype=np.int32)
            h = lib.pkv_bm_create(num_blocks, block_size, order.ctypes.data, int(order.size))
        if not h:
            raise ValueError("pkv_bm_create: bad arguments")
        self._h = ctypes.c_void_p(h)

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and _lib is not None:
            _lib.pkv_bm_destroy(h)
            self._h = None

    @property
    def num_free(self) -> int:
        return int(load().pkv_bm_num_free(self._h))

    def refcount(self, block: int) -> int:
        return int(load().pkv_bm_refcount(self._h, int(block)))

    def add_sequence(self, seq_id: int, num_tokens: int) -> None:
        _check("pkv_bm_add_sequence", load().pkv_bm_add_sequence(self._h, seq_id, num_tokens))

    def fork(self, parent: int, child: int) -> None:
        _check("pkv_bm_fork", load().pkv_bm_fork(self._h, parent, child))

    def append_slot(self, seq_id: int):
        """(slot, (src, dst) copy-on-write pair or None) of the sequence's next token."""
        slot, src, dst = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_bm_append_slot", load().pkv_bm_append_slot(
            self._h, seq_id, ctypes.byref(slot), ctypes.byref(src), ctypes.byref(dst)))
        return int(slot.value), (None if src.value < 0 else (int(src.value), int(dst.value)))

    def free_sequence(self, seq_id: int) -> None:
        _check("pkv_bm_free_sequence", load().pkv_bm_free_sequence(self._h, seq_id))

    def sequence(self, seq_id: int):
        """(block table as a list, number of tokens)."""
        nb, nt = ctypes.c_int(), ctypes.c_int64()
        _check("pkv_bm_sequence", load().pkv_bm_sequence(self._h, seq_id, None, 0,
                                                          ctypes.byref(nb), ctypes.byref(nt)))
        table = np.zeros(max(1, nb.value), dtype=np.int32)
        _check("pkv_bm_sequence", load().pkv_bm_sequence(
            self._h, seq_id, table.ctypes.data, int(table.size), ctypes.byref(nb),
            ctypes.byref(nt)))
        return table[:nb.value].tolist(), int(nt.value)

    def prepare_step(self, seq_ids, max_blocks: int):
        """Append one token to each sequence: (slot_mapping int64[n], cow_pairs int32[k, 2],
        block_tables int32[n, max_blocks], context_lens int32[n])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = int(ids.size)
        slots = np.zeros(n, np.int64)
        pairs = np.zeros((max(n, 1), 2), np.int32)
        tables = np.zeros((max(n, 1), max_blocks), np.int32)
        ctx = np.zeros(max(n, 1), np.int32)
        ncow = ctypes.c_int(0)
        _check("pkv_bm_prepare_step", load().pkv_bm_prepare_step(
            self._h, ids.ctypes.data, n, slots.ctypes.data, pairs.ctypes.data,
            ctypes.byref(ncow), tables.ctypes.data, max_blocks, ctx.ctypes.data))
        return slots, pairs[:ncow.value].copy(), tables[:n], ctx[:n]
