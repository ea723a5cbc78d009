"""The C-ABI library builds, loads and exports what include/pagedkv.h declares;
host-side validation answers without a GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

from paged_kv_cache_87_gb300 import binding, build

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "pagedkv.h")


@pytest.fixture(scope="module")
def lib():
    build.build()
    return binding.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_\w+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("pkv_paged_decode_attention", "pkv_reshape_and_cache", "pkv_copy_blocks",
                 "pkv_decode_workspace_bytes", "pkv_get_device_status", "pkv_status_string",
                 "pkv_paged_multi_query_attention", "pkv_paged_tree_attention",
                 "pkv_selftest_wait_bound"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in binding._SIGNATURES, name


def test_status_strings(lib):
    for st in range(5):
        assert binding.pkv_status_string(st)
    assert binding.pkv_version() >= 100


def test_workspace_sizes(lib):
    # single-chunk contexts need no partial states: the workspace is the fixed
    # per-worker table (32 B x 4096 workers) plus small per-sequence arrays
    small = binding.pkv_decode_workspace_bytes(4, 8, 8, 64, 16, 256, "f32")
    assert 0 < small < 192 * 1024
    # OPT-13B-shaped: 2048 tokens -> 4 chunks of 512 -> partial states for 64*40*4 chunks
    ws = binding.pkv_decode_workspace_bytes(64, 40, 40, 128, 16, 2048, "f16")
    assert ws >= 64 * 40 * 4 * (128 + 2) * 4
    # unsupported / invalid sizes give 0
    assert binding.pkv_decode_workspace_bytes(4, 8, 8, 96, 16, 256, "f32") == 0
    assert binding.pkv_decode_workspace_bytes(4, 8, 3, 64, 16, 256, "f32") == 0
    assert binding.pkv_decode_workspace_bytes(4, 8, 8, 64, 12, 256, "f32") == 0
    # contexts beyond 256 chunks of 64*B tokens are out of range for B=8
    assert binding.pkv_decode_workspace_bytes(1, 8, 8, 64, 8, 200000, "f32") == 0


def _decode(lib, **kw):
    a = dict(query=1024, k=1024, v=1024, bt=1024, cl=1024, S=4, Hq=8, Hkv=8, d=64, B=16, NB=64,
             mb=16, mctx=256, scale=0.125, qt=0, kt=0, kvs=1.0, ws=None, wsb=0, out=1024)
    a.update(kw)
    return lib.pkv_paged_decode_attention(a["query"], a["k"], a["v"], a["bt"], a["cl"], a["S"],
                                          a["Hq"], a["Hkv"], a["d"], a["B"], a["NB"], a["mb"],
                                          a["mctx"], a["scale"], a["qt"], a["kt"], a["kvs"],
                                          a["ws"], a["wsb"], a["out"], None)


def test_decode_host_validation(lib):
    E = binding
    assert _decode(lib, query=None) == E.PKV_ERR_INVALID_ARG
    assert _decode(lib, d=96) == E.PKV_ERR_UNSUPPORTED
    assert _decode(lib, B=12) == E.PKV_ERR_UNSUPPORTED
    assert _decode(lib, Hkv=3) == E.PKV_ERR_INVALID_ARG
    assert _decode(lib, qt=3) == E.PKV_ERR_UNSUPPORTED        # fp8 queries are not built
    assert _decode(lib, qt=1, kt=2) == E.PKV_ERR_UNSUPPORTED  # f16 q with bf16 cache
    assert _decode(lib, kvs=0.0) == E.PKV_ERR_INVALID_ARG
    assert _decode(lib, kvs=float("inf")) == E.PKV_ERR_INVALID_ARG
    assert _decode(lib, scale=float("nan")) == E.PKV_ERR_INVALID_ARG
    assert _decode(lib, mctx=16 * 16 + 1) == E.PKV_ERR_INVALID_ARG
    assert _decode(lib, query=1024 + 8) == E.PKV_ERR_INVALID_ARG   # misaligned
    assert _decode(lib) == E.PKV_ERR_WORKSPACE                     # no workspace
    assert _decode(lib, ws=4096 + 16, wsb=1 << 20) == E.PKV_ERR_WORKSPACE   # misaligned
    assert _decode(lib, ws=4096, wsb=16) == E.PKV_ERR_WORKSPACE    # too small
    assert _decode(lib, S=0, query=None, k=None) == E.PKV_OK       # nothing to do


def _multi_query(lib, **kw):
    a = dict(query=1024, k=1024, v=1024, bt=1024, cl=1024, qs=1024, S=4, tq=16, Hq=8, Hkv=2,
             d=128, B=16, NB=64, mb=16, mctx=256, scale=0.088, qt=2, kt=2, kvs=1.0, ws=None,
             wsb=0, out=1024)
    a.update(kw)
    return lib.pkv_paged_multi_query_attention(
        a["query"], a["k"], a["v"], a["bt"], a["cl"], a["qs"], a["S"], a["tq"], a["Hq"],
        a["Hkv"], a["d"], a["B"], a["NB"], a["mb"], a["mctx"], a["scale"], a["qt"], a["kt"],
        a["kvs"], a["ws"], a["wsb"], a["out"], None)


def test_multi_query_host_validation(lib):
    E = binding
    assert _multi_query(lib, query=None) == E.PKV_ERR_INVALID_ARG
    assert _multi_query(lib, qs=None) == E.PKV_ERR_INVALID_ARG
    assert _multi_query(lib, qt=0, kt=0) == E.PKV_ERR_UNSUPPORTED   # fp32
    assert _multi_query(lib, kt=3) == E.PKV_ERR_UNSUPPORTED          # FP8 K/V
    assert _multi_query(lib, qt=1) == E.PKV_ERR_UNSUPPORTED          # f16 q, bf16 cache
    assert _multi_query(lib, d=64) == E.PKV_ERR_UNSUPPORTED
    assert _multi_query(lib, B=12) == E.PKV_ERR_UNSUPPORTED
    assert _multi_query(lib, Hq=6) == E.PKV_ERR_UNSUPPORTED          # group 3 does not divide 128
    assert _multi_query(lib, Hkv=3) == E.PKV_ERR_INVALID_ARG
    assert _multi_query(lib, kvs=0.0) == E.PKV_ERR_INVALID_ARG
    assert _multi_query(lib, mctx=16 * 16 + 1) == E.PKV_ERR_INVALID_ARG
    assert _multi_query(lib, qs=1024 + 2) == E.PKV_ERR_INVALID_ARG   # misaligned
    assert _multi_query(lib) == E.PKV_ERR_WORKSPACE
    assert _multi_query(lib, ws=4096, wsb=8) == E.PKV_ERR_WORKSPACE
    assert _multi_query(lib, tq=0, query=None) == E.PKV_OK           # nothing to do
    assert binding.pkv_multi_query_workspace_bytes(4) == 768   # item prefix, launch order, counter
    assert binding.pkv_multi_query_workspace_bytes(1000) == 8448


def _tree(lib, tree, **kw):
    a = dict(query=1024, k=1024, v=1024, bt=1024, cl=1024, qs=1024, S=4, tq=16, Hq=8, Hkv=2,
             d=128, B=16, NB=64, mb=16, mctx=256, scale=0.088, qt=2, kt=2, kvs=1.0, ws=4096,
             wsb=4096, out=1024)
    a.update(kw)
    return lib.pkv_paged_tree_attention(
        a["query"], a["k"], a["v"], a["bt"], a["cl"], a["qs"], tree, a["S"], a["tq"], a["Hq"],
        a["Hkv"], a["d"], a["B"], a["NB"], a["mb"], a["mctx"], a["scale"], a["qt"], a["kt"],
        a["kvs"], a["ws"], a["wsb"], a["out"], None)


def test_tree_host_validation(lib):
    """The draft-tree entry validates like the causal one and needs an 8-byte aligned mask
    (checked before any device call)."""
    E = binding
    assert _tree(lib, None) == E.PKV_ERR_INVALID_ARG                 # no mask
    assert _tree(lib, 1028) == E.PKV_ERR_INVALID_ARG                 # misaligned mask
    assert _tree(lib, 1024, qt=0, kt=0) == E.PKV_ERR_UNSUPPORTED      # fp32
    assert _tree(lib, 1024, Hq=6) == E.PKV_ERR_UNSUPPORTED
    assert _tree(lib, 1024, ws=None, wsb=0) == E.PKV_ERR_WORKSPACE
    assert _tree(lib, None, tq=0, query=None) == E.PKV_OK            # nothing to do


def test_reshape_and_copy_host_validation(lib):
    E = binding
    f = lib.pkv_reshape_and_cache
    assert f(None, 16, 16, 16, 16, 3, 8, 128, 16, 64, 2, 2, 1.0, None) == E.PKV_ERR_INVALID_ARG
    assert f(16, 16, 16, 16, 16, 3, 8, 100, 16, 64, 2, 2, 1.0, None) == E.PKV_ERR_UNSUPPORTED
    assert f(16, 16, 16, 16, 16, 3, 8, 128, 16, 64, 2, 3, 0.0, None) == E.PKV_ERR_INVALID_ARG
    assert f(16, 16, 16, 16, 16, 3, 8, 128, 16, 64, 1, 2, 1.0, None) == E.PKV_ERR_UNSUPPORTED
    assert f(16, 16, 16, 16, 12, 3, 8, 128, 16, 64, 2, 2, 1.0, None) == E.PKV_ERR_INVALID_ARG
    assert f(None, None, None, None, None, 0, 8, 128, 16, 64, 2, 2, 1.0, None) == E.PKV_OK
    g = lib.pkv_copy_blocks
    assert g(None, 16, 16, 2, 8, 128, 16, 64, 3, None) == E.PKV_ERR_INVALID_ARG
    assert g(16, 16, 16, 2, 8, 128, 24, 64, 3, None) == E.PKV_ERR_UNSUPPORTED
    assert g(None, None, None, 0, 8, 128, 16, 64, 3, None) == E.PKV_OK


def test_binding_validates_copy_pairs_on_host():
    binding.validate_pairs([[1, 2], [3, 4]], 8)
    for bad in ([[1, 2], [3, 2]], [[1, 2], [2, 5]], [[0, 8]], [[-1, 2]]):
        with pytest.raises(ValueError):
            binding.validate_pairs(bad, 8)


def test_binding_checks_the_tree_mask_before_any_call():
    """The tree mask must be 64-bit, one entry per query row; checked before the library
    is called (no device needed)."""
    import torch
    q = torch.zeros(5, 2, 128, dtype=torch.bfloat16)
    kc = torch.zeros(4, 2, 16, 128, dtype=torch.bfloat16)
    i32 = lambda *s: torch.zeros(*s, dtype=torch.int32)
    for bad in (torch.zeros(5, dtype=torch.int32), torch.zeros(4, dtype=torch.int64),
                torch.zeros(5, 1, dtype=torch.int64)):
        with pytest.raises(ValueError):
            binding.pkv_paged_tree_attention(q, kc, kc, i32(1, 4), i32(1), i32(2), bad, 64, 0.1)


def test_product_path_does_not_import_the_oracle():
    """The package never reaches into oracle/ (test infrastructure only)."""
    pkg = os.path.dirname(binding.__file__)
    for root, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(root, fn)).read()
                assert not re.search(r"^\s*(import|from)\s+oracle\b", src, re.M), fn
                assert "oracle.c" not in src and "liboracle" not in src, fn


def test_missing_library_fails_loudly(tmp_path):
    saved = binding._lib
    binding._lib = None
    try:
        with pytest.raises(RuntimeError):
            binding.load(str(tmp_path / "nope.so"))
    finally:
        binding._lib = saved
