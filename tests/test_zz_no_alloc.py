"""pkv_paged_decode_attention_noalloc: decode for callers that cannot allocate.

Callers inside a host framework that owns every device allocation, under a
device-memory budget fixed at start-up, or in a loop where a cudaMalloc (which
may synchronise the device) is not allowed cannot hand the decode a
cudaMalloc'ed workspace.  This entry point uses the library's static device
scratch instead.  Its output must match the workspace entry point's on the same
inputs, call after call (the scratch keeps the previous call's contents), and
it must refuse sizes that need more scratch than the array holds.

The file is named so pytest collects it last.
"""
import ctypes
import math

import numpy as np
import pytest
import torch

from paged_kv_cache_87_gb300 import binding, inputs
from tests.helpers import gpu_state, tolerance

pytestmark = pytest.mark.gpu


def _call_noalloc(st, out):
    """Through the C ABI directly: plain pointers and sizes."""
    w = st.w
    lib = binding.load()
    return lib.pkv_paged_decode_attention_noalloc(
        st.query.data_ptr(), st.k_cache.data_ptr(), st.v_cache.data_ptr(),
        st.block_tables.data_ptr(), st.context_lens.data_ptr(), w.num_seqs, w.num_q_heads,
        w.num_kv_heads, w.head_dim, w.block_size, w.num_blocks, w.max_blocks,
        w.max_context_len, ctypes.c_float(w.scale), binding.dtype_code(w.q_dtype),
        binding.dtype_code(w.kv_dtype), ctypes.c_float(w.kv_scale), out.data_ptr(),
        torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("make", [
    lambda: inputs.make_config(1, num_seqs=16),                  # multi-chunk fp16 MHA
    lambda: inputs.make_config(4, num_seqs=16, ctx_cap=3000),    # FP8 KV, GQA 4
])
def test_noalloc_matches_workspace_entry_point_twice(make):
    w = make()
    need = binding.pkv_decode_workspace_bytes(w.num_seqs, w.num_q_heads, w.num_kv_heads,
                                              w.head_dim, w.block_size, w.max_context_len,
                                              w.kv_dtype)
    assert 0 < need <= binding.NOALLOC_SCRATCH_BYTES
    st = gpu_state(w)                     # setup + one step with the workspace entry point
    ref = st.out.clone()
    for _ in range(2):                    # two calls in a row on the shared scratch
        out = torch.full_like(st.out, float("nan"))
        assert _call_noalloc(st, out) == binding.PKV_OK
        torch.cuda.synchronize()
        err = (out.double() - ref.double()).abs().max().item()
        assert math.isfinite(err) and err <= tolerance(w)
    assert binding.pkv_get_device_status() == 0


def test_noalloc_rejects_sizes_beyond_the_scratch():
    w = inputs.make_config(0)
    st = gpu_state(w)
    # a batch of 4096 long contexts needs far more split-KV state than the static array
    # holds: the call must refuse before launching anything (the small tensors of `st`
    # are never touched)
    need = binding.pkv_decode_workspace_bytes(4096, 64, 8, 128, 32, 100000, "bf16")
    assert need > binding.NOALLOC_SCRATCH_BYTES
    lib = binding.load()
    rc = lib.pkv_paged_decode_attention_noalloc(
        st.query.data_ptr(), st.k_cache.data_ptr(), st.v_cache.data_ptr(),
        st.block_tables.data_ptr(), st.context_lens.data_ptr(), 4096, 64, 8, 128, 32,
        w.num_blocks, 100000, 100000, ctypes.c_float(0.1), binding.PKV_BF16, binding.PKV_BF16,
        ctypes.c_float(1.0), st.out.data_ptr(), torch.cuda.current_stream().cuda_stream)
    assert rc == binding.PKV_ERR_WORKSPACE
    assert binding.pkv_get_device_status() == 0
