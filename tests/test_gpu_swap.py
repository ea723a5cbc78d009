"""Swapping blocks between the device pool and a pinned host pool ("PagedAttention:
Mathematical Foundations ..." §6 Preemption and Memory Recovery, swapping)."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import binding, inputs
from paged_kv_cache_87_gb300.session import host_tensor, to_numpy_storage
from tests.helpers import TOL, oracle_caches, oracle_decode

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv", ["bf16", "e4m3", "f32"])
def test_swap_out_and_in_bit_exact(kv):
    rng = np.random.default_rng(5)
    NBd, NBh, H, B, d = 60, 40, 4, 16, 128
    nbytes = NBd * H * B * d * inputs.DTYPE_BYTES[kv]
    dev_k = host_tensor(rng.integers(0, 256, nbytes, np.uint8).view(inputs.NP_CONTAINER[kv])
                        .reshape(NBd, H, B, d), kv).cuda()
    dev_v = host_tensor(rng.integers(0, 256, nbytes, np.uint8).view(inputs.NP_CONTAINER[kv])
                        .reshape(NBd, H, B, d), kv).cuda()
    k0, v0 = dev_k.clone(), dev_v.clone()
    host_k = torch.zeros((NBh, H, B, d), dtype=dev_k.dtype).pin_memory()
    host_v = torch.zeros((NBh, H, B, d), dtype=dev_v.dtype).pin_memory()
    out_pairs = np.stack([rng.permutation(NBd)[:25], rng.permutation(NBh)[:25]], 1)
    binding.pkv_swap_blocks(dev_k, dev_v, host_k, host_v, out_pairs)          # swap out
    torch.cuda.synchronize()
    for s, h in out_pairs:
        assert torch.equal(host_k[h].view(torch.uint8), k0[s].cpu().view(torch.uint8))
        assert torch.equal(host_v[h].view(torch.uint8), v0[s].cpu().view(torch.uint8))
    dev_k.view(torch.uint8).fill_(0x7F)
    dev_v.view(torch.uint8).fill_(0x7F)
    in_dst = rng.permutation(NBd)[:25]
    binding.pkv_swap_blocks(host_k, host_v, dev_k, dev_v,
                            np.stack([out_pairs[:, 1], in_dst], 1))           # swap in
    torch.cuda.synchronize()
    for (s, _), t in zip(out_pairs, in_dst):
        assert torch.equal(dev_k[t].view(torch.uint8), k0[s].view(torch.uint8))
        assert torch.equal(dev_v[t].view(torch.uint8), v0[s].view(torch.uint8))
    assert binding.pkv_get_device_status() == 0


def test_decode_after_swap_round_trip():
    """Preempt a whole batch to host, bring it back into other blocks, decode."""
    w = inputs.make_config(2, num_seqs=12)
    from tests.helpers import gpu_state
    st = gpu_state(w)
    ref_out = st.out.clone()
    used = np.unique(w.block_tables[w.block_tables >= 0])
    host_k = torch.empty((len(used),) + tuple(st.k_cache.shape[1:]), dtype=st.k_cache.dtype
                         ).pin_memory()
    host_v = torch.empty_like(host_k).pin_memory()
    binding.pkv_swap_blocks(st.k_cache, st.v_cache, host_k, host_v,
                            np.stack([used, np.arange(len(used))], 1))
    st.k_cache.fill_(float("nan"))
    st.v_cache.fill_(float("nan"))
    new_ids = np.random.default_rng(2).permutation(w.num_blocks)[:len(used)]
    binding.pkv_swap_blocks(host_k, host_v, st.k_cache, st.v_cache,
                            np.stack([np.arange(len(used)), new_ids], 1))
    remap = np.full(w.num_blocks, -1, np.int64)
    remap[used] = new_ids
    tables = np.where(w.block_tables >= 0, remap[np.maximum(w.block_tables, 0)], -1)
    st.block_tables.copy_(torch.from_numpy(tables.astype(np.int32)))
    st.decode()
    torch.cuda.synchronize()
    assert torch.equal(st.out.view(torch.int16), ref_out.view(torch.int16))
    assert binding.pkv_get_device_status() == 0


def test_swap_refuses_pageable_host_memory():
    dev = torch.zeros((4, 1, 16, 64), device="cuda")
    pageable = torch.zeros((4, 1, 16, 64))
    lib = binding.load()
    pairs = torch.tensor([[0, 1]], dtype=torch.int32, device="cuda")
    rc = lib.pkv_swap_blocks(dev.data_ptr(), dev.data_ptr(), 4, pageable.data_ptr(),
                             pageable.data_ptr(), 4, pairs.data_ptr(), 1, 1, 64, 16,
                             binding.PKV_F32, torch.cuda.current_stream().cuda_stream)
    assert rc == binding.PKV_ERR_INVALID_ARG
