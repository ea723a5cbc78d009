"""GPU parity of reshape_and_cache and copy_blocks: byte-exact against the oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_87_gb300 import binding, inputs
from paged_kv_cache_87_gb300.session import host_tensor, poisoned_cache, to_numpy_storage

pytestmark = pytest.mark.gpu


def _pool_pair(shape, dtype):
    return (inputs.poison_array(shape, dtype), inputs.poison_array(shape, dtype),
            poisoned_cache(shape, dtype, "cuda"), poisoned_cache(shape, dtype, "cuda"))


@pytest.mark.parametrize("src,kv,d,B", [
    ("f32", "f32", 64, 16), ("f16", "f16", 128, 16), ("bf16", "bf16", 128, 32),
    ("bf16", "bf16", 64, 8), ("bf16", "e4m3", 128, 16), ("f16", "e4m3", 64, 32),
    ("f32", "e4m3", 128, 8),
])
def test_reshape_and_cache_bit_exact(src, kv, d, B):
    rng = np.random.default_rng(100 + d + B)
    H, NB = 4, 37
    T = min(300, (NB - 2) * B)
    key = inputs.draw_normal(rng, (T, H, d), src)
    val = inputs.draw_normal(rng, (T, H, d), src)
    # scattered slots, some padding (-1), guard blocks 0 and NB-1 never written
    slots = rng.permutation(np.arange(B, (NB - 1) * B))[:T].astype(np.int64)
    slots[rng.random(T) < 0.1] = -1
    scale = 2.0 ** -5 if kv == "e4m3" else 1.0
    hk, hv, dk, dv = _pool_pair((NB, H, B, d), kv)
    oracle.reshape_and_cache(key, val, hk, hv, slots, num_kv_heads=H, head_dim=d, block_size=B,
                             num_blocks=NB, src_dtype=src, kv_dtype=kv, kv_scale=scale)
    binding.pkv_reshape_and_cache(host_tensor(key, src).cuda(), host_tensor(val, src).cuda(), dk,
                                  dv, torch.from_numpy(slots).cuda(), kv_scale=scale)
    assert binding.pkv_get_device_status() == 0
    gk, gv = to_numpy_storage(dk, kv), to_numpy_storage(dv, kv)
    assert gk.view(np.uint8).tobytes() == hk.view(np.uint8).tobytes()
    assert gv.view(np.uint8).tobytes() == hv.view(np.uint8).tobytes()


def test_e4m3_encode_boundaries_bit_exact():
    """Midpoints, neighbours, saturation and subnormals, through the GPU write path."""
    pos = [oracle.e4m3_to_double(c) for c in range(0x7F)]
    vals = []
    for a, b in zip(pos[:-1], pos[1:]):
        mid = np.float32((a + b) / 2)
        vals += [mid, np.nextafter(mid, np.float32(0)), np.nextafter(mid, np.float32(np.inf)), a]
    vals += [448.0, 449.0, 463.99, 464.0, 465.0, 1e5, np.inf, 2.0 ** -10, 2.0 ** -12, 0.0]
    v = np.array(vals, np.float32)
    v = np.concatenate([v, -v])
    d, H, B = 128, 1, 16
    n = -(-v.size // d) * d
    x = np.zeros(n, np.float32)
    x[:v.size] = v
    T = n // d
    key = x.reshape(T, H, d)
    slots = np.arange(T, dtype=np.int64)
    NB = -(-T // B)
    hk, hv, dk, dv = _pool_pair((NB, H, B, d), "e4m3")
    oracle.reshape_and_cache(key, key, hk, hv, slots, num_kv_heads=H, head_dim=d, block_size=B,
                             num_blocks=NB, src_dtype="f32", kv_dtype="e4m3", kv_scale=1.0)
    kt = torch.from_numpy(key).cuda()
    binding.pkv_reshape_and_cache(kt, kt, dk, dv, torch.from_numpy(slots).cuda(), kv_scale=1.0)
    assert (to_numpy_storage(dk, "e4m3") == hk).all()


def test_reshape_flags_slots_outside_the_pool():
    H, d, B, NB = 2, 64, 16, 4
    key = torch.randn(3, H, d, device="cuda")
    dk, dv = poisoned_cache((NB, H, B, d), "f32", "cuda"), poisoned_cache((NB, H, B, d), "f32",
                                                                          "cuda")
    slots = torch.tensor([0, NB * B, 5], dtype=torch.int64, device="cuda")   # middle one bad
    binding.pkv_reshape_and_cache(key, key, dk, dv, slots)
    assert binding.pkv_get_device_status() == binding.DEV_BAD_SLOT
    assert torch.equal(dk[0, :, 0], key[0]) and torch.equal(dk[0, :, 5], key[2])
    assert binding.pkv_get_device_status() == 0   # read clears


@pytest.mark.parametrize("kv,d,B,H", [("e4m3", 128, 16, 8), ("f16", 128, 16, 40),
                                      ("f32", 64, 8, 3)])
def test_copy_blocks_bit_exact(kv, d, B, H):
    rng = np.random.default_rng(7)
    NB = 50
    nbytes = NB * H * B * d * inputs.DTYPE_BYTES[kv]
    raw_k = rng.integers(0, 256, nbytes, dtype=np.uint8)
    raw_v = rng.integers(0, 256, nbytes, dtype=np.uint8)
    hk = raw_k.view(inputs.NP_CONTAINER[kv]).reshape(NB, H, B, d).copy()
    hv = raw_v.view(inputs.NP_CONTAINER[kv]).reshape(NB, H, B, d).copy()
    dk = host_tensor(hk, kv).cuda()
    dv = host_tensor(hv, kv).cuda()
    ids = rng.permutation(NB)
    pairs = np.stack([ids[:20], ids[20:40]], 1).astype(np.int32)
    oracle.copy_blocks(hk, hv, pairs, num_kv_heads=H, head_dim=d, block_size=B, num_blocks=NB,
                       kv_dtype=kv)
    binding.pkv_copy_blocks(dk, dv, pairs)
    assert binding.pkv_get_device_status() == 0
    assert to_numpy_storage(dk, kv).view(np.uint8).tobytes() == hk.view(np.uint8).tobytes()
    assert to_numpy_storage(dv, kv).view(np.uint8).tobytes() == hv.view(np.uint8).tobytes()


def test_copy_blocks_flags_ids_outside_the_pool():
    NB, H, B, d = 6, 2, 16, 64
    dk = torch.randn(NB, H, B, d, device="cuda")
    dv = torch.randn(NB, H, B, d, device="cuda")
    k0 = dk.clone()
    pairs = torch.tensor([[1, 2], [3, NB]], dtype=torch.int32, device="cuda")
    binding.pkv_copy_blocks(dk, dv, pairs)        # device pairs: not host-validated
    assert binding.pkv_get_device_status() == binding.DEV_BAD_PAIR
    assert torch.equal(dk[2], k0[1]) and torch.equal(dk[3], k0[3])


def test_copy_blocks_rejects_overlapping_pairs_on_host():
    dk = torch.zeros(4, 1, 8, 64, device="cuda")
    with pytest.raises(ValueError):
        binding.pkv_copy_blocks(dk, dk.clone(), [[0, 1], [1, 2]])
