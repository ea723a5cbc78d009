"""Test helpers: golden-file parsing and the oracle side of a workload.

The oracle side replays a workload's setup and step with the oracle's own
reshape_and_cache / copy_blocks on host buffers, then runs the oracle's decode.
"""
from __future__ import annotations

import os

import numpy as np

import oracle
from paged_kv_cache_87_gb300 import inputs

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name: str) -> dict:
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (x.strip() for x in line.split("=", 1))
            out[k] = v
    return out


def ints(s: str) -> list[int]:
    return [int(x) for x in s.split()]


def to_f64(a: np.ndarray, dtype: str) -> np.ndarray:
    """Exact fp64 values of stored elements, via numpy / torch (not the oracle's codecs)."""
    if dtype == "f32":
        return a.astype(np.float64)
    if dtype == "f16":
        return a.astype(np.float64)
    if dtype == "bf16":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
        return t.to(torch.float64).numpy()
    if dtype == "e4m3":
        import torch
        t = torch.from_numpy(np.ascontiguousarray(a)).view(torch.float8_e4m3fn)
        return t.to(torch.float64).numpy()
    raise ValueError(dtype)


def oracle_caches(w: inputs.Workload, *, with_step: bool = True, poison: bool = True):
    """Host K/V pools after the workload's setup (and its step's writes) by the oracle."""
    kc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    vc = inputs.poison_array(w.cache_shape, w.kv_dtype)
    if not poison:
        kc[...] = 0
        vc[...] = 0
    common = dict(num_kv_heads=w.num_kv_heads, head_dim=w.head_dim, block_size=w.block_size,
                  num_blocks=w.num_blocks)
    ops = list(w.setup)
    if with_step:
        if len(w.step_pairs):
            ops.append(("copy", w.step_pairs))
        ops.append(("reshape", w.new_vec, w.new_slots))
    for op in ops:
        if op[0] == "reshape":
            idx, slots = op[1], op[2]
            oracle.reshape_and_cache(np.ascontiguousarray(w.key[idx]),
                                     np.ascontiguousarray(w.value[idx]), kc, vc, slots,
                                     src_dtype=w.src_dtype, kv_dtype=w.kv_dtype,
                                     kv_scale=w.kv_scale, **common)
        else:
            oracle.copy_blocks(kc, vc, op[1], kv_dtype=w.kv_dtype, **common)
    return kc, vc


def oracle_decode(w: inputs.Workload, kc, vc, sel=None, nthreads=1, context_lens=None,
                  block_tables=None):
    return oracle.paged_decode_attention(
        w.query, kc, vc, w.block_tables if block_tables is None else block_tables,
        w.context_lens if context_lens is None else context_lens,
        num_q_heads=w.num_q_heads, num_kv_heads=w.num_kv_heads, head_dim=w.head_dim,
        block_size=w.block_size, num_blocks=w.num_blocks, scale=w.scale, q_dtype=w.q_dtype,
        kv_dtype=w.kv_dtype, kv_scale=w.kv_scale, sel=sel, nthreads=nthreads)


def logical_kv_f64(w: inputs.Workload, s: int):
    """Table-free logical K/V of sequence s in fp64 (from the generator's record).

    For an e4m3 cache this is the value the cache holds after quantisation, so
    callers that need it pass the dequantised rows instead.
    """
    idx = w.seq_tokens[s]
    return to_f64(w.key[idx], w.src_dtype), to_f64(w.value[idx], w.src_dtype)


# ------------------------------------------------------------- GPU side --

# max abs error allowed against the fp64 oracle, by the type that limits precision
TOL = {"f32": 1e-4, "f16": 5e-3, "bf16": 1.6e-2, "e4m3": 1.6e-2}


def tolerance(w: inputs.Workload) -> float:
    return TOL["e4m3"] if w.kv_dtype == "e4m3" else TOL[w.q_dtype]


def gpu_state(w: inputs.Workload, steps: int = 1, prefix: bool | None = None):
    """DeviceState after the workload's setup and `steps` hot-path steps.

    prefix: use the prefix-aware decode (default: for shared-prompt workloads)."""
    import torch
    from paged_kv_cache_87_gb300 import binding
    from paged_kv_cache_87_gb300.session import DeviceState
    st = DeviceState(w, "cuda", prefix=prefix)
    st.run_setup()
    for _ in range(steps):
        st.step()
    torch.cuda.synchronize()
    assert binding.pkv_get_device_status() == 0
    return st


def relabel_blocks(w: inputs.Workload, perm: np.ndarray) -> inputs.Workload:
    """The same workload with physical block b renamed perm[b] everywhere."""
    import dataclasses
    B = w.block_size

    def slots(a):
        a = np.asarray(a, np.int64)
        return np.where(a >= 0, perm[np.maximum(a, 0) // B] * B + np.maximum(a, 0) % B, a)

    def pairs(p):
        return perm[np.asarray(p, np.int64)].astype(np.int32).reshape(-1, 2)

    setup = [(op[0], op[1], slots(op[2])) if op[0] == "reshape" else (op[0], pairs(op[1]))
             for op in w.setup]
    tables = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1)
    return dataclasses.replace(w, setup=setup, step_pairs=pairs(w.step_pairs),
                               new_slots=slots(w.new_slots),
                               block_tables=tables.astype(np.int32))
