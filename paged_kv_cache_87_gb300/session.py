"""Device-side state of a workload: the pool, tables and step inputs in HBM.

Allocation is torch's (device memory and streams are torch's job here); every
write into the pool and the decode itself go through the C ABI (``binding``).
"""
from __future__ import annotations

import numpy as np
import torch

from . import binding
from .inputs import MultiQueryWorkload, Workload

TORCH_DTYPE = {"f32": torch.float32, "f16": torch.float16, "bf16": torch.bfloat16,
               "e4m3": torch.float8_e4m3fn}


def host_tensor(a: np.ndarray, dtype: str) -> torch.Tensor:
    """Wrap a numpy storage array (bf16 as uint16, e4m3 as uint8) as a torch tensor."""
    a = np.ascontiguousarray(a)
    if dtype == "bf16":
        return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16)
    if dtype == "e4m3":
        return torch.from_numpy(a.view(np.uint8)).view(torch.float8_e4m3fn)
    return torch.from_numpy(a)


def poisoned_cache(shape, dtype: str, device) -> torch.Tensor:
    t = torch.empty(shape, dtype=TORCH_DTYPE[dtype], device=device)
    if dtype == "e4m3":
        t.view(torch.uint8).fill_(0x7F)        # E4M3 NaN
    else:
        t.fill_(float("nan"))
    return t


def to_numpy_storage(t: torch.Tensor, dtype: str) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if dtype == "bf16":
        return t.view(torch.int16).numpy().view(np.uint16)
    if dtype == "e4m3":
        return t.view(torch.uint8).numpy()
    return t.numpy()


class DeviceState:
    """A workload's pool and step inputs resident on one CUDA device."""

    def __init__(self, w: Workload, device="cuda", keep_vectors: bool = False,
                 prefix: bool | None = None):
        self.w = w
        # prefix-aware decode for workloads built with shared prompts
        self.prefix = w.group_of_seq is not None if prefix is None else prefix
        self.device = torch.device(device)
        dev = self.device
        self.k_cache = poisoned_cache(w.cache_shape, w.kv_dtype, dev)
        self.v_cache = poisoned_cache(w.cache_shape, w.kv_dtype, dev)
        self.query = host_tensor(w.query, w.q_dtype).to(dev)
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.context_lens = torch.from_numpy(w.context_lens).to(dev)
        self.step_pairs = torch.from_numpy(np.ascontiguousarray(w.step_pairs, np.int32)).to(dev)
        self.new_key = host_tensor(w.key[w.new_vec], w.src_dtype).to(dev)
        self.new_value = host_tensor(w.value[w.new_vec], w.src_dtype).to(dev)
        self.new_slots = torch.from_numpy(w.new_slots).to(dev)
        self.out = torch.empty_like(self.query)
        self.workspace = torch.empty(
            max(256, binding.pkv_decode_workspace_bytes(
                w.num_seqs, w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size,
                w.max_context_len, w.kv_dtype)), dtype=torch.uint8, device=dev)
        self.keep_vectors = keep_vectors

    # ---------------------------------------------------------------- setup --
    def run_setup(self, chunk_tokens: int = 1 << 20) -> None:
        """Fill the pool: the workload's prefill writes and fork copies, in order."""
        w = self.w
        for op in w.setup:
            if op[0] == "copy":
                binding.pkv_copy_blocks(self.k_cache, self.v_cache, op[1])
                continue
            idx, slots = op[1], op[2]
            for a in range(0, len(idx), chunk_tokens):
                sl = slice(a, a + chunk_tokens)
                k = host_tensor(w.key[idx[sl]], w.src_dtype).to(self.device)
                v = host_tensor(w.value[idx[sl]], w.src_dtype).to(self.device)
                s = torch.from_numpy(np.ascontiguousarray(slots[sl])).to(self.device)
                binding.pkv_reshape_and_cache(k, v, self.k_cache, self.v_cache, s,
                                              kv_scale=w.kv_scale)
        torch.cuda.synchronize(self.device)

    # ----------------------------------------------------------------- step --
    def copy_step(self, stream=None) -> None:
        if self.step_pairs.numel():
            binding.pkv_copy_blocks(self.k_cache, self.v_cache, self.step_pairs, stream=stream)

    def append_step(self, stream=None) -> None:
        binding.pkv_reshape_and_cache(self.new_key, self.new_value, self.k_cache, self.v_cache,
                                      self.new_slots, kv_scale=self.w.kv_scale, stream=stream)

    def decode(self, stream=None, out=None) -> torch.Tensor:
        w = self.w
        return binding.pkv_paged_decode_attention(
            self.query, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
            w.max_context_len, w.scale, kv_scale=w.kv_scale, workspace=self.workspace,
            out=self.out if out is None else out, stream=stream, prefix=self.prefix)

    def step(self, stream=None) -> torch.Tensor:
        """One pass of the hot path: copy-on-write, append the new tokens, decode."""
        self.copy_step(stream)
        self.append_step(stream)
        return self.decode(stream)

    def prepare(self, stream=None) -> tuple:
        """The step's calls with their arguments marshalled once, for `stream`:
        (copy-on-write + append calls, decode call).  Re-prepare after the inputs
        move (pack_step_inputs)."""
        w = self.w
        pre = []
        if self.step_pairs.numel():
            pre.append(binding.prepare_copy_blocks(self.k_cache, self.v_cache, self.step_pairs,
                                                   stream=stream))
        pre.append(binding.prepare_reshape_and_cache(self.new_key, self.new_value, self.k_cache,
                                                     self.v_cache, self.new_slots,
                                                     kv_scale=w.kv_scale, stream=stream))
        dec = binding.prepare_paged_decode_attention(
            self.query, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
            w.max_context_len, w.scale, kv_scale=w.kv_scale, workspace=self.workspace,
            out=self.out, stream=stream, prefix=self.prefix)
        return tuple(pre), dec

    def out_f64(self) -> np.ndarray:
        return self.out.detach().to(torch.float64).cpu().numpy()

    STEP_INPUTS = ("query", "new_key", "new_value", "new_slots", "context_lens",
                   "block_tables", "step_pairs")

    def pack_step_inputs(self) -> tuple[torch.Tensor, torch.Tensor]:
        """Move the step's inputs into one device buffer and return it with a pinned host
        buffer of the same layout holding their values.

        Each input becomes a 256-byte aligned view of the device buffer, so a single
        host-to-device copy of the host buffer refreshes every input of a step (instead
        of one small copy per tensor)."""
        return pack_views(self, self.STEP_INPUTS)


def pack_views(obj, names) -> tuple[torch.Tensor, torch.Tensor]:
    """Replace the tensors obj.<name> by views of one device byte buffer (256-byte
    aligned offsets, values kept); returns (pinned host copy, device buffer)."""
    tensors = [getattr(obj, n) for n in names]
    offs, off = [], 0
    for t in tensors:
        off = (off + 255) // 256 * 256
        offs.append(off)
        off += t.numel() * t.element_size()
    dev = torch.empty(max(off, 256), dtype=torch.uint8, device=tensors[0].device)
    host = torch.empty(dev.numel(), dtype=torch.uint8).pin_memory()
    host.zero_()
    for n, t, o in zip(names, tensors, offs):
        nb = t.numel() * t.element_size()
        view = dev[o:o + nb].view(t.dtype).view(t.shape)
        view.copy_(t)
        if nb:
            host[o:o + nb].copy_(t.detach().cpu().contiguous().view(-1).view(torch.uint8))
        setattr(obj, n, view)
    torch.cuda.synchronize(dev.device)
    return host, dev


class MultiQueryState:
    """A multi-query workload's pool, tables and queries resident on one CUDA device.

    ``run_setup`` writes the tokens cached before the step; ``step`` writes the
    queries' own K/V rows and runs the multi-query attention.
    """

    def __init__(self, w: MultiQueryWorkload, device="cuda"):
        self.w = w
        dev = self.device = torch.device(device)
        self.k_cache = poisoned_cache(w.cache_shape, w.kv_dtype, dev)
        self.v_cache = poisoned_cache(w.cache_shape, w.kv_dtype, dev)
        self.query = host_tensor(w.query, w.q_dtype).to(dev)
        self.block_tables = torch.from_numpy(w.block_tables).to(dev)
        self.context_lens = torch.from_numpy(w.context_lens).to(dev)
        self.query_start = torch.from_numpy(w.query_start).to(dev)
        self.tree = (torch.from_numpy(w.tree.view(np.int64)).to(dev)
                     if getattr(w, "tree", None) is not None else None)
        self.new_key = host_tensor(w.key[w.new_idx], w.kv_dtype).to(dev)
        self.new_value = host_tensor(w.value[w.new_idx], w.kv_dtype).to(dev)
        self.new_slots = torch.from_numpy(np.ascontiguousarray(w.slots[w.new_idx])).to(dev)
        self.out = torch.empty_like(self.query)
        self.workspace = torch.empty(max(256, binding.pkv_multi_query_workspace_bytes(w.num_seqs)),
                                     dtype=torch.uint8, device=dev)

    def run_setup(self, chunk_tokens: int = 1 << 20) -> None:
        w = self.w
        idx = w.prior_idx
        for a in range(0, len(idx), chunk_tokens):
            sl = idx[a:a + chunk_tokens]
            k = host_tensor(w.key[sl], w.kv_dtype).to(self.device)
            v = host_tensor(w.value[sl], w.kv_dtype).to(self.device)
            s = torch.from_numpy(np.ascontiguousarray(w.slots[sl])).to(self.device)
            binding.pkv_reshape_and_cache(k, v, self.k_cache, self.v_cache, s)
        torch.cuda.synchronize(self.device)

    def append_step(self, stream=None) -> None:
        binding.pkv_reshape_and_cache(self.new_key, self.new_value, self.k_cache, self.v_cache,
                                      self.new_slots, stream=stream)

    def attend(self, stream=None, out=None) -> torch.Tensor:
        w = self.w
        if self.tree is not None:
            return binding.pkv_paged_tree_attention(
                self.query, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
                self.query_start, self.tree, w.max_context_len, w.scale,
                workspace=self.workspace, out=self.out if out is None else out, stream=stream)
        return binding.pkv_paged_multi_query_attention(
            self.query, self.k_cache, self.v_cache, self.block_tables, self.context_lens,
            self.query_start, w.max_context_len, w.scale, workspace=self.workspace,
            out=self.out if out is None else out, stream=stream)

    def step(self, stream=None) -> torch.Tensor:
        """One pass: write the queries' own K/V, then attend."""
        self.append_step(stream)
        return self.attend(stream)

    def pack_step_inputs(self) -> tuple[torch.Tensor, torch.Tensor]:
        """As DeviceState.pack_step_inputs: the step's inputs as views of one device
        buffer, plus a pinned host buffer of the same layout."""
        names = ["query", "new_key", "new_value", "new_slots", "context_lens", "query_start",
                 "block_tables"] + (["tree"] if self.tree is not None else [])
        return pack_views(self, names)

    def out_f64(self) -> np.ndarray:
        return self.out.detach().to(torch.float64).cpu().numpy()
