"""Builds a workload's paged KV state on one GPU and runs decode steps.

Everything goes through the libpagedkv binding: the host block manager
decides slots, tables and copy-on-write pairs; pk_copy_blocks,
pk_reshape_and_cache and pk_paged_attention_decode do the device work. The
seeded inputs come from the ``workloads`` module.

A decode step (one pass of the hot path) is, in order:
  1. host: append one token to every sequence (pk_bm_append_batch), export
     the padded block tables and context lengths, and order the work
     (longest first, or a planned work list: DecodeState.plan);
  2. device: pk_copy_blocks for the step's copy-on-write pairs (if any),
     pk_reshape_and_cache of the new tokens' K/V, pk_paged_attention_decode.
"""
from __future__ import annotations

import dataclasses
from typing import List, Optional

import numpy as np

from . import (BlockManager, cache_desc, pk_attention_plan, pk_cascade_attention_decode,
               pk_cascade_workspace_size, pk_copy_blocks, pk_longest_first_order, pk_paged_attention_decode,
               pk_paged_attention_decode_append, pk_paged_attention_resolve_partition,
               pk_paged_attention_workspace_size, pk_reshape_and_cache)


def to_device(a: np.ndarray, dtype: str, device):
    """A numpy array of workload values (fp32, or bf16 bit patterns) as a CUDA tensor."""
    import torch
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32))
    return t.to(device)


def from_device(t) -> np.ndarray:
    """A CUDA tensor back as numpy (bf16 as uint16 bit patterns)."""
    import torch
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


@dataclasses.dataclass
class StepInputs:
    """Host-side inputs of one decode step."""
    step: int
    q: np.ndarray           # [S, Hq, d]
    k: np.ndarray           # [S, Hk, d]
    v: np.ndarray           # [S, Hk, d]
    slots: np.ndarray       # int64 [S]
    pairs: np.ndarray       # int64 [n, 2]
    tables: np.ndarray      # int32 [S, max_blocks]
    ctx_lens: np.ndarray    # int32 [S]
    order: np.ndarray       # int32 [S], launch order (longest first)

    @property
    def max_context_len(self) -> int:
        return int(self.ctx_lens.max())


class DecodeState:
    """A workload's pool, block manager and prefill, resident on one GPU."""

    def __init__(self, wl, device="cuda", extra_tokens: int = 0, alloc_order: Optional[np.ndarray] = None,
                 init_value: float = 0.0):
        """``alloc_order`` overrides the workload's block hand-out order;
        ``init_value`` fills the pools before the prefill (slots no token
        writes keep it)."""
        import torch
        self.wl = wl
        self.device = torch.device(device)
        self.torch_dtype = torch.float32 if wl.dtype == "f32" else torch.bfloat16
        order = wl.alloc_order() if alloc_order is None else alloc_order
        self.bm = BlockManager(wl.num_blocks, wl.block_size, order)
        shape = (wl.num_blocks, wl.block_size, wl.num_kv_heads, wl.head_dim)
        self.k_cache = torch.full(shape, init_value, dtype=self.torch_dtype, device=self.device)
        self.v_cache = torch.full(shape, init_value, dtype=self.torch_dtype, device=self.device)
        self.desc = cache_desc(self.k_cache)
        self.max_blocks = -(-(int(wl.ctx_lens.max()) + int(extra_tokens)) // wl.block_size)
        self.prefill_slots: List[np.ndarray] = []
        self.prefill_pairs: List[tuple] = []
        self.steps_done = 0
        self.prompt_tokens = 0   # prompt tokens admitted through the prefix cache
        self.cached_tokens = 0   # of which served by the cache
        self._prefill()

    def _prefill(self):
        import torch
        from workloads import prefill_plan
        wl = self.wl
        for op in prefill_plan(wl):
            if op[0] == "add":
                self.bm.add_seq(op[1])
            elif op[0] == "fork":
                self.bm.fork(op[1], op[2])
            elif op[0] == "free":
                self.bm.free_seq(op[1])
            elif op[0] == "admit":
                r = op[1]
                toks = wl.chat_tokens(r)
                n_cached = self.bm.add_seq_cached(r, toks)
                self.cached_tokens += n_cached
                self.prompt_tokens += len(toks)
                if len(toks) > n_cached:
                    slots, _ = self.bm.append(r, len(toks) - n_cached)
                    self.prefill_slots.append(slots)
                    k, v = wl.chat_kv(r, n_cached, len(toks))
                    pk_reshape_and_cache(to_device(k, wl.dtype, self.device), to_device(v, wl.dtype, self.device),
                                         torch.from_numpy(slots).to(self.device), self.k_cache, self.v_cache)
                self.bm.commit(r, toks)
            else:
                _, seq, n, src = op
                slots, cow = self.bm.append(seq, n)
                self.prefill_slots.append(slots)
                if cow is not None:
                    self.prefill_pairs.append(cow)
                    pk_copy_blocks(self.k_cache, self.v_cache,
                                   torch.tensor([cow], dtype=torch.int64, device=self.device))
                k, v = wl.prefix_kv(src[1]) if src[0] == "prefix" else wl.prefill_kv(src[1], n)
                pk_reshape_and_cache(to_device(k, wl.dtype, self.device), to_device(v, wl.dtype, self.device),
                                     torch.from_numpy(slots).to(self.device), self.k_cache, self.v_cache)

    # -- host side of a step --------------------------------------------------
    def prepare_step(self, step: Optional[int] = None) -> StepInputs:
        """Appends one token to every sequence on the host; returns the step's inputs."""
        wl = self.wl
        step = self.steps_done if step is None else step
        q, k, v = wl.step_inputs(step)
        slots, pairs = self.bm.append_batch(range(wl.num_seqs))
        tables, lens = self.bm.export_tables(range(wl.num_seqs), self.max_blocks)
        self.steps_done += 1
        return StepInputs(step, q, k, v, slots, pairs, tables, lens, pk_longest_first_order(lens))

    def upload(self, si: StepInputs) -> dict:
        """The step's inputs as device tensors."""
        import torch
        dev = self.device
        return {
            "q": to_device(si.q, self.wl.dtype, dev),
            "k": to_device(si.k, self.wl.dtype, dev),
            "v": to_device(si.v, self.wl.dtype, dev),
            "slots": torch.from_numpy(si.slots).to(dev),
            "pairs": torch.from_numpy(np.ascontiguousarray(si.pairs, dtype=np.int64).reshape(-1, 2)).to(dev),
            "tables": torch.from_numpy(si.tables).to(dev),
            "ctx_lens": torch.from_numpy(si.ctx_lens).to(dev),
            "order": torch.from_numpy(si.order).to(dev),
            "max_context_len": si.max_context_len,
        }

    # -- device side of a step -------------------------------------------------
    def workspace_bytes(self, max_context_len: int, partition_size: int) -> int:
        wl = self.wl
        return pk_paged_attention_workspace_size(wl.num_seqs, wl.num_q_heads, max_context_len, partition_size,
                                                 self.desc)

    def resolve_partition(self, max_context_len: int, partition_size: int) -> int:
        wl = self.wl
        return pk_paged_attention_resolve_partition(wl.num_seqs, wl.num_q_heads, max_context_len,
                                                    partition_size, self.desc)

    def alloc_workspace(self, max_context_len: int, partition_size: int):
        import torch
        n = self.workspace_bytes(max_context_len, partition_size)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=self.device) if n else None

    def new_out(self):
        import torch
        wl = self.wl
        return torch.empty((wl.num_seqs, wl.num_q_heads, wl.head_dim), dtype=self.torch_dtype,
                           device=self.device)

    def run_step(self, d: dict, out, workspace=None, partition_size: int = -1, impl: str = "auto",
                 stream=None):
        """Enqueues copy_blocks (if pairs), the scatter and the attention of one step."""
        if d["pairs"].shape[0]:
            pk_copy_blocks(self.k_cache, self.v_cache, d["pairs"], stream=stream)
        pk_reshape_and_cache(d["k"], d["v"], d["slots"], self.k_cache, self.v_cache, stream=stream)
        self.attention(d, out, workspace, partition_size, impl, stream)

    def plan(self, si: StepInputs, partition_size: int = -1):
        """The step's planned partition and work list (pk_attention_plan on the
        host lengths); the work list as a device tensor."""
        import torch
        part, items = pk_attention_plan(si.ctx_lens, self.wl.num_q_heads, self.desc, partition_size)
        return part, torch.from_numpy(items).to(self.device)

    def run_step_fused(self, d: dict, out, workspace=None, stream=None):
        """The step with its scatter fused into the attention (needs the plan's
        ``items`` and ``partition`` in ``d``): copy_blocks (if pairs), then
        pk_paged_attention_decode_append."""
        if d["pairs"].shape[0]:
            pk_copy_blocks(self.k_cache, self.v_cache, d["pairs"], stream=stream)
        pk_paged_attention_decode_append(out, d["q"], d["k"], d["v"], d["slots"], self.k_cache, self.v_cache,
                                         d["tables"], d["ctx_lens"], self.wl.scale, d["max_context_len"],
                                         d["partition"], d["items"], workspace, stream)

    def attention(self, d: dict, out, workspace=None, partition_size: int = -1, impl: str = "auto",
                  stream=None, ordered: bool = True):
        """The attention call; ``ordered`` launches the longest work first: by
        the step's work list when ``d`` holds one (``items``), else by the
        sequence order."""
        items = d.get("items") if ordered else None
        if items is not None and "partition" in d:
            partition_size = d["partition"]   # the plan's partition goes with its work list
        pk_paged_attention_decode(out, d["q"], self.k_cache, self.v_cache, d["tables"], d["ctx_lens"],
                                  self.wl.scale, d["max_context_len"], partition_size, workspace, impl,
                                  stream, seq_order=d.get("order") if ordered and items is None else None,
                                  work_items=items)

    # -- cascade (shared-prefix) attention --------------------------------------
    def cascade_groups(self, min_prefix_blocks: int = 1, max_group_size: Optional[int] = None) -> dict:
        """The batch's shared-prefix groups as device tensors (host block manager)."""
        import torch
        wl = self.wl
        mg = max(1, 16 // wl.group) if max_group_size is None else int(max_group_size)
        g = self.bm.prefix_groups(range(wl.num_seqs), mg, min_prefix_blocks)
        dev = self.device
        out = dict(g)
        for k in ("offsets", "members", "prefix_len", "seq_prefix_len"):
            arr = g[k] if len(g[k]) else np.zeros(1, np.int32)
            out[k] = torch.from_numpy(np.ascontiguousarray(arr, dtype=np.int32)).to(dev)
        return out

    def alloc_cascade_workspace(self, max_context_len: int, groups: dict, partition_size: int = -1):
        import torch
        wl = self.wl
        n = pk_cascade_workspace_size(wl.num_seqs, wl.num_q_heads, max_context_len, groups["num_groups"],
                                      groups["max_prefix_len"], partition_size, self.desc)
        return torch.empty(max(n, 16), dtype=torch.uint8, device=self.device)

    def attention_cascade(self, d: dict, out, groups: dict, workspace, partition_size: int = -1, stream=None,
                          ordered: bool = True):
        pk_cascade_attention_decode(out, d["q"], self.k_cache, self.v_cache, d["tables"], d["ctx_lens"],
                                    self.wl.scale, d["max_context_len"], groups, partition_size, workspace,
                                    d.get("order") if ordered else None, stream)
