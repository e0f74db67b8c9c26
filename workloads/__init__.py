"""Seeded synthetic inputs for the paged decode-attention workloads.

This module only draws numbers: sequence lengths, the order in which a pool
hands out its physical blocks, and the query / key / value vectors. It holds
none of the method's arithmetic (no block manager, no address translation, no
attention), so the CUDA path and the CPU oracle can both consume its output
without sharing any code with each other.

Workloads (shapes follow the pages' examples; all data is synthetic):

* ``tiny``   4 sequences, context lengths {1, 17, 33, 100}, 16-token blocks,
             8 query heads = 8 KV heads, head_dim 64, fp32, 64-block pool.
* ``mha7b``  Llama-2-7B-like layer: 64 sequences, 32 = 32 heads, head_dim 128,
             bf16, 16-token blocks, context uniform in [128, 2048], 8192 blocks.
* ``gqa8b``  Llama-3-8B-like layer: 256 sequences, 32 query / 8 KV heads,
             head_dim 128, bf16, 16-token blocks, prompt uniform in [32, 512]
             plus a lognormal output length (mean 200, sigma 1, capped at 4096),
             32768 blocks.
* ``long``   8 sequences of 32768 tokens, 64 query / 8 KV heads, head_dim 128,
             bf16, 16-token blocks in a 20000-block pool, 512-token partitions.
* ``prefix`` 32 groups of 4 parallel samples sharing a 2000-token prompt, then
             1..500 divergent tokens each, 32 / 8 heads, head_dim 128, bf16,
             block size 8, 16 or 32, a pool of 524288 slots.
* ``mixed``  one long request among short ones: 128 sequences, 32 query / 8 KV
             heads, head_dim 128, bf16, 16-token blocks; 127 contexts uniform in
             [256, 1024] and sequence 37 at 32768 tokens; 12288 blocks.
* ``chat``   a chat server's decode batch: 128 requests, each one of 4 system
             prompts (1000, 1536, 2000, 600 tokens; popularity 1 : 1/2 : 1/3 :
             1/4) followed by a lognormal user turn (mean 200, sigma 1, capped
             at 2000), admitted through a prefix cache after 32 earlier
             requests that have already finished; 32 / 8 heads, head_dim 128,
             bf16, 16-token blocks, 32768 blocks. Token ids are drawn from a
             32000-word vocabulary; the K/V of a system-prompt position depend
             only on the prompt and the position, those of the user turn on the
             request.

Every context length is the length *after* the step's new token is appended.
"""
from __future__ import annotations

import dataclasses
import math
from typing import List, Optional

import numpy as np

__all__ = [
    "Workload",
    "make_workload",
    "WORKLOAD_NAMES",
    "f32_to_bf16_bits",
    "bf16_bits_to_f32",
    "normal_values",
    "allocator_trace",
    "ALLOCATOR_TRACES",
]

WORKLOAD_NAMES = ("tiny", "mha7b", "gqa8b", "long", "prefix", "chat", "mixed")


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round finite fp32 values to bfloat16 (round to nearest, ties to even).

    Returns the 16-bit patterns as ``uint16``. This is input preparation: the
    bf16 workloads are defined by these bits, and both sides read them.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    if not np.isfinite(x).all():
        raise ValueError("bf16 rounding of the inputs expects finite values")
    # For finite values the sum stays below 2**32, so uint32 arithmetic is exact.
    r = (u >> 16) & 1
    r += u
    r += 0x7FFF
    r >>= 16
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to fp32 (exact: bf16 is the top half of fp32)."""
    return (np.ascontiguousarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_values(rng: np.random.Generator, shape, dtype: str) -> np.ndarray:
    """N(0, 1) values in the workload's storage type.

    ``dtype`` is ``"f32"`` (returns float32) or ``"bf16"`` (returns the uint16
    bit patterns of the fp32 draw rounded to bf16).
    """
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if dtype == "f32":
        return x
    if dtype == "bf16":
        return f32_to_bf16_bits(x)
    raise ValueError(f"unknown dtype {dtype!r}")


@dataclasses.dataclass
class Workload:
    """One seeded decode workload.

    ``ctx_lens[s]`` is sequence s's context length after the step token.
    ``prefix_groups`` / ``prefix_len`` are non-zero only for ``prefix``: then
    sequences ``g*n .. g*n+n-1`` form group g, whose first member holds the
    shared prompt and whose others are forked from it.
    """

    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    dtype: str  # "f32" | "bf16"
    num_blocks: int
    ctx_lens: np.ndarray  # int64 [S]
    seed: int
    partition_size: int = 512
    prefix_groups: int = 0
    prefix_n: int = 0
    prefix_len: int = 0
    chat_prompt_lens: Optional[np.ndarray] = None  # system prompt lengths (chat)
    chat_choice: Optional[np.ndarray] = None       # prompt of each request, batch then retired
    chat_retired: int = 0                          # earlier requests, ids num_seqs ..
    memo: Optional[dict] = dataclasses.field(default=None, repr=False, compare=False)

    def enable_memo(self) -> "Workload":
        """Keep generated token data so a second consumer does not redraw it."""
        if self.memo is None:
            self.memo = {}
        return self

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def esz(self) -> int:
        return 4 if self.dtype == "f32" else 2

    @property
    def np_dtype(self):
        return np.float32 if self.dtype == "f32" else np.uint16

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def alloc_order(self) -> np.ndarray:
        """The order in which the pool hands out blocks (first entry first)."""
        rng = np.random.default_rng(self.seed + 1000)
        return rng.permutation(self.num_blocks).astype(np.int32)

    # ---- token data -------------------------------------------------------
    def prefill_kv(self, seq: int, n_tokens: int):
        """K and V for the first ``n_tokens`` private tokens of sequence ``seq``.

        Shape ``[n_tokens, Hk, d]`` each. For ``prefix`` these are the
        sequence's divergent tokens (the shared prompt comes from
        :meth:`prefix_kv`).
        """
        key = ("prefill", seq, n_tokens)
        if self.memo is not None and key in self.memo:
            return self.memo[key]
        rng = np.random.default_rng([self.seed, 1, seq])
        shape = (n_tokens, self.num_kv_heads, self.head_dim)
        k = normal_values(rng, shape, self.dtype)
        v = normal_values(rng, shape, self.dtype)
        if self.memo is not None:
            self.memo[key] = (k, v)
        return k, v

    def prefix_kv(self, group: int):
        """K and V of group ``group``'s shared prompt, ``[prefix_len, Hk, d]``."""
        key = ("prefix", group)
        if self.memo is not None and key in self.memo:
            return self.memo[key]
        rng = np.random.default_rng([self.seed, 3, group])
        shape = (self.prefix_len, self.num_kv_heads, self.head_dim)
        k = normal_values(rng, shape, self.dtype)
        v = normal_values(rng, shape, self.dtype)
        if self.memo is not None:
            self.memo[key] = (k, v)
        return k, v

    # ---- chat requests (token ids and their K/V) ----------------------------
    def chat_user_len(self, req: int) -> int:
        """Length of request ``req``'s user turn (batch requests end one token
        before the step token; retired requests have their own draw)."""
        if req < self.num_seqs:
            return int(self.ctx_lens[req]) - 1 - int(self.chat_prompt_lens[self.chat_choice[req]])
        rng = np.random.default_rng([self.seed, 6, req])
        return int(_lognormal_outputs(rng, 1, 200.0, 1.0, 2000)[0])

    def chat_tokens(self, req: int) -> np.ndarray:
        """Token ids of request ``req``'s prompt: system prompt, then user turn (int32)."""
        p = int(self.chat_choice[req])
        sys_ids = np.random.default_rng([self.seed, 4, p]).integers(0, 32000, int(self.chat_prompt_lens[p]))
        user = np.random.default_rng([self.seed, 5, req]).integers(0, 32000, self.chat_user_len(req))
        return np.concatenate([sys_ids, user]).astype(np.int32)

    def chat_kv(self, req: int, start: int, end: int):
        """K and V ``[end - start, Hk, d]`` of positions [start, end) of request ``req``."""
        p = int(self.chat_choice[req])
        S = int(self.chat_prompt_lens[p])
        shape = (self.num_kv_heads, self.head_dim)
        key_s, key_u = ("chat_sys", p), ("chat_user", req)
        if self.memo is not None and key_s in self.memo:
            ks, vs = self.memo[key_s]
        else:
            rng = np.random.default_rng([self.seed, 7, p])
            ks, vs = normal_values(rng, (S,) + shape, self.dtype), normal_values(rng, (S,) + shape, self.dtype)
            if self.memo is not None:
                self.memo[key_s] = (ks, vs)
        if self.memo is not None and key_u in self.memo:
            ku, vu = self.memo[key_u]
        else:
            n = self.chat_user_len(req)
            rng = np.random.default_rng([self.seed, 8, req])
            ku, vu = normal_values(rng, (n,) + shape, self.dtype), normal_values(rng, (n,) + shape, self.dtype)
            if self.memo is not None:
                self.memo[key_u] = (ku, vu)
        return np.concatenate([ks, ku])[start:end], np.concatenate([vs, vu])[start:end]

    def step_inputs(self, step: int):
        """Query ``[S, Hq, d]`` and the new token's K, V ``[S, Hk, d]`` of a step."""
        rng = np.random.default_rng([self.seed, 2, step])
        q = normal_values(rng, (self.num_seqs, self.num_q_heads, self.head_dim), self.dtype)
        k = normal_values(rng, (self.num_seqs, self.num_kv_heads, self.head_dim), self.dtype)
        v = normal_values(rng, (self.num_seqs, self.num_kv_heads, self.head_dim), self.dtype)
        return q, k, v

    def kv_bytes(self, ctx_lens: Optional[np.ndarray] = None) -> int:
        """Algorithmic K+V bytes one decode step must read: sum ctx * Hk * d * esz * 2."""
        c = self.ctx_lens if ctx_lens is None else ctx_lens
        return int(np.sum(c, dtype=np.int64)) * self.num_kv_heads * self.head_dim * self.esz * 2

    def describe(self) -> dict:
        return {
            "workload": self.name,
            "num_seqs": self.num_seqs,
            "num_q_heads": self.num_q_heads,
            "num_kv_heads": self.num_kv_heads,
            "head_dim": self.head_dim,
            "block_size": self.block_size,
            "dtype": self.dtype,
            "num_blocks": self.num_blocks,
            "ctx_mean": float(np.mean(self.ctx_lens)),
            "ctx_max": int(np.max(self.ctx_lens)),
            "seed": self.seed,
        }


def _lognormal_outputs(rng: np.random.Generator, n: int, mean: float, sigma: float, cap: int) -> np.ndarray:
    mu = math.log(mean) - sigma * sigma / 2.0
    x = rng.lognormal(mean=mu, sigma=sigma, size=n)
    return np.clip(np.rint(x), 1, cap).astype(np.int64)


def make_workload(name: str, block_size: Optional[int] = None, num_seqs: Optional[int] = None) -> Workload:
    """Build a named workload. ``block_size`` applies to ``prefix`` (8/16/32).

    ``num_seqs`` truncates the batch (the first sequences, same lengths and
    data) for reduced-size cases; ``prefix`` truncates by whole groups.
    """
    if name == "tiny":
        wl = Workload("tiny", 4, 8, 8, 64, 16, "f32", 64,
                      np.array([1, 17, 33, 100], dtype=np.int64), seed=1131)
    elif name == "mha7b":
        seed = 1132
        rng = np.random.default_rng([seed, 0])
        ctx = rng.integers(128, 2049, size=64).astype(np.int64)
        wl = Workload("mha7b", 64, 32, 32, 128, 16, "bf16", 8192, ctx, seed=seed)
    elif name == "gqa8b":
        seed = 1133
        rng = np.random.default_rng([seed, 0])
        prompt = rng.integers(32, 513, size=256).astype(np.int64)
        out = _lognormal_outputs(rng, 256, 200.0, 1.0, 4096)
        wl = Workload("gqa8b", 256, 32, 8, 128, 16, "bf16", 32768, prompt + out, seed=seed)
    elif name == "long":
        wl = Workload("long", 8, 64, 8, 128, 16, "bf16", 20000,
                      np.full(8, 32768, dtype=np.int64), seed=1134)
    elif name == "prefix":
        seed = 1135
        B = 16 if block_size is None else int(block_size)
        if B not in (8, 16, 32):
            raise ValueError("prefix workload uses block size 8, 16 or 32")
        rng = np.random.default_rng([seed, 0])
        groups, n, plen = 32, 4, 2000
        div = rng.integers(1, 501, size=groups * n).astype(np.int64)
        wl = Workload("prefix", groups * n, 32, 8, 128, B, "bf16", 524288 // B, plen + div,
                      seed=seed, prefix_groups=groups, prefix_n=n, prefix_len=plen)
    elif name == "mixed":
        seed = 1139
        rng = np.random.default_rng([seed, 0])
        ctx = rng.integers(256, 1025, size=128).astype(np.int64)
        ctx[37] = 32768
        wl = Workload("mixed", 128, 32, 8, 128, 16, "bf16", 12288, ctx, seed=seed)
    elif name == "chat":
        seed = 1136
        rng = np.random.default_rng([seed, 0])
        S, retired = 128, 32
        lens = np.array([1000, 1536, 2000, 600], dtype=np.int64)
        w = 1.0 / np.arange(1, 5)
        choice = rng.choice(4, size=S + retired, p=w / w.sum())
        user = _lognormal_outputs(rng, S, 200.0, 1.0, 2000)
        wl = Workload("chat", S, 32, 8, 128, 16, "bf16", 32768, lens[choice[:S]] + user + 1, seed=seed,
                      chat_prompt_lens=lens, chat_choice=choice, chat_retired=retired)
    else:
        raise ValueError(f"unknown workload {name!r}; choose from {WORKLOAD_NAMES}")
    if block_size is not None and name != "prefix":
        raise ValueError("block_size override applies to the prefix workload only")
    if num_seqs is not None and num_seqs < wl.num_seqs:
        if wl.prefix_groups:
            g = max(1, num_seqs // wl.prefix_n)
            wl.prefix_groups = g
            wl.num_seqs = g * wl.prefix_n
        elif wl.chat_choice is not None:
            # keep the retired requests (and their draws) after the shorter batch
            wl.chat_choice = np.concatenate([wl.chat_choice[: int(num_seqs)], wl.chat_choice[wl.num_seqs:]])
            wl.num_seqs = int(num_seqs)
        else:
            wl.num_seqs = int(num_seqs)
        wl.ctx_lens = wl.ctx_lens[: wl.num_seqs].copy()
    return wl


ALLOCATOR_TRACES = ("tight", "serving")


def allocator_trace(name: str, num_requests: Optional[int] = None):
    """A seeded request trace for the allocator policy simulator.

    Returns ``(capacity_slots, requests)``; each request is a dict with
    ``arrival`` (step), ``prompt``, ``max_new``, ``gen`` (tokens it
    generates) and ``completion`` (the step after its last token).

    * ``tight``   the pages' 80-slot cache; 14 requests, arrival gaps
                  U{0..4}, prompts U{4..16}, max_new U{8..24}, gen
                  U{max_new/2 .. max_new}.
    * ``serving`` 131072 slots; 2000 requests, Poisson arrivals (1.5 per
                  step), prompts U{32..512}, max_new 2048, gen lognormal
                  (mean 200, sigma 1, capped at 2048).
    ``num_requests`` keeps the first requests (a reduced case) and scales
    the capacity in proportion.
    """
    if name == "tight":
        rng = np.random.default_rng([1137, 0])
        n, capacity = 14, 80
        arrival = np.cumsum(rng.integers(0, 5, n))
        prompt = rng.integers(4, 17, n)
        max_new = rng.integers(8, 25, n)
        gen = np.array([rng.integers(m // 2, m + 1) for m in max_new])
    elif name == "serving":
        rng = np.random.default_rng([1138, 0])
        n, capacity = 2000, 131072
        arrival = np.cumsum(rng.poisson(1.0 / 1.5, n))
        prompt = rng.integers(32, 513, n)
        max_new = np.full(n, 2048)
        gen = _lognormal_outputs(rng, n, 200.0, 1.0, 2048)
    else:
        raise ValueError(f"unknown trace {name!r}; choose from {ALLOCATOR_TRACES}")
    if num_requests is not None and num_requests < n:
        capacity = max(1, capacity * int(num_requests) // n)
        n = int(num_requests)
    reqs = [dict(arrival=int(arrival[i]), prompt=int(prompt[i]), max_new=int(max_new[i]), gen=int(gen[i]),
                 completion=int(arrival[i] + gen[i] + 1)) for i in range(n)]
    return capacity, reqs


def prefill_plan(wl: Workload) -> List[tuple]:
    """The ordered list of host operations that builds a workload's state.

    Each entry is one of ``("add", seq)``, ``("append", seq, n, source)``,
    ``("fork", parent, child)``, ``("admit", seq)`` or ``("free", seq)``;
    ``source`` says where the appended tokens' K/V come from: ``("prefix",
    group)`` or ``("private", seq)``. ``admit`` (chat) is a request arriving
    with the prompt ``wl.chat_tokens(seq)`` whose K/V are
    ``wl.chat_kv(seq, ...)``: the consumer admits it through its prefix
    cache, writes the positions the cache did not cover and registers the
    prompt's full blocks. After the plan, every batch sequence holds
    ``ctx_lens[s] - 1`` tokens; the decode step then appends one more token
    to each sequence in index order.
    """
    ops: List[tuple] = []
    if wl.chat_choice is not None:
        for r in range(wl.num_seqs, wl.num_seqs + wl.chat_retired):
            ops.append(("admit", r))
            ops.append(("free", r))
        for s in range(wl.num_seqs):
            ops.append(("admit", s))
    elif wl.prefix_groups:
        n = wl.prefix_n
        for g in range(wl.prefix_groups):
            parent = g * n
            ops.append(("add", parent))
            ops.append(("append", parent, wl.prefix_len, ("prefix", g)))
            for c in range(1, n):
                ops.append(("fork", parent, parent + c))
        for s in range(wl.num_seqs):
            ndiv = int(wl.ctx_lens[s]) - wl.prefix_len - 1
            if ndiv > 0:
                ops.append(("append", s, ndiv, ("private", s)))
    else:
        for s in range(wl.num_seqs):
            ops.append(("add", s))
            n0 = int(wl.ctx_lens[s]) - 1
            if n0 > 0:
                ops.append(("append", s, n0, ("private", s)))
    return ops
