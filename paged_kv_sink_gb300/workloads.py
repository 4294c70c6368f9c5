"""Seeded synthetic inputs for attention with an attention sink.

This module only draws random numbers and lays them out; it contains none of the
attention arithmetic.  The CUDA path (through the C ABI) and the CPU oracle both
take their inputs from here, so that they see bit-identical data.

Workloads (shapes from the two forms of the sink described on the pages):

* ``prefill_tiny``   -- causal prefill with a learnable per-head sink
  (flash-attention PR "feat: Implement Sink Attention", Description: a
  ``(nheads,)`` sink logit): B 1, L 256, Hq 4, Hkv 2, d 64, sink ~ N(0,1).
* ``extend_varlen``  -- varlen chunked extend with sink, GPT-OSS-like heads
  (sglang PR "openai oss attention sink support with trtllm-gen backend",
  Highlights: the extend path gets ``sink=``): 8 requests, prefix U{0..16384},
  chunk U{512..8192}, Hq 64, Hkv 8, d 64, sink ~ U(-2, 4).
* ``decode_sink``    -- paged single-token decode with sink (same page,
  decode path): B 64, Hq 64, Hkv 8, d 64, page 16, L U{1024..32768}.
* ``decode_window``  -- paged decode with first-window + last-window selection
  and no learnable sink (sglang PR "To implement attention-sink", Motivation
  and suggested code: first 1024 + last 7168 tokens): B 32, Hq 32, Hkv 8,
  d 128, page 64, L U{8192..65536}.
* ``train``          -- training forward+backward with sink: B 2, L 8192,
  Hq 64, Hkv 8, d 64, sink ~ N(0,1), dO ~ N(0,1).
* ``extend_window``  -- the varlen extend with the first 1024 + last 7168 window
  of sglang PR "To implement attention-sink" (Motivation and suggested code:
  8192 visible tokens per query once a sequence is longer than that): 8
  requests, prefix U{8192..32768} (so that the window skips keys), chunk
  U{512..8192}, Hq 64, Hkv 8, d 64, sink ~ U(-2, 4).
* ``extend_paged``   -- the ``extend_varlen`` shapes with each request's
  prefix in a paged cache (page 16, random page permutation; the serving
  extend path reads its prefix through the page table, sglang PR "To implement
  attention-sink", suggested code) and the chunk's K/V appended by the call.

Recipe: one ``torch.Generator('cpu')`` seeded with ``seed``; draws are taken in
the fixed order lengths -> page permutation -> q -> k -> v -> sink -> dO (for
the paged extend: q -> K cache -> V cache -> new K -> new V -> sink).
Integer "uniform a-b" ranges include both ends.  Floating inputs are drawn in
fp32 and rounded to bf16 (round-to-nearest-even, torch's conversion).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

__all__ = ["Prefill", "Decode", "make_prefill", "make_decode", "WORKLOADS", "workload"]


@dataclass
class Prefill:
    """Varlen prefill / extend / training inputs (all CPU tensors)."""
    name: str
    q: torch.Tensor            # (total_q, hq, d) bf16
    k: torch.Tensor            # (total_k, hkv, d) bf16
    v: torch.Tensor            # (total_k, hkv, d) bf16
    sink: Optional[torch.Tensor]  # (hq,) fp32 or None (= -inf)
    cu_seqlens_q: torch.Tensor  # (B+1,) int32
    cu_seqlens_k: torch.Tensor  # (B+1,) int32
    win_first: int = 0
    win_last: int = 0
    causal: bool = True
    scale: float = 0.0          # 0 -> 1/sqrt(d)
    dout: Optional[torch.Tensor] = None  # (total_q, hq, d) bf16, training only
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.cu_seqlens_q.numel() - 1

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.k.shape[1]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def seqlens_q(self):
        return (self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).tolist()

    @property
    def seqlens_k(self):
        return (self.cu_seqlens_k[1:] - self.cu_seqlens_k[:-1]).tolist()

    @property
    def max_seqlen_q(self) -> int:
        return max(self.seqlens_q) if self.batch else 0

    @property
    def max_seqlen_k(self) -> int:
        return max(self.seqlens_k) if self.batch else 0

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / math.sqrt(self.head_dim)


@dataclass
class Decode:
    """Paged single-token decode inputs (all CPU tensors)."""
    name: str
    q: torch.Tensor            # (B, hq, d) bf16
    k_cache: torch.Tensor      # (num_pages, page_size, hkv, d) bf16
    v_cache: torch.Tensor      # (num_pages, page_size, hkv, d) bf16
    page_table: torch.Tensor   # (B, max_pages) int32, physical page ids
    seqlens: torch.Tensor      # (B,) int32, true cache length incl. the new token
    page_size: int
    sink: Optional[torch.Tensor]
    win_first: int = 0
    win_last: int = 0
    scale: float = 0.0
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.k_cache.shape[2]

    @property
    def head_dim(self) -> int:
        return self.q.shape[2]

    @property
    def num_pages(self) -> int:
        return self.k_cache.shape[0]

    @property
    def max_pages(self) -> int:
        return self.page_table.shape[1]

    @property
    def softmax_scale(self) -> float:
        return self.scale if self.scale > 0 else 1.0 / math.sqrt(self.head_dim)


@dataclass
class PagedExtend:
    """Varlen extend against a paged KV cache (all CPU tensors).

    Request ``b`` has ``seqlens_k[b]`` tokens in the cache: a prefix followed by
    its new chunk of ``Lq_b`` tokens (the query rows, ``cu_seqlens_q``).  The
    chunk's K/V rows are ``k_new``/``v_new``; the cache slots of the chunk hold
    unrelated values until the chunk is appended."""
    name: str
    q: torch.Tensor            # (total_q, hq, d) bf16
    k_new: torch.Tensor        # (total_q, hkv, d) bf16
    v_new: torch.Tensor        # (total_q, hkv, d) bf16
    k_cache: torch.Tensor      # (num_pages, page_size, hkv, d) bf16
    v_cache: torch.Tensor
    page_table: torch.Tensor   # (B, max_pages) int32
    seqlens_k: torch.Tensor    # (B,) int32, prefix + chunk
    cu_seqlens_q: torch.Tensor  # (B+1,) int32
    page_size: int
    sink: Optional[torch.Tensor]
    win_first: int = 0
    win_last: int = 0
    causal: bool = True
    scale: float = 0.0

    @property
    def batch(self) -> int:
        return self.cu_seqlens_q.numel() - 1

    @property
    def hq(self) -> int:
        return self.q.shape[1]

    @property
    def hkv(self) -> int:
        return self.k_cache.shape[2]

    @property
    def seqlens_q(self):
        return (self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).tolist()

    @property
    def max_seqlen_q(self) -> int:
        return max(self.seqlens_q) if self.batch else 0

    @property
    def max_seqlen_k(self) -> int:
        return int(self.seqlens_k.max()) if self.batch else 0


def _randint(g, lo, hi, n):
    """n integers uniform on [lo, hi] (both ends included)."""
    return torch.randint(lo, hi + 1, (n,), generator=g, dtype=torch.int64)


def _normal_bf16(g, shape):
    return torch.randn(*shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def _sink(g, kind, hq):
    if kind is None:
        return None
    if kind == "normal":
        return torch.randn(hq, generator=g, dtype=torch.float32)
    lo, hi = kind
    return (torch.rand(hq, generator=g, dtype=torch.float32) * (hi - lo) + lo).float()


def make_prefill(*, name="prefill", seqlens_q, seqlens_k=None, hq, hkv, d, sink="normal",
                 win_first=0, win_last=0, causal=True, scale=0.0, with_dout=False, seed=0,
                 g=None) -> Prefill:
    """Build a varlen prefill problem.

    ``seqlens_q``/``seqlens_k`` are lists (or callables ``g -> list`` drawn first).
    K/V for request r hold its cached prefix followed by its new chunk, so the
    chunk's rows are the last ``Lq`` key positions (bottom-right causal).
    """
    if g is None:
        g = torch.Generator().manual_seed(seed)
    if callable(seqlens_q):
        seqlens_q, seqlens_k = seqlens_q(g)
    if seqlens_k is None:
        seqlens_k = list(seqlens_q)
    seqlens_q = [int(x) for x in seqlens_q]
    seqlens_k = [int(x) for x in seqlens_k]
    cu_q = torch.zeros(len(seqlens_q) + 1, dtype=torch.int32)
    cu_k = torch.zeros(len(seqlens_k) + 1, dtype=torch.int32)
    cu_q[1:] = torch.tensor(seqlens_q, dtype=torch.int64).cumsum(0).to(torch.int32)
    cu_k[1:] = torch.tensor(seqlens_k, dtype=torch.int64).cumsum(0).to(torch.int32)
    tq, tk = int(cu_q[-1]), int(cu_k[-1])
    q = _normal_bf16(g, (tq, hq, d))
    k = _normal_bf16(g, (tk, hkv, d))
    v = _normal_bf16(g, (tk, hkv, d))
    s = _sink(g, sink, hq)
    dout = _normal_bf16(g, (tq, hq, d)) if with_dout else None
    return Prefill(name=name, q=q, k=k, v=v, sink=s, cu_seqlens_q=cu_q, cu_seqlens_k=cu_k,
                   win_first=win_first, win_last=win_last, causal=causal, scale=scale, dout=dout)


def make_decode(*, name="decode", seqlens, hq, hkv, d, page_size, sink=("uniform", -2.0, 4.0),
                win_first=0, win_last=0, scale=0.0, seed=0, g=None, extra_pages=0) -> Decode:
    """Build a paged single-token decode problem.

    ``seqlens`` is a list or a callable ``g -> list`` (drawn first).  Each request
    owns ceil(L/page_size) pages; the physical pool is the sum of those (plus
    ``extra_pages`` unused ones) and pages are assigned by a random permutation.
    Unused page-table entries are -1.
    """
    if g is None:
        g = torch.Generator().manual_seed(seed)
    if callable(seqlens):
        seqlens = seqlens(g)
    seqlens = [int(x) for x in seqlens]
    B = len(seqlens)
    npages = [(L + page_size - 1) // page_size for L in seqlens]
    pool = sum(npages) + extra_pages
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    max_pages = max(npages) if B else 0
    max_pages = max(max_pages, 1)
    pt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[off:off + n]
        off += n
    q = _normal_bf16(g, (B, hq, d))
    kc = _normal_bf16(g, (pool, page_size, hkv, d))
    vc = _normal_bf16(g, (pool, page_size, hkv, d))
    if isinstance(sink, tuple) and sink and sink[0] == "uniform":
        sink = (sink[1], sink[2])
    s = _sink(g, sink, hq)
    return Decode(name=name, q=q, k_cache=kc, v_cache=vc, page_table=pt,
                  seqlens=torch.tensor(seqlens, dtype=torch.int32), page_size=page_size,
                  sink=s, win_first=win_first, win_last=win_last, scale=scale)


def make_paged_extend(*, name="paged_extend", seqlens_q, seqlens_k, hq, hkv, d, page_size,
                      sink=(-2.0, 4.0), win_first=0, win_last=0, causal=True, scale=0.0, seed=0,
                      g=None, extra_pages=0) -> PagedExtend:
    """Build a paged varlen extend problem.

    Lengths (lists or a callable ``g -> (seqlens_q, seqlens_k)``) are drawn
    first, then the page permutation (as in ``make_decode``), then q, the two
    caches, the chunk's new K and V, and the sink."""
    if g is None:
        g = torch.Generator().manual_seed(seed)
    if callable(seqlens_q):
        seqlens_q, seqlens_k = seqlens_q(g)
    seqlens_q = [int(x) for x in seqlens_q]
    seqlens_k = [int(x) for x in seqlens_k]
    B = len(seqlens_q)
    npages = [(L + page_size - 1) // page_size for L in seqlens_k]
    pool = max(sum(npages) + extra_pages, 1)
    perm = torch.randperm(pool, generator=g).to(torch.int32)
    max_pages = max(max(npages) if B else 0, 1)
    pt = torch.full((B, max_pages), -1, dtype=torch.int32)
    off = 0
    for b, n in enumerate(npages):
        pt[b, :n] = perm[off:off + n]
        off += n
    cu_q = torch.zeros(B + 1, dtype=torch.int32)
    cu_q[1:] = torch.tensor(seqlens_q, dtype=torch.int64).cumsum(0).to(torch.int32)
    tq = int(cu_q[-1])
    q = _normal_bf16(g, (tq, hq, d))
    kc = _normal_bf16(g, (pool, page_size, hkv, d))
    vc = _normal_bf16(g, (pool, page_size, hkv, d))
    kn = _normal_bf16(g, (tq, hkv, d))
    vn = _normal_bf16(g, (tq, hkv, d))
    s = _sink(g, sink, hq)
    return PagedExtend(name=name, q=q, k_new=kn, v_new=vn, k_cache=kc, v_cache=vc, page_table=pt,
                       seqlens_k=torch.tensor(seqlens_k, dtype=torch.int32), cu_seqlens_q=cu_q,
                       page_size=page_size, sink=s, win_first=win_first, win_last=win_last,
                       causal=causal, scale=scale)


# ---------------------------------------------------------------------------
# The five named workloads.


def prefill_tiny(seed=0):
    return make_prefill(name="prefill_tiny B1 L256 Hq4 Hkv2 d64 sink", seqlens_q=[256],
                        hq=4, hkv=2, d=64, sink="normal", seed=seed)


def extend_varlen(seed=0, n_req=8):
    def lens(g):
        prefix = _randint(g, 0, 16384, n_req)
        chunk = _randint(g, 512, 8192, n_req)
        return chunk.tolist(), (prefix + chunk).tolist()
    return make_prefill(name="extend_varlen 8req prefix U0-16384 chunk U512-8192 Hq64 Hkv8 d64 sink",
                        seqlens_q=lens, hq=64, hkv=8, d=64, sink=(-2.0, 4.0), seed=seed)


def extend_window(seed=0, n_req=8):
    def lens(g):
        prefix = _randint(g, 8192, 32768, n_req)
        chunk = _randint(g, 512, 8192, n_req)
        return chunk.tolist(), (prefix + chunk).tolist()
    return make_prefill(name="extend_window 8req prefix U8192-32768 chunk U512-8192 Hq64 Hkv8 d64 sink "
                             "first1024+last7168",
                        seqlens_q=lens, hq=64, hkv=8, d=64, sink=(-2.0, 4.0), win_first=1024, win_last=7168,
                        seed=seed)


def decode_sink(seed=0):
    return make_decode(name="decode_sink B64 Hq64 Hkv8 d64 ps16 L U1024-32768 sink",
                       seqlens=lambda g: _randint(g, 1024, 32768, 64).tolist(),
                       hq=64, hkv=8, d=64, page_size=16, sink=("uniform", -2.0, 4.0), seed=seed)


def decode_window(seed=0):
    return make_decode(name="decode_window B32 Hq32 Hkv8 d128 ps64 L U8192-65536 first1024+last7168",
                       seqlens=lambda g: _randint(g, 8192, 65536, 32).tolist(),
                       hq=32, hkv=8, d=128, page_size=64, sink=None,
                       win_first=1024, win_last=7168, seed=seed)


def extend_paged(seed=0, n_req=8, page_size=16):
    """The varlen-extend shapes with the prefix in a paged cache (page size 16,
    random page permutation) and the chunk appended by the call."""
    def lens(g):
        prefix = _randint(g, 0, 16384, n_req)
        chunk = _randint(g, 512, 8192, n_req)
        return chunk.tolist(), (prefix + chunk).tolist()
    return make_paged_extend(name=f"extend_paged 8req prefix U0-16384 chunk U512-8192 Hq64 Hkv8 d64 ps{page_size} sink",
                             seqlens_q=lens, seqlens_k=None, hq=64, hkv=8, d=64, page_size=page_size,
                             sink=(-2.0, 4.0), seed=seed)


def train(seed=0):
    return make_prefill(name="train B2 L8192 Hq64 Hkv8 d64 causal sink fwd+bwd",
                        seqlens_q=[8192, 8192], hq=64, hkv=8, d=64, sink="normal",
                        with_dout=True, seed=seed)


# Head dim 128 (the width of the models the window form serves): the same
# lengths as extend_varlen and train with 32 query heads over 8 KV heads.
def extend_d128(seed=0, n_req=8):
    def lens(g):
        prefix = _randint(g, 0, 16384, n_req)
        chunk = _randint(g, 512, 8192, n_req)
        return chunk.tolist(), (prefix + chunk).tolist()
    return make_prefill(name="extend_d128 8req prefix U0-16384 chunk U512-8192 Hq32 Hkv8 d128 sink",
                        seqlens_q=lens, hq=32, hkv=8, d=128, sink=(-2.0, 4.0), seed=seed)


def train_d128(seed=0):
    return make_prefill(name="train_d128 B2 L8192 Hq32 Hkv8 d128 causal sink fwd+bwd",
                        seqlens_q=[8192, 8192], hq=32, hkv=8, d=128, sink="normal",
                        with_dout=True, seed=seed)


WORKLOADS = {
    "prefill_tiny": prefill_tiny,
    "extend_varlen": extend_varlen,
    "extend_window": extend_window,
    "decode_sink": decode_sink,
    "decode_window": decode_window,
    "train": train,
    "extend_paged": extend_paged,
    "extend_d128": extend_d128,
    "train_d128": train_d128,
}


def workload(name, seed=0):
    return WORKLOADS[name](seed=seed)
