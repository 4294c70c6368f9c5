"""The seeded synthetic workloads follow their stated recipe (lengths, value
ranges, page permutations, draw order) and the algorithmic work the bench divides
by is the closed form of that recipe: visible (query, key) pairs for the FLOPs,
visible tokens for the KV bytes (the windowed decode sees exactly 1024 + 7168
tokens per request, by the oracle's visibility rule)."""
import pytest
import torch

import bench
from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl


@pytest.fixture
def no_bulk(monkeypatch):
    """Skip drawing the bulk tensors (several GB for the decode caches).  Lengths
    and the page permutation are drawn before them, so everything checked with
    this fixture is what the bench uses; only the later draws (the sink) shift."""
    monkeypatch.setattr(wl, "_normal_bf16", lambda g, shape: torch.empty(shape, dtype=torch.bfloat16))


def _check_page_table(pt, seqlens, page_size, pool):
    used = []
    for b, L in enumerate(seqlens):
        n = -(-L // page_size)
        assert (pt[b, :n] >= 0).all() and (pt[b, n:] == -1).all()
        used += pt[b, :n].tolist()
    assert sorted(used) == list(range(pool))  # every physical page once: a permutation


def test_generators_are_deterministic():
    a, b, c = wl.prefill_tiny(0), wl.prefill_tiny(0), wl.prefill_tiny(1)
    for n in ("q", "k", "v", "sink"):
        assert torch.equal(getattr(a, n), getattr(b, n))
    assert not torch.equal(a.q, c.q)


def test_prefill_tiny():
    p = wl.prefill_tiny()
    assert p.q.shape == (256, 4, 64) and p.k.shape == (256, 2, 64) and p.q.dtype == torch.bfloat16
    assert p.cu_seqlens_q.tolist() == [0, 256] and p.sink.shape == (4,)
    assert bench.fwd_flops(p) == 4 * 64 * 4 * 256 * 257 // 2  # 33.7 MFLOP


def test_extend_varlen_recipe(no_bulk):
    p = wl.extend_varlen()
    C = p.seqlens_q
    P = [k - q for q, k in zip(p.seqlens_q, p.seqlens_k)]
    assert len(C) == 8 and all(512 <= c <= 8192 for c in C) and all(0 <= x <= 16384 for x in P)
    assert (p.hq, p.hkv, p.head_dim) == (64, 8, 64) and p.causal and p.win_last == 0
    assert ((p.sink >= -2.0) & (p.sink < 4.0)).all()
    # bottom-right causal: chunk row t sees P + t + 1 keys
    closed = sum(4 * 64 * 64 * (c * x + c * (c + 1) // 2) for c, x in zip(C, P))
    assert bench.fwd_flops(p) == closed
    assert closed == 4_836_967_579_648  # the bench line's algorithmic TFLOP per step (seed 0)


def test_extend_window_recipe(no_bulk):
    p = wl.extend_window()
    C = p.seqlens_q
    P = [k - q for q, k in zip(p.seqlens_q, p.seqlens_k)]
    assert len(C) == 8 and all(512 <= c <= 8192 for c in C) and all(8192 <= x <= 32768 for x in P)
    assert (p.win_first, p.win_last) == (1024, 7168) and p.causal
    # every query of a request sits at position >= 8191, so it sees exactly 1024 + 7168 keys
    assert bench.fwd_flops(p) == 4 * 64 * 64 * 8192 * sum(C)
    # and the visibility rule of the oracle agrees
    for Lq, Lk in zip(C, p.seqlens_k):
        (a0, b0), (a1, b1) = orc.visible_ranges(Lk - Lq + 1, 1024, 7168)
        assert (b0 - a0) + (b1 - a1) == 8192


def test_extend_paged_shares_the_lengths(no_bulk):
    p, pe = wl.extend_varlen(), wl.extend_paged()
    assert pe.seqlens_q == p.seqlens_q and pe.seqlens_k.tolist() == p.seqlens_k
    assert pe.page_size == 16
    _check_page_table(pe.page_table, pe.seqlens_k.tolist(), 16, pe.k_cache.shape[0])


def test_decode_sink_recipe(no_bulk):
    dc = wl.decode_sink()
    L = dc.seqlens.tolist()
    assert len(L) == 64 and all(1024 <= x <= 32768 for x in L)
    assert (dc.hq, dc.hkv, dc.head_dim, dc.page_size) == (64, 8, 64, 16) and dc.win_last == 0
    assert dc.k_cache.shape == (sum(-(-x // 16) for x in L), 16, 8, 64)
    _check_page_table(dc.page_table, L, 16, dc.k_cache.shape[0])
    assert ((dc.sink >= -2.0) & (dc.sink < 4.0)).all()
    kv_bytes = sum(bench._visible_counts(L, 0, 0)) * 2 * 8 * 64 * 2
    assert kv_bytes == sum(L) * 2048 == 1_942_480_896  # the bench line's kv_bytes (seed 0)


def test_decode_window_recipe(no_bulk):
    dc = wl.decode_window()
    L = dc.seqlens.tolist()
    assert len(L) == 32 and all(8192 <= x <= 65536 for x in L)
    assert (dc.hq, dc.hkv, dc.head_dim, dc.page_size) == (32, 8, 128, 64)
    assert (dc.win_first, dc.win_last) == (1024, 7168) and dc.sink is None
    _check_page_table(dc.page_table, L, 64, dc.k_cache.shape[0])
    for x in L:
        (a0, b0), (a1, b1) = orc.visible_ranges(x, 1024, 7168)
        assert (a0, b0) == (0, 1024) and (a1, b1) == (x - 7168, x)
    counts = bench._visible_counts(L, 1024, 7168)
    assert counts == [8192] * 32
    assert sum(counts) * 2 * 8 * 128 * 2 == 1_073_741_824  # the skipped middle is not counted


def test_train_recipe(no_bulk):
    p = wl.train()
    assert p.cu_seqlens_q.tolist() == [0, 8192, 16384] and p.dout is not None and p.causal
    fwd = bench.fwd_flops(p)
    assert fwd == 2 * 4 * 64 * 64 * (8192 * 8193 // 2)  # 1.10 TFLOP
    assert fwd + 2.5 * fwd == 3_848_760_459_264  # forward + backward (five GEMMs), per step


def test_head_dim_128_recipes(no_bulk):
    """The d-128 bench workloads keep the extend / train lengths at 32 query
    heads over 8 KV heads."""
    e, e128 = wl.extend_varlen(), wl.extend_d128()
    assert e128.seqlens_q == e.seqlens_q and e128.seqlens_k == e.seqlens_k
    assert (e128.hq, e128.hkv, e128.head_dim) == (32, 8, 128)
    assert bench.fwd_flops(e128) == bench.fwd_flops(e)  # 4 d Hq per pair: 4*128*32 = 4*64*64
    t = wl.train_d128()
    assert t.seqlens_q == [8192, 8192] and (t.hq, t.hkv, t.head_dim) == (32, 8, 128) and t.dout is not None
