"""Paged decode (split + combine kernels) and the visible-set plan against the
fp64 oracle, through the C ABI."""
import math

import numpy as np
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl
from parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def _dev(dc):
    d = "cuda"
    return dict(q=dc.q.to(d), k_cache=dc.k_cache.to(d), v_cache=dc.v_cache.to(d),
                page_table=dc.page_table.to(d), seqlens=dc.seqlens.to(d),
                sink=None if dc.sink is None else dc.sink.to(d))


def _run(ext, dc, **kw):
    t = _dev(dc)
    out, lse = ext.attn_sink_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["page_table"],
                                          t["seqlens"], t["sink"], dc.win_first, dc.win_last,
                                          dc.scale, **kw)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    return out.cpu(), lse.cpu()


def _oracle(dc, **kw):
    return orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens,
                                 dc.page_size, dc.sink, dc.win_first, dc.win_last, dc.scale, **kw)


CASES = [
    # (hq, hkv, d, page_size, seqlens, win_first, win_last, sink)
    (8, 1, 64, 16, [1, 2, 15, 16, 17, 100, 1000], 0, 0, ("uniform", -2.0, 4.0)),
    (64, 8, 64, 16, [1024, 3000, 77, 5000], 0, 0, ("uniform", -2.0, 4.0)),
    (32, 8, 128, 64, [8192, 9000, 20000, 100], 1024, 7168, None),
    (32, 8, 128, 64, [8192, 9000, 300], 1024, 7168, ("uniform", -2.0, 4.0)),
    (16, 4, 64, 7, [50, 333, 1], 5, 40, ("uniform", -2.0, 4.0)),      # odd page size, tiny windows
    (12, 12, 64, 8, [40, 70], 0, 0, None),                             # MHA (group 1)
    (48, 4, 64, 16, [500, 1500], 0, 0, ("uniform", -2.0, 4.0)),        # group 12 (two head tiles)
    (40, 2, 128, 32, [700, 65], 0, 0, ("uniform", -2.0, 4.0)),         # group 20 (two head blocks)
    (8, 2, 64, 16, [4000], 0, 100, ("uniform", -2.0, 4.0)),            # pure sliding window
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"hq{c[0]}hkv{c[1]}d{c[2]}ps{c[3]}w{c[5]}-{c[6]}")
def test_decode_matches_oracle(ext, case):
    hq, hkv, d, ps, lens, F_, W, sink = case
    dc = wl.make_decode(seqlens=lens, hq=hq, hkv=hkv, d=d, page_size=ps, sink=sink,
                        win_first=F_, win_last=W, seed=1, extra_pages=5)
    out, lse = _run(ext, dc)
    O, LSE = _oracle(dc)
    assert_out_close(out, O)
    assert_lse_close(lse, LSE)


def test_decode_sink_limits(ext):
    """sigma = -inf (no sink), large finite sigma and sigma = +inf."""
    dc = wl.make_decode(seqlens=[33, 600], hq=8, hkv=2, d=64, page_size=16, sink=None, seed=2)
    out, lse = _run(ext, dc)
    O, LSE = _oracle(dc)
    assert_out_close(out, O)
    assert_lse_close(lse, LSE)
    dc.sink = torch.full((8,), 80.0)
    out, lse = _run(ext, dc)
    O, LSE = _oracle(dc)
    assert_out_close(out, O)
    assert_lse_close(lse, LSE)
    assert float(out.abs().max()) < 1e-20
    dc.sink = torch.full((8,), math.inf)
    out, lse = _run(ext, dc)
    assert torch.all(out.float() == 0) and torch.all(torch.isposinf(lse))


def test_empty_cache_rows(ext):
    """A request with seqlen 0 sees nothing: O = 0, LSE = sink."""
    dc = wl.make_decode(seqlens=[0, 5], hq=4, hkv=1, d=64, page_size=16, sink=("uniform", -2.0, 4.0), seed=3)
    out, lse = _run(ext, dc)
    O, LSE = _oracle(dc)
    assert torch.all(out[0].float() == 0)
    np.testing.assert_allclose(lse[0].numpy(), dc.sink.numpy(), rtol=1e-6)
    assert_out_close(out, O)


def test_sink_counted_once_across_split_counts(ext):
    """One long request decoded alone (many small splits) and inside a batch
    (fewer, larger splits) agrees with the oracle both ways; a sink added per
    split would break it."""
    dc = wl.make_decode(seqlens=[30000] + [1024] * 63, hq=64, hkv=8, d=64, page_size=16,
                        sink=("uniform", -2.0, 4.0), seed=4)
    out_b, lse_b = _run(ext, dc)
    O, LSE = _oracle(dc, requests=[0])
    assert_out_close(out_b[0], O[0])
    assert_lse_close(lse_b[0], LSE[0])
    one = wl.Decode(name="one", q=dc.q[:1], k_cache=dc.k_cache, v_cache=dc.v_cache,
                    page_table=dc.page_table[:1].contiguous(), seqlens=dc.seqlens[:1].contiguous(),
                    page_size=16, sink=dc.sink)
    out_1, lse_1 = _run(ext, one)
    assert_out_close(out_1[0], O[0])
    assert_lse_close(lse_1[0], LSE[0])


def test_page_permutation_is_bitwise_invariant(ext):
    dc = wl.make_decode(seqlens=[777, 2048, 31], hq=16, hkv=2, d=128, page_size=16,
                        sink=("uniform", -2.0, 4.0), seed=5)
    out_a, lse_a = _run(ext, dc)
    perm = torch.randperm(dc.num_pages, generator=torch.Generator().manual_seed(8))
    kc = torch.empty_like(dc.k_cache)
    vc = torch.empty_like(dc.v_cache)
    kc[perm] = dc.k_cache
    vc[perm] = dc.v_cache
    pt = torch.where(dc.page_table >= 0, perm[dc.page_table.clamp(min=0).long()].int(), dc.page_table)
    dc2 = wl.Decode(name="perm", q=dc.q, k_cache=kc, v_cache=vc, page_table=pt.contiguous(),
                    seqlens=dc.seqlens, page_size=16, sink=dc.sink)
    out_b, lse_b = _run(ext, dc2)
    assert torch.equal(out_a, out_b) and torch.equal(lse_a, lse_b)


@pytest.mark.parametrize("F_,W", [(1024, 7168), (0, 0), (3, 5), (0, 64), (100, 0)])
def test_visible_ranges_and_slots_bit_exact(ext, F_, W):
    lens = [0, 1, 2, 63, 64, 65, 1023, 1024, 1025, 8191, 8192, 8193, 9000, 65536]
    dc = wl.make_decode(seqlens=lens, hq=1, hkv=1, d=64, page_size=64, sink=None, seed=6)
    sl = dc.seqlens.cuda()
    ranges = ext.attn_sink_visible_ranges(sl, F_, W).cpu().numpy()
    for b, L in enumerate(lens):
        (a0, b0), (a1, b1) = orc.visible_ranges(L, F_, W)
        assert list(ranges[b]) == [a0, b0, a1, b1], (L, F_, W)
    ref = orc.visible_slots(dc.seqlens, dc.page_table, 64, F_, W)
    maxv = max(len(t) for t, _ in ref)
    slots = ext.attn_sink_visible_slots(sl, dc.page_table.cuda(), 64, dc.num_pages, F_, W,
                                        maxv).cpu().numpy()
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    for b, (t, s) in enumerate(ref):
        np.testing.assert_array_equal(slots[b, :len(s)], s)
        assert np.all(slots[b, len(s):] == -1)


def test_bad_page_ids_and_lengths_raise_device_status(ext):
    """Out-of-range page ids and over-long seqlens are caught by the kernels'
    own bounds checks: the load is skipped and a status bit is set."""
    dc = wl.make_decode(seqlens=[40, 40], hq=4, hkv=1, d=64, page_size=16, sink=None, seed=7)
    pt = dc.page_table.clone()
    pt[1, 1] = dc.num_pages + 100
    t = _dev(dc)
    ext.attn_sink_decode_paged(t["q"], t["k_cache"], t["v_cache"], pt.cuda(), t["seqlens"])
    torch.cuda.synchronize()
    assert ext.device_status() & 1
    assert ext.device_status() == 0  # cleared
    sl = torch.tensor([40, 10_000], dtype=torch.int32, device="cuda")
    ext.attn_sink_decode_paged(t["q"], t["k_cache"], t["v_cache"], t["page_table"], sl)
    torch.cuda.synchronize()
    assert ext.device_status() & 2


def test_bad_page_rows_take_no_weight(ext):
    """Rows read through an out-of-range page id are skipped (status bit) and
    left out of the softmax: the result equals the decode over the request's
    other tokens (built as a shorter request whose page table skips that page)."""
    dc = wl.make_decode(seqlens=[40, 40], hq=4, hkv=1, d=64, page_size=16, sink=("uniform", -2.0, 4.0), seed=7)
    pt = dc.page_table.clone()
    pt[1, 1] = dc.num_pages + 100  # request 1, tokens 16..31
    t = _dev(dc)
    ext.device_status()
    out, lse = ext.attn_sink_decode_paged(t["q"], t["k_cache"], t["v_cache"], pt.cuda(), t["seqlens"], t["sink"])
    torch.cuda.synchronize()
    assert ext.device_status() & ext._lib.DEV_PAGE_OOB
    # request 1 without tokens 16..31: tokens 0..15 (page pt[1,0]) then 32..39 (slots 0..7 of page pt[1,2])
    pt2 = dc.page_table.clone()
    pt2[1, 1] = dc.page_table[1, 2]
    sl2 = torch.tensor([40, 24], dtype=torch.int32)
    O, LSE = orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, pt2, sl2, dc.page_size, dc.sink)
    assert_out_close(out.cpu(), O)
    assert_lse_close(lse.cpu(), LSE)


@pytest.mark.parametrize("name", ["decode_sink", "decode_window"])
def test_full_size_workloads_sampled(ext, name):
    """The full-size decode workloads, in the launch configuration the bench
    times; O and LSE of a sample of requests (all heads) against the oracle."""
    dc = wl.workload(name)
    out, lse = _run(ext, dc)
    g = torch.Generator().manual_seed(123)
    reqs = sorted(torch.randperm(dc.batch, generator=g)[:6].tolist())
    O, LSE = _oracle(dc, requests=reqs)
    for b in reqs:
        assert_out_close(out[b], O[b], what=f"{name} b={b}")
        assert_lse_close(lse[b], LSE[b])
