"""Long contexts against the fp64 oracle: a 256k-key forward (with and without
the first 1024 + last 7168 window), a 128k-key head-dim-128 forward, a 64k-key
backward, a 200k-token paged extend and a 1M-token paged decode.  They run the
kernels' long loops (thousands of key tiles, hundreds of decode splits) and
their index arithmetic far past the lengths of the other tests."""
import numpy as np
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl
from parity import assert_grad_close, assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def _rows(seqlens_q, per_req, seed):
    g = torch.Generator().manual_seed(seed)
    rows = {}
    for b, Lq in enumerate(seqlens_q):
        pick = set(torch.randint(0, Lq, (per_req,), generator=g).tolist())
        rows[b] = sorted(pick | {0, Lq - 1, min(127, Lq - 1), min(128, Lq - 1)})
    return rows


def _index(cu, rows):
    cu = cu.tolist()
    return np.concatenate([np.asarray(r) + cu[b] for b, r in rows.items()])


@pytest.mark.parametrize("d,lk,hq,hkv,win", [(64, 262144, 4, 1, (0, 0)), (64, 262144, 4, 1, (1024, 7168)),
                                            (128, 131072, 4, 2, (0, 0))])
def test_fwd_long_context_sampled(ext, d, lk, hq, hkv, win):
    p = wl.make_prefill(seqlens_q=[300], seqlens_k=[lk], hq=hq, hkv=hkv, d=d, sink=(-2.0, 4.0),
                        win_first=win[0], win_last=win[1], seed=71)
    dev = "cuda"
    out, lse = ext.attn_sink_fwd(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.sink.to(dev), p.cu_seqlens_q.to(dev),
                                 p.cu_seqlens_k.to(dev), p.max_seqlen_q, p.max_seqlen_k, p.win_first, p.win_last)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    rows = _rows(p.seqlens_q, 16, 1)
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first, p.win_last,
                          rows=rows)
    idx = _index(p.cu_seqlens_q, rows)
    assert_out_close(out.cpu()[idx], O[idx], what=f"d{d} Lk{lk} win{win}")
    assert_lse_close(lse.cpu()[:, idx], LSE[:, idx], what=f"d{d} Lk{lk} win{win}")


def test_bwd_long_context(ext):
    """256 query rows over 65536 keys: 512 key-tile CTAs, most of them with a
    single query tile; every gradient against the oracle."""
    p = wl.make_prefill(seqlens_q=[256], seqlens_k=[65536], hq=2, hkv=1, d=64, sink=(-2.0, 4.0),
                        with_dout=True, seed=72)
    dev = "cuda"
    q, k, v, sink = p.q.to(dev), p.k.to(dev), p.v.to(dev), p.sink.to(dev)
    cq, ck = p.cu_seqlens_q.to(dev), p.cu_seqlens_k.to(dev)
    out, lse = ext.attn_sink_fwd(q, k, v, sink, cq, ck, p.max_seqlen_q, p.max_seqlen_k)
    dq, dk, dv, ds = ext.attn_sink_bwd(q, k, v, sink, out, lse, p.dout.to(dev), cq, ck, p.max_seqlen_q,
                                       p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    rq, rk, rv, rs, _, _ = orc.attn_bwd(p.q, p.k, p.v, p.sink, p.dout, p.cu_seqlens_q, p.cu_seqlens_k)
    assert_grad_close(dq.cpu(), rq, "dq")
    assert_grad_close(dk.cpu(), rk, "dk")
    assert_grad_close(dv.cpu(), rv, "dv")
    assert_grad_close(ds.cpu(), rs, "dsink")


def test_paged_extend_long_prefix(ext):
    """A 200k-token prefix in a page-16 cache (12.5k pages, random order) and a
    257-row chunk appended by the call."""
    pe = wl.make_paged_extend(seqlens_q=[257], seqlens_k=[200001], hq=4, hkv=1, d=64, page_size=16, seed=73)
    dev = "cuda"
    kc, vc = pe.k_cache.to(dev), pe.v_cache.to(dev)
    out, lse = ext.attn_sink_fwd_paged(pe.q.to(dev), kc, vc, pe.page_table.to(dev), pe.cu_seqlens_q.to(dev),
                                       pe.seqlens_k.to(dev), pe.max_seqlen_q, pe.max_seqlen_k, pe.sink.to(dev),
                                       pe.k_new.to(dev), pe.v_new.to(dev))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    kw, vw = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new,
                           pe.page_size, cu_new=pe.cu_seqlens_q)
    rows = _rows(pe.seqlens_q, 16, 2)
    O, LSE = orc.attn_fwd_paged(pe.q, kw, vw, pe.page_table, pe.seqlens_k, pe.cu_seqlens_q, pe.page_size,
                                pe.sink, rows=rows)
    idx = _index(pe.cu_seqlens_q, rows)
    assert_out_close(out.cpu()[idx], O[idx])
    assert_lse_close(lse.cpu()[:, idx], LSE[:, idx])


@pytest.mark.parametrize("win", [(0, 0), (1024, 7168)])
def test_decode_million_tokens(ext, win):
    """Two requests of 1,048,576 and 777,777 cached tokens (page 64, random page
    order): hundreds of splits per request, then the combine."""
    dc = wl.make_decode(seqlens=[1048576, 777777], hq=8, hkv=1, d=64, page_size=64, win_first=win[0],
                        win_last=win[1], seed=74)
    dev = "cuda"
    out, lse = ext.attn_sink_decode_paged(dc.q.to(dev), dc.k_cache.to(dev), dc.v_cache.to(dev),
                                          dc.page_table.to(dev), dc.seqlens.to(dev), dc.sink.to(dev),
                                          dc.win_first, dc.win_last, dc.scale)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    O, LSE = orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens, dc.page_size,
                                   dc.sink, dc.win_first, dc.win_last, dc.scale)
    assert_out_close(out.cpu(), O)
    assert_lse_close(lse.cpu(), LSE)
