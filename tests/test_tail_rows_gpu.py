"""Rows that a request's last key tile covers past its own keys must not reach its
output: with NaN in every cache slot no request owns, and NaN in a neighbouring
request's rows and past the end of the K/V buffers, the forward's outputs equal
those of the clean inputs bit for bit.  The backward likewise: NaN in a
neighbouring request and past the end of q, dout, k and v leaves the other
requests' gradients as they are (dK and dV bit for bit; dQ and dsink are sums
of fp32 atomic adds whose order is not fixed)."""
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def _owned_slots(page_table, seqlens_k, page_size, num_slots):
    owned = torch.zeros(num_slots, dtype=torch.bool)
    for b, L in enumerate(seqlens_k.tolist()):
        for t in range(L):
            owned[int(page_table[b, t // page_size]) * page_size + t % page_size] = True
    return owned


@pytest.mark.parametrize("page_size,win", [(16, (0, 0)), (8, (16, 200)), (128, (0, 0))])
def test_fwd_paged_ignores_unowned_slots(ext, page_size, win):
    pe = wl.make_paged_extend(seqlens_q=[77, 1, 130], seqlens_k=[301, 45, 130], hq=8, hkv=2, d=64,
                              page_size=page_size, win_first=win[0], win_last=win[1], seed=17, extra_pages=4)
    kw, vw = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new, page_size,
                           cu_new=pe.cu_seqlens_q)
    n_slots = kw.shape[0] * page_size
    owned = _owned_slots(pe.page_table, pe.seqlens_k, page_size, n_slots)
    assert not owned.all()
    dev = "cuda"
    results = []
    for poison in (False, True):
        kc, vc = kw.clone().view(n_slots, -1), vw.clone().view(n_slots, -1)
        if poison:
            kc[~owned] = float("nan")
            vc[~owned] = float("nan")
        out, lse = ext.attn_sink_fwd_paged(pe.q.to(dev), kc.view_as(kw).to(dev), vc.view_as(vw).to(dev),
                                           pe.page_table.to(dev), pe.cu_seqlens_q.to(dev), pe.seqlens_k.to(dev),
                                           pe.max_seqlen_q, pe.max_seqlen_k, pe.sink.to(dev),
                                           win_first=win[0], win_last=win[1])
        torch.cuda.synchronize()
        assert ext.device_status() == 0
        results.append((out.cpu(), lse.cpu()))
    assert not results[0][0].isnan().any()
    assert torch.equal(results[0][0], results[1][0])
    assert torch.equal(results[0][1], results[1][1])


@pytest.mark.parametrize("d", [64, 128])
def test_fwd_neighbour_and_trailing_rows_do_not_leak(ext, d):
    p = wl.make_prefill(seqlens_q=[100, 77, 129], seqlens_k=[300, 200, 129], hq=8, hkv=2, d=d, sink="normal",
                        seed=23)
    cq, ck = p.cu_seqlens_q.tolist(), p.cu_seqlens_k.tolist()
    dev = "cuda"
    results = []
    for poison in (False, True):
        q, k, v = p.q.clone(), p.k.clone(), p.v.clone()
        if poison:
            # request 1 holds NaN in every row, and the K/V buffers run 64 NaN rows past the last key
            q[cq[1]:cq[2]] = float("nan")
            k[ck[1]:ck[2]] = float("nan")
            v[ck[1]:ck[2]] = float("nan")
            pad = torch.full((64,) + tuple(k.shape[1:]), float("nan"), dtype=k.dtype)
            k, v = torch.cat([k, pad]), torch.cat([v, pad])
        out, lse = ext.attn_sink_fwd(q.to(dev), k.to(dev), v.to(dev), p.sink.to(dev), p.cu_seqlens_q.to(dev),
                                     p.cu_seqlens_k.to(dev), p.max_seqlen_q, p.max_seqlen_k)
        torch.cuda.synchronize()
        assert ext.device_status() == 0
        results.append((out.cpu(), lse.cpu()))
    for lo, hi in ((cq[0], cq[1]), (cq[2], cq[3])):
        assert not results[0][0][lo:hi].isnan().any()
        assert torch.equal(results[0][0][lo:hi], results[1][0][lo:hi])
        assert torch.equal(results[0][1][:, lo:hi], results[1][1][:, lo:hi])


def _fwd_bwd(ext, q, k, v, dout, p, dev="cuda"):
    sink = p.sink.to(dev)
    cq, ck = p.cu_seqlens_q.to(dev), p.cu_seqlens_k.to(dev)
    q, k, v, dout = q.to(dev), k.to(dev), v.to(dev), dout.to(dev)
    out, lse = ext.attn_sink_fwd(q, k, v, sink, cq, ck, p.max_seqlen_q, p.max_seqlen_k)
    dq, dk, dv, ds = ext.attn_sink_bwd(q, k, v, sink, out, lse, dout, cq, ck, p.max_seqlen_q, p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu(), ds.cpu()


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / max(float(b.norm()), 1e-30))


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_trailing_rows_do_not_leak(ext, d):
    """64 NaN rows past the end of q, dout, k and v (the last request's tail tiles
    read them): every gradient, dsink included, is unchanged."""
    p = wl.make_prefill(seqlens_q=[100, 77, 129], seqlens_k=[300, 200, 129], hq=8, hkv=2, d=d, sink="normal",
                        with_dout=True, seed=29)
    res = []
    for poison in (False, True):
        q, k, v, dout = p.q.clone(), p.k.clone(), p.v.clone(), p.dout.clone()
        if poison:
            def pad(x):
                return torch.cat([x, torch.full((64,) + tuple(x.shape[1:]), float("nan"), dtype=x.dtype)])
            q, k, v, dout = pad(q), pad(k), pad(v), pad(dout)
        dq, dk, dv, ds = _fwd_bwd(ext, q, k, v, dout, p)
        res.append((dq[:p.q.shape[0]], dk[:p.k.shape[0]], dv[:p.k.shape[0]], ds))
    (dq0, dk0, dv0, ds0), (dq1, dk1, dv1, ds1) = res
    for x in (dq1, dk1, dv1, ds1):
        assert not x.isnan().any()
    assert torch.equal(dk0, dk1) and torch.equal(dv0, dv1)
    assert _rel(dq1, dq0) <= 1e-5 and _rel(ds1, ds0) <= 1e-5


def test_bwd_neighbour_rows_do_not_leak(ext):
    """Request 1 holds NaN in every row of q, dout, k and v: the gradients of
    requests 0 and 2 (whose tail tiles cover request 1's rows and the buffers'
    end) stay finite and unchanged."""
    p = wl.make_prefill(seqlens_q=[100, 77, 129], seqlens_k=[300, 200, 129], hq=8, hkv=2, d=64, sink="normal",
                        with_dout=True, seed=31)
    cq, ck = p.cu_seqlens_q.tolist(), p.cu_seqlens_k.tolist()
    res = []
    for poison in (False, True):
        q, k, v, dout = p.q.clone(), p.k.clone(), p.v.clone(), p.dout.clone()
        if poison:
            q[cq[1]:cq[2]] = float("nan")
            dout[cq[1]:cq[2]] = float("nan")
            k[ck[1]:ck[2]] = float("nan")
            v[ck[1]:ck[2]] = float("nan")
        res.append(_fwd_bwd(ext, q, k, v, dout, p))
    (dq0, dk0, dv0, _), (dq1, dk1, dv1, _) = res
    for (ql, qh), (kl, kh) in (((cq[0], cq[1]), (ck[0], ck[1])), ((cq[2], cq[3]), (ck[2], ck[3]))):
        assert not dq1[ql:qh].isnan().any() and not dk1[kl:kh].isnan().any() and not dv1[kl:kh].isnan().any()
        assert torch.equal(dk0[kl:kh], dk1[kl:kh]) and torch.equal(dv0[kl:kh], dv1[kl:kh])
        assert _rel(dq1[ql:qh], dq0[ql:qh]) <= 1e-5


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_rows_past_last_request_are_zero(ext, d):
    """q / dout and k / v carry rows past the last request's (cu_seqlens[batch] <
    total): into output buffers that hold NaN, the backward writes zeros there
    (dq, and dk / dv with contiguous rows), and the requests' own gradients
    equal those of the buffers without the extra rows."""
    p = wl.make_prefill(seqlens_q=[100, 77], seqlens_k=[300, 129], hq=8, hkv=2, d=d, sink="normal",
                        with_dout=True, seed=37)
    dev = "cuda"
    nq, nk = p.q.shape[0], p.k.shape[0]
    ref = _fwd_bwd(ext, p.q, p.k, p.v, p.dout, p)

    def pad(x, n):
        return torch.cat([x, torch.randn((n,) + tuple(x.shape[1:])).to(x.dtype)])
    q, dout = pad(p.q, 40).to(dev), pad(p.dout, 40).to(dev)
    k, v = pad(p.k, 150).to(dev), pad(p.v, 150).to(dev)
    sink = p.sink.to(dev)
    cq, ck = p.cu_seqlens_q.to(dev), p.cu_seqlens_k.to(dev)
    out, lse = ext.attn_sink_fwd(q, k, v, sink, cq, ck, p.max_seqlen_q, p.max_seqlen_k)
    dq = torch.full_like(q, float("nan"))
    dk, dv = torch.full_like(k, float("nan")), torch.full_like(v, float("nan"))
    _, _, _, ds = ext.attn_sink_bwd(q, k, v, sink, out, lse, dout, cq, ck, p.max_seqlen_q, p.max_seqlen_k,
                                    dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    dq, dk, dv, ds = dq.cpu(), dk.cpu(), dv.cpu(), ds.cpu()
    assert torch.count_nonzero(dq[nq:]) == 0 and not dq[nq:].isnan().any()
    for x in (dk, dv):
        assert torch.count_nonzero(x[nk:]) == 0 and not x[nk:].isnan().any()
    assert torch.equal(dk[:nk], ref[1]) and torch.equal(dv[:nk], ref[2])
    assert _rel(dq[:nq], ref[0]) <= 1e-5 and _rel(ds, ref[3]) <= 1e-5
