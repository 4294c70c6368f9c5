"""Packed QKV / KV layouts (row strides through the C ABI) against the
contiguous entry points and the fp64 oracle."""
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl
from parity import GRAD_REL_FRO, assert_lse_close, assert_out_close, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def _problem(hq, hkv, seqlens=(300, 129, 1), seed=31, with_dout=False, d=64):
    return wl.make_prefill(seqlens_q=list(seqlens), hq=hq, hkv=hkv, d=d, sink="normal", causal=True,
                           with_dout=with_dout, seed=seed)


def _pack(p):
    return torch.cat([p.q, p.k, p.v], dim=1).contiguous()  # (T, hq + 2 hkv, d)


@pytest.mark.parametrize("hq,hkv,d", [(8, 2, 64), (4, 4, 64), (8, 2, 128)])
def test_fwd_qkvpacked_equals_separate(ext, hq, hkv, d):
    p = _problem(hq, hkv, d=d)
    dev = "cuda"
    qkv = _pack(p).to(dev)
    cq = p.cu_seqlens_q.to(dev)
    out_p, lse_p = ext.attn_sink_fwd_qkvpacked(qkv, hkv, p.sink.to(dev), cq, p.max_seqlen_q)
    out_s, lse_s = ext.attn_sink_fwd(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.sink.to(dev), cq,
                                     p.cu_seqlens_k.to(dev), p.max_seqlen_q, p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(out_p.cpu(), out_s.cpu()) and torch.equal(lse_p.cpu(), lse_s.cpu())
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    assert_out_close(out_p.cpu(), O)
    assert_lse_close(lse_p.cpu(), LSE)


def test_fwd_qkvpacked_mha_4d_layout(ext):
    p = _problem(4, 4, seqlens=(200,))
    dev = "cuda"
    qkv4 = torch.stack([p.q, p.k, p.v], dim=1).contiguous().to(dev)  # (T, 3, H, d)
    out, lse = ext.attn_sink_fwd_qkvpacked(qkv4, 4, p.sink.to(dev), p.cu_seqlens_q.to(dev), p.max_seqlen_q)
    torch.cuda.synchronize()
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    assert_out_close(out.cpu(), O)
    assert_lse_close(lse.cpu(), LSE)


def test_fwd_kvpacked_equals_separate(ext):
    p = wl.make_prefill(seqlens_q=[100, 257], seqlens_k=[900, 257], hq=8, hkv=2, d=64, sink=(-2.0, 4.0),
                        seed=8)
    dev = "cuda"
    kv = torch.stack([p.k, p.v], dim=1).contiguous().to(dev)  # (Tk, 2, hkv, d)
    cq, ck = p.cu_seqlens_q.to(dev), p.cu_seqlens_k.to(dev)
    out_p, lse_p = ext.attn_sink_fwd_kvpacked(p.q.to(dev), kv, p.sink.to(dev), cq, ck, p.max_seqlen_q,
                                              p.max_seqlen_k)
    out_s, lse_s = ext.attn_sink_fwd(p.q.to(dev), p.k.to(dev), p.v.to(dev), p.sink.to(dev), cq, ck,
                                     p.max_seqlen_q, p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(out_p.cpu(), out_s.cpu()) and torch.equal(lse_p.cpu(), lse_s.cpu())


@pytest.mark.parametrize("d", [64, 128])
def test_bwd_qkvpacked(ext, d):
    hq, hkv = 8, 2
    p = _problem(hq, hkv, seqlens=(300, 129), with_dout=True, d=d)
    dev = "cuda"
    qkv = _pack(p).to(dev)
    cq = p.cu_seqlens_q.to(dev)
    sink = p.sink.to(dev)
    out, lse = ext.attn_sink_fwd_qkvpacked(qkv, hkv, sink, cq, p.max_seqlen_q)
    dqkv, dsink = ext.attn_sink_bwd_qkvpacked(qkv, hkv, sink, out, lse, p.dout.to(dev), cq, p.max_seqlen_q)
    dq, dk, dv, ds = ext.attn_sink_bwd(p.q.to(dev), p.k.to(dev), p.v.to(dev), sink, out, lse, p.dout.to(dev), cq,
                                       p.cu_seqlens_k.to(dev), p.max_seqlen_q, p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    dqkv = dqkv.cpu()
    # dK / dV come from TMEM without atomics: identical bits
    assert torch.equal(dqkv[:, hq:hq + hkv], dk.cpu())
    assert torch.equal(dqkv[:, hq + hkv:], dv.cpu())
    # dQ is summed with atomic adds in an unspecified order
    assert rel_fro(dqkv[:, :hq], dq.cpu()) <= 1e-3
    dQ, dK, dV, dS, _, _ = orc.attn_bwd(p.q, p.k, p.v, p.sink, p.dout, p.cu_seqlens_q, p.cu_seqlens_k)
    for got, want, n in ((dqkv[:, :hq], dQ, "dq"), (dqkv[:, hq:hq + hkv], dK, "dk"),
                         (dqkv[:, hq + hkv:], dV, "dv"), (dsink.cpu(), dS, "dsink")):
        assert rel_fro(got, want) <= GRAD_REL_FRO, n


def test_bad_stride_rejected(ext):
    p = _problem(4, 2, seqlens=(64,))
    dev = "cuda"
    lib = ext.lib()
    import ctypes
    q, k, v = p.q.to(dev), p.k.to(dev), p.v.to(dev)
    out = torch.empty_like(q)
    P = lambda t: ctypes.c_void_p(t.data_ptr())
    rc = lib.attn_sink_fwd_strided(P(q), P(k), P(v), 4 * 64 - 8, 0, 0, None, P(p.cu_seqlens_q.to(dev)),
                                   P(p.cu_seqlens_k.to(dev)), 1, 64, 64, 4, 2, 64, 64, 64, 0, 0, 1, 0.0, P(out), None,
                                   ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == -1
