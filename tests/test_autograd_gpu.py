"""The autograd functions (learnable sink, flash-attention PR "feat: Implement
Sink Attention", Key Changes): forward and backward through torch.autograd give
the C-ABI entry points' results and the fp64 oracle's gradients, dsink included."""
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl
from parity import assert_grad_close, assert_out_close, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def _leaf(t):
    return t.to("cuda").requires_grad_(True)


def _oracle(p):
    return orc.attn_bwd(p.q, p.k, p.v, p.sink, p.dout, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first,
                        p.win_last, p.causal, p.scale)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("case", ["ragged_sink", "window_no_sink"])
def test_varlen_func_gradients(ext, d, case):
    if case == "ragged_sink":
        p = wl.make_prefill(seqlens_q=[1, 130, 257], seqlens_k=[40, 300, 257], hq=8, hkv=2, d=d,
                            sink=(-2.0, 4.0), with_dout=True, seed=31)
    else:
        p = wl.make_prefill(seqlens_q=[200], seqlens_k=[700], hq=4, hkv=2, d=d, sink=None, win_first=20,
                            win_last=100, with_dout=True, seed=32)
    q, k, v = _leaf(p.q), _leaf(p.k), _leaf(p.v)
    sink = None if p.sink is None else _leaf(p.sink)
    cq, ck = p.cu_seqlens_q.cuda(), p.cu_seqlens_k.cuda()
    out, lse = ext.attn_sink_varlen_func(q, k, v, cq, ck, p.max_seqlen_q, p.max_seqlen_k, learnable_sink=sink,
                                         causal=p.causal, win_first=p.win_first, win_last=p.win_last,
                                         return_lse=True)
    out.backward(p.dout.cuda())
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert not lse.requires_grad

    # the forward is the entry point's, bit for bit
    ref_out, ref_lse = ext.attn_sink_fwd(q.detach(), k.detach(), v.detach(),
                                         None if sink is None else sink.detach(), cq, ck, p.max_seqlen_q,
                                         p.max_seqlen_k, p.win_first, p.win_last, p.causal)
    assert torch.equal(out.detach(), ref_out) and torch.equal(lse, ref_lse)

    rq, rk, rv, rs, ro, _ = _oracle(p)
    assert_out_close(out.detach().cpu(), ro, "out")
    assert_grad_close(q.grad.cpu(), rq, "dq")
    assert_grad_close(k.grad.cpu(), rk, "dk")
    assert_grad_close(v.grad.cpu(), rv, "dv")
    if sink is not None:
        assert sink.grad is not None and sink.grad.dtype == torch.float32
        assert_grad_close(sink.grad.cpu(), rs, "dsink")


def test_func_batched_equals_varlen(ext):
    """(B, S, H, d) batches run as B equal-length sequences of the varlen path."""
    g = torch.Generator().manual_seed(5)
    B, sq, sk, hq, hkv, d = 3, 150, 260, 4, 2, 64
    q0 = torch.randn(B, sq, hq, d, generator=g).to(torch.bfloat16)
    k0 = torch.randn(B, sk, hkv, d, generator=g).to(torch.bfloat16)
    v0 = torch.randn(B, sk, hkv, d, generator=g).to(torch.bfloat16)
    s0 = torch.randn(hq, generator=g, dtype=torch.float32)
    do = torch.randn(B, sq, hq, d, generator=g).to(torch.bfloat16).cuda()

    q, k, v, s = _leaf(q0), _leaf(k0), _leaf(v0), _leaf(s0)
    out = ext.attn_sink_func(q, k, v, learnable_sink=s)
    assert out.shape == (B, sq, hq, d)
    out.backward(do)

    q2, k2, v2, s2 = (_leaf(q0.reshape(B * sq, hq, d)), _leaf(k0.reshape(B * sk, hkv, d)),
                      _leaf(v0.reshape(B * sk, hkv, d)), _leaf(s0))
    cq = torch.arange(0, (B + 1) * sq, sq, dtype=torch.int32, device="cuda")
    ck = torch.arange(0, (B + 1) * sk, sk, dtype=torch.int32, device="cuda")
    out2 = ext.attn_sink_varlen_func(q2, k2, v2, cq, ck, sq, sk, learnable_sink=s2)
    out2.backward(do.reshape(B * sq, hq, d))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(out.detach().reshape(B * sq, hq, d), out2.detach())
    # dK / dV accumulate in a fixed order; dQ and dsink are summed by reductions
    # whose order varies between runs
    assert torch.equal(k.grad.reshape(B * sk, hkv, d), k2.grad)
    assert torch.equal(v.grad.reshape(B * sk, hkv, d), v2.grad)
    assert rel_fro(q.grad.reshape(B * sq, hq, d).cpu(), q2.grad.cpu()) < 1e-5
    assert rel_fro(s.grad.cpu(), s2.grad.cpu()) < 1e-5


@pytest.mark.parametrize("layout", ["t3hd", "flat"])
def test_varlen_qkvpacked_func_gradients(ext, layout):
    hq = hkv = 4 if layout == "t3hd" else None
    if layout == "t3hd":
        p = wl.make_prefill(seqlens_q=[129, 300], hq=4, hkv=4, d=64, sink="normal", with_dout=True, seed=41)
        qkv0 = torch.stack([p.q, p.k, p.v], dim=1)  # (T, 3, H, d)
    else:
        p = wl.make_prefill(seqlens_q=[129, 300], hq=8, hkv=2, d=64, sink="normal", with_dout=True, seed=42)
        qkv0 = torch.cat([p.q, p.k, p.v], dim=1)  # (T, Hq + 2 Hkv, d)
        hq, hkv = 8, 2
    qkv, s = _leaf(qkv0.contiguous()), _leaf(p.sink)
    cu = p.cu_seqlens_q.cuda()
    out = ext.attn_sink_varlen_qkvpacked_func(qkv, cu, p.max_seqlen_q, hkv=hkv, learnable_sink=s)
    out.backward(p.dout.cuda())
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert qkv.grad.shape == qkv.shape
    g = qkv.grad.reshape(qkv.shape[0], -1, 64).cpu()
    rq, rk, rv, rs, ro, _ = _oracle(p)
    assert_out_close(out.detach().cpu(), ro, "out")
    assert_grad_close(g[:, :hq], rq, "dq")
    assert_grad_close(g[:, hq:hq + hkv], rk, "dk")
    assert_grad_close(g[:, hq + hkv:], rv, "dv")
    assert_grad_close(s.grad.cpu(), rs, "dsink")


def test_sink_trains(ext):
    """SGD on the sink alone lowers a loss that falls as the sink takes weight
    (the output's squared norm), moving every head's sink up."""
    p = wl.make_prefill(seqlens_q=[256], hq=4, hkv=2, d=64, sink=(4.0, 6.0), seed=51)
    q, k, v = p.q.cuda(), p.k.cuda(), p.v.cuda()
    s = torch.nn.Parameter(p.sink.cuda())
    s0 = s.detach().clone()
    cq = p.cu_seqlens_q.cuda()
    opt = torch.optim.SGD([s], lr=0.005)
    losses = []
    for _ in range(5):
        opt.zero_grad()
        out = ext.attn_sink_varlen_func(q, k, v, cq, cq, p.max_seqlen_q, p.max_seqlen_q, learnable_sink=s)
        loss = out.float().square().sum()
        loss.backward()
        opt.step()
        losses.append(loss.item())
    assert ext.device_status() == 0
    assert all(b < a for a, b in zip(losses, losses[1:])), losses
    assert losses[-1] < 0.9 * losses[0], losses
    assert bool((s.detach() > s0).all()), (s0, s.detach())


def test_varlen_kvpacked_func_gradients(ext):
    p = wl.make_prefill(seqlens_q=[100, 257], seqlens_k=[300, 400], hq=8, hkv=2, d=64, sink="normal",
                        with_dout=True, seed=61)
    q = _leaf(p.q)
    kv = _leaf(torch.stack([p.k, p.v], dim=1).contiguous())  # (Tk, 2, Hkv, d)
    s = _leaf(p.sink)
    cq, ck = p.cu_seqlens_q.cuda(), p.cu_seqlens_k.cuda()
    out = ext.attn_sink_varlen_kvpacked_func(q, kv, cq, ck, p.max_seqlen_q, p.max_seqlen_k, learnable_sink=s)
    out.backward(p.dout.cuda())
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert kv.grad.shape == kv.shape
    rq, rk, rv, rs, ro, _ = _oracle(p)
    assert_out_close(out.detach().cpu(), ro, "out")
    assert_grad_close(q.grad.cpu(), rq, "dq")
    assert_grad_close(kv.grad[:, 0].cpu(), rk, "dk")
    assert_grad_close(kv.grad[:, 1].cpu(), rv, "dv")
    assert_grad_close(s.grad.cpu(), rs, "dsink")


def test_fixed_length_packed_forms_equal_varlen(ext):
    """(B, S, 3, H, d) and (B, Sk, 2, Hkv, d) batches give the varlen packed
    functions' results; padding rows past the last sequence get zero gradient."""
    g = torch.Generator().manual_seed(7)
    B, S, H, d = 2, 140, 4, 64
    qkv0 = torch.randn(B, S, 3, H, d, generator=g).to(torch.bfloat16)
    s0 = torch.randn(H, generator=g, dtype=torch.float32)
    do = torch.randn(B, S, H, d, generator=g).to(torch.bfloat16).cuda()
    qkv, s = _leaf(qkv0), _leaf(s0)
    out = ext.attn_sink_qkvpacked_func(qkv, learnable_sink=s)
    out.backward(do)
    # the same sequences inside a buffer with 5 padding rows at the end
    pad = torch.randn(5, 3, H, d, generator=g).to(torch.bfloat16)
    qkv2 = _leaf(torch.cat([qkv0.reshape(B * S, 3, H, d), pad]))
    s2 = _leaf(s0)
    cu = torch.arange(0, (B + 1) * S, S, dtype=torch.int32, device="cuda")
    out2 = ext.attn_sink_varlen_qkvpacked_func(qkv2, cu, S, learnable_sink=s2)
    out2[:B * S].backward(do.reshape(B * S, H, d))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(out.detach().reshape(B * S, H, d), out2.detach()[:B * S])
    g1 = qkv.grad.reshape(B * S, 3, H, d)
    assert torch.equal(g1[:, 1:], qkv2.grad[:B * S, 1:])  # dK, dV: fixed accumulation order
    assert rel_fro(g1[:, 0].cpu(), qkv2.grad[:B * S, 0].cpu()) < 1e-5
    assert torch.count_nonzero(qkv2.grad[B * S:]) == 0
    assert rel_fro(s.grad.cpu(), s2.grad.cpu()) < 1e-5

    # kv-packed: q (B, Sq, Hq, d) against kv (B, Sk, 2, Hkv, d)
    sq, sk, hq, hkv = 90, 150, 8, 2
    q0 = torch.randn(B, sq, hq, d, generator=g).to(torch.bfloat16)
    kv0 = torch.randn(B, sk, 2, hkv, d, generator=g).to(torch.bfloat16)
    s3 = torch.randn(hq, generator=g, dtype=torch.float32)
    do3 = torch.randn(B, sq, hq, d, generator=g).to(torch.bfloat16).cuda()
    q, kv, s = _leaf(q0), _leaf(kv0), _leaf(s3)
    out = ext.attn_sink_kvpacked_func(q, kv, learnable_sink=s)
    out.backward(do3)
    q2, kv2, s2 = _leaf(q0.reshape(B * sq, hq, d)), _leaf(kv0.reshape(B * sk, 2, hkv, d)), _leaf(s3)
    cq = torch.arange(0, (B + 1) * sq, sq, dtype=torch.int32, device="cuda")
    ck = torch.arange(0, (B + 1) * sk, sk, dtype=torch.int32, device="cuda")
    out2 = ext.attn_sink_varlen_kvpacked_func(q2, kv2, cq, ck, sq, sk, learnable_sink=s2)
    out2.backward(do3.reshape(B * sq, hq, d))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(out.detach().reshape(B * sq, hq, d), out2.detach())
    assert torch.equal(kv.grad.reshape(B * sk, 2, hkv, d), kv2.grad)
    assert rel_fro(q.grad.reshape(B * sq, hq, d).cpu(), q2.grad.cpu()) < 1e-5
    # and the packed forward is the unpacked one, bit for bit
    k_, v_ = kv0.reshape(B * sk, 2, hkv, d)[:, 0].contiguous(), kv0.reshape(B * sk, 2, hkv, d)[:, 1].contiguous()
    ref, _ = ext.attn_sink_fwd(q0.reshape(B * sq, hq, d).cuda(), k_.cuda(), v_.cuda(), s3.cuda(), cq, ck, sq, sk)
    assert torch.equal(out2.detach(), ref)
