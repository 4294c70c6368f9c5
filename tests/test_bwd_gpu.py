"""Backward (preprocess + tcgen05 main + dQ convert) against the fp64 oracle,
through the C ABI.  The GPU backward consumes the GPU forward's O and LSE, as
a training step does."""
import math

import numpy as np
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl
from parity import assert_grad_close, rel_fro

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def run_fwd_bwd(ext, p):
    d = "cuda"
    q, k, v = p.q.to(d), p.k.to(d), p.v.to(d)
    sink = None if p.sink is None else p.sink.to(d)
    cq, ck = p.cu_seqlens_q.to(d), p.cu_seqlens_k.to(d)
    out, lse = ext.attn_sink_fwd(q, k, v, sink, cq, ck, p.max_seqlen_q, p.max_seqlen_k, p.win_first,
                                 p.win_last, p.causal, p.scale)
    dq, dk, dv, ds = ext.attn_sink_bwd(q, k, v, sink, out, lse, p.dout.to(d), cq, ck, p.max_seqlen_q,
                                       p.max_seqlen_k, p.win_first, p.win_last, p.causal, p.scale)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    return dq.cpu(), dk.cpu(), dv.cpu(), None if ds is None else ds.cpu()


def oracle_bwd(p, **kw):
    return orc.attn_bwd(p.q, p.k, p.v, p.sink, p.dout, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first,
                        p.win_last, p.causal, p.scale, **kw)


CASES = {
    # name: (seqlens_q, seqlens_k, hq, hkv, sink, win_first, win_last, causal)
    "square_gqa2": ([256], None, 4, 2, "normal", 0, 0, True),
    "ragged_extend": ([1, 127, 129, 300], [1, 200, 129, 700], 8, 2, (-2.0, 4.0), 0, 0, True),
    "mha": ([200], [260], 2, 2, "normal", 0, 0, True),
    "odd_group": ([190], [333], 6, 2, "normal", 0, 0, True),
    "no_sink": ([300], [300], 4, 1, None, 0, 0, True),
    "non_causal": ([150, 33], [290, 140], 4, 2, "normal", 0, 0, False),
    "window_small": ([400], [650], 4, 2, (-2.0, 4.0), 20, 100, True),
    "sliding_only": ([300], [500], 2, 1, "normal", 0, 64, True),
    "more_q_than_k": ([300, 10], [100, 0], 4, 2, "normal", 0, 0, True),
    "group8": ([512], [1024], 16, 2, (-2.0, 4.0), 0, 0, True),
    # the sglang window (first 1024 + last 7168) past 8192 keys: the key tiles in the
    # gap between the windows see no query row, a first window wider than a tile
    "window_1024_7168": ([384], [9000], 2, 1, (-2.0, 4.0), 1024, 7168, True),
    # more than 32 key tiles in several (KV head, request) groups: the head-dim-128
    # kernel launches its key tiles in bands of 16, the head-dim-64 one tile-major
    "banded_groups": ([300, 4100], [5000, 4200], 4, 2, "normal", 0, 0, True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_bwd_matches_oracle(ext, name):
    sq, sk, hq, hkv, sink, F_, W, causal = CASES[name]
    p = wl.make_prefill(seqlens_q=sq, seqlens_k=sk, hq=hq, hkv=hkv, d=64, sink=sink, win_first=F_,
                        win_last=W, causal=causal, with_dout=True, seed=17)
    dq, dk, dv, ds = run_fwd_bwd(ext, p)
    rq, rk, rv, rs, _, _ = oracle_bwd(p)
    assert_grad_close(dq, rq, f"{name} dq")
    assert_grad_close(dk, rk, f"{name} dk")
    assert_grad_close(dv, rv, f"{name} dv")
    if p.sink is None:
        assert ds is None
    else:
        assert_grad_close(ds, rs, f"{name} dsink")


# head_dim 128 (bwd_main128_kernel: 64-query steps, dQ^T with the head dims on the TMEM lanes).
D128_CASES = ["square_gqa2", "ragged_extend", "mha", "no_sink", "non_causal", "window_small", "more_q_than_k",
              "window_1024_7168", "banded_groups"]


@pytest.mark.parametrize("name", D128_CASES)
def test_bwd_d128_matches_oracle(ext, name):
    sq, sk, hq, hkv, sink, F_, W, causal = CASES[name]
    p = wl.make_prefill(seqlens_q=sq, seqlens_k=sk, hq=hq, hkv=hkv, d=128, sink=sink, win_first=F_,
                        win_last=W, causal=causal, with_dout=True, seed=19)
    dq, dk, dv, ds = run_fwd_bwd(ext, p)
    rq, rk, rv, rs, _, _ = oracle_bwd(p)
    assert_grad_close(dq, rq, f"{name} dq")
    assert_grad_close(dk, rk, f"{name} dk")
    assert_grad_close(dv, rv, f"{name} dv")
    if p.sink is not None:
        assert_grad_close(ds, rs, f"{name} dsink")


def test_bwd_sink_plus_infinity(ext):
    p = wl.make_prefill(seqlens_q=[140], hq=4, hkv=2, d=64, sink="normal", with_dout=True, seed=5)
    p.sink = torch.full((4,), math.inf)
    dq, dk, dv, ds = run_fwd_bwd(ext, p)
    for g in (dq, dk, dv, ds):
        assert torch.all(g.float() == 0)


@pytest.mark.slow
def test_train_full_size_sampled(ext):
    """Training workload at full size (B 2, L 8192, Hq 64, Hkv 8): dK/dV of KV
    head 0, dQ of its eight query heads and their dsink, both requests."""
    p = wl.workload("train")
    dq, dk, dv, ds = run_fwd_bwd(ext, p)
    rq, rk, rv, rs, _, _ = oracle_bwd(p, kv_heads=[0], check_identity=False)
    assert_grad_close(dq[:, :8], rq[:, :8], "dq")
    assert_grad_close(dk[:, :1], rk[:, :1], "dk")
    assert_grad_close(dv[:, :1], rv[:, :1], "dv")
    assert_grad_close(ds[:8], rs[:8], "dsink")


@pytest.mark.slow
def test_train_d128_full_size_sampled(ext):
    """Head-dim-128 training workload at full size (B 2, L 8192, Hq 32, Hkv 8; the
    key tiles launched in bands): dK/dV of KV head 0, dQ of its four query heads
    and their dsink, both requests."""
    p = wl.workload("train_d128")
    dq, dk, dv, ds = run_fwd_bwd(ext, p)
    rq, rk, rv, rs, _, _ = oracle_bwd(p, kv_heads=[0], check_identity=False)
    assert_grad_close(dq[:, :4], rq[:, :4], "dq")
    assert_grad_close(dk[:, :1], rk[:, :1], "dk")
    assert_grad_close(dv[:, :1], rv[:, :1], "dv")
    assert_grad_close(ds[:4], rs[:4], "dsink")


def test_train_step_cuda_graph_replay(ext):
    """Forward + backward captured once in a CUDA graph (the backward's scratch
    comes from the stream-ordered pool inside the capture) and replayed on new
    inputs copied into the captured buffers; each replay equals eager calls."""
    p = wl.make_prefill(seqlens_q=[300, 129], seqlens_k=[500, 129], hq=8, hkv=2, d=64, sink="normal",
                        with_dout=True, seed=41)
    d = "cuda"
    bufs = {n: getattr(p, n).to(d) for n in ("q", "k", "v", "sink", "dout", "cu_seqlens_q", "cu_seqlens_k")}
    out = torch.empty_like(bufs["q"])
    lse = torch.empty((p.hq, p.q.shape[0]), dtype=torch.float32, device=d)
    dq, dk, dv = torch.empty_like(bufs["q"]), torch.empty_like(bufs["k"]), torch.empty_like(bufs["v"])
    dsink = torch.empty_like(bufs["sink"])

    def step():
        ext.attn_sink_fwd(bufs["q"], bufs["k"], bufs["v"], bufs["sink"], bufs["cu_seqlens_q"],
                          bufs["cu_seqlens_k"], p.max_seqlen_q, p.max_seqlen_k, out=out, lse=lse)
        ext.attn_sink_bwd(bufs["q"], bufs["k"], bufs["v"], bufs["sink"], out, lse, bufs["dout"],
                          bufs["cu_seqlens_q"], bufs["cu_seqlens_k"], p.max_seqlen_q, p.max_seqlen_k, dq=dq,
                          dk=dk, dv=dv, dsink=dsink)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        step()
    g = torch.Generator().manual_seed(5)
    for _ in range(2):
        for n in ("q", "k", "v", "dout"):
            bufs[n].copy_(torch.randn(bufs[n].shape, generator=g).to(torch.bfloat16))
        graph.replay()
        torch.cuda.synchronize()
        assert ext.device_status() == 0
        got = [t.clone() for t in (out, lse, dk, dv, dq, dsink)]
        step()
        torch.cuda.synchronize()
        assert torch.equal(got[0], out) and torch.equal(got[1], lse)
        assert torch.equal(got[2], dk) and torch.equal(got[3], dv)
        assert rel_fro(got[4], dq) <= 1e-3 and rel_fro(got[5], dsink) <= 1e-4  # fp32 atomics, order not fixed
