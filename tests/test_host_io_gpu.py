"""Forward on host-resident tensors (copies pipelined against the kernels by
the library) against the device entry point and the fp64 oracle."""
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


@pytest.mark.parametrize("pinned,d", [(True, 64), (False, 64), (True, 128)])
def test_fwd_host_equals_device_entry_point(ext, pinned, d):
    p = wl.make_prefill(seqlens_q=[300, 0, 1, 129, 77], seqlens_k=[1000, 20, 1, 129, 400], hq=8, hkv=2, d=d,
                        sink=(-2.0, 4.0), win_first=16, win_last=200, seed=3)
    host = {n: getattr(p, n) for n in ("q", "k", "v", "sink", "cu_seqlens_q", "cu_seqlens_k")}
    if pinned:
        host = {n: t.pin_memory() for n, t in host.items()}
    out_h, lse_h = ext.attn_sink_fwd_host(host["q"], host["k"], host["v"], host["sink"], host["cu_seqlens_q"],
                                          host["cu_seqlens_k"], p.win_first, p.win_last)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    dv = "cuda"
    out_d, lse_d = ext.attn_sink_fwd(p.q.to(dv), p.k.to(dv), p.v.to(dv), p.sink.to(dv), p.cu_seqlens_q.to(dv),
                                     p.cu_seqlens_k.to(dv), p.max_seqlen_q, p.max_seqlen_k, p.win_first,
                                     p.win_last)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu())
    assert torch.equal(lse_h, lse_d.cpu())
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first, p.win_last)
    assert_out_close(out_h, O)
    assert_lse_close(lse_h, LSE)


@pytest.mark.parametrize("causal,win", [(True, (16, 700)), (False, (0, 0)), (True, (0, 0))])
def test_fwd_host_multi_chunk_matches_device_and_oracle(ext, causal, win):
    """Requests longer than one 1024-row chunk, one with fewer keys than queries
    (its first rows see no key): streaming a request chunk by chunk, each chunk
    over its key prefix, gives the device entry point's rows bit for bit."""
    p = wl.make_prefill(seqlens_q=[2500, 1100, 3], seqlens_k=[3000, 900, 50], hq=4, hkv=2, d=64,
                        sink=(-2.0, 4.0), win_first=win[0], win_last=win[1], causal=causal, seed=5)
    host = [t.pin_memory() for t in (p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)]
    out_h, lse_h = ext.attn_sink_fwd_host(*host, win_first=win[0], win_last=win[1], causal=causal)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    d = "cuda"
    out_d, lse_d = ext.attn_sink_fwd(*[t.to(d) for t in host], p.max_seqlen_q, p.max_seqlen_k, win[0], win[1],
                                     causal=causal)
    torch.cuda.synchronize()
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, win[0], win[1], causal=causal)
    assert_out_close(out_h, O)
    assert_lse_close(lse_h, LSE)


def test_fwd_host_full_size_matches_device(ext):
    """The extend_varlen workload (the bench's end-to-end path), bit-identical to
    the device entry point."""
    p = wl.workload("extend_varlen")
    host = [t.pin_memory() for t in (p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)]
    out_h, lse_h = ext.attn_sink_fwd_host(*host)
    torch.cuda.synchronize()
    d = "cuda"
    out_d, lse_d = ext.attn_sink_fwd(*[t.to(d) for t in host], p.max_seqlen_q, p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(out_h, out_d.cpu()) and torch.equal(lse_h, lse_d.cpu())


def test_fwd_host_rejects_device_tensors(ext):
    p = wl.make_prefill(seqlens_q=[10], hq=2, hkv=1, d=64, sink="normal", seed=1)
    with pytest.raises(TypeError):
        ext.attn_sink_fwd_host(p.q.cuda(), p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
