"""Paged-cache append, decode with the new token appended in the same call
(also replayed from a CUDA graph), and varlen extend through a page table,
against the fp64 oracle through the C ABI."""
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


def _new_rows(n, hkv, d, seed):
    g = torch.Generator().manual_seed(seed)
    k = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16)
    v = torch.randn(n, hkv, d, generator=g).to(torch.bfloat16)
    return k, v


@pytest.mark.parametrize("page_size,d", [(16, 64), (7, 128), (64, 64)])
def test_kv_append_bit_exact(ext, page_size, d):
    pe = wl.make_paged_extend(seqlens_q=[3, 1, 40, 0], seqlens_k=[10, 1, 300, 5], hq=4, hkv=2, d=d,
                              page_size=page_size, seed=7, extra_pages=3)
    dev = "cuda"
    kc, vc = pe.k_cache.to(dev), pe.v_cache.to(dev)
    ext.attn_sink_kv_append(pe.k_new.to(dev), pe.v_new.to(dev), kc, vc, pe.page_table.to(dev),
                            pe.seqlens_k.to(dev), cu_new=pe.cu_seqlens_q.to(dev))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    want_k, want_v = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new,
                                   page_size, cu_new=pe.cu_seqlens_q)
    assert torch.equal(kc.cpu(), want_k)
    assert torch.equal(vc.cpu(), want_v)


DECODE_CASES = [
    # (hq, hkv, d, page_size, seqlens, win_first, win_last, sink)
    (8, 2, 64, 16, [1, 17, 300, 4096], 0, 0, ("uniform", -2.0, 4.0)),
    (8, 2, 128, 64, [9000, 100], 1024, 7168, None),
    (16, 4, 64, 5, [33, 2, 700], 0, 64, ("uniform", -2.0, 4.0)),
]


@pytest.mark.parametrize("case", DECODE_CASES, ids=lambda c: f"d{c[2]}ps{c[3]}w{c[5]}-{c[6]}")
def test_decode_append_matches_oracle(ext, case):
    hq, hkv, d, ps, seqlens, F_, W, sink = case
    dc = wl.make_decode(seqlens=seqlens, hq=hq, hkv=hkv, d=d, page_size=ps, sink=sink, win_first=F_,
                        win_last=W, seed=3, extra_pages=2)
    kn, vn = _new_rows(len(seqlens), hkv, d, seed=11)
    dev = "cuda"
    kc, vc = dc.k_cache.to(dev), dc.v_cache.to(dev)
    out, lse = ext.attn_sink_decode_paged_append(dc.q.to(dev), kn.to(dev), vn.to(dev), kc, vc,
                                                 dc.page_table.to(dev), dc.seqlens.to(dev),
                                                 None if dc.sink is None else dc.sink.to(dev), F_, W)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    kw, vw = orc.kv_append(dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens, kn, vn, ps)
    assert torch.equal(kc.cpu(), kw) and torch.equal(vc.cpu(), vw)
    O, LSE = orc.attn_decode_paged(dc.q, kw, vw, dc.page_table, dc.seqlens, ps, dc.sink, F_, W)
    assert_out_close(out.cpu(), O)
    assert_lse_close(lse.cpu(), LSE)


def test_decode_append_cuda_graph_replay(ext):
    """One captured decode-with-append, replayed for three consecutive tokens:
    new q / K / V and lengths are copied into the captured buffers between
    replays, and each replay matches the oracle run on the same inputs."""
    hq, hkv, d, ps = 8, 2, 64, 16
    dc = wl.make_decode(seqlens=[40, 1000, 7], hq=hq, hkv=hkv, d=d, page_size=ps, seed=5, extra_pages=3)
    B = 3
    # room for three more tokens in every request: lengths grow from L-3+1 to L
    seq0 = dc.seqlens - 2
    dev = "cuda"
    q_buf = torch.zeros(B, hq, d, dtype=torch.bfloat16, device=dev)
    kn_buf = torch.zeros(B, hkv, d, dtype=torch.bfloat16, device=dev)
    vn_buf = torch.zeros(B, hkv, d, dtype=torch.bfloat16, device=dev)
    len_buf = seq0.to(dev)
    kc, vc = dc.k_cache.to(dev), dc.v_cache.to(dev)
    pt = dc.page_table.to(dev)
    sink = dc.sink.to(dev)
    out = torch.empty(B, hq, d, dtype=torch.bfloat16, device=dev)
    lse = torch.empty(B, hq, dtype=torch.float32, device=dev)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):  # warm-up outside capture (pool, function attributes)
        ext.attn_sink_decode_paged_append(q_buf, kn_buf, vn_buf, kc.clone(), vc.clone(), pt, len_buf, sink,
                                          out=out, lse=lse)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, capture_error_mode="thread_local"):
        ext.attn_sink_decode_paged_append(q_buf, kn_buf, vn_buf, kc, vc, pt, len_buf, sink, out=out, lse=lse)
    k_ref, v_ref = dc.k_cache.clone(), dc.v_cache.clone()
    g = torch.Generator().manual_seed(77)
    for step in range(3):
        q = torch.randn(B, hq, d, generator=g).to(torch.bfloat16)
        kn = torch.randn(B, hkv, d, generator=g).to(torch.bfloat16)
        vn = torch.randn(B, hkv, d, generator=g).to(torch.bfloat16)
        lens = (seq0 + step).to(torch.int32)
        q_buf.copy_(q)
        kn_buf.copy_(kn)
        vn_buf.copy_(vn)
        len_buf.copy_(lens)
        graph.replay()
        torch.cuda.synchronize()
        assert ext.device_status() == 0
        k_ref, v_ref = orc.kv_append(k_ref, v_ref, dc.page_table, lens, kn, vn, ps)
        O, LSE = orc.attn_decode_paged(q, k_ref, v_ref, dc.page_table, lens, ps, dc.sink)
        assert_out_close(out.cpu(), O, what=f"replay {step}")
        assert_lse_close(lse.cpu(), LSE, what=f"replay {step}")
    assert torch.equal(kc.cpu(), k_ref) and torch.equal(vc.cpu(), v_ref)


FWD_CASES = {
    # name: (seqlens_q, seqlens_k, hq, hkv, page_size, sink, win_first, win_last, append)
    "ps16_append": ([1, 127, 300, 129], [1, 400, 1129, 129], 8, 2, 16, (-2.0, 4.0), 0, 0, True),
    "ps8_prefilled": ([200, 77], [260, 77], 4, 1, 8, "normal", 0, 0, False),
    "ps64_window": ([500, 130], [3000, 130], 4, 2, 64, (-2.0, 4.0), 20, 700, True),
    "ps128_nosink": ([256], [1000], 2, 2, 128, None, 0, 0, True),
    "ps256_sliding": ([300], [900], 4, 2, 256, "normal", 0, 64, True),
    "ps32_first_last": ([384], [9000], 2, 1, 32, (-2.0, 4.0), 1024, 7168, True),
}


@pytest.mark.parametrize("name,d", [(n, 64) for n in FWD_CASES] +
                         [(n, 128) for n in ("ps16_append", "ps8_prefilled", "ps32_first_last")])
def test_fwd_paged_matches_oracle(ext, name, d):
    sq, sk, hq, hkv, ps, sink, F_, W, append = FWD_CASES[name]
    pe = wl.make_paged_extend(seqlens_q=sq, seqlens_k=sk, hq=hq, hkv=hkv, d=d, page_size=ps, sink=sink,
                              win_first=F_, win_last=W, seed=13, extra_pages=4)
    kw, vw = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new, ps,
                           cu_new=pe.cu_seqlens_q)
    dev = "cuda"
    if append:
        kc, vc = pe.k_cache.to(dev), pe.v_cache.to(dev)
        kn, vn = pe.k_new.to(dev), pe.v_new.to(dev)
    else:
        kc, vc = kw.to(dev), vw.to(dev)
        kn = vn = None
    out, lse = ext.attn_sink_fwd_paged(pe.q.to(dev), kc, vc, pe.page_table.to(dev), pe.cu_seqlens_q.to(dev),
                                       pe.seqlens_k.to(dev), pe.max_seqlen_q, pe.max_seqlen_k,
                                       None if pe.sink is None else pe.sink.to(dev), kn, vn, F_, W)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    assert torch.equal(kc.cpu(), kw) and torch.equal(vc.cpu(), vw)
    O, LSE = orc.attn_fwd_paged(pe.q, kw, vw, pe.page_table, pe.seqlens_k, pe.cu_seqlens_q, ps, pe.sink,
                                F_, W, True)
    assert_out_close(out.cpu(), O, what=name)
    assert_lse_close(lse.cpu(), LSE, what=name)


def test_fwd_paged_equals_contiguous_fwd(ext):
    """The paged forward on a cache reproduces attn_sink_fwd on the same tokens
    laid out contiguously (same kernel arithmetic, only the loads differ)."""
    pe = wl.make_paged_extend(seqlens_q=[129, 300], seqlens_k=[700, 300], hq=8, hkv=2, d=64, page_size=16,
                              seed=21)
    kw, vw = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new, 16,
                           cu_new=pe.cu_seqlens_q)
    K, cu_k = orc.gather_paged(kw, pe.page_table, pe.seqlens_k, 16)
    V, _ = orc.gather_paged(vw, pe.page_table, pe.seqlens_k, 16)
    dev = "cuda"
    out_p, lse_p = ext.attn_sink_fwd_paged(pe.q.to(dev), kw.to(dev), vw.to(dev), pe.page_table.to(dev),
                                           pe.cu_seqlens_q.to(dev), pe.seqlens_k.to(dev), pe.max_seqlen_q,
                                           pe.max_seqlen_k, pe.sink.to(dev))
    out_c, lse_c = ext.attn_sink_fwd(pe.q.to(dev), K.contiguous().to(dev), V.contiguous().to(dev),
                                     pe.sink.to(dev), pe.cu_seqlens_q.to(dev),
                                     torch.as_tensor(cu_k, dtype=torch.int32).to(dev), pe.max_seqlen_q,
                                     pe.max_seqlen_k)
    torch.cuda.synchronize()
    assert torch.equal(out_p.cpu(), out_c.cpu())
    assert torch.equal(lse_p.cpu(), lse_c.cpu())


def test_fwd_paged_rejects_page_size(ext):
    pe = wl.make_paged_extend(seqlens_q=[10], seqlens_k=[30], hq=2, hkv=1, d=64, page_size=24, seed=1)
    dev = "cuda"
    with pytest.raises(ext.AttnSinkError) as ei:
        ext.attn_sink_fwd_paged(pe.q.to(dev), pe.k_cache.to(dev), pe.v_cache.to(dev), pe.page_table.to(dev),
                                pe.cu_seqlens_q.to(dev), pe.seqlens_k.to(dev), 10, 30, pe.sink.to(dev))
    assert ei.value.code == -2


def test_extend_paged_full_size_sampled(ext):
    """The extend_paged workload at full size in the bench's launch
    configuration (chunk appended by the call); sampled rows of every head
    against the oracle."""
    pe = wl.workload("extend_paged")
    dev = "cuda"
    kc, vc = pe.k_cache.to(dev), pe.v_cache.to(dev)
    out, lse = ext.attn_sink_fwd_paged(pe.q.to(dev), kc, vc, pe.page_table.to(dev), pe.cu_seqlens_q.to(dev),
                                       pe.seqlens_k.to(dev), pe.max_seqlen_q, pe.max_seqlen_k, pe.sink.to(dev),
                                       pe.k_new.to(dev), pe.v_new.to(dev))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    kw, vw = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new,
                           pe.page_size, cu_new=pe.cu_seqlens_q)
    assert torch.equal(kc.cpu(), kw) and torch.equal(vc.cpu(), vw)
    g = torch.Generator().manual_seed(0)
    rows = {}
    for b, Lq in enumerate(pe.seqlens_q):
        pick = set(torch.randint(0, Lq, (16,), generator=g).tolist()) | {0, Lq - 1}
        rows[b] = sorted(pick)
    O, LSE = orc.attn_fwd_paged(pe.q, kw, vw, pe.page_table, pe.seqlens_k, pe.cu_seqlens_q, pe.page_size,
                                pe.sink, rows=rows)
    cq = pe.cu_seqlens_q.tolist()
    idx = np.concatenate([np.asarray(r) + cq[b] for b, r in rows.items()])
    assert_out_close(out.cpu()[idx], O[idx])
    assert_lse_close(lse.cpu()[:, idx], LSE[:, idx])


def test_kv_append_bad_rows_are_skipped_and_flagged(ext):
    """A page id outside the cache and a request with more new rows than cached
    tokens are skipped (no write anywhere) and raise the device status bits."""
    pe = wl.make_paged_extend(seqlens_q=[2, 3, 1], seqlens_k=[10, 2, 40], hq=2, hkv=2, d=64, page_size=16,
                              seed=9, extra_pages=2)
    pt = pe.page_table.clone()
    pt[2, 2] = pe.k_cache.shape[0] + 7  # request 2's new token (position 39) lands in page index 2
    dev = "cuda"
    kc, vc = pe.k_cache.to(dev), pe.v_cache.to(dev)
    ext.device_status()  # clear
    ext.attn_sink_kv_append(pe.k_new.to(dev), pe.v_new.to(dev), kc, vc, pt.to(dev), pe.seqlens_k.to(dev),
                            cu_new=pe.cu_seqlens_q.to(dev))
    torch.cuda.synchronize()
    bits = ext.device_status()
    assert bits & ext._lib.DEV_PAGE_OOB and bits & ext._lib.DEV_SEQLEN_OOB
    # request 0 is appended normally; request 1 (3 rows, 2 tokens): rows with t >= 0 are written,
    # the one at t = -1 is skipped; request 2's row is skipped
    want_k, _ = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table[:1], pe.seqlens_k[:1], pe.k_new[:2],
                              pe.v_new[:2], 16, cu_new=torch.tensor([0, 2], dtype=torch.int32))
    got = kc.cpu()
    flat_got, flat_want, flat_old = got.reshape(-1, 2, 64), want_k.reshape(-1, 2, 64), pe.k_cache.reshape(-1, 2, 64)
    pt0 = pe.page_table.numpy()
    for t in (8, 9):  # request 0's two new rows
        sl = orc.paged_slot(pt0, 0, t, 16)
        assert torch.equal(flat_got[sl], flat_want[sl])
    for t, r in ((0, 3), (1, 4)):  # request 1: rows 1 and 2 of its three land on tokens 0 and 1
        sl = orc.paged_slot(pt0, 1, t, 16)
        assert torch.equal(flat_got[sl], pe.k_new[r])
    touched = {orc.paged_slot(pt0, 0, t, 16) for t in (8, 9)} | {orc.paged_slot(pt0, 1, t, 16) for t in (0, 1)}
    for sl in range(flat_old.shape[0]):
        if sl not in touched:
            assert torch.equal(flat_got[sl], flat_old[sl])


def test_kv_append_rows_past_max_new_are_flagged(ext):
    """max_new sizes the grid: a request with more new rows than the grid covers
    leaves its extra rows unwritten and raises the sequence-length status bit."""
    pe = wl.make_paged_extend(seqlens_q=[10, 1], seqlens_k=[30, 5], hq=2, hkv=2, d=64, page_size=16, seed=4)
    dev = "cuda"
    kc, vc = pe.k_cache.to(dev), pe.v_cache.to(dev)
    ext.device_status()
    ext.attn_sink_kv_append(pe.k_new.to(dev), pe.v_new.to(dev), kc, vc, pe.page_table.to(dev),
                            pe.seqlens_k.to(dev), cu_new=pe.cu_seqlens_q.to(dev), max_new=2)
    torch.cuda.synchronize()
    assert ext.device_status() & ext._lib.DEV_SEQLEN_OOB
    # the grid covers 8 rows per request: request 0's rows 0..7 land, rows 8 and 9 do not
    pt0 = pe.page_table.numpy()
    flat_got, flat_old = kc.cpu().reshape(-1, 2, 64), pe.k_cache.reshape(-1, 2, 64)
    for r in range(10):
        sl = orc.paged_slot(pt0, 0, 20 + r, 16)
        assert torch.equal(flat_got[sl], pe.k_new[r] if r < 8 else flat_old[sl])


def test_fwd_paged_bad_page_is_flagged(ext):
    pe = wl.make_paged_extend(seqlens_q=[64], seqlens_k=[200], hq=2, hkv=1, d=64, page_size=16, seed=2)
    pt = pe.page_table.clone()
    pt[0, 3] = -5
    dev = "cuda"
    ext.device_status()
    ext.attn_sink_fwd_paged(pe.q.to(dev), pe.k_cache.to(dev), pe.v_cache.to(dev), pt.to(dev),
                            pe.cu_seqlens_q.to(dev), pe.seqlens_k.to(dev), 64, 200, pe.sink.to(dev))
    torch.cuda.synchronize()
    assert ext.device_status() & ext._lib.DEV_PAGE_OOB


def test_fwd_paged_empty_and_zero_length_requests(ext):
    dev = "cuda"
    # a request with no new rows and one with a single token between two regular ones
    pe = wl.make_paged_extend(seqlens_q=[50, 0, 1, 70], seqlens_k=[90, 33, 1, 70], hq=4, hkv=2, d=64,
                              page_size=32, seed=6)
    out, lse = ext.attn_sink_fwd_paged(pe.q.to(dev), pe.k_cache.to(dev), pe.v_cache.to(dev),
                                       pe.page_table.to(dev), pe.cu_seqlens_q.to(dev), pe.seqlens_k.to(dev),
                                       pe.max_seqlen_q, pe.max_seqlen_k, pe.sink.to(dev), pe.k_new.to(dev),
                                       pe.v_new.to(dev))
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    kw, vw = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new, 32,
                           cu_new=pe.cu_seqlens_q)
    O, LSE = orc.attn_fwd_paged(pe.q, kw, vw, pe.page_table, pe.seqlens_k, pe.cu_seqlens_q, 32, pe.sink)
    assert_out_close(out.cpu(), O)
    assert_lse_close(lse.cpu(), LSE)
    # an empty batch is a no-op
    q0 = torch.empty((0, 4, 64), dtype=torch.bfloat16, device=dev)
    out0, _ = ext.attn_sink_fwd_paged(q0, pe.k_cache.to(dev), pe.v_cache.to(dev), pe.page_table[:0].to(dev),
                                      torch.zeros(1, dtype=torch.int32, device=dev),
                                      torch.zeros(0, dtype=torch.int32, device=dev), 0, 0, pe.sink.to(dev))
    assert out0.shape == (0, 4, 64)
