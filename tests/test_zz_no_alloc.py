"""The allocation-free decode entry point against the allocating one and the
oracle (paged decode, sink and first/last window: sglang PR "To implement
attention-sink", Motivation; the sink term: flash-attention PR "feat: Implement
Sink Attention", Key Changes).

Some callers cannot allocate device memory when they call into the library
(an engine that reserved the GPU up front, a latency-critical path that must
not take the allocator's locks or its implicit synchronisation).  For them
attn_sink_decode_paged_noalloc keeps its scratch in a static device array.
This file is collected last on purpose: it must pass run alone in a fresh
process and after every other test.
"""
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
    return [t.cuda() for t in (dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens)], \
        (None if dc.sink is None else dc.sink.cuda())


@pytest.mark.parametrize("case", ["fits", "longer_splits"])
def test_noalloc_matches_allocating_entry_point_twice(ext, case):
    if case == "fits":
        dc = wl.make_decode(seqlens=[9000, 3000, 65, 8192], hq=32, hkv=8, d=128, page_size=64, sink=None,
                            win_first=1024, win_last=7168, seed=21)
    else:  # partials of the default split exceed the static array: fewer, longer splits
        dc = wl.make_decode(seqlens=[20000] * 64, hq=64, hkv=8, d=64, page_size=16,
                            sink=("uniform", -2.0, 4.0), seed=22)
        # the plan sizes splits for the page table's capacity (4096 pages = 65536
        # tokens): 32 splits of 2048 tokens, 34.6 MB of partials > 32 MiB
        pad = torch.full((64, 4096 - dc.page_table.shape[1]), -1, dtype=torch.int32)
        dc.page_table = torch.cat([dc.page_table, pad], dim=1).contiguous()
    (q, kc, vc, pt, sl), sink = _dev(dc)
    ref_o, ref_l = ext.attn_sink_decode_paged(q, kc, vc, pt, sl, sink, dc.win_first, dc.win_last)
    torch.cuda.synchronize()
    # the oracle on every request of the small case, on three requests (all heads) of the large one
    reqs = list(range(dc.q.shape[0])) if case == "fits" else [0, 31, 63]
    O, LSE = orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens, dc.page_size,
                                   dc.sink, dc.win_first, dc.win_last, requests=reqs)
    for _ in range(2):  # two calls in a row share (and reuse) the static scratch
        o, l = ext.attn_sink_decode_paged_noalloc(q, kc, vc, pt, sl, sink, dc.win_first, dc.win_last)
        torch.cuda.synchronize()
        assert ext.device_status() == 0
        assert_out_close(o.cpu(), ref_o.cpu())
        assert_lse_close(l.cpu(), ref_l.cpu())
        assert_out_close(o.cpu()[reqs], O[reqs], "out vs oracle")
        assert_lse_close(l.cpu()[reqs], LSE[reqs], "lse vs oracle")


def test_noalloc_rejects_oversized_requests(ext):
    B, hq, d = 4096, 64, 128  # one split per (request, head) already needs > 32 MiB
    q = torch.zeros((B, hq, d), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 16, hq, d), dtype=torch.bfloat16, device="cuda")
    pt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones(B, dtype=torch.int32, device="cuda")
    with pytest.raises(ext.AttnSinkError) as ei:
        ext.attn_sink_decode_paged_noalloc(q, kc, kc, pt, sl)
    assert ei.value.code == -2 and "scratch" in str(ei.value)
