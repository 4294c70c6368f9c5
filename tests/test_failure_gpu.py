"""The bounded wait behind every pipeline barrier, run on the GPU: a wait on a
barrier that nothing completes gives up after its limit, the host reads
ATTN_SINK_DEV_TIMEOUT, and the same context then runs the forward correctly."""
import time

import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import _lib
from paged_kv_sink_gb300 import workloads as wl
from parity import assert_lse_close, assert_out_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ext():
    from paged_kv_sink_gb300 import build
    build.build()
    import paged_kv_sink_gb300 as ext
    return ext


def test_wait_that_is_completed_returns_without_status(ext):
    ext.device_status()  # clear
    ext.attn_sink_selftest_wait(True)
    torch.cuda.synchronize()
    assert ext.device_status() == 0


def test_wait_that_is_never_completed_times_out_and_the_context_survives(ext):
    ext.device_status()  # clear
    t0 = time.monotonic()
    ext.attn_sink_selftest_wait(False)
    torch.cuda.synchronize()
    waited = time.monotonic() - t0
    assert ext.device_status() == _lib.DEV_TIMEOUT
    assert 0.9 <= waited < 60.0  # the wait limit is 1 s of the device's global timer
    assert ext.device_status() == 0  # reading clears it
    # the context is intact: a forward call right after is correct
    p = wl.make_prefill(seqlens_q=[200, 64], seqlens_k=[300, 64], hq=4, hkv=2, d=64, sink="normal", seed=29)
    d = "cuda"
    out, lse = ext.attn_sink_fwd(p.q.to(d), p.k.to(d), p.v.to(d), p.sink.to(d), p.cu_seqlens_q.to(d),
                                 p.cu_seqlens_k.to(d), p.max_seqlen_q, p.max_seqlen_k)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    assert_out_close(out.cpu(), O)
    assert_lse_close(lse.cpu(), LSE)
