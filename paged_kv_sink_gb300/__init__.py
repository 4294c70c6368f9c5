"""Attention with an attention sink on GB300 (sm_103a).

The compute path is the C-ABI library ``libattn_sink.so`` (hand-written CUDA
kernels); this package holds its thin Python binding, the in-tree build
script and the seeded synthetic workloads used by the tests and the bench.
"""
from ._lib import (  # noqa: F401
    EXPORTS,
    AttnSinkError,
    attn_sink_bwd,
    attn_sink_bwd_kvpacked,
    attn_sink_bwd_qkvpacked,
    attn_sink_decode_paged,
    attn_sink_decode_paged_append,
    attn_sink_decode_paged_noalloc,
    attn_sink_fwd,
    attn_sink_fwd_host,
    attn_sink_fwd_kvpacked,
    attn_sink_fwd_paged,
    attn_sink_fwd_qkvpacked,
    attn_sink_kv_append,
    attn_sink_selftest_wait,
    attn_sink_visible_ranges,
    attn_sink_visible_slots,
    device_status,
    lib,
)
from .autograd import (  # noqa: F401
    attn_sink_func,
    attn_sink_kvpacked_func,
    attn_sink_qkvpacked_func,
    attn_sink_varlen_func,
    attn_sink_varlen_kvpacked_func,
    attn_sink_varlen_qkvpacked_func,
)
