"""Varlen forward (tcgen05 kernel) against the fp64 oracle, through the C ABI."""
import math

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


def run_fwd(ext, p, **kw):
    d = "cuda"
    out, lse = ext.attn_sink_fwd(p.q.to(d), p.k.to(d), p.v.to(d),
                                 None if p.sink is None else p.sink.to(d),
                                 p.cu_seqlens_q.to(d), p.cu_seqlens_k.to(d), p.max_seqlen_q,
                                 p.max_seqlen_k, p.win_first, p.win_last, p.causal, p.scale, **kw)
    torch.cuda.synchronize()
    assert ext.device_status() == 0
    return out.cpu(), lse.cpu()


def oracle_fwd(p, **kw):
    return orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, p.win_first,
                        p.win_last, p.causal, p.scale, **kw)


CASES = {
    # name: (seqlens_q, seqlens_k, hq, hkv, sink, win_first, win_last, causal)
    "square_gqa2": ([256], None, 4, 2, "normal", 0, 0, True),
    "ragged_extend": ([1, 127, 128, 129, 300], [1, 132, 256, 1129, 377], 8, 2, (-2.0, 4.0), 0, 0, True),
    "mha_single_slot": ([200, 77], [260, 77], 3, 3, "normal", 0, 0, True),
    "odd_group": ([190], [400], 6, 2, None, 0, 0, True),
    "non_causal": ([200, 5], [333, 129], 4, 1, "normal", 0, 0, False),
    "window_small": ([500, 130], [700, 130], 4, 2, (-2.0, 4.0), 20, 100, True),
    "window_1024_7168": ([384], [9000], 2, 1, (-2.0, 4.0), 1024, 7168, True),
    "sliding_only": ([300], [600], 2, 2, "normal", 0, 64, True),
    "more_q_than_k": ([300, 10], [100, 0], 4, 2, "normal", 0, 0, True),
    "group8_long": ([1000], [3000], 16, 2, (-2.0, 4.0), 0, 0, True),
    # many key tiles per CTA: the softmax can run ahead of the MMA issuer
    "long_prefix": ([256, 384], [20000, 16384], 4, 2, (-2.0, 4.0), 0, 0, True),
}


@pytest.mark.parametrize("name", list(CASES))
def test_fwd_matches_oracle(ext, name):
    sq, sk, hq, hkv, sink, F_, W, causal = CASES[name]
    p = wl.make_prefill(seqlens_q=sq, seqlens_k=sk, hq=hq, hkv=hkv, d=64, sink=sink,
                        win_first=F_, win_last=W, causal=causal, seed=11)
    out, lse = run_fwd(ext, p)
    O, LSE = oracle_fwd(p)
    assert_out_close(out, O, what=name)
    assert_lse_close(lse, LSE, what=name)


# head_dim 128 (one CTA per SM, two 64-wide swizzle atoms per operand row):
# the window run of sglang PR "To implement attention-sink" serves a model with
# 128-wide heads (Qwen3-8B: 32 query heads over 8 KV heads).
D128_CASES = ["square_gqa2", "ragged_extend", "odd_group", "non_causal", "window_small", "window_1024_7168",
              "sliding_only", "more_q_than_k", "long_prefix"]


@pytest.mark.parametrize("name", D128_CASES)
def test_fwd_d128_matches_oracle(ext, name):
    sq, sk, hq, hkv, sink, F_, W, causal = CASES[name]
    p = wl.make_prefill(seqlens_q=sq, seqlens_k=sk, hq=hq, hkv=hkv, d=128, sink=sink,
                        win_first=F_, win_last=W, causal=causal, seed=12)
    out, lse = run_fwd(ext, p)
    O, LSE = oracle_fwd(p)
    assert_out_close(out, O, what=name)
    assert_lse_close(lse, LSE, what=name)


def test_fwd_d128_gqa4_window(ext):
    """The 128-wide-head shape of the window run (4 query heads per KV head) with
    the first 1024 + last 7168 window over 9000 keys."""
    p = wl.make_prefill(seqlens_q=[300, 129], seqlens_k=[9000, 2000], hq=8, hkv=2, d=128, sink=None,
                        win_first=1024, win_last=7168, causal=True, seed=21)
    out, lse = run_fwd(ext, p)
    O, LSE = oracle_fwd(p)
    assert_out_close(out, O)
    assert_lse_close(lse, LSE)


@pytest.mark.parametrize("sig", [-math.inf, 80.0, math.inf])
def test_fwd_sink_limits(ext, sig):
    p = wl.make_prefill(seqlens_q=[150, 40], hq=4, hkv=2, d=64, sink="normal", seed=3)
    p.sink = None if sig == -math.inf else torch.full((4,), sig)
    out, lse = run_fwd(ext, p)
    O, LSE = oracle_fwd(p)
    if sig == math.inf:
        assert torch.all(out.float() == 0) and torch.all(torch.isposinf(lse))
    else:
        assert_out_close(out, O)
        assert_lse_close(lse, LSE)


def test_fwd_explicit_scale(ext):
    p = wl.make_prefill(seqlens_q=[129], hq=2, hkv=1, d=64, sink="normal", scale=0.3, seed=4)
    out, lse = run_fwd(ext, p)
    O, LSE = oracle_fwd(p)
    assert_out_close(out, O)
    assert_lse_close(lse, LSE)


def _sample_rows(p, per_req, seed=0):
    g = torch.Generator().manual_seed(seed)
    rows = {}
    for b, Lq in enumerate(p.seqlens_q):
        pick = set(torch.randint(0, Lq, (per_req,), generator=g).tolist())
        pick |= {0, Lq - 1, min(127, Lq - 1), min(128, Lq - 1)}
        rows[b] = sorted(pick)
    return rows


@pytest.mark.parametrize("name", ["prefill_tiny", "extend_varlen", "extend_window", "train", "extend_d128",
                                  "train_d128"])
def test_full_size_workloads_sampled(ext, name):
    """The named workloads at full size in the bench's launch configuration;
    sampled rows (all heads) against the oracle, the tiny one completely.  The
    head-dim-128 ones run two query heads per CTA (fwd2_kernel)."""
    p = wl.workload(name)
    out, lse = run_fwd(ext, p)
    if name == "prefill_tiny":
        O, LSE = oracle_fwd(p)
        assert_out_close(out, O)
        assert_lse_close(lse, LSE)
        return
    rows = _sample_rows(p, 24)
    O, LSE = oracle_fwd(p, rows=rows)
    cq = p.cu_seqlens_q.tolist()
    idx = np.concatenate([np.asarray(r) + cq[b] for b, r in rows.items()])
    assert_out_close(out[idx], O[idx], what=name)
    assert_lse_close(lse[:, idx], LSE[:, idx], what=name)
