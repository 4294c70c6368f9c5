"""Pins for the CPU fp64 oracle: each test ties it to something other than itself.

* plain causal softmax attention from torch's own ``scaled_dot_product_attention``
  (sink = -inf reduces to the textbook operation);
* the closed form of the sink: O_sink = O_std * Z / (Z + e^sigma),
  LSE_sink = logaddexp(LSE_std, sigma) (flash-attention PR "feat: Implement
  Sink Attention", Description: an extra logit in the softmax);
* the limit sigma -> +inf (output -> 0);
* the first/last-window rule against brute force and against attention over
  the explicitly gathered first-F + last-W tokens (sglang PR "To implement
  attention-sink", suggested code);
* paging invariances; GQA = MHA with replicated K/V;
* gradients against central finite differences and against torch autograd of
  an appended-sink-column formulation.
"""
import math
import os

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _sdpa_causal(q, k, v, scale):
    """Textbook causal attention for Lq == Lk via torch (fp64, GQA)."""
    qt = torch.as_tensor(q).permute(1, 0, 2)[None]  # (1, Hq, L, d)
    kt = torch.as_tensor(k).permute(1, 0, 2)[None]
    vt = torch.as_tensor(v).permute(1, 0, 2)[None]
    o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True, scale=scale, enable_gqa=True)
    return o[0].permute(1, 0, 2).numpy()


def _lse_causal(q, k, scale):
    """logsumexp of the causal scaled logits, per (head, row), via torch."""
    qt = torch.as_tensor(q).permute(1, 0, 2)  # (Hq, L, d)
    kt = torch.as_tensor(k).permute(1, 0, 2)
    G = qt.shape[0] // kt.shape[0]
    kt = kt.repeat_interleave(G, dim=0)
    s = scale * qt @ kt.transpose(1, 2)
    L = s.shape[-1]
    s = s.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), -math.inf)
    return torch.logsumexp(s, dim=-1).numpy()  # (Hq, L)


def _tiny_prefill(seed, L=37, hq=4, hkv=2, d=16, sink="normal", batch=2):
    p = wl.make_prefill(seqlens_q=[L, L - 11][:batch], hq=hq, hkv=hkv, d=d, sink=sink, seed=seed)
    return p


@pytest.mark.parametrize("seed", [0, 1])
def test_no_sink_is_causal_softmax_attention(seed):
    p = _tiny_prefill(seed, sink=None)
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, None, p.cu_seqlens_q, p.cu_seqlens_k)
    q, k, v = orc.to64(p.q), orc.to64(p.k), orc.to64(p.v)
    for b in range(p.batch):
        a, e = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        ref = _sdpa_causal(q[a:e], k[a:e], v[a:e], p.softmax_scale)
        np.testing.assert_allclose(O[a:e], ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(LSE[:, a:e], _lse_causal(q[a:e], k[a:e], p.softmax_scale),
                                   rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", [0, 3])
def test_sink_closed_form(seed):
    p = _tiny_prefill(seed, sink="normal")
    p.sink = p.sink * 3  # spread the sink logits so they matter
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    q, k, v = orc.to64(p.q), orc.to64(p.k), orc.to64(p.v)
    sig = orc.to64(p.sink)
    for b in range(p.batch):
        a, e = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
        o_std = _sdpa_causal(q[a:e], k[a:e], v[a:e], p.softmax_scale)  # (L, Hq, d)
        lse_std = _lse_causal(q[a:e], k[a:e], p.softmax_scale)          # (Hq, L)
        # Z/(Z + e^sigma) = sigmoid(LSE_std - sigma)
        frac = 1.0 / (1.0 + np.exp(sig[:, None] - lse_std))
        np.testing.assert_allclose(O[a:e], o_std * frac.T[:, :, None], rtol=1e-11, atol=1e-12)
        np.testing.assert_allclose(LSE[:, a:e], np.logaddexp(lse_std, sig[:, None]),
                                   rtol=1e-12, atol=1e-12)


def test_sink_to_plus_infinity():
    p = _tiny_prefill(5, sink="normal")
    vmax = float(orc.to64(p.v).__abs__().max())
    q, k = orc.to64(p.q), orc.to64(p.k)
    for sig in (30.0, 80.0):
        s = torch.full((p.hq,), sig)
        O, LSE = orc.attn_fwd(p.q, p.k, p.v, s, p.cu_seqlens_q, p.cu_seqlens_k)
        for b in range(p.batch):
            a, e = int(p.cu_seqlens_q[b]), int(p.cu_seqlens_q[b + 1])
            Z = np.exp(_lse_causal(q[a:e], k[a:e], p.softmax_scale))  # (Hq, L)
            bound = math.exp(-sig) * Z * vmax * math.sqrt(p.head_dim)
            nrm = np.linalg.norm(O[a:e], axis=-1).T
            assert np.all(nrm <= bound * (1 + 1e-9))
    s = torch.full((p.hq,), math.inf)
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, s, p.cu_seqlens_q, p.cu_seqlens_k)
    assert np.all(O == 0.0) and np.all(LSE == math.inf)
    dq, dk, dv, ds, _, _ = orc.attn_bwd(p.q, p.k, p.v, s, torch.ones_like(p.q), p.cu_seqlens_q,
                                       p.cu_seqlens_k)
    for g in (dq, dk, dv, ds):
        assert np.all(g == 0.0)


def test_extend_rows_equal_tail_of_full_prefill():
    """Bottom-right alignment: a chunk of Lq new rows over Lk keys = the last Lq rows
    of full causal prefill over Lk rows (which the SDPA pin fixes)."""
    g = torch.Generator().manual_seed(7)
    Lk, Lq, hq, hkv, d = 45, 13, 4, 2, 16
    full = wl.make_prefill(seqlens_q=[Lk], hq=hq, hkv=hkv, d=d, sink="normal", g=g)
    Of, Lf = orc.attn_fwd(full.q, full.k, full.v, full.sink, full.cu_seqlens_q, full.cu_seqlens_k)
    cu_q = torch.tensor([0, Lq], dtype=torch.int32)
    Oc, Lc = orc.attn_fwd(full.q[Lk - Lq:], full.k, full.v, full.sink, cu_q, full.cu_seqlens_k)
    np.testing.assert_array_equal(Oc, Of[Lk - Lq:])
    np.testing.assert_array_equal(Lc, Lf[:, Lk - Lq:])


def test_empty_rows_and_keys():
    """Rows with no visible key: O = 0, LSE = sigma (or -inf without a sink)."""
    g = torch.Generator().manual_seed(1)
    p = wl.make_prefill(seqlens_q=[5, 3], seqlens_k=[3, 0], hq=2, hkv=1, d=8, sink="normal", g=g)
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    sig = orc.to64(p.sink)
    # request 0: rows 0,1 sit at positions -2,-1 -> nothing visible
    assert np.all(O[0:2] == 0) and np.allclose(LSE[:, 0:2], sig[:, None])
    assert np.all(O[5:8] == 0) and np.allclose(LSE[:, 5:8], sig[:, None])
    O2, LSE2 = orc.attn_fwd(p.q, p.k, p.v, None, p.cu_seqlens_q, p.cu_seqlens_k)
    assert np.all(O2[5:8] == 0) and np.all(LSE2[:, 5:8] == -math.inf)
    assert np.all(np.isfinite(O2[2:5]))


def _golden_windows():
    rows = []
    with open(os.path.join(GOLDEN, "window_slices.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                rows.append(tuple(int(x) for x in line.split()))
    return rows


def test_window_golden_slices():
    rows = _golden_windows()
    assert len(rows) >= 5
    for L, F_, W, a0, b0, a1, b1 in rows:
        assert orc.visible_ranges(L, F_, W) == [(a0, b0), (a1, b1)], (L, F_, W)


def test_visible_ranges_brute_force():
    for L in range(1, 301):
        for F_ in (0, 1, 3, 8, 64):
            for W in (0, 1, 5, 16, 100):
                (a0, b0), (a1, b1) = orc.visible_ranges(L, F_, W)
                got = set(range(a0, b0)) | set(range(a1, b1))
                assert (b0 - a0) + (b1 - a1) == len(got)  # disjoint
                if W <= 0:
                    want = set(range(L))
                else:
                    want = {t for t in range(L) if t < F_ or t >= L - W}
                assert got == want, (L, F_, W)
                assert a0 <= b0 <= a1 <= b1


def test_visible_mask_matches_ranges():
    Lk = 90
    for F_, W in ((4, 10), (0, 7), (20, 100), (3, 1)):
        m = orc.visible_mask(np.arange(Lk), Lk, F_, W, True)
        for p in range(Lk):
            (a0, b0), (a1, b1) = orc.visible_ranges(p + 1, F_, W)
            want = np.zeros(Lk, bool)
            want[a0:b0] = True
            want[a1:b1] = True
            np.testing.assert_array_equal(m[p], want)


def _decode_case(seed, seqlens, ps, F_=0, W=0, sink=("uniform", -2.0, 4.0), hq=4, hkv=2, d=16):
    return wl.make_decode(seqlens=seqlens, hq=hq, hkv=hkv, d=d, page_size=ps, sink=sink,
                          win_first=F_, win_last=W, seed=seed, extra_pages=3)


@pytest.mark.parametrize("sink", [None, ("uniform", -2.0, 4.0)])
def test_window_equals_gathered_tokens(sink):
    """Decode with the window = plain attention over cat(first F, last W) tokens."""
    F_, W = 5, 9
    dc = _decode_case(2, [3, 14, 15, 40, 77], ps=4, F_=F_, W=W, sink=sink)
    O, LSE = orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens,
                                   dc.page_size, dc.sink, F_, W)
    G = dc.hq // dc.hkv
    kflat = dc.k_cache.reshape(-1, dc.hkv, dc.head_dim).double()
    vflat = dc.v_cache.reshape(-1, dc.hkv, dc.head_dim).double()
    for b, L in enumerate(dc.seqlens.tolist()):
        # the page-table rows of sglang's req_to_token, token-level (page size 1 view)
        tok = [int(dc.page_table[b, t // 4]) * 4 + t % 4 for t in range(L)]
        if L > F_ + W:
            sel = tok[:F_] + tok[L - W:L]
        else:
            sel = tok[:L]
        kk = kflat[sel].permute(1, 0, 2)[None]  # (1, Hkv, n, d)
        vv = vflat[sel].permute(1, 0, 2)[None]
        qq = dc.q[b].double()[None, :, None, :]  # (1, Hq, 1, d)
        o = F.scaled_dot_product_attention(qq, kk, vv, scale=dc.softmax_scale, enable_gqa=True)
        o = o[0, :, 0].numpy()
        s = dc.softmax_scale * (qq[0] @ kk[0].repeat_interleave(G, 0).transpose(1, 2))  # (Hq,1,n)
        lse_std = torch.logsumexp(s[:, 0], -1).numpy()
        if sink is None:
            np.testing.assert_allclose(O[b], o, rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(LSE[b], lse_std, rtol=1e-12, atol=1e-12)
        else:
            sig = orc.to64(dc.sink)
            frac = 1.0 / (1.0 + np.exp(sig - lse_std))
            np.testing.assert_allclose(O[b], o * frac[:, None], rtol=1e-11, atol=1e-12)
            np.testing.assert_allclose(LSE[b], np.logaddexp(lse_std, sig), rtol=1e-12)


def test_prefill_window_rows_equal_gathered():
    """Each prefill row with the window on = attention over its own gathered keys."""
    F_, W = 3, 6
    g = torch.Generator().manual_seed(11)
    p = wl.make_prefill(seqlens_q=[7], seqlens_k=[26], hq=2, hkv=1, d=8, sink="normal",
                        win_first=F_, win_last=W, g=g)
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, F_, W)
    for i in range(7):
        L = 26 - 7 + i + 1  # tokens up to and including this query's position
        sel = list(range(L)) if L <= F_ + W else list(range(F_)) + list(range(L - W, L))
        Od, Ld = orc.attn_fwd(p.q[i:i + 1], p.k[sel], p.v[sel], p.sink,
                              torch.tensor([0, 1], dtype=torch.int32),
                              torch.tensor([0, len(sel)], dtype=torch.int32), causal=True,
                              scale=p.softmax_scale)
        np.testing.assert_allclose(O[i], Od[0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(LSE[:, i], Ld[:, 0], rtol=1e-13)


def test_page_permutation_invariance_and_page_size_one():
    lens = [1, 16, 17, 50, 64]
    a = _decode_case(4, lens, ps=16)
    Oa, La = orc.attn_decode_paged(a.q, a.k_cache, a.v_cache, a.page_table, a.seqlens,
                                   16, a.sink)
    # Re-home every page to a new physical id: identical logical contents.
    g = torch.Generator().manual_seed(99)
    perm = torch.randperm(a.num_pages, generator=g)
    kc = torch.empty_like(a.k_cache)
    vc = torch.empty_like(a.v_cache)
    kc[perm] = a.k_cache
    vc[perm] = a.v_cache
    pt = torch.where(a.page_table >= 0, perm[a.page_table.clamp(min=0).long()].int(),
                     a.page_table)
    Ob, Lb = orc.attn_decode_paged(a.q, kc, vc, pt, a.seqlens, 16, a.sink)
    np.testing.assert_array_equal(Oa, Ob)
    np.testing.assert_array_equal(La, Lb)
    # Page size 1: the token-level req_to_token table of the sglang backend.
    kc1 = a.k_cache.reshape(-1, 1, a.hkv, a.head_dim)
    vc1 = a.v_cache.reshape(-1, 1, a.hkv, a.head_dim)
    pt1 = torch.full((a.batch, max(lens)), -1, dtype=torch.int32)
    for b, L in enumerate(lens):
        for t in range(L):
            pt1[b, t] = int(a.page_table[b, t // 16]) * 16 + t % 16
    Oc, Lc = orc.attn_decode_paged(a.q, kc1, vc1, pt1, a.seqlens, 1, a.sink)
    np.testing.assert_array_equal(Oa, Oc)
    np.testing.assert_array_equal(La, Lc)


def test_decode_equals_last_prefill_row():
    lens = [9, 33]
    dc = _decode_case(6, lens, ps=8)
    O, LSE = orc.attn_decode_paged(dc.q, dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens,
                                   8, dc.sink)
    for b, L in enumerate(lens):
        slots = [int(dc.page_table[b, t // 8]) * 8 + t % 8 for t in range(L)]
        k = dc.k_cache.reshape(-1, dc.hkv, dc.head_dim)[slots]
        v = dc.v_cache.reshape(-1, dc.hkv, dc.head_dim)[slots]
        Op, Lp = orc.attn_fwd(dc.q[b:b + 1], k, v, dc.sink, torch.tensor([0, 1]),
                              torch.tensor([0, L]))
        np.testing.assert_allclose(O[b], Op[0], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(LSE[b], Lp[:, 0], rtol=1e-13)


def test_gqa_equals_mha_replicated():
    p = _tiny_prefill(8, hq=6, hkv=2, d=8, sink="normal")
    p.dout = torch.randn(p.q.shape, generator=torch.Generator().manual_seed(3)).to(torch.bfloat16)
    G = 3
    k_rep = p.k.repeat_interleave(G, dim=1)
    v_rep = p.v.repeat_interleave(G, dim=1)
    Og, Lg = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    Om, Lm = orc.attn_fwd(p.q, k_rep, v_rep, p.sink, p.cu_seqlens_q, p.cu_seqlens_k)
    np.testing.assert_allclose(Og, Om, rtol=1e-13, atol=1e-14)
    gq = orc.attn_bwd(p.q, p.k, p.v, p.sink, p.dout, p.cu_seqlens_q, p.cu_seqlens_k)
    gm = orc.attn_bwd(p.q, k_rep, v_rep, p.sink, p.dout, p.cu_seqlens_q, p.cu_seqlens_k)
    np.testing.assert_allclose(gq[0], gm[0], rtol=1e-11, atol=1e-12)
    tk = p.k.shape[0]
    np.testing.assert_allclose(gq[1], gm[1].reshape(tk, 2, G, 8).sum(2), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(gq[2], gm[2].reshape(tk, 2, G, 8).sum(2), rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(gq[3], gm[3], rtol=1e-11, atol=1e-12)


def _loss(q, k, v, s, dout, cu_q, cu_k, F_, W):
    O, _ = orc.attn_fwd(q, k, v, s, cu_q, cu_k, F_, W)
    return float((O * dout).sum())


@pytest.mark.parametrize("F_,W", [(0, 0), (2, 4)])
def test_backward_central_differences(F_, W):
    rng = np.random.default_rng(5)
    cu_q = np.array([0, 9, 14])
    cu_k = np.array([0, 12, 17])
    hq, hkv, d = 4, 2, 8
    q = rng.standard_normal((14, hq, d))
    k = rng.standard_normal((17, hkv, d))
    v = rng.standard_normal((17, hkv, d))
    s = rng.standard_normal(hq)
    do = rng.standard_normal((14, hq, d))
    dq, dk, dv, ds, _, _ = orc.attn_bwd(q, k, v, s, do, cu_q, cu_k, F_, W)
    h = 1e-6

    def fd(x, name):
        g = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            old = x[idx]
            x[idx] = old + h
            lp = _loss(q, k, v, s, do, cu_q, cu_k, F_, W)
            x[idx] = old - h
            lm = _loss(q, k, v, s, do, cu_q, cu_k, F_, W)
            x[idx] = old
            g[idx] = (lp - lm) / (2 * h)
        return g

    for an, x in ((dq, q), (dk, k), (dv, v), (ds, s)):
        num = fd(x, "")
        err = np.linalg.norm(an - num) / max(np.linalg.norm(num), 1e-30)
        assert err <= 1e-6, err


def test_backward_against_appended_column_autograd():
    """Third opinion: sink as an appended logit column with a zero value row,
    softmax and autograd by torch (fp64)."""
    rng = np.random.default_rng(9)
    L, hq, hkv, d = 21, 4, 2, 8
    G = hq // hkv
    q = torch.tensor(rng.standard_normal((L, hq, d)), requires_grad=True)
    k = torch.tensor(rng.standard_normal((L, hkv, d)), requires_grad=True)
    v = torch.tensor(rng.standard_normal((L, hkv, d)), requires_grad=True)
    s = torch.tensor(rng.standard_normal(hq) * 2, requires_grad=True)
    do = torch.tensor(rng.standard_normal((L, hq, d)))
    scale = 1 / math.sqrt(d)
    kk = k.repeat_interleave(G, 1).permute(1, 0, 2)
    vv = v.repeat_interleave(G, 1).permute(1, 0, 2)
    logits = scale * q.permute(1, 0, 2) @ kk.transpose(1, 2)  # (Hq, L, L)
    logits = logits.masked_fill(~torch.ones(L, L, dtype=torch.bool).tril(), -math.inf)
    col = s[:, None, None].expand(hq, L, 1)
    probs = torch.softmax(torch.cat([logits, col], dim=-1), dim=-1)[..., :L]
    o = (probs @ vv).permute(1, 0, 2)
    (o * do).sum().backward()
    cu = np.array([0, L])
    dq, dk, dv, ds, O, _ = orc.attn_bwd(q.detach().numpy(), k.detach().numpy(),
                                        v.detach().numpy(), s.detach().numpy(), do.numpy(), cu, cu)
    np.testing.assert_allclose(O, o.detach().numpy(), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(dq, q.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dk, k.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(dv, v.grad.numpy(), rtol=1e-10, atol=1e-12)
    np.testing.assert_allclose(ds, s.grad.numpy(), rtol=1e-10, atol=1e-12)


def test_planted_mistakes_are_caught():
    """A dropped sink term or a wrong sign in dsink must fail the pins above."""
    rng = np.random.default_rng(2)
    L, hq, hkv, d = 8, 2, 1, 4
    q = rng.standard_normal((L, hq, d))
    k = rng.standard_normal((L, hkv, d))
    v = rng.standard_normal((L, hkv, d))
    s = np.array([0.7, -0.3])
    do = rng.standard_normal((L, hq, d))
    cu = np.array([0, L])
    dq, dk, dv, ds, _, _ = orc.attn_bwd(q, k, v, s, do, cu, cu)
    h = 1e-6
    num = np.zeros(hq)
    for i in range(hq):
        sp, sm = s.copy(), s.copy()
        sp[i] += h
        sm[i] -= h
        num[i] = (_loss(q, k, v, sp, do, cu, cu, 0, 0) - _loss(q, k, v, sm, do, cu, cu, 0, 0)) / (2 * h)
    assert np.allclose(ds, num, rtol=1e-6)
    assert not np.allclose(-ds, num, rtol=1e-2)   # flipped sign would be caught
    O_sink, _ = orc.attn_fwd(q, k, v, s, cu, cu)
    O_nosink, _ = orc.attn_fwd(q, k, v, None, cu, cu)
    assert not np.allclose(O_sink, O_nosink, rtol=1e-3)  # dropping the sink is visible
