"""CPU fp64 oracle for attention with an attention sink.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
legs of ``bench.py`` may call it.  It shares no code with the CUDA library.

What is computed (the plain definition, written out):

* Learnable sink (flash-attention PR "feat: Implement Sink Attention",
  Description; sglang PR "openai oss attention sink support with trtllm-gen
  backend", Summary of Changes): each query head ``h`` has one extra logit
  ``sigma_h`` that enters the softmax denominator and carries no value vector.
  With ``s_ij = scale * q_i . k_j`` over the visible keys ``V(i)``::

      m_i   = max(sigma, max_{j in V(i)} s_ij)
      Z_i   = exp(sigma - m_i) + sum_{j in V(i)} exp(s_ij - m_i)
      O_i   = sum_{j in V(i)} exp(s_ij - m_i) v_j / Z_i
      LSE_i = m_i + ln Z_i                      (natural log, includes sigma)

  ``sink=None`` means sigma = -inf (plain softmax attention).
* First-window + last-window selection (sglang PR "To implement
  attention-sink", Motivation and the review's suggested code: keep the first
  1024 and the last 7168 cached tokens, per sequence): a query at absolute
  position ``p`` sees ``[0, min(F, p+1)) U [max(p+1-W, 0), p+1)``; ``W <= 0``
  turns the window off (plain causal).  Decode queries sit at ``p = L-1``.
* Paged KV (same page, suggested code: ``req_to_token`` rows become the page
  table): logical token ``t`` of request ``b`` lives at physical slot
  ``page_table[b, t // page_size] * page_size + t % page_size``.
* Backward (flash-attention PR, Key Changes: the backward pass returns the
  sink's gradient): ``P_ij = exp(s_ij - LSE_i)``, ``dP = dO V^T``,
  ``D_i = sum_j P_ij dP_ij``, ``dS = P o (dP - D)``, ``dQ = scale dS K``,
  ``dK = scale dS^T Q`` and ``dV = P^T dO`` summed over the query heads that
  share a KV head, ``dsink_h = -sum_i exp(sigma_h - LSE_i) D_i``.

Readings where the pages are silent (each listed in the design notes):
sigma is in the units of the scaled logits; one sigma per query head; causal
alignment is bottom-right (query row t of a chunk of Lq rows sits at absolute
position Lk - Lq + t); a row with no visible key has O = 0 and LSE = sigma;
sigma = +inf gives O = 0, LSE = +inf and no gradient; windows require causal.

The softmax is deliberately two-pass (materialise the logits of a row, take
the max, then exponentiate).  Rows are handled in groups only to bound
memory; every row is still the definition above.  Matrix products use numpy's
fp64 ``@`` as a library primitive.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence

import numpy as np

__all__ = [
    "visible_ranges", "visible_mask", "visible_slots", "attn_fwd", "attn_decode_paged",
    "attn_bwd", "to64",
]

ROW_BLOCK = 512


def to64(x):
    """Exact up-cast of a torch/numpy tensor (bf16/fp32/int) to a numpy fp64 array."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _ints(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().cpu().to(torch.int64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.int64)


# ---------------------------------------------------------------------------
# Visible set (window selection)

def visible_ranges(L: int, win_first: int, win_last: int):
    """Token ranges a decode query of a request with ``L`` cached tokens sees.

    The query is the newest token (position L-1).  Returns two half-open
    ranges ``[(a0, b0), (a1, b1)]`` that are disjoint and in increasing order;
    an empty range is ``(x, x)``.  With the window off the first range is
    ``[0, L)`` and the second is empty.  The first window is ``[0, F)`` and the
    last window ``[L-W, L)`` (the review's suggested slices ``[:1024]`` and
    ``[L-7168:L]``), clipped to ``[0, L)`` and merged when they overlap.
    """
    L = int(L)
    if win_last <= 0:
        return [(0, L), (L, L)]
    first_end = min(win_first, L)
    last_begin = max(L - win_last, first_end)
    return [(0, first_end), (last_begin, L)]


def visible_mask(pos: np.ndarray, Lk: int, win_first: int, win_last: int, causal: bool):
    """Boolean (len(pos), Lk) mask: key j is visible to a query at position pos."""
    j = np.arange(Lk)[None, :]
    p = np.asarray(pos)[:, None]
    if causal:
        vis = j <= p
    else:
        if win_last > 0:
            raise ValueError("first/last-window selection is defined for causal attention only")
        vis = np.ones((p.shape[0], Lk), dtype=bool)
    if win_last > 0:
        vis = vis & ((j < win_first) | (j >= p + 1 - win_last))
    return vis


def visible_slots(seqlens, page_table, page_size: int, win_first: int, win_last: int):
    """Per request, the visible logical tokens and the physical slots they occupy.

    Returns a list of ``(t, slot)`` int64 array pairs, ``t`` increasing.
    ``slot = page_table[b, t // page_size] * page_size + t % page_size``.
    """
    seqlens = _ints(seqlens)
    pt = _ints(page_table)
    out = []
    for b, L in enumerate(seqlens):
        (a0, b0), (a1, b1) = visible_ranges(int(L), win_first, win_last)
        t = np.concatenate([np.arange(a0, b0), np.arange(a1, b1)]).astype(np.int64)
        slot = pt[b, t // page_size] * page_size + t % page_size
        out.append((t, slot))
    return out


# ---------------------------------------------------------------------------
# Row softmax with a sink logit (two-pass)

def _sink_softmax_rows(s: np.ndarray, vis: np.ndarray, sigma: float):
    """Weights and statistics of the sink softmax for a block of rows.

    ``s``: (R, n) scaled logits, ``vis``: (R, n) visibility.  Returns
    ``(w, Z, m, lse)`` where ``w = exp(s - m)`` on visible entries (0 elsewhere),
    ``Z`` includes ``exp(sigma - m)``, and rows are special-cased when ``m`` is
    infinite (no visible key and no sink, or sigma = +inf).
    """
    R = s.shape[0]
    sm = np.where(vis, s, -np.inf)
    rowmax = sm.max(axis=1) if sm.shape[1] else np.full(R, -np.inf)
    m = np.maximum(rowmax, sigma)
    w = np.zeros_like(s)
    Z = np.zeros(R)
    lse = np.empty(R)
    finite = np.isfinite(m)
    if finite.any():
        mf = m[finite]
        w[finite] = np.where(vis[finite], np.exp(sm[finite] - mf[:, None]), 0.0)
        Z[finite] = w[finite].sum(axis=1) + np.exp(sigma - mf)
        lse[finite] = mf + np.log(Z[finite])
    # m == -inf: nothing visible and no sink -> O = 0, LSE = -inf
    # m == +inf: sigma = +inf takes all the mass -> O = 0, LSE = +inf
    lse[~finite] = m[~finite]
    return w, Z, m, lse


def _sink_value(sink, h):
    if sink is None:
        return -math.inf
    return float(to64(sink)[h])


# ---------------------------------------------------------------------------
# Forward (prefill / extend / training)

def attn_fwd(q, k, v, sink, cu_seqlens_q, cu_seqlens_k, win_first=0, win_last=0, causal=True,
             scale=0.0, heads: Optional[Iterable[int]] = None,
             requests: Optional[Iterable[int]] = None, rows: Optional[dict] = None):
    """Forward attention with a sink over varlen requests.

    q: (total_q, Hq, d); k, v: (total_k, Hkv, d); sink (Hq,) or None.
    Returns ``(O, LSE)`` as fp64 arrays of shapes (total_q, Hq, d) and
    (Hq, total_q).  Entries outside ``heads`` x ``requests`` (or outside the
    per-request ``rows`` dict ``{b: local row indices}``) are NaN.
    """
    Q, K, Vv = to64(q), to64(k), to64(v)
    cq, ck = _ints(cu_seqlens_q), _ints(cu_seqlens_k)
    tq, hq, d = Q.shape
    hkv = K.shape[1]
    if hq % hkv:
        raise ValueError("Hq must be a multiple of Hkv")
    G = hq // hkv
    if scale <= 0:
        scale = 1.0 / math.sqrt(d)
    O = np.full((tq, hq, d), np.nan)
    LSE = np.full((hq, tq), np.nan)
    heads = range(hq) if heads is None else list(heads)
    requests = range(len(cq) - 1) if requests is None else list(requests)
    for b in requests:
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        Lq, Lk = q1 - q0, k1 - k0
        sel = np.arange(Lq) if rows is None else np.asarray(sorted(rows.get(b, [])), dtype=np.int64)
        for h in heads:
            kh = h // G
            sigma = _sink_value(sink, h)
            Kb, Vb = K[k0:k1, kh], Vv[k0:k1, kh]
            for r0 in range(0, len(sel), ROW_BLOCK):
                ii = sel[r0:r0 + ROW_BLOCK]
                pos = (Lk - Lq) + ii
                s = scale * (Q[q0 + ii, h] @ Kb.T)
                vis = visible_mask(pos, Lk, win_first, win_last, causal)
                w, Z, m, lse = _sink_softmax_rows(s, vis, sigma)
                o = np.zeros((len(ii), d))
                fin = np.isfinite(m)
                if fin.any():
                    o[fin] = (w[fin] @ Vb) / Z[fin][:, None]
                O[q0 + ii, h] = o
                LSE[h, q0 + ii] = lse
    return O, LSE


# ---------------------------------------------------------------------------
# Paged single-token decode

def attn_decode_paged(q, k_cache, v_cache, page_table, seqlens, page_size, sink=None,
                      win_first=0, win_last=0, scale=0.0,
                      heads: Optional[Iterable[int]] = None,
                      requests: Optional[Iterable[int]] = None):
    """One new query token per request against its paged KV cache.

    q: (B, Hq, d); caches (num_pages, page_size, Hkv, d); page_table (B, max_pages);
    seqlens (B,) = cache length including the new token.  Returns (O, LSE) fp64
    of shapes (B, Hq, d) and (B, Hq); entries outside the subsets are NaN.
    """
    Q = to64(q)
    B, hq, d = Q.shape
    hkv = k_cache.shape[2]
    G = hq // hkv
    if scale <= 0:
        scale = 1.0 / math.sqrt(d)
    heads = range(hq) if heads is None else list(heads)
    requests = range(B) if requests is None else list(requests)
    slots = visible_slots(seqlens, page_table, page_size, win_first, win_last)
    O = np.full((B, hq, d), np.nan)
    LSE = np.full((B, hq), np.nan)
    try:
        import torch
        kflat = k_cache.reshape(-1, hkv, d)
        vflat = v_cache.reshape(-1, hkv, d)
        def gather(cache, sl, kh):
            return cache[torch.as_tensor(sl, dtype=torch.long), kh].to(torch.float64).numpy()
    except ImportError:  # pragma: no cover
        kflat = np.asarray(k_cache).reshape(-1, hkv, d)
        vflat = np.asarray(v_cache).reshape(-1, hkv, d)
        def gather(cache, sl, kh):
            return np.asarray(cache[sl, kh], dtype=np.float64)
    for b in requests:
        _, sl = slots[b]
        for kh in sorted({h // G for h in heads}):
            Kv = gather(kflat, sl, kh)
            Vv = gather(vflat, sl, kh)
            for h in heads:
                if h // G != kh:
                    continue
                sigma = _sink_value(sink, h)
                s = scale * (Kv @ Q[b, h])[None, :]
                vis = np.ones_like(s, dtype=bool)
                w, Z, m, lse = _sink_softmax_rows(s, vis, sigma)
                O[b, h] = (w[0] @ Vv) / Z[0] if np.isfinite(m[0]) else 0.0
                LSE[b, h] = lse[0]
    return O, LSE


# ---------------------------------------------------------------------------
# Paged cache writes and paged extend

def paged_slot(page_table, b: int, t: int, page_size: int) -> int:
    """Physical slot of logical token ``t`` of request ``b`` (the page-table
    indirection of the sglang attention-sink PR's suggested code)."""
    return int(page_table[b, t // page_size]) * page_size + t % page_size


def kv_append(k_cache, v_cache, page_table, seqlens, k_new, v_new, page_size, cu_new=None):
    """Writes each request's new K/V rows into its pages and returns the new caches.

    Request ``b`` has ``n_b`` new rows (``cu_new[b+1] - cu_new[b]``; one row,
    row ``b`` of ``k_new``, when ``cu_new`` is None) and ``seqlens[b]`` counts
    them: they are logical tokens ``L_b - n_b .. L_b - 1``, written in order.
    This is the cache update that precedes attention in KV-cache decode
    (flash-attention PR "feat: Implement Sink Attention", Description: the
    KV-cache decode path with a sink).  Caches are torch tensors
    (num_pages, page_size, Hkv, d); copies are exact.
    """
    import torch
    kc = k_cache.clone()
    vc = v_cache.clone()
    kflat = kc.view(-1, *kc.shape[2:])
    vflat = vc.view(-1, *vc.shape[2:])
    L = _ints(seqlens)
    pt = _ints(page_table)
    B = len(L)
    cn = np.arange(B + 1) if cu_new is None else _ints(cu_new)
    for b in range(B):
        n = int(cn[b + 1] - cn[b])
        for r in range(n):
            t = int(L[b]) - n + r
            slot = paged_slot(pt, b, t, page_size)
            kflat[slot] = k_new[int(cn[b]) + r]
            vflat[slot] = v_new[int(cn[b]) + r]
    return kc, vc


def gather_paged(cache, page_table, seqlens, page_size):
    """Contiguous (sum L_b, Hkv, d) copy of each request's tokens 0..L_b-1 and
    the matching cu_seqlens (B+1)."""
    import torch
    flat = cache.reshape(-1, *cache.shape[2:])
    L = _ints(seqlens)
    pt = _ints(page_table)
    idx = [paged_slot(pt, b, t, page_size) for b in range(len(L)) for t in range(int(L[b]))]
    cu = np.zeros(len(L) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(L)
    return flat[torch.as_tensor(idx, dtype=torch.long)], cu


def attn_fwd_paged(q, k_cache, v_cache, page_table, seqlens_k, cu_seqlens_q, page_size, sink,
                   win_first=0, win_last=0, causal=True, scale=0.0, heads=None, requests=None,
                   rows=None):
    """Varlen extend / prefill whose keys and values live in a paged cache:
    request ``b``'s query rows (``cu_seqlens_q``) are the last ``Lq_b`` of its
    ``seqlens_k[b]`` cached tokens (bottom-right causal alignment), read through
    the page table.  The same attention as ``attn_fwd`` on the gathered tokens."""
    K, cu_k = gather_paged(k_cache, page_table, seqlens_k, page_size)
    V, _ = gather_paged(v_cache, page_table, seqlens_k, page_size)
    return attn_fwd(q, K, V, sink, cu_seqlens_q, cu_k, win_first, win_last, causal, scale,
                    heads=heads, requests=requests, rows=rows)


# ---------------------------------------------------------------------------
# Backward

def attn_bwd(q, k, v, sink, dout, cu_seqlens_q, cu_seqlens_k, win_first=0, win_last=0,
             causal=True, scale=0.0, kv_heads: Optional[Iterable[int]] = None,
             requests: Optional[Iterable[int]] = None, check_identity=True):
    """Gradients of ``sum(dout * O)`` w.r.t. q, k, v and the sink.

    Returns ``(dQ, dK, dV, dsink, O, LSE)`` in fp64; dQ (total_q, Hq, d), dK/dV
    (total_k, Hkv, d), dsink (Hq,).  Entries outside ``kv_heads`` (and their
    query heads) x ``requests`` are NaN; dsink sums over the chosen requests.
    """
    Q, K, Vv, dO = to64(q), to64(k), to64(v), to64(dout)
    cq, ck = _ints(cu_seqlens_q), _ints(cu_seqlens_k)
    tq, hq, d = Q.shape
    tk, hkv, _ = K.shape
    G = hq // hkv
    if scale <= 0:
        scale = 1.0 / math.sqrt(d)
    kv_heads = range(hkv) if kv_heads is None else list(kv_heads)
    requests = range(len(cq) - 1) if requests is None else list(requests)
    heads = [kh * G + g for kh in kv_heads for g in range(G)]
    O, LSE = attn_fwd(q, k, v, sink, cu_seqlens_q, cu_seqlens_k, win_first, win_last, causal,
                      scale, heads=heads, requests=requests)
    dQ = np.full((tq, hq, d), np.nan)
    dK = np.full((tk, hkv, d), np.nan)
    dV = np.full((tk, hkv, d), np.nan)
    dsink = np.full(hq, np.nan)
    for h in heads:
        dsink[h] = 0.0
    for b in requests:
        q0, q1, k0, k1 = cq[b], cq[b + 1], ck[b], ck[b + 1]
        Lq, Lk = q1 - q0, k1 - k0
        for kh in kv_heads:
            Kb, Vb = K[k0:k1, kh], Vv[k0:k1, kh]
            dKb = np.zeros((Lk, d))
            dVb = np.zeros((Lk, d))
            for h in range(kh * G, kh * G + G):
                sigma = _sink_value(sink, h)
                for r0 in range(0, Lq, ROW_BLOCK):
                    ii = np.arange(r0, min(Lq, r0 + ROW_BLOCK))
                    rows = q0 + ii
                    lse = LSE[h, rows]
                    s = scale * (Q[rows, h] @ Kb.T)
                    vis = visible_mask((Lk - Lq) + ii, Lk, win_first, win_last, causal)
                    fin = np.isfinite(lse)[:, None]
                    arg = np.where(vis & fin, s - np.where(fin, lse[:, None], 0.0), -np.inf)
                    P = np.exp(arg)
                    dP = dO[rows, h] @ Vb.T
                    D = (P * dP).sum(axis=1)
                    if check_identity:
                        D2 = (dO[rows, h] * O[rows, h]).sum(axis=1)
                        assert np.allclose(D, D2, rtol=1e-9, atol=1e-9), "D_i identity failed"
                    dS = P * (dP - D[:, None])
                    dQ[rows, h] = scale * (dS @ Kb)
                    dKb += scale * (dS.T @ Q[rows, h])
                    dVb += P.T @ dO[rows, h]
                    # probability mass on the sink, exp(sigma - LSE_i)
                    if sigma == -math.inf:
                        psink = np.zeros(len(ii))
                    elif sigma == math.inf:
                        psink = np.ones(len(ii))
                    else:
                        psink = np.where(np.isfinite(lse), np.exp(sigma - np.where(
                            np.isfinite(lse), lse, 0.0)), 0.0)
                    dsink[h] += -(psink * D).sum()
            dK[k0:k1, kh] = dKb
            dV[k0:k1, kh] = dVb
    return dQ, dK, dV, dsink, O, LSE
