"""Pins for the oracle's paged-cache functions (cache append, paged extend).

* ``paged_slot`` on a hand-worked example of the page-table indirection (sglang
  PR "To implement attention-sink", suggested code: ``req_to_token`` rows as a
  page table) and against ``visible_slots`` with the window off;
* ``kv_append`` touches exactly the appended slots, and a request's gathered
  tokens end with its new rows;
* ``attn_fwd_paged`` equals ``attn_fwd`` on the contiguous tokens when the
  cache is filled page by page by an independent scatter, for two different
  page permutations;
* decode after appending the new token equals decode on a cache that already
  holds it.
"""
import numpy as np
import pytest
import torch

from oracle import attn_sink_oracle as orc
from paged_kv_sink_gb300 import workloads as wl


def test_paged_slot_hand_example():
    # page size 4; request 0 owns physical pages 2 then 0: token 5 is the second
    # token of its second page -> physical page 0, offset 1 -> slot 1.
    pt = np.array([[2, 0]])
    assert orc.paged_slot(pt, 0, 5, 4) == 1
    assert orc.paged_slot(pt, 0, 0, 4) == 8
    assert orc.paged_slot(pt, 0, 3, 4) == 11


def test_paged_slot_matches_visible_slots():
    dc = wl.make_decode(seqlens=[1, 7, 33, 64], hq=2, hkv=1, d=8, page_size=8, seed=5, extra_pages=3)
    slots = orc.visible_slots(dc.seqlens, dc.page_table, dc.page_size, 0, 0)
    pt = dc.page_table.numpy()
    for b, L in enumerate(dc.seqlens.tolist()):
        toks, sl = slots[b]
        assert list(toks) == list(range(L))
        assert [orc.paged_slot(pt, b, t, 8) for t in range(L)] == list(sl)


def _scatter_pages(chunks, page_size, pool, hkv, d, perm):
    """Independent fill: request b's contiguous rows cut into pages in order,
    page j stored at physical page perm_b[j] by tensor slicing."""
    cache = torch.zeros((pool, page_size, hkv, d), dtype=torch.bfloat16)
    rows = []
    off = 0
    for x in chunks:
        n = (x.shape[0] + page_size - 1) // page_size
        ids = perm[off:off + n]
        off += n
        for j, pg in enumerate(ids.tolist()):
            part = x[j * page_size:(j + 1) * page_size]
            cache[pg, :part.shape[0]] = part
        rows.append(ids.tolist())
    maxp = max(len(r) for r in rows)
    pt = torch.full((len(chunks), maxp), -1, dtype=torch.int32)
    for b, r in enumerate(rows):
        pt[b, :len(r)] = torch.tensor(r, dtype=torch.int32)
    return cache, pt


@pytest.mark.parametrize("page_size", [4, 16])
def test_attn_fwd_paged_equals_contiguous(page_size):
    p = wl.make_prefill(seqlens_q=[9, 30, 1], seqlens_k=[40, 30, 17], hq=4, hkv=2, d=16, sink="normal",
                        win_first=3, win_last=11, causal=True, seed=21)
    ck = p.cu_seqlens_k.tolist()
    ks = [p.k[ck[b]:ck[b + 1]] for b in range(3)]
    vs = [p.v[ck[b]:ck[b + 1]] for b in range(3)]
    pool = sum((x.shape[0] + page_size - 1) // page_size for x in ks) + 2
    O, LSE = orc.attn_fwd(p.q, p.k, p.v, p.sink, p.cu_seqlens_q, p.cu_seqlens_k, 3, 11, True)
    for seed in (1, 2):
        perm = torch.randperm(pool, generator=torch.Generator().manual_seed(seed))
        kc, pt = _scatter_pages(ks, page_size, pool, 2, 16, perm)
        vc, _ = _scatter_pages(vs, page_size, pool, 2, 16, perm)
        seqlens_k = torch.tensor([x.shape[0] for x in ks], dtype=torch.int32)
        Op, LSEp = orc.attn_fwd_paged(p.q, kc, vc, pt, seqlens_k, p.cu_seqlens_q, page_size, p.sink,
                                      3, 11, True)
        np.testing.assert_array_equal(Op, O)
        np.testing.assert_array_equal(LSEp, LSE)


def test_kv_append_touches_only_new_slots():
    pe = wl.make_paged_extend(seqlens_q=[2, 3, 1], seqlens_k=[5, 9, 1], hq=2, hkv=2, d=8, page_size=4,
                              seed=3, extra_pages=2)
    kc, vc = orc.kv_append(pe.k_cache, pe.v_cache, pe.page_table, pe.seqlens_k, pe.k_new, pe.v_new,
                           pe.page_size, cu_new=pe.cu_seqlens_q)
    changed = (kc != pe.k_cache).reshape(-1, 2 * 8).any(dim=1)
    assert int(changed.sum()) <= int(pe.cu_seqlens_q[-1])  # equal unless a new row equals the old one
    K, cu = orc.gather_paged(kc, pe.page_table, pe.seqlens_k, pe.page_size)
    V, _ = orc.gather_paged(vc, pe.page_table, pe.seqlens_k, pe.page_size)
    cq = pe.cu_seqlens_q.tolist()
    for b in range(3):
        n = cq[b + 1] - cq[b]
        assert torch.equal(K[cu[b + 1] - n:cu[b + 1]], pe.k_new[cq[b]:cq[b + 1]])
        assert torch.equal(V[cu[b + 1] - n:cu[b + 1]], pe.v_new[cq[b]:cq[b + 1]])
    # tokens before the new ones are untouched
    K0, _ = orc.gather_paged(pe.k_cache, pe.page_table, pe.seqlens_k, pe.page_size)
    for b in range(3):
        n = cq[b + 1] - cq[b]
        assert torch.equal(K[cu[b]:cu[b + 1] - n], K0[cu[b]:cu[b + 1] - n])
    # untouched slots keep their values exactly
    flat_old = pe.k_cache.reshape(-1, 2, 8)
    flat_new = kc.reshape(-1, 2, 8)
    written = {orc.paged_slot(pe.page_table.numpy(), b, t, 4)
               for b in range(3) for t in range(int(pe.seqlens_k[b]) - (cq[b + 1] - cq[b]), int(pe.seqlens_k[b]))}
    for sl in range(flat_old.shape[0]):
        if sl not in written:
            assert torch.equal(flat_old[sl], flat_new[sl])


def test_decode_after_append_equals_prefilled():
    dc = wl.make_decode(seqlens=[5, 33, 16], hq=4, hkv=2, d=8, page_size=8, seed=9, extra_pages=1)
    g = torch.Generator().manual_seed(4)
    kn = torch.randn(3, 2, 8, generator=g).to(torch.bfloat16)
    vn = torch.randn(3, 2, 8, generator=g).to(torch.bfloat16)
    kc, vc = orc.kv_append(dc.k_cache, dc.v_cache, dc.page_table, dc.seqlens, kn, vn, 8)
    # prefilled cache built directly: the last token of request b sits in its last page
    kp, vp = dc.k_cache.clone(), dc.v_cache.clone()
    for b, L in enumerate(dc.seqlens.tolist()):
        pg = int(dc.page_table[b, (L - 1) // 8])
        kp[pg, (L - 1) % 8] = kn[b]
        vp[pg, (L - 1) % 8] = vn[b]
    assert torch.equal(kc, kp) and torch.equal(vc, vp)
    O1, L1 = orc.attn_decode_paged(dc.q, kc, vc, dc.page_table, dc.seqlens, 8, dc.sink)
    O2, L2 = orc.attn_decode_paged(dc.q, kp, vp, dc.page_table, dc.seqlens, 8, dc.sink)
    np.testing.assert_array_equal(O1, O2)
    np.testing.assert_array_equal(L1, L2)
