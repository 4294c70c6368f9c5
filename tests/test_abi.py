"""The C-ABI library builds, loads and exports every symbol its header
declares; host-side validation rejects bad arguments before any CUDA work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn_sink.h")


@pytest.fixture(scope="module")
def lib():
    from paged_kv_sink_gb300 import build as b
    path = b.build()
    from paged_kv_sink_gb300 import _lib
    return _lib.load(path)


def _declared():
    txt = open(HEADER).read()
    txt = re.sub(r"/\*.*?\*/", "", txt, flags=re.S)
    return sorted(set(re.findall(r"\b(attn_sink_\w+)\s*\(", txt)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("attn_sink_fwd", "attn_sink_decode_paged", "attn_sink_bwd",
              "attn_sink_visible_ranges", "attn_sink_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    for n in _declared():
        assert hasattr(lib, n), n
    from paged_kv_sink_gb300 import _lib
    assert set(_declared()) <= set(_lib.EXPORTS) | {"attn_sink_version"}
    assert b"sm_103a" in lib.attn_sink_version()


def test_validation_without_gpu(lib):
    """Bad arguments come back as status codes, with no CUDA call made."""
    P = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # head_dim 96 is unsupported
    rc = lib.attn_sink_decode_paged(P, P, P, P, 4, P, 1, 8, 2, 96, 16, 4, None, 0, 0, 0.0, P, None, None)
    assert rc == -2
    # hq not a multiple of hkv
    rc = lib.attn_sink_decode_paged(P, P, P, P, 4, P, 1, 6, 4, 64, 16, 4, None, 0, 0, 0.0, P, None, None)
    assert rc == -2
    # negative batch
    rc = lib.attn_sink_decode_paged(P, P, P, P, 4, P, -1, 8, 2, 64, 16, 4, None, 0, 0, 0.0, P, None, None)
    assert rc == -1
    assert b"positive" in lib.attn_sink_last_error()
    # NULL tensors
    rc = lib.attn_sink_decode_paged(None, P, P, P, 4, P, 2, 8, 2, 64, 16, 4, None, 0, 0, 0.0, P, None, None)
    assert rc == -1
    # misaligned cache pointer
    rc = lib.attn_sink_decode_paged(P, ctypes.c_void_p(18), P, P, 4, P, 2, 8, 2, 64, 16, 4, None, 0, 0,
                                    0.0, P, None, None)
    assert rc == -1
    # window without causal is rejected
    rc = lib.attn_sink_fwd(P, P, P, None, P, P, 1, 8, 8, 4, 2, 64, 8, 8, 4, 8, 0, 0.0, P, None, None)
    assert rc == -1
    # forward head_dim 96 unsupported (64 and 128 are)
    rc = lib.attn_sink_fwd(P, P, P, None, P, P, 1, 8, 8, 4, 2, 96, 8, 8, 0, 0, 1, 0.0, P, None, None)
    assert rc == -2
    assert b"64, 128" in lib.attn_sink_last_error()
    # dsink must accompany sink
    rc = lib.attn_sink_bwd(P, P, P, P, P, P, P, P, P, 1, 8, 8, 4, 2, 64, 8, 8, 0, 0, 1, 0.0, P, P, P, None, None)
    assert rc == -1
    # empty batch is a no-op
    rc = lib.attn_sink_decode_paged(None, None, None, None, 4, None, 0, 8, 2, 64, 16, 4, None, 0, 0, 0.0,
                                    None, None, None)
    assert rc == 0


def test_validation_of_the_extended_entry_points_without_gpu(lib):
    """Host-side checks of the strided, paged, append and host-buffer entry points
    return their status codes before any CUDA call."""
    P = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # strided forward: a q row stride below heads*64, and one that breaks 16-byte rows
    for q_rs in (200, 260):
        rc = lib.attn_sink_fwd_strided(P, P, P, q_rs, 0, 0, None, P, P, 1, 8, 8, 4, 2, 64, 8, 8, 0, 0, 1, 0.0,
                                       P, None, None)
        assert rc == -1
        assert b"row stride" in lib.attn_sink_last_error()
    # strided backward: bad k stride
    rc = lib.attn_sink_bwd_strided(P, P, P, 0, 100, 0, None, P, P, P, P, P, 1, 8, 8, 4, 2, 64, 8, 8, 0, 0, 1,
                                   0.0, P, P, P, 0, 0, 0, None, None)
    assert rc == -1
    assert b"k row stride" in lib.attn_sink_last_error()
    # paged forward: page size not a power of two >= 8; k_new without v_new
    for ps in (24, 4):
        rc = lib.attn_sink_fwd_paged(P, None, None, P, P, P, 4, P, P, 1, 8, 4, 2, 64, ps, 16, 8, 40, None, 0, 0,
                                     1, 0.0, P, None, None)
        assert rc == -2
    rc = lib.attn_sink_fwd_paged(P, P, None, P, P, P, 4, P, P, 1, 8, 4, 2, 64, 16, 16, 8, 40, None, 0, 0, 1,
                                 0.0, P, None, None)
    assert rc == -1
    assert b"together" in lib.attn_sink_last_error()
    # paged forward: windows need causal attention
    rc = lib.attn_sink_fwd_paged(P, None, None, P, P, P, 4, P, P, 1, 8, 4, 2, 64, 16, 16, 8, 40, None, 4, 8, 0,
                                 0.0, P, None, None)
    assert rc == -1
    # append: head_dim 96; several rows per request without cu_new; misaligned cache; empty is a no-op
    rc = lib.attn_sink_kv_append(P, P, P, P, P, 4, 2, 2, 96, 16, 8, 3, P, P, None)
    assert rc == -2
    rc = lib.attn_sink_kv_append(P, P, None, P, P, 4, 2, 2, 64, 16, 8, 3, P, P, None)
    assert rc == -1
    assert b"cu_new" in lib.attn_sink_last_error()
    rc = lib.attn_sink_kv_append(P, P, P, P, P, 4, 2, 2, 64, 16, 8, 3, ctypes.c_void_p(24), P, None)
    assert rc == -1
    assert b"aligned" in lib.attn_sink_last_error()
    rc = lib.attn_sink_kv_append(None, None, None, None, None, 4, 0, 2, 64, 16, 8, 0, None, None, None)
    assert rc == 0
    # decode with append: NULL new rows
    rc = lib.attn_sink_decode_paged_append(P, None, None, P, P, P, 4, P, 2, 8, 2, 64, 16, 4, None, 0, 0, 0.0,
                                           P, None, None)
    assert rc == -1
    assert b"k_new" in lib.attn_sink_last_error()
    # host-buffer forward: cu_seqlens are read on the host and checked there
    def fwd_host(cu_q, cu_k, batch, head_dim=64):
        aq = (ctypes.c_int32 * len(cu_q))(*cu_q)
        ak = (ctypes.c_int32 * len(cu_k))(*cu_k)
        return lib.attn_sink_fwd_host(P, P, P, None, ctypes.cast(aq, ctypes.c_void_p),
                                      ctypes.cast(ak, ctypes.c_void_p), batch, 4, 2, head_dim, 0, 0, 1, 0.0, P,
                                      None, None)
    assert fwd_host([1, 5], [0, 5], 1) == -1
    assert b"start at 0" in lib.attn_sink_last_error()
    assert fwd_host([0, 5, 3], [0, 5, 9], 2) == -1
    assert b"non-decreasing" in lib.attn_sink_last_error()
    assert fwd_host([0, 5], [0, 5], 1, head_dim=96) == -2
    assert fwd_host([0], [0], 0) == 0
    assert fwd_host([0, 0, 0], [0, 7, 9], 2) == 0  # no query rows: nothing to do


def test_grid_limits_rejected_on_the_host(lib):
    """More requests (or query rows per request) than a launch grid dimension
    holds come back as -2 with a message, before any CUDA work."""
    P = ctypes.c_void_p(16)  # never dereferenced: validation fails first
    # forward: 65536 requests; then one request of 65535 * 128 + 1 query rows
    rc = lib.attn_sink_fwd(P, P, P, None, P, P, 65536, 1, 1, 4, 2, 64, 1, 1, 0, 0, 1, 0.0, P, None, None)
    assert rc == -2 and b"batch" in lib.attn_sink_last_error()
    rc = lib.attn_sink_fwd(P, P, P, None, P, P, 1, 1, 1, 4, 2, 64, 65535 * 128 + 1, 1, 0, 0, 1, 0.0, P, None, None)
    assert rc == -2 and b"max_seqlen_q" in lib.attn_sink_last_error()
    rc = lib.attn_sink_fwd(P, P, P, None, P, P, 65535, 1, 1, 4, 2, 64, 65535 * 128, 1, 0, 0, 1, 0.0, None, None,
                           None)
    assert rc == -1 and b"out" in lib.attn_sink_last_error()  # at the limits: on to the next check
    # decode and append: 65536 requests
    rc = lib.attn_sink_decode_paged(P, P, P, P, 4, P, 65536, 8, 2, 64, 16, 4, None, 0, 0, 0.0, P, None, None)
    assert rc == -2 and b"batch" in lib.attn_sink_last_error()
    rc = lib.attn_sink_kv_append(P, P, None, P, P, 4, 65536, 2, 64, 16, 8, 1, P, P, None)
    assert rc == -2 and b"batch" in lib.attn_sink_last_error()


def test_autograd_functions_check_arguments_on_the_host(lib):
    """The autograd functions only marshal arguments: host tensors and
    malformed shapes are rejected before any library call."""
    import torch
    import paged_kv_sink_gb300 as ext
    q = torch.zeros(4, 2, 64, dtype=torch.bfloat16)
    kv = torch.zeros(4, 1, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 4], dtype=torch.int32)
    with pytest.raises(TypeError, match="CUDA"):
        ext.attn_sink_varlen_func(q, kv, kv, cu, cu, 4, 4)
    with pytest.raises(TypeError, match="batch, seqlen"):
        ext.attn_sink_func(q, kv, kv)
    with pytest.raises(TypeError, match="hkv"):
        ext.attn_sink_varlen_qkvpacked_func(torch.zeros(4, 6, 64, dtype=torch.bfloat16), cu, 4)
    with pytest.raises(TypeError, match="CUDA"):
        ext.attn_sink_varlen_qkvpacked_func(torch.zeros(4, 3, 2, 64, dtype=torch.bfloat16), cu, 4)
    with pytest.raises(TypeError, match="kv must be"):
        ext.attn_sink_varlen_kvpacked_func(q, kv, cu, cu, 4, 4)
    with pytest.raises(TypeError, match="qkv must be"):
        ext.attn_sink_qkvpacked_func(torch.zeros(4, 3, 2, 64, dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="CUDA"):
        ext.attn_sink_kvpacked_func(q.reshape(1, 4, 2, 64), torch.zeros(1, 4, 2, 1, 64, dtype=torch.bfloat16))
