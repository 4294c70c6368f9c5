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
    # forward head_dim 128 unsupported
    rc = lib.attn_sink_fwd(P, P, P, None, P, P, 1, 8, 8, 4, 2, 128, 8, 8, 0, 0, 1, 0.0, P, None, None)
    assert rc == -2
    # dsink must accompany sink
    rc = lib.attn_sink_bwd(P, P, P, P, P, P, P, P, P, 1, 8, 8, 4, 2, 64, 8, 8, 0, 0, 1, 0.0, P, P, P, None, None)
    assert rc == -1
    # empty batch is a no-op
    rc = lib.attn_sink_decode_paged(None, None, None, None, 4, None, 0, 8, 2, 64, 16, 4, None, 0, 0, 0.0,
                                    None, None, None)
    assert rc == 0
