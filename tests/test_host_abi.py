"""The C-ABI library without a GPU: it builds, loads, exports every declared symbol, and rejects
bad arguments before touching CUDA."""

from __future__ import annotations

import ctypes

import pytest

from sparse_latent_attention_gb300 import _lib, build


@pytest.fixture(scope="module")
def lib():
    build.build()
    return _lib.load()


def test_exports_every_declared_symbol(lib):
    names = _lib.declared_symbols()
    assert set(names) == {"sa_sparse_attn", "sa_sparse_attn_workspace_size", "sa_window_idxs",
                          "sa_act_quant_fp8", "sa_read_status", "sa_status_string", "sa_version",
                          "sa_sparse_attn_static_scratch"}
    for n in names:
        assert hasattr(lib, n), n


def test_status_strings_and_version(lib):
    for code in range(7):
        assert _lib.status_string(code) not in ("", "unknown status")
    assert _lib.status_string(99) == "unknown status"
    assert _lib.version() >= 100


def test_workspace_size_is_host_arithmetic(lib):
    f = lib.sa_sparse_attn_workspace_size
    assert f(1, 4096, 64, 512, 4096, 128, 0) >= _lib.SA_STATUS_BYTES
    # few tokens and many idx tiles: split partials are part of the workspace
    assert f(64, 1, 64, 512, 8320, 1152, 0) > f(1, 4096, 64, 512, 4096, 128, 0)
    assert f(1, 16, 64, 100, 48, 16, 0) == 0     # d not a multiple of 64
    assert f(1, 16, 129, 512, 48, 16, 0) == 0    # more than 128 heads
    assert f(1, 16, 64, 512, 48, 16, 7) == 0     # unknown kv format


FAKE = ctypes.c_void_p(1 << 40)  # never dereferenced: every call below fails validation first


def _attn(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, kv_scale=None, fmt=0, sink=FAKE, idx=FAKE, scale=0.1, b=1, s=2,
             h=4, d=64, rows=8, topk=4, o=ctypes.c_void_p((1 << 40) + (1 << 30)), ws=FAKE,
             ws_bytes=1 << 20, stream=None)
    a.update(kw)
    return lib.sa_sparse_attn(a["q"], a["kv"], a["kv_scale"], a["fmt"], a["sink"], a["idx"],
                              a["scale"], a["b"], a["s"], a["h"], a["d"], a["rows"], a["topk"],
                              a["o"], a["ws"], a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(q=None), _lib.SA_ERR_INVALID_ARG),
    (dict(o=None), _lib.SA_ERR_INVALID_ARG),
    (dict(fmt=1), _lib.SA_ERR_INVALID_ARG),             # fp8 without scales
    (dict(kv_scale=FAKE), _lib.SA_ERR_INVALID_ARG),     # bf16 with scales
    (dict(fmt=3), _lib.SA_ERR_INVALID_ARG),
    (dict(b=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(topk=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(d=96), _lib.SA_ERR_UNSUPPORTED),
    (dict(h=200), _lib.SA_ERR_UNSUPPORTED),
    (dict(q=ctypes.c_void_p((1 << 40) + 2)), _lib.SA_ERR_INVALID_ARG),  # misaligned
    (dict(ws=None), _lib.SA_ERR_WORKSPACE),
    (dict(ws_bytes=16), _lib.SA_ERR_WORKSPACE),
    (dict(o=FAKE), _lib.SA_ERR_INVALID_ARG),            # output overlaps the inputs
])
def test_sparse_attn_rejects_bad_arguments(lib, kw, code):
    assert _attn(lib, **kw) == code


def test_window_idxs_rejects_bad_arguments(lib):
    f = lib.sa_window_idxs
    assert f(0, 4, 0, FAKE, 8, 1, 0, None) == _lib.SA_ERR_INVALID_ARG      # window 0
    assert f(0, 4, 8, FAKE, 4, 1, 0, None) == _lib.SA_ERR_INVALID_ARG      # ld < window
    assert f(4, 3, 8, FAKE, 8, 1, 0, None) == _lib.SA_ERR_UNSUPPORTED      # chunked prefill
    assert f(0, 4, 8, None, 8, 1, 0, None) == _lib.SA_ERR_INVALID_ARG
    assert f(0, 0, 8, None, 8, 1, 0, None) == _lib.SA_OK                   # nothing to write


def test_act_quant_rejects_bad_arguments(lib):
    f = lib.sa_act_quant_fp8
    assert f(FAKE, 4, 33, 33, FAKE, 33, None, 0, None, 0, None) == _lib.SA_ERR_INVALID_ARG
    assert f(FAKE, 4, 64, 64, None, 0, None, 0, None, 0, None) == _lib.SA_ERR_INVALID_ARG
    assert f(FAKE, 4, 64, 32, FAKE, 64, None, 0, None, 0, None) == _lib.SA_ERR_INVALID_ARG
    assert f(None, 0, 64, 64, FAKE, 64, None, 0, None, 0, None) == _lib.SA_OK


def test_read_status_rejects_null(lib):
    assert lib.sa_read_status(None, 0, None) == _lib.SA_ERR_INVALID_ARG
