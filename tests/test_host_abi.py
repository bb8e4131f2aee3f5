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
                          "sa_sparse_attn_static_scratch", "sa_window_write",
                          "sa_sparse_attn_rope", "sa_sparse_attn_family", "sa_indexer_topk",
                          "sa_candidate_blocks", "sa_hc_split_sinkhorn"}
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
FAKE2 = ctypes.c_void_p(1 << 41)  # a second such address, far from the first


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
    (dict(o=FAKE, ws=None), _lib.SA_ERR_INVALID_ARG),   # ... checked before the workspace
])
def test_sparse_attn_rejects_bad_arguments(lib, kw, code):
    assert _attn(lib, **kw) == code


def _attn_family(lib, family, **kw):
    a = dict(q=FAKE, kv=FAKE, kv_scale=None, fmt=0, sink=FAKE, idx=FAKE, scale=0.1, b=1, s=2,
             h=64, d=512, rows=8, topk=4, o=ctypes.c_void_p((1 << 40) + (1 << 30)), ws=None,
             ws_bytes=0, stream=None)
    a.update(kw)
    return lib.sa_sparse_attn_family(a["q"], a["kv"], a["kv_scale"], a["fmt"], a["sink"],
                                     a["idx"], a["scale"], a["b"], a["s"], a["h"], a["d"],
                                     a["rows"], a["topk"], a["o"], a["ws"], a["ws_bytes"], family,
                                     a["stream"])


def test_sparse_attn_family_routing(lib):
    # a valid call without a workspace gets as far as the workspace check in every family that
    # can run the shape
    for fam in (_lib.SA_FAMILY_AUTO, _lib.SA_FAMILY_TCGEN05, _lib.SA_FAMILY_MMA_SYNC):
        assert _attn_family(lib, fam) == _lib.SA_ERR_WORKSPACE
    assert _attn_family(lib, _lib.SA_FAMILY_MMA_SYNC, d=256) == _lib.SA_ERR_WORKSPACE
    assert _attn_family(lib, _lib.SA_FAMILY_TCGEN05, d=256) == _lib.SA_ERR_UNSUPPORTED
    assert _attn_family(lib, 3) == _lib.SA_ERR_INVALID_ARG
    assert _attn_family(lib, -1) == _lib.SA_ERR_INVALID_ARG


def _attn_rope(lib, **kw):
    a = dict(q=FAKE, kv=FAKE, kv_scale=None, fmt=0, sink=FAKE, idx=FAKE, scale=0.1, b=1, s=2,
             h=64, d=512, rows=8, topk=4, o=ctypes.c_void_p((1 << 40) + (1 << 30)), ws=None,
             ws_bytes=0, rot=FAKE2, npos=16, rope_dim=64, start_pos=3, stream=None)
    a.update(kw)
    return lib.sa_sparse_attn_rope(a["q"], a["kv"], a["kv_scale"], a["fmt"], a["sink"], a["idx"],
                                   a["scale"], a["b"], a["s"], a["h"], a["d"], a["rows"],
                                   a["topk"], a["o"], a["ws"], a["ws_bytes"], a["rot"], a["npos"],
                                   a["rope_dim"], a["start_pos"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(), _lib.SA_ERR_WORKSPACE),                    # valid rotation: the shared checks follow
    (dict(rope_dim=63), _lib.SA_ERR_INVALID_ARG),       # odd
    (dict(rope_dim=0), _lib.SA_ERR_INVALID_ARG),
    (dict(rope_dim=514), _lib.SA_ERR_INVALID_ARG),      # wider than the head
    (dict(start_pos=15), _lib.SA_ERR_INVALID_ARG),      # positions 15, 16 past a 16-row table
    (dict(start_pos=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(npos=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(d=256, rope_dim=64), _lib.SA_ERR_UNSUPPORTED),  # only the d = 512 kernel fuses it
    (dict(rot=None), _lib.SA_ERR_INVALID_ARG),
    (dict(rot=ctypes.c_void_p((1 << 41) + 4)), _lib.SA_ERR_INVALID_ARG),  # not 8-byte aligned
    (dict(rot=ctypes.c_void_p((1 << 40) + (1 << 30) + 256)), _lib.SA_ERR_INVALID_ARG),  # in o
    (dict(rot=None, b=0), _lib.SA_OK),                  # no tokens: nothing is read
])
def test_sparse_attn_rope_rejects_bad_arguments(lib, kw, code):
    assert _attn_rope(lib, **kw) == code


def _topk(lib, **kw):
    a = dict(score=FAKE, fmt=0, cand=None, b=2, s=1, n=32, start=127, ratio=4, topk=16,
             offset=128, idx=FAKE2, ld=16, bstride=16, stream=None)
    a.update(kw)
    return lib.sa_indexer_topk(a["score"], a["fmt"], a["cand"], a["b"], a["s"], a["n"], a["start"],
                               a["ratio"], a["topk"], a["offset"], a["idx"], a["ld"], a["bstride"],
                               a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(fmt=2), _lib.SA_ERR_INVALID_ARG),
    (dict(n=33), _lib.SA_ERR_INVALID_ARG),              # not (start_pos + s) // ratio
    (dict(ratio=0), _lib.SA_ERR_INVALID_ARG),
    (dict(offset=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(offset=(1 << 31) - 20), _lib.SA_ERR_INVALID_ARG),  # offset + n past int32
    (dict(s=2, start=126), _lib.SA_ERR_UNSUPPORTED),    # chunked prefill
    (dict(start=4 * 49153 - 1, n=49153), _lib.SA_ERR_UNSUPPORTED),  # past the shared-memory row
    (dict(ld=15), _lib.SA_ERR_INVALID_ARG),             # rows shorter than k
    (dict(bstride=15), _lib.SA_ERR_INVALID_ARG),        # sequences overlap
    (dict(score=None), _lib.SA_ERR_INVALID_ARG),
    (dict(idx=ctypes.c_void_p((1 << 41) + 2)), _lib.SA_ERR_INVALID_ARG),  # misaligned
    (dict(idx=FAKE), _lib.SA_ERR_INVALID_ARG),          # idx overlaps score
    (dict(topk=0, score=None), _lib.SA_OK),             # k == 0: nothing to write
    (dict(b=0, score=None), _lib.SA_OK),
    (dict(cand=ctypes.c_void_p((1 << 41) + 8)), _lib.SA_ERR_INVALID_ARG),  # candidates overlap idx
])
def test_indexer_topk_rejects_bad_arguments(lib, kw, code):
    assert _topk(lib, **kw) == code


def _cand(lib, **kw):
    a = dict(logits=FAKE, fmt=0, b=2, s=1, n=32, start=127, ratio=4, kb=2, bs=8, mask=FAKE2,
             stream=None)
    a.update(kw)
    return lib.sa_candidate_blocks(a["logits"], a["fmt"], a["b"], a["s"], a["n"], a["start"],
                                   a["ratio"], a["kb"], a["bs"], a["mask"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(fmt=5), _lib.SA_ERR_INVALID_ARG),
    (dict(n=31), _lib.SA_ERR_INVALID_ARG),              # not (start_pos + s) // ratio
    (dict(bs=0), _lib.SA_ERR_INVALID_ARG),
    (dict(kb=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(s=2, start=126), _lib.SA_ERR_UNSUPPORTED),    # chunked prefill
    (dict(start=4 * 49153 - 1, n=49153, bs=1), _lib.SA_ERR_UNSUPPORTED),  # too many blocks
    (dict(mask=None), _lib.SA_ERR_INVALID_ARG),
    (dict(logits=None), _lib.SA_ERR_INVALID_ARG),
    (dict(mask=ctypes.c_void_p((1 << 40) + 64)), _lib.SA_ERR_INVALID_ARG),  # inside the logits
    (dict(b=0, logits=None, mask=None), _lib.SA_OK),
])
def test_candidate_blocks_rejects_bad_arguments(lib, kw, code):
    assert _cand(lib, **kw) == code


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


def test_window_write_rejects_bad_arguments(lib):
    f = lib.sa_window_write
    ok_args = [FAKE, 2, 1, 64, 64, 5, 8, FAKE2, 64, 8 * 64, None, 0, 0, None, 0, 0, None]

    def call(**kw):
        a = list(ok_args)
        for k, v in kw.items():
            a[int(k[1:])] = v
        return f(*a)

    assert call(a3=33) == _lib.SA_ERR_INVALID_ARG                   # d not a multiple of 32
    assert call(a6=0) == _lib.SA_ERR_INVALID_ARG                    # window < 1
    assert call(a5=-1) == _lib.SA_ERR_INVALID_ARG                   # negative position
    assert call(a7=None) == _lib.SA_ERR_INVALID_ARG                 # no output at all
    assert call(a4=32) == _lib.SA_ERR_INVALID_ARG                   # x rows shorter than d
    assert call(a8=32) == _lib.SA_ERR_INVALID_ARG                   # ring rows shorter than d
    assert call(a9=7 * 64) == _lib.SA_ERR_INVALID_ARG               # two sequences' rings overlap
    assert call(a7=FAKE) == _lib.SA_ERR_INVALID_ARG                 # the ring overlaps x
    assert call(a7=None, a10=FAKE2, a11=64, a12=8 * 64 - 1) == _lib.SA_ERR_INVALID_ARG
    assert call(a7=None, a13=FAKE2, a14=1, a15=16) == _lib.SA_ERR_INVALID_ARG  # scale rows < d/32
    assert call(a1=0) == _lib.SA_OK and call(a2=0) == _lib.SA_OK   # nothing to write


def test_read_status_rejects_null(lib):
    assert lib.sa_read_status(None, 0, None) == _lib.SA_ERR_INVALID_ARG


def _hc(lib, **kw):
    a = dict(mixes=FAKE, n=100, hc=4, scale=ctypes.c_void_p((1 << 40) + (1 << 20)),
             base=ctypes.c_void_p((1 << 40) + (1 << 21)), iters=20, eps=1e-6,
             pre=ctypes.c_void_p(1 << 41), post=ctypes.c_void_p((1 << 41) + (1 << 20)),
             comb=ctypes.c_void_p((1 << 41) + (1 << 21)), stream=None)
    a.update(kw)
    return lib.sa_hc_split_sinkhorn(a["mixes"], a["n"], a["hc"], a["scale"], a["base"], a["iters"],
                                    a["eps"], a["pre"], a["post"], a["comb"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(hc=3), _lib.SA_ERR_UNSUPPORTED),              # only the model's hc_mult = 4
    (dict(iters=0), _lib.SA_ERR_INVALID_ARG),
    (dict(n=-1), _lib.SA_ERR_INVALID_ARG),
    (dict(n=(2**31 - 1) * 256 + 1), _lib.SA_ERR_INVALID_ARG),  # past the grid
    (dict(mixes=ctypes.c_void_p((1 << 40) + 4)), _lib.SA_ERR_INVALID_ARG),  # not 16-byte aligned
    (dict(comb=None), _lib.SA_ERR_INVALID_ARG),
    (dict(post=ctypes.c_void_p(1 << 41)), _lib.SA_ERR_INVALID_ARG),  # post overlaps pre
    (dict(pre=ctypes.c_void_p((1 << 40) + 96)), _lib.SA_ERR_INVALID_ARG),  # pre inside mixes
    (dict(n=0, mixes=None), _lib.SA_OK),
])
def test_hc_split_sinkhorn_rejects_bad_arguments(lib, kw, code):
    assert _hc(lib, **kw) == code

