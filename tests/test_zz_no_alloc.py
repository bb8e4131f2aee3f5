"""sa_sparse_attn_static_scratch: sparse_attn for callers that cannot allocate device memory
(a plugin whose host runtime owns all device allocations, a serving loop that must not call
cudaMalloc / cudaFree on its request path).  It must give the same result as sa_sparse_attn with
a caller workspace, call after call, while the library's one scratch array carries the previous
call's contents.  Kept last in collection order so a failure here comes after every other test.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

import sparse_latent_attention_gb300 as sa
from sparse_latent_attention_gb300 import _lib, build, workloads
from tests import _gpu
from tests._helpers import assert_close_bf16

pytestmark = pytest.mark.gpu

STATIC_SCRATCH_BYTES = 64 << 20  # SA_STATIC_SCRATCH_BYTES in include/sparse_attn.h


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    lib = _lib.load()
    f = lib.sa_sparse_attn_static_scratch
    P, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    f.restype = i32
    f.argtypes = [P, P, P, i32, P, P, ctypes.c_float, i64, i64, i32, i32, i64, i32, P, P, P]
    return lib


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _call_static(lib, x, wl, o, status):
    fmt = sa.SA_KV_BF16 if x["kv_scale"] is None else sa.SA_KV_FP8_E4M3
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.sa_sparse_attn_static_scratch(
        _p(x["q"]), _p(x["kv"]), _p(x["kv_scale"]), fmt, _p(x["sink"]), _p(x["idx"]), wl.scale,
        wl.b, wl.s, wl.h, wl.d, wl.rows, wl.topk, _p(o), _p(status), stream)


CASES = [
    # decode: idx columns split over CTAs, partials live in the scratch array
    dict(b=3, s=1, h=64, d=512, rows=5000, topk=1152, seed=401),
    # prefill with a ragged tail: only the status word is scratch
    dict(b=1, s=40, h=64, d=512, rows=300, topk=200, seed=402),
    # the long fp8-decode shape at 150 sequences: two head blocks, pieces merged in the kernel
    dict(b=150, s=1, h=128, d=512, rows=2500, topk=2176, seed=404),
]


@pytest.mark.parametrize("case", CASES, ids=["decode_split", "prefill", "decode_b150_h128"])
def test_static_scratch_matches_workspace_call(lib, case):
    dev = torch.device("cuda:0")
    wl = workloads.make_random(case["b"], case["s"], case["h"], case["d"], case["rows"],
                               case["topk"], seed=case["seed"], all_neg_tokens=(0,))
    x = _gpu.prepare(wl, dev, quantise=False)
    ref = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale)
    want = _gpu.bf16_tensor_to_u16(ref)
    status = torch.full((1,), 7, dtype=torch.int32, device=dev)
    for call in range(2):  # the second call runs over the first call's leftovers
        o = torch.full_like(ref, float("nan"))
        assert _call_static(lib, x, wl, o, status) == _lib.SA_OK
        torch.cuda.synchronize()
        # the same kernels on the same inputs as the workspace call: the same bits
        assert torch.equal(o.view(torch.int16), ref.view(torch.int16)), f"call {call}"
        assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, 1e-2, 1e-2,
                          what=f"static scratch call {call}")
        assert int(status.item()) == 0


def test_static_scratch_reports_bad_index_then_clears(lib):
    dev = torch.device("cuda:0")
    wl = workloads.make_random(2, 1, 64, 512, 3000, 900, seed=403)
    x = _gpu.prepare(wl, dev, quantise=False)
    bad = dict(x)
    bad["idx"] = x["idx"].clone()
    bad["idx"][1, 0, 17] = wl.rows
    status = torch.zeros((1,), dtype=torch.int32, device=dev)
    o = torch.empty_like(x["q"])
    assert _call_static(lib, bad, wl, o, status) == _lib.SA_OK
    torch.cuda.synchronize()
    assert int(status.item()) & 1
    ref = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale)
    assert _call_static(lib, x, wl, o, status) == _lib.SA_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0  # cleared at the start of the call
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), _gpu.bf16_tensor_to_u16(ref), 1e-2, 1e-2,
                      what="after a bad call")


def test_static_scratch_rejects_shapes_beyond_the_array(lib):
    # head_dim 448 runs in the mma.sync family, whose split partials for this shape need more
    # than the array holds
    dev = torch.device("cuda:0")
    b, s, h, d, rows, topk = 150, 1, 128, 448, 8, 2176
    need = lib.sa_sparse_attn_workspace_size(b, s, h, d, rows, topk, 0)
    assert need > STATIC_SCRATCH_BYTES
    q = torch.zeros((b, s, h, d), dtype=torch.bfloat16, device=dev)
    kv = torch.zeros((b, rows, d), dtype=torch.bfloat16, device=dev)
    idx = torch.full((b, s, topk), -1, dtype=torch.int32, device=dev)
    sink = torch.zeros(h, device=dev)
    o = torch.empty_like(q)
    x = dict(q=q, kv=kv, kv_scale=None, sink=sink, idx=idx)
    wl = type("W", (), dict(scale=0.1, b=b, s=s, h=h, d=d, rows=rows, topk=topk))
    assert _call_static(lib, x, wl, o, None) == _lib.SA_ERR_WORKSPACE


def test_static_scratch_checks_arguments_first(lib):
    dev = torch.device("cuda:0")
    wl = workloads.make_random(2, 3, 64, 512, 100, 70, seed=405)
    x = _gpu.prepare(wl, dev, quantise=False)
    status = torch.full((1,), 7, dtype=torch.int32, device=dev)
    # o overlapping q: refused before anything is enqueued (status_out untouched)
    assert _call_static(lib, x, wl, x["q"], status) == _lib.SA_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(status.item()) == 7
    # no tokens: nothing computed, and the status word reported as zero
    empty = dict(q=torch.empty((0, 3, 64, 512), dtype=torch.bfloat16, device=dev),
                 kv=x["kv"][:0], kv_scale=None, sink=x["sink"],
                 idx=torch.empty((0, 3, 70), dtype=torch.int32, device=dev))
    w0 = type("W", (), dict(scale=wl.scale, b=0, s=3, h=64, d=512, rows=100, topk=70))
    assert _call_static(lib, empty, w0, empty["q"], status) == _lib.SA_OK
    torch.cuda.synchronize()
    assert int(status.item()) == 0
