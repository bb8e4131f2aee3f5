"""sparse_attn for GB300: DeepSeek V4.1's index-gathered latent attention with an attention sink.

The public calls take torch CUDA tensors and pass their device pointers to the C-ABI library
(libsa.so, include/sparse_attn.h) on the current stream.  PyTorch provides device memory and
streams only; all the arithmetic runs in the library's sm_103a kernels.

    o = sparse_attn(q, kv, sink, idx, softmax_scale)            # bf16 kv
    o = sparse_attn(q, codes, sink, idx, scale, kv_scale=e8m0)  # fp8 e4m3 kv + e8m0 scales
    window_idxs(start_pos, seqlen, window, out=idx[..., :window])
    act_quant_fp8(x, out_rt=x)                                  # in-place block-32 round trip
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import (SA_KV_BF16, SA_KV_FP8_E4M3, SA_SCORE_BF16, SA_SCORE_F32, SA_STATUS_BYTES,
                   SparseAttnError, load, status_string)

__all__ = ["sparse_attn", "window_idxs", "act_quant_fp8", "window_write", "indexer_topk",
           "candidate_blocks", "hc_split_sinkhorn",
           "workspace_size", "new_workspace", "read_status", "SparseAttnError", "SA_KV_BF16",
           "SA_KV_FP8_E4M3", "SA_SCORE_F32", "SA_SCORE_BF16", "load"]


def _ptr(t) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _need(t, name, dtype, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def workspace_size(b, s, h, d, rows, topk, kv_format=SA_KV_BF16) -> int:
    n = int(load().sa_sparse_attn_workspace_size(b, s, h, d, rows, topk, kv_format))
    if n == 0:
        raise SparseAttnError(_lib.SA_ERR_UNSUPPORTED, "sa_sparse_attn_workspace_size")
    return n


def new_workspace(b, s, h, d, rows, topk, kv_format=SA_KV_BF16, device="cuda") -> torch.Tensor:
    """A zeroed uint8 workspace of the size the library asks for (status word cleared)."""
    return torch.zeros(workspace_size(b, s, h, d, rows, topk, kv_format), dtype=torch.uint8,
                       device=device)


FAMILIES = {"auto": _lib.SA_FAMILY_AUTO, "tcgen05": _lib.SA_FAMILY_TCGEN05,
            "mma": _lib.SA_FAMILY_MMA_SYNC}


def sparse_attn(q, kv, sink, idx, softmax_scale, *, kv_scale=None, out=None, workspace=None,
                rope=None, family=None, stream=None) -> torch.Tensor:
    """o[b, s, h, d] (bf16) = sparse_attn(q, kv, sink, idx, softmax_scale).

    q [b, s, h, d] bf16; kv [b, rows, d] bf16, or uint8 e4m3 codes with kv_scale [b, rows, d/32]
    uint8 e8m0; sink [h] f32; idx [b, s, topk] int32 (-1 = empty).
    rope=(rot, start_pos): also rotate o's last rot.shape[1] * 2 dims back by the inverse rotary
    embedding of positions start_pos + si, rot [positions, rope_dim / 2, 2] f32 (cos, sin).
    family: None (= "auto"), "tcgen05" or "mma" -- the kernel family that computes the call."""
    _need(q, "q", torch.bfloat16)
    dev = q.device
    b, s, h, d = q.shape
    fmt = SA_KV_BF16 if kv_scale is None else SA_KV_FP8_E4M3
    _need(kv, "kv", torch.bfloat16 if fmt == SA_KV_BF16 else torch.uint8, dev)
    if kv.dim() != 3 or kv.shape[0] != b or kv.shape[2] != d:
        raise ValueError(f"kv shape {tuple(kv.shape)} does not match q {tuple(q.shape)}")
    rows = kv.shape[1]
    if kv_scale is not None:
        _need(kv_scale, "kv_scale", torch.uint8, dev)
        if tuple(kv_scale.shape) != (b, rows, d // 32):
            raise ValueError(f"kv_scale shape {tuple(kv_scale.shape)} != {(b, rows, d // 32)}")
    _need(sink, "sink", torch.float32, dev)
    if tuple(sink.shape) != (h,):
        raise ValueError(f"sink shape {tuple(sink.shape)} != ({h},)")
    _need(idx, "idx", torch.int32, dev)
    if idx.dim() != 3 or idx.shape[0] != b or idx.shape[1] != s:
        raise ValueError(f"idx shape {tuple(idx.shape)} does not match q {tuple(q.shape)}")
    topk = idx.shape[2]
    if out is None:
        out = torch.empty_like(q)
    else:
        _need(out, "out", torch.bfloat16, dev)
        if out.shape != q.shape:
            raise ValueError("out must have q's shape")
    if workspace is None:
        workspace = new_workspace(b, s, h, d, rows, topk, fmt, device=dev)
    else:
        _need(workspace, "workspace", torch.uint8, dev)
    if family is not None and family not in FAMILIES:
        raise ValueError(f"family must be one of {sorted(FAMILIES)}")
    if rope is not None:
        if family not in (None, "auto", "tcgen05"):
            raise ValueError("the fused rotation runs in the tcgen05 family only")
        rot, start_pos = rope
        _need(rot, "rot", torch.float32, dev)
        if rot.dim() != 3 or rot.shape[2] != 2:
            raise ValueError(f"rot shape {tuple(rot.shape)} is not [positions, rope_dim / 2, 2]")
        st = load().sa_sparse_attn_rope(_ptr(q), _ptr(kv), _ptr(kv_scale), fmt, _ptr(sink),
                                        _ptr(idx), float(softmax_scale), b, s, h, d, rows, topk,
                                        _ptr(out), _ptr(workspace), workspace.numel(), _ptr(rot),
                                        rot.shape[0], 2 * rot.shape[1], int(start_pos),
                                        _stream(stream))
        _lib.check(st, "sa_sparse_attn_rope")
        return out
    if family is not None:
        st = load().sa_sparse_attn_family(_ptr(q), _ptr(kv), _ptr(kv_scale), fmt, _ptr(sink),
                                          _ptr(idx), float(softmax_scale), b, s, h, d, rows, topk,
                                          _ptr(out), _ptr(workspace), workspace.numel(),
                                          FAMILIES[family], _stream(stream))
        _lib.check(st, "sa_sparse_attn_family")
        return out
    st = load().sa_sparse_attn(_ptr(q), _ptr(kv), _ptr(kv_scale), fmt, _ptr(sink), _ptr(idx),
                               float(softmax_scale), b, s, h, d, rows, topk, _ptr(out),
                               _ptr(workspace), workspace.numel(), _stream(stream))
    _lib.check(st, "sa_sparse_attn")
    return out


def _score_format(score, name="score"):
    if not isinstance(score, torch.Tensor) or not score.is_cuda or score.dim() != 3:
        raise TypeError(f"{name} must be a 3-D CUDA tensor")
    if not score.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if score.dtype == torch.float32:
        return SA_SCORE_F32
    if score.dtype == torch.bfloat16:
        return SA_SCORE_BF16
    raise TypeError(f"{name} must be float32 or bfloat16, got {score.dtype}")


def hc_split_sinkhorn(mixes, hc_scale, hc_base, hc=4, sinkhorn_iters=20, eps=1e-6, *,
                      stream=None):
    """hc_split_sinkhorn: mixes [..., (2 + hc) * hc] f32, hc_scale [3], hc_base [(2 + hc) * hc]
    -> (pre [..., hc], post [..., hc], comb [..., hc, hc]), all f32."""
    for t, name in ((mixes, "mixes"), (hc_scale, "hc_scale"), (hc_base, "hc_base")):
        _need(t, name, torch.float32, mixes.device)
    mix = (2 + hc) * hc
    if mixes.shape[-1] != mix or tuple(hc_scale.shape) != (3,) or tuple(hc_base.shape) != (mix,):
        raise ValueError(f"shapes do not fit hc = {hc}: mixes [..., {mix}], hc_scale [3], "
                         f"hc_base [{mix}]")
    lead = tuple(mixes.shape[:-1])
    n = mixes.numel() // mix
    pre = torch.empty(lead + (hc,), dtype=torch.float32, device=mixes.device)
    post = torch.empty_like(pre)
    comb = torch.empty(lead + (hc, hc), dtype=torch.float32, device=mixes.device)
    st = load().sa_hc_split_sinkhorn(_ptr(mixes), n, hc, _ptr(hc_scale), _ptr(hc_base),
                                     int(sinkhorn_iters), float(eps), _ptr(pre), _ptr(post),
                                     _ptr(comb), _stream(stream))
    _lib.check(st, "sa_hc_split_sinkhorn")
    return pre, post, comb


def candidate_blocks(logits, start_pos, ratio, topk_blocks, block_size, *, out=None,
                     stream=None) -> torch.Tensor:
    """select_candidate_blocks: logits [b, s, n_comp] (f32 or bf16) -> bool mask [b, s, n_comp],
    True inside the topk_blocks best blocks of block_size positions (the block of the query's
    newest visible position always kept, -inf blocks never)."""
    fmt = _score_format(logits, "logits")
    b, s, n = logits.shape
    if out is None:
        out = torch.empty((b, s, n), dtype=torch.bool, device=logits.device)
    elif out.dtype != torch.bool or tuple(out.shape) != (b, s, n) or not out.is_contiguous():
        raise ValueError(f"out must be a contiguous bool tensor of shape {(b, s, n)}")
    st = load().sa_candidate_blocks(_ptr(logits), fmt, b, s, n, int(start_pos), int(ratio),
                                    int(topk_blocks), int(block_size), _ptr(out),
                                    _stream(stream))
    _lib.check(st, "sa_candidate_blocks")
    return out


def indexer_topk(score, start_pos, ratio, index_topk, offset, *, candidates=None, out=None,
                 stream=None):
    """The indexer's selection: score [b, s, n_comp] (f32 or bf16, n_comp = (start_pos + s) //
    ratio) -> idx [b, s, k] int32, k = min(index_topk, n_comp): the top-k positions in position
    order, + offset, -1 for a position the query does not see.  ``candidates`` (bool [b, s,
    n_comp], e.g. from candidate_blocks) masks the scores outside it first.  ``out`` may be a
    column slice of a wider idx tensor (its row and batch strides are used)."""
    fmt = _score_format(score)
    b, s, n = score.shape
    if candidates is not None and (candidates.dtype != torch.bool or tuple(candidates.shape) !=
                                   (b, s, n) or not candidates.is_contiguous()):
        raise ValueError(f"candidates must be a contiguous bool tensor of shape {(b, s, n)}")
    k = min(int(index_topk), n)
    if out is None:
        out = torch.empty((b, s, k), dtype=torch.int32, device=score.device)
    if out.dtype != torch.int32 or not out.is_cuda or tuple(out.shape) != (b, s, k) or (
            k > 0 and out.stride(2) != 1):
        raise ValueError(f"out must be a CUDA int32 tensor of shape {(b, s, k)} with unit column "
                         "stride")
    ld = out.stride(1) if s > 1 else max(k, out.stride(1))
    bstride = out.stride(0) if b > 1 else s * ld
    st = load().sa_indexer_topk(_ptr(score), fmt, _ptr(candidates), b, s, n, int(start_pos),
                                int(ratio),
                                int(index_topk), int(offset), _ptr(out), ld, bstride,
                                _stream(stream))
    _lib.check(st, "sa_indexer_topk")
    return out


def window_idxs(start_pos, seqlen, window, *, out=None, nbatch=1, stream=None, device="cuda"):
    """Window index table [nbatch, seqlen, window] (int32), written into ``out`` when given
    (``out`` may be a column slice of a wider idx tensor: its row and batch strides are used)."""
    if out is None:
        out = torch.empty((nbatch, seqlen, window), dtype=torch.int32, device=device)
    if out.dtype != torch.int32 or not out.is_cuda:
        raise TypeError("out must be a CUDA int32 tensor")
    if out.dim() == 2:
        out3 = out.unsqueeze(0)
    else:
        out3 = out
    if tuple(out3.shape) != (nbatch, seqlen, window) or out3.stride(2) != 1:
        raise ValueError(f"out shape {tuple(out.shape)} / strides do not fit ({nbatch}, {seqlen}, "
                         f"{window}) with unit column stride")
    ld = out3.stride(1) if seqlen > 1 else max(window, out3.stride(1))
    bstride = out3.stride(0) if nbatch > 1 else seqlen * ld
    st = load().sa_window_idxs(start_pos, seqlen, window, _ptr(out3), ld, nbatch, bstride,
                               _stream(stream))
    _lib.check(st, "sa_window_idxs")
    return out


def act_quant_fp8(x, *, out_rt=None, codes=None, scales=None, stream=None):
    """Block-32 e4m3 quantisation of the rows of a 2-D bf16 tensor (last dim contiguous).

    Writes the bf16 round trip into ``out_rt`` (may be ``x`` itself), the e4m3 codes into
    ``codes`` and the e8m0 block scales into ``scales`` (each a 2-D tensor with unit column
    stride; rows may be strided, e.g. one ring slot per sequence of a cache)."""
    if x.dim() != 2 or x.stride(1) != 1 or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise ValueError("x must be a 2-D CUDA bf16 tensor with unit column stride")
    n, d = x.shape

    def rows_of(t, name, dtype, width):
        if t is None:
            return None, 0
        if t.dim() != 2 or t.dtype != dtype or t.stride(1) != 1 or tuple(t.shape) != (n, width):
            raise ValueError(f"{name} must be a 2-D {dtype} tensor of shape ({n}, {width}) with "
                             "unit column stride")
        return t, t.stride(0)

    rt, rts = rows_of(out_rt, "out_rt", torch.bfloat16, d)
    cd, cds = rows_of(codes, "codes", torch.uint8, d)
    sc, scs = rows_of(scales, "scales", torch.uint8, d // 32)
    st = load().sa_act_quant_fp8(_ptr(x), n, d, x.stride(0), _ptr(rt), rts, _ptr(cd), cds,
                                 _ptr(sc), scs, _stream(stream))
    _lib.check(st, "sa_act_quant_fp8")


def window_write(x, start_pos, *, ring_rt=None, codes=None, scales=None, stream=None):
    """The ring write with act_quant fused (sa_window_write): row t of x[bi] (the new token at
    position start_pos + t of sequence bi) goes to ring slot (start_pos + t) % window.

    x is a 3-D CUDA bf16 tensor [nbatch, seqlen, d] (last dim contiguous, rows of a sequence
    equally spaced, sequences seqlen rows apart).  The rings are 3-D tensors [nbatch, window, d]
    (bf16 round trip ``ring_rt``, e4m3 ``codes``) or [nbatch, window, d / 32] (e8m0 ``scales``)
    with unit column stride; they may be strided views of a larger cache, e.g. its first window
    rows."""
    if x.dim() != 3 or x.stride(2) != 1 or x.dtype != torch.bfloat16 or not x.is_cuda:
        raise ValueError("x must be a 3-D CUDA bf16 tensor with unit column stride")
    nb, sl, d = x.shape
    if nb > 1 and x.stride(0) != sl * x.stride(1):
        raise ValueError("the sequences of x must be seqlen rows apart")
    window = None

    def ring_of(t, name, dtype, width):
        nonlocal window
        if t is None:
            return None, 0, 0
        if (t.dim() != 3 or t.dtype != dtype or t.stride(2) != 1 or t.shape[0] != nb
                or t.shape[2] != width):
            raise ValueError(f"{name} must be a 3-D {dtype} tensor of shape ({nb}, window, {width})"
                             " with unit column stride")
        if window is None:
            window = t.shape[1]
        elif t.shape[1] != window:
            raise ValueError("the rings must have the same window")
        return t, t.stride(1), t.stride(0)

    rt, rts, rtb = ring_of(ring_rt, "ring_rt", torch.bfloat16, d)
    cd, cds, cdb = ring_of(codes, "codes", torch.uint8, d)
    sc, scs, scb = ring_of(scales, "scales", torch.uint8, d // 32)
    if window is None:
        raise ValueError("give at least one of ring_rt, codes, scales")
    st = load().sa_window_write(_ptr(x), nb, sl, d, x.stride(1) if sl > 1 else d, int(start_pos),
                                window, _ptr(rt), rts, rtb, _ptr(cd), cds, cdb, _ptr(sc), scs, scb,
                                _stream(stream))
    _lib.check(st, "sa_window_write")


def read_status(workspace, clear=False, stream=None) -> int:
    """The workspace status word as an sa_status (synchronises the stream)."""
    return int(load().sa_read_status(_ptr(workspace), int(bool(clear)), _stream(stream)))
