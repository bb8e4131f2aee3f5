"""CPU oracle for DeepSeek V4.1 sparse latent attention -- TEST INFRASTRUCTURE ONLY.

The plain, slow definition of every step on the path, used to check the CUDA library.  Only
``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline / reference leg may
import this package; the product path never does.  The arithmetic lives in ``sa_oracle.c``
(plain C, f64), which shares nothing with the CUDA sources; this module compiles it with gcc on
first use and marshals numpy arrays through ctypes.

Sources (see the header of ``sa_oracle.c``): the "Module attn" API page of the spark_model
deepseek_v41_ref docs (precision paragraph, ring-cache paragraph, act_quant_inplace, pow2_ceil,
sparse_attn, window_topk_idxs), the "DeepSeek V4.1" attention output page (Attention.forward /
__init__, apply_rotary_emb), its source-layer attention page in the indexer view
(Indexer.forward's selection, select_candidate_blocks) and its attention-write page
(hc_split_sinkhorn).
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "sa_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

# Status codes of the C functions
OK, BAD_ARG, UNSUPPORTED, BAD_INDEX = 0, 1, 2, 3


def build(force: bool = False) -> str:
    """Compile ``liboracle.so`` next to its source (gcc, IEEE arithmetic, no FMA contraction)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
               "-fno-fast-math", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.or_bf16_round.restype = ctypes.c_uint16
            lib.or_bf16_round.argtypes = [ctypes.c_double]
            lib.or_bf16_to_f64.restype = ctypes.c_double
            lib.or_bf16_to_f64.argtypes = [ctypes.c_uint16]
            lib.or_e4m3_to_f64.restype = ctypes.c_double
            lib.or_e4m3_to_f64.argtypes = [ctypes.c_uint8]
            lib.or_e4m3_encode.restype = ctypes.c_uint8
            lib.or_e4m3_encode.argtypes = [ctypes.c_float]
            lib.or_pow2_ceil.restype = ctypes.c_float
            lib.or_pow2_ceil.argtypes = [ctypes.c_float]
            lib.or_act_quant.restype = ctypes.c_int
            lib.or_act_quant.argtypes = [P, i64, i64, P, P, P]
            lib.or_window_idxs.restype = ctypes.c_int
            lib.or_window_idxs.argtypes = [i64, i64, i64, P, i64]
            lib.or_rope.restype = ctypes.c_int
            lib.or_rope.argtypes = [P, i64, i64, i64, P, i64, P, ctypes.c_int, P]
            lib.or_ring_write.restype = ctypes.c_int
            lib.or_ring_write.argtypes = [P, P, i64, i64, i64, i64]
            lib.or_indexer_topk.restype = ctypes.c_int
            lib.or_indexer_topk.argtypes = [P, i64, i64, i64, i64, i64, i64, i64, P]
            lib.or_candidate_blocks.restype = ctypes.c_int
            lib.or_candidate_blocks.argtypes = [P, i64, i64, P, i64, i64, P]
            lib.or_hc_split_sinkhorn.restype = ctypes.c_int
            lib.or_hc_split_sinkhorn.argtypes = [P, i64, i64, P, P, i64, ctypes.c_double, P, P, P]
            for name in ("or_bf16_round_array", "or_e4m3_encode_array", "or_e4m3_decode_array",
                         "or_pow2_ceil_array"):
                getattr(lib, name).restype = None
                getattr(lib, name).argtypes = [P, P, i64]
            lib.or_sparse_attn.restype = ctypes.c_int
            lib.or_sparse_attn.argtypes = [P, P, P, P, ctypes.c_int, P, P, ctypes.c_float,
                                           i64, i64, i64, i64, i64, i64, P, i64, P, P,
                                           ctypes.c_int]
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# --------------------------------------------------------------------------------------------
# scalar codecs (vectorised by plain loops over the C scalar functions)
# --------------------------------------------------------------------------------------------

def _array_call(name, x, in_dtype, out_dtype):
    lib = _load()
    a = np.ascontiguousarray(x, dtype=in_dtype)
    out = np.empty(a.shape, out_dtype)
    getattr(lib, name)(_ptr(a), _ptr(out), a.size)
    return out


def bf16_round(x) -> np.ndarray:
    """f64 -> bf16 bits (uint16), round to nearest even."""
    return _array_call("or_bf16_round_array", x, np.float64, np.uint16)


def bf16_to_f64(bits) -> np.ndarray:
    """bf16 bits -> exact f64 (the widening is a bit shift, done here in numpy)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def e4m3_decode(codes) -> np.ndarray:
    """e4m3 byte -> f64 value (NaN for the two NaN codes)."""
    return _array_call("or_e4m3_decode_array", codes, np.uint8, np.float64)


def e4m3_encode(x) -> np.ndarray:
    """f32 -> e4m3 byte, round to nearest even, saturating at +-448."""
    return _array_call("or_e4m3_encode_array", x, np.float32, np.uint8)


def pow2_ceil(v) -> np.ndarray:
    """2 ** ceil(log2 v) for positive normal f32, from the IEEE fields."""
    return _array_call("or_pow2_ceil_array", v, np.float32, np.float32)


# --------------------------------------------------------------------------------------------
# the path's operations
# --------------------------------------------------------------------------------------------

def act_quant(x_bf16: np.ndarray):
    """Block-32 e4m3 / ue8m0 round trip of bf16 rows.

    ``x_bf16`` is uint16 [..., d] (bf16 bits), d % 32 == 0.  Returns (x_rt bf16 bits [..., d],
    codes uint8 [..., d], scales uint8 [..., d/32])."""
    lib = _load()
    x = _c(x_bf16, np.uint16)
    d = x.shape[-1]
    n = x.size // d if d else 0
    x_rt = np.empty_like(x)
    codes = np.empty(x.shape, np.uint8)
    scales = np.empty(x.shape[:-1] + (d // 32,), np.uint8)
    rc = lib.or_act_quant(_ptr(x), n, d, _ptr(x_rt), _ptr(codes), _ptr(scales))
    if rc != OK:
        raise ValueError(f"or_act_quant failed ({rc})")
    return x_rt, codes, scales


def window_idxs(start_pos: int, seqlen: int, window: int) -> np.ndarray:
    """[seqlen][window] int32 slot indices (prefill: start_pos == 0; decode: seqlen == 1)."""
    lib = _load()
    out = np.empty((seqlen, window), np.int32)
    rc = lib.or_window_idxs(start_pos, seqlen, window, _ptr(out), window)
    if rc == UNSUPPORTED:
        raise NotImplementedError("chunked prefill (start_pos > 0 and seqlen > 1)")
    if rc != OK:
        raise ValueError(f"or_window_idxs failed ({rc})")
    return out


def _widen_scores(score) -> np.ndarray:
    score = np.asarray(score)
    if score.dtype == np.uint16:  # bf16 bits, widened exactly
        score = (score.astype(np.uint32) << 16).view(np.float32)
    return _c(score, np.float32)


def visible_positions(s: int, n_comp: int, start_pos: int, ratio: int) -> np.ndarray:
    """[s] positions each query of a call sees (Indexer.forward's compress_lens): (si + 1) //
    ratio at a prefill, all n_comp at a decode step."""
    if start_pos == 0:
        return (np.arange(1, s + 1, dtype=np.int64) // ratio).astype(np.int64)
    return np.full(s, n_comp, np.int64)


def indexer_topk(score, start_pos: int, ratio: int, index_topk: int, offset: int,
                 candidates=None) -> np.ndarray:
    """The indexer's selection on score [b, s, n_comp] (f32, or bf16 bits as uint16, widened
    exactly): idx [b, s, min(index_topk, n_comp)] int32 (see or_indexer_topk).  ``candidates``
    (bool [b, s, n_comp]) first masks every score outside it to -inf, as a layer that uses
    another layer's candidate blocks does (Indexer.forward, the uses_candidates branch)."""
    lib = _load()
    sc = _widen_scores(score)
    if candidates is not None:
        sc = np.where(np.asarray(candidates, bool), sc, np.float32(-np.inf)).astype(np.float32)
    b, s, n = sc.shape
    k = min(index_topk, n)
    out = np.empty((b, s, k), np.int32)
    rc = lib.or_indexer_topk(_ptr(sc), b, s, n, start_pos, ratio, index_topk, offset, _ptr(out))
    if rc == UNSUPPORTED:
        raise NotImplementedError("chunked prefill (start_pos > 0 and seqlen > 1)")
    if rc != OK:
        raise ValueError(f"or_indexer_topk failed ({rc})")
    return out


def candidate_blocks(logits, start_pos: int, ratio: int, topk_blocks: int,
                     block_size: int) -> np.ndarray:
    """select_candidate_blocks on logits [b, s, n_comp] (f32 or bf16 bits) of one indexer call at
    start_pos: the bool mask [b, s, n_comp] of the positions in kept blocks (or_candidate_blocks),
    each query seeing the positions visible_positions() gives it."""
    sc = _widen_scores(logits)
    b, s, n = sc.shape
    vis = np.tile(visible_positions(s, n, start_pos, ratio), b)
    return candidate_blocks_rows(sc.reshape(b * s, n), vis, topk_blocks, block_size).reshape(
        b, s, n)


def candidate_blocks_rows(logits, visible, topk_blocks: int, block_size: int) -> np.ndarray:
    """or_candidate_blocks on rows [rows, width] (f32 or bf16 bits), row r seeing its first
    visible[r] positions: bool mask [rows, width]."""
    lib = _load()
    sc = _widen_scores(logits)
    rows, n = sc.shape
    vis = np.ascontiguousarray(np.asarray(visible, np.int64))
    out = np.empty((rows, n), np.uint8)
    rc = lib.or_candidate_blocks(_ptr(sc), rows, n, _ptr(vis), topk_blocks, block_size,
                                 _ptr(out))
    if rc != OK:
        raise ValueError(f"or_candidate_blocks failed ({rc})")
    return out.astype(bool)


def hc_split_sinkhorn(mixes, hc_scale, hc_base, hc: int = 4, iters: int = 20,
                      eps: float = 1e-6):
    """hc_split_sinkhorn on mixes [..., (2 + hc) * hc] f32 with hc_scale [3], hc_base
    [(2 + hc) * hc] (f32): (pre [..., hc], post [..., hc], comb [..., hc, hc]) in f64."""
    lib = _load()
    m = _c(mixes, np.float32)
    lead = m.shape[:-1]
    mix = (2 + hc) * hc
    if m.shape[-1] != mix:
        raise ValueError(f"mixes rows must have {mix} values")
    n = int(np.prod(lead)) if lead else 1
    sc, bs = _c(hc_scale, np.float32), _c(hc_base, np.float32)
    pre = np.empty((n, hc), np.float64)
    post = np.empty((n, hc), np.float64)
    comb = np.empty((n, hc, hc), np.float64)
    rc = lib.or_hc_split_sinkhorn(_ptr(m), n, hc, _ptr(sc), _ptr(bs), iters, eps, _ptr(pre),
                                  _ptr(post), _ptr(comb))
    if rc != OK:
        raise ValueError(f"or_hc_split_sinkhorn failed ({rc})")
    return pre.reshape(lead + (hc,)), post.reshape(lead + (hc,)), comb.reshape(lead + (hc, hc))


def ring_write(ring: np.ndarray, rows: np.ndarray, start_pos: int) -> None:
    """Write kv rows [seqlen][d] (bf16 bits) for positions start_pos.. into ring [window][d]."""
    lib = _load()
    assert ring.dtype == np.uint16 and ring.flags.c_contiguous
    r = _c(rows, np.uint16)
    rc = lib.or_ring_write(_ptr(ring), _ptr(r), start_pos, r.shape[0], ring.shape[0], ring.shape[1])
    if rc != OK:
        raise ValueError(f"or_ring_write failed ({rc})")


def rope(x, rot, pos, rope_dim, inverse, want_f64=False):
    """apply_rotary_emb on the last ``rope_dim`` elements of each row of x (bf16 bits, [..., d]):
    rows of x flattened in order, row r at position pos[r] of the table rot ([npos, rope_dim/2, 2]
    f32 cos, sin); ``inverse`` conjugates the rotation.  Returns a new array (and, with want_f64,
    the unrounded rotated values [rows, rope_dim])."""
    lib = _load()
    x = np.array(x, dtype=np.uint16, copy=True, order="C")
    d = x.shape[-1]
    n = x.size // d
    r = _c(rot, np.float32)
    p = _c(np.asarray(pos, dtype=np.int64).reshape(-1), np.int64)
    assert p.size == n
    x64 = np.empty((n, rope_dim), np.float64) if want_f64 else None
    rc = lib.or_rope(_ptr(x), n, d, rope_dim, _ptr(r), r.shape[0], _ptr(p), int(bool(inverse)),
                     _ptr(x64) if want_f64 else None)
    if rc != OK:
        raise ValueError(f"or_rope failed ({rc})")
    return (x, x64) if want_f64 else x


def sparse_attn(q, kv, sink, idx, scale, *, kv_scales=None, tokens=None, nthreads=None,
                want_f64=False):
    """The plain definition of sparse_attn.

    q      uint16 [b, s, h, d] bf16 bits
    kv     uint16 [b, rows, d] bf16 bits, or (kv_scales given) uint8 e4m3 codes [b, rows, d]
    kv_scales uint8 [b, rows, d/32] e8m0, or None
    sink   float32 [h]
    idx    int32 [b, s, topk], -1 = empty
    scale  softmax scale, used as the f32 value
    tokens optional int64 list of flat token ids (b_i * s + s_i): only those are computed and the
           result is [len(tokens), h, d]; otherwise [b, s, h, d].
    Returns bf16 bits (uint16) and, with want_f64, the unrounded f64 result as a second value.
    """
    lib = _load()
    q = _c(q, np.uint16)
    b, s, h, d = q.shape
    fmt = 0 if kv_scales is None else 1
    kv = _c(kv, np.uint16 if fmt == 0 else np.uint8)
    rows = kv.shape[1]
    sc = None if kv_scales is None else _c(kv_scales, np.uint8)
    sink = _c(sink, np.float32)
    idx = _c(idx, np.int32)
    topk = idx.shape[-1]
    assert idx.shape == (b, s, topk) and kv.shape == (b, rows, d) and sink.shape == (h,)
    if tokens is None:
        tk = None
        out_shape = (b, s, h, d)
        nt = b * s
    else:
        tk = _c(tokens, np.int64)
        nt = tk.size
        out_shape = (nt, h, d)
    o = np.empty(out_shape, np.uint16)
    o64 = np.empty(out_shape, np.float64) if want_f64 else None
    if nthreads is None:
        nthreads = os.cpu_count() or 1
    rc = lib.or_sparse_attn(_ptr(q), _ptr(kv) if fmt == 0 else None,
                            _ptr(kv) if fmt == 1 else None, _ptr(sc), fmt, _ptr(sink), _ptr(idx),
                            float(np.float32(scale)), b, s, h, d, rows, topk, _ptr(tk), nt,
                            _ptr(o), _ptr(o64), int(nthreads))
    if rc == BAD_INDEX:
        raise IndexError("an index is outside [-1, rows)")
    if rc != OK:
        raise ValueError(f"or_sparse_attn failed ({rc})")
    return (o, o64) if want_f64 else o
