"""Pins of the CPU oracle to facts outside itself: library routines, closed forms, invariants,
brute force and the pages' worked examples.  No GPU needed."""

from __future__ import annotations

import concurrent.futures
import itertools
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from sparse_latent_attention_gb300 import workloads
from tests._helpers import bf16_to_f64, compose_idx_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# --------------------------------------------------------------------------------------------
# small random problems
# --------------------------------------------------------------------------------------------

def _problem(seed, b=2, s=3, h=5, d=32, rows=20, topk=9, neg=0.2, distinct=True):
    rng = np.random.default_rng(seed)
    q = workloads.to_bf16_bits(rng.standard_normal((b, s, h, d), dtype=np.float32))
    kv = workloads.to_bf16_bits(rng.standard_normal((b, rows, d), dtype=np.float32))
    sink = rng.standard_normal(h).astype(np.float32)
    if distinct:
        idx = np.stack([np.stack([rng.choice(rows, topk, replace=False) for _ in range(s)])
                        for _ in range(b)]).astype(np.int32)
    else:
        idx = rng.integers(0, rows, (b, s, topk)).astype(np.int32)
    idx[rng.random(idx.shape) < neg] = -1
    scale = np.float32(d ** -0.5)
    return q, kv, sink, idx, scale


def _dense_reference(q, kv, sink, idx, scale):
    """Brute force: a dense [h, rows] logit matrix per token, every unlisted row masked to -inf,
    listed rows weighted by their multiplicity (log count added), one extra sink column whose
    value row is zero, and scipy's softmax over the lot."""
    b, s, h, d = q.shape
    rows = kv.shape[1]
    qf, kf = bf16_to_f64(q), bf16_to_f64(kv)
    out = np.zeros((b, s, h, d))
    for bi in range(b):
        for si in range(s):
            counts = np.bincount(idx[bi, si][idx[bi, si] >= 0], minlength=rows).astype(float)
            if counts.sum() == 0:
                continue
            logits = float(np.float32(scale)) * (qf[bi, si] @ kf[bi].T)  # [h, rows]
            with np.errstate(divide="ignore"):
                logits = logits + np.log(counts)[None, :]  # -inf where unlisted
            full = np.concatenate([logits, sink.astype(np.float64)[:, None]], axis=1)
            p = scipy.special.softmax(full, axis=1)
            values = np.concatenate([kf[bi], np.zeros((1, d))], axis=0)
            out[bi, si] = p @ values
    return out


@pytest.mark.parametrize("seed,distinct", [(11, True), (12, True), (13, False)])
def test_sparse_attn_matches_dense_masked_softmax(seed, distinct):
    q, kv, sink, idx, scale = _problem(seed, distinct=distinct)
    idx[0, 1, :] = -1  # one token with nothing listed
    o, o64 = oracle.sparse_attn(q, kv, sink, idx, scale, want_f64=True)
    ref = _dense_reference(q, kv, sink, idx, scale)
    np.testing.assert_allclose(o64, ref, rtol=1e-12, atol=1e-13)
    # the bf16 output is the rounding of the f64 result, checked against torch's f64 -> bf16
    # conversion where f32 holds the value exactly
    t = torch.from_numpy(o64.astype(np.float32)).to(torch.bfloat16).view(torch.int16).numpy()
    agree = (t.view(np.uint16) == o).mean()
    assert agree > 0.999


def test_sink_to_minus_inf_is_plain_softmax():
    q, kv, sink, idx, scale = _problem(21, neg=0.0)
    ninf = np.full_like(sink, -np.inf)
    _, o64 = oracle.sparse_attn(q, kv, ninf, idx, scale, want_f64=True)
    qf, kf = bf16_to_f64(q), bf16_to_f64(kv)
    for bi in range(q.shape[0]):
        for si in range(q.shape[1]):
            g = kf[bi, idx[bi, si]]
            p = scipy.special.softmax(float(scale) * qf[bi, si] @ g.T, axis=1)
            np.testing.assert_allclose(o64[bi, si], p @ g, rtol=1e-12, atol=1e-13)
    # a very negative finite sink approaches the same limit
    _, o64b = oracle.sparse_attn(q, kv, np.full_like(sink, -1e4), idx, scale, want_f64=True)
    np.testing.assert_allclose(o64b, o64, rtol=1e-12, atol=1e-13)


def test_index_order_invariance():
    q, kv, sink, idx, scale = _problem(31, topk=15)
    o, o64 = oracle.sparse_attn(q, kv, sink, idx, scale, want_f64=True)
    rng = np.random.default_rng(5)
    perm = np.stack([np.stack([rng.permutation(idx.shape[-1]) for _ in range(idx.shape[1])])
                     for _ in range(idx.shape[0])])
    idx_p = np.take_along_axis(idx, perm, axis=-1)
    o2, o64b = oracle.sparse_attn(q, kv, sink, idx_p, scale, want_f64=True)
    np.testing.assert_allclose(o64b, o64, rtol=1e-12, atol=1e-14)
    same = (o2 == o).mean()
    assert same >= 0.999
    diff = np.abs(o2.astype(np.int32) - o.astype(np.int32))
    assert diff.max() <= 1


def test_all_minus_one_row_is_exact_zero():
    q, kv, sink, idx, scale = _problem(41)
    idx[:] = -1
    o = oracle.sparse_attn(q, kv, sink, idx, scale)
    assert (o == 0).all()
    # also with a sink of -inf (defined as 0)
    o = oracle.sparse_attn(q, kv, np.full_like(sink, -np.inf), idx, scale)
    assert (o == 0).all()


def test_single_row_without_sink_returns_that_row_bit_exact():
    q, kv, sink, idx, scale = _problem(51)
    idx[:] = -1
    idx[..., 3] = 7
    o = oracle.sparse_attn(q, kv, np.full_like(sink, -np.inf), idx, scale)
    for bi in range(q.shape[0]):
        for si in range(q.shape[1]):
            for hh in range(q.shape[2]):
                assert (o[bi, si, hh] == kv[bi, 7]).all()


def test_identical_rows_closed_form():
    """All listed rows equal v: o = v * n / (n + exp(sink - l)), l = scale <q, v>."""
    q, kv, sink, idx, scale = _problem(61, neg=0.0)
    kv[:] = kv[:, :1, :]  # every row is row 0
    _, o64 = oracle.sparse_attn(q, kv, sink, idx, scale, want_f64=True)
    qf, kf = bf16_to_f64(q), bf16_to_f64(kv)
    n = idx.shape[-1]
    for bi in range(q.shape[0]):
        v = kf[bi, 0]
        l = float(scale) * (qf[bi] @ v)  # [s, h]
        w = n / (n + np.exp(sink.astype(np.float64)[None, :] - l))
        np.testing.assert_allclose(o64[bi], w[..., None] * v[None, None, :], rtol=1e-12,
                                   atol=1e-14)


def test_output_bounded_by_gathered_rows():
    q, kv, sink, idx, scale = _problem(71, topk=12)
    _, o64 = oracle.sparse_attn(q, kv, sink, idx, scale, want_f64=True)
    kf = bf16_to_f64(kv)
    for bi in range(q.shape[0]):
        for si in range(q.shape[1]):
            live = idx[bi, si][idx[bi, si] >= 0]
            bound = np.abs(kf[bi, live]).max(axis=0) if live.size else np.zeros(q.shape[-1])
            assert (np.abs(o64[bi, si]) <= bound[None, :] * (1 + 1e-15)).all()


def test_fp8_storage_equals_round_trip():
    """Attention over e4m3 codes + e8m0 scales equals attention over their bf16 round trip."""
    q, kv, sink, idx, scale = _problem(81, d=64)
    rt, codes, scales = oracle.act_quant(kv)
    a = oracle.sparse_attn(q, rt, sink, idx, scale)
    bq = oracle.sparse_attn(q, codes, sink, idx, scale, kv_scales=scales)
    assert (a == bq).all()


def test_out_of_range_index_refused():
    q, kv, sink, idx, scale = _problem(91)
    idx[0, 0, 0] = kv.shape[1]
    with pytest.raises(IndexError):
        oracle.sparse_attn(q, kv, sink, idx, scale)
    idx[0, 0, 0] = -2
    with pytest.raises(IndexError):
        oracle.sparse_attn(q, kv, sink, idx, scale)


def test_token_subset_matches_full():
    q, kv, sink, idx, scale = _problem(101, b=3, s=4)
    full = oracle.sparse_attn(q, kv, sink, idx, scale)
    toks = np.array([0, 5, 11, 7])
    part = oracle.sparse_attn(q, kv, sink, idx, scale, tokens=toks)
    assert (part == full.reshape(-1, *full.shape[2:])[toks]).all()


def test_tiny_workload_against_dense():
    wl = workloads.make_named("tiny")
    idx = compose_idx_oracle(wl)
    assert (idx[0, 11] == -1).all()
    kv = wl.kv_raw_dense()
    _, o64 = oracle.sparse_attn(wl.q, kv, wl.sink, idx, wl.scale, want_f64=True)
    np.testing.assert_allclose(o64, _dense_reference(wl.q, kv, wl.sink, idx, wl.scale),
                               rtol=1e-12, atol=1e-13)


# --------------------------------------------------------------------------------------------
# bf16 rounding
# --------------------------------------------------------------------------------------------

def test_bf16_round_matches_torch_on_f32_values():
    rng = np.random.default_rng(3)
    x = np.concatenate([rng.standard_normal(200000).astype(np.float32),
                        (rng.standard_normal(50000) * 1e-39).astype(np.float32),  # subnormal
                        (rng.standard_normal(50000) * 1e37).astype(np.float32),
                        np.array([0.0, -0.0, 3.3895314e38, -3.3895314e38], np.float32)])
    want = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(x.astype(np.float64))
    assert (got == want).all()


def test_bf16_round_f64_brute_force_nearest():
    """For f64 inputs (finer than f32) the result is the nearest bf16, ties to even mantissa."""
    rng = np.random.default_rng(4)
    # bf16 neighbours and their exact midpoints, nudged by tiny f64 amounts
    base = workloads.to_bf16_bits(rng.standard_normal(20000).astype(np.float32))
    lo = bf16_to_f64(base)
    hi = bf16_to_f64((base.astype(np.int32) + 1).astype(np.uint16))  # next magnitude
    mid = (lo + hi) / 2
    for x in (mid, mid + np.abs(mid) * 1e-12, mid - np.abs(mid) * 1e-12, lo + (hi - lo) * 0.3):
        got = bf16_to_f64(oracle.bf16_round(x))
        dlo, dhi = np.abs(x - lo), np.abs(x - hi)
        want = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi,
                        np.where(base % 2 == 0, lo, hi)))
        assert (got == want).all()


# --------------------------------------------------------------------------------------------
# e4m3 codec
# --------------------------------------------------------------------------------------------

def test_e4m3_decode_all_codes_matches_torch():
    codes = np.arange(256, dtype=np.uint8)
    got = oracle.e4m3_decode(codes)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert set(np.nonzero(nan)[0]) == {0x7F, 0xFF}
    assert np.isnan(got[nan]).all()
    assert (got[~nan] == want[~nan]).all()
    assert got[~nan].max() == 448.0 and got[~nan].min() == -448.0


def _e4m3_finite_values():
    v = oracle.e4m3_decode(np.arange(128, dtype=np.uint8))
    return np.arange(128)[~np.isnan(v)], v[~np.isnan(v)]


def test_e4m3_encode_matches_torch_and_brute_force():
    rng = np.random.default_rng(6)
    codes, vals = _e4m3_finite_values()
    mids = (vals[1:] + vals[:-1]) / 2
    x = np.concatenate([
        rng.standard_normal(300000) * 30, rng.standard_normal(100000) * 0.01,
        rng.uniform(-460, 460, 100000), vals, -vals, mids, -mids,
        np.nextafter(mids, 0), np.nextafter(mids, 1000)]).astype(np.float32)
    x = x[np.abs(x) < 464]  # torch turns larger magnitudes into NaN rather than saturating
    got = oracle.e4m3_encode(x)
    want = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert (got == want).all()
    # brute force on the mids and a sample: nearest finite value, ties to the even code
    xs = np.concatenate([mids, x[:20000].astype(np.float64)])
    a = np.abs(xs)
    dist = np.abs(a[:, None] - vals[None, :])
    best = dist.min(axis=1, keepdims=True)
    cand = dist == best
    pick_even = cand & (codes[None, :] % 2 == 0)
    choose = np.where(cand.sum(1) > 1, pick_even.argmax(1), cand.argmax(1))
    want_code = codes[choose] | np.where(np.signbit(xs), 0x80, 0)
    want_code = np.where(a == 0, np.where(np.signbit(xs), 0x80, 0), want_code)
    assert (oracle.e4m3_encode(xs.astype(np.float32)) == want_code).all()


def test_e4m3_encode_saturates():
    x = np.array([464, 480, 1e6, 3e38, -500, -1e9], np.float32)
    assert (oracle.e4m3_encode(x) == np.array([0x7E] * 4 + [0xFE] * 2, np.uint8)).all()


# --------------------------------------------------------------------------------------------
# pow2_ceil
# --------------------------------------------------------------------------------------------

@pytest.mark.slow
def test_pow2_ceil_exhaustive():
    """Every positive normal f32 against 2 ** ceil(log2 v) from numpy's frexp."""
    lo, hi = 0x00800000, 0x7F7FFFFF
    step = 1 << 22

    def chunk(start):
        bits = np.arange(start, min(start + step, hi + 1), dtype=np.uint32)
        v = bits.view(np.float32)
        m, e = np.frexp(v)  # v = m * 2^e, 0.5 <= m < 1
        ce = np.where(m == 0.5, e - 1, e)
        with np.errstate(over="ignore"):
            want = np.ldexp(np.float32(1.0), ce).astype(np.float32)
        got = oracle.pow2_ceil(v)
        return start, bool((got.view(np.uint32) == want.view(np.uint32)).all())

    # the chunks run on every core (numpy and the ctypes call release the GIL); still every value
    with concurrent.futures.ThreadPoolExecutor(max_workers=os.cpu_count() or 1) as pool:
        for start, ok in pool.map(chunk, range(lo, hi + 1, step)):
            assert ok, hex(start)


# --------------------------------------------------------------------------------------------
# act_quant
# --------------------------------------------------------------------------------------------

def _read_act_quant_examples():
    out = []
    for line in open(os.path.join(GOLDEN, "act_quant_examples.txt")):
        line = line.split("#")[0].strip()
        if not line:
            continue
        head, tail = line.split("|")
        parts = head.split()
        out.append((parts[0], int(parts[1]), [float(t) for t in parts[2:]],
                    [float(t) for t in tail.split()]))
    return out


@pytest.mark.parametrize("case", _read_act_quant_examples(), ids=lambda c: c[0])
def test_act_quant_worked_examples(case):
    name, e8m0, xin, xout = case
    x = np.zeros(32, np.float32)
    x[: len(xin)] = xin
    bits = workloads.to_bf16_bits(x)
    assert (bf16_to_f64(bits)[: len(xin)] == np.array(xin)).all(), "inputs must be bf16 values"
    rt, codes, scales = oracle.act_quant(bits[None])
    assert scales[0, 0] == e8m0
    got = bf16_to_f64(rt[0])
    assert (got[: len(xout)] == np.array(xout)).all(), got[: len(xout)]
    assert (got[len(xout):] == 0).all()


def test_act_quant_properties():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((64, 512)).astype(np.float32)
    x *= np.exp(rng.uniform(-20, 20, (64, 16))).repeat(32, axis=1).astype(np.float32)
    bits = workloads.to_bf16_bits(x)
    rt, codes, scales = oracle.act_quant(bits)
    xf = bf16_to_f64(bits).reshape(64, 16, 32)
    rtf = bf16_to_f64(rt).reshape(64, 16, 32)
    s = np.ldexp(1.0, scales.astype(np.int32) - 127)[..., None]
    amax = np.maximum(np.abs(xf).max(-1, keepdims=True), float(np.float32(1e-4)))
    # the scale is the smallest power of two that brings amax / s to <= 448
    assert (amax / s <= 448).all() and ((amax / (s / 2) > 448) | (s <= 2.0 ** -22)).all()
    # dequantised values are codes times scale, and the codes decode to the round trip
    dec = oracle.e4m3_decode(codes).reshape(64, 16, 32)
    assert (dec * s == rtf).all()
    # round to nearest: error at most half an e4m3 step of the value's binade (or subnormal step)
    y = xf / s
    step = np.where(np.abs(y) < 2.0 ** -6, 2.0 ** -9,
                    np.ldexp(1.0, np.floor(np.log2(np.maximum(np.abs(y), 1e-300))).astype(int) - 3))
    assert (np.abs(dec - y) <= step / 2 + 0.0).all()
    # the round trip is idempotent (codes and scales need not be: a block whose amax rounded
    # down onto 448 * 2^k takes the smaller scale the second time, with the same values)
    rt2, codes2, scales2 = oracle.act_quant(rt)
    assert (rt2 == rt).all()
    s2 = np.ldexp(1.0, scales2.astype(np.int32) - 127)[..., None]
    assert (oracle.e4m3_decode(codes2).reshape(64, 16, 32) * s2 == rtf).all()


# --------------------------------------------------------------------------------------------
# window indices and the ring cache
# --------------------------------------------------------------------------------------------

def _golden_ring():
    g = {}
    for line in open(os.path.join(GOLDEN, "ring_example.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, _kind, *vals = line.split()
            g[k] = [int(v) for v in vals]
    return g


def test_ring_worked_example():
    g = _golden_ring()
    W = g["window"][0]
    n = g["prefill_tokens"][0]
    ring = np.full((W, 1), 0xFFFF, np.uint16)
    tokens = np.arange(n + 2, dtype=np.uint16)[:, None]  # a row's value is its token number
    oracle.ring_write(ring, tokens[:n], 0)
    assert ring[:, 0].tolist() == g["prefill_ring"]
    for p in (12, 13):
        oracle.ring_write(ring, tokens[p:p + 1], p)
        assert int(np.nonzero(ring[:, 0] == p)[0][0]) == g[f"decode{p}_slot"][0]
        assert ring[:, 0].tolist() == g[f"decode{p}_ring"]
        idx = oracle.window_idxs(p, 1, W)[0]
        assert idx.tolist() == g[f"decode{p}_idx"]
        # the ring read in column order is the last W tokens, oldest first
        assert ring[idx, 0].tolist() == list(range(p - W + 1, p + 1))
    assert oracle.window_idxs(0, n, W)[3].tolist() == g["prefill_row3"]


def test_window_idxs_cases():
    # prefill: causal window, row i covers positions i-W+1..i
    w = oracle.window_idxs(0, 300, 128)
    for i in (0, 1, 127, 128, 299):
        row = w[i]
        want = [p if p >= 0 else -1 for p in range(i - 127, i + 1)]
        assert row.tolist() == want
    # shorter chunk than the window: still W columns, -1 first
    assert oracle.window_idxs(0, 3, 8).tolist()[2] == [-1] * 5 + [0, 1, 2]
    # decode before the ring is full: -1 first, then slots of positions 0..p
    assert oracle.window_idxs(5, 1, 8).tolist() == [[-1, -1, 0, 1, 2, 3, 4, 5]]
    # decode with a full ring at a multiple of W: oldest slot is (p+1) mod W
    assert oracle.window_idxs(32768, 1, 128)[0].tolist() == list(range(1, 128)) + [0]
    with pytest.raises(NotImplementedError):
        oracle.window_idxs(4, 3, 8)
    # empty chunk
    assert oracle.window_idxs(0, 0, 8).shape == (0, 8)


# --------------------------------------------------------------------------------------------
# apply_rotary_emb ("DeepSeek V4.1" attention page: the rotation of the output's rope dims)
# --------------------------------------------------------------------------------------------

def _rope_case(seed, n=40, d=512, rd=64, npos=50):
    rng = np.random.default_rng(seed)
    x = oracle.bf16_round(rng.standard_normal((n, d)) * np.exp(rng.uniform(-5, 5, (n, d))))
    ang = rng.uniform(-np.pi, np.pi, (npos, rd // 2))
    rot = np.stack([np.cos(ang), np.sin(ang)], -1).astype(np.float32)
    pos = rng.integers(0, npos, n)
    return x, rot, pos, d, rd


@pytest.mark.parametrize("inverse", [False, True])
def test_rope_is_numpys_complex_multiply(inverse):
    x, rot, pos, d, rd = _rope_case(77)
    n = x.shape[0]
    y, y64 = oracle.rope(x, rot, pos, rd, inverse, want_f64=True)
    xs = oracle.bf16_to_f64(x[:, d - rd:]).reshape(n, rd // 2, 2)
    w = rot[pos].astype(np.float64)
    w = w[..., 0] + 1j * w[..., 1]
    ref = (xs[..., 0] + 1j * xs[..., 1]) * (np.conj(w) if inverse else w)
    ref = np.stack([ref.real, ref.imag], -1).reshape(n, rd)
    scale = np.abs(oracle.bf16_to_f64(x)).max()
    assert np.abs(y64 - ref).max() <= 1e-13 * scale
    assert (y[:, d - rd:] == oracle.bf16_round(ref)).all()
    assert (y[:, : d - rd] == x[:, : d - rd]).all()        # the other dims untouched
    # the rotation keeps each pair's length, times the table entry's
    r2 = (xs ** 2).sum(-1) * np.abs(w) ** 2
    assert np.allclose((y64.reshape(n, rd // 2, 2) ** 2).sum(-1), r2, rtol=1e-12, atol=0)


def test_rope_special_angles_are_exact():
    x, rot, pos, d, rd = _rope_case(78)
    a, b = x[:, d - rd::2], x[:, d - rd + 1::2]
    neg = lambda t: t ^ np.uint16(0x8000)  # noqa: E731
    for c, s_, fwd, inv in [(1.0, 0.0, (a, b), (a, b)),            # angle 0: identity
                            (0.0, 1.0, (neg(b), a), (b, neg(a))),  # pi / 2
                            (-1.0, 0.0, (neg(a), neg(b)), (neg(a), neg(b)))]:  # pi
        r = np.zeros_like(rot)
        r[..., 0], r[..., 1] = c, s_
        for inverse, (ea, eb) in ((False, fwd), (True, inv)):
            y = oracle.rope(x, r, pos, rd, inverse)
            # (a signed zero may come out as +0 where -0 went in: compare values)
            assert np.array_equal(oracle.bf16_to_f64(y[:, d - rd::2]), oracle.bf16_to_f64(ea))
            assert np.array_equal(oracle.bf16_to_f64(y[:, d - rd + 1::2]), oracle.bf16_to_f64(eb))


def test_rope_inverse_undoes_the_rotation():
    x, rot, pos, d, rd = _rope_case(79)
    back = oracle.rope(oracle.rope(x, rot, pos, rd, False), rot, pos, rd, True)
    xv, bv = oracle.bf16_to_f64(x[:, d - rd:]), oracle.bf16_to_f64(back[:, d - rd:])
    # two bf16 roundings and the f32 table's |w| != 1: within a few bf16 steps of the pair's size
    pair = np.sqrt((xv.reshape(-1, rd // 2, 2) ** 2).sum(-1)).repeat(2, -1).reshape(xv.shape)
    assert (np.abs(bv - xv) <= 2 ** -6 * pair + 1e-30).all()


def test_rope_rejects_bad_arguments():
    x, rot, pos, d, rd = _rope_case(80, n=2)
    with pytest.raises(ValueError):
        oracle.rope(x, rot, pos, 63, True)          # odd rope_dim
    with pytest.raises(ValueError):
        oracle.rope(x, rot, [0, 50], rd, True)      # a position past the table


# --------------------------------------------------------------------------------------------
# the indexer's selection ("DeepSeek V4.1" source-layer attention page (indexer view), Indexer.forward)
# --------------------------------------------------------------------------------------------

def _golden_indexer():
    g = {}
    for line in open(os.path.join(GOLDEN, "indexer_topk_example.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, _kind, *vals = line.split()
            g[k] = [float(v) for v in vals]
    return g


def test_indexer_topk_worked_example():
    g = _golden_indexer()
    ratio, k, off = int(g["ratio"][0]), int(g["index_topk"][0]), int(g["offset"][0])
    sc = np.tile(np.array(g["scores"], np.float32), (1, 12, 1))
    got = oracle.indexer_topk(sc, 0, ratio, k, off)[0]
    for q in (0, 2, 3, 6, 7, 10, 11):
        assert got[q].tolist() == [int(v) for v in g[f"prefill_q{q}"]], q
    dec = oracle.indexer_topk(sc[:, :1], 12, ratio, k, off)[0, 0]
    assert dec.tolist() == [int(v) for v in g["decode12"]]
    ties = oracle.indexer_topk(np.ones((1, 1, 4), np.float32), 15, ratio, k, off)[0, 0]
    assert ties.tolist() == [int(v) for v in g["decode_ties"]]


def test_indexer_topk_is_torch_topk_on_distinct_scores():
    # without ties the picked set is unique: torch.topk (a library routine) on the masked scores,
    # sorted, gives the same rows
    rng = np.random.default_rng(91)
    for b, s, start, ratio, topk in ((2, 64, 0, 4, 5), (3, 1, 1023, 4, 64), (1, 33, 0, 1, 40)):
        n = (start + s) // ratio
        sc = rng.permutation(b * s * n).reshape(b, s, n).astype(np.float32) / 7.0  # distinct
        got = oracle.indexer_topk(sc, start, ratio, topk, 1000)
        t = torch.from_numpy(sc.astype(np.float64))
        vis = torch.full((s, 1), n) if start else (torch.arange(1, s + 1) // ratio)[:, None]
        t = t.masked_fill(torch.arange(n)[None, :] >= vis, float("-inf"))
        k = min(topk, n)
        for bi in range(b):
            for si in range(s):
                nv = int(vis[si, 0])
                # finite picks are unique; -inf picks (masked) all become -1
                want = sorted(torch.topk(t[bi, si], min(k, nv)).indices.tolist())
                row = [p + 1000 for p in want] + [-1] * (k - len(want))
                assert got[bi, si].tolist() == row, (b, s, bi, si)


def test_indexer_topk_brute_force_with_ties():
    # every k-subset on tiny rows with heavy ties: the picked set is the one that beats every
    # other position it leaves out (higher score, or equal score at a lower position)
    rng = np.random.default_rng(92)
    for trial in range(200):
        n = int(rng.integers(1, 8))
        k = int(rng.integers(0, 9))
        sc = rng.integers(-2, 3, size=(1, 1, n)).astype(np.float32)
        sc[sc == -2] = -np.inf
        if trial % 3 == 0:
            sc[sc == 0] = -0.0  # -0 ties with +0
        got = oracle.indexer_topk(sc, 4 * n, 4, k, 10)[0, 0]
        kk = min(k, n)
        best = None
        for S in itertools.combinations(range(n), kk):
            out = set(range(n)) - set(S)
            if all(sc[0, 0, i] > sc[0, 0, j] or (sc[0, 0, i] == sc[0, 0, j] and i < j)
                   for i in S for j in out):
                assert best is None  # the rule picks exactly one subset
                best = S
        assert got.tolist() == [p + 10 for p in best], (sc, k)


def test_indexer_topk_row_shape_invariants():
    rng = np.random.default_rng(93)
    s, ratio, topk = 200, 4, 16
    n = s // ratio
    sc = rng.standard_normal((2, s, n)).astype(np.float32)
    got = oracle.indexer_topk(sc, 0, ratio, topk, 7)
    for bi in range(2):
        for si in range(s):
            row = got[bi, si]
            valid = row[row >= 0]
            assert len(valid) == min(topk, (si + 1) // ratio)        # every visible pick kept
            assert (row[len(valid):] == -1).all()                    # -1 only at the tail
            assert (np.diff(valid) > 0).all() and (valid < 7 + (si + 1) // ratio).all()


def test_indexer_topk_bf16_scores_and_bad_arguments():
    rng = np.random.default_rng(94)
    x = rng.standard_normal((1, 1, 50)).astype(np.float32)
    bits = (x.view(np.uint32) >> 16).astype(np.uint16)               # truncated to bf16
    wid = (bits.astype(np.uint32) << 16).view(np.float32)
    assert (oracle.indexer_topk(bits, 200, 4, 9, 0) == oracle.indexer_topk(wid, 200, 4, 9, 0)).all()
    with pytest.raises(ValueError):
        oracle.indexer_topk(x, 0, 4, 9, 0)                           # 50 != (0 + 1) // 4
    with pytest.raises(NotImplementedError):
        oracle.indexer_topk(np.zeros((1, 2, 50), np.float32), 99, 2, 9, 0)  # chunked prefill


# --------------------------------------------------------------------------------------------
# select_candidate_blocks ("DeepSeek V4.1" source-layer attention page (indexer view))
# --------------------------------------------------------------------------------------------

def _golden_candidates():
    g = {}
    for line in open(os.path.join(GOLDEN, "candidate_blocks_example.txt")):
        line = line.split("#")[0].strip()
        if line:
            k, _kind, *vals = line.split()
            g[k] = [float(v) for v in vals]
    return g


def test_candidate_blocks_worked_example():
    g = _golden_candidates()
    row = np.array(g["logits"], np.float32)
    bs = int(g["block_size"][0])
    for key in ("v10_k2", "v5_k2", "v6_k1", "v0_k2", "v10_k5", "v3_k3"):
        vis, k = (int(x) for x in key[1:].split("_k"))
        got = oracle.candidate_blocks_rows(row[None], [vis], k, bs)[0]
        assert got.astype(int).tolist() == [int(v) for v in g[key]], key


def test_candidate_blocks_brute_force_with_ties():
    # every subset of blocks on tiny rows with heavy ties and -inf: the kept blocks are the one
    # subset of size min(k, blocks) that beats every block it leaves out (higher score, or equal
    # at a lower block), the newest reachable block counting as +inf, minus its -inf members
    rng = np.random.default_rng(95)
    for _ in range(300):
        width = int(rng.integers(1, 13))
        bs = int(rng.integers(1, 5))
        k = int(rng.integers(0, 6))
        vis = int(rng.integers(0, width + 1))
        row = rng.integers(-2, 3, size=width).astype(np.float32)
        row[row == -2] = -np.inf
        got = oracle.candidate_blocks_rows(row[None], [vis], k, bs)[0]
        nb = -(-width // bs)
        score = []
        for j in range(nb):
            vals = [row[t] if t < vis else -np.inf for t in range(j * bs, min((j + 1) * bs, width))]
            score.append(max(vals))
        if vis > 0:
            score[(vis - 1) // bs] = np.inf
        kk = min(k, nb)
        picks = [S for S in itertools.combinations(range(nb), kk)
                 if all(score[i] > score[j] or (score[i] == score[j] and i < j)
                        for i in S for j in set(range(nb)) - set(S))]
        assert len(picks) == 1
        kept = {j for j in picks[0] if score[j] > -np.inf}
        want = [t // bs in kept for t in range(width)]
        assert got.tolist() == want, (row, vis, k, bs)


def test_candidate_blocks_invariants_and_level_two():
    rng = np.random.default_rng(96)
    b, s, ratio, bs, kb = 2, 160, 4, 8, 3
    n = s // ratio
    x = rng.standard_normal((b, s, n)).astype(np.float32)
    m = oracle.candidate_blocks(x, 0, ratio, kb, bs)
    vis = oracle.visible_positions(s, n, 0, ratio)
    for si in range(s):
        blocks = m[:, si].reshape(b, -1, bs) if n % bs == 0 else None
        assert blocks is not None and (blocks.all(-1) | ~blocks.any(-1)).all()  # whole blocks
        nkept = blocks.any(-1).sum(-1)
        assert (nkept == min(kb, -(-int(vis[si]) // bs))).all()              # reachable blocks
        if vis[si] > 0:
            assert m[:, si, vis[si] - 1].all()                                 # newest pinned
    # level two: all-True candidates change nothing; the candidates bound every finite pick
    full = np.ones_like(m)
    assert (oracle.indexer_topk(x, 0, ratio, 16, 0, candidates=full) ==
            oracle.indexer_topk(x, 0, ratio, 16, 0)).all()
    two = oracle.indexer_topk(x, 0, ratio, 16, 0, candidates=m)
    for bi in range(b):
        for si in range(s):
            picks = two[bi, si][two[bi, si] >= 0]
            c = int(m[bi, si, :vis[si]].sum())  # visible candidate positions (finite scores)
            assert int(m[bi, si, picks].sum()) == min(16, c)


# --------------------------------------------------------------------------------------------
# hc_split_sinkhorn ("DeepSeek V4.1" attention-write page (decode))
# --------------------------------------------------------------------------------------------

def _hc_case(seed, n=64, hc=4, spread=1.0):
    rng = np.random.default_rng(seed)
    mix = (2 + hc) * hc
    m = (rng.standard_normal((n, mix)) * spread).astype(np.float32)
    sc = rng.uniform(0.5, 2.0, 3).astype(np.float32)
    base = (rng.standard_normal(mix) * 0.5).astype(np.float32)
    return m, sc, base


def test_hc_pre_post_are_library_sigmoids():
    m, sc, base = _hc_case(101)
    pre, post, _ = oracle.hc_split_sinkhorn(m, sc, base, 4, 20, 1e-6)
    a = m.astype(np.float64)
    want_pre = scipy.special.expit(a[:, :4] * np.float64(sc[0]) + base[:4]) + 1e-6
    want_post = 2.0 * scipy.special.expit(a[:, 4:8] * np.float64(sc[1]) + base[4:8])
    assert np.allclose(pre, want_pre, rtol=0, atol=1e-15)
    assert np.allclose(post, want_post, rtol=0, atol=1e-15)


def test_hc_one_round_is_softmax_then_column_normalisation():
    # iters = 1: the row softmax (scipy) plus eps, then each column over (its sum + eps)
    m, sc, base = _hc_case(102, hc=3)
    eps = 1e-3
    _, _, comb = oracle.hc_split_sinkhorn(m, sc, base, 3, 1, eps)
    logits = (m[:, 6:].astype(np.float64) * np.float64(sc[2]) + base[6:]).reshape(-1, 3, 3)
    x = scipy.special.softmax(logits, axis=-1) + eps
    want = x / (x.sum(axis=-2, keepdims=True) + eps)
    assert np.allclose(comb, want, rtol=1e-13, atol=0)
    assert not np.allclose(comb, np.swapaxes(want, -1, -2), atol=1e-3)  # rows and columns differ


def test_hc_uniform_logits_follow_the_scalar_recurrence():
    # equal logits keep every entry equal: x0 = 1/hc + eps, then x <- x / (hc x + eps) once per
    # normalisation (one column step, then a row and a column step per extra round)
    hc, iters, eps = 4, 20, 1e-2
    m = np.zeros((2, 24), np.float32)
    _, _, comb = oracle.hc_split_sinkhorn(m, np.ones(3, np.float32), np.zeros(24, np.float32),
                                          hc, iters, eps)
    x = 1.0 / hc + eps
    for _ in range(2 * iters - 1):
        x = x / (hc * x + eps)
    assert np.allclose(comb, x, rtol=1e-14, atol=0)


def test_hc_sinkhorn_limit_is_doubly_stochastic():
    m, sc, base = _hc_case(103, n=200, spread=2.0)
    _, _, comb = oracle.hc_split_sinkhorn(m, sc, base, 4, 20, 1e-6)
    cols = comb.sum(axis=-2)
    rows = comb.sum(axis=-1)
    assert np.abs(cols - 1).max() < 1e-5           # the last step normalises the columns
    assert np.abs(rows - 1).max() < 5e-3           # 20 rounds: the rows are close ...
    # ... and more rounds move them to the fixed point, where only eps keeps the sums below 1
    _, _, c40 = oracle.hc_split_sinkhorn(m, sc, base, 4, 40, 1e-6)
    _, _, c100 = oracle.hc_split_sinkhorn(m, sc, base, 4, 100, 1e-6)
    assert np.abs(c40.sum(-1) - 1).max() < np.abs(rows - 1).max()
    assert np.abs(c100.sum(-1) - 1).max() < 2e-6 and np.abs(c100.sum(-2) - 1).max() < 2e-6


def test_hc_comb_is_permutation_equivariant():
    # permuting the logits' rows by P and columns by Q permutes comb the same way
    m, sc, base = _hc_case(104, n=16)
    rng = np.random.default_rng(5)
    P, Q = rng.permutation(4), rng.permutation(4)
    sc[2], base[8:] = 1.0, 0.0  # a shared affine map keeps the permutation exact
    logit = m[:, 8:].reshape(-1, 4, 4)
    m2 = m.copy()
    m2[:, 8:] = logit[:, P][:, :, Q].reshape(-1, 16)
    _, _, c1 = oracle.hc_split_sinkhorn(m, sc, base)
    _, _, c2 = oracle.hc_split_sinkhorn(m2, sc, base)
    assert np.allclose(c2, c1[:, P][:, :, Q], rtol=1e-12, atol=0)
