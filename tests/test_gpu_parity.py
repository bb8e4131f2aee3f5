"""GPU parity: the CUDA path (called through the C ABI) against the CPU oracle on the same
seeded inputs.  Indices and act_quant bit-exact; sparse_attn outputs within
|gpu - oracle| <= 1e-2 + 1e-2 * |oracle| per element."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_latent_attention_gb300 as sa
from sparse_latent_attention_gb300 import build, workloads
from tests import _gpu
from tests._helpers import assert_close_bf16, compose_idx_oracle, quantised_kv_oracle

pytestmark = pytest.mark.gpu

ATOL = RTOL = 1e-2


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    sa.load()
    return torch.device("cuda:0")


def _sample_tokens(wl, n, seed=0, runs=False):
    """n sampled query tokens (all of them when n >= the workload's); with runs, also three whole
    runs of 64 consecutive tokens -- at the start, the middle and the end -- so that every
    position of a CTA's token sequence (and the row reuse between consecutive tokens) is met."""
    nt = wl.n_tokens
    if nt <= n:
        return np.arange(nt)
    rng = np.random.default_rng(seed)
    fixed = np.array([0, 1, 2, 63, 64, 127, 128, 129, nt // 2, nt - 2, nt - 1])
    fixed = fixed[fixed < nt]
    rest = rng.choice(nt, size=n - len(fixed), replace=False)
    parts = [fixed, rest]
    if runs:
        mid = nt // 2 - 32
        parts += [np.arange(0, 64), np.arange(mid, mid + 64), np.arange(nt - 64, nt)]
    return np.unique(np.concatenate(parts))


def _oracle_on_tokens(wl, tokens, quantise):
    tokens = np.asarray(tokens)
    bsel = sorted(set((tokens // wl.s).tolist()))
    kv_o, sc_o, idx = _gpu.oracle_inputs(wl, quantise, bsel)
    q = wl.q[bsel]
    idx_sel = idx[bsel]
    pos = {b: i for i, b in enumerate(bsel)}
    local = np.array([pos[t // wl.s] * wl.s + t % wl.s for t in tokens])
    return oracle.sparse_attn(q, kv_o, wl.sink, idx_sel, wl.scale, kv_scales=sc_o,
                              tokens=local), idx


def _gpu_run(wl, dev, quantise):
    x = _gpu.prepare(wl, dev, quantise)
    ws = sa.new_workspace(wl.b, wl.s, wl.h, wl.d, wl.rows, wl.topk,
                          sa.SA_KV_FP8_E4M3 if x["kv_scale"] is not None else sa.SA_KV_BF16,
                          device=dev)
    o = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, kv_scale=x["kv_scale"],
                       workspace=ws)
    torch.cuda.synchronize()
    return o, x, ws


# --------------------------------------------------------------------------------------------
# helpers on the path: bit-exact
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("start_pos,seqlen,window,nbatch,ld", [
    (0, 12, 8, 1, 8), (0, 4096, 128, 1, 128), (0, 300, 128, 2, 640), (0, 3, 8, 1, 8),
    (12, 1, 8, 1, 8), (13, 1, 8, 3, 20), (5, 1, 8, 1, 8), (32768, 1, 128, 64, 1152),
    (131072, 1, 128, 4, 2176), (1, 1, 1, 1, 1)])
def test_window_idxs_bit_exact(dev, start_pos, seqlen, window, nbatch, ld):
    out = torch.full((nbatch, seqlen, ld), -7, dtype=torch.int32, device=dev)
    sa.window_idxs(start_pos, seqlen, window, out=out[:, :, :window], nbatch=nbatch)
    got = out.cpu().numpy()
    want = oracle.window_idxs(start_pos, seqlen, window)
    for bi in range(nbatch):
        assert (got[bi, :, :window] == want).all()
        assert (got[bi, :, window:] == -7).all()  # nothing written past the window columns


def _act_quant_inputs():
    rng = np.random.default_rng(17)
    x = rng.standard_normal((512, 512)).astype(np.float32)
    # blocks spanning the whole bf16 range, exact zeros, tiny values near the 1e-4 floor,
    # values on e4m3 rounding midpoints, negative zeros
    x *= np.exp(rng.uniform(-80, 80, (512, 16))).repeat(32, axis=1).astype(np.float32)
    x[0] = 0.0
    x[1] = -0.0
    x[2, :32] = 1e-4
    x[3, :32] = 448.0 * np.array([1, 3.125 / 448, 1.0625 / 448, 17 / 448] * 8)
    x[4] = rng.uniform(-1e-6, 1e-6, 512)
    x[5, :] = 450.0
    return workloads.to_bf16_bits(x)


def test_act_quant_bit_exact(dev):
    bits = _act_quant_inputs()
    want_rt, want_codes, want_sc = oracle.act_quant(bits)
    x = _gpu.u16_to_bf16_tensor(bits, dev)
    rt = torch.empty_like(x)
    codes = torch.empty(x.shape, dtype=torch.uint8, device=dev)
    sc = torch.empty((x.shape[0], x.shape[1] // 32), dtype=torch.uint8, device=dev)
    sa.act_quant_fp8(x, out_rt=rt, codes=codes, scales=sc)
    assert (_gpu.bf16_tensor_to_u16(rt) == want_rt).all()
    assert (codes.cpu().numpy() == want_codes).all()
    assert (sc.cpu().numpy() == want_sc).all()
    # in place, and rows strided inside a larger buffer (one ring slot per sequence)
    y = x.clone()
    sa.act_quant_fp8(y, out_rt=y)
    assert (_gpu.bf16_tensor_to_u16(y) == want_rt).all()
    cache = torch.zeros((512, 3, 512), dtype=torch.uint8, device=dev)
    cscale = torch.zeros((512, 3, 16), dtype=torch.uint8, device=dev)
    sa.act_quant_fp8(x, codes=cache[:, 1, :], scales=cscale[:, 1, :])
    assert (cache[:, 1].cpu().numpy() == want_codes).all()
    assert (cache[:, 0].cpu().numpy() == 0).all() and (cache[:, 2].cpu().numpy() == 0).all()
    assert (cscale[:, 1].cpu().numpy() == want_sc).all()


def test_act_quant_both_kernel_shapes(dev):
    """Rows whose strides allow 16-byte accesses take the eight-per-thread kernel; others (an odd
    row stride, a misaligned start) the one-element-per-lane kernel: both bit-exact."""
    bits = _act_quant_inputs()[:96, :256]
    want_rt, want_codes, want_sc = oracle.act_quant(bits)
    for stride, offset in ((256, 0), (264, 8), (259, 0), (256, 1)):
        buf = torch.zeros(96 * stride + offset + 8, dtype=torch.bfloat16, device=dev)
        x = buf[offset:offset + 96 * stride].view(96, stride)[:, :256]
        x.copy_(_gpu.u16_to_bf16_tensor(bits, dev))
        rt = torch.empty((96, 256), dtype=torch.bfloat16, device=dev)
        codes = torch.empty((96, 256), dtype=torch.uint8, device=dev)
        sc = torch.empty((96, 8), dtype=torch.uint8, device=dev)
        sa.act_quant_fp8(x, out_rt=rt, codes=codes, scales=sc)
        assert (_gpu.bf16_tensor_to_u16(rt) == want_rt).all(), (stride, offset)
        assert (codes.cpu().numpy() == want_codes).all(), (stride, offset)
        assert (sc.cpu().numpy() == want_sc).all(), (stride, offset)
        sa.act_quant_fp8(x, out_rt=x)  # in place, strided
        assert (_gpu.bf16_tensor_to_u16(x.contiguous()) == want_rt).all(), (stride, offset)


def test_act_quant_every_bf16_value(dev):
    """Each of the 65536 bf16 patterns (NaN and inf excluded) inside a block with a fixed
    amax, so every e4m3 rounding case and both signs are met."""
    allv = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f = (allv.astype(np.uint32) << 16).view(np.float32)
    ok = np.isfinite(f)
    vals = allv[ok]
    for amax in (448.0, 1.0, 3e-3, 1e30):
        fv = (vals.astype(np.uint32) << 16).view(np.float32)
        keep = vals[np.abs(fv) <= amax]
        n = (len(keep) + 30) // 31 * 31
        blk = np.zeros(n, np.uint16)
        blk[: len(keep)] = keep
        blk = blk.reshape(-1, 31)
        amax_bits = workloads.to_bf16_bits(np.float32([amax]))[0]
        rows = np.concatenate([blk, np.full((blk.shape[0], 1), amax_bits, np.uint16)], axis=1)
        rows = rows.reshape(-1, 64) if rows.shape[0] % 2 == 0 else np.concatenate(
            [rows, np.zeros((1, 32), np.uint16)]).reshape(-1, 64)
        want_rt, want_codes, want_sc = oracle.act_quant(rows)
        x = _gpu.u16_to_bf16_tensor(rows, dev)
        codes = torch.empty(x.shape, dtype=torch.uint8, device=dev)
        rt = torch.empty_like(x)
        sc = torch.empty((x.shape[0], 2), dtype=torch.uint8, device=dev)
        sa.act_quant_fp8(x, out_rt=rt, codes=codes, scales=sc)
        assert (codes.cpu().numpy() == want_codes).all(), amax
        assert (_gpu.bf16_tensor_to_u16(rt) == want_rt).all(), amax
        assert (sc.cpu().numpy() == want_sc).all(), amax


@pytest.mark.parametrize("nb,seqlen,start_pos,window,rows", [
    (1, 12, 0, 8, 8),          # the ring-cache paragraph's prefill: 12 tokens into 8 slots
    (2, 12, 0, 8, 20),         # the same for two sequences, the ring the first 8 rows of a cache
    (2, 5, 0, 8, 8),           # fewer tokens than slots
    (3, 1, 13, 8, 30),         # decode at position 13 (slot 5)
    (3, 1, 32768, 128, 300),   # decode at position 32768 (slot 0) into a 128-slot ring
    (1, 300, 0, 128, 128)])    # a long prefill: only the last 128 tokens stay
def test_window_write_bit_exact(dev, nb, seqlen, start_pos, window, rows):
    d = 512
    rng = np.random.default_rng(900 + nb * 31 + seqlen)
    x = rng.standard_normal((nb, seqlen, d)).astype(np.float32)
    x *= np.exp(rng.uniform(-20, 20, (nb, seqlen, d // 32))).repeat(32, axis=2).astype(np.float32)
    bits = workloads.to_bf16_bits(x)
    rt, codes, sc = oracle.act_quant(bits.reshape(-1, d))
    rt, codes, sc = (a.reshape(nb, seqlen, -1) for a in (rt, codes, sc))
    # expected caches: a sentinel everywhere, the ring rows placed by the oracle's ring write
    want_rt = np.full((nb, rows, d), 0x3F80, np.uint16)
    want_c = np.full((nb, rows, d), 0xAB, np.uint8)
    want_s = np.full((nb, rows, d // 32), 0x55, np.uint8)
    for bi in range(nb):
        ring = np.ascontiguousarray(want_rt[bi, :window])
        oracle.ring_write(ring, rt[bi], start_pos)
        want_rt[bi, :window] = ring
        for t in range(seqlen):  # the codes and scales follow the same slot rule
            want_c[bi, (start_pos + t) % window] = codes[bi, t]
            want_s[bi, (start_pos + t) % window] = sc[bi, t]
    cache_rt = torch.full((nb, rows, d), 1.0, dtype=torch.bfloat16, device=dev)
    cache_c = torch.full((nb, rows, d), 0xAB, dtype=torch.uint8, device=dev)
    cache_s = torch.full((nb, rows, d // 32), 0x55, dtype=torch.uint8, device=dev)
    sa.window_write(_gpu.u16_to_bf16_tensor(bits, dev), start_pos, ring_rt=cache_rt[:, :window],
                    codes=cache_c[:, :window], scales=cache_s[:, :window])
    torch.cuda.synchronize()
    assert (_gpu.bf16_tensor_to_u16(cache_rt) == want_rt).all()
    assert (cache_c.cpu().numpy() == want_c).all()
    assert (cache_s.cpu().numpy() == want_s).all()


# --------------------------------------------------------------------------------------------
# sparse_attn on the five named workloads (full size, sampled outputs)
# --------------------------------------------------------------------------------------------

@pytest.mark.parametrize("name,n_sample", [("tiny", 16), ("swa_prefill", 64), ("cmp_prefill", 48),
                                           ("decode", 64), ("fp8_decode", 256)])
def test_named_workload_parity(dev, name, n_sample):
    wl = workloads.make_named(name)
    quantise = name != "tiny"
    o, x, ws = _gpu_run(wl, dev, quantise)
    assert sa.read_status(ws) == 0
    # the whole index table matches the oracle's composition bit for bit
    idx_want = compose_idx_oracle(wl)
    assert (x["idx"].cpu().numpy() == idx_want).all()
    tokens = _sample_tokens(wl, n_sample, runs=wl.s > 1)
    want, _ = _oracle_on_tokens(wl, tokens, quantise)
    got = _gpu.bf16_tensor_to_u16(o.view(wl.n_tokens, wl.h, wl.d)[torch.from_numpy(tokens).to(dev)])
    assert_close_bf16(got, want, ATOL, RTOL, what=name)
    # properties over every output: finite, and zero exactly where a token lists no row
    of = o.float()
    assert torch.isfinite(of).all()
    empty = (x["idx"] < 0).all(dim=-1)
    if empty.any():
        assert (of[empty] == 0).all()


def test_bf16_round_trip_kv_matches_oracle(dev):
    """The kv the attention reads for a named workload is the oracle's act_quant round trip."""
    wl = workloads.make_named("swa_prefill")
    kv = _gpu.device_kv_raw(wl, dev)
    sa.act_quant_fp8(kv.view(-1, wl.d), out_rt=kv.view(-1, wl.d))
    rt, _, _ = oracle.act_quant(wl.kv_raw_dense())
    assert (_gpu.bf16_tensor_to_u16(kv) == rt).all()


# --------------------------------------------------------------------------------------------
# sparse_attn on small problems: every output compared
# --------------------------------------------------------------------------------------------

RANDOM_CASES = [
    # b, s, h, d, rows, topk, extra
    (2, 37, 64, 512, 300, 200, {}),                 # ragged tail over 4 tiles
    (1, 9, 128, 512, 700, 650, {}),                 # two head blocks, 11 tiles
    (3, 1, 64, 512, 5000, 1152, {}),                # decode: split idx columns + merge
    (5, 1, 128, 512, 3000, 2176, {}),               # decode, 128 heads
    (1, 20, 4, 64, 48, 16, {}),                     # tiny head count and head_dim
    (2, 11, 100, 192, 90, 70, {}),                  # ragged heads, odd head_dim
    (1, 13, 64, 256, 64, 64, dict(distinct=False)),  # repeated indices count repeatedly
    (2, 7, 64, 512, 400, 130, dict(q_scale=12.0)),  # large logits: running max moves a lot
    (1, 8, 64, 512, 100, 100, dict(sink_scale=30.0)),  # sinks far from the logits
    (2, 9, 16, 128, 50, 40, dict(neg_frac=0.97)),   # nearly everything masked
    # head_dim 512 (tcgen05 path) with partial head blocks: o's TMA store boxes clipped at h
    (2, 9, 100, 512, 300, 200, {}),                 # 64 + 36 heads, two tiles
    (1, 12, 8, 512, 200, 130, {}),                  # fewer heads than one 32-row store box
    (3, 1, 40, 512, 2000, 600, {}),                 # decode split with a partial head block
    # repeated indices in the tcgen05 family: ring placement falls back to column order, and a
    # row kept from the previous pair may be listed twice
    (1, 13, 64, 512, 64, 64, dict(distinct=False)),
    (2, 30, 64, 512, 90, 200, dict(distinct=False)),
    (3, 1, 64, 512, 300, 1152, dict(distinct=False)),  # cut decode ranges, many repeats
    # cut ranges: few tokens, many pairs, pieces merged in the kernel (ragged last pair)
    (1, 1, 64, 512, 9000, 4100, {}),
    (7, 1, 128, 512, 3000, 2176, {}),
    (2, 2, 64, 512, 5000, 1900, {}),
]


@pytest.mark.parametrize("case", RANDOM_CASES, ids=lambda c: f"b{c[0]}s{c[1]}h{c[2]}d{c[3]}k{c[5]}")
def test_random_parity(dev, case):
    b, s, h, d, rows, topk, extra = case
    empty = (1,) if b * s > 1 else ()
    wl = workloads.make_random(b, s, h, d, rows, topk, seed=1000 + b * 7 + s,
                               all_neg_tokens=empty, **extra)
    o, x, ws = _gpu_run(wl, dev, quantise=False)
    assert sa.read_status(ws) == 0
    want = oracle.sparse_attn(wl.q, wl.kv_raw_dense(), wl.sink, compose_idx_oracle(wl), wl.scale)
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, ATOL, RTOL, what=str(case))
    if empty:
        assert (_gpu.bf16_tensor_to_u16(o.view(-1, h, d)[1]) == 0).all()


ROPE_CASES = [
    # b, s, h, rows, topk, rope_dim, start_pos, quantise
    (2, 37, 64, 300, 200, 64, 0, False),        # prefill, the layer's 64 rope dims
    (3, 1, 64, 5000, 1152, 64, 4000, False),    # decode: split partials rotated, then merged
    (2, 9, 100, 300, 200, 64, 5, False),        # a partial head block
    (2, 9, 64, 300, 200, 64, 11, True),         # fp8 kv
    (1, 12, 64, 200, 130, 512, 3, False),       # the whole head rotated
    (1, 12, 64, 200, 130, 2, 3, False),         # one pair: the last two dims only
    (2, 5, 64, 300, 0, 64, 2, False),           # no idx columns: o = 0 stays 0
]


@pytest.mark.parametrize("case", ROPE_CASES,
                         ids=lambda c: f"b{c[0]}s{c[1]}h{c[2]}k{c[4]}r{c[5]}p{c[6]}{'q' if c[7] else ''}")
def test_inverse_rope_fused(dev, case):
    # sparse_attn followed by apply_rotary_emb(o[..., -rope_dim:], inverse) at the positions
    # start_pos + si ("DeepSeek V4.1" attention page, Attention.forward): the oracle takes the two
    # steps as the page writes them (o rounded to bf16, then rotated and rounded again); the kernel
    # rotates its f32 result before its one rounding, within the tolerance of the two-step form.
    b, s, h, rows, topk, rd, start_pos, quantise = case
    d = 512
    wl = workloads.make_random(b, s, h, d, rows, topk, seed=3000 + rd + start_pos,
                               all_neg_tokens=(1,) if b * s > 1 else (),
                               kv_format="fp8" if quantise else "bf16")
    rot = workloads.rope_table(start_pos + s + 3, rd, seed=rd + start_pos)
    x = _gpu.prepare(wl, dev, quantise)
    fmt = sa.SA_KV_FP8_E4M3 if x["kv_scale"] is not None else sa.SA_KV_BF16
    ws = sa.new_workspace(b, s, h, d, wl.rows, wl.topk, fmt, device=dev)
    plain = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, kv_scale=x["kv_scale"],
                           workspace=ws)
    o = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, kv_scale=x["kv_scale"],
                       workspace=ws, rope=(torch.from_numpy(rot).to(dev), start_pos))
    torch.cuda.synchronize()
    assert sa.read_status(ws) == 0
    # the dims outside the rope slice are the plain call's, bit for bit
    assert torch.equal(o[..., :d - rd].view(torch.int16), plain[..., :d - rd].view(torch.int16))
    kv_o = quantised_kv_oracle(wl, quantise)[0]  # fp8 rows decode to the round trip's values
    o_or = oracle.sparse_attn(wl.q, kv_o, wl.sink, compose_idx_oracle(wl), wl.scale)
    o_or = o_or.reshape(b * s * h, d)
    pos = np.repeat(np.tile(start_pos + np.arange(s), b), h)
    want = oracle.rope(o_or, rot, pos, rd, True).reshape(b, s, h, d)
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, ATOL, RTOL, what=str(case))


GUARD_CASES = [
    # b, s, h, rows, topk, kv fp8, rope dims, start_pos
    (2, 9, 100, 300, 200, False, 0, 0),        # 64 + 36 heads: clipped store boxes
    (1, 12, 8, 200, 130, False, 0, 0),         # fewer heads than one store box
    (3, 1, 40, 2000, 600, False, 0, 0),        # decode pieces merged into a partial head block
    (5, 1, 64, 3000, 1152, False, 0, 0),       # decode pieces, full head block
    (2, 9, 64, 300, 200, False, 64, 5),        # fused rotation
    (3, 1, 64, 3000, 1152, False, 64, 4000),   # fused rotation on merged pieces
    (2, 9, 40, 300, 200, True, 0, 0),          # fp8 kv, partial head block
    (4, 1, 128, 3000, 2176, True, 0, 0),       # fp8 kv, two head blocks, pieces
]


@pytest.mark.parametrize("case", GUARD_CASES, ids=lambda c: f"b{c[0]}s{c[1]}h{c[2]}k{c[4]}"
                         f"{'f8' if c[5] else ''}{'r' if c[6] else ''}")
def test_o_guard_zones(dev, case):
    """o inside a larger buffer filled with a sentinel: nothing outside o is written (clipped TMA
    store boxes, merged pieces, the rotation), and o matches the oracle."""
    b, s, h, rows, topk, fp8, rd, start_pos = case
    d = 512
    wl = workloads.make_random(b, s, h, d, rows, topk, seed=6100 + h + topk,
                               all_neg_tokens=(1,) if b * s > 1 else (),
                               kv_format="fp8" if fp8 else "bf16")
    x = _gpu.prepare(wl, dev, quantise=fp8)
    n = b * s * h * d
    pad = 64 * 1024  # elements on each side (a multiple of 8: o stays 16-byte aligned)
    sentinel = torch.tensor(-12345.0, dtype=torch.bfloat16)
    buf = torch.full((pad + n + pad,), float(sentinel), dtype=torch.bfloat16, device=dev)
    o = buf[pad:pad + n].view(b, s, h, d)
    rope = None
    if rd:
        rot = workloads.rope_table(start_pos + s + 1, rd, seed=rd + start_pos)
        rope = (torch.from_numpy(rot).to(dev), start_pos)
    ws = sa.new_workspace(b, s, h, d, wl.rows, wl.topk,
                          sa.SA_KV_FP8_E4M3 if fp8 else sa.SA_KV_BF16, device=dev)
    sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, kv_scale=x["kv_scale"],
                   out=o, workspace=ws, rope=rope)
    torch.cuda.synchronize()
    assert sa.read_status(ws) == 0
    sent = sentinel.view(torch.int16).item()
    assert (buf[:pad].view(torch.int16) == sent).all(), "written before o"
    assert (buf[pad + n:].view(torch.int16) == sent).all(), "written after o"
    kv_o = quantised_kv_oracle(wl, fp8)[0]
    want = oracle.sparse_attn(wl.q, kv_o, wl.sink, compose_idx_oracle(wl), wl.scale)
    if rd:
        want = oracle.rope(want.reshape(b * s * h, d), rot,
                           np.repeat(np.tile(start_pos + np.arange(s), b), h), rd,
                           True).reshape(b, s, h, d)
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, ATOL, RTOL, what=f"guard {case}")


def test_running_max_raised_every_tile(dev):
    # The logits grow by ~7 nats (> 2^8 in log2 units) from one block of 64 rows to the next, so
    # a token that lists the rows in order raises its running maximum (and rescales O) on every
    # row tile; the reversed order never does, and a shuffled order with holes does sometimes.
    rng = np.random.default_rng(2024)
    b, s, h, d, rows = 1, 3, 64, 512, 704
    scale = d ** -0.5
    q0 = rng.standard_normal(d)
    q = q0[None, None, None, :] + 0.1 * rng.standard_normal((b, s, h, d))
    kv = 0.5 * rng.standard_normal((b, rows, d))
    kv += (np.arange(rows) // 64)[None, :, None] * 7.0 * (q0 / np.linalg.norm(q0))[None, None, :]
    q_bits, kv_bits = oracle.bf16_round(q), oracle.bf16_round(kv)
    sink = rng.standard_normal(h).astype(np.float32)
    idx = np.empty((b, s, rows), dtype=np.int32)
    idx[0, 0] = np.arange(rows)
    idx[0, 1] = np.arange(rows)[::-1]
    perm = rng.permutation(rows).astype(np.int32)
    perm[rng.random(rows) < 0.2] = -1
    idx[0, 2] = perm
    ws = sa.new_workspace(b, s, h, d, rows, rows, device=dev)
    o = sa.sparse_attn(_gpu.u16_to_bf16_tensor(q_bits, dev), _gpu.u16_to_bf16_tensor(kv_bits, dev),
                       torch.from_numpy(sink).to(dev), torch.from_numpy(idx).to(dev), scale,
                       workspace=ws)
    torch.cuda.synchronize()
    assert sa.read_status(ws) == 0
    want = oracle.sparse_attn(q_bits, kv_bits, sink, idx, scale)
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, ATOL, RTOL, what="growing logits")


def test_query_parts_match_the_whole_call(dev):
    # Attending the query tokens in parts (as the benchmark's end-to-end step does, each part its
    # own call on the same kv) gives the whole call's output: bit for bit for a part of many
    # tokens (each CTA takes whole tokens), and within the tolerance for a part of few tokens,
    # whose idx columns the kernel may cut between SMs and merge (a different f32 summation
    # order).  The same call twice gives the same bits: the merge order is fixed.
    wl = workloads.make_random(1, 2600, 64, 512, 2800, 200, seed=4242, window=128)
    x = _gpu.prepare(wl, dev, quantise=False)
    ws = sa.new_workspace(1, 2600, 64, 512, 2800, 200, device=dev)
    whole = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, workspace=ws)
    parts = torch.empty_like(whole)
    bounds = ((0, 1300), (1300, 2600), (0, 256), (256, 512), (512, 1000), (1000, 1300))
    for i, (a, b) in enumerate(bounds):
        wp = sa.new_workspace(1, b - a, 64, 512, 2800, 200, device=dev)
        sa.sparse_attn(x["q"][:, a:b], x["kv"], x["sink"], x["idx"][:, a:b], wl.scale,
                       out=parts[:, a:b], workspace=wp)
        assert sa.read_status(wp) == 0
        torch.cuda.synchronize()
        if i == 1:  # two parts of 1300 tokens, each whole tokens per CTA
            assert torch.equal(whole.view(torch.int16), parts.view(torch.int16))
    assert sa.read_status(ws) == 0
    assert_close_bf16(_gpu.bf16_tensor_to_u16(parts), _gpu.bf16_tensor_to_u16(whole), ATOL, RTOL,
                      what="parts")
    want = oracle.sparse_attn(wl.q, wl.kv_raw_dense(), wl.sink, compose_idx_oracle(wl), wl.scale,
                              tokens=np.arange(0, 1300, 7))
    assert_close_bf16(_gpu.bf16_tensor_to_u16(parts[0, 0:1300:7]), want, ATOL, RTOL, what="parts")
    for a, b in bounds[2:]:  # the few-token parts again: the same bits
        again = sa.sparse_attn(x["q"][:, a:b], x["kv"], x["sink"], x["idx"][:, a:b], wl.scale)
        assert torch.equal(again.view(torch.int16), parts[:, a:b].view(torch.int16))


def test_sink_minus_inf_and_single_row(dev):
    wl = workloads.make_random(2, 5, 64, 512, 40, 24, seed=77, neg_frac=0.0)
    wl.sink[:] = -np.inf
    wl.idx_tail[:] = -1
    wl.idx_tail[..., 5] = 3
    o, x, ws = _gpu_run(wl, dev, quantise=False)
    kvd = wl.kv_raw_dense()
    got = _gpu.bf16_tensor_to_u16(o)
    for bi in range(2):
        assert (got[bi] == kvd[bi, 3][None, None, :]).all()  # one row, no sink: that row exactly


def test_empty_shapes(dev):
    # topk == 0 and rows == 0: nothing listed, o == 0
    for rows, topk in ((10, 0), (0, 7)):
        wl = workloads.make_random(1, 4, 64, 512, max(rows, 1), topk, seed=5, neg_frac=1.0)
        q = _gpu.u16_to_bf16_tensor(wl.q, dev)
        kv = torch.zeros((1, rows, 512), dtype=torch.bfloat16, device=dev)
        idx = torch.full((1, 4, topk), -1, dtype=torch.int32, device=dev)
        sink = torch.from_numpy(wl.sink).to(dev)
        o = torch.full_like(q, 3.0)
        sa.sparse_attn(q, kv, sink, idx, wl.scale, out=o)
        assert (o.view(torch.int16) == 0).all()  # +0 bit patterns, whatever TMEM held before
    # no tokens at all: a no-op
    q = torch.empty((0, 4, 64, 512), dtype=torch.bfloat16, device=dev)
    o = sa.sparse_attn(q, torch.zeros((0, 5, 512), dtype=torch.bfloat16, device=dev),
                       torch.zeros(64, device=dev), torch.zeros((0, 4, 3), dtype=torch.int32,
                                                                device=dev), 0.1)
    assert o.shape == q.shape


def test_out_of_range_index_is_flagged_and_ignored(dev):
    wl = workloads.make_random(2, 6, 64, 512, 90, 70, seed=91)
    x = _gpu.prepare(wl, dev, quantise=False)
    idx_bad = x["idx"].clone()
    idx_bad[0, 2, 5] = 90       # == rows
    idx_bad[1, 4, 0] = -3
    idx_bad[1, 5, 69] = 1 << 30
    ws = sa.new_workspace(wl.b, wl.s, wl.h, wl.d, wl.rows, wl.topk, device=dev)
    o = sa.sparse_attn(x["q"], x["kv"], x["sink"], idx_bad, wl.scale, workspace=ws)
    assert sa.read_status(ws, clear=True) == sa._lib.SA_ERR_INDEX
    assert sa.read_status(ws) == 0
    idx_ok = idx_bad.clone()
    idx_ok[(idx_ok < -1) | (idx_ok >= wl.rows)] = -1
    want = oracle.sparse_attn(wl.q, wl.kv_raw_dense(), wl.sink, idx_ok.cpu().numpy(), wl.scale)
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, ATOL, RTOL, what="bad idx")


@pytest.mark.parametrize("family", ["tcgen05", "mma"])
@pytest.mark.parametrize("b,s,h,topk,window", [(2, 9, 64, 300, 0), (4, 1, 128, 2176, 0),
                                               (3, 1, 64, 1152, 0), (1, 140, 64, 128, 128),
                                               (2, 70, 64, 200, 128), (2, 5, 40, 300, 0)])
def test_fp8_storage_bit_identical_to_round_trip(dev, b, s, h, topk, window, family):
    """Attention over e4m3 codes + e8m0 scales gives the same bits as attention over the bf16
    round trip of the same rows (same kernel family, tiling and order)."""
    wl = workloads.make_random(b, s, h, 512, 2500, topk, seed=300 + topk, kv_format="fp8",
                               window=window)
    raw = _gpu.device_kv_raw(wl, dev)
    codes = torch.empty((b, wl.rows, 512), dtype=torch.uint8, device=dev)
    scales = torch.empty((b, wl.rows, 16), dtype=torch.uint8, device=dev)
    sa.act_quant_fp8(raw.view(-1, 512), codes=codes.view(-1, 512), scales=scales.view(-1, 16))
    rt = raw.clone()
    sa.act_quant_fp8(rt.view(-1, 512), out_rt=rt.view(-1, 512))
    q = _gpu.u16_to_bf16_tensor(wl.q, dev)
    sink = torch.from_numpy(wl.sink).to(dev)
    idx = _gpu.device_idx(wl, dev)
    o_fp8 = sa.sparse_attn(q, codes, sink, idx, wl.scale, kv_scale=scales, family=family)
    o_bf16 = sa.sparse_attn(q, rt, sink, idx, wl.scale, family=family)
    assert torch.equal(o_fp8.view(torch.int16), o_bf16.view(torch.int16))


@pytest.mark.parametrize("case", [(2, 37, 64, 300, 200), (3, 1, 64, 5000, 1152),
                                  (1, 9, 128, 700, 650), (2, 7, 64, 400, 130)],
                         ids=lambda c: f"b{c[0]}s{c[1]}h{c[2]}k{c[4]}")
def test_kernel_families_agree(dev, case):
    """The tcgen05 kernel (head_dim 512, bf16 kv) and the mma.sync kernel on the same inputs."""
    b, s, h, rows, topk = case
    wl = workloads.make_random(b, s, h, 512, rows, topk, seed=500 + topk, all_neg_tokens=(0,),
                               q_scale=4.0)
    x = _gpu.prepare(wl, dev, quantise=False)
    o_tc = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, family="tcgen05")
    o_mma = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, family="mma")
    torch.cuda.synchronize()
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o_tc), _gpu.bf16_tensor_to_u16(o_mma), ATOL, RTOL,
                      what="tc vs mma")


@pytest.mark.parametrize("b,s,start_pos,rows,topk", [
    (400, 1, 300, 300, 200),   # decode: every sequence's ring is rows 0..127, ~3 tasks per CTA
    (3, 300, 0, 300, 128),     # sliding-window prefill of 3 sequences back to back
    (2, 150, 0, 400, 200),     # window + random columns
])
def test_resident_rows_not_reused_across_sequences(dev, b, s, start_pos, rows, topk):
    """Consecutive tasks on one CTA share row numbers but not data when they belong to
    different sequences; rows kept in shared memory between tiles must match both."""
    wl = workloads.make_random(b, s, 64, 512, rows, topk, seed=700 + b, window=128,
                               start_pos=start_pos, neg_frac=0.05)
    o, x, ws = _gpu_run(wl, dev, quantise=False)
    assert sa.read_status(ws) == 0
    want = oracle.sparse_attn(wl.q, wl.kv_raw_dense(), wl.sink, compose_idx_oracle(wl), wl.scale)
    assert_close_bf16(_gpu.bf16_tensor_to_u16(o), want, ATOL, RTOL, what="reuse")
    # the same call again, several times: the producers' placement records are shared between
    # threads that run at their own pace, and a race there shows up only on some runs
    for rep in range(4):
        o2 = sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, workspace=ws)
        torch.cuda.synchronize()
        assert sa.read_status(ws) == 0
        assert_close_bf16(_gpu.bf16_tensor_to_u16(o2), want, ATOL, RTOL, what=f"reuse, run {rep + 2}")


def test_decode_step_replays_from_a_cuda_graph(dev):
    """A decode step -- the window table, the ring write of the step's new rows, and sparse_attn with
    its split merge (programmatic dependent launches) -- captured once into a CUDA graph and
    replayed: the same bits as the eager calls, replay after replay, with new inputs copied into
    the captured buffers between replays."""
    b, d, window, rows, topk, pos = 6, 512, 128, 3000, 1152, 4321
    wl = workloads.make_random(b, 1, 64, d, rows, topk, seed=8080, window=window, start_pos=pos)
    x = _gpu.prepare(wl, dev, quantise=True)
    new_rows = torch.randn((b, 1, d), device=dev).to(torch.bfloat16)
    ws = sa.new_workspace(b, 1, 64, d, rows, topk, device=dev)
    out = torch.empty_like(x["q"])
    stream = torch.cuda.Stream(device=dev)

    def step():
        sa.window_idxs(pos, 1, window, out=x["idx"][:, :, :window], nbatch=b)
        sa.window_write(new_rows, pos, ring_rt=x["kv"][:, :window])
        sa.sparse_attn(x["q"], x["kv"], x["sink"], x["idx"], wl.scale, out=out, workspace=ws)

    with torch.cuda.stream(stream):
        step()  # eager, also configures the kernels before the capture
    torch.cuda.synchronize()
    eager = out.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for rep in range(3):
        out.fill_(0)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), eager.view(torch.int16)), f"replay {rep}"
    # new queries copied into the captured buffer: the replay follows them
    x["q"].copy_(torch.randn_like(x["q"], dtype=torch.float32).to(torch.bfloat16))
    with torch.cuda.stream(stream):
        step()
    torch.cuda.synchronize()
    eager2 = out.clone()
    out.fill_(0)
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager2.view(torch.int16))
    assert not torch.equal(eager2.view(torch.int16), eager.view(torch.int16))
    assert sa.read_status(ws) == 0
