"""Seeded synthetic inputs for sparse_attn.

This module only draws random numbers and lays them out; it holds none of the method's
arithmetic (no window-index rule, no quantisation, no attention).  Both the CUDA path and the
CPU oracle read the same arrays from here.

Every workload is drawn from ``numpy.random.default_rng(seed)`` (PCG64) in a fixed order:
q, sink, the random index columns, then the kv rows.  Normal draws are f32 N(0, 1) rounded to
bf16 by torch's round-to-nearest-even conversion (a library routine).

The five named workloads follow the attention layer's shapes (64 or 128 local heads,
head_dim 512, window 128, compress ratio 4, index_topk-sized compressed selections):

  tiny        b1 s16 h4 d64 rows48: 8 ring columns + 8 distinct random rows from 8..47,
              ~20 % of entries dropped to -1 and query 11 entirely -1
  swa_prefill b1 s4096 h64 d512: 4096 chunk rows, idx = the causal 128-wide window only
  cmp_prefill b1 s8192 h64 d512 ratio 4: 8192 chunk rows + 2048 compressed rows; idx = window
              ++ 512 distinct visible compressed groups (+8192), ascending, -1 tail when fewer
              than 512 are visible
  decode      b64 s1 h64 d512 at position 32768: 128 ring rows + 8192 compressed rows per
              sequence; idx = ring ++ 1024 distinct compressed rows (+128), ascending
  fp8_decode  b256 s1 h128 d512 at position 131072, kv stored e4m3 + e8m0: 128 ring rows +
              32768 compressed rows; idx = ring ++ 2048 distinct compressed rows (+128),
              ascending, 102 of them (5 %) scattered to -1

The window columns themselves are not produced here: they are the method's own
``window_idxs(start_pos, s, window)`` and are put in front of ``idx_tail`` by the caller.
kv rows that no index can reach are left at zero (only their values would differ; no output
depends on them), which keeps the 4 GB fp8 cache cheap to build.
"""

from __future__ import annotations

import dataclasses
import functools

import numpy as np
import torch


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """f32 array -> bf16 bit patterns (uint16), rounded by torch."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


@dataclasses.dataclass
class Workload:
    name: str
    b: int
    s: int
    h: int
    d: int
    rows: int          # kv rows per sequence (window part first, then compressed part)
    topk: int          # idx columns = window + tail
    window: int        # leading idx columns that come from window_idxs
    start_pos: int     # 0 = prefill of an s-token chunk, p = single-token decode at position p
    kv_format: str     # "bf16" or "fp8" (e4m3 codes + e8m0 block scales in storage)
    scale: float       # softmax scale head_dim ** -0.5, as the f32 the kernels receive
    q: np.ndarray      # uint16 [b, s, h, d] bf16 bits
    sink: np.ndarray   # float32 [h]
    idx_tail: np.ndarray   # int32 [b, s, topk - window]: the non-window columns, final values
    drop: np.ndarray | None  # bool [b, s, topk] entries forced to -1 after composing, or None
    kv_rows: np.ndarray    # int64 [b, n_used] kv rows that hold values (ascending)
    kv_vals: np.ndarray    # uint16 [b, n_used, d] raw bf16 N(0,1) values of those rows
    ring_slots: bool = False  # tiny only: the window columns are ring slots (position mod window)
    seed: int = 0

    @property
    def n_tokens(self) -> int:
        return self.b * self.s

    def kv_raw_dense(self, bsel=None) -> np.ndarray:
        """Raw (pre-act_quant) kv as dense bf16 bits [len(bsel), rows, d] (zeros elsewhere)."""
        bs = range(self.b) if bsel is None else bsel
        out = np.zeros((len(bs), self.rows, self.d), np.uint16)
        for i, bi in enumerate(bs):
            out[i, self.kv_rows[bi]] = self.kv_vals[bi]
        return out

    def flops(self) -> float:
        """4 * b * s * h * topk * d (QK^T and PV, every idx column counted)."""
        return 4.0 * self.b * self.s * self.h * self.topk * self.d

    def q_bytes(self) -> int:
        return self.b * self.s * self.h * self.d * 2

    def kv_row_bytes(self) -> int:
        return self.d * 2 if self.kv_format == "bf16" else self.d + self.d // 32


def _normal_bf16(rng, shape) -> np.ndarray:
    return to_bf16_bits(rng.standard_normal(shape, dtype=np.float32))


def _distinct_sorted(rng, n_choices: int, k: int) -> np.ndarray:
    return np.sort(rng.choice(n_choices, size=k, replace=False)).astype(np.int32)


def _fill_rows(rng, b, rows_per_seq, d):
    kv_rows = np.stack([np.asarray(r, np.int64) for r in rows_per_seq])
    kv_vals = _normal_bf16(rng, (b, kv_rows.shape[1], d))
    return kv_rows, kv_vals


@functools.lru_cache(maxsize=4)
def make_named(name: str, visibility: str = "pages", batch: int | None = None) -> Workload:
    """One of the five named workloads, drawn from its fixed seed.  ``batch`` sets the number of
    sequences of the two decode workloads (a smaller case of the same structure, e.g. for a
    profiler capture); the other workloads ignore it."""
    if name == "tiny":
        seed, b, s, h, d, rows, W = 1, 1, 16, 4, 64, 48, 8
        rng = np.random.default_rng(seed)
        q = _normal_bf16(rng, (b, s, h, d))
        sink = rng.standard_normal(h, dtype=np.float32)
        tail = np.stack([_distinct_sorted(rng, rows - W, 8) + W for _ in range(s)])[None]
        drop = rng.random((b, s, W + 8)) < 0.2
        drop[0, 11, :] = True
        kv_rows, kv_vals = _fill_rows(rng, b, [np.arange(rows)], d)
        return Workload(name, b, s, h, d, rows, W + 8, W, 0, "bf16", float(np.float32(d ** -0.5)),
                        q, sink, tail.astype(np.int32), drop, kv_rows, kv_vals, ring_slots=True,
                        seed=seed)
    if name == "swa_prefill":
        seed, b, s, h, d, W = 2, 1, 4096, 64, 512, 128
        rng = np.random.default_rng(seed)
        q = _normal_bf16(rng, (b, s, h, d))
        sink = rng.standard_normal(h, dtype=np.float32)
        tail = np.zeros((b, s, 0), np.int32)
        kv_rows, kv_vals = _fill_rows(rng, b, [np.arange(s)], d)
        return Workload(name, b, s, h, d, s, W, W, 0, "bf16", float(np.float32(d ** -0.5)),
                        q, sink, tail, None, kv_rows, kv_vals, seed=seed)
    if name == "cmp_prefill":
        seed, b, s, h, d, W, ratio, k = 3, 1, 8192, 64, 512, 128, 4, 512
        n_cmp = s // ratio
        rng = np.random.default_rng(seed)
        q = _normal_bf16(rng, (b, s, h, d))
        sink = rng.standard_normal(h, dtype=np.float32)
        tail = np.full((b, s, k), -1, np.int32)
        for p in range(s):
            # compressed groups this query may see: the Indexer's rule (a group becomes visible
            # once the query has passed its last token), or the group-start rule
            n_vis = (p + 1) // ratio if visibility == "pages" else min(p // ratio + 1, n_cmp)
            kk = min(k, n_vis)
            if kk:
                tail[0, p, :kk] = _distinct_sorted(rng, n_vis, kk) + s
        kv_rows, kv_vals = _fill_rows(rng, b, [np.arange(s + n_cmp)], d)
        return Workload(name, b, s, h, d, s + n_cmp, W + k, W, 0, "bf16",
                        float(np.float32(d ** -0.5)), q, sink, tail, None, kv_rows, kv_vals,
                        seed=seed)
    if name in ("decode", "fp8_decode"):
        if name == "decode":
            seed, b, h, pos, k, n_drop, fmt = 4, 64, 64, 32768, 1024, 0, "bf16"
        else:
            seed, b, h, pos, k, n_drop, fmt = 5, 256, 128, 131072, 2048, 102, "fp8"
        if batch is not None:
            b = int(batch)
        s, d, W, ratio = 1, 512, 128, 4
        n_cmp = pos // ratio
        rng = np.random.default_rng(seed)
        q = _normal_bf16(rng, (b, s, h, d))
        sink = rng.standard_normal(h, dtype=np.float32)
        tail = np.stack([_distinct_sorted(rng, n_cmp, k) + W for _ in range(b)])[:, None, :]
        for bi in range(b):
            if n_drop:  # scattered through the compressed columns, not only at the tail
                tail[bi, 0, rng.choice(k, size=n_drop, replace=False)] = -1
        used = []
        for bi in range(b):
            live = tail[bi, 0][tail[bi, 0] >= 0]
            used.append(np.concatenate([np.arange(W), np.sort(live)]))
        width = max(len(u) for u in used)
        # pad every sequence's row list to the same width with further unused rows (values
        # there are never read); keeps the arrays rectangular
        for bi in range(b):
            if len(used[bi]) < width:
                spare = np.setdiff1d(np.arange(W, W + n_cmp), used[bi])[: width - len(used[bi])]
                used[bi] = np.sort(np.concatenate([used[bi], spare]))
        kv_rows, kv_vals = _fill_rows(rng, b, used, d)
        return Workload(name, b, s, h, d, W + n_cmp, W + k, W, pos, fmt,
                        float(np.float32(d ** -0.5)), q, sink, tail.astype(np.int32), None,
                        kv_rows, kv_vals, seed=seed)
    raise KeyError(name)


NAMED = ("tiny", "swa_prefill", "cmp_prefill", "decode", "fp8_decode")


def make_random(b, s, h, d, rows, topk, *, seed, window=0, start_pos=0, kv_format="bf16",
                neg_frac=0.1, all_neg_tokens=(), sink_scale=1.0, q_scale=1.0,
                distinct=True) -> Workload:
    """A free-form workload for parity cases: random idx columns (distinct per token unless
    ``distinct`` is False) drawn from all rows, ``neg_frac`` of them set to -1, and the tokens in
    ``all_neg_tokens`` left with no row at all.  ``window`` > 0 reserves that many leading
    columns for window_idxs, composed by the caller."""
    rng = np.random.default_rng(seed)
    q = to_bf16_bits(rng.standard_normal((b, s, h, d), dtype=np.float32) * np.float32(q_scale))
    sink = (rng.standard_normal(h, dtype=np.float32) * np.float32(sink_scale)).astype(np.float32)
    ntail = topk - window
    tail = np.empty((b, s, ntail), np.int32)
    for bi in range(b):
        for si in range(s):
            if distinct and ntail <= rows:
                tail[bi, si] = rng.choice(rows, size=ntail, replace=False)
            else:
                tail[bi, si] = rng.integers(0, rows, size=ntail)
    drop = rng.random((b, s, topk)) < neg_frac
    for t in all_neg_tokens:
        drop[t // s, t % s, :] = True
    kv_rows, kv_vals = _fill_rows(rng, b, [np.arange(rows)] * b, d)
    return Workload(f"random_b{b}_s{s}_h{h}_d{d}_r{rows}_k{topk}", b, s, h, d, rows, topk, window,
                    start_pos, kv_format, float(np.float32(d ** -0.5)), q, sink, tail, drop,
                    kv_rows, kv_vals, seed=seed)


def rope_table(npos: int, rope_dim: int, *, seed: int) -> np.ndarray:
    """A rotation table for the output's rope dims: [npos, rope_dim / 2, 2] f32 (cos, sin) of
    angles drawn uniformly from [-pi, pi) (the layer's own table holds position times frequency;
    any angle exercises the rotation the same way), computed by numpy's cos / sin."""
    ang = np.random.default_rng(seed).uniform(-np.pi, np.pi, (npos, rope_dim // 2))
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1).astype(np.float32)
