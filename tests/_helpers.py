"""Test-side helpers: compose the oracle's inputs for a workload and compare results."""

from __future__ import annotations

import numpy as np

import oracle


def compose_idx_oracle(wl) -> np.ndarray:
    """idx [b, s, topk]: the oracle's window_idxs columns, then the workload's tail columns, then
    the workload's forced -1 entries."""
    idx = np.empty((wl.b, wl.s, wl.topk), np.int32)
    if wl.window:
        win = oracle.window_idxs(wl.start_pos, wl.s, wl.window)
        if wl.ring_slots:
            win = np.where(win >= 0, win % wl.window, -1).astype(np.int32)
        idx[:, :, : wl.window] = win[None]
    idx[:, :, wl.window:] = wl.idx_tail
    if wl.drop is not None:
        idx[wl.drop] = -1
    return idx


def quantised_kv_oracle(wl, quantise: bool, bsel=None):
    """The kv the attention sees: raw bf16, or the oracle's act_quant round trip.  For fp8 storage
    also returns (codes, scales)."""
    raw = wl.kv_raw_dense(bsel)
    if not quantise:
        return raw, None, None
    rt, codes, scales = oracle.act_quant(raw)
    return rt, codes, scales


def bf16_to_f64(bits):
    return oracle.bf16_to_f64(bits)


def assert_close_bf16(got_bits, want_bits, atol=1e-2, rtol=1e-2, what=""):
    """|got - want| <= atol + rtol * |want| elementwise (bf16 output, f32 accumulate)."""
    g = bf16_to_f64(got_bits)
    w = bf16_to_f64(want_bits)
    err = np.abs(g - w)
    lim = atol + rtol * np.abs(w)
    bad = ~(err <= lim)
    if bad.any():
        where = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} elements out of tolerance; "
                             f"first at {where.tolist()}: got {g[bad][:5]}, want {w[bad][:5]}; "
                             f"max err {err.max():.3e}")
    return float(err.max()) if err.size else 0.0
