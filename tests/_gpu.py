"""GPU-side preparation of a workload through the library (window_idxs, act_quant) and the
matching oracle-side expectations."""

from __future__ import annotations

import numpy as np
import torch

import sparse_latent_attention_gb300 as sa
from tests._helpers import compose_idx_oracle


def u16_to_bf16_tensor(a: np.ndarray, device) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_tensor_to_u16(t: torch.Tensor) -> np.ndarray:
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def device_kv_raw(wl, device) -> torch.Tensor:
    """Dense raw kv [b, rows, d] bf16 on the device (rows no index reaches stay zero)."""
    kv = torch.zeros((wl.b, wl.rows, wl.d), dtype=torch.bfloat16, device=device)
    rows = torch.from_numpy(wl.kv_rows).to(device)
    vals = u16_to_bf16_tensor(wl.kv_vals, device)
    bidx = torch.arange(wl.b, device=device)[:, None].expand_as(rows)
    kv[bidx, rows] = vals
    return kv


def device_idx(wl, device) -> torch.Tensor:
    """idx [b, s, topk] with the window columns written by the library's window_idxs."""
    idx = torch.empty((wl.b, wl.s, wl.topk), dtype=torch.int32, device=device)
    if wl.window:
        sa.window_idxs(wl.start_pos, wl.s, wl.window, out=idx[:, :, : wl.window], nbatch=wl.b)
        if wl.ring_slots:
            w = idx[:, :, : wl.window]
            idx[:, :, : wl.window] = torch.where(w >= 0, w % wl.window, w)
    idx[:, :, wl.window:] = torch.from_numpy(wl.idx_tail).to(device)
    if wl.drop is not None:
        idx[torch.from_numpy(wl.drop).to(device)] = -1
    return idx


def prepare(wl, device, quantise: bool):
    """Device inputs of one workload, built through the library: returns a dict with q, kv (bf16
    round trip, or e4m3 codes for fp8 storage), kv_scale (fp8 only), sink, idx."""
    q = u16_to_bf16_tensor(wl.q, device)
    sink = torch.from_numpy(wl.sink).to(device)
    idx = device_idx(wl, device)
    kv = device_kv_raw(wl, device)
    kv_scale = None
    if quantise and wl.kv_format == "fp8":
        codes = torch.empty((wl.b, wl.rows, wl.d), dtype=torch.uint8, device=device)
        kv_scale = torch.empty((wl.b, wl.rows, wl.d // 32), dtype=torch.uint8, device=device)
        sa.act_quant_fp8(kv.view(-1, wl.d), codes=codes.view(-1, wl.d),
                         scales=kv_scale.view(-1, wl.d // 32))
        del kv
        kv = codes
    elif quantise:
        sa.act_quant_fp8(kv.view(-1, wl.d), out_rt=kv.view(-1, wl.d))
    return dict(q=q, kv=kv, kv_scale=kv_scale, sink=sink, idx=idx)


def oracle_inputs(wl, quantise: bool, bsel):
    """Oracle-side kv for the sequences in bsel and the full composed idx.  Only rows that hold
    values go through the oracle's act_quant; the other rows take the oracle's result for an
    all-zero row."""
    import oracle
    idx = compose_idx_oracle(wl)
    if not quantise:
        return wl.kv_raw_dense(bsel), None, idx
    bsel = list(bsel)
    rt_u, codes_u, sc_u = oracle.act_quant(wl.kv_vals[bsel])
    zrt, zc, zs = oracle.act_quant(np.zeros((1, wl.d), np.uint16))
    nb = len(bsel)
    rt = np.broadcast_to(zrt, (nb, wl.rows, wl.d)).copy()
    codes = np.broadcast_to(zc, (nb, wl.rows, wl.d)).copy()
    scales = np.broadcast_to(zs, (nb, wl.rows, wl.d // 32)).copy()
    for i, bi in enumerate(bsel):
        rt[i, wl.kv_rows[bi]] = rt_u[i]
        codes[i, wl.kv_rows[bi]] = codes_u[i]
        scales[i, wl.kv_rows[bi]] = sc_u[i]
    if wl.kv_format == "fp8":
        return codes, scales, idx
    return rt, None, idx
