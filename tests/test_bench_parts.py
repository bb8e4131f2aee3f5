"""Host logic of the benchmark's end-to-end step: the parts its queries are copied in, attended
and copied out in cover every query once, in order (CPU; the parts' outputs are checked against
the whole call on the GPU in test_gpu_parity)."""

from __future__ import annotations

from types import SimpleNamespace

import numpy as np
import pytest

import bench


def _covered(parts, b, s):
    hit = np.zeros((b, s), np.int32)
    for qs, ks in parts:
        hit[qs[0], qs[1] if len(qs) > 1 else slice(None)] += 1
        if len(qs) == 1:              # a batch split: kv follows the same sequences
            assert ks == qs
        else:                         # a token split: every part reads the whole kv
            assert ks == (slice(None),)
    return hit


@pytest.mark.parametrize("b,s,n", [(1, 4096, 16), (1, 8192, 16), (1, 1000, 7), (1, 5, 16),
                                   (64, 1, 8), (256, 1, 3), (3, 1, 8), (1, 1, 4)])
def test_parts_cover_every_query_once(b, s, n):
    path = SimpleNamespace(wl=SimpleNamespace(b=b, s=s))
    parts = bench.GpuPath.chunks(path, n)
    assert 1 <= len(parts) <= n
    assert (_covered(parts, b, s) == 1).all()
    # parts are contiguous and in order along the split dimension
    dim = 0 if b > 1 else 1
    edges = [p[0][dim] for p in parts]
    assert edges[0].start == 0 and edges[-1].stop == (b if b > 1 else s)
    assert all(x.stop == y.start for x, y in zip(edges, edges[1:]))


def test_roofline_line_binding_and_context():
    import bench
    peaks = {"hbm_gbs": 6659.6, "bf16_tflops": 1922.9, "bf16_tflops_sustained": 1731.3,
             "source": "measured"}
    # an HBM-bound call: 541.1 MB and 68.7 GFLOP in 0.1308 ms
    terms = {"bound": "hbm", "alg_bytes": 541_065_216, "flops": 68_719_476_736.0,
             "t_hbm": 541_065_216 / 6659.6e9, "t_tc": 68_719_476_736.0 / 1922.9e12}
    r = bench.roofline_line(terms, peaks, 0.1308, 500_166_656)
    gbs = 541_065_216 / 0.1308e-3 / 1e9
    assert r["bound"] == "hbm" and r["unit"] == "GB/s" and r["traffic"] == 500_166_656
    assert abs(r["achieved"] - gbs) < 0.1 and abs(r["frac"] - gbs / 6659.6) < 1e-4
    assert r["other"]["unit"] == "TFLOP/s"
    assert abs(r["frac_of_roofline_time"] - terms["t_hbm"] / 0.1308e-3) < 1e-4
    assert abs(r["context"]["hbm_frac_of_nominal"] - gbs / bench.HBM_NOMINAL_GBS) < 1e-4
    # a tensor-bound call; the fallback peaks carry a sustained figure too
    terms = {"bound": "tensor", "alg_bytes": 1e9, "flops": 6.87e14, "t_hbm": 1e9 / 6.8e12,
             "t_tc": 6.87e14 / 1.9e15}
    r = bench.roofline_line(terms, dict(bench.FALLBACK_PEAKS), 1.121, None)
    tfs = 6.87e14 / 1.121e-3 / 1e12
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s" and r["traffic"] is None
    assert abs(r["frac"] - tfs / 1900.0) < 1e-4 and r["peak_source"] == "fallback (burst)"
    assert abs(r["context"]["tensor_frac_of_sustained"] - tfs / 1700.0) < 1e-4


def test_both_arms_print_the_same_config():
    from sparse_latent_attention_gb300 import workloads
    wl = workloads.make_named("tiny")
    a, b = bench.config_of(wl, 1), bench.config_of(wl, 1)
    assert a == b and a["workload"] == "tiny" and "tokens_per_step" not in a
    assert bench.DEFAULT_WORKLOAD == "cmp_prefill"
    assert set(bench.TIMED_WORKLOADS) == {"swa_prefill", "cmp_prefill", "decode", "fp8_decode"}


def test_e2e_link_floor():
    link = {"h2d_gbs": 50.0, "d2h_gbs": 40.0, "duplex_gbs": 60.0}
    # each direction alone: 1 GB in 20 ms, 0.4 GB out in 10 ms; together 1.4 GB at 60 GB/s
    t = bench.e2e_link_floor_ms(link, 1e9, 4e8)
    assert abs(t - 1.4e9 / 60e9 * 1e3) < 1e-9
    assert abs(bench.e2e_link_floor_ms(link, 1e9, 0) - 20.0) < 1e-9
