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
