"""GPU parity of the indexer's selection (sa_indexer_topk) against the CPU oracle: bit-exact idx on
the same seeded scores, ties included (both sides pick equal scores lowest position first)."""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
import sparse_latent_attention_gb300 as sa
from sparse_latent_attention_gb300 import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="session")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    build.build()
    sa.load()
    return torch.device("cuda:0")


def _scores(rng, b, s, n, kind):
    x = rng.standard_normal((b, s, n)).astype(np.float32)
    if kind == "ties":        # eight levels: most picks are decided by the tie rule
        x = np.round(x * 2.0).astype(np.float32)
    elif kind == "specials":  # -0 / +0, -inf inside the visible range, whole rows equal
        x[x > 1.2] = 0.0
        x[x < -1.2] = -0.0
        x[(x > 0.0) & (x < 0.1)] = -np.inf
        x[:, ::7, :] = 0.5
    return x


def _run(dev, score_np, start_pos, ratio, topk, offset, bf16=False):
    if bf16:
        bits = (score_np.view(np.uint32) >> 16).astype(np.uint16)      # truncated to bf16
        t = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
        want = oracle.indexer_topk(bits, start_pos, ratio, topk, offset)
    else:
        t = torch.from_numpy(score_np).to(dev)
        want = oracle.indexer_topk(score_np, start_pos, ratio, topk, offset)
    got = sa.indexer_topk(t, start_pos, ratio, topk, offset)
    torch.cuda.synchronize()
    return got.cpu().numpy(), want


CASES = [
    # b, s, start_pos, ratio, index_topk, offset, kind, bf16
    (1, 8192, 0, 4, 512, 8192, "normal", False),     # the compressed prefill: 2048 positions
    (64, 1, 131071, 4, 2048, 128, "normal", False),  # long decode: 32768 positions
    (1, 1000, 0, 4, 64, 128, "ties", True),          # bf16 scores, heavy ties
    (2, 301, 0, 4, 48, 5, "specials", False),        # -0/+0, -inf, equal rows; ragged s
    (1, 100, 0, 4, 512, 128, "normal", False),       # index_topk above the positions: k = 25
    (3, 1, 40, 4, 1, 0, "ties", False),              # k = 1
    (1, 257, 0, 1, 100, 0, "normal", False),         # ratio 1
    (2, 1, 16383, 4, 700, 9, "ties", True),          # 4096 positions: 128-thread block
    (2, 1, 16387, 4, 700, 9, "ties", True),          # 4097: the shortest 1024-thread row
    (4, 1, 32767, 4, 1024, 128, "normal", False),    # the decode shape's 8192 positions
    (2, 1, 65539, 4, 3000, 9, "normal", False),      # 16385: 1024-thread block
    (2, 1, 4 * 49152 - 1, 4, 2048, 128, "ties", False),  # the largest row (192 KB of keys)
]


@pytest.mark.parametrize("case", CASES, ids=lambda c: f"b{c[0]}s{c[1]}p{c[2]}r{c[3]}k{c[4]}{c[6]}"
                         f"{'-bf16' if c[7] else ''}")
def test_indexer_topk_bit_exact(dev, case):
    b, s, start_pos, ratio, topk, offset, kind, bf16 = case
    n = (start_pos + s) // ratio
    rng = np.random.default_rng(b * 1000 + s + topk)
    got, want = _run(dev, _scores(rng, b, s, n, kind), start_pos, ratio, topk, offset, bf16)
    assert got.shape == want.shape
    bad = np.argwhere(got != want)
    assert bad.size == 0, f"{len(bad)} entries differ; first at {bad[:3].tolist()}"


def test_indexer_topk_into_wider_idx(dev):
    # the k columns written after the window columns of a wider idx tensor, nothing else touched
    b, s, ratio, topk, W = 2, 1, 4, 300, 128
    start_pos = 4 * 1000 - 1
    n = (start_pos + s) // ratio
    rng = np.random.default_rng(5)
    sc = rng.standard_normal((b, s, n)).astype(np.float32)
    idx = torch.full((b, s, W + topk + 3), -7, dtype=torch.int32, device=dev)
    sa.indexer_topk(torch.from_numpy(sc).to(dev), start_pos, ratio, topk, W,
                    out=idx[:, :, W:W + topk])
    torch.cuda.synchronize()
    got = idx.cpu().numpy()
    assert (got[:, :, W:W + topk] == oracle.indexer_topk(sc, start_pos, ratio, topk, W)).all()
    assert (got[:, :, :W] == -7).all() and (got[:, :, W + topk:] == -7).all()


def test_indexer_topk_feeds_sparse_attn(dev):
    # the selection's output is a valid idx for the attention call: window columns from
    # window_idxs, compressed columns from indexer_topk, rows = window + compressed positions
    b, s, h, d, ratio, W, topk = 1, 64, 64, 512, 4, 16, 8
    n = s // ratio
    rng = np.random.default_rng(6)
    sc = torch.from_numpy(rng.standard_normal((b, s, n)).astype(np.float32)).to(dev)
    idx = torch.empty((b, s, W + topk), dtype=torch.int32, device=dev)
    sa.window_idxs(0, s, W, out=idx[:, :, :W])
    sa.indexer_topk(sc, 0, ratio, topk, s, out=idx[:, :, W:])
    q = torch.randn((b, s, h, d), device=dev).to(torch.bfloat16)
    kv = torch.randn((b, s + n, d), device=dev).to(torch.bfloat16)
    ws = sa.new_workspace(b, s, h, d, s + n, W + topk, device=dev)
    sa.sparse_attn(q, kv, torch.zeros(h, device=dev), idx, d ** -0.5, workspace=ws)
    torch.cuda.synchronize()
    assert sa.read_status(ws) == 0  # every index inside [-1, rows)
    comp = idx[:, :, W:].cpu().numpy()
    assert ((comp == -1) | ((comp >= s) & (comp < s + n))).all()


CAND_CASES = [
    # b, s, start_pos, ratio, topk_blocks, block_size, kind, bf16
    (1, 8192, 0, 4, 2048, 8, "normal", False),      # the page's 2048 x 8 over a 2048-position prefill
    (1, 8192, 0, 4, 64, 8, "normal", False),        # 64 of 256 blocks
    (64, 1, 131071, 4, 2048, 8, "normal", False),   # long decode: 4096 blocks, half kept
    (4, 1, 32767, 4, 256, 8, "ties", True),         # 8192 positions (1024 threads), 1024 blocks
    (2, 1, 16387, 4, 300, 8, "normal", False),      # 4097 positions: the shortest 1024-thread row
    (1, 1000, 0, 4, 16, 8, "ties", True),           # bf16, heavy ties between block maxima
    (2, 301, 0, 4, 5, 7, "specials", False),        # -0/+0/-inf, equal rows, a ragged last block
    (1, 64, 0, 4, 0, 8, "normal", False),           # no block wanted: all zeros
    (2, 1, 4095, 4, 100, 1, "ties", False),         # every position its own block
    (1, 40, 0, 1, 3, 64, "normal", False),          # one block, wider than the row
]


@pytest.mark.parametrize("case", CAND_CASES, ids=lambda c: f"b{c[0]}s{c[1]}p{c[2]}kb{c[4]}bs{c[5]}"
                         f"{c[6]}{'-bf16' if c[7] else ''}")
def test_candidate_blocks_bit_exact(dev, case):
    b, s, start_pos, ratio, kb, bs, kind, bf16 = case
    n = (start_pos + s) // ratio
    rng = np.random.default_rng(b * 7 + s + kb + bs)
    x = _scores(rng, b, s, n, kind)
    if bf16:
        bits = (x.view(np.uint32) >> 16).astype(np.uint16)
        t = torch.from_numpy(bits.view(np.int16)).to(dev).view(torch.bfloat16)
        want = oracle.candidate_blocks(bits, start_pos, ratio, kb, bs)
    else:
        t = torch.from_numpy(x).to(dev)
        want = oracle.candidate_blocks(x, start_pos, ratio, kb, bs)
    got = sa.candidate_blocks(t, start_pos, ratio, kb, bs)
    torch.cuda.synchronize()
    bad = np.argwhere(got.cpu().numpy() != want)
    assert bad.size == 0, f"{len(bad)} mask bytes differ; first at {bad[:3].tolist()}"


@pytest.mark.parametrize("b,s,start_pos,kb,topk", [(1, 2048, 0, 8, 64), (8, 1, 32767, 256, 512)])
def test_two_level_selection_bit_exact(dev, b, s, start_pos, kb, topk):
    # level one on one layer's scores, level two on another's inside the candidate blocks
    ratio, bs, offset = 4, 8, 128
    n = (start_pos + s) // ratio
    rng = np.random.default_rng(kb + topk)
    src = rng.standard_normal((b, s, n)).astype(np.float32)
    own = rng.standard_normal((b, s, n)).astype(np.float32)
    cand = sa.candidate_blocks(torch.from_numpy(src).to(dev), start_pos, ratio, kb, bs)
    idx = sa.indexer_topk(torch.from_numpy(own).to(dev), start_pos, ratio, topk, offset,
                          candidates=cand)
    torch.cuda.synchronize()
    cand_o = oracle.candidate_blocks(src, start_pos, ratio, kb, bs)
    assert (cand.cpu().numpy() == cand_o).all()
    want = oracle.indexer_topk(own, start_pos, ratio, topk, offset, candidates=cand_o)
    assert (idx.cpu().numpy() == want).all()
