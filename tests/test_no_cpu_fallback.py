"""The product path has no CPU fallback: every Python entry refuses host tensors with an error
before anything is computed, and the package never imports the oracle."""

from __future__ import annotations

import ast
import os

import pytest
import torch

import sparse_latent_attention_gb300 as sa

PKG = os.path.dirname(sa.__file__)


def _host(*shape, dtype=torch.float32):
    return torch.zeros(shape, dtype=dtype)


@pytest.mark.parametrize("call", [
    lambda: sa.sparse_attn(_host(1, 2, 4, 64, dtype=torch.bfloat16), _host(1, 8, 64, dtype=torch.bfloat16),
                           _host(4), torch.zeros((1, 2, 4), dtype=torch.int32), 0.125),
    lambda: sa.indexer_topk(_host(1, 8, 2), 0, 4, 1, 0),
    lambda: sa.candidate_blocks(_host(1, 8, 2), 0, 4, 1, 1),
    lambda: sa.hc_split_sinkhorn(_host(3, 24), _host(3), _host(24)),
    lambda: sa.act_quant_fp8(_host(2, 64, dtype=torch.bfloat16), out_rt=_host(2, 64, dtype=torch.bfloat16)),
])
def test_host_tensors_are_refused(call):
    with pytest.raises((TypeError, ValueError)):
        call()


def test_package_never_imports_the_oracle():
    for root, _, files in os.walk(PKG):
        for f in files:
            if not f.endswith(".py"):
                continue
            tree = ast.parse(open(os.path.join(root, f)).read())
            for node in ast.walk(tree):
                names = []
                if isinstance(node, ast.Import):
                    names = [a.name for a in node.names]
                elif isinstance(node, ast.ImportFrom):
                    names = [node.module or ""]
                assert not any(n == "oracle" or n.startswith("oracle.") for n in names), (f, names)
