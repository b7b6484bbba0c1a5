"""dt_tree_attention on the GPU against the CPU oracle (fp64): the verify pass's attention over the prefix and the
draft tree with the ancestor-only mask.

Tolerance: the GPU multiplies bf16 inputs exactly and accumulates in fp32, but rounds the softmax weights to bf16
(relative error 2^-9) before they weigh the value rows (|v| <= ~4.5 for N(0,1) draws): the output error is at most
about 2^-9 x 4.5 = 0.009. TOL = 1e-2 absolute, and the mean error must be far below it."""
import math

import numpy as np
import pytest
import torch

from oracle import oracle as orc
from speculative_decoding_tree_top_gb300 import synth

pytestmark = pytest.mark.gpu
TOL = 1e-2


def run(dtlib, B, n, L, Hq, Hkv, d=128, seed=2468, mask=None):
    q, k, v, m = synth.make_attention_inputs(B, n, L, Hq, Hkv, d, seed=seed)
    if mask is not None:
        m = mask
    scale = 1.0 / math.sqrt(d)
    out = dtlib.dt_tree_attention(q.cuda(), k.cuda(), v.cuda(), m.cuda(), scale)
    torch.cuda.synchronize()
    ref = orc.tree_attention(synth.bits_u16(q), synth.bits_u16(k), synth.bits_u16(v), m.numpy(), scale)
    return out.cpu().numpy().astype(np.float64), ref, (q, k, v, m)


@pytest.mark.parametrize("B,n,L,Hq,Hkv", [
    (1, 16, 2048, 32, 8),     # Qwen3-4B's attention shape, a 2048-token prefix: the bench case
    (2, 16, 0, 32, 8),        # no prefix: the tree keys alone
    (3, 7, 100, 8, 2),        # odd sizes: rows 28 of 64, a partial key block
    (1, 16, 5000, 4, 1),      # one key/value head, a long prefix in many chunks
    (4, 1, 63, 2, 2),         # one node, no grouping
    (64, 16, 100, 32, 8),     # pairs of two key blocks: most inside one CTA's share (written directly), the rest
                              # split over two CTAs (combined)
])
def test_tree_attention_parity(dtlib, B, n, L, Hq, Hkv):
    out, ref, _ = run(dtlib, B, n, L, Hq, Hkv)
    err = np.abs(out - ref)
    assert err.max() <= TOL, err.max()
    assert err.mean() <= TOL / 10, err.mean()


def test_tree_attention_diagonal_mask_returns_own_values(dtlib):
    """No prefix and a diagonal mask: each node's only key is itself, its weight 1 exactly, so the output is its own
    value row exactly."""
    B, n, Hq, Hkv = 2, 16, 8, 2
    diag = torch.eye(n, dtype=torch.uint8).expand(B, n, n).contiguous()
    out, _, (q, k, v, m) = run(dtlib, B, n, 0, Hq, Hkv, mask=diag)
    vf = v.float().numpy()
    for h in range(Hq):
        assert np.array_equal(out[:, :, h], vf[:, h // (Hq // Hkv)].astype(np.float64)), h


def test_tree_attention_full_batch_sampled_requests(dtlib):
    """The B = 64 configuration the bench times (its combine takes a warp per row): the whole batch on the GPU, two
    sampled requests against the oracle one by one (requests are independent)."""
    B, n, L, Hq, Hkv, d = 64, 16, 2048, 32, 8, 128
    q, k, v, m = synth.make_attention_inputs(B, n, L, Hq, Hkv, d, seed=77)
    scale = 1.0 / math.sqrt(d)
    out = dtlib.dt_tree_attention(q.cuda(), k.cuda(), v.cuda(), m.cuda(), scale)
    torch.cuda.synchronize()
    out = out.cpu().numpy().astype(np.float64)
    for b in (5, 63):
        ref = orc.tree_attention(synth.bits_u16(q[b:b + 1]), synth.bits_u16(k[b:b + 1]), synth.bits_u16(v[b:b + 1]),
                                 m[b:b + 1].numpy(), scale)
        err = np.abs(out[b:b + 1] - ref)
        assert err.max() <= TOL, (b, err.max())
        assert err.mean() <= TOL / 10, (b, err.mean())
