"""Pins for the oracle's sliding-window branch and gated combination (CPU only).

The sliding-window branch of Native Sparse Attention (window_size in the
Flash-Sparse-Attention README's "Usage"; the three parallel branches of the
papernotes page's 领域现状): every token attends to its last `window` positions,
causal, one softmax.  The oracle expresses it as a block selection (the blocks that
hold those keys) plus a token-level lower bound, so it is pinned to dense banded
attention computed by torch SDPA (fp64) and its autograd.  The gated combination is a
plain weighted sum: it is pinned to its closed form and to finite differences.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import make_cu_seqlens


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _banded_sdpa(q, k, v, seqlens, window, scale, grad_out=None):
    """Dense sliding-window attention per sequence via torch SDPA; with grad_out, also
    (dq, dk, dv) by autograd.  q [N, h_q, d]; k, v [N, h_k, d] (fp64 numpy)."""
    h_q, h_k = q.shape[1], k.shape[1]
    g = h_q // h_k
    tq = torch.from_numpy(q).requires_grad_(grad_out is not None)
    tk = torch.from_numpy(k).requires_grad_(grad_out is not None)
    tv = torch.from_numpy(v).requires_grad_(grad_out is not None)
    outs, base = [], 0
    for L in seqlens:
        i = torch.arange(L)
        mask = (i[None, :] <= i[:, None]) & (i[None, :] > i[:, None] - window)
        qs = tq[base:base + L].permute(1, 0, 2).unsqueeze(0)
        ks = tk[base:base + L].repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
        vs = tv[base:base + L].repeat_interleave(g, dim=1).permute(1, 0, 2).unsqueeze(0)
        o = F.scaled_dot_product_attention(qs, ks, vs, attn_mask=mask, scale=scale)
        outs.append(o.squeeze(0).permute(1, 0, 2))
        base += L
    out = torch.cat(outs, 0)
    if grad_out is None:
        return out.detach().numpy()
    out.backward(torch.from_numpy(grad_out))
    return out.detach().numpy(), tq.grad.numpy(), tk.grad.numpy(), tv.grad.numpy()


@pytest.mark.parametrize("window,block", [(20, 8), (1, 8), (64, 16), (13, 4)])
def test_window_forward_equals_banded_sdpa(window, block):
    seqlens, h_k, g, d = [70, 1, 45], 2, 2, 16
    n = sum(seqlens)
    topk = (window - 1 + block - 1) // block + 1
    q, k, v = _rand((n, h_k * g, d), 1), _rand((n, h_k, d), 2), _rand((n, h_k, d), 3)
    cu = make_cu_seqlens(seqlens)
    sel = oracle.window_select(cu, h_k, block, topk, window)
    out, lse = oracle.fwd(cu, block, sel, q, k, v, 0.25, window=window)
    ref = _banded_sdpa(q, k, v, seqlens, window, 0.25)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    assert np.isfinite(lse).all()


def test_window_backward_equals_banded_autograd():
    seqlens, h_k, g, d, block, window = [50, 33], 1, 3, 8, 8, 17
    n = sum(seqlens)
    topk = (window - 1 + block - 1) // block + 1
    q, k, v, do = (_rand((n, h_k * g, d), 11), _rand((n, h_k, d), 12),
                   _rand((n, h_k, d), 13), _rand((n, h_k * g, d), 14))
    cu = make_cu_seqlens(seqlens)
    sel = oracle.window_select(cu, h_k, block, topk, window)
    dq, dk, dv = oracle.bwd(cu, block, sel, q, k, v, do, 0.4, window=window)
    _, rq, rk, rv = _banded_sdpa(q, k, v, seqlens, window, 0.4, grad_out=do)
    for got, ref in ((dq, rq), (dk, rk), (dv, rv)):
        np.testing.assert_allclose(got, ref, rtol=0, atol=1e-11)


def test_window_longer_than_sequence_is_causal_attention():
    seqlens, h_k, g, d, block = [40, 25], 1, 2, 8, 8
    n = sum(seqlens)
    q, k, v = _rand((n, h_k * g, d), 21), _rand((n, h_k, d), 22), _rand((n, h_k, d), 23)
    cu = make_cu_seqlens(seqlens)
    sel = oracle.window_select(cu, h_k, block, 5, 1000)
    w_out, w_lse = oracle.fwd(cu, block, sel, q, k, v, 0.5, window=1000)
    c_out, c_lse = oracle.fwd(cu, block, sel, q, k, v, 0.5)
    np.testing.assert_array_equal(w_out, c_out)
    np.testing.assert_array_equal(w_lse, c_lse)
    ref = _banded_sdpa(q, k, v, seqlens, 10 ** 6, 0.5)
    np.testing.assert_allclose(w_out, ref, rtol=0, atol=1e-12)


def test_window_select_rows():
    cu = make_cu_seqlens([100, 70])
    sel = oracle.window_select(cu, 1, 32, 4, 70)
    assert list(sel[0, 99]) == [3, 2, 1, 0]          # keys 30..99: blocks 0..3
    assert list(sel[0, 0]) == [0, -1, -1, -1]
    assert list(sel[0, 100 + 69]) == [2, 1, 0, -1]
    assert list(sel[0, 40]) == [1, 0, -1, -1]         # keys 0..40
    with pytest.raises(ValueError):
        oracle.window_select(cu, 1, 32, 2, 70)        # 4 blocks needed


def test_gate_combine_closed_form_and_gradients():
    rng = np.random.default_rng(5)
    o = [rng.standard_normal((6, 4, 8)) for _ in range(3)]
    gates = rng.uniform(size=(6, 4, 3))
    out = oracle.gate_combine(o, gates)
    np.testing.assert_allclose(out, gates[..., :1] * o[0] + gates[..., 1:2] * o[1]
                               + gates[..., 2:3] * o[2], rtol=0, atol=1e-15)
    dy = rng.standard_normal(out.shape)
    d_br, d_g = oracle.gate_combine_bwd(o, gates, dy)
    eps = 1e-6
    for b in range(3):
        gp, gm = gates.copy(), gates.copy()
        gp[..., b] += eps
        gm[..., b] -= eps
        fd = ((oracle.gate_combine(o, gp) - oracle.gate_combine(o, gm)) * dy).sum(-1) / (2 * eps)
        np.testing.assert_allclose(d_g[..., b], fd, rtol=0, atol=1e-8)
        op, om = [x.copy() for x in o], [x.copy() for x in o]
        op[b][0, 0, 0] += eps
        om[b][0, 0, 0] -= eps
        fd_o = ((oracle.gate_combine(op, gates) - oracle.gate_combine(om, gates)) * dy).sum() / (2 * eps)
        np.testing.assert_allclose(d_br[b][0, 0, 0], fd_o, rtol=0, atol=1e-8)
