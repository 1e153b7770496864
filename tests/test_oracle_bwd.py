"""Pins for the oracle's backward (CPU only): finite differences of the oracle's
own forward, torch autograd through SDPA on the dense special case, and closed
forms (sum_j dk_j = 0, constant V, q = 0)."""
import math

import numpy as np
import torch
import torch.nn.functional as F

import oracle
from workloads import make_cu_seqlens, make_selection


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _setup(seqlens=(64,), h_k=1, g=2, d=8, block=16, topk=3, seed=0):
    n = sum(seqlens)
    rng = np.random.default_rng(seed)
    sel = make_selection(list(seqlens), h_k, block, topk, "uniform", rng)
    q, k, v = rng.standard_normal((n, h_k * g, d)), rng.standard_normal((n, h_k, d)), \
        rng.standard_normal((n, h_k, d))
    dout = rng.standard_normal((n, h_k * g, d))
    return make_cu_seqlens(list(seqlens)), block, sel, q, k, v, dout


def test_finite_differences():
    # L = sum(dO * O); central differences, eps = 1e-6, relative error <= 1e-6.
    cu, block, sel, q, k, v, dout = _setup(seqlens=(64,), seed=1)
    scale = 0.35
    dq, dk, dv = oracle.bwd(cu, block, sel, q, k, v, dout, scale)

    def loss(q_, k_, v_):
        out, _ = oracle.fwd(cu, block, sel, q_, k_, v_, scale)
        return float(np.sum(out * dout))

    rng = np.random.default_rng(2)
    eps = 1e-6
    for name, x, grad in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        flat = x.reshape(-1)
        idx = rng.choice(flat.size, size=min(flat.size, 120), replace=False)
        num = np.empty(idx.size)
        for i, j in enumerate(idx):
            xp, xm = flat.copy(), flat.copy()
            xp[j] += eps
            xm[j] -= eps
            args = {"q": q, "k": k, "v": v}
            args[name] = xp.reshape(x.shape)
            lp = loss(args["q"], args["k"], args["v"])
            args[name] = xm.reshape(x.shape)
            lm = loss(args["q"], args["k"], args["v"])
            num[i] = (lp - lm) / (2 * eps)
        ana = grad.reshape(-1)[idx]
        err = np.abs(num - ana) / np.maximum(1.0, np.abs(ana))
        assert err.max() <= 1e-6, (name, err.max())


def test_dense_causal_grads_equal_sdpa_autograd():
    n, h_k, g, d, block, topk = 96, 1, 2, 16, 16, 6
    rng = np.random.default_rng(3)
    sel = np.full((h_k, n, topk), -1, dtype=np.int32)
    for t in range(n):
        sel[0, t, :t // block + 1] = rng.permutation(t // block + 1)
    q, k, v = _rand((n, h_k * g, d), 4), _rand((n, h_k, d), 5), _rand((n, h_k, d), 6)
    dout = _rand((n, h_k * g, d), 7)
    dq, dk, dv = oracle.bwd(make_cu_seqlens([n]), block, sel, q, k, v, dout, 0.25)
    tq = torch.from_numpy(q).permute(1, 0, 2).unsqueeze(0).requires_grad_()
    tk = torch.from_numpy(k).permute(1, 0, 2).unsqueeze(0).requires_grad_()
    tv = torch.from_numpy(v).permute(1, 0, 2).unsqueeze(0).requires_grad_()
    o = F.scaled_dot_product_attention(tq, tk.repeat_interleave(g, 1), tv.repeat_interleave(g, 1),
                                       is_causal=True, scale=0.25)
    o.backward(torch.from_numpy(dout).permute(1, 0, 2).unsqueeze(0))
    np.testing.assert_allclose(dq, tq.grad[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dk, tk.grad[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)
    np.testing.assert_allclose(dv, tv.grad[0].permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


def test_dk_sums_to_zero_per_kv_head():
    # Each row's dS sums to zero and q_t is constant along the row: sum_j dk_j = 0.
    cu, block, sel, q, k, v, dout = _setup(seqlens=(50, 77), h_k=2, g=3, d=8, block=8, topk=4,
                                           seed=8)
    _, dk, _ = oracle.bwd(cu, block, sel, q, k, v, dout, 0.5)
    assert np.abs(dk.sum(axis=0)).max() < 1e-11


def test_constant_v_zero_dq_dk():
    cu, block, sel, q, k, v, dout = _setup(seqlens=(70,), h_k=2, g=2, seed=9)
    v = np.broadcast_to(_rand((1, 2, 8), 10), v.shape).copy()
    dq, dk, _ = oracle.bwd(cu, block, sel, q, k, v, dout, 0.5)
    assert np.abs(dq).max() < 1e-12 and np.abs(dk).max() < 1e-12


def test_zero_query_dv_closed_form():
    # q = 0: P = 1/n(t) on K(t), so dv_j = sum over (t, hq) with j in K(t) of dO_t / |K(t)|.
    seqlens, h_k, g, d, block, topk = (45, 30), 2, 2, 4, 8, 4
    cu, block, sel, q, k, v, dout = _setup(seqlens, h_k, g, d, block, topk, seed=11)
    q = np.zeros_like(q)
    _, _, dv = oracle.bwd(cu, block, sel, q, k, v, dout, 1.0)
    ref = np.zeros_like(dv)
    base = 0
    for L in seqlens:
        for tau in range(L):
            for h in range(h_k):
                blocks = {int(b) for b in sel[h, base + tau] if 0 <= b <= tau // block}
                keys = [kk for kk in range(tau + 1) if kk // block in blocks]
                for j in range(g):
                    for kk in keys:
                        ref[base + kk, h] += dout[base + tau, h * g + j] / len(keys)
        base += L
    np.testing.assert_allclose(dv, ref, rtol=0, atol=1e-13)
