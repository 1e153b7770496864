"""Pins for the oracle's forward (CPU only).

The pages print no worked example, so the oracle is pinned to what the
mathematics fixes: special cases that reduce to a library routine (torch's
scaled_dot_product_attention in fp64), a hand-derived example, closed forms and
invariants of the definition (selected attention of "FSA: An Alternative
Efficient Implementation of Native Sparse Attention Kernel", key designs 1-2:
per-token T selected blocks, causal, one softmax over their union).
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from workloads import CONFIGS, make_cu_seqlens, make_inputs, make_selection


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, mask=None, causal=False, scale=None):
    """q [N, H, d], k/v [N, H, d] fp64 numpy -> [N, H, d] via torch SDPA."""
    tq = torch.from_numpy(q).permute(1, 0, 2).unsqueeze(0)
    tk = torch.from_numpy(k).permute(1, 0, 2).unsqueeze(0)
    tv = torch.from_numpy(v).permute(1, 0, 2).unsqueeze(0)
    m = None if mask is None else torch.from_numpy(mask)
    o = F.scaled_dot_product_attention(tq, tk, tv, attn_mask=m, is_causal=causal, scale=scale)
    return o.squeeze(0).permute(1, 0, 2).numpy()


def _expand_kv(k, g):
    return np.repeat(k, g, axis=1)


def _all_causal_blocks(seqlens, h_k, block, topk, seed):
    """Every causal block selected, in a shuffled slot order, rest -1."""
    rng = np.random.default_rng(seed)
    n = sum(seqlens)
    sel = np.full((h_k, n, topk), -1, dtype=np.int32)
    base = 0
    for L in seqlens:
        for tau in range(L):
            c = tau // block
            assert c + 1 <= topk
            for h in range(h_k):
                sel[h, base + tau, :c + 1] = rng.permutation(c + 1)
        base += L
    return sel


def test_dense_causal_equals_sdpa():
    # T * B_K covers the prefix: selected attention == dense causal attention.
    n, h_k, g, d, block, topk = 256, 1, 2, 64, 32, 8
    q, k, v = _rand((n, h_k * g, d), 1), _rand((n, h_k, d), 2), _rand((n, h_k, d), 3)
    sel = _all_causal_blocks([n], h_k, block, topk, 4)
    cu = make_cu_seqlens([n])
    out, lse = oracle.fwd(cu, block, sel, q, k, v, 1 / math.sqrt(d))
    ref = _sdpa(q, _expand_kv(k, g), _expand_kv(v, g), causal=True)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # lse against an independent logsumexp of the masked dense scores
    s = np.einsum("thd,uhd->htu", q, _expand_kv(k, g)) / math.sqrt(d)
    s = np.where(np.tril(np.ones((n, n), bool))[None], s, -np.inf)
    ref_lse = torch.logsumexp(torch.from_numpy(s), dim=-1).numpy()
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-12)


def test_own_block_only_equals_block_local_sdpa():
    # Only the own block selected: block-aligned local attention (keys floor(t/B)*B .. t).
    n, h_k, g, d, block, topk = 192, 2, 2, 16, 16, 4
    q, k, v = _rand((n, h_k * g, d), 5), _rand((n, h_k, d), 6), _rand((n, h_k, d), 7)
    sel = np.full((h_k, n, topk), -1, dtype=np.int32)
    sel[:, :, 2] = (np.arange(n) // block)[None, :]          # own block in a middle slot
    out, _ = oracle.fwd(make_cu_seqlens([n]), block, sel, q, k, v, 0.3)
    t = np.arange(n)
    mask = (t[None, :] // block == t[:, None] // block) & (t[None, :] <= t[:, None])
    ref = _sdpa(q, _expand_kv(k, g), _expand_kv(v, g), mask=mask, scale=0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_varlen_dense_equals_per_sequence_causal():
    # Block indices are local to each packed sequence; no key crosses a boundary.
    seqlens, h_k, g, d, block, topk = [40, 64, 17], 1, 3, 8, 8, 8
    n = sum(seqlens)
    q, k, v = _rand((n, h_k * g, d), 8), _rand((n, h_k, d), 9), _rand((n, h_k, d), 10)
    sel = _all_causal_blocks(seqlens, h_k, block, topk, 11)
    out, _ = oracle.fwd(make_cu_seqlens(seqlens), block, sel, q, k, v, 0.5)
    base = 0
    for L in seqlens:
        sl = slice(base, base + L)
        ref = _sdpa(q[sl], _expand_kv(k[sl], g), _expand_kv(v[sl], g), causal=True, scale=0.5)
        np.testing.assert_allclose(out[sl], ref, rtol=0, atol=1e-12)
        base += L


def _random_sel(seqlens, h_k, block, topk, seed):
    return make_selection(seqlens, h_k, block, topk, "uniform", np.random.default_rng(seed))


def _key_sets(seqlens, sel, block):
    """Brute force K(t): keys tau' <= tau of the token's sequence whose block it selected."""
    out = []
    h_k, n, topk = sel.shape
    base = 0
    for L in seqlens:
        for tau in range(L):
            row = []
            for h in range(h_k):
                blocks = set(int(b) for b in sel[h, base + tau] if 0 <= b <= tau // block)
                row.append([kk for kk in range(tau + 1) if kk // block in blocks])
            out.append((base, row))
        base += L
    return out


def test_constant_v_gives_constant_output():
    seqlens, h_k, g, d, block, topk = [100, 61], 2, 2, 8, 8, 4
    n = sum(seqlens)
    sel = _random_sel(seqlens, h_k, block, topk, 12)
    q, k = _rand((n, h_k * g, d), 13) * 3, _rand((n, h_k, d), 14)
    c = _rand((1, h_k, d), 15)
    v = np.broadcast_to(c, (n, h_k, d)).copy()
    out, _ = oracle.fwd(make_cu_seqlens(seqlens), block, sel, q, k, v, 0.7)
    np.testing.assert_allclose(out, np.repeat(c, g, axis=1).repeat(n, 0), rtol=0, atol=1e-13)


def test_zero_query_closed_forms():
    # q = 0: uniform softmax, lse = ln |K(t)| and out = mean of v over K(t).
    seqlens, h_k, g, d, block, topk = [77, 50], 2, 2, 4, 8, 5
    n = sum(seqlens)
    sel = _random_sel(seqlens, h_k, block, topk, 16)
    sel[0, 5, 1] = 0          # duplicate of slot 0 (own block = block 0 at c = 0)
    sel[1, 70, 3] = 9         # future block: contributes nothing
    q = np.zeros((n, h_k * g, d))
    k, v = _rand((n, h_k, d), 17), _rand((n, h_k, d), 18)
    out, lse = oracle.fwd(make_cu_seqlens(seqlens), block, sel, q, k, v, 1.0)
    t = 0
    for base, row in _key_sets(seqlens, sel, block):
        for h in range(h_k):
            keys = np.asarray(row[h]) + base
            for j in range(g):
                hq = h * g + j
                assert lse[hq, t] == pytest.approx(math.log(len(keys)), abs=1e-14)
                np.testing.assert_allclose(out[t, hq], v[keys, h].mean(0), rtol=0, atol=1e-14)
        t += 1


def test_slot_order_duplicates_and_padding_do_not_matter():
    seqlens, h_k, g, d, block, topk = [130], 2, 1, 8, 16, 4
    n = sum(seqlens)
    sel = _random_sel(seqlens, h_k, block, topk, 19)
    q, k, v = _rand((n, h_k * g, d), 20), _rand((n, h_k, d), 21), _rand((n, h_k, d), 22)
    cu = make_cu_seqlens(seqlens)
    ref_out, ref_lse = oracle.fwd(cu, block, sel, q, k, v, 0.4)
    rng = np.random.default_rng(23)
    perm = np.stack([np.stack([rng.permutation(topk) for _ in range(n)]) for _ in range(h_k)])
    sel_p = np.take_along_axis(sel, perm, axis=-1)
    # append -1, a duplicate, a future block and an out-of-range block
    extra = np.stack([np.full((h_k, n), -1), sel_p[..., 0],
                      np.broadcast_to(np.arange(n) // block + 1, (h_k, n)),
                      np.full((h_k, n), 10 ** 6)], axis=-1).astype(np.int32)
    sel_x = np.concatenate([sel_p, extra], axis=-1)
    out, lse = oracle.fwd(cu, block, sel_x, q, k, v, 0.4)
    np.testing.assert_allclose(out, ref_out, rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, ref_lse, rtol=0, atol=1e-13)


def test_varlen_equals_separate_runs():
    seqlens, h_k, g, d, block, topk = [33, 96, 64], 1, 2, 8, 16, 3
    n = sum(seqlens)
    sel = _random_sel(seqlens, h_k, block, topk, 24)
    q, k, v = _rand((n, h_k * g, d), 25), _rand((n, h_k, d), 26), _rand((n, h_k, d), 27)
    out, lse = oracle.fwd(make_cu_seqlens(seqlens), block, sel, q, k, v, 0.6)
    base = 0
    for L in seqlens:
        sl = slice(base, base + L)
        o1, l1 = oracle.fwd(make_cu_seqlens([L]), block, np.ascontiguousarray(sel[:, sl]),
                            q[sl], k[sl], v[sl], 0.6)
        np.testing.assert_array_equal(out[sl], o1)
        np.testing.assert_array_equal(lse[:, sl], l1)
        base += L


def test_identical_query_heads_give_identical_outputs():
    seqlens, h_k, g, d, block, topk = [90], 2, 4, 8, 8, 4
    n = sum(seqlens)
    sel = _random_sel(seqlens, h_k, block, topk, 28)
    q1 = _rand((n, h_k, 1, d), 29)
    q = np.repeat(q1, g, axis=2).reshape(n, h_k * g, d)
    k, v = _rand((n, h_k, d), 30), _rand((n, h_k, d), 31)
    out, lse = oracle.fwd(make_cu_seqlens(seqlens), block, sel, q, k, v, 0.5)
    o = out.reshape(n, h_k, g, d)
    for j in range(1, g):
        np.testing.assert_array_equal(o[:, :, j], o[:, :, 0])


def test_empty_key_set():
    # A token that selects nothing valid: o = 0, lse = -inf.
    n, block, topk, d = 20, 4, 2, 4
    sel = np.full((1, n, topk), -1, dtype=np.int32)
    sel[0, :, 0] = np.arange(n) // block
    sel[0, 9] = [3, -1]          # future block only (c(9) = 2)
    q, k, v = _rand((n, 1, d), 32), _rand((n, 1, d), 33), _rand((n, 1, d), 34)
    out, lse = oracle.fwd(make_cu_seqlens([n]), block, sel, q, k, v, 1.0)
    assert np.all(out[9] == 0) and lse[0, 9] == -np.inf
    assert np.all(np.isfinite(np.delete(lse[0], 9)))


def test_hand_worked_example():
    """4 tokens, B_K = 2, d = 1, scale = 1, q = 1, k = ln w with w = (1, 2, 3, 4), v = 10 w.

    t0 selects {0}: keys {0};  t1 selects {0}: keys {0, 1};
    t2 selects {1, 0}: keys {0, 1, 2};  t3 selects {1}: keys {2, 3}.
    Softmax weights are w / sum(w), so out = 10 sum(w^2) / sum(w), lse = ln sum(w).
    """
    w = np.array([1.0, 2.0, 3.0, 4.0])
    q = np.ones((4, 1, 1))
    k = np.log(w).reshape(4, 1, 1)
    v = (10 * w).reshape(4, 1, 1)
    sel = np.array([[[0, -1], [0, -1], [1, 0], [1, -1]]], dtype=np.int32)
    out, lse = oracle.fwd(make_cu_seqlens([4]), 2, sel, q, k, v, 1.0)
    np.testing.assert_allclose(out[:, 0, 0], [10.0, 50 / 3, 70 / 3, 250 / 7], rtol=1e-15)
    np.testing.assert_allclose(lse[0], [0.0, math.log(3), math.log(6), math.log(7)], atol=1e-15)
    # Backward with dO = 1 (worked by hand: dS = P (v - out), dk_j = sum_t dS_tj, dq_t = sum_j dS_tj k_j)
    dq, dk, dv = oracle.bwd(make_cu_seqlens([4]), 2, sel, q, k, v, np.ones((4, 1, 1)), 1.0)
    np.testing.assert_allclose(dv[:, 0, 0], [3 / 2, 1.0, 13 / 14, 4 / 7], rtol=1e-14)
    np.testing.assert_allclose(dk[:, 0, 0], [-40 / 9, 10 / 9, 130 / 147, 120 / 49], rtol=1e-13)
    np.testing.assert_allclose(
        dq[:, 0, 0], [0.0, 20 / 9 * math.log(2), (30 * math.log(3) - 10 * math.log(2)) / 9,
                      120 / 49 * math.log(4 / 3)], rtol=1e-13, atol=1e-14)


def test_fwd_rows_matches_full_forward():
    cfg = CONFIGS["tiny"]
    inp = make_inputs(cfg)
    out, lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"], inp["k"],
                          inp["v"], cfg.scale)
    rng = np.random.default_rng(35)
    rows = np.stack([rng.integers(0, cfg.n, 50), rng.integers(0, cfg.h_q, 50)], axis=1)
    o, l = oracle.fwd_rows(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"], inp["k"],
                           inp["v"], cfg.scale, rows)
    np.testing.assert_array_equal(o, out[rows[:, 0], rows[:, 1]])
    np.testing.assert_array_equal(l, lse[rows[:, 1], rows[:, 0]])


def test_golden_regression_fixture():
    """Oracle output on a fixed tiny input, written by tests/golden/make_golden.py."""
    import json, os
    path = os.path.join(os.path.dirname(__file__), "golden", "oracle_small.json")
    with open(path) as f:
        gold = json.load(f)
    inp = gold["inputs"]
    q, k, v = (np.asarray(inp[x], dtype=np.float64) for x in ("q", "k", "v"))
    sel = np.asarray(inp["sel_idx"], dtype=np.int32)
    out, lse = oracle.fwd(np.asarray(inp["cu_seqlens"], np.int32), inp["block"], sel, q, k, v,
                          inp["scale"])
    np.testing.assert_allclose(out, np.asarray(gold["out"]), rtol=0, atol=1e-13)
    np.testing.assert_allclose(lse, np.asarray(gold["lse"]), rtol=0, atol=1e-13)
