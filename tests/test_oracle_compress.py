"""Pins for the oracle's compressed branch and block selection (CPU only).

The step that produces sel_idx: compression of keys and values over windows of
kernel_size positions every kernel_stride, attention over the compressed tokens,
block importance from those probabilities, and top-T selection with the init and
local blocks forced (Flash-Sparse-Attention README, "Usage -> Instantiate FSA
Module": kernel_size 32, kernel_stride 16, block_size 64, topk 16, init_blocks 1,
local_blocks 2).  Each function is pinned to something other than itself: closed
forms, torch SDPA (fp64) with an explicit mask, and brute-force constructions.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import compress as oc
from workloads import make_cu_seqlens


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def test_window_counts_by_enumeration():
    # C2 by brute force: every start position whose window fits
    for l, s in ((32, 16), (4, 2), (5, 3), (1, 1)):
        for length in range(0, 80):
            brute = sum(1 for a in range(0, length, s) if a + l <= length)
            assert oc.num_compressed(length, l, s) == brute
    cu = make_cu_seqlens([0, 31, 32, 47, 48, 100])
    assert oc.cmp_seqlens(cu, 32, 16).tolist() == [0, 0, 0, 1, 2, 4, 9]


def test_compress_constant_and_linear_keys():
    # C1: the mean of a constant is the constant; of k[t] = t it is a*stride + (l - 1)/2
    seqlens, h_k, d, l, s = [70, 40], 2, 3, 8, 4
    n = sum(seqlens)
    cu = make_cu_seqlens(seqlens)
    k = np.zeros((n, h_k, d))
    base = 0
    for L in seqlens:
        k[base:base + L] = np.arange(L)[:, None, None]
        base += L
    v = np.full((n, h_k, d), 2.5)
    kc, vc = oc.compress_kv(cu, k, v, l, s)
    cc = oc.cmp_seqlens(cu, l, s)
    for si, L in enumerate(seqlens):
        for i in range(oc.num_compressed(L, l, s)):
            np.testing.assert_allclose(kc[cc[si] + i], i * s + (l - 1) / 2, rtol=0, atol=1e-12)
    np.testing.assert_allclose(vc, 2.5, rtol=0, atol=1e-12)


def _masked_sdpa(q, kc, vc, seqlens, cc, l, s, scale):
    """C3/C4 by torch SDPA (fp64): per sequence, queries against its compressed tokens
    with the mask window_end <= tau; rows with nothing visible are left at 0."""
    h_q, h_k = q.shape[1], kc.shape[1]
    g = h_q // h_k
    out = np.zeros_like(q)
    base = 0
    for si, L in enumerate(seqlens):
        nc = int(cc[si + 1] - cc[si])
        if nc == 0:
            base += L
            continue
        tau = torch.arange(L)
        ends = torch.arange(nc) * s + l - 1
        mask = ends[None, :] <= tau[:, None]
        rows = mask.any(1)
        qs = torch.from_numpy(q[base:base + L]).permute(1, 0, 2).unsqueeze(0)
        ks = torch.from_numpy(kc[cc[si]:cc[si + 1]]).repeat_interleave(g, 1).permute(1, 0, 2)
        vs = torch.from_numpy(vc[cc[si]:cc[si + 1]]).repeat_interleave(g, 1).permute(1, 0, 2)
        o = F.scaled_dot_product_attention(qs[:, :, rows], ks.unsqueeze(0), vs.unsqueeze(0),
                                           attn_mask=mask[rows], scale=scale)
        out[base:base + L][rows.numpy()] = o.squeeze(0).permute(1, 0, 2).numpy()
        base += L
    return out


@pytest.mark.parametrize("l,s", [(32, 16), (8, 4), (5, 2)])
def test_cmp_attention_equals_masked_sdpa(l, s):
    seqlens, h_k, g, d = [130, 20, 77], 2, 3, 16
    n = sum(seqlens)
    cu = make_cu_seqlens(seqlens)
    q, k, v = _rand((n, h_k * g, d), 1), _rand((n, h_k, d), 2), _rand((n, h_k, d), 3)
    kc, vc = oc.compress_kv(cu, k, v, l, s)
    out, lse = oc.cmp_attn(cu, q, kc, vc, l, s, 0.3)
    ref = _masked_sdpa(q, kc, vc, seqlens, oc.cmp_seqlens(cu, l, s), l, s, 0.3)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)
    # rows that see no compressed token: out 0, lse -inf; all others finite
    base = 0
    for L in seqlens:
        for tau in range(L):
            assert np.isfinite(lse[:, base + tau]).all() == (tau >= l - 1)
        base += L


def test_unit_window_is_dense_causal_attention():
    # l = stride = 1: every key is its own compressed token, so C4 is causal attention
    seqlens, h_k, g, d = [40, 9], 1, 2, 8
    n = sum(seqlens)
    cu = make_cu_seqlens(seqlens)
    q, k, v = _rand((n, h_k * g, d), 4), _rand((n, h_k, d), 5), _rand((n, h_k, d), 6)
    kc, vc = oc.compress_kv(cu, k, v, 1, 1)
    out, _ = oc.cmp_attn(cu, q, kc, vc, 1, 1, 0.5)
    base = 0
    for L in seqlens:
        qs = torch.from_numpy(q[base:base + L]).permute(1, 0, 2)
        ks = torch.from_numpy(k[base:base + L]).repeat_interleave(g, 1).permute(1, 0, 2)
        vs = torch.from_numpy(v[base:base + L]).repeat_interleave(g, 1).permute(1, 0, 2)
        ref = F.scaled_dot_product_attention(qs, ks, vs, is_causal=True, scale=0.5)
        np.testing.assert_allclose(out[base:base + L], ref.permute(1, 0, 2).numpy(), rtol=0,
                                   atol=1e-12)
        base += L


def test_importance_uniform_probabilities_closed_form():
    # q = 0 gives every visible compressed token probability 1/nv, so the importance
    # of block j is g * (number of visible windows overlapping j) / nv, counted here
    # key by key
    L, h_k, g, d, l, s, B = 300, 2, 4, 8, 32, 16, 64
    cu = make_cu_seqlens([L])
    q = np.zeros((L, h_k * g, d))
    k, v = _rand((L, h_k, d), 7), _rand((L, h_k, d), 8)
    kc, vc = oc.compress_kv(cu, k, v, l, s)
    toks = [31, 47, 63, 64, 127, 200, 299]
    _, imps, _, _ = oc.select_rows(cu, q, kc, vc, l, s, 1.0, B, 4, 1, 2, toks)
    for t, imp in zip(toks, imps):
        nv = oc.visible(t, l, s)
        for j in range(t // B + 1):
            keys = set(range(j * B, j * B + B))
            cnt = sum(1 for i in range(nv) if keys & set(range(i * s, i * s + l)))
            np.testing.assert_allclose(imp[:, j], g * cnt / nv, rtol=0, atol=1e-12)
        # each probability lands once per block its window touches
        twice = sum(1 for i in range(nv) if (i * s) // B != (i * s + l - 1) // B)
        np.testing.assert_allclose(imp.sum(1), g * (nv + twice) / nv, rtol=0, atol=1e-12)


def _select_by_sort(imp_row, tau, B, T, init, local):
    """C6 built independently: forced blocks first, then a stable sort by -importance."""
    c = tau // B
    forced = sorted({j for j in range(c + 1) if j < init or j > c - local})
    rest = [j for j in range(c + 1) if j not in forced]
    order = np.lexsort((np.array(rest), -imp_row[rest])) if rest else []
    picked = (forced + [rest[i] for i in order])[:T]
    return picked + [-1] * (T - len(picked))


def test_select_topk_matches_sort_construction():
    rng = np.random.default_rng(9)
    B, T = 64, 6
    for tau in [0, 63, 64, 130, 700, 1500]:
        for init, local in ((1, 2), (0, 0), (3, 1), (2, 5)):
            nb = tau // B + 1
            imp = np.round(rng.random(nb), 1)      # rounded, so ties occur
            got = oc.select_topk(imp, tau, B, T, init, local)
            assert got.tolist() == _select_by_sort(imp, tau, B, T, init, local)


def test_selection_rows_are_valid_and_forced_blocks_present():
    seqlens, h_k, g, d, l, s, B, T = [600, 100], 2, 2, 16, 32, 16, 64, 5
    n = sum(seqlens)
    cu = make_cu_seqlens(seqlens)
    q, k, v = _rand((n, h_k * g, d), 10), _rand((n, h_k, d), 11), _rand((n, h_k, d), 12)
    kc, vc = oc.compress_kv(cu, k, v, l, s)
    toks = list(range(0, n, 7))
    sel, imps, _, _ = oc.select_rows(cu, q, kc, vc, l, s, 0.25, B, T, 1, 2, toks)
    for n_, t in enumerate(toks):
        tau = t - (0 if t < 600 else 600)
        c = tau // B
        for h in range(h_k):
            row = sel[h, n_]
            kept = row[row >= 0]
            assert len(set(kept.tolist())) == len(kept) == min(T, c + 1)
            assert all(0 <= j <= c for j in kept)
            assert set(oc.forced_blocks(tau, B, 1, 2)) <= set(kept.tolist())
            # every unselected causal block scores no higher than every selected
            # unforced one
            free = [j for j in kept if j not in oc.forced_blocks(tau, B, 1, 2)]
            other = [j for j in range(c + 1) if j not in kept]
            if free and other:
                assert imps[n_][h, free].min() >= imps[n_][h, other].max()
