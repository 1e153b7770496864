"""fp64 CPU oracle for the step before selected attention -- TEST INFRASTRUCTURE ONLY.

The compressed branch and the block selection that produce ``sel_idx``: Native
Sparse Attention's compression, selection and sliding-window branches (papernotes
page, 研究背景与动机 "领域现状"; its 方法详解 flowchart takes the NSA selection
tensor T as input), with the hyperparameters of the Flash-Sparse-Attention README's
"Usage -> Instantiate FSA Module" example: kernel_size = 32, kernel_stride = 16,
block_size = 64, topk = 16, init_blocks = 1, local_blocks = 2.

The pages name these parameters but define no formula, so this module takes the
plainest reading of each step (numbered as in the design notes):
  C1  compression is the mean of the window's keys (values): the weight-free case
      of the learned compression, whose weights no page gives;
  C2  compressed token i of a sequence covers positions [i*stride, i*stride + l)
      and exists when that window lies inside the sequence;
  C3  the query at position tau sees compressed token i when the window ends at
      or before it: i*stride + l - 1 <= tau;
  C4  compressed attention is softmax(scale * q . kc) over the visible compressed
      tokens, times vc; with none visible, out = 0 and lse = -inf;
  C5  the importance of selection block j (keys [j*B, j*B + B)) for a (KV head,
      token) is the sum, over the group's g query heads and over the visible
      compressed tokens whose window overlaps those keys, of their probability;
  C6  top-T among the causal blocks j <= tau // B: the init blocks (j < init) and
      the local blocks (c - local + 1 .. c, c = tau // B) are always kept and come
      first, ascending; then the others by importance, larger first, ties to the
      lower block; slots left over are -1.

Plain numpy in fp64, loops over tokens; only ``tests/`` may import it.  Parity
status: pinned -- compression by closed forms (constant and linear keys) and a
brute-force window enumeration; compressed attention by torch SDPA (fp64) with
an explicit visibility mask, and l = stride = 1 equals dense causal attention;
importance by the uniform-probability closed form and a key-level brute force;
selection by an independent sort-based construction.
"""
from __future__ import annotations

import numpy as np


def num_compressed(length: int, kernel_size: int, stride: int) -> int:
    """C2: windows [i*stride, i*stride + l) that fit in a sequence of `length`."""
    if length < kernel_size:
        return 0
    return (length - kernel_size) // stride + 1


def cmp_seqlens(cu_seqlens, kernel_size: int, stride: int) -> np.ndarray:
    """Offsets of each sequence's compressed tokens in the packed compressed rows."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    out = np.zeros(len(cu), dtype=np.int32)
    for s in range(len(cu) - 1):
        out[s + 1] = out[s] + num_compressed(int(cu[s + 1] - cu[s]), kernel_size, stride)
    return out


def compress_kv(cu_seqlens, k, v, kernel_size: int, stride: int):
    """C1/C2: kc[r, h] = mean of k over the r-th window, likewise vc; fp64.

    k, v: [N, h_k, d].  Returns kc, vc: [N_c, h_k, d] with the compressed tokens of
    sequence s at rows cu_cmp[s] .. cu_cmp[s + 1] - 1."""
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = cmp_seqlens(cu, kernel_size, stride)
    kc = np.zeros((int(cc[-1]),) + k.shape[1:], dtype=np.float64)
    vc = np.zeros_like(kc)
    for s in range(len(cu) - 1):
        for i in range(int(cc[s + 1] - cc[s])):
            a = int(cu[s]) + i * stride
            kc[cc[s] + i] = k[a:a + kernel_size].mean(axis=0)
            vc[cc[s] + i] = v[a:a + kernel_size].mean(axis=0)
    return kc, vc


def visible(tau: int, kernel_size: int, stride: int) -> int:
    """C3: how many compressed tokens the query at position tau sees."""
    if tau < kernel_size - 1:
        return 0
    return (tau - kernel_size + 1) // stride + 1


def _seq_of(cu, t):
    return int(np.searchsorted(cu, t, side="right") - 1)


def cmp_attn_rows(cu_seqlens, q, kc, vc, kernel_size: int, stride: int, scale: float, tokens):
    """C4 for the listed tokens: out [len(tokens), h_q, d], lse [len(tokens), h_q] and
    the probabilities of each token's visible compressed tokens (list of [h_q, nv])."""
    q = np.asarray(q, dtype=np.float64)
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    cc = cmp_seqlens(cu, kernel_size, stride)
    h_q, d = q.shape[1], q.shape[2]
    h_k = kc.shape[1]
    g = h_q // h_k
    outs = np.zeros((len(tokens), h_q, d))
    lses = np.full((len(tokens), h_q), -np.inf)
    probs = []
    for n, t in enumerate(tokens):
        s = _seq_of(cu, t)
        nv = visible(int(t - cu[s]), kernel_size, stride)
        p_t = np.zeros((h_q, nv))
        for hq in range(h_q):
            if nv == 0:
                continue
            keys = kc[cc[s]:cc[s] + nv, hq // g]
            vals = vc[cc[s]:cc[s] + nv, hq // g]
            sc = scale * (keys @ q[t, hq])
            m = sc.max()
            e = np.exp(sc - m)
            z = e.sum()
            p = e / z
            outs[n, hq] = p @ vals
            lses[n, hq] = m + np.log(z)
            p_t[hq] = p
        probs.append(p_t)
    return outs, lses, probs


def cmp_attn(cu_seqlens, q, kc, vc, kernel_size: int, stride: int, scale: float):
    """C4 for every token: out [N, h_q, d] and lse [h_q, N] (the selected path's layouts)."""
    n = np.asarray(q).shape[0]
    out, lse, _ = cmp_attn_rows(cu_seqlens, q, kc, vc, kernel_size, stride, scale, range(n))
    return out, lse.T.copy()


def block_importance(probs_t, tau: int, h_k: int, block: int, kernel_size: int, stride: int):
    """C5 for one token: [h_k, c + 1] importance of its causal blocks, c = tau // B.

    probs_t: [h_q, nv] probabilities of the token's visible compressed tokens."""
    h_q, nv = probs_t.shape
    g = h_q // h_k
    nb = tau // block + 1
    imp = np.zeros((h_k, nb))
    for i in range(nv):
        a, b = i * stride, i * stride + kernel_size      # the window's keys [a, b)
        w = probs_t[:, i].reshape(h_k, g).sum(axis=1)    # summed over each group's heads
        for j in range(a // block, (b - 1) // block + 1):  # the blocks holding those keys
            imp[:, j] += w
    return imp


def forced_blocks(tau: int, block: int, init_blocks: int, local_blocks: int):
    """C6: the blocks kept whatever their importance, ascending."""
    c = tau // block
    keep = set(range(min(init_blocks, c + 1)))
    keep.update(j for j in range(c - local_blocks + 1, c + 1) if j >= 0)
    return sorted(keep)


def select_topk(imp_row, tau: int, block: int, topk: int, init_blocks: int, local_blocks: int):
    """C6 for one (KV head, token): topk block ids, forced ones first, -1 padded."""
    forced = forced_blocks(tau, block, init_blocks, local_blocks)
    chosen = list(forced[:topk])
    taken = set(chosen)
    while len(chosen) < topk:
        best = -1
        for j in range(tau // block + 1):   # ascending, so ties keep the lower block
            if j in taken:
                continue
            if best < 0 or imp_row[j] > imp_row[best]:
                best = j
        if best < 0:
            break
        chosen.append(best)
        taken.add(best)
    return np.array(chosen + [-1] * (topk - len(chosen)), dtype=np.int32)


def select_rows(cu_seqlens, q, kc, vc, kernel_size, stride, scale, block, topk, init_blocks,
                local_blocks, tokens):
    """C4-C6 for the listed tokens: sel [h_k, len(tokens), topk] and importance rows
    (list of [h_k, c + 1]), with the compressed attention's out and lse."""
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    h_k = kc.shape[1]
    out, lse, probs = cmp_attn_rows(cu, q, kc, vc, kernel_size, stride, scale, tokens)
    sel = np.full((h_k, len(tokens), topk), -1, dtype=np.int32)
    imps = []
    for n, t in enumerate(tokens):
        tau = int(t - cu[_seq_of(cu, t)])
        imp = block_importance(probs[n], tau, h_k, block, kernel_size, stride)
        imps.append(imp)
        for h in range(h_k):
            sel[h, n] = select_topk(imp[h], tau, block, topk, init_blocks, local_blocks)
    return sel, imps, out, lse
