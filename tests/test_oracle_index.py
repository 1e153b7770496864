"""Pins for the oracle's index tensors (I_i = the tokens that selected KV block i,
O_i = the compact-buffer position of each kept (token, slot) pair; "FSA: An
Alternative Efficient Implementation of Native Sparse Attention Kernel", key
design 2).  CPU only."""
import numpy as np

import oracle
from workloads import CONFIGS, keys_attended, make_cu_seqlens, make_inputs, make_selection


def _brute_force(cu, block, sel):
    """Dictionary-of-lists construction straight from the definition."""
    h_k, n, topk = sel.shape
    seqs = [(int(cu[s]), int(cu[s + 1])) for s in range(len(cu) - 1)]
    nblk = [(b - a + block - 1) // block for a, b in seqs]
    start = np.concatenate([[0], np.cumsum(nblk)])
    lists = {}
    kept = {}
    for h in range(h_k):
        for s, (a, b) in enumerate(seqs):
            for t in range(a, b):
                tau = t - a
                seen = set()
                for kk in range(topk):
                    blk = int(sel[h, t, kk])
                    if 0 <= blk <= tau // block and blk < nblk[s] and blk not in seen:
                        seen.add(blk)
                        lists.setdefault((h, int(start[s]) + blk), []).append(t)
                        kept[(h, t, kk)] = (h, int(start[s]) + blk)
    nb = int(start[-1])
    counts = np.zeros(h_k * nb, np.int32)
    for (h, gb), lst in lists.items():
        counts[h * nb + gb] = len(lst)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    q_list = np.zeros(int(offsets[-1]), np.int32)
    for (h, gb), lst in lists.items():
        q_list[offsets[h * nb + gb]:offsets[h * nb + gb] + len(lst)] = sorted(lst)
    slot_map = np.full(sel.shape, -1, np.int32)
    for (h, t, kk), (_, gb) in kept.items():
        seg = q_list[offsets[h * nb + gb]:offsets[h * nb + gb + 1]]
        slot_map[h, t, kk] = offsets[h * nb + gb] + int(np.searchsorted(seg, t))
    return counts, offsets, q_list, slot_map, nb


def test_index_matches_brute_force_with_edge_cases():
    seqlens, h_k, block, topk = [37, 64, 5, 90], 3, 8, 5
    rng = np.random.default_rng(0)
    sel = make_selection(seqlens, h_k, block, topk, "uniform", rng)
    n = sum(seqlens)
    # sprinkle duplicates, -1, future blocks, out-of-range values and negatives
    for _ in range(200):
        h, t, kk = rng.integers(h_k), rng.integers(n), rng.integers(topk)
        sel[h, t, kk] = rng.choice([-1, -5, 0, 1, 2, 3, 11, 10 ** 6, sel[h, t, 0]])
    cu = make_cu_seqlens(seqlens)
    got = oracle.index(cu, block, sel)
    counts, offsets, q_list, slot_map, nb = _brute_force(cu, block, sel)
    assert got["num_blocks"] == nb
    np.testing.assert_array_equal(got["counts"], counts)
    np.testing.assert_array_equal(got["offsets"], offsets)
    np.testing.assert_array_equal(got["q_list"], q_list)
    np.testing.assert_array_equal(got["slot_map"], slot_map)


def _check_invariants(cu, block, sel, idx):
    h_k, n, topk = sel.shape
    counts, offsets, q_list, slot_map = idx["counts"], idx["offsets"], idx["q_list"], idx["slot_map"]
    np.testing.assert_array_equal(offsets[1:] - offsets[:-1], counts)
    assert offsets[0] == 0 and offsets[-1] == q_list.size
    for i in range(counts.size):
        seg = q_list[offsets[i]:offsets[i + 1]]
        assert np.all(np.diff(seg) > 0)               # strictly ascending tokens
    kept = slot_map >= 0
    h_idx, t_idx, _ = np.nonzero(kept)
    np.testing.assert_array_equal(q_list[slot_map[kept]], t_idx)   # q_list[slot_map] = t
    assert np.unique(slot_map[kept]).size == q_list.size           # a bijection onto positions


def test_index_invariants_on_configs():
    for name in ("tiny", "fwd8k"):
        cfg = CONFIGS[name]
        inp = make_inputs(cfg)
        idx = oracle.index(inp["cu_seqlens"], cfg.block, inp["sel_idx"])
        _check_invariants(inp["cu_seqlens"], cfg.block, inp["sel_idx"], idx)


def test_pair_count_closed_form():
    # Under the synthetic rule every token keeps min(T, c(t) + 1) distinct blocks.
    for seqlens, block, topk in (([256], 32, 4), ([1000, 333, 64], 64, 16), ([4096], 64, 16)):
        sel = make_selection(seqlens, 2, block, topk, "distance", np.random.default_rng(1))
        idx = oracle.index(make_cu_seqlens(seqlens), block, sel)
        per_tok = []
        for L in seqlens:
            c = np.arange(L) // block
            per_tok.append(np.minimum(topk, c + 1))
        expect = 2 * int(np.concatenate(per_tok).sum())
        assert idx["q_list"].size == expect
        # n(t) of the rule (used for useful-FLOP counts) equals |K(t)| = exp(lse) at q = 0
        n = sum(seqlens)
        rng = np.random.default_rng(2)
        k, v = rng.standard_normal((n, 2, 4)), rng.standard_normal((n, 2, 4))
        _, lse = oracle.fwd(make_cu_seqlens(seqlens), block, sel, np.zeros((n, 2, 4)), k, v, 1.0)
        n_t = keys_attended(seqlens, block, topk)
        np.testing.assert_allclose(np.exp(lse), np.broadcast_to(n_t, (2, n)), rtol=1e-12)
