"""GPU index builder vs the oracle's index tensors: bit-exact (counts, offsets,
I_i = q_list, O_i = slot_map) on every workload and on edge cases."""
import numpy as np
import pytest
import torch

import oracle
from workloads import CONFIGS, make_cu_seqlens, make_selection

pytestmark = pytest.mark.gpu


def _gpu_index(sel, cu, block, h_q_per_k=1, d=128, dtype=torch.bfloat16):
    import block_sparse_attention_nsa_gb300 as nsa
    h_k, n, topk = sel.shape
    dims = nsa.make_dims(len(cu) - 1, n, h_k * h_q_per_k, h_k, d, block, topk, dtype)
    ws = nsa.alloc_workspace(dims)
    s = torch.from_numpy(np.ascontiguousarray(sel)).cuda()
    c = torch.from_numpy(np.ascontiguousarray(cu)).cuda()
    nsa.index(s, c, block, dims, ws)
    view = nsa.index_view(dims, ws)
    code, bits = nsa.get_status(dims, ws)
    return view, code, bits


def _assert_same(view, ref):
    assert view["num_blocks"] == ref["num_blocks"]
    np.testing.assert_array_equal(view["counts"].cpu().numpy(), ref["counts"])
    np.testing.assert_array_equal(view["offsets"].cpu().numpy(), ref["offsets"])
    np.testing.assert_array_equal(view["q_list"].cpu().numpy(), ref["q_list"])
    np.testing.assert_array_equal(view["slot_map"].cpu().numpy(), ref["slot_map"])


@pytest.mark.parametrize("name", ["tiny", "fwd8k", "fwd64k", "varlen", "bwd32k"])
def test_index_bit_exact_on_workloads(name):
    cfg = CONFIGS[name]
    rng = np.random.default_rng(cfg.seed)
    sel = make_selection(cfg.seqlens, cfg.h_k, cfg.block, cfg.topk, cfg.rule, rng)
    cu = make_cu_seqlens(cfg.seqlens)
    view, code, bits = _gpu_index(sel, cu, cfg.block, cfg.g, cfg.d)
    assert code == 0 and bits == 0
    _assert_same(view, oracle.index(cu, cfg.block, sel))


@pytest.mark.parametrize("topk", [1, 3, 16, 32])
@pytest.mark.parametrize("block", [32, 128])
def test_index_edge_cases(topk, block):
    seqlens = [0, 37, 300, 1, 0, 129, 513]          # empty and ragged sequences
    h_k = 3
    n = sum(seqlens)
    rng = np.random.default_rng(topk * 1000 + block)
    sel = make_selection(seqlens, h_k, block, topk, "uniform", rng)
    for _ in range(400):                            # duplicates, -1, future, out of range
        h, t, k = rng.integers(h_k), rng.integers(n), rng.integers(topk)
        sel[h, t, k] = rng.choice([-1, 0, 1, 2, 3, 5, sel[h, t, 0]])
    cu = make_cu_seqlens(seqlens)
    view, code, bits = _gpu_index(sel, cu, block)
    _assert_same(view, oracle.index(cu, block, sel))
    # values -1 .. last block of the token's sequence are legal; others raise bit 1
    nblk = np.concatenate([np.full(L, (L + block - 1) // block) for L in seqlens])
    illegal = bool(np.any((sel < -1) | (sel >= nblk[None, :, None])))
    assert bits == (1 if illegal else 0) and code == (5 if illegal else 0)


def test_index_flags_out_of_range_values():
    seqlens, block, topk = [200, 100], 32, 4
    sel = make_selection(seqlens, 1, block, topk, "uniform", np.random.default_rng(5))
    sel[0, 10, 3] = -7
    sel[0, 250, 2] = 99
    cu = make_cu_seqlens(seqlens)
    view, code, bits = _gpu_index(sel, cu, block)
    assert code == 5 and (bits & 1)
    _assert_same(view, oracle.index(cu, block, sel))
