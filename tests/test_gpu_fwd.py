"""GPU forward vs the fp64 oracle on the same seeded inputs (through the C ABI).

Every workload, the 64K one at g = 1, 2, 4, 8 and the varlen one included, is
compared element by element over the whole output and lse, in the launch
configuration the benchmark times."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_forward, sample_rows, to_device
from workloads import CONFIGS, WorkloadConfig, make_inputs

pytestmark = pytest.mark.gpu


def _run(cfg, inp):
    import block_sparse_attention_nsa_gb300 as nsa
    dv = to_device(inp)
    out, lse = nsa.fwd(dv["q"], dv["k"], dv["v"], dv["sel_idx"], dv["cu_seqlens"], cfg.block,
                       cfg.scale)
    torch.cuda.synchronize()
    return out, lse


@pytest.mark.parametrize("name", ["tiny", "fwd8k"])
def test_forward_full_compare(name):
    cfg = CONFIGS[name]
    inp = make_inputs(cfg)
    out, lse = _run(cfg, inp)
    ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                  inp["k"], inp["v"], cfg.scale)
    check_forward(out, lse, ref_out, ref_lse, name)


@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_forward_64k_full(g):
    # the 64K workload at every group size, in the benchmark's launch configuration,
    # compared element by element over the whole output and lse
    cfg = CONFIGS["fwd64k"].with_g(g)
    inp = make_inputs(cfg)
    out, lse = _run(cfg, inp)
    ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                  inp["k"], inp["v"], cfg.scale)
    check_forward(out, lse, ref_out, ref_lse, cfg.name)


def test_forward_varlen_full():
    cfg = CONFIGS["varlen"]
    inp = make_inputs(cfg)
    out, lse = _run(cfg, inp)
    ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                  inp["k"], inp["v"], cfg.scale)
    check_forward(out, lse, ref_out, ref_lse, "varlen")


def test_forward_64k_sampled_boundaries():
    # quick tier: sequence edges and block boundaries of the 64K workload at g = 4
    cfg = CONFIGS["fwd64k"].with_g(4)
    inp = make_inputs(cfg)
    out, lse = _run(cfg, inp)
    rows = sample_rows(cfg.n, cfg.h_q, 500, seed=4, block=cfg.block)
    ref_o, ref_l = oracle.fwd_rows(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                   inp["k"], inp["v"], cfg.scale, rows)
    check_forward(out[rows[:, 0], rows[:, 1]], lse[rows[:, 1], rows[:, 0]], ref_o, ref_l,
                  cfg.name)


@pytest.mark.parametrize("d", [64, 128, 256])
@pytest.mark.parametrize("block", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_forward_shapes_ragged(d, block, dtype):
    # several sequences with ragged tails, small T, g = 3 (rows not a multiple of 128)
    cfg = WorkloadConfig("ragged", (300, 1, 517, 64, 0, 250), 2, 3, d, block, 5, dtype,
                         "uniform", 1.0, 77)
    inp = make_inputs(cfg)
    if d == 128 and block == 128:
        import block_sparse_attention_nsa_gb300 as nsa
        with pytest.raises(nsa.NsaError) as e:      # outside the supported envelope
            _run(cfg, inp)
        assert e.value.code == 2
        return
    out, lse = _run(cfg, inp)
    ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                  inp["k"], inp["v"], cfg.scale)
    check_forward(out, lse, ref_out, ref_lse, f"d{d} B{block} {dtype}")


def test_forward_degenerate_selections():
    # rows with no valid block (-1 only, future blocks only), duplicates, T = 1 and T = 32
    for topk in (1, 32):
        cfg = WorkloadConfig("degen", (700, 129), 1, 2, 128, 64, topk, "bf16", "uniform", 1.0,
                             11 + topk)
        inp = make_inputs(cfg)
        sel = inp["sel_idx"]
        sel[0, 100, :] = -1
        sel[0, 5, 0] = 3                           # future block only
        sel[0, 600, :] = sel[0, 600, :1]           # all slots the same block
        out, lse = _run(cfg, inp)
        ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, sel, inp["q"], inp["k"],
                                      inp["v"], cfg.scale)
        check_forward(out, lse, ref_out, ref_lse, f"T={topk}")
        assert torch.all(out[100] == 0) and torch.isinf(lse[:, 100]).all()


def test_forward_dense_special_case_matches_sdpa():
    # every causal block selected: the kernel must equal dense causal attention
    n, block = 512, 64
    cfg = WorkloadConfig("dense", (n,), 2, 2, 128, block, n // block, "bf16", "uniform", 1.0, 3)
    inp = make_inputs(cfg)
    sel = np.full((2, n, n // block), -1, dtype=np.int32)
    for t in range(n):
        sel[:, t, : t // block + 1] = np.arange(t // block + 1)[::-1]
    inp["sel_idx"] = sel
    out, lse = _run(cfg, inp)
    ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], block, sel, inp["q"], inp["k"], inp["v"],
                                  cfg.scale)
    check_forward(out, lse, ref_out, ref_lse, "dense")


@pytest.mark.parametrize("which", ["64k_g16", "64k_d64_b128_t8"])
def test_forward_extended_sampled(which):
    # beyond the five workloads: g = 16 at 64K tokens, and the pages' (B_K, T) = (128, 8)
    # pair at d = 64; sampled rows against the oracle, the whole output finite
    import dataclasses
    base = CONFIGS["fwd64k"]
    cfg = base.with_g(16) if which == "64k_g16" else dataclasses.replace(
        base.with_g(4), d=64, block=128, topk=8, name="fwd64k_d64_b128_t8")
    inp = make_inputs(cfg)
    out, lse = _run(cfg, inp)
    assert torch.isfinite(out).all() and torch.isfinite(lse).all()
    rows = sample_rows(cfg.n, cfg.h_q, 400, seed=16, block=cfg.block)
    ref_o, ref_l = oracle.fwd_rows(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                   inp["k"], inp["v"], cfg.scale, rows)
    check_forward(out[rows[:, 0], rows[:, 1]], lse[rows[:, 1], rows[:, 0]], ref_o, ref_l,
                  cfg.name)
