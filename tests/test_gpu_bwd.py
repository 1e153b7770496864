"""GPU backward vs the fp64 oracle's backward (direct differentiation), through
the C ABI.  dQ, dK, dV within relative L2 2e-2 over the whole tensor."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import GRAD_REL_L2, rel_l2, to_device
from workloads import CONFIGS, WorkloadConfig, make_inputs

pytestmark = pytest.mark.gpu


def _run(cfg, inp, index_ready=True):
    import block_sparse_attention_nsa_gb300 as nsa
    d = to_device(inp)
    dims = nsa.make_dims(len(cfg.seqlens), cfg.n, cfg.h_q, cfg.h_k, cfg.d, cfg.block, cfg.topk,
                         d["q"].dtype)
    ws = nsa.alloc_workspace(dims)
    out, lse = nsa.fwd(d["q"], d["k"], d["v"], d["sel_idx"], d["cu_seqlens"], cfg.block,
                       cfg.scale, workspace=ws)
    if not index_ready:
        ws.zero_()           # nothing left from the forward: the backward rebuilds its index
    dq, dk, dv = nsa.bwd(d["q"], d["k"], d["v"], d["sel_idx"], d["cu_seqlens"], cfg.block,
                         cfg.scale, out, lse, d["dout"], workspace=ws, index_ready=index_ready)
    code, bits = nsa.get_status(dims, ws)
    assert code == 0, bits
    return dq, dk, dv


def _check(cfg, inp, grads):
    ref = oracle.bwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"], inp["k"], inp["v"],
                     inp["dout"], cfg.scale)
    for name, got, r in zip(("dq", "dk", "dv"), grads, ref):
        assert torch.isfinite(got).all(), name
        err = rel_l2(got, r)
        assert err <= GRAD_REL_L2, f"{cfg.name} {name}: rel-L2 {err:.3e}"


@pytest.mark.parametrize("block", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_backward_small_ragged(block, dtype):
    cfg = WorkloadConfig("bwd_small", (300, 1, 517, 64, 250), 2, 3, 128, block, 5, dtype,
                         "uniform", 1.0, 5, with_dout=True)
    inp = make_inputs(cfg)
    _check(cfg, inp, _run(cfg, inp))


def test_backward_rebuilds_index():
    cfg = WorkloadConfig("bwd_noidx", (700, 129), 2, 2, 128, 64, 6, "bf16", "uniform", 1.0, 6,
                         with_dout=True)
    inp = make_inputs(cfg)
    _check(cfg, inp, _run(cfg, inp, index_ready=False))


def test_backward_degenerate_selections():
    cfg = WorkloadConfig("bwd_degen", (700, 129), 1, 2, 128, 64, 4, "bf16", "uniform", 1.0, 12,
                         with_dout=True)
    inp = make_inputs(cfg)
    sel = inp["sel_idx"]
    sel[0, 100, :] = -1                 # no key at all: zero gradient for that query
    sel[0, 600, :] = sel[0, 600, :1]    # duplicates
    dq, dk, dv = _run(cfg, inp)
    _check(cfg, inp, (dq, dk, dv))
    assert torch.all(dq[100] == 0)


def test_backward_bwd32k_full():
    cfg = CONFIGS["bwd32k"]
    inp = make_inputs(cfg)
    _check(cfg, inp, _run(cfg, inp))
