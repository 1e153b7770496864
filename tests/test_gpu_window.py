"""Sliding-window branch and gated combination on the GPU against the fp64 oracle.

The window runs on the selected-attention kernels: nsa_sel_attn_window_select writes
the window's block selection (compared bit for bit with the oracle's), and
nsa_sel_attn_fwd_window / _bwd_window add the window's lower key bound to the causal
mask.  The gated combination is the gate-weighted sum of the branch outputs.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import GRAD_REL_L2, check_forward, rel_l2, to_device
from workloads import WorkloadConfig, make_inputs

pytestmark = pytest.mark.gpu


def _case(d, block, window, dtype, seqlens, seed):
    topk = (window - 1 + block - 1) // block + 1
    cfg = WorkloadConfig("window", tuple(seqlens), 2, 2, d, block, topk, dtype, "uniform", 1.0,
                         seed)
    inp = make_inputs(cfg, with_dout=True)
    sel = oracle.window_select(inp["cu_seqlens"], cfg.h_k, block, topk, window)
    inp["sel_idx"] = sel
    return cfg, inp


@pytest.mark.parametrize("d,block,window,dtype", [(128, 64, 512, "bf16"), (64, 32, 100, "fp16"),
                                                  (128, 32, 33, "bf16"), (256, 64, 200, "bf16"),
                                                  (64, 128, 300, "bf16")])
def test_window_forward_and_selection(d, block, window, dtype):
    import block_sparse_attention_nsa_gb300 as nsa
    cfg, inp = _case(d, block, window, dtype, [1000, 3, 700, 2049], 90 + d + block)
    dv = to_device(inp)
    sel_gpu = nsa.window_select(dv["cu_seqlens"], cfg.n, cfg.h_k, block, cfg.topk, window)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(sel_gpu.cpu().numpy(), inp["sel_idx"])
    out, lse = nsa.fwd_window(dv["q"], dv["k"], dv["v"], sel_gpu, dv["cu_seqlens"], block,
                              cfg.scale, window)
    torch.cuda.synchronize()
    ref_o, ref_l = oracle.fwd(inp["cu_seqlens"], block, inp["sel_idx"], inp["q"], inp["k"],
                              inp["v"], cfg.scale, window=window)
    check_forward(out, lse, ref_o, ref_l, f"window d{d} B_K{block} W{window}")


@pytest.mark.parametrize("d,block,window,dtype", [(128, 64, 512, "bf16"), (64, 32, 100, "fp16"),
                                                  (256, 32, 90, "bf16")])
def test_window_backward(d, block, window, dtype):
    import block_sparse_attention_nsa_gb300 as nsa
    cfg, inp = _case(d, block, window, dtype, [900, 1, 1200], 190 + d)
    dv = to_device(inp)
    sel = torch.from_numpy(inp["sel_idx"]).cuda()
    ws = nsa.alloc_workspace(nsa.make_dims(len(cfg.seqlens), cfg.n, cfg.h_q, cfg.h_k, d, block,
                                           cfg.topk, dv["q"].dtype))
    out, lse = nsa.fwd_window(dv["q"], dv["k"], dv["v"], sel, dv["cu_seqlens"], block,
                              cfg.scale, window, workspace=ws)
    dq, dk, dvv = nsa.bwd_window(dv["q"], dv["k"], dv["v"], sel, dv["cu_seqlens"], block,
                                 cfg.scale, window, out, lse, dv["dout"], workspace=ws,
                                 index_ready=True)
    torch.cuda.synchronize()
    gq, gk, gv = oracle.bwd(inp["cu_seqlens"], block, inp["sel_idx"], inp["q"], inp["k"],
                            inp["v"], inp["dout"], cfg.scale, window=window)
    for name, got, ref in (("dq", dq, gq), ("dk", dk, gk), ("dv", dvv, gv)):
        err = rel_l2(got, ref)
        assert err <= GRAD_REL_L2, f"{name} rel-L2 {err:.3e}"


def test_window_select_rejects_small_topk():
    import block_sparse_attention_nsa_gb300 as nsa
    cu = torch.tensor([0, 100], dtype=torch.int32, device="cuda")
    with pytest.raises(nsa.NsaError) as e:
        nsa.window_select(cu, 100, 1, 32, 2, 70)       # 4 blocks needed
    assert e.value.code == 1


@pytest.mark.parametrize("nbr,d,dtype", [(3, 128, torch.bfloat16), (2, 64, torch.float16),
                                         (1, 256, torch.bfloat16)])
def test_gate_combine(nbr, d, dtype):
    import block_sparse_attention_nsa_gb300 as nsa
    g = torch.Generator().manual_seed(nbr * d)
    N, h_q = 1537, 6
    br = [torch.randn(N, h_q, d, generator=g).to(dtype) for _ in range(nbr)]
    gates = torch.rand(N, h_q, nbr, generator=g)
    dout = torch.randn(N, h_q, d, generator=g).to(dtype)
    out = nsa.gate_combine([b.cuda() for b in br], gates.cuda())
    dbr, dg = nsa.gate_combine_bwd([b.cuda() for b in br], gates.cuda(), dout.cuda())
    torch.cuda.synchronize()
    ref = oracle.gate_combine(br, gates)
    ref_dbr, ref_dg = oracle.gate_combine_bwd(br, gates, dout)
    assert np.abs(out.float().cpu().numpy() - ref).max() <= 2e-2
    for got, r in zip(dbr, ref_dbr):
        assert np.abs(got.float().cpu().numpy() - r).max() <= 2e-2
    np.testing.assert_allclose(dg.cpu().numpy(), ref_dg, rtol=1e-4, atol=1e-3)
