"""nsa_sel_attn_step_host: the host-buffer step (the bench's end-to-end call).

It copies the inputs in, runs forward and backward, and copies the results back,
with dout and out/lse on a side stream that overlaps the compute.  Its results must
equal, bit for bit, those of the device-side nsa_sel_attn_fwd + nsa_sel_attn_bwd on
the same inputs (the same kernels run), on consecutive calls; and the fp64 oracle's
within the forward and backward tolerances.
"""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_forward, rel_l2, GRAD_REL_L2, to_device
from workloads import CONFIGS, WorkloadConfig, make_inputs

pytestmark = pytest.mark.gpu


def _device_step(nsa, cfg, d):
    ws = nsa.alloc_workspace(nsa.make_dims(len(cfg.seqlens), cfg.n, cfg.h_q, cfg.h_k, cfg.d,
                                           cfg.block, cfg.topk, d["q"].dtype))
    out, lse = nsa.fwd(d["q"], d["k"], d["v"], d["sel_idx"], d["cu_seqlens"], cfg.block,
                       cfg.scale, workspace=ws)
    dq, dk, dv = nsa.bwd(d["q"], d["k"], d["v"], d["sel_idx"], d["cu_seqlens"], cfg.block,
                         cfg.scale, out, lse, d["dout"], workspace=ws, index_ready=True)
    torch.cuda.synchronize()
    return out, lse, dq, dk, dv


@pytest.mark.parametrize("name", ["tiny", "ragged"])
def test_step_host_equals_device_step(name):
    import block_sparse_attention_nsa_gb300 as nsa
    cfg = CONFIGS["tiny"] if name == "tiny" else WorkloadConfig(
        "ragged_step", (300, 1, 517, 64, 250), 2, 3, 128, 64, 5, "bf16", "uniform", 1.0, 61)
    inp = make_inputs(cfg, with_dout=True)
    d = to_device(inp)
    ref = _device_step(nsa, cfg, d)
    dims = nsa.make_dims(len(cfg.seqlens), cfg.n, cfg.h_q, cfg.h_k, cfg.d, cfg.block, cfg.topk,
                         d["q"].dtype)
    pin = lambda t: t.contiguous().pin_memory()
    host = {"q": pin(inp["q"]), "k": pin(inp["k"]), "v": pin(inp["v"]),
            "dout": pin(inp["dout"]),
            "sel_idx": pin(torch.from_numpy(np.ascontiguousarray(inp["sel_idx"]))),
            "cu_seqlens": pin(torch.from_numpy(np.ascontiguousarray(inp["cu_seqlens"])))}
    staging = torch.empty(nsa.staging_size(dims), dtype=torch.uint8, device="cuda")
    ws = nsa.alloc_workspace(dims)
    for call in range(2):
        for key, like in (("out", "q"), ("dq", "q"), ("dk", "k"), ("dv", "v")):
            host[key] = torch.full_like(host[like], float("nan")).pin_memory()
        host["lse"] = torch.full((cfg.h_q, cfg.n), float("nan"), dtype=torch.float32).pin_memory()
        nsa.step_host(dims, host, cfg.scale, staging, ws)
        for key, r in zip(("out", "lse", "dq", "dk", "dv"), ref):
            got = host[key]
            assert torch.equal(got.view(torch.int16) if got.dtype != torch.float32 else got,
                               (r.cpu().view(torch.int16) if r.dtype != torch.float32
                                else r.cpu())), f"{name} call {call}: {key} differs"
    ref_out, ref_lse = oracle.fwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                  inp["k"], inp["v"], cfg.scale)
    check_forward(host["out"], host["lse"], ref_out, ref_lse, name)
    gq, gk, gv = oracle.bwd(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"], inp["k"],
                            inp["v"], inp["dout"], cfg.scale)
    for key, r in (("dq", gq), ("dk", gk), ("dv", gv)):
        assert rel_l2(host[key], r) <= GRAD_REL_L2, key
