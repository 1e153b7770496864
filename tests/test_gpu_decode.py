"""One-step decode (nsa_sel_attn_decode) against the fp64 oracle.

The decode query of a sequence is its last cached token.  The oracle computes the
forward for exactly those (token, query head) rows of the packed batch, so both sides
see the same inputs: q of the last tokens, the whole caches, and the last tokens'
selection rows.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_forward
from workloads import CONFIGS, WorkloadConfig, make_inputs

pytestmark = pytest.mark.gpu


def _decode_case(cfg):
    import block_sparse_attention_nsa_gb300 as nsa
    inp = make_inputs(cfg)
    cu = np.asarray(inp["cu_seqlens"], dtype=np.int64)
    last = cu[1:] - 1                                   # last token of every sequence
    live = cu[1:] > cu[:-1]
    assert live.all()
    q_dec = inp["q"][torch.from_numpy(last)].contiguous().cuda()             # [B, h_q, d]
    sel_dec = np.ascontiguousarray(inp["sel_idx"][:, last, :])              # [h_k, B, T]
    k, v = inp["k"].cuda(), inp["v"].cuda()
    cu_d = torch.from_numpy(np.ascontiguousarray(inp["cu_seqlens"])).cuda()
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = nsa.decode(q_dec, k, v, torch.from_numpy(sel_dec).cuda(), cu_d, cfg.block,
                          cfg.scale, device_status=status)
    torch.cuda.synchronize()
    rows = np.stack([np.repeat(last, cfg.h_q), np.tile(np.arange(cfg.h_q), len(last))], axis=1)
    ref_o, ref_l = oracle.fwd_rows(inp["cu_seqlens"], cfg.block, inp["sel_idx"], inp["q"],
                                   inp["k"], inp["v"], cfg.scale, rows)
    return out, lse, ref_o, ref_l, status, inp, last


@pytest.mark.parametrize("d,block,g,dtype", [(128, 64, 4, "bf16"), (128, 64, 16, "bf16"),
                                             (64, 32, 2, "fp16"), (128, 128, 1, "bf16"),
                                             (64, 128, 8, "fp16")])
def test_decode_matches_oracle(d, block, g, dtype):
    cfg = WorkloadConfig("decode", (1000, 4097, 64, 1, 2500, 777), 2, g, d, block, 16, dtype,
                         "uniform", 1.0, 77 + g)
    out, lse, ref_o, ref_l, status, _, last = _decode_case(cfg)
    B, h_q = len(last), cfg.h_q
    check_forward(out.reshape(B * h_q, d), lse.t().reshape(B * h_q), ref_o, ref_l,
                  f"decode d{d} B_K{block} g{g}")
    assert int(status.item()) == 0


def test_decode_distance_rule_64k_cache():
    # the 64K workload's distance-rule selection, decoding the last token of a 64K cache
    cfg = dataclasses.replace(CONFIGS["fwd64k"].with_g(4), seqlens=(16384, 32768, 8192, 8192),
                              name="decode_64k")
    out, lse, ref_o, ref_l, status, _, last = _decode_case(cfg)
    check_forward(out.reshape(-1, cfg.d), lse.t().reshape(-1), ref_o, ref_l, "decode 64k")
    assert int(status.item()) == 0


def test_decode_flags_bad_selection_and_handles_empty():
    import block_sparse_attention_nsa_gb300 as nsa
    h_k, g, d, blk, T = 1, 2, 64, 32, 4
    lens = [100, 0, 40]
    cu = torch.tensor([0, 100, 100, 140], dtype=torch.int32, device="cuda")
    torch.manual_seed(3)
    q = torch.randn(3, h_k * g, d, device="cuda").to(torch.bfloat16)
    k = torch.randn(140, h_k, d, device="cuda").to(torch.bfloat16)
    v = torch.randn(140, h_k, d, device="cuda").to(torch.bfloat16)
    sel = torch.tensor([[[3, 0, -1, -1], [-1, -1, -1, -1], [1, 0, 7, -1]]], dtype=torch.int32,
                       device="cuda")                     # 7 is past sequence 2's last block
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse = nsa.decode(q, k, v, sel, cu, blk, d ** -0.5, device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 1                          # NSA_DEVERR_BAD_INDEX
    assert torch.all(out[1] == 0) and torch.all(torch.isneginf(lse[:, 1]))
    assert torch.isfinite(out[0].float()).all() and torch.isfinite(out[2].float()).all()
    # the bad slot is skipped: sequence 2 attends to blocks 1 and 0 only, like the oracle
    sel_full = np.full((h_k, 140, T), -1, dtype=np.int32)
    sel_full[0, 99] = [3, 0, -1, -1]
    sel_full[0, 139] = [1, 0, -1, -1]
    rows = np.array([[99, 0], [99, 1], [139, 0], [139, 1]])
    q_full = torch.zeros(140, h_k * g, d, dtype=torch.bfloat16)
    q_full[99], q_full[139] = q[0].cpu(), q[2].cpu()
    ref_o, ref_l = oracle.fwd_rows(cu.cpu().numpy(), blk, sel_full, q_full, k.cpu(), v.cpu(),
                                   d ** -0.5, rows)
    got_o = torch.stack([out[0, 0], out[0, 1], out[2, 0], out[2, 1]])
    got_l = torch.stack([lse[0, 0], lse[1, 0], lse[0, 2], lse[1, 2]])
    check_forward(got_o, got_l, ref_o, ref_l, "decode edge")


def test_decode_rejects_unsupported_shapes():
    import block_sparse_attention_nsa_gb300 as nsa
    q = torch.zeros(2, 4, 256, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(10, 1, 256, dtype=torch.bfloat16, device="cuda")
    sel = torch.zeros(1, 2, 4, dtype=torch.int32, device="cuda")
    cu = torch.tensor([0, 5, 10], dtype=torch.int32, device="cuda")
    with pytest.raises(nsa.NsaError) as e:
        nsa.decode(q, k, k, sel, cu, 64, 0.1)
    assert e.value.code == 2
