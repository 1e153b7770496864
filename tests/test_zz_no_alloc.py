"""The no-allocation forward, nsa_sel_attn_fwd_noalloc, called through the C ABI.

It exists for callers that cannot allocate device memory (host frameworks that
own all device memory, loops that cannot take an allocation's synchronisation);
its scratch is a fixed array inside the library.  Its output
must match the regular nsa_sel_attn_fwd (given a caller-allocated workspace)
within the forward tolerance, on consecutive calls that reuse the same array.
This file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import LSE_MAX_ABS, OUT_MAX_ABS, OUT_MEAN_ABS, to_device
from workloads import CONFIGS, WorkloadConfig, make_inputs

pytestmark = pytest.mark.gpu

NOALLOC_LIMIT = 16 * 1024 * 1024


def _lib():
    import block_sparse_attention_nsa_gb300 as nsa
    lib = nsa.load()
    fn = lib.nsa_sel_attn_fwd_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(nsa.Dims)] + [ctypes.c_void_p] * 5 + [ctypes.c_float] + \
        [ctypes.c_void_p] * 3
    return nsa, fn


def _case(cfg):
    nsa, _ = _lib()
    inp = make_inputs(cfg)
    d = to_device(inp)
    dims = nsa.make_dims(len(cfg.seqlens), cfg.n, cfg.h_q, cfg.h_k, cfg.d, cfg.block, cfg.topk,
                         d["q"].dtype)
    return d, dims


def _noalloc(d, dims, cfg):
    _, fn = _lib()
    out = torch.full_like(d["q"], float("nan"))
    lse = torch.full((cfg.h_q, cfg.n), float("nan"), dtype=torch.float32, device="cuda")
    st = fn(ctypes.byref(dims), d["q"].data_ptr(), d["k"].data_ptr(), d["v"].data_ptr(),
            d["sel_idx"].data_ptr(), d["cu_seqlens"].data_ptr(), cfg.scale, out.data_ptr(),
            lse.data_ptr(), torch.cuda.current_stream().cuda_stream)
    return st, out, lse


def _regular(d, cfg):
    nsa, _ = _lib()
    return nsa.fwd(d["q"], d["k"], d["v"], d["sel_idx"], d["cu_seqlens"], cfg.block, cfg.scale)


def _close(out, lse, ref_out, ref_lse):
    err = (out.float() - ref_out.float()).abs()
    assert torch.isfinite(out).all()
    assert err.max().item() <= OUT_MAX_ABS and err.mean().item() <= OUT_MEAN_ABS
    fin = torch.isfinite(ref_lse)
    assert torch.equal(torch.isfinite(lse), fin)
    if fin.any():
        assert (lse[fin] - ref_lse[fin]).abs().max().item() <= LSE_MAX_ABS


def test_noalloc_forward_matches_regular_on_consecutive_calls():
    nsa, _ = _lib()
    cfg_a = CONFIGS["tiny"]
    cfg_b = WorkloadConfig("noalloc_b", (300, 517, 250), 2, 3, 128, 64, 5, "bf16", "uniform",
                           1.0, 41)
    cases = []
    for cfg in (cfg_a, cfg_b):
        d, dims = _case(cfg)
        assert nsa.workspace_size(dims)[0] <= NOALLOC_LIMIT
        ref_out, ref_lse = _regular(d, cfg)
        cases.append((cfg, d, dims, ref_out, ref_lse))
    # two different problems back to back, then the first again: the shared
    # scratch keeps the previous call's contents, which must not matter
    for cfg, d, dims, ref_out, ref_lse in cases + cases[:1]:
        st, out, lse = _noalloc(d, dims, cfg)
        assert st == 0
        torch.cuda.synchronize()
        _close(out, lse, ref_out, ref_lse)


def test_noalloc_rejects_problems_above_the_limit():
    nsa, _ = _lib()
    cfg = CONFIGS["fwd8k"]
    d, dims = _case(cfg)
    assert nsa.workspace_size(dims)[0] > NOALLOC_LIMIT
    st, out, _ = _noalloc(d, dims, cfg)
    assert st == 3                       # NSA_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert torch.isnan(out).all()


def _status():
    import block_sparse_attention_nsa_gb300 as nsa
    lib = nsa.load()
    fn = lib.nsa_sel_attn_fwd_noalloc_status
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(nsa.Dims), ctypes.c_void_p, ctypes.POINTER(ctypes.c_int32)]
    return fn


def test_noalloc_status_reports_a_bad_selection_and_clears():
    status = _status()
    cfg = CONFIGS["tiny"]
    d, dims = _case(cfg)
    stream = torch.cuda.current_stream().cuda_stream
    bits = ctypes.c_int32(-1)
    # a clean call first: the word reads 0
    st, _, _ = _noalloc(d, dims, cfg)
    assert st == 0
    assert status(ctypes.byref(dims), stream, ctypes.byref(bits)) == 0 and bits.value == 0
    # one slot past the sequence's last block: skipped by the kernels, flagged in the word
    nb = (cfg.n + cfg.block - 1) // cfg.block
    bad = d["sel_idx"].clone()
    bad[0, cfg.n - 1, cfg.topk - 1] = nb
    d_bad = dict(d, sel_idx=bad)
    st, out, lse = _noalloc(d_bad, dims, cfg)
    assert st == 0
    assert status(ctypes.byref(dims), stream, ctypes.byref(bits)) == 5   # NSA_ERR_BAD_INDEX
    assert bits.value & 1                                                # NSA_DEVERR_BAD_INDEX
    assert torch.isfinite(out).all()
    # read and cleared: the next read is clean, and so is the next good call
    assert status(ctypes.byref(dims), stream, ctypes.byref(bits)) == 0 and bits.value == 0
    st, _, _ = _noalloc(d, dims, cfg)
    assert st == 0
    assert status(ctypes.byref(dims), stream, ctypes.byref(bits)) == 0 and bits.value == 0
