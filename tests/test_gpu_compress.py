"""GPU compressed branch and top-T block selection vs the fp64 oracle (through the C ABI).

The step that produces sel_idx: compression (kernel_size 32, kernel_stride 16),
attention over the compressed tokens, block importance and top-T selection with the
init and local blocks forced (Flash-Sparse-Attention README, "Usage").  Compressed
rows and offsets are compared element by element; out and lse to the forward's
tolerances, with the oracle's compressed tokens rounded once to the 16-bit type the
path stores them in; the selection, whose ranking is decided by fp32 sums on the GPU and fp64
sums in the oracle, is compared where the oracle's ranking is unique and checked
for validity where blocks tie within rounding."""
import numpy as np
import pytest
import torch

from gpu_helpers import check_forward
from oracle import compress as oc
from workloads import WorkloadConfig, make_cu_seqlens, make_inputs

pytestmark = pytest.mark.gpu

L_K, STRIDE = 32, 16


def _inputs(seqlens, h_k, g, d, dtype, seed):
    cfg = WorkloadConfig("cmp", tuple(seqlens), h_k, g, d, 64, 1, dtype, "uniform", 1.0, seed)
    inp = make_inputs(cfg)
    dev = {k: inp[k].cuda().contiguous() for k in ("q", "k", "v")}
    dev["cu"] = torch.from_numpy(inp["cu_seqlens"]).cuda()
    return cfg, inp, dev


def _f64(t):
    return t.float().cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_compress_kv_matches_oracle(d, dtype):
    seqlens = [300, 5, 31, 32, 47, 48, 0, 1000]
    cfg, inp, dev = _inputs(seqlens, 2, 1, d, dtype, 5)
    import block_sparse_attention_nsa_gb300 as nsa
    kc, vc, cu_cmp = nsa.compress_kv(dev["k"], dev["v"], dev["cu"], L_K, STRIDE)
    torch.cuda.synchronize()
    ref_cc = oc.cmp_seqlens(inp["cu_seqlens"], L_K, STRIDE)
    np.testing.assert_array_equal(cu_cmp.cpu().numpy(), ref_cc)
    rk, rv = oc.compress_kv(inp["cu_seqlens"], _f64(inp["k"]), _f64(inp["v"]), L_K, STRIDE)
    nc = int(ref_cc[-1])
    assert kc.shape[0] == cfg.n // STRIDE >= nc
    # fp32 sums of 16-bit inputs, one rounding to 16 bits: within one unit in the last
    # place of the exact mean rounded to that type
    u = 2.0 ** -7 if dtype == "bf16" else 2.0 ** -10
    for got, ref in ((kc[:nc], rk), (vc[:nc], rv)):
        r16 = _round16(ref, dtype)
        ulp = u * 2.0 ** np.floor(np.log2(np.maximum(np.abs(r16), 1e-30)))
        ulp = np.maximum(ulp, 2.0 ** -24 if dtype == "fp16" else 0.0)   # fp16 subnormals
        assert (np.abs(_f64(got) - r16) <= ulp + 1e-30).all()


def _round16(x, dtype):
    """The oracle's exact compressed tokens rounded once to the 16-bit type the path
    stores them in (the header's contract for nsa_compress_kv)."""
    t = {"bf16": torch.bfloat16, "fp16": torch.float16}[dtype]
    return torch.from_numpy(x).to(t).double().numpy()


def _check_selection(sel, ref_sel, imps, taus, block, topk, init, local, what):
    """Forced blocks first (ascending); distinct causal entries, then -1; the unforced
    picks rank by the oracle's fp64 importance up to a rounding tolerance."""
    h_k = sel.shape[0]
    exact = 0
    for n_, tau in enumerate(taus):
        c = tau // block
        forced = oc.forced_blocks(tau, block, init, local)[:topk]
        for h in range(h_k):
            row, ref = sel[h, n_], ref_sel[h, n_]
            kept = row[row >= 0].tolist()
            assert row[len(kept):].tolist() == [-1] * (topk - len(kept)), what
            assert len(kept) == min(topk, c + 1) and len(set(kept)) == len(kept), what
            assert all(0 <= j <= c for j in kept), what
            assert kept[:len(forced)] == forced, what
            imp = imps[n_][h]
            tol = 1e-4 + 2e-3 * float(imp.max())
            free = kept[len(forced):]
            others = [j for j in range(c + 1) if j not in kept]
            if free and others:
                assert imp[free].min() >= imp[others].max() - tol, what
            for x, y in zip(free, free[1:]):
                assert imp[x] >= imp[y] - tol, what
            exact += int((row == ref).all())
    return exact


@pytest.mark.parametrize("g,d,dtype,block", [(1, 128, "bf16", 64), (4, 128, "bf16", 64),
                                             (3, 64, "fp16", 64), (16, 128, "bf16", 64),
                                             (2, 64, "bf16", 32), (1, 64, "fp16", 128)])
def test_cmp_attn_select_matches_oracle(g, d, dtype, block):
    # ragged sequences: empty, shorter than one window, a partial chunk, several chunks;
    # B_K = 64 = 4 strides takes the kernel's aligned importance path, 32 and 128 the
    # general one
    seqlens = [700, 0, 20, 31, 33, 2100, 130]
    topk, init, local = 6, 1, 2
    cfg, inp, dev = _inputs(seqlens, 2, g, d, dtype, 17 + g)
    import block_sparse_attention_nsa_gb300 as nsa
    kc, vc, cu_cmp = nsa.compress_kv(dev["k"], dev["v"], dev["cu"], L_K, STRIDE)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, lse, sel = nsa.cmp_attn_select(dev["q"], kc, vc, dev["cu"], cu_cmp, L_K, STRIDE,
                                        max(seqlens), cfg.scale, block, topk, init, local,
                                        device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rk, rv = oc.compress_kv(inp["cu_seqlens"], _f64(inp["k"]), _f64(inp["v"]), L_K, STRIDE)
    rk, rv = _round16(rk, dtype), _round16(rv, dtype)
    toks = list(range(cfg.n))
    ref_sel, imps, ref_out, ref_lse = oc.select_rows(inp["cu_seqlens"], _f64(inp["q"]), rk, rv,
                                                     L_K, STRIDE, cfg.scale, block, topk, init,
                                                     local, toks)
    check_forward(out, lse, ref_out, ref_lse.T, f"cmp g={g} d={d}")
    cu = inp["cu_seqlens"]
    taus = [t - int(cu[np.searchsorted(cu, t, side="right") - 1]) for t in toks]
    exact = _check_selection(sel.cpu().numpy(), ref_sel, imps, taus, block, topk, init, local,
                             f"g={g}")
    # most rows have a unique ranking and must agree exactly
    assert exact >= 0.9 * len(toks) * cfg.h_k, exact


def test_cmp_attn_select_64k_sampled():
    # the 64K workload's shape (h_k = 4, d = 128, B_K = 64, T = 16, g = 4): sampled
    # tokens against the oracle, every output finite where a compressed token is visible
    seqlens = [65536]
    block, topk, init, local = 64, 16, 1, 2
    cfg, inp, dev = _inputs(seqlens, 4, 4, 128, "bf16", 1002)
    import block_sparse_attention_nsa_gb300 as nsa
    kc, vc, cu_cmp = nsa.compress_kv(dev["k"], dev["v"], dev["cu"], L_K, STRIDE)
    out, lse, sel = nsa.cmp_attn_select(dev["q"], kc, vc, dev["cu"], cu_cmp, L_K, STRIDE,
                                        65536, cfg.scale, block, topk, init, local)
    torch.cuda.synchronize()
    assert torch.isfinite(out).all()
    assert torch.isfinite(lse[:, L_K - 1:]).all() and torch.isinf(lse[:, :L_K - 1]).all()
    rng = np.random.default_rng(3)
    toks = sorted(set(rng.integers(0, 65536, 60).tolist()) | {0, 30, 31, 63, 64, 1023, 65535})
    rk, rv = oc.compress_kv(inp["cu_seqlens"], _f64(inp["k"]), _f64(inp["v"]), L_K, STRIDE)
    rk, rv = _round16(rk, "bf16"), _round16(rv, "bf16")
    ref_sel, imps, ref_out, ref_lse = oc.select_rows(inp["cu_seqlens"], _f64(inp["q"]), rk, rv,
                                                     L_K, STRIDE, cfg.scale, block, topk, init,
                                                     local, toks)
    check_forward(out[toks], lse[:, toks], ref_out, ref_lse.T, "cmp 64k")
    _check_selection(sel[:, toks].cpu().numpy(), ref_sel, imps, toks, block, topk, init, local,
                     "64k")
    # the selection feeds the selected-attention forward
    out2, lse2 = nsa.fwd(dev["q"], dev["k"], dev["v"], sel, dev["cu"], block, cfg.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out2).all() and torch.isfinite(lse2).all()


def test_cmp_attn_select_rejects_long_sequence():
    # a sequence longer than max_seqlen is flagged on the device and skipped
    seqlens = [200, 300]
    cfg, inp, dev = _inputs(seqlens, 1, 2, 64, "bf16", 9)
    import block_sparse_attention_nsa_gb300 as nsa
    kc, vc, cu_cmp = nsa.compress_kv(dev["k"], dev["v"], dev["cu"], L_K, STRIDE)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    nsa.cmp_attn_select(dev["q"], kc, vc, dev["cu"], cu_cmp, L_K, STRIDE, 256, cfg.scale, 64, 4,
                        device_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) & 2        # NSA_DEVERR_BAD_SEQLENS


def test_cmp_attn_select_workspace_rows_match_shared_rows():
    # g = 1 with a 40K-token sequence: in shared memory the importance rows leave a CTA
    # 64 tokens, so the call takes 128-token CTAs with the rows in its workspace.  The
    # per-row arithmetic is the same either way, so both launches agree bit for bit;
    # sampled rows are also checked against the oracle.
    seqlens = [40000, 300, 5000]
    block, topk, init, local = 64, 16, 1, 2
    cfg, inp, dev = _inputs(seqlens, 2, 1, 64, "bf16", 41)
    import block_sparse_attention_nsa_gb300 as nsa
    dims = nsa.make_dims(len(seqlens), cfg.n, cfg.h_q, cfg.h_k, cfg.d, block, topk, dev["q"].dtype)
    assert nsa.cmp_workspace_size(dims, L_K, STRIDE, max(seqlens)) > 0
    kc, vc, cu_cmp = nsa.compress_kv(dev["k"], dev["v"], dev["cu"], L_K, STRIDE)
    args = (dev["q"], kc, vc, dev["cu"], cu_cmp, L_K, STRIDE, max(seqlens), cfg.scale, block,
            topk, init, local)
    out_w, lse_w, sel_w = nsa.cmp_attn_select(*args)
    out_s, lse_s, sel_s = nsa.cmp_attn_select(*args, use_workspace=False)
    torch.cuda.synchronize()
    assert torch.equal(sel_w, sel_s)
    assert torch.equal(out_w, out_s)
    assert torch.equal(torch.nan_to_num(lse_w), torch.nan_to_num(lse_s))
    rng = np.random.default_rng(5)
    toks = sorted(set(rng.integers(0, cfg.n, 120).tolist()) | {0, 31, 39999, 40000, 40299,
                                                                 40300, cfg.n - 1})
    rk, rv = oc.compress_kv(inp["cu_seqlens"], _f64(inp["k"]), _f64(inp["v"]), L_K, STRIDE)
    rk, rv = _round16(rk, "bf16"), _round16(rv, "bf16")
    ref_sel, imps, ref_out, ref_lse = oc.select_rows(inp["cu_seqlens"], _f64(inp["q"]), rk, rv,
                                                     L_K, STRIDE, cfg.scale, block, topk, init,
                                                     local, toks)
    check_forward(out_w[toks], lse_w[:, toks], ref_out, ref_lse.T, "cmp workspace")
    cu = inp["cu_seqlens"]
    taus = [t - int(cu[np.searchsorted(cu, t, side="right") - 1]) for t in toks]
    _check_selection(sel_w[:, toks].cpu().numpy(), ref_sel, imps, taus, block, topk, init,
                     local, "workspace")
