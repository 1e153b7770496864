"""Shared helpers of the GPU parity tests (the oracle side is fp64, CPU)."""
import numpy as np
import torch

# Parity bar (forward): out max-abs <= 2e-2 and mean-abs <= 2e-3 for bf16/fp16
# inputs, lse max-abs <= 1e-3; backward: dQ, dK, dV relative L2 <= 2e-2.
OUT_MAX_ABS, OUT_MEAN_ABS, LSE_MAX_ABS, GRAD_REL_L2 = 2e-2, 2e-3, 1e-3, 2e-2


def to_device(inp, dev="cuda"):
    out = {}
    for key in ("q", "k", "v", "dout"):
        if inp.get(key) is not None:
            out[key] = inp[key].to(dev).contiguous()
    out["sel_idx"] = torch.from_numpy(np.ascontiguousarray(inp["sel_idx"])).to(dev)
    out["cu_seqlens"] = torch.from_numpy(np.ascontiguousarray(inp["cu_seqlens"])).to(dev)
    return out


def check_forward(out, lse, ref_out, ref_lse, what=""):
    """out/ref_out [..., d]; lse/ref_lse matching shapes (numpy or torch)."""
    o = out.float().cpu().numpy() if torch.is_tensor(out) else np.asarray(out, np.float64)
    l = lse.float().cpu().numpy() if torch.is_tensor(lse) else np.asarray(lse, np.float64)
    assert np.isfinite(o).all(), f"{what}: non-finite output"
    # max and mean of |o - ref| over the whole tensor, a slab of rows at a time
    o2, r2 = o.reshape(o.shape[0], -1), np.asarray(ref_out).reshape(o.shape[0], -1)
    emax, esum = 0.0, 0.0
    for i in range(0, o2.shape[0], 4096):
        e = np.abs(o2[i:i + 4096].astype(np.float64) - r2[i:i + 4096])
        emax = max(emax, float(e.max()))
        esum += float(e.sum())
    emean = esum / max(1, o2.size)
    assert emax <= OUT_MAX_ABS, f"{what}: out max-abs {emax:.3e}"
    assert emean <= OUT_MEAN_ABS, f"{what}: out mean-abs {emean:.3e}"
    fin = np.isfinite(ref_lse)
    np.testing.assert_array_equal(np.isfinite(l), fin, err_msg=f"{what}: lse -inf pattern")
    lerr = np.abs(l[fin] - ref_lse[fin]).max() if fin.any() else 0.0
    assert lerr <= LSE_MAX_ABS, f"{what}: lse max-abs {lerr:.3e}"
    return emax, emean, float(lerr)


def rel_l2(got, ref):
    g = got.float().cpu().numpy() if torch.is_tensor(got) else got
    return float(np.linalg.norm(g - ref) / max(np.linalg.norm(ref), 1e-30))


def sample_rows(n, h_q, count, seed, seqlens=None, block=64):
    """(token, query head) rows: random ones plus sequence edges and block boundaries."""
    rng = np.random.default_rng(seed)
    t = list(rng.integers(0, n, count))
    base = 0
    for L in (seqlens or [n]):
        for x in (0, 1, block - 1, block, L // 2, L - block, L - 2, L - 1):
            if 0 <= x < L:
                t.append(base + x)
        base += L
    t = np.asarray(t, dtype=np.int64)
    hq = rng.integers(0, h_q, t.size)
    hq[: min(h_q, t.size)] = np.arange(min(h_q, t.size))
    return np.stack([t, hq], axis=1)
