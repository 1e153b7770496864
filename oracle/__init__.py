"""fp64 CPU oracle for NSA selected attention -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never calls it and the
two share no code.  The arithmetic lives in ``nsa_oracle.c`` (plain loops, fp64,
OpenMP over independent rows); this module compiles it with gcc on first use
and marshals numpy arrays through ctypes.

Parity status per function (pins live in tests/test_oracle_*.py):
  fwd / fwd_rows -- pinned: dense causal attention and block-aligned local
                    attention via torch SDPA (fp64), a hand-derived golden
                    example, constant-V, q = 0 closed forms, slot-order /
                    duplicate / -1 invariance, varlen = separate runs.
  bwd            -- pinned: central finite differences of fwd, torch autograd
                    through SDPA on the dense special case, sum_j dk_j = 0,
                    constant-V and q = 0 closed forms.
  index          -- pinned: brute-force construction on tiny inputs, the
                    scan/segment/inverse invariants, and the closed-form pair
                    counts of the synthetic selection rule.
  window_select, fwd / bwd with window -- pinned: dense sliding-window attention
                    (torch SDPA with a band mask, fp64) and its autograd; window
                    >= sequence length equals plain causal attention.
  gate_combine / gate_combine_bwd -- pinned: closed-form sums and central finite
                    differences of the gates.
  compress (module oracle.compress, numpy fp64) -- compression, compressed
                    attention, block importance and top-T selection; pinned: closed
                    forms, torch SDPA with an explicit mask, l = stride = 1 equals
                    causal attention, key-level and sort-based brute force.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nsa_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libnsa_oracle.so")
_lock = threading.Lock()
_lib = None

_i32p = np.ctypeslib.ndpointer(dtype=np.int32, flags="C_CONTIGUOUS")
_i64p = np.ctypeslib.ndpointer(dtype=np.int64, flags="C_CONTIGUOUS")
_f64p = np.ctypeslib.ndpointer(dtype=np.float64, flags="C_CONTIGUOUS")


def build(force: bool = False) -> str:
    """Compile nsa_oracle.c into oracle/_build/libnsa_oracle.so (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fopenmp", "-std=c11", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        c_int, c_dbl, c_i64 = ctypes.c_int, ctypes.c_double, ctypes.c_int64
        lib.nsa_oracle_fwd.argtypes = [c_int, _i32p, c_int, c_int, c_int, c_int, c_int, _i32p,
                                       _f64p, _f64p, _f64p, c_dbl, _f64p, _f64p, c_int]
        lib.nsa_oracle_fwd.restype = c_int
        lib.nsa_oracle_fwd_rows.argtypes = [c_int, _i32p, c_int, c_int, c_int, c_int, c_int, _i32p,
                                            _f64p, _f64p, _f64p, c_dbl, c_i64, _i64p, _f64p, _f64p,
                                            c_int]
        lib.nsa_oracle_fwd_rows.restype = c_int
        lib.nsa_oracle_bwd.argtypes = [c_int, _i32p, c_int, c_int, c_int, c_int, c_int, _i32p,
                                       _f64p, _f64p, _f64p, _f64p, c_dbl, _f64p, _f64p, _f64p, c_int]
        lib.nsa_oracle_bwd.restype = c_int
        lib.nsa_oracle_index.argtypes = [c_int, _i32p, c_int, c_int, c_int, _i32p, _i32p, _i32p,
                                         _i32p, _i32p]
        lib.nsa_oracle_index.restype = c_i64
        lib.nsa_oracle_num_blocks.argtypes = [c_int, _i32p, c_int]
        lib.nsa_oracle_num_blocks.restype = c_i64
        lib.nsa_oracle_fwd_w.argtypes = [c_int, _i32p, c_int, c_int, c_int, c_int, c_int, c_int,
                                         _i32p, _f64p, _f64p, _f64p, c_dbl, _f64p, _f64p, c_int]
        lib.nsa_oracle_fwd_w.restype = c_int
        lib.nsa_oracle_bwd_w.argtypes = [c_int, _i32p, c_int, c_int, c_int, c_int, c_int, c_int,
                                         _i32p, _f64p, _f64p, _f64p, _f64p, c_dbl, _f64p, _f64p,
                                         _f64p, c_int]
        lib.nsa_oracle_bwd_w.restype = c_int
        lib.nsa_oracle_window_select.argtypes = [c_int, _i32p, c_int, c_int, c_int, c_int, _i32p]
        lib.nsa_oracle_window_select.restype = c_int
        lib.nsa_oracle_max_threads.argtypes = []
        lib.nsa_oracle_max_threads.restype = c_int
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    """Exact upcast of a torch (bf16/fp16/fp32) tensor or numpy array to fp64."""
    if hasattr(x, "detach"):
        x = x.detach().cpu().float().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _i32(x) -> np.ndarray:
    if hasattr(x, "detach"):
        x = x.detach().cpu().numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.int32))


def max_threads() -> int:
    return int(_load().nsa_oracle_max_threads())


def _dims(cu, q, k, sel):
    n = int(cu[-1])
    h_q, d = q.shape[1], q.shape[2]
    h_k = k.shape[1]
    if h_q % h_k:
        raise ValueError("h_q must be a multiple of h_k")
    topk = sel.shape[2]
    if q.shape[0] != n or k.shape[0] != n or sel.shape[:2] != (h_k, n):
        raise ValueError("shape mismatch")
    return n, h_q, h_k, h_q // h_k, d, topk


def fwd(cu_seqlens, block, sel_idx, q, k, v, scale, threads: int = 0, window: int = 0):
    """out [N, h_q, d] and lse [h_q, N] in fp64 (natural log, scale included).  window
    > 0 also restricts every token's keys to its last `window` positions."""
    cu, sel = _i32(cu_seqlens), _i32(sel_idx)
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, h_q, h_k, g, d, topk = _dims(cu, q, k, sel)
    out = np.empty((n, h_q, d))
    lse = np.empty((h_q, n))
    rc = _load().nsa_oracle_fwd_w(len(cu) - 1, cu, h_k, g, d, block, topk, int(window), sel, q,
                                  k, v, float(scale), out, lse, threads)
    if rc:
        raise RuntimeError(f"nsa_oracle_fwd failed ({rc})")
    return out, lse


def fwd_rows(cu_seqlens, block, sel_idx, q, k, v, scale, rows, threads: int = 0):
    """Forward on sampled (token, query head) rows: returns out [n, d], lse [n]."""
    cu, sel = _i32(cu_seqlens), _i32(sel_idx)
    q, k, v = _f64(q), _f64(k), _f64(v)
    n, h_q, h_k, g, d, topk = _dims(cu, q, k, sel)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    out = np.empty((rows.shape[0], d))
    lse = np.empty(rows.shape[0])
    rc = _load().nsa_oracle_fwd_rows(len(cu) - 1, cu, h_k, g, d, block, topk, sel, q, k, v,
                                     float(scale), rows.shape[0], rows, out, lse, threads)
    if rc:
        raise RuntimeError(f"nsa_oracle_fwd_rows failed ({rc})")
    return out, lse


def bwd(cu_seqlens, block, sel_idx, q, k, v, dout, scale, threads: int = 0, window: int = 0):
    """dq [N, h_q, d], dk, dv [N, h_k, d] in fp64 by direct differentiation (window as
    for fwd)."""
    cu, sel = _i32(cu_seqlens), _i32(sel_idx)
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    n, h_q, h_k, g, d, topk = _dims(cu, q, k, sel)
    dq = np.empty((n, h_q, d))
    dk = np.empty((n, h_k, d))
    dv = np.empty((n, h_k, d))
    rc = _load().nsa_oracle_bwd_w(len(cu) - 1, cu, h_k, g, d, block, topk, int(window), sel, q,
                                  k, v, dout, float(scale), dq, dk, dv, threads)
    if rc:
        raise RuntimeError(f"nsa_oracle_bwd failed ({rc})")
    return dq, dk, dv


def window_select(cu_seqlens, h_k, block, topk, window) -> np.ndarray:
    """Selection int32 [h_k, N, topk] of the sliding window: the blocks holding the keys
    of (tau - window, tau] of each token, newest first, the rest -1."""
    cu = _i32(cu_seqlens)
    n = int(cu[-1])
    sel = np.empty((h_k, n, topk), dtype=np.int32)
    if _load().nsa_oracle_window_select(len(cu) - 1, cu, h_k, block, topk, int(window), sel):
        raise ValueError("topk too small for the window")
    return sel


def gate_combine(branches, gates):
    """Gated combination of branch outputs (the three-branch NSA output): out[r] =
    sum_b gates[r, b] * o_b[r].  branches: list of [N, h_q, d]; gates [N, h_q, nb]."""
    g = _f64(gates)
    out = np.zeros(_f64(branches[0]).shape)
    for b, o in enumerate(branches):
        out += g[..., b:b + 1] * _f64(o)
    return out


def gate_combine_bwd(branches, gates, dout):
    """d o_b = gates[..., b] * dout; d gates[..., b] = sum_d dout * o_b."""
    g, dy = _f64(gates), _f64(dout)
    d_br = [g[..., b:b + 1] * dy for b in range(len(branches))]
    d_g = np.stack([(dy * _f64(o)).sum(-1) for o in branches], axis=-1)
    return d_br, d_g


def num_blocks(cu_seqlens, block) -> int:
    cu = _i32(cu_seqlens)
    return int(_load().nsa_oracle_num_blocks(len(cu) - 1, cu, block))


def index(cu_seqlens, block, sel_idx):
    """Index tensors: counts [h_k*NB], offsets [h_k*NB+1], q_list [total], slot_map [h_k,N,T]."""
    cu, sel = _i32(cu_seqlens), _i32(sel_idx)
    h_k, n, topk = sel.shape
    if int(cu[-1]) != n:
        raise ValueError("shape mismatch")
    nb = num_blocks(cu, block)
    counts = np.empty(h_k * nb, dtype=np.int32)
    offsets = np.empty(h_k * nb + 1, dtype=np.int32)
    q_list = np.empty(max(1, h_k * n * topk), dtype=np.int32)
    slot_map = np.empty((h_k, n, topk), dtype=np.int32)
    total = _load().nsa_oracle_index(len(cu) - 1, cu, h_k, block, topk, sel, counts, offsets,
                                     q_list, slot_map)
    if total < 0:
        raise RuntimeError("nsa_oracle_index failed")
    return {"counts": counts, "offsets": offsets, "q_list": q_list[:total].copy(),
            "slot_map": slot_map, "num_blocks": nb}
