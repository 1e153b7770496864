"""Python binding of libnsa_sel.so: NSA selected attention on GB300 (sm_103a).

Argument marshalling only.  Every step of the computation runs in the library's
CUDA kernels; PyTorch provides device memory (outputs and workspace) and the
current stream.  There is no CPU or PyTorch fallback: if the library is missing
or a call fails, an exception is raised.

Names follow the C ABI in include/nsa_sel_attn.h:
  workspace_size, index, index_view, fwd, bwd, decode, step_host, get_status,
  window_select, fwd_window, bwd_window, gate_combine, gate_combine_bwd,
  compress_kv, cmp_attn_select, profile_enable, profile_collect.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = ["Dims", "NsaError", "load", "workspace_size", "index", "index_view", "fwd", "bwd",
           "decode", "window_select", "fwd_window", "bwd_window", "gate_combine",
           "gate_combine_bwd", "compress_kv", "cmp_attn_select", "cmp_workspace_size",
           "staging_size", "step_host", "get_status", "profile_enable", "profile_collect",
           "kernel_names", "make_dims", "LIB_PATH"]

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libnsa_sel.so")

NSA_BF16, NSA_FP16 = 0, 1
_STATUS = {0: "ok", 1: "invalid argument", 2: "unsupported configuration",
           3: "workspace too small", 4: "CUDA error", 5: "bad index", 6: "timeout"}


class NsaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {_STATUS.get(code, code)} (status {code})")
        self.code = code


class Dims(ctypes.Structure):
    _fields_ = [("num_seqs", ctypes.c_int32), ("total_tokens", ctypes.c_int32),
                ("h_q", ctypes.c_int32), ("h_k", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("block_size", ctypes.c_int32), ("topk", ctypes.c_int32),
                ("dtype", ctypes.c_int32)]


_lib = None


def load():
    """Load the in-tree library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} not found: build it with "
                           "`python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i32, sz, f32 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_size_t, ctypes.c_float
    dp = ctypes.POINTER(Dims)
    st = ctypes.c_int
    sig = {
        "nsa_sel_attn_workspace_size": (st, [dp, ctypes.POINTER(sz), ctypes.POINTER(sz)]),
        "nsa_sel_attn_index": (st, [dp, vp, vp, vp, sz, vp]),
        "nsa_sel_attn_index_view": (st, [dp, vp, ctypes.POINTER(vp), ctypes.POINTER(vp),
                                         ctypes.POINTER(vp), ctypes.POINTER(vp),
                                         ctypes.POINTER(vp), ctypes.POINTER(i32)]),
        "nsa_sel_attn_fwd": (st, [dp, vp, vp, vp, vp, vp, f32, vp, vp, vp, sz, vp]),
        "nsa_sel_attn_bwd": (st, [dp, vp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp, vp, vp, sz,
                                  ctypes.c_int, vp]),
        "nsa_sel_attn_staging_size": (st, [dp, ctypes.POINTER(sz)]),
        "nsa_sel_attn_step_host": (st, [dp, vp, vp, vp, vp, vp, vp, f32, vp, vp, vp, vp, vp, vp,
                                        sz, vp, sz, vp]),
        "nsa_sel_attn_get_status": (st, [dp, vp, vp, ctypes.POINTER(i32)]),
        "nsa_sel_attn_decode": (st, [dp, vp, vp, vp, vp, vp, f32, vp, vp, vp, vp]),
        "nsa_sel_attn_window_select": (st, [dp, vp, ctypes.c_int, vp, vp]),
        "nsa_sel_attn_fwd_window": (st, [dp, vp, vp, vp, vp, vp, f32, ctypes.c_int, vp, vp, vp,
                                         sz, vp]),
        "nsa_sel_attn_bwd_window": (st, [dp, vp, vp, vp, vp, vp, f32, ctypes.c_int, vp, vp, vp,
                                         vp, vp, vp, vp, sz, ctypes.c_int, vp]),
        "nsa_gate_combine_fwd": (st, [dp, ctypes.c_int, vp, vp, vp, vp, vp, vp]),
        "nsa_gate_combine_bwd": (st, [dp, ctypes.c_int, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                      vp]),
        "nsa_compress_kv": (st, [dp, vp, ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp, vp,
                                 vp]),
        "nsa_cmp_attn_select": (st, [dp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                     ctypes.c_int, f32, ctypes.c_int, ctypes.c_int, vp, vp, vp,
                                     vp, vp, sz, vp]),
        "nsa_cmp_workspace_size": (st, [dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(sz)]),
        "nsa_sel_attn_num_kernels": (i32, []),
        "nsa_sel_attn_kernel_name": (ctypes.c_char_p, [i32]),
        "nsa_sel_attn_profile_enable": (st, [i32]),
        "nsa_sel_attn_profile_collect": (st, [ctypes.POINTER(i32), ctypes.POINTER(f32)]),
        "nsa_status_string": (ctypes.c_char_p, [st]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def _check(code: int, where: str):
    if code != 0:
        raise NsaError(code, where)


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def make_dims(num_seqs: int, total_tokens: int, h_q: int, h_k: int, head_dim: int,
              block_size: int, topk: int, dtype: torch.dtype) -> Dims:
    code = {torch.bfloat16: NSA_BF16, torch.float16: NSA_FP16}.get(dtype)
    if code is None:
        raise NsaError(2, f"dtype {dtype}")
    return Dims(num_seqs, total_tokens, h_q, h_k, head_dim, block_size, topk, code)


def _dims_of(q, k, sel_idx, cu_seqlens, block_size) -> Dims:
    if q.dim() != 3 or k.dim() != 3 or sel_idx.dim() != 3:
        raise ValueError("q [N, h_q, d], k [N, h_k, d], sel_idx [h_k, N, T] expected")
    return make_dims(cu_seqlens.numel() - 1, q.shape[0], q.shape[1], k.shape[1], q.shape[2],
                     block_size, sel_idx.shape[2], q.dtype)


def workspace_size(dims: Dims):
    f, b = ctypes.c_size_t(), ctypes.c_size_t()
    _check(load().nsa_sel_attn_workspace_size(ctypes.byref(dims), ctypes.byref(f),
                                              ctypes.byref(b)), "workspace_size")
    return f.value, b.value


def alloc_workspace(dims: Dims, device=None) -> torch.Tensor:
    f, b = workspace_size(dims)
    return torch.empty(max(f, b, 256), dtype=torch.uint8, device=device or "cuda")


def _contig(*ts):
    for t in ts:
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def index(sel_idx, cu_seqlens, block_size, dims: Dims, workspace: torch.Tensor, stream=None):
    _contig(sel_idx, cu_seqlens)
    _check(load().nsa_sel_attn_index(ctypes.byref(dims), _ptr(sel_idx), _ptr(cu_seqlens),
                                     _ptr(workspace), workspace.numel(), _stream(stream)), "index")


def index_view(dims: Dims, workspace: torch.Tensor):
    """Copies of the index tensors (synchronises): counts, offsets, q_list, slot_map, nb."""
    ptrs = [ctypes.c_void_p() for _ in range(5)]
    nbmax = ctypes.c_int32()
    _check(load().nsa_sel_attn_index_view(ctypes.byref(dims), _ptr(workspace),
                                          *[ctypes.byref(p) for p in ptrs],
                                          ctypes.byref(nbmax)), "index_view")
    base = workspace.data_ptr()

    def view(ptr, count):
        off = ptr.value - base
        return workspace[off:off + 4 * count].view(torch.int32)

    torch.cuda.synchronize()
    nb = int(view(ptrs[4], 1).item())
    nseg = dims.h_k * nb
    counts = view(ptrs[0], nseg).clone()
    offsets = view(ptrs[1], nseg + 1).clone()
    total = int(offsets[-1].item()) if nseg > 0 else 0
    q_list = view(ptrs[2], total).clone()
    slot_map = view(ptrs[3], dims.h_k * dims.total_tokens * dims.topk).clone().view(
        dims.h_k, dims.total_tokens, dims.topk)
    return {"counts": counts, "offsets": offsets, "q_list": q_list, "slot_map": slot_map,
            "num_blocks": nb}


def fwd(q, k, v, sel_idx, cu_seqlens, block_size: int, scale: float,
        workspace: Optional[torch.Tensor] = None, out=None, lse=None, stream=None):
    """out [N, h_q, d] (q's dtype) and lse float32 [h_q, N]."""
    _contig(q, k, v, sel_idx, cu_seqlens)
    dims = _dims_of(q, k, sel_idx, cu_seqlens, block_size)
    if workspace is None:
        workspace = alloc_workspace(dims, q.device)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device)
    _check(load().nsa_sel_attn_fwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(sel_idx),
                                   _ptr(cu_seqlens), float(scale), _ptr(out), _ptr(lse),
                                   _ptr(workspace), workspace.numel(), _stream(stream)), "fwd")
    return out, lse


def bwd(q, k, v, sel_idx, cu_seqlens, block_size: int, scale: float, out, lse, dout,
        workspace: Optional[torch.Tensor] = None, index_ready: bool = False, dq=None, dk=None,
        dv=None, stream=None):
    """dq, dk, dv (q's dtype).  index_ready reuses the index left in `workspace` by fwd."""
    _contig(q, k, v, sel_idx, cu_seqlens, out, lse, dout)
    dims = _dims_of(q, k, sel_idx, cu_seqlens, block_size)
    if workspace is None:
        workspace = alloc_workspace(dims, q.device)
        index_ready = False
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    _check(load().nsa_sel_attn_bwd(ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(sel_idx),
                                   _ptr(cu_seqlens), float(scale), _ptr(out), _ptr(lse),
                                   _ptr(dout), _ptr(dq), _ptr(dk), _ptr(dv), _ptr(workspace),
                                   workspace.numel(), 1 if index_ready else 0, _stream(stream)),
           "bwd")
    return dq, dk, dv


def staging_size(dims: Dims) -> int:
    n = ctypes.c_size_t()
    _check(load().nsa_sel_attn_staging_size(ctypes.byref(dims), ctypes.byref(n)), "staging_size")
    return n.value


def step_host(dims: Dims, host: dict, scale: float, staging: torch.Tensor,
              workspace: torch.Tensor, stream=None):
    """Forward + backward from host (ideally pinned) tensors; results land in host tensors.

    host: q, k, v, dout, sel_idx, cu_seqlens (inputs) and out, lse, dq, dk, dv (outputs).
    """
    _check(load().nsa_sel_attn_step_host(
        ctypes.byref(dims), _ptr(host["q"]), _ptr(host["k"]), _ptr(host["v"]),
        _ptr(host["sel_idx"]), _ptr(host["cu_seqlens"]), _ptr(host["dout"]), float(scale),
        _ptr(host["out"]), _ptr(host.get("lse")), _ptr(host["dq"]), _ptr(host["dk"]),
        _ptr(host["dv"]), _ptr(staging), staging.numel(), _ptr(workspace), workspace.numel(),
        _stream(stream)), "step_host")


def decode(q, k_cache, v_cache, sel_idx, cu_seqlens, block_size: int, scale: float, out=None,
           lse=None, device_status=None, stream=None):
    """One-step decode: q [B, h_q, d] (the last token of each cached sequence), caches
    [N, h_k, d], sel_idx int32 [h_k, B, T]; returns out [B, h_q, d] and lse [h_q, B]."""
    _contig(q, k_cache, v_cache, sel_idx, cu_seqlens)
    B, h_q, d = q.shape
    h_k, topk = k_cache.shape[1], sel_idx.shape[2]
    dims = make_dims(B, k_cache.shape[0], h_q, h_k, d, block_size, topk, q.dtype)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((h_q, B), dtype=torch.float32, device=q.device)
    _check(load().nsa_sel_attn_decode(
        ctypes.byref(dims), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(sel_idx),
        _ptr(cu_seqlens), float(scale), _ptr(out), _ptr(lse), _ptr(device_status),
        _stream(stream)), "decode")
    return out, lse


def compress_kv(k, v, cu_seqlens, kernel_size: int, kernel_stride: int, device_status=None,
                stream=None):
    """Compressed keys and values: kc, vc [N // kernel_stride, h_k, d] (rows past the
    total are unused) and cu_cmp int32 [S + 1], each sequence's compressed rows."""
    _contig(k, v, cu_seqlens)
    n, h_k, d = k.shape
    dims = make_dims(cu_seqlens.numel() - 1, n, h_k, h_k, d, 64, 1, k.dtype)
    rows = n // kernel_stride
    kc = torch.empty((rows, h_k, d), dtype=k.dtype, device=k.device)
    vc = torch.empty_like(kc)
    cu_cmp = torch.empty(cu_seqlens.numel(), dtype=torch.int32, device=k.device)
    _check(load().nsa_compress_kv(ctypes.byref(dims), _ptr(cu_seqlens), int(kernel_size),
                                  int(kernel_stride), _ptr(k), _ptr(v), _ptr(kc), _ptr(vc),
                                  _ptr(cu_cmp), _ptr(device_status), _stream(stream)),
           "compress_kv")
    return kc, vc, cu_cmp


def cmp_workspace_size(dims: Dims, kernel_size: int, kernel_stride: int,
                       max_seqlen: int) -> int:
    """Workspace bytes of cmp_attn_select (0 when shared memory holds the rows)."""
    b = ctypes.c_size_t()
    _check(load().nsa_cmp_workspace_size(ctypes.byref(dims), int(kernel_size),
                                         int(kernel_stride), int(max_seqlen), ctypes.byref(b)),
           "cmp_workspace_size")
    return b.value


def cmp_attn_select(q, kc, vc, cu_seqlens, cu_cmp, kernel_size: int, kernel_stride: int,
                    max_seqlen: int, scale: float, block_size: int, topk: int,
                    init_blocks: int = 1, local_blocks: int = 2, device_status=None,
                    workspace: Optional[torch.Tensor] = None, use_workspace: bool = True,
                    stream=None):
    """Compressed attention and top-T block selection: out [N, h_q, d], lse float32
    [h_q, N] and sel_idx int32 [h_k, N, topk].  workspace: uint8 device tensor of at
    least cmp_workspace_size bytes; allocated here when None and needed, and never
    passed when use_workspace is False (the importance rows then stay in shared
    memory, in smaller CTAs)."""
    _contig(q, kc, vc, cu_seqlens, cu_cmp)
    n, h_q, d = q.shape
    h_k = kc.shape[1]
    dims = make_dims(cu_seqlens.numel() - 1, n, h_q, h_k, d, block_size, topk, q.dtype)
    if not use_workspace:
        workspace = None
    elif workspace is None:
        need = cmp_workspace_size(dims, kernel_size, kernel_stride, max_seqlen)
        if need:
            workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    out = torch.empty_like(q)
    lse = torch.empty((h_q, n), dtype=torch.float32, device=q.device)
    sel = torch.empty((h_k, n, topk), dtype=torch.int32, device=q.device)
    _check(load().nsa_cmp_attn_select(
        ctypes.byref(dims), _ptr(q), _ptr(kc), _ptr(vc), _ptr(cu_seqlens), _ptr(cu_cmp),
        int(kernel_size), int(kernel_stride), int(max_seqlen), float(scale), int(init_blocks),
        int(local_blocks), _ptr(out), _ptr(lse), _ptr(sel), _ptr(device_status),
        _ptr(workspace), 0 if workspace is None else workspace.numel(),
        _stream(stream)), "cmp_attn_select")
    return out, lse, sel


def window_select(cu_seqlens, total_tokens: int, h_k: int, block_size: int, topk: int,
                  window: int, num_seqs: Optional[int] = None, stream=None):
    """Selection int32 [h_k, N, topk] of the sliding window (newest block first)."""
    num_seqs = cu_seqlens.numel() - 1 if num_seqs is None else num_seqs
    dims = make_dims(num_seqs, total_tokens, h_k, h_k, 64, block_size, topk, torch.bfloat16)
    sel = torch.empty((h_k, total_tokens, topk), dtype=torch.int32, device=cu_seqlens.device)
    _check(load().nsa_sel_attn_window_select(ctypes.byref(dims), _ptr(cu_seqlens), int(window),
                                             _ptr(sel), _stream(stream)), "window_select")
    return sel


def fwd_window(q, k, v, sel_idx, cu_seqlens, block_size: int, scale: float, window: int,
               workspace: Optional[torch.Tensor] = None, out=None, lse=None, stream=None):
    """fwd with the sliding window's lower key bound (keys > t - window)."""
    _contig(q, k, v, sel_idx, cu_seqlens)
    dims = _dims_of(q, k, sel_idx, cu_seqlens, block_size)
    if workspace is None:
        workspace = alloc_workspace(dims, q.device)
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty((q.shape[1], q.shape[0]), dtype=torch.float32, device=q.device) \
        if lse is None else lse
    _check(load().nsa_sel_attn_fwd_window(
        ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(sel_idx), _ptr(cu_seqlens),
        float(scale), int(window), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(),
        _stream(stream)), "fwd_window")
    return out, lse


def bwd_window(q, k, v, sel_idx, cu_seqlens, block_size: int, scale: float, window: int, out,
               lse, dout, workspace: Optional[torch.Tensor] = None, index_ready: bool = False,
               stream=None):
    """bwd with the sliding window's lower key bound; returns dq, dk, dv."""
    _contig(q, k, v, sel_idx, cu_seqlens, out, lse, dout)
    dims = _dims_of(q, k, sel_idx, cu_seqlens, block_size)
    if workspace is None:
        workspace = alloc_workspace(dims, q.device)
        index_ready = False
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    _check(load().nsa_sel_attn_bwd_window(
        ctypes.byref(dims), _ptr(q), _ptr(k), _ptr(v), _ptr(sel_idx), _ptr(cu_seqlens),
        float(scale), int(window), _ptr(out), _ptr(lse), _ptr(dout), _ptr(dq), _ptr(dk),
        _ptr(dv), _ptr(workspace), workspace.numel(), 1 if index_ready else 0, _stream(stream)),
        "bwd_window")
    return dq, dk, dv


def gate_combine(branches, gates, stream=None):
    """out = sum_b gates[..., b] * branches[b]; branches [N, h_q, d], gates fp32 [N, h_q, nb]."""
    _contig(*branches, gates)
    o = list(branches) + [None] * (3 - len(branches))
    N, h_q, d = branches[0].shape
    dims = make_dims(1, N, h_q, h_q, d, 64, 1, branches[0].dtype)
    out = torch.empty_like(branches[0])
    _check(load().nsa_gate_combine_fwd(ctypes.byref(dims), len(branches), _ptr(o[0]), _ptr(o[1]),
                                       _ptr(o[2]), _ptr(gates), _ptr(out), _stream(stream)),
           "gate_combine")
    return out


def gate_combine_bwd(branches, gates, dout, stream=None):
    """(list of d branch, d gates fp32)."""
    _contig(*branches, gates, dout)
    o = list(branches) + [None] * (3 - len(branches))
    N, h_q, d = branches[0].shape
    dims = make_dims(1, N, h_q, h_q, d, 64, 1, branches[0].dtype)
    dbr = [torch.empty_like(b) for b in branches] + [None] * (3 - len(branches))
    dg = torch.empty_like(gates)
    _check(load().nsa_gate_combine_bwd(ctypes.byref(dims), len(branches), _ptr(o[0]), _ptr(o[1]),
                                       _ptr(o[2]), _ptr(gates), _ptr(dout), _ptr(dbr[0]),
                                       _ptr(dbr[1]), _ptr(dbr[2]), _ptr(dg), _stream(stream)),
           "gate_combine_bwd")
    return dbr[:len(branches)], dg


def get_status(dims: Dims, workspace: torch.Tensor, stream=None):
    """(status code, raw device bits); synchronises the stream and clears the word."""
    bits = ctypes.c_int32()
    code = load().nsa_sel_attn_get_status(ctypes.byref(dims), _ptr(workspace), _stream(stream),
                                          ctypes.byref(bits))
    return int(code), int(bits.value)


def kernel_names():
    lib = load()
    return [lib.nsa_sel_attn_kernel_name(i).decode() for i in range(lib.nsa_sel_attn_num_kernels())]


def profile_enable(on: bool = True):
    _check(load().nsa_sel_attn_profile_enable(1 if on else 0), "profile_enable")


def profile_collect():
    """{kernel name: (launches, total ms)} since the last collect (synchronises)."""
    lib = load()
    n = lib.nsa_sel_attn_num_kernels()
    launches = (ctypes.c_int32 * n)()
    ms = (ctypes.c_float * n)()
    _check(lib.nsa_sel_attn_profile_collect(launches, ms), "profile_collect")
    return {name: (int(launches[i]), float(ms[i])) for i, name in enumerate(kernel_names())}
