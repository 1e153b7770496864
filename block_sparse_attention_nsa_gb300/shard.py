"""Splitting one selected-attention problem across ranks without any exchange.

Every KV head, together with its g query heads, its rows of the selection
tensor and its K/V columns, is independent in both forward and backward (the
softmax of a query never mixes KV heads, and dK/dV of a head only receive
contributions from that head's queries).  A rank that owns KV heads
[h_lo, h_hi) therefore computes exactly the slice of out / lse / dq / dk / dv
that a single device would, and the only collective needed is an optional
gather of results.  Sequences of a packed batch are independent as well.
"""
from __future__ import annotations

from typing import Sequence, Tuple


def kv_head_range(h_k: int, world: int, rank: int) -> Tuple[int, int]:
    """Contiguous, balanced KV-head range [lo, hi) of `rank` (may be empty if world > h_k)."""
    if world < 1 or not 0 <= rank < world:
        raise ValueError("bad world/rank")
    base, extra = divmod(h_k, world)
    lo = rank * base + min(rank, extra)
    return lo, lo + base + (1 if rank < extra else 0)


def slice_heads(tensors: dict, h_k: int, g: int, lo: int, hi: int) -> dict:
    """Per-rank views: q/out/dout/dq [N, h_q, d] -> query heads [lo*g, hi*g); k/v/dk/dv
    [N, h_k, d] -> [lo, hi); sel_idx [h_k, N, T] -> [lo, hi); lse [h_q, N] -> rows."""
    out = {}
    for name, t in tensors.items():
        if t is None:
            out[name] = None
        elif name in ("q", "out", "dout", "dq"):
            out[name] = t[:, lo * g:hi * g].contiguous() if hasattr(t, "contiguous") else \
                t[:, lo * g:hi * g].copy()
        elif name in ("k", "v", "dk", "dv"):
            out[name] = t[:, lo:hi].contiguous() if hasattr(t, "contiguous") else t[:, lo:hi].copy()
        elif name == "sel_idx":
            out[name] = t[lo:hi].contiguous() if hasattr(t, "contiguous") else t[lo:hi].copy()
        elif name == "lse":
            out[name] = t[lo * g:hi * g].contiguous() if hasattr(t, "contiguous") else \
                t[lo * g:hi * g].copy()
        else:
            out[name] = t
    return out


def sequence_groups(seqlens: Sequence[int], world: int):
    """Greedy split of packed sequences into `world` groups of similar token counts
    (largest first); returns one list of sequence indices per rank."""
    order = sorted(range(len(seqlens)), key=lambda i: -int(seqlens[i]))
    load = [0] * world
    groups = [[] for _ in range(world)]
    for i in order:
        r = min(range(world), key=lambda x: load[x])
        groups[r].append(i)
        load[r] += int(seqlens[i])
    return [sorted(gr) for gr in groups]
