"""Seeded synthetic inputs for NSA selected attention.

This module is shared by the fp64 oracle's tests, the GPU parity tests and
``bench.py``.  It draws inputs only (q, k, v, dO, the selection tensor and the
packed-sequence offsets); it contains none of the attention arithmetic.

Shapes and layouts (packed variable-length batch, tokens concatenated):
  q, dout     [N, h_q, d]       h_q = h_k * g (query head hq belongs to KV head hq // g)
  k, v        [N, h_k, d]
  sel_idx     int32 [h_k, N, T]  sequence-local KV-block indices, -1 = empty slot
  cu_seqlens  int32 [S + 1]      prefix offsets of the packed sequences

The selection tensor plays the role of NSA's top-k output (the h_K x N x T
selection tensor of "FSA: An Alternative Efficient Implementation of Native
Sparse Attention Kernel", key design 2).  Per (KV head, token) with local
block c = position // block_size:
  slot 0 = the token's own block c; slot 1 = block 0 when c > 0;
  the remaining min(T - 2, c - 1) slots are drawn without replacement from
  blocks 1 .. c-1, with equal weights ("uniform") or weights 1 / (1 + (c - b))
  ("distance"); unused slots are -1.  Draws use Gumbel-top-k, which samples
  the same distribution as sequential weighted sampling without replacement
  (Vieira 2014; Kool, van Hoof & Welling 2019), and are kept in descending
  order of their perturbed keys.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch

__all__ = ["WorkloadConfig", "CONFIGS", "make_selection", "make_cu_seqlens", "make_inputs",
           "config_by_name"]


@dataclasses.dataclass(frozen=True)
class WorkloadConfig:
    name: str
    seqlens: tuple
    h_k: int
    g: int
    d: int
    block: int
    topk: int
    dtype: str          # "bf16" or "fp16"
    rule: str           # "uniform" or "distance"
    std: float
    seed: int
    with_dout: bool = False

    @property
    def n(self) -> int:
        return int(sum(self.seqlens))

    @property
    def h_q(self) -> int:
        return self.h_k * self.g

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_g(self, g: int) -> "WorkloadConfig":
        return dataclasses.replace(self, g=g, name=f"{self.name.split('_g')[0]}_g{g}")


# The five workloads of the hot path (packed batch of one or more sequences).
CONFIGS = {
    "tiny": WorkloadConfig("tiny", (256,), 1, 2, 64, 32, 4, "bf16", "uniform", 1.0, 1000),
    "fwd8k": WorkloadConfig("fwd8k", (8192,), 4, 1, 128, 64, 16, "bf16", "uniform", 1.0, 1001),
    "fwd64k": WorkloadConfig("fwd64k", (65536,), 4, 1, 128, 64, 16, "bf16", "distance", 1.0, 1002),
    "varlen": WorkloadConfig("varlen", (16384, 32768, 8192, 8192), 2, 4, 256, 64, 16, "fp16",
                             "uniform", math.sqrt(0.5), 1003),
    "bwd32k": WorkloadConfig("bwd32k", (32768,), 4, 2, 128, 64, 16, "bf16", "uniform", 1.0, 1004,
                             with_dout=True),
}


def config_by_name(name: str) -> WorkloadConfig:
    """'fwd64k_g4' style names select a group size for the 64K sweep."""
    if "_g" in name:
        base, g = name.split("_g")
        return CONFIGS[base].with_g(int(g))
    return CONFIGS[name]


def make_cu_seqlens(seqlens: Sequence[int]) -> np.ndarray:
    cu = np.zeros(len(seqlens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    return cu


def _draw_one_sequence(rng: np.random.Generator, length: int, h_k: int, block: int, topk: int,
                       rule: str) -> np.ndarray:
    """Selection rows for one sequence, [h_k, length, topk], sequence-local indices."""
    sel = np.full((h_k, length, topk), -1, dtype=np.int32)
    nblk = (length + block - 1) // block
    for c in range(nblk):
        t0, t1 = c * block, min(length, (c + 1) * block)
        rows = t1 - t0
        sel[:, t0:t1, 0] = c
        if topk >= 2 and c > 0:
            sel[:, t0:t1, 1] = 0
        ndraw = min(topk - 2, c - 1) if topk >= 2 else 0
        if ndraw <= 0:
            continue
        cand = np.arange(1, c, dtype=np.int32)               # blocks 1 .. c-1
        if rule == "uniform":
            logw = np.zeros(c - 1)
        elif rule == "distance":
            logw = -np.log1p((c - cand).astype(np.float64))
        else:
            raise ValueError(f"unknown selection rule {rule!r}")
        keys = logw[None, None, :] + rng.gumbel(size=(h_k, rows, c - 1))
        if ndraw < c - 1:
            part = np.argpartition(-keys, ndraw - 1, axis=-1)[..., :ndraw]
        else:
            part = np.broadcast_to(np.arange(c - 1), (h_k, rows, c - 1)).copy()
        pk = np.take_along_axis(keys, part, axis=-1)
        order = np.argsort(-pk, axis=-1, kind="stable")
        picks = np.take_along_axis(part, order, axis=-1)
        sel[:, t0:t1, 2:2 + ndraw] = cand[picks]
    return sel


def make_selection(seqlens: Sequence[int], h_k: int, block: int, topk: int, rule: str,
                   rng: np.random.Generator) -> np.ndarray:
    """Selection tensor int32 [h_k, N, T] for a packed batch (indices local to each sequence)."""
    parts = [_draw_one_sequence(rng, int(L), h_k, block, topk, rule) for L in seqlens]
    return np.ascontiguousarray(np.concatenate(parts, axis=1))


def _draw_last_token(rng: np.random.Generator, length: int, h_k: int, block: int, topk: int,
                     rule: str) -> np.ndarray:
    """Selection row [h_k, topk] of the last token of a sequence of `length` tokens, by
    the same rule as _draw_one_sequence (own block, block 0, draws from 1 .. c-1)."""
    sel = np.full((h_k, topk), -1, dtype=np.int32)
    if length <= 0:
        return sel
    c = (length - 1) // block
    sel[:, 0] = c
    if topk >= 2 and c > 0:
        sel[:, 1] = 0
    ndraw = min(topk - 2, c - 1) if topk >= 2 else 0
    if ndraw > 0:
        cand = np.arange(1, c, dtype=np.int32)
        logw = (np.zeros(c - 1) if rule == "uniform"
                else -np.log1p((c - cand).astype(np.float64)))
        keys = logw[None, :] + rng.gumbel(size=(h_k, c - 1))
        picks = np.argsort(-keys, axis=-1, kind="stable")[:, :ndraw]
        sel[:, 2:2 + ndraw] = cand[picks]
    return sel


def make_decode_inputs(seqlens: Sequence[int], h_k: int, g: int, d: int, block: int, topk: int,
                       rule: str, dtype: str, seed: int, std: float = 1.0):
    """One-step decode inputs: q [B, h_q, d] (the new token of each sequence), k/v caches
    [N, h_k, d] packed by cu_seqlens, sel_idx int32 [h_k, B, T] (the last token's row)."""
    rng = np.random.default_rng(seed)
    td = torch_dtype(dtype)
    B, n = len(seqlens), int(np.sum(seqlens))
    q = _normal(rng, (B, h_k * g, d), std, td)
    k = _normal(rng, (n, h_k, d), std, td)
    v = _normal(rng, (n, h_k, d), std, td)
    sel = np.stack([_draw_last_token(rng, int(L), h_k, block, topk, rule) for L in seqlens],
                   axis=1)
    return {"q": q, "k": k, "v": v, "sel_idx": np.ascontiguousarray(sel),
            "cu_seqlens": make_cu_seqlens(seqlens), "scale": d ** -0.5}


def _normal(rng: np.random.Generator, shape, std: float, dtype: torch.dtype) -> torch.Tensor:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    return torch.from_numpy(x).to(dtype)


def torch_dtype(name: str) -> torch.dtype:
    return {"bf16": torch.bfloat16, "fp16": torch.float16}[name]


def make_inputs(cfg: WorkloadConfig, seed: Optional[int] = None, with_dout: Optional[bool] = None):
    """All inputs of one workload as CPU tensors/arrays (bf16/fp16 rounded once).

    Returns a dict with q, k, v (torch, cfg dtype), dout (torch or None),
    sel_idx (np.int32 [h_k, N, T]), cu_seqlens (np.int32 [S+1]) and scale.
    """
    rng = np.random.default_rng(cfg.seed if seed is None else seed)
    n, dt = cfg.n, torch_dtype(cfg.dtype)
    sel = make_selection(cfg.seqlens, cfg.h_k, cfg.block, cfg.topk, cfg.rule, rng)
    q = _normal(rng, (n, cfg.h_q, cfg.d), cfg.std, dt)
    k = _normal(rng, (n, cfg.h_k, cfg.d), cfg.std, dt)
    v = _normal(rng, (n, cfg.h_k, cfg.d), cfg.std, dt)
    want_dout = cfg.with_dout if with_dout is None else with_dout
    dout = _normal(rng, (n, cfg.h_q, cfg.d), 1.0, dt) if want_dout else None
    return {"q": q, "k": k, "v": v, "dout": dout, "sel_idx": sel,
            "cu_seqlens": make_cu_seqlens(cfg.seqlens), "scale": cfg.scale}


def keys_attended(seqlens: Sequence[int], block: int, topk: int) -> np.ndarray:
    """n(t) for the rule above: keys a token attends (independent of the random picks).

    Own block contributes r + 1 keys, each other selected block a full block:
    n(t) = (t mod B) + 1 + B * min(T - 1, t // B).  Used for useful-FLOP counts.
    """
    out = []
    for L in seqlens:
        t = np.arange(int(L), dtype=np.int64)
        c, r = t // block, t % block
        out.append(r + 1 + block * np.minimum(topk - 1, c))
    return np.concatenate(out)
