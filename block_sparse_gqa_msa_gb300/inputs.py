"""Seeded synthetic inputs for block-sparse causal document-local GQA.

This module only draws random numbers and lays out index structures; it holds
none of the attention arithmetic, so both the CUDA path's tests and the CPU
oracle can consume it without sharing any method code.

Tensor shapes follow the flat-attention interface of the NeMo-Automodel PR
"feat(minimax-m3): add SM100 MSA sparse attention with custom backward"
(section "Design"): compact THD tensors Q[T,64,128], K/V[T,4,128], dO like Q,
an int32 selection q2k[4,T,16] of document-local key-block ids with -1 in
unused slots, and int32 document offsets [D+1].

The five workloads (``config(n)``, n = 1..5):
  1. one document, T=1024; a query in block b selects 0..b (dense causal);
  2. one document, T=16384; per (index head, query in block b >= 16): b, 0 and
     14 distinct blocks uniform on 1..b-1, sorted (all of 0..b when b < 16);
  3. one packed row of T=16384 real tokens, document lengths lognormal
     (median 1500, sigma 1) clipped to [128, 8192], drawn until they reach
     16384 with the last document truncated; selection as in 2, per document;
  4. eight such rows of S=16384, each losing a trailing U(0, 0.15) fraction
     of tokens as padding, concatenated (T ~ 1.2e5);
  5. one document, T=131072; 1 % of key rows scaled by 4; per (index head,
     query in block b >= 16): b, 0, b-1..b-6 and 8 distinct blocks from
     1..b-7 drawn with weight 1/(b-j) without replacement, sorted.
Values of Q, K, V, dO are i.i.d. N(0,1) rounded to bf16.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

NUM_Q_HEADS = 64
NUM_KV_HEADS = 4
HEAD_DIM = 128
BLOCK = 128
TOPK = 16

CONFIG_SEEDS = {1: 1001, 2: 1002, 3: 1003, 4: 1004, 5: 1005}


@dataclasses.dataclass
class Workload:
    name: str
    q: torch.Tensor          # bf16 [T,64,128], CPU
    k: torch.Tensor          # bf16 [T,4,128]
    v: torch.Tensor          # bf16 [T,4,128]
    do: torch.Tensor         # bf16 [T,64,128]
    q2k: torch.Tensor        # int32 [4,T,16]
    doc_offsets: torch.Tensor  # int32 [D+1]
    scale: float

    @property
    def T(self) -> int:
        return int(self.q.shape[0])

    @property
    def num_docs(self) -> int:
        return int(self.doc_offsets.numel() - 1)


def _normal_bf16(shape, seed: int) -> torch.Tensor:
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def dense_tensors(T: int, seed: int):
    """Q, K, V, dO as i.i.d. N(0,1) bf16, each from its own sub-seed."""
    q = _normal_bf16((T, NUM_Q_HEADS, HEAD_DIM), seed * 16 + 0)
    k = _normal_bf16((T, NUM_KV_HEADS, HEAD_DIM), seed * 16 + 1)
    v = _normal_bf16((T, NUM_KV_HEADS, HEAD_DIM), seed * 16 + 2)
    do = _normal_bf16((T, NUM_Q_HEADS, HEAD_DIM), seed * 16 + 3)
    return q, k, v, do


# ----------------------------------------------------------------- selections
def _fill_dense(q2k: np.ndarray, rows: slice, b: int) -> None:
    """All blocks 0..b ascending, then -1 (b < 16)."""
    q2k[:, rows, : b + 1] = np.arange(b + 1, dtype=np.int32)
    q2k[:, rows, b + 1:] = -1


def select_uniform(q2k: np.ndarray, start: int, length: int, rng: np.random.Generator) -> None:
    """Config-2 style selection for one document occupying rows [start, start+length)."""
    nblk = (length + BLOCK - 1) // BLOCK
    for b in range(nblk):
        lo = start + b * BLOCK
        hi = min(start + (b + 1) * BLOCK, start + length)
        rows = slice(lo, hi)
        if b < TOPK:
            _fill_dense(q2k, rows, b)
            continue
        n = hi - lo
        # 14 distinct blocks uniform on 1..b-1: the 14 smallest of b-1 uniform keys.
        keys = rng.random((NUM_KV_HEADS, n, b - 1))
        pick = np.argpartition(keys, 14, axis=2)[:, :, :14] + 1
        sel = np.concatenate(
            [np.full((NUM_KV_HEADS, n, 1), b), np.zeros((NUM_KV_HEADS, n, 1)), pick], axis=2
        ).astype(np.int32)
        q2k[:, rows, :] = np.sort(sel, axis=2)


def select_long(q2k: np.ndarray, start: int, length: int, rng: np.random.Generator) -> None:
    """Config-5 style selection: b, 0, b-1..b-6 and 8 blocks from 1..b-7 with
    weight 1/(b-j), drawn without replacement (Gumbel top-k)."""
    nblk = (length + BLOCK - 1) // BLOCK
    for b in range(nblk):
        lo = start + b * BLOCK
        hi = min(start + (b + 1) * BLOCK, start + length)
        rows = slice(lo, hi)
        if b < TOPK:
            _fill_dense(q2k, rows, b)
            continue
        n = hi - lo
        cand = np.arange(1, b - 6)  # 1..b-7
        logw = -np.log((b - cand).astype(np.float64))
        gumbel = -np.log(-np.log(rng.random((NUM_KV_HEADS, n, cand.size))))
        pick = cand[np.argpartition(-(logw + gumbel), 8, axis=2)[:, :, :8]]
        fixed = np.array([b, 0] + [b - i for i in range(1, 7)], dtype=np.int64)
        sel = np.concatenate(
            [np.broadcast_to(fixed, (NUM_KV_HEADS, n, 8)), pick], axis=2
        ).astype(np.int32)
        q2k[:, rows, :] = np.sort(sel, axis=2)


def packed_doc_lengths(total: int, rng: np.random.Generator) -> list[int]:
    """Lognormal(median 1500, sigma 1) lengths clipped to [128, 8192], drawn
    until they reach ``total``; the last one is truncated to fit."""
    lens: list[int] = []
    acc = 0
    while acc < total:
        x = int(round(rng.lognormal(mean=math.log(1500.0), sigma=1.0)))
        x = min(max(x, 128), 8192)
        x = min(x, total - acc)
        lens.append(x)
        acc += x
    return lens


def offsets_from_lengths(lens) -> np.ndarray:
    return np.concatenate([[0], np.cumsum(np.asarray(lens, dtype=np.int64))]).astype(np.int32)


def selection_for_docs(lens, rng: np.random.Generator, style: str = "uniform") -> np.ndarray:
    T = int(sum(lens))
    q2k = np.full((NUM_KV_HEADS, T, TOPK), -1, dtype=np.int32)
    start = 0
    for L in lens:
        if style == "uniform":
            select_uniform(q2k, start, L, rng)
        elif style == "long":
            select_long(q2k, start, L, rng)
        else:
            raise ValueError(style)
        start += L
    return q2k


# ----------------------------------------------------------------- configs
def config_structure(n: int, seed: int | None = None):
    """(doc lengths, q2k) for workload n, without the dense tensors."""
    seed = CONFIG_SEEDS[n] if seed is None else seed
    rng = np.random.default_rng(seed)
    if n == 1:
        lens = [1024]
        q2k = selection_for_docs(lens, rng)
    elif n == 2:
        lens = [16384]
        q2k = selection_for_docs(lens, rng)
    elif n == 3:
        lens = packed_doc_lengths(16384, rng)
        q2k = selection_for_docs(lens, rng)
    elif n == 4:
        lens = []
        for _ in range(8):
            row = packed_doc_lengths(16384, rng)
            drop = int(math.floor(rng.uniform(0.0, 0.15) * 16384))
            keep = 16384 - drop
            acc = 0
            for L in row:
                if acc >= keep:
                    break
                L = min(L, keep - acc)
                lens.append(L)
                acc += L
        q2k = selection_for_docs(lens, rng)
    elif n == 5:
        lens = [131072]
        q2k = selection_for_docs(lens, rng, style="long")
    else:
        raise ValueError(f"unknown workload {n}")
    return lens, q2k


def config(n: int, seed: int | None = None) -> Workload:
    seed = CONFIG_SEEDS[n] if seed is None else seed
    lens, q2k = config_structure(n, seed)
    T = int(sum(lens))
    q, k, v, do = dense_tensors(T, seed)
    if n == 5:
        rng = np.random.default_rng(seed + 7)
        rows = rng.choice(T, size=T // 100, replace=False)
        k[torch.from_numpy(rows)] = (k[torch.from_numpy(rows)].float() * 4.0).to(torch.bfloat16)
    names = {
        1: "single-doc T=1024 dense-causal top-16",
        2: "single-doc T=16384 top-16 uniform",
        3: "packed-docs T=16384 top-16 doc-local",
        4: "8 packed rows S=16384 minus padding, top-16 doc-local",
        5: "single-doc T=131072 top-16 near+harmonic, K outliers",
    }
    return Workload(
        name=names[n], q=q, k=k, v=v, do=do,
        q2k=torch.from_numpy(q2k), doc_offsets=torch.from_numpy(offsets_from_lengths(lens)),
        scale=1.0 / math.sqrt(HEAD_DIM),
    )


def custom(lens, seed: int, style: str = "uniform", q2k: np.ndarray | None = None,
           scale: float | None = None) -> Workload:
    """Workload with given document lengths (small parity / edge cases)."""
    rng = np.random.default_rng(seed)
    if q2k is None:
        q2k = selection_for_docs(lens, rng, style)
    T = int(sum(lens))
    q, k, v, do = dense_tensors(T, seed)
    return Workload(
        name=f"custom{list(lens)}", q=q, k=k, v=v, do=do,
        q2k=torch.from_numpy(np.ascontiguousarray(q2k, dtype=np.int32)),
        doc_offsets=torch.from_numpy(offsets_from_lengths(lens)),
        scale=(1.0 / math.sqrt(HEAD_DIM)) if scale is None else scale,
    )


def random_selection(lens, rng: np.random.Generator, p_empty: float = 0.2,
                     p_future: float = 0.1) -> np.ndarray:
    """Irregular selection for edge-case tests: uniform draws from the whole
    document (future blocks included), -1 slots and duplicates."""
    T = int(sum(lens))
    q2k = np.empty((NUM_KV_HEADS, T, TOPK), dtype=np.int32)
    start = 0
    for L in lens:
        nblk = (L + BLOCK - 1) // BLOCK
        for t in range(start, start + L):
            b = (t - start) // BLOCK
            hi = nblk if rng.random() < p_future else b + 1
            vals = rng.integers(0, hi, size=(NUM_KV_HEADS, TOPK))
            vals[rng.random((NUM_KV_HEADS, TOPK)) < p_empty] = -1
            q2k[:, t, :] = vals
        start += L
    return q2k
