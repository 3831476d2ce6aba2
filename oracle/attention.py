"""Exact causal softmax attention in float64 (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition (ZYFA post, "Introduction" and "Methodology and Limitations":
causal forward attention with equal query and key lengths; grouped-query
heads as in the Mistral-7B / Qwen3-8B layers it times):

    O[b, i, h, :] = sum_{j <= i} softmax_j( scale * Q[b,i,h] . K[b,j,g(h)] ) V[b,j,g(h)]
    g(h) = h // (Hq / Hkv)

The softmax subtracts the row maximum before exponentiating. Nothing here
models FP8 probabilities, lean P or any kernel-internal rounding: for the FP8
path the oracle is this same definition applied to the dequantised inputs
(the ZYFA post, "Error of a Single Attention Call", compares kernels with fp64
attention on the same quantised inputs).
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np


def kv_head(h: int, Hq: int, Hkv: int) -> int:
    assert Hq % Hkv == 0
    return h // (Hq // Hkv)


def causal_probs(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """Probabilities of one head: q [S, D], k [S, D] -> P [S, S] (rows sum to 1,
    zero above the diagonal)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    S = q.shape[0]
    s = (q @ k.T) * scale
    mask = np.triu(np.ones((S, S), dtype=bool), k=1)
    s = np.where(mask, -np.inf, s)
    s = s - np.max(s, axis=1, keepdims=True)
    p = np.exp(s)
    return p / np.sum(p, axis=1, keepdims=True)


def causal_attention(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """q [B,S,Hq,Dqk], k [B,S,Hkv,Dqk], v [B,S,Hkv,Dv] -> O [B,S,Hq,Dv] float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, S, Hq, _ = q.shape
    Hkv = k.shape[2]
    out = np.empty((B, S, Hq, v.shape[3]), dtype=np.float64)
    for b in range(B):
        for h in range(Hq):
            g = kv_head(h, Hq, Hkv)
            p = causal_probs(q[b, :, h, :], k[b, :, g, :], scale)
            out[b, :, h, :] = p @ v[b, :, g, :]
    return out


def causal_attention_varlen(q: np.ndarray, k: np.ndarray, v: np.ndarray, cu_seqlens, scale: float) -> np.ndarray:
    """Packed variable-length batch: q [T,Hq,Dqk], k [T,Hkv,Dqk], v [T,Hkv,Dv];
    sequence i is tokens cu_seqlens[i] .. cu_seqlens[i+1]-1 and attends
    causally within itself only (the same definition applied to each
    sequence). Returns O [T,Hq,Dv] float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    out = np.zeros((q.shape[0], q.shape[1], v.shape[2]), dtype=np.float64)
    cu = [int(x) for x in cu_seqlens]
    for i in range(len(cu) - 1):
        s, e = cu[i], cu[i + 1]
        if e > s:
            out[s:e] = causal_attention(q[None, s:e], k[None, s:e], v[None, s:e], scale)[0]
    return out


def causal_attention_prefix(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    """Queries that continue a cached sequence (chunked prefill; the pages
    name paged caches as future work, "Methodology and Limitations"):
    q [Lq,Hq,Dqk] holds the last Lq positions of a sequence whose keys and
    values k [L,Hkv,Dqk], v [L,Hkv,Dv] cover all L >= Lq positions, a prefix
    of P = L - Lq cached tokens and then the new ones. Query i sits at
    position P + i and attends to keys 0 .. P + i: the causal definition
    above with the query index offset by P. Returns O [Lq,Hq,Dv] float64."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    Lq, Hq, _ = q.shape
    L, Hkv, _ = k.shape
    P = L - Lq
    assert P >= 0, "more queries than positions"
    allowed = np.arange(L)[None, :] <= (P + np.arange(Lq))[:, None]
    out = np.empty((Lq, Hq, v.shape[2]), dtype=np.float64)
    for h in range(Hq):
        g = kv_head(h, Hq, Hkv)
        s = np.where(allowed, (q[:, h, :] @ k[:, g, :].T) * scale, -np.inf)
        s = s - np.max(s, axis=1, keepdims=True)
        p = np.exp(s)
        out[:, h, :] = (p / np.sum(p, axis=1, keepdims=True)) @ v[:, g, :]
    return out


def causal_attention_rows(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                          b: int, h: int, rows: Iterable[int]) -> np.ndarray:
    """Selected output rows of one (batch, query head), one row at a time:
    row i attends to keys 0..i. Returns [len(rows), Dv] float64."""
    Hq = q.shape[2]
    Hkv = k.shape[2]
    g = kv_head(h, Hq, Hkv)
    res = []
    for i in rows:
        qi = np.asarray(q[b, i, h, :], dtype=np.float64)
        kk = np.asarray(k[b, : i + 1, g, :], dtype=np.float64)
        vv = np.asarray(v[b, : i + 1, g, :], dtype=np.float64)
        s = (kk @ qi) * scale
        s = s - np.max(s)
        p = np.exp(s)
        res.append((p / np.sum(p)) @ vv)
    return np.stack(res)


def causal_attention_rows_pquant(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float,
                                 b: int, h: int, rows: Iterable[int], block: int = 64) -> np.ndarray:
    """Selected output rows with the probabilities quantised the way the ZYFA
    post describes ("Per-Block Scaling and Normalization by the Rounded Row
    Sum"): the row's probabilities p (max-subtracted, as in the exact oracle)
    are cut into blocks of `block` keys; each block is multiplied by 2^kb with
    kb = floor(-log2(block max)), so its largest value lies in (0.5, 1]; the
    products are rounded to e4m3 (nearest, ties to even); the power of two is
    divided back out, giving weights W; the output is sum(W v) / sum(W), i.e.
    normalised by the sum of the rounded weights. A block whose probabilities
    all underflow to zero contributes nothing. Used only for the error-by-stage
    report (P-rounding error as the pages define it), not as a parity gate.
    Returns [len(rows), Dv] float64."""
    from . import fp8 as _fp8

    Hq = q.shape[2]
    Hkv = k.shape[2]
    g = kv_head(h, Hq, Hkv)
    res = []
    for i in rows:
        qi = np.asarray(q[b, i, h, :], dtype=np.float64)
        kk = np.asarray(k[b, : i + 1, g, :], dtype=np.float64)
        vv = np.asarray(v[b, : i + 1, g, :], dtype=np.float64)
        s = (kk @ qi) * scale
        p = np.exp(s - np.max(s))
        w = np.zeros_like(p)
        for c in range(0, p.size, block):
            pb = p[c:c + block]
            mb = float(np.max(pb))
            if mb <= 0.0:
                continue
            kb = math.floor(-math.log2(mb))
            codes = _fp8.e4m3_rne(np.ldexp(pb, kb))
            w[c:c + block] = np.ldexp(_fp8.e4m3_decode(codes), -kb)
        res.append((w @ vv) / np.sum(w))
    return np.stack(res)


def rel_l2(out: np.ndarray, ref: np.ndarray) -> float:
    """||out - ref||_2 / ||ref||_2 -- the relative RMS error of the ZYFA post
    ("Error of a Single Attention Call")."""
    out = np.asarray(out, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    den = np.linalg.norm(ref.ravel())
    return float(np.linalg.norm((out - ref).ravel()) / (den if den > 0 else 1.0))


def max_abs(out: np.ndarray, ref: Optional[np.ndarray]) -> float:
    return float(np.max(np.abs(np.asarray(out, np.float64) - np.asarray(ref, np.float64))))
