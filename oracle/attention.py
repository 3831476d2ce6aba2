"""Exact causal softmax attention in float64 (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Definition (ZYFA post, "Introduction" and "Methodology and Limitations":
causal forward attention with equal query and key lengths; grouped-query
heads as in the Mistral-7B / Qwen3-8B layers it times):

    O[b, i, h, :] = sum_{j <= i} softmax_j( scale * Q[b,i,h] . K[b,j,g(h)] ) V[b,j,g(h)]
    g(h) = h // (Hq / Hkv)

The softmax subtracts the row maximum before exponentiating. For the FP8
path the parity gate is this same definition applied to the dequantised
inputs (the ZYFA post, "Error of a Single Attention Call", compares kernels
with fp64 attention on the same quantised inputs). Three further functions
round the probabilities: causal_attention_rows_pquant the way the pages
describe (per-64-key powers of two; the error-by-stage report),
causal_attention_rows_window under the per-row offset window, the reading of
that scheme the GB300 FP8 path follows, and causal_attention_rows_bf16, the
BF16 path's stale running maximum with bf16 probabilities and their rounded
sum (tighter checks of the two paths' rounding). Nothing here models lean P.
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


# The probability rounding of the GB300 FP8 path, a reading of the ZYFA post
# ("Per-Block Scaling and Normalization by the Rounded Row Sum") for a tensor
# core that applies no per-row scale inside the PV product: each row keeps one
# power-of-two offset o for all its key tiles, moved (with the partial output
# and sum rescaled by the exact power of two) only when a tile's largest
# scaled probability leaves [2^WIN_LO, 2^WIN_HI]; o never drops more than
# WIN_FLOOR binades below the row's largest log2 value seen so far.
WIN_LO, WIN_HI, WIN_FLOOR = -4.0, 8.0, 64.0


def window_step(o: Optional[float], top: Optional[float], bm: float):
    """One key tile of the offset rule. bm: log2 of the tile's largest
    scaled probability before the offset (its largest base-2 score plus
    log2 of the tile's V scale); o, top: the row's offset and largest bm so
    far (None before the first tile). Returns the new (o, top): the first
    tile sets o = bm; a later tile moves o to max(bm, max(top, bm) - WIN_FLOOR)
    when bm - o > WIN_HI, or when bm - o < WIN_LO while bm lies within
    WIN_FLOOR binades of top; otherwise o stays."""
    if o is None:
        return bm, bm
    rel = bm - o
    if rel > WIN_HI or (rel < WIN_LO and bm > top - WIN_FLOOR):
        o = max(bm, max(top, bm) - WIN_FLOOR)
    return o, max(top, bm)


def lean_codes(y: np.ndarray) -> np.ndarray:
    """Lean P ("Lean P: Linear Approximation of the FP8 Code" in the ZYFA
    post): the e4m3 code of 2^t is taken as 8t + 56, which is exact at whole
    t (the code grows by 8 per doubling and 56 encodes 1.0). Here
    y = 1080 + 8t is rounded to the nearest integer, ties to even (float16
    has unit spacing in [1024, 2048)), values below 1024 give code 0, and the
    code is y - 1024. Returns the codes as uint8."""
    y = np.asarray(y, dtype=np.float64)
    n = np.rint(y)                              # nearest, ties to even
    n = np.where(y < 1023.5, 1024.0, n)
    return (n - 1024.0).astype(np.uint8)


def _window_tiles(qc, sq, k8, ks, v8, vs, c2, b, g, i, j_lo, j_hi, block, round_p, trace, lean=False):
    """Row i over key tiles j_lo .. j_hi - 1 in order, starting a fresh
    offset: returns (O, l, o) in units of the final offset o."""
    from . import fp8 as _fp8

    o = top = None
    acc = np.zeros(v8.shape[3], dtype=np.float64)
    l = 0.0
    for j in range(j_lo, j_hi):
        k0, k1 = j * block, min(j * block + block, i + 1)
        kc = _fp8.e4m3_decode(k8[b, k0:k1, g, :])
        vc = _fp8.e4m3_decode(v8[b, k0:k1, g, :])
        sk, sv = float(ks[b, g, j]), float(vs[b, g, j])
        x = (kc @ qc) * (sq * sk * c2)
        lsv = math.log2(sv)
        bm = float(np.max(x)) + lsv
        o_new, top = window_step(o, top, bm)
        if o is not None and o_new != o:
            f = 2.0 ** (o - o_new)
            acc *= f
            l *= f
        o = o_new
        if lean:
            p = _fp8.e4m3_decode(lean_codes(1080.0 + 8.0 * (x + lsv - o)))
        else:
            p = np.exp2(x + lsv - o)
            if round_p:
                p = _fp8.e4m3_decode(_fp8.e4m3_rne(p))
        acc += p @ vc
        l += float(np.sum(p)) / sv
        if trace is not None:
            trace.append((i, j, o))
    return acc, l, o


def causal_attention_rows_window(q8: np.ndarray, qs: np.ndarray, k8: np.ndarray, ks: np.ndarray,
                                 v8: np.ndarray, vs: np.ndarray, scale: float, b: int, h: int,
                                 rows: Iterable[int], block: int = 128, round_p: bool = True,
                                 trace: Optional[list] = None, chunk_tiles: int = 0,
                                 lean: bool = False) -> np.ndarray:
    """Selected output rows of the FP8 path with the probabilities rounded
    under the offset window above. Inputs are the e4m3 codes [B,S,H,D] and
    the per-(batch, head, 128-token block) scales [B,H,nblk] of Q, K, V.

    For row i, key tiles j = 0 .. i // block in order (tile j: keys j*block ..
    min(j*block + block, i + 1) - 1): base-2 scores x = (q_code . k_code) *
    sq * sk * scale / ln 2; bm = max x + log2 sv; the offset o follows
    window_step; the tile's probabilities P' = e4m3_RNE(2^(x + log2 sv - o))
    (unrounded when round_p is False); with earlier tiles scaled by
    2^(o_old - o) at each move, O = sum P' v_code and l = sum P' / sv, and
    the row's output is O / l. The weight on the dequantised value v_code * sv
    is P' 2^o / sv, so the weights sum to one exactly: the output is
    normalised by the sum of the rounded probabilities. With round_p False
    this is exact softmax attention on the dequantised inputs.

    chunk_tiles = C > 0: the key range split into chunks of C tiles (tiles
    cC .. min(cC + C, i // block + 1) - 1), each run as above from a fresh
    offset, and the chunks' (O_c, l_c, o_c) merged exactly: with M = max o_c,
    output = sum O_c 2^(o_c - M) / sum l_c 2^(o_c - M). lean: P' from
    lean_codes(1080 + 8 (x + log2 sv - o)) instead of the rounded
    exponential (same offsets, same normalisation by the sum of P'). trace,
    if given, receives (i, j, o) for every tile. Returns [len(rows), Dv]
    float64."""
    from . import fp8 as _fp8

    Hq = q8.shape[2]
    Hkv = k8.shape[2]
    g = kv_head(h, Hq, Hkv)
    c2 = scale / math.log(2.0)
    res = []
    for i in rows:
        qc = _fp8.e4m3_decode(q8[b, i, h, :])
        sq = float(qs[b, h, i // block])
        n = i // block + 1
        C = chunk_tiles if chunk_tiles > 0 else n
        parts = [_window_tiles(qc, sq, k8, ks, v8, vs, c2, b, g, i, j0, min(j0 + C, n), block, round_p, trace,
                               lean)
                 for j0 in range(0, n, C)]
        M = max(o for _, _, o in parts)
        acc = sum(a * 2.0 ** (o - M) for a, _, o in parts)
        l = sum(x * 2.0 ** (o - M) for _, x, o in parts)
        res.append(acc / l)
    return np.stack(res)


# The BF16 path's probabilities (a reading of the ZYFA post's normalisation
# by the rounded row sum, carried over to BF16): a running maximum m kept
# stale while no tile's maximum exceeds it by more than BF16_STALE binades,
# probabilities 2^(x - m) rounded to bf16 before the PV product, and the row
# sum taken over the rounded values.
BF16_STALE = 8.0


def bf16_rne(x: np.ndarray) -> np.ndarray:
    """Finite non-negative values rounded to float32, then to bf16 (nearest,
    ties to even), returned as float64."""
    f = np.ascontiguousarray(np.asarray(x, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


def stale_max_step(m: Optional[float], xmax: float) -> float:
    """One key tile of the BF16 running maximum: the first tile sets m to
    its maximum; a later tile moves m to its own maximum only when that
    exceeds m by more than BF16_STALE."""
    if m is None or xmax > m + BF16_STALE:
        return xmax
    return m


def causal_attention_rows_bf16(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, b: int, h: int,
                               rows: Iterable[int], block: int = 128, round_p: bool = True) -> np.ndarray:
    """Selected output rows of the BF16 path with its probability rounding:
    for row i, key tiles j = 0 .. i // block in order, base-2 scores
    x = (q . k) * scale / ln 2, m from stale_max_step (earlier tiles scaled by
    2^(m_old - m) when it moves), P = bf16(2^(x - m)) (unrounded when
    round_p is False), O = sum P v, l = sum P, output O / l: the weights sum
    to one exactly. With round_p False this is exact softmax attention.
    Returns [len(rows), Dv] float64."""
    Hq = q.shape[2]
    Hkv = k.shape[2]
    g = kv_head(h, Hq, Hkv)
    c2 = scale / math.log(2.0)
    res = []
    for i in rows:
        qi = np.asarray(q[b, i, h, :], dtype=np.float64)
        m = None
        acc = np.zeros(v.shape[3], dtype=np.float64)
        l = 0.0
        for j in range(i // block + 1):
            k0, k1 = j * block, min(j * block + block, i + 1)
            x = (np.asarray(k[b, k0:k1, g, :], dtype=np.float64) @ qi) * c2
            m_new = stale_max_step(m, float(np.max(x)))
            if m is not None and m_new != m:
                f = 2.0 ** (m - m_new)
                acc *= f
                l *= f
            m = m_new
            p = np.exp2(x - m)
            if round_p:
                p = bf16_rne(p)
            acc += p @ np.asarray(v[b, k0:k1, g, :], dtype=np.float64)
            l += float(np.sum(p))
        res.append(acc / l)
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
