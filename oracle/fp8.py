"""e4m3 format, round-to-nearest-even and per-block FP8 quantisation (oracle).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Format ("FP8 GEMM on CDNA4", section 2.1; ZYFA post footnote 7): one sign
bit, 4 exponent bits with bias 7, 3 mantissa bits. Exponent field 0 holds the
subnormals m * 2^-9; the all-ones exponent with all-ones mantissa is NaN and
there is no infinity, so the largest finite magnitude is 448 (code 0x7E).
Normal values start at 2^-6; values below 2^-10 round to zero (ZYFA post,
"Precision and Underflow of FP8 Probabilities").

Rounding ("FP8 GEMM on CDNA4", section 2.3): round to the nearest code, ties
to the code with an even mantissa. Magnitudes above 448 saturate to 448
(a reading: the quantiser's x / scale never exceeds 448 by more than one
rounding, and the clamp of section 2.2 fixes the saturating behaviour).

Quantiser ("FP8 GEMM on CDNA4", section 2.2, at per-block granularity): for
each (batch, head, 128-token block) over the whole head dimension,
    amax  = max |y|,           y = x  or  y = FWHT128(x) / sqrt(128)
    scale = fl32(amax / 448)   (scale = 1 when amax < 1e-8)
    code  = RNE_e4m3(fl32(y / scale)),   dequantised value = code * scale.
The arithmetic is IEEE float32, emulated with numpy float32 operations, so
that codes and scales are fixed to the bit.

Hadamard rotation (ZYFA post, "FP8 Error in Full-Model Inference"): rows of
Q and K are multiplied by the normalised Sylvester Hadamard matrix
H_128 / sqrt(128) before quantisation; V is never rotated. In float32 the
transform is evaluated as the fast Walsh-Hadamard butterfly with stages of
span 1, 2, 4, ..., 64, each pair (a, b) -> (a + b, a - b) rounded to float32,
followed by one float32 multiply by fl32(1/sqrt(128)). The pages do not fix
the order; this order is the reading both implementations follow.
"""
from __future__ import annotations

import math

import numpy as np

E4M3_MAX = 448.0
BLOCK_TOKENS = 128
ZERO_GUARD = np.float32(1e-8)


def _e4m3_magnitude(code: int) -> float:
    """Value of a non-negative e4m3 code 0..126 from the format definition."""
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0:
        return m * 2.0 ** -9
    return (1.0 + m / 8.0) * 2.0 ** (e - 7)


# Magnitudes of the 127 finite non-negative codes; increasing with the code.
E4M3_VALUES = np.array([_e4m3_magnitude(c) for c in range(127)], dtype=np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """uint8 e4m3 codes -> float64 values (NaN for 0x7F / 0xFF)."""
    codes = np.asarray(codes, dtype=np.uint8)
    mag_code = (codes & 0x7F).astype(np.int64)
    table = np.concatenate([E4M3_VALUES, [np.nan]])
    mag = table[mag_code]
    return np.where(codes & 0x80, -mag, mag)


def e4m3_rne(q: np.ndarray, chunk: int = 1 << 22) -> np.ndarray:
    """Round float values to e4m3 codes: nearest code, ties to even mantissa,
    saturating at 448, sign kept (a negative value that rounds to zero gives
    0x80). The nearest code is found by searching the full table of codes.
    Large arrays are processed in chunks of `chunk` elements."""
    q = np.asarray(q)
    flat = q.reshape(-1)
    out = np.empty(flat.shape, dtype=np.uint8)
    for s in range(0, flat.size, chunk):
        out[s:s + chunk] = _e4m3_rne_flat(flat[s:s + chunk])
    return out.reshape(q.shape)


def _e4m3_rne_flat(q: np.ndarray) -> np.ndarray:
    q = np.asarray(q, dtype=np.float64)
    a = np.abs(q)
    idx = np.searchsorted(E4M3_VALUES, a, side="left")      # first value >= a
    hi = np.clip(idx, 0, 126)
    lo = np.clip(idx - 1, 0, 126)
    d_hi = np.abs(E4M3_VALUES[hi] - a)
    d_lo = np.abs(a - E4M3_VALUES[lo])
    pick_lo = (d_lo < d_hi) | ((d_lo == d_hi) & (lo % 2 == 0))
    mag = np.where(pick_lo, lo, hi)
    mag = np.where(a > E4M3_MAX, 126, mag)                   # saturate
    sign = np.signbit(q)
    return (mag | np.where(sign, 0x80, 0)).astype(np.uint8)


def fwht128_fp32(x: np.ndarray) -> np.ndarray:
    """Normalised 128-point Walsh-Hadamard transform along the last axis in
    float32: butterflies of span 1, 2, ..., 64, then multiply by
    fl32(1/sqrt(128))."""
    y = np.asarray(x, dtype=np.float32)
    n = y.shape[-1]
    assert n == 128, "the rotation is defined for head dimension 128"
    lead = y.shape[:-1]
    h = 1
    while h < n:
        z = y.reshape(lead + (n // (2 * h), 2, h))
        a = z[..., 0, :]
        b = z[..., 1, :]
        y = np.stack([a + b, a - b], axis=-2).reshape(lead + (n,))
        h *= 2
    c = np.float32(1.0 / math.sqrt(128.0))
    return (y * c).astype(np.float32)


def quantize_fp8(x: np.ndarray, hadamard: bool = False, block: int = BLOCK_TOKENS):
    """Per-block FP8 quantisation.

    x: [B, S, H, D] values exactly representable in float32 (the bf16 input).
    Returns (codes uint8 [B, S, H, D], scales float32 [B, H, ceil(S/block)]).
    Each (b, h, token block) is reduced on its own; a ragged last block uses
    only its own rows (the zero padding below cannot raise |y|'s maximum).
    """
    x = np.asarray(x, dtype=np.float32)
    B, S, H, D = x.shape
    y = fwht128_fp32(x) if hadamard else x
    nblk = (S + block - 1) // block
    pad = nblk * block - S
    if pad:
        y = np.concatenate([y, np.zeros((B, pad, H, D), np.float32)], axis=1)
    yb = y.reshape(B, nblk, block, H, D)
    amax = np.abs(yb).max(axis=(2, 4))                                   # [B, nblk, H], float32
    scale = np.where(amax < ZERO_GUARD, np.float32(1.0),
                     (amax / np.float32(E4M3_MAX)).astype(np.float32)).astype(np.float32)
    q = (yb / scale[:, :, None, :, None]).astype(np.float32)              # IEEE float32 division
    codes = e4m3_rne(q).reshape(B, nblk * block, H, D)[:, :S]
    return np.ascontiguousarray(codes), np.ascontiguousarray(scale.transpose(0, 2, 1))


def quantize_fp8_varlen(x: np.ndarray, cu_seqlens, hadamard: bool = False, block: int = BLOCK_TOKENS):
    """Packed variable-length x [T,H,D]: each sequence quantised on its own
    (its 128-token blocks never mix tokens of two sequences). Returns codes
    uint8 [T,H,D] and scales float32 [B,H,ceil(max_len/128)]; entries past a
    sequence's last block are NaN (never written)."""
    x = np.asarray(x)
    cu = [int(c) for c in cu_seqlens]
    B = len(cu) - 1
    max_len = max(cu[i + 1] - cu[i] for i in range(B))
    nb = (max_len + block - 1) // block
    codes = np.zeros(x.shape, dtype=np.uint8)
    scales = np.full((B, x.shape[1], nb), np.nan, dtype=np.float32)
    for i in range(B):
        s, e = cu[i], cu[i + 1]
        if e > s:
            c, sc = quantize_fp8(x[None, s:e], hadamard=hadamard, block=block)
            codes[s:e] = c[0]
            scales[i, :, :sc.shape[2]] = sc[0]
    return codes, scales


def dequantize_fp8_varlen(codes: np.ndarray, scales: np.ndarray, cu_seqlens, block: int = BLOCK_TOKENS):
    """Inverse of quantize_fp8_varlen: float64 [T,H,D]."""
    cu = [int(c) for c in cu_seqlens]
    out = np.zeros(codes.shape, dtype=np.float64)
    for i in range(len(cu) - 1):
        s, e = cu[i], cu[i + 1]
        if e > s:
            nb = (e - s + block - 1) // block
            out[s:e] = dequantize_fp8(codes[None, s:e], scales[i:i + 1, :, :nb], block=block)[0]
    return out


def dequantize_fp8(codes: np.ndarray, scales: np.ndarray, block: int = BLOCK_TOKENS):
    """codes [B,S,H,D] uint8, scales [B,H,nblk] -> float64 [B,S,H,D] = code * scale."""
    vals = e4m3_decode(codes)
    B, S, H, D = codes.shape
    tok_blk = np.arange(S) // block
    sc = np.asarray(scales, dtype=np.float64)[:, :, tok_blk]      # [B, H, S]
    return vals * np.transpose(sc, (0, 2, 1))[..., None]
