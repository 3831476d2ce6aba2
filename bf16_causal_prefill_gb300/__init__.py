"""Causal prefill attention for NVIDIA GB300 (sm_103a): BF16 and per-block FP8.

Python binding of the C-ABI library ``libzyfa.so`` (declared in
``include/zyfa.h``). This module only marshals arguments: every step of the
computation runs in the library's CUDA kernels. There is no CPU fallback; if
the library is missing or the device is not sm_103, calls raise.

Entry points (names follow the C ABI):
  quantize_fp8(x, hadamard=False)            -> (codes uint8, scales float32)
  attn_fwd_bf16(q, k, v, softmax_scale=None) -> o (bf16)
  attn_fwd_fp8(q8, qs, k8, ks, v8, vs, ...)  -> o (bf16)
  prefill_fp8(q, k, v, hadamard=False)       -> o: quantise Q, K, V then FP8 attention
  device_status()                            -> raises ZyfaError on a kernel timeout

Tensors are [B, S, H, D] with the head dimension contiguous.
"""
from __future__ import annotations

import ctypes
import math
import os
from typing import Optional, Tuple

import torch

__all__ = [
    "ZyfaError", "lib", "quantize_fp8", "attn_fwd_bf16", "attn_fwd_fp8", "prefill_fp8",
    "device_status", "set_debug", "scale_blocks", "BLOCK_TOKENS",
]

BLOCK_TOKENS = 128
_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_PKG_DIR, "libzyfa.so")
_lib = None

_i64x3 = ctypes.c_int64 * 3


class ZyfaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"zyfa error {code}: {msg}")
        self.code = code


def lib() -> ctypes.CDLL:
    """Load libzyfa.so (built by ``__graft_entry__.build()`` / ``_build.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(_LIB_PATH):
        raise RuntimeError(
            f"{_LIB_PATH} is missing: build it with bf16_causal_prefill_gb300._build.build()")
    L = ctypes.CDLL(_LIB_PATH)
    vp, i64, c_int, c_float = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_float
    L.zyfa_status_string.restype = ctypes.c_char_p
    L.zyfa_status_string.argtypes = [c_int]
    L.zyfa_last_error_message.restype = ctypes.c_char_p
    L.zyfa_last_error_message.argtypes = []
    L.zyfa_version.restype = c_int
    L.zyfa_quantize_fp8.restype = c_int
    L.zyfa_quantize_fp8.argtypes = [vp, i64, i64, i64, vp, vp, c_int, c_int, c_int, c_int, c_int, vp]
    L.zyfa_attn_fwd_bf16.restype = c_int
    L.zyfa_attn_fwd_bf16.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                     vp, vp, vp, vp, vp]
    L.zyfa_attn_fwd_fp8.restype = c_int
    L.zyfa_attn_fwd_fp8.argtypes = [vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int,
                                    c_float, vp, vp, vp, vp, c_int, vp]
    L.zyfa_attn_fwd_bf16_rows.restype = c_int
    L.zyfa_attn_fwd_bf16_rows.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                          vp, vp, vp, vp, c_int, c_int, vp]
    L.zyfa_attn_fwd_fp8_rows.restype = c_int
    L.zyfa_attn_fwd_fp8_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int,
                                         c_float, vp, vp, vp, vp, c_int, c_int, c_int, vp]
    L.zyfa_attn_workspace_bytes.restype = ctypes.c_size_t
    L.zyfa_attn_workspace_bytes.argtypes = [c_int, c_int, c_int]
    L.zyfa_attn_split_tiles.restype = c_int
    L.zyfa_attn_split_tiles.argtypes = [c_int, c_int, c_int]
    L.zyfa_attn_fwd_bf16_ws.restype = c_int
    L.zyfa_attn_fwd_bf16_ws.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_float,
                                        vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.zyfa_attn_fwd_fp8_ws.restype = c_int
    L.zyfa_attn_fwd_fp8_ws.argtypes = [vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int,
                                       c_float, vp, vp, vp, vp, c_int, vp, ctypes.c_size_t, vp]
    L.zyfa_quantize_fp8_rows.restype = c_int
    L.zyfa_quantize_fp8_rows.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, vp, vp, c_int, c_int,
                                         c_int, c_int, c_int, c_int, c_int, vp]
    L.zyfa_quantize_fp8_qkv.restype = c_int
    L.zyfa_quantize_fp8_qkv.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp] + [c_int] * 7 + [vp]
    L.zyfa_quantize_fp8_qkv_rows.restype = c_int
    L.zyfa_quantize_fp8_qkv_rows.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp] + [c_int] * 9 + [vp]
    L.zyfa_quantize_fp8_qkv_varlen.restype = c_int
    L.zyfa_quantize_fp8_qkv_varlen.argtypes = [vp] * 13 + [c_int] * 6 + [vp]
    L.zyfa_quantize_fp8_qkv_varlen_dev.restype = c_int
    L.zyfa_quantize_fp8_qkv_varlen_dev.argtypes = [vp] * 13 + [c_int] * 8 + [vp, vp]
    L.zyfa_prefill_fp8_host_workspace.restype = ctypes.c_size_t
    L.zyfa_prefill_fp8_host_workspace.argtypes = [c_int] * 6
    L.zyfa_prefill_fp8_host.restype = c_int
    L.zyfa_prefill_fp8_host.argtypes = [vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_float, c_int,
                                        c_int, vp, ctypes.c_size_t, c_int, vp]
    L.zyfa_varlen_workspace_bytes.restype = ctypes.c_size_t
    L.zyfa_varlen_workspace_bytes.argtypes = []
    L.zyfa_quantize_fp8_varlen_dev.restype = c_int
    L.zyfa_quantize_fp8_varlen_dev.argtypes = [vp, ctypes.c_int64, ctypes.c_int64, vp, vp, vp, c_int, c_int, c_int,
                                               c_int, c_int, c_int, vp, vp]
    L.zyfa_attn_fwd_bf16_varlen_dev.restype = c_int
    L.zyfa_attn_fwd_bf16_varlen_dev.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_int, c_int,
                                                c_float, vp, vp, vp, vp, vp, vp]
    L.zyfa_attn_fwd_fp8_varlen_dev.restype = c_int
    L.zyfa_attn_fwd_fp8_varlen_dev.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                               c_int, c_int, c_float, vp, vp, vp, vp, vp, c_int, vp]
    L.zyfa_noalloc_scratch_bytes.restype = ctypes.c_size_t
    L.zyfa_noalloc_scratch_bytes.argtypes = []
    L.zyfa_attn_fwd_fp8_varlen_dev_noalloc.restype = c_int
    L.zyfa_attn_fwd_fp8_varlen_dev_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int,
                                                       c_int, c_int, c_int, c_float, vp, vp, vp, vp, c_int, vp]
    L.zyfa_quantize_fp8_varlen.restype = c_int
    L.zyfa_quantize_fp8_varlen.argtypes = [vp, i64, i64, vp, vp, vp, c_int, c_int, c_int, c_int, vp]
    L.zyfa_attn_fwd_bf16_varlen.restype = c_int
    L.zyfa_attn_fwd_bf16_varlen.argtypes = [vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int, c_float,
                                            vp, vp, vp, vp, vp]
    L.zyfa_attn_fwd_fp8_varlen.restype = c_int
    L.zyfa_attn_fwd_fp8_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, c_int, c_int, c_int, c_int, c_int,
                                           c_float, vp, vp, vp, vp, c_int, vp]
    L.zyfa_attn_fwd_bf16_paged.restype = c_int
    L.zyfa_attn_fwd_bf16_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, c_int, c_int, c_int, c_int, c_int, c_int,
                                           c_float, vp, vp, vp, vp, vp]
    L.zyfa_attn_fwd_fp8_paged.restype = c_int
    L.zyfa_attn_fwd_fp8_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, c_int, c_int, c_int, c_int,
                                          c_int, c_int, c_float, vp, vp, vp, vp, c_int, vp]
    L.zyfa_decode_workspace_bytes.restype = ctypes.c_size_t
    L.zyfa_decode_workspace_bytes.argtypes = [c_int, c_int, c_int]
    L.zyfa_attn_decode_bf16_paged.restype = c_int
    L.zyfa_attn_decode_bf16_paged.argtypes = [vp, vp, vp, vp, vp, vp, i64, c_int, c_int, c_int, c_int, c_int, c_int,
                                              c_float, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    L.zyfa_attn_decode_fp8_paged.restype = c_int
    L.zyfa_attn_decode_fp8_paged.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i64, c_int, c_int, c_int, c_int,
                                             c_int, c_int, c_float, vp, vp, vp, vp, vp, ctypes.c_size_t, c_int, vp]
    L.zyfa_get_device_status.restype = c_int
    L.zyfa_get_device_status.argtypes = [vp, ctypes.POINTER(ctypes.c_uint)]
    L.zyfa_set_debug.restype = c_int
    L.zyfa_set_debug.argtypes = [c_int, ctypes.c_double]
    _lib = L
    return L


def _check(rc: int) -> None:
    if rc != 0:
        L = lib()
        raise ZyfaError(rc, L.zyfa_last_error_message().decode() or L.zyfa_status_string(rc).decode())


def _stream_ptr(t: torch.Tensor, stream: Optional[torch.cuda.Stream]) -> int:
    s = stream if stream is not None else torch.cuda.current_stream(t.device)
    return s.cuda_stream


def _require(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError(f"{name} must be 4-D [B,S,H,D] with a contiguous last dim")


def _strides(t: torch.Tensor):
    return _i64x3(t.stride(0), t.stride(1), t.stride(2))


def scale_blocks(S: int) -> int:
    return (S + BLOCK_TOKENS - 1) // BLOCK_TOKENS


def quantize_fp8(x: torch.Tensor, hadamard: bool = False, out: Optional[torch.Tensor] = None,
                 scales: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None,
                 rows: Optional[Tuple[int, int]] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-(b, h, 128-token block) e4m3 quantisation of a bf16 [B,S,H,D] tensor.
    Returns (codes uint8 [B,S,H,D] dense, scales float32 [B,H,ceil(S/128)]).
    rows=(begin, end): only the blocks covering those tokens are written."""
    _require(x, "x", torch.bfloat16)
    B, S, H, D = x.shape
    if out is None:
        out = torch.empty((B, S, H, D), dtype=torch.uint8, device=x.device)
    if scales is None:
        scales = torch.empty((B, H, scale_blocks(S)), dtype=torch.float32, device=x.device)
    if not out.is_contiguous() or not scales.is_contiguous():
        raise ValueError("out and scales must be contiguous")
    if rows is None:
        _check(lib().zyfa_quantize_fp8(x.data_ptr(), x.stride(0), x.stride(1), x.stride(2), out.data_ptr(),
                                       scales.data_ptr(), B, S, H, D, int(bool(hadamard)),
                                       _stream_ptr(x, stream)))
    else:
        _check(lib().zyfa_quantize_fp8_rows(x.data_ptr(), x.stride(0), x.stride(1), x.stride(2), out.data_ptr(),
                                            scales.data_ptr(), B, S, H, D, int(bool(hadamard)), int(rows[0]),
                                            int(rows[1]), _stream_ptr(x, stream)))
    return out, scales


def quantize_fp8_qkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, hadamard: bool = False,
                     stream: Optional[torch.cuda.Stream] = None, rows: Optional[Tuple[int, int]] = None,
                     out=None):
    """Q, K and V of one attention call quantised in one launch (Q and K
    rotated when hadamard, V never): the bytes of three quantize_fp8 calls.
    Returns ((q8, qs), (k8, ks), (v8, vs)). out: the same structure of
    preallocated tensors to write into; rows=(begin, end) as quantize_fp8."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16)
    B, S, Hq, Dqk = q.shape
    Hkv, Dv = k.shape[2], v.shape[3]
    if out is None:
        out = tuple((torch.empty(t.shape, dtype=torch.uint8, device=t.device),
                     torch.empty((B, t.shape[2], scale_blocks(S)), dtype=torch.float32, device=t.device))
                    for t in (q, k, v))
    for c, sc in out:
        if not c.is_contiguous() or not sc.is_contiguous():
            raise ValueError("out and scales must be contiguous")
    (q8, qs), (k8, ks), (v8, vs) = out
    ptrs = (q.data_ptr(), _strides(q), k.data_ptr(), _strides(k), v.data_ptr(), _strides(v), q8.data_ptr(),
            qs.data_ptr(), k8.data_ptr(), ks.data_ptr(), v8.data_ptr(), vs.data_ptr())
    if rows is None:
        _check(lib().zyfa_quantize_fp8_qkv(*ptrs, B, S, Hq, Hkv, Dqk, Dv, int(bool(hadamard)),
                                           _stream_ptr(q, stream)))
    else:
        _check(lib().zyfa_quantize_fp8_qkv_rows(*ptrs, B, S, Hq, Hkv, Dqk, Dv, int(bool(hadamard)), int(rows[0]),
                                                int(rows[1]), _stream_ptr(q, stream)))
    return out


def _attn_workspace(B: int, S: int, Hq: int, device, split, stream):
    """(pointer, bytes, tensor) of the split-key-range workspace of an
    equal-length call: split=True allocates one when the library could split
    this problem (zyfa_attn_workspace_bytes > 0), a uint8 CUDA tensor is used
    as given, False gives none (the unsplit call)."""
    if split is False or split is None:
        return None, 0, None
    if isinstance(split, torch.Tensor):
        if not split.is_cuda or split.dtype != torch.uint8:
            raise ValueError("workspace must be a uint8 CUDA tensor")
        return split.data_ptr(), split.numel(), split
    n = lib().zyfa_attn_workspace_bytes(B, S, Hq)
    if n == 0:
        return None, 0, None
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    if stream is not None:
        ws.record_stream(stream)
    return ws.data_ptr(), ws.numel(), ws


def attn_fwd_bf16(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, softmax_scale: Optional[float] = None,
                  out: Optional[torch.Tensor] = None,
                  stream: Optional[torch.cuda.Stream] = None,
                  rows: Optional[Tuple[int, int]] = None, split=False) -> torch.Tensor:
    """Causal attention on bf16 q [B,S,Hq,Dqk], k [B,S,Hkv,Dqk], v [B,S,Hkv,Dv] -> o [B,S,Hq,Dv] bf16.
    rows=(begin, end): only those output rows (multiples of 256, or end = S).
    split=True (or a uint8 workspace tensor): small problems split each
    query-tile pair's keys across CTAs (zyfa_attn_fwd_bf16_ws); the result
    differs from the unsplit call in the last bits."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require(t, n, torch.bfloat16)
    B, S, Hq, Dqk = q.shape
    Hkv, Dv = k.shape[2], v.shape[3]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    _require(out, "out", torch.bfloat16)
    ws_ptr, ws_bytes, _ws = _attn_workspace(B, S, Hq, q.device, split, stream) if rows is None else (None, 0, None)
    if ws_ptr is not None:
        _check(lib().zyfa_attn_fwd_bf16_ws(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, Hq,
                                           Hkv, Dqk, Dv, float(softmax_scale), _strides(q), _strides(k),
                                           _strides(v), _strides(out), ws_ptr, ws_bytes, _stream_ptr(q, stream)))
    elif rows is None:
        _check(lib().zyfa_attn_fwd_bf16(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, Hq, Hkv,
                                        Dqk, Dv, float(softmax_scale), _strides(q), _strides(k), _strides(v),
                                        _strides(out), _stream_ptr(q, stream)))
    else:
        _check(lib().zyfa_attn_fwd_bf16_rows(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, Hq,
                                             Hkv, Dqk, Dv, float(softmax_scale), _strides(q), _strides(k),
                                             _strides(v), _strides(out), int(rows[0]), int(rows[1]),
                                             _stream_ptr(q, stream)))
    return out


def attn_fwd_fp8(q8: torch.Tensor, q_scale: torch.Tensor, k8: torch.Tensor, k_scale: torch.Tensor,
                 v8: torch.Tensor, v_scale: torch.Tensor, softmax_scale: Optional[float] = None,
                 out: Optional[torch.Tensor] = None,
                 stream: Optional[torch.cuda.Stream] = None,
                 rows: Optional[Tuple[int, int]] = None, lean_p: bool = False, split=False) -> torch.Tensor:
    """Causal attention on per-block e4m3 inputs (uint8 codes + float32 block scales) -> bf16 o.
    rows=(begin, end): only those output rows (multiples of 256, or end = S).
    split: as attn_fwd_bf16 (zyfa_attn_fwd_fp8_ws)."""
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _require(t, n, torch.uint8)
    for t, n in ((q_scale, "q_scale"), (k_scale, "k_scale"), (v_scale, "v_scale")):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous():
            raise ValueError(f"{n} must be a contiguous float32 CUDA tensor")
    B, S, Hq, Dqk = q8.shape
    Hkv, Dv = k8.shape[2], v8.shape[3]
    nb = scale_blocks(S)
    if q_scale.shape != (B, Hq, nb) or k_scale.shape != (B, Hkv, nb) or v_scale.shape != (B, Hkv, nb):
        raise ValueError("scale tensors must be [B, H, ceil(S/128)]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16, device=q8.device)
    _require(out, "out", torch.bfloat16)
    ws_ptr, ws_bytes, _ws = _attn_workspace(B, S, Hq, q8.device, split, stream) if rows is None else (None, 0, None)
    if ws_ptr is not None:
        _check(lib().zyfa_attn_fwd_fp8_ws(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(),
                                          v8.data_ptr(), v_scale.data_ptr(), out.data_ptr(), B, S, Hq, Hkv, Dqk,
                                          Dv, float(softmax_scale), _strides(q8), _strides(k8), _strides(v8),
                                          _strides(out), _fp8_flags(lean_p), ws_ptr, ws_bytes,
                                          _stream_ptr(q8, stream)))
    elif rows is None:
        _check(lib().zyfa_attn_fwd_fp8(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(),
                                       v8.data_ptr(), v_scale.data_ptr(), out.data_ptr(), B, S, Hq, Hkv, Dqk, Dv,
                                       float(softmax_scale), _strides(q8), _strides(k8), _strides(v8),
                                       _strides(out), _fp8_flags(lean_p), _stream_ptr(q8, stream)))
    else:
        _check(lib().zyfa_attn_fwd_fp8_rows(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(),
                                            v8.data_ptr(), v_scale.data_ptr(), out.data_ptr(), B, S, Hq, Hkv, Dqk,
                                            Dv, float(softmax_scale), _strides(q8), _strides(k8), _strides(v8),
                                            _strides(out), int(rows[0]), int(rows[1]), _fp8_flags(lean_p), _stream_ptr(q8, stream)))
    return out


def prefill_fp8(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, hadamard: bool = False,
                softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                stream: Optional[torch.cuda.Stream] = None, lean_p: bool = False, split=False):
    """The FP8 prefill path: quantise Q and K (optionally rotated) and V in
    one launch, then FP8 attention (split: as attn_fwd_fp8). Returns
    (o, (q8, qs, k8, ks, v8, vs))."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[3])
    (q8, qs), (k8, ks), (v8, vs) = quantize_fp8_qkv(q, k, v, hadamard, stream=stream)
    o = attn_fwd_fp8(q8, qs, k8, ks, v8, vs, softmax_scale, out=out, stream=stream, lean_p=lean_p, split=split)
    return o, (q8, qs, k8, ks, v8, vs)


def prefill_fp8_host_workspace(B: int, S: int, Hq: int, Hkv: int, Dqk: int, Dv: int,
                               device=None) -> torch.Tensor:
    """Device workspace (uint8) for prefill_fp8_host at these sizes."""
    n = lib().zyfa_prefill_fp8_host_workspace(B, S, Hq, Hkv, Dqk, Dv)
    if n == 0:
        raise ValueError("invalid sizes")
    return torch.empty(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def prefill_fp8_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, hadamard: bool = False,
                     softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                     n_chunks: int = 0, workspace: Optional[torch.Tensor] = None,
                     stream: Optional[torch.cuda.Stream] = None, lean_p: bool = False) -> torch.Tensor:
    """The FP8 prefill on page-locked host tensors: copies in, quantisation,
    attention and the copy of O back run as one pipeline along the sequence.
    Returns the page-locked host o; it is valid once the stream (default: the
    current one) has been synchronised."""
    for t, name in ((q, "q"), (k, "k"), (v, "v")):
        if t.dtype != torch.bfloat16 or t.is_cuda or not t.is_contiguous() or not t.is_pinned():
            raise ValueError(f"{name} must be a dense, page-locked host bf16 tensor")
    B, S, Hq, Dqk = q.shape
    Hkv, Dv = k.shape[2], v.shape[3]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((B, S, Hq, Dv), dtype=torch.bfloat16).pin_memory()
    if workspace is None:
        workspace = prefill_fp8_host_workspace(B, S, Hq, Hkv, Dqk, Dv)
    s = stream if stream is not None else torch.cuda.current_stream(workspace.device)
    _check(lib().zyfa_prefill_fp8_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), B, S, Hq, Hkv,
                                       Dqk, Dv, float(softmax_scale), int(bool(hadamard)), int(n_chunks),
                                       workspace.data_ptr(), workspace.numel(), _fp8_flags(lean_p), s.cuda_stream))
    return out


# ------------------------------------------------------ packed varlen batches
def _cu_host(cu_seqlens) -> Tuple[ctypes.Array, int, int]:
    """Host int32 copy of cu_seqlens (list, numpy array or tensor; a CUDA
    tensor is copied to the host, which synchronises). Returns the ctypes
    array, B and the longest sequence."""
    if isinstance(cu_seqlens, torch.Tensor):
        vals = [int(x) for x in cu_seqlens.detach().to("cpu", torch.int64).tolist()]
    else:
        vals = [int(x) for x in cu_seqlens]
    if len(vals) < 2:
        raise ValueError("cu_seqlens needs at least two entries")
    arr = (ctypes.c_int32 * len(vals))(*vals)
    max_len = max(vals[i + 1] - vals[i] for i in range(len(vals) - 1))
    return arr, len(vals) - 1, max_len


def _cu_device(cu_seqlens, max_seqlen: Optional[int], device) -> Optional[Tuple[int, int, int]]:
    """(pointer, B, max_seqlen) when cu_seqlens is an int32 CUDA tensor and the
    caller gave max_seqlen: the offsets stay on the device (no host read, no
    synchronisation). None otherwise (the host path)."""
    if max_seqlen is None or not isinstance(cu_seqlens, torch.Tensor) or not cu_seqlens.is_cuda:
        return None
    if cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or not cu_seqlens.is_contiguous():
        raise ValueError("device cu_seqlens must be a contiguous 1-D int32 CUDA tensor")
    if cu_seqlens.device != device:
        raise ValueError("cu_seqlens must be on the same device as the tensors")
    if cu_seqlens.numel() < 2:
        raise ValueError("cu_seqlens needs at least two entries")
    return cu_seqlens.data_ptr(), cu_seqlens.numel() - 1, int(max_seqlen)


def _varlen_workspace(device, stream: Optional[torch.cuda.Stream]) -> torch.Tensor:
    ws = torch.empty(lib().zyfa_varlen_workspace_bytes(), dtype=torch.uint8, device=device)
    if stream is not None:
        ws.record_stream(stream)
    return ws


def _require_packed(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != 3 or t.stride(2) != 1:
        raise ValueError(f"{name} must be 3-D [T,H,D] with a contiguous last dim")


def _fp8_flags(lean_p: bool) -> int:
    """The flags word of the FP8 attention calls: lean P (head dim 128) or exact P."""
    return 1 if lean_p else 0


def _i64x2(a: int, b: int):
    return (ctypes.c_int64 * 2)(a, b)


def _strides2(t: torch.Tensor):
    return _i64x2(t.stride(0), t.stride(1))


def quantize_fp8_varlen(x: torch.Tensor, cu_seqlens, hadamard: bool = False,
                        stream: Optional[torch.cuda.Stream] = None,
                        max_seqlen: Optional[int] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-(sequence, head, 128-token block) e4m3 quantisation of a packed bf16
    [T,H,D] tensor. Returns (codes uint8 [T,H,D], scales float32
    [B,H,ceil(max_len/128)]). An int32 CUDA cu_seqlens with max_seqlen given
    stays on the device (scales then [B,H,ceil(max_seqlen/128)])."""
    _require_packed(x, "x", torch.bfloat16)
    T, H, D = x.shape
    out = torch.empty((T, H, D), dtype=torch.uint8, device=x.device)
    dev = _cu_device(cu_seqlens, max_seqlen, x.device)
    if dev is not None:
        cu_ptr, B, max_len = dev
        scales = torch.zeros((B, H, scale_blocks(max_len)), dtype=torch.float32, device=x.device)
        ws = _varlen_workspace(x.device, stream)
        _check(lib().zyfa_quantize_fp8_varlen_dev(x.data_ptr(), x.stride(0), x.stride(1), out.data_ptr(),
                                                  scales.data_ptr(), cu_ptr, B, T, max_len, H, D,
                                                  int(bool(hadamard)), ws.data_ptr(), _stream_ptr(x, stream)))
        return out, scales
    cu, B, max_len = _cu_host(cu_seqlens)
    scales = torch.zeros((B, H, scale_blocks(max_len)), dtype=torch.float32, device=x.device)
    _check(lib().zyfa_quantize_fp8_varlen(x.data_ptr(), x.stride(0), x.stride(1), out.data_ptr(), scales.data_ptr(),
                                          cu, B, H, D, int(bool(hadamard)), _stream_ptr(x, stream)))
    return out, scales


def quantize_fp8_qkv_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens, hadamard: bool = False,
                            stream: Optional[torch.cuda.Stream] = None, max_seqlen: Optional[int] = None):
    """Q, K and V of a packed variable-length batch quantised in one launch
    (the bytes of three quantize_fp8_varlen calls). Returns ((q8, qs),
    (k8, ks), (v8, vs)); device offsets as quantize_fp8_varlen."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require_packed(t, n, torch.bfloat16)
    T, Hq, Dqk = q.shape
    Hkv, Dv = k.shape[1], v.shape[2]
    dev = _cu_device(cu_seqlens, max_seqlen, q.device)
    if dev is not None:
        cu_ptr, B, max_len = dev
    else:
        cu, B, max_len = _cu_host(cu_seqlens)
    out = tuple((torch.empty(t.shape, dtype=torch.uint8, device=t.device),
                 torch.zeros((B, t.shape[1], scale_blocks(max_len)), dtype=torch.float32, device=t.device))
                for t in (q, k, v))
    (q8, qs), (k8, ks), (v8, vs) = out
    ptrs = (q.data_ptr(), _strides2(q), k.data_ptr(), _strides2(k), v.data_ptr(), _strides2(v), q8.data_ptr(),
            qs.data_ptr(), k8.data_ptr(), ks.data_ptr(), v8.data_ptr(), vs.data_ptr())
    if dev is not None:
        ws = _varlen_workspace(q.device, stream)
        _check(lib().zyfa_quantize_fp8_qkv_varlen_dev(*ptrs, cu_ptr, B, T, max_len, Hq, Hkv, Dqk, Dv,
                                                      int(bool(hadamard)), ws.data_ptr(), _stream_ptr(q, stream)))
    else:
        _check(lib().zyfa_quantize_fp8_qkv_varlen(*ptrs, cu, B, Hq, Hkv, Dqk, Dv, int(bool(hadamard)),
                                                  _stream_ptr(q, stream)))
    return out


def attn_fwd_bf16_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens,
                         softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                         stream: Optional[torch.cuda.Stream] = None,
                         max_seqlen: Optional[int] = None) -> torch.Tensor:
    """Causal attention over a packed variable-length batch: q [T,Hq,Dqk],
    k [T,Hkv,Dqk], v [T,Hkv,Dv] -> o [T,Hq,Dv] bf16; each sequence attends to
    itself only. An int32 CUDA cu_seqlens with max_seqlen given stays on the
    device."""
    for t, n in ((q, "q"), (k, "k"), (v, "v")):
        _require_packed(t, n, torch.bfloat16)
    T, Hq, Dqk = q.shape
    Hkv, Dv = k.shape[1], v.shape[2]
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    _require_packed(out, "out", torch.bfloat16)
    dev = _cu_device(cu_seqlens, max_seqlen, q.device)
    if dev is not None:
        cu_ptr, B, max_len = dev
        ws = _varlen_workspace(q.device, stream)
        _check(lib().zyfa_attn_fwd_bf16_varlen_dev(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), cu_ptr,
                                                   B, T, max_len, Hq, Hkv, Dqk, Dv, float(softmax_scale),
                                                   _strides2(q), _strides2(k), _strides2(v), _strides2(out),
                                                   ws.data_ptr(), _stream_ptr(q, stream)))
        return out
    cu, B, _ = _cu_host(cu_seqlens)
    _check(lib().zyfa_attn_fwd_bf16_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), cu, B, Hq,
                                           Hkv, Dqk, Dv, float(softmax_scale), _strides2(q), _strides2(k),
                                           _strides2(v), _strides2(out), _stream_ptr(q, stream)))
    return out


def attn_fwd_fp8_varlen(q8: torch.Tensor, q_scale: torch.Tensor, k8: torch.Tensor, k_scale: torch.Tensor,
                        v8: torch.Tensor, v_scale: torch.Tensor, cu_seqlens, softmax_scale: Optional[float] = None,
                        out: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None,
                        max_seqlen: Optional[int] = None, lean_p: bool = False) -> torch.Tensor:
    """FP8 causal attention over a packed variable-length batch (codes and
    scales as written by quantize_fp8_varlen) -> bf16 o [T,Hq,Dv]. An int32
    CUDA cu_seqlens with max_seqlen given stays on the device."""
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _require_packed(t, n, torch.uint8)
    T, Hq, Dqk = q8.shape
    Hkv, Dv = k8.shape[1], v8.shape[2]
    dev = _cu_device(cu_seqlens, max_seqlen, q8.device)
    if dev is not None:
        cu_ptr, B, max_len = dev
        cu = None
    else:
        cu, B, max_len = _cu_host(cu_seqlens)
    nb = scale_blocks(max_len)
    for t, n, h in ((q_scale, "q_scale", Hq), (k_scale, "k_scale", Hkv), (v_scale, "v_scale", Hkv)):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (B, h, nb):
            raise ValueError(f"{n} must be a contiguous float32 CUDA tensor [B, H, ceil(max_len/128)]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=q8.device)
    _require_packed(out, "out", torch.bfloat16)
    if dev is not None:
        ws = _varlen_workspace(q8.device, stream)
        _check(lib().zyfa_attn_fwd_fp8_varlen_dev(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(),
                                                  k_scale.data_ptr(), v8.data_ptr(), v_scale.data_ptr(),
                                                  out.data_ptr(), cu_ptr, B, T, max_len, Hq, Hkv, Dqk, Dv,
                                                  float(softmax_scale), _strides2(q8), _strides2(k8), _strides2(v8),
                                                  _strides2(out), ws.data_ptr(), _fp8_flags(lean_p), _stream_ptr(q8, stream)))
        return out
    _check(lib().zyfa_attn_fwd_fp8_varlen(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(), k_scale.data_ptr(),
                                          v8.data_ptr(), v_scale.data_ptr(), out.data_ptr(), cu, B, Hq, Hkv, Dqk,
                                          Dv, float(softmax_scale), _strides2(q8), _strides2(k8), _strides2(v8),
                                          _strides2(out), _fp8_flags(lean_p), _stream_ptr(q8, stream)))
    return out


def attn_fwd_fp8_varlen_dev_noalloc(q8: torch.Tensor, q_scale: torch.Tensor, k8: torch.Tensor,
                                    k_scale: torch.Tensor, v8: torch.Tensor, v_scale: torch.Tensor,
                                    cu_seqlens: torch.Tensor, max_seqlen: int, out: torch.Tensor,
                                    softmax_scale: Optional[float] = None,
                                    stream: Optional[torch.cuda.Stream] = None, lean_p: bool = False) -> torch.Tensor:
    """attn_fwd_fp8_varlen with device offsets for callers that cannot
    allocate device memory on the call path (a replayed CUDA graph with fixed
    memory, a serving loop drawing only from its own pool): the library keeps
    the call's unit table in a static 32 KB device array instead of a
    workspace, so neither this function nor the library allocates; the caller
    passes every input and the output `out` [T,Hq,Dv] bf16. Calls that can
    overlap on the GPU share that array and must not be issued concurrently.
    Results are bitwise those of attn_fwd_fp8_varlen(..., max_seqlen=...)."""
    for t, n in ((q8, "q8"), (k8, "k8"), (v8, "v8")):
        _require_packed(t, n, torch.uint8)
    _require_packed(out, "out", torch.bfloat16)
    T, Hq, Dqk = q8.shape
    Hkv, Dv = k8.shape[1], v8.shape[2]
    dev = _cu_device(cu_seqlens, max_seqlen, q8.device)
    if dev is None:
        raise ValueError("cu_seqlens must be an int32 CUDA tensor and max_seqlen must be given")
    cu_ptr, B, max_len = dev
    nb = scale_blocks(max_len)
    for t, n, h in ((q_scale, "q_scale", Hq), (k_scale, "k_scale", Hkv), (v_scale, "v_scale", Hkv)):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (B, h, nb):
            raise ValueError(f"{n} must be a contiguous float32 CUDA tensor [B, H, ceil(max_seqlen/128)]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    _check(lib().zyfa_attn_fwd_fp8_varlen_dev_noalloc(q8.data_ptr(), q_scale.data_ptr(), k8.data_ptr(),
                                                      k_scale.data_ptr(), v8.data_ptr(), v_scale.data_ptr(),
                                                      out.data_ptr(), cu_ptr, B, T, max_len, Hq, Hkv, Dqk, Dv,
                                                      float(softmax_scale), _strides2(q8), _strides2(k8),
                                                      _strides2(v8), _strides2(out), _fp8_flags(lean_p), _stream_ptr(q8, stream)))
    return out


def prefill_fp8_varlen(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, cu_seqlens, hadamard: bool = False,
                       softmax_scale: Optional[float] = None, stream: Optional[torch.cuda.Stream] = None,
                       max_seqlen: Optional[int] = None, lean_p: bool = False):
    """The FP8 prefill path over a packed variable-length batch. Returns
    (o, (q8, qs, k8, ks, v8, vs))."""
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(q.shape[2])
    (q8, qs), (k8, ks), (v8, vs) = quantize_fp8_qkv_varlen(q, k, v, cu_seqlens, hadamard, stream=stream,
                                                           max_seqlen=max_seqlen)
    o = attn_fwd_fp8_varlen(q8, qs, k8, ks, v8, vs, cu_seqlens, softmax_scale, stream=stream, max_seqlen=max_seqlen,
                            lean_p=lean_p)
    return o, (q8, qs, k8, ks, v8, vs)


def _require_cache(t: torch.Tensor, name: str, dtype: torch.dtype) -> None:
    _require(t, name, dtype)
    if t.shape[1] != 128:
        raise ValueError(f"{name} must be [num_pages, 128, H, D] (pages of 128 tokens)")


def _paged_meta(cu_seqlens_q, ctx_lens, block_table: torch.Tensor, device):
    cu, B, max_len = _cu_host(cu_seqlens_q)
    if isinstance(ctx_lens, torch.Tensor):
        ctx_vals = [int(x) for x in ctx_lens.detach().to("cpu", torch.int64).tolist()]
    else:
        ctx_vals = [int(x) for x in ctx_lens]
    if len(ctx_vals) != B:
        raise ValueError("ctx_lens needs one entry per sequence")
    ctx = (ctypes.c_int32 * B)(*ctx_vals)
    if (not block_table.is_cuda or block_table.dtype != torch.int32 or block_table.dim() != 2
            or block_table.stride(1) != 1 or block_table.shape[0] != B):
        raise ValueError("block_table must be an int32 CUDA tensor [B, max_pages] with a contiguous last dim")
    if block_table.device != device:
        raise ValueError("block_table must be on the same device as the tensors")
    return cu, ctx, B, max_len


def quantize_fp8_cache(cache: torch.Tensor, hadamard: bool = False,
                       stream: Optional[torch.cuda.Stream] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """Per-(page, head) e4m3 quantisation of a paged bf16 cache
    [num_pages, 128, H, D] (each page is one 128-token block). Returns
    (codes uint8 [num_pages, 128, H, D], scales float32 [num_pages, H])."""
    _require_cache(cache, "cache", torch.bfloat16)
    codes, scales = quantize_fp8(cache, hadamard, stream=stream)
    return codes, scales.view(cache.shape[0], cache.shape[2])


def attn_fwd_bf16_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, cu_seqlens_q, ctx_lens,
                        block_table: torch.Tensor, softmax_scale: Optional[float] = None,
                        out: Optional[torch.Tensor] = None,
                        stream: Optional[torch.cuda.Stream] = None) -> torch.Tensor:
    """Packed queries q [T,Hq,Dqk] of B sequences that continue cached ones:
    sequence i has ctx_lens[i] cached tokens and its new
    tokens' queries are rows cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1; its
    keys/values, new tokens included, are the pages block_table[i] of
    k_cache/v_cache [num_pages,128,Hkv,D]. Query j attends to positions
    0 .. ctx_lens[i] + j. Returns o [T,Hq,Dv] bf16."""
    _require_packed(q, "q", torch.bfloat16)
    _require_cache(k_cache, "k_cache", torch.bfloat16)
    _require_cache(v_cache, "v_cache", torch.bfloat16)
    T, Hq, Dqk = q.shape
    Hkv, Dv = k_cache.shape[2], v_cache.shape[3]
    cu, ctx, B, _ = _paged_meta(cu_seqlens_q, ctx_lens, block_table, q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    _require_packed(out, "out", torch.bfloat16)
    _check(lib().zyfa_attn_fwd_bf16_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(), cu,
                                          ctx, block_table.data_ptr(), block_table.stride(0), k_cache.shape[0], B,
                                          Hq, Hkv, Dqk, Dv, float(softmax_scale), _strides2(q), _strides(k_cache),
                                          _strides(v_cache), _strides2(out), _stream_ptr(q, stream)))
    return out


def attn_fwd_fp8_paged(q8: torch.Tensor, q_scale: torch.Tensor, k_cache8: torch.Tensor, k_scale: torch.Tensor,
                       v_cache8: torch.Tensor, v_scale: torch.Tensor, cu_seqlens_q, ctx_lens,
                       block_table: torch.Tensor, softmax_scale: Optional[float] = None,
                       out: Optional[torch.Tensor] = None,
                       stream: Optional[torch.cuda.Stream] = None, lean_p: bool = False) -> torch.Tensor:
    """FP8 form of attn_fwd_bf16_paged: q8/q_scale from quantize_fp8_varlen on
    the packed queries, k/v caches and their [num_pages, Hkv] scales from
    quantize_fp8_cache. Returns o [T,Hq,Dv] bf16."""
    _require_packed(q8, "q8", torch.uint8)
    _require_cache(k_cache8, "k_cache8", torch.uint8)
    _require_cache(v_cache8, "v_cache8", torch.uint8)
    T, Hq, Dqk = q8.shape
    P, Hkv, Dv = k_cache8.shape[0], k_cache8.shape[2], v_cache8.shape[3]
    cu, ctx, B, max_len = _paged_meta(cu_seqlens_q, ctx_lens, block_table, q8.device)
    if (not q_scale.is_cuda or q_scale.dtype != torch.float32 or not q_scale.is_contiguous()
            or tuple(q_scale.shape) != (B, Hq, scale_blocks(max_len))):
        raise ValueError("q_scale must be a contiguous float32 CUDA tensor [B, Hq, ceil(max_len/128)]")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != P * Hkv:
            raise ValueError(f"{n} must be a contiguous float32 CUDA tensor [num_pages, Hkv]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((T, Hq, Dv), dtype=torch.bfloat16, device=q8.device)
    _require_packed(out, "out", torch.bfloat16)
    _check(lib().zyfa_attn_fwd_fp8_paged(q8.data_ptr(), q_scale.data_ptr(), k_cache8.data_ptr(), k_scale.data_ptr(),
                                         v_cache8.data_ptr(), v_scale.data_ptr(), out.data_ptr(), cu, ctx,
                                         block_table.data_ptr(), block_table.stride(0), P, B, Hq, Hkv, Dqk, Dv,
                                         float(softmax_scale), _strides2(q8), _strides(k_cache8), _strides(v_cache8),
                                         _strides2(out), _fp8_flags(lean_p), _stream_ptr(q8, stream)))
    return out


def _decode_meta(seq_lens, block_table: torch.Tensor, N: int, device):
    if isinstance(seq_lens, torch.Tensor):
        vals = [int(x) for x in seq_lens.detach().to("cpu", torch.int64).tolist()]
    else:
        vals = [int(x) for x in seq_lens]
    if len(vals) != N:
        raise ValueError("seq_lens needs one entry per token of q")
    if (not block_table.is_cuda or block_table.dtype != torch.int32 or block_table.dim() != 2
            or block_table.stride(1) != 1 or block_table.shape[0] != N):
        raise ValueError("block_table must be an int32 CUDA tensor [N, max_pages] with a contiguous last dim")
    if block_table.device != device:
        raise ValueError("block_table must be on the same device as the tensors")
    return (ctypes.c_int32 * N)(*vals)


def _decode_workspace(N: int, Hq: int, Hkv: int, device, split, stream):
    """(pointer, bytes, tensor) of the split-key-range workspace: split=True
    allocates one, a uint8 CUDA tensor is used as given, False/None gives none.
    split=True allocates nothing when the library would use the workspace for
    neither a split (considered only while N*Hkv < 4 x the SM count) nor
    replicated rows (groups of at most 32 query heads)."""
    if split is False or split is None:
        return None, 0, None
    if isinstance(split, torch.Tensor):
        if not split.is_cuda or split.dtype != torch.uint8:
            raise ValueError("workspace must be a uint8 CUDA tensor")
        return split.data_ptr(), split.numel(), split
    sms = torch.cuda.get_device_properties(device).multi_processor_count
    if Hq // Hkv > 32 and N * Hkv >= 4 * sms:
        return None, 0, None
    ws = torch.empty(lib().zyfa_decode_workspace_bytes(N, Hq, Hkv), dtype=torch.uint8, device=device)
    if stream is not None:
        ws.record_stream(stream)
    return ws.data_ptr(), ws.numel(), ws


def quantize_fp8_decode(q: torch.Tensor, stream: Optional[torch.cuda.Stream] = None,
                        hadamard: bool = False) -> Tuple[torch.Tensor, torch.Tensor]:
    """e4m3 codes of decode queries q [N,Hq,D] with one scale per token and
    head. Returns (codes uint8 [N,Hq,D], scales float32 [N,Hq])."""
    _require_packed(q, "q", torch.bfloat16)
    codes, scales = quantize_fp8_varlen(q, list(range(q.shape[0] + 1)), hadamard, stream=stream)
    return codes, scales.view(q.shape[0], q.shape[1])


def attn_decode_bf16_paged(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, seq_lens,
                           block_table: torch.Tensor, softmax_scale: Optional[float] = None,
                           out: Optional[torch.Tensor] = None,
                           stream: Optional[torch.cuda.Stream] = None, split=True) -> torch.Tensor:
    """One decode step: q [N,Hq,Dqk] holds each sequence's new token (its K/V
    already in the cache); sequence i has seq_lens[i] positions, the new one
    included, in pages block_table[i] of k_cache/v_cache [num_pages,128,Hkv,D].
    split: True (allocate a workspace so long key ranges may be split across
    SMs), a uint8 CUDA workspace tensor, or False (no split: the bytes of the
    paged prefill with one new token). Returns o [N,Hq,Dv] bf16."""
    _require_packed(q, "q", torch.bfloat16)
    _require_cache(k_cache, "k_cache", torch.bfloat16)
    _require_cache(v_cache, "v_cache", torch.bfloat16)
    N, Hq, Dqk = q.shape
    Hkv, Dv = k_cache.shape[2], v_cache.shape[3]
    lens = _decode_meta(seq_lens, block_table, N, q.device)
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((N, Hq, Dv), dtype=torch.bfloat16, device=q.device)
    _require_packed(out, "out", torch.bfloat16)
    ws_ptr, ws_bytes, _ws = _decode_workspace(N, Hq, Hkv, q.device, split, stream)
    _check(lib().zyfa_attn_decode_bf16_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), out.data_ptr(),
                                             lens, block_table.data_ptr(), block_table.stride(0), k_cache.shape[0],
                                             N, Hq, Hkv, Dqk, Dv, float(softmax_scale), _strides2(q),
                                             _strides(k_cache), _strides(v_cache), _strides2(out), ws_ptr, ws_bytes,
                                             _stream_ptr(q, stream)))
    return out


def attn_decode_fp8_paged(q8: torch.Tensor, q_scale: torch.Tensor, k_cache8: torch.Tensor, k_scale: torch.Tensor,
                          v_cache8: torch.Tensor, v_scale: torch.Tensor, seq_lens, block_table: torch.Tensor,
                          softmax_scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                          stream: Optional[torch.cuda.Stream] = None, split=True,
                          lean_p: bool = False) -> torch.Tensor:
    """FP8 form of attn_decode_bf16_paged: q8/q_scale from quantize_fp8_decode,
    caches and their [num_pages, Hkv] scales from quantize_fp8_cache."""
    _require_packed(q8, "q8", torch.uint8)
    _require_cache(k_cache8, "k_cache8", torch.uint8)
    _require_cache(v_cache8, "v_cache8", torch.uint8)
    N, Hq, Dqk = q8.shape
    P, Hkv, Dv = k_cache8.shape[0], k_cache8.shape[2], v_cache8.shape[3]
    lens = _decode_meta(seq_lens, block_table, N, q8.device)
    if not q_scale.is_cuda or q_scale.dtype != torch.float32 or not q_scale.is_contiguous() or q_scale.numel() != N * Hq:
        raise ValueError("q_scale must be a contiguous float32 CUDA tensor [N, Hq]")
    for t, n in ((k_scale, "k_scale"), (v_scale, "v_scale")):
        if not t.is_cuda or t.dtype != torch.float32 or not t.is_contiguous() or t.numel() != P * Hkv:
            raise ValueError(f"{n} must be a contiguous float32 CUDA tensor [num_pages, Hkv]")
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(Dqk)
    if out is None:
        out = torch.empty((N, Hq, Dv), dtype=torch.bfloat16, device=q8.device)
    _require_packed(out, "out", torch.bfloat16)
    ws_ptr, ws_bytes, _ws = _decode_workspace(N, Hq, Hkv, q8.device, split, stream)
    _check(lib().zyfa_attn_decode_fp8_paged(q8.data_ptr(), q_scale.data_ptr(), k_cache8.data_ptr(),
                                            k_scale.data_ptr(), v_cache8.data_ptr(), v_scale.data_ptr(),
                                            out.data_ptr(), lens, block_table.data_ptr(), block_table.stride(0), P,
                                            N, Hq, Hkv, Dqk, Dv, float(softmax_scale), _strides2(q8),
                                            _strides(k_cache8), _strides(v_cache8), _strides2(out), ws_ptr, ws_bytes, _fp8_flags(lean_p),
                                            _stream_ptr(q8, stream)))
    return out


def device_status(stream: Optional[torch.cuda.Stream] = None) -> int:
    """Synchronise and read/clear the device status word; raises on a timeout."""
    w = ctypes.c_uint(0)
    s = stream.cuda_stream if stream is not None else torch.cuda.current_stream().cuda_stream
    _check(lib().zyfa_get_device_status(s, ctypes.byref(w)))
    return w.value


def set_debug(stall_loader: bool = False, timeout_seconds: float = 0.0) -> None:
    """Test hook: stall the attention loader warp and/or bound waits (seconds)."""
    _check(lib().zyfa_set_debug(int(bool(stall_loader)), float(timeout_seconds)))
