"""Shared helpers for the GPU parity tests: run the CUDA path, run the oracle
on the same seeded inputs, compare. Inputs come only from ``workloads``; the
oracle never sees a value produced by the CUDA path."""
from __future__ import annotations

import math
import os
from typing import Dict, List, Optional

import numpy as np
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from oracle import attention as oattn
from oracle import fp8 as ofp8

# Gates (tolerances fixed by the benchmark spec for this path).
BF16_REL_L2 = 5e-3
BF16_MAX_ABS = 1e-2
FP8_REL_L2 = 2.5e-2


def f32(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy()


def oracle_quant(x_bf16: torch.Tensor, hadamard: bool):
    return ofp8.quantize_fp8(f32(x_bf16), hadamard=hadamard)


def oracle_dequant(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    return ofp8.dequantize_fp8(codes, scales)


def errors(got: np.ndarray, ref: np.ndarray) -> Dict[str, float]:
    return {"rel_l2": oattn.rel_l2(got, ref), "max_abs": oattn.max_abs(got, ref)}


def assert_bf16_gate(got: np.ndarray, ref: np.ndarray, what: str = "") -> Dict[str, float]:
    e = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert e["rel_l2"] <= BF16_REL_L2 and e["max_abs"] <= BF16_MAX_ABS, f"{what}: {e}"
    return e


def assert_fp8_gate(got: np.ndarray, ref: np.ndarray, what: str = "") -> Dict[str, float]:
    e = errors(got, ref)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    assert e["rel_l2"] <= FP8_REL_L2, f"{what}: {e}"
    return e


def sampled_rows_oracle(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, rows: List[int],
                        heads: Optional[List[int]] = None, batches: Optional[List[int]] = None) -> np.ndarray:
    """Oracle rows [len(batches), len(rows), len(heads), Dv] computed one by one.
    q may be float32 (converted per row); k and v are converted per head once."""
    B, S, Hq, _ = q.shape
    Hkv = k.shape[2]
    heads = list(range(Hq)) if heads is None else heads
    batches = list(range(B)) if batches is None else batches
    out = np.empty((len(batches), len(rows), len(heads), v.shape[3]))
    group = Hq // Hkv
    cache = {}
    for bi, b in enumerate(batches):
        for hi, h in enumerate(heads):
            g = h // group
            if (b, g) not in cache:
                cache = {(b, g): (np.asarray(k[b:b + 1, :, g:g + 1], np.float64),
                                  np.asarray(v[b:b + 1, :, g:g + 1], np.float64))}
            kk, vv = cache[(b, g)]
            qq = np.asarray(q[b:b + 1, :, h:h + 1], np.float32)
            out[bi, :, hi] = oattn.causal_attention_rows(qq, kk, vv, scale, 0, 0, rows)
    return out


def sampled_rows_pquant(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, rows: List[int]) -> np.ndarray:
    """Like sampled_rows_oracle, with the probabilities quantised per 64-key
    block as the pages describe (oracle.attention.causal_attention_rows_pquant)."""
    B, S, Hq, _ = q.shape
    Hkv = k.shape[2]
    out = np.empty((B, len(rows), Hq, v.shape[3]))
    group = Hq // Hkv
    for b in range(B):
        for h in range(Hq):
            g = h // group
            kk = np.asarray(k[b:b + 1, :, g:g + 1], np.float64)
            vv = np.asarray(v[b:b + 1, :, g:g + 1], np.float64)
            qq = np.asarray(q[b:b + 1, :, h:h + 1], np.float32)
            out[b, :, h] = oattn.causal_attention_rows_pquant(qq, kk, vv, scale, 0, 0, rows)
    return out


def gpu_rows(o: torch.Tensor, rows: List[int], heads: Optional[List[int]] = None,
             batches: Optional[List[int]] = None) -> np.ndarray:
    B, S, Hq, _ = o.shape
    heads = list(range(Hq)) if heads is None else heads
    batches = list(range(B)) if batches is None else batches
    idx_r = torch.tensor(rows, device=o.device)
    sel = o[batches][:, idx_r][:, :, heads]
    return sel.float().cpu().numpy()


def fp8_quant_blocks_for_rows(x: torch.Tensor, rows: List[int], hadamard: bool):
    """Oracle codes/scales for only the 128-token blocks that contain `rows`
    (quantisation is per block, so each block is quantised on its own)."""
    blocks = sorted({r // 128 for r in rows})
    res = {}
    for j in blocks:
        sl = x[:, j * 128:(j + 1) * 128]
        res[j] = oracle_quant(sl, hadamard)
    return res


def full_oracle(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float, workers: int = 8) -> np.ndarray:
    """The oracle's full output [B,S,Hq,Dv] (float64), one (batch, head) per
    task over a pool of spawned processes (safe after CUDA is initialised)."""
    import multiprocessing as mp
    import oracle_pool
    B, S, Hq, _ = q.shape
    Hkv = k.shape[2]
    group = Hq // Hkv
    tasks = [(np.asarray(q[b, :, h], np.float64), np.asarray(k[b, :, h // group], np.float64),
              np.asarray(v[b, :, h // group], np.float64), scale) for b in range(B) for h in range(Hq)]
    n = max(1, min(workers, os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(n) as pool:
        outs = pool.map(oracle_pool.head_output, tasks, chunksize=1)
    out = np.empty((B, S, Hq, v.shape[3]))
    for i, o in enumerate(outs):
        out[i // Hq, :, i % Hq] = o
    return out

