"""Pins for the float64 causal attention oracle.

The oracle is checked against brute force on tiny inputs (pure Python, no
numpy), PyTorch's float64 scaled-dot-product attention, closed forms and the
invariants of causal softmax attention. Mutation tests plant plausible
mistakes in local copies and show that the pins catch them.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import attention as A
from oracle import fp8


def _brute(q, k, v, scale):
    B, S, Hq, D = q.shape
    Hkv = k.shape[2]
    Dv = v.shape[3]
    out = np.zeros((B, S, Hq, Dv))
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv)
            for i in range(S):
                sc = []
                for j in range(i + 1):
                    sc.append(sum(float(q[b, i, h, d]) * float(k[b, j, g, d]) for d in range(D)) * scale)
                mx = max(sc)
                w = [math.exp(s - mx) for s in sc]
                tot = sum(w)
                for e in range(Dv):
                    out[b, i, h, e] = sum(w[j] * float(v[b, j, g, e]) for j in range(i + 1)) / tot
    return out


@pytest.mark.parametrize("S,Hq,Hkv,D,Dv", [(1, 1, 1, 3, 2), (5, 2, 1, 4, 3), (8, 4, 2, 3, 5)])
def test_brute_force_tiny(S, Hq, Hkv, D, Dv):
    rng = np.random.default_rng(S * 100 + Hq)
    q = rng.standard_normal((2, S, Hq, D))
    k = rng.standard_normal((2, S, Hkv, D))
    v = rng.standard_normal((2, S, Hkv, Dv))
    np.testing.assert_allclose(A.causal_attention(q, k, v, 0.7), _brute(q, k, v, 0.7),
                               rtol=1e-12, atol=1e-12)


def _sdpa(q, k, v, scale):
    Hq, Hkv = q.shape[2], k.shape[2]
    t = lambda x: torch.from_numpy(np.asarray(x, np.float64)).permute(0, 2, 1, 3)
    kk = t(k).repeat_interleave(Hq // Hkv, dim=1)
    vv = t(v).repeat_interleave(Hq // Hkv, dim=1)
    o = F.scaled_dot_product_attention(t(q), kk, vv, is_causal=True, scale=scale)
    return o.permute(0, 2, 1, 3).numpy()


@pytest.mark.parametrize("Hq,Hkv,D,Dv", [(4, 4, 64, 64), (8, 2, 128, 128), (4, 1, 192, 128)])
def test_matches_torch_sdpa_float64(Hq, Hkv, D, Dv):
    rng = np.random.default_rng(Hq * 7 + D)
    S = 77
    q = rng.standard_normal((2, S, Hq, D))
    k = rng.standard_normal((2, S, Hkv, D))
    v = rng.standard_normal((2, S, Hkv, Dv))
    scale = 1.0 / math.sqrt(D)
    np.testing.assert_allclose(A.causal_attention(q, k, v, scale), _sdpa(q, k, v, scale),
                               rtol=1e-10, atol=1e-12)


def test_probability_rows_sum_to_one_and_are_causal():
    rng = np.random.default_rng(11)
    q = rng.standard_normal((40, 16)) * 4
    k = rng.standard_normal((40, 16)) * 4
    p = A.causal_probs(q, k, 0.5)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, rtol=0, atol=1e-14)
    assert np.all(p[np.triu_indices(40, 1)] == 0)


def test_uniform_v_returns_v():
    rng = np.random.default_rng(12)
    q = rng.standard_normal((1, 50, 2, 8))
    k = rng.standard_normal((1, 50, 1, 8))
    v = np.full((1, 50, 1, 4), 3.25)
    np.testing.assert_allclose(A.causal_attention(q, k, v, 1.0), 3.25, rtol=0, atol=1e-13)


def test_row_zero_returns_v0():
    rng = np.random.default_rng(13)
    q = rng.standard_normal((1, 20, 3, 8))
    k = rng.standard_normal((1, 20, 3, 8))
    v = rng.standard_normal((1, 20, 3, 6))
    o = A.causal_attention(q, k, v, 1.0)
    np.testing.assert_allclose(o[0, 0], v[0, 0], rtol=0, atol=1e-14)


def test_zero_query_gives_prefix_mean():
    rng = np.random.default_rng(14)
    k = rng.standard_normal((1, 30, 1, 8))
    v = rng.standard_normal((1, 30, 1, 5))
    q = np.zeros((1, 30, 1, 8))
    o = A.causal_attention(q, k, v, 1.0)
    prefix_mean = np.cumsum(v[0, :, 0], axis=0) / np.arange(1, 31)[:, None]
    np.testing.assert_allclose(o[0, :, 0], prefix_mean, rtol=0, atol=1e-13)


def test_gqa_equals_repeated_kv_mha():
    rng = np.random.default_rng(15)
    q = rng.standard_normal((1, 25, 6, 8))
    k = rng.standard_normal((1, 25, 2, 8))
    v = rng.standard_normal((1, 25, 2, 4))
    rep = lambda x: np.repeat(x, 3, axis=2)
    np.testing.assert_allclose(A.causal_attention(q, k, v, 0.3),
                               A.causal_attention(q, rep(k), rep(v), 0.3), rtol=0, atol=1e-14)


def test_rows_api_matches_full():
    rng = np.random.default_rng(16)
    q = rng.standard_normal((2, 60, 4, 16))
    k = rng.standard_normal((2, 60, 2, 16))
    v = rng.standard_normal((2, 60, 2, 8))
    full = A.causal_attention(q, k, v, 0.25)
    rows = [0, 1, 31, 59]
    got = A.causal_attention_rows(q, k, v, 0.25, 1, 3, rows)
    np.testing.assert_allclose(got, full[1, rows, 3], rtol=1e-12, atol=1e-14)


def test_rotated_dequantised_inputs_keep_attention():
    # Hadamard rotation of Q and K leaves QK^T, hence the output, unchanged.
    rng = np.random.default_rng(17)
    q = rng.standard_normal((1, 64, 2, 128)).astype(np.float32)
    k = rng.standard_normal((1, 64, 1, 128)).astype(np.float32)
    v = rng.standard_normal((1, 64, 1, 128))
    o = A.causal_attention(q, k, v, 1 / math.sqrt(128))
    orot = A.causal_attention(fp8.fwht128_fp32(q), fp8.fwht128_fp32(k), v, 1 / math.sqrt(128))
    np.testing.assert_allclose(orot, o, rtol=0, atol=1e-5)


def test_rel_l2_is_relative_rms():
    ref = np.array([3.0, 4.0])
    assert A.rel_l2(ref + np.array([0.3, 0.4]), ref) == pytest.approx(0.1)


# ---------------------------------------------------------------- mutations --

def _attn_mutant(q, k, v, scale, *, diag_masked=False, head_map="div", no_max=False):
    B, S, Hq, _ = q.shape
    Hkv = k.shape[2]
    out = np.empty((B, S, Hq, v.shape[3]))
    for b in range(B):
        for h in range(Hq):
            g = h // (Hq // Hkv) if head_map == "div" else h % Hkv
            s = (q[b, :, h] @ k[b, :, g].T) * scale
            mask = np.triu(np.ones((S, S), bool), k=0 if diag_masked else 1)
            if diag_masked:
                mask[0, 0] = False
            s = np.where(mask, -np.inf, s)
            if not no_max:
                s = s - s.max(axis=1, keepdims=True)
            p = np.exp(s)
            out[b, :, h] = (p / p.sum(axis=1, keepdims=True)) @ v[b, :, g]
    return out


def test_mutant_mask_is_caught():
    rng = np.random.default_rng(18)
    q, k, v = (rng.standard_normal((1, 6, 2, 3)) for _ in range(3))
    assert not np.allclose(_attn_mutant(q, k, v, 0.5, diag_masked=True), _brute(q, k, v, 0.5))


def test_mutant_head_mapping_is_caught():
    rng = np.random.default_rng(19)
    q = rng.standard_normal((1, 20, 8, 16))
    k = rng.standard_normal((1, 20, 2, 16))
    v = rng.standard_normal((1, 20, 2, 16))
    assert not np.allclose(_attn_mutant(q, k, v, 0.25, head_map="mod"), _sdpa(q, k, v, 0.25))


def test_mutant_missing_max_subtraction_overflows():
    # Activation-like scores overflow exp() without the row-max shift.
    q = np.full((1, 4, 1, 2), 30.0)
    k = np.full((1, 4, 1, 2), 30.0)
    v = np.ones((1, 4, 1, 1))
    with np.errstate(over="ignore", invalid="ignore"):
        bad = _attn_mutant(q, k, v, 1.0, no_max=True)
    assert not np.all(np.isfinite(bad))
    np.testing.assert_allclose(A.causal_attention(q, k, v, 1.0), 1.0)
