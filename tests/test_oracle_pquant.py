"""Pins for the per-block P quantisation of the oracle (the P-rounding stage
of the error-by-stage report; ZYFA post, "Per-Block Scaling and
Normalization by the Rounded Row Sum").

- probabilities that are e4m3 values times a per-block power of two pass
  through unchanged, so the result equals the exact oracle;
- a constant V comes back (to float64 rounding) whatever the P rounding,
  since the weights are normalised by their own sum;
- on random scores the error is nonzero but within the e4m3 step (2^-4
  relative per weight);
- planted mistakes (no power of two divided back out, normalising by the
  unrounded sum, one scale for the whole row) fail at least one pin.
"""
import math

import numpy as np
import pytest

from oracle import attention as A
from oracle import fp8


def _rows_exact(q, k, v, scale, rows):
    return A.causal_attention_rows(q, k, v, scale, 0, 0, rows)


def _scores_for(p_targets, scale=1.0):
    """A single query row whose probabilities (max-subtracted) are p_targets:
    q = [1, 0, ...], k_j = [log(p_j)/scale, 0, ...]."""
    n = len(p_targets)
    q = np.zeros((1, n, 1, 2))
    k = np.zeros((1, n, 1, 2))
    q[0, n - 1, 0, 0] = 1.0
    k[0, :, 0, 0] = np.log(np.asarray(p_targets, dtype=np.float64)) / scale
    return q, k


# per 4-key block: e4m3 values times 2^-k with different k per block; block max 1, 2^-3, 2^-7 x 1.75 ...
P_EXACT = [1.0, 0.75, 0.5, 0.3125,
           0.125, 0.125 * 0.875, 0.125 * 0.5, 0.125 * 0.625,
           2.0 ** -7 * 1.75, 2.0 ** -7 * 1.5, 2.0 ** -7, 2.0 ** -7 * 1.125]


def _pquant_exact_case(fn):
    q, k = _scores_for(P_EXACT)
    rng = np.random.default_rng(0)
    v = rng.standard_normal((1, len(P_EXACT), 1, 3))
    rows = [len(P_EXACT) - 1]
    return fn(q, k, v, 1.0, 0, 0, rows, block=4), _rows_exact(q, k, v, 1.0, rows)


def test_representable_probabilities_pass_unchanged():
    got, ref = _pquant_exact_case(A.causal_attention_rows_pquant)
    np.testing.assert_allclose(got, ref, rtol=1e-12, atol=1e-14)


def test_constant_v_is_exact():
    rng = np.random.default_rng(1)
    S = 300
    q = rng.standard_normal((1, S, 1, 16)) * 3
    k = rng.standard_normal((1, S, 1, 16)) * 3
    v = np.full((1, S, 1, 4), 0.7)
    got = A.causal_attention_rows_pquant(q, k, v, 0.25, 0, 0, [0, 1, 63, 64, 200, 299])
    np.testing.assert_allclose(got, 0.7, rtol=1e-13, atol=0)


def test_random_scores_error_within_e4m3_step():
    rng = np.random.default_rng(2)
    S = 256
    q = rng.standard_normal((1, S, 1, 32))
    k = rng.standard_normal((1, S, 1, 32))
    v = rng.standard_normal((1, S, 1, 8))
    rows = list(range(0, S, 7))
    got = A.causal_attention_rows_pquant(q, k, v, 1 / math.sqrt(32), 0, 0, rows)
    ref = _rows_exact(q, k, v, 1 / math.sqrt(32), rows)
    e = A.rel_l2(got, ref)
    assert 0 < e < 2.0 ** -4


def _mutant(kind):
    def fn(q, k, v, scale, b, h, rows, block=64):
        res = []
        for i in rows:
            kk = np.asarray(k[b, : i + 1, 0, :], np.float64)
            vv = np.asarray(v[b, : i + 1, 0, :], np.float64)
            s = (kk @ np.asarray(q[b, i, h, :], np.float64)) * scale
            p = np.exp(s - np.max(s))
            w = np.zeros_like(p)
            for c in range(0, p.size, block):
                pb = p[c:c + block]
                mb = np.max(pb) if kind != "row_scale" else np.max(p)
                kb = math.floor(-math.log2(mb))
                wb = fp8.e4m3_decode(fp8.e4m3_rne(np.ldexp(pb, kb)))
                w[c:c + block] = wb if kind == "no_descale" else np.ldexp(wb, -kb)
            den = np.sum(w) if kind != "unrounded_sum" else np.sum(p)
            res.append((w @ vv) / den)
        return np.stack(res)
    return fn


@pytest.mark.parametrize("kind", ["no_descale", "unrounded_sum", "row_scale"])
def test_mutants_are_caught(kind):
    fn = _mutant(kind)
    caught = False
    got, ref = _pquant_exact_case(fn)
    if not np.allclose(got, ref, rtol=1e-12, atol=1e-14):
        caught = True
    rng = np.random.default_rng(1)
    S = 300
    q = rng.standard_normal((1, S, 1, 16)) * 3
    k = rng.standard_normal((1, S, 1, 16)) * 3
    v = np.full((1, S, 1, 4), 0.7)
    g = fn(q, k, v, 0.25, 0, 0, [63, 200, 299])
    if not np.allclose(g, 0.7, rtol=1e-13, atol=0):
        caught = True
    assert caught, kind
