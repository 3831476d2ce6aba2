"""Pins for the cached-prefix oracle (queries that continue a sequence).

- no prefix: the plain causal oracle;
- the new queries' rows of a full causal attention over the whole sequence,
  whatever the prefix positions' own queries are (an offset off by one row
  or a mask on the query index instead of the position fails this);
- closed forms: zero queries average the values at positions 0 .. P + i,
  constant values come back unchanged;
- a key after the query's position is never attended to, however large its
  score, while the same key at the query's own position dominates.
"""
import numpy as np

from oracle import attention as A


def _seq(L, Hq=4, Hkv=2, D=16, Dv=8, seed=0):
    rng = np.random.default_rng(seed)
    return (rng.standard_normal((L, Hq, D)), rng.standard_normal((L, Hkv, D)),
            rng.standard_normal((L, Hkv, Dv)))


def test_no_prefix_is_plain_causal_attention():
    q, k, v = _seq(11)
    got = A.causal_attention_prefix(q, k, v, 0.4)
    ref = A.causal_attention(q[None], k[None], v[None], 0.4)[0]
    np.testing.assert_allclose(got, ref, rtol=1e-13, atol=1e-15)


def test_rows_of_the_full_sequence():
    q, k, v = _seq(23, seed=1)
    full = A.causal_attention(q[None], k[None], v[None], 0.3)[0]
    for P in (1, 9, 22):
        got = A.causal_attention_prefix(q[P:], k, v, 0.3)
        np.testing.assert_allclose(got, full[P:], rtol=1e-12, atol=1e-14)
    # the prefix positions' queries play no part
    q2 = q.copy()
    q2[:9] = 100.0
    np.testing.assert_array_equal(A.causal_attention_prefix(q2[9:], k, v, 0.3),
                                  A.causal_attention_prefix(q[9:], k, v, 0.3))


def test_zero_queries_average_the_visible_values():
    _, k, v = _seq(17, seed=2)
    P, Lq = 12, 5
    got = A.causal_attention_prefix(np.zeros((Lq, 4, 16)), k, v, 1.0)
    for i in range(Lq):
        for h in range(4):
            np.testing.assert_allclose(got[i, h], v[: P + i + 1, h // 2].mean(axis=0), rtol=1e-12, atol=1e-14)


def test_constant_values_come_back():
    q, k, _ = _seq(9, seed=3)
    v = np.full((9, 2, 8), -1.75)
    np.testing.assert_allclose(A.causal_attention_prefix(q[4:], k, v, 2.0), -1.75, rtol=0, atol=1e-13)


def test_future_key_is_masked_own_key_dominates():
    L, P = 8, 5
    q = np.zeros((L - P, 1, 4))
    q[:, 0, 0] = 1.0
    k = np.zeros((L, 1, 4))
    v = np.zeros((L, 1, 2))
    v[:, 0, 0] = np.arange(L)
    k[P + 1, 0, 0] = 1000.0          # position P + 1: visible from query 1 on, not from query 0
    out = A.causal_attention_prefix(q, k, v, 1.0)
    np.testing.assert_allclose(out[0, 0, 0], np.arange(P + 1).mean(), rtol=1e-12)
    np.testing.assert_allclose(out[1:, 0, 0], P + 1, rtol=1e-12)


# ---------------------------------------------------------------- mutations --
# Plausible mistakes planted in a local copy of the prefix oracle; a pin above
# must tell each from the real one.

def _prefix_mutant(q, k, v, scale, *, offset_shift=0, mask_by_query_index=False):
    Lq, Hq, _ = q.shape
    L, Hkv, _ = k.shape
    P = L - Lq + offset_shift
    pos = np.arange(Lq) if mask_by_query_index else P + np.arange(Lq)
    allowed = np.arange(L)[None, :] <= pos[:, None]
    out = np.empty((Lq, Hq, v.shape[2]))
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = np.where(allowed, (q[:, h] @ k[:, g].T) * scale, -np.inf)
        p = np.exp(s - s.max(axis=1, keepdims=True))
        out[:, h] = (p / p.sum(axis=1, keepdims=True)) @ v[:, g]
    return out


def _full_rows(q, k, v, scale, P):
    return A.causal_attention(q[None], k[None], v[None], scale)[0][P:]


def test_mutant_offset_by_one_is_caught():
    q, k, v = _seq(19, seed=7)
    ref = _full_rows(q, k, v, 0.3, 6)
    np.testing.assert_allclose(A.causal_attention_prefix(q[6:], k, v, 0.3), ref, rtol=1e-12, atol=1e-14)
    for shift in (-1, 1):
        assert not np.allclose(_prefix_mutant(q[6:], k, v, 0.3, offset_shift=shift), ref)


def test_mutant_mask_on_the_query_index_is_caught():
    q, k, v = _seq(19, seed=8)
    ref = _full_rows(q, k, v, 0.3, 6)
    assert not np.allclose(_prefix_mutant(q[6:], k, v, 0.3, mask_by_query_index=True), ref)
