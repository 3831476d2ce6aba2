"""Pins of the oracle's emulation of the BF16 path's probability rounding
(oracle.attention.causal_attention_rows_bf16: a stale running maximum moved
only past 2^8, probabilities rounded to bf16, the row sum over the rounded
values), each fixed by something other than the function itself: the
running-maximum rule on hand-worked sequences, bf16 rounding against
torch's conversion, exact softmax attention with the rounding off, and the
exact average of a constant V."""
import numpy as np
import pytest
import torch

import workloads
from oracle import attention as oattn
from parity import f32


def test_stale_maximum_hand_worked():
    m, seen = None, []
    for xmax in (0.0, 8.0, 8.5, 3.0, 20.0, 28.0, 28.01):
        m = oattn.stale_max_step(m, xmax)
        seen.append(m)
    assert seen == [0.0, 0.0, 8.5, 8.5, 20.0, 20.0, 28.01]


def test_bf16_rounding_agrees_with_torch():
    rng = np.random.default_rng(5)
    x = np.concatenate([rng.uniform(0, 256, 200000), np.exp2(rng.uniform(-40, 8, 200000)),
                        1.0 + np.arange(0, 1024) / 2 ** 15])        # ties and near-ties around 1
    want = torch.from_numpy(x).to(torch.float32).to(torch.bfloat16).to(torch.float64).numpy()
    assert np.array_equal(oattn.bf16_rne(x), want)


CASES = [
    workloads.custom(1, 2, 1, 300, seed=51),
    workloads.custom(1, 2, 2, 260, Dqk=192, seed=52),
    workloads.custom(1, 2, 1, 700, seed=53, v_std=0.5, outliers=4, outlier_gain=20.0, rope_theta=1.0e6),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_unrounded_is_exact_attention(w):
    q, k, v = (f32(t) for t in workloads.make_qkv(w))
    rows = sorted(set([0, 1, 127, 128, 255, 256, w.S - 1] + list(range(3, w.S, 37))))
    for h in range(w.Hq):
        un = oattn.causal_attention_rows_bf16(q, k, v, w.softmax_scale, 0, h, rows, round_p=False)
        ex = oattn.causal_attention_rows(q, k, v, w.softmax_scale, 0, h, rows)
        assert oattn.rel_l2(un, ex) < 1e-12
        r = oattn.causal_attention_rows_bf16(q, k, v, w.softmax_scale, 0, h, rows)
        assert np.abs(r[1:] - un[1:]).max() > 0          # the rounding does act


def test_rounded_sum_gives_exact_average():
    w = CASES[0]
    q, k, _ = (f32(t) for t in workloads.make_qkv(w))
    c = 0.6875                                             # a bf16 value
    v = np.full((1, w.S, 1, 128), c)
    out = oattn.causal_attention_rows_bf16(q, k, v, w.softmax_scale, 0, 1, [0, 5, 127, 128, w.S - 1])
    assert np.all(out == c)


# ---------------------------------------------------------------- mutations --

def _bf16_mutant(q, k, v, scale, b, h, rows, round_p, *, no_rescale=False, l_unrounded=False):
    g = oattn.kv_head(h, q.shape[2], k.shape[2])
    c2 = scale / np.log(2.0)
    res = []
    for i in rows:
        qi = q[b, i, h].astype(np.float64)
        m, acc, l = None, np.zeros(v.shape[3]), 0.0
        for j in range(i // 128 + 1):
            k0, k1 = 128 * j, min(128 * j + 128, i + 1)
            x = (k[b, k0:k1, g].astype(np.float64) @ qi) * c2
            m_new = oattn.stale_max_step(m, float(np.max(x)))
            if m is not None and m_new != m and not no_rescale:
                acc *= 2.0 ** (m - m_new)
                l *= 2.0 ** (m - m_new)
            m = m_new
            exact = np.exp2(x - m)
            p = oattn.bf16_rne(exact) if round_p else exact
            acc += p @ v[b, k0:k1, g].astype(np.float64)
            l += float(np.sum(exact if l_unrounded else p))
        res.append(acc / l)
    return np.stack(res)


def test_bf16_mutant_without_rescale_is_caught():
    w = CASES[2]                                   # activation-like: the maximum moves
    q, k, v = (f32(t) for t in workloads.make_qkv(w))
    rows = list(range(5, w.S, 23))
    worst = max(oattn.rel_l2(_bf16_mutant(q, k, v, w.softmax_scale, 0, h, rows, False, no_rescale=True),
                             oattn.causal_attention_rows(q, k, v, w.softmax_scale, 0, h, rows))
                for h in range(w.Hq))
    assert worst > 1e-6


def test_bf16_mutant_unrounded_sum_is_caught_by_the_exact_average():
    w = CASES[0]
    q, k, _ = (f32(t) for t in workloads.make_qkv(w))
    v = np.full((1, w.S, 1, 128), 0.6875)
    bad = _bf16_mutant(q, k, v, w.softmax_scale, 0, 1, [5, 127, 128, w.S - 1], True, l_unrounded=True)
    assert not np.all(bad == 0.6875)
