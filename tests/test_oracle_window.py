"""Pins of the oracle's emulation of the FP8 path's probability rounding
(oracle.attention.causal_attention_rows_window, the offset-window reading of
the ZYFA post's "Per-Block Scaling and Normalization by the Rounded Row
Sum"), each fixed by something other than the function itself:

* the offset rule on hand-worked sequences of tile maxima;
* with rounding switched off, exact softmax attention on the dequantised
  inputs (the float64 definition), on rows whose offsets move up and down,
  so every rescale and the folding of the V scale are checked;
* the pages' exact-average property: V of one value whose block scale is a
  power of two comes out exactly, however P is rounded, because the
  normalisation divides by the sum of the rounded probabilities;
* every tile's largest scaled probability lies in the window (or the tile
  is too far below the row's maximum to move the offset).
"""
import math

import numpy as np
import pytest

import workloads
from oracle import attention as oattn
from oracle import fp8 as ofp8
from parity import f32


def _offsets(bms):
    o = top = None
    out = []
    for bm in bms:
        o, top = oattn.window_step(o, top, bm)
        out.append(o)
    return out


def test_offset_rule_hand_worked():
    # first tile sets o; a jump above the window moves o up to the tile's
    # maximum; a tile more than 4 binades below moves it down; a tile more
    # than 64 binades below the row's maximum leaves it
    assert _offsets([0.0, 10.0, 3.0, -70.0]) == [0.0, 10.0, 3.0, 3.0]
    # edges of the window do not move it
    assert _offsets([0.0, 8.0, -4.0, 5.0]) == [0.0, 0.0, 0.0, 0.0]
    assert _offsets([0.0, 8.5]) == [0.0, 8.5]
    assert _offsets([0.0, -4.5]) == [0.0, -4.5]
    assert _offsets([0.0, 100.0, 20.0]) == [0.0, 100.0, 100.0]
    assert _offsets([0.0, 100.0, 50.0, 55.0, 44.0]) == [0.0, 100.0, 50.0, 50.0, 44.0]


def _quantised(w):
    q, k, v = workloads.make_qkv(w)
    return [ofp8.quantize_fp8(f32(x), hadamard=False) for x in (q, k, v)]


CASES = [
    workloads.custom(1, 2, 1, 300, seed=21),
    workloads.custom(1, 2, 2, 260, Dqk=192, seed=22),
    workloads.custom(1, 2, 1, 700, seed=23, v_std=0.5, outliers=4, outlier_gain=20.0, rope_theta=1.0e6),
]


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_unrounded_window_is_exact_attention(w):
    (cq, sq), (ck, sk), (cv, sv) = _quantised(w)
    dq, dk, dv = (ofp8.dequantize_fp8(c, s) for c, s in ((cq, sq), (ck, sk), (cv, sv)))
    rows = sorted(set([0, 1, 127, 128, 255, 256, w.S - 1] + list(range(3, w.S, 37))))
    moves = 0
    for h in range(w.Hq):
        trace = []
        un = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, h, rows,
                                                round_p=False, trace=trace)
        ex = oattn.causal_attention_rows(dq, dk, dv, w.softmax_scale, 0, h, rows)
        assert oattn.rel_l2(un, ex) < 1e-12
        moves += sum(1 for a, b in zip(trace, trace[1:]) if a[0] == b[0] and a[2] != b[2])
    if "outlier" in w.name or w.outliers:
        assert moves > 0            # the rescales were exercised


def test_rounded_sum_gives_exact_average():
    w = workloads.custom(1, 2, 1, 520, seed=24)
    (cq, sq), (ck, sk), (cg, sg) = _quantised(w)
    c = 448.0 * 2.0 ** -5                       # V = c everywhere: code 448, scale 2^-5
    cv, sv = ofp8.quantize_fp8(np.full((1, w.S, 1, 128), c, dtype=np.float32))
    assert np.all(sv == 2.0 ** -5)
    rows = [0, 5, 127, 128, 300, 519]
    out = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, 1, rows)
    assert np.all(out == c)
    # the pin is not vacuous: on the same rows the rounding moves the output
    # for a V that is not constant (rows past the first, which has one key)
    r = oattn.causal_attention_rows_window(cq, sq, ck, sk, cg, sg, w.softmax_scale, 0, 1, rows)
    u = oattn.causal_attention_rows_window(cq, sq, ck, sk, cg, sg, w.softmax_scale, 0, 1, rows, round_p=False)
    assert np.all(r[0] == u[0])
    assert np.all(np.abs(r[1:] - u[1:]).max(axis=1) > 0)


def test_tile_maxima_stay_in_the_window():
    w = CASES[2]
    (cq, sq), (ck, sk), (cv, sv) = _quantised(w)
    c2 = w.softmax_scale / math.log(2.0)
    rows = list(range(0, w.S, 11))
    for h in range(w.Hq):
        trace = []
        oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, h, rows, trace=trace)
        top = {}
        for i, j, o in trace:
            g = oattn.kv_head(h, w.Hq, w.Hkv)
            k0, k1 = 128 * j, min(128 * j + 128, i + 1)
            x = (ofp8.e4m3_decode(ck[0, k0:k1, g]) @ ofp8.e4m3_decode(cq[0, i, h])) * (
                float(sq[0, h, i // 128]) * float(sk[0, g, j]) * c2)
            bm = float(np.max(x)) + math.log2(float(sv[0, g, j]))
            t = max(top.get(i, bm), bm)
            top[i] = t
            rel = bm - o
            assert rel <= oattn.WIN_HI + 1e-9
            assert rel >= oattn.WIN_LO - 1e-9 or bm <= t - oattn.WIN_FLOOR + 1e-9 or j == 0


@pytest.mark.parametrize("w", CASES[::2], ids=lambda w: w.name)
def test_chunked_window_merges_exactly(w):
    """Key chunks run from fresh offsets and merged by their offsets: exact
    attention with the rounding off (any chunk size), and the unchunked
    emulation itself when one chunk holds every tile."""
    (cq, sq), (ck, sk), (cv, sv) = _quantised(w)
    dq, dk, dv = (ofp8.dequantize_fp8(c, s) for c, s in ((cq, sq), (ck, sk), (cv, sv)))
    rows = sorted(r for r in set([0, 127, 128, 383, 384, w.S - 1] + list(range(7, w.S, 53))) if r < w.S)
    for h in range(w.Hq):
        ex = oattn.causal_attention_rows(dq, dk, dv, w.softmax_scale, 0, h, rows)
        for C in (1, 2, 3):
            un = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, h, rows,
                                                    round_p=False, chunk_tiles=C)
            assert oattn.rel_l2(un, ex) < 1e-12
        whole = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, h, rows)
        one = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, h, rows,
                                                 chunk_tiles=64)
        assert np.array_equal(whole, one)


def _page_codes():
    codes = {}
    import os
    for line in open(os.path.join(os.path.dirname(__file__), "golden", "e4m3_page_values.txt")):
        if line.strip() and not line.startswith("#"):
            val, code = line.split()[:2]
            codes[float(val)] = int(code, 16)
    return codes


def test_lean_codes_at_whole_exponents_are_the_pages_codes():
    page = _page_codes()
    for t, v in ((0, 1.0), (1, 2.0), (2, 4.0)):
        assert int(oattn.lean_codes(np.array([1080.0 + 8 * t]))[0]) == page[v]
    t = np.arange(-6, 9, dtype=np.float64)
    assert np.array_equal(ofp8.e4m3_decode(oattn.lean_codes(1080.0 + 8 * t)), 2.0 ** t)


def test_lean_code_is_the_exact_code_or_the_next():
    """8 t + 56 rounds to the exact nearest code of 2^t or one above it: the
    linear code overshoots the mantissa 8 (2^f - 1) by at most
    8 max(f - 2^f + 1) < 0.7 (format definition, normal range)."""
    t = np.linspace(-6.0, 8.0, 200001)
    lean = oattn.lean_codes(1080.0 + 8.0 * t).astype(int)
    exact = ofp8.e4m3_rne(2.0 ** t).astype(int)
    d = lean - exact
    assert d.min() == 0 and d.max() == 1
    assert 0.2 < np.mean(d) < 0.6


def test_lean_window_keeps_the_exact_average():
    w = workloads.custom(1, 2, 1, 520, seed=25)
    (cq, sq), (ck, sk), _ = _quantised(w)
    c = 448.0 * 2.0 ** -3
    cv, sv = ofp8.quantize_fp8(np.full((1, w.S, 1, 128), c, dtype=np.float32))
    rows = [0, 5, 127, 128, 300, 519]
    out = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, 1, rows, lean=True)
    assert np.all(out == c)


# ---------------------------------------------------------------- mutations --
# Plausible mistakes planted in a local copy of the emulation's tile loop; a
# pin above must catch each of them.

def _window_mutant(q8, qs, k8, ks, v8, vs, scale, b, h, rows, round_p, *, no_rescale=False,
                   l_without_sv=False, no_lsv=False, l_unrounded=False):
    g = oattn.kv_head(h, q8.shape[2], k8.shape[2])
    c2 = scale / math.log(2.0)
    res = []
    for i in rows:
        qc = ofp8.e4m3_decode(q8[b, i, h])
        sq = float(qs[b, h, i // 128])
        o = top = None
        acc, l = np.zeros(v8.shape[3]), 0.0
        for j in range(i // 128 + 1):
            k0, k1 = 128 * j, min(128 * j + 128, i + 1)
            kc, vc = ofp8.e4m3_decode(k8[b, k0:k1, g]), ofp8.e4m3_decode(v8[b, k0:k1, g])
            sk, sv = float(ks[b, g, j]), float(vs[b, g, j])
            x = (kc @ qc) * (sq * sk * c2)
            lsv = 0.0 if no_lsv else math.log2(sv)
            o_new, top = oattn.window_step(o, top, float(np.max(x)) + lsv)
            if o is not None and o_new != o and not no_rescale:
                acc *= 2.0 ** (o - o_new)
                l *= 2.0 ** (o - o_new)
            o = o_new
            exact = np.exp2(x + lsv - o)
            p = ofp8.e4m3_decode(ofp8.e4m3_rne(exact)) if round_p else exact
            acc += p @ vc
            l += float(np.sum(exact if l_unrounded else p)) / (1.0 if l_without_sv else sv)
        res.append(acc / l)
    return np.stack(res)


@pytest.mark.parametrize("flag", ["no_rescale", "l_without_sv", "no_lsv"])
def test_window_mutants_are_caught_by_exact_attention(flag):
    w = CASES[2]                                   # activation-like: offsets move both ways
    (cq, sq), (ck, sk), (cv, sv) = _quantised(w)
    dq, dk, dv = (ofp8.dequantize_fp8(c, s) for c, s in ((cq, sq), (ck, sk), (cv, sv)))
    rows = list(range(5, w.S, 23))
    worst = 0.0
    for h in range(w.Hq):
        bad = _window_mutant(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, h, rows, False, **{flag: True})
        ex = oattn.causal_attention_rows(dq, dk, dv, w.softmax_scale, 0, h, rows)
        worst = max(worst, oattn.rel_l2(bad, ex))
    assert worst > 1e-6


def test_window_mutant_unrounded_sum_is_caught_by_the_exact_average():
    w = workloads.custom(1, 2, 1, 520, seed=24)
    (cq, sq), (ck, sk), _ = _quantised(w)
    c = 448.0 * 2.0 ** -5
    cv, sv = ofp8.quantize_fp8(np.full((1, w.S, 1, 128), c, dtype=np.float32))
    bad = _window_mutant(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, 1, [5, 127, 300, 519], True, l_unrounded=True)
    assert not np.all(bad == c)
