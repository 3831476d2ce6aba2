"""Pins for the packed variable-length oracle (attention and quantiser).

- equal-length sequences packed one after another give the batched oracle's
  output (a different indexing path: [B,S,H,D] batches vs [T,H,D] offsets);
- sequences are independent: changing one sequence's tokens leaves every
  other sequence's outputs, codes and scales bit-identical;
- a single sequence is the plain causal oracle; empty sequences are skipped;
- a mistake that lets a sequence see the previous one's keys, or a block
  that mixes tokens of two sequences, fails these pins.
"""
import numpy as np
import pytest

from oracle import attention as A
from oracle import fp8


def _packed(lens, Hq=2, Hkv=1, D=16, Dv=8, seed=0):
    rng = np.random.default_rng(seed)
    T = sum(lens)
    q = rng.standard_normal((T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((T, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((T, Hkv, Dv)).astype(np.float32)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    return q, k, v, cu


def test_equal_lengths_match_the_batched_oracle():
    q, k, v, cu = _packed([7, 7, 7])
    got = A.causal_attention_varlen(q, k, v, cu, 0.3)
    ref = A.causal_attention(q.reshape(3, 7, 2, 16), k.reshape(3, 7, 1, 16), v.reshape(3, 7, 1, 8), 0.3)
    np.testing.assert_allclose(got, ref.reshape(21, 2, 8), rtol=1e-13, atol=1e-15)


def test_sequences_are_independent():
    q, k, v, cu = _packed([5, 0, 9, 1])
    base = A.causal_attention_varlen(q, k, v, cu, 0.25)
    q2, k2, v2 = q.copy(), k.copy(), v.copy()
    q2[5:14] += 1.0
    k2[5:14] -= 2.0
    v2[5:14] *= 3.0
    other = A.causal_attention_varlen(q2, k2, v2, cu, 0.25)
    np.testing.assert_array_equal(base[:5], other[:5])
    np.testing.assert_array_equal(base[14:], other[14:])
    assert not np.allclose(base[5:14], other[5:14])


def test_single_sequence_is_the_plain_oracle():
    q, k, v, cu = _packed([11])
    got = A.causal_attention_varlen(q, k, v, cu, 0.5)
    ref = A.causal_attention(q[None], k[None], v[None], 0.5)[0]
    np.testing.assert_array_equal(got, ref)


def test_leaky_mutant_is_caught():
    q, k, v, cu = _packed([4, 6])

    def leaky(q, k, v, cu, scale):    # second sequence also sees the first's keys
        return A.causal_attention(q[None], k[None], v[None], scale)[0]

    assert not np.allclose(leaky(q, k, v, cu, 0.3)[4:], A.causal_attention_varlen(q, k, v, cu, 0.3)[4:])


@pytest.mark.parametrize("had", [False, True])
def test_quantiser_blocks_never_mix_sequences(had):
    rng = np.random.default_rng(3)
    lens = [130, 0, 5, 256]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(int)
    x = (rng.standard_normal((sum(lens), 2, 128)) * 2).astype(np.float32)
    codes, scales = fp8.quantize_fp8_varlen(x, cu, had)
    for i, (s, e) in enumerate(zip(cu[:-1], cu[1:])):
        if e > s:
            c, sc = fp8.quantize_fp8(x[None, s:e], hadamard=had)
            np.testing.assert_array_equal(codes[s:e], c[0])
            np.testing.assert_array_equal(scales[i, :, :sc.shape[2]], sc[0])
    # a huge value in sequence 3 changes no scale of sequence 0
    x2 = x.copy()
    x2[cu[3]] *= 1000
    c2, s2 = fp8.quantize_fp8_varlen(x2, cu, had)
    np.testing.assert_array_equal(s2[0], scales[0])
    np.testing.assert_array_equal(c2[:cu[1]], codes[:cu[1]])
    # round trip within the e4m3 step
    back = fp8.dequantize_fp8_varlen(codes, scales, cu)
    ref = x if not had else fp8.fwht128_fp32(x[None])[0]
    assert np.max(np.abs(back - ref)) <= np.nanmax(scales) * 32
