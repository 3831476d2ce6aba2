"""Causal attention on the GPU (BF16 and FP8) against the float64 oracle.

Small shapes are compared element by element over the whole output; they span
several 128-row tiles, ragged tails, GQA and the MLA head shape. The FP8 path
is compared with the oracle run on the oracle's own dequantised inputs. Pins
that hold exactly (rounded-row-sum normalisation, determinism, GQA) are
checked bitwise.
"""
import math

import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from oracle import attention as oattn
from parity import (assert_bf16_gate, assert_fp8_gate, f32, oracle_dequant, oracle_quant)

pytestmark = pytest.mark.gpu

SHAPES = [  # B, Hq, Hkv, S, Dqk
    (1, 1, 1, 1, 128),
    (1, 2, 1, 7, 128),
    (1, 2, 2, 128, 128),
    (2, 4, 2, 129, 128),
    (1, 2, 1, 255, 128),
    (1, 4, 1, 256, 128),
    (1, 3, 3, 300, 192),
    (2, 8, 2, 520, 128),
    (1, 2, 2, 640, 192),
]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _inputs(B, Hq, Hkv, S, D, seed=0):
    w = workloads.custom(B, Hq, Hkv, S, Dqk=D, Dv=128, seed=seed)
    q, k, v = workloads.make_qkv(w)
    return w, (q, k, v), (q.cuda(), k.cuda(), v.cuda())


@pytest.mark.parametrize("B,Hq,Hkv,S,D", SHAPES)
def test_bf16_matches_oracle(B, Hq, Hkv, S, D):
    w, (q, k, v), (qd, kd, vd) = _inputs(B, Hq, Hkv, S, D, seed=S)
    o = zyfa.attn_fwd_bf16(qd, kd, vd, w.softmax_scale)
    zyfa.device_status()
    ref = oattn.causal_attention(f32(q), f32(k), f32(v), w.softmax_scale)
    assert_bf16_gate(f32(o), ref, f"bf16 {B,Hq,Hkv,S,D}")


@pytest.mark.parametrize("B,Hq,Hkv,S,D", SHAPES)
def test_fp8_matches_oracle_on_oracle_codes(B, Hq, Hkv, S, D):
    w, (q, k, v), _ = _inputs(B, Hq, Hkv, S, D, seed=S + 1)
    had = D == 128
    cq, sq = oracle_quant(q, had)
    ck, sk = oracle_quant(k, had)
    cv, sv = oracle_quant(v, False)
    dev = lambda a: torch.from_numpy(a).cuda()
    o = zyfa.attn_fwd_fp8(dev(cq), dev(sq), dev(ck), dev(sk), dev(cv), dev(sv), w.softmax_scale)
    zyfa.device_status()
    ref = oattn.causal_attention(oracle_dequant(cq, sq), oracle_dequant(ck, sk), oracle_dequant(cv, sv),
                                 w.softmax_scale)
    assert_fp8_gate(f32(o), ref, f"fp8 {B,Hq,Hkv,S,D}")


@pytest.mark.parametrize("hadamard", [False, True])
def test_small_workload_end_to_end(hadamard):
    """The whole FP8 path (GPU quantiser + FP8 attention) and the BF16 path on
    the 1K-token Gaussian workload, full output."""
    w = workloads.get(workloads.SMALL)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o8, (q8, qs, k8, ks, v8, vs) = zyfa.prefill_fp8(qd, kd, vd, hadamard=hadamard)
    o16 = zyfa.attn_fwd_bf16(qd, kd, vd)
    zyfa.device_status()
    cq, sq = oracle_quant(q, hadamard)
    ck, sk = oracle_quant(k, hadamard)
    cv, sv = oracle_quant(v, False)
    for got, ref in ((q8, cq), (k8, ck), (v8, cv), (qs, sq), (ks, sk), (vs, sv)):
        assert np.array_equal(got.cpu().numpy(), ref)
    ref8 = oattn.causal_attention(oracle_dequant(cq, sq), oracle_dequant(ck, sk), oracle_dequant(cv, sv),
                                  w.softmax_scale)
    e8 = assert_fp8_gate(f32(o8), ref8, "fp8 small workload")
    ref16 = oattn.causal_attention(f32(q), f32(k), f32(v), w.softmax_scale)
    assert_bf16_gate(f32(o16), ref16, "bf16 small workload")
    # error against unquantised fp64 attention: reported, not gated
    print(f"\nfp8 hadamard={hadamard}: rel_l2 vs dequantised oracle {e8['rel_l2']:.3e}, "
          f"vs unquantised fp64 {oattn.rel_l2(f32(o8), ref16):.3e}")


def test_fp8_rounded_row_sum_gives_exact_average():
    """ZYFA post, footnote 6: dividing by the sum of the rounded probabilities
    makes every output a weighted average whose weights sum to one. With V
    constant at c = 448 * 2^-5 every V block has scale 2^-5 and code 448, so
    the output must be exactly c, even where many probabilities underflow."""
    g = torch.Generator().manual_seed(11)
    B, S, Hq, Hkv, D = 1, 700, 4, 2, 128
    q = (torch.randn(B, S, Hq, D, generator=g) * 4).to(torch.bfloat16)
    k = (torch.randn(B, S, Hkv, D, generator=g) * 4).to(torch.bfloat16)
    c = 448.0 * 2 ** -5
    v = torch.full((B, S, Hkv, 128), c).to(torch.bfloat16)
    o, _ = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda())
    zyfa.device_status()
    got = o.float().cpu()
    bad = (got != c).nonzero()
    assert bad.numel() == 0, (f"{bad.shape[0]} of {got.numel()} outputs differ from {c}; "
                              f"values {sorted(set(got[got != c].tolist()))[:8]}; rows {sorted(set(bad[:, 1].tolist()))[:16]}")


def test_row_zero_and_single_key():
    w, (q, k, v), (qd, kd, vd) = _inputs(1, 2, 1, 256, 128, seed=3)
    o = zyfa.attn_fwd_bf16(qd, kd, vd)
    assert torch.equal(o[0, 0, 0].cpu(), v[0, 0, 0])
    o8, (_, _, _, _, v8, vs) = zyfa.prefill_fp8(qd, kd, vd)
    zyfa.device_status()
    v0 = oracle_dequant(*oracle_quant(v, False))[0, 0, 0]
    np.testing.assert_allclose(f32(o8)[0, 0, 0], v0, rtol=2 ** -8, atol=0)


def test_gqa_equals_repeated_kv_and_is_deterministic():
    w, (q, k, v), (qd, kd, vd) = _inputs(1, 8, 2, 384, 128, seed=4)
    o1 = zyfa.attn_fwd_bf16(qd, kd, vd)
    o2 = zyfa.attn_fwd_bf16(qd, kd, vd)
    rep = lambda t: t.repeat_interleave(4, dim=2).contiguous()
    o3 = zyfa.attn_fwd_bf16(qd, rep(kd), rep(vd))
    zyfa.device_status()
    assert torch.equal(o1, o2) and torch.equal(o1, o3)
    f1, _ = zyfa.prefill_fp8(qd, kd, vd)
    f2, _ = zyfa.prefill_fp8(qd, kd, vd)
    assert torch.equal(f1, f2)


def test_strided_views_of_fused_qkv():
    g = torch.Generator().manual_seed(6)
    B, S, Hq, Hkv, D = 2, 300, 4, 2, 128
    fused = torch.randn(B, S, Hq + 2 * Hkv, D, generator=g).to(torch.bfloat16)
    fd = fused.cuda()
    q, k, v = fd[:, :, :Hq], fd[:, :, Hq:Hq + Hkv], fd[:, :, Hq + Hkv:]
    out = torch.empty(B, S, Hq, 2 * D, dtype=torch.bfloat16, device="cuda")[..., :D]  # strided output
    zyfa.attn_fwd_bf16(q, k, v, out=out)
    zyfa.device_status()
    ref = oattn.causal_attention(f32(fused[:, :, :Hq]), f32(fused[:, :, Hq:Hq + Hkv]),
                                 f32(fused[:, :, Hq + Hkv:]), 1 / math.sqrt(D))
    assert_bf16_gate(f32(out), ref, "strided")


def test_rotation_keeps_attention():
    """Hadamard rotation of Q and K leaves QK^T unchanged: the FP8 outputs with
    and without rotation agree with the unquantised result to FP8 accuracy."""
    w, (q, k, v), (qd, kd, vd) = _inputs(1, 4, 2, 512, 128, seed=9)
    o_plain, _ = zyfa.prefill_fp8(qd, kd, vd, hadamard=False)
    o_rot, _ = zyfa.prefill_fp8(qd, kd, vd, hadamard=True)
    zyfa.device_status()
    ref = oattn.causal_attention(f32(q), f32(k), f32(v), w.softmax_scale)
    assert oattn.rel_l2(f32(o_plain), ref) < 5e-2
    assert oattn.rel_l2(f32(o_rot), ref) < 5e-2


@pytest.mark.parametrize("fp8", [False, True])
def test_more_than_one_wave_with_odd_tile_count(fp8):
    """16 query heads over 21 query tiles: 176 query-tile pairs, more than
    one wave, so the units run from the host's per-CTA lists, and the last
    pair of every head has no second tile. Full output against the oracle."""
    B, Hq, Hkv, S, D = 1, 16, 4, 2688, 128
    w, (q, k, v), (qd, kd, vd) = _inputs(B, Hq, Hkv, S, D, seed=77 + fp8)
    if fp8:
        cq, sq = oracle_quant(q, False)
        ck, sk = oracle_quant(k, False)
        cv, sv = oracle_quant(v, False)
        dev = lambda a: torch.from_numpy(a).cuda()
        o = zyfa.attn_fwd_fp8(dev(cq), dev(sq), dev(ck), dev(sk), dev(cv), dev(sv), w.softmax_scale)
        ref = oattn.causal_attention(oracle_dequant(cq, sq), oracle_dequant(ck, sk), oracle_dequant(cv, sv),
                                     w.softmax_scale)
        zyfa.device_status()
        assert_fp8_gate(f32(o), ref, "fp8 multi-wave odd tiles")
    else:
        o = zyfa.attn_fwd_bf16(qd, kd, vd, w.softmax_scale)
        zyfa.device_status()
        ref = oattn.causal_attention(f32(q), f32(k), f32(v), w.softmax_scale)
        assert_bf16_gate(f32(o), ref, "bf16 multi-wave odd tiles")
