"""Packed variable-length batches on the GPU against the oracle.

Sequences of mixed lengths (empty, one token, ragged tails, several tiles)
are packed along the token dimension; each must attend to itself only. BF16
and FP8 outputs are compared with the oracle element by element; the varlen
quantiser's codes and scales must equal the oracle's bit for bit; packed
equal-length sequences must reproduce the batched kernels' outputs exactly
(same tiles, same arithmetic, only the work order differs).
"""
import math

import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
from oracle import attention as oattn
from oracle import fp8 as ofp8
from parity import assert_bf16_gate, assert_fp8_gate, f32

pytestmark = pytest.mark.gpu

LENS = [1, 127, 0, 128, 129, 300, 1000, 64, 513]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _packed(lens, Hq, Hkv, D, Dv=128, seed=0):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens)
    q = torch.randn(T, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(T, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, Dv, generator=g).to(torch.bfloat16)
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    return q, k, v, cu


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 128), (2, 2, 192)])
def test_bf16_varlen_matches_oracle(Hq, Hkv, D):
    q, k, v, cu = _packed(LENS, Hq, Hkv, D, seed=D)
    o = zyfa.attn_fwd_bf16_varlen(q.cuda(), k.cuda(), v.cuda(), cu)
    zyfa.device_status()
    ref = oattn.causal_attention_varlen(f32(q), f32(k), f32(v), cu, 1 / math.sqrt(D))
    assert_bf16_gate(f32(o), ref, f"bf16 varlen D={D}")


@pytest.mark.parametrize("Hq,Hkv,D,had", [(4, 2, 128, False), (4, 2, 128, True), (2, 2, 192, False)])
def test_fp8_varlen_quantiser_and_attention(Hq, Hkv, D, had):
    q, k, v, cu = _packed(LENS, Hq, Hkv, D, seed=D + had)
    o, (q8, qs, k8, ks, v8, vs) = zyfa.prefill_fp8_varlen(q.cuda(), k.cuda(), v.cuda(), cu, hadamard=had)
    zyfa.device_status()
    refs = []
    for x, got_c, got_s, rot in ((q, q8, qs, had), (k, k8, ks, had), (v, v8, vs, False)):
        rc, rs = ofp8.quantize_fp8_varlen(f32(x), cu, rot)
        np.testing.assert_array_equal(got_c.cpu().numpy(), rc)
        written = ~np.isnan(rs)
        np.testing.assert_array_equal(got_s.cpu().numpy()[written].view(np.uint32), rs[written].view(np.uint32))
        refs.append(ofp8.dequantize_fp8_varlen(rc, rs, cu))
    ref = oattn.causal_attention_varlen(refs[0], refs[1], refs[2], cu, 1 / math.sqrt(D))
    assert_fp8_gate(f32(o), ref, f"fp8 varlen D={D} hadamard={had}")


def test_equal_lengths_reproduce_the_batched_kernels():
    B, S, Hq, Hkv, D = 3, 700, 4, 2, 128
    q, k, v, cu = _packed([S] * B, Hq, Hkv, D, seed=7)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o_var = zyfa.attn_fwd_bf16_varlen(qd, kd, vd, cu)
    o_bat = zyfa.attn_fwd_bf16(qd.view(B, S, Hq, D), kd.view(B, S, Hkv, D), vd.view(B, S, Hkv, 128))
    f_var, _ = zyfa.prefill_fp8_varlen(qd, kd, vd, cu)
    f_bat, _ = zyfa.prefill_fp8(qd.view(B, S, Hq, D), kd.view(B, S, Hkv, D), vd.view(B, S, Hkv, 128))
    zyfa.device_status()
    assert torch.equal(o_var.view(B, S, Hq, 128), o_bat)
    assert torch.equal(f_var.view(B, S, Hq, 128), f_bat)


def test_sequences_do_not_leak():
    """Changing one sequence changes no output row of the others."""
    q, k, v, cu = _packed([200, 333, 129], 2, 1, 128, seed=9)
    o1 = zyfa.attn_fwd_bf16_varlen(q.cuda(), k.cuda(), v.cuda(), cu)
    k2, v2 = k.clone(), v.clone()
    k2[200:533] = -k2[200:533]
    v2[200:533] = 2 * v2[200:533]
    o2 = zyfa.attn_fwd_bf16_varlen(q.cuda(), k2.cuda(), v2.cuda(), cu)
    zyfa.device_status()
    assert torch.equal(o1[:200], o2[:200]) and torch.equal(o1[533:], o2[533:])
    assert not torch.equal(o1[200:533], o2[200:533])


@pytest.mark.parametrize("Hq,Hkv,D,had", [(4, 2, 128, True), (2, 2, 192, False)])
@pytest.mark.parametrize("bound", [0, 300])
def test_device_offsets_reproduce_the_host_tables(Hq, Hkv, D, had, bound):
    """Offsets left on the device (tables built by a kernel) give the bytes of
    the host-offset calls; a looser max_seqlen only widens the scale arrays."""
    q, k, v, cu = _packed(LENS, Hq, Hkv, D, seed=3 * D + bound)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    max_len = max(LENS) + bound
    o_host = zyfa.attn_fwd_bf16_varlen(qd, kd, vd, cu)
    o_dev = zyfa.attn_fwd_bf16_varlen(qd, kd, vd, cu_dev, max_seqlen=max_len)
    f_host, codes_host = zyfa.prefill_fp8_varlen(qd, kd, vd, cu, hadamard=had)
    f_dev, codes_dev = zyfa.prefill_fp8_varlen(qd, kd, vd, cu_dev, hadamard=had, max_seqlen=max_len)
    zyfa.device_status()
    assert torch.equal(o_dev.view(torch.int16), o_host.view(torch.int16))
    assert torch.equal(f_dev.view(torch.int16), f_host.view(torch.int16))
    for i in (0, 2, 4):   # codes
        assert torch.equal(codes_dev[i], codes_host[i])
    for i in (1, 3, 5):   # scales: the host layout is the leading blocks of the device one
        nb = codes_host[i].shape[2]
        for b, n in enumerate(LENS):
            used = (n + 127) // 128
            assert torch.equal(codes_dev[i][b, :, :used].view(torch.int32), codes_host[i][b, :, :used].view(torch.int32))
        assert codes_dev[i].shape[2] >= nb


@pytest.mark.parametrize("bad", ["decreasing", "total", "too_long"])
def test_invalid_device_offsets_compute_nothing_and_are_reported(bad):
    lens = [100, 300, 50]
    q, k, v, cu = _packed(lens, 2, 1, 128, seed=21)
    cu_bad = list(cu)
    max_len = 300
    if bad == "decreasing":
        cu_bad[1], cu_bad[2] = cu_bad[2], cu_bad[1]
    elif bad == "total":
        cu_bad[-1] -= 1
    else:
        max_len = 299
    cu_dev = torch.tensor(cu_bad, dtype=torch.int32, device="cuda")
    zyfa.device_status()
    out = torch.full((q.shape[0], 2, 128), -7.0, dtype=torch.bfloat16, device="cuda")
    zyfa.attn_fwd_bf16_varlen(q.cuda(), k.cuda(), v.cuda(), cu_dev, out=out, max_seqlen=max_len)
    with pytest.raises(zyfa.ZyfaError) as err:
        zyfa.device_status()
    assert err.value.code == 1 and "cu_seqlens" in str(err.value)
    assert bool((out == -7.0).all())
    codes, scales = zyfa.quantize_fp8_varlen(q.cuda(), cu_dev, max_seqlen=max_len)
    with pytest.raises(zyfa.ZyfaError):
        zyfa.device_status()
    assert bool((scales == 0).all())
    assert zyfa.device_status() == 0   # the word was cleared


def test_device_offsets_at_the_sequence_limit():
    """1024 sequences (the table's limit), many empty or one token long:
    the device-built tables give the bytes of the host-built ones."""
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(0, 300, size=1024)]
    lens[17] = 0
    lens[500] = 1
    lens[1023] = 777
    q, k, v, cu = _packed(lens, 2, 1, 128, seed=11)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    cu_dev = torch.tensor(cu, dtype=torch.int32, device="cuda")
    o_host = zyfa.attn_fwd_bf16_varlen(qd, kd, vd, cu)
    o_dev = zyfa.attn_fwd_bf16_varlen(qd, kd, vd, cu_dev, max_seqlen=max(lens))
    c_host, s_host = zyfa.quantize_fp8_varlen(qd, cu)
    c_dev, s_dev = zyfa.quantize_fp8_varlen(qd, cu_dev, max_seqlen=max(lens))
    zyfa.device_status()
    assert torch.equal(o_dev.view(torch.int16), o_host.view(torch.int16))
    assert torch.equal(c_dev, c_host)
    assert torch.equal(s_dev.view(torch.int32), s_host.view(torch.int32))
