"""Row ranges ("chunked prefill") and the prefill from host memory, on the GPU.

A call restricted to query rows [r0, r1) must write exactly those rows, with
the bytes the full call writes there, and leave every other row untouched;
the quantiser's row-range form likewise for its 128-token blocks. The host
prefill pipelines copies, quantisation and attention along the sequence and
must return the bytes of the device-resident FP8 path; a small case is also
held against the oracle directly.
"""
import math

import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
from oracle import attention as oattn
from oracle import fp8 as ofp8
from parity import assert_fp8_gate, f32

pytestmark = pytest.mark.gpu

SENTINEL = -7.0


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _inputs(B, S, Hq, Hkv, D, Dv=128, seed=0):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, S, Hq, D, generator=g).to(torch.bfloat16)
    k = torch.randn(B, S, Hkv, D, generator=g).to(torch.bfloat16)
    v = torch.randn(B, S, Hkv, Dv, generator=g).to(torch.bfloat16)
    return q, k, v


def _bounds(S, pieces):
    """Piece boundaries on 256-row multiples, the last piece ending at S."""
    b = sorted({min(S, p) for p in pieces} | {0, S})
    return list(zip(b[:-1], b[1:]))


CASES = [(2, 1000, 4, 2, 128), (1, 2309, 2, 1, 128), (2, 777, 2, 2, 192)]


@pytest.mark.parametrize("B,S,Hq,Hkv,D", CASES)
@pytest.mark.parametrize("fp8", [False, True])
def test_row_ranges_reproduce_the_full_call(B, S, Hq, Hkv, D, fp8):
    q, k, v = (t.cuda() for t in _inputs(B, S, Hq, Hkv, D, seed=S + D))
    if fp8:
        args = (*zyfa.quantize_fp8(q), *zyfa.quantize_fp8(k), *zyfa.quantize_fp8(v))
        call = lambda **kw: zyfa.attn_fwd_fp8(*args, **kw)
    else:
        call = lambda **kw: zyfa.attn_fwd_bf16(q, k, v, **kw)
    full = call()
    pieced = torch.full_like(full, SENTINEL)
    for r0, r1 in _bounds(S, [256, 768, 1280, 2048]):
        call(out=pieced, rows=(r0, r1))
    zyfa.device_status()
    assert torch.equal(pieced.view(torch.int16), full.view(torch.int16))
    # one range alone touches nothing outside it
    if S > 512:
        one = torch.full_like(full, SENTINEL)
        call(out=one, rows=(256, 512))
        zyfa.device_status()
        assert torch.equal(one[:, 256:512].view(torch.int16), full[:, 256:512].view(torch.int16))
        assert bool((one[:, :256] == SENTINEL).all()) and bool((one[:, 512:] == SENTINEL).all())


@pytest.mark.parametrize("B,S,H,D,had", [(2, 1000, 3, 128, True), (1, 777, 2, 192, False)])
def test_quantiser_row_ranges_reproduce_the_full_call(B, S, H, D, had):
    x = _inputs(B, S, H, H, D, seed=S)[0].cuda()
    codes, scales = zyfa.quantize_fp8(x, had)
    c2 = torch.full_like(codes, 0x5A)
    s2 = torch.full_like(scales, SENTINEL)
    for r0, r1 in _bounds(S, [128, 384, 512]):
        zyfa.quantize_fp8(x, had, out=c2, scales=s2, rows=(r0, r1))
    zyfa.device_status()
    assert torch.equal(c2, codes)
    assert torch.equal(s2.view(torch.int32), scales.view(torch.int32))
    c3 = torch.full_like(codes, 0x5A)
    s3 = torch.full_like(scales, SENTINEL)
    zyfa.quantize_fp8(x, had, out=c3, scales=s3, rows=(128, 384))
    zyfa.device_status()
    assert torch.equal(c3[:, 128:384], codes[:, 128:384])
    assert bool((c3[:, :128] == 0x5A).all()) and bool((c3[:, 384:] == 0x5A).all())
    assert torch.equal(s3[:, :, 1:3].view(torch.int32), scales[:, :, 1:3].view(torch.int32))
    assert bool((s3[:, :, 0] == SENTINEL).all()) and bool((s3[:, :, 3:] == SENTINEL).all())


@pytest.mark.parametrize("B,S,Hq,Hkv,D,had", [(2, 1000, 4, 2, 128, True), (1, 2309, 2, 1, 128, False),
                                              (2, 777, 2, 2, 192, False)])
@pytest.mark.parametrize("n_chunks", [1, 3, 0, 64])
def test_host_prefill_equals_device_path(B, S, Hq, Hkv, D, had, n_chunks):
    q, k, v = (t.pin_memory() for t in _inputs(B, S, Hq, Hkv, D, seed=S + n_chunks))
    o_dev, _ = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda(), hadamard=had)
    o_host = zyfa.prefill_fp8_host(q, k, v, hadamard=had, n_chunks=n_chunks)
    torch.cuda.current_stream().synchronize()
    zyfa.device_status()
    assert not o_host.is_cuda
    assert torch.equal(o_host.view(torch.int16), o_dev.cpu().view(torch.int16))


def test_host_prefill_reuses_its_workspace_back_to_back():
    B, S, Hq, Hkv, D = 1, 1536, 4, 2, 128
    ws = zyfa.prefill_fp8_host_workspace(B, S, Hq, Hkv, D, D)
    outs, refs = [], []
    for seed in range(3):
        q, k, v = (t.pin_memory() for t in _inputs(B, S, Hq, Hkv, D, seed=100 + seed))
        refs.append(zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda())[0].cpu())
        outs.append(zyfa.prefill_fp8_host(q, k, v, n_chunks=4, workspace=ws))
    torch.cuda.current_stream().synchronize()
    zyfa.device_status()
    for o, r in zip(outs, refs):
        assert torch.equal(o.view(torch.int16), r.view(torch.int16))


def test_host_prefill_matches_oracle():
    B, S, Hq, Hkv, D = 1, 600, 2, 1, 128
    q, k, v = (t.pin_memory() for t in _inputs(B, S, Hq, Hkv, D, seed=11))
    o = zyfa.prefill_fp8_host(q, k, v, hadamard=True, n_chunks=3)
    torch.cuda.current_stream().synchronize()
    zyfa.device_status()
    deq = []
    for x, rot in ((q, True), (k, True), (v, False)):
        c, s = ofp8.quantize_fp8(f32(x), rot)
        deq.append(ofp8.dequantize_fp8(c, s))
    ref = oattn.causal_attention(deq[0], deq[1], deq[2], 1 / math.sqrt(D))
    assert_fp8_gate(f32(o), ref, "host prefill")


def test_host_prefill_refuses_pageable_buffers():
    q, k, v = _inputs(1, 256, 2, 1, 128)
    with pytest.raises(ValueError):
        zyfa.prefill_fp8_host(q, k, v)


def test_host_prefill_at_the_bench_size_equals_device_path():
    """The end-to-end configuration the benchmark times (32K GQA, default
    pieces): same bytes as the device-resident FP8 path, whose outputs the
    full-size workload tests hold against the oracle."""
    import workloads
    w = workloads.get(workloads.BENCH)
    q, k, v = workloads.make_qkv(w)
    hq, hk, hv = (t.pin_memory() for t in (q, k, v))
    o_dev, _ = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda(), softmax_scale=w.softmax_scale)
    o_host = zyfa.prefill_fp8_host(hq, hk, hv, softmax_scale=w.softmax_scale)
    torch.cuda.current_stream().synchronize()
    zyfa.device_status()
    assert torch.equal(o_host.view(torch.int16), o_dev.cpu().view(torch.int16))
