"""Few query-tile pairs with split key ranges (zyfa_attn_fwd_{bf16,fp8}_ws)
against the float64 oracle, full outputs.

When a call has fewer query-tile pairs than SMs (long sequences with few
heads), the longest pair's chain of key blocks sets its time; with a caller
workspace the library may split every pair's key blocks into chunks run by
separate CTAs, a second kernel combining the chunks' partial rows. The
shapes below split on a GB300 (chunks of 4, 6 and 10 key blocks): an odd
number of query tiles (the last pair without its second tile), ragged
tails, GQA, batch 2 and the MLA head shape. They are compared with the
oracle under the same gates as the unsplit calls, and with the unsplit
calls. The 1K-token workload does not split (its fixed costs outweigh the
gain) and then the workspace call reproduces the unsplit call's bytes.
"""
import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from oracle import attention as oattn
from parity import assert_bf16_gate, assert_fp8_gate, f32, oracle_dequant, oracle_quant

pytestmark = pytest.mark.gpu

SHAPES = [  # B, Hq, Hkv, S, Dqk
    (1, 1, 1, 4096, 128),     # chunks of 4 key blocks
    (1, 1, 1, 4200, 128),     # 33 query tiles (the last pair has tile A only), ragged, chunks of 6
    (1, 2, 1, 4096, 128),     # GQA
    (2, 1, 1, 4000, 128),     # batch 2, ragged tail
    (1, 1, 1, 4096, 192),     # MLA head shape
    (1, 1, 1, 8192, 128),     # chunks of 10
]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _inputs(B, Hq, Hkv, S, D, seed):
    w = workloads.custom(B, Hq, Hkv, S, Dqk=D, Dv=128, seed=seed)
    q, k, v = workloads.make_qkv(w)
    return w, (q, k, v)


@pytest.mark.parametrize("B,Hq,Hkv,S,D", SHAPES)
def test_split_bf16_matches_oracle(B, Hq, Hkv, S, D):
    assert zyfa.lib().zyfa_attn_workspace_bytes(B, S, Hq) > 0
    assert zyfa.lib().zyfa_attn_split_tiles(B, S, Hq) > 0
    w, (q, k, v) = _inputs(B, Hq, Hkv, S, D, seed=S + 7)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o = zyfa.attn_fwd_bf16(qd, kd, vd, w.softmax_scale, split=True)
    o_plain = zyfa.attn_fwd_bf16(qd, kd, vd, w.softmax_scale)
    zyfa.device_status()
    ref = oattn.causal_attention(f32(q), f32(k), f32(v), w.softmax_scale)
    assert_bf16_gate(f32(o), ref, f"bf16 split {B, Hq, Hkv, S, D}")
    d = (o.float() - o_plain.float()).norm() / o_plain.float().norm()
    assert d < 5e-3, f"split and unsplit calls differ by {d}"


@pytest.mark.parametrize("B,Hq,Hkv,S,D", SHAPES)
def test_split_fp8_matches_oracle(B, Hq, Hkv, S, D):
    w, (q, k, v) = _inputs(B, Hq, Hkv, S, D, seed=S + 8)
    had = D == 128
    cq, sq = oracle_quant(q, had)
    ck, sk = oracle_quant(k, had)
    cv, sv = oracle_quant(v, False)
    dev = lambda a: torch.from_numpy(a).cuda()
    args = (dev(cq), dev(sq), dev(ck), dev(sk), dev(cv), dev(sv), w.softmax_scale)
    o = zyfa.attn_fwd_fp8(*args, split=True)
    o_plain = zyfa.attn_fwd_fp8(*args)
    zyfa.device_status()
    ref = oattn.causal_attention(oracle_dequant(cq, sq), oracle_dequant(ck, sk), oracle_dequant(cv, sv),
                                 w.softmax_scale)
    assert_fp8_gate(f32(o), ref, f"fp8 split {B, Hq, Hkv, S, D}")
    # per-chunk offsets round P differently: the split path really ran
    assert not torch.equal(o, o_plain)


def test_small_workload_does_not_split():
    """The 1K workload through the workspace calls equals the unsplit calls
    bitwise: there the library keeps one CTA per query-tile pair."""
    w = workloads.get(workloads.SMALL)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    assert zyfa.lib().zyfa_attn_workspace_bytes(w.B, w.S, w.Hq) > 0
    assert zyfa.lib().zyfa_attn_split_tiles(w.B, w.S, w.Hq) == 0
    o1, _ = zyfa.prefill_fp8(qd, kd, vd, split=True)
    o2, _ = zyfa.prefill_fp8(qd, kd, vd)
    b1 = zyfa.attn_fwd_bf16(qd, kd, vd, split=True)
    b2 = zyfa.attn_fwd_bf16(qd, kd, vd)
    zyfa.device_status()
    assert torch.equal(o1, o2) and torch.equal(b1, b2)


def test_split_prefill_and_graph():
    """A splitting shape through prefill_fp8(split=True): codes bit-exact,
    within the FP8 gate of the oracle, deterministic, and replayed from a
    CUDA graph with the same bytes."""
    w = workloads.custom(1, 2, 1, 4096, seed=11)
    q, k, v = workloads.make_qkv(w)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o1, (q8, qs, k8, ks, v8, vs) = zyfa.prefill_fp8(qd, kd, vd, split=True)
    o2, _ = zyfa.prefill_fp8(qd, kd, vd, split=True)
    zyfa.device_status()
    assert torch.equal(o1, o2)
    oq = [oracle_quant(x, had) for x, had in ((q, False), (k, False), (v, False))]
    for (c, sc), (gc, gs) in zip(oq, ((q8, qs), (k8, ks), (v8, vs))):
        assert np.array_equal(gc.cpu().numpy(), c) and np.array_equal(gs.cpu().numpy(), sc)
    ref = oattn.causal_attention(*(oracle_dequant(c, sc) for c, sc in oq), w.softmax_scale)
    assert_fp8_gate(f32(o1), ref, "fp8 split prefill")
    o_plain, _ = zyfa.prefill_fp8(qd, kd, vd)
    assert not torch.equal(o1, o_plain)
    ws = torch.empty(zyfa.lib().zyfa_attn_workspace_bytes(w.B, w.S, w.Hq), dtype=torch.uint8, device="cuda")
    out = torch.empty_like(o1)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        zyfa.attn_fwd_fp8(q8, qs, k8, ks, v8, vs, w.softmax_scale, out=out, split=ws)   # warm-up
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=s):
            zyfa.attn_fwd_fp8(q8, qs, k8, ks, v8, vs, w.softmax_scale, out=out, split=ws)
    torch.cuda.current_stream().wait_stream(s)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    zyfa.device_status()
    assert torch.equal(out, o1)


def test_split_workspace_too_small_is_refused():
    w, (q, k, v) = _inputs(1, 1, 1, 4096, 128, seed=3)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    need = zyfa.lib().zyfa_attn_workspace_bytes(1, 4096, 1)
    small = torch.empty(need - 256, dtype=torch.uint8, device="cuda")
    with pytest.raises(zyfa.ZyfaError):
        zyfa.attn_fwd_bf16(qd, kd, vd, w.softmax_scale, split=small)
