"""Q, K and V quantised in one launch (zyfa_quantize_fp8_qkv and its
row-range and packed forms) against the oracle: codes and scales bit-exact,
and the same bytes as one call per tensor."""
import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
from oracle import fp8 as ofp8
from parity import f32, oracle_quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _qkv(B, S, Hq, Hkv, Dqk, Dv, seed):
    g = torch.Generator().manual_seed(seed)
    q = (torch.randn(B, S, Hq, Dqk, generator=g) * 2).to(torch.bfloat16)
    k = (torch.randn(B, S, Hkv, Dqk, generator=g) * 3).to(torch.bfloat16)
    v = torch.randn(B, S, Hkv, Dv, generator=g).to(torch.bfloat16)
    return q, k, v


def _assert_oracle(x_cpu, had, codes, scales, what):
    rc, rs = oracle_quant(x_cpu, had)
    np.testing.assert_array_equal(scales.cpu().numpy().view(np.uint32), rs.view(np.uint32), err_msg=what)
    bad = np.argwhere(codes.cpu().numpy() != rc)
    assert bad.size == 0, f"{what}: {len(bad)} codes differ, first at {bad[:5].tolist()}"


CASES = [(2, 1000, 4, 2, 128, 128, False), (2, 1000, 4, 2, 128, 128, True), (1, 640, 4, 4, 192, 128, False),
         (1, 1, 2, 1, 128, 128, True), (3, 257, 8, 1, 128, 128, True), (1, 3000, 16, 2, 128, 128, False)]


@pytest.mark.parametrize("B,S,Hq,Hkv,Dqk,Dv,had", CASES)
def test_one_launch_matches_the_oracle_and_the_single_calls(B, S, Hq, Hkv, Dqk, Dv, had):
    q, k, v = _qkv(B, S, Hq, Hkv, Dqk, Dv, seed=S + Hq + had)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    got = zyfa.quantize_fp8_qkv(qd, kd, vd, had)
    zyfa.device_status()
    for x, xd, (c, s), rot, n in ((q, qd, got[0], had, "q"), (k, kd, got[1], had, "k"), (v, vd, got[2], False, "v")):
        _assert_oracle(x, rot, c, s, n)
        c1, s1 = zyfa.quantize_fp8(xd, rot)
        assert torch.equal(c, c1) and torch.equal(s.view(torch.int32), s1.view(torch.int32)), n


def test_views_into_a_fused_projection():
    # q, k, v as head slices of one [B, S, Hq + 2 Hkv, D] tensor: tileable
    # strides, so still one launch
    g = torch.Generator().manual_seed(9)
    fused = (torch.randn(2, 700, 12, 128, generator=g) * 2).to(torch.bfloat16)
    dev = fused.cuda()
    got = zyfa.quantize_fp8_qkv(dev[:, :, :8], dev[:, :, 8:10], dev[:, :, 10:], True)
    zyfa.device_status()
    for (lo, hi), (c, s), rot, n in (((0, 8), got[0], True, "q"), ((8, 10), got[1], True, "k"),
                                     ((10, 12), got[2], False, "v")):
        _assert_oracle(fused[:, :, lo:hi].contiguous(), rot, c, s, n)


def test_unaligned_views_fall_back_per_tensor():
    # a 4-byte base offset rules out tiled copies for q only: k and v still
    # stream, q takes the register kernel; same bytes either way
    g = torch.Generator().manual_seed(10)
    big = (torch.randn(1, 300, 4, 132, generator=g) * 2).to(torch.bfloat16)
    q_cpu = big[..., 2:130].contiguous()
    _, k, v = _qkv(1, 300, 4, 2, 128, 128, seed=11)
    got = zyfa.quantize_fp8_qkv(big.cuda()[..., 2:130], k.cuda(), v.cuda(), True)
    zyfa.device_status()
    _assert_oracle(q_cpu, True, *got[0], "q")
    _assert_oracle(k, True, *got[1], "k")
    _assert_oracle(v, False, *got[2], "v")


def test_row_pieces_equal_the_whole_call():
    q, k, v = _qkv(2, 1100, 4, 2, 128, 128, seed=12)
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    whole = zyfa.quantize_fp8_qkv(qd, kd, vd, True)
    pieces = tuple((torch.full(c.shape, 0xAB, dtype=torch.uint8, device="cuda"),
                    torch.full(s.shape, -1.0, device="cuda")) for c, s in whole)
    for r0, r1 in ((0, 256), (256, 768), (768, 1100)):
        zyfa.quantize_fp8_qkv(qd, kd, vd, True, rows=(r0, r1), out=pieces)
    zyfa.device_status()
    for (c, s), (pc, ps) in zip(whole, pieces):
        assert torch.equal(c, pc) and torch.equal(s.view(torch.int32), ps.view(torch.int32))


LENS = [1, 127, 0, 128, 129, 300, 1000, 64, 513]


@pytest.mark.parametrize("Hq,Hkv,Dqk,had", [(4, 2, 128, True), (4, 2, 128, False), (2, 2, 192, False)])
@pytest.mark.parametrize("device_offsets", [False, True])
def test_packed_batch_matches_the_oracle(Hq, Hkv, Dqk, had, device_offsets):
    g = torch.Generator().manual_seed(Dqk + had)
    T = sum(LENS)
    q = torch.randn(T, Hq, Dqk, generator=g).to(torch.bfloat16)
    k = torch.randn(T, Hkv, Dqk, generator=g).to(torch.bfloat16)
    v = torch.randn(T, Hkv, 128, generator=g).to(torch.bfloat16)
    cu = np.concatenate([[0], np.cumsum(LENS)]).astype(np.int32).tolist()
    offs = torch.tensor(cu, dtype=torch.int32, device="cuda") if device_offsets else cu
    got = zyfa.quantize_fp8_qkv_varlen(q.cuda(), k.cuda(), v.cuda(), offs, had,
                                       max_seqlen=max(LENS) if device_offsets else None)
    assert zyfa.device_status() == 0
    for x, (c, s), rot, n in ((q, got[0], had, "q"), (k, got[1], had, "k"), (v, got[2], False, "v")):
        rc, rs = ofp8.quantize_fp8_varlen(f32(x), cu, rot)
        np.testing.assert_array_equal(c.cpu().numpy(), rc, err_msg=n)
        written = ~np.isnan(rs)
        np.testing.assert_array_equal(s.cpu().numpy()[written].view(np.uint32), rs[written].view(np.uint32),
                                      err_msg=n)
