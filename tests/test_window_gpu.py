"""The FP8 path's probability rounding, element by element: the kernel's
output against the oracle's emulation of the offset-window reading of the
ZYFA post's per-block scaling (oracle.attention.causal_attention_rows_window,
pinned on the CPU by tests/test_oracle_window.py), on the same e4m3 codes
and scales, sampled rows of every head, unsplit calls.

The emulation is rounded to bf16 the way the kernel stores its fp32 O / l,
and most outputs must then be bitwise equal (the kernel's fp32 scores,
exponentials and sums move a handful of e4m3 roundings). On Gaussian rows
the exact float64 oracle, which does not round P, matches far fewer: the
check sees the rounding scheme itself, well inside the FP8 gate of the
exact oracle (2.5e-2).
"""
import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from oracle import attention as oattn
from oracle import fp8 as ofp8
from parity import f32, oracle_dequant, oracle_quant

pytestmark = pytest.mark.gpu

CASES = [
    workloads.custom(1, 4, 2, 2048, seed=31),
    workloads.custom(2, 2, 2, 700, seed=32),                     # batch 2, ragged tail
    workloads.custom(1, 2, 2, 1000, Dqk=192, seed=33),           # MLA head shape, ragged tail
    workloads.custom(1, 4, 2, 4096, seed=34, v_std=0.5, outliers=4, outlier_gain=20.0, rope_theta=1.0e6),
]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> float32 -> bf16, nearest-even at each step."""
    t = torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_rounding_matches_the_window_emulation(w):
    q, k, v = workloads.make_qkv(w)
    (cq, sq), (ck, sk), (cv, sv) = (oracle_quant(x, False) for x in (q, k, v))
    dev = lambda a: torch.from_numpy(a).cuda()
    o = zyfa.attn_fwd_fp8(dev(cq), dev(sq), dev(ck), dev(sk), dev(cv), dev(sv), w.softmax_scale)
    zyfa.device_status()
    got = o.float().cpu().numpy().astype(np.float64)
    dq, dk, dv = (oracle_dequant(c, s) for c, s in ((cq, sq), (ck, sk), (cv, sv)))
    rows = sorted(set([0, 1, 127, 128, 129, 255, 256, w.S - 1] + list(range(5, w.S, max(1, w.S // 40)))))
    eq_emu = eq_exact = n = 0
    worst = 0.0
    for b in range(w.B):
        for h in range(w.Hq):
            emu = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, b, h, rows)
            ex = oattn.causal_attention_rows(dq, dk, dv, w.softmax_scale, b, h, rows)
            g = got[b, rows, h, :]
            worst = max(worst, oattn.rel_l2(g, emu))
            eq_emu += int(np.sum(g == _bf16(emu)))
            eq_exact += int(np.sum(g == _bf16(ex)))
            n += g.size
    f_emu, f_exact = eq_emu / n, eq_exact / n
    print(f"\n{w.name}: bitwise equal to the emulation {f_emu:.4f}, to the exact oracle {f_exact:.4f}; "
          f"worst head rel-L2 to the emulation {worst:.2e}")
    assert worst < 3e-3
    assert f_emu >= 0.97
    if not w.outliers:
        assert f_emu > f_exact + 0.3


def _match(got: np.ndarray, emu: np.ndarray) -> float:
    return float(np.mean(got == _bf16(emu)))


def test_split_key_ranges_match_the_chunked_emulation():
    """A call that splits each query-tile pair's keys into chunks of C tiles
    (zyfa_attn_split_tiles): every chunk starts its own offset and the
    partial rows are merged by their offsets, as the chunked emulation
    does."""
    w = workloads.custom(1, 1, 1, 4096, seed=35)
    C = zyfa.lib().zyfa_attn_split_tiles(w.B, w.S, w.Hq)
    assert C > 0
    q, k, v = workloads.make_qkv(w)
    (cq, sq), (ck, sk), (cv, sv) = (oracle_quant(x, False) for x in (q, k, v))
    dev = lambda a: torch.from_numpy(a).cuda()
    o = zyfa.attn_fwd_fp8(dev(cq), dev(sq), dev(ck), dev(sk), dev(cv), dev(sv), w.softmax_scale, split=True)
    zyfa.device_status()
    got = o.float().cpu().numpy().astype(np.float64)
    rows = sorted(set([0, 127, 128, 1023, 1024, w.S - 1] + list(range(9, w.S, 29))))
    g = got[0, rows, 0, :]
    chunked = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, 0, rows, chunk_tiles=C)
    whole = oattn.causal_attention_rows_window(cq, sq, ck, sk, cv, sv, w.softmax_scale, 0, 0, rows)
    f_chunked, f_whole = _match(g, chunked), _match(g, whole)
    print(f"\nsplit into chunks of {C} tiles: bitwise equal to the chunked emulation {f_chunked:.4f}, "
          f"to the unchunked one {f_whole:.4f}")
    assert oattn.rel_l2(g, chunked) < 3e-3
    assert f_chunked >= 0.97


def test_packed_batch_matches_the_window_emulation():
    """Packed sequences (host offsets): each sequence's keys are tiled from
    its own start and quantised on their own, so each sequence is the dense
    emulation on its slice."""
    lens, Hq, Hkv, D = [300, 1000, 129, 700], 4, 2, 128
    gen = torch.Generator().manual_seed(36)
    T = sum(lens)
    q, k, v = (torch.randn(T, H, D, generator=gen).to(torch.bfloat16) for H in (Hq, Hkv, Hkv))
    cu = [0]
    for n in lens:
        cu.append(cu[-1] + n)
    o, (q8, qs, k8, ks, v8, vs) = zyfa.prefill_fp8_varlen(q.cuda(), k.cuda(), v.cuda(), cu)
    zyfa.device_status()
    got = o.float().cpu().numpy().astype(np.float64)
    codes = []
    for x, gc in ((q, q8), (k, k8), (v, v8)):
        rc, rs = ofp8.quantize_fp8_varlen(f32(x), cu)
        np.testing.assert_array_equal(gc.cpu().numpy(), rc)
        codes.append((rc, rs))
    (cq, sq), (ck, sk), (cv, sv) = codes
    scale = 1.0 / np.sqrt(D)
    eq = n = 0
    for i, L in enumerate(lens):
        s0, nb = cu[i], (L + 127) // 128
        sl = lambda c: c[s0:s0 + L][None]
        rows = sorted(set([0, L - 1] + list(range(3, L, 41))))
        for h in range(Hq):
            emu = oattn.causal_attention_rows_window(sl(cq), sq[i:i + 1, :, :nb], sl(ck), sk[i:i + 1, :, :nb],
                                                     sl(cv), sv[i:i + 1, :, :nb], scale, 0, h, rows)
            gr = got[[s0 + r for r in rows], h, :]
            assert oattn.rel_l2(gr, emu) < 3e-3
            eq += int(np.sum(gr == _bf16(emu)))
            n += gr.size
    print(f"\npacked batch {lens}: bitwise equal to the emulation {eq / n:.4f}")
    assert eq / n >= 0.97
