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
from parity import oracle_dequant, oracle_quant

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
