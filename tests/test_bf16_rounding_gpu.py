"""The BF16 path's probability rounding, element by element: the kernel's
output against the oracle's emulation (oracle.attention.
causal_attention_rows_bf16, pinned on the CPU by
tests/test_oracle_bf16_emulation.py) on sampled rows of every head. After
rounding the emulation to bf16 most outputs must be bitwise equal; on
Gaussian rows the exact oracle, which does not round P, matches clearly
fewer, so the check sees the rounding scheme itself."""
import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from oracle import attention as oattn
from parity import f32

pytestmark = pytest.mark.gpu

CASES = [
    workloads.custom(1, 4, 2, 2048, seed=41),
    workloads.custom(2, 2, 2, 700, seed=43),                     # batch 2, ragged tail
    workloads.custom(1, 2, 2, 1000, Dqk=192, seed=44),           # MLA head shape, ragged tail
    workloads.custom(1, 4, 2, 4096, seed=42, v_std=0.5, outliers=4, outlier_gain=20.0, rope_theta=1.0e6),
]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _bf16(x: np.ndarray) -> np.ndarray:
    t = torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.float32).to(torch.bfloat16)
    return t.to(torch.float64).numpy()


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_bf16_rounding_matches_the_emulation(w):
    q, k, v = workloads.make_qkv(w)
    o = zyfa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale)
    zyfa.device_status()
    got = o.float().cpu().numpy().astype(np.float64)
    qf, kf, vf = f32(q), f32(k), f32(v)
    rows = sorted(set([0, 1, 127, 128, 129, 255, 256, w.S - 1] + list(range(5, w.S, max(1, w.S // 40)))))
    eq_emu = eq_exact = n = 0
    worst = 0.0
    for b in range(w.B):
        for h in range(w.Hq):
            emu = oattn.causal_attention_rows_bf16(qf, kf, vf, w.softmax_scale, b, h, rows)
            ex = oattn.causal_attention_rows(qf, kf, vf, w.softmax_scale, b, h, rows)
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
        assert f_emu > f_exact + 0.2
