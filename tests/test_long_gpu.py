"""A 128K-token sequence (4x the longest benchmark configuration): offsets,
row sums and output indexing at 1024 key tiles per row, checked on sampled
rows (including the last) against the oracle, BF16 and FP8 (both modes of
the FP8 probabilities), plus the same sequence through the packed
variable-length entry point next to a short one."""
import math

import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
from oracle import attention as oattn
from parity import (FP8_REL_L2, assert_bf16_gate, assert_fp8_gate, f32, fp8_quant_blocks_for_rows, gpu_rows,
                    oracle_dequant, oracle_quant, sampled_rows_oracle)

pytestmark = pytest.mark.gpu

S = 131072
ROWS = [0, 1, 127, 128, 4095, 65536, 100000, S - 129, S - 1]


@pytest.fixture(scope="module")
def inputs(cuda_device):
    import __graft_entry__
    __graft_entry__.build()
    g = torch.Generator().manual_seed(12)
    q = torch.randn(1, S, 2, 128, generator=g).to(torch.bfloat16)
    k = torch.randn(1, S, 1, 128, generator=g).to(torch.bfloat16)
    v = torch.randn(1, S, 1, 128, generator=g).to(torch.bfloat16)
    return q, k, v


def test_bf16_128k(inputs):
    q, k, v = inputs
    o = zyfa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda())
    zyfa.device_status()
    ref = sampled_rows_oracle(f32(q), f32(k), f32(v), 1 / math.sqrt(128), ROWS)
    assert_bf16_gate(gpu_rows(o, ROWS), ref, "bf16 128K")


@pytest.mark.parametrize("mode", ["exact", "lean"])
def test_fp8_128k(inputs, mode):
    q, k, v = inputs
    o, _ = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda(), lean_p=(mode == "lean"))
    zyfa.device_status()
    kdq = oracle_dequant(*oracle_quant(k, False))
    vdq = oracle_dequant(*oracle_quant(v, False))
    qdq = np.zeros(q.shape, np.float32)
    for j, (cq, sq) in fp8_quant_blocks_for_rows(q, ROWS, False).items():
        qdq[:, j * 128:(j + 1) * 128] = oracle_dequant(cq, sq)
    ref = sampled_rows_oracle(qdq, kdq, vdq, 1 / math.sqrt(128), ROWS)
    assert_fp8_gate(gpu_rows(o, ROWS), ref, f"fp8 128K {mode}")


def test_varlen_128k_next_to_a_short_sequence(inputs):
    q, k, v = inputs
    short = 300
    qp = torch.cat([q[0, :short], q[0]], 0).cuda()
    kp = torch.cat([k[0, :short], k[0]], 0).cuda()
    vp = torch.cat([v[0, :short], v[0]], 0).cuda()
    cu = [0, short, short + S]
    o = zyfa.attn_fwd_bf16_varlen(qp, kp, vp, cu)
    ob = zyfa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda())
    zyfa.device_status()
    assert torch.equal(o[short:], ob[0])
    assert torch.equal(o[:short], ob[0, :short])
