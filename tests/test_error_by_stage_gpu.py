"""Error of the FP8 path split by stage, on sampled rows of full-size
workloads (ZYFA post, "Error of a Single Attention Call" and "FP8 Error in
Full-Model Inference": input quantisation, probability quantisation, the
rest). All errors are relative L2 over the sampled rows, normalised by the
unquantised fp64 output O:

    input   = |O(dq) - O|          oracle on the oracle's dequantised Q, K, V
    P_pages = |O_P(dq) - O(dq)|    the same with P rounded per 64-key block
                                   as the pages describe (power of two, e4m3,
                                   divided back out, rounded-sum normalised)
    kernel  = |O_gpu - O(dq)|      the FP8 kernel's P rounding and arithmetic
    total   = |O_gpu - O|

The activation-like workload (outlier channels, RoPE) runs with and without
the Hadamard rotation; a Gaussian workload is the contrast. The printed table
is the report; the assertions only check what the pages' account implies:
the rotation cuts the input-quantisation error on outlier inputs, and the
kernel's P rounding costs no more than a small multiple of the pages'
scheme."""
import numpy as np
import pytest

import bf16_causal_prefill_gb300 as zyfa
import workloads
from parity import (f32, fp8_quant_blocks_for_rows, gpu_rows, oracle_dequant, oracle_quant,
                    sampled_rows_oracle, sampled_rows_pquant)

pytestmark = pytest.mark.gpu

ROWS_PER_HEAD = 6


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _stage_errors(name, had):
    w = workloads.get(name)
    q, k, v = workloads.make_qkv(w)
    had = had and w.Dqk == 128
    o, _ = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda(), hadamard=had)
    zyfa.device_status()
    rows = workloads.sample_rows(w.S, n=ROWS_PER_HEAD, seed=w.S + 1)
    got = gpu_rows(o, rows)
    del o
    kdq = oracle_dequant(*oracle_quant(k, had))
    vdq = oracle_dequant(*oracle_quant(v, False))
    qdq = np.zeros(q.shape, np.float32)
    for j, (cq, sq) in fp8_quant_blocks_for_rows(q, rows, had).items():
        qdq[:, j * 128:(j + 1) * 128] = oracle_dequant(cq, sq)
    ref = sampled_rows_oracle(f32(q), f32(k), f32(v), w.softmax_scale, rows)
    ref_dq = sampled_rows_oracle(qdq, kdq, vdq, w.softmax_scale, rows)
    ref_pq = sampled_rows_pquant(qdq, kdq, vdq, w.softmax_scale, rows)
    n = np.linalg.norm(ref.ravel())
    e = lambda a, b: float(np.linalg.norm((a - b).ravel()) / n)
    res = {"input": e(ref_dq, ref), "P_pages": e(ref_pq, ref_dq), "kernel": e(got, ref_dq),
           "total": e(got, ref), "pages_total": e(ref_pq, ref)}
    print(f"\nerror by stage {name} hadamard={had}: " + ", ".join(f"{k} {v:.3e}" for k, v in res.items()))
    return res


def test_error_by_stage_activation_like():
    plain = _stage_errors("act_b1_gqa32x8_s16k_d128", False)
    rot = _stage_errors("act_b1_gqa32x8_s16k_d128", True)
    assert rot["input"] < plain["input"]
    for r in (plain, rot):
        assert r["kernel"] <= 3.0 * r["P_pages"] + 2e-3


def test_error_by_stage_gaussian():
    r = _stage_errors("gauss_b2_gqa32x8_s8k_d128", False)
    assert r["kernel"] <= 3.0 * r["P_pages"] + 2e-3
