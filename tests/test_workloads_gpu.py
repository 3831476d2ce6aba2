"""Full-size workloads, in the launch configuration the benchmark times,
checked on sampled query rows that the oracle computes one at a time: all
heads, a set of rows per head that includes row 0, tile edges and the last
row. The FP8 path is checked end to end: the GPU quantiser's codes for K, V
and the sampled Q blocks must equal the oracle's bit for bit, and the output
rows must meet the FP8 gate against the oracle on the oracle's dequantised
inputs. The error against unquantised fp64 attention is printed. The batch-2
8K workload is also checked in full (every output element, BF16 and FP8), the
oracle spread over a pool of processes."""
import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from oracle import attention as oattn
from parity import (assert_bf16_gate, assert_fp8_gate, f32, fp8_quant_blocks_for_rows, full_oracle, gpu_rows,
                    oracle_dequant, oracle_quant, sampled_rows_oracle)

pytestmark = pytest.mark.gpu

LARGE = ["gauss_b2_gqa32x8_s8k_d128", "gauss_b1_gqa32x8_s32k_d128", "gauss_b1_mla16_s32k_d192",
         "act_b1_gqa32x8_s16k_d128"]
ROWS_PER_HEAD = 256   # row 0, the first tiles' edges (t, t + 1, t + 127), the last row, seeded random rows


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


_cache = {}


def _load(name):
    if name not in _cache:
        _cache.clear()
        w = workloads.get(name)
        q, k, v = workloads.make_qkv(w)
        _cache[name] = (w, q, k, v)
    return _cache[name]


def _rows(w):
    return workloads.sample_rows(w.S, n=ROWS_PER_HEAD, seed=w.S)


@pytest.mark.parametrize("name", LARGE)
def test_bf16_sampled_rows(name):
    w, q, k, v = _load(name)
    o = zyfa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale)
    zyfa.device_status()
    rows = _rows(w)
    got = gpu_rows(o, rows)
    del o
    ref = sampled_rows_oracle(f32(q), f32(k), f32(v), w.softmax_scale, rows)
    e = assert_bf16_gate(got, ref, f"bf16 {name}")
    print(f"\n{name} bf16 sampled: {e}")


@pytest.mark.parametrize("name,hadamard", [(n, False) for n in LARGE] +
                         [("act_b1_gqa32x8_s16k_d128", True), ("gauss_b1_gqa32x8_s32k_d128", True)])
def test_fp8_sampled_rows(name, hadamard):
    w, q, k, v = _load(name)
    had = hadamard and w.Dqk == 128
    o, (q8, qs, k8, ks, v8, vs) = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda(), hadamard=had)
    zyfa.device_status()
    rows = _rows(w)
    got = gpu_rows(o, rows)
    del o
    # oracle quantisation: K and V in full, Q only in the blocks of the sampled rows
    ck, sk = oracle_quant(k, had)
    cv, sv = oracle_quant(v, False)
    assert np.array_equal(k8.cpu().numpy(), ck) and np.array_equal(ks.cpu().numpy(), sk)
    assert np.array_equal(v8.cpu().numpy(), cv) and np.array_equal(vs.cpu().numpy(), sv)
    qblocks = fp8_quant_blocks_for_rows(q, rows, had)
    q8c, qsc = q8.cpu().numpy(), qs.cpu().numpy()
    qdq = np.zeros(q.shape, np.float32)
    for j, (cq, sq) in qblocks.items():
        assert np.array_equal(q8c[:, j * 128:(j + 1) * 128], cq)
        assert np.array_equal(qsc[:, :, j:j + 1], sq)
        qdq[:, j * 128:(j + 1) * 128] = oracle_dequant(cq, sq)
    kdq = oracle_dequant(ck, sk)
    vdq = oracle_dequant(cv, sv)
    ref = sampled_rows_oracle(qdq, kdq, vdq, w.softmax_scale, rows)
    e = assert_fp8_gate(got, ref, f"fp8 {name} hadamard={had}")
    ref_exact = sampled_rows_oracle(f32(q), f32(k), f32(v), w.softmax_scale, rows)
    print(f"\n{name} fp8 hadamard={had}: vs dequantised oracle {e}, "
          f"vs unquantised fp64 rel_l2={oattn.rel_l2(got, ref_exact):.3e}")


FULL = "gauss_b2_gqa32x8_s8k_d128"


@pytest.mark.parametrize("path", ["bf16", "fp8"])
def test_full_output_b2_8k(path):
    w, q, k, v = _load(FULL)
    if path == "bf16":
        o = zyfa.attn_fwd_bf16(q.cuda(), k.cuda(), v.cuda(), w.softmax_scale)
        zyfa.device_status()
        qo, ko, vo = f32(q), f32(k), f32(v)
    else:
        o, (q8, qs, k8, ks, v8, vs) = zyfa.prefill_fp8(q.cuda(), k.cuda(), v.cuda())
        zyfa.device_status()
        deq = []
        for x, c8, sc in ((q, q8, qs), (k, k8, ks), (v, v8, vs)):
            c, s = oracle_quant(x, False)
            assert np.array_equal(c8.cpu().numpy(), c) and np.array_equal(sc.cpu().numpy(), s)
            deq.append(oracle_dequant(c, s))
        qo, ko, vo = deq
    got = f32(o)
    del o
    ref = full_oracle(qo, ko, vo, w.softmax_scale)
    gate = assert_bf16_gate if path == "bf16" else assert_fp8_gate
    e = gate(got, ref, f"{path} {FULL} full output")
    print(f"\n{FULL} {path} full output: {e}")

