"""zyfa_quantize_fp8 on the GPU against the oracle: codes and scales bit-exact."""
import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads
from parity import oracle_quant

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _check(x_cpu: torch.Tensor, hadamard: bool, x_dev: torch.Tensor = None):
    x_dev = x_cpu.cuda() if x_dev is None else x_dev
    codes, scales = zyfa.quantize_fp8(x_dev, hadamard)
    zyfa.device_status()
    ref_c, ref_s = oracle_quant(x_cpu, hadamard)
    got_c, got_s = codes.cpu().numpy(), scales.cpu().numpy()
    np.testing.assert_array_equal(got_s.view(np.uint32), ref_s.view(np.uint32))
    bad = np.argwhere(got_c != ref_c)
    assert bad.size == 0, f"{len(bad)} codes differ, first at {bad[:5].tolist()}"


def _all_bf16(limit: float) -> torch.Tensor:
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16)
    x = bits.float()
    x = torch.where(torch.isfinite(x) & (x.abs() <= limit), x, torch.zeros_like(x))
    return x.to(torch.bfloat16).reshape(1, 512, 1, 128)


def test_every_bf16_pattern_plain():
    # includes bf16 subnormals, signed zeros, and the largest finite values
    _check(_all_bf16(3.0e38), hadamard=False)


def test_every_bf16_pattern_rotated():
    _check(_all_bf16(1.0e30), hadamard=True)


def test_every_bf16_pattern_shuffled_blocks():
    x = _all_bf16(3.0e38).reshape(-1)
    g = torch.Generator().manual_seed(3)
    x = x[torch.randperm(x.numel(), generator=g)].reshape(1, 256, 2, 128)
    _check(x, hadamard=False)
    _check(x.clamp(-1e30, 1e30), hadamard=True)


@pytest.mark.parametrize("S,H,D,had", [(1, 1, 128, False), (127, 2, 128, True), (300, 3, 192, False),
                                       (129, 1, 128, False), (1000, 4, 128, True)])
def test_ragged_shapes(S, H, D, had):
    g = torch.Generator().manual_seed(S + H)
    x = (torch.randn(2, S, H, D, generator=g) * 3).to(torch.bfloat16)
    _check(x, had)


def test_strided_input():
    # q, k, v as views into one fused [B, S, Hq + 2 Hkv, D] projection output
    g = torch.Generator().manual_seed(5)
    fused = torch.randn(1, 384, 8, 128, generator=g).to(torch.bfloat16)
    dev = fused.cuda()
    for lo, hi in ((0, 4), (4, 6), (6, 8)):
        _check(fused[:, :, lo:hi].contiguous(), True, dev[:, :, lo:hi])


def test_zero_block_and_signed_zero():
    x = torch.zeros(1, 256, 1, 128)
    x[0, 128:, 0, :] = -1e-6          # rounds to zero: sign kept
    x[0, 200, 0, 5] = 3.0
    x[0, 0, 0, 0] = -0.0
    _check(x.to(torch.bfloat16), False)
    codes, scales = zyfa.quantize_fp8(x.to(torch.bfloat16).cuda())
    assert scales[0, 0, 0].item() == 1.0 and codes[0, :128].eq(0).sum() == 128 * 128 - 1


@pytest.mark.parametrize("name", [workloads.SMALL, "act_b1_gqa32x8_s16k_d128"])
def test_workload_tensors(name):
    w = workloads.get(name)
    q, k, v = workloads.make_qkv(w)
    for t, had in ((q, False), (q, True), (k, True), (v, False)):
        _check(t, had)


@pytest.mark.parametrize("D,had", [(128, False), (128, True), (192, False)])
def test_unaligned_views_use_the_register_kernel(D, had):
    """Views whose base or strides do not allow 16-byte tiled copies go to the
    register kernel; contiguous tensors go to the streaming (TMA) kernel. Both
    must give the oracle's bytes."""
    g = torch.Generator().manual_seed(D + had)
    big = (torch.randn(2, 300, 3, D + 4, generator=g) * 2).to(torch.bfloat16)
    x_cpu = big[..., 2:2 + D].contiguous()
    _check(x_cpu, had, big.cuda()[..., 2:2 + D])      # stride_h = D + 4, base offset 4 bytes
    _check(x_cpu, had)                                # contiguous copy: streaming kernel
