"""The packed FP8 attention call that allocates nothing
(zyfa_attn_fwd_fp8_varlen_dev_noalloc).

Some callers cannot allocate device memory where they call attention: a step
replayed from a CUDA graph whose memory was fixed when it was captured, or a
serving loop that hands out device memory only from its own pool. For them the
library keeps the call's unit table in a static device array instead of a
caller workspace. Every call reuses that array, so this test makes two calls
in a row on two different batches (the second overwrites the first's table)
and checks each output against the workspace form of the same call, within
the FP8 gate the other tests use; the two forms run the same kernels on the
same table, so their bytes agree as well.

The file name sorts last, so a run that stops at the first failure has run
every other test before this one; the test also passes alone in a fresh
process (the first call there looks up the array's device address).
"""
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
from parity import assert_fp8_gate, f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _batch(lens, Hq, Hkv, seed):
    g = torch.Generator().manual_seed(seed)
    T = sum(lens)
    q = torch.randn(T, Hq, 128, generator=g).to(torch.bfloat16).cuda()
    k = torch.randn(T, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    v = torch.randn(T, Hkv, 128, generator=g).to(torch.bfloat16).cuda()
    offs = [0]
    for n in lens:
        offs.append(offs[-1] + n)
    cu = torch.tensor(offs, dtype=torch.int32, device="cuda")
    max_len = max(lens)
    q8, qs = zyfa.quantize_fp8_varlen(q, cu, max_seqlen=max_len)
    k8, ks = zyfa.quantize_fp8_varlen(k, cu, max_seqlen=max_len)
    v8, vs = zyfa.quantize_fp8_varlen(v, cu, max_seqlen=max_len)
    return (q8, qs, k8, ks, v8, vs), cu, max_len


def test_two_calls_in_a_row_match_the_workspace_call():
    cases = [_batch([300, 1, 1000, 129, 0, 513], 4, 2, seed=11), _batch([64, 777, 256], 8, 2, seed=12)]
    refs = [zyfa.attn_fwd_fp8_varlen(*t, cu, max_seqlen=m) for t, cu, m in cases]
    zyfa.device_status()
    # the caller owns the outputs; the two calls below run back to back
    outs = [torch.empty_like(r) for r in refs]
    for (t, cu, m), out in zip(cases, outs):
        zyfa.attn_fwd_fp8_varlen_dev_noalloc(*t, cu, m, out)
    zyfa.device_status()
    for i, (out, ref) in enumerate(zip(outs, refs)):
        assert_fp8_gate(f32(out), f32(ref), f"no-alloc call {i}")
        assert torch.equal(out, ref), f"no-alloc call {i}: bytes differ from the workspace call"
