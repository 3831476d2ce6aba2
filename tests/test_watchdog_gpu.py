"""Failure detection without a GPU fault: a test hook makes the attention
kernel's loader warp issue nothing, so every consumer's bounded wait runs out.
The kernel must record the timeout in the device status word, exit cleanly,
free its tensor memory, and leave the context usable for the next call."""
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def test_stalled_loader_reports_timeout_and_context_survives():
    w = workloads.custom(1, 2, 1, 512, seed=1)
    q, k, v = (t.cuda() for t in workloads.make_qkv(w))
    good = zyfa.attn_fwd_bf16(q, k, v)
    zyfa.device_status()
    try:
        zyfa.set_debug(stall_loader=True, timeout_seconds=0.2)
        zyfa.attn_fwd_bf16(q, k, v)
        with pytest.raises(zyfa.ZyfaError) as ei:
            zyfa.device_status()
        assert ei.value.code == 4
    finally:
        zyfa.set_debug(False, 0.0)
    again = zyfa.attn_fwd_bf16(q, k, v)
    assert zyfa.device_status() == 0
    assert torch.equal(good, again)
