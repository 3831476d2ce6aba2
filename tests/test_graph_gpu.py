"""The calls enqueue only kernels on the caller's stream (no allocation, no
synchronisation, tensor maps passed by value), so a prefill can be captured
into a CUDA graph once and replayed on new inputs; the replay must produce
the bytes of the eager calls."""
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _qkv(seed, B=1, S=1000, Hq=4, Hkv=2, D=128):
    g = torch.Generator().manual_seed(seed)
    mk = lambda h: torch.randn(B, S, h, D, generator=g).to(torch.bfloat16).cuda()
    return mk(Hq), mk(Hkv), mk(Hkv)


def test_graph_replay_matches_eager():
    q, k, v = _qkv(0)
    nb = zyfa.scale_blocks(q.shape[1])
    q8 = torch.empty(q.shape, dtype=torch.uint8, device="cuda")
    k8 = torch.empty(k.shape, dtype=torch.uint8, device="cuda")
    v8 = torch.empty(v.shape, dtype=torch.uint8, device="cuda")
    qs = torch.empty((1, 4, nb), device="cuda")
    ks = torch.empty((1, 2, nb), device="cuda")
    vs = torch.empty((1, 2, nb), device="cuda")
    o8 = torch.empty((1, q.shape[1], 4, 128), dtype=torch.bfloat16, device="cuda")
    o16 = torch.empty_like(o8)

    def step():
        zyfa.quantize_fp8(q, True, out=q8, scales=qs)
        zyfa.quantize_fp8(k, True, out=k8, scales=ks)
        zyfa.quantize_fp8(v, False, out=v8, scales=vs)
        zyfa.attn_fwd_fp8(q8, qs, k8, ks, v8, vs, out=o8)
        zyfa.attn_fwd_bf16(q, k, v, out=o16)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                       # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for seed in (1, 2):
        nq, nk, nv = _qkv(seed)
        q.copy_(nq)
        k.copy_(nk)
        v.copy_(nv)
        graph.replay()
        torch.cuda.synchronize()
        got8, got16 = o8.clone(), o16.clone()
        ref8, _ = zyfa.prefill_fp8(nq, nk, nv, hadamard=True)
        ref16 = zyfa.attn_fwd_bf16(nq, nk, nv)
        zyfa.device_status()
        assert torch.equal(got8.view(torch.int16), ref8.view(torch.int16))
        assert torch.equal(got16.view(torch.int16), ref16.view(torch.int16))
