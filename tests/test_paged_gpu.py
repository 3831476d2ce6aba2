"""Queries that continue a cached sequence, with K/V in a paged cache
(chunked prefill, prefix caching), on the GPU against the oracle.

Sequences with and without a cached prefix (prefixes on and off page
boundaries; chunks that are empty, one token, ragged or several tiles) are
laid out in 128-token pages in a shuffled order; block
table entries past what a sequence needs hold an out-of-range page, so a
read past them would set the device status. BF16 and FP8 outputs are
compared with the oracle element by element (the cache quantiser's codes and
scales bit for bit). Two exact consistency checks: no prefix reproduces the
packed varlen call, and a prefix of r0 tokens reproduces rows r0.. of the
full-sequence row-range call, byte for byte.
"""
import math

import numpy as np
import pytest
import torch

import bf16_causal_prefill_gb300 as zyfa
from oracle import attention as oattn
from oracle import fp8 as ofp8
from parity import assert_bf16_gate, assert_fp8_gate, f32

pytestmark = pytest.mark.gpu

# (cached tokens, new tokens) per sequence: prefixes on and off page
# boundaries, chunks of one token (a decode step) to several tiles
SEQS = [(0, 300), (256, 129), (640, 1000), (128, 0), (384, 1), (0, 128), (1024, 77), (5, 300), (300, 129),
        (127, 1), (1000, 250), (129, 127), (77, 0)]


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    import __graft_entry__
    __graft_entry__.build()


def _sequences(seqs, Hq, Hkv, D, Dv=128, seed=0):
    g = torch.Generator().manual_seed(seed)
    out = []
    for ctx, n in seqs:
        L = ctx + n
        out.append((torch.randn(L, Hq, D, generator=g).to(torch.bfloat16),
                    torch.randn(L, Hkv, D, generator=g).to(torch.bfloat16),
                    torch.randn(L, Hkv, Dv, generator=g).to(torch.bfloat16)))
    return out


def _paged(seqs, full, extra_pages=3, seed=1):
    """Packed new queries, shuffled page caches (unused slots zero), block table."""
    g = torch.Generator().manual_seed(seed)
    need = [(ctx + n + 127) // 128 if n > 0 else 0 for ctx, n in seqs]
    P = sum(need) + extra_pages
    perm = torch.randperm(P, generator=g).tolist()
    Hkv, D = full[0][1].shape[1], full[0][1].shape[2]
    Dv = full[0][2].shape[2]
    kc = torch.zeros(P, 128, Hkv, D, dtype=torch.bfloat16)
    vc = torch.zeros(P, 128, Hkv, Dv, dtype=torch.bfloat16)
    width = max(need) + 2
    bt = torch.full((len(seqs), width), P + 1000, dtype=torch.int32)   # out of range: never read
    at = 0
    for i, ((ctx, n), (_, k, v)) in enumerate(zip(seqs, full)):
        for j in range(need[i]):
            p = perm[at]
            at += 1
            bt[i, j] = p
            cnt = min(128, ctx + n - 128 * j)
            kc[p, :cnt] = k[128 * j:128 * j + cnt]
            vc[p, :cnt] = v[128 * j:128 * j + cnt]
    q = torch.cat([f[0][ctx:] for (ctx, _), f in zip(seqs, full)])
    cu = [0]
    for _, n in seqs:
        cu.append(cu[-1] + n)
    return q, kc, vc, bt, cu


def _oracle(seqs, qs, ks, vs, scale):
    outs = [oattn.causal_attention_prefix(q[ctx:], k, v, scale) for (ctx, n), q, k, v in zip(seqs, qs, ks, vs) if n]
    return np.concatenate(outs)


@pytest.mark.parametrize("Hq,Hkv,D", [(4, 2, 128), (2, 2, 192)])
def test_bf16_paged_matches_oracle(Hq, Hkv, D):
    full = _sequences(SEQS, Hq, Hkv, D, seed=D)
    q, kc, vc, bt, cu = _paged(SEQS, full)
    o = zyfa.attn_fwd_bf16_paged(q.cuda(), kc.cuda(), vc.cuda(), cu, [c for c, _ in SEQS], bt.cuda())
    zyfa.device_status()
    ref = _oracle(SEQS, [f32(f[0]) for f in full], [f32(f[1]) for f in full], [f32(f[2]) for f in full],
                  1 / math.sqrt(D))
    assert_bf16_gate(f32(o), ref, f"bf16 paged D={D}")


def _gather(pages, bt_row, L):
    return np.concatenate([pages[p] for p in bt_row[:(L + 127) // 128]])[:L]


@pytest.mark.parametrize("Hq,Hkv,D,had", [(4, 2, 128, False), (4, 2, 128, True), (2, 2, 192, False)])
def test_fp8_paged_quantiser_and_attention(Hq, Hkv, D, had):
    full = _sequences(SEQS, Hq, Hkv, D, seed=D + had)
    q, kc, vc, bt, cu = _paged(SEQS, full)
    q8, qs = zyfa.quantize_fp8_varlen(q.cuda(), cu, had)
    kc8, ks = zyfa.quantize_fp8_cache(kc.cuda(), had)
    vc8, vs = zyfa.quantize_fp8_cache(vc.cuda(), False)
    o = zyfa.attn_fwd_fp8_paged(q8, qs, kc8, ks, vc8, vs, cu, [c for c, _ in SEQS], bt.cuda())
    zyfa.device_status()
    # quantiser: bit-exact against the oracle, pages as 128-token blocks
    rq, rqs = ofp8.quantize_fp8_varlen(f32(q), cu, had)
    np.testing.assert_array_equal(q8.cpu().numpy(), rq)
    deq = []
    for cache, got_c, got_s, rot in ((kc, kc8, ks, had), (vc, vc8, vs, False)):
        rc, rs = ofp8.quantize_fp8(f32(cache), rot)
        np.testing.assert_array_equal(got_c.cpu().numpy(), rc)
        np.testing.assert_array_equal(got_s.cpu().numpy().view(np.uint32), rs[:, :, 0].view(np.uint32))
        deq.append(ofp8.dequantize_fp8(rc, rs))
    qd = ofp8.dequantize_fp8_varlen(rq, rqs, cu)
    btn = bt.numpy()
    qs_full, ks_full, vs_full = [], [], []
    for i, (ctx, n) in enumerate(SEQS):
        if n == 0:      # no queries: its pages are never read
            qs_full.append(None), ks_full.append(None), vs_full.append(None)
            continue
        qs_full.append(np.concatenate([np.zeros((ctx, Hq, D)), qd[cu[i]:cu[i + 1]]]))
        ks_full.append(_gather(deq[0], btn[i], ctx + n))
        vs_full.append(_gather(deq[1], btn[i], ctx + n))
    ref = _oracle(SEQS, qs_full, ks_full, vs_full, 1 / math.sqrt(D))
    assert_fp8_gate(f32(o), ref, f"fp8 paged D={D} hadamard={had}")


def test_no_prefix_reproduces_the_packed_varlen_call():
    seqs = [(0, n) for n in (1, 127, 0, 128, 129, 300, 1000, 64, 513)]
    full = _sequences(seqs, 4, 2, 128, seed=11)
    q, kc, vc, bt, cu = _paged(seqs, full)
    k = torch.cat([f[1] for f in full]).cuda()
    v = torch.cat([f[2] for f in full]).cuda()
    qd, kcd, vcd, btd = q.cuda(), kc.cuda(), vc.cuda(), bt.cuda()
    ctx = [0] * len(seqs)
    assert torch.equal(zyfa.attn_fwd_bf16_paged(qd, kcd, vcd, cu, ctx, btd), zyfa.attn_fwd_bf16_varlen(qd, k, v, cu))
    q8, qs = zyfa.quantize_fp8_varlen(qd, cu)
    kc8, ks = zyfa.quantize_fp8_cache(kcd)
    vc8, vs = zyfa.quantize_fp8_cache(vcd)
    k8, kss = zyfa.quantize_fp8_varlen(k, cu)
    v8, vss = zyfa.quantize_fp8_varlen(v, cu)
    zyfa.device_status()
    assert torch.equal(zyfa.attn_fwd_fp8_paged(q8, qs, kc8, ks, vc8, vs, cu, ctx, btd),
                       zyfa.attn_fwd_fp8_varlen(q8, qs, k8, kss, v8, vss, cu))
    zyfa.device_status()


@pytest.mark.parametrize("r0", [256, 512])
def test_prefix_reproduces_the_row_range_call(r0):
    S, Hq, Hkv, D = 1000, 4, 2, 128
    (qf, kf, vf), = _sequences([(0, S)], Hq, Hkv, D, seed=r0)
    q, kc, vc, bt, cu = _paged([(r0, S - r0)], [(qf, kf, vf)])
    qd, kcd, vcd, btd = q.cuda(), kc.cuda(), vc.cuda(), bt.cuda()
    qb, kb, vb = qf.cuda()[None], kf.cuda()[None], vf.cuda()[None]
    got16 = zyfa.attn_fwd_bf16_paged(qd, kcd, vcd, cu, [r0], btd)
    ref16 = zyfa.attn_fwd_bf16(qb, kb, vb, rows=(r0, S))[0, r0:]
    assert torch.equal(got16, ref16)
    q8, qs = zyfa.quantize_fp8_varlen(qd, cu)
    kc8, ks = zyfa.quantize_fp8_cache(kcd)
    vc8, vs = zyfa.quantize_fp8_cache(vcd)
    fq8, fqs = zyfa.quantize_fp8(qb)
    fk8, fks = zyfa.quantize_fp8(kb)
    fv8, fvs = zyfa.quantize_fp8(vb)
    got8 = zyfa.attn_fwd_fp8_paged(q8, qs, kc8, ks, vc8, vs, cu, [r0], btd)
    ref8 = zyfa.attn_fwd_fp8(fq8, fqs, fk8, fks, fv8, fvs, rows=(r0, S))[0, r0:]
    zyfa.device_status()
    assert torch.equal(got8, ref8)


@pytest.mark.parametrize("fp8", [False, True])
def test_decode_steps_match_oracle(fp8):
    # one new token per sequence after prefixes of any length: a decode step
    rng = np.random.default_rng(3)
    seqs = [(int(c), 1) for c in rng.integers(0, 3000, size=16)] + [(0, 1), (127, 1), (128, 1)]
    Hq, Hkv, D = 8, 2, 128
    full = _sequences(seqs, Hq, Hkv, D, seed=21 + fp8)
    q, kc, vc, bt, cu = _paged(seqs, full)
    ctx = [c for c, _ in seqs]
    if not fp8:
        o = zyfa.attn_fwd_bf16_paged(q.cuda(), kc.cuda(), vc.cuda(), cu, ctx, bt.cuda())
        zyfa.device_status()
        ref = _oracle(seqs, [f32(f[0]) for f in full], [f32(f[1]) for f in full], [f32(f[2]) for f in full],
                      1 / math.sqrt(D))
        assert_bf16_gate(f32(o), ref, "bf16 decode")
        return
    q8, qs = zyfa.quantize_fp8_varlen(q.cuda(), cu)
    kc8, ks = zyfa.quantize_fp8_cache(kc.cuda())
    vc8, vs = zyfa.quantize_fp8_cache(vc.cuda())
    o = zyfa.attn_fwd_fp8_paged(q8, qs, kc8, ks, vc8, vs, cu, ctx, bt.cuda())
    zyfa.device_status()
    rq, rqs = ofp8.quantize_fp8_varlen(f32(q), cu, False)
    qd = ofp8.dequantize_fp8_varlen(rq, rqs, cu)
    kd = ofp8.dequantize_fp8(*ofp8.quantize_fp8(f32(kc), False))
    vd = ofp8.dequantize_fp8(*ofp8.quantize_fp8(f32(vc), False))
    btn = bt.numpy()
    ref = np.concatenate([oattn.causal_attention_prefix(qd[i:i + 1], _gather(kd, btn[i], c + 1),
                                                        _gather(vd, btn[i], c + 1), 1 / math.sqrt(D))
                          for i, (c, _) in enumerate(seqs)])
    assert_fp8_gate(f32(o), ref, "fp8 decode")


def test_out_of_range_page_sets_the_status_and_reads_zeros():
    seqs = [(128, 200)]
    full = _sequences(seqs, 2, 1, 128, seed=5)
    q, kc, vc, bt, cu = _paged(seqs, full, extra_pages=0)
    bt[0, 1] = kc.shape[0] + 7          # a page past the cache
    o = zyfa.attn_fwd_bf16_paged(q.cuda(), kc.cuda(), vc.cuda(), cu, [128], bt.cuda())
    with pytest.raises(zyfa.ZyfaError):
        zyfa.device_status()
    assert zyfa.device_status() == 0     # the status word was cleared
    assert torch.isfinite(o.float()).all()


# ----------------------------------------------------------------- decode --
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (4, 4, 128), (32, 1, 128), (4, 2, 192)])
@pytest.mark.parametrize("fp8", [False, True])
def test_decode_call_matches_oracle_and_the_paged_prefill(Hq, Hkv, D, fp8):
    """The decode call (query heads of a KV group as tile rows) against the
    oracle, with and without split key ranges; without, byte for byte against
    the paged prefill with one new token."""
    rng = np.random.default_rng(Hq + fp8)
    lens = [int(x) for x in rng.integers(1, 2500, size=13)] + [1, 2, 127, 128, 129, 256]
    seqs = [(L - 1, 1) for L in lens]
    full = _sequences(seqs, Hq, Hkv, D, seed=31 + Hq + fp8)
    q, kc, vc, bt, cu = _paged(seqs, full)
    qd, kcd, vcd, btd = q.cuda(), kc.cuda(), vc.cuda(), bt.cuda()
    ctx = [c for c, _ in seqs]
    btn = bt.numpy()
    if fp8:
        q8, qs = zyfa.quantize_fp8_decode(qd)
        kc8, ks = zyfa.quantize_fp8_cache(kcd)
        vc8, vs = zyfa.quantize_fp8_cache(vcd)
        o = zyfa.attn_decode_fp8_paged(q8, qs, kc8, ks, vc8, vs, lens, btd, split=False)
        o_split = zyfa.attn_decode_fp8_paged(q8, qs, kc8, ks, vc8, vs, lens, btd)
        q8p, qsp = zyfa.quantize_fp8_varlen(qd, cu)
        ref_gpu = zyfa.attn_fwd_fp8_paged(q8p, qsp, kc8, ks, vc8, vs, cu, ctx, btd)
        zyfa.device_status()
        assert torch.equal(q8, q8p) and torch.equal(qs.view(-1), qsp.view(-1))
        rq, rqs = ofp8.quantize_fp8_varlen(f32(q), cu, False)
        qo = ofp8.dequantize_fp8_varlen(rq, rqs, cu)
        ko = ofp8.dequantize_fp8(*ofp8.quantize_fp8(f32(kc), False))
        vo = ofp8.dequantize_fp8(*ofp8.quantize_fp8(f32(vc), False))
    else:
        o = zyfa.attn_decode_bf16_paged(qd, kcd, vcd, lens, btd, split=False)
        o_split = zyfa.attn_decode_bf16_paged(qd, kcd, vcd, lens, btd)
        ref_gpu = zyfa.attn_fwd_bf16_paged(qd, kcd, vcd, cu, ctx, btd)
        zyfa.device_status()
        qo, ko, vo = f32(q), f32(kc), f32(vc)
    ref = np.concatenate([oattn.causal_attention_prefix(qo[i:i + 1], _gather(ko, btn[i], L), _gather(vo, btn[i], L),
                                                        1 / math.sqrt(D)) for i, L in enumerate(lens)])
    gate = assert_fp8_gate if fp8 else assert_bf16_gate
    gate(f32(o), ref, f"decode fp8={fp8} Hq={Hq} Hkv={Hkv}")
    gate(f32(o_split), ref, f"decode, split key ranges, fp8={fp8} Hq={Hq} Hkv={Hkv}")
    assert torch.equal(o, ref_gpu)


@pytest.mark.parametrize("Hq,Hkv,D", [(16, 8, 128), (8, 4, 128), (64, 1, 128), (64, 1, 192)])
@pytest.mark.parametrize("fp8", [False, True])
def test_decode_small_batch_long_context_splits(Hq, Hkv, D, fp8):
    """Two sequences of 9000 and 20000 positions: a handful of tasks for the
    whole GPU, so the key ranges are split into many pieces; against the
    oracle, and within rounding of the unsplit call. 16/8 heads replicate the
    group's rows in the tile; 8/4 heads (8 tasks, too few for replicated
    rows) and 64 query heads per KV head (above 32) take the split path with
    one copy of the rows. Queries are scaled by 3 so the rows
    attend to a few hundred keys rather than near-uniformly to all 20000 (a
    flat average of random values shrinks the output to the size of the FP8
    probability-rounding noise, split or not)."""
    lens = [9000, 20000]
    seqs = [(L - 1, 1) for L in lens]
    full = _sequences(seqs, Hq, Hkv, D, seed=41 + fp8 + Hq + D)
    full = [((q.float() * 3).to(torch.bfloat16), k, v) for q, k, v in full]
    q, kc, vc, bt, cu = _paged(seqs, full)
    qd, kcd, vcd, btd = q.cuda(), kc.cuda(), vc.cuda(), bt.cuda()
    btn = bt.numpy()
    if fp8:
        q8, qs = zyfa.quantize_fp8_decode(qd)
        kc8, ks = zyfa.quantize_fp8_cache(kcd)
        vc8, vs = zyfa.quantize_fp8_cache(vcd)
        o = zyfa.attn_decode_fp8_paged(q8, qs, kc8, ks, vc8, vs, lens, btd)
        o1 = zyfa.attn_decode_fp8_paged(q8, qs, kc8, ks, vc8, vs, lens, btd, split=False)
        rq, rqs = ofp8.quantize_fp8_varlen(f32(q), cu, False)
        qo = ofp8.dequantize_fp8_varlen(rq, rqs, cu)
        ko = ofp8.dequantize_fp8(*ofp8.quantize_fp8(f32(kc), False))
        vo = ofp8.dequantize_fp8(*ofp8.quantize_fp8(f32(vc), False))
    else:
        o = zyfa.attn_decode_bf16_paged(qd, kcd, vcd, lens, btd)
        o1 = zyfa.attn_decode_bf16_paged(qd, kcd, vcd, lens, btd, split=False)
        qo, ko, vo = f32(q), f32(kc), f32(vc)
    zyfa.device_status()
    ref = np.concatenate([oattn.causal_attention_prefix(qo[i:i + 1], _gather(ko, btn[i], L), _gather(vo, btn[i], L),
                                                        1 / math.sqrt(D)) for i, L in enumerate(lens)])
    gate = assert_fp8_gate if fp8 else assert_bf16_gate
    gate(f32(o), ref, f"decode split fp8={fp8} Hq={Hq} Hkv={Hkv} D={D}")
    e_split = oattn.rel_l2(f32(o), ref)
    e_one = oattn.rel_l2(f32(o1), ref)
    assert e_split <= 1.25 * e_one + 1e-4, (e_split, e_one)
