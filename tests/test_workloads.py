"""The seeded input recipe: shapes, determinism and the activation-like structure."""
import math

import torch

import workloads as W


def test_all_workloads_have_expected_shapes():
    w = W.get("gauss_b1_mla16_s32k_d192")
    assert (w.B, w.Hq, w.Hkv, w.S, w.Dqk, w.Dv) == (1, 16, 16, 32768, 192, 128)
    assert math.isclose(w.softmax_scale, 1 / math.sqrt(192))
    assert W.get(W.BENCH).causal_flops == 32 * 32768 ** 2 * 256


def test_generation_is_deterministic_and_bf16():
    w = W.custom(1, 4, 2, 200, seed=3)
    a = W.make_qkv(w)
    b = W.make_qkv(w)
    for x, y in zip(a, b):
        assert x.dtype == torch.bfloat16
        assert torch.equal(x, y)
    assert a[0].shape == (1, 200, 4, 128) and a[1].shape == (1, 200, 2, 128)


def test_activation_like_inputs_have_outliers_and_v_std():
    import dataclasses
    w = W.get("act_b1_gqa32x8_s16k_d128").with_seq(512)
    # before RoPE: per KV head the 4 amplified channels stand out
    q0, k0, _ = W.make_qkv(dataclasses.replace(w, rope_theta=None))
    rms = k0.float().pow(2).mean(dim=(0, 1)).sqrt()          # [Hkv, D]
    top = rms.sort(dim=-1, descending=True).values
    assert torch.all(top[:, 3] > 8 * top[:, 4])
    # the same channels are amplified in every query head of the group
    qrms = q0.float().pow(2).mean(dim=(0, 1)).sqrt()
    for hk in range(w.Hkv):
        kc = set(rms[hk].topk(4).indices.tolist())
        for hq in range(hk * 4, hk * 4 + 4):
            assert set(qrms[hq].topk(4).indices.tolist()) == kc
    # RoPE rotates channel pairs (i, i + D/2): pair norms are kept (up to bf16)
    q, k, v = W.make_qkv(w)
    pn = lambda x: (x.float()[..., :64] ** 2 + x.float()[..., 64:] ** 2)
    torch.testing.assert_close(pn(k), pn(k0), rtol=2e-2, atol=2e-2)
    assert not torch.equal(k, k0)
    assert abs(v.float().std().item() - 0.5) < 0.02


def test_sample_rows_cover_edges():
    rows = W.sample_rows(1000, n=64)
    assert rows[0] == 0 and rows[-1] == 999 and 128 in rows and 127 in rows
    assert len(rows) == len(set(rows)) == 64
