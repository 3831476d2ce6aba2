"""The C-ABI library builds, loads without a GPU, exports every symbol that
include/zyfa.h declares, and rejects bad arguments on the host before any
launch (these calls never reach a GPU)."""
import ctypes
import os
import re

import pytest

import __graft_entry__
import bf16_causal_prefill_gb300 as zyfa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "zyfa.h")


@pytest.fixture(scope="module")
def L():
    __graft_entry__.build()
    return zyfa.lib()


def _declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(zyfa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("zyfa_quantize_fp8", "zyfa_attn_fwd_bf16", "zyfa_attn_fwd_fp8", "zyfa_get_device_status",
              "zyfa_status_string"):
        assert n in names


def test_library_exports_every_declared_symbol(L):
    for n in _declared():
        assert hasattr(L, n), f"libzyfa.so does not export {n}"


def test_status_strings(L):
    assert L.zyfa_status_string(0) == b"ok"
    assert L.zyfa_status_string(4) == b"kernel wait timed out"
    assert L.zyfa_version() >= 100


I3 = ctypes.c_int64 * 3


def _bf16(L, **kw):
    a = dict(q=16, k=16, v=16, o=16, B=1, S=128, Hq=2, Hkv=1, Dqk=128, Dv=128, scale=0.1,
             qs=I3(256, 256, 128), ks=I3(128, 128, 128), vs=I3(128, 128, 128), os_=I3(256, 256, 128))
    a.update(kw)
    return L.zyfa_attn_fwd_bf16(a["q"], a["k"], a["v"], a["o"], a["B"], a["S"], a["Hq"], a["Hkv"], a["Dqk"],
                                a["Dv"], ctypes.c_float(a["scale"]), a["qs"], a["ks"], a["vs"], a["os_"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(q=0), 1),                      # null pointer
    (dict(k=8), 1),                      # misaligned pointer
    (dict(Hq=3, Hkv=2), 1),              # Hq not a multiple of Hkv
    (dict(S=0), 1),
    (dict(Dqk=64, Dv=64), 2),            # unsupported head dims
    (dict(Dqk=192, Dv=192), 2),
    (dict(scale=-1.0), 1),
    (dict(qs=I3(256, 256, 100)), 1),     # stride not 16-byte multiple
    (dict(os_=I3(256, 0, 128)), 1),
])
def test_attention_rejects_bad_arguments_on_host(L, kw, code):
    assert _bf16(L, **kw) == code
    assert L.zyfa_last_error_message()


def test_quantiser_rejects_bad_arguments_on_host(L):
    q = L.zyfa_quantize_fp8
    assert q(None, 1, 1, 1, 16, 16, 1, 1, 1, 128, 0, None) == 1
    assert q(16, 64, 64, 64, 16, 16, 1, 1, 1, 64, 0, None) == 2          # D
    assert q(16, 192, 192, 192, 16, 16, 1, 1, 1, 192, 1, None) == 2       # rotation needs D=128
    assert q(16, 3, 128, 128, 16, 16, 1, 1, 1, 128, 0, None) == 1          # odd stride


def test_fp8_attention_needs_scales(L):
    rc = L.zyfa_attn_fwd_fp8(16, None, 16, 16, 16, 16, 16, 1, 128, 2, 1, 128, 128, ctypes.c_float(0.1),
                             I3(256, 256, 128), I3(128, 128, 128), I3(128, 128, 128), I3(256, 256, 128), 0, None)
    assert rc == 1


@pytest.mark.parametrize("flags", [2, 4, -1, 0x100])
def test_fp8_attention_refuses_unknown_flags(L, flags):
    # the flags word selects exact or lean probabilities per call; other bits are refused
    rc = L.zyfa_attn_fwd_fp8(16, 16, 16, 16, 16, 16, 16, 1, 128, 2, 1, 128, 128, ctypes.c_float(0.1),
                             I3(256, 256, 128), I3(128, 128, 128), I3(128, 128, 128), I3(256, 256, 128), flags,
                             None)
    assert rc == 1
    assert b"flags" in L.zyfa_last_error_message()


def test_python_binding_refuses_cpu_tensors():
    import torch
    x = torch.zeros(1, 128, 1, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        zyfa.quantize_fp8(x)


I2 = ctypes.c_int64 * 2


def _cu(*vals):
    return (ctypes.c_int32 * len(vals))(*vals)


def _varlen(L, cu, B, **kw):
    a = dict(q=16, k=16, v=16, o=16, Hq=2, Hkv=1, Dqk=128, Dv=128, scale=0.1,
             qs=I2(256, 128), ks=I2(128, 128), vs=I2(128, 128), os_=I2(256, 128))
    a.update(kw)
    return L.zyfa_attn_fwd_bf16_varlen(a["q"], a["k"], a["v"], a["o"], cu, B, a["Hq"], a["Hkv"], a["Dqk"], a["Dv"],
                                       ctypes.c_float(a["scale"]), a["qs"], a["ks"], a["vs"], a["os_"], None)


@pytest.mark.parametrize("cu,B,kw,code", [
    (None, 1, {}, 1),                                # null cu_seqlens
    (_cu(1, 5), 1, {}, 1),                           # cu_seqlens[0] != 0
    (_cu(0, 5, 3), 2, {}, 1),                        # decreasing
    (_cu(0, 5), 0, {}, 1),                           # no sequence
    (_cu(0, 300000), 1, {}, 2),                      # longer than the level table
    (_cu(0, 5, 9), 2, dict(Hq=3, Hkv=2), 1),         # Hq not a multiple of Hkv
    (_cu(0, 5, 9), 2, dict(qs=I2(100, 128)), 1),     # token stride not 16-byte multiple
    (_cu(0, 5, 9), 2, dict(Dqk=64, Dv=64), 2),
])
def test_varlen_attention_rejects_bad_arguments_on_host(L, cu, B, kw, code):
    assert _varlen(L, cu, B, **kw) == code
    assert L.zyfa_last_error_message()


def test_varlen_empty_batch_enqueues_nothing(L):
    # every sequence empty: valid, nothing to compute, no device touched
    assert _varlen(L, _cu(0, 0, 0), 2) == 0


def test_varlen_quantiser_rejects_bad_arguments_on_host(L):
    q = L.zyfa_quantize_fp8_varlen
    assert q(16, 128, 128, 16, 16, _cu(0, 4, 2), 2, 1, 128, 0, None) == 1    # decreasing offsets
    assert q(16, 128, 128, 16, 16, _cu(0, 4), 1, 1, 64, 0, None) == 2         # D
    assert q(16, 132, 128, 16, 16, _cu(0, 4), 1, 1, 128, 0, None) == 2        # token stride not a multiple of 8
    assert q(8, 128, 128, 16, 16, _cu(0, 4), 1, 1, 128, 0, None) == 2         # base not 16-byte aligned
    assert q(16, 128, 128, 16, 16, _cu(0, 0), 1, 1, 128, 0, None) == 0        # empty: nothing enqueued


def _rows(L, fp8, r0, r1, S=1000):
    st = (I3(S * 256, 256, 128), I3(S * 128, 128, 128), I3(S * 128, 128, 128), I3(S * 256, 256, 128))
    if fp8:
        return L.zyfa_attn_fwd_fp8_rows(16, 16, 16, 16, 16, 16, 16, 1, S, 2, 1, 128, 128, ctypes.c_float(0.1),
                                        *st, r0, r1, 0, None)
    return L.zyfa_attn_fwd_bf16_rows(16, 16, 16, 16, 1, S, 2, 1, 128, 128, ctypes.c_float(0.1), *st, r0, r1, None)


@pytest.mark.parametrize("fp8", [False, True])
@pytest.mark.parametrize("r0,r1", [(-256, 256), (0, 0), (256, 256), (512, 256), (128, 512), (0, 300),
                                   (0, 1001), (768, 1200)])
def test_row_range_attention_rejects_bad_ranges_on_host(L, fp8, r0, r1):
    # ranges are non-empty, inside [0, S), and on 256-row boundaries (or end at S)
    assert _rows(L, fp8, r0, r1) == 1
    assert "rows" in L.zyfa_last_error_message().decode()


def test_row_range_quantiser_rejects_bad_ranges_on_host(L):
    q = L.zyfa_quantize_fp8_rows
    for r0, r1 in ((-128, 128), (0, 0), (64, 256), (0, 200), (0, 1001), (256, 128)):
        assert q(16, 1000 * 128, 128, 128, 16, 16, 1, 1000, 1, 128, 0, r0, r1, None) == 1, (r0, r1)


def test_host_prefill_workspace_size(L):
    B, S, Hq, Hkv, D = 2, 1000, 4, 2, 128
    r = lambda n: (n + 255) // 256 * 256
    tq, tk = B * S * Hq * D, B * S * Hkv * D
    nb = (S + 127) // 128
    want = r(2 * tq) + 2 * r(2 * tk) + r(tq) + 2 * r(tk) + r(4 * B * Hq * nb) \
        + 2 * r(4 * B * Hkv * nb) + r(2 * tq)
    assert L.zyfa_prefill_fp8_host_workspace(B, S, Hq, Hkv, D, D) == want
    assert L.zyfa_prefill_fp8_host_workspace(0, S, Hq, Hkv, D, D) == 0


def test_host_prefill_rejects_bad_arguments_on_host(L):
    p = L.zyfa_prefill_fp8_host
    n = L.zyfa_prefill_fp8_host_workspace(1, 512, 2, 1, 128, 128)
    ok = dict(q=16, k=16, v=16, o=16, Dqk=128, Dv=128, Hq=2, Hkv=1, scale=0.1, had=0, chunks=0, ws=256, wsn=n)

    def call(**kw):
        a = dict(ok, **kw)
        return p(a["q"], a["k"], a["v"], a["o"], 1, 512, a["Hq"], a["Hkv"], a["Dqk"], a["Dv"],
                 ctypes.c_float(a["scale"]), a["had"], a["chunks"], a["ws"], a["wsn"], 0, None)

    assert call(q=0) == 1                     # null pointer
    assert call(ws=0) == 1                    # no workspace
    assert call(ws=128) == 1                  # workspace not 256-byte aligned
    assert call(wsn=n - 1) == 1               # workspace too small
    assert call(chunks=-1) == 1
    assert call(chunks=65) == 1
    assert call(Dqk=64, Dv=64) == 2
    assert call(Hq=3, Hkv=2) == 1
    assert call(Dqk=192, had=1) == 2          # rotation needs head dim 128
    assert call(scale=0.0) == 1
    assert call() == 1                        # host buffers are not page-locked
    assert "page-locked" in L.zyfa_last_error_message().decode()


def test_device_offset_varlen_rejects_bad_arguments_on_host(L):
    n = L.zyfa_varlen_workspace_bytes()
    assert n >= 4 * (2 + 3 * 1024 + 1025) and n % 256 == 0
    a = L.zyfa_attn_fwd_bf16_varlen_dev

    def call(cu=16, B=2, total=10, max_len=8, ws=256, Hq=2, Hkv=1, D=128):
        return a(16, 16, 16, 16, cu, B, total, max_len, Hq, Hkv, D, 128, ctypes.c_float(0.1), I2(256, 128),
                 I2(128, 128), I2(128, 128), I2(256, 128), ws, None)

    assert call(cu=0) == 1                       # no offsets
    assert call(B=0) == 1
    assert call(B=1025) == 1
    assert call(total=-1) == 1
    assert call(max_len=-1) == 1
    assert call(max_len=300000) == 2             # longer than the level table
    assert call(ws=0) == 1                       # no workspace
    assert call(ws=128) == 1                     # workspace not 256-byte aligned
    assert call(cu=18) == 1                      # offsets not 4-byte aligned
    assert call(Hq=3, Hkv=2) == 1
    assert call(total=0) == 0                    # nothing to compute, nothing enqueued
    q = L.zyfa_quantize_fp8_varlen_dev
    assert q(16, 128, 128, 16, 16, 0, 1, 4, 4, 1, 128, 0, 256, None) == 1
    assert q(16, 128, 128, 16, 16, 16, 1, 4, 4, 1, 64, 0, 256, None) == 2    # D
    assert q(16, 128, 128, 16, 16, 16, 1, 0, 4, 1, 128, 0, 256, None) == 0   # empty


def _paged(L, cu, ctx, B, **kw):
    a = dict(q=16, kc=16, vc=16, o=16, bt=16, bt_stride=4, pages=8, Hq=2, Hkv=1, Dqk=128, Dv=128, scale=0.1,
             qs=I2(256, 128), kcs=I3(128 * 128, 128, 128), vcs=I3(128 * 128, 128, 128), os_=I2(256, 128))
    a.update(kw)
    return L.zyfa_attn_fwd_bf16_paged(a["q"], a["kc"], a["vc"], a["o"], cu, ctx, a["bt"], a["bt_stride"],
                                      a["pages"], B, a["Hq"], a["Hkv"], a["Dqk"], a["Dv"], ctypes.c_float(a["scale"]),
                                      a["qs"], a["kcs"], a["vcs"], a["os_"], None)


@pytest.mark.parametrize("cu,ctx,B,kw,code", [
    (_cu(0, 5, 9), None, 2, {}, 1),                           # null ctx_lens
    (_cu(0, 5, 9), _cu(0, 509), 2, {}, 1),                    # 509 cached + 4 new tokens: 5 pages > 4
    (_cu(0, 5, 9), _cu(0, -128), 2, {}, 1),                   # negative context
    (_cu(0, 5, 9), _cu(0, 512), 2, {}, 1),                    # 4 cached + 1 new page > row stride 4
    (_cu(0, 5, 9), _cu(0, 384), 2, dict(bt=0), 1),            # null block table
    (_cu(0, 5, 9), _cu(0, 384), 2, dict(bt=18), 1),           # misaligned block table
    (_cu(0, 5, 9), _cu(0, 384), 2, dict(pages=0), 1),         # no pages
    (_cu(0, 5, 9), _cu(0, 384), 2, dict(kcs=I3(128 * 128, 100, 128)), 1),   # cache token stride not 16-byte
    (_cu(0, 5, 9), _cu(0, 384), 2, dict(Dqk=64, Dv=64), 2),   # head dims
    (_cu(3, 5, 9), _cu(0, 0), 2, {}, 1),                      # cu_seqlens[0] != 0
])
def test_paged_attention_rejects_bad_arguments_on_host(L, cu, ctx, B, kw, code):
    assert _paged(L, cu, ctx, B, **kw) == code
    assert L.zyfa_last_error_message()


def test_paged_empty_batch_enqueues_nothing(L):
    # no new tokens: valid, nothing to compute, no device touched
    assert _paged(L, _cu(0, 0, 0), _cu(128, 0), 2) == 0


def _decode(L, lens, N, **kw):
    a = dict(q=16, kc=16, vc=16, o=16, bt=16, bt_stride=4, pages=8, Hq=2, Hkv=1, Dqk=128, Dv=128, scale=0.1,
             qs=I2(256, 128), kcs=I3(128 * 128, 128, 128), vcs=I3(128 * 128, 128, 128), os_=I2(256, 128))
    a.update(kw)
    return L.zyfa_attn_decode_bf16_paged(a["q"], a["kc"], a["vc"], a["o"], lens, a["bt"], a["bt_stride"],
                                         a["pages"], N, a["Hq"], a["Hkv"], a["Dqk"], a["Dv"],
                                         ctypes.c_float(a["scale"]), a["qs"], a["kcs"], a["vcs"], a["os_"], None, 0,
                                         None)


@pytest.mark.parametrize("lens,N,kw,code", [
    (None, 1, {}, 1),                                  # null seq_lens
    (_cu(5, 0), 2, {}, 1),                             # a sequence without its new token
    (_cu(5, 513), 2, {}, 1),                           # 513 positions: 5 pages > row stride 4
    (_cu(5), 0, {}, 1),                                # no sequence
    (_cu(5), 1, dict(qs=I2(512, 128)), 1),             # heads of a token not contiguous
    (_cu(5), 1, dict(Hq=3, Hkv=2), 1),                 # Hq not a multiple of Hkv
    (_cu(5), 1, dict(Hq=256, Hkv=1, qs=I2(256 * 128, 128)), 1),   # more than 128 heads per KV head
    (_cu(5), 1, dict(bt=0), 1),                        # null block table
    (_cu(5), 1, dict(Dqk=64, Dv=64), 2),               # head dims
])
def test_decode_rejects_bad_arguments_on_host(L, lens, N, kw, code):
    assert _decode(L, lens, N, **kw) == code
    assert L.zyfa_last_error_message()


def test_decode_workspace_size(L):
    L.zyfa_decode_workspace_bytes.restype = ctypes.c_size_t
    small = L.zyfa_decode_workspace_bytes(1, 32, 8)
    big = L.zyfa_decode_workspace_bytes(64, 32, 8)
    assert small > 0 and big > small and small % 4 == 0


def test_python_paged_and_decode_bindings_check_tensors_before_any_launch():
    # CPU tensors (and a wrong dtype) are refused in the binding, before the
    # library is called
    import torch
    q = torch.zeros(4, 2, 128, dtype=torch.bfloat16)
    cache = torch.zeros(3, 128, 1, 128, dtype=torch.bfloat16)
    bt = torch.zeros(2, 3, dtype=torch.int32)
    with pytest.raises(ValueError):                       # CPU tensors
        zyfa.attn_fwd_bf16_paged(q, cache, cache, [0, 2, 4], [0, 0], bt)
    with pytest.raises(ValueError):
        zyfa.attn_decode_bf16_paged(q, cache, cache, [5, 5, 5, 5], torch.zeros(4, 3, dtype=torch.int32))
    with pytest.raises(ValueError):
        zyfa.quantize_fp8_cache(torch.zeros(3, 64, 1, 128, dtype=torch.bfloat16))
    with pytest.raises(ValueError):
        zyfa.quantize_fp8_decode(torch.zeros(4, 2, 128, dtype=torch.float32))


def test_noalloc_call_refuses_what_its_static_table_cannot_hold(L):
    # the static scratch holds one unit table: at most 1024 sequences of at
    # most 262144 tokens; larger calls fail on the host before any device work
    assert L.zyfa_noalloc_scratch_bytes() == 32768
    s2 = (ctypes.c_int64 * 2)(128, 128)
    def call(B, max_len):
        return L.zyfa_attn_fwd_fp8_varlen_dev_noalloc(16, 16, 16, 16, 16, 16, 16, 16, B, 1000, max_len, 1, 1, 128,
                                                       128, ctypes.c_float(0.1), s2, s2, s2, s2, 0, None)
    assert call(2000, 1000) == 1
    assert b"static scratch" in L.zyfa_last_error_message()
    assert call(0, 1000) == 1
    assert call(4, 300000) == 2
    assert b"static scratch" in L.zyfa_last_error_message()



def test_attn_workspace_size(L):
    """Split key ranges apply to problems of fewer than 256 query-tile pairs
    with more than two query tiles (at most 8 chunks per query tile); the
    size grows with the problem."""
    f = L.zyfa_attn_workspace_bytes
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int] * 3
    assert f(1, 256, 8) == 0                  # one pair of at most two key blocks: nothing to split
    assert f(1, 32768, 32) == 0               # 4096 pairs fill the GPU
    assert f(0, 1024, 2) == 0 and f(1, 0, 2) == 0
    small, big = f(1, 1024, 2), f(1, 16384, 1)
    # 1K, 2 heads: 4 chunks (2 key blocks each) x 1024 rows x 2 heads partial
    # rows of 128 fp32 + (m, l)
    assert small == 4 * 1024 * 2 * 128 * 4 + 4 * 1024 * 2 * 8
    # 16K, 1 head: 8 chunks of 16 key blocks
    assert big == 8 * 16384 * 128 * 4 + 8 * 16384 * 8


def test_attn_ws_calls_refuse_bad_arguments_before_launch(L):
    s3 = (ctypes.c_int64 * 3)(128 * 2, 128, 128)
    rc = L.zyfa_attn_fwd_bf16_ws(None, 16, 16, 16, 1, 128, 2, 2, 128, 128, ctypes.c_float(0.1), s3, s3, s3, s3,
                                 None, 0, None)
    assert rc == 1   # ZYFA_ERR_INVALID_ARG: null q


def test_attn_split_tiles_refuses_bad_sizes(L):
    assert L.zyfa_attn_split_tiles(0, 1024, 2) == -1
    assert L.zyfa_attn_split_tiles(1, 0, 2) == -1
