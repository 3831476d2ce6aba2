// C-ABI entry points: argument validation, TMA descriptor encoding, device
// status word, and the launches of the quantiser and attention kernels.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <queue>
#include <vector>

#include "../../include/zyfa.h"
#include "internal.h"

namespace {

thread_local char g_last_error[512] = "";

int fail(int code, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return code;
}

int fail_cuda(cudaError_t e, const char* what) {
  return fail(ZYFA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// FP8 attention flags: ZYFA_FP8_LEAN_P selects lean P; no other bit is
// defined. Returns 0 (exact P) or 1 (lean P), or -1 for unknown bits.
int fp8_flags_lean(int flags) {
  if (flags & ~ZYFA_FP8_LEAN_P) return -1;
  return (flags & ZYFA_FP8_LEAN_P) ? 1 : 0;
}
int lean_flags_error(int flags) {
  return fail(ZYFA_ERR_INVALID_ARG, "unknown FP8 flags 0x%x (only ZYFA_FP8_LEAN_P is defined)", flags);
}

// Per-device state, filled on first use of a device.
constexpr int kMaxDevices = 64;
struct DeviceInfo {
  bool ready = false;
  int sm_count = 0;
  int cc_major = 0, cc_minor = 0;
  unsigned int* status = nullptr;   // address of the status word on this device
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

uint64_t g_timeout_ns = 2000000000ull;
int g_debug_stall = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

}  // namespace

// One word per device; kernels OR timeout codes into it.
__device__ unsigned int zyfa_device_status_word;

namespace {

int device_info(DeviceInfo** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ZYFA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess)
      return fail_cuda(e, "cudaDeviceGetAttribute(SM count)");
    cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev);
    void* p = nullptr;
    if ((e = cudaGetSymbolAddress(&p, zyfa_device_status_word)) != cudaSuccess)
      return fail_cuda(e, "cudaGetSymbolAddress(status word)");
    d.status = static_cast<unsigned int*>(p);
    if (!g_encode) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
        return fail(ZYFA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    d.ready = true;
  }
  if (!(d.cc_major == 10 && d.cc_minor == 3))
    return fail(ZYFA_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a", dev, d.cc_major,
                d.cc_minor);
  *out = &d;
  return ZYFA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// 5-D tiled map over a [B, S, H, D] tensor that splits D into 128-byte column
// blocks and puts tokens before blocks (dims innermost first: 128 bytes of D,
// S, D / 128 bytes, H, B), so one box = a whole 128-token tile of one head,
// laid out in shared memory as column block after column block of
// 128 rows x 128 bytes (the layout the MMA descriptors expect), 128-byte
// swizzle, out-of-range tokens read as zero.
// A row that is not a whole number of 128-byte blocks (e4m3 at head dim 192)
// keeps a 4-D map (D, H, S, B) with a 128-byte box per column block: its last
// box runs past the row and reads zeros, where a 5-D block would read the
// next head (or past the tensor).
int make_map(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int elt, int D, int H, int S, int B,
             const int64_t strides[3], const char* name, int box_rows = 128) {
  if ((D * elt) % 128 != 0 || box_rows != 128) {
    const cuuint64_t dims[4] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(H), static_cast<cuuint64_t>(S),
                                static_cast<cuuint64_t>(B)};
    const cuuint64_t gstrides[3] = {static_cast<cuuint64_t>(strides[2]) * elt,
                                    static_cast<cuuint64_t>(strides[1]) * elt,
                                    static_cast<cuuint64_t>(strides[0]) * elt};
    const cuuint32_t box[4] = {static_cast<cuuint32_t>(128 / elt), 1u, static_cast<cuuint32_t>(box_rows), 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(map, dt, 4, const_cast<void*>(base), dims, gstrides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(ZYFA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
    return ZYFA_OK;
  }
  const int inner = 128 / elt;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(S),
                              static_cast<cuuint64_t>(D / inner), static_cast<cuuint64_t>(H),
                              static_cast<cuuint64_t>(B)};
  const cuuint64_t gstrides[4] = {static_cast<cuuint64_t>(strides[1]) * elt, 128u,
                                  static_cast<cuuint64_t>(strides[2]) * elt,
                                  static_cast<cuuint64_t>(strides[0]) * elt};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(inner), 128u, static_cast<cuuint32_t>(D / inner), 1u, 1u};
  const cuuint32_t estr[5] = {1u, 1u, 1u, 1u, 1u};
  CUresult r = g_encode(map, dt, 5, const_cast<void*>(base), dims, gstrides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ZYFA_ERR_INVALID_ARG, "cuTensorMapEncodeTiled(%s) failed: %d", name, (int)r);
  return ZYFA_OK;
}

int check_strides(const int64_t s[3], int64_t mult, const char* name) {
  if (!s) return fail(ZYFA_ERR_INVALID_ARG, "%s strides pointer is null", name);
  for (int i = 0; i < 3; ++i) {
    if (s[i] <= 0) return fail(ZYFA_ERR_INVALID_ARG, "%s stride[%d] = %lld must be positive", name, i, (long long)s[i]);
    if (s[i] % mult != 0)
      return fail(ZYFA_ERR_INVALID_ARG, "%s stride[%d] = %lld must be a multiple of %lld elements", name, i,
                  (long long)s[i], (long long)mult);
    if (s[i] >= (int64_t(1) << 38)) return fail(ZYFA_ERR_INVALID_ARG, "%s stride[%d] too large", name, i);
  }
  return ZYFA_OK;
}

struct AttnCommon {
  int B, S, Hq, Hkv, Dqk, Dv;
  float softmax_scale;
};

int validate_attn(const AttnCommon& c, const void* q, const void* k, const void* v, void* o, int64_t in_mult,
                  const int64_t qs[3], const int64_t ks[3], const int64_t vs[3], const int64_t os[3]) {
  if (!q || !k || !v || !o) return fail(ZYFA_ERR_INVALID_ARG, "null tensor pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16))
    return fail(ZYFA_ERR_INVALID_ARG, "tensor pointers must be 16-byte aligned");
  if (c.B < 1 || c.S < 1 || c.Hq < 1 || c.Hkv < 1)
    return fail(ZYFA_ERR_INVALID_ARG, "B, S, Hq, Hkv must be >= 1 (got %d, %d, %d, %d)", c.B, c.S, c.Hq, c.Hkv);
  if (c.Hq % c.Hkv != 0) return fail(ZYFA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", c.Hq, c.Hkv);
  if (!((c.Dqk == 128 && c.Dv == 128) || (c.Dqk == 192 && c.Dv == 128)))
    return fail(ZYFA_ERR_UNSUPPORTED, "head dims (%d, %d) unsupported; use (128, 128) or (192, 128)", c.Dqk, c.Dv);
  if (!(c.softmax_scale > 0.f) || !std::isfinite(c.softmax_scale))
    return fail(ZYFA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  const long long n_qtiles = (c.S + 127) / 128;
  if (static_cast<long long>(c.B) * c.Hq * ((n_qtiles + 1) / 2) >= (1LL << 31))
    return fail(ZYFA_ERR_INVALID_ARG, "problem too large");
  int r;
  if ((r = check_strides(qs, in_mult, "q")) || (r = check_strides(ks, in_mult, "k")) ||
      (r = check_strides(vs, in_mult, "v")) || (r = check_strides(os, 8, "o")))
    return r;
  return ZYFA_OK;
}

}  // namespace

extern "C" {

int zyfa_version(void) { return 100; }

const char* zyfa_status_string(int status) {
  switch (status) {
    case ZYFA_OK: return "ok";
    case ZYFA_ERR_INVALID_ARG: return "invalid argument";
    case ZYFA_ERR_UNSUPPORTED: return "unsupported";
    case ZYFA_ERR_CUDA: return "CUDA error";
    case ZYFA_ERR_TIMEOUT: return "kernel wait timed out";
    default: return "unknown status";
  }
}

const char* zyfa_last_error_message(void) { return g_last_error; }

int zyfa_set_debug(int stall_loader, double timeout_seconds) {
  g_debug_stall = stall_loader ? 1 : 0;
  g_timeout_ns = timeout_seconds > 0 ? static_cast<uint64_t>(timeout_seconds * 1e9) : 2000000000ull;
  return ZYFA_OK;
}

// One tensor of a quantiser call.
struct QuantIn {
  const void* x;            // bf16
  int64_t sb, ss, sh;       // element strides of x (packed: sb unused)
  void* out;                // e4m3 codes, dense
  float* scales;
  int H, D, hadamard;
  const char* name;
};

static int check_quant_in(const QuantIn& t) {
  if (!t.x || !t.out || !t.scales) return fail(ZYFA_ERR_INVALID_ARG, "%s: null pointer", t.name);
  if (t.H < 1 || t.H > 65535) return fail(ZYFA_ERR_INVALID_ARG, "%s: H must be in 1..65535", t.name);
  if (t.D != 128 && t.D != 192) return fail(ZYFA_ERR_UNSUPPORTED, "%s: head dim %d unsupported (128 or 192)", t.name, t.D);
  if (t.hadamard && t.D != 128) return fail(ZYFA_ERR_UNSUPPORTED, "%s: Hadamard rotation needs head dim 128", t.name);
  if (!aligned(t.x, 4) || !aligned(t.out, 2) || !aligned(t.scales, 4))
    return fail(ZYFA_ERR_INVALID_ARG, "%s: misaligned pointer", t.name);
  if (t.sb <= 0 || t.ss <= 0 || t.sh <= 0 || (t.sb | t.ss | t.sh) & 1)
    return fail(ZYFA_ERR_INVALID_ARG, "%s: strides must be positive and even", t.name);
  return ZYFA_OK;
}

// Inputs whose base and strides allow 16-byte tiled copies go to the
// streaming kernel; other views to the register kernel (same bytes).
static bool quant_tileable(const QuantIn& t) {
  const int64_t lim = int64_t(1) << 38;
  return aligned(t.x, 16) && aligned(t.out, 16) && t.sb % 8 == 0 && t.ss % 8 == 0 && t.sh % 8 == 0 && t.sb < lim &&
         t.ss < lim && t.sh < lim;
}

static int quant_stream_tensor(const QuantIn& t, int B, int S, zyfa::QuantMaps* m, zyfa::QuantStreamArgs* a, int i) {
  const int64_t xs[3] = {t.sb, t.ss, t.sh};
  const int64_t os[3] = {static_cast<int64_t>(S) * t.H * t.D, static_cast<int64_t>(t.H) * t.D, t.D};
  int r = make_map(&m->in[i], t.x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, t.D, t.H, S, B, xs, t.name);
  if (!r) r = make_map(&m->out[i], t.out, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, t.D, t.H, S, B, os, t.name);
  if (r) return r;
  a->t[i].out = static_cast<uint8_t*>(t.out);
  a->t[i].scales = t.scales;
  a->t[i].H = t.H;
  a->t[i].D = t.D;
  a->t[i].hadamard = t.hadamard;
  return ZYFA_OK;
}

// Equal-length tensors [B,S,H_t,D_t], 128-token blocks covering rows
// [row_begin, row_end): one streaming launch for all of them when every
// tensor can be tiled, else one launch per tensor.
static int quant_dense(const QuantIn* in, int n, int B, int S, int row_begin, int row_end, void* stream) {
  if (B < 1 || S < 1) return fail(ZYFA_ERR_INVALID_ARG, "B, S, H must be >= 1");
  if (row_begin < 0 || row_end > S || row_begin >= row_end || row_begin % 128 != 0 ||
      (row_end != S && row_end % 128 != 0))
    return fail(ZYFA_ERR_INVALID_ARG, "row range [%d, %d) must be non-empty, inside [0, %d), on 128-token blocks",
                row_begin, row_end, S);
  if ((static_cast<long long>(S) + 127) / 128 > 65535 * 1024LL || B > 65535)
    return fail(ZYFA_ERR_INVALID_ARG, "grid too large");
  bool all_tile = true;
  for (int t = 0; t < n; ++t) {
    if (int r = check_quant_in(in[t])) return r;
    all_tile = all_tile && quant_tileable(in[t]);
  }
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  zyfa::QuantStreamArgs a{};
  a.B = B;
  a.S = S;
  a.blk_lo = row_begin / 128;
  a.blk_hi = (row_end + 127) / 128;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns;
  for (int t0 = 0; t0 < n; t0 = all_tile ? n : t0 + 1) {
    const int t1 = all_tile ? n : t0 + 1;
    cudaError_t e;
    if (quant_tileable(in[t0])) {
      zyfa::QuantMaps m{};
      int dmax = 128;
      for (int t = t0; t < t1; ++t) {
        if (int r = quant_stream_tensor(in[t], B, S, &m, &a, t - t0)) return r;
        dmax = std::max(dmax, in[t].D);
      }
      a.n = t1 - t0;
      e = zyfa::launch_quantize_fp8_stream(m, a, dmax, d->sm_count, st);
    } else {
      const QuantIn& t = in[t0];
      zyfa::QuantArgs r{};
      r.x = t.x;
      r.sb = t.sb;
      r.ss = t.ss;
      r.sh = t.sh;
      r.out = static_cast<uint8_t*>(t.out);
      r.scales = t.scales;
      r.B = B;
      r.S = S;
      r.H = t.H;
      r.D = t.D;
      r.blk_lo = a.blk_lo;
      r.blk_hi = a.blk_hi;
      r.hadamard = t.hadamard;
      r.status = d->status;
      r.timeout_ns = g_timeout_ns;
      r.num_sms = d->sm_count;
      e = zyfa::launch_quantize_fp8(r, st);
    }
    if (e != cudaSuccess) return fail_cuda(e, "quantize_fp8 launch");
  }
  return ZYFA_OK;
}

static int quant_common(const void* x, int64_t stride_b, int64_t stride_s, int64_t stride_h, void* out,
                        float* scales, int B, int S, int H, int D, int hadamard, int row_begin, int row_end,
                        void* stream) {
  const QuantIn t{x, stride_b, stride_s, stride_h, out, scales, H, D, hadamard, "x"};
  return quant_dense(&t, 1, B, S, row_begin, row_end, stream);
}

static int quant_qkv(const void* q, const int64_t qs[3], const void* k, const int64_t ks[3], const void* v,
                     const int64_t vs[3], void* q8, float* q_scale, void* k8, float* k_scale, void* v8,
                     float* v_scale, int B, int S, int Hq, int Hkv, int Dqk, int Dv, int hadamard, int row_begin,
                     int row_end, void* stream) {
  if (!qs || !ks || !vs) return fail(ZYFA_ERR_INVALID_ARG, "null strides pointer");
  if (!((Dqk == 128 || Dqk == 192) && Dv == 128))
    return fail(ZYFA_ERR_UNSUPPORTED, "head dims (%d, %d) unsupported; use (128, 128) or (192, 128)", Dqk, Dv);
  const QuantIn in[3] = {{q, qs[0], qs[1], qs[2], q8, q_scale, Hq, Dqk, hadamard, "q"},
                         {k, ks[0], ks[1], ks[2], k8, k_scale, Hkv, Dqk, hadamard, "k"},
                         {v, vs[0], vs[1], vs[2], v8, v_scale, Hkv, Dv, 0, "v"}};
  return quant_dense(in, 3, B, S, row_begin, row_end, stream);
}

int zyfa_quantize_fp8(const void* x, int64_t stride_b, int64_t stride_s, int64_t stride_h, void* out,
                      float* scales, int B, int S, int H, int D, int hadamard, void* stream) {
  return quant_common(x, stride_b, stride_s, stride_h, out, scales, B, S, H, D, hadamard, 0, S, stream);
}

int zyfa_quantize_fp8_rows(const void* x, int64_t stride_b, int64_t stride_s, int64_t stride_h, void* out,
                           float* scales, int B, int S, int H, int D, int hadamard, int row_begin, int row_end,
                           void* stream) {
  return quant_common(x, stride_b, stride_s, stride_h, out, scales, B, S, H, D, hadamard, row_begin, row_end,
                      stream);
}

int zyfa_quantize_fp8_qkv(const void* q, const int64_t q_strides[3], const void* k, const int64_t k_strides[3],
                          const void* v, const int64_t v_strides[3], void* q8, float* q_scale, void* k8,
                          float* k_scale, void* v8, float* v_scale, int B, int S, int Hq, int Hkv, int Dqk, int Dv,
                          int hadamard, void* stream) {
  return quant_qkv(q, q_strides, k, k_strides, v, v_strides, q8, q_scale, k8, k_scale, v8, v_scale, B, S, Hq, Hkv,
                   Dqk, Dv, hadamard, 0, S, stream);
}

int zyfa_quantize_fp8_qkv_rows(const void* q, const int64_t q_strides[3], const void* k, const int64_t k_strides[3],
                               const void* v, const int64_t v_strides[3], void* q8, float* q_scale, void* k8,
                               float* k_scale, void* v8, float* v_scale, int B, int S, int Hq, int Hkv, int Dqk,
                               int Dv, int hadamard, int row_begin, int row_end, void* stream) {
  return quant_qkv(q, q_strides, k, k_strides, v, v_strides, q8, q_scale, k8, k_scale, v8, v_scale, B, S, Hq, Hkv,
                   Dqk, Dv, hadamard, row_begin, row_end, stream);
}

// Work order of the equal-length kernels: how many (batch, KV head) groups
// have their units interleaved (longest query-tile pairs first within each
// such super-group). Eight, or four when the K/V of eight groups would fill
// more than half of L2 (64 MiB of 129 MB): the query heads sharing a K/V
// tile then find it in L2 instead of re-reading it from HBM (bf16 at 32K
// tokens: 3.0x the algorithmic DRAM bytes with eight groups, 1.26x with
// four). Three, five or six groups ran 2-9% slower than four or eight.
static int groups_in_flight(int S, int Dqk, int Dv, int elt) {
  constexpr double kHalfL2Bytes = 64.0 * (1 << 20);
  const double group_bytes = static_cast<double>(S) * (Dqk + Dv) * elt;
  return 8 * group_bytes > kHalfL2Bytes ? 4 : 8;
}

// Few query-tile pairs (fewer than SMs, e.g. a long sequence with few
// heads): the longest pair's chain of key blocks sets the time while most
// SMs idle. With a caller workspace the key blocks of every pair can be
// split into chunks of C blocks (C even, at most kMaxKeyChunks chunks per
// query tile) that run on separate CTAs, a second kernel combining the
// chunks' partial rows. The host picks C with a cost model in units of one
// key block of a pair (~1.25 us on a GB300): the kernel's static schedule
// simulated (unit u on CTA u mod grid, pairs longest first, kUnitCost per
// unit for its start and its partial-row stores) plus the combine, which
// moves every partial row twice (written, then read: kCombineBytesPerBlock
// per key block of time) after a second launch (kCombineLaunch). It splits
// only where that comes to less than 85% of the unsplit schedule with
// kMinGain blocks to spare. The constants were fitted to GB300 timings of
// split and unsplit calls (FP8, one and two heads, 4K to 32K tokens): one
// head at 4K, 8K, 16K tokens ran 1.8x, 2.1x, 1.7x faster split, two heads
// at 16K 7% slower (left unsplit by the model), the 1K-token 2-head
// workload unsplit.
constexpr int kMaxKeyChunks = 8;
constexpr int kUnitCost = 4;
constexpr int kMinGain = 4;
constexpr double kCombineBytesPerBlock = 2.5e6;
constexpr int kCombineLaunch = 5;

static int pair_key_blocks(int t, int nq) { return (2 * t + 1 < nq) ? 2 * t + 2 : 2 * t + 1; }

// Largest per-CTA cost of the static schedule with chunks of C key blocks
// (C = 0: one unit per pair), and the unit count.
static long long schedule_cost(int B, int Hq, int nq, int sms, int C, long long* units) {
  const int pairs = (nq + 1) / 2;
  const long long bh = static_cast<long long>(B) * Hq;
  long long n = 0;
  for (int t = 0; t < pairs; ++t) n += C ? (pair_key_blocks(t, nq) + C - 1) / C : 1;
  n *= bh;
  *units = n;
  const long long grid = std::min<long long>(n, sms);
  std::vector<long long> load(static_cast<size_t>(std::max<long long>(grid, 1)), 0);
  long long u = 0;
  for (int t = pairs - 1; t >= 0; --t) {
    const int nk = pair_key_blocks(t, nq);
    const int nch = C ? (nk + C - 1) / C : 1;
    for (int c = 0; c < nch; ++c) {
      const int len = C ? std::min(C, nk - c * C) : nk;
      for (long long i = 0; i < bh; ++i, ++u) load[static_cast<size_t>(u % grid)] += len + kUnitCost;
    }
  }
  long long cost = *std::max_element(load.begin(), load.end());
  if (C) {
    // partial rows: both query tiles of pair t write one per chunk of its key blocks
    double rows = 0;
    for (int t = 0; t < pairs; ++t) rows += (2 * t + 1 < nq ? 2 : 1) * 128.0 * ((pair_key_blocks(t, nq) + C - 1) / C);
    rows *= static_cast<double>(bh);
    cost += kCombineLaunch + static_cast<long long>(2.0 * rows * (128 * 4 + 8) / kCombineBytesPerBlock);
  }
  return cost;
}

// Problems of this many query-tile pairs or more never split, whatever the
// SM count: the workspace size does not depend on the GPU.
constexpr int kMaxSmsForPrefillSplit = 256;

static int min_split_tiles(int nq) {
  const int c = (nq + kMaxKeyChunks - 1) / kMaxKeyChunks;
  return std::max(2, (c + 1) & ~1);
}

// C for this problem on `sms` SMs, or 0 (no split); units: the split unit count.
static int prefill_split_tiles(int B, int S, int Hq, int sms, long long* units) {
  if (B < 1 || S < 1 || Hq < 1 || sms < 1) return 0;
  const int nq = (S + 127) / 128, pairs = (nq + 1) / 2;
  if (static_cast<long long>(B) * Hq * pairs >= std::min(sms, kMaxSmsForPrefillSplit)) return 0;
  long long n0;
  const long long plain = schedule_cost(B, Hq, nq, sms, 0, &n0);
  long long best = plain;
  int best_c = 0, prev = 0;
  // candidates: the smallest even C giving the longest query tile k chunks
  for (int k = kMaxKeyChunks; k >= 2; --k) {
    const int c = (nq + k - 1) / k;
    const int C = std::max(min_split_tiles(nq), (c + 1) & ~1);
    if (C >= nq || C == prev) continue;
    prev = C;
    long long n;
    const long long cost = schedule_cost(B, Hq, nq, sms, C, &n) + kMinGain;
    if (cost < best) { best = cost; best_c = C; }
  }
  if (best_c && 100 * best >= 85 * plain) best_c = 0;
  if (best_c) schedule_cost(B, Hq, nq, sms, best_c, units);
  return best_c;
}

// Partial rows of a split call: at most kMaxKeyChunks chunks x B x 128 tiles x
// Hq, for problems of fewer than kMaxSmsForPrefillSplit pairs and more than
// two query tiles (whether the call splits depends on the GPU's SM count);
// 0 otherwise.
static size_t prefill_partial_rows(int B, int S, int Hq) {
  if (B < 1 || S < 1 || Hq < 1) return 0;
  const int nq = (S + 127) / 128, pairs = (nq + 1) / 2;
  if (nq <= 2 || static_cast<long long>(B) * Hq * pairs >= kMaxSmsForPrefillSplit) return 0;
  const int chunks = (nq + min_split_tiles(nq) - 1) / min_split_tiles(nq);
  return static_cast<size_t>(chunks) * B * (static_cast<size_t>(nq) * 128) * Hq;
}

static size_t prefill_ws_bytes(int B, int S, int Hq) {
  // per partial row: 128 fp32 of O, then (m, l) after the O block
  const size_t rows = prefill_partial_rows(B, S, Hq);
  return rows ? ((rows * 128 * 4 + 255) & ~size_t(255)) + rows * 2 * 4 : 0;
}

// Multi-wave equal-length calls: CTA c of the persistent kernel would run
// units c, c + grid, ... (round robin); with query-tile pairs of very
// different lengths that leaves the busiest CTA with several percent more
// work than the average (32K GQA: 3.5%; 8K batch 2 and the activation-like
// 16K: about 10%, by the model below). The host instead hands the units out
// in the kernel's order, each to the CTA with the least work so far (what a
// work queue would do, without one): cost = the pair's key blocks plus
// kListUnitCost for the unit's start. The list goes to the kernel as a
// parameter, cached for the last shape.
constexpr int kListUnitCost = 2;

static int unit_key_blocks(int u, const zyfa::AttnArgs& a, int n_qtiles) {
  const int n_pairs = a.pair_hi - a.pair_lo, G = a.Hq / a.Hkv, n_groups = a.B * a.Hkv;
  const int gif = std::max(1, a.groups_in_flight);
  const int per_sg = gif * G * n_pairs;
  const int sg = u / per_sg, r = u - sg * per_sg;
  const int gs_here = std::min(gif, n_groups - sg * gif);
  const int t = a.pair_hi - 1 - r / (gs_here * G);
  return (2 * t + 1 < n_qtiles) ? 2 * t + 2 : 2 * t + 1;
}

static const zyfa::UnitList* unit_list(const zyfa::AttnArgs& a) {
  const long long n = static_cast<long long>(a.B) * a.Hq * (a.pair_hi - a.pair_lo);
  const int G = a.num_sms;
  if (n <= G || n > zyfa::kMaxListUnits || G > zyfa::kMaxListCtas) return nullptr;
  // Row-range calls (the host pipeline's pieces) keep the round robin: their
  // pairs are of similar length, and consecutive pieces on two streams fill
  // each other's idle SMs (the end-to-end prefill measured 0.2 ms slower
  // with per-piece lists).
  if (a.pair_lo != 0 || a.pair_hi != (a.S + 255) / 256) return nullptr;
  static thread_local zyfa::UnitList list;
  static thread_local long long key[8] = {-1};
  const long long k[8] = {a.B, a.S, a.Hq, a.Hkv, a.pair_lo, a.pair_hi, a.groups_in_flight, G};
  if (std::equal(k, k + 8, key)) return &list;
  const int n_qtiles = (a.S + 127) / 128;
  std::vector<int> owner(static_cast<size_t>(n));
  std::vector<int> count(G, 0);
  using Load = std::pair<long long, int>;
  std::priority_queue<Load, std::vector<Load>, std::greater<Load>> heap;
  for (int c = 0; c < G; ++c) heap.push({0, c});
  for (int u = 0; u < n; ++u) {
    const Load top = heap.top();
    heap.pop();
    owner[u] = top.second;
    ++count[top.second];
    heap.push({top.first + unit_key_blocks(u, a, n_qtiles) + kListUnitCost, top.second});
  }
  list.start[0] = 0;
  for (int c = 0; c < G; ++c) list.start[c + 1] = static_cast<uint16_t>(list.start[c] + count[c]);
  std::vector<int> fill(list.start, list.start + G);
  for (int u = 0; u < n; ++u) list.unit[fill[owner[u]]++] = static_cast<uint16_t>(u);
  std::copy(k, k + 8, key);
  return &list;
}

static int attn_common(bool fp8, int lean, const void* q, const float* qsc, const void* k, const float* ksc, const void* v,
                       const float* vsc, void* o, int B, int S, int Hq, int Hkv, int Dqk, int Dv,
                       float softmax_scale, const int64_t qs[3], const int64_t ks[3], const int64_t vs[3],
                       const int64_t os[3], int row_begin, int row_end, void* stream, void* workspace = nullptr,
                       size_t workspace_bytes = 0) {
  AttnCommon c{B, S, Hq, Hkv, Dqk, Dv, softmax_scale};
  const int elt = fp8 ? 1 : 2;
  if (int r = validate_attn(c, q, k, v, o, 16 / elt, qs, ks, vs, os)) return r;
  if (row_begin < 0 || row_end > S || row_begin >= row_end || row_begin % 256 != 0 ||
      (row_end % 256 != 0 && row_end != S))
    return fail(ZYFA_ERR_INVALID_ARG,
                "rows [%d, %d) must lie in [0, %d) with both ends multiples of 256 (or the end = S)", row_begin,
                row_end, S);
  if (fp8) {
    if (!qsc || !ksc || !vsc) return fail(ZYFA_ERR_INVALID_ARG, "null scale pointer");
    if (!aligned(qsc, 4) || !aligned(ksc, 4) || !aligned(vsc, 4))
      return fail(ZYFA_ERR_INVALID_ARG, "scale pointers must be 4-byte aligned");
  }
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  int r;
  if ((r = make_map(&tq, q, dt, elt, Dqk, Hq, S, B, qs, "q")) || (r = make_map(&tk, k, dt, elt, Dqk, Hkv, S, B, ks, "k")) ||
      (r = make_map(&tv, v, dt, elt, Dv, Hkv, S, B, vs, "v")))
    return r;
  zyfa::AttnArgs a{};
  a.B = B; a.S = S; a.Hq = Hq; a.Hkv = Hkv; a.Dqk = Dqk; a.Dv = Dv;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.o = o; a.o_sb = os[0]; a.o_ss = os[1]; a.o_sh = os[2];
  a.q_scale = qsc; a.k_scale = ksc; a.v_scale = vsc;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns;
  a.debug_stall = g_debug_stall;
  a.num_sms = d->sm_count;
  a.scale_blocks = (S + 127) / 128;
  a.lean_p = lean;
  a.pair_lo = row_begin / 256;
  a.pair_hi = (row_end + 255) / 256;
  a.groups_in_flight = groups_in_flight(S, Dqk, Dv, elt);
  long long split_units = 0;
  const int split = (workspace && row_begin == 0 && row_end == S)
                        ? prefill_split_tiles(B, S, Hq, d->sm_count, &split_units) : 0;
  if (split) {
    if (!aligned(workspace, 256)) return fail(ZYFA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < prefill_ws_bytes(B, S, Hq))
      return fail(ZYFA_ERR_INVALID_ARG, "workspace of %zu bytes is below zyfa_attn_workspace_bytes = %zu",
                  workspace_bytes, prefill_ws_bytes(B, S, Hq));
    const size_t rows = prefill_partial_rows(B, S, Hq);
    a.split_tiles = split;
    a.part_o = static_cast<float*>(workspace);
    a.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows * 128 * 4 + 255) & ~size_t(255)));
    cudaError_t e = fp8 ? zyfa::launch_attn_fp8_split(tq, tk, tv, a, split_units, static_cast<cudaStream_t>(stream))
                        : zyfa::launch_attn_bf16_split(tq, tk, tv, a, split_units, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, fp8 ? "attn_fwd_fp8 launch" : "attn_fwd_bf16 launch");
    e = zyfa::launch_prefill_combine(a, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "prefill_combine launch");
    return ZYFA_OK;
  }
  const zyfa::UnitList* list = unit_list(a);
  cudaError_t e = fp8 ? zyfa::launch_attn_fp8(tq, tk, tv, a, static_cast<cudaStream_t>(stream), list)
                      : zyfa::launch_attn_bf16(tq, tk, tv, a, static_cast<cudaStream_t>(stream), list);
  if (e != cudaSuccess) return fail_cuda(e, fp8 ? "attn_fwd_fp8 launch" : "attn_fwd_bf16 launch");
  return ZYFA_OK;
}

size_t zyfa_attn_workspace_bytes(int B, int S, int Hq) { return prefill_ws_bytes(B, S, Hq); }

int zyfa_attn_split_tiles(int B, int S, int Hq) {
  if (B < 1 || S < 1 || Hq < 1) return -fail(ZYFA_ERR_INVALID_ARG, "B, S and Hq must be >= 1");
  DeviceInfo* d;
  if (int r = device_info(&d)) return -r;
  long long units;
  return prefill_split_tiles(B, S, Hq, d->sm_count, &units);
}

int zyfa_attn_fwd_bf16_ws(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                          int Dqk, int Dv, float softmax_scale, const int64_t q_strides[3],
                          const int64_t k_strides[3], const int64_t v_strides[3], const int64_t o_strides[3],
                          void* workspace, size_t workspace_bytes, void* stream) {
  return attn_common(false, 0, q, nullptr, k, nullptr, v, nullptr, o, B, S, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides,
                     k_strides, v_strides, o_strides, 0, S, stream, workspace, workspace_bytes);
}

int zyfa_attn_fwd_fp8_ws(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                         const void* v8, const float* v_scale, void* o, int B, int S, int Hq, int Hkv, int Dqk,
                         int Dv, float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                         const int64_t v_strides[3], const int64_t o_strides[3], int flags, void* workspace,
                         size_t workspace_bytes, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_common(true, lean, q8, q_scale, k8, k_scale, v8, v_scale, o, B, S, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, 0, S, stream, workspace, workspace_bytes);
}

int zyfa_attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv, int Dqk,
                       int Dv, float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                       const int64_t v_strides[3], const int64_t o_strides[3], void* stream) {
  return attn_common(false, 0, q, nullptr, k, nullptr, v, nullptr, o, B, S, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides,
                     k_strides, v_strides, o_strides, 0, S, stream);
}

int zyfa_attn_fwd_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale, const void* v8,
                      const float* v_scale, void* o, int B, int S, int Hq, int Hkv, int Dqk, int Dv,
                      float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                      const int64_t v_strides[3], const int64_t o_strides[3], int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_common(true, lean, q8, q_scale, k8, k_scale, v8, v_scale, o, B, S, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, 0, S, stream);
}

int zyfa_attn_fwd_bf16_rows(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                            int Dqk, int Dv, float softmax_scale, const int64_t q_strides[3],
                            const int64_t k_strides[3], const int64_t v_strides[3], const int64_t o_strides[3],
                            int row_begin, int row_end, void* stream) {
  return attn_common(false, 0, q, nullptr, k, nullptr, v, nullptr, o, B, S, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides,
                     k_strides, v_strides, o_strides, row_begin, row_end, stream);
}

int zyfa_attn_fwd_fp8_rows(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                           const void* v8, const float* v_scale, void* o, int B, int S, int Hq, int Hkv, int Dqk,
                           int Dv, float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                           const int64_t v_strides[3], const int64_t o_strides[3], int row_begin, int row_end,
                           int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_common(true, lean, q8, q_scale, k8, k_scale, v8, v_scale, o, B, S, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, row_begin, row_end, stream);
}

// ----------------------------------------------------- packed varlen batches
// Host cu_seqlens: B + 1 nondecreasing offsets starting at 0.
static int read_seqlens(const int32_t* cu, int B, int* total, int* max_len) {
  if (!cu) return fail(ZYFA_ERR_INVALID_ARG, "cu_seqlens is null");
  if (B < 1 || B > zyfa::kMaxVarlenSeqs)
    return fail(ZYFA_ERR_INVALID_ARG, "batch %d outside 1..%d", B, zyfa::kMaxVarlenSeqs);
  if (cu[0] != 0) return fail(ZYFA_ERR_INVALID_ARG, "cu_seqlens[0] must be 0");
  int mx = 0;
  for (int i = 0; i < B; ++i) {
    if (cu[i + 1] < cu[i]) return fail(ZYFA_ERR_INVALID_ARG, "cu_seqlens must be nondecreasing (at %d)", i);
    mx = std::max(mx, cu[i + 1] - cu[i]);
  }
  if (mx > 2 * 128 * zyfa::kMaxVarlenLevels)
    return fail(ZYFA_ERR_UNSUPPORTED, "sequence of %d tokens exceeds %d", mx, 2 * 128 * zyfa::kMaxVarlenLevels);
  *total = cu[B];
  *max_len = mx;
  return ZYFA_OK;
}

// Device-resident offsets: the caller states the packed token count and an
// upper bound on the sequence length; the tables are built on the device into
// the caller's workspace ([SeqTable][QuantSeqTable], 256-byte aligned).
static size_t varlen_ws_quant_offset() { return (sizeof(zyfa::SeqTable) + 255) & ~size_t(255); }
static size_t varlen_ws_bytes() { return varlen_ws_quant_offset() + ((sizeof(zyfa::QuantSeqTable) + 255) & ~size_t(255)); }

static int check_dev_seqlens(const int32_t* cu, int B, int total, int max_len, void* workspace) {
  if (!cu) return fail(ZYFA_ERR_INVALID_ARG, "cu_seqlens is null");
  if (B < 1 || B > zyfa::kMaxVarlenSeqs)
    return fail(ZYFA_ERR_INVALID_ARG, "batch %d outside 1..%d", B, zyfa::kMaxVarlenSeqs);
  if (total < 0) return fail(ZYFA_ERR_INVALID_ARG, "total_tokens must be >= 0");
  if (max_len < 0) return fail(ZYFA_ERR_INVALID_ARG, "max_seqlen must be >= 0");
  if (max_len > 2 * 128 * zyfa::kMaxVarlenLevels)
    return fail(ZYFA_ERR_UNSUPPORTED, "max_seqlen %d exceeds %d", max_len, 2 * 128 * zyfa::kMaxVarlenLevels);
  if (!workspace || !aligned(workspace, 256)) return fail(ZYFA_ERR_INVALID_ARG, "workspace must be non-null and 256-byte aligned");
  if (!aligned(cu, 4)) return fail(ZYFA_ERR_INVALID_ARG, "cu_seqlens must be 4-byte aligned");
  return ZYFA_OK;
}

// Unit table of a packed batch: non-empty sequences, longest first (ties in
// batch order); level k holds pair t = n_levels - 1 - k of every sequence
// with more than t pairs. ctx (paged K/V) gives each sequence's cached
// tokens, else none.
static void build_seq_table(const int32_t* cu, const int32_t* ctx, int B, int max_len, int Hq,
                            zyfa::SeqTable* tab) {
  std::vector<int> order;
  for (int i = 0; i < B; ++i)
    if (cu[i + 1] > cu[i]) order.push_back(i);
  std::stable_sort(order.begin(), order.end(),
                   [&](int x, int y) { return (cu[x + 1] - cu[x]) > (cu[y + 1] - cu[y]); });
  tab->n_seqs = static_cast<int>(order.size());
  for (int i = 0; i < tab->n_seqs; ++i) {
    tab->start[i] = cu[order[i]];
    tab->len[i] = cu[order[i] + 1] - cu[order[i]];
    tab->index[i] = order[i];
    tab->ctx[i] = ctx ? ctx[order[i]] : 0;
  }
  auto pairs = [](int len) { return ((len + 127) / 128 + 1) / 2; };
  tab->n_levels = pairs(max_len);
  // cnt[t]: sequences with more than t pairs (a prefix of the sorted order)
  std::vector<int> cnt(tab->n_levels);
  int with = tab->n_seqs;
  for (int t = 0; t < tab->n_levels; ++t) {
    while (with > 0 && pairs(tab->len[with - 1]) <= t) --with;
    cnt[t] = with;
  }
  tab->level_start[0] = 0;
  for (int kl = 0; kl < tab->n_levels; ++kl)
    tab->level_start[kl + 1] = tab->level_start[kl] + cnt[tab->n_levels - 1 - kl] * Hq;
}

static int attn_varlen(bool fp8, int lean, const void* q, const float* qsc, const void* k, const float* ksc, const void* v,
                       const float* vsc, void* o, const int32_t* cu, int B, int Hq, int Hkv, int Dqk, int Dv,
                       float softmax_scale, const int64_t qs[2], const int64_t ks[2], const int64_t vs[2],
                       const int64_t os[2], void* stream, const int32_t* cu_dev = nullptr, int total_dev = 0,
                       int max_len_dev = 0, void* workspace = nullptr) {
  int T = 0, max_len = 0;
  if (cu_dev) {
    if (int r = check_dev_seqlens(cu_dev, B, total_dev, max_len_dev, workspace)) return r;
    T = total_dev;
    max_len = max_len_dev;
  } else if (int r = read_seqlens(cu, B, &T, &max_len)) {
    return r;
  }
  if (!qs || !ks || !vs || !os) return fail(ZYFA_ERR_INVALID_ARG, "strides pointer is null");
  if (T == 0) return ZYFA_OK;   // nothing to compute
  // The packed tensors as one batch of T tokens.
  const int64_t q3[3] = {qs[0] * T, qs[0], qs[1]}, k3[3] = {ks[0] * T, ks[0], ks[1]};
  const int64_t v3[3] = {vs[0] * T, vs[0], vs[1]}, o3[3] = {os[0] * T, os[0], os[1]};
  AttnCommon c{1, T, Hq, Hkv, Dqk, Dv, softmax_scale};
  const int elt = fp8 ? 1 : 2;
  if (int r = validate_attn(c, q, k, v, o, 16 / elt, q3, k3, v3, o3)) return r;
  if (fp8) {
    if (!qsc || !ksc || !vsc) return fail(ZYFA_ERR_INVALID_ARG, "null scale pointer");
    if (!aligned(qsc, 4) || !aligned(ksc, 4) || !aligned(vsc, 4))
      return fail(ZYFA_ERR_INVALID_ARG, "scale pointers must be 4-byte aligned");
  }
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  int r;
  if ((r = make_map(&tq, q, dt, elt, Dqk, Hq, T, 1, q3, "q")) || (r = make_map(&tk, k, dt, elt, Dqk, Hkv, T, 1, k3, "k")) ||
      (r = make_map(&tv, v, dt, elt, Dv, Hkv, T, 1, v3, "v")))
    return r;
  zyfa::AttnArgs a{};
  a.B = 1; a.S = T; a.Hq = Hq; a.Hkv = Hkv; a.Dqk = Dqk; a.Dv = Dv;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.o = o; a.o_sb = o3[0]; a.o_ss = o3[1]; a.o_sh = o3[2];
  a.q_scale = qsc; a.k_scale = ksc; a.v_scale = vsc;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns;
  a.debug_stall = g_debug_stall;
  a.num_sms = d->sm_count;
  a.scale_blocks = (max_len + 127) / 128;
  a.lean_p = lean;
  if (cu_dev) {
    auto* dtab = static_cast<zyfa::SeqTable*>(workspace);
    cudaError_t e = zyfa::launch_build_seq_tables(cu_dev, B, T, max_len, Hq, dtab, nullptr, d->status,
                                                  static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "build_seq_tables launch");
    e = fp8 ? zyfa::launch_attn_fp8_varlen_dev(tq, tk, tv, a, dtab, static_cast<cudaStream_t>(stream))
            : zyfa::launch_attn_bf16_varlen_dev(tq, tk, tv, a, dtab, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, fp8 ? "attn_fwd_fp8_varlen launch" : "attn_fwd_bf16_varlen launch");
    return ZYFA_OK;
  }
  static thread_local zyfa::SeqTable tab;
  build_seq_table(cu, nullptr, B, max_len, Hq, &tab);
  cudaError_t e = fp8 ? zyfa::launch_attn_fp8_varlen(tq, tk, tv, a, tab, static_cast<cudaStream_t>(stream))
                      : zyfa::launch_attn_bf16_varlen(tq, tk, tv, a, tab, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, fp8 ? "attn_fwd_fp8_varlen launch" : "attn_fwd_bf16_varlen launch");
  return ZYFA_OK;
}

int zyfa_attn_fwd_bf16_varlen(const void* q, const void* k, const void* v, void* o, const int32_t* cu_seqlens, int B,
                              int Hq, int Hkv, int Dqk, int Dv, float softmax_scale, const int64_t q_strides[2],
                              const int64_t k_strides[2], const int64_t v_strides[2], const int64_t o_strides[2],
                              void* stream) {
  return attn_varlen(false, 0, q, nullptr, k, nullptr, v, nullptr, o, cu_seqlens, B, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, stream);
}

int zyfa_attn_fwd_fp8_varlen(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                             const void* v8, const float* v_scale, void* o, const int32_t* cu_seqlens, int B, int Hq,
                             int Hkv, int Dqk, int Dv, float softmax_scale, const int64_t q_strides[2],
                             const int64_t k_strides[2], const int64_t v_strides[2], const int64_t o_strides[2],
                             int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_varlen(true, lean, q8, q_scale, k8, k_scale, v8, v_scale, o, cu_seqlens, B, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, stream);
}

// Packed queries over a paged K/V cache (chunked prefill, prefix caching).
static int attn_paged(bool fp8, int lean, const void* q, const float* qsc, const void* kc, const float* ksc, const void* vc,
                      const float* vsc, void* o, const int32_t* cu, const int32_t* ctx_lens,
                      const int32_t* block_table, int64_t bt_stride, int num_pages, int B, int Hq, int Hkv, int Dqk,
                      int Dv, float softmax_scale, const int64_t qs[2], const int64_t kcs[3], const int64_t vcs[3],
                      const int64_t os[2], void* stream) {
  int T = 0, max_len = 0;
  if (int r = read_seqlens(cu, B, &T, &max_len)) return r;
  if (!ctx_lens) return fail(ZYFA_ERR_INVALID_ARG, "ctx_lens is null");
  if (!block_table || !aligned(block_table, 4)) return fail(ZYFA_ERR_INVALID_ARG, "block_table must be non-null and 4-byte aligned");
  if (num_pages < 1) return fail(ZYFA_ERR_INVALID_ARG, "num_pages must be >= 1");
  if (bt_stride < 1) return fail(ZYFA_ERR_INVALID_ARG, "block_table row stride must be >= 1");
  for (int i = 0; i < B; ++i) {
    const int32_t c = ctx_lens[i];
    if (c < 0) return fail(ZYFA_ERR_INVALID_ARG, "ctx_lens[%d] = %d must be non-negative", i, c);
    const int64_t blocks = (static_cast<int64_t>(c) + (cu[i + 1] - cu[i]) + 127) / 128;
    if (blocks > (1 << 23)) return fail(ZYFA_ERR_UNSUPPORTED, "sequence %d is too long", i);
    if (cu[i + 1] > cu[i] && blocks > bt_stride)
      return fail(ZYFA_ERR_INVALID_ARG, "sequence %d needs %lld pages, more than the block_table row stride %lld", i,
                  (long long)blocks, (long long)bt_stride);
  }
  if (!qs || !kcs || !vcs || !os) return fail(ZYFA_ERR_INVALID_ARG, "strides pointer is null");
  if (T == 0) return ZYFA_OK;   // nothing to compute
  const int64_t q3[3] = {qs[0] * T, qs[0], qs[1]}, o3[3] = {os[0] * T, os[0], os[1]};
  AttnCommon c{1, T, Hq, Hkv, Dqk, Dv, softmax_scale};
  const int elt = fp8 ? 1 : 2;
  // the caches pass the same checks as packed K/V (their strides separately)
  if (int r = validate_attn(c, q, kc, vc, o, 16 / elt, q3, q3, q3, o3)) return r;
  if (int r = check_strides(kcs, 16 / elt, "k_cache")) return r;
  if (int r = check_strides(vcs, 16 / elt, "v_cache")) return r;
  if (fp8) {
    if (!qsc || !ksc || !vsc) return fail(ZYFA_ERR_INVALID_ARG, "null scale pointer");
    if (!aligned(qsc, 4) || !aligned(ksc, 4) || !aligned(vsc, 4))
      return fail(ZYFA_ERR_INVALID_ARG, "scale pointers must be 4-byte aligned");
  }
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  int r;
  if ((r = make_map(&tq, q, dt, elt, Dqk, Hq, T, 1, q3, "q")) ||
      (r = make_map(&tk, kc, dt, elt, Dqk, Hkv, 128, num_pages, kcs, "k_cache")) ||
      (r = make_map(&tv, vc, dt, elt, Dv, Hkv, 128, num_pages, vcs, "v_cache")))
    return r;
  zyfa::AttnArgs a{};
  a.B = 1; a.S = T; a.Hq = Hq; a.Hkv = Hkv; a.Dqk = Dqk; a.Dv = Dv;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.o = o; a.o_sb = o3[0]; a.o_ss = o3[1]; a.o_sh = o3[2];
  a.q_scale = qsc; a.k_scale = ksc; a.v_scale = vsc;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns;
  a.debug_stall = g_debug_stall;
  a.num_sms = d->sm_count;
  a.scale_blocks = (max_len + 127) / 128;
  a.lean_p = lean;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.num_pages = num_pages;
  static thread_local zyfa::SeqTable tab;
  build_seq_table(cu, ctx_lens, B, max_len, Hq, &tab);
  cudaError_t e = fp8 ? zyfa::launch_attn_fp8_varlen(tq, tk, tv, a, tab, static_cast<cudaStream_t>(stream))
                      : zyfa::launch_attn_bf16_varlen(tq, tk, tv, a, tab, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, fp8 ? "attn_fwd_fp8_paged launch" : "attn_fwd_bf16_paged launch");
  return ZYFA_OK;
}

int zyfa_attn_fwd_bf16_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                             const int32_t* cu_seqlens_q, const int32_t* ctx_lens, const int32_t* block_table,
                             int64_t block_table_stride, int num_pages, int B, int Hq, int Hkv, int Dqk, int Dv,
                             float softmax_scale, const int64_t q_strides[2], const int64_t k_cache_strides[3],
                             const int64_t v_cache_strides[3], const int64_t o_strides[2], void* stream) {
  return attn_paged(false, 0, q, nullptr, k_cache, nullptr, v_cache, nullptr, o, cu_seqlens_q, ctx_lens, block_table,
                    block_table_stride, num_pages, B, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides, k_cache_strides,
                    v_cache_strides, o_strides, stream);
}

int zyfa_attn_fwd_fp8_paged(const void* q8, const float* q_scale, const void* k_cache8, const float* k_scale,
                            const void* v_cache8, const float* v_scale, void* o, const int32_t* cu_seqlens_q,
                            const int32_t* ctx_lens, const int32_t* block_table, int64_t block_table_stride,
                            int num_pages, int B, int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                            const int64_t q_strides[2], const int64_t k_cache_strides[3],
                            const int64_t v_cache_strides[3], const int64_t o_strides[2], int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_paged(true, lean, q8, q_scale, k_cache8, k_scale, v_cache8, v_scale, o, cu_seqlens_q, ctx_lens, block_table,
                    block_table_stride, num_pages, B, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides, k_cache_strides,
                    v_cache_strides, o_strides, stream);
}

// Decode step: key ranges are split only while there are fewer than
// kSplitTasksPerSm (sequence, KV head) tasks per SM, into splits of at least
// kMinSplitTiles / 2 key blocks; the workspace holds the partial rows of up
// to kSplitTasksPerSm tasks per SM on kMaxSmsForWorkspace SMs, plus one per
// sequence.
constexpr int kSplitTasksPerSm = 4;
constexpr int kMinSplitTiles = 8;
constexpr int kMaxSmsForWorkspace = 256;

// Query rows are replicated (four copies of every split) for groups of at
// most 32 query heads per KV head; larger groups keep one copy.
static int decode_copies(int Hq, int Hkv) { return Hkv >= 1 && Hq / Hkv <= 32 ? 4 : 1; }

static size_t decode_partial_rows_bound(int N, int Hq, int Hkv) {
  return decode_copies(Hq, Hkv) *
         (static_cast<size_t>(kSplitTasksPerSm) * kMaxSmsForWorkspace / std::max(Hkv, 1) + 1 + std::max(N, 0));
}

static size_t decode_ws_bytes(int N, int Hq, int Hkv) {
  // per partial row and head: 128 fp32 of O and (m, l)
  const size_t rows = decode_partial_rows_bound(N, Hq, Hkv) * static_cast<size_t>(std::max(Hq, 0));
  return ((rows * 128 * 4 + 255) & ~size_t(255)) + rows * 2 * 4;
}

// Decode step over a paged cache: one query token per sequence.
static int attn_decode(bool fp8, int lean, const void* q, const float* qsc, const void* kc, const float* ksc, const void* vc,
                       const float* vsc, void* o, const int32_t* seq_lens, const int32_t* block_table,
                       int64_t bt_stride, int num_pages, int N, int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                       const int64_t qs[2], const int64_t kcs[3], const int64_t vcs[3], const int64_t os[2],
                       void* workspace, size_t workspace_bytes, void* stream) {
  if (N < 1 || N > zyfa::kMaxVarlenSeqs)
    return fail(ZYFA_ERR_INVALID_ARG, "batch %d outside 1..%d", N, zyfa::kMaxVarlenSeqs);
  if (!seq_lens) return fail(ZYFA_ERR_INVALID_ARG, "seq_lens is null");
  if (!block_table || !aligned(block_table, 4)) return fail(ZYFA_ERR_INVALID_ARG, "block_table must be non-null and 4-byte aligned");
  if (num_pages < 1) return fail(ZYFA_ERR_INVALID_ARG, "num_pages must be >= 1");
  if (bt_stride < 1) return fail(ZYFA_ERR_INVALID_ARG, "block_table row stride must be >= 1");
  if (Hkv < 1 || Hq < 1 || Hq % Hkv != 0 || Hq / Hkv > 128)
    return fail(ZYFA_ERR_INVALID_ARG, "need Hq a multiple of Hkv with at most 128 query heads per KV head");
  int max_len = 0;
  for (int i = 0; i < N; ++i) {
    const int32_t L = seq_lens[i];
    if (L < 1) return fail(ZYFA_ERR_INVALID_ARG, "seq_lens[%d] = %d must be >= 1 (the new token included)", i, L);
    if ((static_cast<int64_t>(L) + 127) / 128 > bt_stride)
      return fail(ZYFA_ERR_INVALID_ARG, "sequence %d needs %lld pages, more than the block_table row stride %lld", i,
                  (long long)((static_cast<int64_t>(L) + 127) / 128), (long long)bt_stride);
    max_len = std::max(max_len, L);
  }
  if (!qs || !kcs || !vcs || !os) return fail(ZYFA_ERR_INVALID_ARG, "strides pointer is null");
  if (qs[0] != static_cast<int64_t>(Hq) * qs[1])
    return fail(ZYFA_ERR_INVALID_ARG, "q must hold each token's heads contiguously (token stride = Hq x head stride)");
  const int64_t rows = static_cast<int64_t>(N) * Hq;
  // q as one batch of N*Hq rows (batch, row, "head" strides; the unit batch and head dimensions span it all)
  const int64_t q3[3] = {qs[1] * rows, qs[1], qs[1] * rows}, o3[3] = {os[0] * N, os[0], os[1]};
  AttnCommon c{1, N, Hq, Hkv, Dqk, Dv, softmax_scale};
  const int elt = fp8 ? 1 : 2;
  if (int r = validate_attn(c, q, kc, vc, o, 16 / elt, q3, q3, q3, o3)) return r;
  if (int r = check_strides(kcs, 16 / elt, "k_cache")) return r;
  if (int r = check_strides(vcs, 16 / elt, "v_cache")) return r;
  if (fp8) {
    if (!qsc || !ksc || !vsc) return fail(ZYFA_ERR_INVALID_ARG, "null scale pointer");
    if (!aligned(qsc, 4) || !aligned(ksc, 4) || !aligned(vsc, 4))
      return fail(ZYFA_ERR_INVALID_ARG, "scale pointers must be 4-byte aligned");
  }
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  const CUtensorMapDataType dt = fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap tq, tk, tv;
  int r;
  // q as rows of (token, head): the group of a KV head is consecutive rows
  // from its first head; 32-row boxes when the rows are replicated.
  // Replicated rows need at least 16 (token, KV head) tasks to pay: with one
  // 32K-token sequence and 8 KV heads they ran 35.9 us (FP8) against 29.8
  // with full rows, while two sequences and more gain from them.
  const bool replicate = workspace != nullptr && Hq / Hkv <= 32 && static_cast<int64_t>(N) * Hkv >= 16;
  if ((r = make_map(&tq, q, dt, elt, Dqk, 1, static_cast<int>(rows), 1, q3, "q", replicate ? 32 : 128)) ||
      (r = make_map(&tk, kc, dt, elt, Dqk, Hkv, 128, num_pages, kcs, "k_cache")) ||
      (r = make_map(&tv, vc, dt, elt, Dv, Hkv, 128, num_pages, vcs, "v_cache")))
    return r;
  zyfa::AttnArgs a{};
  a.B = 1; a.S = N; a.Hq = Hq; a.Hkv = Hkv; a.Dqk = Dqk; a.Dv = Dv;
  a.scale_log2 = softmax_scale * 1.4426950408889634f;
  a.o = o; a.o_sb = o3[0]; a.o_ss = o3[1]; a.o_sh = o3[2];
  a.q_scale = qsc; a.k_scale = ksc; a.v_scale = vsc;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns;
  a.debug_stall = g_debug_stall;
  a.num_sms = d->sm_count;
  a.scale_blocks = 1;          // q_scale [N, Hq]: one per token and head
  a.lean_p = lean;
  a.block_table = block_table;
  a.bt_stride = bt_stride;
  a.num_pages = num_pages;
  a.one_token = 1;
  // Units: sequences by decreasing length (ties in batch order), KV heads adjacent.
  static thread_local zyfa::SeqTable tab;
  std::vector<int> order(N);
  for (int i = 0; i < N; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return seq_lens[x] > seq_lens[y]; });
  tab.n_seqs = N;
  tab.n_levels = 0;
  tab.level_start[0] = 0;
  for (int i = 0; i < N; ++i) {
    tab.start[i] = order[i];
    tab.len[i] = seq_lens[order[i]];
    tab.index[i] = order[i];
    tab.ctx[i] = 0;
  }
  (void)max_len;
  // Split key ranges when that shortens the schedule: CTA c runs units c,
  // c + num_sms, ... (a unit = two tasks of one sequence and split), so the
  // step takes about the largest sum of unit lengths over the CTAs. Each
  // candidate split length (key blocks) is scored that way, plus a start-up
  // cost per unit; splits of a sequence are nearly equal.
  static thread_local zyfa::CombineTable ct;
  int chunk = 0;
  if (workspace && static_cast<int64_t>(N) * Hkv < static_cast<int64_t>(kSplitTasksPerSm) * d->sm_count) {
    const int G = d->sm_count;
    auto makespan = [&](int c) {   // c = 0: no split
      std::vector<int64_t> load(G, 0);
      int64_t unit = 0;
      for (int k = 0; k < N; ++k) {
        const int n = (tab.len[k] + 127) / 128;
        const int S = c ? (n + c - 1) / c : 1;
        for (int sp = 0; sp < S; ++sp) {
          const int len = n / S + (sp < n % S ? 1 : 0);
          for (int h = 0; h < Hkv; h += 2) load[unit++ % G] += len + 2;
        }
      }
      return *std::max_element(load.begin(), load.end());
    };
    int64_t best = makespan(0);
    for (int c = kMinSplitTiles; c < 1 << 16; c *= 2) {
      bool any = false;
      size_t rows = 0;
      for (int k = 0; k < N; ++k) {
        const int n = (tab.len[k] + 127) / 128;
        any = any || n > c;
        rows += (n + c - 1) / c;
      }
      if (!any) break;
      if (decode_copies(Hq, Hkv) * rows > decode_partial_rows_bound(N, Hq, Hkv)) continue;   // beyond the workspace
      const int64_t m = makespan(c);
      if (m < best) { best = m; chunk = c; }
    }
  }
  if (chunk || replicate) {
    if (!aligned(workspace, 256)) return fail(ZYFA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    if (workspace_bytes < decode_ws_bytes(N, Hq, Hkv))
      return fail(ZYFA_ERR_INVALID_ARG, "workspace of %zu bytes is below zyfa_decode_workspace_bytes = %zu",
                  workspace_bytes, decode_ws_bytes(N, Hq, Hkv));
    const int copies = replicate ? 4 : 1;
    int rows = 0;
    for (int k = 0; k < N; ++k) {
      // splits of at least chunk/2 blocks each (one without a split)
      const int splits = chunk ? ((tab.len[k] + 127) / 128 + chunk - 1) / chunk : 1;
      tab.level_start[k] = rows * Hkv;
      tab.ctx[k] = rows;
      ct.base[tab.index[k]] = copies * rows;
      ct.count[tab.index[k]] = copies * splits;
      rows += splits;
    }
    tab.level_start[N] = rows * Hkv;
    if (static_cast<size_t>(copies) * rows > decode_partial_rows_bound(N, Hq, Hkv))
      return fail(ZYFA_ERR_UNSUPPORTED, "internal: %d partial rows exceed the workspace bound", copies * rows);
    a.split_tiles = 1;
    a.replicate = replicate ? 1 : 0;
    a.part_o = static_cast<float*>(workspace);
    const size_t rows_all = decode_partial_rows_bound(N, Hq, Hkv) * static_cast<size_t>(Hq);
    a.part_ml = reinterpret_cast<float*>(static_cast<char*>(workspace) + ((rows_all * 128 * 4 + 255) & ~size_t(255)));
  }
  cudaError_t e = fp8 ? zyfa::launch_attn_fp8_varlen(tq, tk, tv, a, tab, static_cast<cudaStream_t>(stream))
                      : zyfa::launch_attn_bf16_varlen(tq, tk, tv, a, tab, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, fp8 ? "attn_decode_fp8 launch" : "attn_decode_bf16 launch");
  if (a.split_tiles) {
    e = zyfa::launch_decode_combine(a, ct, N, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return fail_cuda(e, "decode_combine launch");
  }
  return ZYFA_OK;
}

size_t zyfa_decode_workspace_bytes(int N, int Hq, int Hkv) { return decode_ws_bytes(N, Hq, Hkv); }

int zyfa_attn_decode_bf16_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                                const int32_t* seq_lens, const int32_t* block_table, int64_t block_table_stride,
                                int num_pages, int N, int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                                const int64_t q_strides[2], const int64_t k_cache_strides[3],
                                const int64_t v_cache_strides[3], const int64_t o_strides[2], void* workspace,
                                size_t workspace_bytes, void* stream) {
  return attn_decode(false, 0, q, nullptr, k_cache, nullptr, v_cache, nullptr, o, seq_lens, block_table,
                     block_table_stride, num_pages, N, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides, k_cache_strides,
                     v_cache_strides, o_strides, workspace, workspace_bytes, stream);
}

int zyfa_attn_decode_fp8_paged(const void* q8, const float* q_scale, const void* k_cache8, const float* k_scale,
                               const void* v_cache8, const float* v_scale, void* o, const int32_t* seq_lens,
                               const int32_t* block_table, int64_t block_table_stride, int num_pages, int N, int Hq,
                               int Hkv, int Dqk, int Dv, float softmax_scale, const int64_t q_strides[2],
                               const int64_t k_cache_strides[3], const int64_t v_cache_strides[3],
                               const int64_t o_strides[2], void* workspace, size_t workspace_bytes, int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_decode(true, lean, q8, q_scale, k_cache8, k_scale, v_cache8, v_scale, o, seq_lens, block_table,
                     block_table_stride, num_pages, N, Hq, Hkv, Dqk, Dv, softmax_scale, q_strides, k_cache_strides,
                     v_cache_strides, o_strides, workspace, workspace_bytes, stream);
}

// Packed variable-length tensors [T,H_t,D_t] (token strides in in[t].ss,
// head strides in in[t].sh): one streaming launch for all of them. Offsets
// on the host (cu_seqlens) or on the device (cu_dev, with the packed token
// count, a bound on the sequence length and the workspace for the table).
static int quant_packed(const QuantIn* in_, int n, const int32_t* cu_seqlens, int B, void* stream,
                        const int32_t* cu_dev = nullptr, int total_dev = 0, int max_len_dev = 0,
                        void* workspace = nullptr) {
  int T = 0, max_len = 0;
  if (cu_dev) {
    if (int r = check_dev_seqlens(cu_dev, B, total_dev, max_len_dev, workspace)) return r;
    T = total_dev;
    max_len = max_len_dev;
  } else if (int r = read_seqlens(cu_seqlens, B, &T, &max_len)) {
    return r;
  }
  QuantIn in[3];
  int dmax = 128;
  for (int t = 0; t < n; ++t) {
    in[t] = in_[t];
    in[t].sb = in[t].ss * std::max(T, 1);
    if (int r = check_quant_in(in[t])) return r;
    if (!quant_tileable(in[t]))
      return fail(ZYFA_ERR_UNSUPPORTED,
                  "%s: packed input needs 16-byte aligned x/out and token/head strides that are multiples of 8 "
                  "elements", in[t].name);
    dmax = std::max(dmax, in[t].D);
  }
  if (T == 0) return ZYFA_OK;
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  zyfa::QuantMaps m{};
  zyfa::QuantStreamArgs a{};
  for (int t = 0; t < n; ++t)
    if (int r = quant_stream_tensor(in[t], 1, T, &m, &a, t)) return r;
  a.n = n;
  a.B = 1;
  a.S = T;
  a.blk_lo = 0;
  a.blk_hi = (T + 127) / 128;
  a.status = d->status;
  a.timeout_ns = g_timeout_ns;
  if (cu_dev) {
    auto* dtab = reinterpret_cast<zyfa::QuantSeqTable*>(static_cast<char*>(workspace) + varlen_ws_quant_offset());
    cudaError_t e = zyfa::launch_build_seq_tables(cu_dev, B, T, max_len, in[0].H, nullptr, dtab, d->status, st);
    if (e != cudaSuccess) return fail_cuda(e, "build_seq_tables launch");
    e = zyfa::launch_quantize_fp8_stream_varlen_dev(m, a, dmax, dtab, d->sm_count, st);
    if (e != cudaSuccess) return fail_cuda(e, "quantize_fp8_varlen launch");
    return ZYFA_OK;
  }
  static thread_local zyfa::QuantSeqTable tab;
  tab.n_seqs = B;
  tab.max_blocks = (max_len + 127) / 128;
  tab.cum_blocks[0] = 0;
  for (int i = 0; i < B; ++i) {
    tab.start[i] = cu_seqlens[i];
    tab.len[i] = cu_seqlens[i + 1] - cu_seqlens[i];
    tab.cum_blocks[i + 1] = tab.cum_blocks[i] + (tab.len[i] + 127) / 128;
  }
  cudaError_t e = zyfa::launch_quantize_fp8_stream_varlen(m, a, dmax, tab, d->sm_count, st);
  if (e != cudaSuccess) return fail_cuda(e, "quantize_fp8_varlen launch");
  return ZYFA_OK;
}

static int quant_varlen(const void* x, int64_t stride_t, int64_t stride_h, void* out, float* scales,
                        const int32_t* cu_seqlens, int B, int H, int D, int hadamard, void* stream,
                        const int32_t* cu_dev = nullptr, int total_dev = 0, int max_len_dev = 0,
                        void* workspace = nullptr) {
  const QuantIn t{x, 0, stride_t, stride_h, out, scales, H, D, hadamard, "x"};
  return quant_packed(&t, 1, cu_seqlens, B, stream, cu_dev, total_dev, max_len_dev, workspace);
}

static int quant_qkv_packed(const void* q, const int64_t qs[2], const void* k, const int64_t ks[2], const void* v,
                            const int64_t vs[2], void* q8, float* q_scale, void* k8, float* k_scale, void* v8,
                            float* v_scale, const int32_t* cu_seqlens, int B, int Hq, int Hkv, int Dqk, int Dv,
                            int hadamard, void* stream, const int32_t* cu_dev = nullptr, int total_dev = 0,
                            int max_len_dev = 0, void* workspace = nullptr) {
  if (!qs || !ks || !vs) return fail(ZYFA_ERR_INVALID_ARG, "null strides pointer");
  if (!((Dqk == 128 || Dqk == 192) && Dv == 128))
    return fail(ZYFA_ERR_UNSUPPORTED, "head dims (%d, %d) unsupported; use (128, 128) or (192, 128)", Dqk, Dv);
  const QuantIn in[3] = {{q, 0, qs[0], qs[1], q8, q_scale, Hq, Dqk, hadamard, "q"},
                         {k, 0, ks[0], ks[1], k8, k_scale, Hkv, Dqk, hadamard, "k"},
                         {v, 0, vs[0], vs[1], v8, v_scale, Hkv, Dv, 0, "v"}};
  return quant_packed(in, 3, cu_seqlens, B, stream, cu_dev, total_dev, max_len_dev, workspace);
}

int zyfa_quantize_fp8_varlen(const void* x, int64_t stride_t, int64_t stride_h, void* out, float* scales,
                             const int32_t* cu_seqlens, int B, int H, int D, int hadamard, void* stream) {
  return quant_varlen(x, stride_t, stride_h, out, scales, cu_seqlens, B, H, D, hadamard, stream);
}

size_t zyfa_varlen_workspace_bytes(void) { return varlen_ws_bytes(); }

int zyfa_quantize_fp8_varlen_dev(const void* x, int64_t stride_t, int64_t stride_h, void* out, float* scales,
                                 const int32_t* cu_seqlens_dev, int B, int total_tokens, int max_seqlen, int H, int D,
                                 int hadamard, void* workspace, void* stream) {
  return quant_varlen(x, stride_t, stride_h, out, scales, nullptr, B, H, D, hadamard, stream, cu_seqlens_dev,
                      total_tokens, max_seqlen, workspace);
}

int zyfa_quantize_fp8_qkv_varlen(const void* q, const int64_t q_strides[2], const void* k,
                                 const int64_t k_strides[2], const void* v, const int64_t v_strides[2], void* q8,
                                 float* q_scale, void* k8, float* k_scale, void* v8, float* v_scale,
                                 const int32_t* cu_seqlens, int B, int Hq, int Hkv, int Dqk, int Dv, int hadamard,
                                 void* stream) {
  return quant_qkv_packed(q, q_strides, k, k_strides, v, v_strides, q8, q_scale, k8, k_scale, v8, v_scale,
                          cu_seqlens, B, Hq, Hkv, Dqk, Dv, hadamard, stream);
}

int zyfa_quantize_fp8_qkv_varlen_dev(const void* q, const int64_t q_strides[2], const void* k,
                                     const int64_t k_strides[2], const void* v, const int64_t v_strides[2], void* q8,
                                     float* q_scale, void* k8, float* k_scale, void* v8, float* v_scale,
                                     const int32_t* cu_seqlens_dev, int B, int total_tokens, int max_seqlen, int Hq,
                                     int Hkv, int Dqk, int Dv, int hadamard, void* workspace, void* stream) {
  return quant_qkv_packed(q, q_strides, k, k_strides, v, v_strides, q8, q_scale, k8, k_scale, v8, v_scale, nullptr,
                          B, Hq, Hkv, Dqk, Dv, hadamard, stream, cu_seqlens_dev, total_tokens, max_seqlen,
                          workspace);
}

int zyfa_attn_fwd_bf16_varlen_dev(const void* q, const void* k, const void* v, void* o, const int32_t* cu_seqlens_dev,
                                  int B, int total_tokens, int max_seqlen, int Hq, int Hkv, int Dqk, int Dv,
                                  float softmax_scale, const int64_t q_strides[2], const int64_t k_strides[2],
                                  const int64_t v_strides[2], const int64_t o_strides[2], void* workspace,
                                  void* stream) {
  return attn_varlen(false, 0, q, nullptr, k, nullptr, v, nullptr, o, nullptr, B, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, stream, cu_seqlens_dev, total_tokens, max_seqlen,
                     workspace);
}

int zyfa_attn_fwd_fp8_varlen_dev(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                                 const void* v8, const float* v_scale, void* o, const int32_t* cu_seqlens_dev, int B,
                                 int total_tokens, int max_seqlen, int Hq, int Hkv, int Dqk, int Dv,
                                 float softmax_scale, const int64_t q_strides[2], const int64_t k_strides[2],
                                 const int64_t v_strides[2], const int64_t o_strides[2], void* workspace,
                                 int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  return attn_varlen(true, lean, q8, q_scale, k8, k_scale, v8, v_scale, o, nullptr, B, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, stream, cu_seqlens_dev, total_tokens, max_seqlen,
                     workspace);
}

// ----------------------------- packed FP8 attention without a workspace
// For callers that cannot allocate device memory on the call path: a step
// replayed inside a CUDA graph whose memory was fixed at capture, a serving
// loop that hands out memory only from its own pool, or a process that runs
// with the allocator locked. zyfa_attn_fwd_fp8_varlen_dev needs a caller
// workspace for the unit table its first kernel builds; this form keeps that
// table in one array of this file instead. The array holds one table for up
// to kMaxVarlenSeqs sequences of up to 2 * 128 * kMaxVarlenLevels tokens
// (check_dev_seqlens rejects anything larger), stays resident on every device
// that loads the library until the process exits, and is shared by all calls:
// each call rewrites every field the attention kernel reads, and calls whose
// kernels overlap on the GPU race on it.
namespace {
constexpr size_t kNoAllocScratchBytes = 32768;
static_assert(sizeof(zyfa::SeqTable) <= kNoAllocScratchBytes, "the unit table must fit the static scratch");
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device (the host-side
// symbol is only a stand-in). Looked up once per device, with that device
// current, on the first call there.
int noalloc_scratch(void** out) {
  static std::mutex mu;
  static void* addr[64] = {};
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= 64) return fail(ZYFA_ERR_UNSUPPORTED, "device ordinal %d outside 0..63", dev);
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return fail_cuda(e, "cudaGetSymbolAddress(static scratch)");
    addr[dev] = p;
  }
  *out = addr[dev];
  return ZYFA_OK;
}
}  // namespace

size_t zyfa_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

int zyfa_attn_fwd_fp8_varlen_dev_noalloc(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                                         const void* v8, const float* v_scale, void* o,
                                         const int32_t* cu_seqlens_dev, int B, int total_tokens, int max_seqlen,
                                         int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                                         const int64_t q_strides[2], const int64_t k_strides[2],
                                         const int64_t v_strides[2], const int64_t o_strides[2], int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  // The static table bounds the batch: refuse what it cannot hold before
  // touching the device.
  if (B < 1 || B > zyfa::kMaxVarlenSeqs)
    return fail(ZYFA_ERR_INVALID_ARG, "batch %d outside 1..%d (the static scratch holds one table of at most %d sequences)",
                B, zyfa::kMaxVarlenSeqs, zyfa::kMaxVarlenSeqs);
  if (max_seqlen > 2 * 128 * zyfa::kMaxVarlenLevels)
    return fail(ZYFA_ERR_UNSUPPORTED, "max_seqlen %d exceeds %d (the static scratch holds one table of sequences up to that length)",
                max_seqlen, 2 * 128 * zyfa::kMaxVarlenLevels);
  void* scratch = nullptr;
  if (int r = noalloc_scratch(&scratch)) return r;
  return attn_varlen(true, lean, q8, q_scale, k8, k_scale, v8, v_scale, o, nullptr, B, Hq, Hkv, Dqk, Dv, softmax_scale,
                     q_strides, k_strides, v_strides, o_strides, stream, cu_seqlens_dev, total_tokens, max_seqlen,
                     scratch);
}

// ------------------------------------------------ prefill from host memory
// Per-device copy streams and per-chunk events of the host pipeline.
namespace {
constexpr int kMaxChunks = 64;
constexpr int kAttnStreams = 2;
struct HostPipe {
  bool ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, att[kAttnStreams] = {};
  cudaEvent_t start = nullptr, end = nullptr;
  cudaEvent_t in[kMaxChunks] = {}, quant[kMaxChunks] = {}, done[kMaxChunks] = {};
  std::mutex mu;
};
HostPipe g_pipe[kMaxDevices];

int host_pipe(HostPipe** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail_cuda(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(ZYFA_ERR_UNSUPPORTED, "device index %d out of range", dev);
  HostPipe& p = g_pipe[dev];
  std::lock_guard<std::mutex> lock(g_mu);
  if (!p.ready) {
    const unsigned int ef = cudaEventDisableTiming;
    if ((e = cudaStreamCreateWithFlags(&p.h2d, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaStreamCreateWithFlags(&p.d2h, cudaStreamNonBlocking)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&p.start, ef)) != cudaSuccess ||
        (e = cudaEventCreateWithFlags(&p.end, ef)) != cudaSuccess)
      return fail_cuda(e, "host pipeline streams");
    for (int i = 0; i < kAttnStreams; ++i)
      if ((e = cudaStreamCreateWithFlags(&p.att[i], cudaStreamNonBlocking)) != cudaSuccess)
        return fail_cuda(e, "host pipeline streams");
    for (int i = 0; i < kMaxChunks; ++i)
      if ((e = cudaEventCreateWithFlags(&p.in[i], ef)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&p.quant[i], ef)) != cudaSuccess ||
          (e = cudaEventCreateWithFlags(&p.done[i], ef)) != cudaSuccess)
        return fail_cuda(e, "host pipeline events");
    p.ready = true;
  }
  *out = &p;
  return ZYFA_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace carve-up: bf16 staging of Q, K, V; their e4m3 codes and block
// scales; the bf16 output before it goes back to the host.
struct HostWorkspace {
  size_t qd, kd, vd, q8, k8, v8, qs, ks, vs, od, total;
};
HostWorkspace host_workspace(int B, int S, int Hq, int Hkv, int Dqk, int Dv) {
  const size_t tq = size_t(B) * S * Hq * Dqk, tk = size_t(B) * S * Hkv * Dqk, tv = size_t(B) * S * Hkv * Dv;
  const size_t nb = size_t((S + 127) / 128);
  HostWorkspace w;
  size_t off = 0;
  auto take = [&](size_t bytes) { const size_t o = off; off += round256(bytes); return o; };
  w.qd = take(tq * 2);
  w.kd = take(tk * 2);
  w.vd = take(tv * 2);
  w.q8 = take(tq);
  w.k8 = take(tk);
  w.v8 = take(tv);
  w.qs = take(size_t(B) * Hq * nb * 4);
  w.ks = take(size_t(B) * Hkv * nb * 4);
  w.vs = take(size_t(B) * Hkv * nb * 4);
  w.od = take(size_t(B) * S * Hq * Dv * 2);
  w.total = off;
  return w;
}

bool page_locked(const void* p) {
  cudaPointerAttributes at{};
  if (cudaPointerGetAttributes(&at, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return at.type == cudaMemoryTypeHost;
}
}  // namespace

size_t zyfa_prefill_fp8_host_workspace(int B, int S, int Hq, int Hkv, int Dqk, int Dv) {
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1 || Dqk < 1 || Dv < 1) return 0;
  return host_workspace(B, S, Hq, Hkv, Dqk, Dv).total;
}

int zyfa_prefill_fp8_host(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                          int Dqk, int Dv, float softmax_scale, int hadamard, int n_chunks, void* workspace,
                          size_t workspace_bytes, int flags, void* stream) {
  const int lean = fp8_flags_lean(flags);
  if (lean < 0) return lean_flags_error(flags);
  if (!q || !k || !v || !o || !workspace) return fail(ZYFA_ERR_INVALID_ARG, "null pointer");
  if (B < 1 || S < 1 || Hq < 1 || Hkv < 1)
    return fail(ZYFA_ERR_INVALID_ARG, "B, S, Hq, Hkv must be >= 1 (got %d, %d, %d, %d)", B, S, Hq, Hkv);
  if (n_chunks < 0 || n_chunks > kMaxChunks)
    return fail(ZYFA_ERR_INVALID_ARG, "n_chunks = %d must be in [0, %d]", n_chunks, kMaxChunks);
  if (!aligned(workspace, 256)) return fail(ZYFA_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (!((Dqk == 128 && Dv == 128) || (Dqk == 192 && Dv == 128)))
    return fail(ZYFA_ERR_UNSUPPORTED, "head dims (%d, %d) unsupported; use (128, 128) or (192, 128)", Dqk, Dv);
  if (Hq % Hkv != 0) return fail(ZYFA_ERR_INVALID_ARG, "Hq (%d) must be a multiple of Hkv (%d)", Hq, Hkv);
  if (hadamard && Dqk != 128) return fail(ZYFA_ERR_UNSUPPORTED, "Hadamard rotation needs head dim 128");
  if (!(softmax_scale > 0.f) || !std::isfinite(softmax_scale))
    return fail(ZYFA_ERR_INVALID_ARG, "softmax_scale must be positive and finite");
  const HostWorkspace w = host_workspace(B, S, Hq, Hkv, Dqk, Dv);
  if (workspace_bytes < w.total)
    return fail(ZYFA_ERR_INVALID_ARG, "workspace of %zu bytes is smaller than the %zu needed", workspace_bytes,
                w.total);
  if (!page_locked(q) || !page_locked(k) || !page_locked(v) || !page_locked(o))
    return fail(ZYFA_ERR_INVALID_ARG, "q, k, v and o must be page-locked host memory");
  HostPipe* p;
  if (int r = host_pipe(&p)) return r;

  // Chunk boundaries: multiples of 256 rows (attention pairs of query tiles).
  const int pairs = (S + 255) / 256;
  int n = n_chunks ? n_chunks : std::min(16, pairs);
  n = std::max(1, std::min(n, pairs));
  int bound[kMaxChunks + 1];
  for (int c = 0; c <= n; ++c) bound[c] = std::min(S, static_cast<int>((static_cast<long long>(pairs) * c / n) * 256));
  bound[n] = S;

  char* ws = static_cast<char*>(workspace);
  void *qd = ws + w.qd, *kd = ws + w.kd, *vd = ws + w.vd, *q8 = ws + w.q8, *k8 = ws + w.k8, *v8 = ws + w.v8;
  float *qs = reinterpret_cast<float*>(ws + w.qs), *ks = reinterpret_cast<float*>(ws + w.ks),
        *vs = reinterpret_cast<float*>(ws + w.vs);
  void* od = ws + w.od;
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  const int64_t sq[3] = {int64_t(S) * Hq * Dqk, int64_t(Hq) * Dqk, Dqk};
  const int64_t sk[3] = {int64_t(S) * Hkv * Dqk, int64_t(Hkv) * Dqk, Dqk};
  const int64_t sv[3] = {int64_t(S) * Hkv * Dv, int64_t(Hkv) * Dv, Dv};
  const int64_t so[3] = {int64_t(S) * Hq * Dv, int64_t(Hq) * Dv, Dv};

  std::lock_guard<std::mutex> lock(p->mu);
  cudaError_t e;
  int rc = ZYFA_OK;
  // Copy rows [r0, r1) of every batch of a dense [B,S,H,D] bf16 tensor.
  auto copy_rows = [&](void* dst, const void* src, int64_t row_bytes, int r0, int r1, cudaMemcpyKind kind,
                       cudaStream_t s) {
    const size_t pitch = size_t(row_bytes) * S;
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + size_t(row_bytes) * r0, pitch,
                             static_cast<const char*>(src) + size_t(row_bytes) * r0, pitch,
                             size_t(row_bytes) * (r1 - r0), B, kind, s);
  };
  if ((e = cudaEventRecord(p->start, st)) != cudaSuccess) return fail_cuda(e, "cudaEventRecord");
  if ((e = cudaStreamWaitEvent(p->h2d, p->start, 0)) != cudaSuccess) return fail_cuda(e, "cudaStreamWaitEvent");
  for (int c = 0; c < n && rc == ZYFA_OK; ++c) {
    const int r0 = bound[c], r1 = bound[c + 1];
    if ((e = copy_rows(qd, q, int64_t(Hq) * Dqk * 2, r0, r1, cudaMemcpyHostToDevice, p->h2d)) != cudaSuccess ||
        (e = copy_rows(kd, k, int64_t(Hkv) * Dqk * 2, r0, r1, cudaMemcpyHostToDevice, p->h2d)) != cudaSuccess ||
        (e = copy_rows(vd, v, int64_t(Hkv) * Dv * 2, r0, r1, cudaMemcpyHostToDevice, p->h2d)) != cudaSuccess ||
        (e = cudaEventRecord(p->in[c], p->h2d)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, p->in[c], 0)) != cudaSuccess) {
      rc = fail_cuda(e, "host pipeline: copy in");
      break;
    }
    // Quantisers in order on the caller's stream; the attention of piece c on
    // one of two streams, so that the next piece's attention can take the
    // SMs that the tail of this one leaves idle (pieces depend only on the
    // quantised inputs, never on each other's outputs).
    cudaStream_t sa = p->att[c % kAttnStreams];
    if ((rc = quant_qkv(qd, sq, kd, sk, vd, sv, q8, qs, k8, ks, v8, vs, B, S, Hq, Hkv, Dqk, Dv, hadamard, r0, r1,
                        stream)))
      break;
    if ((e = cudaEventRecord(p->quant[c], st)) != cudaSuccess || (e = cudaStreamWaitEvent(sa, p->quant[c], 0)) != cudaSuccess) {
      rc = fail_cuda(e, "host pipeline: order attention");
      break;
    }
    if ((rc = attn_common(true, lean, q8, qs, k8, ks, v8, vs, od, B, S, Hq, Hkv, Dqk, Dv, softmax_scale, sq, sk, sv, so,
                          r0, r1, sa)))
      break;
    if ((e = cudaEventRecord(p->done[c], sa)) != cudaSuccess || (e = cudaStreamWaitEvent(p->d2h, p->done[c], 0)) != cudaSuccess ||
        (e = copy_rows(o, od, int64_t(Hq) * Dv * 2, r0, r1, cudaMemcpyDeviceToHost, p->d2h)) != cudaSuccess)
      rc = fail_cuda(e, "host pipeline: copy out");
  }
  // Join both copy streams back into the caller's stream, also on error, so
  // that nothing of this call is left unordered against the caller's work.
  cudaStream_t side[2 + kAttnStreams] = {p->h2d, p->d2h};
  for (int i = 0; i < kAttnStreams; ++i) side[2 + i] = p->att[i];
  for (cudaStream_t x : side)
    if ((e = cudaEventRecord(p->end, x)) != cudaSuccess || (e = cudaStreamWaitEvent(st, p->end, 0)) != cudaSuccess)
      if (rc == ZYFA_OK) rc = fail_cuda(e, "host pipeline: join");
  return rc;
}

int zyfa_get_device_status(void* stream, unsigned int* word) {
  DeviceInfo* d;
  if (int r = device_info(&d)) return r;
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail_cuda(e, "cudaStreamSynchronize");
  unsigned int w = 0;
  if ((e = cudaMemcpyFromSymbol(&w, zyfa_device_status_word, sizeof(w))) != cudaSuccess)
    return fail_cuda(e, "read status word");
  const unsigned int zero = 0;
  if ((e = cudaMemcpyToSymbol(zyfa_device_status_word, &zero, sizeof(zero))) != cudaSuccess)
    return fail_cuda(e, "clear status word");
  if (word) *word = w;
  if (w & ~(zyfa::kStatusBadSeqlens | zyfa::kStatusBadPage))
    return fail(ZYFA_ERR_TIMEOUT, "device status word 0x%x: a kernel wait timed out", w);
  if (w & zyfa::kStatusBadSeqlens)
    return fail(ZYFA_ERR_INVALID_ARG, "device status word 0x%x: device cu_seqlens were not a valid partition "
                "(nothing was computed for that call)", w);
  if (w) return fail(ZYFA_ERR_INVALID_ARG, "device status word 0x%x: a block_table entry was outside the cache "
                     "(that call's output is meaningless)", w);
  return ZYFA_OK;
}

}  // extern "C"
