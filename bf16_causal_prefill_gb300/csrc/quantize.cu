// Per-block FP8 (e4m3) quantisation of Q, K or V, with an optional
// 128-point Walsh-Hadamard rotation of each row before quantisation.
//
// Method: "FP8 GEMM on CDNA4", section 2.2 (amax per block, scale =
// amax / 448, guard for all-zero blocks) and section 2.3 (round to nearest
// even), at per-(batch, head, 128-token block) granularity. The rotation of Q
// and K over the head dimension, fused into the quantisation pass, follows
// "ZYFA: Fast and Accurate FP8 Attention on AMD MI355X", section "FP8 Error in
// Full-Model Inference" and footnote 2.
//
// Arithmetic (fixed to the bit): fp32 butterflies of span 1, 2, ..., 64 in
// that order, each (a + b, a - b) rounded to fp32, then one multiply by
// fl32(1/sqrt(128)); scale = RN(amax / 448) with IEEE division (scale = 1
// when amax < 1e-8); code = cvt.rn.satfinite.e4m3(RN(y / scale)).
//
// Two kernels give the same bytes. The streaming kernel (below) takes every
// input that allows 16-byte tiled copies. The register kernel takes the
// other views: one CTA of 256 threads per (batch, head, 128-token block);
// each of the 8 warps owns 16 rows and keeps them in registers between the
// amax pass and the conversion pass, so the input is read from HBM exactly
// once. Lane l holds elements 2(l + 32i) and 2(l + 32i) + 1 of a row, so a
// warp reads 128 contiguous bytes per access and the Hadamard stages of span
// 2..32 are lane shuffles while spans 1 and 64 stay in registers.
#include <cuda_bf16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace zyfa {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kRowsPerWarp = kBlockTokens / (kQuantThreads / 32);   // 16
constexpr float kInvSqrt128 = 0.0883883476483184405501055452631f;   // RN to fp32 of 2^-3.5
constexpr float kE4m3Max = 448.0f;
constexpr float kZeroGuard = 1e-8f;

// y / scale rounded to fp32, for a whole block with one scale: Markstein's
// correction step (P. Markstein, "Computation of elementary functions on the
// IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// rinv = RN(1/scale) and the faithful q0 = RN(y * rinv), the remainder
// rem = y - scale * q0 is exact under FMA and RN(q0 + rem * rinv) is the
// correctly rounded quotient whenever no intermediate underflows. Every
// quotient that can round to a nonzero e4m3 code (|q| >= 2^-10, so y, scale
// and rem are normal) is therefore exact; smaller ones round to a signed zero
// code either way. A nonzero quotient has the sign of y; the sign is copied
// from y so that y = -0 keeps it (the corrected sum would give +0).
__device__ __forceinline__ float div_by_scale(float y, float scale, float rinv) {
  const float q0 = __fmul_rn(y, rinv);
  const float rem = __fmaf_rn(-scale, q0, y);
  return copysignf(__fmaf_rn(rem, rinv, q0), y);
}

template <int D, bool kHadamard>
__global__ void __launch_bounds__(kQuantThreads) quantize_fp8_kernel(QuantArgs a) {
  constexpr int kPairs = D / 64;   // bf16 pairs per lane per row
  static_assert(!kHadamard || D == 128, "rotation is defined for head dim 128");
  const int blk = a.blk_lo + blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (a.S + kBlockTokens - 1) / kBlockTokens;
  const __nv_bfloat16* x = static_cast<const __nv_bfloat16*>(a.x);

  float v[kRowsPerWarp][2 * kPairs];
  float amax = 0.f;
#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int s = blk * kBlockTokens + warp * kRowsPerWarp + rr;
    const bool valid = s < a.S;
    const __nv_bfloat16* row = x + b * a.sb + static_cast<int64_t>(s) * a.ss + h * a.sh;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      float2 f = make_float2(0.f, 0.f);
      if (valid) {
        const __nv_bfloat162 p = *reinterpret_cast<const __nv_bfloat162*>(row + 2 * (lane + 32 * i));
        f = __bfloat1622float2(p);
      }
      v[rr][2 * i] = f.x;
      v[rr][2 * i + 1] = f.y;
    }
    if constexpr (kHadamard) {
      // span 1: the two elements of a pair
#pragma unroll
      for (int i = 0; i < kPairs; ++i) {
        const float a0 = v[rr][2 * i], a1 = v[rr][2 * i + 1];
        v[rr][2 * i] = __fadd_rn(a0, a1);
        v[rr][2 * i + 1] = __fsub_rn(a0, a1);
      }
      // spans 2..32: partner lane differs in bit log2(span) - 1
#pragma unroll
      for (int m = 1; m <= 16; m <<= 1) {
        const bool upper = (lane & m) != 0;
#pragma unroll
        for (int e = 0; e < 2 * kPairs; ++e) {
          const float o = __shfl_xor_sync(0xffffffffu, v[rr][e], m);
          v[rr][e] = upper ? __fsub_rn(o, v[rr][e]) : __fadd_rn(v[rr][e], o);
        }
      }
      // span 64: element pairs i = 0 and i = 1 of the same lane
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const float a0 = v[rr][t], a1 = v[rr][2 + t];
        v[rr][t] = __fadd_rn(a0, a1);
        v[rr][2 + t] = __fsub_rn(a0, a1);
      }
#pragma unroll
      for (int e = 0; e < 2 * kPairs; ++e) v[rr][e] = __fmul_rn(v[rr][e], kInvSqrt128);
    }
#pragma unroll
    for (int e = 0; e < 2 * kPairs; ++e) amax = fmaxf(amax, fabsf(v[rr][e]));
  }

  // block-wide amax (max is exact in any order)
  __shared__ float red[kQuantThreads / 32];
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
  if (lane == 0) red[warp] = amax;
  __syncthreads();
  float bmax = red[0];
#pragma unroll
  for (int w = 1; w < kQuantThreads / 32; ++w) bmax = fmaxf(bmax, red[w]);
  const float scale = (bmax < kZeroGuard) ? 1.0f : __fdiv_rn(bmax, kE4m3Max);
  const float rinv = __frcp_rn(scale);
  if (threadIdx.x == 0) a.scales[(static_cast<int64_t>(b) * a.H + h) * nblk + blk] = scale;

#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int s = blk * kBlockTokens + warp * kRowsPerWarp + rr;
    if (s >= a.S) break;
    uint8_t* orow = a.out + ((static_cast<int64_t>(b) * a.S + s) * a.H + h) * D;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const float q0 = div_by_scale(v[rr][2 * i], scale, rinv);
      const float q1 = div_by_scale(v[rr][2 * i + 1], scale, rinv);
      *reinterpret_cast<uint16_t*>(orow + 2 * (lane + 32 * i)) = pack_e4m3x2(q0, q1);
    }
  }
}

// Streaming kernel: one persistent CTA per SM walks the 128-token blocks of
// up to three tensors (Q, K, V of one call: Q's blocks, then K's, then V's),
// every CTA taking blocks blockIdx.x, blockIdx.x + gridDim.x, ...
//
// Roles: one thread of warp 8 issues one TMA load per block into a ring of
// stages (the block as column blocks of 64 elements x 128 rows, 128-byte
// swizzle); two consumer warpgroups take the CTA's blocks in turn, one
// thread per row. A thread loads its whole row into registers (the swizzle
// spreads the 16-byte loads of eight consecutive rows over all banks), so the rotation's
// butterflies are all in registers, in packed float2 arithmetic (spans 2 to
// 64; span 1 pairs the two halves of a float2). The block amax is a warp
// reduction plus one named barrier of the warpgroup; the codes overwrite the
// block's own stage (every row has been read by then), swizzled, and leave
// in one TMA store per 128-byte column block (rows past the tensor's end
// are not written); the stage goes back to the loader once that store has
// read it, checked when the warpgroup starts its next block. A packed sequence's
// last, partial block is stored row by row from registers instead, since
// its box would cover the next sequence's rows.
//
// Division: with rinv = RN(1/scale), q0n = RN(y * -rinv) = -q0 exactly,
// rem = RN(y - scale*q0) is exact (Markstein), and RN(q0n + rem * -rinv)
// is minus the correctly rounded quotient; converting it and flipping the
// sign bit of each code gives the code of y / scale, signed zeros
// included (+0 and -0 inputs come out as 0x00 and 0x80).
//
// 384 threads launched at 168 registers each: the consumer warpgroups raise
// theirs to 232 (a rotated row alone is 128 fp32 values) and the loader
// warpgroup drops to 40: 2 x 128 x 232 + 128 x 40 = 384 x 168.
constexpr int kStreamThreads = 384;       // two consumer warpgroups + the loader warpgroup
constexpr int kLoaderWarp = 8;            // its first warp issues the loads
constexpr uint32_t kConsumerRegs = 232, kLoaderRegs = 40;
static_assert(2 * 128 * kConsumerRegs + 128 * kLoaderRegs <= kStreamThreads * 168, "register split");
constexpr unsigned int kStatusQuantTimeout = 0x8u;

// An even number of stages, so that every stage serves one warpgroup only
// (block k of a CTA goes to stage k mod kStages and warpgroup k mod 2), and
// each warpgroup's waits on a stage's barrier follow that stage's phases in
// order.
template <int DMAX>
struct StreamCfg {
  static constexpr int kStageBytes = kBlockTokens * DMAX * 2;               // bf16 block
  static constexpr int kStages = 2 * ((232448 - 2048) / (2 * kStageBytes));  // 6 at D = 128, 4 at 192
  static constexpr int kSmemBytes = kStages * kStageBytes + 1024;
  static_assert(kStages >= 2 && kStages % 2 == 0, "ring");
};

struct NoQuantTable {};

// One 128-token block of the walk.
struct QBlock {
  int t;               // tensor of the call
  int b, h, tok;       // map coordinates (batch, head, first token)
  int valid;           // rows of the block inside its sequence
  int64_t scale_idx;   // where its scale goes
};

template <bool VARLEN, typename Tab>
__device__ __forceinline__ QBlock stream_coords(long long g, const QuantStreamArgs& a, const Tab* tab,
                                                const long long (&start)[4]) {
  QBlock q;
  q.t = g >= start[2] ? 2 : (g >= start[1] ? 1 : 0);
  const int H = a.t[q.t].H;
  const long long l = g - (q.t == 2 ? start[2] : (q.t == 1 ? start[1] : 0));
  if constexpr (VARLEN) {
    int lo = 0, hi = tab->n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (static_cast<long long>(H) * tab->cum_blocks[mid] <= l) lo = mid; else hi = mid - 1;
    }
    const int nb = tab->cum_blocks[lo + 1] - tab->cum_blocks[lo];
    const int r = static_cast<int>(l - static_cast<long long>(H) * tab->cum_blocks[lo]);
    q.h = r / nb;
    const int blk = r - q.h * nb;
    q.b = 0;
    q.tok = tab->start[lo] + blk * kBlockTokens;
    q.valid = min(kBlockTokens, tab->len[lo] - blk * kBlockTokens);
    q.scale_idx = (static_cast<int64_t>(lo) * H + q.h) * tab->max_blocks + blk;
  } else {
    const int range = a.blk_hi - a.blk_lo;
    const int blk = a.blk_lo + static_cast<int>(l % range);
    const long long bh = l / range;
    q.h = static_cast<int>(bh % H);
    q.b = static_cast<int>(bh / H);
    q.tok = blk * kBlockTokens;
    q.valid = min(kBlockTokens, a.S - q.tok);
    const int nblk = (a.S + kBlockTokens - 1) / kBlockTokens;
    q.scale_idx = (static_cast<int64_t>(q.b) * H + q.h) * nblk + blk;
  }
  return q;
}

// Converts 16 consecutive values (8 float2) of a row to e4m3 codes, as four
// little-endian words, element 0 in the low byte of the first.
__device__ __forceinline__ uint4 codes16(const float2 (&y)[8], float2 sc2, float2 nr2) {
  uint32_t w[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    uint32_t c[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float2 v = y[2 * i + e];
      const float2 q0n = __fmul2_rn(v, nr2);
      const float2 rem = __ffma2_rn(q0n, sc2, v);
      const float2 nq = __ffma2_rn(rem, nr2, q0n);
      c[e] = pack_e4m3x2(nq.x, nq.y);
    }
    w[i] = (c[0] | (c[1] << 16)) ^ 0x80808080u;
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

// One block, one row per thread of the warpgroup. Returns false if the CTA
// is aborting (this warpgroup then leaves its loop).
// `stage` holds the block; its codes are staged there for the store.
template <int D, bool ROT, bool VARLEN>
__device__ __forceinline__ bool stream_block(const QBlock& qb, const QuantStreamArgs& a, const CUtensorMap* out_map,
                                             uint8_t* stage, bool ok, float* red, int wg) {
  const int r = threadIdx.x & 127, warp = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  static_assert(!ROT || D == 128, "rotation is defined for head dim 128");
  const QuantTensor& T = a.t[qb.t];
  constexpr int kWords = D / 2;   // bf16 pairs of the row
  uint32_t raw[kWords];
  if (ok) {
#pragma unroll
    for (int cb = 0; cb < D / 64; ++cb) {
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 v = *reinterpret_cast<const uint4*>(stage + cb * 16384 + r * 128 + ((c ^ (r & 7)) << 4));
        raw[32 * cb + 4 * c] = v.x;
        raw[32 * cb + 4 * c + 1] = v.y;
        raw[32 * cb + 4 * c + 2] = v.z;
        raw[32 * cb + 4 * c + 3] = v.w;
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < kWords; ++j) raw[j] = 0u;
  }
  if constexpr (VARLEN) {
    // rows past the sequence's end belong to the next sequence
    if (r >= qb.valid) {
#pragma unroll
      for (int j = 0; j < kWords; ++j) raw[j] = 0u;
    }
  }
  float2 y[ROT ? kWords : 1];   // the rotated row
  float amax = 0.f;
  if constexpr (ROT) {
#pragma unroll
    for (int j = 0; j < kWords; ++j) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[j]));
      y[j] = make_float2(__fadd_rn(f.x, f.y), __fsub_rn(f.x, f.y));   // span 1
    }
    const float2 m1 = make_float2(-1.f, -1.f);
#pragma unroll
    for (int hs = 1; hs < kWords; hs <<= 1) {   // spans 2, 4, ..., 64
#pragma unroll
      for (int j = 0; j < kWords; ++j) {
        if (j & hs) continue;
        const float2 u = y[j], v = y[j + hs];
        y[j] = __fadd2_rn(u, v);
        y[j + hs] = __ffma2_rn(v, m1, u);   // u - v
      }
    }
    const float2 c2 = make_float2(kInvSqrt128, kInvSqrt128);
#pragma unroll
    for (int j = 0; j < kWords; ++j) {
      y[j] = __fmul2_rn(y[j], c2);
      amax = max3f(amax, fabsf(y[j].x), fabsf(y[j].y));
    }
  } else {
    __nv_bfloat162 m2 = __float2bfloat162_rn(0.f);
#pragma unroll
    for (int j = 0; j < kWords; ++j) m2 = __hmax2(m2, __habs2(*reinterpret_cast<const __nv_bfloat162*>(&raw[j])));
    const float2 mf = __bfloat1622float2(m2);
    amax = fmaxf(mf.x, mf.y);
  }
  // amax >= 0 and never NaN: its bit pattern orders like the value
  amax = __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(amax)));
  if (lane == 0) red[warp] = amax;
  // past this barrier every row of the block is in registers
  if (named_bar_red_or(1 + wg, 128, !ok)) return false;
  const float bmax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float scale = (bmax < kZeroGuard) ? 1.0f : __fdiv_rn(bmax, kE4m3Max);
  const float rinv = __frcp_rn(scale);
  const float2 sc2 = make_float2(scale, scale), nr2 = make_float2(-rinv, -rinv);
  if (r == 0) T.scales[qb.scale_idx] = scale;

  const bool direct = VARLEN && qb.valid < kBlockTokens;
  uint8_t* orow = T.out + ((static_cast<int64_t>(qb.b) * a.S + qb.tok + r) * T.H + qb.h) * D;
#pragma unroll
  for (int c = 0; c < D / 16; ++c) {
    float2 v[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      if constexpr (ROT) v[e] = y[8 * c + e];
      else v[e] = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&raw[8 * c + e]));
    }
    const uint4 w = codes16(v, sc2, nr2);
    if (direct) {
      if (r < qb.valid) *reinterpret_cast<uint4*>(orow + 16 * c) = w;
    } else {
      *reinterpret_cast<uint4*>(stage + (c >> 3) * 16384 + r * 128 + (((c & 7) ^ (r & 7)) << 4)) = w;
    }
  }
  // (also when nothing is staged: the amax slots are rewritten next block)
  fence_proxy_async_smem();
  named_bar_sync(1 + wg, 128);
  if (!direct) {
    if (r == 0) {
      if constexpr (D == 128) {
        tma_store_5d(out_map, stage, 0, qb.tok, 0, qb.h, qb.b);
      } else {
        tma_store_4d(out_map, stage, 0, qb.h, qb.tok, qb.b);
        tma_store_4d(out_map, stage + 16384, 128, qb.h, qb.tok, qb.b);
      }
      bulk_commit_group();
    }
  }
  return true;
}

template <int DMAX, bool VARLEN>
__global__ void __launch_bounds__(kStreamThreads, 1)
    quantize_fp8_stream_kernel(const __grid_constant__ QuantMaps maps, QuantStreamArgs a,
                               const __grid_constant__ typename std::conditional<VARLEN, QuantSeqTable,
                                                                                 NoQuantTable>::type tab_param,
                               const typename std::conditional<VARLEN, QuantSeqTable, NoQuantTable>::type* tab_global) {
  using SC = StreamCfg<DMAX>;
  // The sequence table comes by value (built on the host) or, when the
  // offsets live on the device, from global memory (built by a kernel).
  const auto* tab = tab_global ? tab_global : &tab_param;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = base;
  __shared__ __align__(8) uint64_t full[SC::kStages];
  __shared__ __align__(8) uint64_t empty[SC::kStages];
  __shared__ float red[2][4];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5;

  long long start[4];
  start[0] = 0;
#pragma unroll
  for (int t = 0; t < 3; ++t) {
    long long n = 0;
    if (t < a.n) {
      if constexpr (VARLEN) n = static_cast<long long>(a.t[t].H) * tab->cum_blocks[tab->n_seqs];
      else n = static_cast<long long>(a.B) * a.t[t].H * (a.blk_hi - a.blk_lo);
    }
    start[t + 1] = start[t] + n;
  }
  const long long total = start[3];
  const long long first = blockIdx.x, step = gridDim.x;

  if (threadIdx.x == 0) {
    for (int i = 0; i < SC::kStages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();

  if (warp >= kLoaderWarp) {
    regs_decrease<kLoaderRegs>();
    if (warp == kLoaderWarp && (threadIdx.x & 31) == 0) {
      for (int t = 0; t < a.n; ++t) tma_prefetch_desc(&maps.in[t]);
      long long k = 0;
      for (long long g = first; g < total; g += step, ++k) {
        const int s = static_cast<int>(k % SC::kStages);
        if (k >= SC::kStages &&
            !mbar_wait(&empty[s], static_cast<uint32_t>(k / SC::kStages - 1) & 1u, &abort_flag, a.status,
                       kStatusQuantTimeout, a.timeout_ns))
          break;
        const QBlock q = stream_coords<VARLEN>(g, a, tab, start);
        mbar_arrive_expect_tx(&full[s], kBlockTokens * a.t[q.t].D * 2);
        tma_load_5d(stages + s * SC::kStageBytes, &maps.in[q.t], &full[s], 0, q.tok, 0, q.h, q.b);
      }
      // On abort, let every issued copy land before the CTA exits (bounded):
      // the last block issued on each stage.
      if (abort_flag) {
        for (long long kk = k - 1; kk >= 0 && kk >= k - SC::kStages; --kk) {
          if (!mbar_wait_drain(&full[kk % SC::kStages], static_cast<uint32_t>(kk / SC::kStages) & 1u, 200000000ull))
            atomicOr(a.status, 0x100u);
        }
      }
    }
    return;
  }

  regs_increase<kConsumerRegs>();
  const int wg = warp >> 2;
  const bool leader = (threadIdx.x & 127) == 0;
  int held = -1;   // stage whose store may still be reading it (leader only)
  long long k = wg;
  for (long long g = first + wg * step; g < total; g += 2 * step, k += 2) {
    const int s = static_cast<int>(k % SC::kStages);
    const bool ok = mbar_wait(&full[s], static_cast<uint32_t>(k / SC::kStages) & 1u, &abort_flag, a.status,
                              kStatusQuantTimeout, a.timeout_ns);
    // the previous block's store has read its stage: hand that stage back
    if (leader && held >= 0) {
      bulk_wait_group_read<0>();
      mbar_arrive(&empty[held]);
    }
    held = s;
    const QBlock qb = stream_coords<VARLEN>(g, a, tab, start);
    uint8_t* stage = stages + s * SC::kStageBytes;
    bool go;
    if (DMAX == 192 && a.t[qb.t].D == 192)
      go = stream_block<DMAX == 192 ? 192 : 128, false, VARLEN>(qb, a, &maps.out[qb.t], stage, ok, red[wg], wg);
    else if (a.t[qb.t].hadamard)
      go = stream_block<128, true, VARLEN>(qb, a, &maps.out[qb.t], stage, ok, red[wg], wg);
    else
      go = stream_block<128, false, VARLEN>(qb, a, &maps.out[qb.t], stage, ok, red[wg], wg);
    if (!go) break;
  }
  // every store of this warpgroup complete before the CTA exits, and the
  // last stage handed back (the loader may still be waiting for it)
  if (leader) {
    bulk_wait_group<0>();
    if (held >= 0) mbar_arrive(&empty[held]);
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream) {
  if (a.blk_hi <= a.blk_lo) return cudaSuccess;
  dim3 grid(a.blk_hi - a.blk_lo, a.H, a.B);
  if (a.D == 128 && a.hadamard) {
    quantize_fp8_kernel<128, true><<<grid, kQuantThreads, 0, stream>>>(a);
  } else if (a.D == 128) {
    quantize_fp8_kernel<128, false><<<grid, kQuantThreads, 0, stream>>>(a);
  } else if (a.D == 192) {
    quantize_fp8_kernel<192, false><<<grid, kQuantThreads, 0, stream>>>(a);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

template <int DMAX, bool VARLEN, typename Table>
static cudaError_t launch_stream(const QuantMaps& m, const QuantStreamArgs& a, const Table& tab, int grid,
                                 cudaStream_t stream, const Table* tab_global = nullptr) {
  auto kern = quantize_fp8_stream_kernel<DMAX, VARLEN>;
  // The shared-memory opt-in is per function and device: set it once.
  static bool opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !opted_in[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, StreamCfg<DMAX>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted_in[dev] = true;
  }
  if (grid == 0) return cudaSuccess;
  kern<<<grid, kStreamThreads, StreamCfg<DMAX>::kSmemBytes, stream>>>(m, a, tab, tab_global);
  return cudaGetLastError();
}

static bool stream_args_ok(const QuantStreamArgs& a, int dmax) {
  if (a.n < 1 || a.n > 3 || (dmax != 128 && dmax != 192)) return false;
  for (int t = 0; t < a.n; ++t) {
    const QuantTensor& T = a.t[t];
    if ((T.D != 128 && T.D != 192) || T.D > dmax || (T.hadamard && T.D != 128) || T.H < 1) return false;
  }
  return true;
}

cudaError_t launch_quantize_fp8_stream(const QuantMaps& m, const QuantStreamArgs& a, int dmax, int num_sms,
                                       cudaStream_t stream) {
  if (!stream_args_ok(a, dmax)) return cudaErrorInvalidValue;
  long long total = 0;
  for (int t = 0; t < a.n; ++t) total += static_cast<long long>(a.B) * a.t[t].H * (a.blk_hi - a.blk_lo);
  const int grid = static_cast<int>(total < num_sms ? total : num_sms);
  const NoQuantTable none{};
  if (dmax == 128) return launch_stream<128, false>(m, a, none, grid, stream);
  return launch_stream<192, false>(m, a, none, grid, stream);
}

cudaError_t launch_quantize_fp8_stream_varlen(const QuantMaps& m, const QuantStreamArgs& a, int dmax,
                                              const QuantSeqTable& tab, int num_sms, cudaStream_t stream) {
  if (!stream_args_ok(a, dmax)) return cudaErrorInvalidValue;
  long long total = 0;
  for (int t = 0; t < a.n; ++t) total += static_cast<long long>(a.t[t].H) * tab.cum_blocks[tab.n_seqs];
  const int grid = static_cast<int>(total < num_sms ? total : num_sms);
  if (dmax == 128) return launch_stream<128, true>(m, a, tab, grid, stream);
  return launch_stream<192, true>(m, a, tab, grid, stream);
}

cudaError_t launch_quantize_fp8_stream_varlen_dev(const QuantMaps& m, const QuantStreamArgs& a, int dmax,
                                                  const QuantSeqTable* tab, int num_sms, cudaStream_t stream) {
  // The block count is only known on the device: one CTA per SM, each walks
  // the table's blocks (none when the table is empty).
  if (!stream_args_ok(a, dmax)) return cudaErrorInvalidValue;
  static const QuantSeqTable unused{};
  if (dmax == 128) return launch_stream<128, true>(m, a, unused, num_sms, stream, tab);
  return launch_stream<192, true>(m, a, unused, num_sms, stream, tab);
}

}  // namespace zyfa
