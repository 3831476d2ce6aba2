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
// Layout: one CTA of 256 threads per (batch, head, 128-token block); each of
// the 8 warps owns 16 rows and keeps them in registers between the amax pass
// and the conversion pass, so the input is read from HBM exactly once. Lane l
// holds elements 2(l + 32i) and 2(l + 32i) + 1 of a row, so a warp reads 128
// contiguous bytes per access and the Hadamard stages of span 2..32 are lane
// shuffles while spans 1 and 64 stay in registers.
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

// Streaming variant: one persistent CTA of 512 threads per SM walks the
// (batch, head, block) list; a TMA ring of kStages input blocks keeps several
// blocks in flight per SM while the current one is reduced and converted.
// Eight lanes share a row (a warp holds four rows at a time, two such row
// groups per warp): lane j of a row holds the 8-element groups starting at
// 8j, 64 + 8j (and 128 + 8j at D = 192), read as 16-byte shared-memory loads
// that cover 128 contiguous bytes per row. With the rotation (D = 128) the
// butterflies of span 1, 2, 4 (inside a group) and 64 (between the lane's two
// groups) are in registers and spans 8, 16, 32 are shuffles over the row's
// eight lanes; each butterfly is one rounded add or subtract, applied in the
// order 1, 2, ..., 64 as in the register kernel.
constexpr int kStreamThreads = 512;
constexpr int kStreamRowsPerWarp = kBlockTokens / (kStreamThreads / 32);   // 8
constexpr unsigned int kStatusQuantTimeout = 0x8u;

template <int D>
struct StreamCfg {
  static constexpr int kStages = D == 128 ? 4 : 3;
  static constexpr int kBlockBytes = kBlockTokens * D * 2;
  static constexpr int kSmemBytes = kStages * kBlockBytes + 1024;
};

struct NoQuantTable {};

// One 128-token block of the walk: map coordinates (b, h, tok), the number of
// its rows inside the sequence, and where its scale goes.
struct QBlock {
  int b, h, tok, valid;
  int64_t scale_idx;
};

template <int D, bool kHadamard, bool VARLEN>
__global__ void __launch_bounds__(kStreamThreads, 1)
    quantize_fp8_stream_kernel(const __grid_constant__ CUtensorMap tm_x, QuantArgs a,
                               const __grid_constant__ typename std::conditional<VARLEN, QuantSeqTable,
                                                                                 NoQuantTable>::type tab_param,
                               const typename std::conditional<VARLEN, QuantSeqTable, NoQuantTable>::type* tab_global) {
  // The sequence table comes by value (built on the host) or, when the
  // offsets live on the device, from global memory (built by a kernel).
  const auto* tab = tab_global ? tab_global : &tab_param;
  using SC = StreamCfg<D>;
  constexpr int kGroups = D / 64;   // 8-element groups per lane and row
  static_assert(!kHadamard || D == 128, "rotation is defined for head dim 128");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* buf = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 127) & ~uintptr_t(127));
  __shared__ __align__(8) uint64_t full[SC::kStages];
  __shared__ float red[2][kStreamThreads / 32];
  __shared__ int abort_flag;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = (a.S + kBlockTokens - 1) / kBlockTokens;
  long long total;
  if constexpr (VARLEN) total = static_cast<long long>(a.H) * tab->cum_blocks[tab->n_seqs];
  else total = static_cast<long long>(a.B) * a.H * (a.blk_hi - a.blk_lo);
  const long long first = blockIdx.x, step = gridDim.x;

  // Equal lengths: blocks in (b, h, blk) order. Packed sequences: sequence
  // by sequence (binary search on the block prefix), then (h, blk).
  auto coords = [&](long long g) {
    QBlock q;
    if constexpr (VARLEN) {
      int lo = 0, hi = tab->n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (static_cast<long long>(a.H) * tab->cum_blocks[mid] <= g) lo = mid; else hi = mid - 1;
      }
      const int nb = tab->cum_blocks[lo + 1] - tab->cum_blocks[lo];
      const int r = static_cast<int>(g - static_cast<long long>(a.H) * tab->cum_blocks[lo]);
      q.h = r / nb;
      const int blk = r - q.h * nb;
      q.b = 0;
      q.tok = tab->start[lo] + blk * kBlockTokens;
      q.valid = min(kBlockTokens, tab->len[lo] - blk * kBlockTokens);
      q.scale_idx = (static_cast<int64_t>(lo) * a.H + q.h) * tab->max_blocks + blk;
    } else {
      const int range = a.blk_hi - a.blk_lo;
      const int blk = a.blk_lo + static_cast<int>(g % range);
      const long long bh = g / range;
      q.h = static_cast<int>(bh % a.H);
      q.b = static_cast<int>(bh / a.H);
      q.tok = blk * kBlockTokens;
      q.valid = min(kBlockTokens, a.S - blk * kBlockTokens);
      q.scale_idx = (static_cast<int64_t>(q.b) * a.H + q.h) * nblk + blk;
    }
    return q;
  };
  auto issue = [&](long long g, int st) {
    const QBlock q = coords(g);
    mbar_arrive_expect_tx(&full[st], SC::kBlockBytes);
    tma_load_4d(buf + st * SC::kBlockBytes, &tm_x, &full[st], 0, q.h, q.tok, q.b);
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < SC::kStages; ++i) mbar_init(&full[i], 1);
    abort_flag = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_x);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int i = 0; i < SC::kStages; ++i)
      if (first + i * step < total) issue(first + i * step, i);
  }

  int it = 0;
  for (long long g = first; g < total; g += step, ++it) {
    const int st = it % SC::kStages;
    const uint32_t par = static_cast<uint32_t>(it / SC::kStages) & 1u;
    const QBlock qb = coords(g);
    const bool ok = mbar_wait(&full[st], par, &abort_flag, a.status, kStatusQuantTimeout, a.timeout_ns);

    // v[g][k*8 + e]: row warp*8 + 4*g + lane/8, element 64*k + 8*(lane%8) + e
    float v[2][kGroups * 8];
    float amax = 0.f;
    if (ok) {
      const uint8_t* tile = buf + st * SC::kBlockBytes;
#pragma unroll
      for (int g2 = 0; g2 < 2; ++g2) {
        const int r = warp * kStreamRowsPerWarp + 4 * g2 + (lane >> 3);
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
          const uint4 raw = *reinterpret_cast<const uint4*>(tile + (r * D + 64 * k + 8 * (lane & 7)) * 2);
          const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
            v[g2][8 * k + 2 * e] = f.x;
            v[g2][8 * k + 2 * e + 1] = f.y;
          }
        }
        if constexpr (VARLEN) {
          // rows past the sequence's end belong to the next sequence
          if (r >= qb.valid) {
#pragma unroll
            for (int e = 0; e < kGroups * 8; ++e) v[g2][e] = 0.f;
          }
        }
        if constexpr (kHadamard) {
          // spans 1, 2, 4 inside each group of eight
#pragma unroll
          for (int hs = 1; hs <= 4; hs <<= 1) {
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              if (e & hs) continue;
              const float a0 = v[g2][e], a1 = v[g2][e + hs];
              v[g2][e] = __fadd_rn(a0, a1);
              v[g2][e + hs] = __fsub_rn(a0, a1);
            }
          }
          // spans 8, 16, 32: partner lane differs in bit 0, 1, 2 of the row lane
#pragma unroll
          for (int m = 1; m <= 4; m <<= 1) {
            const float sgn = (lane & m) ? -1.f : 1.f;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float o = __shfl_xor_sync(0xffffffffu, v[g2][e], m);
              v[g2][e] = __fmaf_rn(sgn, v[g2][e], o);   // lower: o + v, upper: o - v
            }
          }
          // span 64: the lane's two groups
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const float a0 = v[g2][e], a1 = v[g2][8 + e];
            v[g2][e] = __fadd_rn(a0, a1);
            v[g2][8 + e] = __fsub_rn(a0, a1);
          }
#pragma unroll
          for (int e = 0; e < 16; ++e) v[g2][e] = __fmul_rn(v[g2][e], kInvSqrt128);
        }
#pragma unroll
        for (int e = 0; e < kGroups * 8; e += 2) amax = max3f(amax, fabsf(v[g2][e]), fabsf(v[g2][e + 1]));
      }
    }
#pragma unroll
    for (int m = 16; m >= 1; m >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, m));
    if (lane == 0) red[it & 1][warp] = amax;
    // Every thread has its rows in registers: the stage may be refilled.
    if (__syncthreads_or(!ok)) break;
    if (threadIdx.x == 0 && g + SC::kStages * step < total) issue(g + SC::kStages * step, st);
    float bmax = red[it & 1][0];
#pragma unroll
    for (int w = 1; w < kStreamThreads / 32; ++w) bmax = fmaxf(bmax, red[it & 1][w]);
    const float scale = (bmax < kZeroGuard) ? 1.0f : __fdiv_rn(bmax, kE4m3Max);
    const float rinv = __frcp_rn(scale);
    if (threadIdx.x == 0) a.scales[qb.scale_idx] = scale;
#pragma unroll
    for (int g2 = 0; g2 < 2; ++g2) {
      const int rr = warp * kStreamRowsPerWarp + 4 * g2 + (lane >> 3);
      if (rr < qb.valid) {
        const int64_t s = static_cast<int64_t>(qb.b) * a.S + qb.tok + rr;
        uint8_t* orow = a.out + (s * a.H + qb.h) * D + 8 * (lane & 7);
#pragma unroll
        for (int k = 0; k < kGroups; ++k) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_e4m3x2(div_by_scale(v[g2][8 * k + 2 * e], scale, rinv),
                               div_by_scale(v[g2][8 * k + 2 * e + 1], scale, rinv));
          *reinterpret_cast<uint2*>(orow + 64 * k) = make_uint2(w[0] | (w[1] << 16), w[2] | (w[3] << 16));
        }
      }
    }
  }
  // On abort, let every issued copy land before the CTA exits (bounded).
  if (threadIdx.x == 0 && abort_flag) {
    int k = 0;
    for (long long g = first; g < total && k < it + SC::kStages; g += step, ++k) {
      if (k < it) continue;
      const int st = k % SC::kStages;
      if (!mbar_wait_drain(&full[st], static_cast<uint32_t>(k / SC::kStages) & 1u, 200000000ull))
        atomicOr(a.status, 0x100u);
    }
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

template <int D, bool H, bool VARLEN, typename Table>
static cudaError_t launch_stream(const CUtensorMap& tm_x, const QuantArgs& a, const Table& tab, long long total,
                                 cudaStream_t stream, const Table* tab_global = nullptr) {
  auto kern = quantize_fp8_stream_kernel<D, H, VARLEN>;
  // The shared-memory opt-in is per function and device: set it once.
  static bool opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !opted_in[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, StreamCfg<D>::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted_in[dev] = true;
  }
  if (total == 0) return cudaSuccess;
  const int grid = static_cast<int>(total < a.num_sms ? total : a.num_sms);
  kern<<<grid, kStreamThreads, StreamCfg<D>::kSmemBytes, stream>>>(tm_x, a, tab, tab_global);
  return cudaGetLastError();
}

cudaError_t launch_quantize_fp8_stream(const CUtensorMap& tm_x, const QuantArgs& a, cudaStream_t stream) {
  const NoQuantTable none{};
  const long long total = static_cast<long long>(a.B) * a.H * (a.blk_hi - a.blk_lo);
  if (a.D == 128 && a.hadamard) return launch_stream<128, true, false>(tm_x, a, none, total, stream);
  if (a.D == 128) return launch_stream<128, false, false>(tm_x, a, none, total, stream);
  if (a.D == 192) return launch_stream<192, false, false>(tm_x, a, none, total, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_fp8_stream_varlen(const CUtensorMap& tm_x, const QuantArgs& a, const QuantSeqTable& tab,
                                              cudaStream_t stream) {
  const long long total = static_cast<long long>(a.H) * tab.cum_blocks[tab.n_seqs];
  if (a.D == 128 && a.hadamard) return launch_stream<128, true, true>(tm_x, a, tab, total, stream);
  if (a.D == 128) return launch_stream<128, false, true>(tm_x, a, tab, total, stream);
  if (a.D == 192) return launch_stream<192, false, true>(tm_x, a, tab, total, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_quantize_fp8_stream_varlen_dev(const CUtensorMap& tm_x, const QuantArgs& a,
                                                  const QuantSeqTable* tab, cudaStream_t stream) {
  // The block count is only known on the device: one CTA per SM, each walks
  // the table's blocks (none when the table is empty).
  static const QuantSeqTable unused{};
  const long long total = a.num_sms;
  if (a.D == 128 && a.hadamard) return launch_stream<128, true, true>(tm_x, a, unused, total, stream, tab);
  if (a.D == 128) return launch_stream<128, false, true>(tm_x, a, unused, total, stream, tab);
  if (a.D == 192) return launch_stream<192, false, true>(tm_x, a, unused, total, stream, tab);
  return cudaErrorInvalidValue;
}

}  // namespace zyfa
