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

#include "internal.h"
#include "ptx.cuh"

namespace zyfa {
namespace {

constexpr int kQuantThreads = 256;
constexpr int kRowsPerWarp = kBlockTokens / (kQuantThreads / 32);   // 16
constexpr float kInvSqrt128 = 0.0883883476483184405501055452631f;   // RN to fp32 of 2^-3.5
constexpr float kE4m3Max = 448.0f;
constexpr float kZeroGuard = 1e-8f;

template <int D, bool kHadamard>
__global__ void __launch_bounds__(kQuantThreads) quantize_fp8_kernel(QuantArgs a) {
  constexpr int kPairs = D / 64;   // bf16 pairs per lane per row
  static_assert(!kHadamard || D == 128, "rotation is defined for head dim 128");
  const int blk = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nblk = gridDim.x;
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
  if (threadIdx.x == 0) a.scales[(static_cast<int64_t>(b) * a.H + h) * nblk + blk] = scale;

#pragma unroll
  for (int rr = 0; rr < kRowsPerWarp; ++rr) {
    const int s = blk * kBlockTokens + warp * kRowsPerWarp + rr;
    if (s >= a.S) break;
    uint8_t* orow = a.out + ((static_cast<int64_t>(b) * a.S + s) * a.H + h) * D;
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
      const float q0 = __fdiv_rn(v[rr][2 * i], scale);
      const float q1 = __fdiv_rn(v[rr][2 * i + 1], scale);
      *reinterpret_cast<uint16_t*>(orow + 2 * (lane + 32 * i)) = pack_e4m3x2(q0, q1);
    }
  }
}

}  // namespace

cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream) {
  const int nblk = (a.S + kBlockTokens - 1) / kBlockTokens;
  dim3 grid(nblk, a.H, a.B);
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

}  // namespace zyfa
