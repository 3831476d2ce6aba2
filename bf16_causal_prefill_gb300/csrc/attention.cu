// Causal forward (prefill) attention for sm_103a, BF16 and FP8 (e4m3).
//
// What it computes ("ZYFA: Fast and Accurate FP8 Attention on AMD MI355X",
// "Introduction" and "Methodology and Limitations"): for every batch b, query
// head h and query row i,
//     O[b,i,h,:] = sum_{j<=i} softmax_j(scale * Q[b,i,h] . K[b,j,g(h)]) V[b,j,g(h)],
// g(h) = h / (Hq/Hkv), equal query and key lengths, output BF16.
//
// FP8 path ("Per-Block Scaling and Normalization by the Rounded Row Sum"):
// Q, K, V arrive as e4m3 codes with one fp32 scale per 128-token block. The
// probabilities of each 128-key tile of a row are multiplied by a power of two
// 2^k so that the largest lies in (0.5, 1], rounded to e4m3 (exact P: ex2 then
// RNE), multiplied by V in fp32 on the tensor cores, and the row is normalised
// by the sum of the ROUNDED probabilities (with 2^k divided back out), so the
// weights that multiply V sum to one. Base-2 softmax: p = 2^x with x the score
// minus the running row maximum in base-2 units ("Lean P" section).
//
// GB300 design (not the pages' MI355X design):
//   * persistent CTAs, one per SM, each owning a pair of 128-row query tiles
//     (2t, 2t+1) of one (batch, head); units are visited longest-first and the
//     heads of a GQA group are adjacent so that K/V tiles are shared in L2;
//   * warp 8 loads Q once per unit and K_j, V_j into separate shared-memory
//     rings with TMA (128-byte swizzle);
//   * warp 9 (one thread) issues tcgen05.mma: S = Q K^T (A, B from shared
//     memory) and O += P V (P from tensor memory, V from shared memory,
//     MN-major); accumulators live in tensor memory (S0, S1, O0, O1 = 512
//     columns) and completion is tracked with tcgen05.commit;
//   * warps 0-3 and 4-7 are the softmax warpgroups of the two query tiles,
//     one thread per row: they read S from tensor memory, write P back over
//     S (bf16 or e4m3), rescale O in tensor memory when needed, and write the
//     normalised BF16 output. While one warpgroup computes probabilities the
//     tensor cores run the other tile's products (two-tile ping-pong);
//   * the causal mask is applied on diagonal tiles only.
// Every barrier wait is bounded: on timeout the CTA raises an abort flag,
// records a code in the device status word, drains in-flight copies and
// tensor-core work, frees its tensor memory and exits.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace zyfa {
namespace {

constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // BF16: keep a stale max while x - m <= 8
constexpr float kMaxBlockShift = 100.0f;    // FP8: bound on the per-tile exponent k

enum StatusCode : unsigned int {
  kStatusLoaderTimeout = 0x1u,
  kStatusMmaTimeout = 0x2u,
  kStatusSoftmaxTimeout = 0x4u,
  kStatusDrainFailed = 0x100u,
};

template <int DQK, bool FP8>
struct Cfg {
  static constexpr int kElt = FP8 ? 1 : 2;
  static constexpr int kDv = 128;
  static constexpr int kQkRowBytes = DQK * kElt;
  static constexpr int kQkBlocks = (kQkRowBytes + 127) / 128;   // 128-byte swizzle columns
  static constexpr int kQkTileBytes = kQkBlocks * 128 * 128;
  static constexpr int kVBlocks = kDv * kElt / 128;
  static constexpr int kVTileBytes = kVBlocks * 128 * 128;
  static constexpr int kQkSteps = kQkRowBytes / 32;             // MMA K = 32 bytes
  static constexpr int kPvSteps = FP8 ? 4 : 8;                  // 128 keys / MMA K
  static constexpr int kPvStepBytes = (FP8 ? 32 : 16) * 128;    // V rows per MMA K step
  static constexpr int kInnerElts = 128 / kElt;                 // TMA box inner extent
  static constexpr int kNK = FP8 ? (DQK == 128 ? 4 : 3) : (DQK == 128 ? 3 : 2);
  static constexpr int kNV = FP8 ? (DQK == 128 ? 4 : 3) : (DQK == 128 ? 2 : 1);
  static constexpr uint32_t kIdescS = make_idesc(128, 128, FP8 ? 0u : 1u, false);
  static constexpr uint32_t kIdescPV = make_idesc(128, kDv, FP8 ? 0u : 1u, true);
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = 2 * kQkTileBytes;
  static constexpr int kOffV = kOffK + kNK * kQkTileBytes;
  static constexpr int kOffBar = kOffV + kNV * kVTileBytes;
  // q_full, q_empty, k_full[NK], k_empty[NK], v_full[NV], v_empty[NV],
  // s_full[2], p_full[2], o_full[2], drain
  static constexpr int kNumBars = 2 + 2 * kNK + 2 * kNV + 7;
  static constexpr int kSmemBytes = kOffBar + kNumBars * 8 + 16 + 1024;
  static_assert(kSmemBytes <= 232448, "shared memory budget");
};

struct Unit {
  int b, hq, t;
  bool has_b;
  int n_a, n_b, n_kv;
};

__device__ __forceinline__ Unit decode_unit(int u, int B, int Hq, int n_qtiles) {
  const int n_pairs = (n_qtiles + 1) / 2;
  const int bh_count = B * Hq;
  Unit w;
  w.t = n_pairs - 1 - u / bh_count;            // longest pairs first
  const int bh = u % bh_count;
  w.b = bh / Hq;
  w.hq = bh % Hq;                               // heads of a GQA group adjacent
  w.has_b = (2 * w.t + 1) < n_qtiles;
  w.n_a = 2 * w.t + 1;
  w.n_b = 2 * w.t + 2;
  w.n_kv = w.has_b ? w.n_b : w.n_a;
  return w;
}

template <int DQK, bool FP8>
struct Smem {
  using C = Cfg<DQK, FP8>;
  uint8_t* base;
  uint64_t* bars;
  __device__ __forceinline__ uint64_t* q_full() const { return bars; }
  __device__ __forceinline__ uint64_t* q_empty() const { return bars + 1; }
  __device__ __forceinline__ uint64_t* k_full(int s) const { return bars + 2 + s; }
  __device__ __forceinline__ uint64_t* k_empty(int s) const { return bars + 2 + C::kNK + s; }
  __device__ __forceinline__ uint64_t* v_full(int s) const { return bars + 2 + 2 * C::kNK + s; }
  __device__ __forceinline__ uint64_t* v_empty(int s) const { return bars + 2 + 2 * C::kNK + C::kNV + s; }
  __device__ __forceinline__ uint64_t* s_full(int t) const { return bars + 2 + 2 * C::kNK + 2 * C::kNV + t; }
  __device__ __forceinline__ uint64_t* p_full(int t) const { return s_full(2) + t; }
  __device__ __forceinline__ uint64_t* o_full(int t) const { return s_full(4) + t; }
  __device__ __forceinline__ uint64_t* drain() const { return s_full(6); }
  __device__ __forceinline__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(bars + C::kNumBars); }
  __device__ __forceinline__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(bars + C::kNumBars) + 1;
  }
  __device__ __forceinline__ uint8_t* q_tile(int t) const { return base + C::kOffQ + t * C::kQkTileBytes; }
  __device__ __forceinline__ uint8_t* k_tile(int s) const { return base + C::kOffK + s * C::kQkTileBytes; }
  __device__ __forceinline__ uint8_t* v_tile(int s) const { return base + C::kOffV + s * C::kVTileBytes; }
};

// ------------------------------------------------------------------ loader --
template <int DQK, bool FP8>
__device__ void loader_role(const Smem<DQK, FP8>& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                            const CUtensorMap* tm_v, const AttnArgs& a, int n_qtiles) {
  using C = Cfg<DQK, FP8>;
  const int n_units = a.B * a.Hq * ((n_qtiles + 1) / 2);
  const int group = a.Hq / a.Hkv;
  volatile int* abort_flag = sm.abort_flag();
  int ks = 0, vs = 0;
  uint32_t kph = 0, vph = 0, qn = 0;
  uint32_t k_issued = 0, v_issued = 0;          // stages written at least once
  uint32_t k_par[C::kNK], v_par[C::kNV];
  bool ok = true;
  for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(u, a.B, a.Hq, n_qtiles);
    const int hkv = w.hq / group;
    if (!(ok = mbar_wait(sm.q_empty(), (qn & 1u) ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)))
      break;
    mbar_arrive_expect_tx(sm.q_full(), (w.has_b ? 2 : 1) * C::kQkTileBytes);
#pragma unroll
    for (int kb = 0; kb < C::kQkBlocks; ++kb)
      tma_load_4d(sm.q_tile(0) + kb * 16384, tm_q, sm.q_full(), kb * C::kInnerElts, w.hq, 2 * w.t * 128, w.b);
    if (w.has_b) {
#pragma unroll
      for (int kb = 0; kb < C::kQkBlocks; ++kb)
        tma_load_4d(sm.q_tile(1) + kb * 16384, tm_q, sm.q_full(), kb * C::kInnerElts, w.hq, (2 * w.t + 1) * 128,
                    w.b);
    }
    ++qn;
    for (int j = 0; j < w.n_kv; ++j) {
      if (!(ok = mbar_wait(sm.k_empty(ks), kph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)))
        break;
      mbar_arrive_expect_tx(sm.k_full(ks), C::kQkTileBytes);
#pragma unroll
      for (int kb = 0; kb < C::kQkBlocks; ++kb)
        tma_load_4d(sm.k_tile(ks) + kb * 16384, tm_k, sm.k_full(ks), kb * C::kInnerElts, hkv, j * 128, w.b);
      k_par[ks] = kph;
      k_issued |= 1u << ks;
      if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
      if (!(ok = mbar_wait(sm.v_empty(vs), vph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)))
        break;
      mbar_arrive_expect_tx(sm.v_full(vs), C::kVTileBytes);
#pragma unroll
      for (int vb = 0; vb < C::kVBlocks; ++vb)
        tma_load_4d(sm.v_tile(vs) + vb * 16384, tm_v, sm.v_full(vs), vb * C::kInnerElts, hkv, j * 128, w.b);
      v_par[vs] = vph;
      v_issued |= 1u << vs;
      if (++vs == C::kNV) { vs = 0; vph ^= 1u; }
    }
  }
  if (ok) {
    // Tail: wait until every stage has been released for the last time, so
    // no tcgen05.commit arrival is still in flight when the CTA exits.
    for (int i = 0; i < C::kNK; ++i) {
      if (!mbar_wait(sm.k_empty(ks), kph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)) break;
      if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
    }
    for (int i = 0; i < C::kNV; ++i) {
      if (!mbar_wait(sm.v_empty(vs), vph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)) break;
      if (++vs == C::kNV) { vs = 0; vph ^= 1u; }
    }
    mbar_wait(sm.q_empty(), (qn & 1u) ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns);
  } else {
    // Abort: let every copy this thread issued land before the CTA exits.
    constexpr uint64_t kDrainNs = 200000000ull;
    for (int s = 0; s < C::kNK; ++s)
      if ((k_issued >> s) & 1u)
        if (!mbar_wait_drain(sm.k_full(s), k_par[s], kDrainNs)) atomicOr(a.status, kStatusDrainFailed);
    for (int s = 0; s < C::kNV; ++s)
      if ((v_issued >> s) & 1u)
        if (!mbar_wait_drain(sm.v_full(s), v_par[s], kDrainNs)) atomicOr(a.status, kStatusDrainFailed);
    if (qn > 0)
      if (!mbar_wait_drain(sm.q_full(), (qn - 1) & 1u, kDrainNs)) atomicOr(a.status, kStatusDrainFailed);
  }
}

// --------------------------------------------------------------------- MMA --
template <int DQK, bool FP8>
__device__ __forceinline__ void issue_s(const Smem<DQK, FP8>& sm, uint32_t tmem_s, int qtile, int kstage) {
  using C = Cfg<DQK, FP8>;
  const uint32_t a_base = smem_u32(sm.q_tile(qtile));
  const uint32_t b_base = smem_u32(sm.k_tile(kstage));
#pragma unroll
  for (int st = 0; st < C::kQkSteps; ++st) {
    const uint32_t off = (st * 32 / 128) * 16384 + (st * 32) % 128;
    const uint64_t ad = smem_desc_sw128(a_base + off, 16, 1024);
    const uint64_t bd = smem_desc_sw128(b_base + off, 16, 1024);
    if constexpr (FP8) mma_ss_f8(tmem_s, ad, bd, C::kIdescS, st > 0 ? 1u : 0u);
    else mma_ss_bf16(tmem_s, ad, bd, C::kIdescS, st > 0 ? 1u : 0u);
  }
}

template <int DQK, bool FP8>
__device__ __forceinline__ void issue_pv(const Smem<DQK, FP8>& sm, uint32_t tmem_p, uint32_t tmem_o, int vstage,
                                         bool accumulate) {
  using C = Cfg<DQK, FP8>;
  const uint32_t b_base = smem_u32(sm.v_tile(vstage));
#pragma unroll
  for (int st = 0; st < C::kPvSteps; ++st) {
    // V is [keys, dv] with dv contiguous: an MN-major B operand. LBO steps
    // between 128-byte dv column blocks, SBO between 8-key row groups.
    const uint64_t bd = smem_desc_sw128(b_base + st * C::kPvStepBytes, 16384, 1024);
    const uint32_t acc = (accumulate || st > 0) ? 1u : 0u;
    if constexpr (FP8) mma_ts_f8(tmem_o, tmem_p + st * 8, bd, C::kIdescPV, acc);
    else mma_ts_bf16(tmem_o, tmem_p + st * 8, bd, C::kIdescPV, acc);
  }
}

template <int DQK, bool FP8>
__device__ void mma_role(const Smem<DQK, FP8>& sm, uint32_t tmem, const AttnArgs& a, int n_qtiles) {
  using C = Cfg<DQK, FP8>;
  const int n_units = a.B * a.Hq * ((n_qtiles + 1) / 2);
  volatile int* abort_flag = sm.abort_flag();
  const uint32_t tS[2] = {tmem, tmem + 128};
  const uint32_t tO[2] = {tmem + 256, tmem + 384};
  int ks = 0, vs = 0;
  uint32_t kph = 0, vph = 0, qn = 0, pph0 = 0, pph1 = 0;
  bool ok = true;
#define ZYFA_WAIT(bar, par)                                                                          \
  if (!(ok = mbar_wait((bar), (par), abort_flag, a.status, kStatusMmaTimeout, a.timeout_ns))) break; \
  tc_fence_after();

  for (int u = blockIdx.x; u < n_units && ok; u += gridDim.x) {
    const Unit w = decode_unit(u, a.B, a.Hq, n_qtiles);
    do {
      ZYFA_WAIT(sm.q_full(), qn & 1u);
      ++qn;
      ZYFA_WAIT(sm.k_full(ks), kph);
      issue_s(sm, tS[0], 0, ks);
      tc_commit(sm.s_full(0));
      if (w.has_b) {
        issue_s(sm, tS[1], 1, ks);
        tc_commit(sm.s_full(1));
      }
      tc_commit(sm.k_empty(ks));
      if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
      if (w.n_kv == 1) tc_commit(sm.q_empty());
      for (int j = 0; j < w.n_kv; ++j) {
        ZYFA_WAIT(sm.v_full(vs), vph);
        bool k_next = false;
        if (j < w.n_a) {
          ZYFA_WAIT(sm.p_full(0), pph0);
          pph0 ^= 1u;
          issue_pv(sm, tS[0], tO[0], vs, j > 0);
          if (j + 1 < w.n_a) {
            ZYFA_WAIT(sm.k_full(ks), kph);
            k_next = true;
            issue_s(sm, tS[0], 0, ks);
            tc_commit(sm.s_full(0));
            if (!w.has_b && j + 1 == w.n_a - 1) tc_commit(sm.q_empty());
          } else {
            tc_commit(sm.o_full(0));
          }
        }
        if (w.has_b) {
          ZYFA_WAIT(sm.p_full(1), pph1);
          pph1 ^= 1u;
          issue_pv(sm, tS[1], tO[1], vs, j > 0);
          if (j + 1 < w.n_b) {
            if (!k_next) {
              ZYFA_WAIT(sm.k_full(ks), kph);
              k_next = true;
            }
            issue_s(sm, tS[1], 1, ks);
            tc_commit(sm.s_full(1));
            if (j + 1 == w.n_b - 1) tc_commit(sm.q_empty());
          } else {
            tc_commit(sm.o_full(1));
          }
        }
        tc_commit(sm.v_empty(vs));
        if (++vs == C::kNV) { vs = 0; vph ^= 1u; }
        if (k_next) {
          tc_commit(sm.k_empty(ks));
          if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
        }
      }
    } while (false);
  }
#undef ZYFA_WAIT
  // Let every issued MMA (and the arrivals of earlier commits) complete.
  tc_commit(sm.drain());
  if (!mbar_wait_drain(sm.drain(), 0, 200000000ull)) atomicOr(a.status, kStatusDrainFailed);
}

// ----------------------------------------------------------------- softmax --
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// Exact sum of four e4m3 codes (bytes of w) scaled by 2^-120: each byte moved
// to bits 20..27 is the float with the same value times 2^-120 (normals and
// subnormals alike), so the fp32 additions of up to 128 such terms are exact.
__device__ __forceinline__ float e4m3x4_sum_scaled(uint32_t w) {
  const float f0 = __uint_as_float((w << 20) & 0x0FF00000u);
  const float f1 = __uint_as_float((w << 12) & 0x0FF00000u);
  const float f2 = __uint_as_float((w << 4) & 0x0FF00000u);
  const float f3 = __uint_as_float((w >> 4) & 0x0FF00000u);
  return __fadd_rn(__fadd_rn(f0, f1), __fadd_rn(f2, f3));
}

__device__ __forceinline__ void rescale_o_row(uint32_t tO, float rho) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tO + 32 * c, r);
#pragma unroll
    for (int e = 0; e < 32; ++e) r[e] = __float_as_uint(u2f(r[e]) * rho);
    tmem_st32(tO + 32 * c, r);
  }
}

template <int DQK, bool FP8>
__device__ void softmax_role(const Smem<DQK, FP8>& sm, uint32_t tmem, const AttnArgs& a, int n_qtiles,
                             int warp, int lane) {
  const int n_units = a.B * a.Hq * ((n_qtiles + 1) / 2);
  const int nblk = n_qtiles;
  const int group = a.Hq / a.Hkv;
  volatile int* abort_flag = sm.abort_flag();
  const int wg = warp >> 2;                      // 0: tile 2t, 1: tile 2t+1
  const int r = (warp & 3) * 32 + lane;          // row within the tile (= TMEM lane)
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + wg * 128 + lane_off;
  const uint32_t tO = tmem + 256 + wg * 128 + lane_off;
  uint32_t sph = 0, oph = 0;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.o);

  for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
    const Unit w = decode_unit(u, a.B, a.Hq, n_qtiles);
    if (wg == 1 && !w.has_b) continue;
    const int qt = 2 * w.t + wg;
    const int n = qt + 1;
    const int hkv = w.hq / group;
    float m = 0.f, l = 0.f, R = 1.f;
    float sq = 1.f;
    const float* ks_row = nullptr;
    const float* vs_row = nullptr;
    if constexpr (FP8) {
      sq = __ldg(a.q_scale + (static_cast<int64_t>(w.b) * a.Hq + w.hq) * nblk + qt);
      ks_row = a.k_scale + (static_cast<int64_t>(w.b) * a.Hkv + hkv) * nblk;
      vs_row = a.v_scale + (static_cast<int64_t>(w.b) * a.Hkv + hkv) * nblk;
    }
    for (int j = 0; j < n; ++j) {
      float sk = 1.f, sv = 1.f;
      if constexpr (FP8) {
        sk = __ldg(ks_row + j);
        sv = __ldg(vs_row + j);
      }
      bool ok = mbar_wait(sm.s_full(wg), sph, abort_flag, a.status, kStatusSoftmaxTimeout, a.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) { *abort_flag = 1; return; }
      sph ^= 1u;
      tc_fence_after();
      uint32_t s[128];
#pragma unroll
      for (int c = 0; c < 4; ++c) tmem_ld32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&s[32 * c]));
      if (j == n - 1) {
#pragma unroll
        for (int c = 0; c < 128; ++c)
          if (c > r) s[c] = 0xff800000u;   // -inf above the diagonal
      }
      float mx = u2f(s[0]);
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, u2f(s[c]));

      if constexpr (!FP8) {
        const float xmax = mx * a.scale_log2;
        float rho = 1.f;
        bool need = false;
        if (j == 0) {
          m = xmax;
        } else if (xmax > m + kRescaleThreshold) {
          rho = ex2_approx(m - xmax);
          m = xmax;
          need = true;
        }
        l *= rho;
        const float neg = -m;
        uint32_t pk[64];
        float l0 = 0.f, l1 = 0.f, l2 = 0.f, l3 = 0.f;
#pragma unroll
        for (int c = 0; c < 64; c += 2) {
          const float p0 = ex2_approx(fmaf(u2f(s[2 * c]), a.scale_log2, neg));
          const float p1 = ex2_approx(fmaf(u2f(s[2 * c + 1]), a.scale_log2, neg));
          const float p2 = ex2_approx(fmaf(u2f(s[2 * c + 2]), a.scale_log2, neg));
          const float p3 = ex2_approx(fmaf(u2f(s[2 * c + 3]), a.scale_log2, neg));
          l0 += p0; l1 += p1; l2 += p2; l3 += p3;
          pk[c] = pack_bf16x2(p0, p1);
          pk[c + 1] = pack_bf16x2(p2, p3);
        }
        l += (l0 + l1) + (l2 + l3);
        tmem_st32(tS, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
        tmem_st32(tS + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
        if (j > 0 && __any_sync(0xffffffffu, need)) rescale_o_row(tO, rho);
      } else {
        const float cj = sq * sk * a.scale_log2;
        const float xmax = mx * cj;
        const float m_new = (j == 0) ? xmax : fmaxf(m, xmax);
        const float kf = fminf(floorf(m_new - xmax), kMaxBlockShift);   // 2^k lifts the tile max into (0.5, 1]
        const int ki = static_cast<int>(kf);
        const float off = m_new - kf;
        uint32_t pk[32];
        float l0 = 0.f, l1 = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float p0 = ex2_approx(fmaf(u2f(s[4 * i]), cj, -off));
          const float p1 = ex2_approx(fmaf(u2f(s[4 * i + 1]), cj, -off));
          const float p2 = ex2_approx(fmaf(u2f(s[4 * i + 2]), cj, -off));
          const float p3 = ex2_approx(fmaf(u2f(s[4 * i + 3]), cj, -off));
          pk[i] = pack_e4m3x4(p0, p1, p2, p3);
          if (i & 1) l1 = __fadd_rn(l1, e4m3x4_sum_scaled(pk[i]));
          else l0 = __fadd_rn(l0, e4m3x4_sum_scaled(pk[i]));
        }
        const float lsum = __fadd_rn(l0, l1);                              // sum of rounded P, times 2^-120
        const float two_m_k = __int_as_float((127 - ki) << 23);           // 2^-k
        const float lift = __int_as_float((127 + 120 - ki) << 23);        // 2^(120-k)
        const float r_new = sv * two_m_k;
        float rho = 1.f;
        if (j == 0) {
          l = lsum * lift;
        } else {
          const float decay = ex2_approx(m - m_new);
          rho = (R / r_new) * decay;
          l = fmaf(l, decay, lsum * lift);
        }
        m = m_new;
        R = r_new;
        tmem_st32(tS, pk);
        if (j > 0) rescale_o_row(tO, rho);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full(wg));
    }

    // epilogue: O / l (FP8: times the accumulator scale R), BF16, global store
    bool ok = mbar_wait(sm.o_full(wg), oph, abort_flag, a.status, kStatusSoftmaxTimeout, a.timeout_ns);
    if (!__all_sync(0xffffffffu, ok)) { *abort_flag = 1; return; }
    oph ^= 1u;
    tc_fence_after();
    const float inv = FP8 ? (R / l) : (1.f / l);
    const int q_row = qt * 128 + r;
    __nv_bfloat16* orow = out + w.b * a.o_sb + static_cast<int64_t>(q_row) * a.o_ss + w.hq * a.o_sh;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      __syncwarp();   // tcgen05.ld is warp-collective; the store below is per-thread
      tmem_ld32(tO + 32 * c, o);
      uint32_t pk[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pk[e] = pack_bf16x2(u2f(o[2 * e]) * inv, u2f(o[2 * e + 1]) * inv);
      if (q_row < a.S) {
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
      }
    }
  }
}

// ------------------------------------------------------------------ kernel --
template <int DQK, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a) {
  using C = Cfg<DQK, FP8>;
  extern __shared__ uint8_t smem_raw[];
  Smem<DQK, FP8> sm;
  sm.base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  sm.bars = reinterpret_cast<uint64_t*>(sm.base + C::kOffBar);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qtiles = (a.S + 127) / 128;

  if (threadIdx.x == 0) {
    mbar_init(sm.q_full(), 1);
    mbar_init(sm.q_empty(), 1);
    for (int s = 0; s < C::kNK; ++s) { mbar_init(sm.k_full(s), 1); mbar_init(sm.k_empty(s), 1); }
    for (int s = 0; s < C::kNV; ++s) { mbar_init(sm.v_full(s), 1); mbar_init(sm.v_empty(s), 1); }
    for (int t = 0; t < 2; ++t) {
      mbar_init(sm.s_full(t), 1);
      mbar_init(sm.p_full(t), 4);   // one arrival per softmax warp
      mbar_init(sm.o_full(t), 1);
    }
    mbar_init(sm.drain(), 1);
    *sm.abort_flag() = 0;
    fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(sm.tmem_slot(), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *sm.tmem_slot();

  if (warp == kLoadWarp) {
    if (lane == 0 && !a.debug_stall) loader_role(sm, &tm_q, &tm_k, &tm_v, a, n_qtiles);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    if (lane == 0) mma_role(sm, tmem, a, n_qtiles);
    __syncwarp();
  } else {
    softmax_role(sm, tmem, a, n_qtiles, warp, lane);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int DQK, bool FP8>
cudaError_t launch(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnArgs& a,
                   cudaStream_t stream) {
  using C = Cfg<DQK, FP8>;
  auto kern = attn_fwd_kernel<DQK, FP8>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
  if (e != cudaSuccess) return e;
  const int n_qtiles = (a.S + 127) / 128;
  const long long n_units = static_cast<long long>(a.B) * a.Hq * ((n_qtiles + 1) / 2);
  const int grid = static_cast<int>(n_units < a.num_sms ? n_units : a.num_sms);
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const AttnArgs& a, cudaStream_t stream) {
  if (a.Dqk == 128) return launch<128, false>(tm_q, tm_k, tm_v, a, stream);
  if (a.Dqk == 192) return launch<192, false>(tm_q, tm_k, tm_v, a, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            const AttnArgs& a, cudaStream_t stream) {
  if (a.Dqk == 128) return launch<128, true>(tm_q, tm_k, tm_v, a, stream);
  if (a.Dqk == 192) return launch<192, true>(tm_q, tm_k, tm_v, a, stream);
  return cudaErrorInvalidValue;
}

}  // namespace zyfa
