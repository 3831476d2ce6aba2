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
#include <cuda_fp16.h>

#include <type_traits>

#include "internal.h"
#include "ptx.cuh"

namespace zyfa {
namespace {

constexpr int kThreads = 384;              // 3 warpgroups: softmax A, softmax B, loaders/MMA
constexpr int kLoadWarp = 8;               // Q and K
constexpr int kMmaWarp = 9;
constexpr int kLoadWarpV = 10;             // V
// Register split per path (launch: 384 x 168 = 64512 registers): the
// softmax warpgroups take kSoftmax and the loader/MMA warpgroup kControl,
// 8*32*kSoftmax + 4*32*kControl <= 64512. Measured on the 32K and 16K
// workloads: 208/88 (FP8 and BF16) beats both the even split and
// starving the control warps (which then spill inside the MMA issue loop).
template <bool FP8>
struct RegSplit {
  static constexpr uint32_t kSoftmax = 208;
  static constexpr uint32_t kControl = 88;
  static_assert(8 * 32 * kSoftmax + 4 * 32 * kControl <= 384 * 168, "register split exceeds the launch");
};
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleThreshold = 8.0f;   // BF16: keep a stale max while x - m <= 8

enum StatusCode : unsigned int {
  kStatusLoaderTimeout = 0x1u,
  kStatusMmaTimeout = 0x2u,
  kStatusSoftmaxTimeout = 0x4u,
  kStatusDrainFailed = 0x100u,
};

// Optional timeline trace for performance work (compile with -DZYFA_TRACE):
// CTA 0 records (clock64 << 8 | event) per role into a device buffer that
// zyfa_trace_read() copies out. Not part of the normal build.
#ifdef ZYFA_TRACE
constexpr int kTraceLen = 8192;
__device__ unsigned long long zyfa_trace_buf[4][kTraceLen];
__device__ __forceinline__ void trace_ev(int role, uint32_t& idx, uint32_t code) {
  if (blockIdx.x == 0 && idx < kTraceLen) zyfa_trace_buf[role][idx++] = (clock64() << 8) | code;
}
#define ZTRACE(role, idx, code) trace_ev(role, idx, code)
#else
#define ZTRACE(role, idx, code) \
  do {                          \
  } while (0)
#endif

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
  // Q/K rows of whole 128-byte blocks load as one 5-D request per tile; e4m3
  // at head dim 192 (1.5 blocks) as one 4-D box per block.
  static constexpr bool kQkWhole = (kQkRowBytes % 128) == 0;
  // MMA order per key tile: PV_A, S_A(next), PV_B, S_B(next) (default), or
  // PV_A, PV_B, S_A(next), S_B(next) where a single V stage fits (bf16, 192).
  static constexpr bool kLateS = !FP8 && DQK == 192;
  // Ring depths (K and V stages of 128 keys).
  static constexpr int kNK = FP8 ? (DQK == 128 ? 4 : 3) : 2;
  static constexpr int kNV = FP8 ? (DQK == 128 ? 6 : 4) : (DQK == 128 ? 3 : 1);
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
  int b, hq, t;            // batch coordinate of the maps (0 for packed input), query head, pair
  bool has_b;
  int n_a, n_b, n_kv;
  int c0, dlt;             // paged K/V: cached tokens before the first query row = 128 c0 + dlt (else 0)
  int j0;                  // decode step: first key block of the task (split key range), else 0
  int part;                // decode step with split key ranges: partial-result row of the task, else -1
  int row0;                // first token of the sequence in the token dimension
  int len;                 // tokens of the sequence
  int sidx;                // sequence index of the scale arrays
};

// Work order. The (batch, KV head) groups are taken `gif` at a time (the
// host picks gif, AttnArgs::groups_in_flight); inside such a super-group the
// longest query-tile pairs come first and, for each pair, the groups and then
// their query heads are adjacent. Units in flight then share a few KV heads
// (K/V stay in L2) without every CTA streaming the very same K/V tile at once.

// Pairs pair_lo .. pair_hi - 1 only (a row range of a chunked prefill).
__device__ __forceinline__ Unit decode_unit(int u, int B, int Hq, int Hkv, int n_qtiles, int pair_lo, int pair_hi,
                                            int gif) {
  const int n_pairs = pair_hi - pair_lo;
  const int G = Hq / Hkv;
  const int n_groups = B * Hkv;
  const int per_sg = gif * G * n_pairs;
  const int sg = u / per_sg;
  const int r = u - sg * per_sg;
  const int gs_here = min(gif, n_groups - sg * gif);
  const int per_t = gs_here * G;
  const int tq = r / per_t;
  const int rr = r - tq * per_t;
  const int gi = rr / G;
  const int group = sg * gif + gi;
  Unit w;
  w.b = group / Hkv;
  const int hkv = group - w.b * Hkv;
  w.t = pair_hi - 1 - tq;
  w.hq = hkv * G + (rr - gi * G);
  w.has_b = (2 * w.t + 1) < n_qtiles;
  w.n_a = 2 * w.t + 1;
  w.n_b = 2 * w.t + 2;
  w.n_kv = w.has_b ? w.n_b : w.n_a;
  w.c0 = 0;
  w.dlt = 0;
  w.j0 = 0;
  w.part = -1;
  w.row0 = 0;
  w.sidx = w.b;
  return w;
}

// Unit lists. Equal lengths: B * Hq * pairs units decoded arithmetically
// (decode_unit). Packed variable lengths: the host-built level table.
struct NoTable {};

// PART: the kernel instantiation's units write partial rows (unnormalised
// O and the row's offset or maximum and sum) that a second kernel combines.
// Packed batches: decode steps (one query token per sequence, key ranges
// split across units); prefill instantiations compile none of that code.
// Equal lengths: query-tile pairs whose key blocks are split into chunks of
// split_tiles blocks (small grids, where pairs alone leave SMs idle).
template <bool VARLEN, bool PART = false, bool LIST = false>
struct Sched {
  using Table = typename std::conditional<VARLEN, SeqTable, NoTable>::type;
  const Table* tab;
  int B, Hq, Hkv, S, n_qtiles, pair_lo, pair_hi;
  int groups_in_flight;    // equal lengths: KV groups per super-group of the work order
  bool one_token;          // decode step: one query token per sequence, its heads as tile rows (PART only)
  __device__ __forceinline__ bool step() const { return VARLEN && PART && one_token; }
  // This CTA's units: LIST, the host's list (equal lengths, more than one
  // wave); else units blockIdx.x, blockIdx.x + gridDim.x, ... below nu.
  // Walked as u = first(); u >= 0; u = next(++i, u).
  const UnitList* list;
  int nu;                  // n_units(), computed once
  __device__ __forceinline__ int first() const {
    if constexpr (LIST) return list->start[blockIdx.x + 1] > list->start[blockIdx.x] ? list->unit[list->start[blockIdx.x]] : -1;
    else return static_cast<int>(blockIdx.x) < nu ? static_cast<int>(blockIdx.x) : -1;
  }
  __device__ __forceinline__ int next(int i, int u) const {
    if constexpr (LIST) {
      const int b = list->start[blockIdx.x];
      return b + i < list->start[blockIdx.x + 1] ? list->unit[b + i] : -1;
    } else {
      return u + static_cast<int>(gridDim.x) < nu ? u + static_cast<int>(gridDim.x) : -1;
    }
  }
  int split_tiles;         // nonzero when key ranges are split (decode: per-sequence split counts in tab;
                           // equal lengths: key blocks per chunk, even)
  // Equal lengths with split key ranges: pairs are taken longest first, each
  // as ceil(key blocks / split_tiles) chunks, each chunk for every (batch,
  // query head). Tile A of a chunk always has a key block: split_tiles is
  // even and so is tile B's key count.
  __device__ __forceinline__ int pair_chunks(int t) const {
    const int nk = (2 * t + 1 < n_qtiles) ? 2 * t + 2 : 2 * t + 1;
    return (nk + split_tiles - 1) / split_tiles;
  }
  __device__ __forceinline__ int split_units() const {
    int n = 0;
    for (int t = pair_lo; t < pair_hi; ++t) n += pair_chunks(t);
    return n * B * Hq;
  }
  __device__ __forceinline__ Unit decode_split(int u) const {
    int rem = u, t = pair_hi - 1, nch = 0;
    for (; t > pair_lo; --t) {
      nch = pair_chunks(t) * B * Hq;
      if (rem < nch) break;
      rem -= nch;
    }
    const int c = rem / (B * Hq), bh = rem - c * (B * Hq);
    Unit w;
    w.b = bh / Hq;
    w.hq = bh - w.b * Hq;
    w.t = t;
    w.has_b = (2 * t + 1) < n_qtiles;
    w.j0 = c * split_tiles;
    w.n_a = min(split_tiles, 2 * t + 1 - w.j0);
    w.n_b = w.has_b ? min(split_tiles, 2 * t + 2 - w.j0) : 0;
    w.n_kv = w.has_b ? w.n_b : w.n_a;
    w.c0 = 0;
    w.dlt = 0;
    w.part = c;
    w.row0 = 0;
    w.len = S;
    w.sidx = w.b;
    return w;
  }
  __device__ __forceinline__ int n_tasks() const {
    return split_tiles ? tab->level_start[tab->n_seqs] : tab->n_seqs * Hkv;
  }
  __device__ __forceinline__ int n_units() const {
    if constexpr (VARLEN) return step() ? (n_tasks() + 1) / 2 : tab->level_start[tab->n_levels];
    else if constexpr (PART) return split_units();
    else return B * Hq * (pair_hi - pair_lo);
  }
  // Decode step: task i = (sequence of rank i / Hkv, KV head i % Hkv), the
  // sequences longest first and KV heads adjacent; unit u runs tasks 2u (as
  // tile A) and 2u + 1 (as tile B), each with its own K/V stream. With split
  // key ranges a sequence of rank k owns tasks level_start[k] ..
  // level_start[k+1] - 1, split-major (split s, head h at s * Hkv + h); its
  // key blocks are cut into that many nearly equal splits, split s writing
  // partial row ctx[k] + s.
  __device__ __forceinline__ Unit decode_task(int i, bool second) const {
    int rank, s = 0;
    if (split_tiles) {
      int lo = 0, hi = tab->n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab->level_start[mid] <= i) lo = mid; else hi = mid - 1;
      }
      rank = lo;
      i -= tab->level_start[rank];
      s = i / Hkv;
      i -= s * Hkv;
    } else {
      rank = i / Hkv;
      i -= rank * Hkv;
    }
    Unit w;
    w.b = 0;
    w.hq = i * (Hq / Hkv);        // first query head of the group: tile row 0
    w.t = 0;
    w.row0 = tab->start[rank];    // the token's row in the packed queries
    w.len = tab->len[rank];       // keys, the new token's included
    w.sidx = tab->index[rank];
    w.c0 = 0;
    w.dlt = 0;
    w.has_b = second;
    const int n_all = (w.len + 127) >> 7;
    if (split_tiles) {
      // the sequence's n_all key blocks in S nearly equal splits
      const int S = (tab->level_start[rank + 1] - tab->level_start[rank]) / Hkv;
      const int base = n_all / S, rem = n_all - base * S;
      w.j0 = s * base + min(s, rem);
      w.n_a = w.n_b = w.n_kv = base + (s < rem ? 1 : 0);
      w.part = tab->ctx[rank] + s;
    } else {
      w.j0 = 0;
      w.n_a = w.n_b = w.n_kv = n_all;
      w.part = -1;
    }
    return w;
  }
  // Tile B of a decode unit (call only when decode(u).has_b).
  __device__ __forceinline__ Unit decode_b(int u) const { return decode_task(2 * u + 1, true); }
  __device__ __forceinline__ Unit decode(int u) const {
    if constexpr (VARLEN) {
      if (step()) return decode_task(2 * u, 2 * u + 1 < n_tasks());
      // level k: the largest with level_start[k] <= u
      int lo = 0, hi = tab->n_levels - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (tab->level_start[mid] <= u) lo = mid; else hi = mid - 1;
      }
      const int r = u - tab->level_start[lo];
      const int rank = r / Hq;
      Unit w;
      w.b = 0;
      w.hq = r - rank * Hq;
      w.t = tab->n_levels - 1 - lo;
      w.row0 = tab->start[rank];
      w.len = tab->len[rank];
      w.sidx = tab->index[rank];
      const int ctx = tab->ctx[rank];
      w.j0 = 0;
      w.part = -1;
      w.c0 = ctx >> 7;
      w.dlt = ctx & 127;
      const int nq = (w.len + 127) / 128;
      w.has_b = (2 * w.t + 1) < nq;
      // Query tile i (positions ctx + 128 i ..) sees key blocks 0 .. c0 + i,
      // and c0 + i + 1 when the prefix ends inside a block, up to the
      // sequence's last block.
      const int nk = (ctx + w.len + 127) >> 7;
      const int ext = w.dlt ? 1 : 0;
      w.n_a = min(w.c0 + 2 * w.t + 1 + ext, nk);
      w.n_b = min(w.c0 + 2 * w.t + 2 + ext, nk);
      w.n_kv = w.has_b ? w.n_b : w.n_a;
      return w;
    } else if constexpr (PART) {
      return decode_split(u);
    } else {
      Unit w = decode_unit(u, B, Hq, Hkv, n_qtiles, pair_lo, pair_hi, groups_in_flight);
      w.len = S;
      return w;
    }
  }
};

template <int DQK, bool FP8>
struct Smem {
  using C = Cfg<DQK, FP8>;
  // Shared-window address of the 1024-byte aligned base: one 32-bit value;
  // the generic pointers below are formed from it where they are used.
  uint32_t sb;
  __device__ __forceinline__ uint8_t* at(uint32_t off) const {
    return static_cast<uint8_t*>(__cvta_shared_to_generic(static_cast<size_t>(sb + off)));
  }
  __device__ __forceinline__ uint64_t* bar(int i) const {
    return reinterpret_cast<uint64_t*>(at(C::kOffBar + 8u * static_cast<uint32_t>(i)));
  }
  __device__ __forceinline__ uint64_t* q_full() const { return bar(0); }
  __device__ __forceinline__ uint64_t* q_empty() const { return bar(1); }
  __device__ __forceinline__ uint64_t* k_full(int s) const { return bar(2 + s); }
  __device__ __forceinline__ uint64_t* k_empty(int s) const { return bar(2 + C::kNK + s); }
  __device__ __forceinline__ uint64_t* v_full(int s) const { return bar(2 + 2 * C::kNK + s); }
  __device__ __forceinline__ uint64_t* v_empty(int s) const { return bar(2 + 2 * C::kNK + C::kNV + s); }
  __device__ __forceinline__ uint64_t* s_full(int t) const { return bar(2 + 2 * C::kNK + 2 * C::kNV + t); }
  __device__ __forceinline__ uint64_t* p_full(int t) const { return s_full(2 + t); }
  __device__ __forceinline__ uint64_t* o_full(int t) const { return s_full(4 + t); }
  __device__ __forceinline__ uint64_t* drain() const { return s_full(6); }
  __device__ __forceinline__ uint32_t* tmem_slot() const { return reinterpret_cast<uint32_t*>(bar(C::kNumBars)); }
  __device__ __forceinline__ volatile int* abort_flag() const {
    return reinterpret_cast<volatile int*>(bar(C::kNumBars)) + 1;
  }
  __device__ __forceinline__ uint8_t* q_tile(int t) const { return at(C::kOffQ + t * C::kQkTileBytes); }
  __device__ __forceinline__ uint8_t* k_tile(int s) const { return at(C::kOffK + s * C::kQkTileBytes); }
  __device__ __forceinline__ uint8_t* v_tile(int s) const { return at(C::kOffV + s * C::kVTileBytes); }
};

// Warp-wide bounded wait: every lane polls; the result is uniform.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* status, unsigned int code, uint64_t timeout_ns) {
  const bool ok = mbar_wait(bar, parity, abort_flag, status, code, timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// Warp-wide bounded wait on two barriers at once (one poll loop, one vote):
// each wait costs the MMA warp a fixed overhead during which the tensor pipe
// drains, so the two TMA barriers of an iteration share one. The abort flag
// and the clock are read every 64 polls, as in mbar_wait.
__device__ __forceinline__ bool warp_wait2(uint64_t* bar1, uint32_t par1, uint64_t* bar2, uint32_t par2,
                                           volatile int* abort_flag, unsigned int* status, unsigned int code,
                                           uint64_t timeout_ns) {
  bool ok1 = mbar_try_wait(bar1, par1), ok2 = mbar_try_wait(bar2, par2);
  if (!(ok1 && ok2)) {
    const uint64_t t0 = global_timer_ns();
    for (uint32_t it = 1;; ++it) {
      if (!ok1) ok1 = mbar_try_wait(bar1, par1);
      if (!ok2) ok2 = mbar_try_wait(bar2, par2);
      if (ok1 && ok2) break;
      if ((it & 63u) == 0) {
        if (*abort_flag) break;
        if (global_timer_ns() - t0 > timeout_ns) {
          *abort_flag = 1;
          if (status) atomicOr(status, code);
          break;
        }
      }
    }
  }
  return __all_sync(0xffffffffu, ok1 && ok2);
}

// ------------------------------------------------------------------ loader --
// Two loader warps: one streams Q and K, the other V. A thread's TMA copies
// are processed one after another at a roughly fixed cost per request (one
// 16 KB box takes ~430 cycles however deep the ring is), so each tile, all
// of its 128-byte column blocks, is one request of a 5-D map, and two
// issuing warps double the rate. Each warp runs its loop uniformly (addresses
// and coordinates stay warp-uniform); one elected lane issues the TMA copies
// and the expect-tx arrivals.
enum LoadStream { kStreamQK = 0, kStreamV = 1 };

template <int DQK, bool FP8, int STREAM, bool VARLEN, bool SLICE, bool PART, bool LIST>
__device__ void loader_role(const Smem<DQK, FP8>& sm, const CUtensorMap* tm_q, const CUtensorMap* tm_kv,
                            const AttnArgs& a, const Sched<VARLEN, PART, LIST>& sc, bool leader) {
  using C = Cfg<DQK, FP8>;
  constexpr bool kIsK = (STREAM == kStreamQK);
  constexpr int kStages = kIsK ? C::kNK : C::kNV;
  constexpr uint32_t kTileBytes = kIsK ? C::kQkTileBytes : C::kVTileBytes;
  const int group = a.Hq / a.Hkv;
  const int lane = threadIdx.x & 31;
  volatile int* abort_flag = sm.abort_flag();
  int st = 0;
  uint32_t ph = 0, qn = 0;
  uint32_t issued = 0;        // stages written at least once
  uint32_t par = 0;           // parity bit of each stage's last issue
  bool ok = true;
  uint32_t tix = 0;
  (void)tix;
  auto full = [&](int i) { return kIsK ? sm.k_full(i) : sm.v_full(i); };
  auto empty = [&](int i) { return kIsK ? sm.k_empty(i) : sm.v_empty(i); };
  auto tile = [&](int i) { return kIsK ? sm.k_tile(i) : sm.v_tile(i); };
  for (int i = 0, u = sc.first(); u >= 0 && ok; u = sc.next(++i, u)) {
    const Unit w = sc.decode(u);
    const int hkv = w.hq / group;
    if constexpr (kIsK) {
      if (!(ok = warp_wait(sm.q_empty(), (qn & 1u) ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)))
        break;
      if (leader) {
        mbar_arrive_expect_tx(sm.q_full(), (w.has_b ? 2 : 1) * C::kQkTileBytes);
        for (int qt = 0; qt < (w.has_b ? 2 : 1); ++qt) {
          int row = w.row0 + (2 * w.t + qt) * 128, qh = w.hq;
          if constexpr (VARLEN) {
            // decode step: the map is over (token, head) rows; a group's
            // heads are consecutive rows; tile B holds the second task
            if (sc.step()) {
              const Unit x = qt ? sc.decode_b(u) : w;
              row = x.row0 * a.Hq + x.hq;
              qh = 0;
            }
          }
          if constexpr (SLICE) {
            // the group's rows four times, at tile rows 0, 32, 64, 96
            // (32-row boxes per 128-byte column block)
            for (int cpy = 0; cpy < 4; ++cpy)
#pragma unroll
              for (int kb = 0; kb < C::kQkBlocks; ++kb)
                tma_load_4d(sm.q_tile(qt) + kb * 16384 + cpy * 4096, tm_q, sm.q_full(), kb * C::kInnerElts, 0, row, 0);
            continue;
          }
          if constexpr (C::kQkWhole) {
            tma_load_5d(sm.q_tile(qt), tm_q, sm.q_full(), 0, row, 0, qh, w.b);
          } else {
#pragma unroll
            for (int kb = 0; kb < C::kQkBlocks; ++kb)
              tma_load_4d(sm.q_tile(qt) + kb * 16384, tm_q, sm.q_full(), kb * C::kInnerElts, qh, row, w.b);
          }
        }
      }
      ++qn;
    }
    if constexpr (VARLEN) {
      if (sc.step()) {
        // Decode step: the two tasks' key blocks alternate in the ring
        // (A0, B0, A1, B1, ...; a finished task drops out), the order in
        // which the MMA warp consumes them.
        const Unit wb = w.has_b ? sc.decode_b(u) : w;
        const int na = w.n_kv, nb = w.has_b ? wb.n_kv : 0;
        int pg[2] = {0, 0};
        for (int j = 0; j < max(na, nb) && ok; ++j) {
          for (int x = 0; x < 2; ++x) {
            const Unit& wx = x ? wb : w;
            if (j >= (x ? nb : na)) continue;
            if ((j & 31) == 0) {
              const int e = j + lane;
              pg[x] = e < wx.n_kv ? __ldg(a.block_table + wx.sidx * a.bt_stride + wx.j0 + e) : 0;
            }
            const int page = __shfl_sync(0xffffffffu, pg[x], j & 31);
            if (leader && (page < 0 || page >= a.num_pages)) atomicOr(a.status, kStatusBadPage);
            if (!(ok = warp_wait(empty(st), ph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)))
              break;
            if (leader) {
              mbar_arrive_expect_tx(full(st), kTileBytes);
              const int hx = wx.hq / group;
              if constexpr (!kIsK || C::kQkWhole) {
                tma_load_5d(tile(st), tm_kv, full(st), 0, 0, 0, hx, page);
              } else {
#pragma unroll
                for (int kb = 0; kb < C::kQkBlocks; ++kb)
                  tma_load_4d(tile(st) + kb * 16384, tm_kv, full(st), kb * C::kInnerElts, hx, 0, page);
              }
            }
            par = (par & ~(1u << st)) | (ph << st);
            issued |= 1u << st;
            if (++st == kStages) { st = 0; ph ^= 1u; }
          }
        }
        continue;
      }
    }
    int pages = 0;   // paged K/V: block-table entries j & ~31 .. + 31, one per lane
    for (int j = 0; j < w.n_kv; ++j) {
      // Key block j: tokens row0 + 128 j of batch b, or all 128 tokens of its page.
      // (equal lengths with split key ranges: the chunk starts at block j0)
      int kv_row = w.row0 + ((!VARLEN && PART) ? w.j0 + j : j) * 128, kv_b = w.b;
      if constexpr (VARLEN) {
        if (a.block_table) {
          if ((j & 31) == 0) {
            const int e = j + lane;
            pages = e < w.n_kv ? __ldg(a.block_table + w.sidx * a.bt_stride + e) : 0;
          }
          kv_b = __shfl_sync(0xffffffffu, pages, j & 31);
          kv_row = 0;
          if (leader && (kv_b < 0 || kv_b >= a.num_pages)) atomicOr(a.status, kStatusBadPage);
        }
      }
      if (leader) ZTRACE(3, tix, kIsK ? 20 : 22);
      if (!(ok = warp_wait(empty(st), ph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns))) break;
      if (leader) {
        ZTRACE(3, tix, kIsK ? 21 : 23);
        mbar_arrive_expect_tx(full(st), kTileBytes);
        if constexpr (!kIsK || C::kQkWhole) {
          tma_load_5d(tile(st), tm_kv, full(st), 0, kv_row, 0, hkv, kv_b);
        } else {
#pragma unroll
          for (int kb = 0; kb < C::kQkBlocks; ++kb)
            tma_load_4d(tile(st) + kb * 16384, tm_kv, full(st), kb * C::kInnerElts, hkv, kv_row, kv_b);
        }
      }
      par = (par & ~(1u << st)) | (ph << st);
      issued |= 1u << st;
      if (++st == kStages) { st = 0; ph ^= 1u; }
    }
  }
  if (ok) {
    // Tail: wait until every stage has been released for the last time, so
    // no tcgen05.commit arrival is still in flight when the CTA exits.
    for (int i = 0; i < kStages; ++i) {
      if (!warp_wait(empty(st), ph ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns)) break;
      if (++st == kStages) { st = 0; ph ^= 1u; }
    }
    if constexpr (kIsK) warp_wait(sm.q_empty(), (qn & 1u) ^ 1u, abort_flag, a.status, kStatusLoaderTimeout, a.timeout_ns);
  } else if (leader) {
    // Abort: let every copy this warp issued land before the CTA exits.
    constexpr uint64_t kDrainNs = 200000000ull;
    for (int i = 0; i < kStages; ++i)
      if ((issued >> i) & 1u)
        if (!mbar_wait_drain(full(i), (par >> i) & 1u, kDrainNs)) atomicOr(a.status, kStatusDrainFailed);
    if (kIsK && qn > 0)
      if (!mbar_wait_drain(sm.q_full(), (qn - 1) & 1u, kDrainNs)) atomicOr(a.status, kStatusDrainFailed);
  }
}

// --------------------------------------------------------------------- MMA --
// Operand descriptors are precomputed per buffer (Q tiles, K stages, V
// stages are at fixed offsets); a K step only adds a constant to the low word.
struct OperandDescs {
  Desc q0;        // Q tile 0; tile 1 is kQkTileBytes further
  Desc k0;        // K stage 0; stage s is s * kQkTileBytes further
  Desc v0;        // V stage 0; stage s is s * kVTileBytes further
};

template <int DQK, bool FP8>
__device__ __forceinline__ void issue_s(const OperandDescs& od, uint32_t tmem_s, int qtile, int kstage) {
  using C = Cfg<DQK, FP8>;
  const uint32_t alo = od.q0.lo + static_cast<uint32_t>(qtile) * (C::kQkTileBytes >> 4);
  const uint32_t blo = od.k0.lo + static_cast<uint32_t>(kstage) * (C::kQkTileBytes >> 4);
#pragma unroll
  for (int st = 0; st < C::kQkSteps; ++st) {
    const uint32_t adv = static_cast<uint32_t>(((st * 32 / 128) * 16384 + (st * 32) % 128) >> 4);
    if constexpr (FP8) mma_ss_f8_h(tmem_s, alo + adv, od.q0.hi, blo + adv, od.k0.hi, C::kIdescS, st > 0 ? 1u : 0u);
    else mma_ss_bf16_h(tmem_s, alo + adv, od.q0.hi, blo + adv, od.k0.hi, C::kIdescS, st > 0 ? 1u : 0u);
  }
}

template <int DQK, bool FP8>
__device__ __forceinline__ void issue_pv(const OperandDescs& od, uint32_t tmem_p, uint32_t tmem_o, int vstage,
                                         bool accumulate) {
  using C = Cfg<DQK, FP8>;
  // V is [keys, dv] with dv contiguous: an MN-major B operand. LBO steps
  // between 128-byte dv column blocks, SBO between 8-key row groups.
  const uint32_t blo = od.v0.lo + static_cast<uint32_t>(vstage) * (C::kVTileBytes >> 4);
#pragma unroll
  for (int st = 0; st < C::kPvSteps; ++st) {
    const uint32_t acc = (accumulate || st > 0) ? 1u : 0u;
    const uint32_t adv = static_cast<uint32_t>((st * C::kPvStepBytes) >> 4);
    if constexpr (FP8) mma_ts_f8_h(tmem_o, tmem_p + st * 8, blo + adv, od.v0.hi, C::kIdescPV, acc);
    else mma_ts_bf16_h(tmem_o, tmem_p + st * 8, blo + adv, od.v0.hi, C::kIdescPV, acc);
  }
}

// The whole warp runs the schedule (waits, stage and phase bookkeeping,
// descriptors: all warp-uniform); one elected lane issues tcgen05.mma and
// tcgen05.commit, so a commit tracks exactly the MMAs of that lane.
template <int DQK, bool FP8, bool VARLEN, bool PART, bool LIST>
__device__ void mma_role(const Smem<DQK, FP8>& sm, uint32_t tmem, const AttnArgs& a, const Sched<VARLEN, PART, LIST>& sc,
                         bool leader) {
  using C = Cfg<DQK, FP8>;
  volatile int* abort_flag = sm.abort_flag();
  const uint32_t tS0 = tmem, tS1 = tmem + 128;
  const uint32_t tO0 = tmem + 256, tO1 = tmem + 384;
  int ks = 0, vs = 0;
  uint32_t kph = 0, vph = 0, qn = 0, pph0 = 0, pph1 = 0;
  bool ok = true;
  OperandDescs od;
  od.q0 = make_desc_sw128(smem_u32(sm.q_tile(0)), 16, 1024);
  od.k0 = make_desc_sw128(smem_u32(sm.k_tile(0)), 16, 1024);
  od.v0 = make_desc_sw128(smem_u32(sm.v_tile(0)), 16384, 1024);
  uint32_t tix = 0;
  (void)tix;
// Waits on TMA barriers need no tcgen05 fence (the mbarrier orders the copy
// before the MMA's shared-memory reads); waits on P (written to tensor memory
// by the softmax warps with tcgen05.st) are followed by
// tcgen05.fence::after_thread_sync.
#define ZYFA_WAIT(bar, par) \
  if (!(ok = warp_wait((bar), (par), abort_flag, a.status, kStatusMmaTimeout, a.timeout_ns))) break;
#define ZYFA_WAIT_P(bar, par)                                                                         \
  if (!(ok = warp_wait((bar), (par), abort_flag, a.status, kStatusMmaTimeout, a.timeout_ns))) break; \
  tc_fence_after();

  for (int i = 0, u = sc.first(); u >= 0 && ok; u = sc.next(++i, u)) {
    const Unit w = sc.decode(u);
    do {
      ZYFA_WAIT(sm.q_full(), qn & 1u);
      ++qn;
      if constexpr (VARLEN) {
        if (sc.step()) {
          // Decode step: tasks A and B of the unit are independent chains
          // (own K/V blocks, interleaved in the rings), ping-ponged like two
          // query tiles: S_A(0), S_B(0), then per block PV_X(j), S_X(j+1).
          const int na = w.n_kv, nb = w.has_b ? sc.decode_b(u).n_kv : 0;
          const int n_s = na + nb;        // S products of the unit; Q is free after the last
          int s_done = 0;
          for (int x = 0; x < 2; ++x) {
            if ((x ? nb : na) == 0) continue;
            ZYFA_WAIT(sm.k_full(ks), kph);
            if (leader) {
              issue_s<DQK, FP8>(od, x ? tS1 : tS0, x, ks);
              tc_commit(sm.s_full(x));
              tc_commit(sm.k_empty(ks));
              if (++s_done == n_s) tc_commit(sm.q_empty());
            } else {
              ++s_done;
            }
            if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
          }
          if (!ok) break;
          for (int j = 0; j < max(na, nb) && ok; ++j) {
            for (int x = 0; x < 2; ++x) {
              const int nx = x ? nb : na;
              if (j >= nx) continue;
              ZYFA_WAIT(sm.v_full(vs), vph);
              if (x) {
                ZYFA_WAIT_P(sm.p_full(1), pph1);
                pph1 ^= 1u;
              } else {
                ZYFA_WAIT_P(sm.p_full(0), pph0);
                pph0 ^= 1u;
              }
              if (leader) {
                issue_pv<DQK, FP8>(od, x ? tS1 : tS0, x ? tO1 : tO0, vs, j > 0);
                if (j + 1 == nx) tc_commit(sm.o_full(x));
                tc_commit(sm.v_empty(vs));
              }
              if (++vs == C::kNV) { vs = 0; vph ^= 1u; }
              if (j + 1 < nx) {
                ZYFA_WAIT(sm.k_full(ks), kph);
                if (leader) {
                  issue_s<DQK, FP8>(od, x ? tS1 : tS0, x, ks);
                  tc_commit(sm.s_full(x));
                  tc_commit(sm.k_empty(ks));
                  if (++s_done == n_s) tc_commit(sm.q_empty());
                } else {
                  ++s_done;
                }
                if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
              }
            }
          }
          break;
        }
      }
      ZYFA_WAIT(sm.k_full(ks), kph);
      if (leader) ZTRACE(2, tix, 26);
      if (leader) {
        issue_s<DQK, FP8>(od, tS0, 0, ks);
        tc_commit(sm.s_full(0));
        if (w.has_b) {
          issue_s<DQK, FP8>(od, tS1, 1, ks);
          tc_commit(sm.s_full(1));
        }
        tc_commit(sm.k_empty(ks));
        if (w.n_kv == 1) tc_commit(sm.q_empty());
      }
      if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
      // The tensor pipe accepts about one MMA ahead of execution, so the
      // issuing thread runs in step with it: every wait is done before a
      // contiguous PV -> S issue block, never between two GEMMs.
      for (int j = 0; j < w.n_kv; ++j) {
        const bool need_k = (j + 1 < w.n_kv);      // K_{j+1} feeds S_A(j+1) and/or S_B(j+1)
        if (leader) ZTRACE(2, tix, 10);
#ifdef ZYFA_TRACE
        if (leader)
          ZTRACE(2, tix, 40 + (mbar_test(sm.v_full(vs), vph) ? 1 : 0) + (!need_k || mbar_test(sm.k_full(ks), kph) ? 2 : 0));
#endif
        if (need_k) {
          if (!(ok = warp_wait2(sm.v_full(vs), vph, sm.k_full(ks), kph, abort_flag, a.status, kStatusMmaTimeout,
                                a.timeout_ns)))
            break;
        } else {
          ZYFA_WAIT(sm.v_full(vs), vph);
        }
        if (leader) ZTRACE(2, tix, 11);
        if constexpr (C::kLateS) {
          // Both PV products of V(j) first, then both next S: V(j) is
          // released before the two S products run, which hides the load of
          // V(j+1) behind them when shared memory holds a single V stage.
          if (j < w.n_a) {
            ZYFA_WAIT_P(sm.p_full(0), pph0);
            pph0 ^= 1u;
            if (leader) {
              issue_pv<DQK, FP8>(od, tS0, tO0, vs, j > 0);
              if (j + 1 >= w.n_a) tc_commit(sm.o_full(0));
            }
          }
          if (w.has_b) {
            ZYFA_WAIT_P(sm.p_full(1), pph1);
            pph1 ^= 1u;
            if (leader) {
              issue_pv<DQK, FP8>(od, tS1, tO1, vs, j > 0);
              if (j + 1 >= w.n_b) tc_commit(sm.o_full(1));
            }
          }
          if (leader) {
            tc_commit(sm.v_empty(vs));
            if (j + 1 < w.n_a) {
              issue_s<DQK, FP8>(od, tS0, 0, ks);
              tc_commit(sm.s_full(0));
              if (!w.has_b && j + 1 == w.n_a - 1) tc_commit(sm.q_empty());
            }
            if (w.has_b && j + 1 < w.n_b) {
              issue_s<DQK, FP8>(od, tS1, 1, ks);
              tc_commit(sm.s_full(1));
              if (j + 1 == w.n_b - 1) tc_commit(sm.q_empty());
            }
          }
          if (++vs == C::kNV) { vs = 0; vph ^= 1u; }
          if (need_k) {
            if (leader) tc_commit(sm.k_empty(ks));
            if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
          }
          continue;
        }
        if (j < w.n_a) {
          if (leader) ZTRACE(2, tix, 12);
          ZYFA_WAIT_P(sm.p_full(0), pph0);
          if (leader) ZTRACE(2, tix, 13);
          pph0 ^= 1u;
          if (leader) {
            issue_pv<DQK, FP8>(od, tS0, tO0, vs, j > 0);
            if (j + 1 < w.n_a) {
              issue_s<DQK, FP8>(od, tS0, 0, ks);
              tc_commit(sm.s_full(0));
              if (!w.has_b && j + 1 == w.n_a - 1) tc_commit(sm.q_empty());
            } else {
              tc_commit(sm.o_full(0));
            }
          }
          if (leader) ZTRACE(2, tix, 14);
        }
        if (w.has_b) {
          if (leader) ZTRACE(2, tix, 15);
          ZYFA_WAIT_P(sm.p_full(1), pph1);
          if (leader) ZTRACE(2, tix, 16);
          pph1 ^= 1u;
          if (leader) {
            issue_pv<DQK, FP8>(od, tS1, tO1, vs, j > 0);
            if (j + 1 < w.n_b) {
              issue_s<DQK, FP8>(od, tS1, 1, ks);
              tc_commit(sm.s_full(1));
              if (j + 1 == w.n_b - 1) tc_commit(sm.q_empty());
            } else {
              tc_commit(sm.o_full(1));
            }
          }
          if (leader) ZTRACE(2, tix, 17);
        }
        if (leader) tc_commit(sm.v_empty(vs));
        if (++vs == C::kNV) { vs = 0; vph ^= 1u; }
        if (need_k) {
          if (leader) tc_commit(sm.k_empty(ks));
          if (++ks == C::kNK) { ks = 0; kph ^= 1u; }
        }
      }
    } while (false);
  }
#undef ZYFA_WAIT
#undef ZYFA_WAIT_P
  // Let every issued MMA (and the arrivals of earlier commits) complete.
  if (leader) {
    tc_commit(sm.drain());
    if (!mbar_wait_drain(sm.drain(), 0, 200000000ull)) atomicOr(a.status, kStatusDrainFailed);
  }
  __syncwarp();
}

// ----------------------------------------------------------------- softmax --
__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }

// Row maximum of 128 scores: eight independent chains of 3-input max.
__device__ __forceinline__ float row_max(const uint32_t (&s)[128]) {
  float a[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fmaxf(u2f(s[i]), u2f(s[8 + i]));
#pragma unroll
  for (int c = 16; c < 128; c += 16) {
#pragma unroll
    for (int i = 0; i < 8; ++i) a[i] = max3f(a[i], u2f(s[c + i]), u2f(s[c + 8 + i]));
  }
  return max3f(max3f(a[0], a[1], a[2]), max3f(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
}

// -inf for the columns col0..col0+31 above lim (the diagonal: lim = row).
__device__ __forceinline__ void mask_chunk(uint32_t* s, int col0, int lim) {
#pragma unroll
  for (int c = 0; c < 32; ++c)
    if (col0 + c > lim) s[c] = 0xff800000u;
}

// Four floats -> four e4m3 codes (RNE, saturating; v0 in bits 0..7), and
// acc += (v0' + v2', v1' + v3') over the rounded values v'. Each pair of codes
// is widened to f16 (exact: e4m3 is a subset of f16) and added to the fp32
// accumulator with a mixed-precision add, where every value, subnormal codes
// included, is a normal number; sums of up to 128 such values are exact in
// fp32 while they stay below 2^15.
__device__ __forceinline__ uint32_t pack_e4m3x4_sum(float v0, float v1, float v2, float v3, float2& acc) {
  uint32_t d;
  asm("{\n\t.reg .b16 lo, hi, a0, a1, a2, a3;\n\t.reg .b32 h01, h23;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 lo, %4, %3;\n\t"
      "cvt.rn.satfinite.e4m3x2.f32 hi, %6, %5;\n\t"
      "mov.b32 %0, {lo, hi};\n\t"
      "cvt.rn.f16x2.e4m3x2 h01, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 h23, hi;\n\t"
      "mov.b32 {a0, a1}, h01;\n\t"
      "mov.b32 {a2, a3}, h23;\n\t"
      "add.rn.f32.f16 %1, a0, %1;\n\t"
      "add.rn.f32.f16 %2, a1, %2;\n\t"
      "add.rn.f32.f16 %1, a2, %1;\n\t"
      "add.rn.f32.f16 %2, a3, %2;\n\t}"
      : "=r"(d), "+f"(acc.x), "+f"(acc.y)
      : "f"(v0), "f"(v1), "f"(v2), "f"(v3));
  return d;
}


// Lean P ("ZYFA ...", "Lean P: Linear Approximation of the FP8 Code"): the
// code of a positive e4m3 number grows by 8 per doubling, so the code of 2^x
// is close to 8x + 56 (56 encodes 1.0). y = 1024 + 8x + 56 arrives from the
// caller's multiply-add; converting it to f16 rounds to the nearest integer
// (f16 spacing is 1 in [1024, 2048)) and leaves that integer in the low byte
// of each half; a packed max with 1024 clamps negative codes to 0 (value 0).
// The offset window keeps 8x <= 64, so codes stay <= 120. The four codes are
// gathered with one byte permute; acc adds their exact values as in
// pack_e4m3x4_sum.
__device__ __forceinline__ uint32_t lean_e4m3x4_sum(float2 y01, float2 y23, float2& acc) {
  uint32_t d;
  asm("{\n\t.reg .b16 lo, hi, a0, a1, a2, a3;\n\t.reg .b32 h01, h23, e01, e23, k;\n\t"
      "mov.b32 k, 0x64006400;\n\t"
      "cvt.rn.f16x2.f32 h01, %4, %3;\n\t"
      "cvt.rn.f16x2.f32 h23, %6, %5;\n\t"
      "max.f16x2 h01, h01, k;\n\t"
      "max.f16x2 h23, h23, k;\n\t"
      "prmt.b32 %0, h01, h23, 0x6420;\n\t"
      "mov.b32 {lo, hi}, %0;\n\t"
      "cvt.rn.f16x2.e4m3x2 e01, lo;\n\t"
      "cvt.rn.f16x2.e4m3x2 e23, hi;\n\t"
      "mov.b32 {a0, a1}, e01;\n\t"
      "mov.b32 {a2, a3}, e23;\n\t"
      "add.rn.f32.f16 %1, a0, %1;\n\t"
      "add.rn.f32.f16 %2, a1, %2;\n\t"
      "add.rn.f32.f16 %1, a2, %1;\n\t"
      "add.rn.f32.f16 %2, a3, %2;\n\t}"
      : "=r"(d), "+f"(acc.x), "+f"(acc.y)
      : "f"(y01.x), "f"(y01.y), "f"(y23.x), "f"(y23.y));
  return d;
}

// Probabilities of one 32-column chunk c, p = 2^(s * ca + cb):
//   BF16: packed bf16 pairs into pk[16c .. 16c+15]; acc sums the rounded p.
//   FP8:  e4m3 codes, four per word, into pk[8c .. 8c+7]; acc sums the
//         rounded values.
template <bool FP8, bool LEAN = false>
__device__ __forceinline__ void probs_chunk(int c, const uint32_t* s, float ca, float cb, uint32_t* pk,
                                            float2 (&acc)[2]) {
  const float2 a2 = make_float2(ca, ca);
  const float2 b2 = make_float2(cb, cb);
  if constexpr (!FP8) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const float s0 = u2f(s[2 * i]), s1 = u2f(s[2 * i + 1]);
      const float2 x = __ffma2_rn(make_float2(s0, s1), a2, b2);
      const float2 p = make_float2(ex2_approx(x.x), ex2_approx(x.y));
      const uint32_t pb = pack_bf16x2(p.x, p.y);
      pk[16 * c + i] = pb;
      // the row sum adds the rounded values the PV product uses
      asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
          "add.rn.f32.bf16 %0, lo, %0;\n\tadd.rn.f32.bf16 %1, hi, %1;\n\t}"
          : "+f"(acc[i & 1].x), "+f"(acc[i & 1].y) : "r"(pb));
    }
  } else {
    // lean P: y = 1024 + 56 + 8x = s * (8 ca) + (8 cb + 1080)
    const float2 la2 = make_float2(8.f * ca, 8.f * ca);
    const float2 lb2 = make_float2(8.f * cb + 1080.f, 8.f * cb + 1080.f);
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float s0 = u2f(s[4 * i]), s1 = u2f(s[4 * i + 1]), s2 = u2f(s[4 * i + 2]), s3 = u2f(s[4 * i + 3]);
      if constexpr (LEAN) {
        const float2 y01 = __ffma2_rn(make_float2(s0, s1), la2, lb2);
        const float2 y23 = __ffma2_rn(make_float2(s2, s3), la2, lb2);
        pk[8 * c + i] = lean_e4m3x4_sum(y01, y23, acc[i & 1]);
      } else {
        const float2 x01 = __ffma2_rn(make_float2(s0, s1), a2, b2);
        const float2 x23 = __ffma2_rn(make_float2(s2, s3), a2, b2);
        pk[8 * c + i] = pack_e4m3x4_sum(ex2_approx(x01.x), ex2_approx(x01.y), ex2_approx(x23.x),
                                        ex2_approx(x23.y), acc[i & 1]);
      }
    }
  }
}

// Exact FP8 probabilities of a whole row, in two passes: the 128
// exponentials in place over the scores, then the e4m3 packing and the
// rounded row sum. Measured 3% faster than converting per group of four
// (the packing's conversions no longer wait on each exponential in turn).
__device__ __forceinline__ void probs_row_fp8(uint32_t (&s)[128], float ca, float cb, uint32_t* pk,
                                              float2 (&acc)[2]) {
  const float2 a2 = make_float2(ca, ca), b2 = make_float2(cb, cb);
#pragma unroll
  for (int i = 0; i < 64; ++i) {
    const float2 x = __ffma2_rn(make_float2(u2f(s[2 * i]), u2f(s[2 * i + 1])), a2, b2);
    s[2 * i] = __float_as_uint(ex2_approx(x.x));
    s[2 * i + 1] = __float_as_uint(ex2_approx(x.y));
  }
#pragma unroll
  for (int i = 31; i >= 0; --i)
    pk[i] = pack_e4m3x4_sum(u2f(s[4 * i]), u2f(s[4 * i + 1]), u2f(s[4 * i + 2]), u2f(s[4 * i + 3]), acc[i & 1]);
}

__device__ __forceinline__ void rescale_o_row(uint32_t tO, float rho) {
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint32_t r[32];
    tmem_ld32(tO + 32 * c, r);
    const float2 rr = make_float2(rho, rho);
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float2 x = __fmul2_rn(make_float2(u2f(r[2 * e]), u2f(r[2 * e + 1])), rr);
      r[2 * e] = __float_as_uint(x.x);
      r[2 * e + 1] = __float_as_uint(x.y);
    }
    tmem_st32(tO + 32 * c, r);
  }
}

// FP8 offset window. With offset o the rounded probabilities are
// P' = e4m3(2^(x + log2 sv - o)). A tile whose largest P', 2^(bm - o), falls
// outside [2^kWinLo, 2^kWinHi] moves o to bm - kWinCentre (and O, l are
// rescaled); o never drops below the row's largest log2 value minus
// kFloorBinades (blocks that far down underflow harmlessly). A tile keeps at
// least two binades of normal e4m3 range below its largest P' (2^-4 down to
// 2^-6); a tighter lower edge (2^-2) moved o back and forth on Gaussian rows
// with no measurable change in the output error.
constexpr float kWinLo = -4.0f, kWinHi = 8.0f, kWinCentre = 0.0f, kFloorBinades = 64.0f;

// Decode step with replicated query rows (the SLICE kernels): warp c of a
// softmax warpgroup holds a copy of the group's rows and takes key columns
// 32c .. 32c + 31 of every block (the other columns of its P are zero), with
// its own offset (or running maximum), sum and O rows; the four copies are
// combined like split key ranges. Same arithmetic per column as the
// full-row pass. A copy can see no key at all (a short sequence's last
// block): it keeps m = -inf, l = 0 and O = 0, which the combine weighs 0.
template <bool FP8>
__device__ __forceinline__ void slice_probs(uint32_t tS, uint32_t tO, int cpy, bool diag, int lim, bool first,
                                            float cj, float lsv, float& m, float& l, float& top, uint32_t (&pk)[FP8 ? 32 : 64],
                                            float& psum) {
  uint32_t s[32];
  tmem_ld32(tS + 32 * cpy, s);
  if (diag) mask_chunk(s, 32 * cpy, lim);
  float a8[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) a8[i] = max3f(u2f(s[i]), u2f(s[8 + i]), fmaxf(u2f(s[16 + i]), u2f(s[24 + i])));
  const float mx = max3f(max3f(a8[0], a8[1], a8[2]), max3f(a8[3], a8[4], a8[5]), fmaxf(a8[6], a8[7]));
  constexpr int kW = FP8 ? 8 : 16;     // P words of one 32-column slice
  uint32_t pw[kW];
  float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
  bool moved = false;
  float rho = 1.f;
  if constexpr (FP8) {
    const float bm = mx * cj + lsv;
    if (first) {
      top = bm;
      m = top - kWinCentre;
    } else {
      const float rel = bm - m;
      const bool need = rel > kWinHi || (rel < kWinLo && bm > top - kFloorBinades);
      const float m_new = need ? fmaxf(bm - kWinCentre, fmaxf(top, bm) - kFloorBinades) : m;
      top = fmaxf(top, bm);
      moved = __any_sync(0xffffffffu, need);
      if (moved) {
        rho = ex2_approx(m - m_new);
        l *= rho;
        m = m_new;
      }
    }
    // a copy whose columns are all hidden so far keeps m = -inf (its
    // probabilities are 0, its partial row is empty); the exponent offset
    // must stay finite there
    probs_chunk<true>(0, s, cj, lsv - (m == -INFINITY ? 0.f : m), pw, acc);
  } else {
    const float xmax = mx * cj;
    if (first) {
      m = xmax;
    } else {
      const bool need = xmax > m + kRescaleThreshold;
      moved = __any_sync(0xffffffffu, need);
      if (moved) {
        const float m_new = need ? xmax : m;
        rho = ex2_approx(m - m_new);
        l *= rho;
        m = m_new;
      }
    }
    probs_chunk<false>(0, s, cj, m == -INFINITY ? 0.f : -m, pw, acc);
  }
  // the slice's words at its columns, zeros elsewhere (static indices keep
  // pk in registers)
#pragma unroll
  for (int c = 0; c < 4; ++c)
#pragma unroll
    for (int i = 0; i < kW; ++i) pk[kW * c + i] = (c == cpy) ? pw[i] : 0u;
  const float2 t = __fadd2_rn(acc[0], acc[1]);
  psum = t.x + t.y;
  if (moved) rescale_o_row(tO, rho);
}

template <int DQK, bool FP8, bool VARLEN, bool LEAN, bool SLICE, bool PART, bool LIST>
__device__ void softmax_role(const Smem<DQK, FP8>& sm, uint32_t tmem, const AttnArgs& a, const Sched<VARLEN, PART, LIST>& sc,
                             int warp, int lane) {
  const int nblk = a.scale_blocks;
  const int group = a.Hq / a.Hkv;
  volatile int* abort_flag = sm.abort_flag();
  const int wg = warp >> 2;                      // 0: tile 2t, 1: tile 2t+1
  const int r = (warp & 3) * 32 + lane;          // row within the tile (= TMEM lane)
  const uint32_t lane_off = static_cast<uint32_t>((warp & 3) * 32) << 16;
  const uint32_t tS = tmem + wg * 128 + lane_off;
  const uint32_t tO = tmem + 256 + wg * 128 + lane_off;
  constexpr int kPk = FP8 ? 32 : 64;
  uint32_t sph = 0, oph = 0;
  uint32_t tix = 0;
  const bool tr = lane == 0 && (warp & 3) == 0;
  (void)tix;
  (void)tr;
  __nv_bfloat16* out = static_cast<__nv_bfloat16*>(a.o);

  for (int i = 0, u = sc.first(); u >= 0; u = sc.next(++i, u)) {
    Unit w = sc.decode(u);
    if (wg == 1 && !w.has_b) continue;
    if constexpr (VARLEN) {
      if (sc.step() && wg == 1) w = sc.decode_b(u);   // decode step: tile B runs the unit's second task
    }
    const int qt = 2 * w.t + wg;
    const int n = wg ? w.n_b : w.n_a;   // key blocks this query tile sees
    const int hkv = w.hq / group;
    // BF16: m = running max in log2 units (kept while a new maximum stays
    //       within 2^8 of it), l = sum of the bf16-rounded probabilities.
    // FP8:  m = offset o, top = largest log2(p * sv) seen, l = sum of P'/sv.
    float m = 0.f, l = 0.f, top = 0.f;
    float sq = 1.f;
    int64_t kv_scale_row = 0;
    int pages = 0;   // paged K/V: block-table entries j & ~31 .. + 31, one per lane
    if constexpr (FP8) {
      int64_t qi = (static_cast<int64_t>(w.sidx) * a.Hq + w.hq) * nblk + qt;
      if constexpr (VARLEN) {
        // decode step: row r is query head hq + r, with its own scale
        if (sc.step()) qi = (static_cast<int64_t>(w.sidx) * a.Hq + w.hq + min(SLICE ? (r & 31) : r, group - 1)) * nblk;
      }
      sq = __ldg(a.q_scale + qi);
      kv_scale_row = (static_cast<int64_t>(w.sidx) * a.Hkv + hkv) * nblk;
    }
    (void)pages;
    // Index of the K/V scales of key block jj (called with jj = 0, 1, ...):
    // per sequence block, or per page (block table read 32 entries at a
    // time, one per lane).
    auto kv_index = [&](int jj) -> int64_t {
      int64_t kv_i = kv_scale_row + jj + ((!VARLEN && PART) ? w.j0 : 0);
      if constexpr (VARLEN) {
        if (a.block_table) {
          if ((jj & 31) == 0) {
            const int e = jj + lane;
            pages = e < n ? __ldg(a.block_table + w.sidx * a.bt_stride + w.j0 + e) : 0;
          }
          const int page = min(max(__shfl_sync(0xffffffffu, pages, jj & 31), 0), a.num_pages - 1);
          kv_i = static_cast<int64_t>(page) * a.Hkv + hkv;
        }
      }
      return kv_i;
    };
    // Decode steps with replicated rows load the next block's scales one
    // tile ahead (S is often ready before these loads would return).
    float sk_next = 0.f, sv_next = 0.f;
    if constexpr (FP8 && SLICE) {
      const int64_t i0 = kv_index(0);
      sk_next = __ldg(a.k_scale + i0);
      sv_next = __ldg(a.v_scale + i0);
    }
    for (int j = 0; j < n; ++j) {
      float cj = a.scale_log2, lsv = 0.f, inv_sv = 1.f;
      if constexpr (FP8) {
        float sk, sv;
        if constexpr (SLICE) {
          sk = sk_next;
          sv = sv_next;
          if (j + 1 < n) {
            const int64_t i1 = kv_index(j + 1);
            sk_next = __ldg(a.k_scale + i1);
            sv_next = __ldg(a.v_scale + i1);
          }
        } else {
          const int64_t kv_i = kv_index(j);
          sk = __ldg(a.k_scale + kv_i);
          sv = __ldg(a.v_scale + kv_i);
        }
        cj = sq * sk * a.scale_log2;
        lsv = __log2f(sv);
        inv_sv = 1.0f / sv;
      }
      if (tr) ZTRACE(wg, tix, 1);
      bool ok = mbar_wait(sm.s_full(wg), sph, abort_flag, a.status, kStatusSoftmaxTimeout, a.timeout_ns);
      if (!__all_sync(0xffffffffu, ok)) { *abort_flag = 1; return; }
      sph ^= 1u;
      tc_fence_after();
      if (tr) ZTRACE(wg, tix, 2);
      // Blocks that reach past a row's position are masked: column c of
      // block j is key 128 j + c, the row's position is ctx + 128 qt + r, so
      // columns above lim = 128 (c0 + qt - j) + dlt + r are hidden.
      bool diag;
      int lim;
      if constexpr (VARLEN) {
        const int jd = j - (w.c0 + qt);
        diag = jd >= 0;
        lim = w.dlt + r - 128 * jd;
        if (sc.step()) {          // every row is the token at position len - 1
          const int ja = w.j0 + j;
          diag = (ja == ((w.len - 1) >> 7));
          lim = w.len - 1 - 128 * ja;
        }
      } else if constexpr (PART) {
        diag = (w.j0 + j == qt);   // the diagonal block ends the chunk that holds it
        lim = r;
      } else {
        diag = (j == n - 1);
        lim = r;
      }
      uint32_t pk[kPk];
      float psum = 0.f;
      const bool first = (j == 0);
      if constexpr (SLICE) {
        slice_probs<FP8>(tS, tO, warp & 3, diag, lim, first, cj, lsv, m, l, top, pk, psum);
      } else if constexpr (FP8) {
        // The whole row of S in one load and its maximum first: the offset is
        // set (first tile) or moved (a tile whose largest P' would leave the
        // window) before any exponential, so no tile computes them twice.
        // Rows whose scores span many binades (activation-like inputs) move
        // the offset on a large share of tiles; there this order is 1.5x
        // faster than computing the exponentials speculatively and redoing
        // them, for a few percent on rows that rarely move it.
        uint32_t s[128];
        tmem_ld128(tS, s);
        if (diag) {
#pragma unroll
          for (int c = 0; c < 4; ++c) mask_chunk(&s[32 * c], 32 * c, lim);
        }
        const float bm = row_max(s) * cj + lsv;
        bool moved = false;
        float rho = 1.f;
        if (first) {
          top = bm;
          m = top - kWinCentre;
        } else {
          const float rel = bm - m;
          const bool need = rel > kWinHi || (rel < kWinLo && bm > top - kFloorBinades);
          const float m_new = need ? fmaxf(bm - kWinCentre, fmaxf(top, bm) - kFloorBinades) : m;
          top = fmaxf(top, bm);
          moved = __any_sync(0xffffffffu, need);
          if (moved) {
            rho = ex2_approx(m - m_new);
            l *= rho;
            m = m_new;
          }
        }
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
        if constexpr (LEAN) {
#pragma unroll
          for (int c = 0; c < 4; ++c) probs_chunk<true, true>(c, &s[32 * c], cj, lsv - m, pk, acc);
        } else {
          probs_row_fp8(s, cj, lsv - m, pk, acc);
        }
        const float2 t = __fadd2_rn(acc[0], acc[1]);
        psum = t.x + t.y;
        // O is final for the previous tiles (their PV completed before this
        // S); rescaling it after the exponentials keeps S out of registers.
        if (moved) rescale_o_row(tO, rho);
      } else {
        // The whole row of S in one load and its maximum first. The first
        // tile sets the running maximum; later tiles keep it stale while
        // their own stays within 2^8 of it, otherwise move it before the
        // exponentials (O is rescaled after them). No tile computes its
        // exponentials twice.
        uint32_t s[128];
        tmem_ld128(tS, s);
        if (diag) {
#pragma unroll
          for (int c = 0; c < 4; ++c) mask_chunk(&s[32 * c], 32 * c, lim);
        }
        const float xmax = row_max(s) * cj;
        bool moved = false;
        float rho = 1.f;
        if (first) {
          m = xmax;
        } else {
          const bool need = xmax > m + kRescaleThreshold;
          moved = __any_sync(0xffffffffu, need);
          if (moved) {
            const float m_new = need ? xmax : m;
            rho = ex2_approx(m - m_new);
            l *= rho;
            m = m_new;
          }
        }
        float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
        for (int c = 0; c < 4; ++c) probs_chunk<false>(c, &s[32 * c], cj, -m, pk, acc);
        const float2 t = __fadd2_rn(acc[0], acc[1]);
        psum = t.x + t.y;
        if (moved) rescale_o_row(tO, rho);
      }
      if (tr) ZTRACE(wg, tix, 3);
      if constexpr (FP8) l = fmaf(psum, inv_sv, l);
      else l += psum;
#pragma unroll
      for (int c = 0; c < kPk / 32; ++c) tmem_st32(tS + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&pk[32 * c]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sm.p_full(wg));
      if (tr) ZTRACE(wg, tix, 4);
    }

    // epilogue: O / l, BF16, global store
    if (tr) ZTRACE(wg, tix, 5);
    bool ok = mbar_wait(sm.o_full(wg), oph, abort_flag, a.status, kStatusSoftmaxTimeout, a.timeout_ns);
    if (!__all_sync(0xffffffffu, ok)) { *abort_flag = 1; return; }
    oph ^= 1u;
    tc_fence_after();
    if constexpr (VARLEN) {
      if (w.part >= 0) {
        // split key range: unnormalised O, the row's offset (or running
        // maximum) m and its sum l, combined across splits afterwards
        // replicated rows: copy c of row i is partial row 4 part + c, head hq + i
        const int rr = SLICE ? (r & 31) : r;
        const int64_t prow = static_cast<int64_t>(SLICE ? 4 * w.part + (warp & 3) : w.part) * a.Hq + w.hq + rr;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t o[32];
          __syncwarp();
          tmem_ld32(tO + 32 * c, o);
          if (rr < group) {
            float4* dst = reinterpret_cast<float4*>(a.part_o + prow * 128 + 32 * c);
#pragma unroll
            for (int e = 0; e < 8; ++e)
              dst[e] = make_float4(u2f(o[4 * e]), u2f(o[4 * e + 1]), u2f(o[4 * e + 2]), u2f(o[4 * e + 3]));
          }
        }
        if (rr < group) reinterpret_cast<float2*>(a.part_ml)[prow] = make_float2(m, l);
        continue;
      }
    }
    if constexpr (!VARLEN && PART) {
      // split key range: unnormalised O and (m, l) of chunk w.part, row
      // ((part * B + b) * Spad + query row) * Hq + query head, Spad = 128 x
      // query tiles; combined by prefill_combine_kernel
      const int q_row = qt * 128 + r;
      const int64_t prow =
          ((static_cast<int64_t>(w.part) * a.B + w.b) * (sc.n_qtiles * 128) + q_row) * a.Hq + w.hq;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        uint32_t o[32];
        __syncwarp();
        tmem_ld32(tO + 32 * c, o);
        if (q_row < a.S) {
          float4* dst = reinterpret_cast<float4*>(a.part_o + prow * 128 + 32 * c);
#pragma unroll
          for (int e = 0; e < 8; ++e)
            dst[e] = make_float4(u2f(o[4 * e]), u2f(o[4 * e + 1]), u2f(o[4 * e + 2]), u2f(o[4 * e + 3]));
        }
      }
      if (q_row < a.S) reinterpret_cast<float2*>(a.part_ml)[prow] = make_float2(m, l);
      continue;
    }
    const float inv = 1.f / l;
    const int q_row = qt * 128 + r;
    __nv_bfloat16* orow = out + w.b * a.o_sb + static_cast<int64_t>(w.row0 + q_row) * a.o_ss + w.hq * a.o_sh;
    bool store = q_row < w.len;
    if constexpr (VARLEN) {
      if (sc.step()) {            // row r: query head hq + r of the token
        orow = out + static_cast<int64_t>(w.row0) * a.o_ss + static_cast<int64_t>(w.hq + r) * a.o_sh;
        store = r < group;
      }
    }
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t o[32];
      __syncwarp();   // tcgen05.ld is warp-collective; the stores below are per-thread
      tmem_ld32(tO + 32 * c, o);
      uint32_t pko[16];
#pragma unroll
      for (int e = 0; e < 16; ++e) pko[e] = pack_bf16x2(u2f(o[2 * e]) * inv, u2f(o[2 * e + 1]) * inv);
      if (store) {
        uint4* dst = reinterpret_cast<uint4*>(orow + 32 * c);
#pragma unroll
        for (int v = 0; v < 4; ++v) dst[v] = make_uint4(pko[4 * v], pko[4 * v + 1], pko[4 * v + 2], pko[4 * v + 3]);
      }
    }
    if (tr) ZTRACE(wg, tix, 7);
  }
}

// ------------------------------------------------------------------ kernel --
// LIST: equal lengths with the host's per-CTA unit lists (a parameter of
// about 17 KB, so calls of one wave keep the round-robin instantiation).
struct NoList {};
template <int DQK, bool FP8, bool VARLEN, bool LEAN, bool SLICE, bool PART, bool LIST>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs a,
                    const __grid_constant__ typename Sched<VARLEN>::Table tab,
                    const typename Sched<VARLEN>::Table* tab_global,
                    const __grid_constant__ typename std::conditional<LIST, UnitList, NoList>::type lst) {
  using C = Cfg<DQK, FP8>;
  extern __shared__ uint8_t smem_raw[];
  Smem<DQK, FP8> sm;
  sm.sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  Sched<VARLEN, PART, LIST> sc;
  // The unit table comes by value (built on the host) or, when the sequence
  // offsets live on the device, from global memory (built by a kernel).
  sc.tab = tab_global ? tab_global : &tab;
  sc.B = a.B;
  sc.Hq = a.Hq;
  sc.Hkv = a.Hkv;
  sc.S = a.S;
  sc.n_qtiles = (a.S + 127) / 128;
  sc.pair_lo = a.pair_lo;
  sc.pair_hi = a.pair_hi;
  sc.groups_in_flight = max(1, a.groups_in_flight);
  sc.one_token = a.one_token != 0;
  sc.split_tiles = a.split_tiles;
  if constexpr (LIST) sc.list = &lst;
  else sc.list = nullptr;
  sc.nu = sc.n_units();

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

  if (warp >= 8) {
    regs_decrease<RegSplit<FP8>::kControl>();
    const bool leader = elect_one_sync();
    if (warp == kLoadWarp) {
      if (!a.debug_stall) loader_role<DQK, FP8, kStreamQK, VARLEN, SLICE, PART, LIST>(sm, &tm_q, &tm_k, a, sc, leader);
    } else if (warp == kLoadWarpV) {
      if (!a.debug_stall) loader_role<DQK, FP8, kStreamV, VARLEN, SLICE, PART, LIST>(sm, &tm_q, &tm_v, a, sc, leader);
    } else if (warp == kMmaWarp) {
      mma_role(sm, tmem, a, sc, leader);
    }
    __syncwarp();
  } else {
    regs_increase<RegSplit<FP8>::kSoftmax>();
    softmax_role<DQK, FP8, VARLEN, LEAN, SLICE, PART, LIST>(sm, tmem, a, sc, warp, lane);
    __syncwarp();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int DQK, bool FP8, bool VARLEN, bool LEAN = false, bool SLICE = false, bool PART = SLICE, bool LIST = false>
cudaError_t launch(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v, const AttnArgs& a,
                   const typename Sched<VARLEN>::Table& tab, long long n_units, cudaStream_t stream,
                   const typename Sched<VARLEN>::Table* tab_global = nullptr,
                   const typename std::conditional<LIST, UnitList, NoList>::type* lst = nullptr) {
  using C = Cfg<DQK, FP8>;
  auto kern = attn_fwd_kernel<DQK, FP8, VARLEN, LEAN, SLICE, PART, LIST>;
  // The shared-memory opt-in is per function and device: set it once.
  static bool opted_in[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || !opted_in[dev]) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) opted_in[dev] = true;
  }
  if (n_units == 0) return cudaSuccess;
  const int grid = static_cast<int>(n_units < a.num_sms ? n_units : a.num_sms);
  const typename std::conditional<LIST, UnitList, NoList>::type none{};
  kern<<<grid, kThreads, C::kSmemBytes, stream>>>(tm_q, tm_k, tm_v, a, tab, tab_global, lst ? *lst : none);
  return cudaGetLastError();
}

long long fixed_units(const AttnArgs& a) {
  return static_cast<long long>(a.B) * a.Hq * (a.pair_hi - a.pair_lo);
}

}  // namespace

cudaError_t launch_attn_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const AttnArgs& a, cudaStream_t stream, const UnitList* list) {
  const NoTable none{};
  const long long n = fixed_units(a);
  if (list && a.Dqk == 128)
    return launch<128, false, false, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n, stream, nullptr, list);
  if (list && a.Dqk == 192)
    return launch<192, false, false, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n, stream, nullptr, list);
  if (a.Dqk == 128) return launch<128, false, false>(tm_q, tm_k, tm_v, a, none, n, stream);
  if (a.Dqk == 192) return launch<192, false, false>(tm_q, tm_k, tm_v, a, none, n, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            const AttnArgs& a, cudaStream_t stream, const UnitList* list) {
  const NoTable none{};
  const long long n = fixed_units(a);
  if (list && a.Dqk == 128 && a.lean_p)
    return launch<128, true, false, true, false, false, true>(tm_q, tm_k, tm_v, a, none, n, stream, nullptr, list);
  if (list && a.Dqk == 128)
    return launch<128, true, false, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n, stream, nullptr, list);
  if (list && a.Dqk == 192)
    return launch<192, true, false, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n, stream, nullptr, list);
  if (a.Dqk == 128 && a.lean_p) return launch<128, true, false, true>(tm_q, tm_k, tm_v, a, none, n, stream);
  if (a.Dqk == 128) return launch<128, true, false>(tm_q, tm_k, tm_v, a, none, n, stream);
  if (a.Dqk == 192) return launch<192, true, false>(tm_q, tm_k, tm_v, a, none, n, stream);
  return cudaErrorInvalidValue;
}

// Equal lengths with split key ranges (a.split_tiles key blocks per chunk,
// even): the PART instantiations write partial rows, prefill_combine_kernel
// merges them. n_units = (batch, query head) x the chunks of every pair.
cudaError_t launch_attn_bf16_split(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const AttnArgs& a, long long n_units, cudaStream_t stream) {
  const NoTable none{};
  if (a.Dqk == 128) return launch<128, false, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n_units, stream);
  if (a.Dqk == 192) return launch<192, false, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n_units, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fp8_split(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                  const AttnArgs& a, long long n_units, cudaStream_t stream) {
  const NoTable none{};
  if (a.Dqk == 128 && a.lean_p)
    return launch<128, true, false, true, false, true>(tm_q, tm_k, tm_v, a, none, n_units, stream);
  if (a.Dqk == 128) return launch<128, true, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n_units, stream);
  if (a.Dqk == 192) return launch<192, true, false, false, false, true>(tm_q, tm_k, tm_v, a, none, n_units, stream);
  return cudaErrorInvalidValue;
}

// Equal lengths with split key ranges: out = sum_c O_c 2^(m_c - M) /
// sum_c l_c 2^(m_c - M), M = max_c m_c, over the key chunks c of the row's
// query-tile pair. One warp per (batch, row, query head), four output
// columns per lane (16-byte loads of the partial rows, 8-byte stores), eight
// rows per 256-thread block. While the device status word records a
// timed-out wait, out is left untouched.
__global__ void __launch_bounds__(256) prefill_combine_kernel(const float* __restrict__ part_o,
                                                              const float2* __restrict__ part_ml, int B, int S,
                                                              int Hq, int n_qtiles, int split_tiles,
                                                              __nv_bfloat16* __restrict__ out, int64_t o_sb,
                                                              int64_t o_ss, int64_t o_sh,
                                                              const unsigned int* status) {
  if (*reinterpret_cast<const volatile unsigned int*>(status) &
      (kStatusLoaderTimeout | kStatusMmaTimeout | kStatusSoftmaxTimeout))
    return;
  const int lane = threadIdx.x & 31;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (idx >= static_cast<int64_t>(B) * S * Hq) return;
  const int h = static_cast<int>(idx % Hq);
  const int row = static_cast<int>((idx / Hq) % S);
  const int b = static_cast<int>(idx / (static_cast<int64_t>(Hq) * S));
  const int t = (row >> 7) >> 1;
  const int nk = (2 * t + 1 < n_qtiles) ? 2 * t + 2 : 2 * t + 1;
  const int cnt = (nk + split_tiles - 1) / split_tiles;
  const int64_t spad = static_cast<int64_t>(n_qtiles) * 128;
  auto prow = [&](int c) { return ((static_cast<int64_t>(c) * B + b) * spad + row) * Hq + h; };
  float mx = -INFINITY;
  for (int c = 0; c < cnt; ++c) mx = fmaxf(mx, part_ml[prow(c)].x);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
  for (int c = 0; c < cnt; ++c) {
    const float2 ml = part_ml[prow(c)];
    const float wgt = exp2f(ml.x - mx);
    den = fmaf(ml.y, wgt, den);
    const float4 o = reinterpret_cast<const float4*>(part_o + prow(c) * 128)[lane];
    acc.x = fmaf(o.x, wgt, acc.x);
    acc.y = fmaf(o.y, wgt, acc.y);
    acc.z = fmaf(o.z, wgt, acc.z);
    acc.w = fmaf(o.w, wgt, acc.w);
  }
  const float inv = 1.f / den;
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
  uint2 pkd;
  pkd.x = *reinterpret_cast<uint32_t*>(&lo);
  pkd.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out + b * o_sb + static_cast<int64_t>(row) * o_ss + static_cast<int64_t>(h) * o_sh +
                            4 * lane) = pkd;
}

cudaError_t launch_prefill_combine(const AttnArgs& a, cudaStream_t stream) {
  const int n_qtiles = (a.S + 127) / 128;
  const long long rows = static_cast<long long>(a.B) * a.S * a.Hq;
  if (rows == 0) return cudaSuccess;
  prefill_combine_kernel<<<static_cast<unsigned>((rows + 7) / 8), 256, 0, stream>>>(
      a.part_o, reinterpret_cast<const float2*>(a.part_ml), a.B, a.S, a.Hq, n_qtiles, a.split_tiles,
      static_cast<__nv_bfloat16*>(a.o), a.o_sb, a.o_ss, a.o_sh, a.status);
  return cudaGetLastError();
}

long long table_units(const AttnArgs& a, const SeqTable& tab) {
  if (!a.one_token) return tab.level_start[tab.n_levels];
  const long long tasks = a.split_tiles ? tab.level_start[tab.n_seqs] : static_cast<long long>(tab.n_seqs) * a.Hkv;
  return (tasks + 1) / 2;
}

// Decode step with split key ranges: out = sum_s O_s 2^(m_s - M) /
// sum_s l_s 2^(m_s - M), M = max_s m_s, for each (token, query head); one
// block of 128 threads (one per output column) per (token, head). While the
// device status word records a timed-out wait (the decode kernel stopped
// before writing every partial row), out is left untouched.
__global__ void __launch_bounds__(128) decode_combine_kernel(const float* __restrict__ part_o,
                                                             const float2* __restrict__ part_ml,
                                                             const __grid_constant__ CombineTable ct, int Hq,
                                                             __nv_bfloat16* __restrict__ out, int64_t o_ss,
                                                             int64_t o_sh, const unsigned int* status) {
  if (*reinterpret_cast<const volatile unsigned int*>(status) &
      (kStatusLoaderTimeout | kStatusMmaTimeout | kStatusSoftmaxTimeout))
    return;
  const int i = blockIdx.x / Hq, h = blockIdx.x - (blockIdx.x / Hq) * Hq;
  const int base = ct.base[i], cnt = ct.count[i];
  float mx = -INFINITY;
  for (int s = 0; s < cnt; ++s) mx = fmaxf(mx, part_ml[static_cast<int64_t>(base + s) * Hq + h].x);
  float acc = 0.f, den = 0.f;
  for (int s = 0; s < cnt; ++s) {
    const int64_t row = static_cast<int64_t>(base + s) * Hq + h;
    const float2 ml = part_ml[row];
    const float wgt = exp2f(ml.x - mx);
    den = fmaf(ml.y, wgt, den);
    acc = fmaf(part_o[row * 128 + threadIdx.x], wgt, acc);
  }
  out[static_cast<int64_t>(i) * o_ss + static_cast<int64_t>(h) * o_sh + threadIdx.x] = __float2bfloat16_rn(acc / den);
}

// Decode steps (a.one_token) run their own instantiations (PART), so the
// packed and paged prefill kernels carry none of the one-token code.
cudaError_t launch_attn_bf16_varlen(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    const AttnArgs& a, const SeqTable& tab, cudaStream_t stream) {
  const long long n = table_units(a, tab);
  if (a.replicate && a.Dqk == 128) return launch<128, false, true, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.replicate && a.Dqk == 192) return launch<192, false, true, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.one_token && a.Dqk == 128) return launch<128, false, true, false, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.one_token && a.Dqk == 192) return launch<192, false, true, false, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.Dqk == 128) return launch<128, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.Dqk == 192) return launch<192, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fp8_varlen(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const AttnArgs& a, const SeqTable& tab, cudaStream_t stream) {
  const long long n = table_units(a, tab);
  if (a.replicate && a.Dqk == 128) return launch<128, true, true, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.replicate && a.Dqk == 192) return launch<192, true, true, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.one_token && a.Dqk == 128) return launch<128, true, true, false, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.one_token && a.Dqk == 192) return launch<192, true, true, false, false, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.Dqk == 128 && a.lean_p) return launch<128, true, true, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.Dqk == 128) return launch<128, true, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  if (a.Dqk == 192) return launch<192, true, true>(tm_q, tm_k, tm_v, a, tab, n, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_decode_combine(const AttnArgs& a, const CombineTable& ct, int N, cudaStream_t stream) {
  decode_combine_kernel<<<N * a.Hq, 128, 0, stream>>>(a.part_o, reinterpret_cast<const float2*>(a.part_ml), ct,
                                                      a.Hq, static_cast<__nv_bfloat16*>(a.o), a.o_ss, a.o_sh,
                                                      a.status);
  return cudaGetLastError();
}

// Device-built tables: the unit count is only known on the device, so one
// CTA per SM; CTAs past the last unit leave at once.
cudaError_t launch_attn_bf16_varlen_dev(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                        const AttnArgs& a, const SeqTable* tab, cudaStream_t stream) {
  static const SeqTable unused{};
  if (a.Dqk == 128) return launch<128, false, true>(tm_q, tm_k, tm_v, a, unused, a.num_sms, stream, tab);
  if (a.Dqk == 192) return launch<192, false, true>(tm_q, tm_k, tm_v, a, unused, a.num_sms, stream, tab);
  return cudaErrorInvalidValue;
}

cudaError_t launch_attn_fp8_varlen_dev(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                       const AttnArgs& a, const SeqTable* tab, cudaStream_t stream) {
  static const SeqTable unused{};
  if (a.Dqk == 128 && a.lean_p) return launch<128, true, true, true>(tm_q, tm_k, tm_v, a, unused, a.num_sms, stream, tab);
  if (a.Dqk == 128) return launch<128, true, true>(tm_q, tm_k, tm_v, a, unused, a.num_sms, stream, tab);
  if (a.Dqk == 192) return launch<192, true, true>(tm_q, tm_k, tm_v, a, unused, a.num_sms, stream, tab);
  return cudaErrorInvalidValue;
}

}  // namespace zyfa

#ifdef ZYFA_TRACE
// Copies the trace out and clears it for the next launch.
extern "C" int zyfa_trace_read(void* dst, size_t bytes) {
  if (cudaMemcpyFromSymbol(dst, zyfa::zyfa_trace_buf, bytes) != cudaSuccess) return 3;
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, zyfa::zyfa_trace_buf) != cudaSuccess) return 3;
  return cudaMemset(p, 0, sizeof(zyfa::zyfa_trace_buf)) == cudaSuccess ? 0 : 3;
}
#endif
