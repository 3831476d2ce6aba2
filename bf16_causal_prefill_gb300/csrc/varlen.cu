// Sequence tables of a packed variable-length batch built on the device, for
// callers whose cu_seqlens live in device memory: the same tables the host
// builds from host offsets (stable order by decreasing length, levels of
// query-tile pairs; per-sequence 128-token block counts for the quantiser),
// written to caller-owned device memory by one CTA.
#include <cuda_runtime.h>

#include "internal.h"

namespace zyfa {
namespace {

constexpr int kThreads = 1024;
static_assert(kMaxVarlenSeqs <= kThreads && kMaxVarlenLevels <= kThreads, "one thread per sequence and level");

__device__ __forceinline__ int pairs_of(int len) { return ((len + 127) / 128 + 1) / 2; }

// In-place inclusive prefix sum of v[0..n) in shared memory (n <= kThreads).
__device__ void block_scan(int* v, int n) {
  for (int off = 1; off < n; off <<= 1) {
    int add = 0;
    if (threadIdx.x < n && threadIdx.x >= off) add = v[threadIdx.x - off];
    __syncthreads();
    if (threadIdx.x < n) v[threadIdx.x] += add;
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kThreads, 1)
    build_seq_tables_kernel(const int32_t* __restrict__ cu, int B, int total, int max_len, int Hq,
                            SeqTable* __restrict__ at, QuantSeqTable* __restrict__ qt, unsigned int* status) {
  __shared__ int len_s[kMaxVarlenSeqs];
  __shared__ int start_s[kMaxVarlenSeqs];
  __shared__ int scan_s[kMaxVarlenLevels + 1];
  __shared__ int bad, n_nonempty, longest;
  const int tid = threadIdx.x;
  if (tid == 0) {
    bad = (cu[0] != 0 || cu[B] != total) ? 1 : 0;
    n_nonempty = 0;
    longest = 0;
  }
  __syncthreads();
  if (tid < B) {
    const int s = cu[tid], e = cu[tid + 1];
    const int len = e - s;
    if (len < 0 || len > max_len || s < 0 || e > total) atomicOr(&bad, 1);
    len_s[tid] = len;
    start_s[tid] = s;
    if (len > 0) atomicAdd(&n_nonempty, 1);
    atomicMax(&longest, len);
  }
  __syncthreads();
  if (bad) {
    // Empty tables: every kernel that reads them computes nothing.
    if (tid == 0) {
      if (at) {
        at->n_seqs = 0;
        at->n_levels = 0;
        at->level_start[0] = 0;
      }
      if (qt) {
        qt->n_seqs = 0;
        qt->max_blocks = (max_len + 127) / 128;
        qt->cum_blocks[0] = 0;
      }
      atomicOr(status, kStatusBadSeqlens);
    }
    return;
  }

  if (qt) {
    // Quantiser: sequences in the caller's order, block counts prefix-summed.
    scan_s[tid] = tid < B ? (len_s[tid] + 127) / 128 : 0;
    __syncthreads();
    block_scan(scan_s, B);
    if (tid < B) {
      qt->start[tid] = start_s[tid];
      qt->len[tid] = len_s[tid];
      qt->cum_blocks[tid + 1] = scan_s[tid];
    }
    if (tid == 0) {
      qt->n_seqs = B;
      qt->max_blocks = (max_len + 127) / 128;
      qt->cum_blocks[0] = 0;
    }
    __syncthreads();
  }

  if (at) {
    // Attention: non-empty sequences, longest first, ties in batch order
    // (the rank of sequence i among the others under that order).
    if (tid < B && len_s[tid] > 0) {
      const int li = len_s[tid];
      int rank = 0;
      for (int j = 0; j < B; ++j) {
        const int lj = len_s[j];
        rank += (lj > li || (lj == li && j < tid)) ? 1 : 0;
      }
      at->start[rank] = start_s[tid];
      at->len[rank] = li;
      at->index[rank] = tid;
      at->ctx[rank] = 0;
    }
    const int n_levels = pairs_of(longest);
    // Level k holds pair t = n_levels - 1 - k of every sequence with more
    // than t pairs, Hq units each.
    if (tid < n_levels) {
      const int t = n_levels - 1 - tid;
      int cnt = 0;
      for (int j = 0; j < B; ++j) cnt += pairs_of(len_s[j]) > t ? 1 : 0;
      scan_s[tid] = cnt * Hq;
    }
    __syncthreads();
    block_scan(scan_s, n_levels);
    if (tid < n_levels) at->level_start[tid + 1] = scan_s[tid];
    if (tid == 0) {
      at->n_seqs = n_nonempty;
      at->n_levels = n_levels;
      at->level_start[0] = 0;
    }
  }
}

}  // namespace

cudaError_t launch_build_seq_tables(const int32_t* cu, int B, int total, int max_len, int Hq, SeqTable* attn_tab,
                                    QuantSeqTable* quant_tab, unsigned int* status, cudaStream_t stream) {
  if (B < 1 || B > kMaxVarlenSeqs) return cudaErrorInvalidValue;
  build_seq_tables_kernel<<<1, kThreads, 0, stream>>>(cu, B, total, max_len, Hq, attn_tab, quant_tab, status);
  return cudaGetLastError();
}

}  // namespace zyfa
