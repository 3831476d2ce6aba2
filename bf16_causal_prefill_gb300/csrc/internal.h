// Internal interface between the C-ABI layer (api.cu) and the kernel
// translation units. Not installed; callers use include/zyfa.h.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace zyfa {

constexpr int kBlockTokens = 128;   // quantisation block and attention tile height
constexpr int kTileKeys = 128;      // keys per K/V tile
constexpr int kMaxVarlenSeqs = 1024;     // sequences of a packed batch
constexpr int kMaxVarlenLevels = 1024;   // pairs of 128-row query tiles: 256K tokens

struct QuantArgs {
  const void* x;          // bf16 [B,S,H,D], element strides sb, ss, sh; last dim contiguous
  int64_t sb, ss, sh;
  uint8_t* out;           // e4m3 [B,S,H,D] dense
  float* scales;          // [B,H,ceil(S/128)]
  int B, S, H, D;
  int blk_lo, blk_hi;     // 128-token blocks processed: [blk_lo, blk_hi) of ceil(S/128)
  int hadamard;
  unsigned int* status;   // device status word (streaming kernel's bounded waits)
  uint64_t timeout_ns;
  int num_sms;
};

// Packed variable-length input to the quantiser: sequence i is tokens
// start[i] .. start[i] + len[i] - 1; its 128-token blocks are numbered from
// cum_blocks[i]; scales are [n_seqs, H, max_blocks].
struct QuantSeqTable {
  int n_seqs;
  int max_blocks;
  int start[kMaxVarlenSeqs];
  int len[kMaxVarlenSeqs];
  int cum_blocks[kMaxVarlenSeqs + 1];
};

// Register kernel: any 4-byte aligned input with even strides.
cudaError_t launch_quantize_fp8(const QuantArgs& a, cudaStream_t stream);

// Streaming kernel: up to three tensors of one call (Q, K, V) in one launch.
struct QuantTensor {
  uint8_t* out;           // e4m3 [B,S,H,D] dense (packed: [T,H,D])
  float* scales;          // [B,H,ceil(S/128)] (packed: [n_seqs,H,max_blocks])
  int H, D;               // heads; head dim 128 or 192
  int hadamard;           // rotate rows before quantising (D = 128 only)
};
struct QuantStreamArgs {
  QuantTensor t[3];
  int n;                  // tensors of the call, 1 to 3
  int B, S;               // packed: B = 1, S = total tokens
  int blk_lo, blk_hi;     // equal lengths: 128-token blocks [blk_lo, blk_hi) of every tensor
  unsigned int* status;   // device status word (bounded waits)
  uint64_t timeout_ns;
};
// in[t]: bf16 5-D map (64, S, D/64, H, B) over tensor t, box 64 x 128 x D/64
// x 1 x 1, 128-byte swizzle (16-byte aligned base, strides multiples of 8
// elements). out[t]: the e4m3 output, D = 128: 5-D map (128, S, 1, H, B),
// box 128 x 128 x 1 x 1 x 1; D = 192: 4-D map (D, H, S, B), box 128 x 1 x
// 128 x 1; both 128-byte swizzle.
struct QuantMaps {
  CUtensorMap in[3];
  CUtensorMap out[3];
};
// dmax: the largest head dim of the call's tensors.
cudaError_t launch_quantize_fp8_stream(const QuantMaps& m, const QuantStreamArgs& a, int dmax, int num_sms,
                                       cudaStream_t stream);
// Packed variable-length tensors (B = 1, S = total tokens; maps over T).
cudaError_t launch_quantize_fp8_stream_varlen(const QuantMaps& m, const QuantStreamArgs& a, int dmax,
                                              const QuantSeqTable& tab, int num_sms, cudaStream_t stream);

// Variable-length batches: sequences packed along the token dimension. The
// host sorts the sequences by length (longest first) and lays out the unit
// list by "levels": level k holds pair index t = n_levels - 1 - k of every
// sequence that has more than t pairs of 128-row query tiles (a prefix of the
// sorted order), query heads adjacent. Passed to the kernels by value.
struct SeqTable {
  int n_seqs;                          // sequences with at least one token
  int n_levels;                        // pairs of query tiles of the longest
  int start[kMaxVarlenSeqs];           // first token, sorted order
  int len[kMaxVarlenSeqs];             // tokens, sorted order (descending)
  int index[kMaxVarlenSeqs];           // position in the caller's batch
  int ctx[kMaxVarlenSeqs];             // paged K/V: cached tokens before the queries (else 0)
  int level_start[kMaxVarlenLevels + 1];   // first unit of each level
};

// Equal-length calls of more than one wave: the host assigns the units
// (in the kernel's order, longest query-tile pairs first within each
// super-group of KV groups) to CTAs one by one, each to the CTA with the
// least work so far (list scheduling, as a dynamic queue would), and passes
// each CTA's units here: CTA c runs unit[start[c]] .. unit[start[c+1]-1].
constexpr int kMaxListCtas = 256;
constexpr int kMaxListUnits = 8192;
struct UnitList {
  uint16_t start[kMaxListCtas + 1];
  uint16_t unit[kMaxListUnits];
};

struct AttnArgs {
  int B, S, Hq, Hkv, Dqk, Dv;         // varlen: B = 1 and S = total tokens (the packed tensor)
  float scale_log2;        // softmax_scale * log2(e)
  void* o;                 // bf16 [B,S,Hq,Dv]
  int64_t o_sb, o_ss, o_sh;
  const float* q_scale;    // fp8 only: [B,Hq,nblk]
  const float* k_scale;    // fp8 only: [B,Hkv,nblk]
  const float* v_scale;    // fp8 only: [B,Hkv,nblk]
  unsigned int* status;    // device status word
  uint64_t timeout_ns;     // bound on every barrier wait
  int debug_stall;         // nonzero: the loader issues nothing (watchdog test)
  int num_sms;
  int scale_blocks;        // fp8: blocks per (sequence, head) row of the scale arrays
  int lean_p;              // fp8, head dim 128: lean P instead of exact P
  int pair_lo, pair_hi;    // equal lengths: only query-tile pairs [pair_lo, pair_hi) (rows 256*lo .. 256*hi)
  int groups_in_flight;    // equal lengths: (batch, KV head) groups interleaved in the work order
  // Paged K/V (packed queries only): key block j of sequence i (caller's
  // order) is page block_table[i * bt_stride + j] of caches viewed as
  // [num_pages, 128, Hkv, D]; fp8 K/V scales are [num_pages, Hkv]. Null: K/V
  // packed like the queries.
  const int32_t* block_table;
  int64_t bt_stride;
  int num_pages;
  // Decode step (packed calls only): one query token per sequence; a unit is
  // (sequence, KV head) and its tile rows are the group's query heads. The
  // q map is over (token, head) rows, H = 1; tab.len holds each sequence's
  // key count (the new token included) and tab.start its token's row.
  int one_token;
  // Decode step with split key ranges (split_tiles > 0): a task covers
  // split_tiles key blocks and writes its rows' unnormalised O (fp32, Dv =
  // 128) to part_o and (m, l) to part_ml (float pairs), row (p * Hq + head)
  // for partial row p; decode_combine then writes o.
  int split_tiles;
  float* part_o;
  float* part_ml;
  // Decode step, groups of at most 32 heads, with partial rows: the q map's
  // box is 32 rows, loaded at tile rows 0, 32, 64 and 96; warp c of a softmax
  // warpgroup takes key columns 32c .. 32c + 31 and writes partial row
  // 4 p + c for the task's partial row p (a separate kernel instantiation).
  int replicate;
};

// Equal lengths with split key ranges (a.split_tiles > 0, even): units are
// (batch, query head, query-tile pair, chunk of split_tiles key blocks); each
// writes unnormalised O to part_o and (m, l) to part_ml at row ((chunk * B +
// b) * Spad + query row) * Hq + head, Spad = 128 * ceil(S / 128), and
// launch_prefill_combine writes o. n_units counts the chunks of all pairs.
cudaError_t launch_attn_bf16_split(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const AttnArgs& a, long long n_units, cudaStream_t stream);
cudaError_t launch_attn_fp8_split(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                  const AttnArgs& a, long long n_units, cudaStream_t stream);
cudaError_t launch_prefill_combine(const AttnArgs& a, cudaStream_t stream);

// Partial rows of each sequence (caller's order) for decode_combine.
struct CombineTable {
  int base[kMaxVarlenSeqs];
  int count[kMaxVarlenSeqs];
};
cudaError_t launch_decode_combine(const AttnArgs& a, const CombineTable& ct, int N, cudaStream_t stream);

// A page index outside [0, num_pages): its keys read as zeros (the copy is
// outside the tensor map) and its fp8 scales are taken from page 0 or the
// last page; the call's results are meaningless and this bit is set.
constexpr unsigned int kStatusBadPage = 0x20u;

// tm_q/tm_k/tm_v: 4-D tiled maps (D, H, S, B), 128-byte swizzle, box of
// 128 bytes x 1 head x 128 tokens x 1 batch.
// list: the per-CTA unit lists (grid = a.num_sms CTAs), or null for the
// round-robin order (CTA c runs units c, c + grid, ...).
cudaError_t launch_attn_bf16(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const AttnArgs& a, cudaStream_t stream, const UnitList* list = nullptr);
cudaError_t launch_attn_fp8(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                            const AttnArgs& a, cudaStream_t stream, const UnitList* list = nullptr);
// Packed variable-length batch: maps over (D, H, T, 1); `tab` as above.
// Paged K/V (a.block_table set): tm_k/tm_v over (D, H, 128, num_pages) and
// tab.ctx gives each sequence's cached tokens.
cudaError_t launch_attn_bf16_varlen(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                    const AttnArgs& a, const SeqTable& tab, cudaStream_t stream);
cudaError_t launch_attn_fp8_varlen(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                   const AttnArgs& a, const SeqTable& tab, cudaStream_t stream);

// Offsets on the device: build_seq_tables writes the same tables the host
// would build into device memory (attn_tab and/or quant_tab, either may be
// null); offsets that are not a valid partition of `total` tokens into B
// sequences of at most max_len set kStatusBadSeqlens in *status and leave
// empty tables, so the kernels that read them do nothing.
constexpr unsigned int kStatusBadSeqlens = 0x10u;
cudaError_t launch_build_seq_tables(const int32_t* cu, int B, int total, int max_len, int Hq, SeqTable* attn_tab,
                                    QuantSeqTable* quant_tab, unsigned int* status, cudaStream_t stream);
cudaError_t launch_attn_bf16_varlen_dev(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                        const AttnArgs& a, const SeqTable* tab, cudaStream_t stream);
cudaError_t launch_attn_fp8_varlen_dev(const CUtensorMap& tm_q, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                       const AttnArgs& a, const SeqTable* tab, cudaStream_t stream);
cudaError_t launch_quantize_fp8_stream_varlen_dev(const QuantMaps& m, const QuantStreamArgs& a, int dmax,
                                                  const QuantSeqTable* tab, int num_sms, cudaStream_t stream);

}  // namespace zyfa
