/*
 * zyfa.h -- C ABI of the GB300 causal prefill attention library.
 *
 * One computation: causal forward (prefill) attention in BF16 and FP8 e4m3,
 * head dim 128 (with grouped-query heads) and the MLA head shape (query-key
 * dim 192, value dim 128), with per-block FP8 scaling of Q, K, V and of the
 * probabilities, normalisation by the rounded row sum, and an optional
 * 128-point Hadamard rotation of Q and K before quantisation.
 *
 * Entry points: the quantiser and the two attention calls on [B, S, H, D]
 * batches (plus query-row ranges, a caller workspace that lets calls with
 * few query tiles split their key ranges across CTAs, and a prefill from
 * page-locked host memory); the same on packed variable-length batches
 * (offsets on the host or on the device); packed queries that continue
 * cached sequences over a paged K/V cache; and a decode step over that
 * cache.
 *
 * Sources of the operations (page title, section):
 *   - "ZYFA: Fast and Accurate FP8 Attention on AMD MI355X": "Introduction"
 *     and "Methodology and Limitations" (causal forward pass, equal query and
 *     key lengths, head dim 128 and the MLA shape); "Per-Block Scaling and
 *     Normalization by the Rounded Row Sum"; "FP8 Error in Full-Model
 *     Inference" and footnote 2 (Hadamard rotation fused into the Q pass).
 *   - "FP8 GEMM on CDNA4": section 2.1 (e4m3, max 448), 2.2 (scale = amax /
 *     max, guard for all-zero blocks), 2.3 (round to nearest even).
 *
 * Conventions shared by every entry point:
 *   - Tensors are [B, S, H, D] with the last (head) dimension contiguous.
 *     Strides are in ELEMENTS for the batch, sequence and head dimensions.
 *   - All data pointers are DEVICE pointers owned by the caller; the library
 *     keeps no reference to them after the call returns and allocates no
 *     device memory on the caller's behalf.
 *   - `stream` is a cudaStream_t (NULL = legacy default stream). Work is
 *     enqueued asynchronously; nothing synchronises unless stated.
 *   - Arguments are validated on the host before anything is launched; on
 *     a validation error nothing is enqueued. The text of the last error of
 *     the calling thread is available from zyfa_last_error_message().
 *   - Kernels are built for sm_103a only; another device returns
 *     ZYFA_ERR_UNSUPPORTED.
 *   - Every wait inside the kernels is bounded. A kernel that times out
 *     writes a code into a per-device status word and exits cleanly; read it
 *     with zyfa_get_device_status().
 *   - The device-pointer calls enqueue kernels only (tensor maps and tables
 *     travel as kernel parameters), so they can be captured into a CUDA
 *     graph once each kernel configuration has run eagerly on the device
 *     (the first launch sets its shared-memory opt-in).
 */
#ifndef ZYFA_H_
#define ZYFA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  ZYFA_OK = 0,
  ZYFA_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, bad size or stride */
  ZYFA_ERR_UNSUPPORTED = 2,  /* valid request this build does not implement */
  ZYFA_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  ZYFA_ERR_TIMEOUT = 4       /* a kernel's bounded wait expired (device status) */
} zyfa_status;

/* Static text for a status code. */
const char* zyfa_status_string(int status);

/* Thread-local description of the last non-OK return on this thread. */
const char* zyfa_last_error_message(void);

/* Library version: major * 10000 + minor * 100 + patch. */
int zyfa_version(void);

/*
 * Per-block FP8 quantisation ("FP8 GEMM on CDNA4" 2.2-2.3; rotation: ZYFA
 * post, "FP8 Error in Full-Model Inference").
 *
 * For every (b, h, 128-token block j) over the whole head dimension:
 *   y     = hadamard ? FWHT_128(x) * fl32(1/sqrt(128)) : x        (fp32)
 *   amax  = max |y|;  scale = (amax < 1e-8f) ? 1 : RN(amax / 448)
 *   out   = e4m3 code of RN(y / scale), round to nearest even, saturating
 *           at +-448, sign kept for results that round to zero
 *   scales[(b*H + h)*ceil(S/128) + j] = scale
 * The FWHT runs butterflies of span 1, 2, ..., 64 in that order, each rounded
 * to fp32; results are bit-exact and deterministic.
 *
 * x      : bf16 [B,S,H,D], strides (stride_b, stride_s, stride_h) elements,
 *          4-byte aligned, stride_* even.
 * out    : uint8 e4m3 codes [B,S,H,D], dense (row-major), caller-allocated.
 * scales : float [B,H,ceil(S/128)], dense, caller-allocated.
 * D      : 128 or 192. hadamard (0/1) requires D == 128.
 * Errors : ZYFA_ERR_INVALID_ARG (null/misaligned pointer, B/S/H < 1, odd
 *          stride), ZYFA_ERR_UNSUPPORTED (other D, hadamard with D != 128,
 *          device not sm_103), ZYFA_ERR_CUDA (launch failure).
 */
int zyfa_quantize_fp8(const void* x, int64_t stride_b, int64_t stride_s, int64_t stride_h, void* out,
                      float* scales, int B, int S, int H, int D, int hadamard, void* stream);

/*
 * Row-range form of zyfa_quantize_fp8: only the 128-token blocks covering
 * tokens [row_begin, row_end) of every (batch, head) are read, quantised and
 * written (their codes into out and their scales into scales, both the
 * full-size [B,S,H,D] / [B,H,ceil(S/128)] arrays); everything else is left
 * untouched. row_begin is a multiple of 128, row_end a multiple of 128 or S,
 * 0 <= row_begin < row_end <= S. The bytes written equal those of the full
 * call, so a tensor arriving in pieces can be quantised piece by piece.
 */
int zyfa_quantize_fp8_rows(const void* x, int64_t stride_b, int64_t stride_s, int64_t stride_h, void* out,
                           float* scales, int B, int S, int H, int D, int hadamard, int row_begin, int row_end,
                           void* stream);

/*
 * Q, K and V of one attention call quantised in one launch: the same bytes
 * as three zyfa_quantize_fp8 calls, Q and K with the rotation when
 * hadamard != 0, V never rotated ("ZYFA ...", "FP8 Error in Full-Model
 * Inference": the rotation cancels in Q K^T, so only Q and K take it).
 *
 * q, k, v     : bf16 [B,S,Hq,Dqk], [B,S,Hkv,Dqk], [B,S,Hkv,Dv]; strides
 *               (batch, token, head) in elements.
 * q8, k8, v8  : uint8 e4m3 codes, dense, same shapes, caller-allocated.
 * *_scale     : float [B,H,ceil(S/128)] for each, caller-allocated.
 * (Dqk, Dv)   : (128, 128) or (192, 128); hadamard requires Dqk == 128.
 * When all three inputs allow 16-byte tiled copies (16-byte aligned bases,
 * strides multiples of 8 elements) this is one launch; otherwise each
 * tensor is quantised by its own launch (same bytes). Errors as
 * zyfa_quantize_fp8.
 */
int zyfa_quantize_fp8_qkv(const void* q, const int64_t q_strides[3], const void* k, const int64_t k_strides[3],
                          const void* v, const int64_t v_strides[3], void* q8, float* q_scale, void* k8,
                          float* k_scale, void* v8, float* v_scale, int B, int S, int Hq, int Hkv, int Dqk, int Dv,
                          int hadamard, void* stream);
/* Row-range form (rows [row_begin, row_end) as zyfa_quantize_fp8_rows). */
int zyfa_quantize_fp8_qkv_rows(const void* q, const int64_t q_strides[3], const void* k, const int64_t k_strides[3],
                               const void* v, const int64_t v_strides[3], void* q8, float* q_scale, void* k8,
                               float* k_scale, void* v8, float* v_scale, int B, int S, int Hq, int Hkv, int Dqk,
                               int Dv, int hadamard, int row_begin, int row_end, void* stream);

/*
 * Causal attention, BF16 in and out ("ZYFA ..." Introduction; grouped-query
 * heads: query head h reads KV head h / (Hq / Hkv)):
 *   O[b,i,h,:] = sum_{j<=i} softmax_j(softmax_scale * Q[b,i,h].K[b,j,g]) V[b,j,g]
 * Probabilities are rounded to bf16 for the PV product and the row sum adds
 * the same rounded values (the weights of a row sum to one); accumulation is
 * fp32; output rounded to bf16.
 *
 * q : bf16 [B,S,Hq,Dqk]; k : bf16 [B,S,Hkv,Dqk]; v : bf16 [B,S,Hkv,Dv];
 * o : bf16 [B,S,Hq,Dv], caller-allocated, must not alias q/k/v.
 * *_strides[3] : (batch, seq, head) strides in elements. q/k/v strides must
 *          be multiples of 8 elements (16 bytes, TMA); o strides multiples of
 *          8 elements. All pointers 16-byte aligned.
 * (Dqk, Dv) : (128, 128) or (192, 128). Hq % Hkv == 0. S >= 1 (any length;
 *          the last tile is masked). softmax_scale > 0 and finite.
 * Errors : ZYFA_ERR_INVALID_ARG, ZYFA_ERR_UNSUPPORTED, ZYFA_ERR_CUDA.
 */
int zyfa_attn_fwd_bf16(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                       int Dqk, int Dv, float softmax_scale, const int64_t q_strides[3],
                       const int64_t k_strides[3], const int64_t v_strides[3], const int64_t o_strides[3],
                       void* stream);

/*
 * Causal attention on per-block FP8 inputs ("ZYFA ...", "Per-Block Scaling
 * and Normalization by the Rounded Row Sum"). Inputs are e4m3 codes with one
 * fp32 scale per (b, h, 128-token block), as written by zyfa_quantize_fp8;
 * the dequantised value is code * scale. Each row keeps an offset: its
 * probabilities, times the key tile's V scale and divided by 2^offset, are
 * rounded to e4m3 (RNE); the offset is set from the first key tile's maximum
 * and moved (rescaling the output so far) when a tile's largest rounded value
 * would leave [2^-4, 2^8]. The rounded values multiply the V codes on the
 * tensor cores with fp32 accumulation, and each row is divided by the sum of
 * the same rounded values (offset and V scale divided back out), so the
 * weights that multiply V sum to one. Output bf16.
 *
 * q8/k8/v8 : uint8 e4m3 [B,S,H,D] with the given strides (multiples of 16
 *            elements), 16-byte aligned.
 * q_scale  : float [B,Hq,ceil(S/128)], k_scale/v_scale: float [B,Hkv,ceil(S/128)].
 * flags    : how this call computes the rounded probabilities (every FP8
 *            attention call takes this argument; it affects that call only):
 *            0 (ZYFA_FP8_EXACT_P): 2^x by the exponential unit, then RNE to
 *            e4m3; ZYFA_FP8_LEAN_P ("ZYFA ...", "Lean P: Linear
 *            Approximation of the FP8 Code"): the e4m3 code of 2^x taken as
 *            round(8x + 56), no exponential, at head dim 128 (at 192, the
 *            MLA shape, and in decode steps exact P is used, as the pages
 *            keep it there); faster, with a larger probability-rounding
 *            error (the normalisation by the rounded row sum still holds
 *            exactly). Any other bit: ZYFA_ERR_INVALID_ARG.
 * Other arguments and errors as zyfa_attn_fwd_bf16.
 */
#define ZYFA_FP8_EXACT_P 0
#define ZYFA_FP8_LEAN_P 1
int zyfa_attn_fwd_fp8(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                      const void* v8, const float* v_scale, void* o, int B, int S, int Hq, int Hkv, int Dqk,
                      int Dv, float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                      const int64_t v_strides[3], const int64_t o_strides[3], int flags, void* stream);

/*
 * The two calls above with a caller workspace, for calls with fewer pairs of
 * 128-row query tiles (B * Hq * ceil(S / 256)) than SMs, such as long
 * sequences with few heads ("ZYFA ...", "Introduction": the same causal
 * attention). There the longest pair's chain of key blocks sets the time
 * while most SMs idle, so each pair's key blocks may be split into chunks of
 * C blocks (C even, at most 8 chunks per query tile) run by separate CTAs:
 * every chunk writes its rows' unnormalised output with the row's offset (or
 * running maximum) and rounded sum to the workspace, and a second kernel
 * combines the chunks, o = sum_c O_c 2^(m_c - M) / sum_c l_c 2^(m_c - M). The
 * host picks C from a model of the kernel's static schedule and splits only
 * where that model predicts a clear gain; otherwise, or with workspace ==
 * NULL, the call is exactly zyfa_attn_fwd_bf16 / _fp8 (same bytes). A split
 * call rounds differently in the last bits (per-chunk offsets and sums); the
 * row-range and host-memory forms below reproduce the unsplit call's bytes.
 *
 * workspace       : device memory, 256-byte aligned, owned by the caller and
 *                   not used by anything else until the call's work is done;
 *                   at least zyfa_attn_workspace_bytes(B, S, Hq) bytes
 *                   (smaller: ZYFA_ERR_INVALID_ARG when the call splits).
 * workspace_bytes : its size.
 * zyfa_attn_workspace_bytes: 0 for problems no GPU would split (256 or more
 *                   query-tile pairs, or S <= 256).
 * Other arguments and errors as the calls above.
 */
size_t zyfa_attn_workspace_bytes(int B, int S, int Hq);
/* The chunk length C (key blocks) a full-sequence workspace call of these
 * sizes would use on the current device, 0 when it runs unsplit; negative:
 * minus a status code (B, S or Hq below 1: -ZYFA_ERR_INVALID_ARG). */
int zyfa_attn_split_tiles(int B, int S, int Hq);
int zyfa_attn_fwd_bf16_ws(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                          int Dqk, int Dv, float softmax_scale, const int64_t q_strides[3],
                          const int64_t k_strides[3], const int64_t v_strides[3], const int64_t o_strides[3],
                          void* workspace, size_t workspace_bytes, void* stream);
int zyfa_attn_fwd_fp8_ws(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                         const void* v8, const float* v_scale, void* o, int B, int S, int Hq, int Hkv, int Dqk,
                         int Dv, float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                         const int64_t v_strides[3], const int64_t o_strides[3], int flags, void* workspace,
                         size_t workspace_bytes, void* stream);

/*
 * Row-range ("chunked prefill") forms of the two calls above: only output rows
 * [row_begin, row_end) of every (batch, head) are computed and written, each
 * attending causally to keys 0..row (so K and V are read for rows
 * [0, row_end) only; Q only for the range). row_begin and row_end are
 * multiples of 256, or row_end = S; 0 <= row_begin < row_end <= S. Results
 * are bitwise equal to the same rows of the full call, so a prefill can be
 * split along the sequence and overlapped with the copies of its inputs.
 * Other arguments and errors as the full calls.
 */
int zyfa_attn_fwd_bf16_rows(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                            int Dqk, int Dv, float softmax_scale, const int64_t q_strides[3],
                            const int64_t k_strides[3], const int64_t v_strides[3], const int64_t o_strides[3],
                            int row_begin, int row_end, void* stream);
int zyfa_attn_fwd_fp8_rows(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                           const void* v8, const float* v_scale, void* o, int B, int S, int Hq, int Hkv, int Dqk,
                           int Dv, float softmax_scale, const int64_t q_strides[3], const int64_t k_strides[3],
                           const int64_t v_strides[3], const int64_t o_strides[3], int row_begin, int row_end,
                           int flags, void* stream);

/*
 * The FP8 prefill from host memory: Q, K, V go to the device, are quantised
 * (zyfa_quantize_fp8, with the rotation when hadamard != 0, V never rotated),
 * attended (zyfa_attn_fwd_fp8) and O comes back, in n_chunks pieces along the
 * sequence, so that the copy of piece c+1 in and of piece c-1 out overlap the
 * kernels of piece c. Pieces are whole multiples of 256 rows (the last one
 * may be shorter); n_chunks = 0 picks min(16, ceil(S/256)). The bytes of o
 * equal those of the device-resident calls on the same inputs.
 *
 * q, k, v : bf16 [B,S,Hq,Dqk], [B,S,Hkv,Dqk], [B,S,Hkv,Dv], dense, in
 *           page-locked host memory; o: bf16 [B,S,Hq,Dv] dense, page-locked.
 * workspace : device memory of at least zyfa_prefill_fp8_host_workspace()
 *           bytes, 256-byte aligned, owned by the caller, not used by anything
 *           else until the call's work has finished.
 * stream  : the call orders itself after the work already on stream and
 *           before work queued on it later (it uses streams of its
 *           own in between); o is valid once stream has been synchronised.
 *           The call itself returns once everything is queued.
 * Errors  : as zyfa_attn_fwd_fp8; ZYFA_ERR_INVALID_ARG for pageable host
 *           buffers or a short workspace. After an error the queued part of
 *           the work is still ordered before later work on stream, and o is
 *           unspecified.
 */
size_t zyfa_prefill_fp8_host_workspace(int B, int S, int Hq, int Hkv, int Dqk, int Dv);
int zyfa_prefill_fp8_host(const void* q, const void* k, const void* v, void* o, int B, int S, int Hq, int Hkv,
                          int Dqk, int Dv, float softmax_scale, int hadamard, int n_chunks, void* workspace,
                          size_t workspace_bytes, int flags, void* stream);

/*
 * Packed variable-length batches. The pages time equal-length batches and
 * name variable lengths as future work ("ZYFA ...", "Methodology and
 * Limitations"); this is the layout serving stacks use. Sequences are packed
 * along the token dimension: sequence i is tokens cu_seqlens[i] ..
 * cu_seqlens[i+1]-1 of q [T,Hq,Dqk], k [T,Hkv,Dqk], v [T,Hkv,Dv] and
 * o [T,Hq,Dv] (T = cu_seqlens[B]) and attends causally within itself only.
 *
 * cu_seqlens : HOST int32 [B+1]: cu_seqlens[0] = 0, nondecreasing;
 *              1 <= B <= 1024, each sequence at most 262144 tokens, empty
 *              sequences allowed (T = 0 enqueues nothing).
 * *_strides  : [2] element strides of the token and head dimensions (the
 *              last dimension contiguous); alignment rules as above.
 * q/k/v_scale (FP8): float [B, H, ceil(max_len/128)], one per (sequence,
 *              head, 128-token block of that sequence), as written by
 *              zyfa_quantize_fp8_varlen.
 * The host builds the work list from cu_seqlens (longest sequences first)
 * and passes it to the kernel by value; nothing is allocated.
 * Errors as the equal-length calls.
 */
int zyfa_attn_fwd_bf16_varlen(const void* q, const void* k, const void* v, void* o, const int32_t* cu_seqlens, int B,
                              int Hq, int Hkv, int Dqk, int Dv, float softmax_scale, const int64_t q_strides[2],
                              const int64_t k_strides[2], const int64_t v_strides[2], const int64_t o_strides[2],
                              void* stream);
int zyfa_attn_fwd_fp8_varlen(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                             const void* v8, const float* v_scale, void* o, const int32_t* cu_seqlens, int B, int Hq,
                             int Hkv, int Dqk, int Dv, float softmax_scale, const int64_t q_strides[2],
                             const int64_t k_strides[2], const int64_t v_strides[2], const int64_t o_strides[2],
                             int flags, void* stream);

/*
 * zyfa_quantize_fp8 for a packed variable-length tensor x [T,H,D] (same
 * arithmetic, bit for bit). Blocks are 128 tokens of one sequence; the last
 * block of a sequence may be short and tokens of the next sequence never
 * enter its amax. out: uint8 e4m3 [T,H,D] dense; scales: float
 * [B, H, ceil(max_len/128)] (entries past a sequence's last block are not
 * written). Needs 16-byte aligned x and out and token/head strides that are
 * multiples of 8 elements (ZYFA_ERR_UNSUPPORTED otherwise).
 */
int zyfa_quantize_fp8_varlen(const void* x, int64_t stride_t, int64_t stride_h, void* out, float* scales,
                             const int32_t* cu_seqlens, int B, int H, int D, int hadamard, void* stream);

/*
 * The three packed variable-length calls with cu_seqlens in DEVICE memory
 * (as a serving stack's batcher leaves them): no host read of the offsets
 * and no synchronisation. The caller states the packed token count
 * total_tokens (T, the leading dimension of the packed tensors) and an upper
 * bound max_seqlen on every sequence's length (it also fixes the scale
 * layout [B, H, ceil(max_seqlen/128)], so pass the same value to the
 * quantiser and the attention call). A small kernel builds, in `workspace`,
 * the same tables the host calls build, so the results are bitwise equal to
 * theirs. If the offsets on the device are not a partition of T tokens into
 * B sequences of at most max_seqlen tokens, that call computes nothing and
 * sets bit 4 of the device status word (zyfa_get_device_status then returns
 * ZYFA_ERR_INVALID_ARG).
 *
 * workspace : device memory of zyfa_varlen_workspace_bytes() bytes, 256-byte
 *             aligned, owned by the caller; calls on one stream may share it,
 *             calls that can run concurrently may not.
 * Other arguments and errors as the host-offset calls.
 */
size_t zyfa_varlen_workspace_bytes(void);
int zyfa_quantize_fp8_varlen_dev(const void* x, int64_t stride_t, int64_t stride_h, void* out, float* scales,
                                 const int32_t* cu_seqlens_dev, int B, int total_tokens, int max_seqlen, int H, int D,
                                 int hadamard, void* workspace, void* stream);
/*
 * Q, K and V of a packed variable-length batch quantised in one launch
 * (the bytes of three zyfa_quantize_fp8_varlen / _varlen_dev calls; Q and K
 * rotated when hadamard != 0, V never). Strides (token, head) in elements;
 * scales [B, H, ceil(max_len/128)]; inputs must allow 16-byte tiled copies
 * (ZYFA_ERR_UNSUPPORTED otherwise). The _dev form takes device offsets as
 * zyfa_quantize_fp8_varlen_dev.
 */
int zyfa_quantize_fp8_qkv_varlen(const void* q, const int64_t q_strides[2], const void* k,
                                 const int64_t k_strides[2], const void* v, const int64_t v_strides[2], void* q8,
                                 float* q_scale, void* k8, float* k_scale, void* v8, float* v_scale,
                                 const int32_t* cu_seqlens, int B, int Hq, int Hkv, int Dqk, int Dv, int hadamard,
                                 void* stream);
int zyfa_quantize_fp8_qkv_varlen_dev(const void* q, const int64_t q_strides[2], const void* k,
                                     const int64_t k_strides[2], const void* v, const int64_t v_strides[2], void* q8,
                                     float* q_scale, void* k8, float* k_scale, void* v8, float* v_scale,
                                     const int32_t* cu_seqlens_dev, int B, int total_tokens, int max_seqlen, int Hq,
                                     int Hkv, int Dqk, int Dv, int hadamard, void* workspace, void* stream);
int zyfa_attn_fwd_bf16_varlen_dev(const void* q, const void* k, const void* v, void* o, const int32_t* cu_seqlens_dev,
                                  int B, int total_tokens, int max_seqlen, int Hq, int Hkv, int Dqk, int Dv,
                                  float softmax_scale, const int64_t q_strides[2], const int64_t k_strides[2],
                                  const int64_t v_strides[2], const int64_t o_strides[2], void* workspace,
                                  void* stream);
int zyfa_attn_fwd_fp8_varlen_dev(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                                 const void* v8, const float* v_scale, void* o, const int32_t* cu_seqlens_dev, int B,
                                 int total_tokens, int max_seqlen, int Hq, int Hkv, int Dqk, int Dv,
                                 float softmax_scale, const int64_t q_strides[2], const int64_t k_strides[2],
                                 const int64_t v_strides[2], const int64_t o_strides[2], void* workspace,
                                 int flags, void* stream);

/*
 * zyfa_attn_fwd_fp8_varlen_dev without a workspace: an addition of this
 * library with no counterpart on the pages. It is meant for callers that
 * cannot allocate device memory where they call attention: a step replayed
 * from a CUDA graph whose memory was fixed when it was captured, a serving
 * loop that hands out device memory only from its own pool, or a process that
 * runs with its allocator locked. The unit table that the workspace form
 * builds in caller memory lives instead in one static array of the library
 * (zyfa_noalloc_scratch_bytes() = 32 KB, 256-byte aligned), so this call
 * allocates nothing (no cudaMalloc, no cudaFree, no allocating library call);
 * the caller still owns every input and output.
 *
 * Limits and sharing: the array holds the table of at most 1024 sequences of
 * at most 262144 tokens each; B outside 1..1024 returns ZYFA_ERR_INVALID_ARG
 * and a larger max_seqlen ZYFA_ERR_UNSUPPORTED, before anything is enqueued.
 * The array is resident on every GPU that loads the library until the
 * process exits. All calls share it and each call rewrites it in full, so two
 * calls whose kernels can overlap on the GPU (different streams without an
 * ordering between them) race on it; calls on one stream are safe. The first
 * call on each device looks up the array's device address (with that device
 * current); make that first call before any stream capture.
 *
 * Arguments, results (bitwise those of zyfa_attn_fwd_fp8_varlen_dev) and the
 * other errors as zyfa_attn_fwd_fp8_varlen_dev, without the workspace.
 */
size_t zyfa_noalloc_scratch_bytes(void);
int zyfa_attn_fwd_fp8_varlen_dev_noalloc(const void* q8, const float* q_scale, const void* k8, const float* k_scale,
                                         const void* v8, const float* v_scale, void* o,
                                         const int32_t* cu_seqlens_dev, int B, int total_tokens, int max_seqlen,
                                         int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                                         const int64_t q_strides[2], const int64_t k_strides[2],
                                         const int64_t v_strides[2], const int64_t o_strides[2], int flags,
                                         void* stream);

/*
 * Packed queries over a PAGED K/V cache: chunked prefill and prefix caching.
 * The pages name paged K/V as future work ("ZYFA ...", "Methodology and
 * Limitations"); this is the cache layout serving stacks use. Sequence i
 * has ctx_lens[i] tokens already cached and L_i = cu_seqlens_q[i+1] -
 * cu_seqlens_q[i] new tokens whose queries are rows cu_seqlens_q[i] ..
 * cu_seqlens_q[i+1]-1 of q [T,Hq,Dqk] (and of o [T,Hq,Dv]); the new tokens'
 * keys and values must already be in the cache. Query j of sequence i sits
 * at position ctx_lens[i] + j and attends to cached-sequence positions
 * 0 .. ctx_lens[i] + j (causal with an offset; ctx_lens[i] = 0 for every i
 * is the packed varlen call over a paged cache).
 *
 * k_cache, v_cache : [num_pages, 128, Hkv, Dqk|Dv], pages of 128 tokens;
 *              *_cache_strides [3] are the element strides of the page,
 *              token and head dimensions (last dimension contiguous; the
 *              alignment rules of the packed calls apply).
 * block_table : DEVICE int32, row i (block_table + i * block_table_stride)
 *              lists the pages of sequence i in position order: position p
 *              is token p % 128 of page row_i[p / 128]. Each row needs
 *              ceil((ctx_lens[i] + L_i)/128) valid entries; the rest are
 *              not read. An entry outside [0, num_pages) reads zeros, sets
 *              bit 5 of the device status word and makes that call's output
 *              meaningless (no fault).
 * ctx_lens   : HOST int32 [B], each >= 0 (any chunk boundary; a chunk of
 *              one token per sequence is a decode step).
 * cu_seqlens_q : HOST int32 [B+1] as in the packed calls.
 * Cache slots past a sequence's last position are never attended to, but
 * the tensor cores still multiply them by a zero probability: keep unused
 * slots finite (e.g. zero-initialised cache).
 * FP8: q_scale [B, Hq, ceil(max L_i/128)] from zyfa_quantize_fp8_varlen on
 *              q; k_scale, v_scale float [num_pages, Hkv], one per page and
 *              head (zyfa_quantize_fp8 on a cache as B = num_pages, S = 128).
 * Errors as the packed calls; ZYFA_ERR_INVALID_ARG also for a null
 * block_table, num_pages < 1, or a row stride too short for a sequence.
 */
int zyfa_attn_fwd_bf16_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                             const int32_t* cu_seqlens_q, const int32_t* ctx_lens, const int32_t* block_table,
                             int64_t block_table_stride, int num_pages, int B, int Hq, int Hkv, int Dqk, int Dv,
                             float softmax_scale, const int64_t q_strides[2], const int64_t k_cache_strides[3],
                             const int64_t v_cache_strides[3], const int64_t o_strides[2], void* stream);
int zyfa_attn_fwd_fp8_paged(const void* q8, const float* q_scale, const void* k_cache8, const float* k_scale,
                            const void* v_cache8, const float* v_scale, void* o, const int32_t* cu_seqlens_q,
                            const int32_t* ctx_lens, const int32_t* block_table, int64_t block_table_stride,
                            int num_pages, int B, int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                            const int64_t q_strides[2], const int64_t k_cache_strides[3],
                            const int64_t v_cache_strides[3], const int64_t o_strides[2], int flags,
                            void* stream);

/*
 * Decode step over a paged K/V cache: one new token per sequence (its keys
 * and values already appended to the cache). Sequence i has seq_lens[i]
 * positions, the new token's included; its query q[i] (all Hq heads)
 * attends to positions 0 .. seq_lens[i]-1. A task is (sequence, KV head):
 * the group's Hq/Hkv query heads are the rows of one 128-row tile, so K/V
 * are read once per KV head; each CTA runs two tasks as its two query tiles.
 * Without a workspace the results are the bytes of the paged prefill with
 * ctx_lens[i] = seq_lens[i] - 1 and one new token.
 *
 * workspace  : optional device memory (256-byte aligned) of at least
 *              zyfa_decode_workspace_bytes(N, Hq, Hkv) bytes, owned by the
 *              caller (calls that can run concurrently need their own). With
 *              it, when the N*Hkv tasks would leave SMs idle, each task's key
 *              range is split (at least 8 key blocks per split, about four
 *              tasks per SM), and with Hq/Hkv <= 32 and at least 16 tasks
 *              the group's rows are
 *              replicated four times in the tile so that each softmax warp
 *              takes a quarter of every key block's columns; every split and
 *              copy writes its unnormalised rows with their offset and sum,
 *              and a second kernel combines them (results within rounding of
 *              the call without a workspace). NULL: neither. The workspace
 *              bound counts the four copies only for Hq/Hkv <= 32. A split
 *              is considered only while N*Hkv < 4 x the SM count, so a call
 *              with Hq/Hkv > 32 and at least that many tasks runs as without
 *              a workspace. If a wait of the decode kernel times out (status
 *              bits 0-2, also while an earlier call's timeout is still
 *              unread), the combine kernel leaves o untouched.
 *
 * q, o       : [N, Hq, Dqk|Dv]; q's token stride must be Hq x its head
 *              stride (each token's heads contiguous).
 * seq_lens   : HOST int32 [N], each >= 1; 1 <= N <= 1024; Hq/Hkv <= 128.
 * block_table, k_cache, v_cache, num_pages: as in the paged prefill.
 * FP8: q_scale float [N, Hq], one per token and head (zyfa_quantize_fp8_varlen
 *              with one-token sequences writes it); k_scale, v_scale
 *              [num_pages, Hkv].
 * Errors as the paged prefill.
 */
size_t zyfa_decode_workspace_bytes(int N, int Hq, int Hkv);
int zyfa_attn_decode_bf16_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                                const int32_t* seq_lens, const int32_t* block_table, int64_t block_table_stride,
                                int num_pages, int N, int Hq, int Hkv, int Dqk, int Dv, float softmax_scale,
                                const int64_t q_strides[2], const int64_t k_cache_strides[3],
                                const int64_t v_cache_strides[3], const int64_t o_strides[2], void* workspace,
                                size_t workspace_bytes, void* stream);
int zyfa_attn_decode_fp8_paged(const void* q8, const float* q_scale, const void* k_cache8, const float* k_scale,
                               const void* v_cache8, const float* v_scale, void* o, const int32_t* seq_lens,
                               const int32_t* block_table, int64_t block_table_stride, int num_pages, int N, int Hq,
                               int Hkv, int Dqk, int Dv, float softmax_scale, const int64_t q_strides[2],
                               const int64_t k_cache_strides[3], const int64_t v_cache_strides[3],
                               const int64_t o_strides[2], void* workspace, size_t workspace_bytes, int flags,
                               void* stream);

/*
 * Synchronises `stream`, then reads and clears the current device's status
 * word. *word receives the raw bits (0 when every kernel finished normally;
 * bit 0: loader wait timed out, bit 1: MMA wait, bit 2: softmax wait,
 * bit 3: quantiser wait, bit 4: invalid device cu_seqlens, bit 5: block_table
 * entry outside the paged cache, bit 8: drain after abort incomplete).
 * Returns ZYFA_ERR_TIMEOUT if a wait bit was set, ZYFA_ERR_INVALID_ARG if
 * only bits 4-5 were, ZYFA_ERR_CUDA if the
 * synchronisation failed, else ZYFA_OK.
 * `word` may be NULL.
 */
int zyfa_get_device_status(void* stream, unsigned int* word);

/*
 * Test hooks (process-wide, not thread-safe). stall_loader != 0 makes the
 * attention kernels' loader warp issue nothing, so every consumer wait runs
 * out; timeout_seconds bounds each wait (default 2.0; <= 0 restores it).
 * Used to test the watchdog path without faulting the GPU.
 */
int zyfa_set_debug(int stall_loader, double timeout_seconds);

#ifdef __cplusplus
}
#endif

#endif /* ZYFA_H_ */
