/*
 * fa_lp.h -- C ABI of the GB300 (sm_103a) low-precision packed-varlen attention forward.
 *
 * The operation (FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4,
 * description; SGLang PR #40175 "add fp8_fa_sm120 FP8 backend for SM120 GPUs", Modifications):
 * for every segment [a, b) of cu_seqlens and every head h,
 *
 *     out[a:b, h] = softmax(q[a:b, h] @ k[a:b, h]^T * softmax_scale) @ v[a:b, h]
 *
 * non-causal, head_dim 128, BF16 in and out, computed on quantized operands:
 *   FA_LP_MODE_FP8   : E4M3 Q/K/V with one amax scale per (tensor, head), FP32 accumulation,
 *                      online softmax, probabilities re-quantized to E4M3 before the PV product.
 *   FA_LP_MODE_NVFP4 : SageAttention3-style NVFP4: E2M1 codes with one UE4M3 scale per 16
 *                      elements, K centred by its segment's per-channel mean, Q by its 128-row
 *                      block mean (the qm K^T term added back), V transposed with per-16-key
 *                      scales, two-level P scaling (row maximum brought to 448*6).
 *   block-sparse      : fa_lp_forward_sparse on an FP8 plan: the FP8 arithmetic over the 64-key
 *                      blocks the caller lists for every 64-row query block (SGLang PR #40116
 *                      "Add SM120 Sage compute for SubBlock sparse attention", Modifications).
 *
 * Conventions (all entry points):
 *   - Every function returns an int status (FA_LP_OK or an FA_LP_ERR_* code); nothing throws
 *     across the ABI. fa_lp_status_string() names a status.
 *   - "device pointer" arguments are CUDA device addresses on the plan's device; "host pointer"
 *     arguments are ordinary host memory. The caller keeps ownership of everything it passes.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream). Work is
 *     enqueued on it and the call returns without synchronizing; no host-device synchronization
 *     happens inside fa_lp_quantize / fa_lp_forward_varlen / fa_lp_attention.
 *   - Strides are in ELEMENTS (BF16 = 2 bytes). The channel (head_dim) axis must be contiguous.
 *   - The quantized operands live in one grow-only workspace per device, shared by every plan and
 *     both modes. Calls that use the same device must therefore be ordered (one stream, or
 *     externally synchronized streams): fa_lp_quantize for one plan followed by fa_lp_quantize for
 *     another plan overwrites the first plan's codes.
 *   - There is no fallback: shapes or devices the kernels do not handle return
 *     FA_LP_ERR_UNSUPPORTED (head_dim != 128 is not expressible; a device other than sm_103 is).
 */
#ifndef FA_LP_H_
#define FA_LP_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FA_LP_API __attribute__((visibility("default")))
#else
#define FA_LP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ---------------------------------------------------------------------------- */
#define FA_LP_OK 0
#define FA_LP_ERR_INVALID_ARG 1     /* bad pointer, size, stride, cu_seqlens or mode            */
#define FA_LP_ERR_UNSUPPORTED 2     /* valid request the kernels do not serve (device arch, ...) */
#define FA_LP_ERR_CUDA 3            /* a CUDA runtime / driver call failed                       */
#define FA_LP_ERR_OOM 4             /* workspace or plan metadata allocation failed              */
#define FA_LP_ERR_DEVICE_TIMEOUT 5  /* a bounded device-side wait expired (see fa_lp_get_last_error) */
#define FA_LP_ERR_STATE 6           /* call out of order (e.g. forward before quantize)          */

/* ---- modes ----------------------------------------------------------------------------------- */
#define FA_LP_MODE_FP8 0
#define FA_LP_MODE_NVFP4 1
/* FP8 with one scale per (segment, tensor, head): the amax of each (tensor, head) is taken over
 * the tokens of one segment instead of the whole packed input, so that in a packed batch a long
 * segment does not set a short one's scale. Everything else is FA_LP_MODE_FP8. */
#define FA_LP_MODE_FP8_SEGMENT 2

#define FA_LP_HEAD_DIM 128

typedef struct fa_lp_plan fa_lp_plan;

/* Human-readable name of a status code. Never NULL; the string is static. */
FA_LP_API const char* fa_lp_status_string(int status);

/*
 * fa_lp_plan_create -- validate a packed-varlen segmentation and build (or fetch from the cache)
 * the plan for it.
 * Passage: FlashInfer docs, minimax_h3_sm120_varlen_attention_nvfp4, Parameters (cu_seqlens:
 * cu_seqlens[0] = 0, non-decreasing entries, cu_seqlens[-1] = tokens; cu_seqlens_host avoids a
 * synchronizing device-to-host copy and the segment plan is cached per (cu_seqlens, heads,
 * device); softmax_scale defaults to 1/sqrt(128)).
 *   tokens          : T, total packed tokens (>= 0).
 *   heads           : H (1..1024).
 *   cu_seqlens_host : host pointer, num_segments + 1 int32 entries. Copied; not retained.
 *   num_segments    : >= 1. Empty segments (cu[s] == cu[s+1]) are allowed and produce no work.
 *                     A batch of B sequences of length S is the segmentation [0, S, 2S, ..., BS]
 *                     over the [B*S, H, 128] token axis (each sequence attends to itself only).
 *   softmax_scale   : > 0 and finite; <= 0 or NaN selects 1/sqrt(128).
 *   mode            : FA_LP_MODE_FP8, FA_LP_MODE_NVFP4 or FA_LP_MODE_FP8_SEGMENT (the FP8 path
 *                     with per-(segment, tensor, head) scales; SGLang PR #40175's fused_prep.py
 *                     takes one amax per head, and this mode is the per-segment reading of it for
 *                     packed batches).
 *   device          : CUDA device ordinal the plan will run on (not touched here).
 *   out             : receives the plan. A plan with an identical key is shared (reference
 *                     counted); every successful create needs one fa_lp_plan_destroy.
 * Host-only: makes no CUDA call, so it also works on a machine without a GPU.
 * Errors: FA_LP_ERR_INVALID_ARG for a malformed cu_seqlens, NULL pointers, bad heads or mode.
 */
FA_LP_API int fa_lp_plan_create(int64_t tokens, int heads, const int32_t* cu_seqlens_host,
                      int num_segments, float softmax_scale, int mode, int device,
                      fa_lp_plan** out);

/* Release one reference. The last release frees the plan's host state and its small device
 * metadata buffer (cudaFree, after synchronizing the device). The shared workspace is kept;
 * see fa_lp_release_workspace. NULL is accepted. */
FA_LP_API int fa_lp_plan_destroy(fa_lp_plan* plan);

/* Plan facts, for callers and tests.
 *   padded_tokens : rows of the padded token axis (every segment starts on a 128-row boundary).
 *   work_items    : attention work items (segment, head, pair of 128-row query tiles).
 *   workspace     : bytes of the per-device workspace this plan needs. */
FA_LP_API int fa_lp_plan_info(const fa_lp_plan* plan, int64_t* padded_tokens, int64_t* work_items,
                    size_t* workspace_bytes);

/* Bytes of workspace the plan needs (cf. the FlashInfer op's workspace_bytes_nvfp4). */
FA_LP_API int fa_lp_workspace_bytes(const fa_lp_plan* plan, size_t* bytes);

/*
 * fa_lp_quantize -- quantize BF16 Q, K, V straight from (possibly strided) device views into the
 * device workspace.
 * Passage: SGLang PR #40175, Modifications (fused_prep.py: quantize strided BF16 Q/K/V views per
 * head straight into the kernel buffers, amax then pack, no FP32 intermediates, no layout copy);
 * review reply (the pack pass writes every padding position). NVFP4: FlashInfer docs (K centred
 * by the segment's per-channel mean, Q by its 128-row block mean, E2M1 + UE4M3 per 16, V
 * transposed with per-16-key scales).
 *   q, k, v       : device pointers to BF16 [tokens, heads, 128] views; element strides
 *                   (*_stride_tok, *_stride_head) may be any positive values (e.g. slices of a
 *                   fused [T, 3, H, 128] buffer); channel stride 1; 16-byte aligned rows.
 *   stream        : cudaStream_t (as void*).
 * FP8 mode: per (tensor, head) amax over all tokens, descale = amax/448, codes
 * E4M3_rn_sat(x * (448/amax)). FP8_SEGMENT mode: the same with the amax of each (segment, tensor,
 * head) over the segment's tokens (an empty segment gets descale 1). NVFP4 mode: K means, Q block
 * means, E2M1/UE4M3 packing.
 * Grows the device workspace if needed (stream-ordered cudaMallocAsync/cudaFreeAsync).
 * Retains no reference to q, k, v after the kernels read them.
 * Errors: INVALID_ARG (NULL, misaligned, non-positive strides), UNSUPPORTED (device not sm_103),
 * OOM, CUDA.
 */
FA_LP_API int fa_lp_quantize(fa_lp_plan* plan, const void* q, int64_t q_stride_tok, int64_t q_stride_head,
                   const void* k, int64_t k_stride_tok, int64_t k_stride_head, const void* v,
                   int64_t v_stride_tok, int64_t v_stride_head, void* stream);

/*
 * fa_lp_forward_varlen -- attention over the quantized operands of the last fa_lp_quantize of
 * this plan (same device, same stream order).
 * Passage: SGLang PR #40175, Modifications (kernel.py: E4M3 QK and PV with FP32 accumulation,
 * online softmax, probabilities packed to E4M3) and FlashInfer docs (description; out: optional
 * pre-allocated output of q's shape and dtype; the output is rounded to BF16 once).
 *   cu_seqlens_dev : device pointer to the same num_segments+1 int32 values the plan was built
 *                    from (accepted for the documented call shape; the kernels index with the
 *                    plan's copy, so its contents are not read).
 *   out            : device pointer, BF16 [tokens, heads, 128] with element strides
 *                    (out_stride_tok, out_stride_head), caller-owned. Only rows inside segments
 *                    are written; other rows are left untouched.
 *   stream         : cudaStream_t (as void*).
 * FP8 arithmetic: S = (E4M3 Q codes . E4M3 K codes) accumulated in FP32 on the tensor cores;
 * online softmax over 64-key tiles counted from each segment start, in log2 units with
 * c = dq*dk*softmax_scale*log2(e); the reference maximum m is the first tile's row maximum and
 * moves to a later tile's maximum M only when (M - m)*c > 8 (then O and l are rescaled by
 * 2^((m - M)*c)); P = E4M3_rn(2^(S*c - m*c)) <= 256; l sums the quantized P; O accumulates
 * P * V codes in FP32; out = BF16_rn(O * dv / l).
 * NVFP4 arithmetic (FlashInfer docs, description: two-level P with the row maximum brought to
 * 448*6): S = deq(Q codes) . deq(K codes) on the block-scaled FP4 tensor cores (FP32
 * accumulation), plus qm . deq(K codes) for the query's 128-row block mean qm (FP32); in log2
 * units s = (S + qm.K) * softmax_scale * log2(e);
 * online softmax over 64-key tiles from each segment start with the exact running row maximum m
 * (O and l rescaled by 2^(m_old - m) whenever it moves); P' = 2^(s - m) * 2688; per 16 keys a
 * UE4M3 scale E4M3_rn(max P' / 6) and E2M1_rn codes of P' / scale; l sums the dequantized P; O
 * accumulates deq(P) * deq(V) in FP32; out = BF16_rn(O / l).
 * Errors: STATE (the device's workspace does not hold this plan's codes: no quantize of this
 * plan yet, or another plan quantized on the device since, or the workspace was released),
 * INVALID_ARG, UNSUPPORTED, CUDA.
 */
FA_LP_API int fa_lp_forward_varlen(fa_lp_plan* plan, const int32_t* cu_seqlens_dev, void* out,
                         int64_t out_stride_tok, int64_t out_stride_head, void* stream);

/*
 * fa_lp_forward_varlen_lse -- fa_lp_forward_varlen that also returns each row's log-sum-exp.
 * Passage: SGLang PR #40175, review thread (the SM120 kernel returns output and LSE; the plan's
 * buffers are "FP8, output/LSE"). The pages give no formula; reading taken here: the natural log of
 * the normalizer the output is divided by, in the units of S = q.k * softmax_scale:
 *   FP8   : LSE = m_ref + ln(l), l = sum of the quantized P = 2^((S - m_ref) log2 e), i.e.
 *           log sum_j exp(s_j) up to the E4M3 rounding of P;
 *   NVFP4 : LSE = m + ln(l / 2688) + (q . km) * softmax_scale, l = sum of deq(P'), q the BF16 query
 *           and km its segment's K mean, so that the K centring is undone.
 * Precision of the FP8 l: each of a row's two softmax threads sums its 32 quantized P of a 64-key
 * tile in f16 pairs (a value passes through at most four f16 additions), then in FP32; P spans
 * 2^-9 .. 2^8, so l may differ from the exact sum of the quantized P by a relative 4 * 2^-11 =
 * 1.95e-3 at most (the LSE by as much in absolute terms; measured on ragged varlen rows: at most
 * 2.1e-4, mean 1.1e-5). An exact FP32 sum of the same values cost 5.6 % of the forward's time at
 * S = 30272, H = 56 and was not kept. The NVFP4 l is accumulated in FP32 by the tensor core.
 *   lse             : device pointer, FP32; the row of token t, head h is written to
 *                     lse[h * lse_stride_head + t] for tokens inside segments only (others are
 *                     left untouched). Caller-owned. NULL: behaves as fa_lp_forward_varlen.
 *   lse_stride_head : elements between heads, >= tokens. lse must be 4-byte aligned.
 * Other arguments, errors and ordering as fa_lp_forward_varlen.
 */
FA_LP_API int fa_lp_forward_varlen_lse(fa_lp_plan* plan, const int32_t* cu_seqlens_dev, void* out,
                                       int64_t out_stride_tok, int64_t out_stride_head, float* lse,
                                       int64_t lse_stride_head, void* stream);

/*
 * fa_lp_forward_sparse -- block-sparse attention on the plan's quantized operands (FP8 plans).
 * Passage: SGLang PR #40116 "Add SM120 Sage compute for SubBlock sparse attention",
 * Modifications (64-row query blocks x 64-key blocks, a key block being 4 pooling cells of 16
 * keys; partial blocks; variable per-row block counts, mixed sparse and dense query rows) and
 * Accuracy Tests (ragged lengths, variable block counts, empty rows). Reading taken here: a
 * query row in the g-th 64-row block of its segment attends to the keys of the 64-key blocks
 * listed for (head, g) -- block kb covers keys [64 kb, min(64 kb + 64, L_s)) of the segment --
 * with the arithmetic of fa_lp_forward_varlen (E4M3 Q K^T and P V, FP32 accumulation, online
 * softmax with the lazy reference maximum over the listed blocks in list order, l from the
 * quantized P); a row whose list is empty is written as 0 (LSE -inf). The pages' SM120 mode
 * takes Q K^T in INT8; sm_103a has no INT8 tensor-core MMA (tcgen05.mma kind::i8 does not
 * assemble for it), so here both products are E4M3, on the same quantized operands as the dense
 * forward (call fa_lp_quantize first; FP8 and FP8_SEGMENT plans).
 *   block_offsets : device int32 [heads * G + 1], non-decreasing, block_offsets[0] >= 0; the list
 *                   of (head h, query block g) is block_indices[block_offsets[h G + g] ..
 *                   block_offsets[h G + g + 1]). G = fa_lp_sparse_query_blocks(plan) = sum over
 *                   segments of ceil(L_s / 64); query blocks are numbered over the segments in
 *                   order (empty segments have none).
 *   block_indices : device int32 [num_indices]; every list strictly ascending, entries in
 *                   [0, ceil(L_s / 64)) of the query block's segment.
 *   num_indices   : length of block_indices; no read goes past it.
 *   out, strides, lse, lse_stride_head : as fa_lp_forward_varlen_lse (lse may be NULL).
 * The lists are read on the device: a list that breaks the contract has its offending entries
 * dropped (its rows' output is then unspecified, but no access leaves the arrays) and
 * fa_lp_get_last_error reports status 0x200 and returns FA_LP_ERR_INVALID_ARG.
 * Device memory: the plan keeps a scratch buffer of 4 * num_indices + 16 * heads * (Tpad / 128)
 * bytes (merged lists and tile tables), grown stream-ordered on `stream` when a call needs more;
 * block-sparse calls on one plan share it, so they must be ordered (one stream, or synchronized).
 * Three kernels per call: the list merge, the tile order and the attention (the quantize
 * kernels belong to fa_lp_quantize).
 * Errors: STATE (as fa_lp_forward_varlen), UNSUPPORTED (NVFP4 plan, or a segment longer
 * than 12.5 M tokens), INVALID_ARG, OOM, CUDA.
 */
FA_LP_API int fa_lp_forward_sparse(fa_lp_plan* plan, const int32_t* cu_seqlens_dev,
                                   const int32_t* block_offsets, const int32_t* block_indices,
                                   int64_t num_indices, void* out, int64_t out_stride_tok,
                                   int64_t out_stride_head, float* lse, int64_t lse_stride_head,
                                   void* stream);

/* Number G of 64-row query blocks of the plan (the block lists of fa_lp_forward_sparse). */
FA_LP_API int fa_lp_sparse_query_blocks(const fa_lp_plan* plan, int64_t* num_query_blocks);

/* fa_lp_attention -- fa_lp_quantize followed by fa_lp_forward_varlen on the same stream: the
 * one-call form out = attention(q, k, v, cu_seqlens) of the FlashInfer op's signature. */
FA_LP_API int fa_lp_attention(fa_lp_plan* plan, const void* q, int64_t q_stride_tok,
                    int64_t q_stride_head, const void* k, int64_t k_stride_tok,
                    int64_t k_stride_head, const void* v, int64_t v_stride_tok,
                    int64_t v_stride_head, const int32_t* cu_seqlens_dev, void* out,
                    int64_t out_stride_tok, int64_t out_stride_head, void* stream);

/*
 * fa_lp_attention_host -- the one-call form from and to host memory: copies Q, K and V to the
 * device, quantizes, runs the attention and copies the output back. The heads are processed in
 * chunks, and the copy-in of chunk c+1, the quantize + attention of chunk c and the copy-out of
 * chunk c-1 overlap on three streams. Every step of the path is independent per head (the FP8
 * scales are per (tensor, head), the NVFP4 means and scales per head), so the result equals
 * fa_lp_attention on the same data bit for bit. The chunked schedule is this library's own
 * design; the operation is the one of fa_lp_attention (FlashInfer docs,
 * minimax_h3_sm120_varlen_attention_nvfp4, Parameters and description).
 *   q, k, v         : host pointers, BF16 [tokens, heads, 128] with element strides (tok, head),
 *                     channels contiguous, 16-byte aligned, strides multiples of 8 (as the device
 *                     form). Page-locked memory (cudaHostAlloc / cudaHostRegister) lets the
 *                     copies overlap the compute; pageable memory is accepted, the copies then
 *                     serialise with it.
 *   out             : host pointer, BF16 [tokens, heads, 128] with element strides; every row
 *                     (all tokens lie in a segment) is written. Caller-owned.
 *   heads_per_chunk : 1..heads for chunks of that many heads (the last may be shorter), or 0 for
 *                     the library's choice: the size n giving 4 to 8 chunks whose CTAs fill the
 *                     GPU's waves best (1-head chunks when heads < 4), with a shorter first
 *                     chunk and the rest of n (the last takes what remains) when heads >= 3 n:
 *                     the first chunk has round(2 n / 3) heads for the FP8 modes, ceil(n / 2)
 *                     for NVFP4 (and in fa_lp_attention_sparse_host).
 *   stream          : the quantize and attention kernels run on it; the copies run on two
 *                     streams of the plan, ordered after the work already on `stream`, and
 *                     `stream` is ordered after the last copy-out: once `stream` completes, `out`
 *                     holds the result. The first chunk's copy-in from page-locked views is a
 *                     gather kernel reading them through their device mapping (a 2D DMA copy
 *                     pays a fixed cost per token row); the other copies are DMA copies.
 *                     Returns after enqueueing.
 * Device memory: two chunk slots of Q, K, V and output (8 x tokens x (largest chunk) x 256
 * bytes), allocated on the first call (or a call with another heads_per_chunk) and kept by the
 * plan, plus plans of the chunk sizes (cached like any plan; each call gives them this plan's
 * NVFP4 table limit, see fa_lp_plan_set_table_limit). Device-side wait
 * expiries are reported by fa_lp_get_last_error on this plan. A plan must not run this call
 * from two host threads at once.
 * Errors: INVALID_ARG (null or misaligned view, heads_per_chunk out of range, wrong device),
 * UNSUPPORTED, OOM, CUDA.
 */
FA_LP_API int fa_lp_attention_host(fa_lp_plan* plan, const void* q, int64_t q_stride_tok,
                                   int64_t q_stride_head, const void* k, int64_t k_stride_tok,
                                   int64_t k_stride_head, const void* v, int64_t v_stride_tok,
                                   int64_t v_stride_head, void* out, int64_t out_stride_tok,
                                   int64_t out_stride_head, int heads_per_chunk, void* stream);

/*
 * fa_lp_attention_sparse_host -- fa_lp_forward_sparse from and to host memory, through the head
 * pipeline of fa_lp_attention_host: the block lists are copied to the device once per call,
 * then every chunk of heads is copied in, quantized and run through the block-sparse forward
 * with its heads' lists (offsets from h0 * G on), and copied out, chunks overlapping as there.
 * Passage and semantics: those of fa_lp_forward_sparse (SGLang PR #40116, Modifications); the
 * result equals fa_lp_quantize + fa_lp_forward_sparse on the same data bit for bit.
 *   q, k, v, out, heads_per_chunk, stream : as fa_lp_attention_host.
 *   block_offsets : host int32 [heads * G + 1]; block_indices: host int32 [num_indices]; the list
 *                   contract of fa_lp_forward_sparse (checked on the device, reported through
 *                   fa_lp_get_last_error on the plan).
 * Device memory: that of fa_lp_attention_host plus a copy of the lists, kept by the plan.
 * Errors: INVALID_ARG, UNSUPPORTED (NVFP4 plan), OOM, CUDA.
 */
FA_LP_API int fa_lp_attention_sparse_host(fa_lp_plan* plan, const void* q, int64_t q_stride_tok,
                                          int64_t q_stride_head, const void* k,
                                          int64_t k_stride_tok, int64_t k_stride_head,
                                          const void* v, int64_t v_stride_tok,
                                          int64_t v_stride_head, const int32_t* block_offsets,
                                          const int32_t* block_indices, int64_t num_indices,
                                          void* out, int64_t out_stride_tok,
                                          int64_t out_stride_head, int heads_per_chunk,
                                          void* stream);

/*
 * Inspection of the quantized operands (for bit-exact tests). `which` selects one array of the
 * workspace; the descriptor gives its device address and layout. Valid until the next call that
 * may grow the workspace.
 */
#define FA_LP_Q_CODES 0     /* FP8: u8 [H][Tpad][128]  NVFP4: u8 [H][Tpad][64] (2 codes/byte)   */
#define FA_LP_K_CODES 1     /* same layout as Q                                                  */
#define FA_LP_V_CODES 2     /* FP8: u8 [H][128][Tpad] (V^T)  NVFP4: u8 [H][128][Tpad/2]          */
#define FA_LP_DESCALE 3     /* FP8: f32 [1][3][H] = amax/448 of q, k, v; FP8_SEGMENT: f32        */
                            /* [3][num_segments][H]                                              */
#define FA_LP_Q_SCALES 4    /* NVFP4: u8 [H][Tpad][8] UE4M3, one per 16 channels                 */
#define FA_LP_K_SCALES 5    /* NVFP4: u8 [H][Tpad][8]                                            */
#define FA_LP_V_SCALES 6    /* NVFP4: u8 [H][Tpad/128][128][8], one per 16 keys per channel      */
#define FA_LP_Q_MEANS 7     /* NVFP4: f32 [H][Tpad/128][128], block means                        */
#define FA_LP_K_MEANS 8     /* NVFP4: f32 [num_segments][H][128], segment means                  */
#define FA_LP_Q_KM 9        /* NVFP4: f32 [H][Tpad], q . km of each query row (LSE term)         */
#define FA_LP_QMK_TABLE 10  /* NVFP4: f32 [1][1][n]: per segment s (in order) [H][nb_s][128 nb_s]  */
                            /* = qm_block . deq(Kc_key) (raw units of the scores)                 */

typedef struct fa_lp_array_desc {
  const void* data;  /* device address                                                     */
  int64_t dims[3];   /* outermost first                                                    */
  int64_t strides[3];/* bytes                                                              */
  int elem_bytes;    /* 1 or 4                                                             */
} fa_lp_array_desc;

/* Padded token axis: segment s occupies rows [row_offset[s], row_offset[s] + L_s) of Tpad, where
 * row_offset[s] = sum over s' < s of roundup(L_s', 128); rows in between hold zero codes.
 * row_offsets must have room for num_segments + 1 entries (host pointer). */
FA_LP_API int fa_lp_plan_row_offsets(const fa_lp_plan* plan, int64_t* row_offsets);

FA_LP_API int fa_lp_get_quantized(const fa_lp_plan* plan, int which, fa_lp_array_desc* desc);

/* Copy one quantized array (see fa_lp_get_quantized) into a caller-owned device buffer of at
 * least dims[0]*dims[1]*dims[2]*elem_bytes bytes, stream-ordered on `stream`.
 * Errors: INVALID_ARG (NULL, buffer too small, bad `which`), STATE (nothing quantized yet). */
FA_LP_API int fa_lp_copy_quantized(const fa_lp_plan* plan, int which, void* dst, size_t dst_bytes,
                         void* stream);

/*
 * fa_lp_get_last_error -- device-side status of the plan's kernels: 0 when every bounded
 * device wait completed and every block list was valid; 0x1RR when a wait expired (RR = the
 * waiting role), returning FA_LP_ERR_DEVICE_TIMEOUT; 0x200 when fa_lp_forward_sparse met a block
 * list that breaks its contract, returning FA_LP_ERR_INVALID_ARG. The first error is kept.
 * Reading it synchronizes the device and clears it.
 */
FA_LP_API int fa_lp_get_last_error(fa_lp_plan* plan, int* device_status);

/* Upper bound on the probes of every device-side barrier wait of this plan's kernels. The first
 * 64 probes of a wait spin; each later probe parks the waiting thread for at most about 100
 * microseconds, so the default 20000 probes bounds a wait at about 2 seconds. With a limit below
 * 64 every probe is a non-blocking poll, so that a test can make a wait expire deterministically. A wait that reaches the bound records an error (see
 * fa_lp_get_last_error), makes every CTA of the launch stop, drains in-flight copies and MMAs,
 * frees tensor memory and returns. Small values are for tests of that path. spins >= 1. */
FA_LP_API int fa_lp_plan_set_wait_limit(fa_lp_plan* plan, int64_t spins);

/*
 * fa_lp_plan_set_table_limit -- the largest qm K^T table (bytes) an NVFP4 plan holds at once.
 *
 * Passage: FlashInfer docs, flashinfer.diffusion_ops.minimax_h3_sm120_varlen_attention_nvfp4,
 * description (Q is centred by its 128-row block mean qm and the qm K^T term is added back to the
 * scores). The term is kept as a table of H x sum over segments of nb_s^2 x 128 floats
 * (nb_s = ceil(L_s / 128)): quadratic in the segment length, 1.63 GB for one 30272-token segment
 * at H = 56.
 *
 * When the whole table fits in `bytes`, fa_lp_quantize writes it and the forward reads it. When
 * it does not, the plan holds two table slots of at most bytes / 2 each (one head's table at the
 * least), and the forward builds the table of one group of heads into a slot right before that
 * group's attention launch. The groups alternate between two internal streams; both start after
 * the work already queued on the caller's stream, and the caller's stream then waits for both.
 * Outputs and LSE are bit-identical either way. bytes = 0 restores the library default (4 GB:
 * the whole table up to one segment of about 49.5k tokens at H = 56).
 *
 * The call re-lays the plan's workspace, so the plan must be quantized again. Plans are shared
 * between identical fa_lp_plan_create calls, and the limit applies to every holder; no kernel of
 * the plan may be running. No effect on FP8 plans. While a plan holds the ring,
 * fa_lp_get_quantized(FA_LP_QMK_TABLE) returns UNSUPPORTED.
 * Errors: INVALID_ARG (NULL plan), CUDA (releasing the plan's device tables failed).
 */
FA_LP_API int fa_lp_plan_set_table_limit(fa_lp_plan* plan, size_t bytes);

/* The NVFP4 table layout of a plan: heads per slot, slots (1: the whole table, written by
 * fa_lp_quantize; 2: the ring filled by the forward) and bytes per slot; zeros for FP8 plans.
 * Any output pointer may be NULL. Errors: INVALID_ARG (NULL plan). */
FA_LP_API int fa_lp_plan_table_layout(const fa_lp_plan* plan, int* heads_per_slot, int* slots,
                                      size_t* slot_bytes);

/* Free the workspace of `device` (stream-ordered on `stream`). Plans stay valid; the next
 * quantize allocates again. */
FA_LP_API int fa_lp_release_workspace(int device, void* stream);

/* Encode `n` fp32 device values with the device's converters (format 0: E4M3 rn satfinite,
 * one byte per value; format 1: E2M1 rn satfinite, one 4-bit code per byte). For tests that pin
 * the hardware conversions against the format definitions. */
FA_LP_API int fa_lp_encode(int format, const float* x, int64_t n, uint8_t* codes, void* stream);

/*
 * fa_lp_fp8_descale_noalloc -- the FP8 per-(tensor, head) descales of fa_lp_quantize
 * (amax / 448 over all tokens, 1 when amax is 0) for callers that cannot let the library
 * allocate device memory: programs whose memory belongs to their own pool or allocator,
 * deployments with a fixed memory footprint after start-up, and latency-critical loops that
 * cannot afford cudaMalloc's implicit synchronization. The pages have no counterpart of this
 * call; it is an addition of this library.
 *   q, k, v       : device pointers to BF16 [tokens, heads, 128] views, as for fa_lp_quantize.
 *   tokens, heads : T >= 0 and 1 <= H <= 1024 (larger H returns FA_LP_ERR_INVALID_ARG).
 *   descale       : device pointer, caller-owned f32 [3][heads] (q, k, v), written.
 *   stream        : cudaStream_t (as void*).
 * It makes no cudaMalloc or cudaFree and calls no allocating library routine: its scratch is
 * a fixed 12 KB device array inside the library, held by every GPU that loads it until the
 * process exits, shared by all calls on a device and cleared by each call. Calls that overlap
 * on the GPU race on it; order them on one stream or synchronize. The first call on a device
 * looks up the array's device address (cudaGetSymbolAddress, with that device current); make it
 * before any stream capture begins. The address is kept per CUDA context: after the device's
 * context is destroyed and re-created (cudaDeviceReset), the next call looks it up again, so
 * that call too must come before any capture.
 * Errors: INVALID_ARG (NULL, misaligned or non-positive strides, heads out of range, descale
 * not 4-byte aligned),
 * UNSUPPORTED (device not sm_103), CUDA.
 */
FA_LP_API int fa_lp_fp8_descale_noalloc(const void* q, int64_t q_stride_tok,
                                        int64_t q_stride_head, const void* k,
                                        int64_t k_stride_tok, int64_t k_stride_head,
                                        const void* v, int64_t v_stride_tok,
                                        int64_t v_stride_head, int64_t tokens, int heads,
                                        float* descale, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_LP_H_ */
