/*
 * fa.h -- C ABI of the fused exact-attention library (libfa.so), sm_103a.
 *
 * Operation. Exact scaled-dot-product attention O = softmax(c * Q K^T [masked]) V computed as one
 * fused, tiled kernel whose N x N score matrix never reaches global memory, plus its backward
 * pass, which recomputes the score tiles from Q, K and the saved per-row log-sum-exp.
 *   - "FlashAttention." (Vol. XVI Kernels and Efficiency, plate 4): intro (tiles of Q, K, V loaded
 *     on chip, a score tile folded into a running output by the online softmax), "Never write the
 *     scores" (same softmax(QK^T/sqrt d)V up to rounding; scores recomputed in the backward pass).
 *   - "Flash Attention: IO-Aware Attention Computation", paragraph 4 (fused QK^T, softmax and
 *     value sum; running max and sum), paragraph 5 (block-sparse: skip zero blocks).
 *   - "FlashAttention: Fast and Memory-Efficient Exact Attention with IO-Awareness", abstract
 *     (exact attention; block-sparse extension).
 * The pages fix no interface, no mask format and no backward formulas; this header states the
 * readings adopted:
 *   masked score  : key j is valid for query i iff (!causal || j <= i) && (j < L_b) &&
 *                   (block_mask == NULL || block_mask[(i/128)*nb + j/128] != 0), nb = ceil(N/128).
 *   LSE           : natural-log log-sum-exp of the scaled, valid scores of each row (fp32);
 *                   a row with no valid key gets O = 0 and LSE = -inf.
 *   gradients     : of L = sum(dO * O): dV = P^T dO, dP = dO V^T, D_i = rowsum(dO * O)_i,
 *                   dS = P * (dP - D), dQ = c dS K, dK = c dS^T Q.
 *
 * Layout. Q, K, V, O, dO, dQ, dK, dV are bf16, contiguous [B, H, N, d] (d innermost); LSE is fp32
 * [B, H, N]. All tensor pointers are device pointers, 16-byte aligned. Supported: d in {64, 128},
 * N >= 1 (any N; tails are masked), B, H >= 1, B*H*N*d < 2^31 elements per tensor.
 *
 * Ownership. The caller owns every buffer and keeps it alive until the work on `stream` has
 * finished. The library allocates nothing on the device and keeps no per-call state.
 *
 * Errors. Every entry point validates its arguments on the host and returns a negative
 * fa_status_t before launching anything; a launch failure returns FA_ERR_CUDA. Work is
 * asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream). Every wait inside a
 * kernel is bounded; a wait that runs out, or (in builds with FA_DEBUG_BOUNDS) an index check
 * that fails, writes its code into *dev_status (a caller-owned device int, nullable) and the
 * kernel returns early with undefined outputs; the caller reads *dev_status after synchronising.
 * Nothing is thrown across the ABI and there is no CPU fallback.
 */
#ifndef FA_H_
#define FA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  FA_OK = 0,
  FA_ERR_INVALID_ARG = -1,    /* null pointer, bad size, bad scale, ... */
  FA_ERR_UNSUPPORTED = -2,    /* d not in {64, 128}, tensor too large */
  FA_ERR_MISALIGNED = -3,     /* a tensor pointer is not 16-byte aligned */
  FA_ERR_CUDA = -4,           /* a CUDA runtime/driver call or launch failed */
  FA_ERR_DEVICE_TIMEOUT = -5, /* written to *dev_status: a bounded in-kernel wait ran out */
  FA_ERR_BOUNDS = -6,         /* written to *dev_status: an in-kernel index check failed */
  FA_ERR_SCRATCH_LIMIT = -7   /* fa_bwd_noalloc: the problem needs more than FA_NOALLOC_SCRATCH_BYTES */
} fa_status_t;

/*
 * Forward pass: O and LSE.
 *   q, k, v     in : bf16 [B, H, N, d] device
 *   o           out: bf16 [B, H, N, d] device
 *   lse         out: fp32 [B, H, N] device (natural log)
 *   causal      0 or 1 (top-left aligned: key j visible to query i iff j <= i)
 *   block_mask  nullable, device uint8 [nb * nb], row-major (query tile, key tile), nonzero = keep
 *   seqlens_k   nullable, device int32 [B], each in [0, N]; keys j >= seqlens_k[b] are masked for
 *               every query row of sequence b (a value outside [0, N] is clamped into it)
 *               Both arrays are read by the kernels, so they live in device memory (or managed or
 *               mapped host memory), not in a host array: the library copies nothing. A pointer to
 *               plain host memory is detected before any launch and returns FA_ERR_INVALID_ARG
 *               (the same holds for the cu_seqlens arrays of fa_varlen_problem).
 *   scale       softmax scale c, finite and > 0 (callers normally pass 1/sqrt(d))
 *   tile_visits nullable, device int32 [B * H * nb]: receives, per (b, h, query tile), the number
 *               of 128 x 128 key tiles the kernel visited (tiles with no valid pair are skipped)
 *   dev_status  nullable, device int (see Errors); left untouched on success
 *   stream      cudaStream_t
 */
int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse,
           int B, int H, int N, int d, int causal,
           const uint8_t* block_mask, const int32_t* seqlens_k, float scale,
           int32_t* tile_visits, int* dev_status, void* stream);

/*
 * FP8 forward pass: O and LSE from e4m3 Q, K, V with per-head descale factors.
 * "FlashAttention." (Vol. XVI Kernels and Efficiency, plate 4), "Never write the scores", names FP8
 * as the direction FlashAttention-3 took and fixes no scheme; the reading adopted:
 *   inputs    q  e4m3 [B, H, N, d];  k  e4m3 [B, Hkv, N, d];  vt  e4m3 V^T [B, Hkv, d, N] (V with
 *             the keys contiguous, the layout of the second product's operand); the attention
 *             inputs are q_descale[b*H + h] * q, k_descale[b*Hkv + hk] * k and
 *             v_descale[b*Hkv + hk] * v (fp32 device arrays [B*H], [B*Hkv], [B*Hkv])
 *   computes  exact attention over those inputs, as fa_fwd_gqa does for bf16 ones (same masks,
 *             scale, causal reading, grouped K/V heads, LSE and tile_visits), up to rounding: the
 *             scores are exact e4m3 products summed in fp32; the probabilities are rounded to e4m3
 *             as 2^8 P (an exact running maximum keeps 2^8 P <= 256) for the P V product, whose
 *             error is at most sum_j max(2^-4 P_ij, 2^-18) |v_jk| per output element
 *   outputs   o bf16 [B, H, N, d]; lse fp32 [B, H, N] (natural log of the scaled scores)
 * Supported: d = 128 and N a multiple of 16 (else FA_ERR_UNSUPPORTED). Errors, stream and
 * ownership as for fa_fwd.
 */
int fa_fwd_fp8(const void* q, const void* k, const void* vt, void* o, float* lse,
               int B, int H, int Hkv, int N, int d, int causal,
               const uint8_t* block_mask, const int32_t* seqlens_k,
               const float* q_descale, const float* k_descale, const float* v_descale,
               float scale, int32_t* tile_visits, int* dev_status, void* stream);

/* Bytes of device workspace fa_bwd needs: D (fp32 [B,H,N]) and the fp32 dQ accumulator
 * ([B,H,N,d]), each rounded up to 256 bytes, then 256 bytes for the main pass's key-tile counter.
 * Returns 0 for invalid sizes. */
size_t fa_bwd_workspace_bytes(int B, int H, int N, int d);

/*
 * Backward pass: dQ, dK, dV from Q, K, V, the forward outputs O and LSE, and dO.
 *   q, k, v, o, dout  in : bf16 [B, H, N, d] device (o and lse exactly as fa_fwd wrote them
 *                          for the same q, k, v, mask and scale)
 *   lse               in : fp32 [B, H, N] device
 *   dq, dk, dv        out: bf16 [B, H, N, d] device
 *   causal, block_mask, seqlens_k, scale: as for fa_fwd (must match the forward call)
 *   workspace         device, >= fa_bwd_workspace_bytes(B, H, N, d) bytes, 256-byte aligned;
 *                     scratch only (its contents on entry are ignored and on exit undefined)
 *   dev_status, stream: as for fa_fwd
 * Launches, in order on `stream`: a pre-pass (D = rowsum(dO * O), dQ accumulator and key-tile
 * counter cleared), the main pass (one CTA per SM, each taking key tiles from the counter and
 * looping over the query tiles that can see them) and a post-pass
 * (dQ fp32 -> bf16). dQ is accumulated with fp32 reduce-adds, so its bits may differ between runs by
 * the order of additions; dK, dV, O and LSE are run-to-run identical.
 */
int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv,
           int B, int H, int N, int d, int causal,
           const uint8_t* block_mask, const int32_t* seqlens_k, float scale,
           void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/*
 * Grouped-query attention (multi-query when Hkv = 1): "Flash Attention: IO-Aware Attention
 * Computation", paragraph 16 (K/V heads shared by groups of query heads, to shrink the K/V cache).
 * The page names the variant only; the reading adopted: H query heads and Hkv K/V heads with
 * H % Hkv == 0 and G = H / Hkv; query head h (of sequence b) attends with K/V head h / G, i.e.
 * exactly fa_fwd on K and V with each K/V head repeated G times along the head axis. The backward
 * gradients dK, dV of a K/V head are the sums over its G query heads of what fa_bwd would give for
 * the repeated tensors.
 *   q, o, dout, dq  bf16 [B, H, N, d];  k, v, dk, dv  bf16 [B, Hkv, N, d];  lse fp32 [B, H, N]
 *   tile_visits     [B * H * nb] (per query head); workspace as fa_bwd_workspace_bytes(B, H, N, d)
 * Every other argument, the launches and the errors are as for fa_fwd / fa_bwd; Hkv outside
 * [1, H] or not dividing H returns FA_ERR_INVALID_ARG. fa_fwd and fa_bwd are the Hkv = H case.
 * The backward main pass owns each (key tile, K/V head) in one CTA; it loops over the group's
 * query heads, so dK and dV stay exact sums in fp32 and are run-to-run identical.
 */
int fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse,
               int B, int H, int Hkv, int N, int d, int causal,
               const uint8_t* block_mask, const int32_t* seqlens_k, float scale,
               int32_t* tile_visits, int* dev_status, void* stream);
int fa_bwd_gqa(const void* q, const void* k, const void* v, const void* o, const void* dout,
               const float* lse, void* dq, void* dk, void* dv,
               int B, int H, int Hkv, int N, int d, int causal,
               const uint8_t* block_mask, const int32_t* seqlens_k, float scale,
               void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/*
 * The backward pass of fa_bwd_gqa with optional extras, for verification and measurement. Every
 * argument but `extras` is as for fa_bwd_gqa; extras == NULL is fa_bwd_gqa.
 *   step_visits       nullable, device int32 [B * Hkv * nb]: receives, per (b, K/V head, 128-key
 *                     tile) in that order, the number of 64-row query steps the main pass visited
 *                     for the key tile, summed over the group's query heads. A step (query rows
 *                     64 v .. 64 v + 63) is visited iff its 128-row query tile and the key tile hold
 *                     at least one valid pair (the skip rule of fa_fwd's tile_visits); written for
 *                     every key tile, 0 where none is visited.
 *   main_begin_event  nullable cudaEvent_t, recorded on `stream` right before the main pass
 *   main_end_event    nullable cudaEvent_t, recorded on `stream` right after it (the pair times
 *                     the main pass alone, without the pre- and post-passes)
 * Errors as for fa_bwd_gqa; an event record that fails returns FA_ERR_CUDA.
 */
typedef struct {
  int32_t* step_visits;
  void* main_begin_event;
  void* main_end_event;
} fa_bwd_extras;

int fa_bwd_ex(const void* q, const void* k, const void* v, const void* o, const void* dout,
              const float* lse, void* dq, void* dk, void* dv,
              int B, int H, int Hkv, int N, int d, int causal,
              const uint8_t* block_mask, const int32_t* seqlens_k, float scale,
              void* workspace, size_t workspace_bytes, const fa_bwd_extras* extras,
              int* dev_status, void* stream);

/*
 * Variable-length and strided batches.
 * The pages fix no tensor layout; frameworks hand attention either padded [B, N, H, d] / [B, H, N, d]
 * tensors or packed sequences (the rows of all sequences concatenated, located by cumulative
 * lengths), often with different query and key lengths (a prompt attending a longer cache). The
 * readings adopted:
 *   layout     every bf16 tensor is addressed as [batch][row][head][d] with d contiguous and the
 *              element strides of fa_strides (row, head, batch: multiples of 8 elements, > 0);
 *              e.g. [B, H, N, d] has (d, N*d, H*N*d), [B, N, H, d] has (H*d, d, N*H*d).
 *   packed     cu_seqlens_q/_k (device int32 [B + 1], nondecreasing from 0): sequence b owns rows
 *              cu[b] .. cu[b+1] of the row dimension (batch strides are then ignored); rows_q and
 *              rows_k are the row extents of the tensors (>= cu[B]); seqlen_q/_k bound the lengths
 *              (longer sequences are truncated to the bound, rows past rows_q/_k are never read
 *              or written). Fixed length: cu_seqlens NULL, every sequence has seqlen_q query rows
 *              and seqlen_k keys.
 *   causal     aligned to the bottom-right corner: with L_q queries and L_k keys, key j is visible
 *              to query i iff j <= i + L_k - L_q (the square case is j <= i). Rows with no visible
 *              key get O = 0 and LSE = -inf.
 *   LSE        fp32, fixed length [B, H, seqlen_q]; packed [H, rows_q] (row r of head h at h * rows_q + r).
 *   workspace  fa_bwd_varlen_workspace_bytes: D and the fp32 dQ accumulator, one row per LSE entry,
 *              and the key-tile counter (laid out as for fa_bwd_workspace_bytes).
 * No block mask, key-padding vector or tile counts here (use fa_fwd / fa_bwd for those). K/V may
 * have Hkv heads as in fa_fwd_gqa. Errors, ownership and launches are as for fa_fwd / fa_bwd; a
 * packed batch's last tile is stored row by row so no write crosses into the next sequence.
 */
typedef struct {
  int64_t row, head, batch;
} fa_strides;

typedef struct {
  int B, H, Hkv, d;
  int seqlen_q, seqlen_k;
  const int32_t* cu_seqlens_q; /* NULL (fixed length) or device int32 [B + 1] */
  const int32_t* cu_seqlens_k; /* NULL exactly when cu_seqlens_q is */
  int rows_q, rows_k;          /* packed only: row extents of the query-side / key-side tensors */
  int causal;
  float scale;
} fa_varlen_problem;

int fa_fwd_varlen(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                  const void* v, fa_strides sv, void* o, fa_strides so, float* lse, int* dev_status, void* stream);
size_t fa_bwd_varlen_workspace_bytes(const fa_varlen_problem* p);
int fa_bwd_varlen(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                  const void* v, fa_strides sv, const void* o, fa_strides so, const void* dout, fa_strides sdo,
                  const float* lse, void* dq, fa_strides sdq, void* dk, fa_strides sdk, void* dv, fa_strides sdv,
                  void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/*
 * fa_bwd_varlen adding fp32 shares into caller accumulators instead of writing bf16 gradients:
 * dq_acc += c dS K, dk_acc += c dS^T Q and dv_acc += P^T dO for this call's problem (sequence-sharded
 * ring attention sums one such share per (query block, key block) pair, and rounding each share to
 * bf16 before the sum would lose precision the kernels hold in fp32). dq_acc, dk_acc and dv_acc are
 * fp32 device tensors in the [batch][row][head][d] views of dq, dk, dv (element strides sdq, sdk, sdv,
 * multiples of 8, 16-byte aligned base); every other argument, the workspace and the errors are as for
 * fa_bwd_varlen. Rows outside every sequence are left as they are. Calls on one stream accumulate in
 * order; dK and dV rows are each owned by one CTA and the dQ rows by one warp of the post-pass, so a
 * call has no races of its own, but calls that overlap on the GPU and share accumulators race.
 */
int fa_bwd_varlen_accumulate(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                             const void* v, fa_strides sv, const void* o, fa_strides so, const void* dout,
                             fa_strides sdo, const float* lse, float* dq_acc, fa_strides sdq, float* dk_acc,
                             fa_strides sdk, float* dv_acc, fa_strides sdv, void* workspace,
                             size_t workspace_bytes, int* dev_status, void* stream);

/*
 * Forward split over keys, for decode-shaped problems (few query rows, long keys), where one CTA
 * per pair of 128-row query tiles would leave most SMs idle. The pages name no decode path; the
 * method is the same online softmax, with the key tiles of each query tile split into
 * num_splits contiguous ranges: every range yields a partial O_s (normalised) and LSE_s over its
 * keys, and a merge pass computes M = max_s LSE_s, w_s = exp(LSE_s - M),
 * O = sum_s w_s O_s / sum_s w_s and LSE = M + ln sum_s w_s (exact up to rounding: the log-sum-exp
 * over a union of key sets). Arguments, layouts and results as for fa_fwd_varlen, plus:
 *   num_splits  1 .. 256 (a split with no visible key contributes w_s = 0);
 *               fa_fwd_splitkv_splits(p, number of SMs) gives 1 when the CTAs without a split
 *               already cover the SMs, else the count (at most one per four key tiles) whose CTAs
 *               fill their waves best
 *   workspace   device, >= fa_fwd_splitkv_workspace_bytes(p, num_splits) bytes, 256-byte aligned:
 *               fp32 partial LSE and O, num_splits per LSE row
 * Launches the forward kernel (split mode) and the merge kernel on `stream`.
 */
int fa_fwd_splitkv_splits(const fa_varlen_problem* p, int num_sms);
size_t fa_fwd_splitkv_workspace_bytes(const fa_varlen_problem* p, int num_splits);
int fa_fwd_splitkv(const fa_varlen_problem* p, int num_splits, const void* q, fa_strides sq, const void* k,
                   fa_strides sk, const void* v, fa_strides sv, void* o, fa_strides so, float* lse,
                   void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/*
 * Partial results and their merge, the pieces of sequence-sharded (ring) attention: the essay and
 * the commentary describe the online softmax as associative over pieces of the key space, so
 * attention over a union of key blocks is the log-sum-exp merge of the attentions over each
 * block. A partial is the normalised fp32 O_b and the LSE_b of one key block, stored in the LSE's
 * row order with d contiguous: fa_partial_rows(p) rows (B*H*seqlen_q fixed, H*rows_q packed),
 * part_o [rows][d], part_lse [rows].
 *   fa_fwd_partial       the forward of p (any layout and causal reading of fa_fwd_varlen) into a
 *                        partial: no O or LSE is written; rows of no sequence are not written
 *   fa_merge_partials    acc <- merge(acc, part) in place: M = max(L_a, L_p), w = exp(L - M),
 *                        O = (w_a O_a + w_p O_p) / (w_a + w_p), L = M + ln(w_a + w_p); a row with
 *                        L = -inf on both sides is left as is
 *   fa_finalize_partials acc -> bf16 O (strides so) and fp32 LSE (layout of fa_fwd_varlen)
 * All pointers are device pointers (16-byte aligned, LSE arrays 4-byte); work is asynchronous on
 * `stream`. Initialise an accumulator with the first block's fa_fwd_partial.
 */
size_t fa_partial_rows(const fa_varlen_problem* p);
int fa_fwd_partial(const fa_varlen_problem* p, const void* q, fa_strides sq, const void* k, fa_strides sk,
                   const void* v, fa_strides sv, float* part_o, float* part_lse, int* dev_status, void* stream);
int fa_merge_partials(const fa_varlen_problem* p, float* acc_o, float* acc_lse, const float* part_o,
                      const float* part_lse, void* stream);
int fa_finalize_partials(const fa_varlen_problem* p, const float* acc_o, const float* acc_lse, void* o,
                         fa_strides so, float* lse, void* stream);

/*
 * Backward pass that allocates nothing, for callers that cannot allocate device memory (a plugin
 * or custom operator inside another framework receives only its input and output buffers; the
 * host framework owns the memory pool, and a cudaMalloc of its own would bypass that pool's
 * accounting, fail when the pool holds the device, or synchronise the device mid-stream).
 * The method's sources have no counterpart to this entry point.
 *
 * Same arguments and results as fa_bwd, without the workspace: the library uses a fixed
 * FA_NOALLOC_SCRATCH_BYTES array of its own device image instead (held on every GPU where the
 * library is loaded, until the process exits). Problems whose fa_bwd_workspace_bytes exceed it
 * return FA_ERR_SCRATCH_LIMIT before anything is launched; e.g. d = 128 fits up to about 65 000
 * rows B*H*N. The first call on a device looks up the array's device address, and so does the
 * first call after a device reset (the address belongs to the device's context); make those calls
 * before any stream capture. Calls share the array: two calls whose work overlaps on the GPU
 * (e.g. on different streams) race. Calls in sequence are safe; every call re-initialises what
 * it reads.
 */
#define FA_NOALLOC_SCRATCH_BYTES (32u << 20)
int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const void* dout,
                   const float* lse, void* dq, void* dk, void* dv,
                   int B, int H, int N, int d, int causal,
                   const uint8_t* block_mask, const int32_t* seqlens_k, float scale,
                   int* dev_status, void* stream);

/* Static, human-readable name of a status code (never NULL). */
const char* fa_status_string(int status);

#ifdef __cplusplus
}
#endif

#endif /* FA_H_ */
