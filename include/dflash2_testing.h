/*
 * dflash2_testing.h — test hooks of libdflash2.so (not part of the stable ABI).
 *
 * They expose the library's internal dense contraction so parity tests can
 * check it directly against a plain matrix product, independently of the
 * rest of the draft step.  Same conventions as dflash2.h: device pointers,
 * caller-owned memory, asynchronous on `stream`, negative status on error.
 */
#ifndef DFLASH2_TESTING_H
#define DFLASH2_TESTING_H

#include <stddef.h>
#include <stdint.h>

#include "dflash2.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * out[n][m] = sum_k W[m][k] * X[n][k]   (or out[n][m] += ... with accumulate),
 * through the library's contraction: W X^T stored transposed, fp32.
 *   dtype      DFLASH2_BF16 (tcgen05 path) or DFLASH2_F32 (SIMT path)
 *   W          [M, K], X [N, K], row-major, element type = dtype
 *   ctas       bf16 work schedule: 0 = the library's own (stream-K shares of
 *              all tile x K-chunk work, one CTA per SM); > 0 = stream-K over
 *              that many CTAs (at most 256; tiles shared by several CTAs are
 *              summed by the last piece to arrive, in CTA order); -1 =
 *              whole tiles, one CTA each, round-robin; -2..-8 = cluster
 *              split-K, -ctas K slices per tile in one thread-block cluster,
 *              summed in rank order through distributed shared memory (the
 *              library's own schedule picks this for contractions whose
 *              tiles x slices fill the SMs).  Ignored for f32.
 *   out        float [N][M]
 *   workspace  zeroed on first use, at least dflash2_test_gemm_workspace bytes
 * Returns the number of CTAs launched (>= 1) or a negative status.
 */
/*
 * Schedule the last dflash2_draft_step call in this process took, as bits:
 *   1  fused sublayer prologue (norm + tap logits + conv in one kernel)
 *   2  embedding prologue beside the feature contraction on split SMs
 *   4  QKV contraction with the fused q/k-norm + RoPE epilogue
 *   8  layer 0's context K/V contraction on the SMs the QKV leaves free
 *  16  appended rows carried by the QKV contractions (merged arrangement)
 * Host only; not synchronised with concurrent draft steps.
 */
int dflash2_test_last_schedule(void);

size_t dflash2_test_gemm_workspace(int M, int N);

/*
 * From now on in this process, every bf16 / fp8-weight contraction that the
 * library schedules itself (not the lm_head's top-k) takes cluster split-K
 * with cs K slices where the shape allows it (at least cs K chunks of 64, an
 * activation tile at most 64 wide), so the fused epilogues run after the
 * distributed-shared-memory reduction at test sizes too.  cs = 0 restores the
 * library's own schedule.  Returns 0, or DFLASH2_ERR_INVALID_ARG for cs
 * outside {0, 2..8}.  Not thread-safe against concurrent draft steps.
 */
int dflash2_test_force_cluster_split(int cs);

/*
 * From now on in this process, the block attention of every bf16 draft step
 * runs on: mode 0, the library's choice; 1, the mma.sync cluster kernel; 2,
 * the tcgen05 kernel wherever it applies (head dimension 128, 16-key pages,
 * at most 80 query rows per kv head; elsewhere the library's choice).
 * Returns 0, or DFLASH2_ERR_INVALID_ARG for another mode.  Not thread-safe
 * against concurrent draft steps.
 */
int dflash2_test_force_attention(int mode);

/*
 * The attention kernel the last bf16 or fp32 draft step of this process
 * launched: 1 the mma.sync cluster kernel, 2 the tcgen05 kernel, 3 the SIMT
 * partial + combine kernels; 0 before any.
 */
int dflash2_test_last_attention(void);
int dflash2_test_gemm(int dtype, const void *W, int M, int K, const void *X, int N, int ctas, int accumulate,
                      float *out, void *workspace, size_t ws_bytes, void *stream);

/*
 * The same contraction with fp8 e4m3 weights (the DFLASH2_FP8W path):
 * out[n][m] = scale[m] * sum_k e4m3(W8[m][k]) * X[n][k], X bf16 [N, K],
 * W8 [M, K] bytes (K a multiple of 16), scale float [M].  Same schedule,
 * workspace and return value as dflash2_test_gemm.
 */
int dflash2_test_gemm_fp8(const void *W8, const float *scale, int M, int K, const void *X, int N, int ctas,
                          int accumulate, float *out, void *workspace, size_t ws_bytes, void *stream);

/*
 * Byte offsets, inside the workspace of a dflash2_draft_step call with these
 * sizes (max_ctx = max_pages * page_size), of the intermediates that call
 * leaves behind, in this order:
 *   [0] f    [n_new, H]        projected features of the appended rows
 *   [1] h    [batch*B, H] fp32 residual stream after the last layer
 *   [2] u    [batch*B, H]      normed input of the last MLP sublayer
 *   [3] u2   [batch*B, H]      that input after the dynamic convolution
 *   [4] q    [batch*B, nq, d]  block queries of the last layer (normed, rotated)
 *   [5] kb   [batch*B, nkv, d] block keys of the last layer (normed, rotated)
 *   [6] vb   [batch*B, nkv, d] block values of the last layer
 *   [7] O    [batch*B, nq*d]   attention output of the last layer
 *   [8] act  [batch*B, I]      SiLU(gate)*up of the last layer
 *   [9] hn   [batch*(B-1), H]  final-normed hidden states of positions 1..B-1
 *  [10] ua   [batch*B, H]      normed input of the last attention sublayer
 *  [11] u2a  [batch*B, H]      that input after the dynamic convolution
 *  [12] cnt  int[]             split-K tile counters of the block branch
 *  [13] cnta int[]             split-K tile counters of the append branch
 * Element type is cfg.dtype except h.  `n` must be >= 14.  Host only.
 * The counters (zero between calls) must sit at the same offsets for every
 * call shape, dflash2_append_context (batch 0) included.
 */
int dflash2_test_layout(const dflash2_config *cfg, int batch, int n_new, int max_ctx, size_t *offsets, int n);

/*
 * Top-k of the rows of z = mult * (X W^T), softcapped when cap > 0, through
 * the lm_head path (bf16: tcgen05 GEMM with the fused streaming top-k, then
 * the merge; f32: SIMT GEMM, scan, merge).
 *   cand_id / cand_logit  [N][k] out, best first (equal logits: smaller id)
 *   debug                 nullable [N][M] out: every transformed logit
 *   workspace             at least dflash2_test_topk_workspace(M, N) bytes
 */
size_t dflash2_test_topk_workspace(int dtype, int M, int N);
int dflash2_test_gemm_topk(int dtype, const void *W, int M, int K, const void *X, int N, int k, float mult,
                           float cap, int32_t *cand_id, float *cand_logit, float *debug, void *workspace,
                           size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_TESTING_H */
