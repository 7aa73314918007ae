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

#ifdef __cplusplus
extern "C" {
#endif

/*
 * partial[s][n][m] = sum over the s-th K range of W[m][k] * X[n][k]
 * (the split-K partials whose sum over s is W X^T, stored transposed).
 *   dtype      DFLASH2_BF16 (tcgen05 path) or DFLASH2_F32 (SIMT path, 1 split)
 *   W          [M, K], X [N, K], row-major, element type = dtype
 *   splits     K splits to use (bf16: 1..64, clamped to ceil(K/64); <= 0 picks
 *              the library's own choice); f32 always uses 1
 *   partial    float [splits_used][N][M]; out_bytes its capacity in bytes
 * Returns the number of splits used (>= 1) or a negative status.
 */
int dflash2_test_gemm(int dtype, const void *W, int M, int K, const void *X, int N, int splits,
                      float *partial, size_t out_bytes, void *stream);

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
