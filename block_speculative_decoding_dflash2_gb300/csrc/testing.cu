// Test hooks declared in include/dflash2_testing.h: the internal contraction
// and the lm_head top-k path, callable on their own for parity tests.
#include <algorithm>
#include <cstring>

#include "../../include/dflash2_testing.h"
#include "common.cuh"
#include "internal.h"

namespace df2 {
namespace {

int test_ctx(Ctx* c, void* stream, unsigned* status) {
  int dev = 0, n = 0, maj = 0, mi = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  if (maj != 10 || mi != 3) return DFLASH2_ERR_UNSUPPORTED;
  c->nsm = std::min(n, kMaxSM);
  c->stream = static_cast<cudaStream_t>(stream);
  c->status = status;
  return DFLASH2_OK;
}

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

}  // namespace
}  // namespace df2

using namespace df2;

extern "C" {

int dflash2_test_last_schedule(void) { return draft_last_schedule(); }

size_t dflash2_test_gemm_workspace(int M, int N) {
  if (M <= 0 || N <= 0) return 0;
  return al((size_t)kMaxSM * sizeof(int)) + al(gemm_partial_bytes(M, N));
}

}  // extern "C"

namespace {

int test_gemm(int dtype, const void* W, const float* wscale, int M, int K, const void* X, int N, int ctas,
              int accumulate, float* out, void* workspace, size_t ws_bytes, void* stream) {
  if (dtype != DFLASH2_BF16 && dtype != DFLASH2_F32) return DFLASH2_ERR_DTYPE;
  if (!W || !X || !out || !workspace) return DFLASH2_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0) return DFLASH2_ERR_SHAPE;
  if (ws_bytes < dflash2_test_gemm_workspace(M, N)) return DFLASH2_ERR_WORKSPACE;
  Ctx c;
  const int rc = test_ctx(&c, stream, nullptr);
  if (rc) return rc;
  GemmOp g;
  std::memset(&g, 0, sizeof(g));
  g.W = W;
  g.wscale = wscale;
  g.M = M;
  g.K = K;
  g.ldw = K;
  g.X = X;
  g.N = N;
  g.ldx = K;
  g.out = out;
  g.accumulate = accumulate != 0;
  g.mult = 1.f;
  g.ctas = ctas < 0 ? -1 : std::min(ctas, kMaxSM);
  char* base = static_cast<char*>(workspace);
  g.counters = reinterpret_cast<int*>(base);
  g.partial = reinterpret_cast<float*>(base + al((size_t)kMaxSM * sizeof(int)));
  if (dtype == DFLASH2_F32) {
    const int r = gemm_f32(g, c);
    return r ? r : 1;
  }
  g.ctas = ctas <= -2 ? ctas : g.ctas;  // <= -2: cluster split-K of -ctas slices per tile
  const int r = gemm_bf16(g, c);
  if (r) return r;
  return gemm_last_grid();  // the CTA count gemm_bf16 launched
}

}  // namespace

extern "C" {

int dflash2_test_gemm(int dtype, const void* W, int M, int K, const void* X, int N, int ctas, int accumulate,
                      float* out, void* workspace, size_t ws_bytes, void* stream) {
  return test_gemm(dtype, W, nullptr, M, K, X, N, ctas, accumulate, out, workspace, ws_bytes, stream);
}

int dflash2_test_gemm_fp8(const void* W8, const float* scale, int M, int K, const void* X, int N, int ctas,
                          int accumulate, float* out, void* workspace, size_t ws_bytes, void* stream) {
  if (!scale) return DFLASH2_ERR_INVALID_ARG;
  return test_gemm(DFLASH2_BF16, W8, scale, M, K, X, N, ctas, accumulate, out, workspace, ws_bytes, stream);
}

int dflash2_test_force_cluster_split(int cs) {
  if (cs != 0 && (cs < 2 || cs > 8)) return DFLASH2_ERR_INVALID_ARG;
  df2::gemm_force_csplit(cs);
  return 0;
}

int dflash2_test_force_attention(int mode) {
  if (mode < 0 || mode > 2) return DFLASH2_ERR_INVALID_ARG;
  df2::attention_force_mode(mode);
  return 0;
}

int dflash2_test_last_attention(void) { return df2::attention_last_kernel(); }

int dflash2_test_layout(const dflash2_config* cfg, int batch, int n_new, int max_ctx, size_t* offsets, int n) {
  return workspace_offsets(cfg, batch, n_new, max_ctx, offsets, n);
}

size_t dflash2_test_topk_workspace(int dtype, int M, int N) {
  const int n_lists = std::max(kMaxSM, topk_scan_lists(M));
  size_t t = al(256) + 2 * al((size_t)n_lists * N * KMAX * 4) + al((size_t)N * kTopkSlots * 8);
  if (dtype == DFLASH2_F32) t += al((size_t)N * M * 4);
  return t;
}

int dflash2_test_gemm_topk(int dtype, const void* W, int M, int K, const void* X, int N, int k, float mult,
                           float cap, int32_t* cand_id, float* cand_logit, float* debug, void* workspace,
                           size_t ws_bytes, void* stream) {
  if (dtype != DFLASH2_BF16 && dtype != DFLASH2_F32) return DFLASH2_ERR_DTYPE;
  if (!W || !X || !cand_id || !cand_logit || !workspace) return DFLASH2_ERR_INVALID_ARG;
  if (M <= 0 || N <= 0 || K <= 0 || k < 1 || k > KMAX || k > M || N > 32 * 256) return DFLASH2_ERR_SHAPE;
  if (ws_bytes < dflash2_test_topk_workspace(dtype, M, N)) return DFLASH2_ERR_WORKSPACE;
  Ctx c;
  int rc = test_ctx(&c, stream, static_cast<unsigned*>(workspace));
  if (rc) return rc;
  const int n_lists_cap = std::max(kMaxSM, topk_scan_lists(M));
  char* base = static_cast<char*>(workspace);
  float* lv = reinterpret_cast<float*>(base + al(256));
  int* li = reinterpret_cast<int*>(base + al(256) + al((size_t)n_lists_cap * N * KMAX * 4));
  int n_lists = 0;
  GemmOp g;
  std::memset(&g, 0, sizeof(g));
  g.W = W;
  g.M = M;
  g.K = K;
  g.ldw = K;
  g.X = X;
  g.N = N;
  g.ldx = K;
  g.mult = mult;
  g.cap = cap;
  if (dtype == DFLASH2_BF16) {
    // the shared per-row thresholds start at zero (a memset node; the draft
    // step zeroes them in the kernel before the lm_head instead)
    unsigned long long* thr =
        reinterpret_cast<unsigned long long*>(base + al(256) + 2 * al((size_t)n_lists_cap * N * KMAX * 4));
    if (cudaMemsetAsync(thr, 0, (size_t)N * kTopkSlots * 8, c.stream) != cudaSuccess) return DFLASH2_ERR_CUDA;
    g.topk = true;
    g.lists_v = lv;
    g.lists_i = li;
    g.thr = thr;
    g.debug = debug;
    rc = gemm_bf16(g, c);
    if (rc) return rc;
    n_lists = gemm_topk_lists(M, N, K, c.nsm, dtype);
  } else {
    float* logits = reinterpret_cast<float*>(base + al(256) + 2 * al((size_t)n_lists_cap * N * KMAX * 4) +
                                             al((size_t)N * kTopkSlots * 8));
    g.out = logits;
    rc = gemm_f32(g, c);
    if (rc) return rc;
    rc = launch_topk_scan(logits, N, M, mult, cap, debug, lv, li, &n_lists, c);
    if (rc) return rc;
  }
  return launch_topk_merge(lv, li, n_lists, N, k, cand_id, cand_logit, c);
}

}  // extern "C"
