// Top-k candidates per block position ("DFlash2 Speculative Decoding"
// (llama-cpp-python wiki), "Configuration Notes": selector_top_k candidates
// per position; "Train a DFlash Drafter for Speculative Decoding", "Key
// Config Fields").  Order: larger logit first, equal logits by smaller id.
//
// The lm_head GEMM (tcgen05 path) already leaves one sorted list of KMAX
// entries per CTA and row.  topk_scan_kernel produces the same lists from
// stored logits (fp32 path).  topk_merge_kernel reduces the lists of a row:
// only entries at least as good as the best of the lists' last entries can
// be in the global top-KMAX, so it gathers those (typically a few dozen)
// and ranks them exactly.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int MAXC = 256 * KMAX;  // candidate slots of the merge (n_lists <= 256)

int scan_chunks(int V) { return std::max(1, std::min(64, (V + 1023) / 1024)); }

// grid (chunks, rows), 128 threads: warp w of chunk c keeps the top-KMAX of
// its strided share of [c*len, (c+1)*len) and writes list c*4 + w.
__global__ void __launch_bounds__(128) topk_scan_kernel(const float* __restrict__ logits, int rows, int V, int len,
                                                        float mult, float cap, float* __restrict__ debug,
                                                        float* __restrict__ lists_v, int* __restrict__ lists_i) {
  const int c = blockIdx.x, row = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int v0 = c * len, v1 = min(V, v0 + len);
  float lv = -INFINITY, tv = -INFINITY;
  int li = INT_MAX, ti = INT_MAX;
  for (int base = v0 + warp * 32; base < v1; base += 128) {
    const int id = base + lane;
    float z = -INFINITY;
    const bool valid = id < v1;
    if (valid) {
      z = mult * logits[(size_t)row * V + id];
      if (cap > 0.f) z = cap * tanhf(z / cap);
      if (debug) debug[(size_t)row * V + id] = z;
    }
    unsigned mask = __ballot_sync(0xffffffffu, valid && beats(z, id, tv, ti));
    while (mask) {
      const int src = __ffs(mask) - 1;
      mask &= mask - 1;
      warp_list_offer(lv, li, tv, ti, __shfl_sync(0xffffffffu, z, src), base + src);
    }
  }
  if (lane < KMAX) {
    const size_t o = (((size_t)(c * 4 + warp)) * rows + row) * KMAX + lane;
    lists_v[o] = lv;
    lists_i[o] = li;
  }
}

__global__ void __launch_bounds__(256) topk_merge_kernel(const float* __restrict__ lists_v,
                                                         const int* __restrict__ lists_i, int n_lists, int rows,
                                                         int k, int32_t* __restrict__ cand_id,
                                                         float* __restrict__ cand_logit) {
  __shared__ float cv[MAXC];
  __shared__ int ci[MAXC];
  __shared__ float rv[32];
  __shared__ int ri[32];
  __shared__ int cnt;
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  // threshold = best of the lists' last entries
  float bv = -INFINITY;
  int bi = INT_MAX;
  for (int l = threadIdx.x; l < n_lists; l += blockDim.x) {
    const size_t o = ((size_t)l * rows + row) * KMAX + (KMAX - 1);
    const float v = lists_v[o];
    const int i = lists_i[o];
    if (beats(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
  for (int o = 16; o > 0; o >>= 1) {
    const float v = __shfl_xor_sync(0xffffffffu, bv, o);
    const int i = __shfl_xor_sync(0xffffffffu, bi, o);
    if (beats(v, i, bv, bi)) {
      bv = v;
      bi = i;
    }
  }
  if (lane == 0) {
    rv[warp] = bv;
    ri[warp] = bi;
  }
  if (threadIdx.x == 0) cnt = 0;
  __syncthreads();
  float tv = rv[0];
  int ti = ri[0];
  for (int w = 1; w < (int)(blockDim.x >> 5); ++w)
    if (beats(rv[w], ri[w], tv, ti)) {
      tv = rv[w];
      ti = ri[w];
    }
  // gather every real entry that is not beaten by the threshold
  for (int idx = threadIdx.x; idx < n_lists * KMAX; idx += blockDim.x) {
    const int l = idx / KMAX, e = idx % KMAX;
    const size_t o = ((size_t)l * rows + row) * KMAX + e;
    const float v = lists_v[o];
    const int i = lists_i[o];
    if (i != INT_MAX && !beats(tv, ti, v, i)) {
      const int p = atomicAdd(&cnt, 1);
      if (p < MAXC) {
        cv[p] = v;
        ci[p] = i;
      }
    }
  }
  __syncthreads();
  const int C = min(cnt, MAXC);
  for (int e = threadIdx.x; e < k; e += blockDim.x) {  // slots no candidate reaches stay empty
    cand_id[(size_t)row * k + e] = -1;
    cand_logit[(size_t)row * k + e] = -INFINITY;
  }
  __syncthreads();
  for (int a = threadIdx.x; a < C; a += blockDim.x) {
    int rank = 0;
    for (int b = 0; b < C; ++b) rank += beats(cv[b], ci[b], cv[a], ci[a]) ? 1 : 0;
    if (rank < k) {
      cand_id[(size_t)row * k + rank] = ci[a];
      cand_logit[(size_t)row * k + rank] = cv[a];
    }
  }
}

}  // namespace

int topk_scan_lists(int V) { return scan_chunks(V) * 4; }

int launch_topk_scan(const float* logits, int rows, int V, float mult, float cap, float* debug, float* lists_v,
                     int* lists_i, int* n_lists, const Ctx& c) {
  const int chunks = scan_chunks(V);
  const int len = (V + chunks - 1) / chunks;
  dim3 grid(chunks, rows);
  topk_scan_kernel<<<grid, 128, 0, c.stream>>>(logits, rows, V, len, mult, cap, debug, lists_v, lists_i);
  *n_lists = chunks * 4;
  count_launch();
  return cudaPeekAtLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

int launch_topk_merge(const float* lists_v, const int* lists_i, int n_lists, int rows, int k, int32_t* cand_id,
                      float* cand_logit, const Ctx& c) {
  if (n_lists > 256 || k > KMAX) return DFLASH2_ERR_SHAPE;
  topk_merge_kernel<<<rows, 256, 0, c.stream>>>(lists_v, lists_i, n_lists, rows, k, cand_id, cand_logit);
  count_launch();
  return cudaPeekAtLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

}  // namespace df2
