// Top-k candidates per block position ("DFlash2 Speculative Decoding"
// (llama-cpp-python wiki), "Configuration Notes": selector_top_k candidates
// per position; "Train a DFlash Drafter for Speculative Decoding", "Key
// Config Fields").  Order: larger logit first, equal logits by smaller id.
//
// The lm_head GEMM (tcgen05 path) already leaves one sorted list of KMAX
// entries per CTA and row.  topk_scan_kernel produces the same lists from
// stored logits (fp32 path).  topk_merge_kernel reduces the lists of a row:
// the 16th best list head bounds the answer from below, and one warp picks
// the top k of the entries it does not beat, so the result does not depend
// on how the vocabulary was split.
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

int scan_chunks(int V) { return std::max(1, std::min(64, (V + 1023) / 1024)); }

// grid (chunks, rows), 128 threads: warp w of chunk c keeps the top-KMAX of
// its strided share of [c*len, (c+1)*len) and writes list c*4 + w.
__global__ void __launch_bounds__(128) topk_scan_kernel(const float* __restrict__ logits, int rows, int V, int len,
                                                        float mult, float cap, float* __restrict__ debug,
                                                        float* __restrict__ lists_v, int* __restrict__ lists_i) {
  pdl_launch_next();
  pdl_wait();
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

// Top KMAX of `n` candidates (v[i], id[i]) in shared memory by one warp: a
// sorted list in lanes 0..15, offered only the candidates that beat its last
// entry (one ballot per 32 candidates).  Returns the list in (lv, li).
__device__ __forceinline__ void warp_topk(const float* v, const int* id, int n, float& lv, int& li, float& tv,
                                          int& ti) {
  const int lane = threadIdx.x & 31;
  lv = -INFINITY;
  li = INT_MAX;
  tv = -INFINITY;
  ti = INT_MAX;
  for (int base = 0; base < n; base += 32) {
    const int i = base + lane;
    const float x = i < n ? v[i] : -INFINITY;
    const int xi = i < n ? id[i] : INT_MAX;
    unsigned mask = __ballot_sync(0xffffffffu, i < n && beats(x, xi, tv, ti));
    while (mask) {
      const int src = __ffs(mask) - 1;
      mask &= mask - 1;
      warp_list_offer(lv, li, tv, ti, __shfl_sync(0xffffffffu, x, src), __shfl_sync(0xffffffffu, xi, src));
    }
  }
}

// One CTA per row.  The row's n_lists sorted lists are staged in shared
// memory in one round of loads.  The 16th best list head tau bounds the
// answer from below (16 distinct entries are at least tau), so only entries
// that tau does not beat can be in the top KMAX; those survivors are
// collected and one warp picks the top k of them.  The result is the exact
// top k under the strict (value, id) order, whatever the vocabulary split.
// dynamic shared memory: 2 * n_lists * KMAX * 8 bytes.
constexpr int MT = 512;  // threads of the merge kernel

__global__ void __launch_bounds__(MT) topk_merge_kernel(const float* __restrict__ lists_v,
                                                        const int* __restrict__ lists_i, int n_lists, int rows,
                                                        int k, int32_t* __restrict__ cand_id,
                                                        float* __restrict__ cand_logit) {
  extern __shared__ float mv[];
  __shared__ float tau_v;
  __shared__ int tau_i, n_surv;
  pdl_launch_next();
  pdl_wait();
  const int total = n_lists * KMAX;
  int* mi = reinterpret_cast<int*>(mv + total);
  float* sv = reinterpret_cast<float*>(mi + total);
  int* si = reinterpret_cast<int*>(sv + total);
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int U = 8;  // loads in flight per thread (n_lists <= 256: one round)
  for (int base = threadIdx.x; base < total; base += MT * U) {
    float v[U];
    int id[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * MT;
      if (idx < total) {
        const size_t o = ((size_t)(idx / KMAX) * rows + row) * KMAX + idx % KMAX;
        v[u] = lists_v[o];
        id[u] = lists_i[o];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * MT;
      if (idx < total) {
        mv[idx] = v[u];
        mi[idx] = id[u];
      }
    }
  }
  if (threadIdx.x == 0) n_surv = 0;
  __syncthreads();
  // tau: the KMAX-th best list head (heads are list entries 0, stride KMAX)
  if (warp == 0) {
    float lv, tv;
    int li, ti;
    // stage the heads contiguously in the survivor buffer, then select
    for (int l = lane; l < n_lists; l += 32) {
      sv[l] = mv[l * KMAX];
      si[l] = mi[l * KMAX];
    }
    __syncwarp();
    warp_topk(sv, si, n_lists, lv, li, tv, ti);
    if (lane == 0) {
      tau_v = n_lists >= KMAX ? tv : -INFINITY;
      tau_i = n_lists >= KMAX ? ti : INT_MAX;
    }
  }
  __syncthreads();
  // survivors: entries that tau does not beat
  const float tv0 = tau_v;
  const int ti0 = tau_i;
  for (int idx = threadIdx.x; idx < total; idx += MT) {
    const float v = mv[idx];
    const int id = mi[idx];
    if (!beats(tv0, ti0, v, id)) {
      const int p = atomicAdd(&n_surv, 1);
      sv[p] = v;
      si[p] = id;
    }
  }
  __syncthreads();
  if (warp == 0) {
    float lv, tv;
    int li, ti;
    warp_topk(sv, si, n_surv, lv, li, tv, ti);
    if (lane < k) {
      cand_id[(size_t)row * k + lane] = li == INT_MAX ? -1 : li;
      cand_logit[(size_t)row * k + lane] = lv;
    }
  }
}

}  // namespace

int topk_scan_lists(int V) { return scan_chunks(V) * 4; }

int launch_topk_scan(const float* logits, int rows, int V, float mult, float cap, float* debug, float* lists_v,
                     int* lists_i, int* n_lists, const Ctx& c) {
  const int chunks = scan_chunks(V);
  const int len = (V + chunks - 1) / chunks;
  *n_lists = chunks * 4;
  return launch_k(topk_scan_kernel, dim3(chunks, rows), dim3(128), 0, c, logits, rows, V, len, mult, cap,
                  debug, lists_v, lists_i);
}

int launch_topk_merge(const float* lists_v, const int* lists_i, int n_lists, int rows, int k, int32_t* cand_id,
                      float* cand_logit, const Ctx& c) {
  if (n_lists < 1 || n_lists > 256 || k > KMAX) return DFLASH2_ERR_SHAPE;
  const size_t smem = 2 * (size_t)n_lists * KMAX * 8;  // lists and survivors, <= 64 KB
  static bool attr = false;  // set once, before any capture
  if (!attr) {
    if (cudaFuncSetAttribute(topk_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 64 * 1024) !=
        cudaSuccess)
      return DFLASH2_ERR_CUDA;
    attr = true;
  }
  return launch_k(topk_merge_kernel, dim3(rows), dim3(MT), smem, c, lists_v, lists_i, n_lists, rows, k, cand_id,
                  cand_logit);
}

}  // namespace df2
