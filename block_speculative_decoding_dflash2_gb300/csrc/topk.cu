// Top-k candidates per block position ("DFlash2 Speculative Decoding"
// (llama-cpp-python wiki), "Configuration Notes": selector_top_k candidates
// per position; "Train a DFlash Drafter for Speculative Decoding", "Key
// Config Fields").  Order: larger logit first, equal logits by smaller id.
//
// The lm_head GEMM (tcgen05 path) already leaves one sorted list of KMAX
// entries per CTA and row.  topk_scan_kernel produces the same lists from
// stored logits (fp32 path).  topk_merge_kernel reduces the lists of a row
// with a tree of two-list merges in shared memory; each merge ranks every
// entry of both lists against the other in one warp, so the result does not
// depend on how the vocabulary was split.
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

// Merges sorted lists a (lanes 0..15 hold a[lane]) and b (lanes 16..31 hold
// b[lane-16]) into the best KMAX, written to out_v/out_i[0..KMAX).  An entry's
// rank in the union is its index in its own list plus the number of entries
// of the other list that beat it (the order is strict: ids are distinct).
__device__ __forceinline__ void warp_merge2(float v, int id, float* out_v, int* out_i) {
  const int lane = threadIdx.x & 31;
  const int other = lane < KMAX ? KMAX : 0;
  int rank = lane & (KMAX - 1);
#pragma unroll
  for (int t = 0; t < KMAX; ++t) {
    const float ov = __shfl_sync(0xffffffffu, v, other + t);
    const int oi = __shfl_sync(0xffffffffu, id, other + t);
    rank += beats(ov, oi, v, id) ? 1 : 0;
  }
  __syncwarp();
  if (rank < KMAX) {
    out_v[rank] = v;
    out_i[rank] = id;
  }
  __syncwarp();
}

// One CTA per row.  The row's n_lists lists are staged in shared memory and
// merged pairwise, level by level (list 2j absorbs list 2j+1), one warp per
// pair.  dynamic shared memory: n_lists * KMAX * 8 bytes.
__global__ void __launch_bounds__(256) topk_merge_kernel(const float* __restrict__ lists_v,
                                                         const int* __restrict__ lists_i, int n_lists, int rows,
                                                         int k, int32_t* __restrict__ cand_id,
                                                         float* __restrict__ cand_logit) {
  extern __shared__ float mv[];
  pdl_launch_next();
  pdl_wait();
  int* mi = reinterpret_cast<int*>(mv + n_lists * KMAX);
  const int row = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  constexpr int U = 8;  // loads in flight per thread
  for (int base = threadIdx.x; base < n_lists * KMAX; base += blockDim.x * U) {
    float v[U];
    int id[U];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx < n_lists * KMAX) {
        const size_t o = ((size_t)(idx / KMAX) * rows + row) * KMAX + idx % KMAX;
        v[u] = lists_v[o];
        id[u] = lists_i[o];
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int idx = base + u * blockDim.x;
      if (idx < n_lists * KMAX) {
        mv[idx] = v[u];
        mi[idx] = id[u];
      }
    }
  }
  __syncthreads();
  for (int stride = 1; stride < n_lists; stride *= 2) {
    for (int a = warp * 2 * stride; a < n_lists; a += nw * 2 * stride) {
      const int b = a + stride;
      if (b >= n_lists) continue;  // odd list out: carried to the next level as is
      const int src = lane < KMAX ? a : b;
      const float v = mv[src * KMAX + (lane & (KMAX - 1))];
      const int id = mi[src * KMAX + (lane & (KMAX - 1))];
      __syncwarp();
      warp_merge2(v, id, mv + a * KMAX, mi + a * KMAX);
    }
    __syncthreads();
  }
  for (int e = threadIdx.x; e < k; e += blockDim.x) {
    const int id = mi[e];
    cand_id[(size_t)row * k + e] = id == INT_MAX ? -1 : id;
    cand_logit[(size_t)row * k + e] = mv[e];
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
  const size_t smem = (size_t)n_lists * KMAX * 8;  // <= 32 KB
  return launch_k(topk_merge_kernel, dim3(rows), dim3(256), smem, c, lists_v, lists_i, n_lists, rows, k,
                  cand_id, cand_logit);
}

}  // namespace df2
