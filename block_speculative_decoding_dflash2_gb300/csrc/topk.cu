// Top-k candidates per block position ("DFlash2 Speculative Decoding"
// (llama-cpp-python wiki), "Configuration Notes": selector_top_k candidates
// per position; "Train a DFlash Drafter for Speculative Decoding", "Key
// Config Fields").  Order: larger logit first, equal logits by smaller id.
//
// The lm_head GEMM (tcgen05 path) already leaves one sorted list of KMAX
// entries per CTA and row.  topk_scan_kernel produces the same lists from
// stored logits (fp32 path).  topk_merge_kernel reduces the lists of a row:
// the 16th best list head bounds the answer from below, and the top k of the
// entries it does not beat are found by counting ranks, so the result does
// not depend on how the vocabulary was split.
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

// Rank of key x at slot sx among keys[0..n) in shared memory: the keys above
// it, plus the equal ones (padding entries) at smaller slots.  One thread per
// key ranked: the threads of a warp read the same key at once (a broadcast).
__device__ __forceinline__ int rank_of(const unsigned long long* keys, int n, unsigned long long x, int sx) {
  int rank = 0;
#pragma unroll 8
  for (int m = 0; m < n; ++m) {
    const unsigned long long y = keys[m];
    rank += (y > x) | ((y == x) & (m < sx));
  }
  return rank;
}

// One CTA per row.  The row's n_lists sorted lists are staged in shared
// memory in one round of loads.  The KMAX-th best list head tau bounds the
// answer from below (KMAX distinct entries are at least tau), so only
// entries that tau does not beat can be in the top KMAX.  Both selections
// are rank counts over 64-bit order keys (a warp per element counts the
// elements above it): tau is the head of rank KMAX-1, and a survivor of rank
// q < k is output q.  The result is the exact top k under the strict
// (value, id) order, whatever the vocabulary split.  Each rank is counted by
// one thread over keys read from shared memory as broadcasts.
// dynamic shared memory: 2 * n_lists * KMAX * 8 bytes.
constexpr int MT = 512;  // threads of the merge kernel

__global__ void __launch_bounds__(MT) topk_merge_kernel(const float* __restrict__ lists_v,
                                                        const int* __restrict__ lists_i, int n_lists, int rows,
                                                        int k, int32_t* __restrict__ cand_id,
                                                        float* __restrict__ cand_logit) {
  extern __shared__ __align__(16) unsigned long long mk[];  // [total] keys of the list entries
  __shared__ unsigned long long hk[256];                     // keys of the list heads
  __shared__ unsigned long long tau;
  __shared__ int n_surv;
  pdl_launch_next();
  pdl_wait();
  const int total = n_lists * KMAX;
  unsigned long long* sk = mk + total;                     // [total] survivor keys
  const int row = blockIdx.x;
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
        const unsigned long long key = order_key(v[u], id[u]);
        mk[idx] = key;
        if (idx % KMAX == 0) hk[idx / KMAX] = key;
      }
    }
  }
  if (threadIdx.x == 0) {
    n_surv = 0;
    tau = 0;  // fewer than KMAX lists: every entry survives
  }
  __syncthreads();
  // tau: the list head of rank KMAX-1
  if (n_lists >= KMAX)
    for (int l = threadIdx.x; l < n_lists; l += MT)
      if (rank_of(hk, n_lists, hk[l], l) == KMAX - 1) tau = hk[l];
  __syncthreads();
  // survivors: entries whose key is at least tau's
  const unsigned long long t0 = tau;
  for (int idx = threadIdx.x; idx < total; idx += MT) {
    const unsigned long long key = mk[idx];
    if (key >= t0) {
      sk[atomicAdd(&n_surv, 1)] = key;
    }
  }
  __syncthreads();
  const int ns = n_surv;
  for (int q = ns + threadIdx.x; q < k; q += MT) {  // fewer survivors than k (tiny vocabularies)
    cand_id[(size_t)row * k + q] = -1;
    cand_logit[(size_t)row * k + q] = -INFINITY;
  }
  for (int i = threadIdx.x; i < ns; i += MT) {
    const unsigned long long key = sk[i];
    const int rank = rank_of(sk, ns, key, i);
    if (rank < k) {
      const int id = key_id(key);
      cand_id[(size_t)row * k + rank] = id == INT_MAX ? -1 : id;
      cand_logit[(size_t)row * k + rank] = key_value(key);
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
  const size_t smem = 2 * (size_t)n_lists * KMAX * 8;  // entry and survivor keys, <= 64 KB
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
