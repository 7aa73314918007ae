// Greedy verification, accept and rollback ("DFlash2 Speculative Decoding"
// (llama-cpp-python wiki), "Prerequisites": the target verifies
// [id_last, draft...] in one batch; "DFlash speculative decoding with vLLM",
// "Validation": the generated token ids equal plain greedy decoding; "DFlash2
// Speculative Decoding | NVIDIA NIM for Alpamayo Documentation", "Observe
// Acceptance": the counters and their identities).
//
// target[s][i] is the target's greedy token after [anchor, path_1..path_i].
// The longest prefix with path == target (of the n_draft[s] drafts kept, all
// B-1 without n_draft) is accepted, the target's own next token is emitted
// after it and becomes the next anchor; the rejected suffix is rolled back by
// advancing the sequence length only by a + 1.
#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

__global__ void verify_kernel(int batch, int B, const int32_t* __restrict__ path, const int32_t* __restrict__ n_draft,
                              const int32_t* __restrict__ target,
                              int32_t* __restrict__ accept_len, int32_t* __restrict__ out_tok,
                              int32_t* __restrict__ n_out, int32_t* __restrict__ next_anchor,
                              int32_t* __restrict__ seq_len, int64_t* __restrict__ counters) {
  pdl_launch_next();
  pdl_wait();
  const int s = blockIdx.x * blockDim.x + threadIdx.x;
  if (s >= batch) return;
  const int D = B - 1;
  const int nd = n_draft ? min(max(n_draft[s], 0), D) : D;
  const int32_t* p = path + (size_t)s * D;
  const int32_t* t = target + (size_t)s * B;
  int a = 0;
  while (a < nd && p[a] == t[a]) ++a;
  for (int i = 0; i < B; ++i) out_tok[(size_t)s * B + i] = i < a ? p[i] : (i == a ? t[a] : -1);
  accept_len[s] = a;
  n_out[s] = a + 1;
  next_anchor[s] = t[a];
  if (seq_len) seq_len[s] += a + 1;
  if (counters) {
    unsigned long long* c = reinterpret_cast<unsigned long long*>(counters);
    atomicAdd(c + 0, 1ull);
    atomicAdd(c + 1, (unsigned long long)nd);
    atomicAdd(c + 2, (unsigned long long)a);
    atomicAdd(c + 3, (unsigned long long)(nd - a));
    atomicAdd(c + 4 + a, 1ull);
    for (int i = 0; i < a; ++i) atomicAdd(c + 4 + B + i, 1ull);
  }
}

// Sampled verification, one CTA per sequence (ST threads).  The acceptance
// draws are compared in parallel (one thread per draft) and thread 0 takes
// the first rejection.  The emitted token is then drawn by an inverse CDF
// over row a of the target distribution (with path_a removed after a
// rejection), in id order:
//   1. the row is cut into segments of 128 ids; warp w sums segments w,
//      w + SW, ... (lane l holds ids 4l..4l+3 of a segment: one float4 load
//      when the row is 16-byte aligned, so every load of a warp is
//      coalesced, and several segments' loads are in flight at once);
//   2. a block scan of the segment sums finds the segment holding the
//      threshold u * total;
//   3. one warp walks that segment: lane prefix sums by shuffles, then each
//      lane its own four ids.
constexpr int ST = 512, SW = ST / 32, SEG = 128;
// segment sums in dynamic shared memory, within the 48 KB a block gets without
// opting in (with the static arrays): V <= 1,536,000
constexpr int kSampledMaxSeg = 12000;

// The four ids 4*lane .. 4*lane+3 of segment g of the row (0 past V or at x).
__device__ __forceinline__ float4 seg_load(const float* row, int V, int x, bool vec, int g, int lane) {
  const int v0 = g * SEG + 4 * lane;
  float4 q;
  if (vec && v0 + 3 < V) {
    q = __ldcg(reinterpret_cast<const float4*>(row + v0));
  } else {
    q.x = v0 < V ? __ldcg(row + v0) : 0.f;
    q.y = v0 + 1 < V ? __ldcg(row + v0 + 1) : 0.f;
    q.z = v0 + 2 < V ? __ldcg(row + v0 + 2) : 0.f;
    q.w = v0 + 3 < V ? __ldcg(row + v0 + 3) : 0.f;
  }
  if (x >= v0 && x < v0 + 4) {
    if (x == v0) q.x = 0.f;
    else if (x == v0 + 1) q.y = 0.f;
    else if (x == v0 + 2) q.z = 0.f;
    else q.w = 0.f;
  }
  return q;
}

__global__ void __launch_bounds__(ST) verify_sampled_kernel(
    int B, int V, const int32_t* __restrict__ path, const int32_t* __restrict__ n_draft,
    const float* __restrict__ prob, const float* __restrict__ u_accept, const float* __restrict__ u_sample,
    int32_t* __restrict__ accept_len, int32_t* __restrict__ out_tok, int32_t* __restrict__ n_out,
    int32_t* __restrict__ next_anchor, int32_t* __restrict__ seq_len, int64_t* __restrict__ counters) {
  extern __shared__ float segsum[];  // [nseg]
  __shared__ int a_s, x_s, pick, gsel, claim;
  __shared__ int ok[32];
  __shared__ float wsum[SW], woff[SW + 1], gbefore;
  pdl_launch_next();
  pdl_wait();
  const int s = blockIdx.x, D = B - 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nd = n_draft ? min(max(n_draft[s], 0), D) : D;
  const int32_t* p = path + (size_t)s * D;
  if (threadIdx.x < 32) {  // draft i accepted when its draw is below p_i(path_i)
    const int i = threadIdx.x;
    bool acc = false;
    if (i < nd) {
      const int xi = p[i];
      const float px = (xi >= 0 && xi < V) ? prob[((size_t)s * B + i) * V + xi] : 0.f;
      acc = u_accept[(size_t)s * D + i] < px;
    }
    ok[i] = acc ? 1 : 0;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int a = 0;
    while (a < nd && ok[a]) ++a;
    a_s = a;
    x_s = a < nd ? p[a] : -1;  // the rejected draft, removed from its row
    pick = -1;
    gsel = -1;
    claim = ST;
  }
  __syncthreads();
  const int a = a_s, x = x_s;
  const float* row = prob + ((size_t)s * B + a) * V;
  const bool vec = (reinterpret_cast<uintptr_t>(row) & 15) == 0;
  const int nseg = (V + SEG - 1) / SEG;
  // 1. segment sums, four segments of a warp in flight at once
  for (int g0 = warp; g0 < nseg; g0 += 4 * SW) {
    float4 q[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int g = g0 + u * SW;
      q[u] = g < nseg ? seg_load(row, V, x, vec, g, lane) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      float t = (q[u].x + q[u].y) + (q[u].z + q[u].w);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
      const int g = g0 + u * SW;
      if (lane == 0 && g < nseg) segsum[g] = t;
    }
  }
  __syncthreads();
  // 2. block scan: thread t owns segments [t*per, (t+1)*per).  Each range's
  //    start is the previous range's end as the same float expression (warp
  //    offsets chained serially), so the ranges tile [0, total) without gaps
  //    and exactly one thread holds the threshold.
  const int per = (nseg + ST - 1) / ST;
  const int ga = min(nseg, threadIdx.x * per), gb = min(nseg, ga + per);
  float mine = 0.f;
  for (int g = ga; g < gb; ++g) mine += segsum[g];
  float inc = mine;  // inclusive scan over the warp's lanes
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float y = __shfl_up_sync(0xffffffffu, inc, o);
    if (lane >= o) inc += y;
  }
  float excl = __shfl_up_sync(0xffffffffu, inc, 1);
  if (lane == 0) excl = 0.f;
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  if (threadIdx.x == 0) {  // warp offsets, chained
    float o = 0.f;
    for (int w = 0; w < SW; ++w) {
      const float t = wsum[w];
      woff[w] = o;
      o = o + t;
    }
    woff[SW] = o;
  }
  __syncthreads();
  const float total = woff[SW];
  const float thr = u_sample[s] * total;
  const float before = woff[warp] + excl, end = woff[warp] + inc;
  // (rounding can make a near-empty range overlap its neighbour: the first
  // claiming thread wins, so the draw is deterministic)
  if (before <= thr && thr < end) atomicMin(&claim, (int)threadIdx.x);
  __syncthreads();
  if ((int)threadIdx.x == claim) {
    float c = before, cl = before;
    int gl = -1;
    for (int g = ga; g < gb; ++g) {
      if (segsum[g] > 0.f) {
        gl = g;
        cl = c;
      }
      if (thr < c + segsum[g]) break;
      c += segsum[g];
    }
    // rounding may leave thr past the range's own sums (then the last
    // segment with mass in it), or the range may hold no mass at all (then
    // the next segment with mass)
    for (int g = gb; gl < 0 && g < nseg; ++g)
      if (segsum[g] > 0.f) {
        gl = g;
        cl = c;
      }
    gsel = gl;
    gbefore = cl;
  }
  __syncthreads();
  // 3. the selected segment, one warp
  if (warp == 0 && gsel >= 0) {
    const int g = gsel;
    const float4 q = seg_load(row, V, x, vec, g, lane);
    const float ls = (q.x + q.y) + (q.z + q.w);
    float li = ls;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const float y = __shfl_up_sync(0xffffffffu, li, o);
      if (lane >= o) li += y;
    }
    float c = gbefore + (li - ls);
    const float e[4] = {q.x, q.y, q.z, q.w};
    int hit = -1, last = -1;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      c += e[j];
      if (e[j] > 0.f) last = j;
      if (hit < 0 && e[j] > 0.f && thr < c) hit = j;  // never a token without mass
    }
    const unsigned hm = __ballot_sync(0xffffffffu, hit >= 0);
    if (hm) {
      const int src = __ffs(hm) - 1;
      const int j = __shfl_sync(0xffffffffu, hit, src);
      if (lane == 0) pick = g * SEG + 4 * src + j;
    } else {
      // rounding left the threshold past the segment's last id with mass
      const unsigned lm = __ballot_sync(0xffffffffu, last >= 0);
      if (lm) {
        const int src = 31 - __clz(lm);
        const int j = __shfl_sync(0xffffffffu, last, src);
        if (lane == 0) pick = g * SEG + 4 * src + j;
      }
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int v = pick;
    if (v < 0) {  // rounding left the threshold at the top: the last token with mass
      v = V - 1;
      while (v > 0 && (v == x || row[v] <= 0.f)) --v;
    }
    for (int i = 0; i < B; ++i) out_tok[(size_t)s * B + i] = i < a ? p[i] : (i == a ? v : -1);
    accept_len[s] = a;
    n_out[s] = a + 1;
    next_anchor[s] = v;
    if (seq_len) seq_len[s] += a + 1;
    if (counters) {
      unsigned long long* c = reinterpret_cast<unsigned long long*>(counters);
      atomicAdd(c + 0, 1ull);
      atomicAdd(c + 1, (unsigned long long)nd);
      atomicAdd(c + 2, (unsigned long long)a);
      atomicAdd(c + 3, (unsigned long long)(nd - a));
      atomicAdd(c + 4 + a, 1ull);
      for (int i = 0; i < a; ++i) atomicAdd(c + 4 + B + i, 1ull);
    }
  }
}

}  // namespace

int launch_verify_sampled(int batch, int B, int V, const int32_t* path, const int32_t* n_draft, const float* prob,
                          const float* u_accept, const float* u_sample, int32_t* accept_len, int32_t* out_tok,
                          int32_t* n_out, int32_t* next_anchor, int32_t* seq_len, int64_t* counters,
                          cudaStream_t st) {
  const Ctx c{st, nullptr, 0, true};
  const int nseg = (V + SEG - 1) / SEG;
  if (nseg > kSampledMaxSeg) return DFLASH2_ERR_SHAPE;
  return launch_k(verify_sampled_kernel, dim3(batch), dim3(ST), (size_t)nseg * sizeof(float), c, B, V, path, n_draft,
                  prob, u_accept, u_sample, accept_len, out_tok, n_out, next_anchor, seq_len, counters);
}

int launch_verify(int batch, int B, const int32_t* path, const int32_t* n_draft, const int32_t* target,
                  int32_t* accept_len, int32_t* out_tok, int32_t* n_out, int32_t* next_anchor, int32_t* seq_len,
                  int64_t* counters, cudaStream_t st) {
  const int threads = 128;
  const Ctx c{st, nullptr, 0, true};
  return launch_k(verify_kernel, dim3((batch + threads - 1) / threads), dim3(threads), 0, c, batch, B, path, n_draft,
                  target, accept_len, out_tok, n_out, next_anchor, seq_len, counters);
}

}  // namespace df2
