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

// Sampled verification, one CTA per sequence (ST threads).  Thread 0 walks
// the acceptance draws; then the whole CTA draws the emitted token by an
// inverse CDF over row a of the target distribution (with path_a removed
// after a rejection): each thread sums a contiguous slice of the vocabulary
// in id order, a block scan of the slice sums finds the slice holding the
// threshold, and that slice's thread walks it to the token.
constexpr int ST = 256;

__global__ void __launch_bounds__(ST) verify_sampled_kernel(
    int B, int V, const int32_t* __restrict__ path, const int32_t* __restrict__ n_draft,
    const float* __restrict__ prob, const float* __restrict__ u_accept, const float* __restrict__ u_sample,
    int32_t* __restrict__ accept_len, int32_t* __restrict__ out_tok, int32_t* __restrict__ n_out,
    int32_t* __restrict__ next_anchor, int32_t* __restrict__ seq_len, int64_t* __restrict__ counters) {
  __shared__ int a_s, x_s, pick;
  __shared__ float part[ST];
  pdl_launch_next();
  pdl_wait();
  const int s = blockIdx.x, D = B - 1;
  const int nd = n_draft ? min(max(n_draft[s], 0), D) : D;
  const int32_t* p = path + (size_t)s * D;
  if (threadIdx.x == 0) {
    int a = 0;
    while (a < nd) {
      const int x = p[a];
      const float px = (x >= 0 && x < V) ? prob[((size_t)s * B + a) * V + x] : 0.f;
      if (!(u_accept[(size_t)s * D + a] < px)) break;
      ++a;
    }
    a_s = a;
    x_s = a < nd ? p[a] : -1;  // the rejected draft, removed from its row
    pick = -1;
  }
  __syncthreads();
  const int a = a_s, x = x_s;
  const float* row = prob + ((size_t)s * B + a) * V;
  const int per = (V + ST - 1) / ST;
  const int v0 = min(V, threadIdx.x * per), v1 = min(V, v0 + per);
  float sum = 0.f;
  for (int v = v0; v < v1; ++v) sum += v == x ? 0.f : row[v];
  part[threadIdx.x] = sum;
  __syncthreads();
  // inclusive scan of the slice sums in thread order (Hillis-Steele)
  for (int off = 1; off < ST; off <<= 1) {
    const float add = threadIdx.x >= off ? part[threadIdx.x - off] : 0.f;
    __syncthreads();
    part[threadIdx.x] += add;
    __syncthreads();
  }
  const float total = part[ST - 1];
  const float thr = u_sample[s] * total;
  const float before = threadIdx.x > 0 ? part[threadIdx.x - 1] : 0.f;
  if (before <= thr && thr < part[threadIdx.x] && v1 > v0) {
    float c = before;
    int v = v0;
    for (; v < v1; ++v) {
      c += v == x ? 0.f : row[v];
      if (thr < c) break;
    }
    pick = min(v, v1 - 1);
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
  return launch_k(verify_sampled_kernel, dim3(batch), dim3(ST), 0, c, B, V, path, n_draft, prob, u_accept, u_sample,
                  accept_len, out_tok, n_out, next_anchor, seq_len, counters);
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
