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

}  // namespace

int launch_verify(int batch, int B, const int32_t* path, const int32_t* n_draft, const int32_t* target,
                  int32_t* accept_len, int32_t* out_tok, int32_t* n_out, int32_t* next_anchor, int32_t* seq_len,
                  int64_t* counters, cudaStream_t st) {
  const int threads = 128;
  const Ctx c{st, nullptr, 0, true};
  return launch_k(verify_kernel, dim3((batch + threads - 1) / threads), dim3(threads), 0, c, batch, B, path, n_draft,
                  target, accept_len, out_tok, n_out, next_anchor, seq_len, counters);
}

}  // namespace df2
