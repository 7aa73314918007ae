// DFlash 2 pairwise path selector ("Train a DFlash Drafter for Speculative
// Decoding", "Variants": pairwise scores between consecutive choices pick one
// of each position's top-k candidates so the picks form one consistent
// sequence; "Objective": trained by a cross-entropy over a position's top-k
// given the true predecessor; "Key Config Fields": selector_rank is its width).
//
// Reading implemented here: factors A = W_a E[tok] and Bf = W_b E[tok] of the
// shared embedding; transition score of candidate j at draft position i
// after predecessor p
//     S_i(p, j) = z_i[j] + <A[prev], Bf[c_ij]>,
//     T_i(p, j) = S_i(p, j) - logsumexp_j' S_i(p, j'),
// and the path maximising sum_i T_i (Viterbi, ties to the smaller
// predecessor index, then to the smaller final index).
//
// sel_gather_kernel lays out E rows of [anchor, all candidates] so the factor
// contraction runs on the same GEMM as the rest of the step; viterbi_kernel
// (one CTA per sequence) stages that sequence's factors, logits and
// candidate ids in shared memory and runs the k x k dynamic programme over
// the B-1 positions without touching global memory again.  With a factor
// table (the factors of every vocabulary token, built once), the kernel
// gathers the rows of its tokens itself and the gather and contraction
// launches drop out.
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

// x[r] = E[token of row r], rows = [anchor, cand(0,0..k-1), cand(1,..), ...]
// per sequence; 16-byte copies (H is a multiple of 8).
template <typename T>
__global__ void __launch_bounds__(256) sel_gather_kernel(const int32_t* __restrict__ anchor,
                                                         const int32_t* __restrict__ cand_id, int D, int k,
                                                         const T* __restrict__ E, int V, int H, T* __restrict__ x,
                                                         unsigned* status) {
  pdl_launch_next();
  pdl_wait();
  const int r = blockIdx.x;
  const int nt = D * k + 1;
  const int s = r / nt, t = r % nt;
  int tok = t == 0 ? anchor[s] : cand_id[(size_t)s * D * k + (t - 1)];
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_TOKEN);
    tok = -1;
  }
  constexpr int PER = 16 / sizeof(T);
  uint4* dst = reinterpret_cast<uint4*>(x + (size_t)r * H);
  const uint4* src = reinterpret_cast<const uint4*>(E + (size_t)(tok < 0 ? 0 : tok) * H);
  for (int m = threadIdx.x; m < H / PER; m += blockDim.x) dst[m] = tok < 0 ? make_uint4(0, 0, 0, 0) : src[m];
}

// Factors: Y [batch][nt][2r] rows in [anchor, candidates] order, or (Y
// null) rows of `table` [V][2r] at those tokens; neither (DFlash v1): no
// pairwise term, so the walk is the per-position top-1.
__global__ void __launch_bounds__(512) viterbi_kernel(const float* __restrict__ Y, const float* __restrict__ table,
                                                      const int32_t* __restrict__ anchor, int V,
                                                      const int32_t* __restrict__ cand_id,
                                                      const float* __restrict__ cand_logit, int D, int k, int r,
                                                      int32_t* __restrict__ path, float* __restrict__ path_score,
                                                      unsigned* status, int Dp, float log_p_min,
                                                      int32_t* __restrict__ n_draft) {
  extern __shared__ __align__(16) float sm[];
  __shared__ int tok0;
  pdl_launch_next();
  pdl_wait();
  const int s = blockIdx.x;
  // padded row stride: rows start on different banks; a multiple of 4 when
  // r is, so the dot products read float4s
  const int nt = D * k + 1, w = 2 * r, ws = (r & 3) == 0 ? w + 4 : w + 1;
  float* F = sm;                               // [nt][ws] factors: A = F[t][0:r], Bf = F[t][r:2r]
  float* zs = F + (size_t)nt * ws;             // [D][k] candidate logits
  float* Sm = zs + D * k;                      // [1 + (D-1)k][k] transition log-probabilities
  int* cid = reinterpret_cast<int*>(Sm + (1 + (D - 1) * k) * k);  // [D][k] candidate ids
  int* bp = cid + D * k;                       // [D][k] back pointers

  for (int idx = threadIdx.x; idx < D * k; idx += blockDim.x) {
    zs[idx] = cand_logit[(size_t)s * D * k + idx];
    cid[idx] = cand_id[(size_t)s * D * k + idx];
  }
  // stage the factors: U vector loads in flight per thread
  constexpr int U = 8;
  const bool pairwise = Y || table;
  if (!Y && table) {
    if (threadIdx.x == 0) tok0 = anchor[s];
    __syncthreads();
    // row t of the sequence's lattice: the anchor, then candidate t-1
    auto row_of = [&](int t) -> const float* {
      const int tok = t == 0 ? tok0 : cid[t - 1];
      if (tok < 0 || tok >= V) {
        flag(status, DFLASH2_DEV_BAD_TOKEN);
        return nullptr;
      }
      return table + (size_t)tok * w;
    };
    if ((w & 3) == 0) {
      const int w4 = w / 4, n4 = nt * w4;
      for (int base = threadIdx.x; base < n4; base += blockDim.x * U) {
        float4 v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int idx = base + u * blockDim.x;
          if (idx < n4) {
            const int t = idx / w4;
            const float* src = row_of(t);
            v[u] = src ? reinterpret_cast<const float4*>(src)[idx - t * w4] : make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int idx = base + u * blockDim.x;
          if (idx < n4) {
            const int t = idx / w4;
            *reinterpret_cast<float4*>(F + t * ws + (idx - t * w4) * 4) = v[u];
          }
        }
      }
    } else {
      for (int idx = threadIdx.x; idx < nt * w; idx += blockDim.x) {
        const int t = idx / w;
        const float* src = row_of(t);
        F[t * ws + idx - t * w] = src ? src[idx - t * w] : 0.f;
      }
    }
  } else if (Y && (w & 3) == 0) {
    const float4* y = reinterpret_cast<const float4*>(Y + (size_t)s * nt * w);
    const int w4 = w / 4, n4 = nt * w4;
    for (int base = threadIdx.x; base < n4; base += blockDim.x * U) {
      float4 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (base + u * blockDim.x < n4) v[u] = y[base + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx < n4) {
          const int t = idx / w4, c = (idx - t * w4) * 4;
          float* f = F + t * ws + c;
          f[0] = v[u].x;
          f[1] = v[u].y;
          f[2] = v[u].z;
          f[3] = v[u].w;
        }
      }
    }
  } else if (Y) {
    const float2* y = reinterpret_cast<const float2*>(Y + (size_t)s * nt * w);
    const int w2 = w / 2, n2 = nt * w2;
    for (int base = threadIdx.x; base < n2; base += blockDim.x * U) {
      float2 v[U];
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (base + u * blockDim.x < n2) v[u] = y[base + u * blockDim.x];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int idx = base + u * blockDim.x;
        if (idx < n2) {
          const int t = idx / w2, c = (idx - t * w2) * 2;
          F[t * ws + c] = v[u].x;
          F[t * ws + c + 1] = v[u].y;
        }
      }
    }
  }
  __syncthreads();
  // 1. every transition score at once (they do not depend on the DP): row 0 is
  //    position 1 after the anchor; row 1 + (i-1)k + p is position i+1 after
  //    candidate p of position i.  A thread computes a TS x TS tile (TS
  //    predecessors x TS candidates of one position): each factor it loads
  //    serves TS products, and the tiles spread over most of the CTA's threads.
  constexpr int TS = 2;
  const int nrow = 1 + (D - 1) * k;
  const int kt = (k + TS - 1) / TS;
  const int n_tiles = kt + (D - 1) * kt * kt;
  for (int tile = threadIdx.x; tile < n_tiles; tile += blockDim.x) {
    int i, p0, j0, np;
    if (tile < kt) {  // position 1: the anchor is the only predecessor
      i = 0;
      p0 = 0;
      np = 1;
      j0 = TS * tile;
    } else {
      const int t = tile - kt;
      i = 1 + t / (kt * kt);
      const int rem = t % (kt * kt);
      p0 = TS * (rem / kt);
      j0 = TS * (rem % kt);
      np = min(TS, k - p0);
    }
    const int nj = min(TS, k - j0);
    const float* arow[TS];
    const float* brow[TS];
#pragma unroll
    for (int a = 0; a < TS; ++a) {
      const int p = p0 + min(a, np - 1), j = j0 + min(a, nj - 1);  // clamped: spare lanes recompute an edge
      arow[a] = F + (size_t)(i == 0 ? 0 : 1 + (i - 1) * k + p) * ws;
      brow[a] = F + (size_t)(1 + i * k + j) * ws + r;
    }
    float acc[TS][TS];
#pragma unroll
    for (int a = 0; a < TS; ++a)
#pragma unroll
      for (int b = 0; b < TS; ++b) acc[a][b] = 0.f;
    if (!pairwise) {
      // no pairwise term: S = the candidate logits alone
    } else if ((r & 3) == 0) {
#pragma unroll 4
      for (int c = 0; c < r; c += 4) {
        float4 x[TS], y[TS];
#pragma unroll
        for (int a = 0; a < TS; ++a) {
          x[a] = *reinterpret_cast<const float4*>(arow[a] + c);
          y[a] = *reinterpret_cast<const float4*>(brow[a] + c);
        }
#pragma unroll
        for (int a = 0; a < TS; ++a)
#pragma unroll
          for (int b = 0; b < TS; ++b) {
            acc[a][b] = fmaf(x[a].x, y[b].x, acc[a][b]);
            acc[a][b] = fmaf(x[a].y, y[b].y, acc[a][b]);
            acc[a][b] = fmaf(x[a].z, y[b].z, acc[a][b]);
            acc[a][b] = fmaf(x[a].w, y[b].w, acc[a][b]);
          }
      }
    } else {
      for (int c = 0; c < r; ++c)
#pragma unroll
        for (int a = 0; a < TS; ++a)
#pragma unroll
          for (int b = 0; b < TS; ++b) acc[a][b] = fmaf(arow[a][c], brow[b][c], acc[a][b]);
    }
    const int row0 = i == 0 ? 0 : 1 + (i - 1) * k + p0;
#pragma unroll
    for (int a = 0; a < TS; ++a)
#pragma unroll
      for (int b = 0; b < TS; ++b)
        if (a < np && b < nj) Sm[(row0 + a) * k + j0 + b] = zs[i * k + j0 + b] + acc[a][b];
  }
  __syncthreads();
  // 2. each row -> log-probabilities (one half-warp per row, lane j of the
  //    half holds column j, k <= 16; shuffles stay in the half)
  {
    const int hw = threadIdx.x >> 4, j = threadIdx.x & 15, nhw = blockDim.x >> 4;
    const unsigned hmask = (threadIdx.x & 16) ? 0xffff0000u : 0x0000ffffu;
    for (int row = hw; row < nrow; row += nhw) {
      const float x = j < k ? Sm[row * k + j] : -INFINITY;
      float m = x;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(hmask, m, o));
      float sum = j < k ? expf(x - m) : 0.f;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) sum += __shfl_xor_sync(hmask, sum, o);
      const float lse = m + logf(sum);
      if (j < k) Sm[row * k + j] = x - lse;
    }
  }
  __syncthreads();
  // 3. the max-plus recurrence over the first Dp positions (draft_n_max):
  //    thread (j, p) of the first 256 forms delta[p] + T_i(p, j), and each
  //    half-warp (one j) reduces its 16 predecessors with shuffles, keeping
  //    the larger value and, on a tie, the smaller predecessor; then the
  //    backtrack and the cut at the first chosen transition whose
  //    log-probability is below log(p_min)
  __shared__ float dsm[2][16];
  if (threadIdx.x < 256) {
    const int j = threadIdx.x >> 4, p = threadIdx.x & 15;
    const unsigned hmask = (threadIdx.x & 16) ? 0xffff0000u : 0x0000ffffu;
    if (p == 0 && j < k) dsm[0][j] = Sm[j];
    asm volatile("bar.sync 1, 256;" ::: "memory");
    for (int i = 1; i < Dp; ++i) {
      const float* T = Sm + (1 + (i - 1) * k) * k;  // [p][j]
      float v = (p < k && j < k) ? dsm[(i - 1) & 1][p] + T[p * k + j] : -INFINITY;
      int arg = p;
#pragma unroll
      for (int o = 8; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(hmask, v, o);
        const int a2 = __shfl_xor_sync(hmask, arg, o);
        if (v2 > v || (v2 == v && a2 < arg)) {
          v = v2;
          arg = a2;
        }
      }
      if (p == 0 && j < k) {
        dsm[i & 1][j] = v;
        bp[i * k + j] = arg;
      }
      asm volatile("bar.sync 1, 256;" ::: "memory");
    }
    if (threadIdx.x == 0) {
      const float* dl = dsm[(Dp - 1) & 1];
      int jb = 0;
      float vb = dl[0];
      for (int jj = 1; jj < k; ++jj)
        if (dl[jj] > vb) {
          vb = dl[jj];
          jb = jj;
        }
      int js[32];
      int j = jb;
      for (int i = Dp - 1; i >= 0; --i) {
        js[i] = j;
        if (i > 0) j = bp[i * k + j];
      }
      // kept drafts: the walk stops before the first transition below p_min
      int n = 0;
      float score = 0.f;
      while (n < Dp) {
        const float t = Sm[(n == 0 ? 0 : 1 + (n - 1) * k + js[n - 1]) * k + js[n]];
        if (t < log_p_min) break;
        score += t;
        ++n;
      }
      if (log_p_min == -INFINITY) score = vb;  // no cut: the recurrence's own maximum
      for (int i = 0; i < D; ++i) path[(size_t)s * D + i] = i < n ? cid[i * k + js[i]] : -1;
      if (path_score) path_score[s] = score;
      if (n_draft) n_draft[s] = n;
    }
  }
}

}  // namespace

size_t viterbi_smem_bytes(int D, int k, int r) {
  const size_t ws = (r & 3) == 0 ? 2 * r + 4 : 2 * r + 1;
  return sizeof(float) * ((size_t)(D * k + 1) * ws + (size_t)D * k + (size_t)(1 + (D - 1) * k) * k) +
         sizeof(int) * 2 * (size_t)D * k;
}

int launch_sel_gather(int dtype, const int32_t* anchor, const int32_t* cand_id, int batch, int D, int k,
                      const void* embed, int V, int H, void* x_out, const Ctx& c) {
  const int rows = batch * (D * k + 1);
  if (dtype == DFLASH2_BF16)
    return launch_k(sel_gather_kernel<bf16>, dim3(rows), dim3(128), 0, c, anchor, cand_id, D, k,
                    static_cast<const bf16*>(embed), V, H, static_cast<bf16*>(x_out), c.status);
  return launch_k(sel_gather_kernel<float>, dim3(rows), dim3(128), 0, c, anchor, cand_id, D, k,
                  static_cast<const float*>(embed), V, H, static_cast<float*>(x_out), c.status);
}

int launch_viterbi(const float* Y, const float* table, const int32_t* anchor, int V, const int32_t* cand_id,
                   const float* cand_logit, int batch, int D, int k, int r, int32_t* path, float* path_score,
                   const Ctx& c, int n_max, float p_min, int32_t* n_draft) {
  if (Y && table) return DFLASH2_ERR_INVALID_ARG;
  if (n_max < 0 || !(p_min >= 0.f) || p_min > 1.f) return DFLASH2_ERR_SHAPE;
  // a request past the block is clamped to its B - 1 drafts ("DFlash2
  // Speculative Decoding" (llama-cpp-python wiki), "Configuration Notes")
  const int Dp = (n_max == 0 || n_max > D) ? D : n_max;
  const float log_p_min = p_min > 0.f ? logf(p_min) : -INFINITY;
  const size_t smem = viterbi_smem_bytes(D, k, r);
  static bool attr = false;
  if (!attr) {
    if (cudaFuncSetAttribute(viterbi_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) != cudaSuccess)
      return DFLASH2_ERR_CUDA;
    attr = true;
  }
  return launch_k(viterbi_kernel, dim3(batch), dim3(512), smem, c, Y, table, anchor, V, cand_id, cand_logit, D, k, r,
                  path, path_score, c.status, Dp, log_p_min, n_draft);
}

}  // namespace df2
