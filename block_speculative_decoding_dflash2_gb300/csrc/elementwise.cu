// Row kernels of the draft step that sit between the contractions: split-K
// reduction fused with the consumer (RMSNorm, q/k-norm + RoPE, paged K/V
// store, residual add, SiLU gate), the block embedding and the DFlash2
// dynamic convolution.  All are HBM/L2-light (a few rows of H values); they
// exist to keep each GEMM's epilogue simple and the stored activations bf16.
//
// Readings of the pages these kernels implement ("Train a DFlash Drafter for
// Speculative Decoding"):
//   "What is DFlash?"  block = [anchor, MASK...]; features from the target's
//                      tapped hidden states condition every draft layer
//                      (as extra keys/values: the context K/V written here);
//   "Variants"         the DFlash 2 two-tap in-block convolution around every
//                      sublayer (dyn_conv_kernel);
//   "Key Config Fields" input_embedding_scale, conv_group_size.
#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int RT = 256;  // threads of the row kernels

__device__ __forceinline__ float sum_parts(const float* P, int S, size_t stride, size_t idx) {
  float x = 0.f;
  for (int s = 0; s < S; ++s) x += P[(size_t)s * stride + idx];
  return x;
}

// f[n] = RMSNorm_hidden(sum_s P[s][n])  -- feature projection epilogue.
template <typename T>
__global__ void __launch_bounds__(RT) feature_norm_kernel(const float* __restrict__ P, int S, int rows, int H,
                                                          const T* __restrict__ gamma, float eps, T* __restrict__ f) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  const int n = blockIdx.x;
  const size_t stride = (size_t)rows * H;
  float ss = 0.f;
  for (int m = threadIdx.x; m < H; m += blockDim.x) {
    const float x = sum_parts(P, S, stride, (size_t)n * H + m);
    xs[m] = x;
    ss += x * x;
  }
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
  for (int m = threadIdx.x; m < H; m += blockDim.x) st(&f[(size_t)n * H + m], xs[m] * r * ld(&gamma[m]));
}

// Sequence that owns appended row n: the largest s with new_off[s] <= n.
__device__ __forceinline__ int owner_of(const int32_t* new_off, int batch, int n) {
  int lo = 0, hi = batch - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (new_off[mid] <= n) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Per-head RMSNorm + RoPE of one d-wide head held by a warp (d = 64 or 128:
// lane holds elements lane + 32 j); pair (i, i + d/2) lives in one lane.
template <typename T>
__device__ __forceinline__ void head_norm_rope(float (&x)[4], int d, const T* gamma, float eps, int pos,
                                               float theta) {
  const int lane = threadIdx.x & 31;
  const int nj = d / 32, hj = d / 64;
  float ss = 0.f;
  for (int j = 0; j < nj; ++j) ss += x[j] * x[j];
  const float r = rsqrtf(warp_sum(ss) / (float)d + eps);
  for (int j = 0; j < nj; ++j) x[j] *= r * ld(&gamma[lane + 32 * j]);
  for (int j = 0; j < hj; ++j) {
    float c, s;
    rope_cs(pos, lane + 32 * j, d, theta, &c, &s);
    const float x1 = x[j], x2 = x[j + hj];
    x[j] = x1 * c - x2 * s;
    x[j + hj] = x2 * c + x1 * s;
  }
}

// Context K/V of appended rows -> paged cache (one CTA per row, one warp per
// kv head): K = RoPE(RMSNorm_k(W_k f)), V = W_v f at the row's absolute position.
template <typename T>
__global__ void __launch_bounds__(RT) kv_append_kernel(const float* __restrict__ P, int S, int rows, int nkv, int d,
                                                       const T* __restrict__ k_norm, float eps, float theta,
                                                       const int32_t* __restrict__ ctx_len,
                                                       const int32_t* __restrict__ new_off, int batch,
                                                       const int32_t* __restrict__ block_table, int max_pages,
                                                       int page_size, int n_pages, T* __restrict__ kc,
                                                       T* __restrict__ vc, unsigned* status) {
  const int n = blockIdx.x;
  const int s = owner_of(new_off, batch, n);
  const int pos = ctx_len[s] + (n - new_off[s]);
  if (pos < 0 || pos >= max_pages * page_size) {
    if (threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
    return;
  }
  const int page = block_table[(size_t)s * max_pages + pos / page_size];
  if (page < 0 || page >= n_pages) {
    if (threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_PAGE);
    return;
  }
  const size_t dst = ((size_t)page * page_size + pos % page_size) * nkv * d;
  const int w2 = 2 * nkv * d;
  const size_t stride = (size_t)rows * w2;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nj = d / 32;
  for (int h = warp; h < nkv; h += nw) {
    float x[4];
    for (int j = 0; j < nj; ++j) x[j] = sum_parts(P, S, stride, (size_t)n * w2 + h * d + lane + 32 * j);
    head_norm_rope(x, d, k_norm, eps, pos, theta);
    for (int j = 0; j < nj; ++j) st(&kc[dst + h * d + lane + 32 * j], x[j]);
    for (int j = 0; j < nj; ++j)
      st(&vc[dst + h * d + lane + 32 * j], sum_parts(P, S, stride, (size_t)n * w2 + nkv * d + h * d + lane + 32 * j));
  }
}

// h[row] = scale * E[token], token = anchor (slot 0) or the mask id.
template <typename T>
__global__ void __launch_bounds__(RT) embed_block_kernel(const int32_t* __restrict__ anchor, int mask_id, int B,
                                                         const T* __restrict__ E, int V, int H, float scale,
                                                         float* __restrict__ h, unsigned* status) {
  const int row = blockIdx.x;
  const int s = row / B, i = row % B;
  int tok = i == 0 ? anchor[s] : mask_id;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_TOKEN);
    tok = -1;
  }
  for (int m = threadIdx.x; m < H; m += blockDim.x)
    h[(size_t)row * H + m] = tok < 0 ? 0.f : scale * ld(&E[(size_t)tok * H + m]);
}

// h[row] += sum_s P[s][row] (if P), then u = RMSNorm_gamma(h[row]).  With
// skip_anchor, block slot 0 is not written and the other rows are packed as
// [batch, B-1, H] (the lm_head input).
template <typename T>
__global__ void __launch_bounds__(RT) residual_norm_kernel(float* __restrict__ h, const float* __restrict__ P, int S,
                                                           int rows, int H, const T* __restrict__ gamma, float eps,
                                                           T* __restrict__ u, int B, int skip_anchor) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  const int row = blockIdx.x;
  const size_t stride = (size_t)rows * H;
  float ss = 0.f;
  for (int m = threadIdx.x; m < H; m += blockDim.x) {
    float x = h[(size_t)row * H + m];
    if (P != nullptr) {
      x += sum_parts(P, S, stride, (size_t)row * H + m);
      h[(size_t)row * H + m] = x;
    }
    xs[m] = x;
    ss += x * x;
  }
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
  int orow = row;
  if (skip_anchor) {
    const int s = row / B, i = row % B;
    if (i == 0) return;
    orow = s * (B - 1) + i - 1;
  }
  for (int m = threadIdx.x; m < H; m += blockDim.x) st(&u[(size_t)orow * H + m], xs[m] * r * ld(&gamma[m]));
}

// DFlash2 dynamic two-tap grouped convolution (one CTA per block row t):
//   alpha[g] = softmax(lambda[2g], lambda[2g+1]),  lambda = sum_s P[s][t]
//   u2[ch]   = u_t[ch] + alpha[g][0] u_t[ch] + alpha[g][1] u_{t-1}[ch]
// u_{t-1} = 0 at the anchor (block slot 0): the window stays inside the block.
template <typename T>
__global__ void __launch_bounds__(RT) dyn_conv_kernel(const T* __restrict__ u, const float* __restrict__ P, int S,
                                                      int rows, int H, int gs, int B, T* __restrict__ u2) {
  extern __shared__ float alpha[];  // [G][2]
  const int row = blockIdx.x;
  const int i = row % B;
  const int G = H / gs;
  const size_t stride = (size_t)rows * 2 * G;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const float l0 = sum_parts(P, S, stride, (size_t)row * 2 * G + 2 * g);
    const float l1 = sum_parts(P, S, stride, (size_t)row * 2 * G + 2 * g + 1);
    const float mx = fmaxf(l0, l1);
    const float e0 = expf(l0 - mx), e1 = expf(l1 - mx);
    const float inv = 1.f / (e0 + e1);
    alpha[2 * g] = e0 * inv;
    alpha[2 * g + 1] = e1 * inv;
  }
  __syncthreads();
  for (int m = threadIdx.x; m < H; m += blockDim.x) {
    const int g = m / gs;
    const float ut = ld(&u[(size_t)row * H + m]);
    const float up = i > 0 ? ld(&u[(size_t)(row - 1) * H + m]) : 0.f;
    st(&u2[(size_t)row * H + m], ut + alpha[2 * g] * ut + alpha[2 * g + 1] * up);
  }
}

// Block Q/K/V: reduce split-K partials, per-head RMSNorm + RoPE of q and k at
// the block positions (anchor at the context length after the append).
template <typename T>
__global__ void __launch_bounds__(RT) qkv_epi_kernel(const float* __restrict__ P, int S, int rows, int B, int nq,
                                                     int nkv, int d, const T* __restrict__ qn,
                                                     const T* __restrict__ kn, float eps, float theta,
                                                     const int32_t* __restrict__ ctx_len,
                                                     const int32_t* __restrict__ new_off, T* __restrict__ q,
                                                     T* __restrict__ kb, T* __restrict__ vb) {
  const int row = blockIdx.x;
  const int s = row / B, i = row % B;
  const int pos = ctx_len[s] + (new_off[s + 1] - new_off[s]) + i;
  const int w3 = (nq + 2 * nkv) * d;
  const size_t stride = (size_t)rows * w3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nj = d / 32;
  for (int hh = warp; hh < nq + nkv; hh += nw) {
    float x[4];
    for (int j = 0; j < nj; ++j) x[j] = sum_parts(P, S, stride, (size_t)row * w3 + hh * d + lane + 32 * j);
    head_norm_rope(x, d, hh < nq ? qn : kn, eps, pos, theta);
    T* dst = hh < nq ? q + (size_t)row * nq * d + hh * d : kb + (size_t)row * nkv * d + (hh - nq) * d;
    for (int j = 0; j < nj; ++j) st(&dst[lane + 32 * j], x[j]);
  }
  for (int e = threadIdx.x; e < nkv * d; e += blockDim.x)
    st(&vb[(size_t)row * nkv * d + e], sum_parts(P, S, stride, (size_t)row * w3 + (nq + nkv) * d + e));
}

// act = SiLU(gate) * up from the split-K partials of the stacked gate/up GEMM.
template <typename T>
__global__ void __launch_bounds__(RT) act_kernel(const float* __restrict__ P, int S, int rows, int I,
                                                 T* __restrict__ act) {
  const size_t total = (size_t)rows * I;
  const size_t stride = (size_t)rows * 2 * I;
  for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += (size_t)gridDim.x * blockDim.x) {
    const size_t row = idx / I, j = idx % I;
    const float g = sum_parts(P, S, stride, row * 2 * I + j);
    const float up = sum_parts(P, S, stride, row * 2 * I + I + j);
    st(&act[idx], g / (1.f + expf(-g)) * up);
  }
}

inline int check() {
  count_launch();
  return cudaPeekAtLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

}  // namespace

#define DF2_DISPATCH(dtype, ...)            \
  do {                                       \
    if ((dtype) == DFLASH2_BF16) {           \
      using T = bf16;                        \
      __VA_ARGS__;                           \
    } else {                                 \
      using T = float;                       \
      __VA_ARGS__;                           \
    }                                        \
  } while (0)

int launch_rows_feature_norm(int dtype, const float* P, int S, int rows, int H, const void* gamma, float eps,
                             void* f_out, const Ctx& c) {
  if (rows <= 0) return DFLASH2_OK;
  DF2_DISPATCH(dtype, feature_norm_kernel<T><<<rows, RT, H * sizeof(float), c.stream>>>(
                          P, S, rows, H, static_cast<const T*>(gamma), eps, static_cast<T*>(f_out)));
  return check();
}

int launch_kv_append(int dtype, const float* P, int S, int rows, int nkv, int d, const void* k_norm, float eps,
                     float theta, const int32_t* ctx_len, const int32_t* new_off, int batch,
                     const int32_t* block_table, int max_pages, int page_size, int n_pages, void* kc, void* vc,
                     const Ctx& c) {
  if (rows <= 0) return DFLASH2_OK;
  DF2_DISPATCH(dtype, kv_append_kernel<T><<<rows, RT, 0, c.stream>>>(
                          P, S, rows, nkv, d, static_cast<const T*>(k_norm), eps, theta, ctx_len, new_off, batch,
                          block_table, max_pages, page_size, n_pages, static_cast<T*>(kc), static_cast<T*>(vc),
                          c.status));
  return check();
}

int launch_embed_block(int dtype, const int32_t* anchor, int mask_id, int batch, int B, const void* embed, int V,
                       int H, float scale, float* h_out, const Ctx& c) {
  DF2_DISPATCH(dtype, embed_block_kernel<T><<<batch * B, RT, 0, c.stream>>>(
                          anchor, mask_id, B, static_cast<const T*>(embed), V, H, scale, h_out, c.status));
  return check();
}

int launch_residual_norm(int dtype, float* h, const float* P, int S, int rows, int H, const void* gamma, float eps,
                         void* u_out, int B, int skip_anchor, const Ctx& c) {
  DF2_DISPATCH(dtype, residual_norm_kernel<T><<<rows, RT, H * sizeof(float), c.stream>>>(
                          h, P, S, rows, H, static_cast<const T*>(gamma), eps, static_cast<T*>(u_out), B,
                          skip_anchor));
  return check();
}

int launch_dyn_conv(int dtype, const void* u, const float* P, int S, int rows, int H, int group_size, int B,
                    void* u2_out, const Ctx& c) {
  const int G = H / group_size;
  DF2_DISPATCH(dtype, dyn_conv_kernel<T><<<rows, RT, 2 * G * sizeof(float), c.stream>>>(
                          static_cast<const T*>(u), P, S, rows, H, group_size, B, static_cast<T*>(u2_out)));
  return check();
}

int launch_qkv_epilogue(int dtype, const float* P, int S, int rows, int B, int nq, int nkv, int d,
                        const void* q_norm, const void* k_norm, float eps, float theta, const int32_t* ctx_len,
                        const int32_t* new_off, void* q, void* kb, void* vb, const Ctx& c) {
  DF2_DISPATCH(dtype, qkv_epi_kernel<T><<<rows, RT, 0, c.stream>>>(
                          P, S, rows, B, nq, nkv, d, static_cast<const T*>(q_norm), static_cast<const T*>(k_norm),
                          eps, theta, ctx_len, new_off, static_cast<T*>(q), static_cast<T*>(kb),
                          static_cast<T*>(vb)));
  return check();
}

int launch_act(int dtype, const float* P, int S, int rows, int I, void* act, const Ctx& c) {
  const size_t total = (size_t)rows * I;
  const int blocks = (int)std::min<size_t>((total + RT - 1) / RT, (size_t)c.nsm * 8);
  DF2_DISPATCH(dtype, act_kernel<T><<<blocks, RT, 0, c.stream>>>(P, S, rows, I, static_cast<T*>(act)));
  return check();
}

}  // namespace df2
