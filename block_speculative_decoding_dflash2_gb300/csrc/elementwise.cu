// Row kernels of the draft step that sit between the contractions: the
// consumers of each GEMM's final fp32 output (RMSNorm, q/k-norm + RoPE, paged
// K/V store, SiLU gate), the block embedding and the DFlash2 dynamic
// convolution.  Each touches a few rows of H values: they are latency-bound,
// so every load is a 16-byte vector and the per-row RoPE angles are computed
// once per row, not per head.
//
// Readings of the pages these kernels implement ("Train a DFlash Drafter for
// Speculative Decoding"):
//   "What is DFlash?"  block = [anchor, MASK...]; features from the target's
//                      tapped hidden states condition every draft layer
//                      (as extra keys/values: the context K/V written here);
//   "Variants"         the DFlash 2 two-tap in-block convolution around every
//                      sublayer (dyn_conv_kernel);
//   "Key Config Fields" input_embedding_scale, conv_group_size.
#include <algorithm>
#include <cmath>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int RT = 256;  // threads of the row kernels

// ---------------------------------------------------------------- vector I/O
// 4 consecutive elements of T as floats / back (H, d, I are multiples of 8).
template <typename T> __device__ __forceinline__ float4 ld4(const T* p);
template <> __device__ __forceinline__ float4 ld4<float>(const float* p) { return *reinterpret_cast<const float4*>(p); }
template <> __device__ __forceinline__ float4 ld4<bf16>(const bf16* p) {
  const uint2 u = *reinterpret_cast<const uint2*>(p);
  const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&u.x);
  const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&u.y);
  const float2 fa = __bfloat1622float2(a), fb = __bfloat1622float2(b);
  return make_float4(fa.x, fa.y, fb.x, fb.y);
}
template <typename T> __device__ __forceinline__ void st4(T* p, float4 v);
template <> __device__ __forceinline__ void st4<float>(float* p, float4 v) { *reinterpret_cast<float4*>(p) = v; }
template <> __device__ __forceinline__ void st4<bf16>(bf16* p, float4 v) {
  __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y), b = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<uint32_t*>(&a);
  u.y = *reinterpret_cast<uint32_t*>(&b);
  *reinterpret_cast<uint2*>(p) = u;
}

__device__ __forceinline__ float4 scale4(float4 x, float r, float4 g) {
  return make_float4(x.x * r * g.x, x.y * r * g.y, x.z * r * g.z, x.w * r * g.w);
}

// RMSNorm of one row held in shared memory as fp32 x[H]; writes u = x*r*gamma.
template <typename T>
__device__ __forceinline__ void norm_row(const float* xs, int H, const T* gamma, float eps, T* u, float* red) {
  float ss = 0.f;
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4) {
    const float4 x = *reinterpret_cast<const float4*>(xs + m);
    ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
  }
  const float r = rsqrtf(block_sum(ss, red) / (float)H + eps);
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4)
    st4(u + m, scale4(*reinterpret_cast<const float4*>(xs + m), r, ld4(gamma + m)));
}

// ---------------------------------------------------------------- rope
// cos/sin of position pos for rotary pair i of a d-wide head:
// angle = pos * theta^(-2i/d).  The angle is formed and reduced modulo 2*pi
// in double (a few operations), then sincosf of the reduced fp32 angle, so
// long contexts keep full fp32 accuracy.
__device__ __forceinline__ void rope_cs(int pos, int i, int d, double log2_theta, float* c, float* s) {
  const double inv = exp2(-(2.0 * (double)i / (double)d) * log2_theta);
  double a = (double)pos * inv;
  a -= 6.283185307179586 * rint(a * 0.15915494309189535);
  sincosf((float)a, s, c);
}

// Per-head RMSNorm + RoPE of one d-wide head held by a warp: lane holds
// elements lane + 32 j (j < d/32); pair (i, i + d/2) lives in one lane, and
// cs/sn hold that lane's pair angles (j < d/64).
template <typename T>
__device__ __forceinline__ void head_norm_rope(float (&x)[4], int d, const T* gamma, float eps, const float* cs,
                                               const float* sn) {
  const int lane = threadIdx.x & 31;
  const int nj = d / 32, hj = d / 64;
  float ss = 0.f;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nj) ss += x[j] * x[j];
  const float r = rsqrtf(warp_sum(ss) / (float)d + eps);
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nj) x[j] *= r * ld(&gamma[lane + 32 * j]);
#pragma unroll
  for (int j = 0; j < 2; ++j)
    if (j < hj) {
      const float x1 = x[j], x2 = x[j + hj];
      x[j] = x1 * cs[j] - x2 * sn[j];
      x[j + hj] = x2 * cs[j] + x1 * sn[j];
    }
}

// ---------------------------------------------------------------- kernels

// f[n] = RMSNorm_hidden(Y[n])  -- feature projection epilogue.
template <typename T>
__global__ void __launch_bounds__(RT) feature_norm_kernel(const float* __restrict__ Y, int H,
                                                          const T* __restrict__ gamma, float eps, T* __restrict__ f) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  pdl_launch_next();
  pdl_wait();
  const size_t n = blockIdx.x;
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4)
    *reinterpret_cast<float4*>(xs + m) = *reinterpret_cast<const float4*>(Y + n * H + m);
  norm_row(xs, H, gamma, eps, f + n * H, red);
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

// Context K/V of appended rows -> paged cache (one CTA per row, one warp per
// kv head): K = RoPE(RMSNorm_k(W_k f)), V = W_v f at the row's absolute position.
template <typename T>
__global__ void __launch_bounds__(RT) kv_append_kernel(const float* __restrict__ Y, int nkv, int d,
                                                       const T* __restrict__ k_norm, float eps, double log2_theta,
                                                       const int32_t* __restrict__ ctx_len,
                                                       const int32_t* __restrict__ new_off, int batch,
                                                       const int32_t* __restrict__ block_table, int max_pages,
                                                       int page_size, int n_pages, T* __restrict__ kc,
                                                       T* __restrict__ vc, unsigned* status) {
  pdl_launch_next();
  pdl_wait();
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
  const float* y = Y + (size_t)n * 2 * nkv * d;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nj = d / 32;
  float cs[2], sn[2];
  for (int j = 0; j < d / 64; ++j) rope_cs(pos, lane + 32 * j, d, log2_theta, &cs[j], &sn[j]);
  for (int h = warp; h < nkv; h += nw) {
    float x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nj) x[j] = y[h * d + lane + 32 * j];
    head_norm_rope(x, d, k_norm, eps, cs, sn);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nj) st(&kc[dst + h * d + lane + 32 * j], x[j]);
  }
  for (int e = threadIdx.x * 4; e < nkv * d; e += blockDim.x * 4)
    st4(vc + dst + e, *reinterpret_cast<const float4*>(y + nkv * d + e));
}

// h[row] = scale * E[token], token = anchor (slot 0) or the mask id; then
// u = RMSNorm_gamma(h[row]) for the first sublayer.
template <typename T>
__global__ void __launch_bounds__(RT) embed_norm_kernel(const int32_t* __restrict__ anchor, int mask_id, int B,
                                                        const T* __restrict__ E, int V, int H, float scale,
                                                        const T* __restrict__ gamma, float eps, float* __restrict__ h,
                                                        T* __restrict__ u, unsigned* status) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  pdl_launch_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int s = row / B, i = row % B;
  int tok = i == 0 ? anchor[s] : mask_id;
  if (tok < 0 || tok >= V) {
    if (threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_TOKEN);
    tok = -1;
  }
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4) {
    float4 x = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tok >= 0) {
      x = ld4(E + (size_t)tok * H + m);
      x = make_float4(scale * x.x, scale * x.y, scale * x.z, scale * x.w);
    }
    *reinterpret_cast<float4*>(xs + m) = x;
    *reinterpret_cast<float4*>(h + (size_t)row * H + m) = x;
  }
  norm_row(xs, H, gamma, eps, u + (size_t)row * H, red);
}

// u = RMSNorm_gamma(h[row]).  With skip_anchor, block slot 0 is not written
// and the other rows are packed as [batch, B-1, H] (the lm_head input).
template <typename T>
__global__ void __launch_bounds__(RT) rownorm_kernel(const float* __restrict__ h, int H, const T* __restrict__ gamma,
                                                     float eps, T* __restrict__ u, int B, int skip_anchor) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  pdl_launch_next();
  pdl_wait();
  const int row = blockIdx.x;
  int orow = row;
  if (skip_anchor) {
    const int s = row / B, i = row % B;
    if (i == 0) return;  // the whole CTA leaves together
    orow = s * (B - 1) + i - 1;
  }
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4)
    *reinterpret_cast<float4*>(xs + m) = *reinterpret_cast<const float4*>(h + (size_t)row * H + m);
  norm_row(xs, H, gamma, eps, u + (size_t)orow * H, red);
}

// DFlash2 dynamic two-tap grouped convolution (one CTA per block row t):
//   alpha[g] = softmax(lambda[2g], lambda[2g+1]),  lambda = Y[t] (tap logits)
//   u2[ch]   = u_t[ch] + alpha[g][0] u_t[ch] + alpha[g][1] u_{t-1}[ch]
// u_{t-1} = 0 at the anchor (block slot 0): the window stays inside the block.
template <typename T>
__global__ void __launch_bounds__(RT) dyn_conv_kernel(const T* __restrict__ u, const float* __restrict__ Y, int H,
                                                      int gs, int B, T* __restrict__ u2) {
  extern __shared__ float alpha[];  // [G][2]
  pdl_launch_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int i = row % B;
  const int G = H / gs;
  const float* lam = Y + (size_t)row * 2 * G;
  for (int g = threadIdx.x; g < G; g += blockDim.x) {
    const float l0 = lam[2 * g], l1 = lam[2 * g + 1];
    const float mx = fmaxf(l0, l1);
    const float e0 = expf(l0 - mx), e1 = expf(l1 - mx);
    const float inv = 1.f / (e0 + e1);
    alpha[2 * g] = e0 * inv;
    alpha[2 * g + 1] = e1 * inv;
  }
  __syncthreads();
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4) {
    const int g = m / gs;  // gs is a multiple of 4: the 4 channels share a group
    const float a0 = alpha[2 * g], a1 = alpha[2 * g + 1];
    const float4 ut = ld4(u + (size_t)row * H + m);
    const float4 up = i > 0 ? ld4(u + (size_t)(row - 1) * H + m) : make_float4(0.f, 0.f, 0.f, 0.f);
    st4(u2 + (size_t)row * H + m, make_float4(ut.x + a0 * ut.x + a1 * up.x, ut.y + a0 * ut.y + a1 * up.y,
                                              ut.z + a0 * ut.z + a1 * up.z, ut.w + a0 * ut.w + a1 * up.w));
  }
}

// Block Q/K/V: per-head RMSNorm + RoPE of q and k at the block positions
// (anchor at the context length after the append), v copied.
template <typename T>
__global__ void __launch_bounds__(RT) qkv_epi_kernel(const float* __restrict__ Y, int B, int nq, int nkv, int d,
                                                     const T* __restrict__ qn, const T* __restrict__ kn, float eps,
                                                     double log2_theta, const int32_t* __restrict__ ctx_len,
                                                     const int32_t* __restrict__ new_off, T* __restrict__ q,
                                                     T* __restrict__ kb, T* __restrict__ vb) {
  pdl_launch_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int s = row / B, i = row % B;
  const int pos = ctx_len[s] + (new_off[s + 1] - new_off[s]) + i;
  const int w3 = (nq + 2 * nkv) * d;
  const float* y = Y + (size_t)row * w3;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  const int nj = d / 32;
  float cs[2], sn[2];
  for (int j = 0; j < d / 64; ++j) rope_cs(pos, lane + 32 * j, d, log2_theta, &cs[j], &sn[j]);
  for (int hh = warp; hh < nq + nkv; hh += nw) {
    float x[4];
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nj) x[j] = y[hh * d + lane + 32 * j];
    head_norm_rope(x, d, hh < nq ? qn : kn, eps, cs, sn);
    T* dst = hh < nq ? q + (size_t)row * nq * d + hh * d : kb + (size_t)row * nkv * d + (hh - nq) * d;
#pragma unroll
    for (int j = 0; j < 4; ++j)
      if (j < nj) st(&dst[lane + 32 * j], x[j]);
  }
  for (int e = threadIdx.x * 4; e < nkv * d; e += blockDim.x * 4)
    st4(vb + (size_t)row * nkv * d + e, *reinterpret_cast<const float4*>(y + (nq + nkv) * d + e));
}

// act = SiLU(gate) * up from the stacked gate/up output Y [rows][2I].
template <typename T>
__global__ void __launch_bounds__(RT) act_kernel(const float* __restrict__ Y, int rows, int I, T* __restrict__ act) {
  pdl_launch_next();
  pdl_wait();
  const size_t total4 = (size_t)rows * I / 4;
  for (size_t q4 = (size_t)blockIdx.x * blockDim.x + threadIdx.x; q4 < total4; q4 += (size_t)gridDim.x * blockDim.x) {
    const size_t idx = q4 * 4;
    const size_t row = idx / I, j = idx % I;
    const float4 g = *reinterpret_cast<const float4*>(Y + row * 2 * I + j);
    const float4 up = *reinterpret_cast<const float4*>(Y + row * 2 * I + I + j);
    st4(act + idx, make_float4(g.x / (1.f + expf(-g.x)) * up.x, g.y / (1.f + expf(-g.y)) * up.y,
                               g.z / (1.f + expf(-g.z)) * up.z, g.w / (1.f + expf(-g.w)) * up.w));
  }
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

int launch_rows_feature_norm(int dtype, const float* Y, int rows, int H, const void* gamma, float eps, void* f_out,
                             const Ctx& c) {
  if (rows <= 0) return DFLASH2_OK;
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(feature_norm_kernel<T>, dim3(rows), dim3(RT), H * sizeof(float), c.stream, Y, H,
                                    static_cast<const T*>(gamma), eps, static_cast<T*>(f_out)));
  return rc;
}

int launch_kv_append(int dtype, const float* Y, int rows, int nkv, int d, const void* k_norm, float eps, float theta,
                     const int32_t* ctx_len, const int32_t* new_off, int batch, const int32_t* block_table,
                     int max_pages, int page_size, int n_pages, void* kc, void* vc, const Ctx& c) {
  if (rows <= 0) return DFLASH2_OK;
  const double l2t = std::log2((double)theta);
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(kv_append_kernel<T>, dim3(rows), dim3(RT), 0, c.stream, Y, nkv, d,
                                    static_cast<const T*>(k_norm), eps, l2t, ctx_len, new_off, batch, block_table,
                                    max_pages, page_size, n_pages, static_cast<T*>(kc), static_cast<T*>(vc),
                                    c.status));
  return rc;
}

int launch_embed_norm(int dtype, const int32_t* anchor, int mask_id, int batch, int B, const void* embed, int V, int H,
                      float scale, const void* gamma, float eps, float* h_out, void* u_out, const Ctx& c) {
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(embed_norm_kernel<T>, dim3(batch * B), dim3(RT), H * sizeof(float), c.stream,
                                    anchor, mask_id, B, static_cast<const T*>(embed), V, H, scale,
                                    static_cast<const T*>(gamma), eps, h_out, static_cast<T*>(u_out), c.status));
  return rc;
}

int launch_rownorm(int dtype, const float* h, int rows, int H, const void* gamma, float eps, void* u_out, int B,
                   int skip_anchor, const Ctx& c) {
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(rownorm_kernel<T>, dim3(rows), dim3(RT), H * sizeof(float), c.stream, h, H,
                                    static_cast<const T*>(gamma), eps, static_cast<T*>(u_out), B, skip_anchor));
  return rc;
}

int launch_dyn_conv(int dtype, const void* u, const float* Y, int rows, int H, int group_size, int B, void* u2_out,
                    const Ctx& c) {
  const int G = H / group_size;
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(dyn_conv_kernel<T>, dim3(rows), dim3(RT), 2 * G * sizeof(float), c.stream,
                                    static_cast<const T*>(u), Y, H, group_size, B, static_cast<T*>(u2_out)));
  return rc;
}

int launch_qkv_epilogue(int dtype, const float* Y, int rows, int B, int nq, int nkv, int d, const void* q_norm,
                        const void* k_norm, float eps, float theta, const int32_t* ctx_len, const int32_t* new_off,
                        void* q, void* kb, void* vb, const Ctx& c) {
  const double l2t = std::log2((double)theta);
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(qkv_epi_kernel<T>, dim3(rows), dim3(RT), 0, c.stream, Y, B, nq, nkv, d,
                                    static_cast<const T*>(q_norm), static_cast<const T*>(k_norm), eps, l2t, ctx_len,
                                    new_off, static_cast<T*>(q), static_cast<T*>(kb), static_cast<T*>(vb)));
  return rc;
}

int launch_act(int dtype, const float* Y, int rows, int I, void* act, const Ctx& c) {
  const size_t total4 = (size_t)rows * I / 4;
  const int blocks = (int)std::min<size_t>((total4 + RT - 1) / RT, (size_t)c.nsm * 4);
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(act_kernel<T>, dim3(blocks), dim3(RT), 0, c.stream, Y, rows, I,
                                    static_cast<T*>(act)));
  return rc;
}

}  // namespace df2
