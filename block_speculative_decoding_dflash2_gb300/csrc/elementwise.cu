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
//   "Variants"         DFlash 2's short (two-tap) convolution along the block
//                      around each sublayer (conv_prologue_kernel, or
//                      dyn_conv_kernel after a separate norm and tap GEMM);
//   "Key Config Fields" input_embedding_scale, conv_group_size.
#include <algorithm>
#include <cmath>
#include <type_traits>

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
// cos/sin of position pos for a rotary pair with inverse frequency inv
// (= theta^(-2i/d)): the angle pos * inv is formed and reduced modulo 2*pi
// in double (three operations), then sincosf of the reduced fp32 angle, so
// long contexts keep full fp32 accuracy.
__device__ __forceinline__ void rope_cs(int pos, double inv, float* c, float* s) {
  double a = (double)pos * inv;
  a -= 6.283185307179586 * rint(a * 0.15915494309189535);
  sincosf((float)a, s, c);
}

// RoPE table entries of block row t of sequence sq (position: the context
// length after the append, plus t), pairs i = tid, tid + nt, ... < d/2.
__device__ __forceinline__ void rope_table_block(const RopeTab& rt, int sq, int B, int t, int tid, int nt) {
  const int pos = rt.ctx_len[sq] + (rt.new_off[sq + 1] - rt.new_off[sq]) + t;
  float2* row = rt.cs + ((size_t)sq * B + t) * (rt.d / 2);
  for (int i = tid; i < rt.d / 2; i += nt) {
    float c, sn;
    rope_cs(pos, rt.freq.inv[i], &c, &sn);
    row[i] = make_float2(c, sn);
  }
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

// f[n] = RMSNorm_hidden(Y[n])  -- feature projection epilogue.  With
// rt.cs, also the RoPE table entries of appended row n and its paged-cache
// destination (for the fused K/V epilogue of the context projection).
template <typename T>
__global__ void __launch_bounds__(RT) feature_norm_kernel(const float* __restrict__ Y, int H,
                                                          const T* __restrict__ gamma, float eps, T* __restrict__ f,
                                                          const __grid_constant__ RopeTab rt, unsigned* status) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  __shared__ int pos_s;
  pdl_launch_next();
  pdl_wait();
  const size_t n = blockIdx.x;
  if (rt.cs) {
    if (threadIdx.x == 0) {
      const int sq = owner_of(rt.new_off, rt.batch, (int)n);
      int pos = rt.ctx_len[sq] + ((int)n - rt.new_off[sq]);
      long long dst = -1;
      if (pos < 0 || pos >= rt.max_pages * rt.page_size) {
        flag(status, DFLASH2_DEV_BAD_LENGTH);
        pos = 0;
      } else {
        const int page = rt.block_table[(size_t)sq * rt.max_pages + pos / rt.page_size];
        if (page < 0 || page >= rt.n_pages) flag(status, DFLASH2_DEV_BAD_PAGE);
        else dst = ((long long)page * rt.page_size + pos % rt.page_size) * rt.nkv * rt.d;
      }
      rt.dst[n] = dst;
      pos_s = pos;
    }
    __syncthreads();
    float2* row = rt.cs + n * (rt.d / 2);
    for (int i = threadIdx.x; i < rt.d / 2; i += blockDim.x) {
      float c, sn;
      rope_cs(pos_s, rt.freq.inv[i], &c, &sn);
      row[i] = make_float2(c, sn);
    }
  }
  for (int m = threadIdx.x * 4; m < H; m += blockDim.x * 4)
    *reinterpret_cast<float4*>(xs + m) = *reinterpret_cast<const float4*>(Y + n * H + m);
  norm_row(xs, H, gamma, eps, f + n * H, red);
}

// Context K/V of appended rows -> paged cache, one warp per (row, head):
// K = RoPE(RMSNorm_k(W_k f)) and V = W_v f at the row's absolute position.
// grid = (rows, ceil(2 nkv / warps per CTA)); warps past 2 nkv idle.
template <typename T>
__global__ void __launch_bounds__(RT) kv_append_kernel(const float* __restrict__ Y, int nkv, int d,
                                                       const T* __restrict__ k_norm, float eps, const __grid_constant__ RopeFreq freq,
                                                       const int32_t* __restrict__ ctx_len,
                                                       const int32_t* __restrict__ new_off, int batch,
                                                       const int32_t* __restrict__ block_table, int max_pages,
                                                       int page_size, int n_pages, T* __restrict__ kc,
                                                       T* __restrict__ vc, unsigned* status) {
  pdl_launch_next();
  pdl_wait();
  const int n = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hh = blockIdx.y * (RT / 32) + warp;  // 0..nkv-1: K heads, nkv..2nkv-1: V heads
  if (hh >= 2 * nkv) return;
  const int s = owner_of(new_off, batch, n);
  const int pos = ctx_len[s] + (n - new_off[s]);
  if (pos < 0 || pos >= max_pages * page_size) {
    if (lane == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
    return;
  }
  const int page = block_table[(size_t)s * max_pages + pos / page_size];
  if (page < 0 || page >= n_pages) {
    if (lane == 0) flag(status, DFLASH2_DEV_BAD_PAGE);
    return;
  }
  const size_t dst = ((size_t)page * page_size + pos % page_size) * nkv * d;
  const float* y = Y + (size_t)n * 2 * nkv * d + (size_t)hh * d;
  const int nj = d / 32;
  float x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nj) x[j] = y[lane + 32 * j];
  if (hh < nkv) {
    float cs[2], sn[2];
    for (int j = 0; j < d / 64; ++j) rope_cs(pos, freq.inv[lane + 32 * j], &cs[j], &sn[j]);
    head_norm_rope(x, d, k_norm, eps, cs, sn);
  }
  T* out = (hh < nkv ? kc : vc) + dst + (size_t)(hh < nkv ? hh : hh - nkv) * d;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nj) st(&out[lane + 32 * j], x[j]);
}

// h[row] = scale * E[token], token = anchor (slot 0) or the mask id; then
// u = RMSNorm_gamma(h[row]) for the first sublayer.
template <typename T>
__global__ void __launch_bounds__(RT) embed_norm_kernel(const int32_t* __restrict__ anchor, int mask_id, int B,
                                                        const T* __restrict__ E, int V, int H, float scale,
                                                        const T* __restrict__ gamma, float eps, float* __restrict__ h,
                                                        T* __restrict__ u, const __grid_constant__ RopeTab rt,
                                                        unsigned* status) {
  extern __shared__ float xs[];
  __shared__ float red[32];
  pdl_launch_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int s = row / B, i = row % B;
  if (rt.cs) rope_table_block(rt, s, B, i, threadIdx.x, blockDim.x);
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
// and the other rows are packed as [batch, B-1, H] (the lm_head input); then
// zero_key (nullable, [rows][kTopkSlots]) receives zeros at each packed row:
// the lm_head's shared top-k bounds start from nothing.
template <typename T>
__global__ void __launch_bounds__(RT) rownorm_kernel(const float* __restrict__ h, int H, const T* __restrict__ gamma,
                                                     float eps, T* __restrict__ u, int B, int skip_anchor,
                                                     unsigned long long* __restrict__ zero_key) {
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
    if (zero_key && threadIdx.x < kTopkSlots) zero_key[(size_t)orow * kTopkSlots + threadIdx.x] = 0ull;
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

// DFlash2 sublayer prologue, fused into one kernel: u = RMSNorm_gamma(x) with
// x the residual row h (or, for the first sublayer, the scaled block
// embedding), the dynamic tap logits lambda = W_tap u, their two-way softmax
// alpha, and the two-tap grouped convolution u2 = u + alpha0 u_t + alpha1 u_{t-1}
// (u_{-1} = 0 at the anchor).  One CTA per (run of gpc channel groups,
// sequence): it normalises the B rows of its sequence into shared memory (as
// stored, so the tap logits see the stored u), forms the tap logits of its
// groups, and writes u and u2 of its groups' channels (and h, for the
// embedding).  Tap row 2g + j of W_tap is tap j of group g.
//
// The kernel is latency-bound (a few hundred KB per CTA), so it is built
// around one round of loads: the CTA's tap rows are copied to shared memory
// (cp.async) before the dependency wait, since no kernel writes the weights;
// each row is split over NW / B warps, and a lane issues all its loads of x
// and gamma at once and keeps x in registers across the 1/rms reduction.
constexpr int PT = 512;  // threads of the prologue kernel
constexpr int PUB = 16;  // 4-element vectors per lane and round (bf16)

// Bytes of a row of H elements of es bytes in the prologue's shared memory:
// whole 16-byte units plus 16 bytes of padding.
__host__ __device__ __forceinline__ int prologue_row_bytes(int H, int es) { return (H * es + 15) / 16 * 16 + 16; }

// bf16 tensor-core helpers (mma.sync m16n8k16, ldmatrix), for the tap logits
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// four 8x8 b16 matrices, lane i supplying the address of row i % 8 of matrix i / 8
__device__ __forceinline__ void ldmatrix_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

template <typename T>
struct Vec4Raw;  // 4 elements as loaded, converted to float4 at use
template <>
struct Vec4Raw<float> {
  float4 v;
  __device__ __forceinline__ void load(const float* p) { v = *reinterpret_cast<const float4*>(p); }
  __device__ __forceinline__ float4 f() const { return v; }
};
template <>
struct Vec4Raw<bf16> {
  uint2 v;
  __device__ __forceinline__ void load(const bf16* p) { v = *reinterpret_cast<const uint2*>(p); }
  __device__ __forceinline__ float4 f() const {
    const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.x));
    const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v.y));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

template <>
struct Vec4Raw<uint8_t> {  // fp8 e4m3 tap weights (scaled per row after the dot product)
  uint32_t v;
  __device__ __forceinline__ void load(const uint8_t* p) { v = *reinterpret_cast<const uint32_t*>(p); }
  __device__ __forceinline__ float4 f() const {
    const float2 a = __bfloat1622float2(e4m3x2_to_bf16x2((uint16_t)(v & 0xffffu)));
    const float2 b = __bfloat1622float2(e4m3x2_to_bf16x2((uint16_t)(v >> 16)));
    return make_float4(a.x, a.y, b.x, b.y);
  }
};

// WT: element type of the tap weights (T, or uint8_t e4m3 codes with the
// per-row scales wsc: lambda = wsc[row] * sum_h q[row][h] u[h]).
template <typename T, bool EMBED, typename WT = T>
__global__ void __launch_bounds__(PT) conv_prologue_kernel(
    const float* __restrict__ h_in, const int32_t* __restrict__ anchor, int mask_id, const T* __restrict__ E, int V,
    float scale, const T* __restrict__ gamma, float eps, const WT* __restrict__ Wt, const float* __restrict__ wsc,
    int H, int gs, int gpc, int B, int stage_w, float* __restrict__ h_out, T* __restrict__ u_out,
    T* __restrict__ u2_out, const __grid_constant__ RopeTab rt, unsigned* status) {
  extern __shared__ __align__(16) uint8_t smraw[];
  constexpr int NW = PT / 32;
  constexpr int PU = sizeof(T) == 2 ? PUB : PUB / 2;  // fp32 rows: half, to stay in registers
  using XT = typename std::conditional<EMBED, T, float>::type;  // element type of the source rows
  const int s = blockIdx.y, G = H / gs;
  const int g0 = blockIdx.x * gpc, ng = min(gpc, G - g0);
  // rows are padded by 16 bytes (HP elements apart) so the 8 rows an
  // ldmatrix reads start in different banks
  const int HP = prologue_row_bytes(H, sizeof(T)) / (int)sizeof(T);
  const int WP = prologue_row_bytes(H, sizeof(WT)) / (int)sizeof(WT);
  T* us = reinterpret_cast<T*>(smraw);                 // [B][HP] normed rows as stored
  WT* wsm = reinterpret_cast<WT*>(us + (size_t)B * HP); // [2 gpc][WP] tap rows (stage_w)
  float* rinv = reinterpret_cast<float*>(wsm + (stage_w ? (size_t)2 * gpc * WP : 0));  // [B]
  float* lam = rinv + B;                               // [B][2 gpc] tap logits, then alpha
  float* red = lam + B * 2 * gpc;                      // [B][NW] partial sums of squares
  float* red2 = red + B * NW;                          // [NW][2][16][8] tensor-core partial logits
  __shared__ int toks[32];
  pdl_launch_next();
  if (stage_w) {  // the weights are not written by any kernel of the stream
    constexpr int E16 = 16 / sizeof(WT);
    const WT* src = Wt + (size_t)2 * g0 * H;
    const int per_row = H / E16;
    for (int i = threadIdx.x; i < 2 * ng * per_row; i += PT) {
      const int row = i / per_row, c = (i - row * per_row) * E16;
      cp_async16(wsm + (size_t)row * WP + c, src + (size_t)row * H + c, true);
    }
    cp_async_commit();
  }
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (EMBED && rt.cs && blockIdx.x == 0) {  // the block rows' RoPE table, by one CTA per sequence
    const int hp = rt.d / 2;
    const int pos0 = rt.ctx_len[s] + (rt.new_off[s + 1] - rt.new_off[s]);
    for (int idx = threadIdx.x; idx < B * hp; idx += PT) {
      const int t = idx / hp, i = idx - t * hp;
      float c, sn;
      rope_cs(pos0 + t, rt.freq.inv[i], &c, &sn);
      rt.cs[((size_t)s * B + t) * hp + i] = make_float2(c, sn);
    }
  }
  if (EMBED) {
    for (int t = threadIdx.x; t < B; t += PT) {
      int tok = t == 0 ? anchor[s] : mask_id;
      if (tok < 0 || tok >= V) {
        flag(status, DFLASH2_DEV_BAD_TOKEN);
        tok = -1;
      }
      toks[t] = tok;
    }
    __syncthreads();
  }
  // source row t (nullptr: a zero row, for an invalid token) and its scale
  auto src_row = [&](int t) -> const XT* {
    if constexpr (EMBED) return toks[t] < 0 ? nullptr : E + (size_t)toks[t] * H;
    else return h_in + ((size_t)s * B + t) * H;
  };
  const float xs = EMBED ? scale : 1.f;
  // row t is split into wpr contiguous segments of sl columns, one warp each
  const int wpr = max(1, NW / B), rows_at_once = NW / wpr;
  const int sl = (H / 4 + wpr - 1) / wpr * 4;
  const bool one_round = sl <= 128 * PU;  // uniform: each lane's x fits its registers
  for (int t0 = 0; t0 < B; t0 += rows_at_once) {
    const int t = t0 + warp / wpr, seg = warp % wpr;
    const bool active = warp / wpr < rows_at_once && t < B;
    const XT* x = active ? src_row(t) : nullptr;
    const int m1 = min(H, (seg + 1) * sl);
    Vec4Raw<XT> xv[PU];
    Vec4Raw<T> gv[PU];
    float ss = 0.f;
    // 1. sums of squares (one round of loads when the segment fits)
    if (active) {
      for (int m0 = seg * sl + lane * 4; m0 < m1; m0 += 128 * PU) {
#pragma unroll
        for (int k = 0; k < PU; ++k)
          if (m0 + 128 * k < m1) {
            if (x) xv[k].load(x + m0 + 128 * k);
            if (one_round) gv[k].load(gamma + m0 + 128 * k);
          }
#pragma unroll
        for (int k = 0; k < PU; ++k)
          if (m0 + 128 * k < m1 && x) {
            const float4 v = xv[k].f();
            ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
          }
      }
      ss = warp_sum(ss) * xs * xs;
      if (lane == 0) red[t * NW + seg] = ss;
    }
    __syncthreads();
    if (threadIdx.x < B && threadIdx.x >= t0 && threadIdx.x < t0 + rows_at_once) {
      float sum = 0.f;
      for (int k = 0; k < wpr; ++k) sum += red[threadIdx.x * NW + k];
      rinv[threadIdx.x] = rsqrtf(sum / (float)H + eps);
    }
    __syncthreads();
    // 2. the stored u rows into shared memory
    if (active) {
      const float r = rinv[t];
      for (int m0 = seg * sl + lane * 4; m0 < m1; m0 += 128 * PU) {
        if (!one_round) {
#pragma unroll
          for (int k = 0; k < PU; ++k)
            if (m0 + 128 * k < m1) {
              if (x) xv[k].load(x + m0 + 128 * k);
              gv[k].load(gamma + m0 + 128 * k);
            }
        }
#pragma unroll
        for (int k = 0; k < PU; ++k)
          if (m0 + 128 * k < m1) {
            float4 v = x ? xv[k].f() : make_float4(0.f, 0.f, 0.f, 0.f);
            v = make_float4(xs * v.x, xs * v.y, xs * v.z, xs * v.w);
            st4(us + (size_t)t * HP + m0 + 128 * k, scale4(v, r, gv[k].f()));
          }
      }
    }
  }
  if (stage_w) cp_async_wait<0>();
  __syncthreads();
  // 3. tap logits of this CTA's groups.  bf16 rows staged in shared memory:
  //    on the tensor cores, lambda[t][jj] = sum_h u[t][h] W[jj][h] as
  //    m16n8k16 tiles (A = 16 block rows, B = 16 tap rows as two n8 tiles;
  //    rows past the real ones repeat the last real row and their results
  //    are dropped), the K range split across the warps and the partial
  //    tiles summed through shared memory.  Otherwise one warp per (row,
  //    tap row) on the CUDA cores.
  constexpr bool MMA = std::is_same<T, bf16>::value && std::is_same<WT, bf16>::value;
  const int mtiles = (B + 15) / 16, ntiles = (2 * ng + 15) / 16, tiles = mtiles * ntiles;
  if (MMA && stage_w && H % 16 == 0 && tiles <= NW) {
    const int ksplit = NW / tiles;  // warps per tile (the K range in slices)
    const int tile = warp / ksplit, ks = warp % ksplit;
    if (tile < tiles) {
      const int mt = tile / ntiles, nt = tile % ntiles;
      const int nk = H / 16, kb = ks * nk / ksplit, ke = (ks + 1) * nk / ksplit;
      const int mi = lane >> 3;
      const int ar = min(mt * 16 + (mi & 1) * 8 + (lane & 7), B - 1);            // A row (block row)
      const int br = min(nt * 16 + (mi >> 1) * 8 + (lane & 7), 2 * ng - 1);      // B row (tap row)
      const bf16* ap = reinterpret_cast<const bf16*>(us) + (size_t)ar * HP + (mi >> 1) * 8;
      const bf16* bp = reinterpret_cast<const bf16*>(wsm) + (size_t)br * WP + (mi & 1) * 8;
      float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
      for (int kk = kb; kk < ke; ++kk) {
        uint32_t a[4], b[4];
        ldmatrix_x4(a, ap + kk * 16);
        ldmatrix_x4(b, bp + kk * 16);
        mma_bf16_16816(c0, a, b[0], b[1]);
        mma_bf16_16816(c1, a, b[2], b[3]);
      }
      // partial tile -> red2[warp]: [n8 tile][row 16][col 8]
      float* o = red2 + (size_t)warp * 256;
      const int r0 = lane >> 2, cc = (lane & 3) * 2;
      o[r0 * 8 + cc] = c0[0];
      o[r0 * 8 + cc + 1] = c0[1];
      o[(r0 + 8) * 8 + cc] = c0[2];
      o[(r0 + 8) * 8 + cc + 1] = c0[3];
      o[128 + r0 * 8 + cc] = c1[0];
      o[128 + r0 * 8 + cc + 1] = c1[1];
      o[128 + (r0 + 8) * 8 + cc] = c1[2];
      o[128 + (r0 + 8) * 8 + cc + 1] = c1[3];
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < B * 2 * ng; idx += PT) {
      const int t = idx / (2 * ng), jj = idx % (2 * ng);
      const int mt = t / 16, nt = jj / 16, tl = mt * ntiles + nt;
      const int e = ((jj % 16) / 8) * 128 + (t % 16) * 8 + jj % 8;
      float acc = 0.f;
      for (int k2 = 0; k2 < ksplit; ++k2) acc += red2[(size_t)(tl * ksplit + k2) * 256 + e];
      lam[t * 2 * gpc + jj] = wsc ? acc * wsc[2 * g0 + jj] : acc;
    }
  } else
  for (int p = warp; p < B * 2 * ng; p += NW) {
    const int t = p / (2 * ng), jj = p % (2 * ng);
    const WT* w = stage_w ? wsm + (size_t)jj * WP : Wt + (size_t)(2 * g0 + jj) * H;
    float acc = 0.f;
    for (int m0 = lane * 4; m0 < H; m0 += 128 * PU) {
      Vec4Raw<WT> wv[PU];
#pragma unroll
      for (int k = 0; k < PU; ++k)
        if (m0 + 128 * k < H) wv[k].load(w + m0 + 128 * k);
#pragma unroll
      for (int k = 0; k < PU; ++k)
        if (m0 + 128 * k < H) {
          const float4 wf = wv[k].f(), uv = ld4(us + (size_t)t * HP + m0 + 128 * k);
          acc += wf.x * uv.x + wf.y * uv.y + wf.z * uv.z + wf.w * uv.w;
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) lam[t * 2 * gpc + jj] = wsc ? acc * wsc[2 * g0 + jj] : acc;
  }
  __syncthreads();
  // 4. alpha = softmax over the two taps of each (row, group)
  for (int idx = threadIdx.x; idx < B * ng; idx += PT) {
    const int t = idx / ng, gl = idx % ng;
    float* l = lam + t * 2 * gpc + 2 * gl;
    const float mx = fmaxf(l[0], l[1]);
    const float e0 = expf(l[0] - mx), e1 = expf(l[1] - mx);
    const float inv = 1.f / (e0 + e1);
    l[0] = e0 * inv;
    l[1] = e1 * inv;
  }
  __syncthreads();
  // 5. the convolution over this CTA's channels; u (and h) stored alongside
  const int c0 = g0 * gs, nc = ng * gs;
  for (int idx = threadIdx.x * 4; idx < B * nc; idx += PT * 4) {
    const int t = idx / nc, cc = idx % nc, m = c0 + cc;
    const float* a = lam + t * 2 * gpc + 2 * (cc / gs);  // gs % 4 == 0: the 4 channels share a group
    const float a0 = a[0], a1 = a[1];
    const float4 ut = ld4(us + (size_t)t * HP + m);
    const float4 up = t > 0 ? ld4(us + (size_t)(t - 1) * HP + m) : make_float4(0.f, 0.f, 0.f, 0.f);
    const size_t o = ((size_t)s * B + t) * H + m;
    st4(u_out + o, ut);
    st4(u2_out + o, make_float4(ut.x + a0 * ut.x + a1 * up.x, ut.y + a0 * ut.y + a1 * up.y,
                                ut.z + a0 * ut.z + a1 * up.z, ut.w + a0 * ut.w + a1 * up.w));
    if (EMBED) {
      const XT* x = src_row(t);
      float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
      if (x) {
        Vec4Raw<XT> xr;
        xr.load(x + m);
        v = xr.f();
        v = make_float4(xs * v.x, xs * v.y, xs * v.z, xs * v.w);
      }
      *reinterpret_cast<float4*>(h_out + o) = v;
    }
  }
}

// Block Q/K/V, one warp per (row, head): per-head RMSNorm + RoPE of q and k
// at the block positions (anchor at the context length after the append), v
// copied.  grid = (rows, ceil((nq + 2 nkv) / warps per CTA)).
template <typename T>
__global__ void __launch_bounds__(RT) qkv_epi_kernel(const float* __restrict__ Y, int B, int nq, int nkv, int d,
                                                     const T* __restrict__ qn, const T* __restrict__ kn, float eps,
                                                     const __grid_constant__ RopeFreq freq,
                                                     const int32_t* __restrict__ ctx_len,
                                                     const int32_t* __restrict__ new_off, T* __restrict__ q,
                                                     T* __restrict__ kb, T* __restrict__ vb) {
  pdl_launch_next();
  pdl_wait();
  const int row = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int hh = blockIdx.y * (RT / 32) + warp;  // q heads, then k heads, then v heads
  if (hh >= nq + 2 * nkv) return;
  const int s = row / B, i = row % B;
  const float* y = Y + (size_t)row * (nq + 2 * nkv) * d + (size_t)hh * d;
  const int nj = d / 32;
  float x[4];
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nj) x[j] = y[lane + 32 * j];
  if (hh < nq + nkv) {
    const int pos = ctx_len[s] + (new_off[s + 1] - new_off[s]) + i;
    float cs[2], sn[2];
    for (int j = 0; j < d / 64; ++j) rope_cs(pos, freq.inv[lane + 32 * j], &cs[j], &sn[j]);
    head_norm_rope(x, d, hh < nq ? qn : kn, eps, cs, sn);
  }
  T* dst = hh < nq         ? q + ((size_t)row * nq + hh) * d
           : hh < nq + nkv ? kb + ((size_t)row * nkv + hh - nq) * d
                           : vb + ((size_t)row * nkv + hh - nq - nkv) * d;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    if (j < nj) st(&dst[lane + 32 * j], x[j]);
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
                             const RopeTab& rt, const Ctx& c) {
  if (rows <= 0) return DFLASH2_OK;
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(feature_norm_kernel<T>, dim3(rows), dim3(RT), H * sizeof(float), c, Y, H,
                                    static_cast<const T*>(gamma), eps, static_cast<T*>(f_out), rt, c.status));
  return rc;
}

int launch_kv_append(int dtype, const float* Y, int rows, int nkv, int d, const void* k_norm, float eps, float theta,
                     const int32_t* ctx_len, const int32_t* new_off, int batch, const int32_t* block_table,
                     int max_pages, int page_size, int n_pages, void* kc, void* vc, const Ctx& c) {
  if (rows <= 0) return DFLASH2_OK;
  const RopeFreq freq = rope_freq(d, theta);
  int rc;
  const dim3 grid(rows, (2 * nkv + RT / 32 - 1) / (RT / 32));
  DF2_DISPATCH(dtype, rc = launch_k(kv_append_kernel<T>, grid, dim3(RT), 0, c, Y, nkv, d,
                                    static_cast<const T*>(k_norm), eps, freq, ctx_len, new_off, batch, block_table,
                                    max_pages, page_size, n_pages, static_cast<T*>(kc), static_cast<T*>(vc),
                                    c.status));
  return rc;
}

int launch_embed_norm(int dtype, const int32_t* anchor, int mask_id, int batch, int B, const void* embed, int V, int H,
                      float scale, const void* gamma, float eps, float* h_out, void* u_out, const RopeTab& rt,
                      const Ctx& c) {
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(embed_norm_kernel<T>, dim3(batch * B), dim3(RT), H * sizeof(float), c,
                                    anchor, mask_id, B, static_cast<const T*>(embed), V, H, scale,
                                    static_cast<const T*>(gamma), eps, h_out, static_cast<T*>(u_out), rt,
                                    c.status));
  return rc;
}

int launch_rownorm(int dtype, const float* h, int rows, int H, const void* gamma, float eps, void* u_out, int B,
                   int skip_anchor, const Ctx& c, unsigned long long* zero_key) {
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(rownorm_kernel<T>, dim3(rows), dim3(RT), H * sizeof(float), c, h, H,
                                    static_cast<const T*>(gamma), eps, static_cast<T*>(u_out), B, skip_anchor,
                                    zero_key));
  return rc;
}

int launch_dyn_conv(int dtype, const void* u, const float* Y, int rows, int H, int group_size, int B, void* u2_out,
                    const Ctx& c) {
  const int G = H / group_size;
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(dyn_conv_kernel<T>, dim3(rows), dim3(RT), 2 * G * sizeof(float), c,
                                    static_cast<const T*>(u), Y, H, group_size, B, static_cast<T*>(u2_out)));
  return rc;
}

// Shared memory of the prologue: the B normed rows, the CTA's tap rows when
// staged, 1/rms, tap logits and the per-warp partial sums.
size_t conv_prologue_smem(int dtype, int B, int H, int gpc, bool stage_w, bool w8) {
  const int es = dtype == DFLASH2_BF16 ? 2 : 4, ws = w8 ? 1 : es;
  return (size_t)B * prologue_row_bytes(H, es) + (stage_w ? (size_t)2 * gpc * prologue_row_bytes(H, ws) : 0) +
         (size_t)B * (1 + 2 * gpc + PT / 32) * sizeof(float) + (size_t)(PT / 32) * 256 * sizeof(float);
}

int conv_prologue_groups(int G, int batch, int nsm) {
  // about two CTAs per SM: groups per CTA grows with the batch
  const long want = std::max(1L, (long)2 * nsm / std::max(1, batch));
  return (int)std::max(1L, std::min<long>(G, ((long)G + want - 1) / want));
}

constexpr size_t kPrologueSmem = 200 * 1024;

bool conv_prologue_fits(int dtype, int batch, int B, int H, int G, int nsm) {
  // the fused kernel pays off only with its CTA's tap rows staged in shared
  // memory (tensor-core tap logits); past that (wide batches, where a CTA
  // would take many groups) the rownorm + tap contraction + conv kernels run
  return B <= 32 && conv_prologue_smem(dtype, B, H, conv_prologue_groups(G, batch, nsm), true, false) <= kPrologueSmem;
}

int launch_conv_prologue(int dtype, const float* h_in, const int32_t* anchor, int mask_id, const void* embed, int V,
                         float scale, const void* gamma, float eps, const void* w_tap, const float* tap_scale,
                         int batch, int B, int H, int group_size, float* h_out, void* u_out, void* u2_out,
                         const RopeTab& rt, const Ctx& c) {
  const int G = H / group_size;
  const int gpc = conv_prologue_groups(G, batch, c.nsm);
  const bool w8 = tap_scale != nullptr;
  if (w8 && dtype != DFLASH2_BF16) return DFLASH2_ERR_DTYPE;
  const bool stage_w = conv_prologue_smem(dtype, B, H, gpc, true, w8) <= kPrologueSmem;
  const size_t smem = conv_prologue_smem(dtype, B, H, gpc, stage_w, w8);
  if (smem > kPrologueSmem || B > 32) return DFLASH2_ERR_SHAPE;
  static bool attr = false;  // set once, before any capture
  if (!attr) {
    if (cudaFuncSetAttribute(conv_prologue_kernel<bf16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPrologueSmem) ||
        cudaFuncSetAttribute(conv_prologue_kernel<bf16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPrologueSmem) ||
        cudaFuncSetAttribute(conv_prologue_kernel<float, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPrologueSmem) ||
        cudaFuncSetAttribute(conv_prologue_kernel<float, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPrologueSmem) ||
        cudaFuncSetAttribute(conv_prologue_kernel<bf16, true, uint8_t>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kPrologueSmem) ||
        cudaFuncSetAttribute(conv_prologue_kernel<bf16, false, uint8_t>,
                             cudaFuncAttributeMaxDynamicSharedMemorySize, kPrologueSmem))
      return DFLASH2_ERR_CUDA;
    attr = true;
  }
  const dim3 grid((G + gpc - 1) / gpc, batch);
  int rc;
  if (w8) {
    const uint8_t* wq = static_cast<const uint8_t*>(w_tap);
    if (h_in)
      return launch_k(conv_prologue_kernel<bf16, false, uint8_t>, grid, dim3(PT), smem, c, h_in, anchor, mask_id,
                      static_cast<const bf16*>(embed), V, scale, static_cast<const bf16*>(gamma), eps, wq, tap_scale,
                      H, group_size, gpc, B, stage_w ? 1 : 0, h_out, static_cast<bf16*>(u_out),
                      static_cast<bf16*>(u2_out), rt, c.status);
    return launch_k(conv_prologue_kernel<bf16, true, uint8_t>, grid, dim3(PT), smem, c, h_in, anchor, mask_id,
                    static_cast<const bf16*>(embed), V, scale, static_cast<const bf16*>(gamma), eps, wq, tap_scale, H,
                    group_size, gpc, B, stage_w ? 1 : 0, h_out, static_cast<bf16*>(u_out), static_cast<bf16*>(u2_out),
                    rt, c.status);
  }
  if (h_in)
    DF2_DISPATCH(dtype, rc = launch_k(conv_prologue_kernel<T, false>, grid, dim3(PT), smem, c, h_in, anchor, mask_id,
                                      static_cast<const T*>(embed), V, scale, static_cast<const T*>(gamma), eps,
                                      static_cast<const T*>(w_tap), nullptr, H, group_size, gpc, B, stage_w ? 1 : 0, h_out,
                                      static_cast<T*>(u_out), static_cast<T*>(u2_out), rt, c.status));
  else
    DF2_DISPATCH(dtype, rc = launch_k(conv_prologue_kernel<T, true>, grid, dim3(PT), smem, c, h_in, anchor, mask_id,
                                      static_cast<const T*>(embed), V, scale, static_cast<const T*>(gamma), eps,
                                      static_cast<const T*>(w_tap), nullptr, H, group_size, gpc, B, stage_w ? 1 : 0, h_out,
                                      static_cast<T*>(u_out), static_cast<T*>(u2_out), rt, c.status));
  return rc;
}

int launch_qkv_epilogue(int dtype, const float* Y, int rows, int B, int nq, int nkv, int d, const void* q_norm,
                        const void* k_norm, float eps, float theta, const int32_t* ctx_len, const int32_t* new_off,
                        void* q, void* kb, void* vb, const Ctx& c) {
  const RopeFreq freq = rope_freq(d, theta);
  int rc;
  const dim3 grid(rows, (nq + 2 * nkv + RT / 32 - 1) / (RT / 32));
  DF2_DISPATCH(dtype, rc = launch_k(qkv_epi_kernel<T>, grid, dim3(RT), 0, c, Y, B, nq, nkv, d,
                                    static_cast<const T*>(q_norm), static_cast<const T*>(k_norm), eps, freq, ctx_len,
                                    new_off, static_cast<T*>(q), static_cast<T*>(kb), static_cast<T*>(vb)));
  return rc;
}

int launch_act(int dtype, const float* Y, int rows, int I, void* act, const Ctx& c) {
  const size_t total4 = (size_t)rows * I / 4;
  const int blocks = (int)std::min<size_t>((total4 + RT - 1) / RT, (size_t)c.nsm * 4);
  int rc;
  DF2_DISPATCH(dtype, rc = launch_k(act_kernel<T>, dim3(blocks), dim3(RT), 0, c, Y, rows, I,
                                    static_cast<T*>(act)));
  return rc;
}

}  // namespace df2
