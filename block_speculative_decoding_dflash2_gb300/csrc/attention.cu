// Non-causal block attention over the paged context K/V plus the block's own
// K/V ("Train a DFlash Drafter for Speculative Decoding", "What is DFlash?":
// one non-causal forward over the block; "DFlash speculative decoding with
// vLLM", "Requirements": the attention must support non-causal drafting).
//
// Every query of the block (B positions x nq heads) sees every committed
// context key 0..P-1 and every block key P..P+B-1, with no mask, scale
// 1/sqrt(d), grouped-query sharing (q head h reads kv head h / (nq/nkv)).
//
// Work split: one CTA per (key chunk, kv head, sequence) holds the grp*B
// query rows that share that kv head (GQA packing), streams its key chunk
// through shared memory with an online softmax and writes an unnormalised
// partial (acc, running max, running sum).  A second kernel combines the
// chunks.  No CTA waits on another.  Keys are gathered row by row (one page
// lookup per key, then 16-byte loads of its d contiguous elements).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int AT = 256;  // threads
constexpr int KT = 32;   // keys per shared-memory tile

size_t attn_smem(int R, int d) {
  return sizeof(float) * ((size_t)R * d          /* Qs */
                          + (size_t)KT * (d + 1) /* Ks */
                          + (size_t)KT * d       /* Vs */
                          + (size_t)R * KT       /* Ss */
                          + (size_t)R * d        /* acc */
                          + 3 * (size_t)R + 1)   /* m, l, fac (+ alignment) */
         + sizeof(long long) * KT;               /* per-key row offsets */
}

// 8 consecutive elements as floats (16 bytes of bf16, or two float4).
__device__ __forceinline__ void load8(const bf16* p, float* o) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 f = __bfloat1622float2(h[i]);
    o[2 * i] = f.x;
    o[2 * i + 1] = f.y;
  }
}
__device__ __forceinline__ void load8(const float* p, float* o) {
  const float4 a = *reinterpret_cast<const float4*>(p), b = *reinterpret_cast<const float4*>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}

template <typename T>
__global__ void __launch_bounds__(AT) attn_partial_kernel(
    const T* __restrict__ q, const T* __restrict__ kb, const T* __restrict__ vb, const T* __restrict__ kc,
    const T* __restrict__ vc, const int32_t* __restrict__ block_table, int max_pages, int page_size, int n_pages,
    const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ new_off, int B, int nq, int nkv, int d, int CH,
    int nsplit, float* __restrict__ part, unsigned* status) {
  extern __shared__ float sm[];
  const int sp = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int grp = nq / nkv, R = grp * B;
  float* Qs = sm;
  float* Ks = Qs + R * d;
  float* Vs = Ks + KT * (d + 1);
  float* Ss = Vs + KT * d;
  float* acc = Ss + R * KT;
  float* mrow = acc + R * d;
  float* lrow = mrow + R;
  float* fac = lrow + R;
  // every region above has an even float count except m, l, fac (3R): pad to 8 bytes
  long long* koff = reinterpret_cast<long long*>(fac + R + (R & 1));

  const int P = ctx_len[s] + (new_off[s + 1] - new_off[s]);
  const int L = P + B;
  const int k0 = sp * CH, k1 = min(k0 + CH, L);
  float* out = part + ((((size_t)s * nkv + g) * nsplit + sp) * R) * (d + 2);
  if (k0 >= L) {
    for (int r = threadIdx.x; r < R; r += blockDim.x) {
      out[(size_t)r * (d + 2) + d] = -INFINITY;
      out[(size_t)r * (d + 2) + d + 1] = 0.f;
    }
    return;
  }
  if (P > max_pages * page_size && sp == 0 && threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
  const float scale = rsqrtf((float)d);
  const int c8 = d / 8;  // 8-element chunks per row
  for (int idx = threadIdx.x; idx < R * c8; idx += blockDim.x) {
    const int r = idx / c8, c = (idx % c8) * 8;
    const int i = r / grp, h = g * grp + r % grp;
    float v[8];
    load8(q + (((size_t)s * B + i) * nq + h) * d + c, v);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      Qs[r * d + c + e] = v[e] * scale;
      acc[r * d + c + e] = 0.f;
    }
  }
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    mrow[r] = -INFINITY;
    lrow[r] = 0.f;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nw = blockDim.x >> 5;
  // a key's row offset: into the paged cache, or (bit 62 set) into kb/vb
  constexpr long long BLOCK_BIT = 1LL << 62;
  for (int t0 = k0; t0 < k1; t0 += KT) {
    const int nk = min(KT, k1 - t0);
    __syncthreads();
    if (threadIdx.x < nk) {
      const int j = t0 + threadIdx.x;
      long long o = -1;
      if (j < P) {
        const int pi = j / page_size;
        const int page = pi < max_pages ? block_table[(size_t)s * max_pages + pi] : -1;
        if (page >= 0 && page < n_pages)
          o = (((long long)page * page_size + j % page_size) * nkv + g) * d;
        else
          flag(status, DFLASH2_DEV_BAD_PAGE);
      } else {
        o = BLOCK_BIT | ((((long long)s * B + (j - P)) * nkv + g) * d);
      }
      koff[threadIdx.x] = o;
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < nk * c8; idx += blockDim.x) {
      const int kk = idx / c8, c = (idx % c8) * 8;
      const long long o = koff[kk];
      float kv[8], vv[8];
      if (o < 0) {
#pragma unroll
        for (int e = 0; e < 8; ++e) kv[e] = vv[e] = 0.f;
      } else if (o & BLOCK_BIT) {
        const long long oo = o & ~BLOCK_BIT;
        load8(kb + oo + c, kv);
        load8(vb + oo + c, vv);
      } else {
        load8(kc + o + c, kv);
        load8(vc + o + c, vv);
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        Ks[kk * (d + 1) + c + e] = kv[e];
        Vs[kk * d + c + e] = vv[e];
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < R * nk; idx += blockDim.x) {
      const int r = idx / nk, kk = idx % nk;
      const float* qr = Qs + r * d;
      const float* kr = Ks + kk * (d + 1);
      float a = 0.f;
      for (int c = 0; c < d; ++c) a = fmaf(qr[c], kr[c], a);
      Ss[r * KT + kk] = a;
    }
    __syncthreads();
    for (int r = warp; r < R; r += nw) {
      const float x = lane < nk ? Ss[r * KT + lane] : -INFINITY;
      const float mx = warp_max(x);
      const float m_old = mrow[r];
      const float m_new = fmaxf(m_old, mx);
      const float p = lane < nk ? expf(x - m_new) : 0.f;
      const float ps = warp_sum(p);
      if (lane < nk) Ss[r * KT + lane] = p;
      if (lane == 0) {
        const float f = expf(m_old - m_new);
        fac[r] = f;
        lrow[r] = lrow[r] * f + ps;
        mrow[r] = m_new;
      }
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < R * d; idx += blockDim.x) {
      const int r = idx / d, c = idx % d;
      float a = acc[idx] * fac[r];
      const float* pr = Ss + r * KT;
      for (int kk = 0; kk < nk; ++kk) a = fmaf(pr[kk], Vs[kk * d + c], a);
      acc[idx] = a;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < R * d; idx += blockDim.x) {
    const int r = idx / d, c = idx % d;
    out[(size_t)r * (d + 2) + c] = acc[idx];
  }
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    out[(size_t)r * (d + 2) + d] = mrow[r];
    out[(size_t)r * (d + 2) + d + 1] = lrow[r];
  }
}

// O[s, i, h, :] = sum_chunks acc e^(m - M) / sum_chunks l e^(m - M)
template <typename T>
__global__ void attn_combine_kernel(const float* __restrict__ part, int B, int nq, int nkv, int d, int nsplit,
                                    T* __restrict__ o) {
  const int h = blockIdx.x % nq;
  const int si = blockIdx.x / nq;  // s*B + i
  const int s = si / B, i = si % B;
  const int grp = nq / nkv, g = h / grp, R = grp * B;
  const int r = i * grp + h % grp;
  const float* base = part + (((size_t)s * nkv + g) * nsplit) * R * (d + 2) + (size_t)r * (d + 2);
  const size_t sstride = (size_t)R * (d + 2);
  float M = -INFINITY;
  for (int sp = 0; sp < nsplit; ++sp) {
    const float* p = base + sp * sstride;
    if (p[d + 1] > 0.f) M = fmaxf(M, p[d]);
  }
  float den = 0.f;
  for (int sp = 0; sp < nsplit; ++sp) {
    const float* p = base + sp * sstride;
    if (p[d + 1] > 0.f) den += p[d + 1] * expf(p[d] - M);
  }
  for (int c = threadIdx.x; c < d; c += blockDim.x) {
    float num = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const float* p = base + sp * sstride;
      if (p[d + 1] > 0.f) num += p[c] * expf(p[d] - M);
    }
    st(&o[(size_t)si * nq * d + h * d + c], num / den);
  }
}

int chunk_of(int max_ctx, int B, int batch, int nkv, int nsm) {
  const long L = (long)max_ctx + B;
  long ch = (L * batch * nkv + 4L * nsm - 1) / (4L * nsm);
  ch = ((ch + 63) / 64) * 64;
  return (int)std::max(64L, std::min(1024L, ch));
}

}  // namespace

// Upper bound over every batch <= max_batch and SM count <= kMaxSM (the
// chunk grows with the SM count's inverse, so kMaxSM gives the most chunks).
size_t attn_part_bytes(int max_batch, int B, int nq, int nkv, int d, int max_ctx) {
  size_t best = 0;
  for (int b = 1; b <= max_batch; ++b) {
    const int ch = chunk_of(max_ctx, B, b, nkv, kMaxSM);
    const int nsplit = (max_ctx + B + ch - 1) / ch;
    best = std::max(best, (size_t)b * nkv * nsplit * (size_t)(nq / nkv) * B * (d + 2) * sizeof(float));
  }
  return best;
}

int launch_attention(int dtype, const void* q, const void* kb, const void* vb, const void* kc, const void* vc,
                     const int32_t* block_table, int max_pages, int page_size, int n_pages,
                     const int32_t* ctx_len, const int32_t* new_off, int batch, int B, int nq, int nkv, int d,
                     int max_ctx, float* part, void* o_out, const Ctx& c) {
  const int ch = chunk_of(max_ctx, B, batch, nkv, c.nsm);
  const int nsplit = (max_ctx + B + ch - 1) / ch;
  const int R = (nq / nkv) * B;
  const size_t smem = attn_smem(R, d);
  dim3 grid(nsplit, nkv, batch);
  static bool attr = false;  // set once, before any capture, to the largest size the config check allows
  if (!attr) {
    if (cudaFuncSetAttribute(attn_partial_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
            cudaSuccess ||
        cudaFuncSetAttribute(attn_partial_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024) !=
            cudaSuccess)
      return DFLASH2_ERR_CUDA;
    attr = true;
  }
  if (smem > 200 * 1024) return DFLASH2_ERR_SHAPE;
  if (dtype == DFLASH2_BF16) {
    attn_partial_kernel<bf16><<<grid, AT, smem, c.stream>>>(
        static_cast<const bf16*>(q), static_cast<const bf16*>(kb), static_cast<const bf16*>(vb),
        static_cast<const bf16*>(kc), static_cast<const bf16*>(vc), block_table, max_pages, page_size, n_pages,
        ctx_len, new_off, B, nq, nkv, d, ch, nsplit, part, c.status);
    attn_combine_kernel<bf16><<<batch * B * nq, 128, 0, c.stream>>>(part, B, nq, nkv, d, nsplit,
                                                                      static_cast<bf16*>(o_out));
  } else {
    attn_partial_kernel<float><<<grid, AT, smem, c.stream>>>(
        static_cast<const float*>(q), static_cast<const float*>(kb), static_cast<const float*>(vb),
        static_cast<const float*>(kc), static_cast<const float*>(vc), block_table, max_pages, page_size, n_pages,
        ctx_len, new_off, B, nq, nkv, d, ch, nsplit, part, c.status);
    attn_combine_kernel<float><<<batch * B * nq, 128, 0, c.stream>>>(part, B, nq, nkv, d, nsplit,
                                                                       static_cast<float*>(o_out));
  }
  count_launch(2);
  return cudaGetLastError() == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

}  // namespace df2
