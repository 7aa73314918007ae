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
#include <atomic>
#include <cstring>

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
    int nsplit, int window, float* __restrict__ part, unsigned* status) {
  extern __shared__ float sm[];
  pdl_launch_next();
  pdl_wait();
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
  const int w0 = window > 0 ? max(0, P - window) : 0;  // first context key read (sliding window)
  const int k0 = w0 + sp * CH, k1 = min(k0 + CH, L);
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

// ------------------------------------------------------------------------
// bf16 path: one thread-block cluster per (kv head, sequence).  The NS CTAs
// of the cluster split the keys [0, P + B) into NS contiguous chunks.  Each
// CTA runs a flash-attention pass over its chunk on the tensor cores
// (mma.sync m16n8k16, fp32 accumulation), with its 128-key K/V tiles
// double-buffered in shared memory by cp.async (page ids loaded once),
// and leaves an unnormalised partial (acc, running max, running sum) for each
// of the grp*B query rows in shared memory.  After a cluster barrier every
// CTA merges the cluster's partials of its share of the rows through
// distributed shared memory and writes O: no partial goes to global memory
// and no second kernel runs.
//
// Within a CTA the query rows form 16-row blocks and each tile's keys are cut
// into ksplit shares; each of the 16 warps owns one (row block, key share)
// combination with its own online-softmax state in registers.  The CTA
// first merges a row's shares in shared memory, so the cluster-wide merge
// reads one partial per CTA.  For every
// 16-key step: S = Q K^T (K rows read with ldmatrix as the col-major B
// operand), scale, mask, online softmax, then O += P V with P split into
// bf16 hi + lo parts (two MMAs), so the probabilities keep ~16 bits.

__device__ __forceinline__ void mma16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&v);
}

constexpr int kMaxStages = 4;    // K/V tile stages at most
constexpr int kMaxCluster = 8;   // CTAs per cluster (portable)
constexpr int CLW = 16;          // warps per CTA
constexpr int CLT = 32 * CLW;    // threads
constexpr int kMaxShares = 8;    // key shares per 16-row block (16 keys each per tile)
constexpr size_t kAttnSmem = 227 * 1024;

// Key shares per 16-row block: enough (row block, share) combinations to
// give nearly every warp one (at most CLW combinations, at most kMaxShares
// shares).  The tile takes mkt = shares x 16 x steps keys, steps the fewest
// 16-key steps per share that make the tile at least 64 keys, so every share
// is a whole number of steps.
inline int attn_ksplit(int nrb) { return std::max(1, std::min(kMaxShares, CLW / nrb)); }
inline int attn_tile_keys(int ksplit) {
  const int unit = 16 * ksplit;
  return unit * ((64 + unit - 1) / unit);
}

// Shared memory: Q rows; the kst K/V stages of mkt keys, which after the key
// loop hold the per-combination partial states (read by the whole cluster);
// the merge weights of this CTA's rows; the page ids of its key chunk (npg).
template <int DH>
__host__ __device__ inline size_t attn_kv_bytes(int R, int mkt, int kst, int ksplit) {
  const int nrb = (R + 15) / 16;
  const size_t kvb = (size_t)kst * 2 * mkt * (DH + 8) * 2;
  const size_t comb = (size_t)nrb * ksplit * 16 * (DH + 2) * 4;
  return kvb > comb ? kvb : comb;
}
template <int DH>
size_t attn_cl_smem(int R, int npg, int mkt, int kst, int ksplit) {
  const int nrb = (R + 15) / 16;
  const size_t qb = (size_t)nrb * 16 * (DH + 8) * 2;
  return qb + 128 /* K/V ring alignment */ + attn_kv_bytes<DH>(R, mkt, kst, ksplit) +
         (size_t)(R + kMaxCluster) * kMaxShares * 2 * 4 + (size_t)npg * 4 + 8 + kMaxStages * sizeof(uint64_t);
}

template <int DH>
__global__ void __launch_bounds__(CLT, 1) attn_cluster_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ kb, const bf16* __restrict__ vb, const bf16* __restrict__ kc,
    const bf16* __restrict__ vc, const int32_t* __restrict__ block_table, int max_pages, int page_size, int n_pages,
    const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ new_off, int B, int nq, int nkv, int npg,
    int window, int MKT, int KST, int ksplit, const __grid_constant__ CUtensorMap tmK,
    const __grid_constant__ CUtensorMap tmV, int page_tma, bf16* __restrict__ o, unsigned* status) {
  // MKT keys per K/V tile, KST tile stages (KST - 1 tiles in flight while one
  // is consumed), ksplit key shares of MKT / ksplit keys per 16-row block
  constexpr int MCPW = 1;  // (row block, key share) combinations per warp
  constexpr int LD = DH + 8;  // padded smem row (elements): ldmatrix rows hit distinct banks
  constexpr int NT = DH / 8;  // n8 tiles across the head dimension
  constexpr int C8 = DH / 8;  // 16-byte chunks per row
  constexpr int FS = DH + 2;  // partial row: acc[DH], m, l
  extern __shared__ __align__(16) uint8_t smraw[];
  pdl_launch_next();
  const int NS = gridDim.x;  // the cluster spans x
  const int sp = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int grp = nq / nkv, R = grp * B;
  const int nrb = (R + 15) / 16;
  const int ncombo = nrb * ksplit;
  bf16* Qs = reinterpret_cast<bf16*>(smraw);
  // [KST][K, V][MKT][LD], 128-byte aligned: a page of rows is one TMA box
  bf16* KV = reinterpret_cast<bf16*>((reinterpret_cast<uintptr_t>(Qs + nrb * 16 * LD) + 127) & ~uintptr_t(127));
  float* comb = reinterpret_cast<float*>(KV);            // [ncombo][16][FS], after the key loop
  float* wts = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(KV) + attn_kv_bytes<DH>(R, MKT, KST, ksplit));  // merge weights
  int* pg = reinterpret_cast<int*>(wts + (size_t)(R + kMaxCluster) * kMaxShares * 2);  // page ids of the chunk
  uint64_t* kvbar = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(pg + npg) + 7) & ~uintptr_t(7));
  if (threadIdx.x == 0) {  // one K/V stage completes when its 2*MKT row copies have landed
    for (int i = 0; i < KST; ++i) mbar_init(kvbar + i, 2 * MKT);
    fence_barrier_init();
  }

  pdl_wait();
  const int P = ctx_len[s] + (new_off[s + 1] - new_off[s]);
  const int L = P + B;
  const int w0 = window > 0 ? max(0, P - window) : 0;  // first context key read (sliding window)
  const int CH = (((L - w0 + NS - 1) / NS) + 15) & ~15;
  const int k0 = w0 + min(sp * CH, L - w0), k1 = min(k0 + CH, L);
  if (P > max_pages * page_size && sp == 0 && threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
  // scores are kept in base-2 units (1/sqrt(d) times log2(e)), so each
  // exponential is one exp2 and the softmax is unchanged: 2^(x log2 e) = e^x
  constexpr float kLog2e = 1.4426950408889634f;
  const float scale = rsqrtf((float)DH) * kLog2e;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  // page ids of the chunk's context keys, once (-1: past the table)
  const int pbase = k0 / page_size;
  const int pend = k0 < min(k1, P) ? (min(k1, P) - 1) / page_size + 1 : pbase;
  for (int i = threadIdx.x; i < pend - pbase && i < npg; i += blockDim.x) {
    const int pi = pbase + i;
    pg[i] = pi < max_pages ? block_table[(size_t)s * max_pages + pi] : -1;
  }
  if (pend - pbase > npg && threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
  __syncthreads();
  // query rows (zero padding to whole 16-row blocks)
  for (int idx = threadIdx.x; idx < nrb * 16 * C8; idx += blockDim.x) {
    const int r = idx / C8, c = (idx % C8) * 8;
    const bf16* src = q;
    if (r < R) src = q + (((size_t)s * B + r / grp) * nq + g * grp + r % grp) * DH + c;
    cp_async16(Qs + r * LD + c, src, r < R);
  }
  // K/V rows of keys t0 .. t0 + MKT - 1 into stage stg.  With page_tma (16-key
  // pages and a page-aligned chunk start), each whole context page of the
  // tile is one TMA box per K and V (16 rows of DH + 8 elements from the
  // cache viewed as [pages * 16][nkv * DH]: the row's DH values of this kv
  // head plus 8 ignored ones, which lands them at the padded row pitch);
  // threads 0 .. 2p-1 issue those.  The other rows (the tile's last partial
  // context page, the block's own keys, keys past k1) are copied one row per
  // thread, one 16-byte-aligned bulk copy of DH elements each.  Each of the
  // first 2*MKT threads arrives once per tile on the stage barrier with the
  // bytes it issued (0 when it has none); keys past k1, and rows of an
  // invalid page (flagged), are written as zeros instead.
  const bool tma_ok = page_tma && (k0 % 16) == 0;
  auto issue = [&](int t0, int stg) {
    if (threadIdx.x >= 2 * MKT) return;
    bf16* sbase = KV + (size_t)stg * 2 * MKT * LD;
    const int cend = min(min(t0 + MKT, k1), P);  // context keys of this tile end here
    const int nfull = tma_ok ? max(0, (cend - t0) / 16) : 0;  // whole pages by TMA
    const int nrow = MKT - 16 * nfull;                         // rows copied one by one
    const int tid = threadIdx.x;
    if (tid < 2 * nfull) {
      const bool is_v = tid >= nfull;
      const int pi = is_v ? tid - nfull : tid;
      bf16* dst = sbase + (is_v ? MKT * LD : 0) + (size_t)pi * 16 * LD;
      const int li = (t0 + pi * 16) / 16 - pbase;
      const int page = li < npg ? pg[li] : -1;
      if (page >= 0 && page < n_pages) {
        mbar_arrive_expect_tx(kvbar + stg, 16 * LD * 2);
        fence_proxy_async_smem();
        tma_load_2d(dst, is_v ? &tmV : &tmK, kvbar + stg, g * DH, page * 16, policy_evict_first());
      } else {
        if (!is_v) flag(status, DFLASH2_DEV_BAD_PAGE);
        mbar_arrive_expect_tx(kvbar + stg, 0);
        for (int c = 0; c < 16 * LD / 8; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
      }
      return;
    }
    const int tr = tid - 2 * nfull;
    if (tr >= 2 * nrow) {  // nothing left for this thread this tile
      mbar_arrive_expect_tx(kvbar + stg, 0);
      return;
    }
    const bool is_v = tr >= nrow;
    const int kk = 16 * nfull + (is_v ? tr - nrow : tr);
    bf16* dst = sbase + (is_v ? MKT * LD : 0) + (size_t)kk * LD;
    const int j = t0 + kk;
    const bf16* src = nullptr;
    if (j < k1) {
      if (j < P) {
        const int li = j / page_size - pbase;
        const int page = li < npg ? pg[li] : -1;
        if (page >= 0 && page < n_pages)
          src = (is_v ? vc : kc) + (((size_t)page * page_size + j % page_size) * nkv + g) * DH;
        else if (!is_v)
          flag(status, DFLASH2_DEV_BAD_PAGE);
      } else {
        src = (is_v ? vb : kb) + (((size_t)s * B + (j - P)) * nkv + g) * DH;
      }
    }
    mbar_arrive_expect_tx(kvbar + stg, src ? DH * 2 : 0);
    if (src) {
      bulk_g2s(dst, src, DH * 2, kvbar + stg);
    } else {
#pragma unroll
      for (int c = 0; c < C8; ++c) reinterpret_cast<uint4*>(dst)[c] = make_uint4(0, 0, 0, 0);
    }
  };
  const int ntiles = (k1 - k0 + MKT - 1) / MKT;  // 0 for an empty chunk
  cp_async_commit();  // the Q rows
  for (int i = 0; i < KST && i < ntiles; ++i) issue(k0 + i * MKT, i);  // every stage starts filling
  volatile int never = 0;

  // per-combination online-softmax state: rows lane/4 and lane/4 + 8 of the block
  float m_st[MCPW][2], l_st[MCPW][2], acc[MCPW][NT][4];
#pragma unroll
  for (int c = 0; c < MCPW; ++c) {
    m_st[c][0] = m_st[c][1] = -INFINITY;
    l_st[c][0] = l_st[c][1] = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) acc[c][n][0] = acc[c][n][1] = acc[c][n][2] = acc[c][n][3] = 0.f;
  }
  cp_async_wait<0>();
  __syncthreads();  // the Q rows and the zero-filled rows of the first tiles are visible to every warp
  for (int t = 0; t < ntiles; ++t) {
    // tile t has landed (bounded wait: on a timeout the status says so)
    if (!mbar_wait(kvbar + t % KST, (uint32_t)((t / KST) & 1), &never, 1000000000ull) && threadIdx.x == 0)
      flag(status, DFLASH2_DEV_WAIT_TIMEOUT);
    const bf16* Ks = KV + (size_t)(t % KST) * 2 * MKT * LD;
    const bf16* Vs = Ks + MKT * LD;
    const int nk = min(MKT, k1 - (k0 + t * MKT));
#pragma unroll
    for (int slot = 0; slot < MCPW; ++slot) {
      const int combo = warp + slot * CLW;
      if (combo >= ncombo) break;
      const int rb = combo / ksplit, ks = combo % ksplit;
      const int kbeg = ks * (MKT / ksplit), kend = min(nk, (ks + 1) * (MKT / ksplit));
      for (int j0 = kbeg; j0 < kend; j0 += 16) {
        // S = Q K^T for 16 rows x 16 keys (two n8 tiles)
        float S0[4] = {0.f, 0.f, 0.f, 0.f}, S1[4] = {0.f, 0.f, 0.f, 0.f};
        const int mi = lane >> 3;
#pragma unroll
        for (int kk = 0; kk < DH / 16; ++kk) {
          uint32_t a[4], bk[4];
          ldsm4(a, Qs + (rb * 16 + (mi & 1) * 8 + (lane & 7)) * LD + kk * 16 + (mi >> 1) * 8);
          ldsm4(bk, Ks + (j0 + (mi >> 1) * 8 + (lane & 7)) * LD + kk * 16 + (mi & 1) * 8);
          mma16816(S0, a, bk[0], bk[1]);
          mma16816(S1, a, bk[2], bk[3]);
        }
        // scale and mask keys past the share
        const int cbase = j0 + (lane & 3) * 2;
        float sv[8] = {S0[0], S0[1], S0[2], S0[3], S1[0], S1[1], S1[2], S1[3]};
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const int key = cbase + (e >= 4 ? 8 : 0) + (e & 1);
          sv[e] = key < kend ? sv[e] * scale : -INFINITY;
        }
        // online softmax for the two rows this lane holds (row A: e = 0,1,4,5; row B: 2,3,6,7)
        float mx0 = fmaxf(fmaxf(sv[0], sv[1]), fmaxf(sv[4], sv[5]));
        float mx1 = fmaxf(fmaxf(sv[2], sv[3]), fmaxf(sv[6], sv[7]));
#pragma unroll
        for (int o2 = 1; o2 <= 2; o2 <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o2));
        }
        const float mn0 = fmaxf(m_st[slot][0], mx0), mn1 = fmaxf(m_st[slot][1], mx1);
        // the accumulators are rescaled only when a row's running max grew
        // (after the first keys it rarely does)
        if (__any_sync(0xffffffffu, mn0 > m_st[slot][0] || mn1 > m_st[slot][1])) {
          const float f0 = exp2f(m_st[slot][0] - mn0), f1 = exp2f(m_st[slot][1] - mn1);
          l_st[slot][0] *= f0;
          l_st[slot][1] *= f1;
#pragma unroll
          for (int n = 0; n < NT; ++n) {
            acc[slot][n][0] *= f0;
            acc[slot][n][1] *= f0;
            acc[slot][n][2] *= f1;
            acc[slot][n][3] *= f1;
          }
          m_st[slot][0] = mn0;
          m_st[slot][1] = mn1;
        }
        float p[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) p[e] = exp2f(sv[e] - ((e & 2) ? mn1 : mn0));
        // each lane keeps the sum of its own keys' weights; the four lanes of
        // a row are summed once, after the key loop
        l_st[slot][0] += (p[0] + p[1]) + (p[4] + p[5]);
        l_st[slot][1] += (p[2] + p[3]) + (p[6] + p[7]);
        // P as the A operand, split hi + lo
        float lo[8];
        uint32_t ph[4], pl[4];
#pragma unroll
        for (int e = 0; e < 8; ++e) lo[e] = p[e] - __bfloat162float(__float2bfloat16_rn(p[e]));
        ph[0] = pack_bf16(p[0], p[1]);
        ph[1] = pack_bf16(p[2], p[3]);
        ph[2] = pack_bf16(p[4], p[5]);
        ph[3] = pack_bf16(p[6], p[7]);
        pl[0] = pack_bf16(lo[0], lo[1]);
        pl[1] = pack_bf16(lo[2], lo[3]);
        pl[2] = pack_bf16(lo[4], lo[5]);
        pl[3] = pack_bf16(lo[6], lo[7]);
#pragma unroll
        for (int n2 = 0; n2 < DH / 16; ++n2) {
          uint32_t bv[4];
          ldsm4_t(bv, Vs + (j0 + (mi & 1) * 8 + (lane & 7)) * LD + n2 * 16 + (mi >> 1) * 8);
          mma16816(acc[slot][2 * n2], ph, bv[0], bv[1]);
          mma16816(acc[slot][2 * n2], pl, bv[0], bv[1]);
          mma16816(acc[slot][2 * n2 + 1], ph, bv[2], bv[3]);
          mma16816(acc[slot][2 * n2 + 1], pl, bv[2], bv[3]);
        }
      }
    }
    __syncthreads();  // tile t is consumed: its stage takes tile t + KST
    if (t + KST < ntiles) issue(k0 + (t + KST) * MKT, t % KST);
  }
  // (the last iteration's barrier: every warp is done with the K/V stages,
  // which now hold the partial states)
  // each combination's partial state -> shared memory (empty ones: m = -inf, l = 0)
#pragma unroll
  for (int slot = 0; slot < MCPW; ++slot) {
    const int combo = warp + slot * CLW;
    if (combo >= ncombo) break;
#pragma unroll
    for (int o2 = 1; o2 <= 2; o2 <<= 1) {  // a row's weight sum over its four lanes
      l_st[slot][0] += __shfl_xor_sync(0xffffffffu, l_st[slot][0], o2);
      l_st[slot][1] += __shfl_xor_sync(0xffffffffu, l_st[slot][1], o2);
    }
    float* cb = comb + (size_t)combo * 16 * FS;
    const int r0 = lane >> 2, c0 = (lane & 3) * 2;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      cb[r0 * FS + n * 8 + c0] = acc[slot][n][0];
      cb[r0 * FS + n * 8 + c0 + 1] = acc[slot][n][1];
      cb[(r0 + 8) * FS + n * 8 + c0] = acc[slot][n][2];
      cb[(r0 + 8) * FS + n * 8 + c0 + 1] = acc[slot][n][3];
    }
    if ((lane & 3) == 0) {
      cb[r0 * FS + DH] = m_st[slot][0];
      cb[r0 * FS + DH + 1] = l_st[slot][0];
      cb[(r0 + 8) * FS + DH] = m_st[slot][1];
      cb[(r0 + 8) * FS + DH + 1] = l_st[slot][1];
    }
  }
  __syncthreads();
  // 1. merge each row's key shares in place, into its share-0 slot: weights
  //    e^(m_ks - M) per share (wk), merged (m, l) written by the row's thread
  float* wk = wts;  // [R][ksplit] in-CTA share weights
  for (int r = threadIdx.x; r < R; r += blockDim.x) {
    float* base = comb + ((size_t)(r / 16) * ksplit * 16 + r % 16) * FS + DH;
    float M = -INFINITY;
    for (int ks = 0; ks < ksplit; ++ks) {
      const float* b = base + (size_t)ks * 16 * FS;
      if (b[1] > 0.f) M = fmaxf(M, b[0]);
    }
    float l = 0.f;
    for (int ks = 0; ks < ksplit; ++ks) {
      const float* b = base + (size_t)ks * 16 * FS;
      const float w = b[1] > 0.f ? exp2f(b[0] - M) : 0.f;  // base-2 maxima
      wk[r * ksplit + ks] = w;
      l += b[1] * w;
    }
    base[0] = M;
    base[1] = l;
  }
  __syncthreads();
  if (ksplit > 1) {
    for (int idx = threadIdx.x; idx < R * (DH / 2); idx += blockDim.x) {
      const int r = idx / (DH / 2), c = (idx % (DH / 2)) * 2;
      float2* base = reinterpret_cast<float2*>(comb + ((size_t)(r / 16) * ksplit * 16 + r % 16) * FS + c);
      float2 acc2 = make_float2(0.f, 0.f);
      for (int ks = 0; ks < ksplit; ++ks) {
        const float w = wk[r * ksplit + ks];
        if (w != 0.f) {
          const float2 v = base[(size_t)ks * 16 * FS / 2];
          acc2.x += v.x * w;
          acc2.y += v.y * w;
        }
      }
      *base = acc2;
    }
  }
  cluster_sync();  // every CTA's merged partials are complete and visible to the cluster

  // 2. row r's partials: one per CTA p of the cluster, in its share-0 slot.
  //    This CTA merges rows r = sp, sp + NS, ...: weights e^(m_p - M) / den.
  const int nmine = sp < R ? (R - sp + NS - 1) / NS : 0;
  float* cw = wts + (size_t)R * ksplit;  // [rows of this CTA][NS]
  for (int mi = threadIdx.x; mi < nmine; mi += blockDim.x) {
    const int r = sp + mi * NS;
    const float* base = comb + ((size_t)(r / 16) * ksplit * 16 + r % 16) * FS + DH;
    float2 ml[kMaxCluster];
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p)
      if (p < NS) ml[p] = ld_dsmem2(dsmem_addr(base, p));
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p)
      if (p < NS && ml[p].y > 0.f) M = fmaxf(M, ml[p].x);
    float den = 0.f;
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p)
      if (p < NS) {
        ml[p].x = ml[p].y > 0.f ? exp2f(ml[p].x - M) : 0.f;  // base-2 maxima
        den += ml[p].y * ml[p].x;
      }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p)
      if (p < NS) cw[mi * NS + p] = ml[p].x * inv;
  }
  __syncthreads();
  // O = sum over the cluster's partials of acc * weight, two elements per thread
  for (int idx = threadIdx.x; idx < nmine * (DH / 2); idx += blockDim.x) {
    const int mi = idx / (DH / 2), c = (idx % (DH / 2)) * 2;
    const int r = sp + mi * NS;
    const float* base = comb + ((size_t)(r / 16) * ksplit * 16 + r % 16) * FS + c;
    float2 v[kMaxCluster];
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p)
      if (p < NS) v[p] = ld_dsmem2(dsmem_addr(base, p));
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int p = 0; p < kMaxCluster; ++p)
      if (p < NS) {
        const float w = cw[mi * NS + p];
        if (w != 0.f) {
          a0 += v[p].x * w;
          a1 += v[p].y * w;
        }
      }
    const int i = r / grp, h = g * grp + r % grp;
    *reinterpret_cast<__nv_bfloat162*>(o + ((size_t)s * B + i) * nq * DH + h * DH + c) = __floats2bfloat162_rn(a0, a1);
  }
  cluster_sync();  // the other CTAs may still be reading this CTA's partials
}

// O[s, i, h, :] = sum_chunks acc e^(m - M) / sum_chunks l e^(m - M).
// One CTA per (sequence, kv head, group of CR query rows): the chunk weights
// e^(m - M) / den of its rows are formed once in shared memory, then every
// output element sums its chunks with coalesced, batched loads.
constexpr int CR = 8;

template <typename T>
__global__ void __launch_bounds__(256) attn_combine_kernel(const float* __restrict__ part, int B, int nq, int nkv,
                                                           int d, int nsplit, T* __restrict__ o) {
  extern __shared__ float cw[];  // [nsplit][CR] weights
  pdl_launch_next();
  pdl_wait();
  const int nrg = (nq / nkv * B + CR - 1) / CR;
  const int rg = blockIdx.x % nrg, g = (blockIdx.x / nrg) % nkv, s = blockIdx.x / (nrg * nkv);
  const int grp = nq / nkv, R = grp * B;
  const int r0 = rg * CR, nr = min(CR, R - r0);
  const float* base = part + (((size_t)s * nkv + g) * nsplit) * R * (d + 2);
  const size_t sstride = (size_t)R * (d + 2);
  // m and l of every (chunk, row) into shared memory (cw = m, cl = l)
  float* cl = cw + nsplit * CR;
  for (int idx = threadIdx.x; idx < nsplit * CR; idx += blockDim.x) {
    const int sp = idx / CR, rr = idx % CR;
    float m = -INFINITY, l = 0.f;
    if (rr < nr) {
      const float* p = base + sp * sstride + (size_t)(r0 + rr) * (d + 2);
      l = p[d + 1];
      m = l > 0.f ? p[d] : -INFINITY;
    }
    cw[idx] = m;
    cl[idx] = l;
  }
  __syncthreads();
  if (threadIdx.x < CR) {
    const int rr = threadIdx.x;
    float M = -INFINITY;
    for (int sp = 0; sp < nsplit; ++sp) M = fmaxf(M, cw[sp * CR + rr]);
    float den = 0.f;
    for (int sp = 0; sp < nsplit; ++sp) {
      const float m = cw[sp * CR + rr];
      if (m > -INFINITY && rr < nr) {
        const float e = expf(m - M);
        den += cl[sp * CR + rr] * e;
        cw[sp * CR + rr] = e;
      } else {
        cw[sp * CR + rr] = 0.f;
      }
    }
    const float inv = den > 0.f ? 1.f / den : 0.f;
    for (int sp = 0; sp < nsplit; ++sp) cw[sp * CR + rr] *= inv;
  }
  __syncthreads();
  constexpr int U = 8;
  for (int idx = threadIdx.x; idx < nr * d; idx += blockDim.x) {
    const int rr = idx / d, c = idx % d;
    const float* p = base + (size_t)(r0 + rr) * (d + 2) + c;
    float num = 0.f;
    for (int sp0 = 0; sp0 < nsplit; sp0 += U) {
      float v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) v[u] = sp0 + u < nsplit ? p[(sp0 + u) * sstride] : 0.f;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (sp0 + u < nsplit) {
          const float w = cw[(sp0 + u) * CR + rr];
          if (w != 0.f) num += v[u] * w;  // empty chunks leave acc unwritten
        }
    }
    const int r = r0 + rr, i = r / grp, h = g * grp + r % grp;
    st(&o[((size_t)s * B + i) * nq * d + h * d + c], num);
  }
}

int chunk_of(int max_ctx, int B, int batch, int nkv, int nsm) {
  const long L = (long)max_ctx + B;
  long ch = (L * batch * nkv + 4L * nsm - 1) / (4L * nsm);
  ch = ((ch + 63) / 64) * 64;
  return (int)std::max(64L, std::min(1024L, ch));
}

template <int DH>
int launch_cluster(int R, int max_ctx, int page_size, int batch, int nkv, const Ctx& c, const bf16* q,
                   const bf16* kb, const bf16* vb, const bf16* kc, const bf16* vc, const int32_t* block_table,
                   int max_pages, int n_pages, const int32_t* ctx_len, const int32_t* new_off, int B, int nq,
                   int window, bf16* o) {
  static bool attr = false;  // set once, before any capture
  if (!attr) {
    if (cudaFuncSetAttribute(attn_cluster_kernel<DH>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kAttnSmem))
      return DFLASH2_ERR_CUDA;
    attr = true;
  }
  const int ns = attn_cluster_ctas(max_ctx, B, batch, nkv, c.nsm);
  // chunk length bound (keys), then its pages
  const long ch = ((((long)max_ctx + B + ns - 1) / ns) + 15) & ~15L;
  const int npg = (int)((ch + page_size - 1) / page_size + 1);
  // K/V ring: tiles of mkt keys (the share geometry above), as many stages
  // (up to four) as the shared memory holds beside the Q tile and page list
  const int nrb = (R + 15) / 16;
  const int ksplit = attn_ksplit(nrb), mkt = attn_tile_keys(ksplit);
  int kst = kMaxStages;
  size_t smem = attn_cl_smem<DH>(R, npg, mkt, kst, ksplit);
  while (smem > kAttnSmem && kst > 2) smem = attn_cl_smem<DH>(R, npg, mkt, --kst, ksplit);
  if (smem > kAttnSmem) return DFLASH2_ERR_SHAPE;
  // whole 16-key pages of the cache by TMA: the cache viewed as
  // [n_pages * 16 rows][nkv * DH], a box of 16 rows x (DH + 8) elements
  CUtensorMap tmK, tmV;
  std::memset(&tmK, 0, sizeof(tmK));
  std::memset(&tmV, 0, sizeof(tmV));
  int page_tma = page_size == 16 && (long long)n_pages * 16 < (1LL << 31);
  if (page_tma)
    page_tma = make_rows_map(&tmK, kc, (long long)n_pages * 16, nkv * DH, (long long)nkv * DH, DH + 8, 16) == 0 &&
               make_rows_map(&tmV, vc, (long long)n_pages * 16, nkv * DH, (long long)nkv * DH, DH + 8, 16) == 0;
  return launch_kx(attn_cluster_kernel<DH>, dim3(ns, nkv, batch), dim3(CLT), smem, c, ns, q, kb, vb, kc, vc,
                   block_table, max_pages, page_size, n_pages, ctx_len, new_off, B, nq, nkv, npg, window, mkt, kst,
                   ksplit, tmK, tmV, page_tma, o, c.status);
}

}  // namespace

// CTAs per cluster: at most 8 (the portable cluster size) and one per 64
// keys of the longest sequence.  A CTA takes a whole SM, so while the (kv
// head, sequence) pairs fit the SMs the clusters fill one wave; beyond that,
// enough CTAs for about two per SM, finer pieces for the scheduler to
// balance ragged contexts.
int attn_cluster_ctas(int max_ctx, int B, int batch, int nkv, int nsm) {
  const long L = (long)max_ctx + B;
  const long pairs = (long)nkv * batch;
  const long fill = pairs <= nsm ? nsm / pairs : (2L * nsm + pairs - 1) / pairs;
  return (int)std::max(1L, std::min<long>({8L, (L + 63) / 64, fill}));
}

std::atomic<int> g_attn_mode{0};
std::atomic<int> g_attn_last{0};
void attention_force_mode(int mode) { g_attn_mode.store(mode); }
int attention_last_kernel() { return g_attn_last.load(); }

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
                     int max_ctx, int window, float* part, void* o_out, const Ctx& c) {
  const int R = (nq / nkv) * B;
  const int nrb = (R + 15) / 16;
  const int mode = g_attn_mode.load();
  // the tcgen05 kernel where it was measured faster: more than 32 query rows
  // per kv head and chunks of at least 1024 keys per CTA (27B b=8 ctx 8192:
  // +8% per step; 30B-A3B ctx 8192: +2% at b=1, +8% at b=8, +27% at b=64,
  // +37% at b=256).  With shorter chunks (every 1k-context point, 258-516
  // keys per CTA) and at 32 rows (the 8B shapes) the mma.sync cluster kernel
  // is 1-4% faster: its per-CTA start-up is shorter.
  const long ns = attn_cluster_ctas(max_ctx, B, batch, nkv, c.nsm);
  const long chunk = ((long)max_ctx + B + ns - 1) / ns;
  if ((mode == 2 || (mode == 0 && R > 32 && chunk >= 1024)) && attention_tc_fits(dtype, d, page_size, R)) {
    // (a page list too long for its shared memory: the cluster kernel below)
    const int rc = launch_attention_tc(q, kb, vb, kc, vc, block_table, max_pages, page_size, n_pages, ctx_len,
                                       new_off, batch, B, nq, nkv, max_ctx, window, o_out, c);
    if (rc != DFLASH2_ERR_SHAPE) {
      g_attn_last.store(2);
      return rc;
    }
  }
  if (dtype == DFLASH2_BF16 && (d == 64 || d == 128) && nrb <= CLW) {  // a warp per (row block, key share)
    g_attn_last.store(1);
    const bf16 *q_ = static_cast<const bf16*>(q), *kb_ = static_cast<const bf16*>(kb),
               *vb_ = static_cast<const bf16*>(vb), *kc_ = static_cast<const bf16*>(kc),
               *vc_ = static_cast<const bf16*>(vc);
    bf16* o_ = static_cast<bf16*>(o_out);
    if (d == 64)
      return launch_cluster<64>(R, max_ctx, page_size, batch, nkv, c, q_, kb_, vb_, kc_, vc_, block_table, max_pages,
                                n_pages, ctx_len, new_off, B, nq, window, o_);
    return launch_cluster<128>(R, max_ctx, page_size, batch, nkv, c, q_, kb_, vb_, kc_, vc_, block_table, max_pages,
                               n_pages, ctx_len, new_off, B, nq, window, o_);
  }
  // SIMT path (fp32 storage, or row counts beyond the tensor-core kernel):
  // key-chunk partials in global memory, then the combine kernel
  g_attn_last.store(3);
  const int ch = chunk_of(max_ctx, B, batch, nkv, c.nsm);
  const int nsplit = (max_ctx + B + ch - 1) / ch;
  const size_t smem = attn_smem(R, d);
  const dim3 grid(nsplit, nkv, batch);
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
  int rc;
  if (dtype == DFLASH2_BF16)
    rc = launch_k(attn_partial_kernel<bf16>, grid, dim3(AT), smem, c, static_cast<const bf16*>(q),
                  static_cast<const bf16*>(kb), static_cast<const bf16*>(vb), static_cast<const bf16*>(kc),
                  static_cast<const bf16*>(vc), block_table, max_pages, page_size, n_pages, ctx_len, new_off, B, nq,
                  nkv, d, ch, nsplit, window, part, c.status);
  else
    rc = launch_k(attn_partial_kernel<float>, grid, dim3(AT), smem, c, static_cast<const float*>(q),
                  static_cast<const float*>(kb), static_cast<const float*>(vb), static_cast<const float*>(kc),
                  static_cast<const float*>(vc), block_table, max_pages, page_size, n_pages, ctx_len, new_off, B, nq,
                  nkv, d, ch, nsplit, window, part, c.status);
  if (rc) return rc;
  Ctx cc = c;
  cc.pdl = true;  // same-stream successor of the partial kernel
  const dim3 cgrid(batch * nkv * ((R + CR - 1) / CR));
  const size_t csm = 2 * (size_t)nsplit * CR * sizeof(float);
  if (dtype == DFLASH2_BF16)
    return launch_k(attn_combine_kernel<bf16>, cgrid, dim3(256), csm, cc, (const float*)part, B, nq, nkv, d, nsplit,
                    static_cast<bf16*>(o_out));
  return launch_k(attn_combine_kernel<float>, cgrid, dim3(256), csm, cc, (const float*)part, B, nq, nkv, d, nsplit,
                  static_cast<float*>(o_out));
}

}  // namespace df2
