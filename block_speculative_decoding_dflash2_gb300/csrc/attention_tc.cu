// Non-causal block attention on the 5th-generation tensor cores (tcgen05
// with TMEM accumulators), head dimension 128, bf16 storage ("Train a DFlash
// Drafter for Speculative Decoding", "What is DFlash?": one non-causal
// forward over the block, which attends to the committed context and to
// itself; grouped-query sharing of the kv heads).
//
// The work split is the cluster kernel's: one CTA per (key chunk, kv head,
// sequence), the chunks of a (kv head, sequence) pair in one thread-block
// cluster, the unnormalised partials merged through distributed shared
// memory, O written once.  The query rows of a kv head (grp heads x B block
// positions, R <= 80) are the N dimension of every MMA, so the keys and the
// head dimension take the 128-row M side:
//
//   S^T = K Q^T     M = 128 keys, N = the query rows, K = 128 dims
//   O^T += V^T P^T  M = 128 dims, N = the query rows, K = 128 keys
//
// K, Q and P^T are K-major operands; V^T is read MN-major straight from the
// V tile (each key a 128-byte row of 64 dims).  P is split into bf16 hi + lo
// parts (two MMAs), so the probabilities keep ~16 bits as in the mma.sync
// kernel.  Roles by warp:
//   warp 0      K/V tiles of 128 keys into a two-stage ring: whole 16-key
//               cache pages by TMA (128-byte swizzle, one box per page, half
//               head and K or V), the rest (a partial last page, the block's
//               own keys, zero rows past the chunk, every row when the chunk
//               does not start on a page) by cp.async into the same
//               swizzled layout;
//   warp 1      TMEM allocation and the MMA issue, S^T into two buffers so
//               the next tile's scores are ready while P of this one is formed;
//   warps 2..9  the softmax, thread = (key of the tile, half of the query
//               rows): scores in base-2 units against a per-row reference
//               maximum that moves only when a score passes it by more than
//               2^8 (then the tile's column maxima are formed and the O^T
//               accumulator and the weight sums are rescaled); P = 2^(x - m)
//               as hi + lo into shared memory; per-thread weight sums,
//               reduced over the keys once at the end.
#include <cstring>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int TK = 128;          // keys per K/V tile (M of S^T)
constexpr int TD = 128;          // head dimension (M of O^T)
constexpr int TST = 2;           // K/V stages
constexpr int TW = 10;           // warps: loads, MMA, 8 softmax
constexpr int TT = 32 * TW;      // threads
constexpr int TSW = 8;           // softmax warps
constexpr int TNS = 8;           // CTAs per cluster at most
constexpr int kTcMaxRows = 80;   // query rows per kv head
constexpr uint64_t kTcWaitNs = 1000000000ull;
constexpr float kRescaleAt = 8.f;  // base-2 headroom of the reference maximum

constexpr int KV_STAGE = 2 * TK * TD * 2;  // K and V tiles of a stage (64 KB)
constexpr int HALF = TK * 128;             // one 64-dim half of a K or V tile (16 KB)

// Shared-memory layout (offsets from the 1024-byte aligned base).
template <int NP>
struct TcSmem {
  static constexpr int KV = 0;                         // [TST][K, V][2 halves][TK][128 B]
  static constexpr int Q = TST * KV_STAGE;             // [2 halves][NP][128 B]
  static constexpr int P = Q + 2 * NP * 128;           // [hi, lo][2 key halves][NP][128 B]
  static constexpr int RED = P + 4 * NP * 128;         // float [4 lane quarters][NP]
  static constexpr int MS = RED + 4 * NP * 4;          // float [NP] reference maxima of the rows
  static constexpr int CW = MS + NP * 4;               // float [rows of this CTA][TNS] merge weights
  static constexpr int PG = CW + (NP + TNS) * TNS * 4;  // int page ids of the chunk
  static size_t bytes(int npg) { return 1024 + PG + (size_t)npg * 4 + 16 * 8 + 16; }
};

__device__ __forceinline__ void sm_bar_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
__device__ __forceinline__ bool sm_bar_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, 256, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

template <int NP>
__global__ void __launch_bounds__(TT, 1) attn_tc_kernel(
    const bf16* __restrict__ q, const bf16* __restrict__ kb, const bf16* __restrict__ vb,
    const bf16* __restrict__ kc, const bf16* __restrict__ vc, const int32_t* __restrict__ block_table,
    int max_pages, int page_size, int n_pages, const int32_t* __restrict__ ctx_len,
    const int32_t* __restrict__ new_off, int B, int nq, int nkv, int npg, int window,
    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV, int page_tma,
    bf16* __restrict__ o, unsigned* status) {
  using L = TcSmem<NP>;
  constexpr int HC = NP / 2;  // query rows (TMEM columns) per softmax thread
  constexpr int FS = TD + 2;  // partial row: acc[TD], m, l
  static_assert(NP % 16 == 0 && NP <= kTcMaxRows, "query rows");
  extern __shared__ uint8_t smraw[];
  uint8_t* sm = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smraw) + 1023) & ~uintptr_t(1023));
  float* red = reinterpret_cast<float*>(sm + L::RED);
  float* msh = reinterpret_cast<float*>(sm + L::MS);
  float* cw = reinterpret_cast<float*>(sm + L::CW);
  int* pg = reinterpret_cast<int*>(sm + L::PG);
  uint64_t* bars = reinterpret_cast<uint64_t*>((reinterpret_cast<uintptr_t>(pg + npg) + 7) & ~uintptr_t(7));
  uint64_t* kvfull = bars;       // [TST] a tile landed (1 arrival + TMA bytes)
  uint64_t* kvempty = bars + 2;  // [TST] its PV MMAs completed (commit)
  uint64_t* sfull = bars + 4;    // [2] S^T of a tile in TMEM (commit)
  uint64_t* sempty = bars + 6;   // [2] S^T read by the softmax warps (8 arrivals)
  uint64_t* pready = bars + 8;   // P of a tile in shared memory (8 arrivals)
  uint64_t* odone = bars + 9;    // a tile's PV MMAs completed (commit)
  uint64_t* qready = bars + 10;  // Q rows in shared memory (8 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 11);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* comb = reinterpret_cast<float*>(sm + L::KV);  // [R][FS] after the key loop (aliases the ring)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = gridDim.x, sp = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int grp = nq / nkv, R = grp * B;
  pdl_launch_next();
  if (threadIdx.x == 0) {
    for (int i = 0; i < TST; ++i) {
      mbar_init(kvfull + i, 1);
      mbar_init(kvempty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sfull + i, 1);
      mbar_init(sempty + i, TSW);
    }
    mbar_init(pready, TSW);
    mbar_init(odone, 1);
    mbar_init(qready, TSW);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 256);
    tmem_relinquish();
  }

  pdl_wait();
  const int P = ctx_len[s] + (new_off[s + 1] - new_off[s]);
  const int Lk = P + B;
  const int w0 = window > 0 ? max(0, P - window) : 0;
  const int CH = (((Lk - w0 + NS - 1) / NS) + 15) & ~15;
  const int k0 = w0 + min(sp * CH, Lk - w0), k1 = min(k0 + CH, Lk);
  if (P > max_pages * page_size && sp == 0 && threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
  const int pbase = k0 / page_size;
  const int pend = k0 < min(k1, P) ? (min(k1, P) - 1) / page_size + 1 : pbase;
  for (int i = threadIdx.x; i < pend - pbase && i < npg; i += blockDim.x) {
    const int pi = pbase + i;
    pg[i] = pi < max_pages ? block_table[(size_t)s * max_pages + pi] : -1;
  }
  if (pend - pbase > npg && threadIdx.x == 0) flag(status, DFLASH2_DEV_BAD_LENGTH);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int ntiles = (k1 - k0 + TK - 1) / TK;  // 0 for an empty chunk
  auto fail = [&]() {
    *abort_flag = 1;
    flag(status, DFLASH2_DEV_WAIT_TIMEOUT);
  };

  if (warp == 0) {
    // ---------------------------------------------------------------- K/V loads
    // Lane c < 16 moves 16-byte chunk c of a key's K row, lane 16 + c the
    // same chunk of its V row; chunk c lands in half c / 8, at position
    // (c % 8) ^ (row % 8) of the row's 128 bytes (the TMA's 128-byte swizzle).
    const bool tma_ok = page_tma && (k0 % 16) == 0;
    const uint64_t pol = policy_evict_first();
    const bool isv = lane >= 16;
    const int c = lane & 15;
    int issued = 0;
    for (int t = 0; t < ntiles; ++t) {
      const int st = t % TST;
      if (t >= TST) {
        const bool free_ = __all_sync(0xffffffffu, mbar_wait(kvempty + st, (uint32_t)(((t / TST) - 1) & 1),
                                                             abort_flag, kTcWaitNs));
        if (!free_) {
          if (lane == 0) fail();
          break;
        }
      }
      const int t0 = k0 + t * TK;
      uint8_t* Kst = sm + L::KV + st * KV_STAGE;
      uint8_t* Vst = Kst + KV_STAGE / 2;
      // whole context pages of the tile: TMA boxes where the page id is valid
      const int cend = max(t0, min(min(t0 + TK, k1), P));
      const int nfull = tma_ok ? (cend - t0) / 16 : 0;
      uint32_t vmask = 0;
      for (int i = 0; i < nfull; ++i) {
        const int li = (t0 + 16 * i) / 16 - pbase;
        const int page = li < npg ? pg[li] : -1;
        if (page >= 0 && page < n_pages) vmask |= 1u << i;
      }
      // every other row by cp.async (zero-filled where nothing is read)
      bool manual = false;
      for (int r = 0; r < TK; ++r) {
        if ((r >> 4) < nfull && ((vmask >> (r >> 4)) & 1)) continue;
        manual = true;
        const int j = t0 + r;
        const bf16* src = kc;
        bool ok = false;
        if (j < k1) {
          if (j < P) {
            const int li = j / page_size - pbase;
            const int page = li < npg ? pg[li] : -1;
            if (page >= 0 && page < n_pages) {
              src = (isv ? vc : kc) + (((size_t)page * page_size + j % page_size) * nkv + g) * TD + c * 8;
              ok = true;
            } else if (lane == 0) {
              flag(status, DFLASH2_DEV_BAD_PAGE);
            }
          } else {
            src = (isv ? vb : kb) + (((size_t)s * B + (j - P)) * nkv + g) * TD + c * 8;
            ok = true;
          }
        }
        cp_async16((isv ? Vst : Kst) + (c >> 3) * HALF + r * 128 + (((c & 7) ^ (r & 7)) << 4), src, ok);
      }
      if (manual) {
        cp_async_commit();
        cp_async_wait<0>();
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(kvfull + st, (uint32_t)__popc(vmask) * 4u * 2048u);
      __syncwarp();
      // lane 4i + w: page i, box w (K half 0, K half 1, V half 0, V half 1)
      if (lane < 4 * nfull && ((vmask >> (lane >> 2)) & 1)) {
        const int i = lane >> 2, w = lane & 3;
        const int page = pg[(t0 + 16 * i) / 16 - pbase];
        uint8_t* dst = (w < 2 ? Kst : Vst) + (w & 1) * HALF + i * 16 * 128;
        tma_load_2d(dst, w < 2 ? &tmK : &tmV, kvfull + st, g * TD + (w & 1) * 64, page * 16, pol);
      }
      ++issued;
    }
    // copies still in flight (after an abort) land before the CTA moves on
    for (int t = max(0, issued - TST); t < issued; ++t) {
      volatile int never = 0;
      mbar_wait(kvfull + t % TST, (uint32_t)((t / TST) & 1), &never, kTcWaitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    // One thread issues every MMA.  It polls for whichever of the next PV
    // (P of tile t formed) or the next S^T (tile landed, its S buffer read)
    // can go, PV first, so a PV never waits behind a load.
    if (lane == 0 && ntiles > 0) {
      const uint32_t id_s = idesc_bf16_f32(TK, NP);
      const uint32_t id_o = idesc_bf16_f32(TD, NP) | (1u << 15);  // A = V^T read MN-major
      const uint32_t q_base = smem_u32(sm + L::Q), p_base = smem_u32(sm + L::P);
      bool ok = mbar_wait(qready, 0, abort_flag, kTcWaitNs);
      tc_fence_after();
      int ns_ = 0, npv = 0;
      uint64_t t_last = globaltimer();
      while (ok && npv < ntiles) {
        bool did = false;
        if (npv < ns_ && mbar_try_wait(smem_u32(pready), (uint32_t)(npv & 1))) {
          tc_fence_after();
          const int st = npv % TST;
          const uint32_t v_base = smem_u32(sm + L::KV + st * KV_STAGE + KV_STAGE / 2);
          const uint32_t od = tmem + 2 * NP;
#pragma unroll
          for (int part = 0; part < 2; ++part) {  // P hi, then P lo
#pragma unroll
            for (int j = 0; j < TK / 16; ++j) {
              const uint64_t ad = sdesc_mn_sw128(v_base + j * 2048, HALF, 1024);
              const uint64_t bd = sdesc_sw128(p_base + part * 2 * NP * 128 + (j >> 2) * NP * 128 + (j & 3) * 32);
              umma_bf16(od, ad, bd, id_o, (npv > 0 || part > 0 || j > 0) ? 1u : 0u);
            }
          }
          umma_commit(odone);
          umma_commit(kvempty + st);
          ++npv;
          did = true;
        } else if (ns_ < ntiles && ns_ < npv + 2 &&
                   mbar_try_wait(smem_u32(kvfull + ns_ % TST), (uint32_t)((ns_ / TST) & 1)) &&
                   (ns_ < 2 || mbar_try_wait(smem_u32(sempty + (ns_ & 1)), (uint32_t)(((ns_ >> 1) - 1) & 1)))) {
          tc_fence_after();
          const uint32_t k_base = smem_u32(sm + L::KV + (ns_ % TST) * KV_STAGE);
          const uint32_t sd = tmem + (uint32_t)((ns_ & 1) * NP);
#pragma unroll
          for (int kk = 0; kk < TD / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(k_base + (kk >> 2) * HALF + (kk & 3) * 32);
            const uint64_t bd = sdesc_sw128(q_base + (kk >> 2) * NP * 128 + (kk & 3) * 32);
            umma_bf16(sd, ad, bd, id_s, kk > 0 ? 1u : 0u);
          }
          umma_commit(sfull + (ns_ & 1));
          ++ns_;
          did = true;
        }
        if (did) {
          t_last = globaltimer();
        } else if (*abort_flag || globaltimer() - t_last > kTcWaitNs) {
          ok = false;
        }
      }
      if (!ok) fail();
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------------- softmax
    const int qd = warp & 3;      // TMEM lane quarter this warp may access
    const int h = (warp - 2) >> 2;  // half of the query rows
    const int kl = qd * 32 + lane;  // key of the tile (S^T lane) = head dim (O^T lane)
    const int n0 = h * HC;
    const uint32_t lane_base = tmem + ((uint32_t)(qd * 32) << 16);
    // query rows -> shared memory, K-major with the 128-byte swizzle, zero padding
    for (int idx = (warp - 2) * 32 + lane; idx < NP * 16; idx += TSW * 32) {
      const int r = idx >> 4, cc = idx & 15;
      const bool ok = r < R;
      const bf16* src = ok ? q + (((size_t)s * B + r / grp) * nq + g * grp + r % grp) * TD + cc * 8 : q;
      cp_async16(sm + L::Q + (cc >> 3) * NP * 128 + r * 128 + (((cc & 7) ^ (r & 7)) << 4), src, ok);
    }
    cp_async_commit();
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(qready);

    constexpr float kLog2e = 1.4426950408889634f;
    const float scale = rsqrtf((float)TD) * kLog2e;
    // the rows' reference maxima live in shared memory (one copy for the 128
    // key lanes that use them); the weight sums in registers, per key lane
    float l[HC];
#pragma unroll
    for (int i = 0; i < HC; ++i) l[i] = 0.f;
    if (qd == 0 && lane == 0)
      for (int i = 0; i < HC; ++i) msh[n0 + i] = -INFINITY;
    sm_bar_sync();
    // this thread's P^T element (row n, key kl): key half kl / 64, 16-byte
    // chunk (kl % 64) / 8 swizzled by the row, element kl % 8
    uint8_t* p_hi = sm + L::P + (kl >> 6) * NP * 128 + (kl & 7) * 2;
    uint8_t* p_lo = p_hi + 2 * NP * 128;
    const int pchunk = (kl & 63) >> 3;
    // ok stays uniform over the 256 softmax threads: a failed wait only
    // clears it, and the threads leave the key loop together, at the vote at
    // the top of the next tile, so every named barrier sees all of them
    bool ok = true;
    for (int t = 0; t < ntiles; ++t) {
      if (sm_bar_or(!ok)) break;
      const bool valid = k0 + t * TK + kl < k1;
      if (!mbar_wait(sfull + (t & 1), (uint32_t)((t >> 1) & 1), abort_flag, kTcWaitNs)) {
        fail();
        ok = false;
      }
      ok = __all_sync(0xffffffffu, ok);  // warp-collective TMEM loads below
      tc_fence_after();
      float x[HC];
      {
        uint32_t r[HC];
#pragma unroll
        for (int c8 = 0; c8 < HC / 8; ++c8)
          tmem_ld8_nowait(lane_base + (uint32_t)((t & 1) * NP + n0 + c8 * 8),
                          *reinterpret_cast<uint32_t(*)[8]>(&r[c8 * 8]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < HC; ++i) x[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty + (t & 1));
      bool need = false;
#pragma unroll
      for (int i = 0; i < HC; ++i) {
        x[i] = valid ? x[i] * scale : -INFINITY;
        need |= x[i] > msh[n0 + i] + kRescaleAt;
      }
      bool have_o = false;  // waited for the previous tile's PV
      if (sm_bar_or(need)) {
        // new reference maxima: the tile's column maxima over its 128 keys
#pragma unroll
        for (int i = 0; i < HC; ++i) {
          const float v = warp_max(x[i]);
          if (lane == 0) red[qd * NP + n0 + i] = v;
        }
        sm_bar_sync();
        if (t > 0) {  // O^T holds the earlier tiles: rescale it once their PV is done
          if (!mbar_wait(odone, (uint32_t)((t - 1) & 1), abort_flag, kTcWaitNs)) {
            fail();
            ok = false;
          }
          ok = __all_sync(0xffffffffu, ok);
          tc_fence_after();
          have_o = true;
        }
#pragma unroll
        for (int c8 = 0; c8 < HC / 8; ++c8) {
          float f[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int i = c8 * 8 + e, n = n0 + i;
            const float mt = fmaxf(fmaxf(red[n], red[NP + n]), fmaxf(red[2 * NP + n], red[3 * NP + n]));
            const float mo = msh[n], mn = fmaxf(mo, mt);
            f[e] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
            l[i] *= f[e];
          }
          if (t > 0 && ok) {
            uint32_t r8[8];
            const uint32_t ta = lane_base + (uint32_t)(2 * NP + n0 + c8 * 8);
            tmem_ld8_nowait(ta, r8);
            tmem_ld_wait();
#pragma unroll
            for (int e = 0; e < 8; ++e) r8[e] = __float_as_uint(__uint_as_float(r8[e]) * f[e]);
            tmem_st8(ta, r8);
          }
        }
        if (t > 0 && ok) tmem_st_wait();
        sm_bar_sync();  // every thread has its factors: the maxima move
        if (qd == 0 && lane == 0)
          for (int i = 0; i < HC; ++i) {
            const int n = n0 + i;
            msh[n] = fmaxf(msh[n], fmaxf(fmaxf(red[n], red[NP + n]), fmaxf(red[2 * NP + n], red[3 * NP + n])));
          }
        sm_bar_sync();
      }
      if (t > 0 && !have_o) {  // P of the previous tile read by its PV before it is overwritten
        if (!mbar_wait(odone, (uint32_t)((t - 1) & 1), abort_flag, kTcWaitNs)) {
          fail();
          ok = false;
        }
        tc_fence_after();
      }
      // P = 2^(x - m), split hi + lo, into P^T (row n, key kl)
#pragma unroll
      for (int i = 0; i < HC; ++i) {
        const int n = n0 + i;
        const float p = x[i] == -INFINITY ? 0.f : exp2f(x[i] - msh[n]);
        l[i] += p;
        const __nv_bfloat16 hi = __float2bfloat16_rn(p);
        const __nv_bfloat16 lo = __float2bfloat16_rn(p - __bfloat162float(hi));
        const int off = n * 128 + ((pchunk ^ (n & 7)) << 4);
        *reinterpret_cast<__nv_bfloat16*>(p_hi + off) = hi;
        *reinterpret_cast<__nv_bfloat16*>(p_lo + off) = lo;
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pready);
    }
    // the last PV, then this CTA's partial rows: O^T columns, m and the
    // weight sums (over the 32 keys of a warp, then the 4 lane quarters)
    if (ntiles > 0 && ok) {
      if (!mbar_wait(odone, (uint32_t)((ntiles - 1) & 1), abort_flag, kTcWaitNs)) fail();
      tc_fence_after();
    }
    sm_bar_sync();  // every read of red by the last tile is done
#pragma unroll
    for (int i = 0; i < HC; ++i) {
      const float v = warp_sum(l[i]);
      if (lane == 0) red[qd * NP + n0 + i] = v;
    }
    sm_bar_sync();
#pragma unroll
    for (int c8 = 0; c8 < HC / 8; ++c8) {
      float ov[8];
      if (ntiles > 0) {
        uint32_t r8[8];
        tmem_ld8_nowait(lane_base + (uint32_t)(2 * NP + n0 + c8 * 8), r8);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) ov[e] = __uint_as_float(r8[e]);
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) ov[e] = 0.f;
      }
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        const int n = n0 + c8 * 8 + e;
        if (n < R) comb[(size_t)n * FS + kl] = ov[e];
      }
    }
    if (qd == 0 && lane == 0) {  // one thread per half: the rows' m and weight sums
#pragma unroll
      for (int i = 0; i < HC; ++i) {
        const int n = n0 + i;
        if (n < R) {
          comb[(size_t)n * FS + TD] = msh[n];
          comb[(size_t)n * FS + TD + 1] = red[n] + red[NP + n] + red[2 * NP + n] + red[3 * NP + n];
        }
      }
    }
  }

  // ------------------------------------------------------------ cluster merge
  // Row r's partials, one per CTA p of the cluster: this CTA merges rows
  // r = sp, sp + NS, ... with weights 2^(m_p - M) / den (base-2 maxima).
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // every CTA's partial rows are complete and visible to the cluster
  const int nmine = sp < R ? (R - sp + NS - 1) / NS : 0;
  for (int mi = threadIdx.x; mi < nmine; mi += blockDim.x) {
    const int r = sp + mi * NS;
    const float* base = comb + (size_t)r * FS + TD;
    float2 ml[TNS];
#pragma unroll
    for (int p = 0; p < TNS; ++p)
      if (p < NS) ml[p] = ld_dsmem2(dsmem_addr(base, p));
    float M = -INFINITY;
#pragma unroll
    for (int p = 0; p < TNS; ++p)
      if (p < NS && ml[p].y > 0.f) M = fmaxf(M, ml[p].x);
    float den = 0.f;
#pragma unroll
    for (int p = 0; p < TNS; ++p)
      if (p < NS) {
        ml[p].x = ml[p].y > 0.f ? exp2f(ml[p].x - M) : 0.f;
        den += ml[p].y * ml[p].x;
      }
    const float inv = den > 0.f ? 1.f / den : 0.f;
#pragma unroll
    for (int p = 0; p < TNS; ++p)
      if (p < NS) cw[mi * TNS + p] = ml[p].x * inv;
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < nmine * (TD / 2); idx += blockDim.x) {
    const int mi = idx / (TD / 2), c = (idx % (TD / 2)) * 2;
    const int r = sp + mi * NS;
    const float* base = comb + (size_t)r * FS + c;
    float2 v[TNS];
#pragma unroll
    for (int p = 0; p < TNS; ++p)
      if (p < NS) v[p] = ld_dsmem2(dsmem_addr(base, p));
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int p = 0; p < TNS; ++p)
      if (p < NS) {
        const float w = cw[mi * TNS + p];
        if (w != 0.f) {
          a0 += v[p].x * w;
          a1 += v[p].y * w;
        }
      }
    const int i = r / grp, hh = g * grp + r % grp;
    *reinterpret_cast<__nv_bfloat162*>(o + ((size_t)s * B + i) * nq * TD + hh * TD + c) =
        __floats2bfloat162_rn(a0, a1);
  }
  cluster_sync();  // the other CTAs may still be reading this CTA's partials
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

template <int NP>
int launch_np(int max_ctx, int page_size, int batch, int nkv, const Ctx& c, const bf16* q, const bf16* kb,
              const bf16* vb, const bf16* kc, const bf16* vc, const int32_t* block_table, int max_pages,
              int n_pages, const int32_t* ctx_len, const int32_t* new_off, int B, int nq, int window, bf16* o) {
  const int ns = attn_cluster_ctas(max_ctx, B, batch, nkv, c.nsm);
  const long ch = ((((long)max_ctx + B + ns - 1) / ns) + 15) & ~15L;
  const int npg = (int)((ch + page_size - 1) / page_size + 1);
  const size_t smem = TcSmem<NP>::bytes(npg);
  if (smem > 227 * 1024) return DFLASH2_ERR_SHAPE;
  static bool attr = false;  // set once, before any capture
  if (!attr) {
    if (cudaFuncSetAttribute(attn_tc_kernel<NP>, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024))
      return DFLASH2_ERR_CUDA;
    attr = true;
  }
  // whole 16-key pages by TMA: the cache viewed as [n_pages * 16][nkv * 128],
  // a box of 16 rows x 64 elements (one half of a head), 128-byte swizzle
  CUtensorMap tmK, tmV;
  std::memset(&tmK, 0, sizeof(tmK));
  std::memset(&tmV, 0, sizeof(tmV));
  int page_tma = page_size == 16 && (long long)n_pages * 16 < (1LL << 31);
  if (page_tma)
    page_tma = make_sw128_map(&tmK, kc, (long long)n_pages * 16, nkv * TD, (long long)nkv * TD, 16) == 0 &&
               make_sw128_map(&tmV, vc, (long long)n_pages * 16, nkv * TD, (long long)nkv * TD, 16) == 0;
  return launch_kx(attn_tc_kernel<NP>, dim3(ns, nkv, batch), dim3(TT), smem, c, ns, q, kb, vb, kc, vc,
                   block_table, max_pages, page_size, n_pages, ctx_len, new_off, B, nq, nkv, npg, window, tmK, tmV,
                   page_tma, o, c.status);
}

}  // namespace

bool attention_tc_fits(int dtype, int d, int page_size, int R) {
  return dtype == DFLASH2_BF16 && d == TD && page_size == 16 && R >= 1 && R <= kTcMaxRows;
}

int launch_attention_tc(const void* q_, const void* kb_, const void* vb_, const void* kc_, const void* vc_,
                        const int32_t* block_table, int max_pages, int page_size, int n_pages,
                        const int32_t* ctx_len, const int32_t* new_off, int batch, int B, int nq, int nkv,
                        int max_ctx, int window, void* o_, const Ctx& c) {
  const bf16 *q = static_cast<const bf16*>(q_), *kb = static_cast<const bf16*>(kb_),
             *vb = static_cast<const bf16*>(vb_), *kc = static_cast<const bf16*>(kc_),
             *vc = static_cast<const bf16*>(vc_);
  bf16* o = static_cast<bf16*>(o_);
  const int R = (nq / nkv) * B;
  switch ((R + 15) / 16 * 16) {
    case 16: return launch_np<16>(max_ctx, page_size, batch, nkv, c, q, kb, vb, kc, vc, block_table, max_pages,
                                  n_pages, ctx_len, new_off, B, nq, window, o);
    case 32: return launch_np<32>(max_ctx, page_size, batch, nkv, c, q, kb, vb, kc, vc, block_table, max_pages,
                                  n_pages, ctx_len, new_off, B, nq, window, o);
    case 48: return launch_np<48>(max_ctx, page_size, batch, nkv, c, q, kb, vb, kc, vc, block_table, max_pages,
                                  n_pages, ctx_len, new_off, B, nq, window, o);
    case 64: return launch_np<64>(max_ctx, page_size, batch, nkv, c, q, kb, vb, kc, vc, block_table, max_pages,
                                  n_pages, ctx_len, new_off, B, nq, window, o);
    case 80: return launch_np<80>(max_ctx, page_size, batch, nkv, c, q, kb, vb, kc, vc, block_table, max_pages,
                                  n_pages, ctx_len, new_off, B, nq, window, o);
    default: return DFLASH2_ERR_SHAPE;
  }
}

}  // namespace df2
