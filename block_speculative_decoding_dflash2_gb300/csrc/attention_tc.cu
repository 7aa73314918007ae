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
//   O^T += V^T P^T  M = 128 dims, N = 2 x the query rows, K = 128 keys
//
// K and Q are K-major operands; V^T is read MN-major straight from the V
// tile (each key a 128-byte row of 64 dims), and P^T MN-major as the softmax
// threads write it (each key a 128-byte row of 64 columns, so a thread
// stores its key's probabilities as 16-byte vectors).  P is split into bf16
// hi + lo parts (hi the top 16 bits of p, lo the remainder rounded), side by
// side along N (one MMA per 16 keys reads V once), so the probabilities keep
// ~15 bits; the two halves of O^T are added at the end.  Roles by warp:
//   warp 0      K and V tiles of 128 keys, each into a two-stage ring of its
//               own (K reloads once its S^T is done, V once its PV is): whole 16-key
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
  // P^T of a tile: the hi parts as columns 0 .. NP-1 and the lo parts as
  // NP .. 2NP-1 of one N = 2NP operand, in 64-column blocks
  static constexpr int NB = (2 * NP + 63) / 64;
  static constexpr int P = Q + 2 * NP * 128;           // [PB][NB][TK keys][128 B]
  // two P buffers (the softmax of a tile overlaps the PV of the one before)
  // where they fit beside two K/V stages
  static constexpr int PB = P + 2 * NB * TK * 128 + 8 * 1024 <= 227 * 1024 ? 2 : 1;
  static constexpr int RED = P + PB * NB * TK * 128;   // float [4 lane quarters][NP]
  static constexpr int MS = RED + 4 * NP * 4;          // float [NP] reference maxima of the rows
  static constexpr int CW = MS + NP * 4;               // float [rows of this CTA][TNS] merge weights
  static constexpr int PG = CW + (NP + TNS) * TNS * 4;  // int page ids of the chunk
  static size_t bytes(int npg) { return 1024 + PG + (size_t)npg * 4 + 8 + 18 * 8 + 16; }
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

// 2^x by the special-function unit (ex2.approx: relative error near 2^-22,
// far below the ~2^-15 the hi + lo split of P keeps; 2^-inf = 0)
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
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
  constexpr int PB = L::PB;
  // TMEM columns: O^T (hi, lo halves: 2NP) at 0, the two S^T buffers at 256
  constexpr uint32_t kOCol = 0, kSCol = 256;
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
  uint64_t* kfull = bars;        // [TST] a K tile landed (1 arrival + TMA bytes)
  uint64_t* kempty = bars + 2;   // [TST] its S^T MMAs completed (commit)
  uint64_t* vfull = bars + 4;    // [TST] a V tile landed
  uint64_t* vempty = bars + 6;   // [TST] its PV MMAs completed (commit)
  uint64_t* sfull = bars + 8;    // [2] S^T of a tile in TMEM (commit)
  uint64_t* sempty = bars + 10;  // [2] S^T read by the softmax warps (8 arrivals)
  // P buffer b = t % PB has a barrier pair of its own: with two buffers the
  // softmax may finish tile t + 1 before the MMA thread has seen tile t's
  // phase, which one shared barrier would then have passed
  uint64_t* pready = bars + 12;  // [PB] P of tile t in buffer t % PB (8 arrivals)
  uint64_t* odone = bars + 14;   // [PB] the PV MMAs reading buffer t % PB completed (commit)
  uint64_t* qready = bars + 16;  // Q rows in shared memory (8 arrivals)
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 17);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  float* comb = reinterpret_cast<float*>(sm + L::KV);  // [R][FS] after the key loop (aliases the ring)

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = gridDim.x, sp = blockIdx.x, g = blockIdx.y, s = blockIdx.z;
  const int grp = nq / nkv, R = grp * B;
  pdl_launch_next();
  if (threadIdx.x == 0) {
    for (int i = 0; i < TST; ++i) {
      mbar_init(kfull + i, 1);
      mbar_init(kempty + i, 1);
      mbar_init(vfull + i, 1);
      mbar_init(vempty + i, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(sfull + i, 1);
      mbar_init(sempty + i, TSW);
    }
    mbar_init(pready, TSW);
    mbar_init(pready + 1, TSW);
    mbar_init(odone, 1);
    mbar_init(odone + 1, 1);
    mbar_init(qready, TSW);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
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
    // K and V of a tile have stages (and barriers) of their own: K(t + 2)
    // loads as soon as S^T(t) is done, V(t + 2) once PV(t) is, so the K
    // load overlaps the softmax of the tiles in between.  Whole context
    // pages with a valid id go by TMA (one box per 64-dim half); the other
    // rows by cp.async, chunk c of a row in half c / 8 at position
    // (c % 8) ^ (row % 8) of its 128 bytes (the TMA's 128-byte swizzle).
    const bool tma_ok = page_tma && (k0 % 16) == 0;
    const uint64_t pol = policy_evict_first();
    int issued = 0;
    bool stop = false;
    for (int t = 0; t < ntiles && !stop; ++t) {
      const int st = t % TST;
      const int t0 = k0 + t * TK;
      // (worked out before the stages are free: lane i < 8 checks page i)
      const int cend = max(t0, min(min(t0 + TK, k1), P));
      const int nfull = tma_ok ? (cend - t0) / 16 : 0;
      int my_page = -1;
      if (lane < nfull) {
        const int li = (t0 + 16 * lane) / 16 - pbase;
        my_page = li < npg ? pg[li] : -1;
      }
      const uint32_t vmask = __ballot_sync(0xffffffffu, my_page >= 0 && my_page < n_pages) & 0xffu;
      const uint32_t full_mask = (1u << nfull) - 1u;
      const bool manual = vmask != full_mask || nfull * 16 < TK;
      const int box_page = __shfl_sync(0xffffffffu, my_page, (lane >> 1) & 7);
      for (int part = 0; part < 2; ++part) {  // K, then V
        uint64_t* full = (part ? vfull : kfull) + st;
        if (t >= TST) {
          const bool free_ = __all_sync(0xffffffffu, mbar_wait((part ? vempty : kempty) + st,
                                                               (uint32_t)(((t / TST) - 1) & 1), abort_flag,
                                                               kTcWaitNs));
          if (!free_) {
            if (lane == 0) fail();
            stop = true;
            break;
          }
        }
        uint8_t* dstb = sm + L::KV + st * KV_STAGE + part * (KV_STAGE / 2);
        if (manual) {
          // the pages with an invalid id, then the rows past the whole pages
          for (int idx = (vmask == full_mask ? nfull * 256 : 0) + lane; idx < TK * 16; idx += 32) {
            const int r = idx >> 4, c = idx & 15;
            if ((r >> 4) < nfull && ((vmask >> (r >> 4)) & 1)) continue;
            const int j = t0 + r;
            const bf16* src = kc;
            bool ok = false;
            if (j < k1) {
              if (j < P) {
                const int li = j / page_size - pbase;
                const int page = li < npg ? pg[li] : -1;
                if (page >= 0 && page < n_pages) {
                  src = (part ? vc : kc) + (((size_t)page * page_size + j % page_size) * nkv + g) * TD + c * 8;
                  ok = true;
                } else if (c == 0 && part == 0) {
                  flag(status, DFLASH2_DEV_BAD_PAGE);
                }
              } else {
                src = (part ? vb : kb) + (((size_t)s * B + (j - P)) * nkv + g) * TD + c * 8;
                ok = true;
              }
            }
            cp_async16(dstb + (c >> 3) * HALF + r * 128 + (((c & 7) ^ (r & 7)) << 4), src, ok);
          }
          cp_async_commit();
          cp_async_wait<0>();
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive_expect_tx(full, (uint32_t)__popc(vmask) * 2u * 2048u);
        __syncwarp();
        // lane 2i + hh: page i, half hh
        if (lane < 2 * nfull && ((vmask >> (lane >> 1)) & 1)) {
          const int i = lane >> 1, hh = lane & 1;
          tma_load_2d(dstb + hh * HALF + i * 16 * 128, part ? &tmV : &tmK, full, g * TD + hh * 64, box_page * 16,
                      pol);
        }
      }
      if (!stop) ++issued;
    }
    // copies still in flight (after an abort) land before the CTA moves on
    for (int t = max(0, issued - TST); t < issued; ++t) {
      volatile int never = 0;
      mbar_wait(kfull + t % TST, (uint32_t)((t / TST) & 1), &never, kTcWaitNs);
      mbar_wait(vfull + t % TST, (uint32_t)((t / TST) & 1), &never, kTcWaitNs);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------------- MMA issue
    // One thread issues every MMA.  It polls for whichever of the next PV
    // (P of tile t formed) or the next S^T (tile landed, its S buffer read)
    // can go, PV first, so a PV never waits behind a load.
    if (lane == 0 && ntiles > 0) {
      const uint32_t id_s = idesc_bf16_f32(TK, NP);
      // A = V^T and B = P^T both read MN-major; N = hi and lo columns
      const uint32_t id_o = idesc_bf16_f32(TD, 2 * NP) | (1u << 15) | (1u << 16);
      // operand descriptors of the stage / buffer bases; a k step adds its
      // offset in 16-byte units to the start-address field (no carry: shared
      // addresses stay below 2^18 bytes)
      const uint32_t kv0 = smem_u32(sm + L::KV), p_base = smem_u32(sm + L::P);
      const uint64_t q_desc = sdesc_sw128(smem_u32(sm + L::Q));
      // (stage / buffer 1 is stage / buffer 0 plus a fixed offset)
      const uint64_t k_desc = sdesc_sw128(kv0), v_desc = sdesc_mn_sw128(kv0 + KV_STAGE / 2, HALF, 1024);
      const uint64_t p_desc = sdesc_mn_sw128(p_base, HALF, 1024);
      constexpr uint64_t kStageStep = KV_STAGE >> 4, kBufStep = (L::NB * HALF) >> 4;
      bool ok = mbar_wait(qready, 0, abort_flag, kTcWaitNs);
      tc_fence_after();
      int ns_ = 0, npv = 0;
      uint64_t t_last = globaltimer();
      while (ok && npv < ntiles) {
        bool did = false;
        if (npv < ns_ && mbar_test_wait(smem_u32(pready + npv % PB), (uint32_t)((npv / PB) & 1)) &&
            mbar_test_wait(smem_u32(vfull + npv % TST), (uint32_t)((npv / TST) & 1))) {
          tc_fence_after();
          const int st = npv % TST, pb = npv % PB;
          const uint64_t vd = v_desc + (uint64_t)st * kStageStep;
          const uint64_t pd = p_desc + (uint64_t)pb * kBufStep;
#pragma unroll
          for (int j = 0; j < TK / 16; ++j)  // 16 keys = two 1024-byte atoms
            umma_bf16(tmem + kOCol, vd + (uint64_t)(j * 128), pd + (uint64_t)(j * 128), id_o,
                      (npv > 0 || j > 0) ? 1u : 0u);
          umma_commit(odone + npv % PB);
          umma_commit(vempty + st);
          ++npv;
          did = true;
        } else if (ns_ < ntiles && ns_ < npv + 2 &&
                   mbar_test_wait(smem_u32(kfull + ns_ % TST), (uint32_t)((ns_ / TST) & 1)) &&
                   (ns_ < 2 || mbar_test_wait(smem_u32(sempty + (ns_ & 1)), (uint32_t)(((ns_ >> 1) - 1) & 1)))) {
          tc_fence_after();
          const uint32_t sd = tmem + (uint32_t)(kSCol + (ns_ & 1) * NP);
          const uint64_t kd = k_desc + (uint64_t)(ns_ % TST) * kStageStep;
#pragma unroll
          for (int kk = 0; kk < TD / 16; ++kk)  // 16 dims: 32 bytes within the half's 128-byte rows
            umma_bf16(sd, kd + (uint64_t)((kk >> 2) * (HALF >> 4) + (kk & 3) * 2),
                      q_desc + (uint64_t)((kk >> 2) * (NP * 8) + (kk & 3) * 2), id_s, kk > 0 ? 1u : 0u);
          umma_commit(sfull + (ns_ & 1));
          umma_commit(kempty + ns_ % TST);
          ++ns_;
          did = true;
        }
        if (did) {
          t_last = globaltimer();
        } else {
          // back off: this warp shares its scheduler with two softmax warps
          __nanosleep(40);
          if (*abort_flag || globaltimer() - t_last > kTcWaitNs) ok = false;
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
    // this thread's row of P^T: key kl, query rows n0 .. n0 + HC - 1 in
    // 16-byte chunks of 8 rows (chunk c of a 64-row block at position
    // c ^ (kl % 8) of the key's 128-byte row)
    uint8_t* p_row = sm + L::P + kl * 128;
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
          tmem_ld8_nowait(lane_base + (uint32_t)(kSCol + (t & 1) * NP + n0 + c8 * 8),
                          *reinterpret_cast<uint32_t(*)[8]>(&r[c8 * 8]));
        tmem_ld_wait();
#pragma unroll
        for (int i = 0; i < HC; ++i) x[i] = __uint_as_float(r[i]);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(sempty + (t & 1));
      // rescale test: a score passes its row's reference maximum by more
      // than the headroom (valid keys only; the key is this thread's)
      bool need = false;
      if (valid) {
#pragma unroll
        for (int i = 0; i < HC; i += 4) {
          const float4 m4 = *reinterpret_cast<const float4*>(msh + n0 + i);
          need |= fmaf(x[i], scale, -m4.x) > kRescaleAt;
          need |= fmaf(x[i + 1], scale, -m4.y) > kRescaleAt;
          need |= fmaf(x[i + 2], scale, -m4.z) > kRescaleAt;
          need |= fmaf(x[i + 3], scale, -m4.w) > kRescaleAt;
        }
      }
      bool have_o = false;  // waited for the previous tile's PV
      if (sm_bar_or(need)) {
        // new reference maxima: the tile's column maxima over its 128 keys
#pragma unroll
        for (int i = 0; i < HC; ++i) {
          const float v = warp_max(valid ? x[i] * scale : -INFINITY);
          if (lane == 0) red[qd * NP + n0 + i] = v;
        }
        sm_bar_sync();
        if (t > 0) {  // O^T holds the earlier tiles: rescale it once their PV is done
          if (!mbar_wait(odone + (t - 1) % PB, (uint32_t)(((t - 1) / PB) & 1), abort_flag, kTcWaitNs)) {
            fail();
            ok = false;
          }
          ok = __all_sync(0xffffffffu, ok);
          tc_fence_after();
          have_o = PB == 1;
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
          if (t > 0 && ok) {  // the hi and the lo columns of these rows
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              uint32_t r8[8];
              const uint32_t ta = lane_base + (uint32_t)(kOCol + part * NP + n0 + c8 * 8);
              tmem_ld8_nowait(ta, r8);
              tmem_ld_wait();
#pragma unroll
              for (int e = 0; e < 8; ++e) r8[e] = __float_as_uint(__uint_as_float(r8[e]) * f[e]);
              tmem_st8(ta, r8);
            }
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
      // P buffer t % PB is free once the PV of tile t - PB is done
      if (t >= PB && !have_o) {
        if (!mbar_wait(odone + t % PB, (uint32_t)(((t - PB) / PB) & 1), abort_flag, kTcWaitNs)) {
          fail();
          ok = false;
        }
        tc_fence_after();
      }
      // P = 2^(x - m), split hi + lo, into P^T (key kl, rows n0 ..)
      uint8_t* pb = p_row + (t % PB) * (L::NB * HALF);
#pragma unroll
      for (int c8 = 0; c8 < HC / 8; ++c8) {
        const int nc = n0 + c8 * 8;
        uint32_t hi[4], lo[4];
        if (valid) {
          const float4 ma = *reinterpret_cast<const float4*>(msh + nc);
          const float4 mb = *reinterpret_cast<const float4*>(msh + nc + 4);
          const float mm[8] = {ma.x, ma.y, ma.z, ma.w, mb.x, mb.y, mb.z, mb.w};
#pragma unroll
          for (int e = 0; e < 8; e += 2) {
            const int i = c8 * 8 + e;
            const float p0 = ex2_approx(fmaf(x[i], scale, -mm[e]));
            const float p1 = ex2_approx(fmaf(x[i + 1], scale, -mm[e + 1]));
            l[i] += p0;
            l[i + 1] += p1;
            // hi = p truncated to bf16 (its top 16 bits), lo = the exact
            // remainder rounded to bf16: hi + lo keeps ~15 bits of p
            const uint32_t b0 = __float_as_uint(p0), b1 = __float_as_uint(p1);
            const __nv_bfloat162 l2 = __floats2bfloat162_rn(p0 - __uint_as_float(b0 & 0xffff0000u),
                                                            p1 - __uint_as_float(b1 & 0xffff0000u));
            hi[e >> 1] = __byte_perm(b0, b1, 0x7632);
            lo[e >> 1] = *reinterpret_cast<const uint32_t*>(&l2);
          }
        } else {
#pragma unroll
          for (int e = 0; e < 4; ++e) hi[e] = lo[e] = 0u;
        }
        // column nc (hi) and NP + nc (lo): block c / 64, chunk (c % 64) / 8
        const int ch = nc, cl = NP + nc;
        *reinterpret_cast<uint4*>(pb + (ch >> 6) * HALF + ((((ch & 63) >> 3) ^ (kl & 7)) << 4)) =
            make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4*>(pb + (cl >> 6) * HALF + ((((cl & 63) >> 3) ^ (kl & 7)) << 4)) =
            make_uint4(lo[0], lo[1], lo[2], lo[3]);
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(pready + t % PB);
    }
    // the last PV, then this CTA's partial rows: O^T columns, m and the
    // weight sums (over the 32 keys of a warp, then the 4 lane quarters)
    if (ntiles > 0 && ok) {
      if (!mbar_wait(odone + (ntiles - 1) % PB, (uint32_t)(((ntiles - 1) / PB) & 1), abort_flag, kTcWaitNs))
        fail();
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
      if (ntiles > 0) {  // hi + lo halves
        uint32_t rh[8], rl[8];
        tmem_ld8_nowait(lane_base + (uint32_t)(kOCol + n0 + c8 * 8), rh);
        tmem_ld8_nowait(lane_base + (uint32_t)(kOCol + NP + n0 + c8 * 8), rl);
        tmem_ld_wait();
#pragma unroll
        for (int e = 0; e < 8; ++e) ov[e] = __uint_as_float(rh[e]) + __uint_as_float(rl[e]);
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
    tmem_dealloc(tmem, 512);
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
