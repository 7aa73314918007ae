// Weight-streaming GEMM on the 5th-generation tensor cores (tcgen05) fed by
// TMA, for the dense contractions of the draft step: feature projection,
// context K/V, conv tap generators, QKV, O, gate/up, down, the selector
// factors and the lm_head ("Train a DFlash Drafter for Speculative
// Decoding", "What is DFlash?": a draft stack plus the target's shared
// lm_head).
//
// Shape of the problem: M (weight rows) is large, N (activation rows = the
// block positions of the batch) is small, K is the hidden width.  The MMA
// therefore runs swap-AB: a 128-row weight tile is operand A (MMA M = 128),
// the activation tile is operand B (MMA N = BN in 16..256), the fp32
// accumulator lives in TMEM.  At batch 1 the kernel is HBM-bound: every
// weight byte is read once per step, so the design goal is to keep enough
// TMA bytes in flight per SM (a 4..12-stage ring) on a persistent grid of
// one CTA per SM.
//
// Work schedule.  A contraction is (tiles) x (K chunks of 64).  With few
// tiles per SM, whole tiles leave SMs idle in the last wave, so every
// non-top-k contraction is split "stream-K" style: the tiles' chunks are laid
// end to end and CTA g streams the contiguous share [g W / G, (g+1) W / G) of
// all W = tiles x chunks, crossing tile boundaries.  A tile covered by one
// CTA is written directly; a tile shared by several CTAs is written by its
// pieces as fp32 partials, and the last piece to arrive (arrival counter,
// indexed by the tile's first CTA) sums them in CTA order, so the result is
// deterministic and no CTA waits for another.  The top-k contraction (the
// lm_head) needs whole tiles: its CTAs take whole tiles round-robin.
// Contractions whose tiles fill the SMs a few times over in K slices run as
// cluster split-K instead: one thread-block cluster per tile, CTA r of the
// cluster takes K slice r, and the cluster's first CTA sums the slices'
// partial tiles in rank order through distributed shared memory and runs the
// epilogue (no partial leaves the SMs, no arrival counter).
//
// Epilogues: the plain fp32 output (stored or added to), the streaming top-k
// of the lm_head, and two fused ones that remove a kernel each:
//   SWIGLU  the gate/up contraction: a 128-row tile holds 64 gate rows and
//           the 64 matching up rows (two 64-row TMA boxes), and the epilogue
//           writes SiLU(gate) * up in bf16;
//   HEADS   the q/k/v contractions: a tile holds one 128-wide head (or two
//           64-wide), and the epilogue applies the per-head RMSNorm and
//           RoPE of q and k and stores bf16 q, k, v: to the block's q/k/v
//           buffers, or, for appended context rows, into the paged cache.
//
// Warp roles (192 threads; 320 for the top-k of tiles wider than 16; 64
// more with fp8 weights):
//   warp 0      TMA producer (one lane): weight + activation tiles -> ring
//   warp 1      MMA issuer (one lane) and TMEM owner
//   warps 2..5  epilogue: TMEM -> registers -> the output tile, a partial
//               piece (coalesced over m), or the streaming top-k (wide top-k
//               tiles: warps 2..9, two sets of four on alternate chunks).
//   next 2      fp8 weights only: converters.  The weight tile arrives as
//               e4m3 bytes in a staging slot (half the bytes of bf16); the
//               converters rewrite it as bf16 in the MMA operand layout
//               (exact: every e4m3 value is a bf16 value), and the epilogue
//               multiplies each output row by its weight row's fp32 scale.
// The accumulator is double-buffered in TMEM so the epilogue of one unit
// overlaps the MMAs of the next.
//
// Every wait is bounded (1 s); on timeout the kernel records
// DFLASH2_DEV_WAIT_TIMEOUT, lets the other roles bail out, waits (bounded)
// for its own TMA copies and MMAs in flight, frees TMEM and returns.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <climits>
#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace df2 {

namespace {

constexpr int BM = 128;     // MMA M: weight rows per tile
constexpr int BK = 64;      // K elements per ring stage (128 bytes of bf16)
constexpr int SMEM_BUDGET = 227 * 1024;
constexpr uint64_t WAIT_NS = 1000000000ull;
enum { EPI_PLAIN = 0, EPI_TOPK = 1, EPI_SWIGLU = 2, EPI_HEADS = 3 };
// Epilogue warps: 4 (one per TMEM lane quarter), or 8 (two sets of 4, each
// taking every other 16-column chunk) for the top-k epilogue of wide tiles.
__host__ __device__ constexpr int epi_warps(int epi, int bn) { return (epi == EPI_TOPK && bn > 16) ? 8 : 4; }
// fp8 weights: threads of the converter warps, four warps, or two for the
// q/k-norm + RoPE epilogue (its registers: the block stays at 256 threads,
// so every role may use up to 255 registers)
__host__ __device__ constexpr int conv_threads(int epi) { return epi == EPI_HEADS ? 64 : 128; }
// producer + MMA warps, the epilogue warps, and (fp8 weights) the converters
__host__ __device__ constexpr int threads_of(int epi, int bn, bool fp8) {
  return 64 + 32 * epi_warps(epi, bn) + (fp8 ? conv_threads(epi) : 0);
}
constexpr int TOPK_SLOTS = kTopkSlots;  // shared bound slots per lm_head row (see the top-k epilogue)

struct TcArgs {
  int M, N, K;
  int n_chunks, m_tiles, n_tiles, tiles;
  long work;        // tiles * n_chunks
  int stream;       // 1: stream-K shares of the work; 0: whole tiles round-robin
  int csplit;       // > 1: cluster split-K, csplit CTAs (one cluster) per tile
  float* out;       // final [N][M] fp32 (stored, or added to when accumulate)
  float* partial;   // stream: [gridDim.x][2][BN][BM] pieces of shared tiles
  int* counters;    // stream: [gridDim.x] arrival counters, zero between launches
  int accumulate;
  float* lists_v;
  int* lists_i;
  unsigned long long* thr;  // [N][TOPK_SLOTS] shared bound slots of the top-k (0 at launch)
  float* debug;
  float mult, cap;
  unsigned* status;
  const float* wscale;  // fp8 weights: [M] per-row dequantisation scales (null: bf16 weights)
  // SWIGLU
  bf16* act;  // [N][I], I = M / 2
  int I;
  // HEADS: M rows = n_qh q heads, n_kh k heads, n_kh v heads of width hd
  int hd, n_qh, n_kh;
  const bf16* qn;  // [hd] q-norm gain (n_qh > 0)
  const bf16* kn;  // [hd] k-norm gain
  float eps;
  // Columns n < nblk are block rows (outputs q/kb/vb [n][heads][hd]); columns
  // n >= nblk are appended context rows (k and v to the paged cache; their q
  // heads are not needed and not stored).
  int nblk;
  const float2* rope;      // [nblk][hd/2] (cos, sin) at each block column's position
  const float2* rope_app;  // [N - nblk][hd/2] the same for appended columns
  const long long* dst;    // [N - nblk] element offset of an appended row in the paged cache, -1: skip
  bf16 *q, *kb, *vb;  // block rows: [nblk][heads][hd]
  bf16 *kc, *vc;      // appended rows: paged cache [pages][page_size][n_kh][hd]
};

template <int BN, bool FP8 = false>
struct TcCfg {
  static constexpr int A_BYTES = BM * BK * 2;
  static constexpr int A8_BYTES = FP8 ? BM * BK : 0;  // e4m3 staging of a weight tile
  static constexpr int B_BYTES = BN * BK * 2;
  static constexpr int STAGE = A_BYTES + A8_BYTES + B_BYTES;
  // top-k: 16-column staging (narrow tiles) or the candidate queues of each
  // warp set (wide tiles), the lists, the per-column thresholds, queue counts
  static constexpr int TOPK_SETS = epi_warps(EPI_TOPK, BN) / 4;
  static constexpr int TOPK_EXTRA = (BN > 16 ? TOPK_SETS * 16 * BM * 8 : 16 * BM * 4) + BN * KMAX * 8 + BN * 8 +
                                    TOPK_SETS * 16 * 4 + TOPK_SETS * 4 * 16 * 4;
  static constexpr int FUSE_EXTRA = 16 * BM * 4 + 4 * 16 * 4;  // exchange tile, column sums
  static constexpr int FIXED = 1024 /* alignment slack */ + 1024 /* barriers */;
  __host__ __device__ static constexpr int extra(int epi) {
    return epi == EPI_TOPK ? TOPK_EXTRA : (epi >= EPI_SWIGLU ? FUSE_EXTRA : 0);
  }
  __host__ __device__ static constexpr int stages(int epi) {
    return ((SMEM_BUDGET - FIXED - extra(epi)) / STAGE) > 12 ? 12 : ((SMEM_BUDGET - FIXED - extra(epi)) / STAGE);
  }
  __host__ __device__ static constexpr int smem_bytes(int epi) { return FIXED + stages(epi) * STAGE + extra(epi); }
  static constexpr uint32_t TMEM_COLS = (2 * BN <= 32)    ? 32
                                        : (2 * BN <= 64)  ? 64
                                        : (2 * BN <= 128) ? 128
                                        : (2 * BN <= 256) ? 256
                                                          : 512;
};

// The units of this CTA in order: (tile, first chunk, end chunk).
struct UnitIter {
  long c, cend;  // stream: chunk cursor and end; tiles: tile cursor and count
  int nc, step, stream;
  __device__ __forceinline__ bool next(int& t, int& k0, int& k1) {
    if (c >= cend) return false;
    if (stream) {
      t = (int)(c / nc);
      k0 = (int)(c - (long)t * nc);
      k1 = (int)min((long)nc, (long)k0 + (cend - c));
      c += k1 - k0;
    } else {
      t = (int)c;
      k0 = 0;
      k1 = nc;
      c += step;
    }
    return true;
  }
};

__device__ __forceinline__ long share_start(long work, int G, int g) { return (long)g * work / G; }

__device__ __forceinline__ UnitIter unit_iter(const TcArgs& a) {
  UnitIter it;
  it.nc = a.n_chunks;
  it.stream = a.stream;
  if (a.csplit > 1) {  // one unit: K slice blockIdx.x % csplit of tile blockIdx.x / csplit
    const long t = blockIdx.x / a.csplit, ks = blockIdx.x % a.csplit;
    it.stream = 1;
    it.c = t * a.n_chunks + ks * a.n_chunks / a.csplit;
    it.cend = t * a.n_chunks + (ks + 1) * a.n_chunks / a.csplit;
    it.step = 0;
  } else if (a.stream) {
    it.c = share_start(a.work, gridDim.x, blockIdx.x);
    it.cend = share_start(a.work, gridDim.x, blockIdx.x + 1);
    it.step = 0;
  } else {
    it.c = blockIdx.x;
    it.cend = a.tiles;
    it.step = gridDim.x;
  }
  return it;
}

// CTA whose share holds chunk c: the largest g with share_start(g) <= c.
__device__ __forceinline__ int share_of(long c, long work, int G) { return (int)(((c + 1) * G - 1) / work); }

// Named barrier 1 over the NT epilogue threads; barriers 2, 3 over one set of
// 4 epilogue warps (the top-k epilogue of wide tiles).
template <int NT = 128>
__device__ __forceinline__ void named_sync_epi() { asm volatile("bar.sync 1, %0;" ::"n"(NT) : "memory"); }
__device__ __forceinline__ void named_sync_set(int set) { asm volatile("bar.sync %0, 128;" ::"r"(2 + set) : "memory"); }

// Named barrier over the 4 epilogue warps that also ORs a predicate, so the
// warps take the same branch after it (no warp left waiting on a barrier
// the others skipped).
template <int NT = 128>
__device__ __forceinline__ bool named_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 q, %1, 0;\n\t"
      "bar.red.or.pred p, 1, %2, q;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(NT)
      : "memory");
  return r != 0;
}

template <int BN, int EPI, bool FP8>
__global__ void __launch_bounds__(threads_of(EPI, BN, FP8), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB, TcArgs a) {
  using C = TcCfg<BN, FP8>;
  constexpr bool TOPK = EPI == EPI_TOPK;
  constexpr int EW = epi_warps(EPI, BN);  // epilogue warps
  constexpr int EPT = 32 * EW;            // epilogue threads
  constexpr int SETS = EW / 4;
  constexpr int CONV_THREADS = conv_threads(EPI);
  constexpr int STAGES = C::stages(EPI);
  constexpr int A_BYTES = C::A_BYTES, B_BYTES = C::B_BYTES, A8_BYTES = C::A8_BYTES;
  static_assert(STAGES >= 2, "ring too small");
  static_assert(B_BYTES % 1024 == 0, "B tile must keep 1024-byte swizzle atoms aligned");

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stA = smem;
  uint8_t* stB = smem + STAGES * A_BYTES;
  uint8_t* stA8 = stB + STAGES * B_BYTES;  // fp8: [STAGES][BM][BK] e4m3 staging (rows of 64 bytes)
  uint64_t* bars = reinterpret_cast<uint64_t*>(stA8 + STAGES * A8_BYTES);
  uint64_t* full = bars;
  uint64_t* empty = bars + STAGES;
  uint64_t* tfull = bars + 2 * STAGES;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* last_flag = abort_flag + 1;
  // fp8: the TMA barriers of the staging slots (full then means "converted")
  uint64_t* full8 = drain + 4;
  uint64_t* tma_full = FP8 ? full8 : full;
  float* stg = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 1024);  // [16][BM]
  float* ssb = stg + 16 * BM;  // fused: [4 warps][16 columns] sums
  // top-k: per-set queues [SETS][16][BM] keys (wide tiles; narrow ones stage
  // values in stg), lists [BN][KMAX], thresholds [BN], queue counts [SETS][16]
  unsigned long long* q_s = reinterpret_cast<unsigned long long*>(stg);
  unsigned long long* lk_s =
      reinterpret_cast<unsigned long long*>(reinterpret_cast<uint8_t*>(stg) + (BN > 16 ? SETS * 16 * BM * 8 : 16 * BM * 4));
  unsigned long long* thr_s = lk_s + BN * KMAX;
  int* qn_s = reinterpret_cast<int*>(thr_s + BN);
  float* tau_s = reinterpret_cast<float*>(qn_s + SETS * 16);  // [SETS][4 warps][16] first-tile bounds

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_launch_next();

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      mbar_init(full + s, FP8 ? CONV_THREADS : 1);  // fp8: every converter thread arrives
      mbar_init(empty + s, 1);
      if (FP8) mbar_init(full8 + s, 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(tfull + i, 1);
      mbar_init(tempty + i, EPT);
    }
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  auto fail = [&]() {
    *abort_flag = 1;
    flag(a.status, DFLASH2_DEV_WAIT_TIMEOUT);
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_x = policy_evict_last();
      // weight tile of chunk kc for m-tile mt (SWIGLU: 64 gate rows + the 64 matching up rows)
      // (fp8: into the staging slot; a byte per element, so the x
      // coordinate is the same element index)
      uint8_t* dstA = FP8 ? stA8 : stA;
      constexpr int AB = FP8 ? A8_BYTES : A_BYTES;
      auto load_a = [&](int st, int kc_, int mt_) {
        if constexpr (EPI == EPI_SWIGLU) {
          tma_load_2d(dstA + st * AB, &tmA, tma_full + st, kc_ * BK, mt_ * (BM / 2), pol_w);
          tma_load_2d(dstA + st * AB + AB / 2, &tmA, tma_full + st, kc_ * BK, a.I + mt_ * (BM / 2), pol_w);
        } else {
          tma_load_2d(dstA + st * AB, &tmA, tma_full + st, kc_ * BK, mt_ * BM, pol_w);
        }
      };
      UnitIter it = unit_iter(a);
      int t = 0, kc = 0, k1 = 0;
      bool have = it.next(t, kc, k1);
      // 1. weight tiles of the first ring's worth of chunks, before waiting for
      //    the previous kernel (no kernel on the stream writes the weights)
      int pre = 0;
      {
        UnitIter pit = it;
        int tt = t, kk = kc, kk1 = k1;
        bool h = have;
        while (pre < STAGES && h) {
          mbar_arrive_expect_tx(tma_full + pre, AB + B_BYTES);
          load_a(pre, kk, tt % a.m_tiles);
          ++pre;
          if (++kk == kk1) h = pit.next(tt, kk, kk1);
        }
      }
      pdl_wait();
      // 2. the activation tiles of those chunks
      long issued = 0;
      for (int i = 0; i < pre; ++i) {
        tma_load_2d(stB + i * B_BYTES, &tmB, tma_full + i, kc * BK, (t / a.m_tiles) * BN, pol_x);
        ++issued;
        if (++kc == k1) have = it.next(t, kc, k1);
      }
      int stage = pre % STAGES;
      uint32_t phase = pre == STAGES ? 1u : 0u;
      // 3. steady state
      while (have && !*abort_flag) {
        bool ok = true;
        const int mt = t % a.m_tiles, nt = t / a.m_tiles;
        for (; kc < k1; ++kc) {
          if (!mbar_wait(empty + stage, phase ^ 1u, abort_flag, WAIT_NS)) {
            fail();
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(tma_full + stage, AB + B_BYTES);
          load_a(stage, kc, mt);
          tma_load_2d(stB + stage * B_BYTES, &tmB, tma_full + stage, kc * BK, nt * BN, pol_x);
          ++issued;
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        have = it.next(t, kc, k1);
      }
      if (*abort_flag) {
        // wait (bounded) for every copy this thread issued to land
        for (int s = 0; s < STAGES; ++s) {
          const long cnt = issued / STAGES + (s < issued % STAGES ? 1 : 0);
          if (cnt > 0) {
            volatile int never = 0;
            mbar_wait(tma_full + s, (uint32_t)((cnt - 1) & 1), &never, WAIT_NS);
          }
        }
      }
    }
    __syncwarp();  // lanes 1..31 wait here for the producer lane: the warp reaches the final barrier whole
    if (a.csplit > 1) {  // the two cluster barriers of the slice reduction (see the epilogue)
      cluster_sync();
      cluster_sync();
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      UnitIter it = unit_iter(a);
      int t, k0, k1;
      while (ok && it.next(t, k0, k1)) {
        if (!mbar_wait(tempty + acc, acc_phase ^ 1u, abort_flag, WAIT_NS)) {
          fail();
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem + (uint32_t)(acc * BN);
        for (int kc = k0; kc < k1; ++kc) {
          if (!mbar_wait(full + stage, phase, abort_flag, WAIT_NS) ||
              (FP8 && !mbar_wait(full8 + stage, phase, abort_flag, WAIT_NS))) {
            fail();
            ok = false;
            break;
          }
          tc_fence_after();
          const uint64_t ad = sdesc_sw128(smem_u32(stA + stage * A_BYTES));
          const uint64_t bd = sdesc_sw128(smem_u32(stB + stage * B_BYTES));
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d, ad + 2u * kk, bd + 2u * kk, idesc, (kc > k0 || kk > 0) ? 1u : 0u);
          umma_commit(empty + stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(tfull + acc);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // every MMA issued by this thread completes before TMEM can be freed
      umma_commit(drain);
      volatile int never = 0;
      mbar_wait(drain, 0, &never, WAIT_NS);
    }
    __syncwarp();  // as for the producer warp
    if (a.csplit > 1) {
      cluster_sync();
      cluster_sync();
    }
  } else if (FP8 && warp >= 2 + EW) {
    // ------------------------------------------------------------ fp8 converters
    // Slot s holds rows of 64 e4m3 bytes; thread ct rewrites 16-byte pieces
    // (16 elements of row r) as two 16-byte bf16 chunks of the 128-byte
    // swizzled operand row (chunk c of row r lives at chunk c ^ (r & 7)).
    const int ct = threadIdx.x - (64 + EPT);
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    UnitIter it = unit_iter(a);
    int t, k0, k1;
    while (ok && it.next(t, k0, k1)) {
      for (int kc = k0; kc < k1; ++kc) {
        if (!mbar_wait(full8 + stage, phase, abort_flag, WAIT_NS)) {
          fail();
          ok = false;
          break;
        }
        const uint8_t* src = stA8 + stage * A8_BYTES;
        uint8_t* dst = stA + stage * A_BYTES;
#pragma unroll
        for (int i = 0; i < A8_BYTES / 16 / CONV_THREADS; ++i) {
          const int piece = ct + i * CONV_THREADS;
          const int r = piece >> 2, c0 = (piece & 3) * 2;
          const uint4 q = *reinterpret_cast<const uint4*>(src + piece * 16);
          const uint32_t w[4] = {q.x, q.y, q.z, q.w};
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 lo = e4m3x2_to_bf16x2((uint16_t)(w[e] & 0xffffu));
            const __nv_bfloat162 hi = e4m3x2_to_bf16x2((uint16_t)(w[e] >> 16));
            o[2 * e] = *reinterpret_cast<const uint32_t*>(&lo);
            o[2 * e + 1] = *reinterpret_cast<const uint32_t*>(&hi);
          }
          uint8_t* row = dst + r * 128;
          *reinterpret_cast<uint4*>(row + ((c0 ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(row + (((c0 + 1) ^ (r & 7)) << 4)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();  // the operand is read by tcgen05.mma (async proxy)
        mbar_arrive(full + stage);
        if (++stage == STAGES) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    if (a.csplit > 1) {
      cluster_sync();
      cluster_sync();
    }
  } else {
    // ------------------------------------------------------------ epilogue
    pdl_wait();  // outputs, partials and counters may still be in use by the previous kernel
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int row = q * 32 + lane;
    const int ew = warp - 2;
    int acc = 0;
    uint32_t acc_phase = 0;
    int cur_nt = -1;
    uint32_t touched = 0;

    auto reset_lists = [&]() {
      for (int i = threadIdx.x - 64; i < BN * KMAX; i += EPT) lk_s[i] = 0ull;
      for (int i = threadIdx.x - 64; i < BN; i += EPT) thr_s[i] = 0ull;
      for (int i = threadIdx.x - 64; i < SETS * 16; i += EPT) qn_s[i] = 0;
    };
    auto flush_lists = [&](int nt, bool sentinel) {
      for (int i = threadIdx.x - 64; i < BN * KMAX; i += EPT) {
        const int c = i / KMAX, e = i % KMAX;
        const int n = nt * BN + c;
        if (n < a.N) {
          const size_t o = ((size_t)blockIdx.x * a.N + n) * KMAX + e;
          const unsigned long long key = sentinel ? 0ull : lk_s[i];
          a.lists_v[o] = key ? key_value(key) : -INFINITY;  // empty slots: the (-inf, INT_MAX) sentinel
          a.lists_i[o] = key ? key_id(key) : INT_MAX;
        }
      }
    };

    bool cl_done = false;  // cluster split-K: this CTA took part in both cluster barriers
    UnitIter it = unit_iter(a);
    int t, k0, k1;
    while (it.next(t, k0, k1)) {
      const int mt = t % a.m_tiles, nt = t / a.m_tiles;
      const bool got = mbar_wait(tfull + acc, acc_phase, abort_flag, WAIT_NS);
      if (!got) fail();
      if (named_sync_or<EPT>(!got || *abort_flag)) break;
      tc_fence_after();
      const int m = mt * BM + row;
      const uint32_t tbase = tmem + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * BN);
      // fp8 weights: the dequantisation scale of this thread's weight row
      // (SWIGLU: row < 64 is gate row mt*64 + row, else up row I + mt*64 + row - 64)
      float wsc = 1.f;
      if constexpr (FP8) {
        const int wr = EPI == EPI_SWIGLU ? (row < BM / 2 ? mt * (BM / 2) + row : a.I + mt * (BM / 2) + row - BM / 2) : m;
        wsc = (EPI == EPI_SWIGLU || m < a.M) ? a.wscale[wr] : 0.f;
      }
      if constexpr (!TOPK) {
        // pieces of tile t: CTAs g_first .. g_last share its chunks
        int g_first = blockIdx.x, g_last = blockIdx.x;
        if (a.stream) {
          const long c0t = (long)t * a.n_chunks;
          g_first = share_of(c0t, a.work, gridDim.x);
          g_last = share_of(c0t + a.n_chunks - 1, a.work, gridDim.x);
        }
        const bool direct = g_first == g_last;
        // a CTA's piece of a shared tile is its first unit (slot 0) when its
        // share starts inside the tile, else its last unit (slot 1)
        auto piece = [&](int g) {
          const int slot = share_start(a.work, gridDim.x, g) / a.n_chunks == t ? 0 : 1;
          return a.partial + ((size_t)g * 2 + slot) * BN * BM;
        };
        float* pc = direct ? nullptr : piece(blockIdx.x);
        // final values of columns nt*BN + c0 .. +15 of this thread's row m.
        // All loads of a step are issued before its stores, so they overlap
        // instead of queueing.  The fused epilogues synchronise the four
        // epilogue warps; every call site is uniform across them.
        // (pre_old: the old output values when the caller already loaded them)
        auto finish = [&](float(&v)[16], int c0, const float* pre_old) {
          const int nb = nt * BN + c0;       // first column
          const int nj = min(16, a.N - nb);  // valid columns (may be <= 0)
          if constexpr (FP8) {
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] *= wsc;
          }
          if constexpr (EPI == EPI_PLAIN) {
            if (m < a.M && nj > 0) {
              float* p0 = a.out + (size_t)nb * a.M + m;
              if (a.accumulate) {
                float old[16];
#pragma unroll
                for (int j = 0; j < 16; ++j) old[j] = pre_old ? pre_old[j] : (j < nj ? p0[(size_t)j * a.M] : 0.f);
#pragma unroll
                for (int j = 0; j < 16; ++j) v[j] = old[j] + v[j];
              }
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j < nj) p0[(size_t)j * a.M] = v[j];
            }
          } else if constexpr (EPI == EPI_SWIGLU) {
            // rows 0..63: gate of index i = mt*64 + row; rows 64..127: up of the same i
            constexpr int HB = BM / 2;
            const int hr = row & (HB - 1);
            if (row >= HB) {
#pragma unroll
              for (int j = 0; j < 16; ++j) stg[j * HB + hr] = v[j];
            }
            named_sync_epi();
            if (row < HB) {
              const int i = mt * HB + hr;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j < nj) {
                  const float gt = v[j], up = stg[j * HB + hr];
                  a.act[(size_t)(nb + j) * a.I + i] = __float2bfloat16_rn(gt / (1.f + expf(-gt)) * up);
                }
            }
            named_sync_epi();
          } else if constexpr (EPI == EPI_HEADS) {
            const int tid = threadIdx.x - 64, wq = tid >> 5;
            const int d = a.hd, half = d / 2;
            const int hg = m / d, di = m - hg * d, ip = di % half;
            const bool valid = m < a.M;
            const int kind = hg < a.n_qh ? 0 : (hg < a.n_qh + a.n_kh ? 1 : 2);  // q, k, v
            const bool rot = kind < 2 && valid;
            // every global value this epilogue reads, issued together up front:
            // the norm weight, the RoPE angles of the 16 columns and, for
            // appended rows, their cache offsets (issued after a global store
            // they would each wait for it, the store may alias them)
            const float gdi = rot ? ld((kind == 0 ? a.qn : a.kn) + di) : 1.f;
            float2 cs[16];
            long long dj[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = max(0, min(nb + j, a.N - 1));  // columns past N: clamped, unused
              const bool blk = n < a.nblk;
              const float2* src =
                  blk ? a.rope + (size_t)n * half + ip : a.rope_app + (size_t)(n - a.nblk) * half + ip;
              cs[j] = rot ? __ldcg(src) : make_float2(1.f, 0.f);
              dj[j] = (valid && kind > 0 && !blk) ? __ldcg(a.dst + (n - a.nblk)) : -1;
            }
            // per-column sums of squares over this warp's 32 rows, by a
            // transposing butterfly: each exchange halves the columns a lane
            // keeps (16 shuffles instead of 16 x 5); lane L ends with column
            // (L >> 1)'s sum
            {
              float t8[8], t4[4], t2[2];
              const bool b4 = lane & 16, b3 = lane & 8, b2 = lane & 4, b1 = lane & 2;
#pragma unroll
              for (int i = 0; i < 8; ++i) {
                const float lo = valid ? v[i] * v[i] : 0.f, hi = valid ? v[8 + i] * v[8 + i] : 0.f;
                t8[i] = (b4 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b4 ? lo : hi, 16);
              }
#pragma unroll
              for (int i = 0; i < 4; ++i)
                t4[i] = (b3 ? t8[4 + i] : t8[i]) + __shfl_xor_sync(0xffffffffu, b3 ? t8[i] : t8[4 + i], 8);
#pragma unroll
              for (int i = 0; i < 2; ++i)
                t2[i] = (b2 ? t4[2 + i] : t4[i]) + __shfl_xor_sync(0xffffffffu, b2 ? t4[i] : t4[2 + i], 4);
              float t1 = (b1 ? t2[1] : t2[0]) + __shfl_xor_sync(0xffffffffu, b1 ? t2[0] : t2[1], 2);
              t1 += __shfl_xor_sync(0xffffffffu, t1, 1);
              if (!(lane & 1)) ssb[wq * 16 + (lane >> 1)] = t1;
            }
            named_sync_epi();
            // RMSNorm of q/k heads (a head spans all 128 rows, or a 64-row half)
            float x[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const float ss = d == BM ? (ssb[j] + ssb[16 + j]) + (ssb[32 + j] + ssb[48 + j])
                                       : (wq < 2 ? ssb[j] + ssb[16 + j] : ssb[32 + j] + ssb[48 + j]);
              x[j] = kind < 2 ? v[j] * (rsqrtf(ss / (float)d + a.eps) * gdi) : v[j];
              stg[j * BM + row] = x[j];
            }
            named_sync_epi();
            // RoPE: rotate-half pairs (di, di + d/2)
            if (rot) {
              const float sgn = di < half ? -1.f : 1.f;
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j < nj) x[j] = x[j] * cs[j].x + sgn * (stg[j * BM + (row ^ half)] * cs[j].y);
            }
            if (valid) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                if (j >= nj) continue;
                const bf16 val = __float2bfloat16_rn(x[j]);
                const size_t n = (size_t)(nb + j);
                if ((int)n < a.nblk) {
                  if (kind == 0) a.q[(n * a.n_qh + hg) * d + di] = val;
                  else if (kind == 1) a.kb[(n * a.n_kh + (hg - a.n_qh)) * d + di] = val;
                  else a.vb[(n * a.n_kh + (hg - a.n_qh - a.n_kh)) * d + di] = val;
                } else if (kind > 0 && dj[j] >= 0) {
                  if (kind == 1) a.kc[dj[j] + (size_t)(hg - a.n_qh) * d + di] = val;
                  else a.vc[dj[j] + (size_t)(hg - a.n_qh - a.n_kh) * d + di] = val;
                }
              }
            }
            named_sync_epi();  // the exchange tile and column info are reused next
          }
        };
        const bool clus = a.csplit > 1;
        // cluster split-K: this slice's partial tile in the idle operand ring,
        // as float4 groups [BN / 4][BM][4] (a warp's 16-byte accesses of one
        // column group are consecutive: no bank conflicts at any BN)
        float* part_s = reinterpret_cast<float*>(stA);
        static_assert(EPI == EPI_TOPK || STAGES * (A_BYTES + B_BYTES + A8_BYTES) >= BM * BN * 4,
                      "the operand ring must hold a partial tile");
#pragma unroll 1
        for (int c0 = 0; c0 < BN; c0 += 16) {
          float v[16];
          tmem_ld16(tbase + c0, v);
          if (clus) {
            // (the operand ring is idle: the MMAs of the CTA's only unit are done)
#pragma unroll
            for (int j = 0; j < 16; j += 4)
              *reinterpret_cast<float4*>(part_s + ((size_t)((c0 + j) >> 2) * BM + row) * 4) =
                  make_float4(v[j], v[j + 1], v[j + 2], v[j + 3]);
          } else if (!direct) {
#pragma unroll
            for (int j = 0; j < 16; ++j) pc[(c0 + j) * BM + row] = v[j];
          } else {
            finish(v, c0, nullptr);
          }
        }
        tc_fence_before();
        mbar_arrive(tempty + acc);
        if (clus) {
          cluster_sync();  // every slice's partial is in its CTA's shared memory
          // The cluster's CTAs share the reduction and the epilogue: CTA r sums
          // the slices of column chunks r, r + cs, ... in rank order (the same
          // order whichever CTA sums) and finishes them.
#pragma unroll 1
          for (int c0 = (int)(blockIdx.x % a.csplit) * 16; c0 < BN; c0 += 16 * a.csplit) {
            float v[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) v[j] = 0.f;
#pragma unroll 1
            constexpr int QF = FP8 ? 1 : 2;  // slices whose loads are in flight at once (registers)
            for (int q0 = 0; q0 < a.csplit; q0 += QF) {
              float4 x[QF][4];
#pragma unroll
              for (int qq = 0; qq < QF; ++qq)
                if (q0 + qq < a.csplit) {
#pragma unroll
                  for (int j = 0; j < 4; ++j)
                    x[qq][j] = ld_dsmem4(dsmem_addr(part_s + ((size_t)((c0 >> 2) + j) * BM + row) * 4,
                                                    (uint32_t)(q0 + qq)));
                }
#pragma unroll
              for (int qq = 0; qq < QF; ++qq)
                if (q0 + qq < a.csplit) {
#pragma unroll
                  for (int j = 0; j < 4; ++j) {
                    v[4 * j] += x[qq][j].x;
                    v[4 * j + 1] += x[qq][j].y;
                    v[4 * j + 2] += x[qq][j].z;
                    v[4 * j + 3] += x[qq][j].w;
                  }
                }
            }
            finish(v, c0, nullptr);
          }
          cluster_sync();  // every partial has been read
          cl_done = true;
        } else if (!direct) {
          // the piece is written; one thread publishes it (the barrier orders the
          // other threads' stores before its cumulative fence) and counts it
          named_sync_epi();
          if (threadIdx.x == 64) {
            __threadfence();
            const bool last = atomicAdd(a.counters + g_first, 1) == g_last - g_first;
            if (last) __threadfence();  // acquire: the other pieces are visible to the CTA after the barrier
            *last_flag = last ? 1 : 0;
          }
          named_sync_epi();
          if (*last_flag) {
            // sum the pieces in CTA order, 16 columns at a time
#pragma unroll 1
            for (int c0 = 0; c0 < BN && nt * BN + c0 < a.N; c0 += 16) {
              float sum[16], old[16];
#pragma unroll
              for (int j = 0; j < 16; ++j) sum[j] = 0.f;
              // the old output values load in the same round as the pieces
              const bool pre = EPI == EPI_PLAIN && a.accumulate && m < a.M;
              if (pre) {
                const int nj = min(16, a.N - (nt * BN + c0));
                const float* p0 = a.out + (size_t)(nt * BN + c0) * a.M + m;
#pragma unroll
                for (int j = 0; j < 16; ++j) old[j] = j < nj ? p0[(size_t)j * a.M] : 0.f;
              }
              constexpr int PB = FP8 ? 2 : (EPI == EPI_HEADS ? 4 : 8);  // pieces per round of loads (registers)
              for (int g0 = g_first; g0 <= g_last; g0 += PB) {
                float v[PB][16];
#pragma unroll
                for (int q2 = 0; q2 < PB; ++q2)
                  if (g0 + q2 <= g_last) {
                    const float* pg = piece(g0 + q2) + (size_t)c0 * BM + row;
#pragma unroll
                    for (int j = 0; j < 16; ++j) v[q2][j] = __ldcg(pg + j * BM);
                  }
#pragma unroll
                for (int q2 = 0; q2 < PB; ++q2)
                  if (g0 + q2 <= g_last) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) sum[j] += v[q2][j];
                  }
              }
              finish(sum, c0, pre ? old : nullptr);
            }
            if (threadIdx.x == 64) a.counters[g_first] = 0;
          }
        }
      } else {
        // ---------------------------------------------- streaming top-k
        // Each CTA keeps, per column (lm_head row) of its current column
        // tile, a sorted list of its best KMAX (vocabulary id, logit) entries
        // as 64-bit order keys in shared memory.  An entry is offered only
        // when it beats the column's threshold: the larger of the list's
        // KMAX-th key and a bound shared by all CTAs through global memory.
        // That bound is the smallest of TOPK_SLOTS slots; CTA g raises slot
        // g % TOPK_SLOTS to its list's best key, so the slots hold the keys
        // of TOPK_SLOTS distinct entries (one per slot, from distinct CTAs),
        // and an entry below their minimum has KMAX better ones: it is not in
        // the column's top KMAX.  The slots start at zero (no bound).
        const int ewq = ew & 3;                 // warp within its set
        const int set = SETS > 1 ? ew >> 2 : 0;  // which chunks its set takes
        const bool fresh = nt != cur_nt;        // the lists start empty at this tile
        if (nt != cur_nt) {
          named_sync_epi<EPT>();
          if (cur_nt >= 0) flush_lists(cur_nt, false);
          named_sync_epi<EPT>();
          reset_lists();
          cur_nt = nt;
          touched |= 1u << nt;
          named_sync_epi<EPT>();
        }
        // the shared bound slots of the 4 columns this warp merges in a chunk
        // (columns ewq + 4i, i = 0..3), lane l holding slot l % 16 of column
        // i = 2r + l / 16, loaded ahead of their use in the merge step
        auto slots_load = [&](int c0, unsigned long long (&gs)[2]) {
#pragma unroll
          for (int r2 = 0; r2 < 2; ++r2) {
            const int n = nt * BN + c0 + ewq + 4 * (2 * r2 + (lane >> 4));
            gs[r2] = n < a.N ? __ldcg(a.thr + (size_t)n * TOPK_SLOTS + (lane & 15)) : ~0ull;
          }
        };
        // the minimum of column i's slots, on every lane
        auto slots_min = [&](const unsigned long long (&gs)[2], int i) {
          unsigned long long x = (i & 2) ? gs[1] : gs[0];
#pragma unroll
          for (int o = 1; o < 16; o <<= 1) {
            const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, o);
            x = y < x ? y : x;
          }
          return __shfl_sync(0xffffffffu, x, (i & 1) * 16);
        };
        auto publish = [&](int n, unsigned long long top_before, unsigned long long lk) {
          const unsigned long long top = __shfl_sync(0xffffffffu, lk, 0);
          if (lane == 0 && top > top_before) atomicMax(a.thr + (size_t)n * TOPK_SLOTS + (blockIdx.x % TOPK_SLOTS), top);
        };
        if constexpr (BN <= 16) {
          // narrow tiles (a few rows, the batch-1 step): one chunk per tile,
          // staged in shared memory; warp ew scans columns ew, ew + 4, ...
          // over the 128 rows, 32 at a time
          unsigned long long gs[2];
          slots_load(0, gs);
          float v[16];
          tmem_ld16(tbase, v);
          tc_fence_before();
          mbar_arrive(tempty + acc);
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            float z = a.mult * (FP8 ? wsc * v[j] : v[j]);
            if (a.cap > 0.f) z = a.cap * tanhf(z / a.cap);
            v[j] = z;
          }
          if (a.debug != nullptr && m < a.M) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int n = nt * BN + j;
              if (n < a.N) a.debug[(size_t)n * a.M + m] = v[j];
            }
          }
          named_sync_epi();  // previous tile's scans are done with the staging tile
#pragma unroll
          for (int j = 0; j < 16; ++j) stg[j * BM + row] = v[j];
          named_sync_epi();
#pragma unroll 1
          for (int i = 0; i < 4; ++i) {
            const int c = ewq + 4 * i;
            const int n = nt * BN + c;
            const unsigned long long gk = slots_min(gs, i);  // every lane takes part
            if (n >= a.N) continue;
            unsigned long long* Lk = lk_s + c * KMAX;
            unsigned long long lk = lane < KMAX ? Lk[lane] : 0ull;
            unsigned long long tk = __shfl_sync(0xffffffffu, lk, KMAX - 1);
            const unsigned long long top_before = __shfl_sync(0xffffffffu, lk, 0);
#pragma unroll 1
            for (int r = 0; r < 4; ++r) {
              const int rr = r * 32 + lane;
              const int mm = mt * BM + rr;
              const unsigned long long key = mm < a.M ? order_key(stg[c * BM + rr], mm) : 0ull;
              const bool pass = key > tk && key > gk;
              unsigned mask = __ballot_sync(0xffffffffu, pass);
              if (__popc(mask) > 3) {
                warp_key_merge(lk, tk, pass ? key : 0ull);
              } else {
                while (mask) {
                  const int src = __ffs(mask) - 1;
                  mask &= mask - 1;
                  warp_key_offer(lk, tk, __shfl_sync(0xffffffffu, key, src));
                }
              }
            }
            if (lane < KMAX) Lk[lane] = lk;
            publish(n, top_before, lk);
            __syncwarp();
          }
        } else {
          // wide tiles: the two warp sets take alternate 16-column chunks.  Each
          // thread filters its own row's 16 values against the columns'
          // thresholds (kept current in shared memory) and appends the few
          // that pass to the column's queue; after the set's barrier warp ewq
          // merges the queues of columns ewq + 4i into their lists and renews
          // their thresholds.
          unsigned long long* qset = q_s + (size_t)set * 16 * BM;
          int* qn = qn_s + set * 16;
          const unsigned idk = (unsigned)(0x7fffffff - m);  // low half of this row's keys
#pragma unroll 1
          for (int c0 = set * 16; c0 < BN; c0 += 16 * SETS) {
            unsigned long long gs[2];
            slots_load(c0, gs);
            float v[16];
            tmem_ld16(tbase + c0, v);
            if (c0 + 16 * SETS >= BN) {  // this set's last chunk of the tile
              tc_fence_before();
              mbar_arrive(tempty + acc);
            }
            const int nj = min(16, a.N - (nt * BN + c0));  // valid columns of the chunk
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              float z = a.mult * (FP8 ? wsc * v[j] : v[j]);
              if (a.cap > 0.f) z = a.cap * tanhf(z / a.cap);
              v[j] = z;
            }
            if (a.debug != nullptr && m < a.M) {
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j < nj) a.debug[(size_t)(nt * BN + c0 + j) * a.M + m] = v[j];
            }
            // First tile (empty lists): a lower bound of each column's 16th
            // largest value in this tile, the smallest of its 16 group
            // maxima (8 consecutive rows each: every group maximum is a
            // distinct row at least that large).  Only values at least this
            // bound can be in the tile's top 16, so the rest are not queued.
            float tau[16];
#pragma unroll
            for (int j = 0; j < 16; ++j) tau[j] = -INFINITY;
            if (fresh) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                float x = m < a.M ? v[j] : -INFINITY;
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 1));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 2));
                x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, 4));
                x = fminf(x, __shfl_xor_sync(0xffffffffu, x, 8));
                x = fminf(x, __shfl_xor_sync(0xffffffffu, x, 16));
                if (lane == 0) tau_s[(set * 4 + ewq) * 16 + j] = x;
              }
              named_sync_set(set);
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                const float* tw = tau_s + set * 64 + j;
                tau[j] = fminf(fminf(tw[0], tw[16]), fminf(tw[32], tw[48]));
              }
            }
            if (m < a.M) {
#pragma unroll
              for (int j = 0; j < 16; ++j) {
                unsigned u = __float_as_uint(v[j] + 0.f);
                u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
                const unsigned long long key = ((unsigned long long)u << 32) | idk;
                if (j < nj && v[j] >= tau[j] && key > thr_s[c0 + j]) qset[j * BM + atomicAdd(qn + j, 1)] = key;
              }
            }
            named_sync_set(set);
#pragma unroll 1
            for (int i = 0; i < 4; ++i) {
              const int jj = ewq + 4 * i, c = c0 + jj, n = nt * BN + c;
              const unsigned long long gk = slots_min(gs, i);  // every lane takes part
              if (jj >= nj) continue;
              const int cnt = qn[jj];
              unsigned long long* Lk = lk_s + c * KMAX;
              unsigned long long lk = lane < KMAX ? Lk[lane] : 0ull;
              unsigned long long tk = __shfl_sync(0xffffffffu, lk, KMAX - 1);
              if (cnt > 0) {
                const unsigned long long top_before = __shfl_sync(0xffffffffu, lk, 0);
#pragma unroll 1
                for (int b0 = 0; b0 < cnt; b0 += 32) {
                  unsigned long long ck = b0 + lane < cnt ? qset[jj * BM + b0 + lane] : 0ull;
                  if (ck <= tk || ck <= gk) ck = 0ull;  // no longer beats the list or the shared bound
                  unsigned mask = __ballot_sync(0xffffffffu, ck != 0ull);
                  if (__popc(mask) > 3) {
                    warp_key_merge(lk, tk, ck);
                  } else {
                    while (mask) {
                      const int src = __ffs(mask) - 1;
                      mask &= mask - 1;
                      warp_key_offer(lk, tk, __shfl_sync(0xffffffffu, ck, src));
                    }
                  }
                }
                if (lane < KMAX) Lk[lane] = lk;
                publish(n, top_before, lk);
              }
              if (lane == 0) {
                thr_s[c] = tk > gk ? tk : gk;
                qn[jj] = 0;
              }
            }
            named_sync_set(set);  // queues emptied and thresholds renewed before the next chunk's filter
          }
        }
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (a.csplit > 1 && !cl_done) {  // bailed out before the slice reduction: keep the cluster's barriers
      cluster_sync();
      cluster_sync();
    }
    if constexpr (TOPK) {
      if (!named_sync_or<EPT>(*abort_flag != 0)) {
        if (cur_nt >= 0) flush_lists(cur_nt, false);
        for (int nt = 0; nt < a.n_tiles; ++nt)
          if (!(touched & (1u << nt))) flush_lists(nt, true);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, []() {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 tensor map over rows x cols (row stride ld elements), box of
// 64 columns x box_rows rows, 128-byte swizzle, zero fill out of bounds.
int make_map(CUtensorMap* map, const void* base, int rows, int cols, int ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return DFLASH2_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ((size_t)ld * 2) % 16) return DFLASH2_ERR_SHAPE;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

// 2-D e4m3 tensor map over rows x cols bytes (row stride ld bytes), box of
// 64 columns x box_rows rows, no swizzle (the converters read it row by row).
int make_map8(CUtensorMap* map, const void* base, int rows, int cols, int ld, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return DFLASH2_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || ld % 16) return DFLASH2_ERR_SHAPE;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

// Activation rows per tile.  With very few weight tiles (M <= 512) the rows
// are spread over 16-row tiles so the grid still fills the SMs; otherwise the
// smallest MMA width that holds all rows (at most 256).
int pick_bn(int M, int N) {
  if (N <= 16) return 16;
  if ((M + BM - 1) / BM <= 4 && N <= 256) return 16;
  if (N <= 32) return 32;
  if (N <= 64) return 64;
  if (N <= 128) return 128;
  return 256;
}

template <int BN, int EPI, bool FP8>
int set_smem_attr() {
  static bool attr_set = false;
  if (!attr_set) {
    if (cudaFuncSetAttribute(tc_gemm_kernel<BN, EPI, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             TcCfg<BN, FP8>::smem_bytes(EPI)) != cudaSuccess)
      return DFLASH2_ERR_CUDA;
    attr_set = true;
  }
  return DFLASH2_OK;
}

template <int BN, int EPI, bool FP8>
int launch_bn(const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& args, int grid, const Ctx& c) {
  constexpr int smem = TcCfg<BN, FP8>::smem_bytes(EPI);
  const int rc = set_smem_attr<BN, EPI, FP8>();
  if (rc) return rc;
  return launch_kx(tc_gemm_kernel<BN, EPI, FP8>, dim3(grid), dim3(threads_of(EPI, BN, FP8)), smem, c,
                   args.csplit > 1 ? args.csplit : 1, ma, mb, args);
}

// Clusters of cs CTAs of this instantiation that fit the device at once
// (0 when the query fails), cached per cluster size.
template <int BN, int EPI, bool FP8>
int max_clusters(int cs) {
  static int cache[9] = {-1, -1, -1, -1, -1, -1, -1, -1, -1};
  if (cs < 2 || cs > 8) return 0;
  if (cache[cs] >= 0) return cache[cs];
  if (set_smem_attr<BN, EPI, FP8>()) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs * 64);
  cfg.blockDim = dim3(threads_of(EPI, BN, FP8));
  cfg.dynamicSmemBytes = TcCfg<BN, FP8>::smem_bytes(EPI);
  cudaLaunchAttribute at;
  at.id = cudaLaunchAttributeClusterDimension;
  at.val.clusterDim.x = cs;
  at.val.clusterDim.y = 1;
  at.val.clusterDim.z = 1;
  cfg.attrs = &at;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, tc_gemm_kernel<BN, EPI, FP8>, &cfg) != cudaSuccess) {
    (void)cudaGetLastError();
    n = 0;
  }
  cache[cs] = n;
  return n;
}

template <int BN, bool FP8>
int max_clusters_epi(int epi, int cs) {
  switch (epi) {
    case EPI_SWIGLU:
      if constexpr (BN <= 64) return max_clusters<BN, EPI_SWIGLU, FP8>(cs);
      return 0;
    case EPI_HEADS:
      if constexpr (BN <= 64) return max_clusters<BN, EPI_HEADS, FP8>(cs);
      return 0;
    case EPI_PLAIN: return max_clusters<BN, EPI_PLAIN, FP8>(cs);
    default: return 0;
  }
}

int max_clusters_of(int bn, int epi, bool fp8, int cs) {
  switch (bn) {
    case 16: return fp8 ? max_clusters_epi<16, true>(epi, cs) : max_clusters_epi<16, false>(epi, cs);
    case 32: return fp8 ? max_clusters_epi<32, true>(epi, cs) : max_clusters_epi<32, false>(epi, cs);
    case 64: return fp8 ? max_clusters_epi<64, true>(epi, cs) : max_clusters_epi<64, false>(epi, cs);
    case 128: return fp8 ? max_clusters_epi<128, true>(epi, cs) : max_clusters_epi<128, false>(epi, cs);
    case 256: return fp8 ? max_clusters_epi<256, true>(epi, cs) : max_clusters_epi<256, false>(epi, cs);
    default: return 0;
  }
}

// Cluster split-K size for a contraction, or 1 (stream-K / whole tiles).
// Activation tiles up to 64 wide stream weights with a short MMA per chunk:
// the largest cs in 2..8 (at most the K chunks) whose tiles x cs CTAs fill
// at least three quarters of the SMs without exceeding them.  At 128 and 256
// wide, a chunk's MMA is 8-16x longer than at 16 and each slice hands a
// 64-128 KB fp32 partial through distributed shared memory: the largest cs in 2..4
// whose tiles x cs CTAs fit the SMs in one wave, however few (measured at
// 128 and 256 rows: a 16-tile K/V contraction takes 20-24 us in 4 slices,
// 30-34 us in 8 and 32-33 us as whole tiles; a 48-56-tile QKV contraction
// 27-28 us in 2 slices against 35-38 us whole and 41-54 us stream-K).
// Either way every tile's cluster must fit the device at once.  ctas <= -2
// forces cs = -ctas.
int pick_csplit(int tiles, int n_chunks, int bn, int epi, bool fp8, int nsm, int ctas) {
  if (epi == EPI_TOPK) return 1;
  if (ctas <= -2) {
    const int cs = -ctas;
    return cs <= 8 && cs <= n_chunks && max_clusters_of(bn, epi, fp8, cs) >= 1 ? cs : 1;
  }
  if (ctas != 0) return 1;
  const bool narrow = bn <= 64;
  for (int cs = narrow ? 8 : 4; cs >= 2; --cs) {
    if (cs > n_chunks || (long)tiles * cs > nsm) continue;
    if (narrow && (long)tiles * cs * 4 < (long)nsm * 3) continue;
    if (max_clusters_of(bn, epi, fp8, cs) >= tiles) return cs;
  }
  // so few narrow tiles that no split fills three quarters of the SMs (at
  // most 18 tiles): the widest split with at least two K chunks per slice
  // still beats stream-K, whose pieces meet through global memory
  if (narrow)
    for (int cs = std::min(8, n_chunks / 2); cs >= 2; --cs)
      if ((long)tiles * cs <= nsm && max_clusters_of(bn, epi, fp8, cs) >= tiles) return cs;
  return 1;
}

template <int BN, bool FP8>
int launch_epi(int epi, const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& args, int grid, const Ctx& c) {
  switch (epi) {
    case EPI_TOPK: return launch_bn<BN, EPI_TOPK, FP8>(ma, mb, args, grid, c);
    case EPI_SWIGLU:
      if constexpr (BN <= 64) return launch_bn<BN, EPI_SWIGLU, FP8>(ma, mb, args, grid, c);
      return DFLASH2_ERR_SHAPE;
    case EPI_HEADS:
      if constexpr (BN <= 64) return launch_bn<BN, EPI_HEADS, FP8>(ma, mb, args, grid, c);
      return DFLASH2_ERR_SHAPE;
    default: return launch_bn<BN, EPI_PLAIN, FP8>(ma, mb, args, grid, c);
  }
}

template <int BN>
int launch_epi(int epi, bool fp8, const CUtensorMap& ma, const CUtensorMap& mb, const TcArgs& args, int grid,
               const Ctx& c) {
  return fp8 ? launch_epi<BN, true>(epi, ma, mb, args, grid, c) : launch_epi<BN, false>(epi, ma, mb, args, grid, c);
}

}  // namespace

int make_rows_map(CUtensorMap* map, const void* base, long long rows, int cols, long long ld_elems, int box_cols,
                  int box_rows) {
  auto fn = encode_fn();
  if (!fn) return DFLASH2_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (ld_elems * 2) % 16 || (box_cols * 2) % 16) return DFLASH2_ERR_SHAPE;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld_elems * 2};
  cuuint32_t box[2] = {(cuuint32_t)box_cols, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

int make_sw128_map(CUtensorMap* map, const void* base, long long rows, int cols, long long ld_elems, int box_rows) {
  auto fn = encode_fn();
  if (!fn) return DFLASH2_ERR_CUDA;
  if ((reinterpret_cast<uintptr_t>(base) & 15) || (ld_elems * 2) % 16) return DFLASH2_ERR_SHAPE;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)ld_elems * 2};
  cuuint32_t box[2] = {(cuuint32_t)BK, (cuuint32_t)box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

bool gemm_fusable(int M, int N, int epi) {
  // wider activation tiles run the plain epilogue and a row kernel: their
  // fused epilogues (16 columns per step, each step's norm/RoPE loads and
  // barriers in series) measured slower than the two kernels at 128 and 256
  if (pick_bn(M, N) > 64) return false;
  return epi != kEpiSwiglu || M % BM == 0;
}

size_t gemm_partial_bytes(int M, int N) { return (size_t)kMaxSM * 2 * BM * pick_bn(M, N) * sizeof(float); }

int gemm_tiles(int M, int N) {
  const int bn = pick_bn(M, N);
  return ((M + BM - 1) / BM) * ((N + bn - 1) / bn);
}

int gemm_topk_lists(int M, int N, int K, int nsm, int dtype) {
  (void)K;
  if (dtype == DFLASH2_BF16) {
    const int bn = pick_bn(M, N);
    const long units = (long)((M + BM - 1) / BM) * ((N + bn - 1) / bn);
    return (int)std::min<long>(units, nsm);
  }
  return topk_scan_lists(M);
}

int gemm_max_lists() { return std::max(kMaxSM, 0); }

thread_local int g_last_grid = 0;
int gemm_last_grid() { return g_last_grid; }
std::atomic<int> g_force_csplit{0};
void gemm_force_csplit(int cs) { g_force_csplit.store(cs); }

int gemm_bf16(const GemmOp& g, const Ctx& c) {
  if (g.M <= 0 || g.N <= 0 || g.K <= 0) return DFLASH2_ERR_SHAPE;
  const int bn = pick_bn(g.M, g.N);
  const int epi = g.topk ? EPI_TOPK : g.epi;
  if (epi >= EPI_SWIGLU && !gemm_fusable(g.M, g.N, epi)) return DFLASH2_ERR_SHAPE;
  TcArgs a;
  std::memset(&a, 0, sizeof(a));
  a.M = g.M;
  a.N = g.N;
  a.K = g.K;
  a.n_chunks = (g.K + BK - 1) / BK;
  a.m_tiles = (g.M + BM - 1) / BM;
  a.n_tiles = (g.N + bn - 1) / bn;
  a.tiles = a.m_tiles * a.n_tiles;
  a.work = (long)a.tiles * a.n_chunks;
  a.stream = (!g.topk && g.ctas >= 0) ? 1 : 0;
  const int fcs = g_force_csplit.load();
  a.csplit = kClusterSplit && !g.topk ? pick_csplit(a.tiles, a.n_chunks, bn, epi, g.wscale != nullptr, c.nsm,
                                                    fcs >= 2 && g.ctas == 0 ? -fcs : g.ctas)
                                      : 1;
  // 128- and 256-wide tiles without a cluster split run whole: the fix-up of
  // a stream-K piece reads a 64-128 KB fp32 partial serially, which costs
  // more than the SMs it fills (at 192-272 tiles: 64-72 us whole against
  // 74-83 us stream-K)
  if (a.csplit > 1 || (g.ctas == 0 && bn >= 128)) a.stream = 0;
  a.out = g.out;
  a.partial = g.partial;
  a.counters = g.counters;
  a.accumulate = g.accumulate ? 1 : 0;
  if (a.stream && (!g.partial || !g.counters)) return DFLASH2_ERR_INVALID_ARG;
  // stream-K: one CTA per SM, but at least kMinChunks chunks per CTA, so a
  // shared tile has few pieces to sum (each piece costs its last CTA a load)
  constexpr long kMinChunks = 8;
  const long want = a.stream ? (g.ctas > 0 ? std::min(g.ctas, kMaxSM)
                                           : std::max(1L, std::min<long>(c.nsm, a.work / kMinChunks)))
                             : c.nsm;
  const int grid = a.csplit > 1 ? a.tiles * a.csplit : (int)std::min<long>(want, a.stream ? a.work : a.tiles);
  g_last_grid = grid;
  a.lists_v = g.lists_v;
  a.lists_i = g.lists_i;
  a.thr = g.thr;
  if (g.topk && !g.thr) return DFLASH2_ERR_INVALID_ARG;
  a.debug = g.debug;
  a.mult = g.mult;
  a.cap = g.cap;
  a.status = c.status;
  a.wscale = g.wscale;
  if (g.topk && a.n_tiles > 32) return DFLASH2_ERR_SHAPE;
  if (epi == EPI_SWIGLU) {
    if (!g.act) return DFLASH2_ERR_INVALID_ARG;
    a.act = static_cast<bf16*>(g.act);
    a.I = g.M / 2;
  } else if (epi == EPI_HEADS) {
    if (g.hd * (g.n_qh + 2 * g.n_kh) != g.M || (g.hd != 64 && g.hd != BM) || !g.kn || (g.n_qh > 0 && !g.qn) ||
        g.nblk < 0 || g.nblk > g.N)
      return DFLASH2_ERR_INVALID_ARG;
    if (g.nblk > 0 && (!g.rope || !g.q || !g.kb || !g.vb || g.n_qh == 0)) return DFLASH2_ERR_INVALID_ARG;
    if (g.nblk < g.N && (!g.rope_app || !g.dst || !g.kc || !g.vc)) return DFLASH2_ERR_INVALID_ARG;
    a.hd = g.hd;
    a.n_qh = g.n_qh;
    a.n_kh = g.n_kh;
    a.qn = static_cast<const bf16*>(g.qn);
    a.kn = static_cast<const bf16*>(g.kn);
    a.eps = g.eps;
    a.nblk = g.nblk;
    a.rope = g.rope;
    a.rope_app = g.rope_app;
    a.dst = g.dst;
    a.q = static_cast<bf16*>(g.q);
    a.kb = static_cast<bf16*>(g.kb);
    a.vb = static_cast<bf16*>(g.vb);
    a.kc = static_cast<bf16*>(g.kc);
    a.vc = static_cast<bf16*>(g.vc);
  }

  CUtensorMap ma, mb;
  const bool fp8 = g.wscale != nullptr;
  int rc = fp8 ? make_map8(&ma, g.W, g.M, g.K, g.ldw, epi == EPI_SWIGLU ? BM / 2 : BM)
               : make_map(&ma, g.W, g.M, g.K, g.ldw, epi == EPI_SWIGLU ? BM / 2 : BM);
  if (rc) return rc;
  rc = make_map(&mb, g.X, g.N, g.K, g.ldx, bn);
  if (rc) return rc;

  switch (bn) {
    case 16: return launch_epi<16>(epi, fp8, ma, mb, a, grid, c);
    case 32: return launch_epi<32>(epi, fp8, ma, mb, a, grid, c);
    case 64: return launch_epi<64>(epi, fp8, ma, mb, a, grid, c);
    case 128: return launch_epi<128>(epi, fp8, ma, mb, a, grid, c);
    default: return launch_epi<256>(epi, fp8, ma, mb, a, grid, c);
  }
}

}  // namespace df2
