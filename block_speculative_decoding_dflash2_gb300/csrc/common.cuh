// Device helpers shared by the DFlash2 kernels: element I/O, reductions,
// the device status word, and thin PTX wrappers for mbarrier, TMA and
// tcgen05 (sm_103a).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dflash2.h"

namespace df2 {

typedef __nv_bfloat16 bf16;

// ----------------------------------------------------------------- elements

template <typename T> __device__ __forceinline__ float ld(const T* p);
template <> __device__ __forceinline__ float ld<float>(const float* p) { return *p; }
template <> __device__ __forceinline__ float ld<bf16>(const bf16* p) { return __bfloat162float(*p); }

template <typename T> __device__ __forceinline__ void st(T* p, float v);
template <> __device__ __forceinline__ void st<float>(float* p, float v) { *p = v; }
template <> __device__ __forceinline__ void st<bf16>(bf16* p, float v) { *p = __float2bfloat16_rn(v); }

// ----------------------------------------------------------------- reductions

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Block-wide sum; `sh` needs 32 floats.  Every thread gets the result.
__device__ __forceinline__ float block_sum(float v, float* sh) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = (blockDim.x + 31) >> 5;
  v = warp_sum(v);
  __syncthreads();
  if (lane == 0) sh[wid] = v;
  __syncthreads();
  float t = 0.f;
  for (int i = 0; i < nw; ++i) t += sh[i];
  return t;
}

// ----------------------------------------------------------------- PDL
// Programmatic dependent launch: let the next kernel of the stream start its
// launch now, and wait for the previous kernel's completion (and memory) here.
__device__ __forceinline__ void pdl_launch_next() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ----------------------------------------------------------------- status

__device__ __forceinline__ void flag(unsigned* status, unsigned code) {
  if (status) atomicOr(status, code);
}

// ----------------------------------------------------------------- top-k order
// Candidate a "beats" b: larger value, or equal value and smaller id.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

constexpr int KMAX = 16;  // entries per partial top-k list (top_k <= 16)

// Offer candidate (cv, ci) to a warp-held sorted list: lanes 0..15 hold
// entry `lane` (best first) in (lv, li); (tv, ti) is entry 15, kept current.
// Must be called by all 32 lanes with the same (cv, ci).
__device__ __forceinline__ void warp_list_offer(float& lv, int& li, float& tv, int& ti,
                                                float cv, int ci) {
  if (!beats(cv, ci, tv, ti)) return;  // uniform across the warp
  const int lane = threadIdx.x & 31;
  const bool ahead = (lane < KMAX) && beats(lv, li, cv, ci);
  const int pos = __popc(__ballot_sync(0xffffffffu, ahead) & 0xffffu);
  const float pv = __shfl_up_sync(0xffffffffu, lv, 1);
  const int pi = __shfl_up_sync(0xffffffffu, li, 1);
  if (lane < KMAX && lane > pos) { lv = pv; li = pi; }
  if (lane == pos) { lv = cv; li = ci; }
  tv = __shfl_sync(0xffffffffu, lv, KMAX - 1);
  ti = __shfl_sync(0xffffffffu, li, KMAX - 1);
}

// 64-bit order key of a candidate: a larger key is a better candidate under
// the (value descending, id ascending) order, so one integer compare replaces
// the two-field one.  Value bits are mapped to an unsigned order (negative
// zero first folded onto zero, which compares equal to it).  Key 0 is below
// every candidate with a non-NaN value: it marks an empty list slot.
__device__ __forceinline__ unsigned long long order_key(float v, int id) {
  unsigned u = __float_as_uint(v + 0.f);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return ((unsigned long long)u << 32) | (unsigned)(0x7fffffff - id);
}
__device__ __forceinline__ float key_value(unsigned long long key) {
  const unsigned u = (unsigned)(key >> 32);
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}
__device__ __forceinline__ int key_id(unsigned long long key) { return 0x7fffffff - (int)(unsigned)key; }

// Offer key ck to a warp-held sorted list of keys: lanes 0..15 hold entry
// `lane` (best first, 0 = empty), lanes 16..31 hold 0; tk is entry 15, kept
// current.  Called by all 32 lanes with the same ck.
__device__ __forceinline__ void warp_key_offer(unsigned long long& lk, unsigned long long& tk,
                                               unsigned long long ck) {
  if (ck <= tk) return;  // uniform across the warp
  const int lane = threadIdx.x & 31;
  const int pos = __popc(__ballot_sync(0xffffffffu, lane < KMAX && lk > ck) & 0xffffu);
  const unsigned long long pk = __shfl_up_sync(0xffffffffu, lk, 1);
  if (lane < KMAX && lane > pos) lk = pk;
  if (lane == pos) lk = ck;
  tk = __shfl_sync(0xffffffffu, lk, KMAX - 1);
}

// Merge one key per lane (0 = none) into the warp-held list above in one
// pass: a bitonic sort of the 32 offered keys (descending), then a bitonic
// merge of the list with the best 16 of them (the list descending in lanes
// 0..15, the offers ascending in lanes 16..31 form one bitonic sequence).
__device__ __forceinline__ void warp_key_merge(unsigned long long& lk, unsigned long long& tk,
                                               unsigned long long ck) {
  const int lane = threadIdx.x & 31;
  unsigned long long x = ck;
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1)
#pragma unroll
    for (int j = k >> 1; j > 0; j >>= 1) {
      const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
      // blocks with (lane & k) == 0 sort descending (the whole warp at k = 32)
      const bool keep_max = ((lane & j) == 0) == ((lane & k) == 0);
      x = keep_max ? (x > y ? x : y) : (x < y ? x : y);
    }
  const unsigned long long rev = __shfl_sync(0xffffffffu, x, 31 - lane);
  x = lane < KMAX ? lk : rev;
#pragma unroll
  for (int j = 16; j > 0; j >>= 1) {
    const unsigned long long y = __shfl_xor_sync(0xffffffffu, x, j);
    x = (lane & j) == 0 ? (x > y ? x : y) : (x < y ? x : y);
  }
  lk = lane < KMAX ? x : 0ull;
  tk = __shfl_sync(0xffffffffu, lk, KMAX - 1);
}

// ----------------------------------------------------------------- PTX: smem

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// 16-byte asynchronous global -> shared copy; with valid == false nothing is
// read and the 16 destination bytes are zero-filled (src must still be a
// mapped address).
__device__ __forceinline__ void cp_async16(void* dst, const void* src, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)), "l"(src),
               "r"(valid ? 16 : 0)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

// Contiguous global -> shared copy of `bytes` (a multiple of 16; both
// addresses 16-byte aligned) by the bulk-copy engine, completing on mbarrier
// `bar` (complete_tx).  Preceded by a proxy fence so that earlier generic
// accesses to the destination are ordered before the async write.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "fence.proxy.async.shared::cta;\n\t"
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy shared-memory writes before
// later async-proxy accesses (TMA, tcgen05.mma operand reads).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ----------------------------------------------------------------- fp8 weights
// Two fp8 e4m3 codes (byte 0 -> .x, byte 1 -> .y) as bf16x2, exactly: every
// finite e4m3 value (3 mantissa bits, exponents 2^-9..2^8) is a bf16 value.
__device__ __forceinline__ __nv_bfloat162 e4m3x2_to_bf16x2(uint16_t q) {
  const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(q), __NV_E4M3);
  return __float22bfloat162_rn(__half22float2(__half2(h)));
}
__device__ __forceinline__ float e4m3_to_float(uint8_t q) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw(static_cast<__nv_fp8_storage_t>(q), __NV_E4M3);
  return __half2float(__half(h));
}

// ----------------------------------------------------------------- PTX: clusters
// Whole-cluster barrier with release/acquire ordering of shared memory (every
// thread of every CTA of the cluster must reach it, like __syncthreads).
__device__ __forceinline__ void cluster_sync() {
  __syncwarp();
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Address in CTA `rank`'s shared memory of the same offset as local `p`.
__device__ __forceinline__ uint32_t dsmem_addr(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ float4 ld_dsmem4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float2 ld_dsmem2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}

// ----------------------------------------------------------------- PTX: mbarrier

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Non-blocking test for the phase with the given parity (for a thread that
// polls several barriers: try_wait may suspend the thread for a while on a
// phase that is not complete yet).
__device__ __forceinline__ bool mbar_test_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase with the given parity.  Gives up (returns
// false) after `limit_ns` or as soon as *abort becomes non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort,
                                          uint64_t limit_ns) {
  const uint32_t a = smem_u32(bar);
  if (mbar_try_wait(a, parity)) return true;
  const uint64_t t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(a, parity)) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ----------------------------------------------------------------- PTX: TMA

__device__ __forceinline__ void tma_prefetch_desc(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}

__device__ __forceinline__ void tma_load_2d(void* dst, const void* map, uint64_t* bar, int x, int y,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
      "l"(map), "r"(x), "r"(y), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// ----------------------------------------------------------------- PTX: tcgen05

__device__ __forceinline__ void tmem_alloc(uint32_t* dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst)),
               "r"(ncols)
               : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulation.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// 32 lanes x 16 consecutive 32-bit TMEM columns -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 lanes x 8 consecutive 32-bit TMEM columns -> 8 registers per thread,
// without waiting (tmem_ld_wait() before the registers are read).
__device__ __forceinline__ void tmem_ld8_nowait(uint32_t taddr, uint32_t (&r)[8]) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// 8 registers per thread -> 32 lanes x 8 consecutive TMEM columns
// (tmem_st_wait() before the columns are read by another agent).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of an MN-major operand with the 128-byte
// swizzle: each K index is a 128-byte row of 64 consecutive M (or N)
// elements, 8 such rows form a 1024-byte atom; atoms along K are sbo bytes
// apart and 64-element blocks along M (N) lbo bytes apart.
__device__ __forceinline__ uint64_t sdesc_mn_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)2 << 61;
  return d;
}

// Shared-memory matrix descriptor of a K-major tile written by TMA with the
// 128-byte swizzle: 8-row atoms of 128 bytes, atoms 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);  // start address
  d |= (uint64_t)1 << 16;                    // leading-dimension offset (unused for this layout)
  d |= (uint64_t)(1024 >> 4) << 32;          // stride-dimension offset: 8 rows x 128 B
  d |= (uint64_t)1 << 46;                    // descriptor version (sm_100 family)
  d |= (uint64_t)2 << 61;                    // 128-byte swizzle
  return d;
}

// Instruction descriptor: kind::f16 with bf16 A/B, fp32 D, both K-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

}  // namespace df2
