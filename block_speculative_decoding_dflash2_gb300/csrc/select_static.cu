// dflash2_select_path_static: the path selector for callers that cannot
// allocate device memory.
//
// Some callers cannot hand the library a workspace: code that runs where the
// device allocator may not be called (inside a custom allocator's own
// callbacks, from a runtime that owns all device memory and forbids other
// allocations, or from a plugin host that gives a plugin only its inputs and
// outputs).  For them this entry point keeps its scratch in one file-scope
// device array, sized here, that every GPU loading the library holds until
// the process exits.  Nothing is allocated and no allocating library routine
// is called.
//
// The array's host-side name is only a stand-in for the symbol: its device
// address is looked up with cudaGetSymbolAddress the first time the entry
// point runs on a device (with that device current) and cached per device.
// Every call shares the array, so two calls that overlap on the GPU (other
// streams, other threads) race and corrupt each other; calls on one stream
// are ordered and safe.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace df2 {
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;  // 8 MiB
static __device__ __align__(256) unsigned char g_select_scratch[kStaticScratchBytes];

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

// Device address of g_select_scratch on the current device (looked up once
// per device), or nullptr with *err set.
void* scratch_address(int* err) {
  static std::mutex mu;
  static void* addr[64] = {nullptr};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *err = DFLASH2_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_select_scratch) != cudaSuccess || !p) {
      (void)cudaGetLastError();
      *err = DFLASH2_ERR_CUDA;
      return nullptr;
    }
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace
}  // namespace df2

using namespace df2;

extern "C" {

size_t dflash2_select_path_static_capacity(void) { return kStaticScratchBytes; }

// The device status word of the last dflash2_select_path_static call on the
// current device (the first word of the fixed array): read, then cleared,
// ordered after the work already on `stream`, which this call synchronises.
int dflash2_select_path_static_read_status(void* stream) {
  int err = DFLASH2_OK;
  void* base = scratch_address(&err);
  if (!base) return err;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, base, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if (cudaMemsetAsync(base, 0, sizeof(v), st) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DFLASH2_ERR_CUDA;
  return (int)(v & 0x7fffffffu);
}

int dflash2_select_path_static(const dflash2_config* cfg, const dflash2_weights* w, int batch, const int32_t* anchor,
                               const int32_t* cand_id, const float* cand_logit, int32_t* path, float* path_score,
                               void* stream) {
  const int vc = dflash2_validate_config(cfg);
  if (vc != DFLASH2_OK) return vc;
  if (!w || !w->embed || !w->sel) return DFLASH2_ERR_INVALID_ARG;
  if (batch <= 0) return DFLASH2_ERR_SHAPE;
  if (!anchor || !cand_id || !cand_logit || !path) return DFLASH2_ERR_INVALID_ARG;
  const bool fp8 = cfg->dtype == DFLASH2_FP8W;
  if (fp8 && (!w->scales || !w->scales->sel)) return DFLASH2_ERR_INVALID_ARG;
  dflash2_config c = *cfg;
  if (fp8) c.dtype = DFLASH2_BF16;  // bf16 embedding rows; e4m3 selector weights with row scales
  const int D = c.block_size - 1, k = c.top_k, r = c.selector_rank, H = c.hidden;
  const int es = c.dtype == DFLASH2_BF16 ? 2 : 4;
  // bound the batch before any int product: one sequence's gathered rows
  // alone take (D*k+1)*H*es bytes, so a batch past this cannot fit
  const size_t per_seq = (size_t)(D * k + 1) * ((size_t)H * es + 2 * (size_t)r * sizeof(float));
  if ((size_t)batch > kStaticScratchBytes / per_seq) return DFLASH2_ERR_WORKSPACE;
  const int nsel = batch * (D * k + 1);
  // scratch layout: status word | tile counters | gathered rows | factors | split partials
  int dev = 0, nsm = 0, maj = 0, mi = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return DFLASH2_ERR_CUDA;
  if (maj != 10 || mi != 3) return DFLASH2_ERR_UNSUPPORTED;
  nsm = std::min(nsm, kMaxSM);
  // the factor contraction runs on whole tiles (no stream-K pieces), so the
  // scratch holds only the gathered rows and the factors
  const size_t o_x = 256;
  const size_t o_y = o_x + al((size_t)nsel * H * es);
  const size_t need = o_y + al((size_t)nsel * 2 * r * sizeof(float));
  if (need > kStaticScratchBytes) return DFLASH2_ERR_WORKSPACE;  // batch too large for the fixed scratch
  int err = DFLASH2_OK;
  char* base = static_cast<char*>(scratch_address(&err));
  if (!base) return err;
  Ctx ctx;
  ctx.stream = static_cast<cudaStream_t>(stream);
  ctx.status = reinterpret_cast<unsigned*>(base);
  ctx.nsm = nsm;
  // the status word must start at zero
  if (cudaMemsetAsync(base, 0, o_x, ctx.stream) != cudaSuccess) return DFLASH2_ERR_CUDA;
  int rc = launch_sel_gather(c.dtype, anchor, cand_id, batch, D, k, w->embed, c.vocab, H, base + o_x, ctx);
  if (rc) return rc;
  GemmOp g;
  std::memset(&g, 0, sizeof(g));
  g.W = w->sel;
  g.wscale = fp8 ? w->scales->sel : nullptr;
  g.M = 2 * r;
  g.K = H;
  g.ldw = H;
  g.X = base + o_x;
  g.N = nsel;
  g.ldx = H;
  g.out = reinterpret_cast<float*>(base + o_y);
  g.ctas = -1;
  g.mult = 1.f;
  rc = c.dtype == DFLASH2_BF16 ? gemm_bf16(g, ctx) : gemm_f32(g, ctx);
  if (rc) return rc;
  return launch_viterbi(reinterpret_cast<const float*>(base + o_y), nullptr, anchor, c.vocab, cand_id, cand_logit,
                        batch, D, k, r, path, path_score, ctx);
}

}  // extern "C"
