// C ABI of the DFlash2 draft step: argument checks, workspace plan and the
// launch sequence of each entry point (declared in include/dflash2.h).
//
// Step order on the caller's stream ("Train a DFlash Drafter for
// Speculative Decoding", "What is DFlash?" and "Variants"):
//   (a) fc GEMM -> RMSNorm -> per layer [W_k;W_v] GEMM -> k-norm/RoPE -> paged K/V
//   (b) embed [anchor, MASK...] -> per layer:
//         norm -> tap GEMM -> dyn conv -> QKV GEMM -> q/k norm + RoPE
//         -> attention(context + block) -> O GEMM -> +residual, norm
//         -> tap GEMM -> dyn conv -> gate/up GEMM -> SiLU*up -> down GEMM
//         -> +residual, next norm (final norm packs positions 1..B-1)
//   (c) lm_head GEMM with streaming top-k -> merge
//   (d) selector gather -> factor GEMM -> Viterbi;  verify/accept
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstring>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace df2 {
namespace {

constexpr int kVersion = 10000;

std::atomic<long long> g_launches{0};
std::atomic<int> g_last_schedule{0};
void* volatile g_stage_events[DFLASH2_N_STAGE_EVENTS] = {nullptr};
std::atomic<int> g_stage_on{0};

// Records stage event i on the call's stream.  While the stream is being
// captured the record is made external, so it stays in the graph as an event
// node that later replays fire; otherwise it is a plain record.
int stage_event(int i, cudaStream_t st) {
  if (!g_stage_on.load(std::memory_order_relaxed)) return DFLASH2_OK;
  cudaEvent_t ev = static_cast<cudaEvent_t>(g_stage_events[i]);
  if (!ev) return DFLASH2_OK;
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  cudaError_t e = cudaStreamIsCapturing(st, &cs);
  if (e == cudaSuccess)
    e = cs == cudaStreamCaptureStatusActive ? cudaEventRecordWithFlags(ev, st, cudaEventRecordExternal)
                                            : cudaEventRecord(ev, st);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return DFLASH2_ERR_CUDA;
  }
  return DFLASH2_OK;
}

// Bytes of an activation / cache element (fp8 weights run on bf16 activations).
int esize(int dtype) { return dtype == DFLASH2_F32 ? 4 : 2; }

// The config as the activation path sees it: fp8-weight configs compute with
// bf16 activations, cache and norm gains.
dflash2_config act_config(const dflash2_config& c) {
  dflash2_config a = c;
  if (a.dtype == DFLASH2_FP8W) a.dtype = DFLASH2_BF16;
  return a;
}

// Row scales of the fp8 weights (all null for F32 / BF16 configs).
struct Scales {
  const float *lm_head = nullptr, *fc = nullptr, *sel = nullptr;
  const dflash2_layer_scales* layers = nullptr;
  const float* of(const float* dflash2_layer_scales::*f, int l) const { return layers ? layers[l].*f : nullptr; }
};
Scales scales_of(const dflash2_config& cfg, const dflash2_weights& w) {
  Scales s;
  if (cfg.dtype == DFLASH2_FP8W && w.scales) {
    s.lm_head = w.scales->lm_head;
    s.fc = w.scales->fc;
    s.sel = w.scales->sel;
    s.layers = w.scales->layers;
  }
  return s;
}

size_t al(size_t x) { return (x + 255) & ~size_t(255); }

int check_config(const dflash2_config* c) {
  if (!c) return DFLASH2_ERR_INVALID_ARG;
  if (c->dtype != DFLASH2_F32 && c->dtype != DFLASH2_BF16 && c->dtype != DFLASH2_FP8W) return DFLASH2_ERR_DTYPE;
  if (c->block_size < 2 || c->block_size > 32) return DFLASH2_ERR_BLOCK_SIZE;
  if (c->hidden <= 0 || c->n_q_heads <= 0 || c->n_kv_heads <= 0 || c->intermediate <= 0 || c->vocab <= 0 ||
      c->n_layers <= 0 || c->n_taps <= 0 || c->page_size <= 0)
    return DFLASH2_ERR_SHAPE;
  if (c->head_dim != 64 && c->head_dim != 128) return DFLASH2_ERR_SHAPE;
  if (c->n_q_heads % c->n_kv_heads) return DFLASH2_ERR_SHAPE;
  if (c->conv_kernel_size != 2 && c->conv_kernel_size != 0) return DFLASH2_ERR_SHAPE;  // DFlash 2, or v1 (none)
  if (c->sliding_window < 0) return DFLASH2_ERR_SHAPE;
  // fp8 weight rows are read in 16-byte units (TMA rows, staged tap rows)
  if (c->dtype == DFLASH2_FP8W && (c->hidden % 16 || c->intermediate % 16)) return DFLASH2_ERR_SHAPE;
  if (c->conv_group_size <= 0 || c->hidden % c->conv_group_size) return DFLASH2_ERR_SHAPE;
  if (c->top_k < 1 || c->top_k > KMAX || c->top_k > c->vocab) return DFLASH2_ERR_SHAPE;
  if (c->selector_rank < 1 || c->selector_rank > 128) return DFLASH2_ERR_SHAPE;
  if (c->mask_token_id < 0 || c->mask_token_id >= c->vocab) return DFLASH2_ERR_SHAPE;
  if (!(c->rms_eps >= 0.f) || !(c->rope_theta > 0.f)) return DFLASH2_ERR_SHAPE;
  // 16-byte vector access of rows and channel groups
  if (c->hidden % 8 || c->intermediate % 8 || c->conv_group_size % 4) return DFLASH2_ERR_SHAPE;
  const int R = (c->n_q_heads / c->n_kv_heads) * c->block_size;
  if (R * c->head_dim > 128 * 128) return DFLASH2_ERR_SHAPE;  // attention rows held in shared memory
  if (viterbi_smem_bytes(c->block_size - 1, c->top_k, c->selector_rank) > 200 * 1024) return DFLASH2_ERR_SHAPE;
  // element counts used as 32-bit ints by the launchers
  if ((long long)c->vocab * c->hidden > (1LL << 40)) return DFLASH2_ERR_SHAPE;
  return DFLASH2_OK;
}

// Most lm_head rows (batch * drafts) a draft step takes.
constexpr int kMaxTopkRows = 32 * 256;

struct Layout {
  size_t status, cnt, cnta, thr, f, Y, P, Ya, Pa, h, u, u2, ua, u2a, q, kb, vb, attn, O, act, hn, logits, lv, li, selx,
      rope, ropea, dsta, total;
};

Layout plan(const dflash2_config& c0, int batch, int n_new, int max_ctx) {
  const dflash2_config c = act_config(c0);
  const int H = c.hidden, B = c.block_size, D = B - 1, es = esize(c.dtype);
  const int nq = c.n_q_heads, nkv = c.n_kv_heads, d = c.head_dim, I = c.intermediate;
  const int G = H / c.conv_group_size, r = c.selector_rank, k = c.top_k;
  const int rows = batch * B;
  const int nsel = batch * (D * k + 1);
  // every contraction of a call: {M, N, K, writes Y}
  struct Shape {
    int M, N, K;
    bool y;
  };
  const Shape shapes[8] = {{H, n_new, c.n_taps * H, true},      {2 * nkv * d, n_new, H, true},
                           {2 * G, rows, H, true},              {(nq + 2 * nkv) * d, rows + n_new, H, true},
                           {H, rows, nq * d, false},            {2 * I, rows, H, true},
                           {H, rows, I, false},                 {2 * r, nsel, H, true}};
  // the append branch (shapes 0-1) runs concurrently with the block branch
  // (shapes 2-7), so each has its own output, partial and counter regions
  size_t P = 0, Yb = 0, Pa = 0, Yba = 0;
  for (int i = 0; i < 8; ++i) {
    const Shape& sh = shapes[i];
    if (sh.N <= 0) continue;
    size_t& p = i < 2 ? Pa : P;
    size_t& y = i < 2 ? Yba : Yb;
    p = std::max(p, c.dtype == DFLASH2_BF16 ? gemm_partial_bytes(sh.M, sh.N) : 0);
    if (sh.y) y = std::max(y, (size_t)sh.N * sh.M * sizeof(float));
  }
  const int n_lists = std::max(kMaxSM, topk_scan_lists(c.vocab));
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o += al(bytes);
    return at;
  };
  // the status word and both counter arrays sit at the same offsets for every
  // call and size, so counters left at zero by one call are zero for the next
  L.status = take(256);
  L.cnt = take(kMaxSM * sizeof(int));
  L.cnta = take(kMaxSM * sizeof(int));
  L.thr = take((size_t)kMaxTopkRows * kTopkSlots * sizeof(unsigned long long));  // the lm_head's shared top-k bounds
  L.Y = take(Yb);
  L.P = take(P);
  L.Ya = take(Yba);
  L.Pa = take(Pa);
  L.h = take((size_t)rows * H * 4);
  L.u = take((size_t)rows * H * es);
  L.u2 = take((size_t)rows * H * es);
  L.ua = take((size_t)rows * H * es);
  // u2a and f are one region: the merged QKV contraction reads the block's
  // conv output and the appended rows' features as one activation matrix
  L.u2a = take((size_t)(rows + n_new) * H * es);
  L.f = L.u2a + (size_t)rows * H * es;
  L.q = take((size_t)rows * nq * d * es);
  L.kb = take((size_t)rows * nkv * d * es);
  L.vb = take((size_t)rows * nkv * d * es);
  L.attn = take(batch > 0 ? attn_part_bytes(batch, B, nq, nkv, d, max_ctx) : 0);
  L.O = take((size_t)rows * nq * d * es);
  L.act = take((size_t)rows * I * es);
  L.hn = take((size_t)batch * D * H * es);
  L.logits = take(c.dtype == DFLASH2_F32 ? (size_t)batch * D * c.vocab * 4 : 0);
  L.lv = take((size_t)n_lists * batch * D * KMAX * 4);
  L.li = take((size_t)n_lists * batch * D * KMAX * 4);
  L.selx = take((size_t)nsel * H * es);
  L.rope = take((size_t)rows * (d / 2) * sizeof(float2));     // block rows' RoPE table
  L.ropea = take((size_t)n_new * (d / 2) * sizeof(float2));   // appended rows' RoPE table
  L.dsta = take((size_t)n_new * sizeof(long long));           // appended rows' cache offsets
  L.total = o;
  return L;
}

// Per-device facts: SM count and whether it is the sm_103 part this library targets.
int device_ctx(Ctx* ctx, void* stream, void* ws) {
  static int nsm_cache[64] = {0};
  static int ok_cache[64] = {0};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DFLASH2_ERR_CUDA;
  {
    std::lock_guard<std::mutex> g(mu);
    if (!nsm_cache[dev]) {
      int n = 0, maj = 0, mi = 0;
      if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&maj, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&mi, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return DFLASH2_ERR_CUDA;
      nsm_cache[dev] = std::min(n, kMaxSM);
      ok_cache[dev] = (maj == 10 && mi == 3) ? 1 : 0;
    }
    if (!ok_cache[dev]) return DFLASH2_ERR_UNSUPPORTED;
    ctx->nsm = nsm_cache[dev];
  }
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->status = static_cast<unsigned*>(ws);
  return DFLASH2_OK;
}

// Per-device side stream and fork/join events of the draft step (created on
// first use; the enqueue of one draft step holds g_side_mu).
struct SideStream {
  cudaStream_t s;
  cudaEvent_t fork, join;
  int prio = 0;  // the device's greatest stream priority
};
std::mutex g_side_mu;

int side_stream(SideStream* out) {
  static SideStream per_dev[64];
  static bool made[64] = {false};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return DFLASH2_ERR_CUDA;
  if (!made[dev]) {
    SideStream sd;
    int least = 0;
    if (cudaDeviceGetStreamPriorityRange(&least, &sd.prio) != cudaSuccess ||
        cudaStreamCreateWithFlags(&sd.s, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.fork, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&sd.join, cudaEventDisableTiming) != cudaSuccess)
      return DFLASH2_ERR_CUDA;
    per_dev[dev] = sd;
    made[dev] = true;
  }
  *out = per_dev[dev];
  return DFLASH2_OK;
}

#define TRY(x)                    \
  do {                            \
    const int rc_ = (x);          \
    if (rc_ != DFLASH2_OK) return rc_; \
  } while (0)

template <typename P>
P* at(void* ws, size_t off) {
  return reinterpret_cast<P*>(static_cast<char*>(ws) + off);
}

// out[n][m] (= or +=) sum_k W[m][k] X[n][k]; split-K partials and tile
// counters live in the workspace regions of L (the append branch's own
// regions when `append_branch`, since it runs concurrently with the block).
GemmOp gemm_op(const void* W, int M, int K, const void* X, int N, const float* wscale = nullptr) {
  GemmOp g;
  std::memset(&g, 0, sizeof(g));
  g.W = W;
  g.wscale = wscale;
  g.M = M;
  g.K = K;
  g.ldw = K;
  g.X = X;
  g.N = N;
  g.ldx = K;
  g.mult = 1.f;
  return g;
}

// A bf16 contraction with a fused epilogue (partials/counters of its branch).
int gemm_fused(GemmOp g, const Ctx& ctx, void* ws, const Layout& L, bool append_branch) {
  g.partial = reinterpret_cast<float*>(static_cast<char*>(ws) + (append_branch ? L.Pa : L.P));
  g.counters = reinterpret_cast<int*>(static_cast<char*>(ws) + (append_branch ? L.cnta : L.cnt));
  return gemm_bf16(g, ctx);
}

// c: the activation config (act_config); wscale: the fp8 row scales of W, or null.
int gemm(const dflash2_config& c, const Ctx& ctx, void* ws, const Layout& L, const void* W, int M, int K,
         const void* X, int N, float* out, bool accumulate, bool append_branch = false,
         const float* wscale = nullptr) {
  GemmOp g;
  std::memset(&g, 0, sizeof(g));
  g.W = W;
  g.wscale = wscale;
  g.M = M;
  g.K = K;
  g.ldw = K;
  g.X = X;
  g.N = N;
  g.ldx = K;
  g.out = out;
  g.accumulate = accumulate;
  g.partial = reinterpret_cast<float*>(static_cast<char*>(ws) + (append_branch ? L.Pa : L.P));
  g.counters = reinterpret_cast<int*>(static_cast<char*>(ws) + (append_branch ? L.cnta : L.cnt));
  g.mult = 1.f;
  if (c.dtype == DFLASH2_BF16) return gemm_bf16(g, ctx);
  return gemm_f32(g, ctx);
}

const char* elem_ptr(const void* base, size_t elems, int dtype) {
  return static_cast<const char*>(base) + elems * esize(dtype);
}

int check_weights(const dflash2_config& c, const dflash2_weights* w) {
  if (!w || !w->embed || !w->lm_head || !w->fc || !w->hidden_norm || !w->final_norm || !w->sel || !w->layers)
    return DFLASH2_ERR_INVALID_ARG;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& L = w->layers[l];
    if (!L.attn_norm || !L.qkv || !L.q_norm || !L.k_norm || !L.o || !L.mlp_norm || !L.gate_up || !L.down)
      return DFLASH2_ERR_INVALID_ARG;
    if (c.conv_kernel_size > 0 && (!L.tapgen_attn || !L.tapgen_mlp)) return DFLASH2_ERR_INVALID_ARG;
  }
  if (c.dtype == DFLASH2_FP8W) {
    const dflash2_scales* s = w->scales;
    if (!s || !s->lm_head || !s->fc || !s->sel || !s->layers) return DFLASH2_ERR_INVALID_ARG;
    for (int l = 0; l < c.n_layers; ++l) {
      const dflash2_layer_scales& L = s->layers[l];
      if (!L.qkv || !L.o || !L.gate_up || !L.down) return DFLASH2_ERR_INVALID_ARG;
      if (c.conv_kernel_size > 0 && (!L.tapgen_attn || !L.tapgen_mlp)) return DFLASH2_ERR_INVALID_ARG;
    }
  }
  return DFLASH2_OK;
}

// Stage (a), first half: the feature projection of the n_new appended rows
// into f (fc contraction, then the hidden norm).  With want_tables, the norm
// kernel also leaves the rows' RoPE angles and paged-cache offsets for a fused
// K/V epilogue.
int project_features(const dflash2_config& c, const dflash2_weights& w, const Scales& sc, int n_pages,
                     const int32_t* block_table, int max_pages, int batch, const int32_t* ctx_len, int n_new,
                     const void* taps, const int32_t* new_off, void* ws, const Layout& L, bool want_tables,
                     const Ctx& ctx, Ctx* rest_out) {
  const int H = c.hidden, nkv = c.n_kv_heads, d = c.head_dim;
  float* Y = at<float>(ws, L.Ya);
  // the first launch keeps the caller's ctx.pdl (false right after a fork)
  TRY(gemm(c, ctx, ws, L, w.fc, H, c.n_taps * H, taps, n_new, Y, false, true, sc.fc));
  Ctx rest = ctx;
  rest.pdl = true;
  RopeTab rt;
  std::memset(&rt, 0, sizeof(rt));
  if (want_tables) {
    rt.cs = at<float2>(ws, L.ropea);
    rt.dst = at<long long>(ws, L.dsta);
    rt.d = d;
    rt.freq = rope_freq(d, c.rope_theta);
    rt.ctx_len = ctx_len;
    rt.new_off = new_off;
    rt.batch = batch;
    rt.block_table = block_table;
    rt.max_pages = max_pages;
    rt.page_size = c.page_size;
    rt.n_pages = n_pages;
    rt.nkv = nkv;
  }
  TRY(launch_rows_feature_norm(c.dtype, Y, n_new, H, w.hidden_norm, c.rms_eps, at<char>(ws, L.f), rt, rest));
  if (rest_out) *rest_out = rest;
  return DFLASH2_OK;
}

// Stage (a), whole: features, then every layer's context K/V of the appended
// rows into the paged cache (a contraction per layer, K/V epilogue fused when
// its shape allows).
int run_append(const dflash2_config& c, const dflash2_weights& w, const Scales& sc, void* kc, void* vc, int n_pages,
               const int32_t* block_table, int max_pages, int batch, const int32_t* ctx_len, int n_new,
               const void* taps, const int32_t* new_off, void* ws, const Layout& L, const Ctx& ctx,
               int kv_nsm = 0) {
  if (n_new == 0) return DFLASH2_OK;
  const int H = c.hidden, nq = c.n_q_heads, nkv = c.n_kv_heads, d = c.head_dim;
  float* Y = at<float>(ws, L.Ya);
  void* f = at<char>(ws, L.f);
  const bool fused_kv = c.dtype == DFLASH2_BF16 && gemm_fusable(2 * nkv * d, n_new, kEpiHeads);
  Ctx rest;
  TRY(project_features(c, w, sc, n_pages, block_table, max_pages, batch, ctx_len, n_new, taps, new_off, ws, L,
                       fused_kv, ctx, &rest));
  const size_t layer_elems = (size_t)n_pages * c.page_size * nkv * d;
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& Lw = w.layers[l];
    // layer 0's K/V contraction fits the SMs the block's first QKV
    // contraction leaves free; later layers run beside nothing and take all
    Ctx lrest = rest;
    if (kv_nsm > 0 && l == 0) lrest.nsm = kv_nsm;
    // the k and v rows of the qkv matrix (fp8: bytes, and their scales)
    const float* skv = sc.layers ? sc.layers[l].qkv + (size_t)nq * d : nullptr;
    const void* wkv = skv ? static_cast<const void*>(static_cast<const uint8_t*>(Lw.qkv) + (size_t)nq * d * H)
                          : static_cast<const void*>(elem_ptr(Lw.qkv, (size_t)nq * d * H, c.dtype));
    char* kcl = const_cast<char*>(elem_ptr(kc, l * layer_elems, c.dtype));
    char* vcl = const_cast<char*>(elem_ptr(vc, l * layer_elems, c.dtype));
    if (fused_kv) {
      // K/V epilogue fused: k-norm + RoPE + paged store of the appended rows
      GemmOp g = gemm_op(wkv, 2 * nkv * d, H, f, n_new, skv);
      g.epi = kEpiHeads;
      g.hd = d;
      g.n_kh = nkv;
      g.kn = Lw.k_norm;
      g.eps = c.rms_eps;
      g.nblk = 0;
      g.rope_app = at<float2>(ws, L.ropea);
      g.dst = at<long long>(ws, L.dsta);
      g.kc = kcl;
      g.vc = vcl;
      TRY(gemm_fused(g, lrest, ws, L, true));
    } else {
      TRY(gemm(c, lrest, ws, L, wkv, 2 * nkv * d, H, f, n_new, Y, false, true, skv));
      TRY(launch_kv_append(c.dtype, Y, n_new, nkv, d, Lw.k_norm, c.rms_eps, c.rope_theta, ctx_len, new_off, batch,
                           block_table, max_pages, c.page_size, n_pages, kcl, vcl, lrest));
    }
  }
  return DFLASH2_OK;
}

int check_cache_args(void* kc, void* vc, int n_pages, const int32_t* block_table, int max_pages, int batch,
                     const int32_t* ctx_len, int n_new, const void* taps, const int32_t* new_off) {
  if (batch <= 0 || n_new < 0 || n_pages <= 0 || max_pages <= 0) return DFLASH2_ERR_SHAPE;
  if (!kc || !vc || !block_table || !ctx_len || !new_off) return DFLASH2_ERR_INVALID_ARG;
  if (n_new > 0 && !taps) return DFLASH2_ERR_INVALID_ARG;
  return DFLASH2_OK;
}

}  // namespace

RopeFreq rope_freq(int d, float theta) {
  RopeFreq f;
  const double l2t = std::log2((double)theta);
  for (int i = 0; i < 64; ++i) f.inv[i] = 2 * i < d ? std::exp2(-(2.0 * i / d) * l2t) : 0.0;
  return f;
}

void count_launch(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }

int draft_last_schedule() { return g_last_schedule.load(); }

int workspace_offsets(const dflash2_config* c, int batch, int n_new, int max_ctx, size_t* out, int n) {
  if (check_config(c) != DFLASH2_OK) return DFLASH2_ERR_SHAPE;
  if (!out || n < 14) return DFLASH2_ERR_INVALID_ARG;
  const Layout L = plan(*c, batch, n_new, max_ctx);
  const size_t v[14] = {L.f, L.h, L.u, L.u2, L.q, L.kb, L.vb, L.O, L.act, L.hn, L.ua, L.u2a, L.cnt, L.cnta};
  for (int i = 0; i < 14; ++i) out[i] = v[i];
  return DFLASH2_OK;
}

}  // namespace df2

using namespace df2;

extern "C" {

const char* dflash2_status_string(int s) {
  switch (s) {
    case DFLASH2_OK: return "ok";
    case DFLASH2_ERR_INVALID_ARG: return "invalid argument (null pointer, negative size or bad enum)";
    case DFLASH2_ERR_SHAPE: return "inconsistent or unsupported dimensions";
    case DFLASH2_ERR_BLOCK_SIZE: return "block size out of range or not drafts + 1";
    case DFLASH2_ERR_DTYPE: return "unsupported dtype";
    case DFLASH2_ERR_WORKSPACE: return "workspace missing or too small";
    case DFLASH2_ERR_CUDA: return "a CUDA call failed";
    case DFLASH2_ERR_UNSUPPORTED: return "unsupported device or request (this library targets sm_103a)";
    default: return "unknown status";
  }
}

int dflash2_version(void) { return kVersion; }

int64_t dflash2_launch_count(void) { return g_launches.load(); }

void dflash2_set_stage_events(void* const* events) {
  if (!events) {
    g_stage_on.store(0);
    return;
  }
  for (int i = 0; i < DFLASH2_N_STAGE_EVENTS; ++i) g_stage_events[i] = events[i];
  g_stage_on.store(1);
}

int dflash2_validate_config(const dflash2_config* cfg) { return check_config(cfg); }

size_t dflash2_workspace_size(const dflash2_config* cfg, int max_batch, int max_new_rows, int max_ctx) {
  if (check_config(cfg) != DFLASH2_OK || max_batch < 0 || max_new_rows < 0 || max_ctx < 0) return 0;
  return plan(*cfg, max_batch, max_new_rows, max_ctx).total;
}

int dflash2_append_context(const dflash2_config* cfg, const dflash2_weights* w, void* k_cache, void* v_cache,
                           int n_pages, const int32_t* block_table, int max_pages, int batch,
                           const int32_t* ctx_len, int n_new, const void* new_taps, const int32_t* new_off,
                           void* workspace, size_t ws_bytes, void* stream) {
  TRY(check_config(cfg));
  TRY(check_weights(*cfg, w));
  TRY(check_cache_args(k_cache, v_cache, n_pages, block_table, max_pages, batch, ctx_len, n_new, new_taps, new_off));
  if (!workspace) return DFLASH2_ERR_WORKSPACE;
  const Layout L = plan(*cfg, 0, n_new, 0);
  if (ws_bytes < L.total) return DFLASH2_ERR_WORKSPACE;
  Ctx ctx;
  TRY(device_ctx(&ctx, stream, workspace));
  return run_append(act_config(*cfg), *w, scales_of(*cfg, *w), k_cache, v_cache, n_pages, block_table, max_pages,
                    batch, ctx_len, n_new, new_taps, new_off, workspace, L, ctx);
}

int dflash2_draft_step(const dflash2_config* cfg, const dflash2_weights* w, void* k_cache, void* v_cache,
                       int n_pages, const int32_t* block_table, int max_pages, int batch, const int32_t* ctx_len,
                       int n_new, const void* new_taps, const int32_t* new_off, const int32_t* anchor,
                       int32_t* cand_id, float* cand_logit, float* debug_logits, void* workspace, size_t ws_bytes,
                       void* stream) {
  TRY(check_config(cfg));
  TRY(check_weights(*cfg, w));
  TRY(check_cache_args(k_cache, v_cache, n_pages, block_table, max_pages, batch, ctx_len, n_new, new_taps, new_off));
  if (!anchor || !cand_id || !cand_logit) return DFLASH2_ERR_INVALID_ARG;
  if (!workspace) return DFLASH2_ERR_WORKSPACE;
  const dflash2_config c = act_config(*cfg);
  const Scales sc = scales_of(*cfg, *w);
  const int max_ctx = max_pages * c.page_size;
  const Layout L = plan(c, batch, n_new, max_ctx);
  if (ws_bytes < L.total) return DFLASH2_ERR_WORKSPACE;
  if ((long long)batch * (c.block_size - 1) > kMaxTopkRows) return DFLASH2_ERR_SHAPE;
  Ctx ctx;
  TRY(device_ctx(&ctx, stream, workspace));

  const int H = c.hidden, B = c.block_size, D = B - 1, nq = c.n_q_heads, nkv = c.n_kv_heads, d = c.head_dim;
  const int I = c.intermediate, G = H / c.conv_group_size, rows = batch * B;
  // Stage (a) runs on the device's side stream, forked from and joined back
  // into the caller's stream (event edges, so graph capture records two
  // parallel branches), in one of two arrangements:
  //  separate: the side stream runs the feature projection and every
  //    layer's K/V contraction and joins before the first attention, so with
  //    one layer the K/V work overlaps the block's own QKV contraction
  //    (measured faster at one layer: the join stays late);
  //  merged: with several layers, when the QKV contraction can take the
  //    appended rows as extra activation columns (u2a and f are adjacent),
  //    the side stream runs the feature projection only and joins before
  //    layer 0's QKV contraction, and each layer's QKV contraction also
  //    projects the appended rows' k/v into the cache (W_k and W_v read once
  //    per layer instead of twice).
  const int qkvM = (nq + 2 * nkv) * d;
  // conv_kernel_size 0 (DFlash v1): no convolution, each sublayer reads its
  // normed rows (u2 aliases u); the merged arrangement needs u2a next to f,
  // so v1 runs the separate one
  const bool conv = c.conv_kernel_size > 0;
  const bool merged =
      conv && c.n_layers > 1 && c.dtype == DFLASH2_BF16 && gemm_fusable(qkvM, rows + n_new, kEpiHeads);
  std::unique_lock<std::mutex> side_lock(g_side_mu, std::defer_lock);
  SideStream side;
  const bool forked = n_new > 0;
  // The fused embedding prologue is latency-bound and the feature
  // contraction bandwidth-bound, and neither fits an SM beside the other: a
  // forked step splits the SMs, kForkPrologueSMs for the prologue (on fewer,
  // wider CTAs) and the rest for the contraction, so the two overlap.
  const bool fused = conv && conv_prologue_fits(c.dtype, batch, B, H, G, ctx.nsm);
  const bool split_sms = forked && fused && ctx.nsm > 2 * kForkPrologueSMs &&
                         conv_prologue_fits(c.dtype, batch, B, H, G, kForkPrologueSMs / 2);
  // sublayer prologues: one fused kernel (norm, tap logits, conv) when the
  // sequence's B rows fit its shared memory, else norm + tap GEMM + conv;
  // the QKV contraction with its q/k-norm + RoPE epilogue when its
  // activation tile allows
  const bool fused_qkv = merged || (c.dtype == DFLASH2_BF16 && gemm_fusable(qkvM, rows, kEpiHeads));
  // separate arrangement with the fused QKV: the block's first QKV
  // contraction leaves kForkKvSMs SMs free, where the side stream's K/V
  // contraction runs beside it instead of waiting for the QKV's CTAs to exit
  const bool kv_split = split_sms && !merged && fused_qkv && kForkKvSMs > 0 && ctx.nsm > 2 * kForkKvSMs;
  g_last_schedule.store((fused ? kSchedFusedPrologue : 0) | (split_sms ? kSchedSplitSMs : 0) |
                        (fused_qkv ? kSchedFusedQKV : 0) | (kv_split ? kSchedKvBesideQKV : 0) |
                        (merged ? kSchedMerged : 0));
  TRY(stage_event(0, ctx.stream));
  if (forked) {
    side_lock.lock();
    TRY(side_stream(&side));
    if (cudaEventRecord(side.fork, ctx.stream) != cudaSuccess || cudaStreamWaitEvent(side.s, side.fork, 0) != cudaSuccess)
      return DFLASH2_ERR_CUDA;
    Ctx actx = ctx;
    actx.stream = side.s;
    actx.pdl = false;  // full dependency on the fork event
    actx.prio = kSidePriority ? side.prio : 0;
    if (split_sms) actx.nsm = ctx.nsm - kForkPrologueSMs;
    if (merged)
      TRY(project_features(c, *w, sc, n_pages, block_table, max_pages, batch, ctx_len, n_new, new_taps, new_off,
                           workspace, L, true, actx, nullptr));
    else
      TRY(run_append(c, *w, sc, k_cache, v_cache, n_pages, block_table, max_pages, batch, ctx_len, n_new, new_taps,
                     new_off, workspace, L, actx, kv_split ? kForkKvSMs : 0));
    TRY(stage_event(1, side.s));
    if (cudaEventRecord(side.join, side.s) != cudaSuccess) return DFLASH2_ERR_CUDA;
  } else {
    TRY(stage_event(1, ctx.stream));
  }

  float* Y = at<float>(workspace, L.Y);
  float* h = at<float>(workspace, L.h);
  void* u = at<char>(workspace, L.u);    // MLP sublayer: normed input
  void* u2 = conv ? at<char>(workspace, L.u2) : u;  // MLP sublayer: after the conv
  void* ua = at<char>(workspace, L.ua);   // attention sublayer: normed input
  void* u2a = conv ? at<char>(workspace, L.u2a) : ua;  // attention sublayer: after the conv
  void* q = at<char>(workspace, L.q);
  void* kb = at<char>(workspace, L.kb);
  void* vb = at<char>(workspace, L.vb);
  void* O = at<char>(workspace, L.O);
  void* act = at<char>(workspace, L.act);
  void* hn = at<char>(workspace, L.hn);
  const size_t layer_elems = (size_t)n_pages * c.page_size * nkv * d;
  void* ws = workspace;

  RopeTab rt;  // the block rows' RoPE angles, left by the first kernel for the fused QKV epilogues
  std::memset(&rt, 0, sizeof(rt));
  if (fused_qkv) {
    rt.cs = at<float2>(workspace, L.rope);
    rt.d = d;
    rt.freq = rope_freq(d, c.rope_theta);
    rt.ctx_len = ctx_len;
    rt.new_off = new_off;
    rt.batch = batch;
  }
  if (fused) {
    Ctx ectx = ctx;
    if (split_sms) ectx.nsm = kForkPrologueSMs / 2;  // the prologue sizes its grid at two CTAs per SM
    TRY(launch_conv_prologue(c.dtype, nullptr, anchor, c.mask_token_id, w->embed, c.vocab, c.input_embedding_scale,
                             w->layers[0].attn_norm, c.rms_eps, w->layers[0].tapgen_attn,
                             sc.of(&dflash2_layer_scales::tapgen_attn, 0), batch, B, H, c.conv_group_size, h, ua, u2a,
                             rt, ectx));
  }
  else
    TRY(launch_embed_norm(c.dtype, anchor, c.mask_token_id, batch, B, w->embed, c.vocab, H, c.input_embedding_scale,
                          w->layers[0].attn_norm, c.rms_eps, h, ua, rt, ctx));
  const int n_app = merged ? n_new : 0;  // appended rows the QKV contractions carry
  for (int l = 0; l < c.n_layers; ++l) {
    const dflash2_layer_weights& Lw = w->layers[l];
    const float* s_tap_a = sc.of(&dflash2_layer_scales::tapgen_attn, l);
    const float* s_qkv = sc.of(&dflash2_layer_scales::qkv, l);
    const float* s_o = sc.of(&dflash2_layer_scales::o, l);
    const float* s_tap_m = sc.of(&dflash2_layer_scales::tapgen_mlp, l);
    const float* s_gu = sc.of(&dflash2_layer_scales::gate_up, l);
    const float* s_down = sc.of(&dflash2_layer_scales::down, l);
    // attention sublayer: conv around the normed input, QKV, attention, O (+= residual)
    if (fused) {
      if (l > 0)
        TRY(launch_conv_prologue(c.dtype, h, nullptr, 0, w->embed, c.vocab, 1.f, Lw.attn_norm, c.rms_eps,
                                 Lw.tapgen_attn, s_tap_a, batch, B, H, c.conv_group_size, nullptr, ua, u2a, RopeTab{},
                                 ctx));
    } else {
      if (l > 0) TRY(launch_rownorm(c.dtype, h, rows, H, Lw.attn_norm, c.rms_eps, ua, B, 0, ctx));
      if (conv) {
        TRY(gemm(c, ctx, ws, L, Lw.tapgen_attn, 2 * G, H, ua, rows, Y, false, false, s_tap_a));
        TRY(launch_dyn_conv(c.dtype, ua, Y, rows, H, c.conv_group_size, B, u2a, ctx));
      }
    }
    // merged: the QKV contraction reads the appended rows' features, a full
    // dependency on the join
    Ctx qctx = ctx;
    if (kv_split && l == 0) qctx.nsm = ctx.nsm - kForkKvSMs;
    if (forked && merged && l == 0) {
      if (cudaStreamWaitEvent(ctx.stream, side.join, 0) != cudaSuccess) return DFLASH2_ERR_CUDA;
      qctx.pdl = false;
    }
    if (fused_qkv) {
      // q/k-norm + RoPE fused into the QKV epilogue; merged: the appended rows'
      // features ride along as extra columns and their k/v go to the cache
      GemmOp g = gemm_op(Lw.qkv, qkvM, H, u2a, rows + n_app, s_qkv);
      g.epi = kEpiHeads;
      g.hd = d;
      g.n_qh = nq;
      g.n_kh = nkv;
      g.qn = Lw.q_norm;
      g.kn = Lw.k_norm;
      g.eps = c.rms_eps;
      g.nblk = rows;
      g.rope = at<float2>(ws, L.rope);
      g.q = q;
      g.kb = kb;
      g.vb = vb;
      if (n_app > 0) {
        g.rope_app = at<float2>(ws, L.ropea);
        g.dst = at<long long>(ws, L.dsta);
        g.kc = const_cast<char*>(elem_ptr(k_cache, l * layer_elems, c.dtype));
        g.vc = const_cast<char*>(elem_ptr(v_cache, l * layer_elems, c.dtype));
      }
      TRY(gemm_fused(g, qctx, ws, L, false));
    } else {
      TRY(gemm(c, ctx, ws, L, Lw.qkv, (nq + 2 * nkv) * d, H, u2a, rows, Y, false, false, s_qkv));
      TRY(launch_qkv_epilogue(c.dtype, Y, rows, B, nq, nkv, d, Lw.q_norm, Lw.k_norm, c.rms_eps, c.rope_theta,
                              ctx_len, new_off, q, kb, vb, ctx));
    }
    // separate: the attention reads the appended K/V, a full dependency on the join
    Ctx jctx = ctx;
    if (forked && !merged && l == 0) {
      if (cudaStreamWaitEvent(ctx.stream, side.join, 0) != cudaSuccess) return DFLASH2_ERR_CUDA;
      jctx.pdl = false;
    }
    TRY(launch_attention(c.dtype, q, kb, vb, elem_ptr(k_cache, l * layer_elems, c.dtype),
                         elem_ptr(v_cache, l * layer_elems, c.dtype), block_table, max_pages, c.page_size, n_pages,
                         ctx_len, new_off, batch, B, nq, nkv, d, max_ctx, c.sliding_window, at<float>(workspace, L.attn),
                         O, jctx));
    TRY(gemm(c, ctx, ws, L, Lw.o, H, nq * d, O, rows, h, true, false, s_o));
    // MLP sublayer: conv around the normed input, gate/up, SiLU*up, down (+= residual)
    if (fused) {
      TRY(launch_conv_prologue(c.dtype, h, nullptr, 0, w->embed, c.vocab, 1.f, Lw.mlp_norm, c.rms_eps, Lw.tapgen_mlp, s_tap_m,
                               batch, B, H, c.conv_group_size, nullptr, u, u2, RopeTab{}, ctx));
    } else {
      TRY(launch_rownorm(c.dtype, h, rows, H, Lw.mlp_norm, c.rms_eps, u, B, 0, ctx));
      if (conv) {
        TRY(gemm(c, ctx, ws, L, Lw.tapgen_mlp, 2 * G, H, u, rows, Y, false, false, s_tap_m));
        TRY(launch_dyn_conv(c.dtype, u, Y, rows, H, c.conv_group_size, B, u2, ctx));
      }
    }
    if (c.dtype == DFLASH2_BF16 && gemm_fusable(2 * I, rows, kEpiSwiglu)) {
      GemmOp g = gemm_op(Lw.gate_up, 2 * I, H, u2, rows, s_gu);  // SiLU(gate) * up fused into the epilogue
      g.epi = kEpiSwiglu;
      g.act = act;
      TRY(gemm_fused(g, ctx, ws, L, false));
    } else {
      TRY(gemm(c, ctx, ws, L, Lw.gate_up, 2 * I, H, u2, rows, Y, false, false, s_gu));
      TRY(launch_act(c.dtype, Y, rows, I, act, ctx));
    }
    TRY(gemm(c, ctx, ws, L, Lw.down, H, I, act, rows, h, true, false, s_down));
  }
  TRY(launch_rownorm(c.dtype, h, rows, H, w->final_norm, c.rms_eps, hn, B, 1, ctx,
                     at<unsigned long long>(workspace, L.thr)));

  TRY(stage_event(2, ctx.stream));
  // (c) lm_head over block positions 1..B-1 with the streaming top-k
  float* lv = at<float>(workspace, L.lv);
  int* li = at<int>(workspace, L.li);
  int n_lists = 0;
  const int nrow = batch * D;
  if (c.dtype == DFLASH2_BF16) {
    GemmOp g;
    std::memset(&g, 0, sizeof(g));
    g.W = w->lm_head;
    g.wscale = sc.lm_head;
    g.M = c.vocab;
    g.K = H;
    g.ldw = H;
    g.X = hn;
    g.N = nrow;
    g.ldx = H;
    g.topk = true;
    g.lists_v = lv;
    g.lists_i = li;
    g.thr = at<unsigned long long>(workspace, L.thr);
    g.debug = debug_logits;
    g.mult = c.output_multiplier;
    g.cap = c.final_logit_softcap;
    TRY(gemm_bf16(g, ctx));
    n_lists = gemm_topk_lists(c.vocab, nrow, H, ctx.nsm, c.dtype);
  } else {
    float* logits = at<float>(workspace, L.logits);
    TRY(gemm(c, ctx, workspace, L, w->lm_head, c.vocab, H, hn, nrow, logits, false));
    TRY(launch_topk_scan(logits, nrow, c.vocab, c.output_multiplier, c.final_logit_softcap, debug_logits, lv, li,
                         &n_lists, ctx));
  }
  TRY(stage_event(3, ctx.stream));
  TRY(launch_topk_merge(lv, li, n_lists, nrow, c.top_k, cand_id, cand_logit, ctx));
  TRY(stage_event(4, ctx.stream));
  return DFLASH2_OK;
}

int dflash2_select_path_ex(const dflash2_config* cfg, const dflash2_weights* w, int batch, const int32_t* anchor,
                           const int32_t* cand_id, const float* cand_logit, const dflash2_draft_opts* opts,
                           int32_t* path, float* path_score, int32_t* n_draft, void* workspace, size_t ws_bytes,
                           void* stream) {
  TRY(check_config(cfg));
  if (!w || !w->embed || !w->sel) return DFLASH2_ERR_INVALID_ARG;
  if (batch <= 0) return DFLASH2_ERR_SHAPE;
  if (!anchor || !cand_id || !cand_logit || !path) return DFLASH2_ERR_INVALID_ARG;
  if (!workspace) return DFLASH2_ERR_WORKSPACE;
  if (cfg->dtype == DFLASH2_FP8W && (!w->scales || !w->scales->sel)) return DFLASH2_ERR_INVALID_ARG;
  const dflash2_config c = act_config(*cfg);
  const Scales sc = scales_of(*cfg, *w);
  const Layout L = plan(c, batch, 0, 0);
  if (ws_bytes < L.total) return DFLASH2_ERR_WORKSPACE;
  Ctx ctx;
  TRY(device_ctx(&ctx, stream, workspace));
  const int D = c.block_size - 1, k = c.top_k, r = c.selector_rank, H = c.hidden;
  void* x = at<char>(workspace, L.selx);
  float* Y = at<float>(workspace, L.Y);
  TRY(launch_sel_gather(c.dtype, anchor, cand_id, batch, D, k, w->embed, c.vocab, H, x, ctx));
  TRY(gemm(c, ctx, workspace, L, w->sel, 2 * r, H, x, batch * (D * k + 1), Y, false, false, sc.sel));
  return launch_viterbi(Y, nullptr, anchor, c.vocab, cand_id, cand_logit, batch, D, k, r, path, path_score, ctx,
                        opts ? opts->n_max : 0, opts ? opts->p_min : 0.f, n_draft);
}

int dflash2_select_path(const dflash2_config* cfg, const dflash2_weights* w, int batch, const int32_t* anchor,
                        const int32_t* cand_id, const float* cand_logit, int32_t* path, float* path_score,
                        void* workspace, size_t ws_bytes, void* stream) {
  return dflash2_select_path_ex(cfg, w, batch, anchor, cand_id, cand_logit, nullptr, path, path_score, nullptr,
                                workspace, ws_bytes, stream);
}

size_t dflash2_selector_table_bytes(const dflash2_config* cfg) {
  if (check_config(cfg) != DFLASH2_OK) return 0;
  return (size_t)cfg->vocab * 2 * cfg->selector_rank * sizeof(float);
}

int dflash2_build_selector_table(const dflash2_config* cfg, const dflash2_weights* w, float* table, void* stream) {
  TRY(check_config(cfg));
  if (!w || !w->embed || !w->sel || !table) return DFLASH2_ERR_INVALID_ARG;
  if (cfg->dtype == DFLASH2_FP8W && (!w->scales || !w->scales->sel)) return DFLASH2_ERR_INVALID_ARG;
  Ctx ctx;
  TRY(device_ctx(&ctx, stream, nullptr));
  const dflash2_config c = act_config(*cfg);
  // table[v][m] = sum_h sel[m][h] E[v][h]: the selector contraction with the
  // whole vocabulary as its activation rows (whole tiles: no workspace)
  GemmOp g = gemm_op(w->sel, 2 * c.selector_rank, c.hidden, w->embed, c.vocab, scales_of(*cfg, *w).sel);
  g.out = table;
  g.ctas = -1;
  if (c.dtype == DFLASH2_BF16) return gemm_bf16(g, ctx);
  return gemm_f32(g, ctx);
}

int dflash2_select_path_table_ex(const dflash2_config* cfg, int batch, const int32_t* anchor,
                                 const int32_t* cand_id, const float* cand_logit, const float* table,
                                 const dflash2_draft_opts* opts, int32_t* path, float* path_score, int32_t* n_draft,
                                 void* workspace, void* stream) {
  TRY(check_config(cfg));
  if (batch <= 0) return DFLASH2_ERR_SHAPE;
  if (!anchor || !cand_id || !cand_logit || !table || !path) return DFLASH2_ERR_INVALID_ARG;
  Ctx ctx;
  TRY(device_ctx(&ctx, stream, workspace));
  const dflash2_config& c = *cfg;
  return launch_viterbi(nullptr, table, anchor, c.vocab, cand_id, cand_logit, batch, c.block_size - 1, c.top_k,
                        c.selector_rank, path, path_score, ctx, opts ? opts->n_max : 0, opts ? opts->p_min : 0.f,
                        n_draft);
}

int dflash2_select_top1(const dflash2_config* cfg, int batch, const int32_t* cand_id, const float* cand_logit,
                        const dflash2_draft_opts* opts, int32_t* path, float* path_score, int32_t* n_draft,
                        void* workspace, void* stream) {
  TRY(check_config(cfg));
  if (batch <= 0) return DFLASH2_ERR_SHAPE;
  if (!cand_id || !cand_logit || !path) return DFLASH2_ERR_INVALID_ARG;
  Ctx ctx;
  TRY(device_ctx(&ctx, stream, workspace));
  const dflash2_config& c = *cfg;
  return launch_viterbi(nullptr, nullptr, nullptr, c.vocab, cand_id, cand_logit, batch, c.block_size - 1, c.top_k,
                        c.selector_rank, path, path_score, ctx, opts ? opts->n_max : 0, opts ? opts->p_min : 0.f,
                        n_draft);
}

int dflash2_select_path_table(const dflash2_config* cfg, int batch, const int32_t* anchor, const int32_t* cand_id,
                              const float* cand_logit, const float* table, int32_t* path, float* path_score,
                              void* workspace, void* stream) {
  return dflash2_select_path_table_ex(cfg, batch, anchor, cand_id, cand_logit, table, nullptr, path, path_score,
                                      nullptr, workspace, stream);
}

int dflash2_verify_accept(int batch, int block_size, const int32_t* path, const int32_t* target,
                          int32_t* accept_len, int32_t* out_tok, int32_t* n_out, int32_t* next_anchor,
                          int32_t* seq_len, int64_t* counters, void* stream) {
  if (block_size < 2 || block_size > 32) return DFLASH2_ERR_BLOCK_SIZE;
  if (batch <= 0) return DFLASH2_ERR_SHAPE;
  if (!path || !target || !accept_len || !out_tok || !n_out || !next_anchor) return DFLASH2_ERR_INVALID_ARG;
  return launch_verify(batch, block_size, path, nullptr, target, accept_len, out_tok, n_out, next_anchor, seq_len,
                       counters, static_cast<cudaStream_t>(stream));
}

int dflash2_verify_accept_ex(int batch, int block_size, const int32_t* path, const int32_t* n_draft,
                             const int32_t* target, int32_t* accept_len, int32_t* out_tok, int32_t* n_out,
                             int32_t* next_anchor, int32_t* seq_len, int64_t* counters, void* stream) {
  if (block_size < 2 || block_size > 32) return DFLASH2_ERR_BLOCK_SIZE;
  if (batch <= 0) return DFLASH2_ERR_SHAPE;
  if (!path || !target || !accept_len || !out_tok || !n_out || !next_anchor) return DFLASH2_ERR_INVALID_ARG;
  return launch_verify(batch, block_size, path, n_draft, target, accept_len, out_tok, n_out, next_anchor, seq_len,
                       counters, static_cast<cudaStream_t>(stream));
}

int dflash2_verify_sampled(int batch, int block_size, int vocab, const int32_t* path, const int32_t* n_draft,
                           const float* target_prob, const float* u_accept, const float* u_sample,
                           int32_t* accept_len, int32_t* out_tok, int32_t* n_out, int32_t* next_anchor,
                           int32_t* seq_len, int64_t* counters, void* stream) {
  if (block_size < 2 || block_size > 32) return DFLASH2_ERR_BLOCK_SIZE;
  if (batch <= 0 || vocab < 2) return DFLASH2_ERR_SHAPE;
  if (!path || !target_prob || !u_accept || !u_sample || !accept_len || !out_tok || !n_out || !next_anchor)
    return DFLASH2_ERR_INVALID_ARG;
  return launch_verify_sampled(batch, block_size, vocab, path, n_draft, target_prob, u_accept, u_sample, accept_len,
                               out_tok, n_out, next_anchor, seq_len, counters, static_cast<cudaStream_t>(stream));
}

int dflash2_read_device_status(void* workspace, size_t ws_bytes, void* stream) {
  if (!workspace || ws_bytes < 256) return DFLASH2_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  unsigned v = 0;
  if (cudaMemcpyAsync(&v, workspace, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if (cudaMemsetAsync(workspace, 0, sizeof(v), st) != cudaSuccess) return DFLASH2_ERR_CUDA;
  if (cudaStreamSynchronize(st) != cudaSuccess) return DFLASH2_ERR_CUDA;
  return (int)(v & 0x7fffffffu);
}

}  // extern "C"
