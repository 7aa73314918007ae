// Host-side interfaces between the C ABI layer and the kernel launchers.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dflash2.h"

namespace df2 {

struct Ctx {
  cudaStream_t stream;
  unsigned* status;  // device status word (workspace offset 0)
  int nsm;           // SMs of the current device
  bool pdl = true;   // launch with programmatic stream serialization
  int prio = 0;      // launch priority (0: the stream's own; lower numbers run first)
};

// One dense contraction out[n][m] = sum_k W[m][k] * X[n][k]  (swap-AB: the
// weight rows stream along the MMA M axis, the few activation rows form N).
struct GemmOp {
  const void* W;  // [M, K] row stride ldw elements (bf16, or e4m3 bytes with wscale)
  int M, K, ldw;
  const float* wscale;  // nullable [M]: W is fp8 e4m3 and row m is scaled by wscale[m]
  const void* X;  // [N, K] row stride ldx elements
  int N, ldx;
  // plain epilogue: out[n][m] fp32 (ld = M), stored or, with accumulate,
  // added to.  The bf16 path splits the work stream-K style over `ctas`
  // CTAs (0: one per SM; -1: whole tiles, no pieces); tiles shared between
  // CTAs go through `partial` (gemm_partial_bytes) and `counters`
  // (kMaxSM ints, zero on entry and on exit).
  float* out;
  int ctas;
  float* partial;
  int* counters;
  bool accumulate;
  // top-k epilogue (lm_head): per-CTA sorted lists of KMAX entries
  bool topk;
  float* lists_v;  // [n_lists][N][KMAX]
  int* lists_i;
  unsigned long long* thr;  // [N][kTopkSlots] bound slots shared by the CTAs, zero at launch
  float* debug;  // nullable [N][M] logits after the transform
  float mult, cap;
  // fused epilogues (bf16 path, activation tiles of at most 64 rows; see
  // gemm_fusable): 0 = plain fp32 out; kEpiSwiglu = gate/up rows [0, M/2) and
  // [M/2, M) -> act [N][M/2] bf16 = SiLU(gate) * up; kEpiHeads = per-head
  // RMSNorm + RoPE of q/k heads and copy of v heads, to q/kb/vb (block rows)
  // or to the paged cache (appended rows).
  int epi;
  void* act;
  int hd, n_qh, n_kh;
  const void* qn;
  const void* kn;
  float eps;
  int nblk;                // columns [0, nblk): block rows -> q/kb/vb; [nblk, N): appended rows -> cache
  const float2* rope;      // [nblk][hd/2] (cos, sin) per block column (RopeTab::cs)
  const float2* rope_app;  // [N - nblk][hd/2] per appended column
  const long long* dst;    // [N - nblk] paged-cache offsets of the appended rows (RopeTab::dst)
  void *q, *kb, *vb, *kc, *vc;
};
constexpr int kEpiSwiglu = 2, kEpiHeads = 3;
constexpr int kTopkSlots = 16;  // shared top-k bound slots per lm_head row

// Whether an M x N contraction can take a fused epilogue (activation tiles of
// at most 64 rows; the gate/up pairing also needs M % 128 == 0).
bool gemm_fusable(int M, int N, int epi);

// Bytes of stream-K partial pieces an M x N contraction can need (any SM count).
size_t gemm_partial_bytes(int M, int N);
// Number of partial top-k lists a top-k GEMM of this shape writes.
int gemm_topk_lists(int M, int N, int K, int nsm, int dtype);
// Upper bound of the above over every SM count this library accepts.
int gemm_max_lists();
constexpr int kMaxSM = 256;  // CTAs of a stream-K launch, and its counter array length
// SMs left to the fused embedding prologue while the side stream's feature
// contraction runs beside it (the contraction takes the rest).
constexpr int kForkPrologueSMs = 32;
// SMs the block's first QKV contraction leaves to the side stream's K/V
// contraction when the two run side by side (0: the QKV takes every SM).
constexpr int kForkKvSMs = 32;
// Whether the side stream's stage (a) kernels launch at the device's
// greatest priority, so that the block scheduler places their CTAs before
// the block branch's when SMs free up.
constexpr bool kSidePriority = true;
// Whether contractions whose tiles x K slices fill the SMs run as cluster
// split-K (slices summed in distributed shared memory) instead of stream-K.
constexpr bool kClusterSplit = true;

// Host-side count of kernel launches (instrumentation).
void count_launch(int n = 1);

// Launches `kern` on c.stream, counting the launch.  With c.pdl the launch
// uses programmatic stream serialization: it may start while the previous
// kernel of the stream drains.  Every kernel of this library calls pdl_wait()
// (griddepcontrol.wait) before it touches memory that an earlier kernel
// writes, so only prologues (and, in the GEMM, the weight stream, which
// nothing on the stream writes) overlap.  The first kernel after a
// cross-stream event wait is launched with c.pdl = false: its dependency on
// the other stream must be a full one.  cluster_x > 1 groups the CTAs into
// thread-block clusters of that many CTAs along x.
template <typename... KArgs, typename... Args>
inline int launch_kx(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, const Ctx& c, int cluster_x,
                     Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute at[3];
  int n = 0;
  if (c.prio != 0) {
    at[n].id = cudaLaunchAttributePriority;
    at[n].val.priority = c.prio;
    ++n;
  }
  if (c.pdl) {
    at[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    at[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  if (cluster_x > 1) {
    at[n].id = cudaLaunchAttributeClusterDimension;
    at[n].val.clusterDim.x = cluster_x;
    at[n].val.clusterDim.y = 1;
    at[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = at;
  cfg.numAttrs = n;
  count_launch();
  return cudaLaunchKernelEx(&cfg, kern, args...) == cudaSuccess ? DFLASH2_OK : DFLASH2_ERR_CUDA;
}

template <typename... KArgs, typename... Args>
inline int launch_k(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, const Ctx& c, Args... args) {
  return launch_kx(kern, grid, block, smem, c, 1, args...);
}

// Byte offsets in the workspace of the draft step's intermediates
// {f, h, u, u2, q, kb, vb, O, act, hn} for a call of these sizes (test hook).
int workspace_offsets(const dflash2_config* c, int batch, int n_new, int max_ctx, size_t* out, int n);

int gemm_bf16(const GemmOp& g, const Ctx& c);  // tcgen05 + TMA (sm_103a)
// 2-D bf16 tensor map over rows x cols (row stride ld_elems elements), box of
// box_cols x box_rows, no swizzle, zero fill past the edges (the attention's
// page loads); DFLASH2_ERR_SHAPE for unaligned bases or strides.
int make_rows_map(CUtensorMap* map, const void* base, long long rows, int cols, long long ld_elems, int box_cols,
                  int box_rows);
// The same view with a box of 64 columns x box_rows rows and the 128-byte
// swizzle (tiles that tcgen05.mma reads as K-major or MN-major operands).
int make_sw128_map(CUtensorMap* map, const void* base, long long rows, int cols, long long ld_elems, int box_rows);
// Schedule bits of the last dflash2_draft_step call (test hook)
enum {
  kSchedFusedPrologue = 1,  // sublayer prologue fused (norm + tap logits + conv)
  kSchedSplitSMs = 2,       // embedding prologue beside the feature contraction on split SMs
  kSchedFusedQKV = 4,       // QKV contraction with the q/k-norm + RoPE epilogue
  kSchedKvBesideQKV = 8,    // layer 0's context K/V contraction on the SMs the QKV leaves free
  kSchedMerged = 16,        // appended rows ride in the QKV contractions
};
int draft_last_schedule();
int gemm_last_grid();  // CTAs of this thread's last gemm_bf16 launch
void gemm_force_csplit(int cs);  // test hook: cluster split-K of cs slices where it applies (0 = off)
int gemm_f32(const GemmOp& g, const Ctx& c);   // exact fp32 FMA, SIMT

// Tiles (m_tiles * n_tiles) of a contraction, the size of its counter array.
int gemm_tiles(int M, int N);

// Inverse frequencies theta^(-2i/d) of the rotary pairs i < d/2, in double,
// computed once on the host and passed to the kernels that form angles.
struct RopeFreq {
  double inv[64];
};
RopeFreq rope_freq(int d, float theta);

// RoPE angles (and, for appended rows, paged-cache destinations) that the
// row kernels running ahead of a fused heads epilogue store for it: the
// block rows' table comes from the first sublayer prologue (or the embedding
// kernel), the appended rows' from the feature norm.
struct RopeTab {
  float2* cs;       // [rows][d/2] (cos, sin) of pair i at the row's position; nullptr: not wanted
  long long* dst;   // appended rows: element offset of the row in the paged cache (-1: invalid)
  int d;
  RopeFreq freq;
  const int32_t* ctx_len;
  const int32_t* new_off;
  int batch;
  const int32_t* block_table;  // appended rows only
  int max_pages, page_size, n_pages, nkv;
};

// element-wise / row kernels (elementwise.cu); T = float or bf16 by dtype.
// Y is the producing contraction's final fp32 output, row-major [rows][width].
int launch_rows_feature_norm(int dtype, const float* Y, int rows, int H, const void* gamma, float eps, void* f_out,
                             const RopeTab& rt, const Ctx& c);
int launch_kv_append(int dtype, const float* Y, int rows, int nkv, int d, const void* k_norm, float eps, float theta,
                     const int32_t* ctx_len, const int32_t* new_off, int batch, const int32_t* block_table,
                     int max_pages, int page_size, int n_pages, void* kc, void* vc, const Ctx& c);
int launch_embed_norm(int dtype, const int32_t* anchor, int mask_id, int batch, int B, const void* embed, int V, int H,
                      float scale, const void* gamma, float eps, float* h_out, void* u_out, const RopeTab& rt,
                      const Ctx& c);
int launch_rownorm(int dtype, const float* h, int rows, int H, const void* gamma, float eps, void* u_out, int B,
                   int skip_anchor, const Ctx& c, unsigned long long* zero_key = nullptr);
int launch_dyn_conv(int dtype, const void* u, const float* Y, int rows, int H, int group_size, int B, void* u2_out,
                    const Ctx& c);
int launch_qkv_epilogue(int dtype, const float* Y, int rows, int B, int nq, int nkv, int d, const void* q_norm,
                        const void* k_norm, float eps, float theta, const int32_t* ctx_len, const int32_t* new_off,
                        void* q, void* kb, void* vb, const Ctx& c);
int launch_act(int dtype, const float* Y, int rows, int I, void* act, const Ctx& c);
// Fused sublayer prologue (RMSNorm, tap logits, two-tap conv) for each
// sequence's B rows: from the residual h_in, or, with h_in == nullptr, from
// the block embedding [anchor, mask...] (then h_out receives it).  Writes u
// (normed, as stored) and u2 (after the conv).  conv_prologue_fits says
// whether the B rows and the CTA's tap rows fit its shared memory;
// otherwise the caller runs rownorm + tap GEMM + dyn_conv.
bool conv_prologue_fits(int dtype, int batch, int B, int H, int G, int nsm);
// w_tap: [2G, H] of dtype, or (tap_scale != nullptr, bf16 activations) e4m3
// codes whose row r is scaled by tap_scale[r].
int launch_conv_prologue(int dtype, const float* h_in, const int32_t* anchor, int mask_id, const void* embed, int V,
                         float scale, const void* gamma, float eps, const void* w_tap, const float* tap_scale,
                         int batch, int B, int H, int group_size, float* h_out, void* u_out, void* u2_out,
                         const RopeTab& rt, const Ctx& c);

// attention (attention.cu)
int launch_attention(int dtype, const void* q, const void* kb, const void* vb, const void* kc, const void* vc,
                     const int32_t* block_table, int max_pages, int page_size, int n_pages,
                     const int32_t* ctx_len, const int32_t* new_off, int batch, int B, int nq, int nkv, int d,
                     int max_ctx, int window, float* part, void* o_out, const Ctx& c);
size_t attn_part_bytes(int batch, int B, int nq, int nkv, int d, int max_ctx);
// CTAs per cluster (key chunks per (kv head, sequence)) of the cluster kernels
int attn_cluster_ctas(int max_ctx, int B, int batch, int nkv, int nsm);
// test hook: 0 = the library's choice, 1 = the mma.sync cluster kernel,
// 2 = the tcgen05 kernel wherever it applies
void attention_force_mode(int mode);
int attention_last_kernel();  // test hook: 1 mma.sync cluster, 2 tcgen05, 3 SIMT (0 before any launch)
// tcgen05 attention (attention_tc.cu): bf16 storage, head dimension 128,
// 16-key pages, at most 80 query rows per kv head
bool attention_tc_fits(int dtype, int d, int page_size, int R);
int launch_attention_tc(const void* q, const void* kb, const void* vb, const void* kc, const void* vc,
                        const int32_t* block_table, int max_pages, int page_size, int n_pages,
                        const int32_t* ctx_len, const int32_t* new_off, int batch, int B, int nq, int nkv,
                        int max_ctx, int window, void* o, const Ctx& c);

// top-k (topk.cu)
int launch_topk_scan(const float* logits, int rows, int V, float mult, float cap, float* debug, float* lists_v,
                     int* lists_i, int* n_lists, const Ctx& c);
int topk_scan_lists(int V);
int launch_topk_merge(const float* lists_v, const int* lists_i, int n_lists, int rows, int k, int32_t* cand_id,
                      float* cand_logit, const Ctx& c);

// selector and verify (selector.cu, verify.cu)
int launch_sel_gather(int dtype, const int32_t* anchor, const int32_t* cand_id, int batch, int D, int k,
                      const void* embed, int V, int H, void* x_out, const Ctx& c);
// Y: per-step factors [batch][D*k+1][2r]; or Y null and table [V][2r]
// (factors of every token, gathered by the kernel).
// Drafting knobs: the walk covers positions 1..n_max (<= D) and the path is
// cut before the first chosen transition with probability < p_min; n_draft
// (nullable) receives the drafts kept.  launch_viterbi = n_max D, no cut.
int launch_viterbi(const float* Y, const float* table, const int32_t* anchor, int V, const int32_t* cand_id,
                   const float* cand_logit, int batch, int D, int k, int r, int32_t* path, float* path_score,
                   const Ctx& c, int n_max = 0, float p_min = 0.f, int32_t* n_draft = nullptr);
size_t viterbi_smem_bytes(int D, int k, int r);
int launch_verify_sampled(int batch, int B, int V, const int32_t* path, const int32_t* n_draft, const float* prob,
                          const float* u_accept, const float* u_sample, int32_t* accept_len, int32_t* out_tok,
                          int32_t* n_out, int32_t* next_anchor, int32_t* seq_len, int64_t* counters,
                          cudaStream_t st);
// n_draft: nullable [batch] drafts kept per sequence (B-1 when null).
int launch_verify(int batch, int B, const int32_t* path, const int32_t* n_draft, const int32_t* target,
                  int32_t* accept_len, int32_t* out_tok, int32_t* n_out, int32_t* next_anchor, int32_t* seq_len,
                  int64_t* counters, cudaStream_t st);

}  // namespace df2
