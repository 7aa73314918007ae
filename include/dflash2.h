/*
 * dflash2.h — C ABI of the DFlash2 block-parallel draft step on GB300 (sm_103a).
 *
 * One speculative step of a batch of independent sequences is
 *
 *   dflash2_draft_step     stages (a)-(c): feature projection + context K/V
 *                          append, one non-causal block forward, lm_head with
 *                          a fused streaming top-k (the candidate lattice);
 *   dflash2_select_path    stage (d): pairwise low-rank selector (factors +
 *                          Viterbi);
 *   dflash2_verify_accept  stage (d): greedy verify, accept, rollback and
 *                          counters.
 *
 * dflash2_append_context runs stage (a) alone (e.g. to prefill a prompt).
 *
 * Sources, cited by page title and section:
 *   "Train a DFlash Drafter for Speculative Decoding" — "What is DFlash?",
 *     "Variants", "Objective", "Data", "Key Config Fields";
 *   "DFlash speculative decoding with vLLM" — "Requirements",
 *     "DFlash2 inference", "Validation";
 *   "DFlash2 Speculative Decoding" (llama-cpp-python wiki) — "Prerequisites",
 *     "Configuration Notes";
 *   "DFlash2 Speculative Decoding | NVIDIA NIM for Alpamayo Documentation" —
 *     "Observe Acceptance", "Bring Your Own DFlash2 Head".
 *
 * Conventions shared by every entry point
 *   - Every array argument is a DEVICE pointer owned by the caller unless it
 *     is documented as a host pointer (the config and weight structs are host
 *     structs whose members are device pointers).  The library allocates no
 *     device memory; scratch lives in the caller's workspace.
 *   - Row-major layouts; "[a, b]" means b is the contiguous dimension.
 *   - Calls are asynchronous on the given stream (a cudaStream_t passed as
 *     void*; NULL is the legacy default stream) and launch only kernels, so a
 *     step can be captured in a CUDA graph.
 *   - Return value: DFLASH2_OK or a negative status; a non-OK status means no
 *     kernel was launched by that call (argument checks run before any
 *     launch), except DFLASH2_ERR_CUDA, which reports a failed launch.
 *   - Device-side checks (a page id outside [0, n_pages), a token id outside
 *     [0, vocab), a bounded wait that ran out) do not fault: the kernel skips
 *     the access and records a code in the workspace's status word, read with
 *     dflash2_read_device_status.
 *   - The device status word is the first 4 bytes of the workspace: zero the
 *     workspace once before its first use.
 *   - No C++ exception crosses this interface.
 */
#ifndef DFLASH2_H
#define DFLASH2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- status */
#define DFLASH2_OK                    0
#define DFLASH2_ERR_INVALID_ARG      -1  /* null pointer, negative size, bad enum */
#define DFLASH2_ERR_SHAPE            -2  /* inconsistent or unsupported dimensions */
#define DFLASH2_ERR_BLOCK_SIZE       -3  /* block_size != drafts + 1, or out of range */
#define DFLASH2_ERR_DTYPE            -4  /* unsupported dtype */
#define DFLASH2_ERR_WORKSPACE        -5  /* workspace null or smaller than required */
#define DFLASH2_ERR_CUDA             -6  /* a CUDA runtime/driver call failed */
#define DFLASH2_ERR_UNSUPPORTED      -7  /* valid request this library does not serve (e.g. not sm_103a) */

/* device status word bits (dflash2_read_device_status) */
#define DFLASH2_DEV_BAD_PAGE        0x1  /* block_table entry outside [0, n_pages) */
#define DFLASH2_DEV_BAD_TOKEN       0x2  /* token id outside [0, vocab) */
#define DFLASH2_DEV_WAIT_TIMEOUT    0x4  /* a bounded pipeline wait gave up */
#define DFLASH2_DEV_BAD_LENGTH      0x8  /* a context length beyond the block table */

/* ---------------------------------------------------------------- types */
#define DFLASH2_F32   0  /* float32 weights, activations and cache */
#define DFLASH2_BF16  1  /* bfloat16 weights, activations and cache; fp32 accumulation */
#define DFLASH2_FP8W  2  /* fp8 e4m3 linear weights with fp32 per-output-channel scales
                            (dflash2_scales); bfloat16 embed, norm gains, activations and
                            cache; fp32 accumulation.  A weight element is q * scale[row]:
                            the contractions run on the exact bf16 value of q and apply
                            the row's scale to the fp32 result. */

/*
 * Draft model configuration ("Key Config Fields"; dflash_config of
 * "DFlash2 inference").  Host struct.
 *   hidden                 H, draft (and target embedding) width
 *   n_q_heads, n_kv_heads  draft attention heads (n_q_heads % n_kv_heads == 0)
 *   head_dim               d (64 or 128)
 *   intermediate           I, MLP width
 *   vocab                  V, shared embed_tokens / lm_head rows
 *   n_layers               draft decoder layers (>= 1)
 *   n_taps                 T, number of target layers tapped (target_layer_ids)
 *   block_size             B = 1 anchor + (B-1) drafts, 2..32
 *   conv_kernel_size       taps of the in-block convolution: 2 (DFlash 2), or 0 for
 *                          DFlash (v1): no convolution, tapgen_* unused ("Variants")
 *   conv_group_size        channels sharing one set of dynamic taps; H % it == 0
 *   top_k                  selector_top_k, 1..16
 *   selector_rank          r, 1..128
 *   page_size              context KV page length (tokens per page)
 *   mask_token_id          token filling block slots 1..B-1 ("Data" note)
 *   dtype                  DFLASH2_F32, DFLASH2_BF16 or DFLASH2_FP8W
 *   rms_eps                RMSNorm epsilon
 *   rope_theta             rotary base
 *   input_embedding_scale  multiplies the embedded block (1 = identity)
 *   output_multiplier      multiplies the logits (1 = identity)
 *   final_logit_softcap    cap*tanh(z/cap) when > 0, on the multiplied logits
 *                          (0 = off)
 *   sliding_window         draft_sliding_window ("Key Config Fields"): when > 0 the
 *                          block reads only the last sliding_window context
 *                          positions (and all its own); 0 = the whole prefix
 */
typedef struct dflash2_config {
    int hidden, n_q_heads, n_kv_heads, head_dim, intermediate, vocab;
    int n_layers, n_taps, block_size, conv_kernel_size, conv_group_size;
    int top_k, selector_rank, page_size, mask_token_id, dtype;
    float rms_eps, rope_theta, input_embedding_scale, output_multiplier,
          final_logit_softcap;
    int sliding_window;
} dflash2_config;

/*
 * Weights of one draft layer (device pointers, element type = cfg.dtype;
 * with DFLASH2_FP8W the matrices are e4m3 bytes and the norm gains bf16).
 * G = hidden / conv_group_size.  Matrices are [out_features, in_features].
 *   attn_norm    [H]                      RMSNorm gain before attention
 *   tapgen_attn  [2G, H]                  conv tap generator, row 2g+j = tap j of group g
 *   qkv          [(nq + 2 nkv) d, H]      W_q rows, then W_k rows, then W_v rows
 *   q_norm       [d]                      per-head RMSNorm gain of q
 *   k_norm       [d]                      per-head RMSNorm gain of k (block and context)
 *   o            [H, nq d]
 *   mlp_norm     [H]
 *   tapgen_mlp   [2G, H]
 *   gate_up      [2I, H]                  W_gate rows, then W_up rows
 *   down         [H, I]
 * Base addresses must be 16-byte aligned.
 */
typedef struct dflash2_layer_weights {
    const void *attn_norm, *tapgen_attn, *qkv, *q_norm, *k_norm, *o;
    const void *mlp_norm, *tapgen_mlp, *gate_up, *down;
} dflash2_layer_weights;

/*
 * DFLASH2_FP8W only: the fp32 per-output-channel scales of the e4m3 matrices
 * (device pointers; one float per matrix row, in the row order of the
 * matrix: qkv scales are q rows, then k rows, then v rows).
 */
typedef struct dflash2_layer_scales {
    const float *tapgen_attn, *qkv, *o, *tapgen_mlp, *gate_up, *down;
} dflash2_layer_scales;

/* `layers` is a HOST array of n_layers entries. */
typedef struct dflash2_scales {
    const float *lm_head, *fc, *sel;
    const dflash2_layer_scales *layers;
} dflash2_scales;

/*
 * All draft weights.  Host struct of device pointers; `layers` is a HOST
 * array of n_layers entries.
 *   embed        [V, H]     the target's frozen embed_tokens (shared)
 *   lm_head      [V, H]     the target's frozen lm_head (shared)
 *   fc           [H, T H]   feature projection of the concatenated taps
 *   hidden_norm  [H]        RMSNorm gain after the projection
 *   final_norm   [H]        RMSNorm gain before the lm_head
 *   sel          [2r, H]    selector factors: rows 0..r-1 = W_a (predecessor),
 *                           rows r..2r-1 = W_b (candidate)
 * With DFLASH2_FP8W, lm_head, fc, sel and the layer matrices are e4m3 bytes
 * with the row scales of `scales`; embed and the norm gains are bf16.
 */
typedef struct dflash2_weights {
    const void *embed, *lm_head, *fc, *hidden_norm, *final_norm, *sel;
    const dflash2_layer_weights *layers;
    const dflash2_scales *scales;  /* host pointer; DFLASH2_FP8W only (NULL otherwise) */
} dflash2_weights;

/*
 * Paged context K/V cache (device, caller-owned, element type = cfg.dtype):
 *   k_cache, v_cache  [n_layers, n_pages, page_size, n_kv_heads, head_dim]
 *   block_table       [batch, max_pages] int32: logical page p of sequence s
 *                     lives in physical page block_table[s*max_pages + p].
 * The cache is append-only and holds committed positions only: keys are
 * stored after k_norm and RoPE at their absolute positions.
 */

/* ------------------------------------------------------------- functions */

/* Human-readable text of a status code (static string, never NULL). */
const char *dflash2_status_string(int status);

/* Library ABI version (major*10000 + minor*100 + patch). */
int dflash2_version(void);

/*
 * Checks a configuration against what this library serves.  Returns
 * DFLASH2_OK, DFLASH2_ERR_INVALID_ARG (null), DFLASH2_ERR_SHAPE,
 * DFLASH2_ERR_BLOCK_SIZE or DFLASH2_ERR_DTYPE.  Host only, no CUDA call.
 */
int dflash2_validate_config(const dflash2_config *cfg);

/*
 * Bytes of workspace the entry points need for at most `max_batch`
 * sequences, `max_new_rows` appended context rows per call (sum over the
 * batch) and contexts of at most `max_ctx` positions (the block-table
 * capacity max_pages*page_size).  Returns 0 for an invalid config.
 * Host only.  One workspace may serve all entry points of a step, used one
 * call at a time on one stream.
 */
size_t dflash2_workspace_size(const dflash2_config *cfg, int max_batch,
                              int max_new_rows, int max_ctx);

/*
 * Stage (a): feature projection and context K/V append.
 * "What is DFlash?": the draft reads hidden states tapped from the frozen
 * target at target_layer_ids, mapped by a trained projection.
 *   n_new      host int, total appended rows (sum over the batch), >= 0
 *   new_taps   [n_new, T*H] target taps of the newly committed positions,
 *              concatenated in target_layer_ids order, rows grouped by
 *              sequence in batch order
 *   new_off    [batch+1] int32 row offsets of each sequence into new_taps
 *              (new_off[0] = 0, new_off[batch] = n_new)
 *   ctx_len    [batch] int32 committed context positions BEFORE the append;
 *              sequence s gets positions ctx_len[s] .. ctx_len[s]+n_s-1.
 *              Not modified.
 * Requires ctx_len[s] + n_s <= max_pages*page_size (else the rows are
 * skipped and DFLASH2_DEV_BAD_LENGTH is recorded).
 */
int dflash2_append_context(const dflash2_config *cfg, const dflash2_weights *w,
                           void *k_cache, void *v_cache, int n_pages,
                           const int32_t *block_table, int max_pages,
                           int batch, const int32_t *ctx_len,
                           int n_new, const void *new_taps, const int32_t *new_off,
                           void *workspace, size_t ws_bytes, void *stream);

/*
 * Stages (a)-(c): append (as dflash2_append_context, n_new may be 0), then
 * one non-causal forward over the block [anchor, MASK x (B-1)] of every
 * sequence ("What is DFlash?"; the DFlash 2 convolution of "Variants"), then
 * the shared lm_head over block positions 1..B-1 and the top-k candidates
 * ("Key Config Fields": selector_top_k).
 *   anchor      [batch] int32, the real token at block position 0; it sits at
 *               position ctx_len[s] + n_s (the context length after the append)
 *   cand_id     [batch, B-1, top_k] int32 out: candidate token ids, best first
 *   cand_logit  [batch, B-1, top_k] float out: their logits (after the
 *               output multiplier and softcap)
 *   debug_logits  nullable [batch, B-1, V] float out: every logit of the
 *               block positions, for parity checks (costs a full write)
 * Candidates are ordered by logit descending, equal logits by smaller id.
 */
int dflash2_draft_step(const dflash2_config *cfg, const dflash2_weights *w,
                       void *k_cache, void *v_cache, int n_pages,
                       const int32_t *block_table, int max_pages,
                       int batch, const int32_t *ctx_len,
                       int n_new, const void *new_taps, const int32_t *new_off,
                       const int32_t *anchor,
                       int32_t *cand_id, float *cand_logit, float *debug_logits,
                       void *workspace, size_t ws_bytes, void *stream);

/*
 * Stage (d1): the DFlash 2 pairwise path selector ("Variants": it walks one
 * coherent path through each position's top-k candidates; "Key Config
 * Fields": selector_rank is its width).  With A = W_a E[tok], Bf = W_b E[tok]:
 *   S_i(p, j) = cand_logit[i][j] + <A[prev_p], Bf[cand_id[i][j]]>,
 *   T_i(p, j) = S_i(p, j) - logsumexp_j' S_i(p, j'),
 * prev of position 1 = the anchor; the path maximises sum_i T_i (Viterbi;
 * ties to the smaller predecessor index, then the smaller final index).
 *   path        [batch, B-1] int32 out: chosen token per draft position
 *   path_score  nullable [batch] float out: the path's summed log-probability
 */
int dflash2_select_path(const dflash2_config *cfg, const dflash2_weights *w,
                        int batch, const int32_t *anchor,
                        const int32_t *cand_id, const float *cand_logit,
                        int32_t *path, float *path_score,
                        void *workspace, size_t ws_bytes, void *stream);

/*
 * dflash2_select_path without a workspace, for callers that cannot allocate
 * device memory: code running inside a custom device allocator's callbacks,
 * or inside a host runtime or plugin interface that owns all device memory
 * and hands the library only its inputs and outputs.  The pages have no
 * counterpart of this entry point; it exists only for such callers.
 *
 * Same arguments, results and return codes as dflash2_select_path, minus the
 * workspace.  Device-side flags (DFLASH2_DEV_BAD_TOKEN for a candidate or
 * anchor id outside [0, vocab), DFLASH2_DEV_WAIT_TIMEOUT) land in the fixed
 * array's own status word, which the next call clears: read them with
 * dflash2_select_path_static_read_status before the next call.  Its scratch is one fixed device array inside the library
 * (dflash2_select_path_static_capacity() bytes, 8 MiB), which every GPU that
 * loads the library keeps until the process exits.  A call whose batch needs
 * more scratch than that returns DFLASH2_ERR_WORKSPACE without launching
 * anything (at the Qwen3-8B selector shape, hidden 4096, 7 drafts, top-16,
 * rank 64, the limit is 8 sequences per call).  The call allocates nothing
 * and calls no allocating library routine.
 *
 * The first call on each device looks up the array's device address
 * (cudaGetSymbolAddress, with that device current); make that first call
 * before capturing a stream into a CUDA graph.  All calls share the one
 * array: calls that overlap on the GPU (different streams or threads) race
 * and must not be issued; calls ordered on one stream are safe.  Each call
 * clears the part of the array that must start at zero.
 */
int dflash2_select_path_static(const dflash2_config *cfg, const dflash2_weights *w, int batch,
                               const int32_t *anchor, const int32_t *cand_id, const float *cand_logit,
                               int32_t *path, float *path_score, void *stream);

/* Bytes of the fixed scratch array dflash2_select_path_static uses. */
size_t dflash2_select_path_static_capacity(void);

/*
 * Device status word of the last dflash2_select_path_static call on the
 * current device: a bitwise OR of DFLASH2_DEV_* codes (>= 0), read after the
 * work already queued on `stream` and then cleared.  Synchronises `stream`.
 * Returns DFLASH2_ERR_CUDA on a failed copy or a failed address lookup.
 * Allocates nothing.
 */
int dflash2_select_path_static_read_status(void *stream);

/*
 * The selector's factors of a token depend on nothing but the frozen
 * embedding and W_sel, so they can be computed once for the whole
 * vocabulary and looked up at every step instead of gathered and
 * contracted per step.  The table is
 *   table[v][0:r]  = W_a E[v],   table[v][r:2r] = W_b E[v]     (fp32)
 * for v = 0..vocab-1, row-major [vocab, 2r] (selector_rank = r), computed
 * with the same contraction (cfg.dtype inputs, fp32 accumulation) the
 * per-step selector uses.
 *
 * dflash2_selector_table_bytes: bytes of the table (vocab * 2r * 4), 0 for
 *   an invalid config.  Host only.
 * dflash2_build_selector_table: fills `table` (device, caller-owned,
 *   16-byte aligned) on `stream`; rebuild it whenever embed or sel change.
 *   Needs no workspace.  Returns DFLASH2_OK, DFLASH2_ERR_INVALID_ARG (null
 *   config, weights or table), a config error, or DFLASH2_ERR_CUDA.
 */
size_t dflash2_selector_table_bytes(const dflash2_config *cfg);
int dflash2_build_selector_table(const dflash2_config *cfg, const dflash2_weights *w, float *table,
                                 void *stream);

/*
 * dflash2_select_path on a factor table from dflash2_build_selector_table:
 * same definition, outputs, tie rules and status codes, in one kernel per
 * call (one CTA per sequence).  The factors of each sequence's anchor and
 * candidates are rows of `table`; a token outside [0, vocab) gets zero
 * factors and, when `workspace` is given, sets DFLASH2_DEV_BAD_TOKEN in its
 * device status word (dflash2_read_device_status).  `workspace` is nullable:
 * the call needs no scratch.
 */
int dflash2_select_path_table(const dflash2_config *cfg, int batch, const int32_t *anchor,
                              const int32_t *cand_id, const float *cand_logit, const float *table,
                              int32_t *path, float *path_score, void *workspace, void *stream);

/*
 * Drafting knobs ("DFlash2 Speculative Decoding" (llama-cpp-python wiki),
 * "Configuration Notes": draft_n_max bounds the tokens drafted per step;
 * drafting stops early at a low-confidence selector transition,
 * draft_p_min).  Host struct.
 *   n_max  drafts per step (0 = B-1; a request above B-1 is clamped to B-1,
 *          as the same section says the engine does): the selector walks
 *          positions 1..n_max only (the max-score path over that shorter
 *          lattice)
 *   p_min  in [0, 1]: the path is cut before the first position whose chosen
 *          transition has probability exp(T_i(prev, chosen)) < p_min
 *          (0 = never cut)
 */
typedef struct dflash2_draft_opts {
    int n_max;
    float p_min;
} dflash2_draft_opts;

/*
 * dflash2_select_path / dflash2_select_path_table with drafting knobs (opts
 * nullable: no knobs).  n_draft: nullable [batch] int32 out, the drafts kept
 * (0..n_max); path slots from n_draft on are -1; path_score is the kept
 * positions' summed log-probability.  DFLASH2_ERR_SHAPE for a negative n_max
 * or p_min outside [0, 1].
 */
int dflash2_select_path_ex(const dflash2_config *cfg, const dflash2_weights *w, int batch,
                           const int32_t *anchor, const int32_t *cand_id, const float *cand_logit,
                           const dflash2_draft_opts *opts, int32_t *path, float *path_score, int32_t *n_draft,
                           void *workspace, size_t ws_bytes, void *stream);
int dflash2_select_path_table_ex(const dflash2_config *cfg, int batch, const int32_t *anchor,
                                 const int32_t *cand_id, const float *cand_logit, const float *table,
                                 const dflash2_draft_opts *opts, int32_t *path, float *path_score,
                                 int32_t *n_draft, void *workspace, void *stream);

/*
 * DFlash (v1) selection ("Variants": DFlash 2 adds the pairwise selector to
 * the block-parallel baseline, which takes each position's best candidate):
 * path[s][i] = cand_id[s][i][0], the per-position top-1, with the same
 * drafting knobs (opts nullable), whose transition probabilities are then
 * the softmax of the k candidate logits.  Same outputs as the _ex selectors;
 * needs no factors, no weights and no scratch (workspace nullable: its
 * status word only).
 */
int dflash2_select_top1(const dflash2_config *cfg, int batch, const int32_t *cand_id, const float *cand_logit,
                        const dflash2_draft_opts *opts, int32_t *path, float *path_score, int32_t *n_draft,
                        void *workspace, void *stream);

/*
 * Stage (d2): greedy verification ("Prerequisites": the target verifies
 * [id_last, draft...] in one batch; "Validation": output token ids equal
 * plain greedy decoding).
 *   path          [batch, B-1] int32 proposed tokens
 *   target        [batch, B] int32: target[s][i] is the target's greedy token
 *                 after [anchor, path_1..path_i] (i = 0..B-1)
 *   accept_len    [batch] int32 out: a = longest prefix with path == target
 *   out_tok       [batch, B] int32 out: path_1..path_a, target_a, then -1s
 *   n_out         [batch] int32 out: a + 1
 *   next_anchor   [batch] int32 out: target[s][a]
 *   seq_len       nullable [batch] int32 in/out: += a + 1 (the rejected
 *                 suffix is rolled back simply by not being counted)
 *   counters      nullable int64 [4 + B + (B-1)] in/out, accumulated
 *                 ("Observe Acceptance"): [0] steps, [1] drafted tokens,
 *                 [2] accepted draft tokens, [3] rolled-back tokens,
 *                 [4 .. 4+B-1] histogram of a = 0..B-1,
 *                 [4+B .. 4+2B-2] accepted count by draft position 1..B-1.
 * block_size must be in 2..32.
 */
int dflash2_verify_accept(int batch, int block_size, const int32_t *path,
                          const int32_t *target, int32_t *accept_len,
                          int32_t *out_tok, int32_t *n_out, int32_t *next_anchor,
                          int32_t *seq_len, int64_t *counters, void *stream);

/*
 * dflash2_verify_accept for paths of n_draft[s] drafts (from the _ex
 * selectors; nullable: B-1 each): a <= n_draft[s], and the counters add
 * n_draft[s] drafted and n_draft[s] - a rolled-back tokens.
 */
int dflash2_verify_accept_ex(int batch, int block_size, const int32_t *path, const int32_t *n_draft,
                             const int32_t *target, int32_t *accept_len, int32_t *out_tok, int32_t *n_out,
                             int32_t *next_anchor, int32_t *seq_len, int64_t *counters, void *stream);

/*
 * Sampled verification (temperature > 0): lossless speculative sampling
 * against the target's distribution ([Train]: spec_generate's temperature,
 * top_p and top_k truncate the TARGET's distribution, the one rejection
 * sampling verifies against, so sampled decoding stays lossless with
 * respect to the target sampling on its own).  The selector's proposal is
 * deterministic (a point mass on its path), so draft i is accepted when
 * u_accept[s][i] < p_i(path_i); at the first rejection the emitted token is
 * drawn from p_i with path_i removed (renormalised), and when every kept
 * draft is accepted the bonus token is drawn from the next position's p.
 * A draw maps u_sample[s] to the first token, in id order, whose cumulative
 * mass exceeds u_sample[s] times the total (inverse CDF).
 *   target_prob  [batch, B, vocab] float: p_i for i = 0..B-1, the target's
 *                distribution after [anchor, path_1..path_i] with its own
 *                temperature / top-p / top-k applied (zeros outside)
 *   u_accept     [batch, B-1] float in [0, 1): the acceptance draws
 *   u_sample     [batch] float in [0, 1): the draw of the emitted token
 *   n_draft      nullable [batch]: drafts kept per sequence (B-1 when null)
 * Outputs, seq_len and counters as dflash2_verify_accept_ex.  Random numbers
 * are inputs, so a call is deterministic.  DFLASH2_ERR_SHAPE for vocab < 2
 * or vocab > 1,536,000.
 */
int dflash2_verify_sampled(int batch, int block_size, int vocab, const int32_t *path, const int32_t *n_draft,
                           const float *target_prob, const float *u_accept, const float *u_sample,
                           int32_t *accept_len, int32_t *out_tok, int32_t *n_out, int32_t *next_anchor,
                           int32_t *seq_len, int64_t *counters, void *stream);

/*
 * Instrumentation.  Number of kernel launches the library has issued since
 * it was loaded (host-side counter; a launch recorded into a CUDA graph
 * counts once, at capture).
 */
int64_t dflash2_launch_count(void);

/*
 * Optional stage events (process-wide setting, not thread-safe).  When
 * `events` is non-NULL it must hold DFLASH2_N_STAGE_EVENTS cudaEvent_t
 * handles created with timing enabled; dflash2_draft_step then records them
 * on its stream (as external event records, so they survive CUDA-graph
 * capture): [0] step start, [1] after the context append, [2] after the
 * block forward, [3] after the lm_head contraction with its fused top-k,
 * [4] after the top-k merge.  Pass NULL to stop.
 */
#define DFLASH2_N_STAGE_EVENTS 5
void dflash2_set_stage_events(void *const *events);

/*
 * Reads (synchronising `stream`) and clears the device status word of a
 * workspace: a bitwise OR of DFLASH2_DEV_* codes recorded since the last
 * read, or a negative status if the read itself failed.
 */
int dflash2_read_device_status(void *workspace, size_t ws_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH2_H */
