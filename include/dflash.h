/*
 * dflash.h -- C ABI of libdflash: the one-pass block-diffusion draft step
 * (DFlash drafter with KV injection, DFlow relay in plain and FiLM form, DFlash 2
 * selector and conv, greedy accept or sampling with rejection-sampling verify,
 * contiguous or paged KV cache) on one NVIDIA GB300 GPU (sm_103a).
 *
 * Sources (page title, section):
 *   [DFlash]  "DFlash 投机解码：块扩散草稿与 KV 注入" (caijizhuo.github.io)
 *   [DFlow]   "DFlow 完全拆解" (pinghaoyang.com.cn/aigc/posts/dflow)
 *   [DFlash2] "DFlash 2：正确 token 已在候选里" (bowenzhou.top/papers/2026/DFlash2)
 *
 * Conventions shared by every call
 *   - Every tensor argument is a DEVICE pointer owned by the caller: weights, KV
 *     caches, inputs, outputs and the workspace. The library allocates no device
 *     memory. Weights are borrowed by dflash_set_weights and must outlive the handle.
 *   - Matrices are row-major. Weight matrices are [out_features, in_features] bf16.
 *     "bf16" tensors hold IEEE bfloat16 bit patterns; "f32" tensors hold float.
 *   - Every step call is asynchronous on the given stream and performs no host
 *     synchronisation; a handle and its workspace serve one stream at a time.
 *   - Every call returns DFLASH_OK (0) or a negative DFLASH_ERR_* code; on error
 *     dflash_last_error() returns a thread-local message. Argument errors are
 *     detected on the host before any launch. Errors found on the device (a bounded
 *     wait that ran out, a context length beyond the hint or capacity) are recorded
 *     in a status word inside the workspace and read back by dflash_status().
 *   - No C++ exception crosses the ABI.
 *
 * KV cache layout (both K and V): bf16 [N][max_batch][Hkv][Cmax][hd]; sequence i of
 * a call uses slot i. K rows hold RoPE-rotated keys.
 *
 * Paged KV cache (cfg.num_pages > 0; reading of [DFlash] 四、推理流程, the engineering
 * note: the projected K/V are what the drafter's cache keeps, and requests with a common
 * prefix reuse them through a radix cache): both caches are pools of pages,
 * bf16 [N][num_pages][Hkv][DFLASH_PAGE_ROWS][hd]. Row r of sequence i (every layer, every
 * kv head) is row r % DFLASH_PAGE_ROWS of page table[i][r / DFLASH_PAGE_ROWS] of the
 * block table registered by dflash_set_block_table. Sequences may share pages for rows
 * that no call of the step writes (a common prefix); the rows a call appends (context
 * rows ctx_len .. ctx_len + n_commit - 1, block rows ctx_len .. ctx_len + B - 1) must
 * lie in pages no other sequence of the call reads or writes.
 *
 * Block layout (reading of [DFlash] 符号约定 and 四、推理流程): block i is
 * [anchor, mask_id x (B-1)] at absolute positions ctx_len[i] .. ctx_len[i]+B-1,
 * where ctx_len counts the context rows in the cache; offsets 1..B-1 carry the
 * B-1 draft candidates.
 */
#ifndef DFLASH_H
#define DFLASH_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define DFLASH_API __attribute__((visibility("default")))
#else
#define DFLASH_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st *dflash_stream_t;

enum dflash_status_code {
  DFLASH_OK = 0,
  DFLASH_ERR_INVALID_ARG = -1,       /* null pointer, negative size, bad index */
  DFLASH_ERR_UNSUPPORTED_SHAPE = -2, /* a shape outside what the kernels support */
  DFLASH_ERR_CUDA = -3,              /* a CUDA runtime or driver call failed */
  DFLASH_ERR_TIMEOUT = -4,           /* a bounded device-side wait ran out */
  DFLASH_ERR_DEVICE_CHECK = -5       /* a device-side bounds check failed */
};

enum dflash_flags {
  DFLASH_FLAG_RELAY = 1,  /* DFlow relay rows are accepted by ctx_project / draft_block */
  DFLASH_FLAG_CONV = 2,   /* DFlash 2 two-tap dynamic conv, 4 per layer */
  DFLASH_FLAG_SELECT = 4, /* DFlash 2 path selector weights are registered */
  DFLASH_FLAG_FILM = 8,   /* DFlow FiLM relay weights are registered (requires RELAY) */
  /* Test hook for the failure path: the GEMM producers issue no loads, so every
   * wait on them runs out after max_spin polls, DFLASH_ERR_TIMEOUT is recorded and
   * the kernels return with the context intact. Never set in production. */
  DFLASH_FLAG_TEST_STALL = 1 << 30
};

typedef struct dflash_config {
  int D;        /* drafter hidden size, multiple of 64 */
  int Dt;       /* target hidden size of each of the L selected layers */
  int L;        /* number of target layers concatenated into the W_c input */
  int N;        /* drafter layers, 1..16 */
  int Hq;       /* query heads */
  int Hkv;      /* key/value heads; Hq % Hkv == 0; query head h reads kv head h/(Hq/Hkv) */
  int hd;       /* head dim: 64 or 128 */
  int F;        /* SwiGLU FFN width, multiple of 8 */
  int V;        /* vocabulary size */
  int B;        /* block size: anchor + B-1 masks, 2..16 */
  int k_top;    /* candidates kept per position by dflash_lm_head_topk, 1..16 */
  float rope_base; /* RoPE base (theta_d = base^(-2d/hd), rotate-half pairing) */
  float eps;    /* RMSNorm epsilon */
  int mask_id;  /* token id of the mask embedding row in E */
  int Cmax;     /* context capacity per sequence (cache rows) */
  int max_batch;      /* sequences the cache and workspace are sized for */
  int max_proj_rows;  /* largest R (rows per sequence) passed to dflash_ctx_project */
  int conv_group;     /* channels sharing one conv correction (16); used with CONV */
  int sel_dim;        /* selector embedding width (256); used with SELECT */
  unsigned flags;     /* DFLASH_FLAG_* */
  int max_spin;       /* iteration bound of every device-side wait; 0 = default */
  int film_dim;       /* FILM: hidden width of the relay MLP, multiple of 64 */
  int num_pages;      /* 0: contiguous caches; > 0: paged caches of this many pages
                         (Cmax a multiple of DFLASH_PAGE_ROWS; see the layout above) */
} dflash_config;

/* Rows per page of a paged cache (one 64-key unit of the attention). */
#define DFLASH_PAGE_ROWS 64

typedef struct dflash_layer_weights {
  const void *W_qkv;  /* bf16 [(Hq+2*Hkv)*hd, D]: rows q heads, then k_b heads, then v_b heads */
  const void *Wk_c;   /* bf16 [Hkv*hd, D]: context-key projection W_c^K of this layer */
  const void *Wv_c;   /* bf16 [Hkv*hd, D]: context-value projection W_c^V of this layer */
  const void *W_o;    /* bf16 [D, Hq*hd] */
  const void *W_gate; /* bf16 [F, D] */
  const void *W_up;   /* bf16 [F, D] */
  const void *W_down; /* bf16 [D, F] */
  const void *g_attn; /* bf16 [D] RMSNorm gain before attention */
  const void *g_ffn;  /* bf16 [D] RMSNorm gain before the FFN */
  const void *conv_W0[4];   /* CONV: bf16 [D/conv_group, D], correction of tap 0 */
  const void *conv_W1[4];   /* CONV: bf16 [D/conv_group, D], correction of tap 1 */
  const void *conv_base[4]; /* CONV: bf16 [2, D], base kernel (tap 0, tap 1) */
} dflash_layer_weights;

typedef struct dflash_weights {
  const void *W_c;     /* bf16 [D, L*Dt]: fused target-context projection */
  const void *g_ctx;   /* bf16 [D]: RMSNorm gain after W_c */
  const void *E;       /* bf16 [V, D]: shared token embedding */
  const void *W_lm;    /* bf16 [V, D]: shared LM head */
  const void *g_final; /* bf16 [D]: final RMSNorm gain */
  const void *W_A;     /* SELECT: bf16 [sel_dim, D] */
  const void *W_B;     /* SELECT: bf16 [sel_dim, D] */
  const void *W_G;     /* SELECT: bf16 [sel_dim, D] */
  const dflash_layer_weights *layers; /* N entries; copied by dflash_set_weights */
  const void *film_W1; /* FILM: bf16 [film_dim, 3*D], first layer of the relay MLP */
  const void *film_W2; /* FILM: bf16 [2*D, film_dim], second layer; rows [0,D) beta, [D,2D) gamma */
} dflash_weights;

typedef struct dflash_handle_s *dflash_handle_t;

/* ------------------------------------------------------------------ lifecycle */

/* Validate cfg and create a handle bound to the current CUDA device.
 * Unsupported: hd not in {64,128}, Hq % Hkv != 0, B outside 2..16, k_top outside
 * 1..16, D or L*Dt or Hq*hd not a multiple of 64, F not a multiple of 8. */
DFLASH_API int dflash_create(const dflash_config *cfg, dflash_handle_t *out);

/* Destroy a handle. Safe on NULL. Does not touch borrowed weights. */
DFLASH_API int dflash_destroy(dflash_handle_t h);

/* Register weight pointers (borrowed). Builds the TMA descriptors of every weight
 * matrix. All pointers must be 16-byte aligned; optional groups (conv, selector,
 * FiLM relay) must be non-NULL when their flag is set. */
DFLASH_API int dflash_set_weights(dflash_handle_t h, const dflash_weights *w);

/* Register the block table of a paged cache (the layout above: a reading of [DFlash]
 * 四、推理流程, the note on reusing the projected cache across requests with a common
 * prefix). The table is a borrowed device pointer, int32
 * [max_batch][Cmax / DFLASH_PAGE_ROWS], 4-byte aligned. Kernels read it when they run,
 * so the caller may change entries between calls in stream order. Every call that
 * touches the caches needs it when cfg.num_pages > 0 (DFLASH_ERR_INVALID_ARG before
 * any launch otherwise). An entry outside [0, num_pages) that a call reaches is
 * reported as DFLASH_ERR_DEVICE_CHECK by dflash_status: its rows are not written and
 * are read from page 0. DFLASH_ERR_INVALID_ARG for a contiguous handle. */
DFLASH_API int dflash_set_block_table(dflash_handle_t h, const int32_t *table);

/* Bytes of workspace every step call of this handle needs (sized for max_batch,
 * max_proj_rows and Cmax). The caller allocates it (256-byte aligned) and zero-fills it
 * once before the first call: its first word is the device status word, which the
 * kernels only OR into (dflash_status reads and clears it). */
DFLASH_API int dflash_workspace_size(dflash_handle_t h, size_t *bytes);

/* Synchronise `stream`, read and clear the device status word in `ws`.
 * *code = DFLASH_OK, DFLASH_ERR_TIMEOUT or DFLASH_ERR_DEVICE_CHECK. */
DFLASH_API int dflash_status(dflash_handle_t h, void *ws, dflash_stream_t stream, int *code);

/* Thread-local message for the last error returned on this thread. */
DFLASH_API const char *dflash_last_error(void);

/* ------------------------------------------------------------------ step calls */

/* Fused target-context projection and context-KV append, plus the DFlow relay
 * input ([DFlash] 三、KV 注入 H_c equation and the engineering note that the
 * projected K/V, not H_c, are cached; [DFlow] 第一步 / 第二步).
 *   hv        bf16 [nb, R, L*Dt]: verifier hidden states of R consecutive rows per
 *             sequence, the L selected layers concatenated along features.
 *   n_commit  int32 [nb]: rows 0..n_commit[i]-1 of sequence i become context rows at
 *             positions ctx_len[i]+j: h = RMSNorm(W_c hv), K_c = RoPE(Wk_c h),
 *             V_c = Wv_c h are written into every layer's cache. 0 <= n_commit <= R.
 *   relay_a   int32 [nb] or NULL (requires DFLASH_FLAG_RELAY when non-NULL): the
 *             previous round's accepted count a; rows k in [a+2, B-1] (k < R) are
 *             relayed to block offset j = k - a of the next block.
 *   ctx_len   int32 [nb], device, updated in place to ctx_len + n_commit.
 *   kcache, vcache  the caches (layout above); ctx_len + n_commit must stay <= Cmax.
 *   x0_relay  bf16 [nb, B, D] output or NULL: h_k at the relayed offsets, 0 elsewhere.
 * Prefill is the same call with R = the prompt length (R <= max_proj_rows). */
DFLASH_API int dflash_ctx_project(dflash_handle_t h, int nb, int R, const void *hv,
                       const int32_t *n_commit, const int32_t *relay_a, int32_t *ctx_len,
                       void *kcache, void *vcache, void *x0_relay, void *ws, size_t ws_bytes,
                       dflash_stream_t stream);

/* dflash_ctx_project with the FiLM form of the DFlow relay ([DFlow] 第三步, the
 * [beta; gamma] = MLP_phi([E(b); E(y_{a+1}); h_i]) and x = E_mask + beta * LN(h_i) + gamma
 * equations). Requires DFLASH_FLAG_RELAY | DFLASH_FLAG_FILM and registered film weights.
 * Every argument of dflash_ctx_project keeps its meaning (relay_a is required), plus
 *   relay_b   int32 [nb], device: the verifier's correction token b at the first rejection
 *   relay_y   int32 [nb], device: the draft's rejected guess y_{a+1} there
 * and x0_relay (required) receives, at each relayed offset j (row k = j + a),
 *   beta * LN(h_k) + gamma with [beta; gamma] = W2 silu(W1 [E(b); E(y); h_k]),
 * LN(v) = (v - mean v) / sqrt(var v + eps) (population variance, no gain or bias),
 * rounded to bf16; 0 at every other offset. A token id outside [0, V) is reported as
 * DFLASH_ERR_DEVICE_CHECK by dflash_status and its embedding read as zeros. */
DFLASH_API int dflash_ctx_project_film(dflash_handle_t h, int nb, int R, const void *hv,
                       const int32_t *n_commit, const int32_t *relay_a,
                       const int32_t *relay_b, const int32_t *relay_y, int32_t *ctx_len,
                       void *kcache, void *vcache, void *x0_relay, void *ws, size_t ws_bytes,
                       dflash_stream_t stream);

/* One-pass draft of nb blocks through the N drafter layers ([DFlash] 二、块扩散草稿
 * attention equations and 四、推理流程 draft_forward): x = E[block_ids] (+ x0_relay);
 * per layer x += Attn(RMSNorm(x)) with Q from the block only, K = [K_c; K_b],
 * V = [V_c; V_b] and no mask; x += W_down(silu(W_gate u) * W_up u), u = RMSNorm(x);
 * with CONV a two-tap dynamic conv before and after each sublayer ([DFlash2] 洞察二).
 *   block_ids    int32 [nb, B] token ids (anchor, then mask ids)
 *   x0_relay     bf16 [nb, B, D] or NULL: added to the embeddings (DFlow relay)
 *   kcache, vcache  the caches: every layer's K_b / V_b (K_b rotated) are written to
 *                rows [ctx_len[i], ctx_len[i] + B) of sequence i, which the attention
 *                then reads with the context rows; those rows are scratch (the next
 *                dflash_ctx_project overwrites the committed ones).
 *   ctx_len      int32 [nb]: context rows per sequence (after this step's append);
 *                ctx_len[i] + B must be <= Cmax.
 *   max_ctx_hint host int: an upper bound on every ctx_len[i] (0 = Cmax - B). A
 *                ctx_len[i] above min(hint, Cmax - B), or negative, is reported as
 *                DFLASH_ERR_DEVICE_CHECK by dflash_status (and clamped).
 *   out_hidden   bf16 [nb, B, D]: final RMSNorm output (input of the LM head).
 * Results are bitwise reproducible for the same inputs and the same ctx_len of every
 * sequence of the call: the attention splits the keys over CTAs by the lengths alone.
 * Other sequences' lengths move those split points, so a sequence's output may then
 * differ in rounding (within the stated tolerance), never more. */
DFLASH_API int dflash_draft_block(dflash_handle_t h, int nb, const int32_t *block_ids, const void *x0_relay,
                       void *kcache, void *vcache, const int32_t *ctx_len,
                       int max_ctx_hint, void *out_hidden, void *ws, size_t ws_bytes,
                       dflash_stream_t stream);

/* Shared LM head on offsets 1..B-1 with a fused per-position top-k ([DFlash]
 * dflash_cycle argmax(...)[1:]; [DFlash2] 洞察一 top-16 candidates).
 *   hidden     bf16 [nb, B, D] (dflash_draft_block output)
 *   k          1..k_top
 *   out_ids    int32 [nb, B-1, k]: ids sorted by logit descending, ties to the lower id
 *   out_vals   f32   [nb, B-1, k]: their fp32 logits
 *   out_logits f32   [nb, B-1, V] or NULL: every logit (for parity checks). */
DFLASH_API int dflash_lm_head_topk(dflash_handle_t h, int nb, const void *hidden, int k, int32_t *out_ids,
                        float *out_vals, float *out_logits, void *ws, size_t ws_bytes,
                        dflash_stream_t stream);

/* Allocation-free variant of dflash_lm_head_topk, for callers that cannot hand the
 * library a workspace: code running inside a CUDA-graph capture (a cudaMalloc there
 * is not allowed), hosts whose device memory is entirely owned by another pool
 * allocator, and latency-critical threads that must not risk the implicit device
 * synchronisation an allocation can cause. The pages describe no such call; it
 * exists only for these callers.
 *   Same inputs and outputs as dflash_lm_head_topk, minus out_logits and the
 *   workspace. Scratch (the per-range partial top-k lists) lives in a 4 MiB
 *   file-scope device array that every GPU loading the library holds until exit;
 *   any shape whose lists need more is rejected with DFLASH_ERR_UNSUPPORTED_SHAPE.
 *   out_status: int32 device word or NULL. When given, device-side errors are
 *   OR-ed into it (value 1: a bounded wait ran out; value 2: a bounds check
 *   failed); the caller clears it. When NULL they are not reported, and out_ids /
 *   out_vals are undefined after such an error (they may hold another call's lists).
 *   The first call on a device looks up the array's device address
 *   (cudaGetSymbolAddress) with that device current; make that first call before
 *   any stream capture. The call allocates nothing. All calls share the one array,
 *   so calls that overlap on the GPU (different streams, or different handles on
 *   the same device, not ordered by the caller) race and must not be issued. */
DFLASH_API int dflash_lm_head_topk_noalloc(dflash_handle_t h, int nb, const void *hidden, int k,
                                           int32_t *out_ids, float *out_vals, int32_t *out_status,
                                           dflash_stream_t stream);

/* The drafter layer's context attention alone ([DFlash] 二、块扩散草稿 attention
 * equations): the stage dflash_draft_block runs between its QKV and O GEMMs, exposed
 * for stage-wise checks on given q, K and V.
 *   layer      0..N-1: the layer whose cache rows are read
 *   q          bf16 [nb, B, Hq, hd]: rotated queries of the block rows
 *   kcache, vcache  the caches; sequence i attends to rows [0, ctx_len[i] + B) of its
 *              kv head in layer `layer` (context rows, then the block's own K_b / V_b at
 *              rows ctx_len[i] + j, where dflash_draft_block writes them); no mask
 *   ctx_len, max_ctx_hint  as for dflash_draft_block
 *   out_o      bf16 [nb, B, Hq, hd]: softmax(q K^T / sqrt(hd)) V, query head h reading
 *              kv head h / (Hq/Hkv) */
DFLASH_API int dflash_attention(dflash_handle_t h, int nb, int layer, const void *q,
                                const void *kcache, const void *vcache, const int32_t *ctx_len,
                                int max_ctx_hint, void *out_o, void *ws, size_t ws_bytes,
                                dflash_stream_t stream);

/* Top-k of each row of an fp32 matrix with the same ordering rule as
 * dflash_lm_head_topk (value descending, ties to the lower column; [DFlash2] 洞察一 keeps
 * the top-16 per position). No counterpart call on the pages: it checks the selection rule
 * on exact inputs.
 *   logits f32 [rows, cols]; out_ids int32 [rows, k]; out_vals f32 [rows, k]; k 1..16. */
DFLASH_API int dflash_topk(dflash_handle_t h, int rows, int cols, const float *logits, int k,
                int32_t *out_ids, float *out_vals, void *ws, size_t ws_bytes,
                dflash_stream_t stream);

/* Greedy exact-match accept ([DFlash] 符号约定: 1 <= tau <= B; dflash_cycle step ④;
 * [DFlow] 问题不在拒绝).
 *   draft   int32 [nb, B-1]: candidates c_1..c_{B-1}
 *   target  int32 [nb, B]: verifier greedy tokens; T[j] verifies c_{j+1}
 *   out_tau int32 [nb]: n + 1 with n the number of leading matches
 *   out_bonus int32 [nb]: T[n] */
DFLASH_API int dflash_accept(dflash_handle_t h, int nb, const int32_t *draft, const int32_t *target,
                  int32_t *out_tau, int32_t *out_bonus, dflash_stream_t stream);

/* dflash_accept on the draft's top-k lists as dflash_lm_head_topk writes them: candidate
 * c_j of sequence i is the first (best) entry of offset j's list, topk_ids[(i*(B-1) + j-1)*k]
 * ([DFlash] dflash_cycle: the draft takes the argmax at every offset). No counterpart call
 * on the pages: it reads the lists in place instead of a contiguous copy of their first
 * column.
 *   topk_ids int32 [nb, B-1, k], k 1..16; target, out_tau, out_bonus as dflash_accept.
 * Errors: DFLASH_ERR_INVALID_ARG for a NULL tensor, nb < 0 or k outside 1..16. */
DFLASH_API int dflash_accept_topk(dflash_handle_t h, int nb, const int32_t *topk_ids, int k,
                  const int32_t *target, int32_t *out_tau, int32_t *out_bonus,
                  dflash_stream_t stream);

/* Draft sampling at temperature T > 0 ([DFlash2] 洞察一 and Results: sampling at T = 1;
 * each block offset draws independently from its own distribution, as the one-pass draft
 * predicts every position independently). Row r of `logits` draws
 *   out_ids[r] ~ softmax(logits[r] / T)
 * by Gumbel-max, argmax_v logits[r][v]/T - log(-log u_v) (ties to the lower id), with u_v
 * from Philox4x32-10 (Salmon et al., SC 2011) keyed by `seed`: word v % 4 of the block at
 * counter (v / 4, row0 + r, 0, 0), u = ((w >> 9) + 1/2) / 2^23.
 *   rows      number of rows, <= max_batch * B (for a draft: nb * (B-1), row0 = 0, so that
 *             offset t of sequence i is row i*(B-1) + t-1)
 *   logits    f32 [rows, V] (e.g. the out_logits of dflash_lm_head_topk)
 *   out_ids   int32 [rows]; -1 only for a row whose every logit is NaN
 *   out_lse   f32 [rows]: log sum_v exp(logits[r][v] / T)
 *   out_logq  f32 [rows] or NULL: log q(out_ids[r]) = logits[r][id] / T - out_lse[r] */
DFLASH_API int dflash_sample(dflash_handle_t h, int rows, const float *logits, float temperature,
                  uint64_t seed, int row0, int32_t *out_ids, float *out_lse, float *out_logq,
                  void *ws, size_t ws_bytes, dflash_stream_t stream);

/* The LM head with the draft draw fused into its epilogue: the logits of offsets 1..B-1
 * ([DFlash] dflash_cycle, [1:]) are drawn from as dflash_sample draws from them, while
 * they are computed, so they need not be written or read again.
 *   hidden     bf16 [nb, B, D] (out_hidden of dflash_draft_block)
 *   out_cand   int32 [nb, B-1]: c_t ~ softmax(U_t / T), Philox row i*(B-1) + t-1, stream 0
 *   out_lse    f32 [nb, B-1]: log sum_v exp(U_t(v) / T)
 *   out_logq   f32 [nb, B-1] or NULL: log q_t(c_t)
 *   out_logits f32 [nb, B-1, V] or NULL: U_t (dflash_verify_sample needs them)
 *   k, out_ids, out_vals: the top-k of dflash_lm_head_topk, or out_ids = NULL for none. */
DFLASH_API int dflash_lm_head_sample(dflash_handle_t h, int nb, const void *hidden, float temperature,
                  uint64_t seed, int32_t *out_cand, float *out_lse, float *out_logq,
                  float *out_logits, int k, int32_t *out_ids, float *out_vals, void *ws,
                  size_t ws_bytes, dflash_stream_t stream);

/* The random numbers every draw uses, for checking them (the pages fix no generator:
 * Philox4x32-10, Salmon et al., SC 2011): for v < n, out_u[v] = the Philox
 * uniform of element v of (seed, stream_id, row) (word v % 4 of the block at counter
 * (v / 4, row, stream_id, 0)) and out_g[v] = its Gumbel value -log(-log u) as the draws
 * compute it (absolute error about 1e-6). Needs no handle. */
DFLASH_API int dflash_draw_gumbel(int n, uint64_t seed, int stream_id, int row, float *out_u,
                  float *out_g, dflash_stream_t stream);

/* Lossless rejection-sampling verify of nb drafted blocks at temperature T > 0 ([DFlash2]
 * Results: lossless rejection sampling; [DFlash] 四、推理流程 dflash_cycle step ④: the
 * rejected position is re-drawn from the target, the last step yields the bonus token).
 * With p_j = softmax(target_logits[i][j] / T) and q_t = softmax(draft_logits[i][t-1] / T):
 * step j = 0..B-2 accepts c = cand[i][j] when log u_j < log p_j(c) - log q_{j+1}(c),
 * u_j = Philox uniform of counter (j / 4, i, 1, 0); n = the first rejected step (B-1 when
 * none). out_token[i] is a draw (Gumbel-max, Philox counter (v / 4, i, 2, 0)) from
 * max(0, p_n - q_{n+1}) renormalised, from p_n when that residual is zero everywhere,
 * or from p_{B-1} when every candidate was accepted. out_tau[i] = n + 1.
 *   draft_logits   f32 [nb, B-1, V]: U_t for offsets 1..B-1
 *   draft_lse      f32 [nb, B-1]: log sum exp(U_t / T) (out_lse of dflash_sample)
 *   cand           int32 [nb, B-1]: the drafted candidates (an id outside [0, V) is rejected)
 *   target_logits  f32 [nb, B, V]: row j = the target's logits after block offset j */
DFLASH_API int dflash_verify_sample(dflash_handle_t h, int nb, const float *draft_logits,
                  const float *draft_lse, const int32_t *cand, const float *target_logits,
                  float temperature, uint64_t seed, int32_t *out_tau, int32_t *out_token,
                  void *ws, size_t ws_bytes, dflash_stream_t stream);

/* DFlash 2 sampling walk ([DFlash2] 洞察一: sampling draws from the same score
 * distribution the greedy walk maximises): the scores S_t(a, b) of dflash2_select, then
 * from a_0 = the anchor each offset t draws slot c among its k candidates from
 * softmax_c(S_t(a_{t-1}, b_c) / T) by Gumbel-max (Philox counter (c / 4, i*(B-1) + t-1, 3, 0);
 * ties to the lower token id) and a_t = b_c.
 *   out_path       int32 [nb, B-1]: the drawn tokens
 *   out_walk_logq  f32 [nb, B-1, k]: log softmax_c(S_t(a_{t-1}, b_c) / T) along the drawn
 *                  path: the walk's draft distribution for dflash_verify_sample_walk.
 * Other arguments as dflash2_select. */
DFLASH_API int dflash2_select_sample(dflash_handle_t h, int nb, int k, const int32_t *topk_ids,
                  const float *topk_vals, const void *hidden, const int32_t *block_ids,
                  float temperature, uint64_t seed, int32_t *out_path, float *out_walk_logq,
                  void *ws, size_t ws_bytes, dflash_stream_t stream);

/* dflash_verify_sample with the sampling walk's draft distribution ([DFlash2] 洞察一: the
 * walk samples from the same score distribution, and Results: lossless rejection sampling
 * restores the target's distribution): q_t(v) =
 * exp(walk_logq[t-1][c]) for v = cand_ids[t-1][c], 0 for every other token (so the
 * residual of a non-candidate is p itself, and a drawn token outside the candidates is
 * rejected). Acceptance, residual, fallback and bonus draws as dflash_verify_sample.
 *   cand_ids   int32 [nb, B-1, k] (the top-k ids the walk chose from)
 *   walk_logq  f32 [nb, B-1, k] (out_walk_logq of dflash2_select_sample)
 *   path       int32 [nb, B-1] (out_path of dflash2_select_sample) */
DFLASH_API int dflash_verify_sample_walk(dflash_handle_t h, int nb, int k, const int32_t *cand_ids,
                  const float *walk_logq, const int32_t *path, const float *target_logits,
                  float temperature, uint64_t seed, int32_t *out_tau, int32_t *out_token,
                  void *ws, size_t ws_bytes, dflash_stream_t stream);

/* Recall@k instrumentation ([DFlash2] Why DFlash 2, the Recall@1 / Recall@16 table,
 * conditioned on every earlier position being right): for each block, offsets t = 1, 2, ...
 * count eligible[t-1] += 1 and, while target[i][t-1] is among cand_ids[i][t-1][0..k),
 * hits[t-1] += 1; the first miss ends the block. hits and eligible (int32 [B-1], device)
 * are accumulated atomically: the caller zeroes them to start a tally.
 *   cand_ids  int32 [nb, B-1, k]; target int32 [nb, B] (T[j] is the token after offset j) */
DFLASH_API int dflash_recall_at_k(dflash_handle_t h, int nb, int k, const int32_t *cand_ids,
                  const int32_t *target, int32_t *hits, int32_t *eligible, dflash_stream_t stream);

/* DFlash 2 two-tap dynamic depthwise conv ([DFlash2] 洞察二), in place:
 * x'_t = k_{t,0} * x_t + k_{t,1} * x_{t-1}, k_{t,j} = base_j + expand(W_j x_t),
 * one correction per conv_group channels, x_{-1} = 0 at block offset 0.
 *   layer 0..N-1, which 0..3 (before attention, after attention, before FFN, after FFN)
 *   x  f32 [nb*B, D]: residual stream rows, blocks of B consecutive rows. */
DFLASH_API int dflash2_conv(dflash_handle_t h, int layer, int which, int nb, float *x, void *ws,
                 size_t ws_bytes, dflash_stream_t stream);

/* DFlash 2 path selector, greedy walk ([DFlash2] 洞察一):
 * S_t(a,b) = U_t(b) + <A(a) * G(z_t), B(b)>, A = W_A E[a], B = W_B E[b],
 * G = sigmoid(W_G z_t); a_0 = anchor, a_t = argmax over the candidates of offset t
 * (ties to the lower id).
 *   topk_ids int32 [nb, B-1, k], topk_vals f32 [nb, B-1, k] (dflash_lm_head_topk output)
 *   hidden bf16 [nb, B, D]; block_ids int32 [nb, B] (column 0 is the anchor)
 *   out_path int32 [nb, B-1]: the selected draft. */
DFLASH_API int dflash2_select(dflash_handle_t h, int nb, int k, const int32_t *topk_ids,
                   const float *topk_vals, const void *hidden, const int32_t *block_ids,
                   int32_t *out_path, void *ws, size_t ws_bytes, dflash_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* DFLASH_H */
