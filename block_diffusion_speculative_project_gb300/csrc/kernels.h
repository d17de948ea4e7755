// Internal interface between the C-ABI layer (dflash_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace df {

// Launch with programmatic stream serialization: the kernel may start while the
// previous kernel in the stream drains; every libdflash kernel calls
// griddepcontrol.wait before it touches data produced upstream.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t s, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Programmatic launch of a kernel in thread-block clusters of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t s, int cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = cluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Bits of the device status word (first word of the workspace).
constexpr int kStatusTimeout = 1;  // a bounded wait ran out
constexpr int kStatusCheck = 2;    // a bounds check failed (index skipped)

constexpr int kNumSMsDefault = 152;
constexpr int kPageRows = 64;      // rows per page of a paged cache (one attention key unit)

// ---------------------------------------------------------------- GEMM engine

enum GemmEpi : int {
  EPI_BF16 = 0,   // out bf16 [M, ldo] = acc
  EPI_F32 = 1,    // out f32  [M, ldo] = acc
  EPI_RESID = 2,  // xres f32 [M, ldo] += acc
  EPI_ROPE = 3,   // q|k|v of the block: RoPE on columns < rope_cols (per hd-wide head);
                  // columns < q_cols to out bf16, the k and v heads to the layer's
                  // caches kc / vc at rows ctx_len + j
  EPI_SWIGLU = 4, // dual: out bf16 [M, ldo] = silu(acc_gate) * acc_up
  EPI_DUAL_F32 = 5, // dual: out f32 [M, ldo]: cols [0,N) from B0, [N,2N) from B1
  EPI_KV = 6,     // grouped: scatter rows into the K/V caches (RoPE on K groups)
  EPI_TOPK = 7,   // per-row running top-k over the CTA's vocab range
};

constexpr int kMaxBMaps = 12;
constexpr int kMaxBlock = 16;  // largest block size B (dflash_create checks 2 <= B <= 16)
constexpr int kTopkMax = 16;

// Kernel parameters of the tcgen05 GEMM  D[M, N] = A[M, K] * B[N, K]^T.
// A: bf16 rows, read through a 3D tensor map {K, R, G} (plain matrices use G = 1).
// B: bf16 weights [N, K], one 2D tensor map per group (or two for dual).
struct GemmParams {
  CUtensorMap tmA;
  CUtensorMap tmB[kMaxBMaps];
  int M;           // logical rows
  int tile_rows;   // logical rows per 128-lane block (<= 128); an m-tile holds MS blocks
  int a_grouped;   // 0: tile m loads rows [128m, 128m+128) of dim1; 1: groups [m*S, m*S+S)
  int a_S;         // groups per tile when a_grouped
  int N;           // output columns per group (per weight when dual)
  int K;
  int m_tiles, n_tiles, groups, dual, splits;
  int kt_total, kt_per_split;
  int items;       // m_tiles * n_tiles * groups * splits
  int rast_gm;     // persistent tile order: groups of rast_gm m-tiles, m fastest inside a
                   // group, then the column tile, then the weight group (rast_gm = m_tiles:
                   // plain m-fastest order)
  uint32_t stage_tx_bytes;
  int epi;
  void *out;
  long long ldo;
  float *xres;
  // RoPE (EPI_ROPE, EPI_KV)
  const int *ctx_len;
  int rows_per_seq;
  int rope_cols;
  int q_cols;      // EPI_ROPE: columns written to out; the rest are Hkv k then Hkv v heads
  int hd;
  float inv_freq[64];
  // K/V scatter (EPI_KV): group g -> layer g/2, g%2 == 0 keys (rotated), 1 values;
  // EPI_ROPE: the current layer's caches
  void *kc;
  void *vc;
  const int *n_commit;
  int Hkv, Cmax, max_batch;
  // Paged cache (page_table non-null): row pos of sequence seq lives in page
  // page_table[seq * pages_per_seq + pos / kPageRows], row pos % kPageRows; a page holds
  // the kPageRows rows of every kv head. Pages outside [0, num_pages) are reported and
  // not written.
  const int *page_table;
  int pages_per_seq, num_pages;
  long long layer_rows;  // EPI_KV: cache rows of one layer (the layer stride, in rows)
  // top-k (EPI_TOPK)
  int topk_k;
  int tiles_per_cta;
  float *part_vals;  // [ranges][M][topk_k]
  int *part_ids;
  float *logits_out; // [M][N] or null
  int *status;
  int max_spin;
  int stall;         // test hook: issue no loads so the waits run out
  // Deferred RMSNorm (pre-norm residual stream): the EPI_RESID epilogue also writes
  // xg = bf16(x_new * g_next) (bf16(x_new) when g_next is null) and, when ss_out is set,
  // per-(row, column tile) partial sums of x_new^2 (ss_out [M][n_tiles]); a consumer GEMM reading xg as A scales its accumulator row i
  // by rsqrt(sum(ss_in[i][0..ss_n)) * inv_d + eps) before its epilogue (ROPE, SWIGLU),
  // which equals the GEMM of RMSNorm(x) * g.
  uint16_t *xg_out;
  const uint16_t *g_next;
  float *ss_out;
  const float *ss_in;
  int ss_n;
  float inv_d, eps;
  int csplit;        // >1: split K across the CTAs of a cluster, reduce through DSMEM
  int slabs;         // 2: A and B maps carry a 64-column slab dimension and each stage
                     // loads two slabs per copy (plain 128-wide GEMMs with K % 64 == 0)
  int act;           // EPI_BF16: 1 = silu(acc) before rounding
  // EPI_TOPK draw at temperature 1 / smp_inv_T (smp_part set): per (vocabulary range, row)
  // the partial draw of Philox stream smp_stream, row = the LM-head row, two float4 per
  // entry at smp_part[2 * (range * M + row)]
  float4 *smp_part;
  float smp_inv_T;
  int smp_stream;
  unsigned long long smp_seed;
};

struct GemmLaunch {
  int BN;
  int grid;
  size_t smem;
};

// Fills the derived fields of p (tiles, cluster split, grid) and launches; the
// GEMM needs no global scratch (a split K is reduced inside its cluster).
cudaError_t gemm_launch(GemmParams &p, int BN, int num_sms, cudaStream_t s);
// cluster_cap[S] (S = 2..8): clusters of S CTAs the device keeps resident at once,
// 0 = unknown; may be null.
void gemm_plan(int M, int tile_rows, int N, int K, int groups, int dual, int BN, int slabs, int num_sms,
               int epi, const int *cluster_cap, int *splits, int *kt_per_split, int *items, int *grid,
               int *csplit);
int gemm_tiles(int M, int tile_rows, int N, int groups, int dual, int BN);
// Vocabulary ranges of the LM head's top-k GEMM: the n_tiles column tiles are cut into
// *ranges contiguous ranges of *tiles_per_cta tiles, one CTA per (range, row tile), with
// ranges <= max(1, num_sms / m_tiles). The launch and every buffer sized per range use
// this one plan.
void topk_range_plan(int n_tiles, int m_tiles, int num_sms, int *tiles_per_cta, int *ranges);
// 128-row blocks per tile (1 or 2) gemm_launch takes for these launch parameters (tile_rows:
// rows per 128-lane block); a launch's m_tiles = ceil(M / (blocks * tile_rows)).
int gemm_mstack(int epi, int BN, int M, int tile_rows, int N, int groups, int a_grouped, int dual, int num_sms);

// ---------------------------------------------------------------- small kernels

cudaError_t launch_embed_rmsnorm(const int *ids, const uint16_t *E, const uint16_t *relay, int M,
                                 int D, int V, float *x, const uint16_t *g, float eps, uint16_t *u,
                                 int *status, cudaStream_t s);
cudaError_t launch_rmsnorm(const float *x, int M, int D, const uint16_t *g, float eps, uint16_t *u,
                           cudaStream_t s);
cudaError_t launch_rmsnorm_rows(const float *x, int M, int D, const uint16_t *g, float eps,
                                uint16_t *u, int B, int skip_first, cudaStream_t s);
cudaError_t launch_relay_and_len(const uint16_t *h, int nb, int R, int B, int D,
                                 const int *relay_a, const int *n_commit, int *ctx_len,
                                 uint16_t *x0_relay, int Cmax, int *status, cudaStream_t s);
// FiLM relay ([DFlow] 第三步): conditioning rows and the modulated relay rows, one row
// per block offset (i, j); rows that are not relayed get zeros.
cudaError_t launch_film_cond(const uint16_t *h, const uint16_t *E, int nb, int R, int B, int D,
                             int V, const int *relay_a, const int *relay_b, const int *relay_y,
                             uint16_t *cond, int *status, cudaStream_t s);
cudaError_t launch_film_apply(const uint16_t *h, const float *bg, int nb, int R, int B, int D,
                              const int *relay_a, float eps, uint16_t *x0, cudaStream_t s);
// draft position j of sequence i at draft[(i * (B - 1) + j) * draft_stride]
cudaError_t launch_accept(const int *draft, int draft_stride, const int *target, int nb, int B, int *tau,
                          int *bonus, cudaStream_t s);
cudaError_t launch_topk_merge(const float *vals, const int *ids, int rows, int ncand_per_row,
                              long long row_stride, long long part_stride, int parts, int k,
                              int *out_ids, float *out_vals, cudaStream_t s);
cudaError_t launch_f32_to_bf16(const float *x, uint16_t *y, long long n, cudaStream_t s);
cudaError_t launch_conv_apply(float *x, uint16_t *xb_out, const float *corr, const uint16_t *base, int M, int D,
                              int B, int group, cudaStream_t s);
cudaError_t launch_gather_select(const int *block_ids, const int *cand_ids, int nb, int B, int k,
                                 const uint16_t *E, int D, int V, uint16_t *out, int *status,
                                 cudaStream_t s);
// The selector's score table [nb][B-1][k][k] alone (the sampling walk reads it).
cudaError_t launch_select_table(const float *cand_vals, const float *AB, const float *G, float *table,
                                int nb, int B, int k, int sel_dim, cudaStream_t s);
// Sampling walk over the table (sampling.cu): path [nb][B-1] and walk_logq [nb][B-1][k].
cudaError_t launch_select_walk_sample(const int *cand_ids, const float *table, int nb, int B, int k,
                                      float inv_T, unsigned long long seed, int *path, float *walk_logq,
                                      cudaStream_t s);
// Recall@k counts (atomic adds into hits[B-1], eligible[B-1]).
cudaError_t launch_recall_at_k(const int *cand_ids, const int *target, int nb, int B, int k, int *hits,
                               int *eligible, cudaStream_t s);
cudaError_t launch_select_walk(const int *cand_ids, const float *cand_vals, const float *AB,
                               const float *G, float *table, int nb, int B, int k, int sel_dim, int *path,
                               cudaStream_t s);

// ---------------------------------------------------------------- sampling (sampling.cu)

constexpr int kSampleMaxSlices = 64;
// Slices per logit row of the sampling passes (rows * S CTAs, at least 1024 elements each).
int sample_slices(int rows, int V, int num_sms);
// Draws ids[r] ~ softmax(logits[r] * inv_T) (Philox stream `stream`, row row0 + r) and
// writes lse[r] (and logq[r] = log q(ids[r])); stream < 0: lse only (ids, logq unused).
// part: rows * S * 2 float4 of scratch.
cudaError_t launch_sample(const float *logits, long long ld, int rows, int V, float inv_T,
                          unsigned long long seed, int stream, int row0, int S, float4 *part,
                          int *ids, float *lse, float *logq, cudaStream_t s);
// Merge of partial draws (two float4 each) at entries r * row_stride + k * slice_stride.
cudaError_t launch_draw_merge(const float4 *part, int rows, int S, long long row_stride,
                              long long slice_stride, int *ids, float *lse, float *logq, cudaStream_t s);
// Philox uniforms and Gumbel values of (seed, stream, row) for v < n (a check of the random
// numbers every draw uses).
cudaError_t launch_draw_gumbel(int n, unsigned long long seed, int stream, int row, float *u, float *g,
                               cudaStream_t s);
// Rejection-sampling verify against the sampling walk's sparse draft distribution.
cudaError_t launch_verify_walk(const int *cand_ids, const float *walk_logq, int k, const int *path,
                               const float *target_logits, const float *target_lse, int nb, int B, int V,
                               float inv_T, unsigned long long seed, int S, float4 *part, int *nrej,
                               int *tau, int *token, cudaStream_t s);
// Rejection-sampling verify of nb blocks; part: nb * S float4, nrej: nb ints of scratch.
cudaError_t launch_verify(const float *draft_logits, const float *draft_lse, const int *cand,
                          const float *target_logits, const float *target_lse, int nb, int B, int V,
                          float inv_T, unsigned long long seed, int S, float4 *part, int *nrej,
                          int *tau, int *token, cudaStream_t s);

// ---------------------------------------------------------------- attention

// Context attention of one drafter layer (see attention.cu). The block's own K/V rows
// have already been written to cache rows [ctx_len, ctx_len + B) by the QKV GEMM, so
// every sequence attends to cache rows [0, ctx_len + B) of its heads (contiguous, or
// through the page table).
struct AttnParams {
  CUtensorMap tmQ;      // qkv buffer as {hd, Hq heads, nb*B rows}, box {64, Hq/Hkv, B}
  CUtensorMap tmK;      // key cache of every layer: {64, N*max_batch*Hkv*Cmax rows, hd/64}, box {64, 128, hd/64}
                        // (paged: {64, N*num_pages*Hkv*64 rows, hd/64}, box {64, 64, 1})
  CUtensorMap tmV;      // value cache, same shape
  const int *ctx_len;   // [nb]
  uint16_t *o;          // [nb*B, Hq*hd] bf16
  float *part_o;        // [slots][G*B rows][hd] unnormalised partial outputs
  float *part_ml;       // [slots][G*B rows][2] (running max, running sum)
  int nb, B, Hq, Hkv, hd, Cmax, max_batch;
  int layer_row0;       // first cache row of this layer: layer * (rows of one layer)
  // Paged cache (page_table non-null): tmK / tmV are {64, pool rows, hd/64} with box
  // {64, 64, 1}, and unit u of sequence i is page page_table[i * pages_per_seq + u].
  const int *page_table;
  int pages_per_seq, num_pages;
  int max_ctx;          // caller's bound on ctx_len (larger values are reported and clamped)
  int grid;             // CTAs of the attention launch (work is split evenly over them)
  int *status;
  int max_spin;
  int stall;            // test hook: issue no loads so the waits run out
};

// Slots of partial outputs the attention of nb sequences may write: at most one per
// (pair, CTA) boundary, i.e. nb * Hkv + grid.
inline size_t attention_slots(int nb, int Hkv, int grid) { return (size_t)nb * Hkv + grid; }
cudaError_t launch_attention(const AttnParams &p, cudaStream_t s);

}  // namespace df
