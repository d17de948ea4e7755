// C ABI of libdflash (declared in include/dflash.h): argument validation, TMA
// descriptor encoding, workspace layout and the launch sequence of each step call.
// All compute runs in the kernels of gemm_tc.cu, attention.cu, sampling.cu and
// small_ops.cu.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/dflash.h"
#include "kernels.h"

using namespace df;

namespace {

thread_local std::string g_last_error;

int fail(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
int fail(int code, const char *fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_last_error = buf;
  return code;
}

#define DF_CUDA(call)                                                                          \
  do {                                                                                         \
    cudaError_t e_ = (call);                                                                   \
    if (e_ != cudaSuccess)                                                                     \
      return fail(DFLASH_ERR_CUDA, "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_),     \
                  __FILE__, __LINE__);                                                         \
  } while (0)

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// 2D bf16 map over a row-major [rows, cols] matrix (row stride in elements), box
// {64 columns, box_rows rows}, 128-byte swizzle.
int encode_2d(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols, uint64_t stride,
              uint32_t box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  if (reinterpret_cast<uintptr_t>(ptr) % 16 || (stride * 2) % 16)
    return fail(DFLASH_ERR_INVALID_ARG, "tensor %p (row stride %llu) is not 16-byte aligned", ptr,
                (unsigned long long)stride);
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {stride * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(ptr), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled (2D) failed: %d", (int)r);
  return DFLASH_OK;
}

// 3D bf16 map {cols, R, G}: row r of group g at ptr + g*gstride + r*rstride (elements).
int encode_3d(CUtensorMap *m, const void *ptr, uint64_t cols, uint64_t R, uint64_t G, uint64_t rstride,
              uint64_t gstride, uint32_t box_r, uint32_t box_g) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled is unavailable");
  if (reinterpret_cast<uintptr_t>(ptr) % 16 || (rstride * 2) % 16 || (gstride * 2) % 16)
    return fail(DFLASH_ERR_INVALID_ARG, "activation tensor %p is not 16-byte aligned", ptr);
  cuuint64_t dims[3] = {cols, R, G};
  cuuint64_t strides[2] = {rstride * 2, gstride * 2};
  cuuint32_t box[3] = {64, box_r, box_g};
  cuuint32_t es[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(ptr), dims, strides, box,
                  es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(DFLASH_ERR_CUDA, "cuTensorMapEncodeTiled (3D) failed: %d", (int)r);
  return DFLASH_OK;
}

// A plain activation matrix [rows, cols] (row stride = cols) as a 3D map with G = 1.
int encode_act(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t cols) {
  return encode_3d(m, ptr, cols, rows, 1, cols, rows * cols, 128, 1);
}

// Slab maps of the two-slab GEMM stages: a bf16 [rows, K] matrix (row stride K, K a
// multiple of 64) as {64, rows, K/64} with the slab stride 128 bytes; one box = two
// 64-column slabs of box_rows rows, stacked slab after slab.
int encode_slabs(CUtensorMap *m, const void *ptr, uint64_t rows, uint64_t K, uint32_t box_rows) {
  if (K % 64) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "slab map needs K %% 64 == 0 (K=%llu)",
                          (unsigned long long)K);
  return encode_3d(m, ptr, 64, rows, K / 64, K, 64, box_rows, 2);
}

constexpr int kBN = 128;       // tile width of the generic GEMMs
constexpr int kBNTopk = 256;   // tile width of the LM head
constexpr int kBNGateUp = 192; // gate|up GEMM: 96 gate + 96 up rows per tile (F/96 tiles)
// Context projection of a large prefill: 256 x 256 tiles (two stacked 128-row blocks and
// 256 weight rows per tile, twice the FLOPs per operand byte an SM takes in of the 256 x 128
// tiles) once they give at least two waves.
constexpr int kBNWide = 256;
bool wide_tiles(int num_sms, int M, int N, int groups, int epi) {
  const long long tiles = (long long)((M + 255) / 256) * ((N + kBNWide - 1) / kBNWide) * groups;
  return tiles >= 2LL * num_sms && gemm_mstack(epi, kBNWide, M, 128, N, groups, 0, 0, num_sms) == 2;
}
constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

struct WsLayout {
  size_t status = 0;
  size_t pre = 0, h = 0;                       // ctx_project
  size_t x = 0, u = 0, qkv = 0, o = 0, act = 0, xb = 0, corr = 0, ss = 0;  // draft_block
  size_t apart = 0, aml = 0;                   // attention partials
  size_t tk_vals = 0, tk_ids = 0;              // LM head top-k partial lists
  size_t sel_e = 0, sel_ab = 0, sel_g = 0, sel_t = 0;  // selector
  size_t film_cond = 0, film_hid = 0, film_bg = 0;     // FiLM relay
  size_t smp_part = 0, smp_lse = 0, ver_part = 0, ver_nrej = 0;  // sampling
  size_t total = 0;
  size_t apart_bytes = 0, apart_ctas = 0;
};

}  // namespace

struct dflash_handle_s {
  dflash_config cfg{};
  int device = 0;
  int num_sms = kNumSMsDefault;
  bool have_weights = false;
  dflash_weights w{};
  std::vector<dflash_layer_weights> layers;
  CUtensorMap tm_Wc, tm_lm, tm_A, tm_B, tm_G, tm_f1, tm_f2;
  std::vector<CUtensorMap> tm_qkv, tm_kc, tm_vc, tm_o, tm_gate, tm_up, tm_down;
  // 256-row boxes of the context projection's weights, for the wide tiles of large prefills
  CUtensorMap tm_Wc_wide;
  std::vector<CUtensorMap> tm_kc_wide, tm_vc_wide;
  std::vector<CUtensorMap> tm_c0, tm_c1;  // [layer*4 + which]
  float inv_freq[64];
  WsLayout ws;
  const int32_t *block_table = nullptr;  // paged caches: [max_batch][Cmax / kPageRows]
};

namespace {

void plan_workspace(dflash_handle_s *h) {
  const auto &c = h->cfg;
  WsLayout &L = h->ws;
  const int Mb = c.max_batch * c.B;                     // draft rows
  const int Mp = c.max_batch * c.max_proj_rows;         // projection rows
  const int Ml = c.max_batch * (c.B - 1);               // LM-head rows
  const int qkv_n = (c.Hq + 2 * c.Hkv) * c.hd;
  const size_t apart_max = attention_slots(c.max_batch, c.Hkv, h->num_sms);
  const size_t rows_attn = (size_t)(c.Hq / c.Hkv) * c.B;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 1));
    return o;
  };
  L.status = take(256);
  L.pre = take((size_t)Mp * c.D * 4);
  L.h = take((size_t)Mp * c.D * 2);
  L.x = take((size_t)Mb * c.D * 4);
  L.u = take((size_t)Mb * c.D * 2);
  L.qkv = take((size_t)Mb * qkv_n * 2);
  L.o = take((size_t)Mb * c.Hq * c.hd * 2);
  L.act = take((size_t)Mb * c.F * 2);
  L.xb = take((size_t)Mb * c.D * 2);
  L.ss = take((size_t)Mb * ((c.D + 127) / 128) * 4);  // deferred RMSNorm partial sums
  L.corr = take((c.flags & DFLASH_FLAG_CONV) ? (size_t)Mb * 2 * (c.D / c.conv_group) * 4 : 0);
  L.apart_ctas = apart_max;
  L.apart_bytes = apart_max * rows_attn * c.hd * 4;
  L.apart = take(L.apart_bytes);
  L.aml = take(apart_max * rows_attn * 2 * 4);
  const int ranges = h->num_sms;
  L.tk_vals = take((size_t)ranges * Ml * c.k_top * 4);
  L.tk_ids = take((size_t)ranges * Ml * c.k_top * 4);
  if (c.flags & DFLASH_FLAG_SELECT) {
    const int sel_rows = c.max_batch * (1 + (c.B - 1) * c.k_top);
    L.sel_e = take((size_t)sel_rows * c.D * 2);
    L.sel_ab = take((size_t)sel_rows * 2 * c.sel_dim * 4);
    L.sel_g = take((size_t)Ml * c.sel_dim * 4);
    L.sel_t = take((size_t)Ml * c.k_top * c.k_top * 4);  // step score tables
  }
  L.smp_part = take((size_t)std::max(Mb * kSampleMaxSlices, h->num_sms * Ml) * 32);
  L.smp_lse = take((size_t)Mb * 4);
  L.ver_part = take((size_t)c.max_batch * kSampleMaxSlices * 16);
  L.ver_nrej = take((size_t)c.max_batch * 4);
  if (c.flags & DFLASH_FLAG_FILM) {
    L.film_cond = take((size_t)Mb * 3 * c.D * 2);
    L.film_hid = take((size_t)Mb * c.film_dim * 2);
    L.film_bg = take((size_t)Mb * 2 * c.D * 4);
  }
  L.total = off;
}

struct Ws {
  uint8_t *base;
  const WsLayout &L;
  template <class T>
  T *at(size_t off) const {
    return reinterpret_cast<T *>(base + off);
  }
  int *status() const { return at<int>(L.status); }
};

int check_ws(const dflash_handle_s *h, void *ws, size_t ws_bytes) {
  if (!ws) return fail(DFLASH_ERR_INVALID_ARG, "workspace is NULL");
  if (reinterpret_cast<uintptr_t>(ws) % kAlign)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
  if (ws_bytes < h->ws.total)
    return fail(DFLASH_ERR_INVALID_ARG, "workspace too small: %zu < %zu bytes", ws_bytes, h->ws.total);
  return DFLASH_OK;
}

GemmParams base_params(const dflash_handle_s *h, const Ws &w) {
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.groups = 1;
  p.status = w.status();
  p.max_spin = h->cfg.max_spin;
  p.stall = (h->cfg.flags & DFLASH_FLAG_TEST_STALL) ? 1 : 0;
  p.hd = h->cfg.hd;
  std::memcpy(p.inv_freq, h->inv_freq, sizeof(p.inv_freq));
  return p;
}

int run_gemm(const dflash_handle_s *h, GemmParams &p, int BN, cudaStream_t s) {
  DF_CUDA(gemm_launch(p, BN, h->num_sms, s));
  return DFLASH_OK;
}

#define DF_TRY(expr)              \
  do {                            \
    int rc_ = (expr);             \
    if (rc_ != DFLASH_OK) return rc_; \
  } while (0)

const uint16_t *bf(const void *p) { return static_cast<const uint16_t *>(p); }

// Cache rows (of hd elements) of one layer: [max_batch][Hkv][Cmax], or the page pool
// [num_pages][Hkv][kPageRows].
size_t cache_layer_rows(const dflash_config &c) {
  return c.num_pages > 0 ? (size_t)c.num_pages * c.Hkv * kPageRows : (size_t)c.max_batch * c.Hkv * c.Cmax;
}
size_t cache_layer_elems(const dflash_config &c) { return cache_layer_rows(c) * c.hd; }

// A call that touches a paged cache needs the block table.
int check_paging(const dflash_handle_s *h) {
  if (h->cfg.num_pages > 0 && !h->block_table)
    return fail(DFLASH_ERR_INVALID_ARG, "paged caches need dflash_set_block_table first");
  return DFLASH_OK;
}

// Page-table fields of a GEMM that writes cache rows.
void set_paging(const dflash_handle_s *h, GemmParams &p) {
  const auto &c = h->cfg;
  p.page_table = c.num_pages > 0 ? h->block_table : nullptr;
  p.pages_per_seq = c.Cmax / kPageRows;
  p.num_pages = c.num_pages;
  p.layer_rows = (long long)cache_layer_rows(c);
}

// Attention launch parameters for nb sequences: q rows of stride ldq (elements) with
// the queries in their first Hq*hd columns, caches of every layer, output o.
int attention_params(const dflash_handle_s *h, const Ws &w, int nb, const void *q, int ldq,
                     const void *kcache, const void *vcache, const int32_t *ctx_len, int max_ctx,
                     void *o, AttnParams *out) {
  const auto &c = h->cfg;
  AttnParams &ap = *out;
  DF_TRY(encode_3d(&ap.tmQ, q, c.hd, c.Hq, (uint64_t)nb * c.B, c.hd, ldq, c.Hq / c.Hkv, c.B));
  const uint64_t cache_rows = (uint64_t)c.N * cache_layer_rows(c);
  const bool paged = c.num_pages > 0;
  // {64 of hd, cache rows, hd/64 halves}: one box = 128 rows of every half, stacked
  // half after half as the MMA reads them; paged: one box = one page (64 rows) of one half
  DF_TRY(encode_3d(&ap.tmK, kcache, 64, cache_rows, c.hd / 64, c.hd, 64, paged ? 64 : 128,
                   paged ? 1 : c.hd / 64));
  DF_TRY(encode_3d(&ap.tmV, vcache, 64, cache_rows, c.hd / 64, c.hd, 64, paged ? 64 : 128,
                   paged ? 1 : c.hd / 64));
  ap.page_table = paged ? h->block_table : nullptr;
  ap.pages_per_seq = c.Cmax / kPageRows;
  ap.num_pages = c.num_pages;
  ap.ctx_len = ctx_len;
  ap.o = static_cast<uint16_t *>(o);
  ap.part_o = w.at<float>(h->ws.apart);
  ap.part_ml = w.at<float>(h->ws.aml);
  ap.nb = nb;
  ap.B = c.B;
  ap.Hq = c.Hq;
  ap.Hkv = c.Hkv;
  ap.hd = c.hd;
  ap.Cmax = c.Cmax;
  ap.max_batch = c.max_batch;
  ap.max_ctx = max_ctx;
  ap.grid = h->num_sms;
  ap.status = w.status();
  ap.max_spin = c.max_spin;
  ap.stall = (c.flags & DFLASH_FLAG_TEST_STALL) ? 1 : 0;
  if (attention_slots(nb, c.Hkv, ap.grid) > h->ws.apart_ctas)
    return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "attention partials exceed the workspace plan");
  return DFLASH_OK;
}

// One DFlash 2 conv on the fp32 residual rows x [M, D].
// xb_ready: the bf16 copy of x (workspace xb) was written by the producer of x (a
// residual epilogue or the previous conv); write_next: also leave bf16(x') in xb for a
// conv that follows directly.
int run_conv(const dflash_handle_s *h, const Ws &w, int layer, int which, int M, float *x,
             cudaStream_t s, bool xb_ready = false, bool write_next = false) {
  const auto &c = h->cfg;
  const int ng = c.D / c.conv_group;
  uint16_t *xb = w.at<uint16_t>(w.L.xb);
  float *corr = w.at<float>(w.L.corr);
  if (!xb_ready) DF_CUDA(launch_f32_to_bf16(x, xb, (long long)M * c.D, s));
  GemmParams p = base_params(h, w);
  DF_TRY(encode_act(&p.tmA, xb, M, c.D));
  p.tmB[0] = h->tm_c0[layer * 4 + which];
  p.tmB[1] = h->tm_c1[layer * 4 + which];
  p.M = M;
  p.N = ng;
  p.K = c.D;
  p.dual = 1;
  p.epi = EPI_DUAL_F32;
  p.out = corr;
  p.ldo = 2 * ng;
  DF_TRY(run_gemm(h, p, kBN, s));
  DF_CUDA(launch_conv_apply(x, write_next ? xb : nullptr, corr, bf(h->layers[layer].conv_base[which]), M, c.D,
                            c.B, c.conv_group, s));
  return DFLASH_OK;
}

// ---------------------------------------------------------------- allocation-free LM head
//
// Scratch of dflash_lm_head_topk_noalloc: the per-range partial top-k lists (and a
// fallback status word) live in this file-scope device array instead of a
// caller-provided workspace. Every GPU that loads the library holds it until the
// process exits. Host code may not use the symbol as a device address: its device
// address is looked up once per device with cudaGetSymbolAddress.
constexpr size_t kNoallocScratchBytes = size_t(4) << 20;  // 4 MiB
static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
uint8_t *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (looked up on the
// first call for that device, with the device current).
int noalloc_scratch(int device, uint8_t **out) {
  if (device < 0 || device >= kMaxDevices) return fail(DFLASH_ERR_CUDA, "device index %d out of range", device);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_ptr[device]) {
    void *ptr = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr)
      return fail(DFLASH_ERR_CUDA, "cudaGetSymbolAddress of the scratch array failed: %s",
                  cudaGetErrorString(e));
    g_noalloc_ptr[device] = static_cast<uint8_t *>(ptr);
  }
  *out = g_noalloc_ptr[device];
  return DFLASH_OK;
}

}  // namespace

// ====================================================================== C ABI

extern "C" {

const char *dflash_last_error(void) { return g_last_error.c_str(); }

int dflash_create(const dflash_config *cfg, dflash_handle_t *out) {
  if (!cfg || !out) return fail(DFLASH_ERR_INVALID_ARG, "cfg and out must be non-NULL");
  *out = nullptr;
  const dflash_config &c = *cfg;
  if (c.D <= 0 || c.Dt <= 0 || c.L <= 0 || c.N <= 0 || c.Hq <= 0 || c.Hkv <= 0 || c.F <= 0 ||
      c.V <= 1 || c.Cmax <= 0 || c.max_batch <= 0 || c.max_proj_rows <= 0)
    return fail(DFLASH_ERR_INVALID_ARG, "every size in dflash_config must be positive");
  if (c.N > 16) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "N must be <= 16");
  if (c.hd != 64 && c.hd != 128) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "hd must be 64 or 128");
  if (c.Hq % c.Hkv) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "Hq must be a multiple of Hkv");
  if (c.B < 2 || c.B > 16) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "B must be in 2..16");
  if ((c.Hq / c.Hkv) * c.B > 128)
    return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "(Hq/Hkv)*B must be <= 128 (query rows per kv head)");
  if (c.Cmax <= c.B) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "Cmax must exceed B");
  if ((long long)c.N * c.max_batch * c.Hkv * c.Cmax >= (1LL << 31))
    return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "N*max_batch*Hkv*Cmax cache rows must be < 2^31");
  if (c.num_pages < 0) return fail(DFLASH_ERR_INVALID_ARG, "num_pages must be >= 0");
  if (c.num_pages > 0) {
    if (c.Cmax % kPageRows)
      return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "a paged cache needs Cmax %% %d == 0", kPageRows);
    if ((long long)c.N * c.num_pages * c.Hkv * kPageRows >= (1LL << 31))
      return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "N*num_pages*Hkv*%d cache rows must be < 2^31", kPageRows);
  }
  if (c.k_top < 1 || c.k_top > kTopkMax) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "k_top must be in 1..16");
  if (c.D % 64 || (c.L * c.Dt) % 64 || (c.Hq * c.hd) % 64 || c.F % 8)
    return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "D, L*Dt, Hq*hd must be multiples of 64 and F of 8");
  if (c.mask_id < 0 || c.mask_id >= c.V) return fail(DFLASH_ERR_INVALID_ARG, "mask_id outside [0, V)");
  if (!(c.eps > 0.f) || !(c.rope_base > 1.f)) return fail(DFLASH_ERR_INVALID_ARG, "eps and rope_base");
  if (c.flags & DFLASH_FLAG_CONV) {
    if (c.conv_group <= 0 || c.D % c.conv_group || (c.D / c.conv_group) % 8)
      return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "conv_group must divide D into a multiple of 8 groups");
  }
  if (c.flags & DFLASH_FLAG_SELECT) {
    if (c.sel_dim <= 0 || c.sel_dim % 32) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "sel_dim must be a multiple of 32");
  }
  if (c.flags & DFLASH_FLAG_FILM) {
    if (!(c.flags & DFLASH_FLAG_RELAY)) return fail(DFLASH_ERR_INVALID_ARG, "DFLASH_FLAG_FILM requires DFLASH_FLAG_RELAY");
    if (c.film_dim <= 0 || c.film_dim % 64) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "film_dim must be a positive multiple of 64");
  }
  if (2LL * c.N > kMaxBMaps) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "2*N must be <= 12 (grouped K/V projection)");
  auto *h = new (std::nothrow) dflash_handle_s();
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "out of host memory");
  h->cfg = c;
  if (h->cfg.max_spin <= 0) h->cfg.max_spin = 1 << 24;
  if (cudaGetDevice(&h->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device) != cudaSuccess) {
    delete h;
    return fail(DFLASH_ERR_CUDA, "no CUDA device");
  }
  for (int d = 0; d < 64; ++d)
    h->inv_freq[d] = d < c.hd / 2 ? (float)std::pow((double)c.rope_base, -2.0 * d / c.hd) : 0.f;
  plan_workspace(h);
  *out = h;
  return DFLASH_OK;
}

int dflash_destroy(dflash_handle_t h) {
  delete h;
  return DFLASH_OK;
}

int dflash_workspace_size(dflash_handle_t h, size_t *bytes) {
  if (!h || !bytes) return fail(DFLASH_ERR_INVALID_ARG, "handle and bytes must be non-NULL");
  *bytes = h->ws.total;
  return DFLASH_OK;
}

int dflash_set_weights(dflash_handle_t h, const dflash_weights *w) {
  if (!h || !w) return fail(DFLASH_ERR_INVALID_ARG, "handle and weights must be non-NULL");
  const auto &c = h->cfg;
  if (!w->W_c || !w->g_ctx || !w->E || !w->W_lm || !w->g_final || !w->layers)
    return fail(DFLASH_ERR_INVALID_ARG, "a required weight pointer is NULL");
  h->w = *w;
  h->layers.assign(w->layers, w->layers + c.N);
  h->w.layers = h->layers.data();
  const int qkv_n = (c.Hq + 2 * c.Hkv) * c.hd;
  DF_TRY(encode_slabs(&h->tm_Wc, w->W_c, c.D, (uint64_t)c.L * c.Dt, kBN));
  DF_TRY(encode_2d(&h->tm_Wc_wide, w->W_c, c.D, (uint64_t)c.L * c.Dt, (uint64_t)c.L * c.Dt, kBNWide));
  h->tm_kc_wide.resize(c.N);
  h->tm_vc_wide.resize(c.N);
  DF_TRY(encode_2d(&h->tm_lm, w->W_lm, c.V, c.D, c.D, kBNTopk));
  h->tm_qkv.resize(c.N);
  h->tm_kc.resize(c.N);
  h->tm_vc.resize(c.N);
  h->tm_o.resize(c.N);
  h->tm_gate.resize(c.N);
  h->tm_up.resize(c.N);
  h->tm_down.resize(c.N);
  h->tm_c0.resize(4 * c.N);
  h->tm_c1.resize(4 * c.N);
  for (int n = 0; n < c.N; ++n) {
    const dflash_layer_weights &L = h->layers[n];
    if (!L.W_qkv || !L.Wk_c || !L.Wv_c || !L.W_o || !L.W_gate || !L.W_up || !L.W_down || !L.g_attn ||
        !L.g_ffn)
      return fail(DFLASH_ERR_INVALID_ARG, "layer %d: a weight pointer is NULL", n);
    DF_TRY(encode_slabs(&h->tm_qkv[n], L.W_qkv, qkv_n, c.D, kBN));
    DF_TRY(encode_slabs(&h->tm_kc[n], L.Wk_c, (uint64_t)c.Hkv * c.hd, c.D, kBN));
    DF_TRY(encode_slabs(&h->tm_vc[n], L.Wv_c, (uint64_t)c.Hkv * c.hd, c.D, kBN));
    DF_TRY(encode_2d(&h->tm_kc_wide[n], L.Wk_c, (uint64_t)c.Hkv * c.hd, c.D, c.D, kBNWide));
    DF_TRY(encode_2d(&h->tm_vc_wide[n], L.Wv_c, (uint64_t)c.Hkv * c.hd, c.D, c.D, kBNWide));
    DF_TRY(encode_slabs(&h->tm_o[n], L.W_o, c.D, (uint64_t)c.Hq * c.hd, kBN));
    DF_TRY(encode_2d(&h->tm_gate[n], L.W_gate, c.F, c.D, c.D, kBNGateUp / 2));
    DF_TRY(encode_2d(&h->tm_up[n], L.W_up, c.F, c.D, c.D, kBNGateUp / 2));
    if (c.F % 64 == 0)
      DF_TRY(encode_slabs(&h->tm_down[n], L.W_down, c.D, c.F, kBN));
    else
      DF_TRY(encode_2d(&h->tm_down[n], L.W_down, c.D, c.F, c.F, kBN));
    if (c.flags & DFLASH_FLAG_CONV) {
      for (int q = 0; q < 4; ++q) {
        if (!L.conv_W0[q] || !L.conv_W1[q] || !L.conv_base[q])
          return fail(DFLASH_ERR_INVALID_ARG, "layer %d conv %d: a weight pointer is NULL", n, q);
        DF_TRY(encode_2d(&h->tm_c0[4 * n + q], L.conv_W0[q], c.D / c.conv_group, c.D, c.D, kBN / 2));
        DF_TRY(encode_2d(&h->tm_c1[4 * n + q], L.conv_W1[q], c.D / c.conv_group, c.D, c.D, kBN / 2));
      }
    }
  }
  if (c.flags & DFLASH_FLAG_SELECT) {
    if (!w->W_A || !w->W_B || !w->W_G) return fail(DFLASH_ERR_INVALID_ARG, "selector weights are NULL");
    DF_TRY(encode_2d(&h->tm_A, w->W_A, c.sel_dim, c.D, c.D, kBN / 2));
    DF_TRY(encode_2d(&h->tm_B, w->W_B, c.sel_dim, c.D, c.D, kBN / 2));
    DF_TRY(encode_2d(&h->tm_G, w->W_G, c.sel_dim, c.D, c.D, kBN));
  }
  if (c.flags & DFLASH_FLAG_FILM) {
    if (!w->film_W1 || !w->film_W2) return fail(DFLASH_ERR_INVALID_ARG, "FiLM relay weights are NULL");
    DF_TRY(encode_slabs(&h->tm_f1, w->film_W1, c.film_dim, 3ULL * c.D, kBN));
    DF_TRY(encode_slabs(&h->tm_f2, w->film_W2, 2ULL * c.D, c.film_dim, kBN));
  }
  h->have_weights = true;
  return DFLASH_OK;
}

int dflash_set_block_table(dflash_handle_t h, const int32_t *table) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle must be non-NULL");
  if (h->cfg.num_pages <= 0) return fail(DFLASH_ERR_INVALID_ARG, "the handle's caches are not paged");
  if (!table || reinterpret_cast<uintptr_t>(table) % 4)
    return fail(DFLASH_ERR_INVALID_ARG, "block table must be a non-NULL 4-byte aligned device pointer");
  h->block_table = table;
  return DFLASH_OK;
}

int dflash_status(dflash_handle_t h, void *ws, dflash_stream_t stream, int *code) {
  if (!h || !ws || !code) return fail(DFLASH_ERR_INVALID_ARG, "handle, ws and code must be non-NULL");
  int v = 0;
  DF_CUDA(cudaStreamSynchronize(stream));
  DF_CUDA(cudaMemcpy(&v, static_cast<uint8_t *>(ws) + h->ws.status, sizeof(int), cudaMemcpyDeviceToHost));
  DF_CUDA(cudaMemset(static_cast<uint8_t *>(ws) + h->ws.status, 0, sizeof(int)));
  *code = (v & kStatusTimeout) ? DFLASH_ERR_TIMEOUT : (v & kStatusCheck) ? DFLASH_ERR_DEVICE_CHECK : DFLASH_OK;
  return DFLASH_OK;
}

namespace {

// relay_b / relay_y non-null selects the FiLM form of the relay rows.
int ctx_project_impl(dflash_handle_t h, int nb, int R, const void *hv, const int32_t *n_commit,
                     const int32_t *relay_a, const int32_t *relay_b, const int32_t *relay_y,
                     int32_t *ctx_len, void *kcache, void *vcache, void *x0_relay, void *ws,
                     size_t ws_bytes, dflash_stream_t stream) {
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (R < 0 || R > c.max_proj_rows) return fail(DFLASH_ERR_INVALID_ARG, "R=%d outside [0, max_proj_rows]", R);
  if (nb == 0 || R == 0) return DFLASH_OK;
  DF_TRY(check_paging(h));
  if (!hv || !n_commit || !ctx_len || !kcache || !vcache)
    return fail(DFLASH_ERR_INVALID_ARG, "hv, n_commit, ctx_len and the caches must be non-NULL");
  if (relay_a && !(c.flags & DFLASH_FLAG_RELAY))
    return fail(DFLASH_ERR_INVALID_ARG, "relay_a given but DFLASH_FLAG_RELAY is not set");
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  cudaStream_t s = stream;
  const int rows = nb * R;
  float *pre = w.at<float>(h->ws.pre);
  uint16_t *hh = w.at<uint16_t>(h->ws.h);
  {  // pre = hv * W_c^T
    GemmParams p = base_params(h, w);
    const bool wide = wide_tiles(h->num_sms, rows, c.D, 1, EPI_F32);
    if (wide) {
      DF_TRY(encode_act(&p.tmA, hv, rows, (uint64_t)c.L * c.Dt));
      p.slabs = 1;
      p.tmB[0] = h->tm_Wc_wide;
    } else {
      DF_TRY(encode_slabs(&p.tmA, hv, rows, (uint64_t)c.L * c.Dt, 128));
      p.slabs = 2;
      p.tmB[0] = h->tm_Wc;
    }
    p.M = rows;
    p.N = c.D;
    p.K = c.L * c.Dt;
    p.epi = EPI_F32;
    p.out = pre;
    p.ldo = c.D;
    DF_TRY(run_gemm(h, p, wide ? kBNWide : kBN, s));
  }
  DF_CUDA(launch_rmsnorm(pre, rows, c.D, bf(h->w.g_ctx), c.eps, hh, s));
  {  // K_c / V_c of every layer, scattered into the caches (committed rows only)
    GemmParams p = base_params(h, w);
    const bool wide = wide_tiles(h->num_sms, rows, c.Hkv * c.hd, 2 * c.N, EPI_KV);
    if (wide) {
      DF_TRY(encode_act(&p.tmA, hh, rows, c.D));
      p.slabs = 1;
    } else {
      DF_TRY(encode_slabs(&p.tmA, hh, rows, c.D, 128));
      p.slabs = 2;
    }
    for (int n = 0; n < c.N; ++n) {
      p.tmB[2 * n] = wide ? h->tm_kc_wide[n] : h->tm_kc[n];
      p.tmB[2 * n + 1] = wide ? h->tm_vc_wide[n] : h->tm_vc[n];
    }
    p.groups = 2 * c.N;
    p.M = rows;
    p.N = c.Hkv * c.hd;
    p.K = c.D;
    p.epi = EPI_KV;
    p.ctx_len = ctx_len;
    p.rows_per_seq = R;
    p.kc = kcache;
    p.vc = vcache;
    p.n_commit = n_commit;
    p.Hkv = c.Hkv;
    p.Cmax = c.Cmax;
    p.max_batch = c.max_batch;
    set_paging(h, p);
    DF_TRY(run_gemm(h, p, wide ? kBNWide : kBN, s));
  }
  const bool film = relay_b != nullptr;
  DF_CUDA(launch_relay_and_len(hh, nb, R, c.B, c.D, relay_a, n_commit, ctx_len,
                               film ? nullptr : static_cast<uint16_t *>(x0_relay), c.Cmax,
                               w.status(), s));
  if (film) {
    const int M = nb * c.B;
    uint16_t *cond = w.at<uint16_t>(h->ws.film_cond);
    uint16_t *hid = w.at<uint16_t>(h->ws.film_hid);
    float *bg = w.at<float>(h->ws.film_bg);
    DF_CUDA(launch_film_cond(hh, bf(h->w.E), nb, R, c.B, c.D, c.V, relay_a, relay_b, relay_y, cond,
                             w.status(), s));
    {  // hidden = silu(W1 cond)
      GemmParams p = base_params(h, w);
      DF_TRY(encode_slabs(&p.tmA, cond, M, 3ULL * c.D, 128));
      p.slabs = 2;
      p.tmB[0] = h->tm_f1;
      p.M = M;
      p.N = c.film_dim;
      p.K = 3 * c.D;
      p.epi = EPI_BF16;
      p.act = 1;
      p.out = hid;
      p.ldo = c.film_dim;
      DF_TRY(run_gemm(h, p, kBN, s));
    }
    {  // [beta | gamma] = W2 hidden
      GemmParams p = base_params(h, w);
      DF_TRY(encode_slabs(&p.tmA, hid, M, c.film_dim, 128));
      p.slabs = 2;
      p.tmB[0] = h->tm_f2;
      p.M = M;
      p.N = 2 * c.D;
      p.K = c.film_dim;
      p.epi = EPI_F32;
      p.out = bg;
      p.ldo = 2 * c.D;
      DF_TRY(run_gemm(h, p, kBN, s));
    }
    DF_CUDA(launch_film_apply(hh, bg, nb, R, c.B, c.D, relay_a, c.eps,
                              static_cast<uint16_t *>(x0_relay), s));
  }
  return DFLASH_OK;
}

}  // namespace

int dflash_ctx_project(dflash_handle_t h, int nb, int R, const void *hv, const int32_t *n_commit,
                       const int32_t *relay_a, int32_t *ctx_len, void *kcache, void *vcache,
                       void *x0_relay, void *ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  return ctx_project_impl(h, nb, R, hv, n_commit, relay_a, nullptr, nullptr, ctx_len, kcache,
                          vcache, x0_relay, ws, ws_bytes, stream);
}

int dflash_ctx_project_film(dflash_handle_t h, int nb, int R, const void *hv,
                            const int32_t *n_commit, const int32_t *relay_a, const int32_t *relay_b,
                            const int32_t *relay_y, int32_t *ctx_len, void *kcache, void *vcache,
                            void *x0_relay, void *ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  const unsigned need = DFLASH_FLAG_RELAY | DFLASH_FLAG_FILM;
  if ((h->cfg.flags & need) != need)
    return fail(DFLASH_ERR_INVALID_ARG, "the FiLM relay needs DFLASH_FLAG_RELAY | DFLASH_FLAG_FILM");
  if (!relay_a || !relay_b || !relay_y || !x0_relay)
    return fail(DFLASH_ERR_INVALID_ARG, "relay_a, relay_b, relay_y and x0_relay must be non-NULL");
  return ctx_project_impl(h, nb, R, hv, n_commit, relay_a, relay_b, relay_y, ctx_len, kcache,
                          vcache, x0_relay, ws, ws_bytes, stream);
}

int dflash_draft_block(dflash_handle_t h, int nb, const int32_t *block_ids, const void *x0_relay,
                       void *kcache, void *vcache, const int32_t *ctx_len,
                       int max_ctx_hint, void *out_hidden, void *ws, size_t ws_bytes,
                       dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (nb == 0) return DFLASH_OK;
  if (!block_ids || !kcache || !vcache || !ctx_len || !out_hidden)
    return fail(DFLASH_ERR_INVALID_ARG, "block_ids, caches, ctx_len and out_hidden must be non-NULL");
  DF_TRY(check_paging(h));
  if (x0_relay && !(c.flags & DFLASH_FLAG_RELAY))
    return fail(DFLASH_ERR_INVALID_ARG, "x0_relay given but DFLASH_FLAG_RELAY is not set");
  if (max_ctx_hint < 0 || max_ctx_hint > c.Cmax)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ctx_hint=%d outside [0, Cmax]", max_ctx_hint);
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  cudaStream_t s = stream;
  const bool conv = (c.flags & DFLASH_FLAG_CONV) != 0;
  const int M = nb * c.B;
  const int qkv_n = (c.Hq + 2 * c.Hkv) * c.hd;
  const int max_ctx = max_ctx_hint > 0 ? std::min(max_ctx_hint, c.Cmax - c.B) : c.Cmax - c.B;
  float *x = w.at<float>(h->ws.x);
  uint16_t *u = w.at<uint16_t>(h->ws.u);
  uint16_t *qkv = w.at<uint16_t>(h->ws.qkv);
  uint16_t *o = w.at<uint16_t>(h->ws.o);
  uint16_t *act = w.at<uint16_t>(h->ws.act);

  CUtensorMap tm_u, tm_u2, tm_o, tm_act;
  const bool down_slabs = c.F % 64 == 0;
  DF_TRY(encode_act(&tm_u, u, M, c.D));          // gate|up (one slab per stage)
  DF_TRY(encode_slabs(&tm_u2, u, M, c.D, 128));  // QKV
  DF_TRY(encode_slabs(&tm_o, o, M, (uint64_t)c.Hq * c.hd, 128));
  if (down_slabs)
    DF_TRY(encode_slabs(&tm_act, act, M, c.F, 128));
  else
    DF_TRY(encode_act(&tm_act, act, M, c.F));

  DF_CUDA(launch_embed_rmsnorm(block_ids, bf(h->w.E), static_cast<const uint16_t *>(x0_relay), M, c.D,
                               c.V, x, conv ? nullptr : bf(h->layers[0].g_attn), c.eps, u, w.status(), s));
  AttnParams ap{};
  DF_TRY(attention_params(h, w, nb, qkv, qkv_n, kcache, vcache, ctx_len, max_ctx, o, &ap));

  // Without the DFlash 2 convs the pre-norms after layer 0's attention norm are deferred:
  // the residual GEMMs write u = bf16(x * g) and partial sums of x^2 (ss), and the next
  // GEMM (gate|up, or the next layer's QKV) scales its rows by rsqrt(mean x^2 + eps).
  // With the convs, x changes after those epilogues, so the norms stay separate kernels.
  const bool deferred = !conv;
  float *ss = w.at<float>(h->ws.ss);
  const int ss_n = (c.D + kBN - 1) / kBN;
  auto defer_out = [&](GemmParams &p, const void *g_next) {
    if (!deferred || !g_next) return;
    p.xg_out = u;
    p.g_next = static_cast<const uint16_t *>(g_next);
    p.ss_out = ss;
  };
  auto defer_in = [&](GemmParams &p) {
    if (!deferred) return;
    p.ss_in = ss;
    p.ss_n = ss_n;
    p.inv_d = 1.0f / static_cast<float>(c.D);
    p.eps = c.eps;
  };
  for (int n = 0; n < c.N; ++n) {
    const dflash_layer_weights &Lw = h->layers[n];
    if (conv) {
      DF_TRY(run_conv(h, w, n, 0, M, x, s, /*xb_ready=*/n > 0));
      DF_CUDA(launch_rmsnorm(x, M, c.D, bf(Lw.g_attn), c.eps, u, s));
    }
    uint16_t *kc_n = static_cast<uint16_t *>(kcache) + n * cache_layer_elems(c);
    uint16_t *vc_n = static_cast<uint16_t *>(vcache) + n * cache_layer_elems(c);
    {  // q -> qkv buffer; k_b, v_b -> cache rows ctx_len + j; RoPE on q and k_b
      GemmParams p = base_params(h, w);
      p.tmA = tm_u2;
      p.slabs = 2;
      p.tmB[0] = h->tm_qkv[n];
      p.M = M;
      p.N = qkv_n;
      p.K = c.D;
      p.epi = EPI_ROPE;
      p.out = qkv;
      p.ldo = qkv_n;
      p.ctx_len = ctx_len;
      p.rows_per_seq = c.B;
      p.rope_cols = (c.Hq + c.Hkv) * c.hd;
      p.q_cols = c.Hq * c.hd;
      p.kc = kc_n;
      p.vc = vc_n;
      p.Hkv = c.Hkv;
      p.Cmax = c.Cmax;
      set_paging(h, p);
      if (n > 0) defer_in(p);
      DF_TRY(run_gemm(h, p, kBN, s));
    }
    ap.layer_row0 = static_cast<int>(n * cache_layer_rows(c));
    DF_CUDA(launch_attention(ap, s));
    {  // x += o W_O^T
      GemmParams p = base_params(h, w);
      p.tmA = tm_o;
      p.slabs = 2;
      p.tmB[0] = h->tm_o[n];
      p.M = M;
      p.N = c.D;
      p.K = c.Hq * c.hd;
      p.epi = EPI_RESID;
      p.xres = x;
      p.ldo = c.D;
      defer_out(p, Lw.g_ffn);
      if (conv) p.xg_out = w.at<uint16_t>(w.L.xb);  // bf16(x) for conv1
      DF_TRY(run_gemm(h, p, kBN, s));
    }
    if (conv) {
      DF_TRY(run_conv(h, w, n, 1, M, x, s, true, /*write_next=*/true));
      DF_TRY(run_conv(h, w, n, 2, M, x, s, true));
      DF_CUDA(launch_rmsnorm(x, M, c.D, bf(Lw.g_ffn), c.eps, u, s));
    }
    {  // act = silu(u W_gate^T) * (u W_up^T)
      GemmParams p = base_params(h, w);
      p.tmA = tm_u;
      p.tmB[0] = h->tm_gate[n];
      p.tmB[1] = h->tm_up[n];
      p.dual = 1;
      p.M = M;
      p.N = c.F;
      p.K = c.D;
      p.epi = EPI_SWIGLU;
      p.out = act;
      p.ldo = c.F;
      defer_in(p);
      DF_TRY(run_gemm(h, p, kBNGateUp, s));
    }
    {  // x += act W_down^T
      GemmParams p = base_params(h, w);
      p.tmA = tm_act;
      p.slabs = down_slabs ? 2 : 1;
      p.tmB[0] = h->tm_down[n];
      p.M = M;
      p.N = c.D;
      p.K = c.F;
      p.epi = EPI_RESID;
      p.xres = x;
      p.ldo = c.D;
      if (n + 1 < c.N) defer_out(p, h->layers[n + 1].g_attn);
      if (conv) p.xg_out = w.at<uint16_t>(w.L.xb);  // bf16(x) for conv3
      DF_TRY(run_gemm(h, p, kBN, s));
    }
    if (conv) DF_TRY(run_conv(h, w, n, 3, M, x, s, true, /*write_next=*/n + 1 < c.N));
  }
  DF_CUDA(launch_rmsnorm(x, M, c.D, bf(h->w.g_final), c.eps, static_cast<uint16_t *>(out_hidden), s));
  return DFLASH_OK;
}

namespace {

// LM head on block offsets 1..B-1 with the fused top-k; with temperature > 0 also the fused
// draw (out_cand, out_lse, out_logq). out_ids == NULL skips the top-k merge.
int lm_head_impl(dflash_handle_t h, int nb, const void *hidden, int k, int32_t *out_ids,
                 float *out_vals, float *out_logits, float temperature, uint64_t seed,
                 int32_t *out_cand, float *out_lse, float *out_logq, void *ws, size_t ws_bytes,
                 cudaStream_t s) {
  const auto &c = h->cfg;
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  const int R = c.B - 1;
  const int S = 128 / R;
  const int Ml = nb * R;
  GemmParams p = base_params(h, w);
  // rows 1..B-1 of every block: 3D map {D, B-1, nb} starting at row 1
  DF_TRY(encode_3d(&p.tmA, static_cast<const uint16_t *>(hidden) + c.D, c.D, R, nb, c.D,
                   (uint64_t)c.B * c.D, R, S));
  p.tmB[0] = h->tm_lm;
  p.a_grouped = 1;
  p.a_S = S;
  p.tile_rows = S * R;
  p.M = Ml;
  p.N = c.V;
  p.K = c.D;
  p.epi = EPI_TOPK;
  p.topk_k = k;
  p.part_vals = w.at<float>(h->ws.tk_vals);
  p.part_ids = w.at<int>(h->ws.tk_ids);
  p.logits_out = out_logits;
  if (temperature > 0.f) {
    p.smp_part = w.at<float4>(h->ws.smp_part);
    p.smp_inv_T = 1.f / temperature;
    p.smp_stream = 0;
    p.smp_seed = seed;
  }
  // the per-range partial lists in the workspace hold num_sms ranges: check the plan
  // before the launch writes them
  int tpc = 0, ranges = 0;
  const int ms = gemm_mstack(EPI_TOPK, kBNTopk, Ml, p.tile_rows, c.V, 1, 1, 0, h->num_sms);
  topk_range_plan((c.V + kBNTopk - 1) / kBNTopk, (Ml + ms * p.tile_rows - 1) / (ms * p.tile_rows), h->num_sms,
                  &tpc, &ranges);
  if (ranges > h->num_sms) return fail(DFLASH_ERR_UNSUPPORTED_SHAPE, "top-k ranges exceed the workspace plan");
  DF_TRY(run_gemm(h, p, kBNTopk, s));
  if (p.items / p.m_tiles != ranges) return fail(DFLASH_ERR_CUDA, "LM-head range plan mismatch");
  if (out_ids)
    DF_CUDA(launch_topk_merge(p.part_vals, p.part_ids, Ml, k, k, (long long)Ml * k, ranges, k, out_ids,
                              out_vals, s));
  if (temperature > 0.f)
    DF_CUDA(launch_draw_merge(p.smp_part, Ml, ranges, 1, Ml, out_cand, out_lse,
                              out_logq ? out_logq : w.at<float>(h->ws.smp_lse), s));
  return DFLASH_OK;
}

}  // namespace

int dflash_lm_head_topk(dflash_handle_t h, int nb, const void *hidden, int k, int32_t *out_ids,
                        float *out_vals, float *out_logits, void *ws, size_t ws_bytes,
                        dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (k < 1 || k > c.k_top) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, k_top]", k);
  if (nb == 0) return DFLASH_OK;
  if (!hidden || !out_ids || !out_vals) return fail(DFLASH_ERR_INVALID_ARG, "hidden and outputs must be non-NULL");
  return lm_head_impl(h, nb, hidden, k, out_ids, out_vals, out_logits, 0.f, 0, nullptr, nullptr, nullptr,
                      ws, ws_bytes, stream);
}

int dflash_lm_head_sample(dflash_handle_t h, int nb, const void *hidden, float temperature,
                          uint64_t seed, int32_t *out_cand, float *out_lse, float *out_logq,
                          float *out_logits, int k, int32_t *out_ids, float *out_vals, void *ws,
                          size_t ws_bytes, dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be positive and finite");
  if (out_ids && (k < 1 || k > c.k_top)) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, k_top]", k);
  if (out_ids && !out_vals) return fail(DFLASH_ERR_INVALID_ARG, "out_vals must accompany out_ids");
  if (nb == 0) return DFLASH_OK;
  if (!hidden || !out_cand || !out_lse) return fail(DFLASH_ERR_INVALID_ARG, "hidden, out_cand and out_lse must be non-NULL");
  return lm_head_impl(h, nb, hidden, out_ids ? k : c.k_top, out_ids, out_vals, out_logits, temperature,
                      seed, out_cand, out_lse, out_logq, ws, ws_bytes, stream);
}

int dflash_draw_gumbel(int n, uint64_t seed, int stream_id, int row, float *out_u, float *out_g,
                       dflash_stream_t stream) {
  if (n < 0 || stream_id < 0 || row < 0) return fail(DFLASH_ERR_INVALID_ARG, "n, stream_id and row must be >= 0");
  if (n == 0) return DFLASH_OK;
  if (!out_u || !out_g) return fail(DFLASH_ERR_INVALID_ARG, "out_u and out_g must be non-NULL");
  DF_CUDA(launch_draw_gumbel(n, seed, stream_id, row, out_u, out_g, stream));
  return DFLASH_OK;
}

int dflash_lm_head_topk_noalloc(dflash_handle_t h, int nb, const void *hidden, int k, int32_t *out_ids,
                                float *out_vals, int32_t *out_status, dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (k < 1 || k > c.k_top) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, k_top]", k);
  if (nb == 0) return DFLASH_OK;
  if (!hidden || !out_ids || !out_vals) return fail(DFLASH_ERR_INVALID_ARG, "hidden and outputs must be non-NULL");
  int dev = 0;
  DF_CUDA(cudaGetDevice(&dev));
  uint8_t *scratch = nullptr;
  DF_TRY(noalloc_scratch(dev, &scratch));
  const int R = c.B - 1;
  const int S = 128 / R;
  const int Ml = nb * R;
  // The LM-head launch's own work split (vocabulary ranges x row tiles), from the planner
  // the launch uses, so the size check below holds for what the kernel writes.
  const int ms = gemm_mstack(EPI_TOPK, kBNTopk, Ml, S * R, c.V, 1, 1, 0, h->num_sms);
  const int m_tiles = (Ml + ms * S * R - 1) / (ms * S * R);
  const int n_tiles = (c.V + kBNTopk - 1) / kBNTopk;
  int tpc = 0, ranges = 0;
  topk_range_plan(n_tiles, m_tiles, h->num_sms, &tpc, &ranges);
  const size_t list_bytes = (size_t)ranges * Ml * k * sizeof(float);
  const size_t need = 256 + 2 * list_bytes;
  if (need > kNoallocScratchBytes)
    return fail(DFLASH_ERR_UNSUPPORTED_SHAPE,
                "dflash_lm_head_topk_noalloc needs %zu bytes of scratch (%d ranges x %d rows x k=%d); "
                "its static scratch holds %zu bytes",
                need, ranges, Ml, k, kNoallocScratchBytes);
  cudaStream_t s = stream;
  int *status = reinterpret_cast<int *>(scratch);
  if (out_status) {
    status = out_status;
  } else {
    DF_CUDA(cudaMemsetAsync(status, 0, sizeof(int), s));  // the array keeps the last call's word
  }
  GemmParams p;
  std::memset(&p, 0, sizeof(p));
  p.groups = 1;
  p.status = status;
  p.max_spin = c.max_spin;
  p.stall = (c.flags & DFLASH_FLAG_TEST_STALL) ? 1 : 0;
  p.hd = c.hd;
  DF_TRY(encode_3d(&p.tmA, static_cast<const uint16_t *>(hidden) + c.D, c.D, R, nb, c.D,
                   (uint64_t)c.B * c.D, R, S));
  p.tmB[0] = h->tm_lm;
  p.a_grouped = 1;
  p.a_S = S;
  p.tile_rows = S * R;
  p.M = Ml;
  p.N = c.V;
  p.K = c.D;
  p.epi = EPI_TOPK;
  p.topk_k = k;
  p.part_vals = reinterpret_cast<float *>(scratch + 256);
  p.part_ids = reinterpret_cast<int *>(scratch + 256 + list_bytes);
  DF_CUDA(gemm_launch(p, kBNTopk, h->num_sms, s));
  // gemm_launch planned with topk_range_plan on the same (n_tiles, m_tiles, num_sms), so the
  // ranges it launched are the ones checked above
  if (p.items / p.m_tiles != ranges || p.m_tiles != m_tiles)
    return fail(DFLASH_ERR_CUDA, "LM-head range plan mismatch");
  DF_CUDA(launch_topk_merge(p.part_vals, p.part_ids, Ml, k, k, (long long)Ml * k, ranges, k, out_ids,
                            out_vals, s));
  return DFLASH_OK;
}

int dflash_attention(dflash_handle_t h, int nb, int layer, const void *q, const void *kcache,
                     const void *vcache, const int32_t *ctx_len, int max_ctx_hint, void *out_o, void *ws,
                     size_t ws_bytes, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (layer < 0 || layer >= c.N) return fail(DFLASH_ERR_INVALID_ARG, "layer=%d outside [0, N)", layer);
  if (max_ctx_hint < 0 || max_ctx_hint > c.Cmax)
    return fail(DFLASH_ERR_INVALID_ARG, "max_ctx_hint=%d outside [0, Cmax]", max_ctx_hint);
  if (nb == 0) return DFLASH_OK;
  if (!q || !kcache || !vcache || !ctx_len || !out_o) return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor");
  DF_TRY(check_paging(h));
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  const int max_ctx = max_ctx_hint > 0 ? std::min(max_ctx_hint, c.Cmax - c.B) : c.Cmax - c.B;
  AttnParams ap{};
  DF_TRY(attention_params(h, w, nb, q, c.Hq * c.hd, kcache, vcache, ctx_len, max_ctx, out_o, &ap));
  ap.layer_row0 = static_cast<int>(layer * cache_layer_rows(c));
  DF_CUDA(launch_attention(ap, stream));
  return DFLASH_OK;
}

int dflash_topk(dflash_handle_t h, int rows, int cols, const float *logits, int k, int32_t *out_ids,
                float *out_vals, void *ws, size_t ws_bytes, dflash_stream_t stream) {
  (void)ws;
  (void)ws_bytes;
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  if (rows < 0 || cols < 1 || k < 1 || k > kTopkMax || k > cols)
    return fail(DFLASH_ERR_INVALID_ARG, "rows=%d cols=%d k=%d", rows, cols, k);
  if (rows == 0) return DFLASH_OK;
  if (!logits || !out_ids || !out_vals) return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor");
  DF_CUDA(launch_topk_merge(logits, nullptr, rows, cols, cols, 0, 1, k, out_ids, out_vals, stream));
  return DFLASH_OK;
}

int dflash_accept(dflash_handle_t h, int nb, const int32_t *draft, const int32_t *target,
                  int32_t *out_tau, int32_t *out_bonus, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  if (nb < 0) return fail(DFLASH_ERR_INVALID_ARG, "nb < 0");
  if (nb == 0) return DFLASH_OK;
  if (!draft || !target || !out_tau || !out_bonus) return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor");
  DF_CUDA(launch_accept(draft, 1, target, nb, h->cfg.B, out_tau, out_bonus, stream));
  return DFLASH_OK;
}

int dflash_accept_topk(dflash_handle_t h, int nb, const int32_t *topk_ids, int k, const int32_t *target,
                       int32_t *out_tau, int32_t *out_bonus, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  if (nb < 0) return fail(DFLASH_ERR_INVALID_ARG, "nb < 0");
  if (k < 1 || k > kTopkMax) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside 1..%d", k, kTopkMax);
  if (nb == 0) return DFLASH_OK;
  if (!topk_ids || !target || !out_tau || !out_bonus) return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor");
  DF_CUDA(launch_accept(topk_ids, k, target, nb, h->cfg.B, out_tau, out_bonus, stream));
  return DFLASH_OK;
}

int dflash_sample(dflash_handle_t h, int rows, const float *logits, float temperature,
                  uint64_t seed, int row0, int32_t *out_ids, float *out_lse, float *out_logq,
                  void *ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  const auto &c = h->cfg;
  if (rows < 0 || rows > c.max_batch * c.B)
    return fail(DFLASH_ERR_INVALID_ARG, "rows=%d outside [0, max_batch*B]", rows);
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be positive and finite");
  if (row0 < 0) return fail(DFLASH_ERR_INVALID_ARG, "row0 must be >= 0");
  if (rows == 0) return DFLASH_OK;
  if (!logits || !out_ids || !out_lse) return fail(DFLASH_ERR_INVALID_ARG, "logits, out_ids and out_lse must be non-NULL");
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  const int S = sample_slices(rows, c.V, h->num_sms);
  DF_CUDA(launch_sample(logits, c.V, rows, c.V, 1.f / temperature, seed, 0, row0, S,
                        w.at<float4>(h->ws.smp_part), out_ids, out_lse,
                        out_logq ? out_logq : w.at<float>(h->ws.smp_lse), stream));
  return DFLASH_OK;
}

int dflash_verify_sample(dflash_handle_t h, int nb, const float *draft_logits, const float *draft_lse,
                         const int32_t *cand, const float *target_logits, float temperature,
                         uint64_t seed, int32_t *out_tau, int32_t *out_token, void *ws,
                         size_t ws_bytes, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be positive and finite");
  if (nb == 0) return DFLASH_OK;
  if (!draft_logits || !draft_lse || !cand || !target_logits || !out_tau || !out_token)
    return fail(DFLASH_ERR_INVALID_ARG, "every verify argument must be non-NULL");
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  const float inv_T = 1.f / temperature;
  const int rows = nb * c.B;
  float *tlse = w.at<float>(h->ws.smp_lse);
  DF_CUDA(launch_sample(target_logits, c.V, rows, c.V, inv_T, seed, -1, 0,
                        sample_slices(rows, c.V, h->num_sms), w.at<float4>(h->ws.smp_part), nullptr,
                        tlse, nullptr, stream));
  DF_CUDA(launch_verify(draft_logits, draft_lse, cand, target_logits, tlse, nb, c.B, c.V, inv_T, seed,
                        sample_slices(nb, c.V, h->num_sms), w.at<float4>(h->ws.ver_part),
                        w.at<int>(h->ws.ver_nrej), out_tau, out_token, stream));
  return DFLASH_OK;
}

int dflash2_conv(dflash_handle_t h, int layer, int which, int nb, float *x, void *ws, size_t ws_bytes,
                 dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  const auto &c = h->cfg;
  if (!(c.flags & DFLASH_FLAG_CONV)) return fail(DFLASH_ERR_INVALID_ARG, "DFLASH_FLAG_CONV is not set");
  if (layer < 0 || layer >= c.N || which < 0 || which > 3)
    return fail(DFLASH_ERR_INVALID_ARG, "layer=%d which=%d", layer, which);
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (nb == 0) return DFLASH_OK;
  if (!x) return fail(DFLASH_ERR_INVALID_ARG, "x is NULL");
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  return run_conv(h, w, layer, which, nb * c.B, x, stream);
}

namespace {

// The selector's scores for every (offset, previous candidate, candidate), then the greedy
// walk (walk_logq == NULL) or the sampling walk at temperature T.
int select_impl(dflash_handle_t h, int nb, int k, const int32_t *topk_ids, const float *topk_vals,
                const void *hidden, const int32_t *block_ids, float temperature, uint64_t seed,
                int32_t *out_path, float *walk_logq, void *ws, size_t ws_bytes, cudaStream_t s) {
  const auto &c = h->cfg;
  if (!(c.flags & DFLASH_FLAG_SELECT)) return fail(DFLASH_ERR_INVALID_ARG, "DFLASH_FLAG_SELECT is not set");
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (k < 1 || k > c.k_top) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, k_top]", k);
  if (nb == 0) return DFLASH_OK;
  if (!topk_ids || !topk_vals || !hidden || !block_ids || !out_path)
    return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor");
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  const int per = 1 + (c.B - 1) * k;
  const int rows = nb * per;
  uint16_t *eg = w.at<uint16_t>(h->ws.sel_e);
  float *ab = w.at<float>(h->ws.sel_ab);
  float *gp = w.at<float>(h->ws.sel_g);
  DF_CUDA(launch_gather_select(block_ids, topk_ids, nb, c.B, k, bf(h->w.E), c.D, c.V, eg, w.status(), s));
  {  // A | B projections of the gathered embeddings
    GemmParams p = base_params(h, w);
    DF_TRY(encode_act(&p.tmA, eg, rows, c.D));
    p.tmB[0] = h->tm_A;
    p.tmB[1] = h->tm_B;
    p.dual = 1;
    p.M = rows;
    p.N = c.sel_dim;
    p.K = c.D;
    p.epi = EPI_DUAL_F32;
    p.out = ab;
    p.ldo = 2 * c.sel_dim;
    DF_TRY(run_gemm(h, p, kBN, s));
  }
  {  // G pre-activation from the hidden rows of offsets 1..B-1
    const int R = c.B - 1;
    const int S = 128 / R;
    GemmParams p = base_params(h, w);
    DF_TRY(encode_3d(&p.tmA, static_cast<const uint16_t *>(hidden) + c.D, c.D, R, nb, c.D,
                     (uint64_t)c.B * c.D, R, S));
    p.tmB[0] = h->tm_G;
    p.a_grouped = 1;
    p.a_S = S;
    p.tile_rows = S * R;
    p.M = nb * R;
    p.N = c.sel_dim;
    p.K = c.D;
    p.epi = EPI_F32;
    p.out = gp;
    p.ldo = c.sel_dim;
    DF_TRY(run_gemm(h, p, kBN, s));
  }
  float *table = w.at<float>(h->ws.sel_t);
  if (!walk_logq) {
    DF_CUDA(launch_select_walk(topk_ids, topk_vals, ab, gp, table, nb, c.B, k, c.sel_dim, out_path, s));
  } else {
    DF_CUDA(launch_select_table(topk_vals, ab, gp, table, nb, c.B, k, c.sel_dim, s));
    DF_CUDA(launch_select_walk_sample(topk_ids, table, nb, c.B, k, 1.f / temperature, seed, out_path,
                                      walk_logq, s));
  }
  return DFLASH_OK;
}

}  // namespace

int dflash2_select(dflash_handle_t h, int nb, int k, const int32_t *topk_ids, const float *topk_vals,
                   const void *hidden, const int32_t *block_ids, int32_t *out_path, void *ws,
                   size_t ws_bytes, dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  return select_impl(h, nb, k, topk_ids, topk_vals, hidden, block_ids, 0.f, 0, out_path, nullptr, ws,
                     ws_bytes, stream);
}

int dflash2_select_sample(dflash_handle_t h, int nb, int k, const int32_t *topk_ids,
                          const float *topk_vals, const void *hidden, const int32_t *block_ids,
                          float temperature, uint64_t seed, int32_t *out_path, float *out_walk_logq,
                          void *ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!h || !h->have_weights) return fail(DFLASH_ERR_INVALID_ARG, "handle without weights");
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be positive and finite");
  if (!out_walk_logq && nb > 0) return fail(DFLASH_ERR_INVALID_ARG, "out_walk_logq must be non-NULL");
  return select_impl(h, nb, k, topk_ids, topk_vals, hidden, block_ids, temperature, seed, out_path,
                     out_walk_logq, ws, ws_bytes, stream);
}

int dflash_verify_sample_walk(dflash_handle_t h, int nb, int k, const int32_t *cand_ids,
                              const float *walk_logq, const int32_t *path, const float *target_logits,
                              float temperature, uint64_t seed, int32_t *out_tau, int32_t *out_token,
                              void *ws, size_t ws_bytes, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (k < 1 || k > kTopkMax) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, 16]", k);
  if (!(temperature > 0.f) || !std::isfinite(temperature))
    return fail(DFLASH_ERR_INVALID_ARG, "temperature must be positive and finite");
  if (nb == 0) return DFLASH_OK;
  if (!cand_ids || !walk_logq || !path || !target_logits || !out_tau || !out_token)
    return fail(DFLASH_ERR_INVALID_ARG, "every verify argument must be non-NULL");
  DF_TRY(check_ws(h, ws, ws_bytes));
  Ws w{static_cast<uint8_t *>(ws), h->ws};
  const float inv_T = 1.f / temperature;
  const int rows = nb * c.B;
  float *tlse = w.at<float>(h->ws.smp_lse);
  DF_CUDA(launch_sample(target_logits, c.V, rows, c.V, inv_T, seed, -1, 0,
                        sample_slices(rows, c.V, h->num_sms), w.at<float4>(h->ws.smp_part), nullptr,
                        tlse, nullptr, stream));
  DF_CUDA(launch_verify_walk(cand_ids, walk_logq, k, path, target_logits, tlse, nb, c.B, c.V, inv_T, seed,
                             sample_slices(nb, c.V, h->num_sms), w.at<float4>(h->ws.ver_part),
                             w.at<int>(h->ws.ver_nrej), out_tau, out_token, stream));
  return DFLASH_OK;
}

int dflash_recall_at_k(dflash_handle_t h, int nb, int k, const int32_t *cand_ids, const int32_t *target,
                       int32_t *hits, int32_t *eligible, dflash_stream_t stream) {
  if (!h) return fail(DFLASH_ERR_INVALID_ARG, "handle is NULL");
  const auto &c = h->cfg;
  if (nb < 0 || nb > c.max_batch) return fail(DFLASH_ERR_INVALID_ARG, "nb=%d outside [0, max_batch]", nb);
  if (k < 1 || k > kTopkMax) return fail(DFLASH_ERR_INVALID_ARG, "k=%d outside [1, 16]", k);
  if (nb == 0) return DFLASH_OK;
  if (!cand_ids || !target || !hits || !eligible) return fail(DFLASH_ERR_INVALID_ARG, "NULL tensor");
  DF_CUDA(launch_recall_at_k(cand_ids, target, nb, c.B, k, hits, eligible, stream));
  return DFLASH_OK;
}

}  // extern "C"
