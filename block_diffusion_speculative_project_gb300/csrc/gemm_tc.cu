// tcgen05 tensor-core GEMM for the draft step's dense contractions:
//   D[M, N] = A[M, K] * B[N, K]^T,  A = activations (bf16), B = weights (bf16),
//   fp32 accumulation in TMEM, fused epilogues.
//
// Hardware mapping (sm_103a):
//   * one CTA = 6 warps (10 for the LM head's top-k): warp 0 issues TMA tile loads (128B
//     swizzle, K-major), warp 1 allocates TMEM and one thread issues tcgen05.mma (M=128,
//     N=BN, K=16), the other warps drain the fp32 accumulator with tcgen05.ld (32x32b)
//     and run the epilogue; each epilogue warp reads the TMEM lane quarter (warp % 4), and
//     the top-k's two groups of four split each tile's 32-column chunks.
//   * an mbarrier ring of STAGES smem slots couples TMA and MMA; tcgen05.commit
//     frees a slot when the MMAs that read it complete.
//   * two TMEM accumulator sets let the epilogue of one work item run under the MMAs
//     of the next (one set when two do not fit the 512 columns); CTAs are persistent
//     over work items, visited in groups of row tiles (rast_gm) so that the tiles of one
//     wave share their A blocks and weight tiles through L2.
//   * M-stacking (template MS = 2): a work item is two 128-row blocks; each weight tile in
//     smem feeds two M = 128 MMAs into two accumulators (more FLOPs per operand byte an
//     SM takes in), for launches with many row tiles (gemm_mstack).
//   * split-K across a thread-block cluster: the S CTAs of a cluster each reduce a
//     1/S slice of K for the same output tile, stage their fp32 partial in their own
//     (now idle) pipeline smem, and after a hardware cluster barrier every CTA sums
//     a 1/S row slice of the tile over all S partials through distributed shared
//     memory, in rank order (deterministic), and runs the epilogue on it.
//   * weights are streamed with an L2 evict-first policy, activations evict-last.
#include <algorithm>
#include <cmath>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"
#include "sampling.cuh"

namespace df {

constexpr int BM = 128;
constexpr int BK = 64;
// Epilogue warps per CTA: eight for the LM head's top-k (two per TMEM lane quarter, each
// taking every other 32-column chunk of a tile: with one warp per SM sub-partition this
// branchy, dependent code runs latency-bound), else four. Warps 0 and 1 are the TMA
// producer and the MMA issuer.
template <int EPI>
__host__ __device__ constexpr int gemm_epi_warps() {
  return EPI == EPI_TOPK ? 8 : 4;
}
template <int EPI>
__host__ __device__ constexpr int gemm_threads() {
  return 64 + 32 * gemm_epi_warps<EPI>();
}
// Bound of the teardown waits for this CTA's own TMA copies and MMAs, which finish
// without help from any other thread; independent of the caller's max_spin.
constexpr int kDrainSpin = 1 << 22;
// K slabs (64 columns each) one stage holds: two for the plain 128-wide GEMMs, whose
// A and B tiles are then each one 32 KB copy (a tensor copy from one SM costs about
// one DRAM round trip whatever its size, so the small-M GEMMs were bound by the copy
// count), one for the dual and top-k tiles.
template <int BN, int EPI>
__host__ __device__ constexpr int gemm_slabs() {
  return (BN == 128 && EPI != EPI_SWIGLU && EPI != EPI_DUAL_F32 && EPI != EPI_TOPK) ? 2 : 1;
}

// MS: 128-row blocks per tile (M-stacking). With MS = 2 a tile is 256 rows: each weight
// tile in shared memory feeds two M = 128 MMAs into two accumulators, which doubles the
// FLOPs per operand byte an SM takes in when there are enough tiles to fill the GPU.
template <int BN, int SL, int MS = 1>
struct TileCfg {
  static constexpr int A_SLAB = BM * BK * 2;
  static constexpr int B_SLAB = BN * BK * 2;
  static constexpr int A_BLOCK = SL * A_SLAB;  // one 128-row block of A in a stage
  static constexpr int A_BYTES = MS * A_BLOCK;
  static constexpr int B_BYTES = SL * B_SLAB;
  static constexpr int STAGE = A_BYTES + B_BYTES;
  static constexpr int STAGES = (200 * 1024 / STAGE) > 8 ? 8 : (200 * 1024 / STAGE);
  static constexpr int ACC = MS * BN;  // TMEM columns of one accumulator set
  // Two accumulator sets (the epilogue of one tile runs under the MMAs of the next) when
  // they fit in the 512 TMEM columns, else one.
  static constexpr int NBUF = 2 * ACC <= 512 ? 2 : 1;
  static constexpr int TMEM_COLS = (NBUF * ACC <= 256) ? 256 : 512;  // power of two >= the sets
  // Cluster split-K reuses the pipeline smem: the staged partial tile (BM rows of
  // RED_STRIDE floats) followed by the reduced row slice (at most BM / 2 rows). The
  // pipeline region is the larger of the stage ring and that; barriers follow it.
  static constexpr int RED_STRIDE = BN + 4;
  static constexpr size_t RED_BYTES = size_t(BM + BM / 2) * RED_STRIDE * 4;
  static constexpr bool SPLITS = BN <= 192 && MS == 1;  // top-k and M-stacked tiles never split K
  static constexpr size_t PIPE =
      (!SPLITS || size_t(STAGES) * STAGE > RED_BYTES) ? size_t(STAGES) * STAGE : RED_BYTES;
  static constexpr size_t SMEM = 1024 + PIPE + 256;
  static constexpr bool RED_FITS = !SPLITS || RED_BYTES <= PIPE;
};

// Top-k epilogue: a per-thread stash of one 32-value chunk (stride 33 floats, so the
// 32 threads of a warp hit distinct banks), for each of the 256 epilogue threads.
constexpr size_t kTopkStashBytes = 256 * 33 * sizeof(float);
// Row stride (floats, odd: no bank conflicts) of the exchange through which the two
// epilogue groups of the top-k GEMM see each other's members: group g's values at
// [32 g, 32 g + 16) and ids at [32 g + 16, 32 g + 32), then the second group's draw
// (m, s, best, x, id) at [64, 69).
constexpr int kTopkXchg = 69;

// Slabs per stage: as the unstacked tile (an M-stacked 128-wide tile takes two 32 KB A
// copies and one 32 KB B copy per 96 KB stage, two stages in flight).
template <int BN, int EPI, int MS>
__host__ __device__ constexpr int gemm_slabs_ms() {
  return gemm_slabs<BN, EPI>();
}

template <int BN, int EPI, int MS = 1>
constexpr size_t gemm_smem_bytes() {
  return TileCfg<BN, gemm_slabs_ms<BN, EPI, MS>(), MS>::SMEM + (EPI == EPI_TOPK ? kTopkStashBytes : 0);
}

struct Item {
  int m, n, g, s;
};

__device__ __forceinline__ int item_count(const GemmParams &p) {
  if (p.csplit > 1) return 1;
  if (p.epi == EPI_TOPK) {
    const int range = blockIdx.x / p.m_tiles;
    const int n0 = range * p.tiles_per_cta;
    const int n1 = min(p.n_tiles, n0 + p.tiles_per_cta);
    return max(0, n1 - n0);
  }
  if (static_cast<int>(blockIdx.x) >= p.items) return 0;
  return (p.items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1;
}

__device__ __forceinline__ Item item_at(const GemmParams &p, int j) {
  Item r;
  if (p.epi == EPI_TOPK) {
    r.m = blockIdx.x % p.m_tiles;
    r.n = (blockIdx.x / p.m_tiles) * p.tiles_per_cta + j;
    r.g = 0;
    r.s = 0;
    return r;
  }
  int it;
  if (p.csplit > 1) {
    it = blockIdx.x / p.csplit;
    r.m = it % p.m_tiles;
    it /= p.m_tiles;
    r.n = it % p.n_tiles;
    r.g = it / p.n_tiles;
    r.s = static_cast<int>(cluster_ctarank());
    return r;
  }
  it = blockIdx.x + j * gridDim.x;
  {
    const int per_group = p.rast_gm * p.n_tiles * p.groups;
    const int grp = it / per_group, rem = it - grp * per_group;
    const int gm = min(p.rast_gm, p.m_tiles - grp * p.rast_gm);  // the last group may be short
    r.m = grp * p.rast_gm + rem % gm;
    const int ng = rem / gm;
    r.n = ng % p.n_tiles;
    r.g = ng / p.n_tiles;
    r.s = 0;
  }
  return r;
}

// ------------------------------------------------------------------ epilogue helpers

// Vector stores need 16-byte alignment; rows of odd width (e.g. the logits of a
// vocabulary that is not a multiple of 4) fall back to scalar stores.
__device__ __forceinline__ bool aligned16(const void *p) {
  return (reinterpret_cast<uintptr_t>(p) & 15) == 0;
}

__device__ __forceinline__ void store_bf16_32(uint16_t *dst, const float (&v)[32], int nvalid) {
  if (nvalid >= 32 && aligned16(dst)) {
    uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      uint4 w;
      w.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
      w.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
      w.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
      w.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
      d4[q] = w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      if (i < nvalid) {
        __nv_bfloat16 b = __float2bfloat16_rn(v[i]);
        dst[i] = *reinterpret_cast<uint16_t *>(&b);
      }
    }
  }
}

__device__ __forceinline__ void store_f32_32(float *dst, const float (&v)[32], int nvalid) {
  if (nvalid >= 32 && aligned16(dst)) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) d4[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) dst[i] = v[i];
  }
}

// dst += v; the new values are also returned in out (which may alias v).
__device__ __forceinline__ void add_f32_32(float *dst, const float (&v)[32], int nvalid, float (&out)[32]) {
  if (nvalid >= 32 && aligned16(dst)) {
    float4 *d4 = reinterpret_cast<float4 *>(dst);
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      float4 x = d4[q];
      x.x += v[4 * q];
      x.y += v[4 * q + 1];
      x.z += v[4 * q + 2];
      x.w += v[4 * q + 3];
      d4[q] = x;
      out[4 * q] = x.x;
      out[4 * q + 1] = x.y;
      out[4 * q + 2] = x.z;
      out[4 * q + 3] = x.w;
    }
  } else {
#pragma unroll
    for (int i = 0; i < 32; ++i)
      if (i < nvalid) {
        const float x = dst[i] + v[i];
        dst[i] = x;
        out[i] = x;
      }
  }
}

__device__ __forceinline__ float bf16_bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

// Deferred RMSNorm factor of a row: rsqrt(mean of squares + eps) from its partial sums.
__device__ __forceinline__ float deferred_rms(const GemmParams &p, int row) {
  const float *s = p.ss_in + (size_t)row * p.ss_n;
  float a[4] = {0.f, 0.f, 0.f, 0.f};
  int i = 0;
  if ((p.ss_n & 3) == 0 && aligned16(s)) {
    // eight float4 loads in flight at a time (one pass for ss_n <= 32), then the adds in
    // the same order as one at a time; the loads past ss_n are zeros, and adding +0 to
    // these non-negative sums changes nothing
    constexpr int kV = 8;
    for (; i < p.ss_n; i += 4 * kV) {
      float4 x[kV];
#pragma unroll
      for (int k = 0; k < kV; ++k)
        x[k] = i + 4 * k < p.ss_n ? *reinterpret_cast<const float4 *>(s + i + 4 * k) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int k = 0; k < kV; ++k) {
        a[0] += x[k].x;
        a[1] += x[k].y;
        a[2] += x[k].z;
        a[3] += x[k].w;
      }
    }
  } else {
    for (; i < p.ss_n; ++i) a[i & 3] += s[i];
  }
  return rsqrtf(((a[0] + a[1]) + (a[2] + a[3])) * p.inv_d + p.eps);
}

// Rotation angle pos * inv_freq reduced to [-pi, pi] with a two-constant split of
// 2*pi (Cody and Waite's method): 6.28125 has 8 significant bits, so k * 6.28125 is
// exact for the k that occur here (|k| < 2^15) and only the small second constant
// rounds. The reduced angle then goes to the fast sine/cosine intrinsic.
__device__ __forceinline__ void rope_sincos(float angle, float *sn, float *cs) {
  const float k = rintf(angle * 0.15915494309189535f);
  const float r = fmaf(-k, 1.9353071795864769e-3f, fmaf(-k, 6.28125f, angle));
  __sincosf(r, sn, cs);
}

// Row of (sequence, kv head, position) inside one layer's cache, in units of hd elements:
// [max_batch][Hkv][Cmax] contiguous, or through the page table [num_pages][Hkv][kPageRows].
// -1 when the page table names a page outside the pool (the caller skips the row).
__device__ __forceinline__ long long cache_row(const GemmParams &p, int seq, int head, int pos) {
  if (p.page_table == nullptr) return ((long long)seq * p.Hkv + head) * p.Cmax + pos;
  const int pg = p.page_table[(long long)seq * p.pages_per_seq + pos / kPageRows];
  if (pg < 0 || pg >= p.num_pages) return -1;
  return ((long long)pg * p.Hkv + head) * kPageRows + pos % kPageRows;
}

__device__ __forceinline__ void rope_pair(const GemmParams &p, int pos, int d0, float (&a)[32],
                                          float (&b)[32]) {
  const float fpos = static_cast<float>(pos);
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    float sn, cs;
    rope_sincos(fpos * p.inv_freq[d0 + i], &sn, &cs);
    const float x1 = a[i], x2 = b[i];
    a[i] = x1 * cs - x2 * sn;
    b[i] = x2 * cs + x1 * sn;
  }
}

// Per-thread top-k state of the LM-head epilogue: the kTopkMax best (value, id) pairs
// seen so far, kept sorted in registers (v[0] ranks first: value descending, ties to the
// lower id), so the last member is the threshold a new value has to beat. Fillers are
// (-FLT_MAX, id_base + s) with distinct ids. Every step is written as compares and
// selects: a taken branch costs a lone warp tens of cycles, and the epilogue runs one
// or two warps per SM sub-partition.
struct TopkState {
  float v[kTopkMax];
  int id[kTopkMax];
  DrawState dr;  // the draw at temperature T when sampling (smp_part set)
};

__device__ __forceinline__ void topk_init(TopkState &tk, int id_base) {
#pragma unroll
  for (int s = 0; s < kTopkMax; ++s) {
    tk.v[s] = -FLT_MAX;
    tk.id[s] = id_base + s;  // ascending ids: sorted
  }
  draw_init(tk.dr);
}

// Insert (x, xi), which ranks before the last member: it goes to the first position it
// ranks before, the members from there on move down one place and the last drops out.
// The compares all read the old members, so they are independent of one another.
__device__ __forceinline__ void topk_insert(TopkState &tk, float x, int xi) {
  bool b[kTopkMax];
#pragma unroll
  for (int s = 0; s < kTopkMax; ++s) b[s] = topk_before(x, xi, tk.v[s], tk.id[s]);
#pragma unroll
  for (int s = kTopkMax - 1; s > 0; --s) {
    tk.v[s] = b[s - 1] ? tk.v[s - 1] : (b[s] ? x : tk.v[s]);
    tk.id[s] = b[s - 1] ? tk.id[s - 1] : (b[s] ? xi : tk.id[s]);
  }
  tk.v[0] = b[0] ? x : tk.v[0];
  tk.id[0] = b[0] ? xi : tk.id[0];
}

// Runs the epilogue of one output tile. `fetch(c, v)` returns the 32 fp32 values of
// accumulator columns [32c, 32c+32) of this thread's row; it is called by every lane
// (tcgen05.ld is warp-collective); only the stores depend on row validity.
// cpart / nparts: this thread runs the row's 32-column chunks c with c % nparts == cpart
// (nparts threads share the row: adjacent lanes in the split-K epilogue, whose residual
// RMS partial sums are combined by shuffles, or the two epilogue groups of the top-k;
// nparts = 1 when one thread owns the whole row). Every lane of the warp must call it.
template <int BN, int EPI, class Fetch>
__device__ __forceinline__ void epilogue_tile(const GemmParams &p, const Item &t, int row,
                                              bool row_ok, Fetch &&fetch, TopkState &tk,
                                              float *stash, int cpart = 0, int nparts = 1) {
  if constexpr (EPI == EPI_BF16 || EPI == EPI_F32) {
#pragma unroll 1
    for (int c = cpart; c < BN / 32; c += nparts) {
      float v[32];
      fetch(c, v);
      const int col0 = t.n * BN + c * 32;
      const int nval = min(32, p.N - col0);
      if (row_ok && nval > 0) {
        if constexpr (EPI == EPI_BF16) {
          if (p.act) {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = v[i] / (1.0f + expf(-v[i]));
          }
          store_bf16_32(static_cast<uint16_t *>(p.out) + row * p.ldo + col0, v, nval);
        }
        else
          store_f32_32(static_cast<float *>(p.out) + row * p.ldo + col0, v, nval);
      }
    }
  } else if constexpr (EPI == EPI_RESID) {
    float ss = 0.f;
#pragma unroll 1
    for (int c = cpart; c < BN / 32; c += nparts) {
      float v[32];
      fetch(c, v);
      const int col0 = t.n * BN + c * 32;
      const int nval = min(32, p.N - col0);
      if (row_ok && nval > 0) {
        add_f32_32(p.xres + row * p.ldo + col0, v, nval, v);  // v <- x_new
        if (p.xg_out) {
          float gv[32];
          if (!p.g_next) {  // plain bf16 copy of x (input of a DFlash 2 conv)
#pragma unroll
            for (int i = 0; i < 32; ++i) gv[i] = 1.f;
          } else if (nval >= 32 && aligned16(p.g_next + col0)) {
            const uint4 *g4 = reinterpret_cast<const uint4 *>(p.g_next + col0);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const uint4 w = g4[q];
              const uint32_t wd[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                gv[8 * q + 2 * h] = __uint_as_float(wd[h] << 16);
                gv[8 * q + 2 * h + 1] = __uint_as_float(wd[h] & 0xFFFF0000u);
              }
            }
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) gv[i] = i < nval ? bf16_bits_to_f32(p.g_next[col0 + i]) : 0.f;
          }
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float x0 = i < nval ? v[i] : 0.f, x1 = i + 1 < nval ? v[i + 1] : 0.f;
            s0 = fmaf(x0, x0, s0);
            s1 = fmaf(x1, x1, s1);
            v[i] = x0 * gv[i];
            v[i + 1] = x1 * gv[i + 1];
          }
          ss += s0 + s1;
          store_bf16_32(p.xg_out + row * p.ldo + col0, v, nval);
        }
      }
    }
    for (int o = 1; o < nparts; o <<= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if (p.ss_out && row_ok && cpart == 0) p.ss_out[(size_t)row * p.n_tiles + t.n] = ss;
  } else if constexpr (EPI == EPI_ROPE) {
    const int half = p.hd >> 1;
    int seq = 0, pos = 0;
    bool pos_ok = false;
    if (row_ok) {  // issued before the norm factor's loads: independent, so both are in flight
      seq = row / p.rows_per_seq;
      pos = p.ctx_len[seq] + row % p.rows_per_seq;
      pos_ok = pos >= 0 && pos < p.Cmax;
    }
    const float rs = (p.ss_in && row_ok) ? deferred_rms(p, row) : 1.f;
#pragma unroll 1
    for (int h0 = 0; h0 < BN; h0 += p.hd) {
      const int gcol = t.n * BN + h0;
      const bool rot = gcol < p.rope_cols;
      // destination row of this head: the q part of the qkv buffer, or the block's
      // cache row ctx_len + j of a k / v head
      uint16_t *o = nullptr;
      if (row_ok && gcol < p.N) {
        if (gcol < p.q_cols) {
          o = static_cast<uint16_t *>(p.out) + row * p.ldo + gcol;
        } else if (pos_ok) {
          const int kvh = (gcol - p.q_cols) / p.hd;  // 0..2*Hkv-1
          const bool isv = kvh >= p.Hkv;
          const int head = isv ? kvh - p.Hkv : kvh;
          const long long cr = cache_row(p, seq, head, pos);
          if (cr >= 0)
            o = static_cast<uint16_t *>(isv ? p.vc : p.kc) + cr * p.hd;
          else
            flag_status(p.status, kStatusCheck);
        } else {
          flag_status(p.status, kStatusCheck);
        }
      }
#pragma unroll 1
      for (int cc = 32 * cpart; cc < half; cc += 32 * nparts) {
        float a[32], b[32];
        fetch((h0 + cc) >> 5, a);
        fetch((h0 + half + cc) >> 5, b);
        if (o) {
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] *= rs;
            b[i] *= rs;
          }
          if (rot) rope_pair(p, pos, cc, a, b);
          store_bf16_32(o + cc, a, 32);
          store_bf16_32(o + half + cc, b, 32);
        }
      }
    }
  } else if constexpr (EPI == EPI_SWIGLU) {
    const float rs = (p.ss_in && row_ok) ? deferred_rms(p, row) : 1.f;
#pragma unroll 1
    for (int c = cpart; c < BN / 64; c += nparts) {
      float g[32], u[32];
      fetch(c, g);
      fetch(c + BN / 64, u);
      const int col0 = t.n * (BN / 2) + c * 32;
      const int nval = min(32, p.N - col0);
      if (row_ok && nval > 0) {
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float gi = g[i] * rs;
          // rounded to bf16 below: the fast exponential and divide (~1e-6 relative) stay far
          // under that rounding, and the full-precision forms cost ~4 us per launch here
          g[i] = __fdividef(gi, 1.0f + __expf(-gi)) * (u[i] * rs);
        }
        store_bf16_32(static_cast<uint16_t *>(p.out) + row * p.ldo + col0, g, nval);
      }
    }
  } else if constexpr (EPI == EPI_DUAL_F32) {
#pragma unroll 1
    for (int c = cpart; c < BN / 32; c += nparts) {
      float v[32];
      fetch(c, v);
      const int which = c >= BN / 64 ? 1 : 0;
      const int col0 = t.n * (BN / 2) + (c - which * (BN / 64)) * 32;
      const int nval = min(32, p.N - col0);
      if (row_ok && nval > 0)
        store_f32_32(static_cast<float *>(p.out) + row * p.ldo + which * p.N + col0, v, nval);
    }
  } else if constexpr (EPI == EPI_KV) {
    const int layer = t.g >> 1;
    const bool isk = (t.g & 1) == 0;
    const int half = p.hd >> 1;
    int seq = 0, pos = 0;
    bool live = false;
    if (row_ok) {
      seq = row / p.rows_per_seq;
      const int j = row % p.rows_per_seq;
      live = j < p.n_commit[seq];
      pos = p.ctx_len[seq] + j;
      if (live && (pos < 0 || pos >= p.Cmax)) {
        flag_status(p.status, kStatusCheck);
        live = false;
      }
    }
    uint16_t *cache = static_cast<uint16_t *>(isk ? p.kc : p.vc);
#pragma unroll 1
    for (int h0 = 0; h0 < BN; h0 += p.hd) {
      const int head = (t.n * BN + h0) / p.hd;
#pragma unroll 1
      for (int cc = 32 * cpart; cc < half; cc += 32 * nparts) {
        float a[32], b[32];
        fetch((h0 + cc) >> 5, a);
        fetch((h0 + half + cc) >> 5, b);
        if (live && head < p.Hkv) {
          const long long cr = cache_row(p, seq, head, pos);
          if (cr < 0) {
            flag_status(p.status, kStatusCheck);
            continue;
          }
          if (isk) rope_pair(p, pos, cc, a, b);
          uint16_t *o = cache + (layer * p.layer_rows + cr) * p.hd;
          store_bf16_32(o + cc, a, 32);
          store_bf16_32(o + half + cc, b, 32);
        }
      }
    }
  } else if constexpr (EPI == EPI_TOPK) {
#pragma unroll 1
    for (int c = cpart; c < BN / 32; c += nparts) {
      float v[32];
      fetch(c, v);
      const int col0 = t.n * BN + c * 32;
      const int nval = row_ok ? min(32, p.N - col0) : 0;
      if (p.logits_out && nval > 0) store_f32_32(p.logits_out + (size_t)row * p.N + col0, v, nval);
      // branch-free filter: which of the 32 values beat the current worst member
      uint32_t mask = 0;
#pragma unroll
      for (int i = 0; i < 32; ++i)
        mask |= static_cast<uint32_t>((i < nval) & topk_before(v[i], col0 + i, tk.v[kTopkMax - 1], tk.id[kTopkMax - 1]))
                << i;
      if (mask) {
#pragma unroll
        for (int i = 0; i < 32; ++i) stash[i] = v[i];
#pragma unroll 1
        while (mask) {
          const int i = __ffs(mask) - 1;
          mask &= mask - 1;
          const float x = stash[i];
          if (topk_before(x, col0 + i, tk.v[kTopkMax - 1], tk.id[kTopkMax - 1])) topk_insert(tk, x, col0 + i);
        }
      }
      // the draw at temperature T (scales v in place, so it runs after the top-k)
      if (p.smp_part && nval > 0)
        draw_chunk32(tk.dr, v, p.smp_inv_T, col0, nval, (uint32_t)row, (uint32_t)p.smp_stream, p.smp_seed);
    }
  }
}

// ------------------------------------------------------------------ kernel

template <int BN, int EPI, int MS>
__global__ void __launch_bounds__(gemm_threads<EPI>(), 1) gemm_tc_kernel(const __grid_constant__ GemmParams p) {
  constexpr int SLABS = gemm_slabs_ms<BN, EPI, MS>();
  using C = TileCfg<BN, SLABS, MS>;
  static_assert(EPI == EPI_TOPK || MS > 1 || C::RED_FITS, "cluster reduction buffers exceed the pipeline smem");
  static_assert(MS == 1 || EPI != EPI_DUAL_F32, "M-stacked tiles: no dual fp32 epilogue");
  static_assert(MS == 1 || EPI != EPI_TOPK, "M-stacked tiles: no top-k epilogue");
  static_assert(EPI != EPI_TOPK || size_t(BM) * kTopkXchg * 4 <= C::PIPE, "top-k exchange exceeds the pipeline smem");
  static_assert(C::NBUF * C::ACC <= 512, "accumulators exceed tensor memory");
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sA = smem;
  uint8_t *sB = smem + C::STAGES * C::A_BYTES;
  uint64_t *full = reinterpret_cast<uint64_t *>(smem + C::PIPE);
  uint64_t *empty = full + C::STAGES;
  uint64_t *acc_full = empty + C::STAGES;
  uint64_t *acc_empty = acc_full + 2;
  uint64_t *mma_done = acc_empty + 2;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 1);
  float *stash_base = reinterpret_cast<float *>(smem + C::PIPE + 256);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nitems = item_count(p);

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&acc_full[b], 1);
      mbar_init(&acc_empty[b], 32 * gemm_epi_warps<EPI>());
    }
    mbar_init(mma_done, 1);
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (threadIdx.x == 0) griddep_launch();

  if (warp == 0) {
    if (lane == 0 && nitems > 0 && !p.stall) {
      // ---------------- TMA producer
      tma_prefetch_desc(&p.tmA);
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      // Iteration cursor over (work item, k-tile) in this CTA's order.
      struct Cursor {
        int j, kt, kt1;
        Item t;
      };
      auto begin = [&](Cursor &c) {
        c.j = 0;
        c.t = item_at(p, 0);
        c.kt = c.t.s * p.kt_per_split;
        c.kt1 = min(p.kt_total, c.kt + p.kt_per_split);
      };
      auto advance = [&](Cursor &c) -> bool {
        if (++c.kt < c.kt1) return true;
        if (++c.j >= nitems) return false;
        c.t = item_at(p, c.j);
        c.kt = c.t.s * p.kt_per_split;
        c.kt1 = min(p.kt_total, c.kt + p.kt_per_split);
        return true;
      };
      auto load_a = [&](const Cursor &c, int st) {
        uint8_t *a = sA + st * C::A_BYTES;
#pragma unroll
        for (int ms = 0; ms < MS; ++ms) {
          const int row0 = c.t.m * (MS * BM) + ms * BM;
          if (p.slabs == 2)  // A map {64, rows, K/64}: both slabs of the stage in one copy
            tma_load_3d(a + ms * C::A_BLOCK, &p.tmA, &full[st], 0, row0, c.kt * 2, pol_a);
          else if (p.a_grouped)
            tma_load_3d(a + ms * C::A_BLOCK, &p.tmA, &full[st], c.kt * BK, 0, (c.t.m * MS + ms) * p.a_S, pol_a);
          else
            tma_load_3d(a + ms * C::A_BLOCK, &p.tmA, &full[st], c.kt * BK, row0, 0, pol_a);
        }
      };
      auto load_b = [&](const Cursor &c, int st) {
        uint8_t *b = sB + st * C::B_BYTES;
        if (p.slabs == 2) {  // weight maps {64, N, K/64}
          tma_load_3d(b, &p.tmB[c.t.g], &full[st], 0, c.t.n * BN, c.kt * 2, pol_w);
        } else if (p.dual) {
          tma_load_2d(b, &p.tmB[0], &full[st], c.kt * BK, c.t.n * (BN / 2), pol_w);
          tma_load_2d(b + (BN / 2) * 128, &p.tmB[1], &full[st], c.kt * BK, c.t.n * (BN / 2), pol_w);
        } else {
          tma_load_2d(b, &p.tmB[c.t.g], &full[st], c.kt * BK, c.t.n * BN, pol_w);
        }
      };
      // Weights do not depend on earlier kernels: fill every stage's weight tile
      // before waiting for the producer of the activations.
      Cursor c;
      begin(c);
      int pre = 0;
      bool more = true;
      while (more && pre < C::STAGES) {
        mbar_arrive_expect_tx(&full[pre], p.stage_tx_bytes);
        load_b(c, pre);
        ++pre;
        more = advance(c);
      }
      griddep_wait();
      {
        Cursor ca;
        begin(ca);
        for (int k = 0; k < pre; ++k) {
          load_a(ca, k);
          advance(ca);
        }
      }
      int it = pre;
      bool ok = true;
      while (more) {
        const int st = it % C::STAGES;
        const uint32_t ph = (it / C::STAGES) & 1;
        if (!mbar_wait(&empty[st], ph ^ 1, p.max_spin)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[st], p.stage_tx_bytes);
        load_a(c, st);
        load_b(c, st);
        ++it;
        more = advance(c);
      }
      if (!ok) flag_status(p.status, kStatusTimeout);
      // Every issued load must land before the CTA may exit (bounded).
      for (int k = max(0, it - C::STAGES); k < it; ++k)
        mbar_wait(&full[k % C::STAGES], (k / C::STAGES) & 1, kDrainSpin);
    }
  } else if (warp == 1) {
    if (lane == 0 && nitems > 0) {
      // ---------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16_f32(BM, BN);
      const uint64_t a_desc0 = sw128_kmajor_desc(smem_u32(sA));
      const uint64_t b_desc0 = sw128_kmajor_desc(smem_u32(sB));
      int it = 0;
      bool ok = true;
      for (int j = 0; j < nitems && ok; ++j) {
        const Item t = item_at(p, j);
        const int buf = j % C::NBUF;
        const uint32_t use = j / C::NBUF;
        if (!mbar_wait(&acc_empty[buf], (use & 1) ^ 1, p.max_spin)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d = tmem_base + buf * C::ACC;
        const int kt0 = t.s * p.kt_per_split;
        const int kt1 = min(p.kt_total, kt0 + p.kt_per_split);
        for (int kt = kt0; kt < kt1; ++kt, ++it) {
          const int st = it % C::STAGES;
          const uint32_t ph = (it / C::STAGES) & 1;
          if (!mbar_wait(&full[st], ph, p.max_spin)) {
            ok = false;
            break;
          }
          tc_fence_after();
          // descriptors differ only in their start-address field (16-byte units)
          const uint64_t ad = a_desc0 + static_cast<uint64_t>((st * C::A_BYTES) >> 4);
          const uint64_t bd = b_desc0 + static_cast<uint64_t>((st * C::B_BYTES) >> 4);
#pragma unroll
          for (int sl = 0; sl < SLABS; ++sl) {
            if (sl >= p.slabs) break;
            const uint64_t bs = bd + static_cast<uint64_t>((sl * C::B_SLAB) >> 4);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k)
#pragma unroll
              for (int ms = 0; ms < MS; ++ms) {
                const uint64_t as = ad + static_cast<uint64_t>((ms * C::A_BLOCK + sl * C::A_SLAB) >> 4);
                tc_mma_bf16(d + ms * BN, as + 2 * k, bs + 2 * k, idesc, (kt > kt0 || sl > 0 || k > 0) ? 1u : 0u);
              }
          }
          tc_commit(&empty[st]);
        }
        if (!ok) break;
        tc_commit(&acc_full[buf]);
      }
      if (!ok) flag_status(p.status, kStatusTimeout);
      // Every issued MMA must complete before TMEM is freed (bounded).
      tc_commit(mma_done);
      mbar_wait(mma_done, 0, kDrainSpin);
    }
  } else {
    // ---------------- epilogue warps 2..5 (2..9 for the top-k)
    griddep_wait();
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const int eg = (warp - 2) >> 2;  // epilogue group: 0, or 1 for the second top-k group
    float *stash = stash_base + ((warp - 2) * 32 + lane) * 33;
    TopkState tks[MS];
    TopkState &tk = tks[0];
    if constexpr (EPI == EPI_TOPK) {
#pragma unroll
      for (int ms = 0; ms < MS; ++ms) topk_init(tks[ms], INT_MAX - 2 * kTopkMax + 1 + eg * kTopkMax);
    }
    bool ok = true;
    for (int j = 0; j < nitems; ++j) {
      const Item t = item_at(p, j);
      const int buf = j % C::NBUF;
      const uint32_t use = j / C::NBUF;
      if (!mbar_wait(&acc_full[buf], use & 1, p.max_spin)) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * C::ACC;
      const int row = t.m * p.tile_rows + r;
      const bool row_ok = (r < p.tile_rows) && (row < p.M);
      if (MS > 1) {
        // 128-row block ms of the tile: rows (t.m * MS + ms) * tile_rows + r
#pragma unroll
        for (int ms = 0; ms < MS; ++ms) {
          const int row_ms = (t.m * MS + ms) * p.tile_rows + r;
          auto fetch = [&](int c, float (&v)[32]) { tmem_ld32(taddr + ms * BN + c * 32, v); };
          epilogue_tile<BN, EPI>(p, t, row_ms, (r < p.tile_rows) && (row_ms < p.M), fetch, tks[ms], stash);
        }
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
      } else if (EPI != EPI_TOPK && p.csplit > 1) {
        // Stage this CTA's partial tile, row r at red[r * RED_STRIDE], in the
        // pipeline smem (every TMA write has landed and every MMA has completed).
        float *red = reinterpret_cast<float *>(smem) + r * C::RED_STRIDE;
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          float v[32];
          tmem_ld32(taddr + c * 32, v);
          float4 *d4 = reinterpret_cast<float4 *>(red + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) d4[k] = make_float4(v[4 * k], v[4 * k + 1], v[4 * k + 2], v[4 * k + 3]);
        }
      } else {
        auto fetch = [&](int c, float (&v)[32]) { tmem_ld32(taddr + c * 32, v); };
        constexpr int ng = gemm_epi_warps<EPI>() / 4;  // groups sharing a row's chunks
        epilogue_tile<BN, EPI>(p, t, row, row_ok, fetch, tk, stash, ng > 1 ? eg : 0, ng);
        tc_fence_before();
        mbar_arrive(&acc_empty[buf]);
      }
    }
    if (!ok) flag_status(p.status, kStatusTimeout);
    if constexpr (EPI == EPI_TOPK) {
      // The two groups' sorted sets meet through the pipeline smem (every MMA has completed
      // and every copy has landed once the last accumulator was ready). A member's rank in
      // the union is its place in its own set plus the other set's members that rank before
      // it; the members of rank < k are the CTA's partial, written straight to their
      // places. The fillers' ids are distinct across the groups, so the ranks are too. The
      // first group also merges the second group's draw. Every epilogue thread reaches the
      // barrier.
      float *xg = reinterpret_cast<float *>(smem) + r * kTopkXchg;
#pragma unroll
      for (int s2 = 0; s2 < kTopkMax; ++s2) {
        xg[eg * 32 + s2] = tk.v[s2];
        xg[eg * 32 + kTopkMax + s2] = __int_as_float(tk.id[s2]);
      }
      if (eg == 1) {
        xg[64] = tk.dr.m;
        xg[65] = tk.dr.s;
        xg[66] = tk.dr.best;
        xg[67] = tk.dr.x;
        xg[68] = __int_as_float(tk.dr.id);
      }
      named_bar_sync(2, 32 * gemm_epi_warps<EPI>());
      const int m = blockIdx.x % p.m_tiles;
      const int range = blockIdx.x / p.m_tiles;
      const int row = m * p.tile_rows + r;
      if (ok && nitems > 0 && r < p.tile_rows && row < p.M) {
        const float *ov = xg + (1 - eg) * 32;
        float w[kTopkMax];
        int wi[kTopkMax];
#pragma unroll
        for (int s2 = 0; s2 < kTopkMax; ++s2) {
          w[s2] = ov[s2];
          wi[s2] = __float_as_int(ov[kTopkMax + s2]);
        }
        float *pv = p.part_vals + ((size_t)range * p.M + row) * p.topk_k;
        int *pi = p.part_ids + ((size_t)range * p.M + row) * p.topk_k;
#pragma unroll
        for (int s2 = 0; s2 < kTopkMax; ++s2) {
          int rank = s2;
#pragma unroll
          for (int t2 = 0; t2 < kTopkMax; ++t2) rank += topk_before(w[t2], wi[t2], tk.v[s2], tk.id[s2]) ? 1 : 0;
          if (rank < p.topk_k) {
            pv[rank] = tk.v[s2];
            pi[rank] = tk.id[s2];
          }
        }
        if (p.smp_part && eg == 0) {
          DrawState o;
          o.m = xg[64];
          o.s = xg[65];
          o.best = xg[66];
          o.x = xg[67];
          o.id = __float_as_int(xg[68]);
          draw_merge(tk.dr, o);
          draw_store(p.smp_part + 2 * ((size_t)range * p.M + row), tk.dr);
        }
      }
    }
  }

  if (EPI != EPI_TOPK && p.csplit > 1) {
    // Every partial of the cluster is staged; sum this CTA's row slice over the
    // cluster in rank order and run the epilogue on it.
    __syncwarp();
    cluster_sync_all();
    if (warp >= 2 && nitems > 0) {
      const int q = warp & 3;
      const int r = q * 32 + lane;
      const int rank = static_cast<int>(cluster_ctarank());
      const int row0 = rank * BM / p.csplit;               // this CTA's rows [row0, row1)
      const int per = (rank + 1) * BM / p.csplit - row0;
      // Phase 1: the 128 epilogue threads sum this CTA's row slice over the S staged
      // partials (float4 units, loads of two ranks in flight) into a local buffer
      // placed after the staged partial; the sum runs in rank order.
      float *slice = reinterpret_cast<float *>(smem) + BM * C::RED_STRIDE;
      const uint32_t red0 = smem_u32(smem);
      const int units = per * (BN / 4);
      // four units per thread at a time, two ranks' loads each (8 cluster loads in
      // flight): the sum is latency-bound, and each unit's additions stay in rank order
      constexpr int kU = 4;
      for (int e0 = threadIdx.x - 64; e0 < units; e0 += 128 * kU) {
        uint32_t off[kU];
        float4 acc[kU];
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int e = min(e0 + k * 128, units - 1);  // a clamped duplicate is not stored
          const int rr = e / (BN / 4), c4 = e % (BN / 4);
          off[k] = static_cast<uint32_t>(((row0 + rr) * C::RED_STRIDE + c4 * 4) * 4);
          acc[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
        for (int src0 = 0; src0 < p.csplit; src0 += 2) {
          float4 x0[kU], x1[kU];
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            x0[k] = ld_cluster_f4(cluster_map(red0 + off[k], static_cast<uint32_t>(src0)));
            x1[k] = make_float4(0.f, 0.f, 0.f, 0.f);
            if (src0 + 1 < p.csplit)
              x1[k] = ld_cluster_f4(cluster_map(red0 + off[k], static_cast<uint32_t>(src0 + 1)));
          }
#pragma unroll
          for (int k = 0; k < kU; ++k) {
            acc[k].x += x0[k].x;
            acc[k].y += x0[k].y;
            acc[k].z += x0[k].z;
            acc[k].w += x0[k].w;
            acc[k].x += x1[k].x;
            acc[k].y += x1[k].y;
            acc[k].z += x1[k].z;
            acc[k].w += x1[k].w;
          }
        }
#pragma unroll
        for (int k = 0; k < kU; ++k) {
          const int e = e0 + k * 128;
          if (e < units) {
            const int rr = e / (BN / 4), c4 = e % (BN / 4);
            *reinterpret_cast<float4 *>(slice + rr * C::RED_STRIDE + c4 * 4) = acc[k];
          }
        }
      }
      named_bar_sync(1, 128);
      // Phase 2: the slice's rows spread over the 128 epilogue threads, nparts adjacent
      // lanes per row, each running the epilogue on its share of the row's chunks.
      {
        const int nparts = per * 4 <= 128 ? 4 : per * 2 <= 128 ? 2 : 1;
        const int rl = r / nparts, cpart = r % nparts;
        const bool active = rl < per;
        const int rt = row0 + rl;  // row inside the tile
        const Item t = item_at(p, 0);
        const int row = t.m * p.tile_rows + rt;
        const bool row_ok = active && (rt < p.tile_rows) && (row < p.M);
        const float *mine = slice + (active ? rl : 0) * C::RED_STRIDE;
        auto fetch = [&](int c, float (&v)[32]) {
          if (!active) {
#pragma unroll
            for (int k = 0; k < 32; ++k) v[k] = 0.f;
            return;
          }
          const float4 *src = reinterpret_cast<const float4 *>(mine + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const float4 x = src[k];
            v[4 * k] = x.x;
            v[4 * k + 1] = x.y;
            v[4 * k + 2] = x.z;
            v[4 * k + 3] = x.w;
          }
        };
        TopkState tk;
        float *stash = nullptr;
        epilogue_tile<BN, EPI>(p, t, row, row_ok, fetch, tk, stash, cpart, nparts);
      }
    }
    __syncwarp();
    cluster_sync_all();  // peers may still be reading this CTA's partial
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// ------------------------------------------------------------------ host side

int gemm_tiles(int M, int tile_rows, int N, int groups, int dual, int BN) {
  const int m_tiles = (M + tile_rows - 1) / tile_rows;
  const int ncols = dual ? BN / 2 : BN;
  const int n_tiles = (N + ncols - 1) / ncols;
  return m_tiles * n_tiles * groups;
}

void topk_range_plan(int n_tiles, int m_tiles, int num_sms, int *tiles_per_cta, int *ranges) {
  const int ranges0 = std::max(1, num_sms / std::max(1, m_tiles));
  const int tpc = (n_tiles + ranges0 - 1) / ranges0;
  *tiles_per_cta = std::max(1, tpc);
  *ranges = (n_tiles + *tiles_per_cta - 1) / *tiles_per_cta;
}

// Chooses the cluster split S: the largest S <= 8 such that every tile's cluster of
// S CTAs is resident at once (cluster_cap[S] = clusters of that size the device
// holds concurrently; 0 = unknown, then tiles * S <= num_sms) and every split keeps
// >= 8 k-tiles. Multi-wave cluster launches measured slower than one persistent
// unsplit wave, so larger tile counts stay unsplit.
void gemm_plan(int M, int tile_rows, int N, int K, int groups, int dual, int BN, int slabs, int num_sms,
               int epi, const int *cluster_cap, int *splits_out, int *kps_out, int *items_out,
               int *grid_out, int *csplit_out) {
  const int tiles = gemm_tiles(M, tile_rows, N, groups, dual, BN);
  const int kt = (K + BK - 1) / BK;                            // 64-column k-tiles
  const int kst = (K + BK * slabs - 1) / (BK * slabs);         // pipeline stages along K
  int best_s = 1;
  if (epi != EPI_TOPK)
    for (int S = 2; S <= 8; ++S) {
      const bool fits = cluster_cap && cluster_cap[S] > 0 ? tiles <= cluster_cap[S]
                                                          : (long long)tiles * S <= num_sms;
      if (fits && kt >= 8 * S) best_s = S;
    }
  *splits_out = 1;
  *csplit_out = best_s;
  *kps_out = (kst + best_s - 1) / best_s;
  *items_out = best_s > 1 ? tiles * best_s : tiles;
  *grid_out = best_s > 1 ? tiles * best_s : std::max(1, std::min(tiles, num_sms));
}

// Per-instantiation launch set-up, done once per process: the dynamic shared memory
// opt-in and, for each cluster size 2..8, how many clusters of this kernel the device
// keeps resident at once (cluster placement is limited by the GPCs, so tiles * S <=
// SMs alone does not guarantee a single wave).
struct KernelSetup {
  cudaError_t err = cudaSuccess;
  int cluster_cap[9] = {0, 0, 0, 0, 0, 0, 0, 0, 0};
};

template <int BN, int EPI, int MS>
static const KernelSetup &kernel_setup() {
  static const KernelSetup setup = [] {
    KernelSetup k;
    constexpr size_t smem = gemm_smem_bytes<BN, EPI, MS>();
    k.err = cudaFuncSetAttribute(gemm_tc_kernel<BN, EPI, MS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
    if (k.err != cudaSuccess || EPI == EPI_TOPK || MS > 1) return k;
    for (int S = 2; S <= 8; ++S) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(S);
      cfg.blockDim = dim3(gemm_threads<EPI>());
      cfg.dynamicSmemBytes = smem;
      cudaLaunchAttribute attr;
      attr.id = cudaLaunchAttributeClusterDimension;
      attr.val.clusterDim.x = S;
      attr.val.clusterDim.y = 1;
      attr.val.clusterDim.z = 1;
      cfg.attrs = &attr;
      cfg.numAttrs = 1;
      int n = 0;
      if (cudaOccupancyMaxActiveClusters(&n, gemm_tc_kernel<BN, EPI, MS>, &cfg) != cudaSuccess) {
        (void)cudaGetLastError();
        n = 0;
      }
      k.cluster_cap[S] = n;
    }
    return k;
  }();
  return setup;
}

template <int BN, int EPI, int MS = 1>
static cudaError_t plan_and_launch(GemmParams &p, int num_sms, cudaStream_t s) {
  const KernelSetup &ks = kernel_setup<BN, EPI, MS>();
  if (ks.err != cudaSuccess) return ks.err;
  if (p.slabs > gemm_slabs<BN, EPI>() || (p.slabs == 2 && (p.a_grouped || p.dual)))
    return cudaErrorInvalidValue;
  if (MS > 1 && !p.a_grouped && p.tile_rows != BM) return cudaErrorInvalidValue;
  int grid;
  p.csplit = 1;
  if (EPI == EPI_TOPK) {
    p.splits = 1;
    p.kt_per_split = p.kt_total;
    int ranges = 0;
    topk_range_plan(p.n_tiles, p.m_tiles, num_sms, &p.tiles_per_cta, &ranges);
    grid = ranges * p.m_tiles;
    p.items = grid;
  } else if (MS > 1) {
    // M-stacked tiles never split K (chosen only when the tiles fill the GPU)
    p.splits = 1;
    p.kt_per_split = p.kt_total;
    p.items = p.m_tiles * p.n_tiles * p.groups;
    grid = std::max(1, std::min(p.items, num_sms));
  } else {
    gemm_plan(p.M, p.tile_rows, p.N, p.K, p.groups, p.dual, BN, p.slabs, num_sms, p.epi, ks.cluster_cap,
              &p.splits, &p.kt_per_split, &p.items, &grid, &p.csplit);
  }
  p.rast_gm = std::max(1, p.m_tiles);
  if (EPI != EPI_TOPK && p.csplit == 1) {
    // The tiles in flight at once (one per CTA) read A blocks of rast_gm m-tiles and the
    // weight tiles of grid / rast_gm columns; each block is fetched from DRAM once per
    // group and shared through L2. rast_gm = sqrt(grid * B tile / A tile) minimises the
    // bytes one wave of tiles fetches.
    const double a_tile = (double)MS * BM, b_tile = (double)BN;
    const int gm = (int)std::lround(std::sqrt((double)grid * b_tile / a_tile));
    p.rast_gm = std::max(1, std::min(p.m_tiles, gm));
  }
  constexpr size_t smem = gemm_smem_bytes<BN, EPI, MS>();
  if (p.csplit > 1)
    return launch_pdl_cluster(gemm_tc_kernel<BN, EPI, MS>, dim3(grid), dim3(gemm_threads<EPI>()), smem, s, p.csplit,
                              p);
  return launch_pdl(gemm_tc_kernel<BN, EPI, MS>, dim3(grid), dim3(gemm_threads<EPI>()), smem, s, p);
}

// 128-row blocks per tile (1 or 2) a launch takes. The stackable GEMMs (128-wide: W_c's
// fp32 store and the K/V cache scatter; the 192-wide SwiGLU pair) stack when the CTA that
// takes the most tiles (persistent rounds) then takes in fewer operand rows per k column
// (A rows + B rows per tile times rounds): each stacked tile reads its weight tile once for
// 256 rows instead of 128. The 128-wide ones hold two 96 KB stages when stacked, so they
// also need a stacked tile for every SM. Measured and left out: the stacked QKV at 512 rows
// (96 tiles on 96 SMs, 40 -> 43 us) and a stacked LM head (two 256-wide accumulators fill
// the tensor memory, and its top-k epilogue, no longer under the next tile's MMAs, made the
// 448-row LM head 0.44 -> 0.72 ms).
int gemm_mstack(int epi, int BN, int M, int tile_rows, int N, int groups, int a_grouped, int dual, int num_sms) {
  (void)tile_rows;
  if (epi == EPI_TOPK) return 1;
  const bool plain = (BN == 128 || BN == 256) && !dual && (epi == EPI_F32 || epi == EPI_KV);
  const bool swiglu = BN == 192 && dual && epi == EPI_SWIGLU;
  if (a_grouped || !(plain || swiglu) || M <= BM) return 1;
  const long long cols = (long long)((N + (dual ? BN / 2 : BN) - 1) / (dual ? BN / 2 : BN)) * groups;
  const long long t1 = (long long)((M + BM - 1) / BM) * cols, t2 = (long long)((M + 2 * BM - 1) / (2 * BM)) * cols;
  const long long G = std::max(1, num_sms);
  if (plain && t2 < G) return 1;
  return ((t2 + G - 1) / G) * (2 * BM + BN) < ((t1 + G - 1) / G) * (BM + BN) ? 2 : 1;
}

static bool use_mstack(const GemmParams &p, int BN, int num_sms) {
  return gemm_mstack(p.epi, BN, p.M, p.a_grouped ? p.tile_rows : BM, p.N, p.groups, p.a_grouped, p.dual,
                     num_sms) == 2;
}

cudaError_t gemm_launch(GemmParams &p, int BN, int num_sms, cudaStream_t s) {
  const int ms = use_mstack(p, BN, num_sms) ? 2 : 1;
  if (p.a_grouped == 0) p.tile_rows = BM;  // rows per 128-lane block; a tile has ms blocks
  p.m_tiles = (p.M + ms * p.tile_rows - 1) / (ms * p.tile_rows);
  const int ncols = p.dual ? BN / 2 : BN;
  p.n_tiles = (p.N + ncols - 1) / ncols;
  if (p.slabs != 2) p.slabs = 1;
  p.kt_total = (p.K + BK * p.slabs - 1) / (BK * p.slabs);  // stages along K
  // expect-tx bytes of one stage: the A box(es) plus the B box(es), per slab (a slab past
  // K or rows past M are zero-filled by the copy and still counted)
  const uint32_t a_rows = p.a_grouped ? (uint32_t)p.tile_rows : (uint32_t)BM;
  p.stage_tx_bytes = (uint32_t)p.slabs * ((uint32_t)ms * a_rows * BK * 2 + (uint32_t)BN * BK * 2);
  if (ms == 2) {
    switch (BN * 16 + p.epi) {
      case 128 * 16 + EPI_F32: return plan_and_launch<128, EPI_F32, 2>(p, num_sms, s);
      case 128 * 16 + EPI_KV: return plan_and_launch<128, EPI_KV, 2>(p, num_sms, s);
      case 256 * 16 + EPI_F32: return plan_and_launch<256, EPI_F32, 2>(p, num_sms, s);
      case 256 * 16 + EPI_KV: return plan_and_launch<256, EPI_KV, 2>(p, num_sms, s);
      case 192 * 16 + EPI_SWIGLU: return plan_and_launch<192, EPI_SWIGLU, 2>(p, num_sms, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (BN * 16 + p.epi) {
    case 128 * 16 + EPI_BF16: return plan_and_launch<128, EPI_BF16>(p, num_sms, s);
    case 128 * 16 + EPI_F32: return plan_and_launch<128, EPI_F32>(p, num_sms, s);
    case 128 * 16 + EPI_RESID: return plan_and_launch<128, EPI_RESID>(p, num_sms, s);
    case 128 * 16 + EPI_ROPE: return plan_and_launch<128, EPI_ROPE>(p, num_sms, s);
    case 128 * 16 + EPI_SWIGLU: return plan_and_launch<128, EPI_SWIGLU>(p, num_sms, s);
    case 192 * 16 + EPI_SWIGLU: return plan_and_launch<192, EPI_SWIGLU>(p, num_sms, s);
    case 128 * 16 + EPI_DUAL_F32: return plan_and_launch<128, EPI_DUAL_F32>(p, num_sms, s);
    case 128 * 16 + EPI_KV: return plan_and_launch<128, EPI_KV>(p, num_sms, s);
    case 256 * 16 + EPI_TOPK: return plan_and_launch<256, EPI_TOPK>(p, num_sms, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace df
