// Context attention of the drafter layer with KV injection, on the tcgen05 tensor cores:
//   for each sequence i and query head h (kv head g = h / (Hq/Hkv)):
//   o = softmax(q K^T / sqrt(hd)) V,  K = [K_c (cached context rows); K_b (block rows)],
//   V likewise, with no mask (the block is bidirectional).
// Source: "DFlash 投机解码：块扩散草稿与 KV 注入", 二、块扩散草稿 (attention equations).
//
// K_b and V_b were written by the QKV GEMM into cache rows [ctx_len, ctx_len + B), so a
// (sequence, kv head) pair attends to cache rows [0, ctx_len + B): one contiguous range,
// or 64-row pages named by the block table (one page per 64-key unit).
//
// Work decomposition (even split of the streamed bytes): the keys of every pair are cut
// into 64-key units; the units of all pairs, in (sequence, kv head) order, are divided
// into `grid` contiguous ranges of equal size, one per CTA (one CTA per SM). A CTA walks
// its range; each maximal run of units of one pair is a segment. A segment that covers
// its whole pair writes the final output; otherwise it writes an unnormalised partial
// (o, running max, running sum) to slot pair + cta, and a merge kernel combines the
// partials of the pair in CTA order. The split points depend on the batch's context
// lengths only, so results are deterministic for a given batch.
//
// One CTA, 7 warps when G*B <= 64 query rows, else 11 (AttnRoles below):
//   TMA producer  Q tile of the segment's pair ({64 of hd, Hq/Hkv heads, B rows} boxes
//                 from the qkv buffer) and K and V tiles of two units (128 cache rows x hd,
//                 128-byte swizzle; one copy each, or one per unit and 64-column half when
//                 paged) into a 3-stage ring.
//   S issuer      S = Q K^T (M = 128 query rows, the G*B real ones zero-padded, N = 64
//                 keys, K = hd) into TMEM S buffer j % 2; owns the TMEM allocation.
//   PV issuer     O_{j%2} += P V (N = hd, K = 64 keys; P read from TMEM buffer j % 4, V
//                 MN-major straight from its TMA tile); its commit on P buffer j % 4 also
//                 tells the softmax half that PV(j) is complete.
//   softmax       two halves; half h takes the units j with j % 2 == h and keeps its own
//                 running max, running sum and O_h, so the two halves work on consecutive
//                 units at once. Thread r of a half owns query row r (its TMEM lane): it
//                 reads S, masks keys beyond L, updates its max and sum in fp32 (exp2 with
//                 the 1/sqrt(hd) * log2(e) scale folded in) and writes P (bf16) to TMEM.
//                 O_h is rescaled in TMEM only when the row's max grows by more than 2^8
//                 in probability scale, so P stays <= 256 and most units need no O round
//                 trip. At the end of a segment half 0 merges (m, l, O) of both halves and
//                 writes the output or the partial.
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace df {

// Warp roles for NQ TMEM lane quarters of real query rows (NQ = 2 when G*B <= 64, else
// 4): half 0 = warps [0, NQ), half 1 = warps [4, 4 + NQ) (warp w reads TMEM lanes of
// quarter w % 4), then the producer and the two MMA-issuing warps (S and PV: one
// thread issuing both streams was the bottleneck, each tcgen05.mma taking tens of cycles
// to issue).
template <int NQ>
struct AttnRoles {
  static constexpr int PRODUCER = NQ == 4 ? 8 : 2;
  static constexpr int MMA = PRODUCER + 1;              // S = Q K^T issuer (and TMEM owner)
  static constexpr int PV = NQ == 4 ? 10 : 6;           // O += P V issuer
  static constexpr int THREADS = (PV + 1) * 32;
  static constexpr int HALF_THREADS = NQ * 32;
};
constexpr int kKeys = 64;           // keys per unit
constexpr int kAttnStages = 3;    // ring stages of two units each
constexpr int kQRows = 128;         // MMA M: query rows, zero-padded beyond G*B
constexpr int kAttnDrainSpin = 1 << 22;
constexpr float kRescaleLog2 = 8.0f;

template <int HD>
struct AttnCfg {
  static constexpr int ATOMS = HD / 64;               // 128-byte swizzle atoms across hd
  static constexpr int ATOM_Q = kQRows * 128;         // one atom of the Q tile
  static constexpr int ATOM_KV = 2 * kKeys * 128;     // one atom of a two-unit K or V tile
  static constexpr int UNIT_KV = kKeys * 128;         // one unit's rows inside an atom
  static constexpr int Q_BYTES = ATOMS * ATOM_Q;
  static constexpr int KV_TILE = ATOMS * ATOM_KV;
  static constexpr int STAGE = 2 * KV_TILE;           // K tile then V tile: [atom][2 units x 64 rows][128 B]
  static constexpr int OFF_KV = Q_BYTES;
  static constexpr int OFF_BAR = OFF_KV + kAttnStages * STAGE;
  static constexpr int OFF_ML = OFF_BAR + 512;        // half 1's (max, sum) per row
  static constexpr size_t SMEM = 1024 + OFF_ML + kQRows * 8;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t S_COL = 0;                // two S buffers of 64 columns
  static constexpr uint32_t O_COL = 128;              // O_0, O_1: hd columns each
  static constexpr uint32_t P_COL = 128 + 2 * HD;     // 4 P buffers (unit j in j % 4): 64 bf16 keys = 32 columns each
};

__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Context rows of sequence i used by the attention: ctx_len clamped to the caller's
// bound and to the cache (the block occupies the B rows after it).
__device__ __forceinline__ int attn_ctx(const AttnParams &p, int i) {
  const int hi = min(p.max_ctx, p.Cmax - p.B);
  return max(0, min(p.ctx_len[i], hi));
}
__device__ __forceinline__ int attn_units(const AttnParams &p, int i) {
  return (attn_ctx(p, i) + p.B + kKeys - 1) / kKeys;
}

// Warp-collective: Hkv * (sum of units of sequences [0, n)).
__device__ long long attn_units_before(const AttnParams &p, int n, int lane) {
  long long s = 0;
  for (int i = lane; i < n; i += 32) s += attn_units(p, i);
#pragma unroll
  for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  return s * p.Hkv;
}

// First unit of CTA c when T units are split over G CTAs.
__device__ __forceinline__ long long attn_cta_start(long long T, int G, int c) {
  return (long long)c * T / G;
}
// The CTA whose range holds unit u.
__device__ __forceinline__ int attn_cta_of(long long T, int G, long long u) {
  return static_cast<int>(((u + 1) * G + T - 1) / T - 1);
}

// Position of a CTA in its unit range.
struct AttnWalk {
  int pair;   // i * Hkv + g
  int unit;   // unit index inside the pair
  int L, U;   // keys and units of the pair
  int seg;    // segment index inside this CTA
  int seg_unit0;  // first unit of the current segment inside the pair
  int left;   // units left in this CTA's range, including the current one
  int slot;   // 0: first unit of its ring stage, 1: second (same segment, next 64 keys)
  int stage;  // ring stages used before this unit's stage
};

// Context rows of the first kCtxCache sequences, copied to shared memory with the schedule
// (before griddepcontrol.wait), so the walks' pair changes read no global memory.
constexpr int kCtxCache = 64;
__device__ __forceinline__ int walk_ctx(const AttnParams &p, const int *sctx, int i) {
  return i < kCtxCache ? sctx[i] : attn_ctx(p, i);
}

__device__ __forceinline__ void walk_set_pair(AttnWalk &w, const AttnParams &p, const int *sctx) {
  const int i = w.pair / p.Hkv;
  w.L = walk_ctx(p, sctx, i) + p.B;
  w.U = (w.L + kKeys - 1) / kKeys;
}
__device__ __forceinline__ bool walk_first(const AttnWalk &w) { return w.unit == w.seg_unit0; }
__device__ __forceinline__ bool walk_last(const AttnWalk &w) { return w.left == 1 || w.unit == w.U - 1; }
__device__ __forceinline__ void walk_next(AttnWalk &w, const AttnParams &p, const int *sctx) {
  // the next unit shares this unit's stage when this is its first slot and the
  // segment continues (then its keys follow directly)
  const bool share = w.slot == 0 && !walk_last(w);
  w.slot = share ? 1 : 0;
  w.stage += share ? 0 : 1;
  --w.left;
  if (++w.unit == w.U) {
    ++w.pair;
    w.unit = 0;
    w.seg_unit0 = 0;
    ++w.seg;
    if (w.left > 0) walk_set_pair(w, p, sctx);
  }
}

template <int HD, int NQ>
__global__ void __launch_bounds__(AttnRoles<NQ>::THREADS, 1)
    attn_tc_kernel(const __grid_constant__ AttnParams p) {
  using C = AttnCfg<HD>;
  using Ro = AttnRoles<NQ>;
  constexpr int HT = Ro::HALF_THREADS;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                              ~static_cast<uintptr_t>(1023));
  uint8_t *sQ = smem;
  uint8_t *sKV = smem + C::OFF_KV;
  uint64_t *kv_full = reinterpret_cast<uint64_t *>(smem + C::OFF_BAR);
  uint64_t *kv_empty = kv_full + kAttnStages;
  uint64_t *s_full = kv_empty + kAttnStages;   // [2]
  uint64_t *s_empty = s_full + 2;              // [2]
  uint64_t *p_full = s_empty + 2;              // [4]: P of unit j in buffer j % 4
  // [4]: PV of unit j (and every MMA before it) completed. Each buffer's phases are waited
  // in order by the half that owns it, so one parity wait is exact for any PV that half
  // has issued P for: the PV four units earlier is already known complete.
  uint64_t *p_empty = p_full + 4;
  uint64_t *q_full = p_empty + 4;
  uint64_t *q_empty = q_full + 1;
  uint64_t *o_free = q_empty + 1;             // both O read at a segment end
  uint64_t *ml_ready = o_free + 1;            // half 1's (max, sum) written
  uint64_t *mma_done = ml_ready + 1;          // [2]: drain of the S and the PV issuer
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(mma_done + 2);
  int *sched = reinterpret_cast<int *>(tmem_slot + 1);  // [pair, unit, count]
  int *sctx = reinterpret_cast<int *>(smem + C::OFF_BAR + 256);  // [kCtxCache] context rows
  static_assert((2 * kAttnStages + 2 + 2 + 4 + 4 + 2 + 4) * 8 + 4 + 12 <= 256 &&
                    256 + kCtxCache * 4 <= C::OFF_ML - C::OFF_BAR,
                "barrier region overflows");
  float2 *ml1 = reinterpret_cast<float2 *>(smem + C::OFF_ML);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;
  const int R = G * p.B;  // real query rows

  if (threadIdx.x == 0) {
    for (int s = 0; s < kAttnStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&s_full[b], 1);
      mbar_init(&s_empty[b], HT);
      mbar_init(&p_full[b], HT);
      mbar_init(&p_full[b + 2], HT);
      mbar_init(&p_empty[b], 1);
      mbar_init(&p_empty[b + 2], 1);
    }
    mbar_init(q_full, 1);
    mbar_init(q_empty, 1);
    mbar_init(o_free, HT);
    mbar_init(ml_ready, HT);
    mbar_init(&mma_done[0], 1);
    mbar_init(&mma_done[1], 1);
    fence_mbar_init();
  }
  if (warp == Ro::PRODUCER && lane == 0) {
    tma_prefetch_desc(&p.tmQ);
    tma_prefetch_desc(&p.tmK);
    tma_prefetch_desc(&p.tmV);
  }
  if (warp == Ro::MMA) {
    tmem_alloc(tmem_slot, C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp < NQ) {
    // Zero the padding rows of Q (rows >= R are never loaded), so the padded MMA rows
    // compute on zeros.
    const int t = threadIdx.x;
    for (int a = 0; a < C::ATOMS; ++a)
      for (int e = R * 8 + t; e < kQRows * 8; e += HT)
        *reinterpret_cast<uint4 *>(sQ + a * C::ATOM_Q + e * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }

  // The schedule reads only ctx_len, final before any kernel of the drafter starts (the
  // first one waits for the context append before it lets the next launch): it is
  // computed while the QKV GEMM still runs; the q / k_b / v_b inputs are read after the
  // griddepcontrol.wait below.
  if (warp == Ro::PRODUCER) {
    for (int i = lane; i < p.nb && i < kCtxCache; i += 32) sctx[i] = attn_ctx(p, i);
    // Schedule: total units, this CTA's range, and the pair/unit it starts at.
    const long long T = attn_units_before(p, p.nb, lane);
    const int Ge = T < p.grid ? static_cast<int>(T) : p.grid;
    int count = 0, pair0 = 0, unit0 = 0;
    if (static_cast<int>(blockIdx.x) < Ge) {
      const long long u0 = attn_cta_start(T, Ge, blockIdx.x);
      const long long u1 = attn_cta_start(T, Ge, blockIdx.x + 1);
      count = static_cast<int>(u1 - u0);
      // find the sequence holding u0: inclusive scan of Hkv * units, 32 sequences at a time
      long long base = 0;
      int seq = -1;
      for (int b = 0; b < p.nb && seq < 0; b += 32) {
        const int i = b + lane;
        long long v = i < p.nb ? (long long)p.Hkv * attn_units(p, i) : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const long long y = __shfl_up_sync(0xffffffffu, v, o);
          if (lane >= o) v += y;
        }
        const unsigned hit = __ballot_sync(0xffffffffu, i < p.nb && base + v > u0);
        if (hit) {
          const int l = __ffs(hit) - 1;
          const long long before = base + __shfl_sync(0xffffffffu, v, l) -
                                   (long long)p.Hkv * attn_units(p, b + l);
          seq = b + l;
          const int U = attn_units(p, seq);
          const long long off = u0 - before;
          pair0 = seq * p.Hkv + static_cast<int>(off / U);
          unit0 = static_cast<int>(off % U);
        }
        base += __shfl_sync(0xffffffffu, v, 31);
      }
      if (seq < 0) count = 0;  // unreachable when T counts every unit
    }
    if (lane == 0) {
      sched[0] = pair0;
      sched[1] = unit0;
      sched[2] = count;
    }
  }
  if (warp == Ro::MMA && lane == 0) {
    // Report context lengths outside [0, min(max_ctx, Cmax - B)] once per launch.
    if (blockIdx.x == 0)
      for (int i = 0; i < p.nb; ++i) {
        const int c = p.ctx_len[i];
        if (c < 0 || c > p.max_ctx || c > p.Cmax - p.B) flag_status(p.status, kStatusCheck);
      }
  }
  griddep_wait();
  if (threadIdx.x == 0) griddep_launch();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int nunits = sched[2];
  AttnWalk w0;
  w0.pair = sched[0];
  w0.unit = sched[1];
  w0.seg = 0;
  w0.seg_unit0 = w0.unit;
  w0.left = nunits;
  w0.slot = 0;
  w0.stage = 0;
  if (nunits > 0) walk_set_pair(w0, p, sctx);

  if (warp == Ro::PRODUCER) {
    if (lane == 0 && nunits > 0 && !p.stall) {
      // ---------------- TMA producer
      const uint64_t pol_kv = policy_evict_first();
      const uint64_t pol_q = policy_evict_last();
      const uint32_t q_bytes = static_cast<uint32_t>(C::ATOMS * R * 128);
      AttnWalk w = w0;
      bool ok = true;
      int j = 0, q_loads = 0, stages = 0;
      for (; j < nunits; ++j) {
        const int i = w.pair / p.Hkv, g = w.pair % p.Hkv;
        if (walk_first(w)) {
          if (w.seg > 0 && !mbar_wait(q_empty, (w.seg - 1) & 1, p.max_spin)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(q_full, q_bytes);
#pragma unroll
          for (int a = 0; a < C::ATOMS; ++a)
            tma_load_3d(sQ + a * C::ATOM_Q, &p.tmQ, q_full, a * 64, g * G, i * p.B, pol_q);
          ++q_loads;
        }
        if (w.slot == 0) {
          // one copy each for K and V: 128 rows (this unit and the next 64 keys) of
          // every 64-wide half of hd. A tensor copy from one SM costs about one DRAM
          // round trip whatever its size, so the copies are made as large as smem allows.
          const int st = w.stage % kAttnStages;
          if (w.stage >= kAttnStages &&
              !mbar_wait(&kv_empty[st], ((w.stage / kAttnStages) & 1) ^ 1, p.max_spin)) {
            ok = false;
            break;
          }
          uint8_t *kt = sKV + st * C::STAGE;
          if (p.page_table == nullptr) {
            mbar_arrive_expect_tx(&kv_full[st], C::STAGE);
            const int row = p.layer_row0 + (i * p.Hkv + g) * p.Cmax + w.unit * kKeys;
            tma_load_3d(kt, &p.tmK, &kv_full[st], 0, row, 0, pol_kv);
            tma_load_3d(kt + C::KV_TILE, &p.tmV, &kv_full[st], 0, row, 0, pol_kv);
          } else {
            // paged: each unit is one page; its 64 rows of every atom land where the
            // two-unit copy puts them (atom a, unit slot u)
            const int nu = walk_last(w) ? 1 : 2;
            mbar_arrive_expect_tx(&kv_full[st], static_cast<uint32_t>(nu * 2 * C::ATOMS * C::UNIT_KV));
            for (int u = 0; u < nu; ++u) {
              int pg = p.page_table[(long long)i * p.pages_per_seq + w.unit + u];
              if (pg < 0 || pg >= p.num_pages) {
                flag_status(p.status, kStatusCheck);
                pg = 0;
              }
              const int row = p.layer_row0 + (pg * p.Hkv + g) * kPageRows;
#pragma unroll
              for (int a = 0; a < C::ATOMS; ++a) {
                uint8_t *dst = kt + a * C::ATOM_KV + u * C::UNIT_KV;
                tma_load_3d(dst, &p.tmK, &kv_full[st], 0, row, a, pol_kv);
                tma_load_3d(dst + C::KV_TILE, &p.tmV, &kv_full[st], 0, row, a, pol_kv);
              }
            }
          }
          stages = w.stage + 1;
        }
        walk_next(w, p, sctx);
      }
      if (!ok) flag_status(p.status, kStatusTimeout);
      // Every issued load must land before the CTA may exit (bounded).
      for (int k = max(0, stages - kAttnStages); k < stages; ++k)
        mbar_wait(&kv_full[k % kAttnStages], (k / kAttnStages) & 1, kAttnDrainSpin);
      if (q_loads > 0) mbar_wait(q_full, (q_loads - 1) & 1, kAttnDrainSpin);
    }
  } else if (warp == Ro::MMA) {
    if (lane == 0 && nunits > 0) {
      // ---------------- S issuer: S(j) once its K tile has landed and S buffer j % 2 has
      // been read by the softmax
      constexpr uint32_t id_s = idesc_bf16_f32(kQRows, kKeys);
      const uint64_t q_desc0 = sw128_kmajor_desc(smem_u32(sQ));
      const uint64_t kv_desc0 = sw128_kmajor_desc(smem_u32(sKV));
      AttnWalk ws = w0;
      bool ok = true;
      for (int js = 0; js < nunits; ++js) {
        const int st = ws.stage % kAttnStages, sb = js & 1;
        if (walk_first(ws) && !mbar_wait(q_full, ws.seg & 1, p.max_spin)) ok = false;
        // (the second unit of a stage landed with the first)
        if (ok && ws.slot == 0 && !mbar_wait(&kv_full[st], (ws.stage / kAttnStages) & 1, p.max_spin)) ok = false;
        if (ok && js >= 2 && !mbar_wait(&s_empty[sb], ((js >> 1) - 1) & 1, p.max_spin)) ok = false;
        if (!ok) break;
        tc_fence_after();
        // descriptors differ only in their start-address field: add the k-step offset
        const uint64_t kd = kv_desc0 + static_cast<uint64_t>((st * C::STAGE + ws.slot * C::UNIT_KV) >> 4);
        const uint32_t d_s = tmem_base + C::S_COL + sb * kKeys;
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint64_t qo = static_cast<uint64_t>(((kk >> 2) * C::ATOM_Q + (kk & 3) * 32) >> 4);
          const uint64_t ko = static_cast<uint64_t>(((kk >> 2) * C::ATOM_KV + (kk & 3) * 32) >> 4);
          tc_mma_bf16(d_s, q_desc0 + qo, kd + ko, id_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(&s_full[sb]);
        if (walk_last(ws)) tc_commit(q_empty);
        walk_next(ws, p, sctx);
      }
      if (!ok) flag_status(p.status, kStatusTimeout);
      // Every issued MMA must complete before TMEM is freed (bounded).
      tc_commit(&mma_done[0]);
      mbar_wait(&mma_done[0], 0, kAttnDrainSpin);
    }
  } else if (warp == Ro::PV) {
    if (lane == 0 && nunits > 0) {
      // ---------------- PV issuer: O_{j%2} += P(j) V(j) once P(j) is in tensor memory; the
      // first unit of each half in a segment starts the accumulator (after both O of the
      // previous segment were read); the last unit of a stage releases it
      constexpr uint32_t id_pv = idesc_bf16_f32(kQRows, HD) | kIdescBMajorMN;
      const uint64_t v_desc0 = sw128_mnmajor_desc(smem_u32(sKV + C::KV_TILE), C::ATOM_KV);
      AttnWalk wp = w0;
      int jf = 0;
      bool ok = true;
      for (int jp = 0; jp < nunits; ++jp) {
        const int st = wp.stage % kAttnStages, pb = jp & 1, pq = jp & 3;
        if (walk_first(wp)) jf = jp;
        const bool start = jp < jf + 2;
        if (!mbar_wait(&p_full[pq], (jp >> 2) & 1, p.max_spin)) ok = false;
        if (ok && start && wp.seg > 0 && !mbar_wait(o_free, (wp.seg - 1) & 1, p.max_spin)) ok = false;
        if (!ok) break;
        tc_fence_after();
        const uint64_t vd = v_desc0 + static_cast<uint64_t>((st * C::STAGE + wp.slot * C::UNIT_KV) >> 4);
        const uint32_t d_o = tmem_base + C::O_COL + pb * HD;
        const uint32_t a_p = tmem_base + C::P_COL + pq * 32;
#pragma unroll
        for (int kk = 0; kk < kKeys / 16; ++kk)
          tc_mma_bf16_tmem_a(d_o, a_p + kk * 8, vd + static_cast<uint64_t>((kk * 16 * 128) >> 4), id_pv,
                             (!start || kk > 0) ? 1u : 0u);
        tc_commit(&p_empty[pq]);
        if (wp.slot == 1 || walk_last(wp)) tc_commit(&kv_empty[st]);  // last unit of its stage
        walk_next(wp, p, sctx);
      }
      if (!ok) flag_status(p.status, kStatusTimeout);
      tc_commit(&mma_done[1]);
      mbar_wait(&mma_done[1], 0, kAttnDrainSpin);
    }
  } else if ((warp & 3) < NQ) {
    // ---------------- softmax warps: half h = warp / 4 takes units j % 2 == h; thread r
    // of a half owns query row r = TMEM lane r
    const int half = warp >> 2;
    const int q = warp & 3;
    const int r = q * 32 + lane;
    const bool real = r < R;
    const bool warp_real = q * 32 < R;
    const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
    const uint32_t o_mine = trow + C::O_COL + half * HD;
    const float sl2 = rsqrtf(static_cast<float>(HD)) * 1.4426950408889634f;
    // row r of the Q tile is block position r / G of query head g * G + r % G
    const int jq = r / G, hq = r % G;
    AttnWalk w = w0;
    float m_run = -FLT_MAX, l_run = 0.f;
    bool ok = true;
    int jf = 0;
    for (int j = 0; j < nunits && ok; ++j) {
      const int st = w.stage % kAttnStages;
      if (walk_first(w)) {
        jf = j;
        m_run = -FLT_MAX;
        l_run = 0.f;
      }
      if ((j & 1) == half) {
        const bool first = j < jf + 2;  // first unit of this half in the segment
        const int nv = min(kKeys, w.L - w.unit * kKeys);
        ok = mbar_wait(&s_full[half], (j >> 1) & 1, p.max_spin);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        tc_fence_after();
        float sv[kKeys];
        if (warp_real) {
          float t0[32], t1[32];
          tmem_ld32(trow + C::S_COL + half * kKeys, t0);
          tmem_ld32(trow + C::S_COL + half * kKeys + 32, t1);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            sv[c] = t0[c];
            sv[c + 32] = t1[c];
          }
        }
        tc_fence_before();
        mbar_arrive(&s_empty[half]);

        bool need = false;
        float alpha = 1.f;
        if (warp_real) {
          if (nv < kKeys) {
#pragma unroll
            for (int c = 0; c < kKeys; ++c) sv[c] = c < nv ? sv[c] : -FLT_MAX;
          }
          float m8[8];
#pragma unroll
          for (int a = 0; a < 8; ++a) m8[a] = fmaxf(sv[a], sv[a + 8]);
#pragma unroll
          for (int c = 16; c < kKeys; ++c) m8[c & 7] = fmaxf(m8[c & 7], sv[c]);
          const float mx = fmaxf(fmaxf(fmaxf(m8[0], m8[1]), fmaxf(m8[2], m8[3])),
                                 fmaxf(fmaxf(m8[4], m8[5]), fmaxf(m8[6], m8[7])));
          need = real && (mx - m_run) * sl2 > kRescaleLog2;
          if (need) {
            alpha = ex2_approx((m_run - mx) * sl2);
            m_run = mx;
            l_run *= alpha;
          }
        }
        if (!first && __any_sync(0xffffffffu, need)) {
          // O_h *= alpha once PV of this half's previous unit has completed
          ok = mbar_wait(&p_empty[(j - 2) & 3], ((j - 2) >> 2) & 1, p.max_spin);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int cc = 0; cc < HD / 32; ++cc) {
            float ov[32];
            tmem_ld32(o_mine + cc * 32, ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] *= alpha;
            tmem_st32(o_mine + cc * 32, ov);
          }
        }
        // P buffer j % 4 is free once PV of unit j - 4 has completed
        ok = j < 4 || mbar_wait(&p_empty[j & 3], ((j >> 2) - 1) & 1, p.max_spin);
        if (!__all_sync(0xffffffffu, ok)) {
          ok = false;
          break;
        }
        if (warp_real) {
          // P (bf16 pairs) into this half's P columns of the row's TMEM lane
          float pk[kKeys / 2];
          float ls[4] = {0.f, 0.f, 0.f, 0.f};
          const float mb = m_run * sl2;
#pragma unroll
          for (int c = 0; c < kKeys; c += 2) {
            const float p0 = ex2_approx(fmaf(sv[c], sl2, -mb));
            const float p1 = ex2_approx(fmaf(sv[c + 1], sl2, -mb));
            ls[(c >> 1) & 3] += p0 + p1;
            pk[c >> 1] = real ? __uint_as_float(pack_bf16x2(p0, p1)) : 0.f;
          }
          if (real) l_run += (ls[0] + ls[1]) + (ls[2] + ls[3]);
          tmem_st32(trow + C::P_COL + (j & 3) * 32, pk);
        }
        if (nv < kKeys) {
          // V rows beyond the last key may hold anything (even NaN): zero them, P is 0 there.
          ok = mbar_wait(&kv_full[st], (w.stage / kAttnStages) & 1, p.max_spin);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          uint8_t *vt = sKV + st * C::STAGE + C::KV_TILE + w.slot * C::UNIT_KV;
          const int nz = (kKeys - nv) * 8;  // 16-byte chunks per atom
          for (int e = r; e < C::ATOMS * nz; e += HT) {
            const int a = e / nz, x = e % nz;
            *reinterpret_cast<uint4 *>(vt + a * C::ATOM_KV + nv * 128 + x * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        if (nv < kKeys) fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[j & 3]);
      }

      if (walk_last(w)) {
        // segment [jf, j]: the last unit of each half in it, or -1
        const int seg = w.seg;
        const int last_h[2] = {(j & 1) == 0 ? j : (j - 1 >= jf ? j - 1 : -1),
                               (j & 1) == 1 ? j : (j - 1 >= jf ? j - 1 : -1)};
        if (half == 1) {
          // hand (max, sum) to half 0 once O_1 is final; the slot is free once half 0
          // has read the previous segment's
          ok = seg == 0 || mbar_wait(o_free, (seg - 1) & 1, p.max_spin);
          if (ok && last_h[1] >= 0) ok = mbar_wait(&p_empty[last_h[1] & 3], (last_h[1] >> 2) & 1, p.max_spin);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          ml1[r] = last_h[1] >= 0 ? make_float2(m_run, l_run) : make_float2(-FLT_MAX, 0.f);
          tc_fence_before();
          mbar_arrive(ml_ready);
        } else {
          ok = last_h[0] < 0 || mbar_wait(&p_empty[last_h[0] & 3], (last_h[0] >> 2) & 1, p.max_spin);
          if (ok) ok = mbar_wait(ml_ready, seg & 1, p.max_spin);
          if (!__all_sync(0xffffffffu, ok)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const float2 o1 = ml1[r];
          const bool has0 = last_h[0] >= 0, has1 = last_h[1] >= 0;
          const float m0 = has0 ? m_run : -FLT_MAX;
          const float M = fmaxf(m0, o1.x);
          const float a0 = has0 ? ex2_approx((m0 - M) * sl2) : 0.f;
          const float a1 = has1 ? ex2_approx((o1.x - M) * sl2) : 0.f;
          const float L = (has0 ? l_run * a0 : 0.f) + o1.y * a1;
          const bool whole = w.seg_unit0 == 0 && w.unit == w.U - 1;
          const int i = w.pair / p.Hkv, g = w.pair % p.Hkv;
          const int slot = w.pair + static_cast<int>(blockIdx.x);
          const float inv = 1.0f / L;
          if (warp_real) {
#pragma unroll 1
            for (int cc = 0; cc < HD / 32; ++cc) {
              float ov[32], o1v[32];
              if (has0) tmem_ld32(trow + C::O_COL + cc * 32, ov);
              if (has1) tmem_ld32(trow + C::O_COL + HD + cc * 32, o1v);
#pragma unroll
              for (int c = 0; c < 32; ++c)
                ov[c] = (has0 ? ov[c] * a0 : 0.f) + (has1 ? o1v[c] * a1 : 0.f);
              if (!real) continue;
              if (whole) {
                uint16_t *dst = p.o + ((size_t)i * p.B + jq) * ((size_t)p.Hq * HD) +
                                (size_t)(g * G + hq) * HD + cc * 32;
#pragma unroll
                for (int v = 0; v < 4; ++v)
                  reinterpret_cast<uint4 *>(dst)[v] =
                      make_uint4(pack_bf16x2(ov[8 * v] * inv, ov[8 * v + 1] * inv),
                                 pack_bf16x2(ov[8 * v + 2] * inv, ov[8 * v + 3] * inv),
                                 pack_bf16x2(ov[8 * v + 4] * inv, ov[8 * v + 5] * inv),
                                 pack_bf16x2(ov[8 * v + 6] * inv, ov[8 * v + 7] * inv));
              } else {
                float *dst = p.part_o + ((size_t)slot * R + r) * HD + cc * 32;
#pragma unroll
                for (int v = 0; v < 8; ++v)
                  reinterpret_cast<float4 *>(dst)[v] =
                      make_float4(ov[4 * v], ov[4 * v + 1], ov[4 * v + 2], ov[4 * v + 3]);
              }
            }
          }
          if (real && !whole)
            *reinterpret_cast<float2 *>(p.part_ml + ((size_t)slot * R + r) * 2) = make_float2(M, L);
          tc_fence_before();
          mbar_arrive(o_free);
        }
      }
      walk_next(w, p, sctx);
    }
    if (!ok) flag_status(p.status, kStatusTimeout);
  }

  tc_fence_before();
  __syncthreads();
  if (warp == Ro::MMA) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::TMEM_COLS);
  }
}

// Combine the partials of every pair whose units were split over several CTAs, in CTA
// order, and write o (bf16). One CTA per (pair, 8 query rows); one warp per row; each
// lane owns hd/32 consecutive output elements.
constexpr int kMergeWarps = 8;

template <int HD>
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const AttnParams p) {
  constexpr int E = HD / 32;
  // The schedule (which CTAs share this pair) reads only ctx_len, written long before by
  // the context append: the attention triggers this launch after its own
  // griddepcontrol.wait, so every kernel before the attention has completed. It is
  // computed before waiting for the attention; pairs written whole return at once.
  const int pair = blockIdx.x;
  const int i = pair / p.Hkv, g = pair % p.Hkv;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int G = p.Hq / p.Hkv;
  const int R = G * p.B;
  const int r = blockIdx.y * kMergeWarps + warp;
  // This grid's completion (what the next launch's griddepcontrol.wait waits for) must imply
  // the attention's, whose output o the next launch reads, even when no pair needs a merge:
  // CTA (0, 0) always waits for the attention; other CTAs with nothing to merge leave at once
  // (thousands of them waiting would hold the SMs' CTA slots).
  const bool anchor = blockIdx.x == 0 && blockIdx.y == 0;
  if (r >= R) {
    if (anchor) griddep_wait();
    return;
  }
  // total units and the units before this pair, in one pass over the sequences
  long long T = 0, before = 0;
  for (int q = lane; q < p.nb; q += 32) {
    const int u = attn_units(p, q);
    T += u;
    before += q < i ? u : 0;
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    T += __shfl_xor_sync(0xffffffffu, T, o);
    before += __shfl_xor_sync(0xffffffffu, before, o);
  }
  T *= p.Hkv;
  const int Ge = T < p.grid ? static_cast<int>(T) : p.grid;
  const int U = attn_units(p, i);
  const long long A = before * p.Hkv + (long long)g * U;
  const int c0 = attn_cta_of(T, Ge, A), c1 = attn_cta_of(T, Ge, A + U - 1);
  if (c0 == c1) {  // written whole by the attention kernel
    if (anchor) griddep_wait();
    return;
  }
  griddep_wait();
  griddep_launch();
  const float sl2 = rsqrtf(static_cast<float>(HD)) * 1.4426950408889634f;
  {
    // one pass, rescaling to the running maximum (the partials' loads do not depend on
    // each other, so they are in flight together)
    float M = -FLT_MAX, L = 0.f, acc[E];
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
#pragma unroll 4
    for (int c = c0; c <= c1; ++c) {
      const size_t row = (size_t)(pair + c) * R + r;
      const float2 ml = *reinterpret_cast<const float2 *>(p.part_ml + row * 2);
      float v[E];
      const float *src = p.part_o + row * HD + lane * E;
      if constexpr (E == 4) {
        const float4 x = *reinterpret_cast<const float4 *>(src);
        v[0] = x.x;
        v[1] = x.y;
        v[2] = x.z;
        v[3] = x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2 *>(src);
        v[0] = x.x;
        v[1] = x.y;
      }
      const float Mn = fmaxf(M, ml.x);
      const float a_old = exp2f((M - Mn) * sl2), a_new = exp2f((ml.x - Mn) * sl2);
      L = L * a_old + ml.y * a_new;
#pragma unroll
      for (int e = 0; e < E; ++e) acc[e] = acc[e] * a_old + v[e] * a_new;
      M = Mn;
    }
    const float inv = 1.0f / L;
    const int jq = r / G, hq = r % G;
    uint16_t *dst = p.o + ((size_t)i * p.B + jq) * ((size_t)p.Hq * HD) + (size_t)(g * G + hq) * HD + lane * E;
    if constexpr (E == 4) {
      *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                   pack_bf16x2(acc[2] * inv, acc[3] * inv));
    } else {
      *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
    }
  }
}

template <int HD, int NQ>
static cudaError_t launch_attn(const AttnParams &p, cudaStream_t s) {
  using C = AttnCfg<HD>;
  static const cudaError_t configured = cudaFuncSetAttribute(
      attn_tc_kernel<HD, NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
  if (configured != cudaSuccess) return configured;
  cudaError_t e = launch_pdl(attn_tc_kernel<HD, NQ>, dim3(p.grid), dim3(AttnRoles<NQ>::THREADS), C::SMEM,
                             s, p);
  if (e != cudaSuccess) return e;
  const int R = (p.Hq / p.Hkv) * p.B;
  return launch_pdl(attn_merge_kernel<HD>, dim3(p.nb * p.Hkv, (R + kMergeWarps - 1) / kMergeWarps),
                    dim3(kMergeWarps * 32), 0, s, p);
}

cudaError_t launch_attention(const AttnParams &p, cudaStream_t s) {
  if (p.Hq % p.Hkv != 0) return cudaErrorInvalidValue;
  const int R = (p.Hq / p.Hkv) * p.B;
  if (R > kQRows) return cudaErrorInvalidValue;
  const bool wide = R > 64;
  switch (p.hd) {
    case 64: return wide ? launch_attn<64, 4>(p, s) : launch_attn<64, 2>(p, s);
    case 128: return wide ? launch_attn<128, 4>(p, s) : launch_attn<128, 2>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace df
