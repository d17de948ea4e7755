// Split-K context attention of the drafter layer with KV injection:
//   for each sequence i and query head h (kv head g = h / (Hq/Hkv)):
//   o = softmax(q K^T / sqrt(hd)) V,  K = [K_c (cached context rows); K_b (block rows)],
//   V likewise, with no mask (the block is bidirectional).
// Source: "DFlash 投机解码：块扩散草稿与 KV 注入", 二、块扩散草稿 (attention equations).
//
// Work decomposition: one CTA per (context split s, kv head g, sequence i). The
// Hq/Hkv query heads that share g and the B block offsets form the rows of one
// query tile (64 rows at B=16, GQA 4:1), so every K/V byte streamed from HBM is
// used by all of them. Split 0 also owns the B block keys. Each CTA writes an
// unnormalised partial (o, running max m, running sum l); a merge kernel combines
// the splits in split order.
//
// Inner loop: 64-key sub-chunks of K and V are staged into shared memory with
// 16-byte cp.async (2-stage ring, XOR-swizzled rows for conflict-free ldmatrix; three
// CTAs share an SM so twelve warps hide the MMA and shared-memory latencies);
// each warp owns 16 query rows and runs QK^T and PV on tensor cores with
// mma.sync m16n8k16 (bf16 in, fp32 accumulate), keeping P in registers, with an
// online softmax in fp32 (exp2 with the 1/sqrt(hd) * log2(e) scale folded in).
#include <cfloat>

#include "common.cuh"
#include "kernels.h"

namespace df {

constexpr int kAttnThreads = 128;
constexpr int kSub = 64;  // keys per sub-chunk

template <int HD>
struct AttnCfg {
  static constexpr int ROW_BYTES = HD * 2;
  static constexpr int TILE_BYTES = kSub * ROW_BYTES;
  static constexpr int STAGES = 2;
  static constexpr size_t SMEM = size_t(STAGES) * 2 * TILE_BYTES;
};

// Byte offset of 16-byte chunk `chunk` inside a staged row: XOR with the row's low
// three bits so the 8 rows read by one ldmatrix phase hit distinct banks.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return static_cast<uint32_t>((chunk ^ (row & 7)) * 16);
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid) {
  const int n = valid ? 16 : 0;
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

template <int HD>
__global__ void __launch_bounds__(kAttnThreads, 3) attn_split_kernel(const AttnParams p) {
  using C = AttnCfg<HD>;
  extern __shared__ __align__(128) uint8_t smem[];
  griddep_wait();
  griddep_launch();
  const int s = blockIdx.x, g = blockIdx.y, i = blockIdx.z;
  const int grp = p.Hq / p.Hkv;
  const int nrows = grp * p.B;
  const int ctx = p.ctx_len[i];
  if (ctx < 0 || ctx > p.max_ctx || ctx > p.Cmax) {
    if (s == 0 && g == 0 && threadIdx.x == 0) flag_status(p.status, kStatusCheck);
  }
  const int ctx_used = max(0, min(ctx, min(p.max_ctx, p.Cmax)));
  const int nsplit = max(1, (ctx_used + p.chunk - 1) / p.chunk);
  if (s >= nsplit) return;
  const int key0 = s * p.chunk;
  const int key1 = min(ctx_used, key0 + p.chunk);
  const int nctx = max(0, key1 - key0);
  const int has_block = (s == 0) ? 1 : 0;
  const int nsub = has_block + (nctx + kSub - 1) / kSub;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ldq = (p.Hq + 2 * p.Hkv) * HD;
  const uint16_t *kbase = p.kc + (((size_t)i * p.Hkv + g) * p.Cmax) * HD;
  const uint16_t *vbase = p.vc + (((size_t)i * p.Hkv + g) * p.Cmax) * HD;
  const uint32_t sbase = smem_u32(smem);

  // Stage sub-chunk u into ring slot `slot`: K tile then V tile, rows of HD bf16.
  auto load_sub = [&](int u, int slot) {
    const uint32_t kdst = sbase + slot * 2 * C::TILE_BYTES;
    const uint32_t vdst = kdst + C::TILE_BYTES;
    constexpr int CHUNKS = HD / 8;  // 16-byte chunks per row
    for (int e = tid; e < kSub * CHUNKS; e += kAttnThreads) {
      const int row = e / CHUNKS, ch = e % CHUNKS;
      const uint16_t *ks;
      const uint16_t *vs;
      bool valid;
      if (has_block && u == 0) {
        valid = row < p.B;
        const size_t qrow = (size_t)i * p.B + (valid ? row : 0);
        ks = p.qkv + qrow * ldq + (size_t)(p.Hq + g) * HD + ch * 8;
        vs = p.qkv + qrow * ldq + (size_t)(p.Hq + p.Hkv + g) * HD + ch * 8;
      } else {
        const int key = key0 + (u - has_block) * kSub + row;
        valid = key < key1;
        const size_t kr = valid ? (size_t)key : 0;
        ks = kbase + kr * HD + ch * 8;
        vs = vbase + kr * HD + ch * 8;
      }
      const uint32_t off = row * C::ROW_BYTES + swz(row, ch);
      cp_async16(kdst + off, ks, valid);
      cp_async16(vdst + off, vs, valid);
    }
  };
  auto nvalid_of = [&](int u) -> int {
    if (has_block && u == 0) return p.B;
    return min(kSub, nctx - (u - has_block) * kSub);
  };

  // Query fragments (A operand of m16n8k16) for this warp's 16 rows.
  const int wrow0 = warp * 16;
  const bool active = wrow0 < nrows;
  uint32_t qf[HD / 16][4];
  {
    const int r0 = wrow0 + (lane >> 2), r1 = r0 + 8;
    const int c = (lane & 3) * 2;
    const uint32_t *q32[2] = {nullptr, nullptr};
    const int rr[2] = {r0, r1};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (rr[h] < nrows) {
        const int hh = rr[h] / p.B, j = rr[h] % p.B;
        q32[h] = reinterpret_cast<const uint32_t *>(p.qkv + ((size_t)i * p.B + j) * ldq +
                                                    (size_t)(g * grp + hh) * HD);
      }
    }
#pragma unroll
    for (int ks = 0; ks < HD / 16; ++ks) {
      const int col = ks * 16 + c;
      qf[ks][0] = q32[0] ? q32[0][col / 2] : 0u;
      qf[ks][1] = q32[1] ? q32[1][col / 2] : 0u;
      qf[ks][2] = q32[0] ? q32[0][(col + 8) / 2] : 0u;
      qf[ks][3] = q32[1] ? q32[1][(col + 8) / 2] : 0u;
    }
  }

  float o[HD / 8][4];
#pragma unroll
  for (int n = 0; n < HD / 8; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -FLT_MAX, m1 = -FLT_MAX, l0 = 0.f, l1 = 0.f;
  const float sl2 = rsqrtf(static_cast<float>(HD)) * 1.4426950408889634f;

  // prologue: fill STAGES-1 slots
#pragma unroll
  for (int u = 0; u < C::STAGES - 1; ++u) {
    if (u < nsub) load_sub(u, u);
    cp_async_commit();
  }

  for (int u = 0; u < nsub; ++u) {
    {
      const int un = u + C::STAGES - 1;
      if (un < nsub) load_sub(un, un % C::STAGES);
      cp_async_commit();
    }
    cp_async_wait<C::STAGES - 1>();
    __syncthreads();
    const int slot = u % C::STAGES;
    const uint32_t ksm = sbase + slot * 2 * C::TILE_BYTES;
    const uint32_t vsm = ksm + C::TILE_BYTES;
    const int nv = nvalid_of(u);
    if (active) {
      float sc[8][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) sc[n][0] = sc[n][1] = sc[n][2] = sc[n][3] = 0.f;
      const int mi = lane >> 3, rr = lane & 7;
#pragma unroll
      for (int ks = 0; ks < HD / 16; ++ks) {
#pragma unroll
        for (int ntp = 0; ntp < 4; ++ntp) {
          const int key = ntp * 16 + (mi >> 1) * 8 + rr;
          const int ch = ks * 2 + (mi & 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(ksm + key * C::ROW_BYTES + swz(key, ch), b0, b1, b2, b3);
          mma_bf16(sc[2 * ntp], qf[ks], b0, b1);
          mma_bf16(sc[2 * ntp + 1], qf[ks], b2, b3);
        }
      }
      // mask keys beyond the valid count, then online softmax update
      float mx0 = -FLT_MAX, mx1 = -FLT_MAX;
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int k0 = n * 8 + (lane & 3) * 2;
        if (k0 >= nv) sc[n][0] = sc[n][2] = -FLT_MAX;
        if (k0 + 1 >= nv) sc[n][1] = sc[n][3] = -FLT_MAX;
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
      }
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
      mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
      mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
      const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
      const float al0 = exp2f((m0 - mn0) * sl2), al1 = exp2f((m1 - mn1) * sl2);
      m0 = mn0;
      m1 = mn1;
      l0 *= al0;
      l1 *= al1;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
      uint32_t pa[4][4];
#pragma unroll
      for (int n = 0; n < 8; ++n) {
        const int k0 = n * 8 + (lane & 3) * 2;
        const float p0 = (k0 < nv) ? exp2f((sc[n][0] - mn0) * sl2) : 0.f;
        const float p1 = (k0 + 1 < nv) ? exp2f((sc[n][1] - mn0) * sl2) : 0.f;
        const float p2 = (k0 < nv) ? exp2f((sc[n][2] - mn1) * sl2) : 0.f;
        const float p3 = (k0 + 1 < nv) ? exp2f((sc[n][3] - mn1) * sl2) : 0.f;
        l0 += p0 + p1;
        l1 += p2 + p3;
        const int kk = n >> 1;
        if ((n & 1) == 0) {
          pa[kk][0] = pack_bf16x2(p0, p1);
          pa[kk][1] = pack_bf16x2(p2, p3);
        } else {
          pa[kk][2] = pack_bf16x2(p0, p1);
          pa[kk][3] = pack_bf16x2(p2, p3);
        }
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        if (kk * 16 >= nv) break;
#pragma unroll
        for (int ndp = 0; ndp < HD / 16; ++ndp) {
          const int key = kk * 16 + (mi & 1) * 8 + rr;
          const int ch = ndp * 2 + (mi >> 1);
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(vsm + key * C::ROW_BYTES + swz(key, ch), b0, b1, b2, b3);
          mma_bf16(o[2 * ndp], pa[kk], b0, b1);
          mma_bf16(o[2 * ndp + 1], pa[kk], b2, b3);
        }
      }
    }
    __syncthreads();
  }
  cp_async_wait<0>();

  if (active) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const size_t pbase = (((size_t)i * p.Hkv + g) * p.splits + s) * nrows;
    const int r0 = wrow0 + (lane >> 2), r1 = r0 + 8;
    const int c = (lane & 3) * 2;
    if (r0 < nrows) {
      float *dst = p.part_o + (pbase + r0) * HD;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n)
        *reinterpret_cast<float2 *>(dst + n * 8 + c) = make_float2(o[n][0], o[n][1]);
      if ((lane & 3) == 0) *reinterpret_cast<float2 *>(p.part_ml + (pbase + r0) * 2) = make_float2(m0, l0);
    }
    if (r1 < nrows) {
      float *dst = p.part_o + (pbase + r1) * HD;
#pragma unroll
      for (int n = 0; n < HD / 8; ++n)
        *reinterpret_cast<float2 *>(dst + n * 8 + c) = make_float2(o[n][2], o[n][3]);
      if ((lane & 3) == 0) *reinterpret_cast<float2 *>(p.part_ml + (pbase + r1) * 2) = make_float2(m1, l1);
    }
  }
}

// Combine the splits of one (sequence, kv head) in split order and write o (bf16).
// One warp per query row; each lane owns HD/32 consecutive output elements, so the
// partial rows are read with vector loads and the split weights are computed once
// per row.
constexpr int kMergeWarps = 8;

template <int HD>
__global__ void __launch_bounds__(kMergeWarps * 32) attn_merge_kernel(const AttnParams p) {
  constexpr int E = HD / 32;
  griddep_wait();
  griddep_launch();
  const int g = blockIdx.y, i = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int grp = p.Hq / p.Hkv;
  const int nrows = grp * p.B;
  const int t = blockIdx.x * kMergeWarps + warp;
  if (t >= nrows) return;
  const int ctx_used = max(0, min(p.ctx_len[i], min(p.max_ctx, p.Cmax)));
  const int nsplit = max(1, (ctx_used + p.chunk - 1) / p.chunk);
  const float sl2 = rsqrtf(static_cast<float>(HD)) * 1.4426950408889634f;
  const size_t pbase = ((size_t)i * p.Hkv + g) * p.splits * nrows + t;
  float M = -FLT_MAX;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p.part_ml[(pbase + (size_t)s * nrows) * 2]);
  float L = 0.f, acc[E];
#pragma unroll
  for (int e = 0; e < E; ++e) acc[e] = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const size_t r = pbase + (size_t)s * nrows;
    const float2 ml = *reinterpret_cast<const float2 *>(p.part_ml + r * 2);
    const float wgt = exp2f((ml.x - M) * sl2);
    L += ml.y * wgt;
    const float *src = p.part_o + r * HD + lane * E;
    if constexpr (E == 4) {
      const float4 v = *reinterpret_cast<const float4 *>(src);
      acc[0] += v.x * wgt;
      acc[1] += v.y * wgt;
      acc[2] += v.z * wgt;
      acc[3] += v.w * wgt;
    } else {
      const float2 v = *reinterpret_cast<const float2 *>(src);
      acc[0] += v.x * wgt;
      acc[1] += v.y * wgt;
    }
  }
  const float inv = 1.0f / L;
  const int hh = t / p.B, j = t % p.B;
  uint16_t *dst = p.o + ((size_t)i * p.B + j) * (p.Hq * HD) + (size_t)(g * grp + hh) * HD + lane * E;
  if constexpr (E == 4) {
    *reinterpret_cast<uint2 *>(dst) = make_uint2(pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                                 pack_bf16x2(acc[2] * inv, acc[3] * inv));
  } else {
    *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
  }
}

size_t attention_partial_bytes(int nb, int Hq, int Hkv, int hd, int B, int splits) {
  const size_t rows = (size_t)(Hq / Hkv) * B;
  return (size_t)nb * Hkv * splits * rows * ((size_t)hd + 2) * sizeof(float);
}

template <int HD>
static cudaError_t launch_attn_hd(const AttnParams &p, cudaStream_t s) {
  using C = AttnCfg<HD>;
  static bool configured = false;
  if (!configured) {
    cudaError_t e = cudaFuncSetAttribute(attn_split_kernel<HD>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)C::SMEM);
    if (e != cudaSuccess) return e;
    configured = true;
  }
  dim3 grid(p.splits, p.Hkv, p.nb);
  cudaError_t e = launch_pdl(attn_split_kernel<HD>, grid, dim3(kAttnThreads), C::SMEM, s, p);
  if (e != cudaSuccess) return e;
  const int nrows = (p.Hq / p.Hkv) * p.B;
  dim3 mgrid((nrows + kMergeWarps - 1) / kMergeWarps, p.Hkv, p.nb);
  return launch_pdl(attn_merge_kernel<HD>, mgrid, dim3(kMergeWarps * 32), 0, s, p);
}

cudaError_t launch_attention(const AttnParams &p, cudaStream_t s) {
  if (p.hd == 128) return launch_attn_hd<128>(p, s);
  if (p.hd == 64) return launch_attn_hd<64>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace df
