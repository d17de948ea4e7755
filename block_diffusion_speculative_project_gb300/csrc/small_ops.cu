// CUDA-core kernels of the draft step: embedding gather, RMSNorm, relay placement,
// FiLM relay rows, greedy accept, top-k merge, DFlash 2 conv application and selector walk.
// All are memory- or latency-bound row operations; each reads its inputs once with
// 16-byte vector accesses where the row layout allows.
#include <algorithm>
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace df {

__device__ __forceinline__ float bits_to_f32(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t f32_to_bits(float x) {
  __nv_bfloat16 b = __float2bfloat16_rn(x);
  return *reinterpret_cast<uint16_t *>(&b);
}

// Sum over a CTA of 256 threads.
__device__ __forceinline__ float block_sum_256(float v, float *red) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) red[w] = v;
  __syncthreads();
  float t = 0.f;
#pragma unroll
  for (int k = 0; k < 8; ++k) t += red[k];
  __syncthreads();
  return t;
}

// ---------------------------------------------------------------- RMSNorm
// y = g * x / sqrt(mean(x^2) + eps), fp32 statistics, bf16 output.
// Mode 0: x given (f32). Mode 1: x = E[ids[r]] (+ relay[r]) is built, stored to x,
// and normalised when g != nullptr.
template <int MODE>
__global__ void __launch_bounds__(256) rmsnorm_kernel(const float *xin, const int *ids,
                                                      const uint16_t *E, const uint16_t *relay,
                                                      float *xout, int D, const uint16_t *g,
                                                      float eps, uint16_t *u, int B, int skip,
                                                      int rows_out_per_seq, int V, int *status) {
  griddep_wait();
  griddep_launch();
  __shared__ float red[8];
  const int r = blockIdx.x;
  extern __shared__ float row[];  // D floats
  int id = 0;
  if (MODE == 1) {
    id = ids[r];
    if (id < 0 || id >= V) {
      if (threadIdx.x == 0) flag_status(status, kStatusCheck);
      id = 0;
    }
  }
  float ss = 0.f;
  // unrolled so that a thread's loads of the row (4 at D = 4096) are in flight together;
  // the squares are still summed in column order
#pragma unroll 4
  for (int c = threadIdx.x * 4; c < D; c += 256 * 4) {
    float4 v;
    if (MODE == 0) {
      v = *reinterpret_cast<const float4 *>(xin + (size_t)r * D + c);
    } else {
      const uint2 e = *reinterpret_cast<const uint2 *>(E + (size_t)id * D + c);
      v = make_float4(bits_to_f32(e.x & 0xFFFF), bits_to_f32(e.x >> 16), bits_to_f32(e.y & 0xFFFF),
                      bits_to_f32(e.y >> 16));
      if (relay) {
        const uint2 q = *reinterpret_cast<const uint2 *>(relay + (size_t)r * D + c);
        v.x += bits_to_f32(q.x & 0xFFFF);
        v.y += bits_to_f32(q.x >> 16);
        v.z += bits_to_f32(q.y & 0xFFFF);
        v.w += bits_to_f32(q.y >> 16);
      }
      *reinterpret_cast<float4 *>(xout + (size_t)r * D + c) = v;
    }
    *reinterpret_cast<float4 *>(row + c) = v;
    ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
  }
  if (g == nullptr) return;
  const float tot = block_sum_256(ss, red);
  const float inv = rsqrtf(tot / static_cast<float>(D) + eps);
  // optional row remap: skip the first `skip` rows of every block of B rows
  int orow = r;
  if (skip) {
    const int j = r % B;
    if (j < skip) return;
    orow = (r / B) * rows_out_per_seq + (j - skip);
  }
#pragma unroll 4
  for (int c = threadIdx.x * 4; c < D; c += 256 * 4) {
    const float4 v = *reinterpret_cast<const float4 *>(row + c);
    const uint2 gg = *reinterpret_cast<const uint2 *>(g + c);
    uint2 o;
    o.x = static_cast<uint32_t>(f32_to_bits(v.x * inv * bits_to_f32(gg.x & 0xFFFF))) |
          (static_cast<uint32_t>(f32_to_bits(v.y * inv * bits_to_f32(gg.x >> 16))) << 16);
    o.y = static_cast<uint32_t>(f32_to_bits(v.z * inv * bits_to_f32(gg.y & 0xFFFF))) |
          (static_cast<uint32_t>(f32_to_bits(v.w * inv * bits_to_f32(gg.y >> 16))) << 16);
    *reinterpret_cast<uint2 *>(u + (size_t)orow * D + c) = o;
  }
}

cudaError_t launch_embed_rmsnorm(const int *ids, const uint16_t *E, const uint16_t *relay, int M,
                                 int D, int V, float *x, const uint16_t *g, float eps, uint16_t *u,
                                 int *status, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(rmsnorm_kernel<1>, dim3(M), dim3(256), D * sizeof(float), s, nullptr, ids, E,
                             relay, x, D, g, eps, u, 1, 0, 0, V, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm(const float *x, int M, int D, const uint16_t *g, float eps, uint16_t *u,
                           cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(rmsnorm_kernel<0>, dim3(M), dim3(256), D * sizeof(float), s, x, nullptr,
                             nullptr, nullptr, nullptr, D, g, eps, u, 1, 0, 0, 0, nullptr);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_rows(const float *x, int M, int D, const uint16_t *g, float eps,
                                uint16_t *u, int B, int skip_first, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(rmsnorm_kernel<0>, dim3(M), dim3(256), D * sizeof(float), s, x, nullptr,
                             nullptr, nullptr, nullptr, D, g, eps, u, B, skip_first, B - skip_first, 0,
                             nullptr);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- relay placement
// x0_relay[i, j] = h[i*R + j + a] for j in [2, B-1-a] (j + a < R), else 0;
// then ctx_len[i] += n_commit[i].
__global__ void __launch_bounds__(256) relay_len_kernel(const uint16_t *h, int R, int B, int D,
                                                        const int *relay_a, const int *n_commit,
                                                        int *ctx_len, uint16_t *x0, int Cmax,
                                                        int *status) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x, j = blockIdx.y;  // sequence, block offset (one row per CTA)
  if (x0) {
    const int a = relay_a ? relay_a[i] : INT_MAX / 2;
    const int k = j + a;
    const bool take = relay_a && j >= 2 && j <= B - 1 - a && k < R && a >= 0;
    uint4 *dst = reinterpret_cast<uint4 *>(x0 + ((size_t)i * B + j) * D);
    const uint4 *src = take ? reinterpret_cast<const uint4 *>(h + ((size_t)i * R + k) * D) : nullptr;
    for (int c = threadIdx.x; c < D / 8; c += 256) dst[c] = take ? src[c] : make_uint4(0, 0, 0, 0);
  }
  if (j == 0 && threadIdx.x == 0 && n_commit) {
    const int nl = ctx_len[i] + n_commit[i];
    if (nl > Cmax || n_commit[i] < 0 || n_commit[i] > R) flag_status(status, kStatusCheck);
    ctx_len[i] = min(nl, Cmax);
  }
}

cudaError_t launch_relay_and_len(const uint16_t *h, int nb, int R, int B, int D,
                                 const int *relay_a, const int *n_commit, int *ctx_len,
                                 uint16_t *x0_relay, int Cmax, int *status, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(relay_len_kernel, dim3(nb, x0_relay ? B : 1), dim3(256), 0, s, h, R, B, D, relay_a,
                             n_commit, ctx_len, x0_relay, Cmax, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- FiLM relay
// [DFlow] 第三步. One CTA per block offset r = i*B + j of the next block. Offset j of
// sequence i is relayed from previous row k = j + a_i when 2 <= j <= B-1-a_i and k < R
// (the same placement as the plain relay).
__device__ __forceinline__ bool film_relayed(const int *relay_a, int r, int B, int R, int &i,
                                             int &k) {
  i = r / B;
  const int j = r - i * B;
  const int a = relay_a[i];
  k = j + a;
  return a >= 0 && j >= 2 && j <= B - 1 - a && k < R;
}

// cond[r] = [E[b_i]; E[y_i]; h[i*R + k]] (bf16, 3D wide), zeros for offsets not relayed.
__global__ void __launch_bounds__(256) film_cond_kernel(const uint16_t *h, const uint16_t *E, int R,
                                                        int B, int D, int V, const int *relay_a,
                                                        const int *relay_b, const int *relay_y,
                                                        uint16_t *cond, int *status) {
  griddep_wait();
  griddep_launch();
  const int r = blockIdx.x;
  int i, k;
  const bool take = film_relayed(relay_a, r, B, R, i, k);
  const int n8 = D / 8;
  uint4 *dst = reinterpret_cast<uint4 *>(cond + (size_t)r * 3 * D);
  const uint4 zero = make_uint4(0, 0, 0, 0);
  if (!take) {
    for (int c = threadIdx.x; c < 3 * n8; c += 256) dst[c] = zero;
    return;
  }
  const int b = relay_b[i];
  const int y = relay_y[i];
  const bool bok = b >= 0 && b < V;
  const bool yok = y >= 0 && y < V;
  if (threadIdx.x == 0 && !(bok && yok)) flag_status(status, kStatusCheck);
  const uint4 *eb = reinterpret_cast<const uint4 *>(E + (size_t)(bok ? b : 0) * D);
  const uint4 *ey = reinterpret_cast<const uint4 *>(E + (size_t)(yok ? y : 0) * D);
  const uint4 *hk = reinterpret_cast<const uint4 *>(h + ((size_t)i * R + k) * D);
  for (int c = threadIdx.x; c < n8; c += 256) {
    dst[c] = bok ? eb[c] : zero;
    dst[n8 + c] = yok ? ey[c] : zero;
    dst[2 * n8 + c] = hk[c];
  }
}

// x0[r] = bf16(beta * (h_k - mean) / sqrt(var + eps) + gamma), beta = bg[r][0..D),
// gamma = bg[r][D..2D); zeros for offsets not relayed. Two-pass fp32 statistics.
__global__ void __launch_bounds__(256) film_apply_kernel(const uint16_t *h, const float *bg, int R,
                                                         int B, int D, const int *relay_a, float eps,
                                                         uint16_t *x0) {
  griddep_wait();
  griddep_launch();
  __shared__ float red[8];
  const int r = blockIdx.x;
  int i, k;
  const bool take = film_relayed(relay_a, r, B, R, i, k);
  uint4 *dst = reinterpret_cast<uint4 *>(x0 + (size_t)r * D);
  const int n8 = D / 8;
  if (!take) {
    for (int c = threadIdx.x; c < n8; c += 256) dst[c] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4 *hk = reinterpret_cast<const uint4 *>(h + ((size_t)i * R + k) * D);
  float s = 0.f;
  for (int c = threadIdx.x; c < n8; c += 256) {
    const uint4 v = hk[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q)
      s += bits_to_f32(uint16_t(w[q] & 0xFFFFu)) + bits_to_f32(uint16_t(w[q] >> 16));
  }
  const float mean = block_sum_256(s, red) / D;
  float ss = 0.f;
  for (int c = threadIdx.x; c < n8; c += 256) {
    const uint4 v = hk[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float d0 = bits_to_f32(uint16_t(w[q] & 0xFFFFu)) - mean;
      const float d1 = bits_to_f32(uint16_t(w[q] >> 16)) - mean;
      ss += d0 * d0 + d1 * d1;
    }
  }
  const float rstd = rsqrtf(block_sum_256(ss, red) / D + eps);
  const float *beta = bg + (size_t)r * 2 * D;
  const float *gamma = beta + D;
  for (int c = threadIdx.x; c < n8; c += 256) {
    const uint4 v = hk[c];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    const float4 b0 = reinterpret_cast<const float4 *>(beta)[2 * c];
    const float4 b1 = reinterpret_cast<const float4 *>(beta)[2 * c + 1];
    const float4 g0 = reinterpret_cast<const float4 *>(gamma)[2 * c];
    const float4 g1 = reinterpret_cast<const float4 *>(gamma)[2 * c + 1];
    const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
    const float gg[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
    uint32_t o[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float n0 = (bits_to_f32(uint16_t(w[q] & 0xFFFFu)) - mean) * rstd;
      const float n1 = (bits_to_f32(uint16_t(w[q] >> 16)) - mean) * rstd;
      o[q] = pack_bf16x2(bb[2 * q] * n0 + gg[2 * q], bb[2 * q + 1] * n1 + gg[2 * q + 1]);
    }
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

cudaError_t launch_film_cond(const uint16_t *h, const uint16_t *E, int nb, int R, int B, int D,
                             int V, const int *relay_a, const int *relay_b, const int *relay_y,
                             uint16_t *cond, int *status, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(film_cond_kernel, dim3(nb * B), dim3(256), 0, s, h, E, R, B, D, V,
                             relay_a, relay_b, relay_y, cond, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_film_apply(const uint16_t *h, const float *bg, int nb, int R, int B, int D,
                              const int *relay_a, float eps, uint16_t *x0, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(film_apply_kernel, dim3(nb * B), dim3(256), 0, s, h, bg, R, B, D,
                             relay_a, eps, x0);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- accept
__global__ void accept_kernel(const int *draft, int draft_stride, const int *target, int nb, int B,
                              int *tau, int *bonus) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nb) return;
  const int *d = draft + (size_t)i * (B - 1) * draft_stride;
  const int *t = target + (size_t)i * B;
  // every load first (in flight together), then the longest matching prefix by compares
  // and selects: a loop that loads as it compares pays one memory round trip per position
  int dv[kMaxBlock], tv[kMaxBlock];
#pragma unroll
  for (int j = 0; j < kMaxBlock; ++j) {
    dv[j] = j < B - 1 ? d[(size_t)j * draft_stride] : 0;
    tv[j] = j < B ? t[j] : 0;
  }
  int n = 0;
  bool run = true;
#pragma unroll
  for (int j = 0; j < kMaxBlock - 1; ++j) {
    run = run & (j < B - 1) & (dv[j] == tv[j]);
    n += run ? 1 : 0;
  }
  int b = tv[0];
#pragma unroll
  for (int j = 1; j < kMaxBlock; ++j) b = j == n ? tv[j] : b;
  tau[i] = n + 1;
  bonus[i] = b;
}

cudaError_t launch_accept(const int *draft, int draft_stride, const int *target, int nb, int B, int *tau,
                          int *bonus, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(accept_kernel, dim3((nb + 127) / 128), dim3(128), 0, s, draft, draft_stride, target,
                             nb, B, tau, bonus);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- top-k merge
// One CTA (8 warps) per row. Candidate c of part q of row r:
// vals[q*part_stride + r*row_stride + c] (ids from `ids` at the same index, or c itself
// when ids == nullptr). Each thread keeps a sorted top-16 of its strided candidates;
// each warp merges its 32 lists with shuffle-only arg-best rounds; warp 0 merges the
// 8 warp lists the same way. Order: value descending, ties to the lower id.
__device__ __forceinline__ void warp_pop_best(float &hv, int &hi, int lane, float &best_v,
                                              int &best_i, int &best_lane) {
  best_v = hv;
  best_i = hi;
  best_lane = lane;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, best_v, o);
    const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
    const int ol = __shfl_xor_sync(0xffffffffu, best_lane, o);
    if (topk_before(ov, oi, best_v, best_i) || (ov == best_v && oi == best_i && ol < best_lane)) {
      best_v = ov;
      best_i = oi;
      best_lane = ol;
    }
  }
}

__global__ void __launch_bounds__(256) topk_merge_kernel(const float *vals, const int *ids,
                                                         int ncand, long long row_stride,
                                                         long long part_stride, int parts, int k,
                                                         int *out_ids, float *out_vals) {
  griddep_wait();
  griddep_launch();
  __shared__ float sv[256 * kTopkMax];
  __shared__ int si[256 * kTopkMax];
  __shared__ float wv[8 * kTopkMax];
  __shared__ int wi[8 * kTopkMax];
  const int r = blockIdx.x;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float kv[kTopkMax];
  int ki[kTopkMax];
#pragma unroll
  for (int s = 0; s < kTopkMax; ++s) {
    kv[s] = -FLT_MAX;
    ki[s] = INT_MAX;
  }
  const long long total = (long long)parts * ncand;
  for (long long e = threadIdx.x; e < total; e += 256) {
    const int q = static_cast<int>(e / ncand), c = static_cast<int>(e % ncand);
    const long long idx = (long long)q * part_stride + (long long)r * row_stride + c;
    const float v = vals[idx];
    const int id = ids ? ids[idx] : c;
    if (!topk_before(v, id, kv[kTopkMax - 1], ki[kTopkMax - 1])) continue;
    float cv = v;
    int ci = id;
#pragma unroll
    for (int s = 0; s < kTopkMax; ++s) {
      if (topk_before(cv, ci, kv[s], ki[s])) {
        const float tv = kv[s];
        const int ti = ki[s];
        kv[s] = cv;
        ki[s] = ci;
        cv = tv;
        ci = ti;
      }
    }
  }
#pragma unroll
  for (int s = 0; s < kTopkMax; ++s) {
    sv[threadIdx.x * kTopkMax + s] = kv[s];
    si[threadIdx.x * kTopkMax + s] = ki[s];
  }
  __syncwarp();
  // warp level: pop the best head of the 32 lane lists k times
  {
    int head = 0;
    for (int round = 0; round < k; ++round) {
      float hv = head < kTopkMax ? sv[threadIdx.x * kTopkMax + head] : -FLT_MAX;
      int hi = head < kTopkMax ? si[threadIdx.x * kTopkMax + head] : INT_MAX;
      float bv;
      int bi, bl;
      warp_pop_best(hv, hi, lane, bv, bi, bl);
      if (lane == 0) {
        wv[warp * kTopkMax + round] = bv;
        wi[warp * kTopkMax + round] = bi;
      }
      if (lane == bl) ++head;
    }
  }
  __syncthreads();
  if (warp == 0) {
    int head = 0;
    const int src = lane < 8 ? lane : -1;
    for (int round = 0; round < k; ++round) {
      float hv = (src >= 0 && head < k) ? wv[src * kTopkMax + head] : -FLT_MAX;
      int hi = (src >= 0 && head < k) ? wi[src * kTopkMax + head] : INT_MAX;
      float bv;
      int bi, bl;
      warp_pop_best(hv, hi, lane, bv, bi, bl);
      if (lane == 0) {
        out_vals[(size_t)r * k + round] = bv;
        out_ids[(size_t)r * k + round] = bi;
      }
      if (lane == bl) ++head;
    }
  }
}

// Merge of sorted per-part lists (the LM head's per-range top-k lists, parts <= 1024,
// k <= 16): one CTA of 1024 threads per row. A candidate below the k-th best list head
// cannot be in the top k (the k best heads already beat it), so (1) the k-th best head is
// found by rank counting among the heads, (2) every candidate at or above it survives -
// at most k lists x k entries - and (3) the survivors are placed by rank counting. All
// comparisons use the strict order (value descending, then id ascending).
constexpr int kHeadsThreads = 1024;
constexpr int kHeadsMaxSurv = kTopkMax * kTopkMax;

__global__ void __launch_bounds__(kHeadsThreads) topk_merge_heads_kernel(
    const float *vals, const int *ids, int ncand, long long row_stride, long long part_stride, int parts,
    int k, int *out_ids, float *out_vals) {
  griddep_wait();
  griddep_launch();
  __shared__ float hv[kHeadsThreads];
  __shared__ int hi[kHeadsThreads];
  __shared__ float sv[kHeadsMaxSurv];
  __shared__ int si[kHeadsMaxSurv];
  __shared__ float thr_v;
  __shared__ int thr_i, nsurv;
  const int r = blockIdx.x, t = threadIdx.x;
  const long long rowbase = (long long)r * row_stride;
  if (t == 0) {
    thr_v = -FLT_MAX;
    thr_i = INT_MAX;
    nsurv = 0;
  }
  if (t < parts) {
    hv[t] = vals[(long long)t * part_stride + rowbase];
    hi[t] = ids[(long long)t * part_stride + rowbase];
  }
  __syncthreads();
  // (1) the k-th best head (when there are fewer than k lists every candidate survives).
  // Ranks are counted by `sub` adjacent lanes per entry (each taking every sub-th entry),
  // summed by shuffles: the counting loops are short and unrolled (a lone warp pays tens
  // of cycles per taken branch).
  const int sub1 = parts * 4 <= kHeadsThreads ? 4 : parts * 2 <= kHeadsThreads ? 2 : 1;
  if (parts >= k) {
    const int h = t / sub1, part = t % sub1;
    const bool live = h < parts;
    const float v = live ? hv[h] : 0.f;
    const int id = live ? hi[h] : 0;
    int rank = 0;
    if (live) {
#pragma unroll 8
      for (int q = part; q < parts; q += sub1) rank += topk_before(hv[q], hi[q], v, id) ? 1 : 0;
    }
    for (int o = 1; o < sub1; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (live && part == 0 && rank == k - 1) {
      thr_v = v;
      thr_i = id;
    }
  }
  __syncthreads();
  // (2) survivors: candidates not after the threshold
  const float tv = thr_v;
  const int ti = thr_i;
  const int total = parts * ncand;
  for (int e = t; e < total; e += kHeadsThreads) {
    const int part = e / ncand, c = e % ncand;
    const long long idx = (long long)part * part_stride + rowbase + c;
    const float v = vals[idx];
    const int id = ids[idx];
    if (!topk_before(tv, ti, v, id)) {
      const int slot = atomicAdd(&nsurv, 1);
      if (slot < kHeadsMaxSurv) {
        sv[slot] = v;
        si[slot] = id;
      }
    }
  }
  __syncthreads();
  // (3) place the survivors by rank (counted as in (1))
  const int ns = min(nsurv, kHeadsMaxSurv);
  const int sub3 = ns * 4 <= kHeadsThreads ? 4 : ns * 2 <= kHeadsThreads ? 2 : 1;
  {
    const int h = t / sub3, part = t % sub3;
    const bool live = h < ns;
    const float v = live ? sv[h] : 0.f;
    const int id = live ? si[h] : 0;
    int rank = 0;
    if (live) {
#pragma unroll 8
      for (int q = part; q < ns; q += sub3) rank += topk_before(sv[q], si[q], v, id) ? 1 : 0;
    }
    for (int o = 1; o < sub3; o <<= 1) rank += __shfl_xor_sync(0xffffffffu, rank, o);
    if (live && part == 0 && rank < k) {
      out_vals[(size_t)r * k + rank] = v;
      out_ids[(size_t)r * k + rank] = id;
    }
  }
}

cudaError_t launch_topk_merge(const float *vals, const int *ids, int rows, int ncand_per_row,
                              long long row_stride, long long part_stride, int parts, int k,
                              int *out_ids, float *out_vals, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e;
  if (ids && parts > 1 && parts <= kHeadsThreads && ncand_per_row == k && k <= kTopkMax)
    e = launch_pdl(topk_merge_heads_kernel, dim3(rows), dim3(kHeadsThreads), 0, s, vals, ids, ncand_per_row,
                   row_stride, part_stride, parts, k, out_ids, out_vals);
  else
    e = launch_pdl(topk_merge_kernel, dim3(rows), dim3(256), 0, s, vals, ids, ncand_per_row, row_stride,
                   part_stride, parts, k, out_ids, out_vals);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- misc
__global__ void f32_to_bf16_kernel(const float *x, uint16_t *y, long long n) {
  griddep_wait();
  griddep_launch();
  for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
       e += (long long)gridDim.x * blockDim.x)
    y[e] = f32_to_bits(x[e]);
}

cudaError_t launch_f32_to_bf16(const float *x, uint16_t *y, long long n, cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  const int blocks = static_cast<int>(std::min<long long>((n + 255) / 256, 152 * 16));
  cudaError_t e = launch_pdl(f32_to_bf16_kernel, dim3(blocks), dim3(256), 0, s, x, y, n);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Two-tap conv apply, in place on x [M, D] (blocks of B rows):
// x'[t] = (b0 + c0[t][ch/group]) * x[t] + (b1 + c1[t][ch/group]) * x[t-1], x[-1] = 0.
// corr [M, 2*D/group] holds c0 in columns [0, D/group) and c1 after them.
// Rows are visited from last to first so x[t-1] is read before it is overwritten.
// Also writes bf16(x') into xb_out (when set): the input of the next conv's GEMM.
__global__ void conv_apply_kernel(float *x, uint16_t *xb_out, const float *corr, const uint16_t *base, int D,
                                  int B, int group) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x;
  const int ch = blockIdx.y * blockDim.x + threadIdx.x;
  if (ch >= D) return;
  const int ng = D / group;
  const float b0 = bits_to_f32(base[ch]), b1 = bits_to_f32(base[D + ch]);
  float *xb = x + (size_t)i * B * D;
  uint16_t *ob = xb_out ? xb_out + (size_t)i * B * D : nullptr;
  const float *cb = corr + (size_t)i * B * 2 * ng + ch / group;
  // every row of this channel and its two corrections are loaded before any is written
  // (independent loads in flight together); x_{t-1} is the old row t-1, x_{-1} = 0
  float xv[kMaxBlock], k0[kMaxBlock], k1[kMaxBlock];
#pragma unroll
  for (int t = 0; t < kMaxBlock; ++t) {
    if (t < B) {
      xv[t] = xb[(size_t)t * D + ch];
      k0[t] = b0 + cb[(size_t)t * 2 * ng];
      k1[t] = b1 + cb[(size_t)t * 2 * ng + ng];
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxBlock; ++t) {
    if (t < B) {
      const float y = k0[t] * xv[t] + k1[t] * (t > 0 ? xv[t - 1] : 0.f);
      xb[(size_t)t * D + ch] = y;
      if (ob) ob[(size_t)t * D + ch] = f32_to_bits(y);
    }
  }
}

cudaError_t launch_conv_apply(float *x, uint16_t *xb_out, const float *corr, const uint16_t *base, int M, int D,
                              int B, int group, cudaStream_t s) {
  if (M <= 0) return cudaSuccess;
  if (B > kMaxBlock) return cudaErrorInvalidValue;
  dim3 grid(M / B, (D + 255) / 256);
  cudaError_t e = launch_pdl(conv_apply_kernel, grid, dim3(256), 0, s, x, xb_out, corr, base, D, B, group);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Row r of sequence i = r / per, e = r % per: the anchor (e == 0) or candidate e-1.
__global__ void gather_select_kernel(const int *block_ids, const int *cand_ids, int B, int k,
                                     const uint16_t *E, int D, int V, uint16_t *out, int *status) {
  griddep_wait();
  griddep_launch();
  const int r = blockIdx.x;
  const int per = 1 + (B - 1) * k;
  const int i = r / per, e = r % per;
  int id = e == 0 ? block_ids[(size_t)i * B] : cand_ids[(size_t)i * (B - 1) * k + (e - 1)];
  if (id < 0 || id >= V) {
    if (threadIdx.x == 0) flag_status(status, kStatusCheck);
    id = 0;
  }
  const uint4 *src = reinterpret_cast<const uint4 *>(E + (size_t)id * D);
  uint4 *dst = reinterpret_cast<uint4 *>(out + (size_t)r * D);
  for (int c = threadIdx.x; c < D / 8; c += blockDim.x) dst[c] = src[c];
}

cudaError_t launch_gather_select(const int *block_ids, const int *cand_ids, int nb, int B, int k,
                                 const uint16_t *E, int D, int V, uint16_t *out, int *status,
                                 cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(gather_select_kernel, dim3(nb * (1 + (B - 1) * k)), dim3(128), 0, s,
                             block_ids, cand_ids, B, k, E, D, V, out, status);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Selector walk, one CTA per sequence. AB [rows, 2*sel]: A | B projections of the
// gathered tokens; per sequence the rows are [anchor, then candidate (t, c) for
// t = 1..B-1, c = 0..k-1]. G [nb*(B-1), sel]: W_G z_t before the sigmoid.
// The scores of every step do not depend on the walk: for each offset t and each
// possible previous choice a (the anchor at t = 1, one of the k candidates of t - 1
// after that), S_t(a, b) = U_t(b) + sum_d A(a)_d G_t,d B(b)_d for the k candidates b of t.
// select_table_kernel computes all of them at once (one CTA per (t, sequence), one thread
// per (a, b)); select_walk_kernel then walks each sequence's table in shared memory:
// a_t = argmax_b S_t(a_{t-1}, b), ties to the lower id.
__global__ void __launch_bounds__(256) select_table_kernel(const float *cand_vals, const float *AB,
                                                           const float *G, int B, int k, int sel,
                                                           float *table) {
  griddep_wait();
  griddep_launch();
  // shared memory: the gate (sel), then the A rows of the previous offset's candidates and
  // the B rows of this offset's candidates, each row padded to sel + 1 floats so that the
  // 16 candidate rows a warp reads at once fall in distinct banks
  extern __shared__ float sm[];
  const int t = blockIdx.x + 1, i = blockIdx.y;
  const int ld = sel + 1;
  float *gate = sm;
  float *As = sm + sel;
  float *Bs = As + k * ld;
  const float *Gt = G + ((size_t)i * (B - 1) + (t - 1)) * sel;
  const int per = 1 + (B - 1) * k;
  const float *ABi = AB + (size_t)i * per * 2 * sel;
  const int na = t == 1 ? 1 : k;  // offset 1 starts from the anchor (row 0)
  for (int d = threadIdx.x; d < sel; d += blockDim.x) gate[d] = 1.0f / (1.0f + expf(-Gt[d]));
  for (int e = threadIdx.x; e < k * sel; e += blockDim.x) {
    const int b = e / sel, d = e - b * sel;
    Bs[b * ld + d] = ABi[(size_t)(1 + (t - 1) * k + b) * 2 * sel + sel + d];
  }
  __syncthreads();
  // the A rows are stored already multiplied by the gate (the same rounded products the
  // dot products below would form), so the inner loop reads two operands, not three
  for (int e = threadIdx.x; e < na * sel; e += blockDim.x) {
    const int a = e / sel, d = e - a * sel;
    const int arow = t == 1 ? 0 : 1 + (t - 2) * k + a;
    As[a * ld + d] = ABi[(size_t)arow * 2 * sel + d] * gate[d];
  }
  __syncthreads();
  const int ai = threadIdx.x >> 4, b = threadIdx.x & 15;
  if (b >= k || ai >= na) return;
  const float *ar = As + ai * ld, *br = Bs + b * ld;
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 4
  for (int d = 0; d < sel; ++d) acc[d & 3] = fmaf(ar[d], br[d], acc[d & 3]);
  const size_t tr = (size_t)i * (B - 1) + (t - 1);
  table[(tr * k + ai) * k + b] = cand_vals[tr * k + b] + ((acc[0] + acc[1]) + (acc[2] + acc[3]));
}

__global__ void __launch_bounds__(256) select_walk_kernel(const int *cand_ids, const float *table, int B,
                                                          int k, int *path) {
  griddep_wait();
  griddep_launch();
  extern __shared__ float tab[];  // [B-1][k][k] scores, then [B-1][k] candidate ids
  const int i = blockIdx.x;
  const int n = (B - 1) * k * k;
  int *sid = reinterpret_cast<int *>(tab + n);
  const float *ti = table + (size_t)i * n;
  for (int e = threadIdx.x; e < n; e += blockDim.x) tab[e] = ti[e];
  for (int e = threadIdx.x; e < (B - 1) * k; e += blockDim.x) sid[e] = cand_ids[(size_t)i * (B - 1) * k + e];
  __syncthreads();
  // Warp 0 walks: lane c holds candidate c of the offset, and a butterfly of shuffles finds
  // the first candidate by (score descending, id ascending), the one a scan over c keeping
  // the best would find: the ids of one offset are distinct, so that order is strict. A NaN
  // score would make the scan depend on its order; an offset holding one is scanned by
  // lane 0 instead.
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int ai = 0;
  for (int t = 1; t < B; ++t) {
    const float *row = tab + ((t - 1) * k + ai) * k;
    const int *ids = sid + (t - 1) * k;
    const bool on = lane < k;
    const float v = on ? row[lane] : -INFINITY;
    const int id = on ? ids[lane] : INT_MAX;
    int best;
    if (__any_sync(0xffffffffu, on && isnan(v))) {
      best = 0;
      if (lane == 0)
        for (int c = 1; c < k; ++c)
          if (topk_before(row[c], ids[c], row[best], ids[best])) best = c;
      best = __shfl_sync(0xffffffffu, best, 0);
    } else {
      float bv = v;
      int bi = id, bs = lane;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float v2 = __shfl_xor_sync(0xffffffffu, bv, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
        const int s2 = __shfl_xor_sync(0xffffffffu, bs, o);
        const bool take = topk_before(v2, i2, bv, bi);
        bv = take ? v2 : bv;
        bi = take ? i2 : bi;
        bs = take ? s2 : bs;
      }
      best = bs;
    }
    if (lane == 0) path[(size_t)i * (B - 1) + (t - 1)] = ids[best];
    ai = best;
  }
}

cudaError_t launch_select_table(const float *cand_vals, const float *AB, const float *G, float *table,
                                int nb, int B, int k, int sel_dim, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  if (k > 16 || sel_dim % 4 || B < 2) return cudaErrorInvalidValue;
  const size_t smem = ((size_t)sel_dim + 2 * (size_t)k * (sel_dim + 1)) * sizeof(float);
  static size_t opted = 48 * 1024;  // dynamic shared memory the kernel is configured for
  if (smem > opted) {
    cudaError_t a = cudaFuncSetAttribute(select_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (a != cudaSuccess) return a;
    opted = smem;
  }
  cudaError_t e = launch_pdl(select_table_kernel, dim3(B - 1, nb), dim3(256), smem, s, cand_vals, AB, G, B, k,
                             sel_dim, table);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ---------------------------------------------------------------- Recall@k
// One thread per block: offsets t = 1.. while the target token T[t-1] is among the k
// candidates of offset t: eligible[t-1] and hits[t-1] count it; the first miss is counted
// as eligible only and ends the block.
__global__ void recall_at_k_kernel(const int *cand_ids, const int *target, int nb, int B, int k,
                                   int *hits, int *eligible) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nb) return;
  for (int t = 0; t < B - 1; ++t) {
    atomicAdd(&eligible[t], 1);
    const int want = target[(size_t)i * B + t];
    const int *c = cand_ids + ((size_t)i * (B - 1) + t) * k;
    bool hit = false;
    for (int q = 0; q < k; ++q) hit |= c[q] == want;
    if (!hit) break;
    atomicAdd(&hits[t], 1);
  }
}

cudaError_t launch_recall_at_k(const int *cand_ids, const int *target, int nb, int B, int k, int *hits,
                               int *eligible, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(recall_at_k_kernel, dim3((nb + 127) / 128), dim3(128), 0, s, cand_ids, target, nb,
                             B, k, hits, eligible);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_select_walk(const int *cand_ids, const float *cand_vals, const float *AB,
                               const float *G, float *table, int nb, int B, int k, int sel_dim, int *path,
                               cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  if (k > 16 || sel_dim % 4 || B < 2) return cudaErrorInvalidValue;
  const size_t smem = ((size_t)sel_dim + 2 * (size_t)k * (sel_dim + 1)) * sizeof(float);
  static size_t opted = 48 * 1024;  // dynamic shared memory the kernel is configured for
  if (smem > opted) {
    cudaError_t a = cudaFuncSetAttribute(select_table_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (a != cudaSuccess) return a;
    opted = smem;
  }
  cudaError_t e = launch_pdl(select_table_kernel, dim3(B - 1, nb), dim3(256), smem, s, cand_vals, AB, G, B, k,
                             sel_dim, table);
  if (e != cudaSuccess) return e;
  e = launch_pdl(select_walk_kernel, dim3(nb), dim3(256), (size_t)(B - 1) * k * (k + 1) * sizeof(float), s, cand_ids,
                 static_cast<const float *>(table), B, k, path);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
