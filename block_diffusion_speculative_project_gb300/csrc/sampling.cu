// Sampling at temperature T: draft candidates drawn from softmax(U_t / T) and the
// lossless rejection-sampling verify of a drafted block ("DFlash 2：正确 token 已在候选里",
// 洞察一 and Results: sampling at T = 1 with lossless rejection sampling; "DFlash 投机解码",
// 四、推理流程 dflash_cycle step ④: the rejected position is re-drawn from the target).
//
// Every random number comes from Philox4x32-10 (Salmon et al., "Parallel random numbers:
// as easy as 1, 2, 3", SC 2011) keyed by the 64-bit seed: element v of (stream, row) is
// word v % 4 of the block at counter (v / 4, row, stream, 0), and u = ((w >> 9) + 1/2) / 2^23,
// which fp32 holds exactly. Gumbel-max: a draw from softmax(x) is argmax_v x_v - log(-log u_v),
// ties to the lower id.
//
// All kernels are HBM-bound passes over fp32 logit rows: a row is split into S slices, one
// CTA per (slice, row); each keeps a running (max, sum of exp) and the best Gumbel score of
// its slice, and a merge combines the slices.
#include <cfloat>
#include <climits>

#include "common.cuh"
#include "kernels.h"

namespace df {

namespace {

constexpr uint32_t kPhiloxM0 = 0xD2511F53u;
constexpr uint32_t kPhiloxM1 = 0xCD9E8D57u;
constexpr uint32_t kPhiloxW0 = 0x9E3779B9u;
constexpr uint32_t kPhiloxW1 = 0xBB67AE85u;

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint32_t k0, uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += kPhiloxW0;
      k1 += kPhiloxW1;
    }
    const uint32_t hi0 = __umulhi(kPhiloxM0, c.x), lo0 = kPhiloxM0 * c.x;
    const uint32_t hi1 = __umulhi(kPhiloxM1, c.z), lo1 = kPhiloxM1 * c.z;
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
  }
  return c;
}

__device__ __forceinline__ float philox_u(uint32_t w) {
  return (static_cast<float>(w >> 9) + 0.5f) * 1.1920928955078125e-07f;  // 2^-23
}

// Gumbel value of one uniform; logf (not the fast approximation): the largest scores come
// from u close to 1, where log u is tiny and needs full relative precision.
__device__ __forceinline__ float gumbel_of(float u) { return -logf(-logf(u)); }

// Uniform of element v of (stream, row).
__device__ __forceinline__ float philox_uniform(unsigned long long seed, int stream, int row, int v) {
  const uint4 w = philox4x32_10(make_uint4((uint32_t)(v >> 2), (uint32_t)row, (uint32_t)stream, 0u),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  const int q = v & 3;
  return philox_u(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
}

struct Best {
  float v;
  int id;
};

__device__ __forceinline__ void best_take(Best &b, float v, int id) {
  if (v > b.v || (v == b.v && id < b.id)) {
    b.v = v;
    b.id = id;
  }
}

// Online log-sum-exp state: sum of exp(x - m).
__device__ __forceinline__ void lse_add(float &m, float &s, float x) {
  if (x == -INFINITY) return;  // probability 0
  if (x > m) {
    s = s * __expf(m - x) + 1.f;
    m = x;
  } else {
    s += __expf(x - m);
  }
}

__device__ __forceinline__ void lse_merge(float &m, float &s, float m2, float s2) {
  if (m2 == -INFINITY) return;
  if (m2 > m) {
    s = s * __expf(m - m2) + s2;
    m = m2;
  } else {
    s += s2 * __expf(m2 - m);
  }
}

// CTA-wide reduction (256 threads) of (m, s, best); result valid in thread 0.
__device__ __forceinline__ void cta_reduce(float &m, float &s, Best &b) {
  __shared__ float rm[8], rs[8], rb[8];
  __shared__ int ri[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float b2 = __shfl_xor_sync(0xffffffffu, b.v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, b.id, o);
    lse_merge(m, s, m2, s2);
    best_take(b, b2, i2);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    rm[w] = m;
    rs[w] = s;
    rb[w] = b.v;
    ri[w] = b.id;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < 8; ++k) {
      lse_merge(m, s, rm[k], rs[k]);
      best_take(b, rb[k], ri[k]);
    }
  }
}

}  // namespace

// Partial statistics of row r, slice s: part[r * S + s] = {max, sum exp(x - max), best
// Gumbel score, best id} over x = logits[r * ld + v] * inv_T, v in the slice. With
// stream < 0 no Gumbel score is formed (best = -inf, id = INT_MAX).
__global__ void __launch_bounds__(256) sample_partial_kernel(const float *logits, long long ld, int V,
                                                             int chunk, float inv_T,
                                                             unsigned long long seed, int stream,
                                                             int row0, float4 *part) {
  griddep_wait();
  griddep_launch();
  const int s = blockIdx.x, r = blockIdx.y, S = gridDim.x;
  const int lo = s * chunk;
  const int hi = min(V, lo + chunk);
  const float *x = logits + (long long)r * ld;
  float m = -INFINITY, sum = 0.f;
  Best b{-INFINITY, INT_MAX};
  // groups of four consecutive elements share one Philox block (chunk is a multiple of 4)
  for (int g = lo + 4 * threadIdx.x; g < hi; g += 4 * 256) {
    uint4 w = make_uint4(0, 0, 0, 0);
    if (stream >= 0)
      w = philox4x32_10(make_uint4((uint32_t)(g >> 2), (uint32_t)(row0 + r), (uint32_t)stream, 0u),
                        (uint32_t)seed, (uint32_t)(seed >> 32));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = g + q;
      if (v < hi) {
        const float xv = x[v] * inv_T;
        lse_add(m, sum, xv);
        if (stream >= 0) best_take(b, xv + gumbel_of(philox_u(ww[q])), v);
      }
    }
  }
  cta_reduce(m, sum, b);
  if (threadIdx.x == 0) part[(long long)r * S + s] = make_float4(m, sum, b.v, __int_as_float(b.id));
}

// One warp per row: combine the S slices. Writes lse[r] = max + log(sum) and, when ids is
// set, ids[r] = the Gumbel argmax and logq[r] = logits[r][id] * inv_T - lse[r].
__global__ void __launch_bounds__(128) sample_merge_kernel(const float4 *part, int rows, int S,
                                                           const float *logits, long long ld,
                                                           float inv_T, int *ids, float *lse,
                                                           float *logq) {
  griddep_wait();
  griddep_launch();
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float m = -INFINITY, s = 0.f;
  Best b{-INFINITY, INT_MAX};
  for (int k = lane; k < S; k += 32) {
    const float4 p = part[(long long)r * S + k];
    lse_merge(m, s, p.x, p.y);
    best_take(b, p.z, __float_as_int(p.w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    const float b2 = __shfl_xor_sync(0xffffffffu, b.v, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, b.id, o);
    lse_merge(m, s, m2, s2);
    best_take(b, b2, i2);
  }
  if (lane == 0) {
    const float l = m + logf(s);
    lse[r] = l;
    if (ids) {  // no winner only when every score is NaN: id -1
      const bool ok = b.id != INT_MAX;
      ids[r] = ok ? b.id : -1;
      logq[r] = ok ? logits[(long long)r * ld + b.id] * inv_T - l : -INFINITY;
    }
  }
}

// Rejection-sampling verify, one CTA per (slice, sequence). Every CTA of sequence i first
// finds the first rejection n: step j < B-1 accepts c = cand[i][j] when
// log u_j < log p_j(c) - log q_{j+1}(c), u_j = uniform(STREAM_ACCEPT = 1, row i, index j).
// Its slice then scores the emitted draw (stream 2, row i): over r(v) = p_n(v) - q_{n+1}(v) > 0
// the score log r(v) + g_v, and the fallback score log p_n(v) + g_v for the case that r is
// nowhere positive; after B-1 acceptances, log p_{B-1}(v) + g_v.
// part[i * S + s] = {best, id, fallback best, fallback id}; nrej[i] = n (slice 0).
__global__ void __launch_bounds__(256) verify_partial_kernel(
    const float *draft_logits, const float *draft_lse, const int *cand, const float *target_logits,
    const float *target_lse, int B, int V, int chunk, float inv_T, unsigned long long seed,
    float4 *part, int *nrej) {
  griddep_wait();
  griddep_launch();
  __shared__ int n_sh;
  const int s = blockIdx.x, i = blockIdx.y, S = gridDim.x;
  const int bm1 = B - 1;
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    bool acc = true;
    if (j < bm1) {
      const int c = cand[i * bm1 + j];
      if (c >= 0 && c < V) {
        const float lp = target_logits[((long long)i * B + j) * V + c] * inv_T - target_lse[i * B + j];
        const float lq = draft_logits[((long long)i * bm1 + j) * V + c] * inv_T - draft_lse[i * bm1 + j];
        acc = logf(philox_uniform(seed, 1, i, j)) < lp - lq;
      } else {
        acc = false;  // an id outside the vocabulary is never accepted
      }
    }
    const unsigned rej = __ballot_sync(0xffffffffu, !acc);
    if (threadIdx.x == 0) {
      const int n = rej ? __ffs(rej) - 1 : bm1;
      n_sh = n < bm1 ? n : bm1;
    }
  }
  __syncthreads();
  const int n = n_sh;
  if (s == 0 && threadIdx.x == 0) nrej[i] = n;
  const float *zp = target_logits + ((long long)i * B + n) * V;
  const float lzp = target_lse[i * B + n];
  const bool all = n == bm1;
  const float *zq = all ? zp : draft_logits + ((long long)i * bm1 + n) * V;
  const float lzq = all ? 0.f : draft_lse[i * bm1 + n];
  const int lo = s * chunk;
  const int hi = min(V, lo + chunk);
  Best b{-INFINITY, INT_MAX}, f{-INFINITY, INT_MAX};
  for (int g = lo + 4 * threadIdx.x; g < hi; g += 4 * 256) {
    const uint4 w = philox4x32_10(make_uint4((uint32_t)(g >> 2), (uint32_t)i, 2u, 0u), (uint32_t)seed,
                                  (uint32_t)(seed >> 32));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = g + q;
      if (v < hi) {
        const float gv = gumbel_of(philox_u(ww[q]));
        const float lp = zp[v] * inv_T - lzp;
        best_take(f, lp + gv, v);
        if (!all) {
          const float r = __expf(lp) - __expf(zq[v] * inv_T - lzq);
          if (r > 0.f) best_take(b, logf(r) + gv, v);
        }
      }
    }
  }
  // reduce both bests over the CTA
  __shared__ float rb[8], rf[8];
  __shared__ int rbi[8], rfi[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, b.v, o);
    const int bi2 = __shfl_xor_sync(0xffffffffu, b.id, o);
    const float f2 = __shfl_xor_sync(0xffffffffu, f.v, o);
    const int fi2 = __shfl_xor_sync(0xffffffffu, f.id, o);
    best_take(b, b2, bi2);
    best_take(f, f2, fi2);
  }
  const int wp = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    rb[wp] = b.v;
    rbi[wp] = b.id;
    rf[wp] = f.v;
    rfi[wp] = f.id;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < 8; ++k) {
      best_take(b, rb[k], rbi[k]);
      best_take(f, rf[k], rfi[k]);
    }
    part[(long long)i * S + s] = make_float4(b.v, __int_as_float(b.id), f.v, __int_as_float(f.id));
  }
}

// One thread per sequence: tau = n + 1; token = the residual draw when some r(v) > 0 (and
// n < B-1), else the fallback draw.
__global__ void verify_merge_kernel(const float4 *part, const int *nrej, int nb, int B, int S,
                                    int *tau, int *token) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nb) return;
  Best b{-INFINITY, INT_MAX}, f{-INFINITY, INT_MAX};
  for (int k = 0; k < S; ++k) {
    const float4 p = part[(long long)i * S + k];
    best_take(b, p.x, __float_as_int(p.y));
    best_take(f, p.z, __float_as_int(p.w));
  }
  const int n = nrej[i];
  tau[i] = n + 1;
  const int t = (n < B - 1 && b.id != INT_MAX) ? b.id : f.id;
  token[i] = t != INT_MAX ? t : -1;  // -1 only when every score is NaN
}

int sample_slices(int rows, int V, int num_sms) {
  int S = (4 * num_sms + rows - 1) / max(rows, 1);
  const int max_s = (V + 1023) / 1024;  // at least 1024 elements per slice
  S = max(1, min(S, min(max_s, kSampleMaxSlices)));
  return S;
}

static int slice_chunk(int V, int S) { return ((V + S - 1) / S + 3) & ~3; }

cudaError_t launch_sample(const float *logits, long long ld, int rows, int V, float inv_T,
                          unsigned long long seed, int stream, int row0, int S, float4 *part,
                          int *ids, float *lse, float *logq, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(sample_partial_kernel, dim3(S, rows), dim3(256), 0, s, logits, ld, V,
                             slice_chunk(V, S), inv_T, seed, stream, row0, part);
  if (e != cudaSuccess) return e;
  e = launch_pdl(sample_merge_kernel, dim3((rows + 3) / 4), dim3(128), 0, s, (const float4 *)part, rows,
                 S, logits, ld, inv_T, ids, lse, logq);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_verify(const float *draft_logits, const float *draft_lse, const int *cand,
                          const float *target_logits, const float *target_lse, int nb, int B, int V,
                          float inv_T, unsigned long long seed, int S, float4 *part, int *nrej,
                          int *tau, int *token, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(verify_partial_kernel, dim3(S, nb), dim3(256), 0, s, draft_logits,
                             draft_lse, cand, target_logits, target_lse, B, V, slice_chunk(V, S),
                             inv_T, seed, part, nrej);
  if (e != cudaSuccess) return e;
  e = launch_pdl(verify_merge_kernel, dim3((nb + 127) / 128), dim3(128), 0, s, (const float4 *)part,
                 (const int *)nrej, nb, B, S, tau, token);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
