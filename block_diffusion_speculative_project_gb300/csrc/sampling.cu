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
#include "sampling.cuh"

namespace df {

namespace {

// CTA-wide merge (256 threads) of a draw state; the result is valid in thread 0.
__device__ __forceinline__ void cta_reduce(DrawState &d) {
  __shared__ float rm[8], rs[8], rb[8], rx[8];
  __shared__ int ri[8];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DrawState e;
    e.m = __shfl_xor_sync(0xffffffffu, d.m, o);
    e.s = __shfl_xor_sync(0xffffffffu, d.s, o);
    e.best = __shfl_xor_sync(0xffffffffu, d.best, o);
    e.x = __shfl_xor_sync(0xffffffffu, d.x, o);
    e.id = __shfl_xor_sync(0xffffffffu, d.id, o);
    draw_merge(d, e);
  }
  const int w = threadIdx.x >> 5;
  if ((threadIdx.x & 31) == 0) {
    rm[w] = d.m;
    rs[w] = d.s;
    rb[w] = d.best;
    rx[w] = d.x;
    ri[w] = d.id;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    for (int k = 1; k < 8; ++k) {
      DrawState e;
      e.m = rm[k];
      e.s = rs[k];
      e.best = rb[k];
      e.x = rx[k];
      e.id = ri[k];
      draw_merge(d, e);
    }
  }
}

}  // namespace

// Partial draw of row r, slice s (entry (r * S + s) of two float4, see draw_store) over
// x = logits[r * ld + v] * inv_T, v in the slice; Philox row row0 + r of `stream`. With
// stream < 0 only the log-sum-exp is formed (no Gumbel values). Each thread takes groups
// of four consecutive elements (one Philox block), four groups per iteration so that four
// 16-byte loads are in flight; vec: rows start 16-byte aligned and ld % 4 == 0.
__global__ void __launch_bounds__(256) sample_partial_kernel(const float *logits, long long ld, int V,
                                                             int chunk, float inv_T,
                                                             unsigned long long seed, int stream,
                                                             int row0, int vec, float4 *part) {
  griddep_wait();
  griddep_launch();
  const int s = blockIdx.x, r = blockIdx.y, S = gridDim.x;
  const int lo = s * chunk;
  const int hi = min(V, lo + chunk);
  const float *x = logits + (long long)r * ld;
  DrawState d;
  draw_init(d);
  auto load4 = [&](int g, float (&o)[4]) {
    if (vec && g + 4 <= hi) {
      const float4 f = *reinterpret_cast<const float4 *>(x + g);
      o[0] = f.x; o[1] = f.y; o[2] = f.z; o[3] = f.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) o[q] = (g + q < hi) ? x[g + q] : -INFINITY;
    }
  };
  auto take4 = [&](int g, const float (&o)[4]) {
    float x[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) x[q] = (g + q < hi) ? o[q] * inv_T : -INFINITY;
    const float m4 = fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
    if (m4 == -INFINITY) return;
    // log-sum-exp: one rescale per group when its max is a new maximum
    if (m4 > d.m) {
      d.s = (d.m == -INFINITY) ? 0.f : d.s * __expf(d.m - m4);
      d.m = m4;
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) d.s += __expf(x[q] - d.m);
    if (stream < 0) return;
    // the draw: nothing in the group can reach the best score -> no random numbers needed
    const float d_min = d.best - m4;
    if (d_min > kGumbelMax) return;
    const uint4 w = philox4x32_10(make_uint4((uint32_t)(g >> 2), (uint32_t)(row0 + r), (uint32_t)stream, 0u),
                                  (uint32_t)seed, (uint32_t)(seed >> 32));
    const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
    const float tthr = draw_t_threshold(d_min);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if (x[q] != -INFINITY && philox_t(ww[q]) <= tthr) {
        const float sc = x[q] + gumbel_fast(ww[q]);
        if (sc > d.best || (sc == d.best && g + q < d.id)) {
          d.best = sc;
          d.id = g + q;
          d.x = x[q];
        }
      }
    }
  };
  constexpr int kStep = 4 * 256;
  int g = lo + 4 * threadIdx.x;
  for (; g + 3 * kStep < hi; g += 4 * kStep) {  // four 16-byte loads in flight
    float a[4][4];
#pragma unroll
    for (int u = 0; u < 4; ++u) load4(g + u * kStep, a[u]);
#pragma unroll
    for (int u = 0; u < 4; ++u) take4(g + u * kStep, a[u]);
  }
  for (; g < hi; g += kStep) {
    float a0[4];
    load4(g, a0);
    take4(g, a0);
  }
  cta_reduce(d);
  if (threadIdx.x == 0) draw_store(part + 2 * ((long long)r * S + s), d);
}

// One warp per row r: merge the partial draws at entries r * row_stride + k * slice_stride,
// k < S. Writes lse[r] and, when ids is set, ids[r] (-1 when every score is NaN) and
// logq[r] = x[id] - lse[r].
__global__ void __launch_bounds__(128) sample_merge_kernel(const float4 *part, int rows, int S,
                                                           long long row_stride, long long slice_stride,
                                                           int *ids, float *lse, float *logq) {
  griddep_wait();
  griddep_launch();
  const int r = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  DrawState d;
  draw_init(d);
  for (int k = lane; k < S; k += 32) draw_merge(d, draw_load(part + 2 * (r * row_stride + k * slice_stride)));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    DrawState e;
    e.m = __shfl_xor_sync(0xffffffffu, d.m, o);
    e.s = __shfl_xor_sync(0xffffffffu, d.s, o);
    e.best = __shfl_xor_sync(0xffffffffu, d.best, o);
    e.x = __shfl_xor_sync(0xffffffffu, d.x, o);
    e.id = __shfl_xor_sync(0xffffffffu, d.id, o);
    draw_merge(d, e);
  }
  if (lane == 0) {
    const float l = d.m + logf(d.s);
    lse[r] = l;
    if (ids) {
      const bool ok = d.id != INT_MAX;
      ids[r] = ok ? d.id : -1;
      logq[r] = ok ? d.x - l : -INFINITY;
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
//
// With walk_ids set, the draft distribution of offset t is the sampling walk's: q_t(v) =
// exp(walk_logq[t-1][c]) for v = walk_ids[t-1][c] (c < wk), 0 elsewhere (draft_logits and
// draft_lse unused); a non-candidate's residual is then p itself.
__global__ void __launch_bounds__(256) verify_partial_kernel(
    const float *draft_logits, const float *draft_lse, const int *cand, const float *target_logits,
    const float *target_lse, int B, int V, int chunk, float inv_T, unsigned long long seed,
    float4 *part, int *nrej, const int *walk_ids, const float *walk_logq, int wk) {
  griddep_wait();
  griddep_launch();
  __shared__ int n_sh;
  __shared__ int sid[kTopkMax];
  __shared__ float sq[kTopkMax];
  const int s = blockIdx.x, i = blockIdx.y, S = gridDim.x;
  const int bm1 = B - 1;
  const bool walk = walk_ids != nullptr;
  if (threadIdx.x < 32) {
    const int j = threadIdx.x;
    bool acc = true;
    if (j < bm1) {
      const int c = cand[i * bm1 + j];
      if (c >= 0 && c < V) {
        const float lp = target_logits[((long long)i * B + j) * V + c] * inv_T - target_lse[i * B + j];
        float lq = INFINITY;  // a token the walk could not have drawn is rejected
        if (walk) {
          const int *ids = walk_ids + ((long long)i * bm1 + j) * wk;
          for (int q = 0; q < wk; ++q)
            if (ids[q] == c) lq = walk_logq[((long long)i * bm1 + j) * wk + q];
        } else {
          lq = draft_logits[((long long)i * bm1 + j) * V + c] * inv_T - draft_lse[i * bm1 + j];
        }
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
  if (walk && n < bm1 && threadIdx.x < wk) {
    sid[threadIdx.x] = walk_ids[((long long)i * bm1 + n) * wk + threadIdx.x];
    sq[threadIdx.x] = __expf(walk_logq[((long long)i * bm1 + n) * wk + threadIdx.x]);
  }
  __syncthreads();
  const float *zp = target_logits + ((long long)i * B + n) * V;
  const float lzp = target_lse[i * B + n];
  const bool all = n == bm1;
  const float *zq = (all || walk) ? zp : draft_logits + ((long long)i * bm1 + n) * V;
  const float lzq = (all || walk) ? 0.f : draft_lse[i * bm1 + n];
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
        const float gv = gumbel_fast(ww[q]);
        const float lp = zp[v] * inv_T - lzp;
        best_take(f, lp + gv, v);
        if (!all) {
          if (walk) {
            bool is_cand = false;
            float qv = 0.f;
            for (int q = 0; q < wk; ++q)
              if (sid[q] == v) {
                is_cand = true;
                qv = sq[q];
              }
            if (!is_cand) {
              best_take(b, lp + gv, v);
            } else {
              const float r = __expf(lp) - qv;
              if (r > 0.f) best_take(b, logf(r) + gv, v);
            }
          } else {
            const float r = __expf(lp) - __expf(zq[v] * inv_T - lzq);
            if (r > 0.f) best_take(b, logf(r) + gv, v);
          }
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

// One warp per sequence: tau = n + 1; token = the residual draw when some r(v) > 0 (and
// n < B-1), else the fallback draw.
__global__ void __launch_bounds__(128) verify_merge_kernel(const float4 *part, const int *nrej, int nb,
                                                           int B, int S, int *tau, int *token) {
  griddep_wait();
  griddep_launch();
  const int i = blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (i >= nb) return;
  Best b{-INFINITY, INT_MAX}, f{-INFINITY, INT_MAX};
  for (int k = lane; k < S; k += 32) {
    const float4 p = part[(long long)i * S + k];
    best_take(b, p.x, __float_as_int(p.y));
    best_take(f, p.z, __float_as_int(p.w));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float b2 = __shfl_xor_sync(0xffffffffu, b.v, o);
    const int bi2 = __shfl_xor_sync(0xffffffffu, b.id, o);
    const float f2 = __shfl_xor_sync(0xffffffffu, f.v, o);
    const int fi2 = __shfl_xor_sync(0xffffffffu, f.id, o);
    best_take(b, b2, bi2);
    best_take(f, f2, fi2);
  }
  if (lane == 0) {
    const int n = nrej[i];
    tau[i] = n + 1;
    const int t = (n < B - 1 && b.id != INT_MAX) ? b.id : f.id;
    token[i] = t != INT_MAX ? t : -1;  // -1 only when every score is NaN
  }
}

// u[v] and g[v] = Gumbel value of element v < n of (seed, stream, row).
__global__ void __launch_bounds__(256) draw_gumbel_kernel(int n, unsigned long long seed, int stream,
                                                          int row, float *u, float *g) {
  const int v = blockIdx.x * 256 + threadIdx.x;
  if (v >= n) return;
  const uint4 w = philox4x32_10(make_uint4((uint32_t)(v >> 2), (uint32_t)row, (uint32_t)stream, 0u),
                                (uint32_t)seed, (uint32_t)(seed >> 32));
  const int q = v & 3;
  const uint32_t word = q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w;
  u[v] = philox_u(word);
  g[v] = gumbel_fast(word);
}

cudaError_t launch_draw_gumbel(int n, unsigned long long seed, int stream, int row, float *u, float *g,
                               cudaStream_t s) {
  if (n <= 0) return cudaSuccess;
  draw_gumbel_kernel<<<(n + 255) / 256, 256, 0, s>>>(n, seed, stream, row, u, g);
  return cudaGetLastError();
}

int sample_slices(int rows, int V, int num_sms) {
  // one resident wave of the slice kernel: SMs x CTAs per SM (from its register use)
  static int per_sm = [] {
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, sample_partial_kernel, 256, 0) != cudaSuccess || n < 1)
      n = 4;
    return n;
  }();
  int S = (per_sm * num_sms) / max(rows, 1);
  const int max_s = (V + 1023) / 1024;  // at least 1024 elements per slice
  S = max(1, min(S, min(max_s, kSampleMaxSlices)));
  return S;
}

static int slice_chunk(int V, int S) { return ((V + S - 1) / S + 3) & ~3; }

cudaError_t launch_sample(const float *logits, long long ld, int rows, int V, float inv_T,
                          unsigned long long seed, int stream, int row0, int S, float4 *part,
                          int *ids, float *lse, float *logq, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  const int vec = (ld % 4 == 0) && (reinterpret_cast<uintptr_t>(logits) % 16 == 0);
  cudaError_t e = launch_pdl(sample_partial_kernel, dim3(S, rows), dim3(256), 0, s, logits, ld, V,
                             slice_chunk(V, S), inv_T, seed, stream, row0, vec, part);
  if (e != cudaSuccess) return e;
  return launch_draw_merge(part, rows, S, S, 1, ids, lse, logq, s);
}

cudaError_t launch_draw_merge(const float4 *part, int rows, int S, long long row_stride,
                              long long slice_stride, int *ids, float *lse, float *logq, cudaStream_t s) {
  if (rows <= 0) return cudaSuccess;
  cudaError_t e = launch_pdl(sample_merge_kernel, dim3((rows + 3) / 4), dim3(128), 0, s, part, rows, S,
                             row_stride, slice_stride, ids, lse, logq);
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
                             inv_T, seed, part, nrej, (const int *)nullptr, (const float *)nullptr, 0);
  if (e != cudaSuccess) return e;
  e = launch_pdl(verify_merge_kernel, dim3((nb + 3) / 4), dim3(128), 0, s, (const float4 *)part,
                 (const int *)nrej, nb, B, S, tau, token);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_verify_walk(const int *cand_ids, const float *walk_logq, int k, const int *path,
                               const float *target_logits, const float *target_lse, int nb, int B, int V,
                               float inv_T, unsigned long long seed, int S, float4 *part, int *nrej,
                               int *tau, int *token, cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  if (k < 1 || k > kTopkMax) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(verify_partial_kernel, dim3(S, nb), dim3(256), 0, s, (const float *)nullptr,
                             (const float *)nullptr, path, target_logits, target_lse, B, V, slice_chunk(V, S),
                             inv_T, seed, part, nrej, cand_ids, walk_logq, k);
  if (e != cudaSuccess) return e;
  e = launch_pdl(verify_merge_kernel, dim3((nb + 3) / 4), dim3(128), 0, s, (const float4 *)part,
                 (const int *)nrej, nb, B, S, tau, token);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// Sampling walk of the DFlash 2 selector: one CTA per sequence; the sequence's score table
// [B-1][k][k] and candidate ids are staged in shared memory, then warp 0 walks: lane c < k
// scores x_c = S_t(a_{t-1}, b_c) / T plus its Gumbel value (Philox stream 3, row
// i*(B-1) + t-1, element c), the warp takes the best (ties to the lower token id), and
// every lane writes log q_c = x_c - logsumexp(x).
__global__ void __launch_bounds__(128) select_walk_sample_kernel(const int *cand_ids, const float *table,
                                                                 int B, int k, float inv_T,
                                                                 unsigned long long seed, int *path,
                                                                 float *walk_logq) {
  griddep_wait();
  griddep_launch();
  extern __shared__ float tab[];  // [B-1][k][k] scores, then [B-1][k] candidate ids
  const int i = blockIdx.x;
  const int bm1 = B - 1;
  const int n = bm1 * k * k;
  int *sid = reinterpret_cast<int *>(tab + n);
  const float *ti = table + (size_t)i * n;
  for (int e = threadIdx.x; e < n; e += blockDim.x) tab[e] = ti[e];
  for (int e = threadIdx.x; e < bm1 * k; e += blockDim.x) sid[e] = cand_ids[(size_t)i * bm1 * k + e];
  __syncthreads();
  if (threadIdx.x >= 32) return;
  const int lane = threadIdx.x;
  int a = 0;  // slot of the previous choice (offset 1 reads the anchor's row 0)
  for (int t = 1; t < B; ++t) {
    const int row = i * bm1 + t - 1;
    const bool on = lane < k;
    const float x = on ? tab[((t - 1) * k + a) * k + lane] * inv_T : -INFINITY;
    const int id = on ? sid[(t - 1) * k + lane] : INT_MAX;
    float sc = -INFINITY;
    if (on) {
      const uint4 w = philox4x32_10(make_uint4((uint32_t)(lane >> 2), (uint32_t)row, 3u, 0u), (uint32_t)seed,
                                    (uint32_t)(seed >> 32));
      const int q = lane & 3;
      sc = x + gumbel_fast(q == 0 ? w.x : q == 1 ? w.y : q == 2 ? w.z : w.w);
    }
    float bsc = sc, m = x;
    int bid = id, bslot = lane;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float sc2 = __shfl_xor_sync(0xffffffffu, bsc, o);
      const int id2 = __shfl_xor_sync(0xffffffffu, bid, o);
      const int sl2 = __shfl_xor_sync(0xffffffffu, bslot, o);
      if (sc2 > bsc || (sc2 == bsc && id2 < bid)) {
        bsc = sc2;
        bid = id2;
        bslot = sl2;
      }
      m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    }
    float e = on ? __expf(x - m) : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) e += __shfl_xor_sync(0xffffffffu, e, o);
    if (on) walk_logq[(size_t)row * k + lane] = x - (m + logf(e));
    if (lane == 0) path[row] = bid;
    a = bslot;
  }
}

cudaError_t launch_select_walk_sample(const int *cand_ids, const float *table, int nb, int B, int k,
                                      float inv_T, unsigned long long seed, int *path, float *walk_logq,
                                      cudaStream_t s) {
  if (nb <= 0) return cudaSuccess;
  if (k < 1 || k > 16 || B < 2) return cudaErrorInvalidValue;
  cudaError_t e = launch_pdl(select_walk_sample_kernel, dim3(nb), dim3(128),
                             (size_t)(B - 1) * k * (k + 1) * sizeof(float), s, cand_ids, table, B, k, inv_T,
                             seed, path, walk_logq);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace df
