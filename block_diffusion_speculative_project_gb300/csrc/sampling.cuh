// Device helpers of the sampling path, shared by the sampling passes (sampling.cu) and the
// LM-head epilogue that draws while it computes the logits (gemm_tc.cu).
//
// Philox4x32-10 (Salmon et al., "Parallel random numbers: as easy as 1, 2, 3", SC 2011):
// element v of (stream, row) is word v % 4 of the block at counter (v / 4, row, stream, 0),
// key (seed low, seed high); u = ((w >> 9) + 1/2) / 2^23, exact in fp32. A draw from
// softmax(x) is argmax_v x_v - log(-log u_v) (Gumbel-max), ties to the lower id.
#pragma once

#include <climits>
#include <cmath>
#include <cstdint>

namespace df {

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

// Gumbel value -log(-log u) of the uniform carried by Philox word w, in about 16
// instructions instead of two full-precision logarithms. E = -log u is needed to full
// relative precision (g = -log E; u close to 1 gives the largest g):
//  * u >= 1/2: t = 1 - u = (2^23 - k - 1/2) 2^-23 is exact, and
//    -log(1 - t) = 2 atanh(z) = 2 (z + z^3/3 + z^5/5 + ...), z = t / (2 - t) <= 1/3
//    (the series of log((1 + z) / (1 - z))); terms to z^13 leave a relative error below
//    1e-8;
//  * u < 1/2: E >= log 2, so the fast logarithm's absolute error (about 2^-21 in the log)
//    stays a relative error below 1e-6.
// Then g = -log E with the fast logarithm: an absolute error of about 1e-6 in g.
__device__ __forceinline__ float gumbel_fast(uint32_t w) {
  const uint32_t k = w >> 9;
  float E;
  if (k >= (1u << 22)) {
    const float t = (static_cast<float>((1u << 23) - k) - 0.5f) * 1.1920928955078125e-07f;
    const float z = __fdividef(t, 2.f - t);
    const float z2 = z * z;
    float sr = 1.f / 13.f;
    sr = fmaf(sr, z2, 1.f / 11.f);
    sr = fmaf(sr, z2, 1.f / 9.f);
    sr = fmaf(sr, z2, 1.f / 7.f);
    sr = fmaf(sr, z2, 1.f / 5.f);
    sr = fmaf(sr, z2, 1.f / 3.f);
    sr = fmaf(sr, z2, 1.f);
    E = 2.f * z * sr;
  } else {
    E = -__logf(philox_u(w));
  }
  return -__logf(E);
}

// Largest Gumbel value gumbel_fast returns (u = 1 - 2^-24 gives 16.636), rounded up.
constexpr float kGumbelMax = 16.7f;

// Draw pruning. An element of logit x can beat the running best score `best` only if its
// Gumbel value reaches d = best - x, i.e. E = -log u <= exp(-d). Since -log u >= t = 1 - u,
// t > exp(-d) (1 + 1e-5) rules it out; the factor covers the fast exponential (relative
// error ~5e-7) and gumbel_fast's own error (~2e-6), so a pruned element's computed score is
// strictly below best. t = (2^23 - k - 1/2) 2^-23 is exact for k = w >> 9.
__device__ __forceinline__ float draw_t_threshold(float d_min) {
  return d_min <= 0.f ? 2.f : __expf(-d_min) * 1.00001f;
}
__device__ __forceinline__ float philox_t(uint32_t w) {
  return (static_cast<float>((1u << 23) - (w >> 9)) - 0.5f) * 1.1920928955078125e-07f;
}

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



// Running state of one row's draw: log-sum-exp (m, s) of x = logit / T and the best
// Gumbel score with its id and its x.
struct DrawState {
  float m, s, best, x;
  int id;
};

__device__ __forceinline__ void draw_init(DrawState &d) {
  d.m = -INFINITY;
  d.s = 0.f;
  d.best = -INFINITY;
  d.x = -INFINITY;
  d.id = INT_MAX;
}

__device__ __forceinline__ void draw_add(DrawState &d, float x, float g, int id) {
  lse_add(d.m, d.s, x);
  const float sc = x + g;
  if (sc > d.best || (sc == d.best && id < d.id)) {
    d.best = sc;
    d.id = id;
    d.x = x;
  }
}

__device__ __forceinline__ void draw_merge(DrawState &d, const DrawState &o) {
  lse_merge(d.m, d.s, o.m, o.s);
  if (o.best > d.best || (o.best == d.best && o.id < d.id)) {
    d.best = o.best;
    d.id = o.id;
    d.x = o.x;
  }
}

// A partial draw in memory: two float4, {m, s, best, id bits} and {x, 0, 0, 0}.
__device__ __forceinline__ void draw_store(float4 *p, const DrawState &d) {
  p[0] = make_float4(d.m, d.s, d.best, __int_as_float(d.id));
  p[1] = make_float4(d.x, 0.f, 0.f, 0.f);
}

__device__ __forceinline__ DrawState draw_load(const float4 *p) {
  const float4 a = p[0];
  DrawState d;
  d.m = a.x;
  d.s = a.y;
  d.best = a.z;
  d.id = __float_as_int(a.w);
  d.x = p[1].x;
  return d;
}

// Draw over the 32 consecutive columns col0..col0+31 (col0 a multiple of 4) of one row:
// logits v[] (scaled by inv_T in place), nval of them valid. Written for instruction-level
// parallelism, since the caller may be one warp per SM sub-partition: the four Philox blocks
// of a 16-column half, its 16 Gumbel values and scores are independent; the half's max, sum
// of exponentials and best score (ties to the lower column) are trees; the running state
// takes one merge per half.
__device__ __forceinline__ void draw_chunk32(DrawState &d, float (&v)[32], float inv_T, int col0,
                                             int nval, uint32_t row, uint32_t stream,
                                             unsigned long long seed) {
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t w[16];
#pragma unroll
    for (int g4 = 0; g4 < 4; ++g4) {
      const uint4 q = philox4x32_10(make_uint4((uint32_t)((col0 + 16 * h + 4 * g4) >> 2), row, stream, 0u),
                                    (uint32_t)seed, (uint32_t)(seed >> 32));
      w[4 * g4] = q.x;
      w[4 * g4 + 1] = q.y;
      w[4 * g4 + 2] = q.z;
      w[4 * g4 + 3] = q.w;
    }
    float sc[16], sx[16];
    int ix[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = 16 * h + i;
      v[c] = c < nval ? v[c] * inv_T : -INFINITY;
    }
    float mx = v[16 * h];
#pragma unroll
    for (int i = 1; i < 16; ++i) mx = fmaxf(mx, v[16 * h + i]);
    if (mx == -INFINITY) continue;  // nothing valid in this half
    const float tthr = draw_t_threshold(d.best - mx);
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int c = 16 * h + i;
      sc[i] = -INFINITY;
      if (v[c] != -INFINITY && philox_t(w[i]) <= tthr) sc[i] = v[c] + gumbel_fast(w[i]);
      sx[i] = v[c];
      ix[i] = i;
    }
    float e[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) e[i] = __expf(v[16 * h + i] - mx);
#pragma unroll
    for (int st = 8; st > 0; st >>= 1) {
#pragma unroll
      for (int i = 0; i < st; ++i) {
        e[i] += e[i + st];
        const bool right = sc[i + st] > sc[i] || (sc[i + st] == sc[i] && ix[i + st] < ix[i]);
        sc[i] = right ? sc[i + st] : sc[i];
        sx[i] = right ? sx[i + st] : sx[i];
        ix[i] = right ? ix[i + st] : ix[i];
      }
    }
    lse_merge(d.m, d.s, mx, e[0]);
    const int id = col0 + 16 * h + ix[0];
    if (sc[0] > d.best || (sc[0] == d.best && id < d.id)) {
      d.best = sc[0];
      d.id = id;
      d.x = sx[0];
    }
  }
}

}  // namespace df
