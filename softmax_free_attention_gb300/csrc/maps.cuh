// maps.cuh -- the three score-to-weight maps over one 32-key chunk of one
// query row (one thread = one row, the chunk's raw dot products in registers),
// as the tensor-core forward applies them between the two MMAs.
//
//   Yat      kappa = (q.k + b)^2 / max(|q|^2 + |k|^2 - 2 q.k + eps, eps)
//            ("Softmax-Free Attention in JAX/Flax NNX", section "One module,
//            two compatibility functions": (dots + b)^2 / (max(d2, 0) + eps),
//            with d2 assembled from the norms and the same dot products)
//   softmax  2^(scale log2(e) q.k - m)
//   s^tau    2^(tau log2(softplus(scale q.k) + eps) - m)  ("s^tau: a focal-length
//            knob for attention": phi^tau with phi = softplus(s) + eps, taken in
//            the log domain so that phi^tau cannot overflow; softplus's log1p
//            by a polynomial, phi2)
#pragma once

#include <stdint.h>

#include "ptx.cuh"

namespace cattn {
namespace tc {

__device__ __forceinline__ float2 f2(uint32_t a, uint32_t b) {
  return make_float2(__uint_as_float(a), __uint_as_float(b));
}

// Yat kernel of one pair of keys: kappa = (dot + b)^2 / max(|q|^2 + |k|^2 -
// 2 dot + eps, eps) with qe = |q|^2 + eps.
// FAST: one reciprocal per pair, 1/den0 = den1 / (den0 den1), which halves
// the SFU work, and no clamp.  The caller takes it only when it is exact up
// to rounding: the assembled |q-k|^2 can fall below zero only by the rounding
// of |q|^2 + |k|^2 - 2 q.k, which is far below eps when
// (|q|^2 + max |k|^2) 2^-16 <= eps, and then every den0 den1 is a normal fp32
// number if also eps >= 2^-60 and |q|^2 + max |k|^2 <= 2^61.
// M: the numerator is (dot + b)^{2M} ("The Kernel Between the Roles", section
// "The run": raising the numerator's power sharpens the kernel's peak).
template <bool FAST, int M = 1>
__device__ __forceinline__ float2 yat_pair(float2 d, float2 nk, float2 b2, float2 qe2, float yeps) {
  const float2 t = __fadd2_rn(d, b2);
  float2 num = __fmul2_rn(t, t);
  if constexpr (M == 2) num = __fmul2_rn(num, num);
  if constexpr (M == 3) num = __fmul2_rn(__fmul2_rn(num, num), num);
  const float2 den = __ffma2_rn(make_float2(-2.f, -2.f), d, __fadd2_rn(qe2, nk));
  if (FAST) {
    const float r = rcp_approx(den.x * den.y);
    return __fmul2_rn(__fmul2_rn(num, make_float2(den.y, den.x)), make_float2(r, r));
  }
  return __fmul2_rn(num, make_float2(rcp_approx(fmaxf(den.x, yeps)), rcp_approx(fmaxf(den.y, yeps))));
}

// kappa of one (query row, key) pair straight from the stored bf16 rows, the
// dot product and |q - k|^2 each summed over the components in fp32 (no norm
// expansion, so nothing cancels), for the few keys whose assembled distance
// may have lost its digits (see yat_near_threshold).
template <int DK, int M>
__device__ __forceinline__ float yat_direct(const uint4 *q4, const uint4 *k4, float b, float eps) {
  float2 dot = make_float2(0.f, 0.f), d2 = dot;
#pragma unroll 2
  for (int i = 0; i < DK / 8; ++i) {
    const uint4 a = __ldg(q4 + i), c = __ldg(k4 + i);
    const uint32_t qa[4] = {a.x, a.y, a.z, a.w}, ka[4] = {c.x, c.y, c.z, c.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {
      const float2 qf = make_float2(__uint_as_float(qa[w] << 16), __uint_as_float(qa[w] & 0xffff0000u));
      const float2 kf = make_float2(__uint_as_float(ka[w] << 16), __uint_as_float(ka[w] & 0xffff0000u));
      dot = __ffma2_rn(qf, kf, dot);
      const float2 df = make_float2(qf.x - kf.x, qf.y - kf.y);
      d2 = __ffma2_rn(df, df, d2);
    }
  }
  const float t = (dot.x + dot.y) + b;
  float num = t * t;
  if constexpr (M == 2) num = num * num;
  if constexpr (M == 3) num = num * num * num;
  return num / (fmaxf(d2.x + d2.y, 0.f) + eps);
}

// Whether yat_pair<true> (one reciprocal per key pair, no clamp) is exact up
// to rounding for every row of the warp against keys whose squared norms are
// at most nk_max (qe = |q|^2 + eps of the lane's row): the assembled distance
// is then off by at most 2^-16 (qe + nk_max) <= eps from the true one, so
// den >= eps / 2 > 0, and den0 * den1 <= (qe + nk_max)^2 stays finite.
// Warp-uniform.
__device__ __forceinline__ bool yat_fast_ok(float nk_max, float qe, float yeps) {
  const float span = qe + nk_max;
  return yeps >= 0x1p-60f && __all_sync(0xffffffffu, span <= 0x1p61f && span * 0x1p-16f <= yeps);
}

// yat_direct as a called function, for call sites that take it key by key
// (the row statistics pass) and should not each carry a copy of the loop.
template <int DK, int M>
__device__ __noinline__ float yat_direct_call(const uint4 *q4, const uint4 *k4, float b, float eps) {
  return yat_direct<DK, M>(q4, k4, b, eps);
}

// Guard of the assembled distance for one query row.  |q|^2 + |k|^2 - 2 q.k
// is three fp32 sums of at most 128 terms, together off by at most
// E = 2^-16 (|q|^2 + |k|^2) from the true squared distance; that is below
// 2^-12 of den = d^2 + eps unless den < (|q|^2 + |k|^2) / 16.  Such a key has
// 0.695 |q| < |k| < 1.44 |q| and q.k > (15/32)(|q|^2 + |k|^2), so its computed
// kappa exceeds thr = (b + (15/32)|q|^2)^(2M) / (0.2 |q|^2) (b >= 0).  Keys of
// random direction sit far below thr (kappa of order |q|^2 / (2 d)).  A row
// whose computed max kappa passes thr is recomputed by the plain definition
// (the forward's near-key pass, near_fix_kernel; the row statistics pass key
// by key).  nq = 0 gives +inf (no key can be at risk).
__device__ __forceinline__ float yat_near_threshold(float nq, float b, int M) {
  const float a = fmaf(0.46875f, nq, b);
  float num = a * a;
  if (M == 2) num = num * num;
  if (M == 3) num = num * num * num;
  return a > 0.f ? num / (0.2f * nq) : 0.f;
}

// top > yat_near_threshold(nq, b, M) without the division (the forward's
// finalise takes it once per row on the way to releasing O).
__device__ __forceinline__ bool yat_near_flag(float top, float nq, float b, int M) {
  const float a = fmaf(0.46875f, nq, b);
  float num = a * a;
  if (M == 2) num = num * num;
  if (M == 3) num = num * num * num;
  return a > 0.f ? top * (0.2f * nq) > num : top > 0.f;
}

// Masks, accumulates and packs one pair: masked keys (col >= limit) get
// kappa = 0; mass (two chains) and top take kappa; returns P = bf16(kappa).
// ENT: ent also takes kappa log2 kappa (0 for kappa = 0), the row's
// sum f log2 f for its entropy.
template <bool PARTIAL, bool ENT = false>
__device__ __forceinline__ uint32_t yat_fold(float2 k, int col, int limit, float2 &mass, float &top,
                                             float2 &ent) {
  if (PARTIAL) {
    k.x = col < limit ? k.x : 0.f;
    k.y = col + 1 < limit ? k.y : 0.f;
  }
  mass = __fadd2_rn(mass, k);
  top = max3(top, k.x, k.y);
  if (ENT) {
    // (the clamp keeps the flush-to-zero log finite, so that kappa = 0 adds
    // 0 without a select)
    const float2 lk = make_float2(lg2_approx(fmaxf(k.x, 1e-30f)), lg2_approx(fmaxf(k.y, 1e-30f)));
    ent = __ffma2_rn(k, lk, ent);
  }
  return pack_bf16x2(k.x, k.y);
}

// Yat map over one 32-key chunk (columns 32c .. 32c+31 of the tile) of one row.  sr: raw
// dots; nk4: squared key norms of the tile (groups of four).
template <bool PARTIAL, bool FAST, int M = 1, bool ENT = false>
__device__ __forceinline__ void yat_chunk(const uint32_t (&sr)[32], int c, const float4 *nk4,
                                          float yb, float qe, float yeps, int limit,
                                          float2 (&mass)[2], float (&top)[2],
                                          uint32_t (&pk)[16], float2 (&ent)[2]) {
  const float2 b2 = make_float2(yb, yb), qe2 = make_float2(qe, qe);
#pragma unroll
  for (int i = 0; i < 32; i += 4) {
    const float4 n4 = nk4[(c * 32 + i) >> 2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int ii = i + 2 * h;
      const float2 k = yat_pair<FAST, M>(f2(sr[ii], sr[ii + 1]),
                                      h ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y), b2, qe2,
                                      yeps);
      pk[ii >> 1] = yat_fold<PARTIAL, ENT>(k, c * 32 + ii, limit, mass[h], top[h], ent[h]);
    }
  }
}

// Max of the raw dot over the allowed keys of one 32-key chunk (masked -> -inf).
template <bool PARTIAL>
__device__ __forceinline__ float chunk_max(const uint32_t (&sr)[32], int c, int limit) {
  float m[2] = {-INFINITY, -INFINITY};
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const int col = c * 32 + i;
    float x0 = __uint_as_float(sr[i]), x1 = __uint_as_float(sr[i + 1]);
    if (PARTIAL) {
      x0 = col < limit ? x0 : -INFINITY;
      x1 = col + 1 < limit ? x1 : -INFINITY;
    }
    m[(i >> 1) & 1] = max3(m[(i >> 1) & 1], x0, x1);
  }
  return fmaxf(m[0], m[1]);
}

// softmax over one 32-key chunk: p = 2^(dot * c2 - m), c2 = scale * log2(e).
// ENT: ent also takes p (dot c2 - m), the row's sum p log2 p (relative to m).
template <bool PARTIAL, bool ENT = false>
__device__ __forceinline__ void softmax_chunk(const uint32_t (&sr)[32], int c, float c2,
                                              float neg_m, int limit, float2 (&l)[2],
                                              uint32_t (&pk)[16], float2 (&ent)[2]) {
  const float2 c22 = make_float2(c2, c2), nm2 = make_float2(neg_m, neg_m);
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const int col = c * 32 + i;
    const float2 x = __ffma2_rn(f2(sr[i], sr[i + 1]), c22, nm2);
    float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    if (PARTIAL) {
      pr.x = col < limit ? pr.x : 0.f;
      pr.y = col + 1 < limit ? pr.y : 0.f;
    }
    l[(i >> 1) & 1] = __fadd2_rn(l[(i >> 1) & 1], pr);
    if (ENT) ent[(i >> 1) & 1] = __ffma2_rn(pr, x, ent[(i >> 1) & 1]);
    pk[i >> 1] = pack_bf16x2(pr.x, pr.y);
  }
}

// log1p(e) for e in [0, 1] as e P(e), P the degree-5 Chebyshev interpolant
// of log1p(x)/x on [0, 1] (interpolation at the Chebyshev points, converted
// to powers of x): relative error below 1e-5 over the whole interval, tiny e
// included, on the FMA pipe.  Every tensor-core path that forms phi(s) (the
// s^tau forward map, its running max, the row statistics, tau* and the
// backward) does it through phi1 / phi2 below, so that a backward's weights
// match the forward's normaliser.  The coefficients are numpy's
// Chebyshev.interpolate(lambda x: log1p(x) / x, 5, domain=[0, 1]) converted
// to the power basis and rounded to fp32.
constexpr float kL1p0 = 0.999990582f, kL1p1 = -0.499314666f, kL1p2 = 0.324849576f,
                kL1p3 = -0.209079534f, kL1p4 = 0.10013973f, kL1p5 = -0.023443656f;
// phi = softplus(s) + eps = max(s, 0) + log1p(e) + eps, e = 2^(-|s| log2 e),
// with max(s, 0) formed as (s + |s|) / 2 (exact in fp32) and eps folded into
// the polynomial's last multiply: three operations after P(e).
__device__ __forceinline__ float phi1(float s, float e, float eps) {
  float p = fmaf(kL1p5, e, kL1p4);
  p = fmaf(p, e, kL1p3);
  p = fmaf(p, e, kL1p2);
  p = fmaf(p, e, kL1p1);
  p = fmaf(p, e, kL1p0);
  return fmaf(0.5f, s + fabsf(s), fmaf(e, p, eps));
}
__device__ __forceinline__ float2 phi2(float2 s, float2 e, float eps) {
  float2 p = __ffma2_rn(make_float2(kL1p5, kL1p5), e, make_float2(kL1p4, kL1p4));
  p = __ffma2_rn(p, e, make_float2(kL1p3, kL1p3));
  p = __ffma2_rn(p, e, make_float2(kL1p2, kL1p2));
  p = __ffma2_rn(p, e, make_float2(kL1p1, kL1p1));
  p = __ffma2_rn(p, e, make_float2(kL1p0, kL1p0));
  const float2 l = __ffma2_rn(e, p, make_float2(eps, eps));
  const float2 u = __fadd2_rn(s, make_float2(fabsf(s.x), fabsf(s.y)));
  return __ffma2_rn(make_float2(0.5f, 0.5f), u, l);
}

// log2(softplus(s) + eps).
__device__ __forceinline__ float log2_phi(float s, float abs_s_log2e, float eps) {
  return lg2_approx(phi1(s, ex2_approx(-abs_s_log2e), eps));
}

// log2 phi(s) of two scores with the non-SFU arithmetic in f32x2 pairs (the
// map is bound by instruction issue): two SFU operations per score.
__device__ __forceinline__ float2 log2_phi2(float2 d, float scale, float c2, float eps) {
  const float2 s = __fmul2_rn(d, make_float2(scale, scale));
  const float2 a = __fmul2_rn(make_float2(fabsf(d.x), fabsf(d.y)), make_float2(c2, c2));
  const float2 phi = phi2(s, make_float2(ex2_approx(-a.x), ex2_approx(-a.y)), eps);
  return make_float2(lg2_approx(phi.x), lg2_approx(phi.y));
}

// s^tau over one 32-key chunk: p = 2^(tau log2 phi(s) - m).
template <bool PARTIAL, bool ENT = false>
__device__ __forceinline__ void stau_chunk(const uint32_t (&sr)[32], int c, float scale, float c2,
                                           float tau, float eps, float neg_m, int limit,
                                           float2 (&l)[2], uint32_t (&pk)[16], float2 (&ent)[2]) {
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const int col = c * 32 + i;
    const float2 g = log2_phi2(f2(sr[i], sr[i + 1]), scale, c2, eps);
    const float2 x = __ffma2_rn(make_float2(tau, tau), g, make_float2(neg_m, neg_m));
    float2 pr = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    if (PARTIAL) {
      pr.x = col < limit ? pr.x : 0.f;
      pr.y = col + 1 < limit ? pr.y : 0.f;
    }
    l[(i >> 1) & 1] = __fadd2_rn(l[(i >> 1) & 1], pr);
    if (ENT) ent[(i >> 1) & 1] = __ffma2_rn(pr, x, ent[(i >> 1) & 1]);
    pk[i >> 1] = pack_bf16x2(pr.x, pr.y);
  }
}

// tau* statistics of one 32-key chunk ("s^tau: a focal-length knob for
// attention", tau* = Cov(s, ln phi(s)) / Var(ln phi(s))): for every allowed
// key, s = scale dot and g = ln phi(s) - g0 (the shift g0 = ln(ln 2 + eps),
// the value at s = 0, keeps the second moments well conditioned); adds 1, s,
// g, s g and g^2 to st.
template <bool PARTIAL>
__device__ __forceinline__ void tau_chunk(const uint32_t (&sr)[32], int c, float scale, float c2,
                                          float eps, float g0, int limit, float (&st)[5]) {
  constexpr float LN2 = 0.6931471805599453f;
  // two keys at a time in f32x2 pairs; the sums of each half kept apart
  float2 sum_s = make_float2(0.f, 0.f), sum_g = sum_s, sum_sg = sum_s, sum_gg = sum_s;
  float n = 0.f;
#pragma unroll
  for (int i = 0; i < 32; i += 2) {
    const float2 d = f2(sr[i], sr[i + 1]);
    float2 s = __fmul2_rn(d, make_float2(scale, scale));
    const float2 a = __fmul2_rn(make_float2(fabsf(d.x), fabsf(d.y)), make_float2(c2, c2));
    const float2 phi = phi2(s, make_float2(ex2_approx(-a.x), ex2_approx(-a.y)), eps);
    float2 g = __ffma2_rn(make_float2(lg2_approx(phi.x), lg2_approx(phi.y)), make_float2(LN2, LN2),
                          make_float2(-g0, -g0));
    if (PARTIAL) {
      const bool ok0 = c * 32 + i < limit, ok1 = c * 32 + i + 1 < limit;
      s = make_float2(ok0 ? s.x : 0.f, ok1 ? s.y : 0.f);
      g = make_float2(ok0 ? g.x : 0.f, ok1 ? g.y : 0.f);
      n += (ok0 ? 1.f : 0.f) + (ok1 ? 1.f : 0.f);
    }
    sum_s = __fadd2_rn(sum_s, s);
    sum_g = __fadd2_rn(sum_g, g);
    sum_sg = __ffma2_rn(s, g, sum_sg);
    sum_gg = __ffma2_rn(g, g, sum_gg);
  }
  st[0] += PARTIAL ? n : 32.f;
  st[1] += sum_s.x + sum_s.y;
  st[2] += sum_g.x + sum_g.y;
  st[3] += sum_sg.x + sum_sg.y;
  st[4] += sum_gg.x + sum_gg.y;
}

// Row statistics of the map over one thread's keys (normalised entropy: "The
// Kernel Between the Roles", section "The run"; sparsity below 1e-6 and top-10
// concentration: the s^tau page's fine-tuning comparison), kept on the map's
// unnormalised values so that the row's normaliser is applied once at the
// end.  Yat takes kappa: hs = sum kappa log2 kappa and sk = sum kappa, so that
// sum w ln w = (ln 2 hs - ln Z' sk) / Z' with w = kappa / Z'; softmax and s^tau
// take x = log2 w: hs = sum 2^x x, so that sum w ln w = ln 2 hs.  small counts
// the allowed keys under the row's threshold (Yat 1e-6 Z', else log2 1e-6);
// top holds the ten largest kappa (or x), in descending order.
struct RowStats {
  float2 hs, sk;
  float small;
  float top[10];
};

// The top-10 insert is a bubble through the sorted list, taken only when some
// lane of the warp has a value above its tenth largest.
__device__ __forceinline__ void top10_insert(float (&top)[10], float v) {
  if (__any_sync(0xffffffffu, v > top[9])) {
#pragma unroll
    for (int i = 0; i < 10; ++i) {
      const float hi = fmaxf(top[i], v);
      v = fminf(top[i], v);
      top[i] = hi;
    }
  }
}

// Two keys of the Yat map: kappa (0 for keys that are not allowed; al0 / al1
// tell them apart for the count when PARTIAL).
template <bool PARTIAL>
__device__ __forceinline__ void stats_pair_yat(RowStats &st, float2 k, float thr, bool al0, bool al1) {
  // kappa log2 kappa is 0 for kappa = 0 (the clamp keeps the log finite)
  const float2 lk = make_float2(lg2_approx(fmaxf(k.x, 1e-30f)), lg2_approx(fmaxf(k.y, 1e-30f)));
  st.hs = __ffma2_rn(k, lk, st.hs);
  st.sk = __fadd2_rn(st.sk, k);
  st.small += ((!PARTIAL || al0) && k.x < thr) ? 1.f : 0.f;
  st.small += ((!PARTIAL || al1) && k.y < thr) ? 1.f : 0.f;
  top10_insert(st.top, k.x);
  top10_insert(st.top, k.y);
}

// Two keys of softmax or s^tau: x = log2 of the weight (a large negative
// finite value for keys that are not allowed, so that 2^x x is 0).
template <bool PARTIAL>
__device__ __forceinline__ void stats_pair_log(RowStats &st, float2 x, float thr, bool al0, bool al1) {
  const float2 w = make_float2(ex2_approx(x.x), ex2_approx(x.y));
  st.hs = __ffma2_rn(w, x, st.hs);
  st.small += ((!PARTIAL || al0) && x.x < thr) ? 1.f : 0.f;
  st.small += ((!PARTIAL || al1) && x.y < thr) ? 1.f : 0.f;
  top10_insert(st.top, x.x);
  top10_insert(st.top, x.y);
}

}  // namespace tc
}  // namespace cattn
