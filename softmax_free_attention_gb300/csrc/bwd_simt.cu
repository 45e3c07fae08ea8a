// bwd_simt.cu -- attention backward on the CUDA cores.
//
// The CUDA-core counterpart of bwd_tc.cu (same gradients, full fp32 FMA
// arithmetic): fp32 inputs (held to 1e-4 of each tensor's largest magnitude)
// and bf16 inputs whose widths have no tensor-core tiles (widened to fp32 on
// load, gradients rounded to bf16 on store).  Two passes, one warp per row; lane l owns columns l, l+32, ...
// of the row vectors, and every dot product is a warp reduction:
//
//   dQ pass   one warp per query row t: first D_t = sum_j w_tj dW_tj from its
//             own weights (and, for Yat, its own row mass), written to the
//             workspace for the second pass, then dq_t = sum_j C_tj k_j (+
//             Yat's distance term).
//   dK/dV     one warp per key row j of one kv head: every query row of every
//             query head sharing it, dk_j += C_tj q_t (+ Yat's distance term),
//             dv_j += w_tj dout_t, and the per-head parameter sums.
//
// Per pair (s = q.k, dW = dout . v):
//   softmax  w = exp(scale s - L_t), L_t the forward's log-sum-exp;
//            C = scale w (dW - D)
//   s^tau    phi = softplus(scale s) + eps, w = exp(tau ln phi - L_t);
//            C = scale w (dW - D) tau sigma(scale s) / phi,
//            dtau += w (dW - D) ln phi, deps += w (dW - D) tau / phi
//   Yat      d2 = |q - k|^2 (summed directly), den = max(d2, 0) + eps,
//            kappa = (s + b)^{2m} / den, Z = sum_j kappa_j + 1e-9 (this pass's
//            own sum, not the forward's M, and s accumulated in fp64: on a row
//            whose numerator s + b nearly cancels, both the numerator's
//            rounding and any mismatch between Z and the kappas reach the
//            gradient through its factor 2 / (s + b)), w = kappa / Z,
//            g = (dW - D) / Z, a = 2m g (s + b)^{2m-1} / den, e = -g kappa / den;
//            dq += a k + 2 e [d2 > 0] (q - k), dk += a q + 2 e [d2 > 0] (k - q),
//            db += a, deps += e
// (the chain rule through the maps of "Softmax-Free Attention in JAX/Flax
// NNX", section "One module, two compatibility functions", and "s^tau: a
// focal-length knob for attention", core formula).
#include <cuda_bf16.h>

#include "bwd.h"
#include "kernels.h"

namespace cattn {
namespace bwds {

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

constexpr unsigned FULL = 0xffffffffu;
constexpr int WARPS = 4;  // rows per 128-thread block

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}

struct Pair {
  float w, c, e, a;  // weight, score gradient, Yat's e [d2 > 0] and a (or s^tau's terms)
  float g1, g2;      // parameter-gradient terms: Yat (a, e); s^tau (deps, dtau)
};

// One pair from its dot products: dot = q.k (Yat: the numerator q.k + b,
// rounded once from fp64), dw = dout . v, d2 = |q - k|^2 (Yat).  Lt: the
// row's normaliser (softmax, s^tau: the forward's log-sum-exp; Yat: the dQ
// pass's Z = sum kappa + 1e-9); Dt: the row's D.
template <int VARIANT, int YM>
__device__ __forceinline__ Pair pair(float dot, float dw, float d2, float Lt, float Dt,
                                     float scale, float b, float eps, float tau) {
  Pair r{0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if constexpr (VARIANT == kSoftmax) {
    r.w = expf(scale * dot - Lt);
    r.c = scale * r.w * (dw - Dt);
  } else if constexpr (VARIANT == kStau) {
    const float s = scale * dot;
    const float phi = fmaxf(s, 0.f) + log1pf(expf(-fabsf(s))) + eps;
    const float lp = logf(phi);
    r.w = expf(tau * lp - Lt);
    const float sig = 1.f / (1.f + expf(-s));
    const float base = r.w * (dw - Dt);
    r.c = scale * base * tau * sig / phi;
    r.g1 = base * tau / phi;
    r.g2 = base * lp;
  } else {
    const float num = dot;
    float nodd = num;
    for (int i = 1; i < YM; ++i) nodd *= num * num;  // num^{2m-1}
    const float den = fmaxf(d2, 0.f) + eps;
    const float kap = nodd * num / den;
    r.w = kap / Lt;
    const float g = (dw - Dt) / Lt;
    r.a = (float)(2 * YM) * g * nodd / den;
    const float e = -g * kap / den;
    r.e = d2 > 0.f ? e : 0.f;
    r.c = r.a;  // the distance term is applied to the row vectors directly
    r.g1 = r.a;
    r.g2 = e;
  }
  return r;
}

template <int VARIANT, int DK, int DV, int YM, typename T>
__global__ void __launch_bounds__(WARPS * 32) dq_kernel(const BwdSimtParams p) {
  const T *gq = static_cast<const T *>(p.q), *gk = static_cast<const T *>(p.k);
  const T *gv = static_cast<const T *>(p.v), *gdo = static_cast<const T *>(p.dout);
  constexpr int KC = DK / 32, VC = DV / 32;
  const int lane = threadIdx.x & 31;
  const long long row = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (row >= (long long)p.B * p.h * p.Tq) return;
  const int t = (int)(row % p.Tq);
  const int bh = (int)(row / p.Tq);
  const int head = bh % p.h, batch = bh / p.h;
  const int bhk = batch * p.hkv + head / (p.h / p.hkv);
  const float b = VARIANT == kYat ? p.b[head] : 0.f;
  const float eps = VARIANT != kSoftmax ? p.eps[head] : 0.f;
  const float tau = VARIANT == kStau ? p.tau[head] : 1.f;
  float Lt = VARIANT == kYat ? 0.f : p.row_mass[row];
  float q[KC], dout[VC];
#pragma unroll
  for (int i = 0; i < KC; ++i) q[i] = ldf(gq + row * DK + lane + 32 * i);
#pragma unroll
  for (int i = 0; i < VC; ++i) dout[i] = ldf(gdo + row * DV + lane + 32 * i);
  const int n = p.causal ? min(t + 1, p.Tk) : p.Tk;
  const T *kb = gk + (size_t)bhk * p.Tk * DK;
  const T *vb = gv + (size_t)bhk * p.Tk * DV;
  auto dots = [&](int j, float &dot, float &dw, float &d2) {
    float a = 0.f, c = 0.f, e = 0.f;
    double a64 = 0.0;
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      const float kv = ldf(kb + (size_t)j * DK + lane + 32 * i);
      if (VARIANT == kYat) {
        a64 = fma((double)q[i], (double)kv, a64);
        e = fmaf(q[i] - kv, q[i] - kv, e);
      } else {
        a = fmaf(q[i], kv, a);
      }
    }
#pragma unroll
    for (int i = 0; i < VC; ++i) c = fmaf(dout[i], ldf(vb + (size_t)j * DV + lane + 32 * i), c);
    if (VARIANT == kYat) {
      dot = (float)(warp_sum_d(a64) + (double)b);  // the numerator q.k + b
    } else {
      dot = warp_sum(a);
    }
    dw = warp_sum(c);
    d2 = VARIANT == kYat ? warp_sum(e) : 0.f;
  };
  // D_t (and, for Yat, Z_t) from this pass's own weights
  float D = 0.f;
  if constexpr (VARIANT == kYat) {
    double z = 0.0, zd = 0.0;
    for (int j = 0; j < n; ++j) {
      float dot, dw, d2;
      dots(j, dot, dw, d2);
      const Pair r = pair<VARIANT, YM>(dot, dw, d2, 1.f, 0.f, p.scale, b, eps, tau);
      z += r.w;  // kappa
      zd += (double)r.w * dw;
    }
    Lt = (float)(z + 1e-9);
    D = (float)(zd / (z + 1e-9));
  } else {
    for (int j = 0; j < n; ++j) {
      float dot, dw, d2;
      dots(j, dot, dw, d2);
      const Pair r = pair<VARIANT, YM>(dot, dw, d2, Lt, 0.f, p.scale, b, eps, tau);
      D = fmaf(r.w, dw, D);
    }
  }
  if (lane == 0) {
    p.Dbuf[row] = D;
    if (VARIANT == kYat) p.Dbuf[(long long)p.B * p.h * p.Tq + row] = Lt;
  }
  float dq[KC];
#pragma unroll
  for (int i = 0; i < KC; ++i) dq[i] = 0.f;
  for (int j = 0; j < n; ++j) {
    float dot, dw, d2;
    dots(j, dot, dw, d2);
    const Pair r = pair<VARIANT, YM>(dot, dw, d2, Lt, D, p.scale, b, eps, tau);
#pragma unroll
    for (int i = 0; i < KC; ++i) {
      const float kv = ldf(kb + (size_t)j * DK + lane + 32 * i);
      dq[i] = fmaf(r.c, kv, dq[i]);
      if (VARIANT == kYat) dq[i] = fmaf(2.f * r.e, q[i] - kv, dq[i]);
    }
  }
#pragma unroll
  for (int i = 0; i < KC; ++i) stf(static_cast<T *>(p.dq) + row * DK + lane + 32 * i, dq[i]);
}

template <int VARIANT, int DK, int DV, int YM, typename T>
__global__ void __launch_bounds__(WARPS * 32) dkv_kernel(const BwdSimtParams p) {
  const T *gq = static_cast<const T *>(p.q), *gk = static_cast<const T *>(p.k);
  const T *gv = static_cast<const T *>(p.v), *gdo = static_cast<const T *>(p.dout);
  constexpr int KC = DK / 32, VC = DV / 32;
  const int lane = threadIdx.x & 31;
  const long long krow = (long long)blockIdx.x * WARPS + (threadIdx.x >> 5);
  if (krow >= (long long)p.B * p.hkv * p.Tk) return;
  const int j = (int)(krow % p.Tk);
  const int bhk = (int)(krow / p.Tk);
  const int g = bhk % p.hkv, batch = bhk / p.hkv;
  const int group = p.h / p.hkv;
  float k[KC], v[VC], dk[KC], dv[VC];
#pragma unroll
  for (int i = 0; i < KC; ++i) {
    k[i] = ldf(gk + krow * DK + lane + 32 * i);
    dk[i] = 0.f;
  }
#pragma unroll
  for (int i = 0; i < VC; ++i) {
    v[i] = ldf(gv + krow * DV + lane + 32 * i);
    dv[i] = 0.f;
  }
  for (int hi = 0; hi < group; ++hi) {
    const int head = g * group + hi;
    const int bh = batch * p.h + head;
    const float b = VARIANT == kYat ? p.b[head] : 0.f;
    const float eps = VARIANT != kSoftmax ? p.eps[head] : 0.f;
    const float tau = VARIANT == kStau ? p.tau[head] : 1.f;
    float g1 = 0.f, g2 = 0.f;
    for (int t = p.causal ? j : 0; t < p.Tq; ++t) {
      const long long row = (long long)bh * p.Tq + t;
      float q[KC], dout[VC];
      float a = 0.f, c = 0.f, e = 0.f;
      double a64 = 0.0;
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        q[i] = ldf(gq + row * DK + lane + 32 * i);
        if (VARIANT == kYat) {
          a64 = fma((double)q[i], (double)k[i], a64);
          e = fmaf(q[i] - k[i], q[i] - k[i], e);
        } else {
          a = fmaf(q[i], k[i], a);
        }
      }
#pragma unroll
      for (int i = 0; i < VC; ++i) {
        dout[i] = ldf(gdo + row * DV + lane + 32 * i);
        c = fmaf(dout[i], v[i], c);
      }
      const float dot = VARIANT == kYat ? (float)(warp_sum_d(a64) + (double)b) : warp_sum(a);
      const float dw = warp_sum(c);
      const float d2 = VARIANT == kYat ? warp_sum(e) : 0.f;
      const float Lt = VARIANT == kYat ? p.Dbuf[(long long)p.B * p.h * p.Tq + row]
                                       : p.row_mass[row];
      const Pair r = pair<VARIANT, YM>(dot, dw, d2, Lt, p.Dbuf[row], p.scale, b, eps, tau);
#pragma unroll
      for (int i = 0; i < KC; ++i) {
        dk[i] = fmaf(r.c, q[i], dk[i]);
        if (VARIANT == kYat) dk[i] = fmaf(2.f * r.e, k[i] - q[i], dk[i]);
      }
#pragma unroll
      for (int i = 0; i < VC; ++i) dv[i] = fmaf(r.w, dout[i], dv[i]);
      g1 += r.g1;
      g2 += r.g2;
    }
    if (VARIANT != kSoftmax && lane == 0) {
      atomicAdd(p.dpar + 2 * head, (double)g1);
      atomicAdd(p.dpar + 2 * head + 1, (double)g2);
    }
  }
#pragma unroll
  for (int i = 0; i < KC; ++i) stf(static_cast<T *>(p.dk) + krow * DK + lane + 32 * i, dk[i]);
#pragma unroll
  for (int i = 0; i < VC; ++i) stf(static_cast<T *>(p.dv) + krow * DV + lane + 32 * i, dv[i]);
}

template <int VARIANT, int DK, int DV, int YM, typename T>
cudaError_t launch(const BwdSimtParams &p, cudaStream_t s) {
  const long long qrows = (long long)p.B * p.h * p.Tq;
  const long long krows = (long long)p.B * p.hkv * p.Tk;
  if (qrows > 0)
    dq_kernel<VARIANT, DK, DV, YM, T>
        <<<(unsigned)((qrows + WARPS - 1) / WARPS), WARPS * 32, 0, s>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || krows <= 0) return e;
  dkv_kernel<VARIANT, DK, DV, YM, T>
      <<<(unsigned)((krows + WARPS - 1) / WARPS), WARPS * 32, 0, s>>>(p);
  return cudaGetLastError();
}

template <int DK, int DV, typename T>
cudaError_t launch_for(int variant, int yat_m, const BwdSimtParams &p, cudaStream_t s) {
  if (variant == kSoftmax) return launch<kSoftmax, DK, DV, 1, T>(p, s);
  if (variant == kStau) return launch<kStau, DK, DV, 1, T>(p, s);
  if (yat_m == 2) return launch<kYat, DK, DV, 2, T>(p, s);
  if (yat_m == 3) return launch<kYat, DK, DV, 3, T>(p, s);
  return launch<kYat, DK, DV, 1, T>(p, s);
}

template <typename T>
cudaError_t by_shape(int variant, int dk, int dv, int yat_m, const BwdSimtParams &p,
                     cudaStream_t s) {
  switch (dk * 1000 + dv) {
    case 32032: return launch_for<32, 32, T>(variant, yat_m, p, s);
    case 32064: return launch_for<32, 64, T>(variant, yat_m, p, s);
    case 32128: return launch_for<32, 128, T>(variant, yat_m, p, s);
    case 64032: return launch_for<64, 32, T>(variant, yat_m, p, s);
    case 64064: return launch_for<64, 64, T>(variant, yat_m, p, s);
    case 64128: return launch_for<64, 128, T>(variant, yat_m, p, s);
    case 128032: return launch_for<128, 32, T>(variant, yat_m, p, s);
    case 128064: return launch_for<128, 64, T>(variant, yat_m, p, s);
    case 128128: return launch_for<128, 128, T>(variant, yat_m, p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace bwds

cudaError_t launch_bwd_simt(int variant, bool bf16, int dk, int dv, int yat_m,
                            const BwdSimtParams &p, cudaStream_t s) {
  return bf16 ? bwds::by_shape<__nv_bfloat16>(variant, dk, dv, yat_m, p, s)
              : bwds::by_shape<float>(variant, dk, dv, yat_m, p, s);
}

}  // namespace cattn
