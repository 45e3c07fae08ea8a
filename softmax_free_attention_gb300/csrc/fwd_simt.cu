// fwd_simt.cu -- attention forward on the CUDA cores.
//
// bf16 inputs whose head widths the tensor-core kernel has no tiles for (any
// (dk, dv) in {32, 64, 128}^2 other than (64, 64), (128, 128), (128, 64))
// take this path, widened to fp32 on load and rounded to bf16 on store.
// (fp32 inputs run on the tensor cores as three-pass tf32, fwd_tf32.cu; the
// kernel here is instantiated for fp32 as well.)  One CTA holds 32 query rows of
// one (batch, head); 8 warps take 4 rows each.  Keys stream through shared
// memory 32 at a time; lane l owns key l of the tile for the score and owns
// value columns l, l+32, ... for the weighted sum.
//
// Maps (same definitions as the tensor-core path):
//   Yat      kappa = (q.k + b)^2 / (max(|q-k|^2, 0) + eps) on the raw q.k,
//            with |q-k|^2 summed directly; row mass kept in fp32, no max trick.
//   softmax  online softmax of s = scale * q.k (running max per key tile).
//   s^tau    online softmax of sigma = tau * ln(softplus(s) + eps), which is
//            phi^tau / sum phi^tau ("s^tau: a focal-length knob for attention",
//            the equivalence with softmax of tau log phi + C).
#include <cuda_bf16.h>

#include "kernels.h"

namespace cattn {
namespace simt {

__device__ __forceinline__ float ldf(const float *p) { return *p; }
__device__ __forceinline__ float ldf(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void stf(float *p, float v) { *p = v; }
__device__ __forceinline__ void stf(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

constexpr int ROWS = 32;  // query rows per CTA
constexpr int RPW = 4;    // rows per warp
constexpr int KT = 32;    // keys per tile
constexpr int THREADS = 256;
constexpr unsigned FULL = 0xffffffffu;

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
  return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, o));
  return v;
}

template <int DK, int DV>
struct Smem {
  static constexpr int Q = ROWS * DK;
  static constexpr int K = KT * (DK + 1);
  static constexpr int V = KT * DV;
  static constexpr int BYTES = (Q + K + V) * 4;
};

template <int VARIANT, int DK, int DV, typename T>
__global__ void __launch_bounds__(THREADS) fwd_kernel(const FwdParams p) {
  using S = Smem<DK, DV>;
  extern __shared__ float sm[];
  float *sq = sm;
  float *sk = sm + S::Q;
  float *sv = sk + S::K;
  constexpr int VC = DV / 32;  // value columns per lane

  const int bh = blockIdx.y;
  const int head = bh % p.h;
  const int batch = bh / p.h;
  const int bh_kv = batch * p.hkv + head / (p.h / p.hkv);
  const int row0 = blockIdx.x * ROWS;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const T *q = reinterpret_cast<const T *>(p.q) + (size_t)bh * p.Tq * DK;
  const T *k = reinterpret_cast<const T *>(p.k) + (size_t)bh_kv * p.Tk * DK;
  const T *v = reinterpret_cast<const T *>(p.v) + (size_t)bh_kv * p.Tk * DV;

  for (int i = threadIdx.x; i < ROWS * DK; i += THREADS) {
    const int r = i / DK, c = i - r * DK;
    sq[i] = (row0 + r < p.Tq) ? ldf(q + (size_t)(row0 + r) * DK + c) : 0.f;
  }

  float b = 0.f, eps = 0.f, tau = 1.f;
  if (VARIANT == kYat) {
    b = p.b[head];
    eps = p.eps[head];
  } else if (VARIANT == kStau) {
    eps = p.eps[head];
    tau = p.tau[head];
  }

  float m[RPW], l[RPW], top[RPW], acc[RPW][VC];
#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    m[rr] = -INFINITY;
    l[rr] = 0.f;
    top[rr] = -INFINITY;
#pragma unroll
    for (int c = 0; c < VC; ++c) acc[rr][c] = 0.f;
  }

  const int kend = p.causal ? min(p.Tk, row0 + ROWS) : p.Tk;
  for (int kt = 0; kt < kend; kt += KT) {
    __syncthreads();
    for (int i = threadIdx.x; i < KT * DK; i += THREADS) {
      const int r = i / DK, c = i - r * DK;
      sk[r * (DK + 1) + c] = (kt + r < p.Tk) ? ldf(k + (size_t)(kt + r) * DK + c) : 0.f;
    }
    for (int i = threadIdx.x; i < KT * DV; i += THREADS) {
      const int r = i / DV;
      sv[i] = (kt + r < p.Tk) ? ldf(v + (size_t)kt * DV + i) : 0.f;
    }
    __syncthreads();

#pragma unroll
    for (int rr = 0; rr < RPW; ++rr) {
      const int lr = warp * RPW + rr;
      const int row = row0 + lr;
      const int key = kt + lane;
      const bool allowed = key < p.Tk && (!p.causal || key <= row);
      const float *qr = sq + lr * DK;
      const float *kr = sk + lane * (DK + 1);
      float dot = 0.f, d2 = 0.f;
#pragma unroll 8
      for (int d = 0; d < DK; ++d) {
        const float a = qr[d], c = kr[d];
        dot = fmaf(a, c, dot);
        if (VARIANT == kYat) {
          const float diff = a - c;
          d2 = fmaf(diff, diff, d2);
        }
      }
      float w;  // this lane's key weight before normalisation
      if (VARIANT == kYat) {
        const float t = dot + b;
        float num = t * t;  // (dot + b)^{2m}
        const float t2 = num;
        for (int i = 1; i < p.yat_m; ++i) num *= t2;
        w = allowed ? num / (fmaxf(d2, 0.f) + eps) : 0.f;
        l[rr] += warp_sum(w);
        top[rr] = fmaxf(top[rr], warp_max(allowed ? w : -INFINITY));
      } else {
        const float s = dot * p.scale;
        float x;  // exponent of the weight
        if (VARIANT == kSoftmax) {
          x = s;
        } else {
          const float sp = fmaxf(s, 0.f) + log1pf(expf(-fabsf(s)));
          x = tau * logf(sp + eps);
        }
        x = allowed ? x : -INFINITY;
        top[rr] = fmaxf(top[rr], warp_max(allowed ? s : -INFINITY));
        const float tmax = warp_max(x);
        const float mn = fmaxf(m[rr], tmax);
        const float corr = (m[rr] == -INFINITY) ? 0.f : expf(m[rr] - mn);
        w = allowed ? expf(x - mn) : 0.f;
        l[rr] = l[rr] * corr + warp_sum(w);
#pragma unroll
        for (int c = 0; c < VC; ++c) acc[rr][c] *= corr;
        m[rr] = mn;
      }
      // acc[c] += sum_key w_key * v[key][lane + 32c]
#pragma unroll 8
      for (int kk = 0; kk < KT; ++kk) {
        const float wk = __shfl_sync(FULL, w, kk);
#pragma unroll
        for (int c = 0; c < VC; ++c) acc[rr][c] = fmaf(wk, sv[kk * DV + lane + 32 * c], acc[rr][c]);
      }
    }
  }

#pragma unroll
  for (int rr = 0; rr < RPW; ++rr) {
    const int row = row0 + warp * RPW + rr;
    if (row >= p.Tq) continue;
    const float inv = VARIANT == kYat ? 1.f / (l[rr] + 1e-9f) : 1.f / l[rr];
    T *orow = reinterpret_cast<T *>(p.out) + ((size_t)bh * p.Tq + row) * DV;
#pragma unroll
    for (int c = 0; c < VC; ++c) stf(orow + lane + 32 * c, acc[rr][c] * inv);
    if (lane == 0) {
      const size_t ti = (size_t)bh * p.Tq + row;
      if (p.row_mass) p.row_mass[ti] = VARIANT == kYat ? l[rr] : m[rr] + logf(l[rr]);
      if (p.row_max) p.row_max[ti] = top[rr];
    }
  }
}

template <int VARIANT, int DK, int DV, typename T>
cudaError_t launch(const FwdParams &p, cudaStream_t s) {
  auto kern = fwd_kernel<VARIANT, DK, DV, T>;
  constexpr int bytes = Smem<DK, DV>::BYTES;
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  dim3 grid((unsigned)((p.Tq + ROWS - 1) / ROWS), (unsigned)(p.B * p.h));
  if (grid.x == 0 || grid.y == 0) return cudaSuccess;
  kern<<<grid, THREADS, bytes, s>>>(p);
  return cudaGetLastError();
}

template <typename T, int V>
cudaError_t by_shape(int dk, int dv, const FwdParams &p, cudaStream_t s) {
  switch (dk * 1000 + dv) {
    case 32032: return launch<V, 32, 32, T>(p, s);
    case 32064: return launch<V, 32, 64, T>(p, s);
    case 32128: return launch<V, 32, 128, T>(p, s);
    case 64032: return launch<V, 64, 32, T>(p, s);
    case 64064: return launch<V, 64, 64, T>(p, s);
    case 64128: return launch<V, 64, 128, T>(p, s);
    case 128032: return launch<V, 128, 32, T>(p, s);
    case 128064: return launch<V, 128, 64, T>(p, s);
    case 128128: return launch<V, 128, 128, T>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename T>
cudaError_t by_variant(int variant, int dk, int dv, const FwdParams &p, cudaStream_t s) {
  if (variant == kSoftmax) return by_shape<T, kSoftmax>(dk, dv, p, s);
  if (variant == kYat) return by_shape<T, kYat>(dk, dv, p, s);
  return by_shape<T, kStau>(dk, dv, p, s);
}

}  // namespace simt

bool fwd_simt_supported(int dk, int dv) {
  auto ok = [](int d) { return d == 32 || d == 64 || d == 128; };
  return ok(dk) && ok(dv);
}

cudaError_t launch_fwd_simt(int variant, bool bf16, int dk, int dv, const FwdParams &p,
                            cudaStream_t s) {
  return bf16 ? simt::by_variant<__nv_bfloat16>(variant, dk, dv, p, s)
              : simt::by_variant<float>(variant, dk, dv, p, s);
}

}  // namespace cattn
