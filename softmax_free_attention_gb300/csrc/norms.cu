// norms.cu -- squared L2 norm of every row of a bf16 [BH, T, d] tensor.
//
// The Yat map needs |q - k|^2 for every score; it is assembled as
// |q|^2 + |k|^2 - 2 q.k from the dot products the scores already need
// ("Softmax-Free Attention in JAX/Flax NNX", section "One module, two
// compatibility functions").  This kernel supplies the two norm vectors, in
// fp32 from the stored bf16 values.  It is bandwidth bound: d/8 threads share
// a row, each reading one 16-byte vector, then a shuffle reduction.
#include <cuda_bf16.h>

#include "kernels.h"

namespace cattn {
namespace {

template <int G>  // threads per row = d / 8
__global__ void __launch_bounds__(256) row_sqnorm_kernel(const uint4 *__restrict__ x,
                                                         float *__restrict__ out, int T, int T_pad,
                                                         long long n_out) {
  const long long gtid = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  const long long slot = gtid / G;
  const int part = (int)(gtid % G);
  float acc = 0.f;
  if (slot < n_out) {
    const long long bh = slot / T_pad;
    const int t = (int)(slot - bh * T_pad);
    if (t < T) {
      const uint4 raw = __ldg(x + (bh * T + t) * G + part);
      const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float2 f = __bfloat1622float2(h2[i]);
        acc = fmaf(f.x, f.x, acc);
        acc = fmaf(f.y, f.y, acc);
      }
    }
  }
#pragma unroll
  for (int o = G / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (part == 0 && slot < n_out) out[slot] = acc;
}

}  // namespace

cudaError_t launch_row_sqnorm_bf16(const void *x, float *out, int BH, int T, int T_pad, int d,
                                   cudaStream_t s) {
  const long long n_out = (long long)BH * T_pad;
  if (n_out == 0) return cudaSuccess;
  const int G = d / 8;
  const long long threads = n_out * G;
  const unsigned blocks = (unsigned)((threads + 255) / 256);
  const uint4 *xv = reinterpret_cast<const uint4 *>(x);
  if (G == 16)
    row_sqnorm_kernel<16><<<blocks, 256, 0, s>>>(xv, out, T, T_pad, n_out);
  else if (G == 8)
    row_sqnorm_kernel<8><<<blocks, 256, 0, s>>>(xv, out, T, T_pad, n_out);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace cattn
