// norms.cu -- squared L2 norm of every row of a bf16 [BH, T, d] tensor.
//
// The Yat map needs |q - k|^2 for every score; it is assembled as
// |q|^2 + |k|^2 - 2 q.k from the dot products the scores already need
// ("Softmax-Free Attention in JAX/Flax NNX", section "One module, two
// compatibility functions").  This kernel supplies the key norms, in fp32
// from the stored bf16 values, and the largest of them (the forward uses it
// to check that products of two distances stay in the fp32 range).  It is
// bandwidth bound: d/8 threads share a row, each reading one 16-byte vector
// of it; every thread keeps ROWS such loads in flight before the shuffle
// reductions, and the grid strides over the rows with a few CTAs per SM.
#include <cuda_bf16.h>

#include "kernels.h"

namespace cattn {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 4;  // row groups per thread per pass

template <int G>  // threads per row = d / 8
__global__ void __launch_bounds__(kThreads) row_sqnorm_kernel(const uint4 *__restrict__ x,
                                                              float *__restrict__ out, int T,
                                                              int T_pad, long long n_out,
                                                              unsigned long long *__restrict__ max64,
                                                              unsigned int gen,
                                                              unsigned int *__restrict__ zero_words,
                                                              int n_zero) {
  if (blockIdx.x == 0 && threadIdx.x < n_zero) zero_words[threadIdx.x] = 0u;
  // One pass of a block covers SPAN consecutive output slots; T_pad is a
  // multiple of 128 >= SPAN, so a span never crosses from one head to the next.
  constexpr int RPB = kThreads / G;
  constexpr int SPAN = RPB * kRows;
  static_assert(128 % SPAN == 0, "a span stays inside one head");
  const int part = threadIdx.x % G;
  const int sub = threadIdx.x / G;
  float running_max = 0.f;
  for (long long base = (long long)blockIdx.x * SPAN; base < n_out;
       base += (long long)gridDim.x * SPAN) {
    const long long bh = base / T_pad;
    const int t0 = (int)(base - bh * T_pad);
    const uint4 *xh = x + bh * T * G;
    uint4 raw[kRows];
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const int t = t0 + i * RPB + sub;
      raw[i] = t < T ? __ldg(xh + (long long)t * G + part) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int i = 0; i < kRows; ++i) {
      const __nv_bfloat162 *h2 = reinterpret_cast<const __nv_bfloat162 *>(&raw[i]);
      float acc = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(h2[e]);
        acc = fmaf(f.x, f.x, acc);
        acc = fmaf(f.y, f.y, acc);
      }
#pragma unroll
      for (int o = G / 2; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
      if (part == 0) out[base + i * RPB + sub] = acc;  // padded rows get zero
      running_max = fmaxf(running_max, acc);
    }
  }
  // one update per CTA; non-negative floats order like their bit patterns
  __shared__ float warp_max[kThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    running_max = fmaxf(running_max, __shfl_xor_sync(0xffffffffu, running_max, o));
  if ((threadIdx.x & 31) == 0) warp_max[threadIdx.x >> 5] = running_max;
  __syncthreads();
  if (threadIdx.x == 0) {
    float m = warp_max[0];
#pragma unroll
    for (int w = 1; w < kThreads / 32; ++w) m = fmaxf(m, warp_max[w]);
    // a word of another generation (an earlier call's maximum, or whatever
    // the workspace held) is replaced; within this generation it only grows
    const unsigned long long mine = ((unsigned long long)gen << 32) | __float_as_uint(m);
    unsigned long long old = *reinterpret_cast<volatile unsigned long long *>(max64);
    while (!((unsigned)(old >> 32) == gen && old >= mine)) {
      const unsigned long long seen = atomicCAS(max64, old, mine);
      if (seen == old) break;
      old = seen;
    }
  }
}

}  // namespace

cudaError_t launch_row_sqnorm_bf16(const void *x, float *out, int BH, int T, int T_pad, int d,
                                   unsigned long long *max64, unsigned int gen,
                                   unsigned int *zero_words, int n_zero, cudaStream_t s) {
  const long long n_out = (long long)BH * T_pad;
  if (n_out == 0) return cudaSuccess;
  const int G = d / 8;
  if (G != 16 && G != 8) return cudaErrorInvalidValue;
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long per_block = (long long)(kThreads / G) * kRows;
  long long blocks = (n_out + per_block - 1) / per_block;
  if (blocks > 8LL * sms) blocks = 8LL * sms;
  const uint4 *xv = reinterpret_cast<const uint4 *>(x);
  if (G == 16)
    row_sqnorm_kernel<16><<<(unsigned)blocks, kThreads, 0, s>>>(xv, out, T, T_pad, n_out, max64, gen,
                                                                 zero_words, n_zero);
  else
    row_sqnorm_kernel<8><<<(unsigned)blocks, kThreads, 0, s>>>(xv, out, T, T_pad, n_out, max64, gen,
                                                                zero_words, n_zero);
  return cudaGetLastError();
}

}  // namespace cattn
