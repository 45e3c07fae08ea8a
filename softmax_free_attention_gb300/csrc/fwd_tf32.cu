// fwd_tf32.cu -- attention forward for fp32 inputs on the sm_103a tensor cores.
//
// Both contractions run as tcgen05.mma kind::tf32 in three passes.  Every
// fp32 operand x is split as x = hi + lo, hi = x rounded to the 10-bit tf32
// significand and lo = x - hi (exact in fp32); the tensor core reads lo at
// tf32 precision too, so hi*hi + hi*lo + lo*hi carries each product to about
// 2^-20 of its size (the dropped lo*lo term is below 2^-22), against 2^-11
// for a single tf32 pass.  That keeps the output within the fp32 target of
// 1e-4 max|v|.
//
//   split pass   q, k -> (hi, lo) arrays; v -> its transpose (hi, lo), keys
//                contiguous, so that every MMA operand is K-major; Yat: |k|^2
//                of the fp32 keys (accumulated in fp64)
//   S  = Qh Kh^T + Qh Kl^T + Ql Kh^T   A, B from shared memory -> TMEM fp32
//   P  = map(S)                         four map warps, one query row each,
//                                       the whole 32-key tile per thread;
//                                       P written to TMEM as (hi, lo)
//   O += Ph Vh + Ph Vl + Pl Vh          A = P from TMEM, B = V^T from shared
//                                       memory -> TMEM fp32
//
// The maps are those of the bf16 path ("Softmax-Free Attention in JAX/Flax
// NNX", section "One module, two compatibility functions"; "s^tau: a
// focal-length knob for attention", core formula), in fp32 with the accurate
// math library functions: Yat kappa = (q.k + b)^{2m} / max(|q|^2 + |k|^2 -
// 2 q.k + eps, eps) with a plain row mass and the near-key guard of the bf16
// path (a row whose max kappa passes yat_near_threshold is recomputed by the
// plain definition afterwards); softmax and s^tau with a running max (exact
// rescale of O and l whenever the max grows).
//
// One CTA per (batch * head, 128-row query tile), 160 threads: warps 0-3 map
// (thread r = query row r of the tile = TMEM lane r), warp 4 lane 0 issues the
// TMA loads and the MMAs.  The pipeline is serial per key tile of 32 keys: S
// MMAs, map, PV MMAs; the next key tile's K is loaded once S is done and its
// V once PV is done, so the loads overlap the map and the other MMA.  Every
// mbarrier wait is bounded (2 s of %globaltimer); on expiry the kernel records
// a site code, raises a CTA-wide abort flag, and every role leaves its loop
// (copies in flight landed first, tensor memory released).
#include <cuda_bf16.h>

#include "kernels.h"
#include "maps.cuh"
#include "ptx.cuh"

namespace cattn {

__device__ unsigned int g_status_tf32;

namespace tf32 {

constexpr int BM = 128;  // query rows per CTA
constexpr int BN = 32;   // keys per tile
constexpr int THREADS = 160;
constexpr int MAP_THREADS = 128;
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr unsigned FULL = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

// TMEM columns: S [0, 32), P hi [32, 64), P lo [64, 96), O [128, 128 + dv)
constexpr uint32_t TM_S = 0, TM_PH = 32, TM_PL = 64, TM_O = 128;

// x rounded to nearest (ties to even) at the tf32 significand (10 bits
// after the point): the "hi" part, exactly representable in tf32.
__device__ __forceinline__ float tf32_hi(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0xfffu + ((u >> 13) & 1u);
  u &= 0xffffe000u;
  return __uint_as_float(u);
}

// D (+)= A[smem] B[smem], kind::tf32
__device__ __forceinline__ void mma_ss_tf32(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D (+)= A[tmem] B[smem], kind::tf32
__device__ __forceinline__ void mma_ts_tf32(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                            uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// Instruction descriptor, kind::tf32: fp32 D, tf32 A and B, both K-major.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N) {
  return (1u << 4)                       // D format: f32
         | (2u << 7)                     // A format: tf32
         | (2u << 10)                    // B format: tf32
         | ((uint32_t)(N >> 3) << 17)    // N / 8
         | ((uint32_t)(M >> 4) << 24);   // M / 16
}

template <int DK, int DV>
struct Layout {
  static constexpr int Q_BYTES = BM * DK * 4;   // DK/32 boxes of 128 rows x 128 B
  static constexpr int K_BYTES = BN * DK * 4;   // DK/32 boxes of 32 rows x 128 B
  static constexpr int V_BYTES = DV * BN * 4;   // one box of DV rows x 128 B
  static constexpr int OFF_QH = 0;
  static constexpr int OFF_QL = OFF_QH + Q_BYTES;
  static constexpr int OFF_KH = OFF_QL + Q_BYTES;
  static constexpr int OFF_KL = OFF_KH + K_BYTES;
  static constexpr int OFF_VH = OFF_KL + K_BYTES;
  static constexpr int OFF_VL = OFF_VH + V_BYTES;
  static constexpr int OFF_BAR = OFF_VL + V_BYTES;
  // q_full, k_full, v_full, s_full, s_free, p_full, pv_done, k_free, drain
  static constexpr int NBAR = 9;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;  // TMEM base, abort flag
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(K_BYTES % 1024 == 0 && V_BYTES % 1024 == 0, "swizzle atoms stay 1024-B aligned");
};

__device__ __forceinline__ bool bwait(uint32_t bar, uint32_t parity, volatile int *abort,
                                      unsigned site, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((honor_abort && *abort != 0) || (globaltimer_ns() - t0 > WAIT_LIMIT_NS)) {
      atomicCAS(&g_status_tf32, 0u, site | 1u);
      *abort = 1;
      return false;
    }
  }
}

// Warp-collective form (every lane polls, the decision is warp-uniform).
__device__ __forceinline__ bool bwait_warp(uint32_t bar, uint32_t parity, volatile int *abort,
                                           unsigned site) {
  if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
    const int bad = (*abort != 0) || (globaltimer_ns() - t0 > WAIT_LIMIT_NS);
    if (__any_sync(FULL, bad)) {
      if ((threadIdx.x & 31) == 0) {
        atomicCAS(&g_status_tf32, 0u, site | 1u);
        *abort = 1;
      }
      return false;
    }
  }
}

template <int VARIANT, int DK, int DV, int YM>
__global__ void __launch_bounds__(THREADS, 1)
    fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_qh,
               const __grid_constant__ CUtensorMap tm_ql, const __grid_constant__ CUtensorMap tm_kh,
               const __grid_constant__ CUtensorMap tm_kl, const __grid_constant__ CUtensorMap tm_vh,
               const __grid_constant__ CUtensorMap tm_vl) {
  using L = Layout<DK, DV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const uint32_t bar_q_full = sb + L::OFF_BAR, bar_k_full = bar_q_full + 8,
                 bar_v_full = bar_q_full + 16, bar_s_full = bar_q_full + 24,
                 bar_s_free = bar_q_full + 32, bar_p_full = bar_q_full + 40,
                 bar_pv_done = bar_q_full + 48, bar_k_free = bar_q_full + 56,
                 bar_drain = bar_q_full + 64;
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  const int bh = blockIdx.y;
  const int head = bh % p.h, batch = bh / p.h;
  const int bh_kv = batch * p.hkv + head / (p.h / p.hkv);
  const int row0 = blockIdx.x * BM;
  // key tiles this query tile needs
  const int kend = p.causal ? min(p.Tk, row0 + BM) : p.Tk;
  const int n_kt = (kend + BN - 1) / BN;

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    mbar_init(bar_k_full, 1);
    mbar_init(bar_v_full, 1);
    mbar_init(bar_s_full, 1);
    mbar_init(bar_s_free, MAP_THREADS);
    mbar_init(bar_p_full, MAP_THREADS);
    mbar_init(bar_pv_done, 1);
    mbar_init(bar_k_free, 1);
    mbar_init(bar_drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == 4) {
    tmem_alloc(smem_u32(tmem_holder), 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == 4) {
    // ------------------------------------------------------------ loads and MMAs
    if (lane == 0) {
      tma_prefetch_desc(&tm_qh);
      tma_prefetch_desc(&tm_kh);
      tma_prefetch_desc(&tm_vh);
      constexpr uint32_t IDS = idesc_tf32(BM, BN), IDO = idesc_tf32(BM, DV);
      uint32_t k_loads = 0, v_loads = 0;  // copies started (for the drain)
      auto load_k = [&](int j) {
        mbar_arrive_expect_tx(bar_k_full, 2u * (uint32_t)L::K_BYTES);
#pragma unroll
        for (int c = 0; c < DK / 32; ++c) {
          tma_load_3d(sb + L::OFF_KH + c * BN * 128, &tm_kh, 32 * c, j * BN, bh_kv, bar_k_full);
          tma_load_3d(sb + L::OFF_KL + c * BN * 128, &tm_kl, 32 * c, j * BN, bh_kv, bar_k_full);
        }
        ++k_loads;
      };
      auto load_v = [&](int j) {
        mbar_arrive_expect_tx(bar_v_full, 2u * (uint32_t)L::V_BYTES);
        tma_load_3d(sb + L::OFF_VH, &tm_vh, j * BN, 0, bh_kv, bar_v_full);
        tma_load_3d(sb + L::OFF_VL, &tm_vl, j * BN, 0, bh_kv, bar_v_full);
        ++v_loads;
      };
      mbar_arrive_expect_tx(bar_q_full, 2u * (uint32_t)L::Q_BYTES);
#pragma unroll
      for (int c = 0; c < DK / 32; ++c) {
        tma_load_3d(sb + L::OFF_QH + c * BM * 128, &tm_qh, 32 * c, row0, bh, bar_q_full);
        tma_load_3d(sb + L::OFF_QL + c * BM * 128, &tm_ql, 32 * c, row0, bh, bar_q_full);
      }
      if (n_kt > 0) {
        load_k(0);
        load_v(0);
      }
      const uint64_t dqh = smem_desc_sw128(sb + L::OFF_QH, 16, 1024);
      const uint64_t dql = smem_desc_sw128(sb + L::OFF_QL, 16, 1024);
      const uint64_t dkh = smem_desc_sw128(sb + L::OFF_KH, 16, 1024);
      const uint64_t dkl = smem_desc_sw128(sb + L::OFF_KL, 16, 1024);
      const uint64_t dvh = smem_desc_sw128(sb + L::OFF_VH, 16, 1024);
      const uint64_t dvl = smem_desc_sw128(sb + L::OFF_VL, 16, 1024);
      bool ok = bwait(bar_q_full, 0, abort, 0x10);
      for (int j = 0; ok && j < n_kt; ++j) {
        const uint32_t ph = (uint32_t)j & 1u;
        if (!(ok = bwait(bar_k_full, ph, abort, 0x20))) break;
        if (j > 0 && !(ok = bwait(bar_s_free, ph ^ 1u, abort, 0x30))) break;
        tc_fence_after();
        // S = Qh Kh^T + Qh Kl^T + Ql Kh^T; 8-element k steps, 32-element boxes
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
          const uint64_t da = pass == 2 ? dql : dqh, db = pass == 1 ? dkl : dkh;
#pragma unroll
          for (int kk = 0; kk < DK / 8; ++kk) {
            const uint64_t ao = (uint64_t)(((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4);
            const uint64_t bo = (uint64_t)(((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4);
            mma_ss_tf32(tmem + TM_S, da + ao, db + bo, IDS, (pass > 0 || kk > 0) ? 1u : 0u);
          }
        }
        mma_commit(bar_s_full);
        mma_commit(bar_k_free);
        // the K tile has been read once S is done: bring in the next one
        if (!(ok = bwait(bar_k_free, ph, abort, 0x40))) break;
        if (j + 1 < n_kt) load_k(j + 1);
        if (!(ok = bwait(bar_p_full, ph, abort, 0x50))) break;
        if (!(ok = bwait(bar_v_full, ph, abort, 0x60))) break;
        tc_fence_after();
        // O += Ph Vh + Ph Vl + Pl Vh; A = P (32 keys) from TMEM, 8 columns per k step
#pragma unroll
        for (int pass = 0; pass < 3; ++pass) {
          const uint32_t pa = tmem + (pass == 2 ? TM_PL : TM_PH);
          const uint64_t db = pass == 1 ? dvl : dvh;
#pragma unroll
          for (int kk = 0; kk < BN / 8; ++kk)
            mma_ts_tf32(tmem + TM_O, pa + (uint32_t)kk * 8, db + (uint64_t)((kk * 32) >> 4), IDO,
                        (j > 0 || pass > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(bar_pv_done);
        // P and the V tile have been read once PV is done
        if (!(ok = bwait(bar_pv_done, ph, abort, 0x70))) break;
        if (j + 1 < n_kt) load_v(j + 1);
      }
      // every MMA issued has completed once `drain` flips (this wait ignores
      // the abort flag), and every copy started has landed
      mma_commit(bar_drain);
      bwait(bar_drain, 0, abort, 0x80, false);
      bwait(bar_q_full, 0, abort, 0x90, false);
      if (k_loads > 0) bwait(bar_k_full, (k_loads - 1u) & 1u, abort, 0x90, false);
      if (v_loads > 0) bwait(bar_v_full, (v_loads - 1u) & 1u, abort, 0x90, false);
    }
  } else {
    // ------------------------------------------------------------ map warps
    const int r = threadIdx.x;  // row of the tile == TMEM lane
    const int row = row0 + r;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const uint32_t t_s = tmem + lane_off + TM_S, t_ph = tmem + lane_off + TM_PH,
                   t_pl = tmem + lane_off + TM_PL, t_o = tmem + lane_off + TM_O;
    float yb = 0.f, yeps = 0.f, tau = 1.f, seps = 0.f, nq = 0.f;
    if (VARIANT == kYat) {
      yb = p.b[head];
      yeps = p.eps[head];
      if (row < p.Tq) {  // |q|^2 of this row in fp64, from the stored fp32 values
        const float *qr = static_cast<const float *>(p.q) + ((size_t)bh * p.Tq + row) * DK;
        double s = 0.0;
        for (int d = 0; d < DK; ++d) s = fma((double)qr[d], (double)qr[d], s);
        nq = (float)s;
      }
    } else if (VARIANT == kStau) {
      tau = p.tau[head];
      seps = p.eps[head];
    }
    const float qe = nq + yeps;
    const float *nk = p.nk + (size_t)bh_kv * p.Tk_pad;
    float m = -INFINITY;  // softmax / s^tau: running max, log2 units
    float l = 0.f;        // Yat: mass; else the sum of 2^(x - m)
    float top = VARIANT == kYat ? 0.f : -INFINITY;  // Yat: max kappa; else max scaled score
    bool ok = true;
    for (int j = 0; j < n_kt; ++j) {
      const uint32_t ph = (uint32_t)j & 1u;
      if (!(ok = bwait_warp(bar_s_full, ph, abort, 0x100))) break;
      tc_fence_after();
      uint32_t sr[32];
      tmem_ld32(t_s, sr);
      tmem_wait_ld();
      tmem_ld_fence(sr);
      tc_fence_before();
      mbar_arrive(bar_s_free);  // S read: the next S may land
      float w[32];
      float corr = 1.f;
      bool rescale = false;
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int key = j * BN + i;
        const bool allowed = key < p.Tk && (!p.causal || key <= row);
        const float dot = __uint_as_float(sr[i]);
        if (VARIANT == kYat) {
          const float t = dot + yb;
          float num = t * t;
          if (YM == 2) num = num * num;
          if (YM == 3) num = num * num * num;
          const float den = fmaxf(fmaf(-2.f, dot, qe + (allowed ? nk[key] : 0.f)), yeps);
          w[i] = allowed ? num / den : 0.f;
          l += w[i];
          top = fmaxf(top, w[i]);
        } else {
          const float s = dot * p.scale;
          float x;
          if (VARIANT == kSoftmax) {
            x = s * LOG2E;
          } else {
            const float sp = fmaxf(s, 0.f) + log1pf(exp2f(-fabsf(s) * LOG2E));
            x = tau * log2f(sp + seps);
          }
          w[i] = allowed ? x : -INFINITY;
          if (allowed) top = fmaxf(top, s);
        }
      }
      if (VARIANT != kYat) {
        float mt = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) mt = fmaxf(mt, w[i]);
        const float mn = fmaxf(m, mt);
        if (mn > m) {
          corr = m == -INFINITY ? 0.f : exp2f(m - mn);
          rescale = j > 0 && m != -INFINITY;
          l *= corr;
          m = mn;
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          w[i] = w[i] == -INFINITY ? 0.f : exp2f(w[i] - m);
          l += w[i];
        }
      }
      // PV of the previous tile has read P and updated O
      if (j > 0 && !(ok = bwait_warp(bar_pv_done, ph ^ 1u, abort, 0x110))) break;
      tc_fence_after();
      // tcgen05.ld / st are warp-collective: the warp rescales together when
      // any of its rows needs it (the others multiply by 1)
      if (__any_sync(FULL, rescale)) {
        if (!rescale) corr = 1.f;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          tmem_wait_ld();
          tmem_ld_fence(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * corr);
          tmem_st32(t_o + c * 32, o);
        }
      }
      uint32_t hi[32], lo[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float h = tf32_hi(w[i]);
        hi[i] = __float_as_uint(h);
        lo[i] = __float_as_uint(w[i] - h);
      }
      tmem_st32(t_ph, hi);
      tmem_st32(t_pl, lo);
      tmem_wait_st();
      tc_fence_before();
      mbar_arrive(bar_p_full);
    }
    if (ok && n_kt > 0) {
      ok = bwait_warp(bar_pv_done, (uint32_t)(n_kt - 1) & 1u, abort, 0x120);
      tc_fence_after();
    }
    if (ok) {  // warp-uniform: the TMEM loads below are collective
      const bool row_ok = row < p.Tq;
      const float inv = VARIANT == kYat ? 1.f / (l + 1e-9f) : 1.f / l;
      float *orow = static_cast<float *>(p.out) + ((size_t)bh * p.Tq + (row_ok ? row : 0)) * DV;
#pragma unroll
      for (int c = 0; c < DV / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_o + c * 32, o);
        tmem_wait_ld();
        tmem_ld_fence(o);
        float4 *dst = reinterpret_cast<float4 *>(orow + c * 32);
        if (row_ok) {
#pragma unroll
          for (int i = 0; i < 8; ++i)
            dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv, __uint_as_float(o[4 * i + 1]) * inv,
                                 __uint_as_float(o[4 * i + 2]) * inv,
                                 __uint_as_float(o[4 * i + 3]) * inv);
        }
      }
    }
    if (ok && row < p.Tq) {
      const size_t ti = (size_t)bh * p.Tq + row;
      if (p.row_mass) p.row_mass[ti] = VARIANT == kYat ? l : (m + log2f(l)) * LN2;
      if (p.row_max) p.row_max[ti] = top;
      if (VARIANT == kYat && top > tc::yat_near_threshold(nq, yb, YM)) {
        // a key may sit close enough to q for the assembled distance to have
        // cancelled: the near-key pass recomputes this row
        const unsigned slot = atomicAdd(p.near_count, 1u);
        if (slot < p.near_cap) p.near_rows[slot] = make_uint2((unsigned)bh, (unsigned)row);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tmem, 256);
  }
}

// ---------------------------------------------------------------- split pass

// One launch prepares every operand of the fp32 forward.  Blocks [0, nb_e)
// split q then k element by element (hi, lo in the input's layout); blocks
// [nb_e, nb_e + nb_v) each transpose one 32 keys x 32 columns tile of v into
// v^T hi / lo [BHkv, dv, Tk_pad] (keys contiguous, zero past Tk) through
// shared memory; the remaining blocks (Yat) take |k|^2 of 256 key rows each
// (fp64 accumulation, rounded once; zero for padded rows).  Block 0 also
// zeroes the near-key count the forward appends to.
struct PrepArgs {
  const float *q, *k, *v;
  Tf32Split w;
  unsigned int *near_count;
  size_t nq, nk;          // elements of q and of k
  int nb_e, nb_v;         // blocks of the element split and of the transpose
  int tiles_k, tiles_c;   // transpose tiles per (bh_kv) along keys and columns
  int BHkv, Tk, Tk_pad, dk, dv;
};

__global__ void __launch_bounds__(256) prep_kernel(const __grid_constant__ PrepArgs a) {
  __shared__ float tile[32][33];
  const int blk = blockIdx.x;
  if (blk == 0 && threadIdx.x == 0 && a.near_count) *a.near_count = 0u;
  if (blk < a.nb_e) {
    const size_t n = a.nq + a.nk;
    for (size_t i = (size_t)blk * 256 + threadIdx.x; i < n; i += (size_t)a.nb_e * 256) {
      const bool isq = i < a.nq;
      const size_t j = isq ? i : i - a.nq;
      const float x = isq ? a.q[j] : a.k[j], h = tf32_hi(x);
      (isq ? a.w.qh : a.w.kh)[j] = h;
      (isq ? a.w.ql : a.w.kl)[j] = x - h;
    }
    return;
  }
  if (blk < a.nb_e + a.nb_v) {
    int t = blk - a.nb_e;
    const int tk = t % a.tiles_k;
    t /= a.tiles_k;
    const int tc = t % a.tiles_c;
    const int bhkv = t / a.tiles_c;
    const int k0 = tk * 32, c0 = tc * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;  // 32 x 8
    const float *vb = a.v + (size_t)bhkv * a.Tk * a.dv;
    for (int i = ty; i < 32; i += 8) {
      const int key = k0 + i, col = c0 + tx;
      tile[i][tx] = (key < a.Tk && col < a.dv) ? vb[(size_t)key * a.dv + col] : 0.f;
    }
    __syncthreads();
    for (int i = ty; i < 32; i += 8) {
      const int col = c0 + i, key = k0 + tx;
      if (col < a.dv && key < a.Tk_pad) {
        const float val = tile[tx][i], h = tf32_hi(val);
        const size_t o = ((size_t)bhkv * a.dv + col) * a.Tk_pad + key;
        a.w.vth[o] = h;
        a.w.vtl[o] = val - h;
      }
    }
    return;
  }
  const int i = (blk - a.nb_e - a.nb_v) * 256 + threadIdx.x;
  if (i >= a.BHkv * a.Tk_pad) return;
  const int bhkv = i / a.Tk_pad, t = i - bhkv * a.Tk_pad;
  if (t >= a.Tk) {
    a.w.nk[i] = 0.f;
    return;
  }
  const float *kr = a.k + ((size_t)bhkv * a.Tk + t) * a.dk;
  double s = 0.0;
  for (int c = 0; c < a.dk; ++c) s = fma((double)kr[c], (double)kr[c], s);
  a.w.nk[i] = (float)s;
}

template <int VARIANT, int DK, int DV, int YM>
cudaError_t launch(const FwdParams &p, const Tf32Maps &m, cudaStream_t s) {
  using L = Layout<DK, DV>;
  auto kern = fwd_kernel<VARIANT, DK, DV, YM>;
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  dim3 grid((unsigned)((p.Tq + BM - 1) / BM), (unsigned)(p.B * p.h));
  kern<<<grid, THREADS, L::ALLOC, s>>>(p, m.qh, m.ql, m.kh, m.kl, m.vh, m.vl);
  return cudaGetLastError();
}

template <int VARIANT, int YM>
cudaError_t by_shape(int dk, int dv, const FwdParams &p, const Tf32Maps &m, cudaStream_t s) {
  switch (dk * 1000 + dv) {
    case 32032: return launch<VARIANT, 32, 32, YM>(p, m, s);
    case 32064: return launch<VARIANT, 32, 64, YM>(p, m, s);
    case 32128: return launch<VARIANT, 32, 128, YM>(p, m, s);
    case 64032: return launch<VARIANT, 64, 32, YM>(p, m, s);
    case 64064: return launch<VARIANT, 64, 64, YM>(p, m, s);
    case 64128: return launch<VARIANT, 64, 128, YM>(p, m, s);
    case 128032: return launch<VARIANT, 128, 32, YM>(p, m, s);
    case 128064: return launch<VARIANT, 128, 64, YM>(p, m, s);
    case 128128: return launch<VARIANT, 128, 128, YM>(p, m, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace tf32

cudaError_t launch_split_tf32(const FwdParams &p, const Tf32Split &w, int variant, int dk,
                              int dv, cudaStream_t s) {
  tf32::PrepArgs a;
  a.q = static_cast<const float *>(p.q);
  a.k = static_cast<const float *>(p.k);
  a.v = static_cast<const float *>(p.v);
  a.w = w;
  a.near_count = variant == kYat ? p.near_count : nullptr;
  a.nq = (size_t)p.B * p.h * p.Tq * dk;
  a.nk = (size_t)p.B * p.hkv * p.Tk * dk;
  const size_t ne = a.nq + a.nk;
  a.nb_e = (int)((ne + 255) / 256 < 2048 ? (ne + 255) / 256 : 2048);
  if (a.nb_e < 1) a.nb_e = 1;
  a.BHkv = p.B * p.hkv;
  a.Tk = p.Tk;
  a.Tk_pad = p.Tk_pad;
  a.dk = dk;
  a.dv = dv;
  a.tiles_k = (p.Tk_pad + 31) / 32;
  a.tiles_c = (dv + 31) / 32;
  a.nb_v = a.BHkv * a.tiles_k * a.tiles_c;
  const int nb_n = variant == kYat ? (a.BHkv * p.Tk_pad + 255) / 256 : 0;
  const long long blocks = (long long)a.nb_e + a.nb_v + nb_n;
  if (blocks <= 0) return cudaSuccess;
  tf32::prep_kernel<<<(unsigned)blocks, 256, 0, s>>>(a);
  return cudaGetLastError();
}

cudaError_t launch_fwd_tf32(int variant, int dk, int dv, const FwdParams &p, const Tf32Maps &m,
                            cudaStream_t s) {
  if (p.B * p.h == 0 || p.Tq == 0) return cudaSuccess;
  if (variant == kSoftmax) return tf32::by_shape<kSoftmax, 1>(dk, dv, p, m, s);
  if (variant == kStau) return tf32::by_shape<kStau, 1>(dk, dv, p, m, s);
  switch (p.yat_m) {
    case 2: return tf32::by_shape<kYat, 2>(dk, dv, p, m, s);
    case 3: return tf32::by_shape<kYat, 3>(dk, dv, p, m, s);
    default: return tf32::by_shape<kYat, 1>(dk, dv, p, m, s);
  }
}

cudaError_t read_and_clear_tf32_status(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status_tf32, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status_tf32, &zero, sizeof(unsigned int));
}

}  // namespace cattn
