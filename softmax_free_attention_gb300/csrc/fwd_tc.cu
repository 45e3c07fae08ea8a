// fwd_tc.cu -- fused attention forward on the sm_103a tensor cores.
//
// One CTA owns two 128-row query tiles (Q0, Q1) of one (batch, head) and
// streams 128-key K/V tiles through shared memory.  Per KV tile j:
//
//   S_x = Q_x K_j^T          tcgen05.mma (A, B from smem)  -> TMEM, fp32
//   P_x = map(S_x)           epilogue warpgroup x: tcgen05.ld S, apply the
//                            score-to-weight map, tcgen05.st P (bf16) over S
//   O_x += P_x V_j           tcgen05.mma (A = P from TMEM, B = V from smem)
//
// The maps ("Softmax-Free Attention in JAX/Flax NNX", section "One module,
// two compatibility functions"; "s^tau: a focal-length knob for attention",
// core formula):
//   Yat      kappa = (q.k + b)^2 / (max(|q|^2 + |k|^2 - 2 q.k, 0) + eps), the
//            distance assembled from the same dot products as the score; a
//            plain fp32 row mass, no running max and no rescale of O.
//   softmax  exp2((s - m) log2 e) with a running max m; O and l rescaled only
//            when m grows by more than 2^8 (the stale m stays exact because
//            l and O share it).
//   s^tau    exp2(tau log2 phi(s) - m) with phi = softplus(s) + eps and m the
//            running max of tau log2 phi, taken from the max raw score since
//            phi is increasing.
//
// Warp roles (320 threads): warps 0-3 epilogue for Q0, warps 4-7 epilogue
// for Q1 (one query row per thread = one TMEM lane), warp 8 TMA producer,
// warp 9 TMEM allocation + MMA issue (lane 0).  K and V tiles share one ring
// of shared-memory slots guarded by full/empty mbarriers; the squared key
// norms of the Yat map ride in a small ring of their own.
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,256+dv) O1 [384,384+dv).
// P_x is written over the first 64 columns of S_x; the MMA pipe executes a
// CTA's MMAs in issue order, so PV_x(j) reads P_x before S_x(j+1) lands.
//
// Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the kernel
// records a site code in g_status, raises a CTA-wide abort flag, and all roles
// leave their loops so that TMEM is still released.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace cattn {

__device__ unsigned int g_status;

namespace tc {

constexpr int BM = 128;  // query rows per tile
constexpr int BN = 128;  // keys per tile
constexpr int NUM_THREADS = 320;
constexpr int PRODUCER_WARP = 8;
constexpr int MMA_WARP = 9;
constexpr int NKS = 4;  // stages of the key-norm ring
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr unsigned FULL = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

// wait-site codes recorded in g_status
enum : unsigned {
  SITE_PRODUCER = 0x100,
  SITE_MMA = 0x200,
  SITE_EPI = 0x300,
  SITE_FINAL = 0x400,
};

template <int DK, int DV>
struct Layout {
  static constexpr int Q_TILE = BM * DK * 2;
  static constexpr int K_TILE = BN * DK * 2;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int SLOT = K_TILE > V_TILE ? K_TILE : V_TILE;
  static constexpr int NS = (DK == 64 && DV == 64) ? 6 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + 2 * Q_TILE;
  static constexpr int OFF_NK = OFF_RING + NS * SLOT;
  static constexpr int OFF_BAR = OFF_NK + NKS * BN * 4;
  // q_full, kv_full[NS], kv_empty[NS], nk_full[NKS], nk_empty[NKS],
  // s_full[2], p_full[2], o_full[2], drain
  static constexpr int NBAR = 1 + 2 * NS + 2 * NKS + 7;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
};

// Warp-collective bounded wait.  Every lane polls (so every lane acquires the
// phase), the exit decision is warp-uniform.  Returns false on timeout/abort.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned site, bool honor_abort = true) {
  if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
    if ((it & 63u) == 0) {
      const int bad =
          (honor_abort && *abort != 0) || (globaltimer_ns() - t0 > WAIT_LIMIT_NS);
      if (__any_sync(FULL, bad)) {
        if ((threadIdx.x & 31) == 0) {
          atomicCAS(&g_status, 0u, site | 1u);
          *abort = 1;
        }
        return false;
      }
    }
  }
}

template <int DK>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false);
#pragma unroll
  for (int kk = 0; kk < DK / 16; ++kk) {
    // 64-column boxes of 128 rows x 128 B; 16-element k steps are 32 B apart
    const uint32_t off = (uint32_t)(kk >> 2) * (BM * 128) + (uint32_t)(kk & 3) * 32;
    mma_ss(d_tmem, smem_desc_sw128(q_smem + off, 16, 1024), smem_desc_sw128(k_smem + off, 16, 1024),
           IDESC, kk > 0 ? 1u : 0u);
  }
}

template <int DV>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, DV, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    // V is N-major: 16 keys = 16 rows of 128 B; 64-wide dv boxes are BN*128 B apart
    mma_ts(d_tmem, p_tmem + (uint32_t)kk * 8, smem_desc_sw128(v_smem + (uint32_t)kk * 2048, BN * 128, 1024),
           IDESC, (accumulate || kk > 0) ? 1u : 0u);
  }
}

template <int DV>
__device__ __forceinline__ void scale_o_tmem(uint32_t t_o, float f) {
#pragma unroll
  for (int c = 0; c < DV / 32; ++c) {
    uint32_t r[32];
    tmem_ld32(t_o + c * 32, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
    tmem_st32(t_o + c * 32, r);
  }
}

template <int VARIANT, int DK, int DV>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = Layout<DK, DV>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t bar_q = bar0;
  auto kv_full = [&](int s) { return bar0 + 8u * (1 + s); };
  auto kv_empty = [&](int s) { return bar0 + 8u * (1 + L::NS + s); };
  auto nk_full = [&](int s) { return bar0 + 8u * (1 + 2 * L::NS + s); };
  auto nk_empty = [&](int s) { return bar0 + 8u * (1 + 2 * L::NS + NKS + s); };
  auto s_full = [&](int x) { return bar0 + 8u * (1 + 2 * L::NS + 2 * NKS + x); };
  auto p_full = [&](int x) { return bar0 + 8u * (3 + 2 * L::NS + 2 * NKS + x); };
  auto o_full = [&](int x) { return bar0 + 8u * (5 + 2 * L::NS + 2 * NKS + x); };
  const uint32_t bar_drain = bar0 + 8u * (7 + 2 * L::NS + 2 * NKS);
  auto q_smem = [&](int x) { return sb + L::OFF_Q + (uint32_t)x * L::Q_TILE; };
  auto slot_smem = [&](int s) { return sb + L::OFF_RING + (uint32_t)s * L::SLOT; };
  const float *nk_ring = reinterpret_cast<const float *>(smem + L::OFF_NK);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  // ---- work unit: (query-tile pair, batch, head); causal pairs heaviest first
  const int BH = p.B * p.h;
  int pair = blockIdx.x / BH;
  const int bh = blockIdx.x - pair * BH;
  if (p.causal) pair = p.n_pairs - 1 - pair;
  const int head = bh % p.h;
  const int batch = bh / p.h;
  const int bh_kv = batch * p.hkv + head / (p.h / p.hkv);
  const int q0 = pair * 2 * BM;
  const bool q1_valid = (q0 + BM) < p.Tq;
  int nkv0, nkv1;
  if (p.causal) {
    nkv0 = min(2 * pair + 1, p.n_kv_tiles);
    nkv1 = q1_valid ? min(2 * pair + 2, p.n_kv_tiles) : 0;
  } else {
    nkv0 = p.n_kv_tiles;
    nkv1 = q1_valid ? p.n_kv_tiles : 0;
  }
  const int nkv = max(nkv0, nkv1);

  if (threadIdx.x == 0) {
    mbar_init(bar_q, 1);
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(kv_full(s), 1);
      mbar_init(kv_empty(s), 1);
    }
    for (int s = 0; s < NKS; ++s) {
      mbar_init(nk_full(s), 1);
      mbar_init(nk_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), BM);
      mbar_init(o_full(x), 1);
    }
    mbar_init(bar_drain, 1);
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_q);
    tma_prefetch_desc(&tm_k);
    tma_prefetch_desc(&tm_v);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_q, (q1_valid ? 2u : 1u) * (uint32_t)L::Q_TILE);
#pragma unroll
      for (int c = 0; c < DK / 64; ++c) {
        tma_load_3d(q_smem(0) + c * BM * 128, &tm_q, c * 64, q0, bh, bar_q);
        if (q1_valid) tma_load_3d(q_smem(1) + c * BM * 128, &tm_q, c * 64, q0 + BM, bh, bar_q);
      }
    }
    __syncwarp();
    for (int j = 0; j < nkv; ++j) {
      {  // K_j
        const int idx = 2 * j, s = idx % L::NS;
        const uint32_t use = (uint32_t)(idx / L::NS);
        if (!warp_wait(kv_empty(s), (use & 1u) ^ 1u, abort, SITE_PRODUCER | 0x10)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(kv_full(s), L::K_TILE);
#pragma unroll
          for (int c = 0; c < DK / 64; ++c)
            tma_load_3d(slot_smem(s) + c * BN * 128, &tm_k, c * 64, j * BN, bh_kv, kv_full(s));
        }
        __syncwarp();
      }
      if (VARIANT == kYat) {  // squared key norms of tile j
        const int s = j % NKS;
        const uint32_t use = (uint32_t)(j / NKS);
        if (!warp_wait(nk_empty(s), (use & 1u) ^ 1u, abort, SITE_PRODUCER | 0x20)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(nk_full(s), BN * 4);
          bulk_load(sb + L::OFF_NK + (uint32_t)s * BN * 4,
                    p.nk + (size_t)bh_kv * p.Tk_pad + (size_t)j * BN, BN * 4, nk_full(s));
        }
        __syncwarp();
      }
      {  // V_j
        const int idx = 2 * j + 1, s = idx % L::NS;
        const uint32_t use = (uint32_t)(idx / L::NS);
        if (!warp_wait(kv_empty(s), (use & 1u) ^ 1u, abort, SITE_PRODUCER | 0x30)) break;
        if (lane == 0) {
          mbar_arrive_expect_tx(kv_full(s), L::V_TILE);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c)
            tma_load_3d(slot_smem(s) + c * BN * 128, &tm_v, c * 64, j * BN, bh_kv, kv_full(s));
        }
        __syncwarp();
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    bool ok = warp_wait(bar_q, 0, abort, SITE_MMA | 0x10);
    tc_fence_after();
    uint32_t pph0 = 0, pph1 = 0;
    const int release_limit = 2 * nkv - L::NS;  // later slots are never reloaded
    for (int j = 0; ok && j <= nkv; ++j) {
      const int vidx = 2 * (j - 1) + 1;
      const int vs = j >= 1 ? vidx % L::NS : 0;
      if (j >= 1) {
        if (!(ok = warp_wait(kv_full(vs), (uint32_t)(vidx / L::NS) & 1u, abort, SITE_MMA | 0x20)))
          break;
        tc_fence_after();
      }
      if (j >= 1 && j - 1 < nkv0) {  // O0 += P0(j-1) V(j-1)
        if (!(ok = warp_wait(p_full(0), pph0, abort, SITE_MMA | 0x30))) break;
        pph0 ^= 1u;
        tc_fence_after();
        if (lane == 0) {
          issue_pv<DV>(tmem + 256, tmem + 0, slot_smem(vs), j - 1 > 0);
          if (j - 1 == nkv0 - 1) mma_commit(o_full(0));
        }
        __syncwarp();
      }
      const int kidx = 2 * j;
      const int ks = kidx % L::NS;
      if (j < nkv) {
        if (!(ok = warp_wait(kv_full(ks), (uint32_t)(kidx / L::NS) & 1u, abort, SITE_MMA | 0x40)))
          break;
        tc_fence_after();
      }
      if (j < nkv0) {  // S0 = Q0 K(j)^T
        if (lane == 0) {
          issue_qk<DK>(tmem + 0, q_smem(0), slot_smem(ks));
          mma_commit(s_full(0));
        }
        __syncwarp();
      }
      if (j >= 1 && j - 1 < nkv1) {  // O1 += P1(j-1) V(j-1)
        if (!(ok = warp_wait(p_full(1), pph1, abort, SITE_MMA | 0x50))) break;
        pph1 ^= 1u;
        tc_fence_after();
        if (lane == 0) {
          issue_pv<DV>(tmem + 384, tmem + 128, slot_smem(vs), j - 1 > 0);
          if (j - 1 == nkv1 - 1) mma_commit(o_full(1));
        }
        __syncwarp();
      }
      if (j < nkv1) {  // S1 = Q1 K(j)^T
        if (lane == 0) {
          issue_qk<DK>(tmem + 128, q_smem(1), slot_smem(ks));
          mma_commit(s_full(1));
        }
        __syncwarp();
      }
      if (lane == 0) {
        if (j < nkv && kidx < release_limit) mma_commit(kv_empty(ks));
        if (j >= 1 && vidx < release_limit) mma_commit(kv_empty(vs));
        // both epilogues delivered P for tile j-1, so they are done with its key norms
        if (VARIANT == kYat && j >= 1) mbar_arrive(nk_empty((j - 1) % NKS));
      }
      __syncwarp();
    }
    // all MMAs issued by this thread have completed once `drain` flips; this
    // wait ignores the abort flag so TMEM is never released under a live MMA
    if (lane == 0) mma_commit(bar_drain);
    __syncwarp();
    warp_wait(bar_drain, 0, abort, SITE_MMA | 0x60, false);
  } else {
    // ------------------------------------------------------------ epilogue
    const int x = warp >> 2;  // query tile of this warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row in tile == TMEM lane
    const int nkv_x = x ? nkv1 : nkv0;
    if (nkv_x > 0) {
      const int qrow0 = q0 + x * BM;
      const int row = qrow0 + r;
      const int qt = qrow0 / BM;
      const bool row_ok = row < p.Tq;
      const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
      const uint32_t t_s = tmem + lane_off + (uint32_t)x * 128;
      const uint32_t t_o = tmem + lane_off + 256u + (uint32_t)x * 128;

      // per-row state
      float acc_a = 0.f, acc_b = 0.f;  // Yat: row mass (two partial sums); else l
      float row_top = -INFINITY;       // Yat: max kappa; else max scaled score
      float m_used = -INFINITY;        // softmax / s^tau: running max, log2 units
      float yb = 0.f, yeps = 0.f, qe = 0.f, tau = 1.f, seps = 0.f;
      if (VARIANT == kYat) {
        yb = p.b[head];
        yeps = p.eps[head];
        const float nq = row_ok ? p.nq[(size_t)bh * p.Tq + row] : 0.f;
        qe = nq + yeps;
      } else if (VARIANT == kStau) {
        tau = p.tau[head];
        seps = p.eps[head];
      }
      const float c2 = p.scale * LOG2E;  // scaled score in log2 units per raw dot

      uint32_t sph = 0;
      bool ok = true;
      for (int j = 0; j < nkv_x; ++j) {
        if (!(ok = warp_wait(s_full(x), sph, abort, SITE_EPI | 0x10))) break;
        sph ^= 1u;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(t_s + c * 32, sr[c]);
        tmem_wait_ld();

        int limit = BN;
        if (j == p.n_kv_tiles - 1) limit = min(limit, p.Tk - j * BN);
        if (p.causal && j == qt) limit = min(limit, r + 1);
        const bool partial = limit < BN;

        uint32_t pk[2][32];  // P as bf16 pairs: columns [0,32) and [32,64)
        if (VARIANT == kYat) {
          const int ns = j % NKS;
          if (!(ok = warp_wait(nk_full(ns), (uint32_t)(j / NKS) & 1u, abort, SITE_EPI | 0x20)))
            break;
          const float2 *nk2 = reinterpret_cast<const float2 *>(nk_ring + ns * BN);
          float top = row_top;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const int col = c * 32 + i;
              const float2 nkv = nk2[col >> 1];
              const float d0 = __uint_as_float(sr[c][i]);
              const float d1 = __uint_as_float(sr[c][i + 1]);
              const float t0 = d0 + yb, t1 = d1 + yb;
              const float den0 = fmaxf(fmaf(-2.f, d0, qe + nkv.x), yeps);
              const float den1 = fmaxf(fmaf(-2.f, d1, qe + nkv.y), yeps);
              float k0 = t0 * t0 * rcp_approx(den0);
              float k1 = t1 * t1 * rcp_approx(den1);
              if (partial) {
                k0 = col < limit ? k0 : 0.f;
                k1 = col + 1 < limit ? k1 : 0.f;
              }
              acc_a += k0;
              acc_b += k1;
              top = fmaxf(top, fmaxf(k0, k1));
              pk[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_bf16x2(k0, k1);
            }
          }
          row_top = top;
        } else {
          // max of the raw dot over allowed keys (scale > 0 keeps the order)
          float mt = -INFINITY;
#pragma unroll
          for (int c = 0; c < 4; ++c)
#pragma unroll
            for (int i = 0; i < 32; ++i) {
              const float d = __uint_as_float(sr[c][i]);
              if (!partial || c * 32 + i < limit) mt = fmaxf(mt, d);
            }
          const float s_top = mt * p.scale;
          row_top = fmaxf(row_top, s_top);
          float m_new;
          if (VARIANT == kSoftmax) {
            m_new = mt * c2;
          } else {
            const float e = ex2_approx(-fabsf(s_top) * LOG2E);
            const float l1p = e < 0x1p-12f ? e : lg2_approx(1.f + e) * LN2;
            m_new = tau * lg2_approx(fmaxf(s_top, 0.f) + l1p + seps);
          }
          if (__any_sync(FULL, m_new > m_used + RESCALE_THRESHOLD)) {
            const float mn = fmaxf(m_used, m_new);
            const float corr = ex2_approx(m_used - mn);
            acc_a *= corr;
            acc_b *= corr;
            if (j > 0) scale_o_tmem<DV>(t_o, corr);
            m_used = mn;
          }
          const float neg_m = -m_used;
#pragma unroll
          for (int c = 0; c < 4; ++c) {
#pragma unroll
            for (int i = 0; i < 32; i += 2) {
              const int col = c * 32 + i;
              const float d0 = __uint_as_float(sr[c][i]);
              const float d1 = __uint_as_float(sr[c][i + 1]);
              float p0, p1;
              if (VARIANT == kSoftmax) {
                p0 = ex2_approx(fmaf(d0, c2, neg_m));
                p1 = ex2_approx(fmaf(d1, c2, neg_m));
              } else {
                const float s0 = d0 * p.scale, s1 = d1 * p.scale;
                const float e0 = ex2_approx(-fabsf(d0) * c2);
                const float e1 = ex2_approx(-fabsf(d1) * c2);
                const float l0 = e0 < 0x1p-12f ? e0 : lg2_approx(1.f + e0) * LN2;
                const float l1 = e1 < 0x1p-12f ? e1 : lg2_approx(1.f + e1) * LN2;
                const float g0 = lg2_approx(fmaxf(s0, 0.f) + l0 + seps);
                const float g1 = lg2_approx(fmaxf(s1, 0.f) + l1 + seps);
                p0 = ex2_approx(fmaf(tau, g0, neg_m));
                p1 = ex2_approx(fmaf(tau, g1, neg_m));
              }
              if (partial) {
                p0 = col < limit ? p0 : 0.f;
                p1 = col + 1 < limit ? p1 : 0.f;
              }
              acc_a += p0;
              acc_b += p1;
              pk[c >> 1][(c & 1) * 16 + (i >> 1)] = pack_bf16x2(p0, p1);
            }
          }
        }
        // P (bf16 pairs) over the first 64 columns of S_x
        tmem_st32(t_s + 0, pk[0]);
        tmem_st32(t_s + 32, pk[1]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(p_full(x));
      }

      if (ok && warp_wait(o_full(x), 0, abort, SITE_EPI | 0x30)) {
        tc_fence_after();
        const float total = acc_a + acc_b;
        const float inv = VARIANT == kYat ? 1.f / (total + 1e-9f) : 1.f / total;
        __nv_bfloat16 *orow =
            reinterpret_cast<__nv_bfloat16 *>(p.out) + ((size_t)bh * p.Tq + row) * DV;
#pragma unroll
        for (int c = 0; c < DV / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(t_o + c * 32, o);
          tmem_wait_ld();
          uint32_t packed[16];
#pragma unroll
          for (int i = 0; i < 16; ++i)
            packed[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv,
                                    __uint_as_float(o[2 * i + 1]) * inv);
          if (row_ok) {
            uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                  packed[4 * i + 3]);
          }
        }
        if (row_ok) {
          const size_t ti = (size_t)bh * p.Tq + row;
          if (p.row_mass)
            p.row_mass[ti] = VARIANT == kYat ? total : (m_used + log2f(total)) * LN2;
          if (p.row_max) p.row_max[ti] = row_top;
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int VARIANT, int DK, int DV>
cudaError_t launch(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                   const CUtensorMap &tv, cudaStream_t s) {
  using L = Layout<DK, DV>;
  auto kern = fwd_kernel<VARIANT, DK, DV>;
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  const long long units = (long long)p.B * p.h * p.n_pairs;
  if (units <= 0) return cudaSuccess;
  kern<<<(unsigned)units, NUM_THREADS, L::ALLOC, s>>>(p, tq, tk, tv);
  return cudaGetLastError();
}

}  // namespace tc

bool fwd_tc_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 128 && dv == 64);
}

cudaError_t launch_fwd_tc(int variant, int dk, int dv, const FwdParams &p, const CUtensorMap &tq,
                          const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t s) {
#define CATTN_TC_CASE(V, DK_, DV_) \
  if (variant == V && dk == DK_ && dv == DV_) return tc::launch<V, DK_, DV_>(p, tq, tk, tv, s);
  CATTN_TC_CASE(kSoftmax, 64, 64)
  CATTN_TC_CASE(kSoftmax, 128, 128)
  CATTN_TC_CASE(kSoftmax, 128, 64)
  CATTN_TC_CASE(kYat, 64, 64)
  CATTN_TC_CASE(kYat, 128, 128)
  CATTN_TC_CASE(kYat, 128, 64)
  CATTN_TC_CASE(kStau, 64, 64)
  CATTN_TC_CASE(kStau, 128, 128)
  CATTN_TC_CASE(kStau, 128, 64)
#undef CATTN_TC_CASE
  return cudaErrorInvalidValue;
}

cudaError_t read_and_clear_status(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace cattn
