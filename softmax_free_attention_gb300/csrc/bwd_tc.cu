// bwd_tc.cu -- attention backward on the sm_103a tensor cores.
//
// Gradients of L = sum(dout * out) through the forward of the three maps.
// Per query row t the forward's weights are w_tj = f_tj / Z_t, recomputed here
// from the scores and the forward's own row_mass (softmax and s^tau: the log
// of Z; Yat: the mass itself).  With dW_tj = dout_t . v_j and D_t = dout_t .
// out_t, the chain rule through the normalisation gives dL/df_tj =
// (dW_tj - D_t) / Z_t, and then per map
//
//   softmax  C = scale w (dW - D)
//   s^tau    C = scale w (dW - D) tau sigma(s) / phi(s),       s = scale q.k
//            dtau += w (dW - D) ln phi,  deps += w (dW - D) tau / phi
//   Yat      g = (dW - D) / Z,  a = 2m g (q.k + b)^{2m-1} / den,
//            e = -g kappa / den (the gradient on den = max(d2, 0) + eps),
//            C = a - 2 e [d2 > 0],  db += a,  deps += e
//
// and the three products
//
//   dq_t = sum_j C_tj k_j (+ 2 q_t sum_j e_tj [d2 > 0] for Yat)
//   dk_j = sum_t C_tj q_t (+ 2 k_j sum_t e_tj [d2 > 0] for Yat)
//   dv_j = sum_t w_tj dout_t
//
// (the Yat distance term: d|q - k|^2 / dq = 2 (q - k), whose k part joins C).
// The maps themselves: "Softmax-Free Attention in JAX/Flax NNX", section "One
// module, two compatibility functions"; "s^tau: a focal-length knob for
// attention", core formula.
//
// Two passes of one kernel template, each a dense tile loop:
//
//   SIDE_KV  one CTA per 128-key tile of one (batch, kv head).  K and V stay
//            in shared memory; 64-row tiles of Q and dout, of every query
//            head that shares the kv head, stream through a two-stage ring
//            with the per-row D, normaliser and |q|^2.  Per tile:
//              S^T = K Q^T and dP^T = V dout^T     tcgen05, into TMEM
//              W^T and C^T                          the map warps, into TMEM and smem
//              dV += W^T dout and dK += C^T Q       tcgen05, accumulators in TMEM
//   SIDE_Q   one CTA per 128-query tile of one (batch, head): Q and dout stay,
//            64-key tiles of K and V (and the squared key norms) stream.
//              S = Q K^T and dP = dout V^T, then C, then dQ += C K.
//
// The dQ pass computes S, dP and C again rather than exchanging partial dQ
// through global atomics: both passes write each output element once, in a
// fixed order, so the backward is deterministic.  S and dP have two TMEM
// buffers each, so the MMAs of tile n+1 run while the warps map tile n, and
// the accumulating MMAs of tile n run while they map tile n+1.
//
// TMEM (512 columns): S[2] at 0 and 64, dP[2] at 128 and 192, the first
// accumulator (dV, or dQ) at 256, the second (dK) at 256 + DV.  In the dK/dV
// pass the map warps write W^T (bf16) over the dP columns they have read, and
// the dV MMAs take it from there; C^T goes through shared memory.
//
// Warp roles (608 threads): warps 0-15 map (warp w: TMEM lanes 32 (w % 4)..+31
// = rows of the resident tile, tile columns [16 (w / 4), +16); four warps per
// SM sub-partition hide each other's TMEM and SFU latencies), warp 16 issues
// the TMA loads, warp 17 allocates TMEM and issues the accumulating MMAs,
// warp 18 issues the S and dP MMAs.
// Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the kernel
// records a site code, raises a CTA-wide abort flag and every role leaves its
// loop, waits for its own copies and MMAs in flight, and TMEM is released.
#include <cuda_bf16.h>

#include <type_traits>

#include "bwd.h"
#include "kernels.h"
#include "maps.cuh"
#include "ptx.cuh"

namespace cattn {

__device__ unsigned int g_bwd_status;

namespace bwd {

constexpr int RT = 128;  // rows of the resident tile (TMEM lanes)
constexpr int CT = 64;   // rows of a streamed tile = columns of S
constexpr int NUM_THREADS = 608;
constexpr int MAP_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;    // the accumulating MMAs (and TMEM allocation)
constexpr int SCORE_WARP = 18;  // the S and dP MMAs
constexpr int NQ = MAP_WARPS / 4;  // column slices of a tile: four map warps per TMEM lane quadrant
constexpr int CW = CT / NQ;        // columns per map warp (16)
static_assert(CW == 16, "a map warp's W^T slice is one K step of the dV MMAs");
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
constexpr unsigned FULL = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;

constexpr int SIDE_KV = 0;
constexpr int SIDE_Q = 1;

constexpr uint32_t TM_S = 0;     // + 64 b
constexpr uint32_t TM_DP = 128;  // + 64 b
constexpr uint32_t TM_A1 = 256;

enum : unsigned { SITE_PRODUCER = 0x1100, SITE_MMA = 0x1200, SITE_MAP = 0x1300 };

// DK: width of q and k rows; DV: width of v and dout rows.  The resident tile
// R and the streamed tile X have rows of DK (K and Q, or Q and K), their
// partners RP and XP rows of DV (V and dout, or dout and V).
template <int DK, int DV, int SIDE>
struct Layout {
  static constexpr int R_TILE = RT * DK * 2;
  static constexpr int RP_TILE = RT * DV * 2;
  static constexpr int X_TILE = CT * DK * 2;
  static constexpr int XP_TILE = CT * DV * 2;
  static constexpr int AUX = 1024;  // up to three 64-float planes (SIDE_KV) or 64 floats (SIDE_Q)
  static constexpr int STAGE = X_TILE + XP_TILE + AUX;
  static constexpr int W_TILE = RT * CT * 2;  // one 128-byte swizzle box per row
  // Four stages in the streamed-tile ring: a stage is held from the tile's S
  // MMAs to its accumulating MMAs and a load takes about two thousand cycles,
  // so the ring runs three tiles ahead of the map warps.  One C buffer in
  // shared memory (the map warps of tile n+1 finish long after the MMAs of
  // tile n have read it); W^T goes to TMEM over the dP columns the map warps
  // have read, which is what leaves room for the fourth stage.
  static constexpr int NS = 4;
  static constexpr int OFF_R = 0;
  static constexpr int OFF_RP = R_TILE;
  static constexpr int OFF_ST = R_TILE + RP_TILE;
  static constexpr int OFF_C = OFF_ST + NS * STAGE;
  static constexpr int OFF_XCH = OFF_C + W_TILE;  // [2][NQ slices][128] floats
  static constexpr int OFF_BAR = OFF_XCH + 2 * NQ * RT * 4;
  // r_full, x_full[NS], x_empty[NS], s_full[2], s_empty[2], wc_full, wc_empty,
  // acc_full, drain
  static constexpr int NBAR = 1 + 2 * NS + 4 + 2 + 2;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr int BYTES = OFF_MISC + 16;
  // at least 120 KB, so that a second CTA (which would wait for this one's
  // 512 TMEM columns) never shares the SM
  static constexpr int ALLOC = BYTES + 1024 > 120 * 1024 ? BYTES + 1024 : 120 * 1024;
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(STAGE % 1024 == 0 && R_TILE % 1024 == 0 && RP_TILE % 1024 == 0 &&
                    X_TILE % 1024 == 0 && XP_TILE % 1024 == 0,
                "swizzle atoms stay 1024-B aligned");
};

__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned site, bool honor_abort = true) {
  if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
    const int bad = (honor_abort && *abort != 0) || (globaltimer_ns() - t0 > WAIT_LIMIT_NS);
    if (__any_sync(FULL, bad)) {
      if ((threadIdx.x & 31) == 0) {
        atomicCAS(&g_bwd_status, 0u, site | 1u);
        *abort = 1;
      }
      return false;
    }
  }
}

__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                            unsigned site, bool honor_abort = true) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((honor_abort && *abort != 0) || (globaltimer_ns() - t0 > WAIT_LIMIT_NS)) {
      atomicCAS(&g_bwd_status, 0u, site | 1u);
      *abort = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void sts128(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                       uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_fence16(uint32_t (&r)[16]) {
#pragma unroll
  for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i])::"memory");
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ void stg128(void *ptr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(ptr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// The MMA lane shares its SM sub-partition with four busy map warps, so its
// instruction count sets how fast it can issue: descriptors are built once
// and every MMA adds a compile-time offset to them (the start-address field
// is the low 14 bits of the descriptor, in 16-byte units; shared-memory
// offsets stay far below its range).

// S[128 x 64] = A[128 x D] B[64 x D]^T from descriptors of a resident tile
// (64-column boxes RT*128 bytes apart) and a streamed tile (CT*128 apart).
template <int D>
__device__ __forceinline__ void issue_scores(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc) {
  constexpr uint32_t IDESC = idesc_bf16_f32(RT, CT, false);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t ao = (uint64_t)(((kk >> 2) * (RT * 128) + (kk & 3) * 32) >> 4);
    const uint64_t bo = (uint64_t)(((kk >> 2) * (CT * 128) + (kk & 3) * 32) >> 4);
    mma_ss_e(d_tmem, adesc + ao, bdesc + bo, IDESC, kk > 0 ? 1u : 0u);
  }
}

// Acc[128 x D] (+)= A[128 x 64] B[64 x D]: A the map warps' tile (one 128-byte
// box per row, K-major), B a streamed tile read N-major (descriptor with the
// 64-column boxes CT*128 bytes apart as its leading offset).
template <int D>
__device__ __forceinline__ void issue_acc(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc_n,
                                          bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(RT, D, true);
#pragma unroll
  for (int kk = 0; kk < CT / 16; ++kk)
    mma_ss_e(d_tmem, adesc + (uint64_t)((kk * 32) >> 4), bdesc_n + (uint64_t)((kk * 2048) >> 4),
           IDESC, (accumulate || kk > 0) ? 1u : 0u);
}

// Acc[128 x D] (+)= A[128 x 64] B[64 x D] with A in TMEM (bf16 pairs; K
// step kk, indices 16 kk .. 16 kk + 15, at columns 16 kk .. 16 kk + 7 from
// a_tmem) and B a streamed tile read N-major.
template <int D>
__device__ __forceinline__ void issue_acc_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc_n,
                                             bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(RT, D, true);
#pragma unroll
  for (int kk = 0; kk < CT / 16; ++kk)
    mma_ts_e(d_tmem, a_tmem + (uint32_t)kk * 16u, bdesc_n + (uint64_t)((kk * 2048) >> 4), IDESC,
             (accumulate || kk > 0) ? 1u : 0u);
}

struct HeadP {
  float b, eps, tau;
};

// Two (row, column) pairs of one row, as f32x2 lanes: the weights w (the
// forward's, recomputed) and the score gradients c, plus the accumulators.
// X, Y, Z: the query row's scalars as the prep and row-sum passes leave them
//   softmax  X = -D scale,   Y = -log2 Z
//   s^tau    X = -D,         Y = -log2 Z
//   Yat      X = -D / Z,     Y = 1 / Z,     Z = |q|^2 + eps + |k|^2
// Accumulators: Yat acc0 = -sum e [d2 > 0] (the rank-one term), acc1 = db,
// acc2 = -deps; s^tau acc1 = deps, acc2 = dtau / ln 2.  FULL: every pair is
// allowed (no mask).  WONLY: the weights only (the row-sum pass).
template <int VARIANT, int YM, bool FULL, bool WONLY>
__device__ __forceinline__ void pair2(float2 s, float2 dp, float2 X, float2 Y, float2 Z,
                                      const HeadP &hp, float scale, float c2, bool al0, bool al1,
                                      float2 &w, float2 &c, float2 &acc0, float2 &acc1,
                                      float2 &acc2) {
  if constexpr (VARIANT == kSoftmax) {
    const float2 x = __ffma2_rn(s, make_float2(c2, c2), Y);
    w = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    if (!FULL) {
      w.x = al0 ? w.x : 0.f;
      w.y = al1 ? w.y : 0.f;
    }
    if constexpr (!WONLY) c = __fmul2_rn(w, __ffma2_rn(dp, make_float2(scale, scale), X));
  } else if constexpr (VARIANT == kStau) {
    const float2 sc = __fmul2_rn(s, make_float2(scale, scale));
    const float e0 = ex2_approx(-fabsf(s.x) * c2), e1 = ex2_approx(-fabsf(s.y) * c2);
    // phi as the forward computes it, so the weights match its normaliser
    const float2 phi = tc::phi2(sc, make_float2(e0, e1), hp.eps);
    const float2 lp = make_float2(lg2_approx(phi.x), lg2_approx(phi.y));
    const float2 x = __ffma2_rn(make_float2(hp.tau, hp.tau), lp, Y);
    w = make_float2(ex2_approx(x.x), ex2_approx(x.y));
    if (!FULL) {
      w.x = al0 ? w.x : 0.f;
      w.y = al1 ? w.y : 0.f;
    }
    if constexpr (!WONLY) {
      // 1 / (1 + e) and 1 / phi from one reciprocal of their product
      const float2 ope = __fadd2_rn(make_float2(e0, e1), make_float2(1.f, 1.f));
      const float2 pq = __fmul2_rn(ope, phi);
      const float2 rq = make_float2(rcp_approx(pq.x), rcp_approx(pq.y));
      const float2 r01 = __fmul2_rn(phi, rq);
      const float2 sig = make_float2(sc.x >= 0.f ? r01.x : e0 * r01.x, sc.y >= 0.f ? r01.y : e1 * r01.y);
      const float2 trphi = __fmul2_rn(make_float2(hp.tau, hp.tau), __fmul2_rn(ope, rq));
      const float2 base = __fmul2_rn(w, __fadd2_rn(dp, X));  // w (dW - D)
      const float2 bt = __fmul2_rn(base, trphi);
      c = __fmul2_rn(__fmul2_rn(bt, sig), make_float2(scale, scale));
      acc1 = __fadd2_rn(acc1, bt);
      acc2 = __ffma2_rn(base, lp, acc2);
    }
  } else {  // Yat
    const float2 num = __fadd2_rn(s, make_float2(hp.b, hp.b));
    const float2 num2 = __fmul2_rn(num, num);
    float2 nodd = num, neven = num2;  // num^{2m-1}, num^{2m}
    if constexpr (YM == 2) {
      nodd = __fmul2_rn(num, num2);
      neven = __fmul2_rn(num2, num2);
    }
    if constexpr (YM == 3) {
      const float2 num4 = __fmul2_rn(num2, num2);
      nodd = __fmul2_rn(num, num4);
      neven = __fmul2_rn(num2, num4);
    }
    const float2 den = __ffma2_rn(make_float2(-2.f, -2.f), s, Z);  // |q - k|^2 + eps
    const bool a0 = den.x > hp.eps, a1 = den.y > hp.eps;
    const float2 rd =
        make_float2(rcp_approx(a0 ? den.x : hp.eps), rcp_approx(a1 ? den.y : hp.eps));
    const float2 kap = __fmul2_rn(neven, rd);
    w = __fmul2_rn(kap, Y);
    if (!FULL) {
      w.x = al0 ? w.x : 0.f;
      w.y = al1 ? w.y : 0.f;
    }
    if constexpr (!WONLY) {
      float2 g = __ffma2_rn(dp, Y, X);  // (dW - D) / Z
      if (!FULL) {
        g.x = al0 ? g.x : 0.f;
        g.y = al1 ? g.y : 0.f;
      }
      const float2 gr = __fmul2_rn(g, rd);
      const float2 a = __fmul2_rn(gr, __fmul2_rn(nodd, make_float2(2.f * YM, 2.f * YM)));
      const float2 ne = __fmul2_rn(gr, kap);  // -e
      const float2 nea = make_float2(a0 ? ne.x : 0.f, a1 ? ne.y : 0.f);
      c = __ffma2_rn(nea, make_float2(2.f, 2.f), a);
      acc0 = __fadd2_rn(acc0, nea);
      acc1 = __fadd2_rn(acc1, a);
      acc2 = __fadd2_rn(acc2, ne);
    }
  }
}

// DP: the row-sum pass (SIDE_Q only): D_t = sum_j w_tj dW_tj from the
// backward's own weights, written over the aux array's D; no C, no dQ.
template <int VARIANT, int DK, int DV, int SIDE, int YM = 1, bool DP = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    bwd_kernel(const __grid_constant__ BwdParams p, const __grid_constant__ CUtensorMap tm_r,
               const __grid_constant__ CUtensorMap tm_rp, const __grid_constant__ CUtensorMap tm_x,
               const __grid_constant__ CUtensorMap tm_xp) {
  using L = Layout<DK, DV, SIDE>;
  constexpr bool KV = SIDE == SIDE_KV;
  static_assert(!DP || SIDE == SIDE_Q, "the row-sum pass runs on the query side");
  constexpr bool HAS_PAR = KV && VARIANT != kSoftmax;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = sb + L::OFF_BAR;
  constexpr int NS = L::NS;
  const uint32_t bar_r_full = bar0;
  auto x_full = [&](int st) { return bar0 + 8u * (1 + st); };
  auto x_empty = [&](int st) { return bar0 + 8u * (1 + NS + st); };
  auto s_full = [&](int b) { return bar0 + 8u * (1 + 2 * NS + b); };
  auto s_empty = [&](int b) { return bar0 + 8u * (3 + 2 * NS + b); };
  const uint32_t bar_wc_full = bar0 + 8u * (5 + 2 * NS);
  const uint32_t bar_wc_empty = bar0 + 8u * (6 + 2 * NS);
  const uint32_t bar_acc = bar0 + 8u * (7 + 2 * NS);
  const uint32_t bar_drain = bar0 + 8u * (8 + 2 * NS);
  const uint32_t r_smem = sb + L::OFF_R, rp_smem = sb + L::OFF_RP;
  auto x_smem = [&](int st) { return sb + L::OFF_ST + (uint32_t)st * L::STAGE; };
  auto xp_smem = [&](int st) { return x_smem(st) + L::X_TILE; };
  auto aux_smem = [&](int st) { return x_smem(st) + L::X_TILE + L::XP_TILE; };
  const uint32_t c_smem = sb + L::OFF_C;
  float *xch = reinterpret_cast<float *>(smem + L::OFF_XCH);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);

  // ---- this CTA's tile and its list of streamed tiles
  int rt, bh_r, n_tiles, first = 0, per_head = 0, group = 1, b_idx;
  if constexpr (KV) {
    const int nb = p.B * p.hkv;
    rt = blockIdx.x / nb;  // key tile; heavy (low) tiles first under a causal mask
    bh_r = blockIdx.x % nb;
    b_idx = bh_r / p.hkv;
    group = p.h / p.hkv;
    first = p.causal ? 2 * rt : 0;
    per_head = p.n_q64 - first;
    n_tiles = group * per_head;
  } else {
    const int nb = p.B * p.h;
    rt = p.n_q128 - 1 - (int)(blockIdx.x / nb);  // query tile, heavy (high) tiles first
    bh_r = blockIdx.x % nb;
    b_idx = bh_r / p.h;
    n_tiles = p.causal ? min(2 * rt + 2, p.n_k64) : p.n_k64;
  }
  // head and row of streamed tile n (SIDE_KV: (query head, query tile); SIDE_Q: key tile)
  auto stream_tile = [&](int n, int &bh_x, int &row0, int &head) {
    if constexpr (KV) {
      const int g = bh_r % p.hkv;
      head = g * group + n / per_head;
      bh_x = b_idx * p.h + head;
      row0 = (first + n % per_head) * CT;
    } else {
      head = bh_r % p.h;
      bh_x = b_idx * p.hkv + head / (p.h / p.hkv);
      row0 = n * CT;
    }
  };

  if (threadIdx.x == 0) {
    mbar_init(bar_r_full, 1);
    for (int st = 0; st < NS; ++st) {
      mbar_init(x_full(st), 1);
      // DP: released by the map warps (lane 0 of each) once they have read the
      // stage's key norms; else by the commit after the tile's last MMA
      mbar_init(x_empty(st), DP ? MAP_WARPS : 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(s_full(b), 1);
      // SIDE_KV: the commit after the tile's dV MMAs, which read W^T out of
      // the dP columns; else every map thread once it has read S and dP
      mbar_init(s_empty(b), KV ? 1 : MAP_WARPS * 32);
    }
    mbar_init(bar_wc_full, MAP_WARPS * 32);
    mbar_init(bar_wc_empty, 1);
    mbar_init(bar_acc, 1);
    mbar_init(bar_drain, 2);  // the commits of both issuing warps
    *abort = 0;
    fence_mbar_init();
  }
  if (warp == MMA_WARP) {
    tmem_alloc(smem_u32(tmem_holder), 512);
    tmem_relinquish();
  }
  if (warp == PRODUCER_WARP && lane == 0) {
    tma_prefetch_desc(&tm_r);
    tma_prefetch_desc(&tm_rp);
    tma_prefetch_desc(&tm_x);
    tma_prefetch_desc(&tm_xp);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == PRODUCER_WARP) {
    if (lane == 0) {
      mbar_arrive_expect_tx(bar_r_full, (uint32_t)(L::R_TILE + L::RP_TILE));
#pragma unroll
      for (int c = 0; c < DK / 64; ++c)
        tma_load_3d(r_smem + c * RT * 128, &tm_r, c * 64, rt * RT, bh_r, bar_r_full);
#pragma unroll
      for (int c = 0; c < DV / 64; ++c)
        tma_load_3d(rp_smem + c * RT * 128, &tm_rp, c * 64, rt * RT, bh_r, bar_r_full);
      // the streamed rows' aux: (dK/dV pass) -D, 1 / Z and, for Yat, |q|^2 +
      // eps, one plane after another; (dQ pass, Yat) the key norms
      constexpr uint32_t AUX_PLANES = KV ? (VARIANT == kYat ? 3u : 2u) : (VARIANT == kYat ? 1u : 0u);
      constexpr uint32_t AUXB = AUX_PLANES * CT * 4;
      int issued = 0;
      for (int n = 0; n < n_tiles; ++n) {
        const int st = n % NS;
        if (n >= NS &&
            !thread_wait(x_empty(st), ((n / NS) & 1) ^ 1, abort, SITE_PRODUCER | 0x10))
          break;
        int bh_x, row0, head;
        stream_tile(n, bh_x, row0, head);
        mbar_arrive_expect_tx(x_full(st), (uint32_t)(L::X_TILE + L::XP_TILE) + AUXB);
#pragma unroll
        for (int c = 0; c < DK / 64; ++c)
          tma_load_3d(x_smem(st) + c * CT * 128, &tm_x, c * 64, row0, bh_x, x_full(st));
#pragma unroll
        for (int c = 0; c < DV / 64; ++c)
          tma_load_3d(xp_smem(st) + c * CT * 128, &tm_xp, c * 64, row0, bh_x, x_full(st));
        if constexpr (KV) {
#pragma unroll
          for (uint32_t k = 0; k < AUX_PLANES; ++k)
            bulk_load(aux_smem(st) + k * CT * 4u, p.aux + k * p.aux_plane + (size_t)bh_x * p.Tq_pad + row0,
                      CT * 4u, x_full(st));
        } else if constexpr (VARIANT == kYat) {
          bulk_load(aux_smem(st), p.nk + (size_t)bh_x * p.Tk_pad + row0, AUXB, x_full(st));
        }
        issued = n + 1;
      }
      // copies still in flight land before the CTA can exit
      thread_wait(bar_r_full, 0, abort, SITE_PRODUCER | 0x20, false);
      for (int m = issued >= NS ? issued - NS : 0; m < issued; ++m)
        thread_wait(x_full(m % NS), (m / NS) & 1, abort, SITE_PRODUCER | 0x30, false);
    }
  } else if (warp == MMA_WARP || warp == SCORE_WARP) {
    // Two issuing warps, each converged with an elected lane issuing: the
    // score warp issues S and dP of tile n as soon as its stage has landed
    // and the map warps have read tile n-2 out of its TMEM buffer; the MMA
    // warp issues the accumulating MMAs of tile m once the map warps have
    // written its W and C.  (A single issuer serialised the two streams; the
    // issuing warps share their SM sub-partitions with busy map warps, so each
    // MMA takes tens of cycles to issue.)  Neither stream reads what the other
    // writes except through the mbarriers: S(n) has completed before the map
    // warps start tile n, so the commit after acc(n) also frees its stage.
    bool ok = warp_wait(bar_r_full, 0, abort, SITE_MMA | 0x10);
    auto stage_off = [](int st) { return (uint64_t)((st * L::STAGE) >> 4); };
    if (warp == SCORE_WARP) {
      // descriptors: K-major views of the resident tiles and stage 0's streamed tiles
      const uint64_t dR = smem_desc_sw128(r_smem, 16, 1024);
      const uint64_t dRP = smem_desc_sw128(rp_smem, 16, 1024);
      const uint64_t dX0 = smem_desc_sw128(x_smem(0), 16, 1024);
      const uint64_t dXP0 = smem_desc_sw128(xp_smem(0), 16, 1024);
      for (int n = 0; ok && n < n_tiles; ++n) {
        const int b = n & 1, st = n % NS;
        if (!(ok = warp_wait(x_full(st), (n / NS) & 1, abort, SITE_MMA | 0x30))) break;
        if (n >= 2 && !(ok = warp_wait(s_empty(b), ((n >> 1) & 1) ^ 1, abort, SITE_MMA | 0x40)))
          break;
        tc_fence_after();
        issue_scores<DK>(tmem + TM_S + 64u * b, dR, dX0 + stage_off(st));
        issue_scores<DV>(tmem + TM_DP + 64u * b, dRP, dXP0 + stage_off(st));
        mma_commit_e(s_full(b));
      }
    } else if constexpr (!DP) {
      // descriptors: the C tile (K-major) and stage 0's streamed tiles (N-major)
      const uint64_t dC = smem_desc_sw128(c_smem, 16, 1024);
      const uint64_t nX0 = smem_desc_sw128(x_smem(0), CT * 128, 1024);
      const uint64_t nXP0 = smem_desc_sw128(xp_smem(0), CT * 128, 1024);
      for (int m = 0; ok && m < n_tiles; ++m) {
        const int st = m % NS;
        if (!(ok = warp_wait(bar_wc_full, m & 1, abort, SITE_MMA | 0x20))) break;
        tc_fence_after();
        if constexpr (KV) {
          // dV += W^T dout (W^T from TMEM), dK += C^T Q
          issue_acc_ts<DV>(tmem + TM_A1, tmem + TM_DP + 64u * (m & 1), nXP0 + stage_off(st),
                           m > 0);
          issue_acc<DK>(tmem + TM_A1 + DV, dC, nX0 + stage_off(st), m > 0);
        } else {
          issue_acc<DK>(tmem + TM_A1, dC, nX0 + stage_off(st), m > 0);  // dQ += C K
        }
        mma_commit_e(x_empty(st));
        mma_commit_e(bar_wc_empty);
        if constexpr (KV) mma_commit_e(s_empty(m & 1));  // S / dP / W^T buffer free
      }
      if (ok) mma_commit_e(bar_acc);
    }
    // every MMA either warp issued has completed once `drain` flips
    mma_commit_e(bar_drain);
    warp_wait(bar_drain, 0, abort, SITE_MMA | 0x50, false);
  } else {
    // ---- map warps
    const int qd = warp & 3, hf = warp >> 2;  // lane quadrant, column slice
    const int r = 32 * qd + lane;  // row of the resident tile
    const uint32_t t_lane = tmem + ((uint32_t)(32 * qd) << 16);
    const float scale = p.scale, c2 = p.scale * LOG2E;
    const int grow = rt * RT + r;  // key j (SIDE_KV) or query t (SIDE_Q)
    // row scalars
    float row_nk = 0.f;
    float4 row_aux = make_float4(0.f, 0.f, 0.f, 0.f);
    HeadP hp{0.f, 1.f, 1.f};
    if constexpr (KV) {
      if (VARIANT == kYat) row_nk = p.nk[(size_t)bh_r * p.Tk_pad + grow];
    } else {
      const size_t ri = (size_t)bh_r * p.Tq_pad + grow;
      row_aux = make_float4(p.aux[ri], p.aux[p.aux_plane + ri], p.aux[2 * p.aux_plane + ri], 0.f);
      const int head = bh_r % p.h;
      if (VARIANT == kYat) hp.b = p.b[head];
      if (VARIANT != kSoftmax) hp.eps = p.eps[head];
      if (VARIANT == kStau) hp.tau = p.tau[head];
    }
    float2 acc0 = make_float2(0.f, 0.f), acc1 = acc0, acc2 = acc0, dsum = acc0, wsum = acc0;
    bool ok = true;
    for (int n = 0; n < n_tiles; ++n) {
      const int b = n & 1, st = n % NS;
      int bh_x, row0, head;
      stream_tile(n, bh_x, row0, head);
      if constexpr (KV) {
        if (n % per_head == 0) {
          if (VARIANT == kYat) hp.b = p.b[head];
          if (VARIANT != kSoftmax) hp.eps = p.eps[head];
          if (VARIANT == kStau) hp.tau = p.tau[head];
        }
      }
      if (!(ok = warp_wait(s_full(b), (n >> 1) & 1, abort, SITE_MAP | 0x10))) break;
      tc_fence_after();
      uint32_t sr[CW], dr[CW];
      tmem_ld16(t_lane + TM_S + 64u * b + (uint32_t)(CW * hf), sr);
      tmem_ld16(t_lane + TM_DP + 64u * b + (uint32_t)(CW * hf), dr);
      tmem_wait_ld();
      tmem_ld_fence16(sr);
      tmem_ld_fence16(dr);
      tc_fence_before();
      if constexpr (!KV) mbar_arrive(s_empty(b));

      const int col0 = row0 + CW * hf;  // global index of this thread's first column
      // warp-uniform: is every pair of this warp's 32 x CW block allowed?
      bool full;
      {
        const int r_lo = rt * RT + 32 * qd, r_hi = r_lo + 31;
        if constexpr (KV)
          full = col0 + CW <= p.Tq && r_hi < p.Tk && (!p.causal || col0 >= r_hi);
        else
          full = col0 + CW <= p.Tk && r_hi < p.Tq && (!p.causal || col0 + CW - 1 <= r_lo);
      }
      uint32_t wpk[CW / 2], cpk[CW / 2];
      auto chunk = [&](auto full_c) {
        constexpr bool FULL = decltype(full_c)::value;
#pragma unroll
        for (int i = 0; i < CW; i += 2) {
          float2 X, Y, Z = make_float2(0.f, 0.f);
          bool al0 = true, al1 = true;
          if constexpr (KV) {
            // the two columns' -D, 1 / Z (and |q|^2 + eps) as pairs, one plane each
            const uint32_t ao = aux_smem(st) + 4u * (CW * hf + i);
            const uint2 ux = lds64(ao), uy = lds64(ao + CT * 4u);
            X = make_float2(__uint_as_float(ux.x), __uint_as_float(ux.y));
            Y = make_float2(__uint_as_float(uy.x), __uint_as_float(uy.y));
            if (VARIANT == kYat) {
              const uint2 uz = lds64(ao + 2u * CT * 4u);
              Z = __fadd2_rn(make_float2(__uint_as_float(uz.x), __uint_as_float(uz.y)),
                             make_float2(row_nk, row_nk));
            }
            if (!FULL) {
              const int t = col0 + i;
              al0 = t < p.Tq && grow < p.Tk && (!p.causal || grow <= t);
              al1 = t + 1 < p.Tq && grow < p.Tk && (!p.causal || grow <= t + 1);
            }
          } else {
            X = make_float2(row_aux.x, row_aux.x);
            Y = make_float2(row_aux.y, row_aux.y);
            if (VARIANT == kYat) {
              const uint2 u = lds64(aux_smem(st) + 4u * (CW * hf + i));
              Z = __fadd2_rn(make_float2(row_aux.z, row_aux.z),
                             make_float2(__uint_as_float(u.x), __uint_as_float(u.y)));
            }
            if (!FULL) {
              const int j = col0 + i;
              al0 = j < p.Tk && grow < p.Tq && (!p.causal || j <= grow);
              al1 = j + 1 < p.Tk && grow < p.Tq && (!p.causal || j + 1 <= grow);
            }
          }
          const float2 sv = tc::f2(sr[i], sr[i + 1]), dv = tc::f2(dr[i], dr[i + 1]);
          float2 w, c = make_float2(0.f, 0.f);
          pair2<VARIANT, YM, FULL, DP>(sv, dv, X, Y, Z, hp, scale, c2, al0, al1, w, c, acc0,
                                       acc1, acc2);
          if constexpr (DP) {
            dsum = __ffma2_rn(w, dv, dsum);
            if (VARIANT == kYat) wsum = __fadd2_rn(wsum, w);
          }
          wpk[i >> 1] = pack_bf16x2(w.x, w.y);
          cpk[i >> 1] = pack_bf16x2(c.x, c.y);
        }
      };
      if (full)
        chunk(std::true_type{});
      else
        chunk(std::false_type{});
      if constexpr (DP) {
        __syncwarp();
        if (lane == 0) mbar_arrive(x_empty(st));
        continue;
      }
      // W^T of this thread's 16 queries (K step hf of the dV MMAs), as bf16
      // pairs, over the first 8 of the 16 dP columns this warp itself read
      if constexpr (KV) tmem_st8(t_lane + TM_DP + 64u * b + 16u * hf, wpk);
      // the accumulating MMAs of tile n-1 have read the C buffer
      if (n >= 1 && !(ok = warp_wait(bar_wc_empty, (n - 1) & 1, abort, SITE_MAP | 0x20))) break;
      // row r of the 128-byte-swizzled box: logical 16-byte chunk 2 hf + q at
      // physical chunk (2 hf + q) ^ (r % 8)
#pragma unroll
      for (int q4 = 0; q4 < CW / 8; ++q4) {
        const uint32_t off =
            (uint32_t)r * 128u + (uint32_t)((((CW / 8) * hf + q4) ^ (r & 7)) * 16);
        sts128(c_smem + off, cpk[4 * q4], cpk[4 * q4 + 1], cpk[4 * q4 + 2], cpk[4 * q4 + 3]);
      }
      if constexpr (KV) tmem_wait_st();
      tc_fence_before();
      fence_proxy_async_smem();
      mbar_arrive(bar_wc_full);
      if constexpr (HAS_PAR) {
        if (n % per_head == per_head - 1) {  // last tile of this query head
          // Yat: (db, deps) = (acc1, -acc2); s^tau: (deps, dtau) = (acc1, acc2 ln 2)
          float a = acc1.x + acc1.y, e = acc2.x + acc2.y;
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            a += __shfl_xor_sync(FULL, a, o);
            e += __shfl_xor_sync(FULL, e, o);
          }
          if (lane == 0) {
            atomicAdd(p.dpar + 2 * head, (double)a);
            atomicAdd(p.dpar + 2 * head + 1, (double)(VARIANT == kYat ? -e : e * LN2));
          }
          acc1 = make_float2(0.f, 0.f);
          acc2 = acc1;
        }
      }
    }
    if constexpr (DP) {
      // the two column halves' partial sums, then D_t over the aux array's D
      // Yat also replaces the forward's 1 / Z by 1 / (sum kappa + 1e-9) of
      // this pass's own kappas, so that a row's weights, normaliser and D all
      // come from the same kappa (on a row whose only keys have a nearly
      // cancelling numerator, a mismatch between the forward's mass and these
      // kappas reaches the gradient through 2 / (q.k + b))
      xch[hf * RT + r] = dsum.x + dsum.y;
      xch[(NQ + hf) * RT + r] = wsum.x + wsum.y;
      named_barrier_sync(1, MAP_WARPS * 32);
      if (ok && hf == 0 && grow < p.Tq) {
        float D_t = 0.f, W_t = 0.f;
#pragma unroll
        for (int x = 0; x < NQ; ++x) {
          D_t += xch[x * RT + r];
          W_t += xch[(NQ + x) * RT + r];
        }
        float *a = p.aux_w + (size_t)bh_r * p.Tq_pad + grow;
        if (VARIANT == kYat) {
          const float zf = 1.f / row_aux.y;          // the forward's M + 1e-9
          const float inv = 1.f / fmaf(W_t, zf, 1e-9f);  // 1 / (sum kappa + 1e-9)
          a[0] = -D_t * zf * inv * inv;              // -D / Z, D = sum kappa dW / Z
          a[p.aux_plane] = inv;
        } else {
          a[0] = -D_t;
        }
      }
    } else {
    // ---- epilogue: accumulators out of TMEM, Yat's rank-one term, bf16 stores
    if (ok) ok = warp_wait(bar_acc, 0, abort, SITE_MAP | 0x30);
    float esum = 0.f;  // sum e [d2 > 0] over the row (Yat)
    if (VARIANT == kYat) {
      xch[hf * RT + r] = acc0.x + acc0.y;
      named_barrier_sync(1, MAP_WARPS * 32);
#pragma unroll
      for (int x = 0; x < NQ; ++x) esum -= xch[x * RT + r];
    }
    if (ok) {
      tc_fence_after();
      const bool row_ok = KV ? grow < p.Tk : grow < p.Tq;
      // one accumulator: NC columns at TMEM column tcol, rows of dst; rank1:
      // add 2 esum times this row of the resident tile (k_j or q_t, DK wide)
      auto emit = [&](auto nc_c, uint32_t tcol, __nv_bfloat16 *dst, bool rank1) {
        constexpr int NC = decltype(nc_c)::value;
#pragma unroll
        for (int cc = 0; cc < NC / (16 * NQ); ++cc) {
          const int col = hf * (NC / NQ) + 16 * cc;  // this thread's next 16 columns
          uint32_t ar[16];
          tmem_ld16(t_lane + tcol + (uint32_t)col, ar);
          tmem_wait_ld();
          tmem_ld_fence16(ar);
          float v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(ar[i]);
          if (rank1) {
            const float f = 2.f * esum;
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4) {
              const int chunk = ((col & 63) >> 3) + q4;
              const uint4 x = lds128(r_smem + (uint32_t)(col >> 6) * (RT * 128) +
                                     (uint32_t)r * 128u + (uint32_t)((chunk ^ (r & 7)) * 16));
              const uint32_t xs[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float lo = __uint_as_float(xs[u] << 16);
                const float hi = __uint_as_float(xs[u] & 0xffff0000u);
                v[8 * q4 + 2 * u] = fmaf(f, lo, v[8 * q4 + 2 * u]);
                v[8 * q4 + 2 * u + 1] = fmaf(f, hi, v[8 * q4 + 2 * u + 1]);
              }
            }
          }
          if (row_ok) {
#pragma unroll
            for (int q4 = 0; q4 < 2; ++q4)
              stg128(dst + col + 8 * q4, pack_bf16x2(v[8 * q4], v[8 * q4 + 1]),
                     pack_bf16x2(v[8 * q4 + 2], v[8 * q4 + 3]),
                     pack_bf16x2(v[8 * q4 + 4], v[8 * q4 + 5]),
                     pack_bf16x2(v[8 * q4 + 6], v[8 * q4 + 7]));
          }
        }
      };
      if constexpr (KV) {
        emit(std::integral_constant<int, DV>{}, TM_A1,
             reinterpret_cast<__nv_bfloat16 *>(p.dv) + ((size_t)bh_r * p.Tk + grow) * DV, false);
        emit(std::integral_constant<int, DK>{}, TM_A1 + DV,
             reinterpret_cast<__nv_bfloat16 *>(p.dk) + ((size_t)bh_r * p.Tk + grow) * DK,
             VARIANT == kYat);
      } else {
        emit(std::integral_constant<int, DK>{}, TM_A1,
             reinterpret_cast<__nv_bfloat16 *>(p.dq) + ((size_t)bh_r * p.Tq + grow) * DK,
             VARIANT == kYat);
      }
    }
    }  // !DP
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// Per query row, the scalars the map warps read (zeros for the padding rows
// up to Tq_pad): softmax (-D scale, -log2 Z, 0) with D = dout . out; s^tau
// (0, -log2 Z, 0); Yat (0, 1 / Z, |q|^2 + eps), Z = row_mass + 1e-9.  The
// row-sum pass fills the first field for Yat (-D / Z) and s^tau (-D).
// Eight lanes per row.
template <int VARIANT, int DK, int DV>
__global__ void __launch_bounds__(256) bwd_prep_kernel(const __nv_bfloat16 *__restrict__ q,
                                                       const __nv_bfloat16 *__restrict__ out,
                                                       const __nv_bfloat16 *__restrict__ dout,
                                                       const float *__restrict__ row_mass,
                                                       const float *__restrict__ eps,
                                                       float *__restrict__ aux, size_t plane,
                                                       int BH, int h, int Tq, int Tq_pad,
                                                       float scale) {
  const long long row = ((long long)blockIdx.x * 256 + threadIdx.x) >> 3;
  const int sub = threadIdx.x & 7;
  const bool live = row < (long long)BH * Tq_pad;
  const int bh = live ? (int)(row / Tq_pad) : 0;
  const int t = live ? (int)(row % Tq_pad) : 0;
  const bool valid = live && t < Tq;
  float dsum = 0.f, qsum = 0.f;
  if (valid && VARIANT == kSoftmax) {
    const size_t base = ((size_t)bh * Tq + t) * DV;
#pragma unroll
    for (int c = sub * 8; c < DV; c += 64) {
      {
        const uint4 o4 = *reinterpret_cast<const uint4 *>(out + base + c);
        const uint4 d4 = *reinterpret_cast<const uint4 *>(dout + base + c);
        const uint32_t os[4] = {o4.x, o4.y, o4.z, o4.w}, ds[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          dsum = fmaf(__uint_as_float(os[u] << 16), __uint_as_float(ds[u] << 16), dsum);
          dsum = fmaf(__uint_as_float(os[u] & 0xffff0000u), __uint_as_float(ds[u] & 0xffff0000u),
                      dsum);
        }
      }
    }
  }
  if (valid && VARIANT == kYat) {
    const size_t base = ((size_t)bh * Tq + t) * DK;
#pragma unroll
    for (int c = sub * 8; c < DK; c += 64) {
      {
        const uint4 q4 = *reinterpret_cast<const uint4 *>(q + base + c);
        const uint32_t qs[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const float lo = __uint_as_float(qs[u] << 16), hi = __uint_as_float(qs[u] & 0xffff0000u);
          qsum = fmaf(lo, lo, qsum);
          qsum = fmaf(hi, hi, qsum);
        }
      }
    }
  }
#pragma unroll
  for (int o = 4; o > 0; o >>= 1) {
    dsum += __shfl_xor_sync(FULL, dsum, o);
    qsum += __shfl_xor_sync(FULL, qsum, o);
  }
  if (live && sub == 0) {
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    if (valid) {
      const float m = row_mass[(size_t)bh * Tq + t];
      a.x = VARIANT == kSoftmax ? -dsum * scale : 0.f;  // the others: the row-sum pass
      a.y = VARIANT == kYat ? 1.f / (m + 1e-9f) : -m * LOG2E;
      a.z = VARIANT == kYat ? qsum + eps[bh % h] : 0.f;
    }
    aux[row] = a.x;
    aux[plane + row] = a.y;
    aux[2 * plane + row] = a.z;
  }
}

__global__ void bwd_param_finalize(const double *dpar, int h, int variant, float *db, float *deps,
                                   float *dtau) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= h) return;
  const double a = dpar[2 * i], e = dpar[2 * i + 1];
  if (variant == kYat) {
    if (db) db[i] = (float)a;
    if (deps) deps[i] = (float)e;
  } else if (variant == kStau) {
    if (deps) deps[i] = (float)a;
    if (dtau) dtau[i] = (float)e;
  }
}

template <int VARIANT, int DK, int DV, int SIDE, int YM, bool DP = false>
cudaError_t launch_side(const BwdParams &p, const CUtensorMap &r, const CUtensorMap &rp,
                        const CUtensorMap &x, const CUtensorMap &xp, cudaStream_t s) {
  using L = Layout<DK, DV, SIDE>;
  auto kern = bwd_kernel<VARIANT, DK, DV, SIDE, YM, DP>;
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  const long long grid = SIDE == SIDE_KV ? (long long)p.B * p.hkv * p.n_k128
                                         : (long long)p.B * p.h * p.n_q128;
  if (grid <= 0) return cudaSuccess;
  kern<<<(unsigned)grid, NUM_THREADS, L::ALLOC, s>>>(p, r, rp, x, xp);
  return cudaGetLastError();
}

// Yat and s^tau first replace the D of dout . out (from the bf16 forward
// output, whose weights were rounded to bf16 before the PV product) with the
// row sum of the backward's own weights times dW, so that sum_j w_j (dW_j - D)
// is zero for the weights actually used.  Yat's score gradient carries the
// factor 2 / (q.k + b) and s^tau's parameter gradients the factors 1 / phi
// and ln phi: on rows whose mass sits on keys where those are large (a causal
// row's first keys; strongly negative scores) a 2^-9 error in D would be
// amplified far beyond the bf16 tolerance.  Softmax's gradient is bounded by
// w <= 1 and keeps dout . out.
template <int VARIANT, int DK, int DV, int YM>
cudaError_t launch_all(const BwdParams &p, const BwdMaps &m, cudaStream_t s) {
  cudaError_t e = cudaSuccess;
  if constexpr (VARIANT != kSoftmax) {
    e = launch_side<VARIANT, DK, DV, SIDE_Q, YM, true>(p, m.q128, m.do128, m.k64, m.v64, s);
    if (e != cudaSuccess) return e;
  }
  e = launch_side<VARIANT, DK, DV, SIDE_KV, YM>(p, m.k128, m.v128, m.q64, m.do64, s);
  if (e != cudaSuccess) return e;
  return launch_side<VARIANT, DK, DV, SIDE_Q, YM>(p, m.q128, m.do128, m.k64, m.v64, s);
}

template <int VARIANT, int DK, int DV>
cudaError_t launch_prep(const BwdParams &p, const void *q, const void *out, const void *dout,
                        const float *row_mass, cudaStream_t s) {
  const long long rows = (long long)p.B * p.h * p.Tq_pad;
  const unsigned blocks = (unsigned)((rows * 8 + 255) / 256);
  bwd_prep_kernel<VARIANT, DK, DV><<<blocks, 256, 0, s>>>(
      static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(out),
      static_cast<const __nv_bfloat16 *>(dout), row_mass, p.eps, p.aux_w, p.aux_plane,
      p.B * p.h, p.h, p.Tq, p.Tq_pad, p.scale);
  return cudaGetLastError();
}

template <int DK, int DV>
cudaError_t prep_for(int variant, const BwdParams &p, const void *q, const void *out,
                     const void *dout, const float *row_mass, cudaStream_t s) {
  if (variant == kSoftmax) return launch_prep<kSoftmax, DK, DV>(p, q, out, dout, row_mass, s);
  if (variant == kYat) return launch_prep<kYat, DK, DV>(p, q, out, dout, row_mass, s);
  return launch_prep<kStau, DK, DV>(p, q, out, dout, row_mass, s);
}

template <int DK, int DV>
cudaError_t all_for(int variant, int yat_m, const BwdParams &p, const BwdMaps &m,
                    cudaStream_t s) {
  if (variant == kSoftmax) return launch_all<kSoftmax, DK, DV, 1>(p, m, s);
  if (variant == kStau) return launch_all<kStau, DK, DV, 1>(p, m, s);
  if (yat_m == 2) return launch_all<kYat, DK, DV, 2>(p, m, s);
  if (yat_m == 3) return launch_all<kYat, DK, DV, 3>(p, m, s);
  return launch_all<kYat, DK, DV, 1>(p, m, s);
}

}  // namespace bwd

bool bwd_tc_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 128 && dv == 64);
}

cudaError_t launch_bwd_prep(int variant, int dk, int dv, const BwdParams &p, const void *q,
                            const void *out, const void *dout, const float *row_mass,
                            cudaStream_t s) {
  using namespace bwd;
  if (dk == 64) return prep_for<64, 64>(variant, p, q, out, dout, row_mass, s);
  if (dv == 64) return prep_for<128, 64>(variant, p, q, out, dout, row_mass, s);
  return prep_for<128, 128>(variant, p, q, out, dout, row_mass, s);
}

cudaError_t launch_bwd_tc(int variant, int dk, int dv, int yat_m, const BwdParams &p,
                          const BwdMaps &m, cudaStream_t s) {
  using namespace bwd;
  if (dk == 64) return all_for<64, 64>(variant, yat_m, p, m, s);
  if (dv == 64) return all_for<128, 64>(variant, yat_m, p, m, s);
  return all_for<128, 128>(variant, yat_m, p, m, s);
}

cudaError_t launch_bwd_param_finalize(int variant, const double *dpar, int h, float *db,
                                      float *deps, float *dtau, cudaStream_t s) {
  if (variant == kSoftmax || h <= 0) return cudaSuccess;
  bwd::bwd_param_finalize<<<(h + 127) / 128, 128, 0, s>>>(dpar, h, variant, db, deps, dtau);
  return cudaGetLastError();
}

cudaError_t read_and_clear_bwd_status(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_bwd_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(unsigned int));
}

}  // namespace cattn
