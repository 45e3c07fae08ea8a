// fwd_tc.cu -- fused attention forward on the sm_103a tensor cores.
//
// A persistent kernel: one CTA per SM works through a list of units, each
// unit two 128-row query tiles (Q0, Q1) of one (batch, head) -- and, for
// non-causal problems with few units, one split of the keys.  K/V tiles of
// 128 keys stream through shared memory, so every tile that reaches the SM
// serves 256 query rows.  Per key tile j and query tile x:
//
//   S_x = Q_x K_j^T     tcgen05.mma, A and B from shared memory -> TMEM fp32
//   P_x = map(S_x)      eight map warps of tile x: tcgen05.ld S, apply the
//                       score-to-weight map, tcgen05.st P (bf16) over S_x
//   O_x += P_x V_j      tcgen05.mma, A = P from TMEM, B = V from shared memory
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
// Schedule.  The producer warp hands out units: its CTA's first unit is
// blockIdx.x, every later one comes from an atomic ticket in the workspace,
// so CTAs that drew light units take more of them.  Units are ordered so that
// the units of a group of (batch, head) pairs run together (their K/V stays in
// L2) and, for causal problems, heaviest first.  A two-entry unit ring in
// shared memory passes each unit number to the MMA warp and the map warps.
// Key splits leave unnormalised partial outputs and per-row statistics in the
// workspace; a small combine kernel merges them (Yat: plain sums of O and of
// the mass; softmax and s^tau: onto the largest running max first).
//
// TMEM (512 columns): S0 [0,128) S1 [128,256) O0 [256,384) O1 [384,512).  P_x
// is written over S_x; the MMA pipe executes a CTA's MMAs in issue order, so
// PV_x(j) reads P_x before S_x(j+1) lands, and the commit that signals S_x(j)
// also covers PV_x(j-1).  The MMA order PV0(j-1) S0(j) PV1(j-1) S1(j) lets
// one query tile's MMAs run while the other tile is being mapped.  For Yat
// and s^tau each PV is issued in two halves: the map warps signal once the
// first 32-key chunk of their P is written, so half of PV_x runs while they
// map the second chunk and only the other half stands between the map and
// S_x(j+1).  (PV reads P from TMEM, and that form of the MMA runs markedly
// slower than one with both operands in shared memory, so its latency is
// worth hiding.)  Between units the next unit's S MMAs follow the last PVs
// at once; its first PV_x waits (o_empty) until the map warps have read O_x
// out.
//
// Warp roles (576 threads): warps 0-15 map (warp w: query tile x = w/8, TMEM
// lanes 32*(w%4)..+31 = those query rows, key columns [64h, 64h+64) with
// h = (w/4)%2, so each tile has two warps per SM sub-partition), warp 16 issues
// TMA loads, warp 17 allocates TMEM and issues the MMAs (lane 0).  K and V
// tiles share one ring of shared-memory slots guarded by full/empty mbarriers;
// the squared key norms of the Yat map ride in a small ring of their own.
//
// Every mbarrier wait is bounded (2 s of %globaltimer); on expiry the kernel
// records a site code in g_status, raises a CTA-wide abort flag, and all roles
// leave their loops so that TMEM is still released.
#include <cuda_bf16.h>

#include <type_traits>

#include "kernels.h"
#include "maps.cuh"
#include "ptx.cuh"

namespace cattn {

__device__ unsigned int g_status;

#ifdef CATTN_TRACE
// Optional clock64 timeline of the first CTAs' steps (compiled out by
// default): [CTA][event][running step].
__device__ unsigned long long g_trace[4][16][512];
extern "C" int cattn_trace_read(void *host, size_t bytes) {
  return (int)cudaMemcpyFromSymbol(host, g_trace, bytes);
}
#define CATTN_TR(ev, idx)                                                     \
  do {                                                                        \
    if (blockIdx.x < 4 && (idx) < 512) g_trace[blockIdx.x][ev][(idx)] = clock64(); \
  } while (0)
#else
#define CATTN_TR(ev, idx) \
  do {                    \
  } while (0)
#endif


namespace tc {

constexpr int BM = kTcQueryTile;  // 128 query rows per tile
constexpr int BN = kTcKeyTile;    // 128 keys per tile
constexpr int NUM_THREADS = 576;
constexpr int MAP_WARPS = 16;
constexpr int PRODUCER_WARP = 16;
constexpr int MMA_WARP = 17;
constexpr int NKS = 4;  // stages of the key-norm ring
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;
// the limit of the test-only wait that nothing completes (FwdParams::test_stall)
constexpr uint64_t STALL_LIMIT_NS = 20000000ull;
constexpr unsigned FULL = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;
constexpr float LN2 = 0.6931471805599453f;
constexpr float RESCALE_THRESHOLD = 8.0f;  // log2 units

// TMEM column map: S_x (and P_x over it) at 128 x, O_x at 256 + 128 x.  Keys
// [64h, 64h+64) of P_x sit at columns [64h, 64h+32) of S_x.
constexpr uint32_t TM_S = 0;
constexpr uint32_t TM_O = 256;

// wait-site codes recorded in g_status
enum : unsigned {
  SITE_PRODUCER = 0x100,
  SITE_MMA = 0x200,
  SITE_EPI = 0x300,
};

template <int DK, int DV>
struct Layout {
  static constexpr int Q_TILE = BM * DK * 2;
  static constexpr int K_TILE = BN * DK * 2;
  static constexpr int V_TILE = BN * DV * 2;
  static constexpr int SLOT = K_TILE > V_TILE ? K_TILE : V_TILE;
  static constexpr int NS = DK == 64 ? 8 : 4;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_RING = OFF_Q + 2 * Q_TILE;
  static constexpr int OFF_NK = OFF_RING + NS * SLOT;
  // row-max exchange of the two column halves: per tile [2 uses][2 tiles][2 halves][BM],
  // final [2 tiles][2 values][2 halves][BM], the entropy sums [2 tiles][2 halves][BM]
  static constexpr int OFF_XCHG = OFF_NK + NKS * BN * 4;
  // (the row statistics pass uses [13 values][2 tiles][BM] of it)
  static constexpr int XCHG_FLOATS = 26 * BM;
  // one-launch Yat forward: each map warp's key norms of the current tile
  // (BN floats per warp, its 64 keys filled), the unit's rows listed for the
  // near-key recompute and their count
  static constexpr int OFF_NKU = OFF_XCHG + XCHG_FLOATS * 4;
  static constexpr int OFF_NEAR = OFF_NKU + MAP_WARPS * BN * 4;
  static constexpr int OFF_NEAR_N = OFF_NEAR + 2 * BM * 4;
  static constexpr int OFF_BAR = OFF_NEAR_N + 16;
  // q_full, q_empty, kv_full[NS], kv_empty[NS], nk_full[NKS], nk_empty[NKS],
  // s_full[2], p_full[2], o_full[2], o_empty[2], unit_full[2], unit_empty[2], drain,
  // p_half[2], never (nothing arrives on it: the test-only stall), and for the
  // one-launch Yat forward rows_done (every row of the unit written)
  static constexpr int NBAR = 2 + 2 * NS + 2 * NKS + 17;
  static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
  // TMEM base address, abort flag, unit ring[2]
  static constexpr int BYTES = OFF_MISC + 16;
  static constexpr int ALLOC = BYTES + 1024;  // room to align the base to 1024 B
  static_assert(ALLOC <= 227 * 1024, "shared memory budget");
  static_assert(SLOT % 1024 == 0 && Q_TILE % 1024 == 0, "swizzle atoms stay 1024-B aligned");
};

// Warp-collective bounded wait.  Every lane polls (so every lane acquires the
// phase), the exit decision is warp-uniform.  Returns false on timeout/abort.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          unsigned site, bool honor_abort = true,
                                          uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (__all_sync(FULL, mbar_try_wait(bar, parity))) return true;
    const int bad = (honor_abort && *abort != 0) || (globaltimer_ns() - t0 > limit_ns);
    if (__any_sync(FULL, bad)) {
      if ((threadIdx.x & 31) == 0) {
        atomicCAS(&g_status, 0u, site | 1u);
        *abort = 1;
      }
      return false;
    }
  }
}

// Single-thread bounded wait (the MMA issuer runs on one lane).  Returns
// false on timeout or abort.
__device__ __forceinline__ bool thread_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                            unsigned site, bool honor_abort = true,
                                            uint64_t limit_ns = WAIT_LIMIT_NS) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((honor_abort && *abort != 0) || (globaltimer_ns() - t0 > limit_ns)) {
      atomicCAS(&g_status, 0u, site | 1u);
      *abort = 1;
      return false;
    }
  }
}

// S = Q K^T for one 128 x 128 tile from prebuilt descriptors of the Q tile
// and the K slot: 16-element k steps, 64-column boxes.
// CONV: issued by a converged MMA warp (elected lane), else by one lane.
template <int DK, bool CONV = false>
__device__ __forceinline__ void issue_qk_d(uint32_t d_tmem, uint64_t qdesc, uint64_t kdesc) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false);
#pragma unroll
  for (int kk = 0; kk < DK / 16; ++kk) {
    const uint64_t qo = (uint64_t)(((kk >> 2) * (BM * 128) + (kk & 3) * 32) >> 4);
    const uint64_t ko = (uint64_t)(((kk >> 2) * (BN * 128) + (kk & 3) * 32) >> 4);
    if constexpr (CONV)
      mma_ss_e(d_tmem, qdesc + qo, kdesc + ko, IDESC, kk > 0 ? 1u : 0u);
    else
      mma_ss(d_tmem, qdesc + qo, kdesc + ko, IDESC, kk > 0 ? 1u : 0u);
  }
}

// Half of O += P V: PART 0 takes keys [0, 32) and [64, 96) (the first
// 32-key chunk of each column half, which the map warps finish first), PART 1
// the other two chunks.
template <int DV, int PART, bool CONV = false>
__device__ __forceinline__ void issue_pv_part(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc,
                                              bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, DV, true);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int kk = (i >> 1) * 4 + PART * 2 + (i & 1);
    (CONV ? mma_ts_e : mma_ts)(d_tmem, p_tmem + (uint32_t)(kk >> 2) * 64 + (uint32_t)(kk & 3) * 8,
           vdesc + (uint64_t)((kk * 2048) >> 4), IDESC, (accumulate || PART == 1 || i > 0) ? 1u : 0u);
  }
}

// O += P V from a prebuilt descriptor of the V slot.
template <int DV, bool CONV = false>
__device__ __forceinline__ void issue_pv_d(uint32_t d_tmem, uint32_t p_tmem, uint64_t vdesc,
                                           bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, DV, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    (CONV ? mma_ts_e : mma_ts)(d_tmem, p_tmem + (uint32_t)(kk >> 2) * 64 + (uint32_t)(kk & 3) * 8,
           vdesc + (uint64_t)((kk * 2048) >> 4), IDESC, (accumulate || kk > 0) ? 1u : 0u);
  }
}

// S = Q K^T for one 128 x 128 tile: 16-element k steps, 64-column boxes.
template <int DK>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint32_t q_smem, uint32_t k_smem) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, BN, false);
#pragma unroll
  for (int kk = 0; kk < DK / 16; ++kk) {
    const uint32_t qa = q_smem + (uint32_t)(kk >> 2) * (BM * 128) + (uint32_t)(kk & 3) * 32;
    const uint32_t ka = k_smem + (uint32_t)(kk >> 2) * (BN * 128) + (uint32_t)(kk & 3) * 32;
    mma_ss(d_tmem, smem_desc_sw128(qa, 16, 1024), smem_desc_sw128(ka, 16, 1024), IDESC,
           kk > 0 ? 1u : 0u);
  }
}

// O += P V for one 128-key tile; P (bf16 pairs) over S (keys [64h, 64h+64)
// at columns [64h, 64h+32)), V N-major with its 64-wide dv boxes BN*128 bytes
// apart.
template <int DV>
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint32_t p_tmem, uint32_t v_smem,
                                         bool accumulate) {
  constexpr uint32_t IDESC = idesc_bf16_f32(BM, DV, true);
#pragma unroll
  for (int kk = 0; kk < BN / 16; ++kk) {
    mma_ts(d_tmem, p_tmem + (uint32_t)(kk >> 2) * 64 + (uint32_t)(kk & 3) * 8,
           smem_desc_sw128(v_smem + (uint32_t)kk * 2048, BN * 128, 1024), IDESC,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

// Multiply dv/2 columns of this thread's row of O by f in place, 16 columns
// at a time (for callers that still hold other registers).
template <int DV>
__device__ __forceinline__ void scale_o_half16(uint32_t t_o, float f) {
#pragma unroll
  for (int c = 0; c < DV / 32; ++c) {
    uint32_t r[16];
    tmem_ld16(t_o + c * 16, r);
    tmem_wait_ld();
#pragma unroll
    for (int i = 0; i < 16; ++i) asm volatile("" : "+r"(r[i])::"memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
    tmem_st16(t_o + c * 16, r);
  }
}

// Multiply dv/2 columns of this thread's row of O by f in place.
template <int DV>
__device__ __forceinline__ void scale_o_half(uint32_t t_o, float f) {
#pragma unroll
  for (int c = 0; c < DV / 64; ++c) {
    uint32_t r[32];
    tmem_ld32(t_o + c * 32, r);
    tmem_wait_ld();
    tmem_ld_fence(r);
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __float_as_uint(__uint_as_float(r[i]) * f);
    tmem_st32(t_o + c * 32, r);
  }
}

// One work unit: (batch*head, query-tile pair, key split), decoded the same
// way by every role.
struct Unit {
  int bh, batch, head, bh_kv;
  int q0;          // first query row of the pair
  int split;       // key split (0 without splits)
  int kv_begin;    // first key tile
  int n[2];        // key tiles of query tile 0 and 1 (0: the tile does not exist)
  int nkv;         // key tiles loaded for the pair: max(n[0], n[1])
};

// Units are ordered group by group of p.head_group (batch, head) pairs; inside
// a group by pair (causal: heaviest first), then split, then (batch, head).  A
// group's K/V stays in L2 while its units run, and the light units come last.
__device__ __forceinline__ Unit decode_unit(const FwdParams &p, int u) {
  Unit t;
  const int BH = p.B * p.h;
  const int per_bh = p.n_pairs * p.n_splits;
  const int g = u / (p.head_group * per_bh);
  const int base = g * p.head_group;
  const int gs = min(p.head_group, BH - base);
  int rem = u - g * p.head_group * per_bh;
  const int pp = rem / (p.n_splits * gs);
  rem -= pp * p.n_splits * gs;
  t.split = rem / gs;
  t.bh = base + (rem - t.split * gs);
  const int pair = p.causal ? p.n_pairs - 1 - pp : pp;
  t.head = t.bh % p.h;
  t.batch = t.bh / p.h;
  t.bh_kv = t.batch * p.hkv + t.head / (p.h / p.hkv);
  t.q0 = pair * 2 * BM;
  const bool q1_valid = (t.q0 + BM) < p.Tq;
  if (p.causal) {  // keys 0 .. last row of the query tile
    t.kv_begin = 0;
    t.n[0] = min(2 * pair + 1, p.n_kv_tiles);
    t.n[1] = q1_valid ? min(2 * pair + 2, p.n_kv_tiles) : 0;
  } else {
    t.kv_begin = t.split * p.kv_per_split;
    t.n[0] = min(p.n_kv_tiles - t.kv_begin, p.kv_per_split);
    t.n[1] = q1_valid ? t.n[0] : 0;
  }
  t.nkv = max(t.n[0], t.n[1]);
  return t;
}

// YM: Yat numerator exponent 2 YM (1 for the other maps).  STATS: the row
// statistics pass (no V, no PV, no O; the weights' statistics per row).
// ENT: the forward also accumulates each row's sum f log2 f of its weights'
// numerators f (Yat kappa; softmax, s^tau 2^(x - m) on the running max m) and
// writes the row's normalised entropy.
// Squared norms of keys 64 half + lane and 64 half + 32 + lane of a K tile
// in shared memory (rows of DK bf16 in 64-column boxes BN rows apart, each
// 128-byte box row swizzled in 16-byte units; the sum does not depend on
// where a unit sits, and the order of a row's units is rotated by lane so
// that a warp's loads fall in distinct banks): written to nkw at those key
// offsets; returns the largest over the warp's 64 keys (zero rows past Tk
// give zero).
template <int DK>
__device__ __forceinline__ float inorm_tile_norms(uint32_t slot, int half, int lane, float *nkw) {
  float mx = 0.f;
#pragma unroll
  for (int h2 = 0; h2 < 2; ++h2) {
    const int key = 64 * half + 32 * h2 + lane;
    float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
    for (int c = 0; c < DK / 64; ++c) {
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const uint4 v = lds128(slot + (uint32_t)(c * (BN * 128) + key * 128) +
                               ((uint32_t)((k + lane) & 7) << 4));
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = make_float2(__uint_as_float(w4[e] << 16), __uint_as_float(w4[e] & 0xffff0000u));
          s2 = __ffma2_rn(f, f, s2);
        }
      }
    }
    const float nrm = s2.x + s2.y;
    nkw[key] = nrm;
    mx = fmaxf(mx, nrm);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
  return mx;
}

// One row of the Yat map by its plain definition, by one warp (the lanes
// share the components of q and k and the columns of v; the keys in order):
// the output row, its mass and max kappa (the near-key recompute of the
// one-launch path; the separate near-key pass spreads a row over 8 warps).
template <int DK, int DV, int YM>
__device__ __noinline__ void near_row_warp(const FwdParams &p, int bh, int row, int lane) {
  constexpr int QE = DK / 32, VE = DV / 32;
  if (row >= p.Tq) return;
  const int head = bh % p.h, batch = bh / p.h;
  const size_t bh_kv = (size_t)batch * p.hkv + head / (p.h / p.hkv);
  const float b = p.b[head], eps = p.eps[head];
  const __nv_bfloat16 *qg = static_cast<const __nv_bfloat16 *>(p.q);
  const __nv_bfloat16 *kg = static_cast<const __nv_bfloat16 *>(p.k);
  const __nv_bfloat16 *vg = static_cast<const __nv_bfloat16 *>(p.v);
  float qf[QE];
#pragma unroll
  for (int i = 0; i < QE; ++i)
    qf[i] = __bfloat162float(qg[((size_t)bh * p.Tq + row) * DK + lane * QE + i]);
  const int lim = p.causal ? min(row + 1, p.Tk) : p.Tk;
  float mass = 0.f, top = 0.f, o[VE];
#pragma unroll
  for (int c = 0; c < VE; ++c) o[c] = 0.f;
  for (int j = 0; j < lim; ++j) {
    const __nv_bfloat16 *kr = kg + (bh_kv * p.Tk + j) * DK + lane * QE;
    float dot = 0.f, d2 = 0.f;
#pragma unroll
    for (int i = 0; i < QE; ++i) {
      const float kf = __bfloat162float(kr[i]);
      dot = fmaf(qf[i], kf, dot);
      const float df = qf[i] - kf;
      d2 = fmaf(df, df, d2);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      dot += __shfl_xor_sync(FULL, dot, off);
      d2 += __shfl_xor_sync(FULL, d2, off);
    }
    const float tt = dot + b;
    float num = tt * tt;
    if constexpr (YM == 2) num = num * num;
    if constexpr (YM == 3) num = num * num * num;
    const float kap = num / (fmaxf(d2, 0.f) + eps);
    mass += kap;
    top = fmaxf(top, kap);
    const __nv_bfloat16 *vr = vg + (bh_kv * p.Tk + j) * DV + lane * VE;
#pragma unroll
    for (int c = 0; c < VE; ++c) o[c] = fmaf(kap, __bfloat162float(vr[c]), o[c]);
  }
  const float inv = 1.f / (mass + 1e-9f);
  const size_t ti = (size_t)bh * p.Tq + row;
  __nv_bfloat16 *orow = static_cast<__nv_bfloat16 *>(p.out) + ti * DV + lane * VE;
#pragma unroll
  for (int c = 0; c < VE; ++c) orow[c] = __float2bfloat16_rn(o[c] * inv);
  if (lane == 0) {
    if (p.row_mass) p.row_mass[ti] = mass;
    if (p.row_max) p.row_max[ti] = top;
  }
}

// INORM: the one-launch Yat forward for problems whose units all run in one
// wave with short rows (one unit per CTA, no key splits, key tiles x dk <=
// 256): the map warps take each key tile's norms from the K tile in shared
// memory, and recompute the rows they flag for the near-key guard at the
// unit's end, so no other launch is needed.
template <int VARIANT, int DK, int DV, int YM = 1, bool STATS = false, bool ENT = false,
          bool INORM = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    fwd_kernel(const __grid_constant__ FwdParams p, const __grid_constant__ CUtensorMap tm_q,
               const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v) {
  using L = Layout<DK, DV>;
  static_assert(!INORM || (VARIANT == kYat && !STATS && !ENT), "one-launch path: Yat forward only");
  // Yat and s^tau split each PV in two: half of it runs while the map warps
  // work on the second half of P (softmax, whose map is the shortest, keeps
  // one PV and its rescale after the map)
  constexpr bool SPLIT_PV = VARIANT == kYat || VARIANT == kStau;
  // the tau* pass (kTau) and the row statistics pass read no V and issue no
  // PV: one ring slot per key tile
  constexpr bool HAS_V = VARIANT != kTau && !STATS;
  constexpr uint32_t STEP = HAS_V ? 2u : 1u;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_s = smem_u32(smem_raw);
  uint8_t *smem = smem_raw + ((1024u - (raw_s & 1023u)) & 1023u);
  const uint32_t sb = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const uint32_t bar0 = sb + L::OFF_BAR;
  const uint32_t bar_q_full = bar0;
  const uint32_t bar_q_empty = bar0 + 8u;
  auto kv_full = [&](uint32_t s) { return bar0 + 8u * (2 + s); };
  auto kv_empty = [&](uint32_t s) { return bar0 + 8u * (2 + L::NS + s); };
  auto nk_full = [&](uint32_t s) { return bar0 + 8u * (2 + 2 * L::NS + s); };
  auto nk_empty = [&](uint32_t s) { return bar0 + 8u * (2 + 2 * L::NS + NKS + s); };
  constexpr int B2 = 2 + 2 * L::NS + 2 * NKS;
  auto s_full = [&](int x) { return bar0 + 8u * (B2 + x); };
  auto p_full = [&](int x) { return bar0 + 8u * (B2 + 2 + x); };
  auto o_full = [&](int x) { return bar0 + 8u * (B2 + 4 + x); };
  auto o_empty = [&](int x) { return bar0 + 8u * (B2 + 6 + x); };
  auto unit_full = [&](uint32_t s) { return bar0 + 8u * (B2 + 8 + s); };
  auto unit_empty = [&](uint32_t s) { return bar0 + 8u * (B2 + 10 + s); };
  const uint32_t bar_drain = bar0 + 8u * (B2 + 12);
  auto p_half = [&](int x) { return bar0 + 8u * (B2 + 13 + x); };
  const uint32_t bar_never = bar0 + 8u * (B2 + 15);
  const uint32_t bar_rows_done = bar0 + 8u * (B2 + 16);
  float *nku = reinterpret_cast<float *>(smem + L::OFF_NKU);
  unsigned int *near_list = reinterpret_cast<unsigned int *>(smem + L::OFF_NEAR);
  unsigned int *near_n = reinterpret_cast<unsigned int *>(smem + L::OFF_NEAR_N);
  auto q_smem = [&](int x) { return sb + L::OFF_Q + (uint32_t)x * L::Q_TILE; };
  auto slot_smem = [&](uint32_t s) { return sb + L::OFF_RING + s * L::SLOT; };
  const float *nk_ring = reinterpret_cast<const float *>(smem + L::OFF_NK);
  uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + L::OFF_MISC);
  volatile int *abort = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 4);
  volatile int *unit_ring = reinterpret_cast<volatile int *>(smem + L::OFF_MISC + 8);

  if (threadIdx.x == 0) {
    mbar_init(bar_q_full, 1);
    // the last S MMAs of a unit, plus (Yat) every map warp once it has read
    // its row's |q|^2 out of the Q tile
    mbar_init(bar_q_empty, VARIANT == kYat ? 1 + MAP_WARPS : 1);
    for (int s = 0; s < L::NS; ++s) {
      mbar_init(kv_full(s), 1);
      // one-launch Yat: a K slot (the even positions) is also released by
      // every map warp once it has taken its keys' norms out of it
      mbar_init(kv_empty(s), INORM && (s % 2) == 0 ? 1 + MAP_WARPS : 1);
    }
    for (int s = 0; s < NKS; ++s) {
      mbar_init(nk_full(s), 1);
      mbar_init(nk_empty(s), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), 8 * 32);  // every thread of the eight map warps of tile x
      mbar_init(p_half(x), 8 * 32);  // the same, once the first chunk of P is written (Yat, s^tau)
      mbar_init(o_full(x), 1);
      mbar_init(o_empty(x), 8);      // lane 0 of each of those warps
      mbar_init(unit_full(x), 1);
      mbar_init(unit_empty(x), 1 + MAP_WARPS);  // the MMA lane and every map warp
    }
    mbar_init(bar_drain, 1);
    mbar_init(bar_never, 1);
    mbar_init(bar_rows_done, MAP_WARPS);  // lane 0 of every map warp
    *near_n = 0u;
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

  // Every consumer role reads unit number uc from the two-entry unit ring
  // (-1 at the end of the schedule, or on abort) and releases the entry when
  // it has finished the unit, so the entry stays readable meanwhile.
  auto peek_unit = [&](uint32_t uc, unsigned site) -> int {
    if (!warp_wait(unit_full(uc & 1u), (uc >> 1) & 1u, abort, site)) return -1;
    return unit_ring[uc & 1u];
  };
  auto release_unit = [&](uint32_t uc) {
    __syncwarp();
    if (lane == 0) mbar_arrive(unit_empty(uc & 1u));
  };

  if (warp == PRODUCER_WARP) {
    // ------------------------------------------------------------ producer
    // One lane hands out units (its CTA's first unit is blockIdx.x, later
    // ones come from the global ticket, fetched one unit ahead so that the
    // atomic's latency hides behind the current unit's loads) and loads each
    // unit's Q pair, then its K/V tiles (and key norms) through the rings.
    // Ring positions run on across units.
    if (lane == 0) {
      int u = blockIdx.x;
      uint32_t kv_pos = 0, nk_pos = 0;
      // copies started: Q pairs, K/V ring positions, key-norm ring positions
      uint32_t q_armed = 0, kv_issued = 0, nk_issued = 0;
      for (uint32_t uc = 0;; ++uc) {
        const uint32_t us = uc & 1u;
        if (!thread_wait(unit_empty(us), ((uc >> 1) & 1u) ^ 1u, abort, SITE_PRODUCER | 0x40)) break;
        unit_ring[us] = u < p.n_units ? u : -1;
        mbar_arrive(unit_full(us));
        if (u >= p.n_units) break;
        const Unit t = decode_unit(p, u);
        // the previous unit's last S MMAs have read both Q tiles
        if (!thread_wait(bar_q_empty, (uc & 1u) ^ 1u, abort, SITE_PRODUCER | 0x50)) break;
        mbar_arrive_expect_tx(bar_q_full, (t.n[1] > 0 ? 2u : 1u) * (uint32_t)L::Q_TILE);
#pragma unroll
        for (int c = 0; c < DK / 64; ++c) {
          tma_load_3d(q_smem(0) + c * BM * 128, &tm_q, c * 64, t.q0, t.bh, bar_q_full);
          if (t.n[1] > 0)
            tma_load_3d(q_smem(1) + c * BM * 128, &tm_q, c * 64, t.q0 + BM, t.bh, bar_q_full);
        }
        ++q_armed;
        bool ok = true;
        for (int j = 0; j < t.nkv; ++j) {
          const int jt = t.kv_begin + j;  // key tile
          {  // K
            const uint32_t pos = kv_pos + STEP * j, s = pos % L::NS;
            if (!(ok = thread_wait(kv_empty(s), ((pos / L::NS) & 1u) ^ 1u, abort,
                                   SITE_PRODUCER | 0x10)))
              break;
            mbar_arrive_expect_tx(kv_full(s), L::K_TILE);
#pragma unroll
            for (int c = 0; c < DK / 64; ++c)
              tma_load_3d(slot_smem(s) + c * BN * 128, &tm_k, c * 64, jt * BN, t.bh_kv, kv_full(s));
            kv_issued = pos + 1;
          }
          if (VARIANT == kYat && !INORM) {  // squared key norms of the tile
            const uint32_t pos = nk_pos + j, s = pos % NKS;
            if (!(ok = thread_wait(nk_empty(s), ((pos / NKS) & 1u) ^ 1u, abort,
                                   SITE_PRODUCER | 0x20)))
              break;
            mbar_arrive_expect_tx(nk_full(s), BN * 4);
            bulk_load(sb + L::OFF_NK + s * BN * 4,
                      p.nk + (size_t)t.bh_kv * p.Tk_pad + (size_t)jt * BN, BN * 4, nk_full(s));
            nk_issued = pos + 1;
          }
          if (HAS_V) {  // V
            const uint32_t pos = kv_pos + 2u * j + 1u, s = pos % L::NS;
            if (!(ok = thread_wait(kv_empty(s), ((pos / L::NS) & 1u) ^ 1u, abort,
                                   SITE_PRODUCER | 0x30)))
              break;
            mbar_arrive_expect_tx(kv_full(s), L::V_TILE);
#pragma unroll
            for (int c = 0; c < DV / 64; ++c)
              tma_load_3d(slot_smem(s) + c * BN * 128, &tm_v, c * 64, jt * BN, t.bh_kv, kv_full(s));
            kv_issued = pos + 1;
          }
        }
        if (!ok) break;
        kv_pos += STEP * t.nkv;
        nk_pos += t.nkv;
        // with no more units than CTAs every unit was handed out at launch
        // and the ticket is never read (nor needs zeroing)
        u = p.n_units <= (int)gridDim.x ? p.n_units
                                        : (int)atomicAdd(p.tile_counter, 1u) + (int)gridDim.x;
      }
      {
        // every copy this lane started lands in shared memory before the CTA
        // can exit: long since consumed when the schedule ran to its end,
        // possibly still in flight after an abort (each the latest use of its
        // barrier; bounded waits that ignore the abort flag)
        if (q_armed > 0)
          thread_wait(bar_q_full, (q_armed - 1u) & 1u, abort, SITE_PRODUCER | 0x60, false);
        for (uint32_t pos = kv_issued > (uint32_t)L::NS ? kv_issued - L::NS : 0u; pos < kv_issued; ++pos)
          thread_wait(kv_full(pos % L::NS), (pos / L::NS) & 1u, abort, SITE_PRODUCER | 0x60, false);
        for (uint32_t pos = nk_issued > (uint32_t)NKS ? nk_issued - NKS : 0u; pos < nk_issued; ++pos)
          thread_wait(nk_full(pos % NKS), (pos / NKS) & 1u, abort, SITE_PRODUCER | 0x60, false);
      }
    }
  } else if (warp == MMA_WARP) {
    // ------------------------------------------------------------ MMA issue
    // Per unit, iteration j: PV0(j-1) S0(j) PV1(j-1) S1(j).  The softmax
    // forward runs the warp converged with an elected lane issuing each MMA
    // and commit (its descriptors then live in uniform registers, which
    // measured 8% faster); the other maps issue from lane 0 alone, which
    // measured about 1% faster for them (their split PV adds waits, each
    // polled by every lane of a converged warp).
    // The next unit's S MMAs follow the last PVs of this one directly; its
    // first PV_x waits until the map warps have read O_x out.  Shared-memory
    // descriptors are built once; a slot's descriptor is the base plus the
    // slot offset in 16-byte units.
    constexpr bool CONV = VARIANT == kSoftmax && !STATS;
    auto mwait = [&](uint32_t bar, uint32_t parity, unsigned site, bool honor = true) {
      return CONV ? warp_wait(bar, parity, abort, site, honor)
                  : thread_wait(bar, parity, abort, site, honor);
    };
    auto mcommit = [&](uint32_t bar) {
      if constexpr (CONV)
        mma_commit_e(bar);
      else
        mma_commit(bar);
    };
    if (CONV || lane == 0) {
      const uint64_t dq0 = smem_desc_sw128(q_smem(0), 16, 1024);
      const uint64_t dq1 = smem_desc_sw128(q_smem(1), 16, 1024);
      const uint64_t dk0 = smem_desc_sw128(slot_smem(0), 16, 1024);
      const uint64_t dv0 = smem_desc_sw128(slot_smem(0), BN * 128, 1024);
      constexpr uint32_t SLOT16 = L::SLOT >> 4;
      uint32_t kv_pos = 0, nk_pos = 0, pph = 0u, ou = 0u;  // bit x: tile x
      bool ok = true;
#ifdef CATTN_TRACE
      int ms = 0;  // running MMA iteration
#endif
      for (uint32_t uc = 0; ok; ++uc) {
        if (uc == 0 && p.test_stall) {
          // test-only: a wait on a barrier that nothing arrives on runs out
          // after a short limit, and every role takes the abort path
          ok = CONV ? warp_wait(bar_never, 0u, abort, SITE_MMA | 0x80, true, STALL_LIMIT_NS)
                    : thread_wait(bar_never, 0u, abort, SITE_MMA | 0x80, true, STALL_LIMIT_NS);
          if (!ok) break;
        }
        if (!mwait(unit_full(uc & 1u), (uc >> 1) & 1u, SITE_MMA | 0x70)) break;
        const int u = unit_ring[uc & 1u];
        if (u < 0) break;
        const Unit t = decode_unit(p, u);
        if (CONV) __syncwarp();
        if (!CONV || lane == 0) mbar_arrive(unit_empty(uc & 1u));  // the unit is decoded
        if (!(ok = mwait(bar_q_full, uc & 1u, SITE_MMA | 0x10))) break;
        for (int j = 0; ok && j <= t.nkv; ++j) {
          const uint32_t vpos = kv_pos + 2u * j - 1u, vs = vpos % L::NS;
          const uint32_t kpos = kv_pos + STEP * j, ks = kpos % L::NS;
          if (HAS_V && j >= 1 &&
              !(ok = mwait(kv_full(vs), (vpos / L::NS) & 1u, SITE_MMA | 0x20)))
            break;
#pragma unroll
          for (int x = 0; x < 2; ++x) {
            if (!HAS_V) {  // tau*: S_x(j) may land once the map warps have read S_x(j-1)
              if (j >= 1 && j - 1 < t.n[x]) {
                if (!(ok = mwait(p_full(x), (pph >> x) & 1u, SITE_MMA | 0x30))) break;
                pph ^= 1u << x;
              }
            } else if (j >= 1 && j - 1 < t.n[x] && SPLIT_PV) {  // O_x += P_x(j-1) V(j-1), in two halves
              if (!(ok = mwait(p_half(x), (pph >> x) & 1u, SITE_MMA | 0x34))) break;
              if (j == 1 &&
                  !(ok = mwait(o_empty(x), ((ou >> x) & 1u) ^ 1u, SITE_MMA | 0x50)))
                break;
              tc_fence_after();
#ifdef CATTN_TRACE
              CATTN_TR(4 + 2 * x, ms);
#endif
              issue_pv_part<DV, 0, CONV>(tmem + TM_O + 128u * x, tmem + TM_S + 128u * x,
                                   dv0 + vs * SLOT16, j > 1);
              if (!(ok = mwait(p_full(x), (pph >> x) & 1u, SITE_MMA | 0x30))) break;
              pph ^= 1u << x;
              tc_fence_after();
              issue_pv_part<DV, 1, CONV>(tmem + TM_O + 128u * x, tmem + TM_S + 128u * x,
                                   dv0 + vs * SLOT16, true);
              if (j == t.n[x]) mcommit(o_full(x));
            } else if (j >= 1 && j - 1 < t.n[x]) {  // O_x += P_x(j-1) V(j-1)
              if (!(ok = mwait(p_full(x), (pph >> x) & 1u, SITE_MMA | 0x30))) break;
              pph ^= 1u << x;
              if (j == 1 &&
                  !(ok = mwait(o_empty(x), ((ou >> x) & 1u) ^ 1u, SITE_MMA | 0x50)))
                break;
              tc_fence_after();
#ifdef CATTN_TRACE
              CATTN_TR(4 + 2 * x, ms);
#endif
              issue_pv_d<DV, CONV>(tmem + TM_O + 128u * x, tmem + TM_S + 128u * x, dv0 + vs * SLOT16,
                             j > 1);
              if (j == t.n[x]) mcommit(o_full(x));
            }
            if (x == 0 && j < t.nkv &&
                !(ok = mwait(kv_full(ks), (kpos / L::NS) & 1u, SITE_MMA | 0x40)))
              break;
            if (j < t.n[x]) {  // S_x = Q_x K(j)^T
              tc_fence_after();
#ifdef CATTN_TRACE
              CATTN_TR(5 + 2 * x, ms);
#endif
              issue_qk_d<DK, CONV>(tmem + TM_S + 128u * x, x ? dq1 : dq0, dk0 + ks * SLOT16);
              mcommit(s_full(x));
            }
          }
          if (!ok) break;
          if (j == t.nkv - 1) mcommit(bar_q_empty);  // the unit's last S MMAs
          if (j < t.nkv) mcommit(kv_empty(ks));
          if (HAS_V && j >= 1) mcommit(kv_empty(vs));
          // every map warp delivered P for tile j-1, so all are done with its key norms
          if (VARIANT == kYat && !INORM && j >= 1 && (!CONV || lane == 0))
            mbar_arrive(nk_empty((nk_pos + j - 1) % NKS));
#ifdef CATTN_TRACE
          ++ms;
#endif
        }
        kv_pos += STEP * t.nkv;
        nk_pos += t.nkv;
        ou ^= (t.n[0] > 0 ? 1u : 0u) | (t.n[1] > 0 ? 2u : 0u);
      }
      // all MMAs issued by this thread have completed once `drain` flips; this
      // wait ignores the abort flag so TMEM is never released under a live MMA
      mcommit(bar_drain);
      mwait(bar_drain, 0, SITE_MMA | 0x60, false);
    }
  } else if (warp < MAP_WARPS) {
    // ------------------------------------------------------------ map warps
    const int x = warp >> 3;          // query tile
    const int half = (warp >> 2) & 1;  // key columns [64 half, 64 half + 64)
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row in tile == TMEM lane
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const uint32_t t_s = tmem + lane_off + TM_S + 128u * x + 64u * half;
    const uint32_t t_o = tmem + lane_off + TM_O + 128u * x + (uint32_t)half * (DV / 2);
    const uint32_t named_bar = 1u + (uint32_t)(x * 4 + quarter);  // warps w and w^4
    float *xchg = reinterpret_cast<float *>(smem + L::OFF_XCHG);
    const float c2 = p.scale * LOG2E;  // scaled score in log2 units per raw dot
    // phase bits: 1 = s_full parity, 2 = o_full parity, 4 = row-max exchange buffer
    uint32_t ph = 0, nk_pos = 0;
    bool ok = true;
#ifdef CATTN_TRACE
    int tr_step = 0;
    const bool tr_warp = (warp & 7) == 0 && lane == 0;  // warps 0 and 8
#endif

    for (uint32_t uc = 0; ok; ++uc) {
      const int u = peek_unit(uc, SITE_EPI | 0x70);
      if (u < 0) break;
      // per unit: key tiles of this query tile, and the allowed-key bound of
      // this row relative to the unit's first key tile
      int nk_tiles, lim_base, nkv;
      float2 acc[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // Yat: mass; else l
      float2 ent[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // ENT: sum f log2 f
      float top[2] = {-INFINITY, -INFINITY};  // Yat: max kappa; else max raw dot
      float m_used = -INFINITY;               // softmax / s^tau: running max, log2 units
      float yb = 0.f, yeps = 0.f, qe = 0.f, tau = 1.f, seps = 0.f;
      bool fast = false;  // Yat: the fast map path is exact up to rounding for this unit
      // Yat row statistics: this row's guard against a cancelled distance and
      // where its query row and the unit's first key sit in memory
      float st_thr = INFINITY;
      const uint4 *st_q4 = nullptr, *st_k4 = nullptr;
      {
        const Unit t = decode_unit(p, u);
        nk_tiles = x ? t.n[1] : t.n[0];
        nkv = t.nkv;
        const int row = t.q0 + x * BM + r;
        lim_base = (p.causal ? min(row + 1, p.Tk) : p.Tk) - t.kv_begin * BN;
        if (VARIANT == kYat && STATS) {
          if (row < p.Tq)
            st_q4 = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.q) +
                                                    ((size_t)t.bh * p.Tq + row) * DK);
          st_k4 = reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p.k) +
                                                  ((size_t)t.bh_kv * p.Tk + (size_t)t.kv_begin * BN) * DK);
        }
        // tau* counts scores of real rows only (the forward just drops the
        // outputs of rows past Tq)
        if (VARIANT == kTau && row >= p.Tq) lim_base = 0;
        if (VARIANT == kYat) {
          yb = p.b[t.head];
          yeps = p.eps[t.head];
        } else if (VARIANT == kStau) {
          tau = p.tau[t.head];
          seps = p.eps[t.head];
        } else if (VARIANT == kTau) {
          seps = p.eps[t.head];
        }
      }
      // tau*: this thread's partial sums of 1, s, g, s g, g^2 over the unit
      float st[5] = {0.f, 0.f, 0.f, 0.f, 0.f};
      // row statistics: this thread's share of the row, the row's normaliser
      // from the forward (Yat: 1 / Z' and ln Z', Z' = M + 1e-9; softmax /
      // s^tau: the log-sum-exp in log2 units) and the threshold of the count
      // below 1e-6 in the accumulated domain (Yat 1e-6 Z', else log2 1e-6)
      RowStats rs;
      float nz_scale = 0.f, nz_log = 0.f, small_thr = 0.f;
      if constexpr (STATS) {
        rs.hs = rs.sk = make_float2(0.f, 0.f);
        rs.small = 0.f;
#pragma unroll
        for (int i = 0; i < 10; ++i) rs.top[i] = VARIANT == kYat ? 0.f : -INFINITY;
        const Unit t = decode_unit(p, u);
        const int row = t.q0 + x * BM + r;
        const float z = row < p.Tq ? p.norm_in[(size_t)t.bh * p.Tq + row] : 0.f;
        if (VARIANT == kYat) {
          nz_scale = 1.f / (z + 1e-9f);
          nz_log = logf(z + 1e-9f);
          small_thr = 1e-6f * (z + 1e-9f);
        } else {
          nz_log = z * LOG2E;
          small_thr = -19.931568569324174f;  // log2(1e-6)
        }
        if (row >= p.Tq) lim_base = 0;  // rows past Tq have no keys
      }
      const float g0 = VARIANT == kTau ? logf(0.6931472f + seps) : 0.f;
      if (VARIANT == kYat) {
        // |q|^2 of this thread's row, in fp32 from the bf16 Q tile in shared
        // memory (rows past Tq were loaded as zeros).  The order of a row's
        // 16-byte units is rotated by lane so that a warp's loads fall in
        // distinct banks; the sum does not depend on where a unit sits in the
        // swizzled row.  The Q tiles are released once every map warp has
        // read them.
        if (!(ok = warp_wait(bar_q_full, uc & 1u, abort, SITE_EPI | 0x40))) break;
        if (nk_tiles > 0) {
          const uint32_t qrow = q_smem(x) + (uint32_t)r * 128u;
          float2 s2 = make_float2(0.f, 0.f);
#pragma unroll
          for (int c = 0; c < DK / 64; ++c) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              const uint4 v = lds128(qrow + (uint32_t)c * (BM * 128) + ((uint32_t)((k + lane) & 7) << 4));
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float2 f = make_float2(__uint_as_float(w[i] << 16),
                                             __uint_as_float(w[i] & 0xffff0000u));
                s2 = __ffma2_rn(f, f, s2);
              }
            }
          }
          qe = (s2.x + s2.y) + yeps;
          // the bounds under which the map's fast path is exact up to rounding
          // (a maximum of another generation of norms bounds nothing: the
          // exact path then)
          if constexpr (!INORM) {  // (the one-launch path bounds each key tile itself)
            const unsigned long long nkw = *p.nk_max;
            const float nkm = p.nk_gen == 0u || (unsigned)(nkw >> 32) == p.nk_gen
                                  ? __uint_as_float((unsigned)nkw)
                                  : INFINITY;
            const float span = qe + nkm;
            fast = yeps >= 0x1p-60f && __all_sync(FULL, span <= 0x1p61f && span * 0x1p-16f <= yeps);
          }
          if (STATS && st_q4) st_thr = yat_near_threshold(s2.x + s2.y, yb, YM);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_q_empty);
      }

      // one-launch Yat: this warp's norms of key tile j, taken from the K slot
      // (ring position 2j of the CTA's only unit) while the S MMAs run; then
      // the slot may be refilled.  A tile this warp does not map is only
      // released (every map warp releases every K slot of the unit).
      auto inorm_tile = [&](int j, bool take) -> bool {
        if constexpr (INORM) {
          const uint32_t kpos = 2u * (uint32_t)j, ks = kpos % L::NS;
          if (!warp_wait(kv_full(ks), (kpos / L::NS) & 1u, abort, SITE_EPI | 0x50)) return false;
          if (take) {
            const float mx = inorm_tile_norms<DK>(slot_smem(ks), half, lane, nku + warp * BN);
            fast = yat_fast_ok(mx, qe, yeps);
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(kv_empty(ks));
        }
        return true;
      };
      for (int j = 0; j < nk_tiles; ++j, ph ^= 1u) {
        if constexpr (INORM) {
          if (!(ok = inorm_tile(j, true))) break;
        }
        if (!(ok = warp_wait(s_full(x), ph & 1u, abort, SITE_EPI | 0x10))) break;
        tc_fence_after();
#ifdef CATTN_TRACE
        if (tr_warp) CATTN_TR(2 * x, tr_step);
#endif

        // keys of tile j allowed for col < limit (col counts the whole tile)
        const int limit = min(BN, lim_base - j * BN);
        const bool partial = __any_sync(FULL, limit < BN);  // warp-uniform path choice
        // Yat takes one path per 32-key chunk: every key allowed for all the
        // warp's rows, none allowed (P = 0, nothing to compute), or per key
        auto chunk_kind = [&](int c) -> int {  // 0 all allowed, 1 none, 2 mixed
          const int c0 = 32 * (half * 2 + c);
          if (!partial || __all_sync(FULL, c0 + 32 <= limit)) return 0;
          if (__all_sync(FULL, c0 >= limit)) return 1;
          return 2;
        };

        if constexpr (VARIANT == kTau) {
          // read S out, free the buffer for S(j+1), then take the statistics
          uint32_t sr[2][32];
          tmem_ld32(t_s, sr[0]);
          tmem_ld32(t_s + 32, sr[1]);
          tmem_wait_ld();
          tmem_ld_fence(sr[0]);
          tmem_ld_fence(sr[1]);
          tc_fence_before();
          mbar_arrive(p_full(x));
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (partial)
              tau_chunk<true>(sr[c], half * 2 + c, p.scale, c2, seps, g0, limit, st);
            else
              tau_chunk<false>(sr[c], half * 2 + c, p.scale, c2, seps, g0, limit, st);
          }
          continue;
        }
        if constexpr (STATS) {
          // the row statistics over the allowed keys, one 32-key chunk at a
          // time; tiles with no masked key take the unmasked path
          const float4 *nk4 = nullptr;
          if (VARIANT == kYat) {
            const uint32_t npos = nk_pos + j, ns = npos % NKS;
            if (!(ok = warp_wait(nk_full(ns), (npos / NKS) & 1u, abort, SITE_EPI | 0x20))) break;
            nk4 = reinterpret_cast<const float4 *>(nk_ring + ns * BN);
          }
          auto stats_tile = [&](auto partial_tag) {
            constexpr bool PARTIAL = decltype(partial_tag)::value;
#pragma unroll
            for (int c = 0; c < 2; ++c) {
              const int cc = half * 2 + c;
              uint32_t sr1[32];
              tmem_ld32(t_s + 32 * c, sr1);
              tmem_wait_ld();
              tmem_ld_fence(sr1);
              if (VARIANT == kYat) {
                // kappa of the chunk's keys in place of their dots, then the
                // guard against a cancelled distance: the (rare) allowed keys
                // whose kappa passed the row's bound are recomputed by the
                // plain definition, outside the accumulation loop below
#pragma unroll
                for (int i = 0; i < 32; i += 2) {
                  const float4 n4 = nk4[(cc * 32 + i) >> 2];
                  const float2 nk2 = (i & 2) ? make_float2(n4.z, n4.w) : make_float2(n4.x, n4.y);
                  const float2 kk =
                      fast ? yat_pair<true, YM>(f2(sr1[i], sr1[i + 1]), nk2, make_float2(yb, yb),
                                                make_float2(qe, qe), yeps)
                           : yat_pair<false, YM>(f2(sr1[i], sr1[i + 1]), nk2, make_float2(yb, yb),
                                                 make_float2(qe, qe), yeps);
                  sr1[i] = __float_as_uint(kk.x);
                  sr1[i + 1] = __float_as_uint(kk.y);
                }
                unsigned flag = 0u;
#pragma unroll
                for (int i = 0; i < 32; ++i)
                  flag |= ((!PARTIAL || cc * 32 + i < limit) && __uint_as_float(sr1[i]) > st_thr) ? 1u << i
                                                                                                 : 0u;
                // (allowed keys only: the others may lie past the end of k;
                // one call site, the result put in place by a select chain so
                // that the chunk stays in registers)
                const uint4 *kt4 = st_k4 + ((size_t)j * BN + (size_t)cc * 32) * (DK / 8);
                while (flag != 0u) {
                  const int i = __ffs(flag) - 1;
                  flag &= flag - 1u;
                  const uint32_t v = __float_as_uint(
                      yat_direct_call<DK, YM>(st_q4, kt4 + (size_t)i * (DK / 8), yb, yeps));
#pragma unroll
                  for (int t = 0; t < 32; ++t) sr1[t] = t == i ? v : sr1[t];
                }
              }
#pragma unroll
              for (int i = 0; i < 32; i += 2) {
                const int col = cc * 32 + i;
                const bool al0 = !PARTIAL || col < limit, al1 = !PARTIAL || col + 1 < limit;
                if (VARIANT == kYat) {
                  // (kappa of the chunk, over the raw dots: see below)
                  float k0 = __uint_as_float(sr1[i]), k1 = __uint_as_float(sr1[i + 1]);
                  if (PARTIAL) {
                    k0 = al0 ? k0 : 0.f;
                    k1 = al1 ? k1 : 0.f;
                  }
                  stats_pair_yat<PARTIAL>(rs, make_float2(k0, k1), small_thr, al0, al1);
                } else {
                  const float d0 = __uint_as_float(sr1[i]), d1 = __uint_as_float(sr1[i + 1]);
                  float x0, x1;  // log2 of the weights
                  if (VARIANT == kSoftmax) {
                    x0 = fmaf(d0, c2, -nz_log);
                    x1 = fmaf(d1, c2, -nz_log);
                  } else {
                    x0 = fmaf(tau, log2_phi(d0 * p.scale, fabsf(d0) * c2, seps), -nz_log);
                    x1 = fmaf(tau, log2_phi(d1 * p.scale, fabsf(d1) * c2, seps), -nz_log);
                  }
                  if (PARTIAL) {
                    x0 = al0 ? x0 : -1e30f;
                    x1 = al1 ? x1 : -1e30f;
                  }
                  stats_pair_log<PARTIAL>(rs, make_float2(x0, x1), small_thr, al0, al1);
                }
              }
            }
          };
          if (partial)
            stats_tile(std::true_type{});
          else
            stats_tile(std::false_type{});
          // S (and, for Yat, the tile's key norms) read: S(j+1) may land
          tc_fence_before();
          mbar_arrive(p_full(x));
          continue;
        }
        bool rescale = false;
        float corr = 1.f;
        if (VARIANT == kYat) {
          const float4 *nk4;
          if constexpr (INORM) {
            nk4 = reinterpret_cast<const float4 *>(nku + warp * BN);
          } else {
            const uint32_t npos = nk_pos + j, ns = npos % NKS;
            if (!(ok = warp_wait(nk_full(ns), (npos / NKS) & 1u, abort, SITE_EPI | 0x20))) break;
            nk4 = reinterpret_cast<const float4 *>(nk_ring + ns * BN);
          }
          // chunk by chunk: P chunk c lands on S columns this warp has read
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            const int kind = chunk_kind(c);
            uint32_t hk[16];
            if (kind == 1) {
#pragma unroll
              for (int i = 0; i < 16; ++i) hk[i] = 0u;
            } else {
              uint32_t sr[32];
              tmem_ld32(t_s + 32 * c, sr);
              tmem_wait_ld();
              tmem_ld_fence(sr);
              if (fast) {
                if (kind == 2)
                  yat_chunk<true, true, YM, ENT>(sr, half * 2 + c, nk4, yb, qe, yeps, limit, acc, top, hk,
                                                ent);
                else
                  yat_chunk<false, true, YM, ENT>(sr, half * 2 + c, nk4, yb, qe, yeps, limit, acc, top, hk,
                                                ent);
              } else {
                if (kind == 2)
                  yat_chunk<true, false, YM, ENT>(sr, half * 2 + c, nk4, yb, qe, yeps, limit, acc, top, hk,
                                                ent);
                else
                  yat_chunk<false, false, YM, ENT>(sr, half * 2 + c, nk4, yb, qe, yeps, limit, acc, top, hk,
                                                ent);
              }
            }
            tmem_st16(t_s + 16 * c, hk);
            if (c == 0) {  // the first chunk of P: half of PV may start
              tmem_wait_st();
              tc_fence_before();
              mbar_arrive(p_half(x));
            }
          }
        } else {
          uint32_t sr[2][32];
          tmem_ld32(t_s, sr[0]);
          tmem_ld32(t_s + 32, sr[1]);
          tmem_wait_ld();
          tmem_ld_fence(sr[0]);
          tmem_ld_fence(sr[1]);
          float mt = partial ? fmaxf(chunk_max<true>(sr[0], half * 2, limit),
                                     chunk_max<true>(sr[1], half * 2 + 1, limit))
                             : fmaxf(chunk_max<false>(sr[0], half * 2, limit),
                                     chunk_max<false>(sr[1], half * 2 + 1, limit));
          // the row max over the whole tile: swap halves with the partner warp
          float *xb = xchg + ((((ph >> 2) & 1u) * 2 + (uint32_t)x) * 2) * BM;
          xb[half * BM + r] = mt;
          named_barrier_sync(named_bar, 64);
          mt = fmaxf(mt, xb[(half ^ 1) * BM + r]);
          ph ^= 4u;
          top[0] = fmaxf(top[0], mt);
          float m_new = -INFINITY;
          if (mt > -INFINITY) {
            if (VARIANT == kSoftmax)
              m_new = mt * c2;
            else
              m_new = tau * log2_phi(mt * p.scale, fabsf(mt) * c2, seps);
          }
          if (__any_sync(FULL, m_new > m_used + RESCALE_THRESHOLD)) {
            const float mn = fmaxf(m_used, m_new);
            corr = ex2_approx(m_used - mn);
            if (ENT && m_used > -INFINITY) {
              // sum p (x - m) onto the new max: each p scales by corr and each
              // exponent drops by mn - m_used
              const float dm = m_used - mn;
#pragma unroll
              for (int hh = 0; hh < 2; ++hh) {
                ent[hh].x = corr * fmaf(dm, acc[hh].x, ent[hh].x);
                ent[hh].y = corr * fmaf(dm, acc[hh].y, ent[hh].y);
              }
            }
            acc[0].x *= corr;
            acc[0].y *= corr;
            acc[1].x *= corr;
            acc[1].y *= corr;
            m_used = mn;
            rescale = j > 0;
          }
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            if (VARIANT == kStau && c == 1) {
              // s^tau holds more temporaries: read the second chunk again
              // rather than keep it live through the first one's map and the
              // rescale of O
              tmem_ld32(t_s + 32, sr[1]);
              tmem_wait_ld();
              tmem_ld_fence(sr[1]);
            }
            uint32_t hk[16];
            if (VARIANT == kSoftmax) {
              if (partial)
                softmax_chunk<true, ENT>(sr[c], half * 2 + c, c2, -m_used, limit, acc, hk, ent);
              else
                softmax_chunk<false, ENT>(sr[c], half * 2 + c, c2, -m_used, limit, acc, hk, ent);
            } else {
              if (partial)
                stau_chunk<true, ENT>(sr[c], half * 2 + c, p.scale, c2, tau, seps, -m_used, limit,
                                      acc, hk, ent);
              else
                stau_chunk<false, ENT>(sr[c], half * 2 + c, p.scale, c2, tau, seps, -m_used, limit,
                                       acc, hk, ent);
            }
            if (SPLIT_PV && c == 0) {
              // O holds every tile before j (S_x(j) landed after PV_x(j-1)):
              // bring this warp's dv/2 columns onto the new max before the
              // first half of PV(j) adds to it
              if (rescale) scale_o_half16<DV>(t_o, corr);
              tmem_st16(t_s, hk);
              tmem_wait_st();
              tc_fence_before();
              mbar_arrive(p_half(x));  // the first chunk of P: half of PV may start
            } else {
              tmem_st16(t_s + 16 * c, hk);
            }
          }
          // softmax: O_x holds every tile before j (S_x(j) landed after
          // PV_x(j-1)): bring this warp's dv/2 columns onto the new max
          if (!SPLIT_PV && rescale) scale_o_half<DV>(t_o, corr);
        }
        tmem_wait_st();
        tc_fence_before();
#ifdef CATTN_TRACE
        if (tr_warp) CATTN_TR(2 * x + 1, tr_step);
        ++tr_step;
#endif
        mbar_arrive(p_full(x));
      }
      if constexpr (INORM) {  // the unit's K slots this warp does not map
        for (int j = nk_tiles; ok && j < nkv; ++j) ok = inorm_tile(j, false);
      }

      if constexpr (STATS) {
        if (ok && nk_tiles > 0) {
          // merge the two column halves of each row: half 1 hands its share to
          // half 0 through shared memory, half 0 writes the row's statistics
          float *sx = xchg + (uint32_t)x * BM;  // [13 values][2 tiles][BM]
          if (half == 1) {
            sx[(0 * 2) * BM + r] = rs.hs.x + rs.hs.y;
            sx[(1 * 2) * BM + r] = rs.sk.x + rs.sk.y;
            sx[(2 * 2) * BM + r] = rs.small;
#pragma unroll
            for (int i = 0; i < 10; ++i) sx[((3 + i) * 2) * BM + r] = rs.top[i];
          }
          named_barrier_sync(named_bar, 64);
          if (half == 0) {
            const float hs = (rs.hs.x + rs.hs.y) + sx[(0 * 2) * BM + r];
            const float sk = (rs.sk.x + rs.sk.y) + sx[(1 * 2) * BM + r];
            rs.small += sx[(2 * 2) * BM + r];
#pragma unroll
            for (int i = 0; i < 10; ++i) {
              float v = sx[((3 + i) * 2) * BM + r];
#pragma unroll
              for (int k2 = 0; k2 < 10; ++k2) {
                const float hi = fmaxf(rs.top[k2], v);
                v = fminf(rs.top[k2], v);
                rs.top[k2] = hi;
              }
            }
            const Unit t = decode_unit(p, unit_ring[uc & 1u]);
            const int row = t.q0 + x * BM + r;
            if (row < p.Tq) {
              const size_t ti = (size_t)t.bh * p.Tq + row;
              // the row's allowed keys
              const float n = (float)(p.causal ? min(row + 1, p.Tk) : p.Tk);
              float top10 = 0.f;
#pragma unroll
              for (int i = 0; i < 10; ++i) top10 += VARIANT == kYat ? rs.top[i] : ex2_approx(rs.top[i]);
              // sum w ln w over the row
              const float hsum = VARIANT == kYat ? nz_scale * (LN2 * hs - nz_log * sk) : LN2 * hs;
              if (VARIANT == kYat) top10 *= nz_scale;
              if (p.st_entropy) p.st_entropy[ti] = n > 1.f ? -hsum / logf(n) : 0.f;
              if (p.st_small) p.st_small[ti] = rs.small / n;
              if (p.st_top10) p.st_top10[ti] = top10;
            }
          }
          // half 0 has read the buffer before half 1 writes it for the next unit
          named_barrier_sync(named_bar, 64);
        }
      }
      if (VARIANT == kTau && ok && nk_tiles > 0) {
        // tau*: the warp's sums, then one fp64 atomic per moment and warp
#pragma unroll
        for (int i = 0; i < 5; ++i) {
          float v = st[i];
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(FULL, v, o);
          st[i] = v;
        }
        if (lane == 0) {
          const Unit t = decode_unit(p, unit_ring[uc & 1u]);
          double *m = p.moments + (size_t)t.head * 6;
#pragma unroll
          for (int i = 0; i < 5; ++i) atomicAdd(m + i, (double)st[i]);
        }
      }
      // ---- finalise: combine the two halves of the row, then normalise and
      // store (or, with key splits, store the unnormalised partial)
      if (VARIANT != kTau && !STATS && ok && nk_tiles > 0) {
        const float part = (acc[0].x + acc[0].y) + (acc[1].x + acc[1].y);
        const float ptop = fmaxf(top[0], top[1]);
        float *fb = xchg + (8 + (uint32_t)x * 4) * BM;  // [2 values][2 halves][BM]
        float *eb = xchg + (16 + (uint32_t)x * 2) * BM;  // ENT: [2 halves][BM]
        fb[(0 * 2 + half) * BM + r] = part;
        fb[(1 * 2 + half) * BM + r] = ptop;
        const float pent = ENT ? (ent[0].x + ent[0].y) + (ent[1].x + ent[1].y) : 0.f;
        if (ENT) eb[half * BM + r] = pent;
        named_barrier_sync(named_bar, 64);
        const float total = part + fb[(0 * 2 + (half ^ 1)) * BM + r];
        const float all_top = fmaxf(ptop, fb[(1 * 2 + (half ^ 1)) * BM + r]);
        const float all_ent = ENT ? pent + eb[(half ^ 1) * BM + r] : 0.f;
        // the partner reads fb before either warp writes it for the next unit
        named_barrier_sync(named_bar, 64);
        // everything that does not need O before the wait, while the last PV runs
        const Unit t = decode_unit(p, unit_ring[uc & 1u]);
        const int row = t.q0 + x * BM + r;
        const bool row_ok = row < p.Tq;
        const float inv = VARIANT == kYat ? 1.f / (total + 1e-9f) : 1.f / total;
        // Yat: a key may sit close enough to q for the assembled distance to
        // have cancelled; the near-key pass then recomputes this row (the
        // one-launch path: this CTA, after its unit).  Taken here, ahead of
        // the wait and without a division: on the unit boundary the guard
        // measured about 1% of the kernel as an IEEE division after the wait.
        const bool near_row =
            VARIANT == kYat && row_ok && half == 0 && yat_near_flag(all_top, qe - yeps, yb, YM);
        if (!(ok = warp_wait(o_full(x), (ph >> 1) & 1u, abort, SITE_EPI | 0x30))) break;
        tc_fence_after();
        if (p.n_splits == 1) {
          __nv_bfloat16 *orow = reinterpret_cast<__nv_bfloat16 *>(p.out) +
                                ((size_t)t.bh * p.Tq + row) * DV + half * (DV / 2);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c) {
            uint32_t o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
            tmem_ld_fence(o);
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i)
              packed[i] = pack_bf16x2(__uint_as_float(o[2 * i]) * inv,
                                      __uint_as_float(o[2 * i + 1]) * inv);
            if (row_ok) {
              // each thread writes its own row: whole 32-byte sectors when the
              // output allows it
              if (p.out_align32) {
#pragma unroll
                for (int i = 0; i < 2; ++i)
                  stg256(orow + c * 32 + 16 * i, packed[8 * i], packed[8 * i + 1], packed[8 * i + 2],
                         packed[8 * i + 3], packed[8 * i + 4], packed[8 * i + 5], packed[8 * i + 6],
                         packed[8 * i + 7]);
              } else {
                uint4 *dst = reinterpret_cast<uint4 *>(orow + c * 32);
#pragma unroll
                for (int i = 0; i < 4; ++i)
                  dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                      packed[4 * i + 3]);
              }
            }
          }
          if (row_ok && half == 0) {
            const size_t ti = (size_t)t.bh * p.Tq + row;
            if (ENT) {
              // normalised entropy of the row's weights f / Z from Z and
              // sum f log2 f: -sum w ln w = ln Z - ln 2 (sum f log2 f) / Z
              // (Yat: w = kappa / Z', Z' = M + 1e-9, so the first term is
              // M ln Z' / Z')
              const int n = p.causal ? min(row + 1, p.Tk) : p.Tk;
              float hrow;
              if (VARIANT == kYat) {
                const float z = total + 1e-9f;
                hrow = (total * logf(z) - LN2 * all_ent) / z;
              } else {
                hrow = logf(total) - LN2 * all_ent / total;
              }
              p.row_entropy[ti] = n > 1 ? hrow / logf((float)n) : 0.f;
            }
            if (near_row) {
              if constexpr (INORM) {
                near_list[atomicAdd(near_n, 1u)] = (unsigned)(x * BM + r);
              } else {
                const unsigned slot = atomicAdd(p.near_count, 1u);
                if (slot < p.near_cap) p.near_rows[slot] = make_uint2((unsigned)t.bh, (unsigned)row);
              }
            }
            if (p.row_mass)
              p.row_mass[ti] = VARIANT == kYat ? total : (m_used + log2f(total)) * LN2;
            if (p.row_max) p.row_max[ti] = VARIANT == kYat ? all_top : all_top * p.scale;
          }
        } else {
          const size_t ti = ((size_t)t.split * p.B * p.h + t.bh) * p.Tq + row;
          float *prow = p.part_o + ti * DV + half * (DV / 2);
#pragma unroll
          for (int c = 0; c < DV / 64; ++c) {
            uint32_t o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
            tmem_ld_fence(o);
            if (row_ok) {  // the workspace is 256-byte aligned
#pragma unroll
              for (int i = 0; i < 4; ++i)
                stg256(prow + c * 32 + 8 * i, o[8 * i], o[8 * i + 1], o[8 * i + 2], o[8 * i + 3],
                       o[8 * i + 4], o[8 * i + 5], o[8 * i + 6], o[8 * i + 7]);
            }
          }
          if (row_ok && half == 0) {
            reinterpret_cast<float4 *>(p.part_stat)[ti] = make_float4(total, m_used, all_top, all_ent);
            if (near_row) {
              const unsigned slot = atomicAdd(p.near_count, 1u);
              if (slot < p.near_cap) p.near_rows[slot] = make_uint2((unsigned)t.bh, (unsigned)row);
            }
          }
        }
        // O_x has been read: the next unit's first PV_x may overwrite it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(o_empty(x));
        ph ^= 2u;
      }
      nk_pos += nkv;
      release_unit(uc);
    }
    if constexpr (INORM) {
      // every row of the CTA's unit written: the rows listed for the
      // near-key guard are recomputed by the plain definition, one per warp
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_rows_done);
      if (ok && warp_wait(bar_rows_done, 0u, abort, SITE_EPI | 0x58)) {
        const Unit t = decode_unit(p, (int)blockIdx.x);
        const unsigned n = *near_n;
        for (unsigned e = (unsigned)warp; e < n; e += MAP_WARPS)
          near_row_warp<DK, DV, YM>(p, t.bh, t.q0 + (int)near_list[e], lane);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == MMA_WARP) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // the key-split combine or the near-key pass may start launching (they
  // wait for this grid's completion before they read anything)
  griddep_launch_dependents();
}

// Key-split combine: one warp per query row merges the n_splits partials.
// Yat adds masses and outputs (the mass is a plain sum); softmax and s^tau
// bring each partial onto the largest running max first.
template <int VARIANT, int DV>
__global__ void __launch_bounds__(256) combine_kernel(const __grid_constant__ FwdParams p) {
  griddep_wait();  // the fused kernel's partials
  const long long rows = (long long)p.B * p.h * p.Tq;
  const long long rrow = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
  if (rrow >= rows) return;
  const int lane = threadIdx.x & 31;
  const float4 *stat = reinterpret_cast<const float4 *>(p.part_stat);
  float m_all = -INFINITY, top = -INFINITY;
  for (int s = 0; s < p.n_splits; ++s) {
    const float4 st = stat[(long long)s * rows + rrow];
    m_all = fmaxf(m_all, st.y);
    top = fmaxf(top, st.z);
  }
  float total = 0.f, ent = 0.f;  // ent: sum f log2 f on m_all (ENT)
  constexpr int PER_LANE = DV / 32;  // 2 or 4 columns per lane
  float o[PER_LANE];
#pragma unroll
  for (int i = 0; i < PER_LANE; ++i) o[i] = 0.f;
  for (int s = 0; s < p.n_splits; ++s) {
    const float4 st = stat[(long long)s * rows + rrow];
    const float w = VARIANT == kYat ? 1.f : (st.y == -INFINITY ? 0.f : exp2f(st.y - m_all));
    total += w * st.x;
    if (p.row_entropy && w > 0.f)
      ent += VARIANT == kYat ? st.w : w * fmaf(st.y - m_all, st.x, st.w);
    const float *src = p.part_o + ((long long)s * rows + rrow) * DV + lane * PER_LANE;
#pragma unroll
    for (int i = 0; i < PER_LANE; ++i) o[i] += w * src[i];
  }
  const float inv = VARIANT == kYat ? 1.f / (total + 1e-9f) : 1.f / total;
  __nv_bfloat16 *dst = reinterpret_cast<__nv_bfloat16 *>(p.out) + rrow * DV + lane * PER_LANE;
#pragma unroll
  for (int i = 0; i < PER_LANE; i += 2) {
    const uint32_t v = pack_bf16x2(o[i] * inv, o[i + 1] * inv);
    *reinterpret_cast<uint32_t *>(dst + i) = v;
  }
  if (lane == 0) {
    if (p.row_mass) p.row_mass[rrow] = VARIANT == kYat ? total : (m_all + log2f(total)) * LN2;
    if (p.row_max) p.row_max[rrow] = VARIANT == kYat ? top : top * p.scale;
    if (p.row_entropy) {  // key splits are non-causal: every row has Tk keys
      float hrow;
      if (VARIANT == kYat) {
        const float z = total + 1e-9f;
        hrow = (total * logf(z) - LN2 * ent) / z;
      } else {
        hrow = logf(total) - LN2 * ent / total;
      }
      p.row_entropy[rrow] = p.Tk > 1 ? hrow / logf((float)p.Tk) : 0.f;
    }
  }
}

// The near-key pass of the Yat forward.  A row whose computed max kappa
// passed yat_near_threshold may hold a key so close to its query that the
// assembled distance |q|^2 + |k|^2 - 2 q.k cancelled; the fused kernel listed
// it (near_rows), and here one CTA per listed row recomputes the whole row by
// the plain definition: kappa_j = (q.k_j + b)^{2M} / (max(|q - k_j|^2, 0) +
// eps) with the dot product and the distance summed over the components in
// fp32 (eight warps take every eighth key; a warp's lanes split the
// components, then each lane accumulates its dv/32 columns of kappa v), and
// writes out = sum kappa v / (sum kappa + 1e-9), the row mass and max kappa
// over what the fused kernel (and, with key splits, the combine) stored.  A
// row listed twice (once per key split) is recomputed twice, with the same
// result.  With no row listed every CTA returns at once.
__device__ __forceinline__ float elem_f(const float *p) { return *p; }
__device__ __forceinline__ float elem_f(const __nv_bfloat16 *p) { return __bfloat162float(*p); }
__device__ __forceinline__ void elem_st(float *p, float v) { *p = v; }
__device__ __forceinline__ void elem_st(__nv_bfloat16 *p, float v) { *p = __float2bfloat16_rn(v); }

template <int DK, int DV, int YM, typename T>
__global__ void __launch_bounds__(256) near_fix_kernel(const __grid_constant__ FwdParams p) {
  constexpr int QE = DK / 32;  // q and k components per lane
  constexpr int VE = DV / 32;  // v columns per lane
  __shared__ float s_mass[8], s_top[8], s_slog[8];
  __shared__ float s_o[8][DV];
  griddep_wait();  // the fused kernel's list, outputs and telemetry
  const unsigned n = min(*p.near_count, p.near_cap);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const T *qg = static_cast<const T *>(p.q);
  const T *kg = static_cast<const T *>(p.k);
  const T *vg = static_cast<const T *>(p.v);
  for (unsigned e = blockIdx.x; e < n; e += gridDim.x) {
    const uint2 id = p.near_rows[e];
    const int bh = (int)id.x, row = (int)id.y;
    const int head = bh % p.h, batch = bh / p.h;
    const size_t bh_kv = (size_t)batch * p.hkv + head / (p.h / p.hkv);
    const float b = p.b[head], eps = p.eps[head];
    float qf[QE];
#pragma unroll
    for (int i = 0; i < QE; ++i)
      qf[i] = elem_f(qg + ((size_t)bh * p.Tq + row) * DK + lane * QE + i);
    const int lim = p.causal ? min(row + 1, p.Tk) : p.Tk;
    float mass = 0.f, top = 0.f, slog = 0.f, o[VE];  // slog: sum kappa ln kappa
#pragma unroll
    for (int c = 0; c < VE; ++c) o[c] = 0.f;
    for (int j = warp; j < lim; j += 8) {
      const T *kr = kg + (bh_kv * p.Tk + j) * DK + lane * QE;
      float dot = 0.f, d2 = 0.f;
#pragma unroll
      for (int i = 0; i < QE; ++i) {
        const float kf = elem_f(kr + i);
        dot = fmaf(qf[i], kf, dot);
        const float df = qf[i] - kf;
        d2 = fmaf(df, df, d2);
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        dot += __shfl_xor_sync(FULL, dot, off);
        d2 += __shfl_xor_sync(FULL, d2, off);
      }
      const float tt = dot + b;
      float num = tt * tt;
      if constexpr (YM == 2) num = num * num;
      if constexpr (YM == 3) num = num * num * num;
      const float kap = num / (fmaxf(d2, 0.f) + eps);
      mass += kap;
      top = fmaxf(top, kap);
      if (kap > 0.f) slog = fmaf(kap, logf(kap), slog);
      const T *vr = vg + (bh_kv * p.Tk + j) * DV + lane * VE;
#pragma unroll
      for (int c = 0; c < VE; ++c) o[c] = fmaf(kap, elem_f(vr + c), o[c]);
    }
    if (lane == 0) {
      s_mass[warp] = mass;
      s_top[warp] = top;
      s_slog[warp] = slog;
    }
#pragma unroll
    for (int c = 0; c < VE; ++c) s_o[warp][lane * VE + c] = o[c];
    __syncthreads();
    if (warp == 0) {
      float m_all = 0.f, t_all = 0.f, l_all = 0.f;
#pragma unroll
      for (int w = 0; w < 8; ++w) {
        m_all += s_mass[w];
        t_all = fmaxf(t_all, s_top[w]);
        l_all += s_slog[w];
      }
      const float inv = 1.f / (m_all + 1e-9f);
      const size_t ti = (size_t)bh * p.Tq + row;
      T *orow = static_cast<T *>(p.out) + ti * DV + lane * VE;
#pragma unroll
      for (int c = 0; c < VE; ++c) {
        float acc = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) acc += s_o[w][lane * VE + c];
        elem_st(orow + c, acc * inv);
      }
      if (lane == 0) {
        if (p.row_mass) p.row_mass[ti] = m_all;
        if (p.row_max) p.row_max[ti] = t_all;
        if (p.row_entropy) {  // -sum w ln w with w = kappa / (M + 1e-9)
          const float z = m_all + 1e-9f;
          const float hrow = (m_all * logf(z) - l_all) / z;
          p.row_entropy[ti] = lim > 1 ? hrow / logf((float)lim) : 0.f;
        }
      }
    }
    __syncthreads();
  }
}

// tau* = (sum s g - sum s sum g / n) / (sum g^2 - (sum g)^2 / n), one thread
// per head, in fp64 (the shift g0 cancels).
__global__ void tau_finalize_kernel(const double *moments, const float *eps, int h, float *tau,
                                    double *moments_out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= h) return;
  const double *m = moments + (size_t)i * 6;
  const double n = m[0], ss = m[1], sg = m[2], ssg = m[3], sgg = m[4];
  const double cov = ssg - ss * sg / n, var = sgg - sg * sg / n;
  tau[i] = (n >= 2.0 && var > 0.0) ? (float)(cov / var) : __int_as_float(0x7fc00000);
  if (moments_out) {
    for (int j = 0; j < 5; ++j) moments_out[(size_t)i * 6 + j] = m[j];
    moments_out[(size_t)i * 6 + 5] = (double)logf(0.6931472f + eps[i]);
  }
}

// Launch of a kernel that follows the fused kernel on the stream: with the
// programmatic serialisation attribute it may begin launching while the
// fused kernel's last CTAs finish; it waits (griddepcontrol.wait) before it
// reads their results.
template <typename Kern>
cudaError_t launch_dependent(Kern kern, unsigned grid, cudaStream_t s, const FwdParams &p) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int VARIANT, int DK, int DV, int YM = 1, bool STATS = false, bool ENT = false,
          bool INORM = false>
cudaError_t launch(const FwdParams &p, const CUtensorMap &tq, const CUtensorMap &tk,
                   const CUtensorMap &tv, cudaStream_t s) {
  using L = Layout<DK, DV>;
  auto kern = fwd_kernel<VARIANT, DK, DV, YM, STATS, ENT, INORM>;
  static int configured_for = -1;
  static int sm_count = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::ALLOC);
    if (e != cudaSuccess) return e;
    e = cudaDeviceGetAttribute(&sm_count, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  if (p.n_units <= 0) return cudaSuccess;
  const int grid = p.n_units < sm_count ? p.n_units : sm_count;  // one CTA per SM
  // (an ordinary launch: as a programmatic dependent of the key-norm kernel
  // it measured 3% slower on a causal B=16, 16-head, 4096-token problem)
  kern<<<grid, NUM_THREADS, L::ALLOC, s>>>(p, tq, tk, tv);
  e = cudaGetLastError();
  if constexpr (VARIANT == kTau || STATS) {
    return e;
  } else {
    if (e != cudaSuccess) return e;
    if (p.n_splits > 1) {
      const long long rows = (long long)p.B * p.h * p.Tq;
      if ((e = launch_dependent(combine_kernel<VARIANT, DV>, (unsigned)((rows + 7) / 8), s, p)) !=
          cudaSuccess)
        return e;
    }
    if constexpr (VARIANT == kYat && !INORM)  // (the one-launch path recomputes its rows itself)
      e = launch_dependent(near_fix_kernel<DK, DV, YM, __nv_bfloat16>, (unsigned)sm_count, s, p);
    return e;
  }
}

}  // namespace tc

TcSchedule tc_schedule(int B, int h, int Tq, int Tk, int causal) {
  TcSchedule s;
  const int n_qtiles = (Tq + kTcQueryTile - 1) / kTcQueryTile;
  s.n_pairs = (n_qtiles + 1) / 2;
  s.n_kv_tiles = (Tk + kTcKeyTile - 1) / kTcKeyTile;
  s.head_group = 16;
  const long long pairs = (long long)B * h * s.n_pairs;
  // Without a causal mask every unit costs the same, so a problem with few
  // units would leave SMs idle in its last wave: split the keys until there
  // are about seven units per SM (at most 64 splits, at least 8 key tiles each).
  int splits = 1;
  if (!causal)
    while (pairs * splits < 1024 && splits < 64 && s.n_kv_tiles >= 16 * splits) splits *= 2;
  s.kv_per_split = (s.n_kv_tiles + splits - 1) / splits;
  s.n_splits = s.n_kv_tiles > 0 ? (s.n_kv_tiles + s.kv_per_split - 1) / s.kv_per_split : 1;
  s.n_units = pairs * s.n_splits;
  return s;
}

int tc_grid_size(long long n_units) {
  constexpr int kMaxDev = 64;
  static int sms[kMaxDev];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDev) return -1;
  if (sms[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    sms[dev] = n;
  }
  return n_units < sms[dev] ? (int)n_units : sms[dev];
}

bool fwd_tc_supported(int dk, int dv) {
  return (dk == 64 && dv == 64) || (dk == 128 && dv == 128) || (dk == 128 && dv == 64);
}

cudaError_t launch_fwd_tc(int variant, int dk, int dv, const FwdParams &p, const CUtensorMap &tq,
                          const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t s) {
#define CATTN_TC_CASE(V, DK_, DV_)                                                   \
  if (variant == V && dk == DK_ && dv == DV_)                                        \
    return p.row_entropy ? tc::launch<V, DK_, DV_, 1, false, true>(p, tq, tk, tv, s) \
                         : tc::launch<V, DK_, DV_>(p, tq, tk, tv, s);
#define CATTN_TC_INORM(DK_, DV_)                                                      \
  if (variant == kYat && p.inline_norms && p.yat_m == 1 && !p.row_entropy && dk == DK_ && \
      dv == DV_)                                                                      \
    return tc::launch<kYat, DK_, DV_, 1, false, false, true>(p, tq, tk, tv, s);
  CATTN_TC_INORM(64, 64)
  CATTN_TC_INORM(128, 128)
  CATTN_TC_INORM(128, 64)
#undef CATTN_TC_INORM
#define CATTN_TC_YAT_M(DK_, DV_, M_)                            \
  if (variant == kYat && p.yat_m == M_ && dk == DK_ && dv == DV_) \
    return tc::launch<kYat, DK_, DV_, M_>(p, tq, tk, tv, s);
  CATTN_TC_YAT_M(64, 64, 2)
  CATTN_TC_YAT_M(128, 128, 2)
  CATTN_TC_YAT_M(128, 64, 2)
  CATTN_TC_YAT_M(64, 64, 3)
  CATTN_TC_YAT_M(128, 128, 3)
  CATTN_TC_YAT_M(128, 64, 3)
#undef CATTN_TC_YAT_M
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
  if (variant == kTau && dk == 64 && dv == 64) return tc::launch<kTau, 64, 64>(p, tq, tk, tv, s);
  if (variant == kTau && dk == 128 && dv == 128) return tc::launch<kTau, 128, 128>(p, tq, tk, tv, s);
  return cudaErrorInvalidValue;
}

cudaError_t launch_row_stats_tc(int variant, int dk, const FwdParams &p, const CUtensorMap &tq,
                                const CUtensorMap &tk, cudaStream_t s) {
#define CATTN_TC_STATS(V, DK_) \
  if (variant == V && dk == DK_) return tc::launch<V, DK_, DK_, 1, true>(p, tq, tk, tk, s);
  CATTN_TC_STATS(kSoftmax, 64)
  CATTN_TC_STATS(kSoftmax, 128)
  CATTN_TC_STATS(kYat, 64)
  CATTN_TC_STATS(kYat, 128)
  CATTN_TC_STATS(kStau, 64)
  CATTN_TC_STATS(kStau, 128)
#undef CATTN_TC_STATS
  return cudaErrorInvalidValue;
}

cudaError_t launch_near_fix_f32(int dk, int dv, int ym, const FwdParams &p, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
#define CATTN_NEAR_F32(DK_, DV_)                                                        \
  if (dk == DK_ && dv == DV_) {                                                         \
    if (ym == 2)                                                                        \
      tc::near_fix_kernel<DK_, DV_, 2, float><<<sms, 256, 0, s>>>(p);                   \
    else if (ym == 3)                                                                   \
      tc::near_fix_kernel<DK_, DV_, 3, float><<<sms, 256, 0, s>>>(p);                   \
    else                                                                                \
      tc::near_fix_kernel<DK_, DV_, 1, float><<<sms, 256, 0, s>>>(p);                   \
    return cudaGetLastError();                                                          \
  }
  CATTN_NEAR_F32(32, 32)
  CATTN_NEAR_F32(32, 64)
  CATTN_NEAR_F32(32, 128)
  CATTN_NEAR_F32(64, 32)
  CATTN_NEAR_F32(64, 64)
  CATTN_NEAR_F32(64, 128)
  CATTN_NEAR_F32(128, 32)
  CATTN_NEAR_F32(128, 64)
  CATTN_NEAR_F32(128, 128)
#undef CATTN_NEAR_F32
  return cudaErrorInvalidValue;
}

cudaError_t launch_tau_finalize(const double *moments, const float *eps, int h, float *tau,
                                double *moments_out, cudaStream_t s) {
  if (h <= 0) return cudaSuccess;
  tc::tau_finalize_kernel<<<(h + 127) / 128, 128, 0, s>>>(moments, eps, h, tau, moments_out);
  return cudaGetLastError();
}

cudaError_t read_and_clear_status(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_status, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_status, &zero, sizeof(unsigned int));
}

}  // namespace cattn
