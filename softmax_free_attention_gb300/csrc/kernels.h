// kernels.h -- host-side launch interface between the C ABI (api.cu) and the
// kernel translation units.  Internal to the library.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace cattn {

// kTau is not a map: the tau* statistics pass over the softmax scores.
enum Variant { kSoftmax = 0, kYat = 1, kStau = 2, kTau = 3 };

// Tile shape of the tensor-core forward: query rows per tile, keys per tile.
constexpr int kTcQueryTile = 128;
constexpr int kTcKeyTile = 128;

// Everything a forward kernel reads besides the tensor maps.
struct FwdParams {
  const void *q, *k, *v;        // element pointers (the tensor-core path reads through TMA)
  void *out;                    // [B, h, Tq, dv]
  int out_align32;              // out is 32-byte aligned (whole-sector stores)
  float *row_mass, *row_max;    // [B, h, Tq] or NULL
  float *row_entropy;           // [B, h, Tq] normalised entropy of the map, or NULL (bf16, yat_m 1)
  const float *b, *eps, *tau;   // [h]
  int yat_m;                    // Yat numerator exponent 2 yat_m (1, 2 or 3)
  const float *nk;              // [B*hkv, Tk_pad]  squared k row norms (Yat, bf16), zero padded
  // the largest of them as (generation << 32) | fp32 bits, and the
  // generation of this call's norms (0: take the word as it is, the caller
  // computed the norms)
  const unsigned long long *nk_max;
  unsigned int nk_gen;
  int B, h, hkv, Tq, Tk, Tk_pad;
  int causal;
  float scale;
  int n_qtiles;    // query tiles per head: ceil(Tq / kTcQueryTile)
  int n_pairs;     // query-tile pairs per head: ceil(n_qtiles / 2)
  int n_kv_tiles;  // ceil(Tk / kTcKeyTile)
  // persistent schedule of the tensor-core forward: one work unit is
  // (batch*head, query-tile pair, key split)
  int n_splits;      // key splits per pair (non-causal only; 1 = no split)
  int kv_per_split;  // key tiles per split
  int head_group;    // (batch, head) pairs whose units are scheduled together
  int n_units;       // B * h * n_pairs * n_splits
  unsigned int *tile_counter;  // next unit to hand out (zero at launch; unread when the units fit in one wave)
  float *part_o;     // [n_splits, B*h, Tq, dv] unnormalised partial outputs (n_splits > 1)
  float *part_stat;  // [n_splits, B*h, Tq, 4]: mass or l, running max (log2), top score
  double *moments;   // kTau: [h][6] sums n, s, g, s g, g^2 (g = ln phi(s) - g0), zeroed
  // row statistics pass: the forward's row_mass as input, three [B, h, Tq]
  // outputs (any may be NULL)
  const float *norm_in;
  float *st_entropy, *st_small, *st_top10;
  // Yat: rows whose max kappa passed the near-key guard, listed by the fused
  // kernel for the near-key pass: (batch * h + head, row) pairs, their count
  // (zeroed before launch) and the list's capacity
  unsigned int *near_count;
  uint2 *near_rows;
  unsigned int near_cap;
  // Yat (bf16, yat_m 1, no entropy): every unit runs in one wave with no key
  // split and at most 256 / dk key tiles, so the fused kernel takes each key
  // tile's norms and recomputes its flagged rows itself; nk, nk_max and the
  // near-key list are not used and no other launch is made
  int inline_norms;
  // test only (CATTN_FLAG_TEST_STALL): the tensor-core forward's MMA warp
  // first waits on a barrier that nothing completes, so that the bounded wait
  // runs out and the kernel takes its abort path
  int test_stall;
};

// Split count and grouping of the persistent tensor-core schedule; a pure
// function of the problem so that the workspace size is known on the host.
struct TcSchedule {
  int n_pairs, n_kv_tiles, n_splits, kv_per_split, head_group;
  long long n_units;
};
TcSchedule tc_schedule(int B, int h, int Tq, int Tk, int causal);

// Tensor-core (tcgen05) forward for bf16 inputs.  Returns a cudaError_t.
// Launches the persistent kernel (and, with key splits, the combine kernel);
// p.tile_counter must already be zero on stream s.
cudaError_t launch_fwd_tc(int variant, int dk, int dv, const FwdParams &p, const CUtensorMap &tq,
                          const CUtensorMap &tk, const CUtensorMap &tv, cudaStream_t s);
bool fwd_tc_supported(int dk, int dv);
// CTAs the persistent forward launches for n_units units (one per SM at
// most), -1 if the device cannot be queried.
int tc_grid_size(long long n_units);

// The row statistics pass: the map's S and weights again (no V), per-row
// normalised entropy, fraction below 1e-6 and top-10 mass.  dk 64 or 128.
cudaError_t launch_row_stats_tc(int variant, int dk, const FwdParams &p, const CUtensorMap &tq,
                                const CUtensorMap &tk, cudaStream_t s);

// tau* per head from the moments the kTau pass accumulated: writes tau[h]
// and, if moments_out is not NULL, the moments with g0 = ln(ln 2 + eps) in
// the sixth slot.
cudaError_t launch_tau_finalize(const double *moments, const float *eps, int h, float *tau,
                                double *moments_out, cudaStream_t s);

// CUDA-core forward: fp32 inputs, and bf16 inputs whose widths have no
// tensor-core tiles; any (dk, dv) in {32, 64, 128}^2.
cudaError_t launch_fwd_simt(int variant, bool bf16, int dk, int dv, const FwdParams &p,
                            cudaStream_t s);
bool fwd_simt_supported(int dk, int dv);

// fp32 inputs on the tensor cores (kind::tf32 in three passes).  The split
// pass writes the hi / lo parts of q and k (their own layouts), of v
// transposed to [B*hkv, dv, Tk_pad] (keys contiguous, zero past Tk) and, for
// Yat, |k|^2 [B*hkv, Tk_pad]; the forward reads them through these maps
// (32-element boxes, 128-byte swizzle): q, k boxes of 128 and 32 rows, v^T
// boxes of 32 keys by dv rows.
struct Tf32Split {
  float *qh, *ql, *kh, *kl, *vth, *vtl, *nk;
};
struct Tf32Maps {
  CUtensorMap qh, ql, kh, kl, vh, vl;
};
// (one launch; it also zeroes p.near_count for Yat)
cudaError_t launch_split_tf32(const FwdParams &p, const Tf32Split &w, int variant, int dk, int dv,
                              cudaStream_t s);
cudaError_t launch_fwd_tf32(int variant, int dk, int dv, const FwdParams &p, const Tf32Maps &m,
                            cudaStream_t s);
cudaError_t read_and_clear_tf32_status(unsigned int *value);
// The near-key pass for fp32 inputs (the bf16 forward launches its own).
cudaError_t launch_near_fix_f32(int dk, int dv, int ym, const FwdParams &p, cudaStream_t s);

// Squared row norms of a bf16 [BH, T, d] tensor into out[BH, T_pad] (zeros
// for padded rows).  Their maximum is folded into *max64 as (gen << 32) |
// fp32 bits by compare-and-swap: a word of another generation (an earlier
// call's, or the workspace's old contents) is replaced and within gen the
// value only grows, so the word needs no zeroing.  Block 0
// also zeroes n_zero words at zero_words (the control words of the kernel
// that follows).
cudaError_t launch_row_sqnorm_bf16(const void *x, float *out, int BH, int T, int T_pad, int d,
                                   unsigned long long *max64, unsigned int gen,
                                   unsigned int *zero_words, int n_zero, cudaStream_t s);
// A generation for launch_row_sqnorm_bf16: strictly increasing over the
// process's calls, never 0.
unsigned int next_norm_generation();

// Device status word set by the forward kernels whose bounded waits gave up.
cudaError_t read_and_clear_status(unsigned int *value);

}  // namespace cattn
