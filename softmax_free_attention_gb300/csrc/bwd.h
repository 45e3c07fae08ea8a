// bwd.h -- host-side launch interface of the backward kernels (bwd_tc.cu,
// bwd_simt.cu).  Internal to the library.
#pragma once

#include "kernels.h"

namespace cattn {

// Everything the backward kernels read besides the tensor maps.
struct BwdParams {
  // per query row, three planes of [B*h, Tq_pad] floats aux_plane apart:
  // D = dout . out (as -D or -D / Z), the normaliser, |q|^2 + eps (Yat), so
  // that a pass streaming query rows reads each quantity of two adjacent
  // rows as one pair
  const float *aux;
  float *aux_w;                // the same planes, written (the row-sum pass rewrites D and 1 / Z)
  size_t aux_plane;
  const float *nk;             // [B*hkv, Tk_pad] squared k row norms (Yat), zero padded
  const float *b, *eps, *tau;  // [h]
  void *dq, *dk, *dv;          // bf16, shaped like q, k, v
  double *dpar;                // [h][2]: Yat (b, eps), s^tau (eps, tau); zeroed
  int B, h, hkv, Tq, Tk, Tq_pad, Tk_pad, causal;
  float scale;
  int n_q64, n_q128, n_k64, n_k128;  // tiles of 64 and 128 rows
};
// Tensor maps of the backward: q, dout, k, v with 128-row and 64-row boxes
// (q and k rows dk wide, v and dout rows dv wide).
struct BwdMaps {
  CUtensorMap q128, do128, k128, v128, q64, do64, k64, v64;
};
bool bwd_tc_supported(int dk, int dv);
// The per-row D, normaliser and |q|^2 (into p.aux) from q, out, dout and
// the forward's row_mass.
cudaError_t launch_bwd_prep(int variant, int dk, int dv, const BwdParams &p, const void *q,
                            const void *out, const void *dout, const float *row_mass,
                            cudaStream_t s);
// The dK/dV pass, then the dQ pass.
cudaError_t launch_bwd_tc(int variant, int dk, int dv, int yat_m, const BwdParams &p,
                          const BwdMaps &m, cudaStream_t s);
// Backward on the CUDA cores: fp32 inputs, and bf16 inputs whose widths have
// no tensor-core tiles; any (dk, dv) in {32, 64, 128}^2.
struct BwdSimtParams {
  const void *q, *k, *v, *dout;  // fp32 or bf16
  const float *row_mass, *b, *eps, *tau;
  void *dq, *dk, *dv;            // the inputs' element type
  float *Dbuf;   // [2][B*h*Tq] the rows' D and (Yat) Z, written by the dQ pass
  double *dpar;  // [h][2], zeroed
  int B, h, hkv, Tq, Tk, causal;
  float scale;
};
cudaError_t launch_bwd_simt(int variant, bool bf16, int dk, int dv, int yat_m,
                            const BwdSimtParams &p, cudaStream_t s);

// The fp64 per-head parameter sums into the fp32 outputs (any may be NULL).
cudaError_t launch_bwd_param_finalize(int variant, const double *dpar, int h, float *db,
                                      float *deps, float *dtau, cudaStream_t s);

// Device status word set by the backward kernels whose bounded waits gave up.
cudaError_t read_and_clear_bwd_status(unsigned int *value);

}  // namespace cattn
