/*
 * cattn.h -- C ABI of the pluggable-map attention forward for GB300 (sm_103a).
 *
 * One call computes, for every batch b, query head i and query row t,
 *
 *     out[b,i,t,:] = sum_j w_tj * v[b,g,j,:],    g = i / (h / hkv)
 *
 * where the weights w_tj come from one of three score-to-weight maps:
 *
 *   CATTN_SOFTMAX  scaled dot-product softmax: s_j = scale * q.k_j, masked
 *                  keys excluded, w = exp(s - max) / sum exp(s - max).
 *                  ("Softmax-Free Attention in JAX/Flax NNX", section "One
 *                  module, two compatibility functions", softmax branch;
 *                  "NNX Scaled Dot-Product Attention", "Shapes and the three
 *                  steps").
 *   CATTN_YAT      the Yat compatibility kernel
 *                  kappa_j = (q.k_j + b_i)^2 / (max(|q - k_j|^2, 0) + eps_i)
 *                  on the raw (unscaled) dot product, masked keys get
 *                  kappa = 0, w = kappa / (sum kappa + 1e-9): no exponential
 *                  and no max subtraction.  (Same page, kernel branch; "The
 *                  Kernel Between the Roles", "What the exponential was hired
 *                  to do".)
 *   CATTN_STAU     the s^tau power-law map: s_j = scale * q.k_j,
 *                  phi = softplus(s) + eps_i, w = phi^tau_i / sum phi^tau_i,
 *                  masked keys excluded.  ("s^tau: a focal-length knob for
 *                  attention", core formula.)
 *
 * Telemetry (optional outputs, fp32, [B, h, Tq]):
 *   row_mass       Yat: sum_j kappa_j (the row mass kept as its own channel,
 *                  "What each normalizer forgets").  softmax: log-sum-exp of
 *                  the scaled scores.  s^tau: log sum_j phi_j^tau.
 *   row_max_score  Yat: max_j kappa_j.  softmax and s^tau: max_j s_j (scaled).
 *
 * Memory layout.  All tensors are dense row-major, innermost index last:
 *   q   [B, h,   Tq, dk]      k [B, hkv, Tk, dk]      v [B, hkv, Tk, dv]
 *   out [B, h,   Tq, dv]      (same element type as q, k, v)
 *   b, eps, tau: fp32 [h], one value per query head.
 * All data pointers are DEVICE pointers on the current CUDA device and must
 * be 16-byte aligned (cattn_forward_host also takes host buffers, named so).
 * The caller owns every buffer; the library never allocates, frees or keeps
 * a reference to them after the call returns.
 *
 * Execution.  Every call is asynchronous on `stream` (NULL = legacy default
 * stream) and never synchronises, except cattn_check_status.  Argument
 * errors are reported before anything is enqueued.
 *
 * Errors.  Every entry point returns an int status: CATTN_OK or one of the
 * CATTN_ERR_* codes below; cattn_error_string() names them.
 */
#ifndef CATTN_H
#define CATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same object as cudaStream_t / CUstream. */
typedef struct CUstream_st *cattn_stream_t;

/* Score-to-weight maps. */
enum { CATTN_SOFTMAX = 0, CATTN_YAT = 1, CATTN_STAU = 2 };

/* Element type of q, k, v and out.  Head widths dk, dv: any of 32, 64, 128.
 * bf16 with (dk, dv) = (64, 64), (128, 128) or (128, 64) runs on the tensor
 * cores (tcgen05 kind::f16, fp32 accumulation); bf16 with the other width
 * pairs runs on the CUDA cores in fp32 (widened on load, rounded on store).
 * fp32 runs on the tensor cores as tcgen05 kind::tf32 in three passes (each
 * operand split into tf32 hi and lo parts: hi*hi + hi*lo + lo*hi), which
 * carries products to about 2^-20 of their size. */
enum { CATTN_F32 = 0, CATTN_BF16 = 1 };

/* cattn_problem_t.flags */
enum {
  /* Yat only: the workspace already holds the squared row norms of this k,
   * written by cattn_key_norms for the same problem; skip them. */
  CATTN_FLAG_NORMS_READY = 1,
  /* Testing only: the tensor-core forward (bf16 inputs) starts with a wait on
   * a barrier that nothing completes.  The bounded wait gives up after 20 ms,
   * every role of the kernel leaves its loop (copies already started are
   * waited for, tensor memory is released), the outputs are left undefined,
   * and the next cattn_check_status returns CATTN_ERR_TIMEOUT.  It exercises
   * the kernel's timeout path without a fault; other entry points and the
   * CUDA-core path ignore it. */
  CATTN_FLAG_TEST_STALL = 2
};

/* Status codes. */
enum {
  CATTN_OK = 0,
  CATTN_ERR_INVALID_ARG = 1, /* NULL required pointer, unknown enum, negative size, bad scale */
  CATTN_ERR_SHAPE = 2,       /* h % hkv != 0, causal with Tq != Tk, Tk < 1, workspace too small */
  CATTN_ERR_UNSUPPORTED = 3, /* head width not in the supported set, pointer not 16-byte
                                aligned, device is not sm_103 */
  CATTN_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  CATTN_ERR_TIMEOUT = 5,     /* a kernel gave up on a bounded wait (reported by
                                cattn_check_status) */
  CATTN_ERR_SCRATCH_LIMIT = 6 /* the problem needs more scratch than cattn_forward_noalloc's
                                 fixed array holds */
};

typedef struct {
  int B;      /* batch size (>= 0; 0 is a no-op) */
  int h;      /* query heads (>= 0; 0 is a no-op) */
  int hkv;    /* key/value heads, h % hkv == 0; query head i reads kv head i / (h/hkv) */
  int Tq;     /* query rows per head (>= 0; 0 is a no-op) */
  int Tk;     /* key rows per head (>= 1) */
  int dk;     /* query/key width: 32, 64 or 128 */
  int dv;     /* value width: 32, 64 or 128 (any pair; see the element types above) */
  int dtype;  /* CATTN_F32 or CATTN_BF16 */
  int causal; /* nonzero: key j is allowed for query row t only when j <= t; needs Tq == Tk */
  float scale; /* softmax and s^tau multiply q.k by this (> 0, e.g. 1/sqrt(dk)); Yat ignores it */
  int flags;  /* CATTN_FLAG_* */
  int yat_m;  /* Yat only: numerator (q.k + b)^{2m}, m in {1, 2, 3}; 0 means 1 ("The Kernel
                 Between the Roles", section "The run"); ignored by the other maps */
} cattn_problem_t;

/* Library version, 100*major + minor. */
int cattn_version(void);

/* Static name of a status code. Never NULL. */
const char *cattn_error_string(int status);

/* Bytes of device workspace cattn_forward / cattn_key_norms need for this
 * problem and variant (0 if none), 256-byte aligned.  The bf16 tensor-core
 * path needs a 256-byte control block (its work-unit ticket and, for
 * CATTN_YAT, the count of rows listed for the near-key pass and the largest
 * key norm), plus, for
 * CATTN_YAT, the fp32 squared norms of every key row (padded to a multiple of
 * 128 rows per head) and the near-key list (8 bytes per row and key split),
 * plus, for non-causal problems with few (batch, head, 256-row) units, the
 * fp32 partial outputs and per-row statistics of a fixed split of the keys (at
 * most 64 splits, chosen from the shape alone).  The fp32 path needs the
 * control block, the tf32 hi / lo parts of q, k and of v transposed (keys
 * padded to a multiple of 128): twice the inputs' size, plus, for CATTN_YAT,
 * the key norms and the near-key list.  bf16 widths without tensor-core tiles
 * need none.  The contents need not be initialised.  Returns 0 for an invalid
 * problem as well; cattn_validate says why. */
size_t cattn_workspace_bytes(int variant, const cattn_problem_t *p);

/* Host-side argument checks only: never touches the GPU, never dereferences
 * a pointer.  Returns the status cattn_forward would return before launching
 * anything (CATTN_OK if the arguments are acceptable). */
int cattn_validate(int variant, const cattn_problem_t *p, const void *q, const void *k,
                   const void *v, const float *b, const float *eps, const float *tau,
                   const void *out, const void *workspace, size_t workspace_bytes);

/* Squared L2 norms of the k rows, fp32, computed from the stored bf16 values
 * and written into the workspace: the key half of the Yat map's norm
 * prologue.  |q - k|^2 = |q|^2 + |k|^2 - 2 q.k is assembled from the same dot
 * products the scores need ("Softmax-Free Attention in JAX/Flax NNX", section
 * "One module, two compatibility functions"); the forward kernel takes |q|^2
 * itself from the query tiles it holds, |k|^2 from here because every key
 * tile serves many query tiles.  bf16 problems only.  cattn_forward(CATTN_YAT,
 * ...) runs this itself unless CATTN_FLAG_NORMS_READY is set, except for a
 * problem whose work units all run in one wave with short rows (no key split,
 * Tk <= 512 at dk 64 or 256 at dk 128, yat_m 1), where the forward kernel
 * takes the key norms itself and makes no other launch. */
int cattn_key_norms(const cattn_problem_t *p, const void *k, void *workspace,
                    size_t workspace_bytes, cattn_stream_t stream);

/* The attention forward.  b and eps are required for CATTN_YAT (b >= 0,
 * eps > 0), eps and tau for CATTN_STAU (eps > 0, tau > 0); unused ones may be
 * NULL.  These device values are not read on the host, so their ranges are
 * preconditions, not checked.  row_mass and row_max_score may be NULL.
 * workspace may be NULL when cattn_workspace_bytes() is 0. */
int cattn_forward(int variant, const cattn_problem_t *p, const void *q, const void *k,
                  const void *v, const float *b, const float *eps, const float *tau, void *out,
                  float *row_mass, float *row_max_score, void *workspace,
                  size_t workspace_bytes, cattn_stream_t stream);

/* The forward of cattn_forward, plus each row's normalised entropy of the
 * map's weights written into row_entropy (device fp32 [B, h, Tq], required):
 * -sum_j w_j ln w_j / ln n over the row's n allowed keys, 0 when n = 1 ("The
 * Kernel Between the Roles", section "The run": zero for a row on one key,
 * one for a row spread evenly; Yat weights kappa / (M + 1e-9), as the row
 * statistics pass).  Accumulated in the same pass as the output: each row
 * keeps sum_j f_j log2 f_j of its weights' numerators f (Yat kappa; softmax
 * and s^tau the exponentials on their running max, moved onto a new max
 * exactly as the normaliser is) and writes ln Z - ln 2 (sum f log2 f) / Z
 * (Yat: (M ln Z' - ln 2 sum f log2 f) / Z', Z' = M + 1e-9).  bf16 inputs on
 * the tensor cores with yat_m = 1 only (else CATTN_ERR_UNSUPPORTED); other
 * arguments, the workspace and the errors are those of cattn_forward.  The
 * fraction of weights below 1e-6 and the top-10 mass still need
 * cattn_row_stats. */
int cattn_forward_entropy(int variant, const cattn_problem_t *p, const void *q, const void *k,
                          const void *v, const float *b, const float *eps, const float *tau,
                          void *out, float *row_mass, float *row_max_score, float *row_entropy,
                          void *workspace, size_t workspace_bytes, cattn_stream_t stream);

/* The same forward for callers that cannot allocate device memory (a plug-in
 * whose host engine plans all device memory at start-up and forbids later
 * allocations, or a latency-critical loop that cannot afford cudaMalloc's
 * implicit synchronisation).  The source pages have no counterpart: this is a
 * library convenience, not part of the method.
 *
 * Arguments as cattn_forward, minus the workspace: the scratch comes from a
 * fixed 16 MiB array of device memory inside the library, which every GPU that
 * loads the library holds until the process exits.  Problems whose
 * cattn_workspace_bytes() exceeds 16 MiB (for causal bf16 Yat: B*hkv*Tk_pad
 * above about 4.19 million key rows; non-causal problems whose keys are split
 * need room for the partial outputs as well) are rejected with
 * CATTN_ERR_SCRATCH_LIMIT before anything is enqueued;
 * CATTN_FLAG_NORMS_READY is rejected with CATTN_ERR_INVALID_ARG.  Nothing is
 * allocated or freed.
 *
 * The first call on a device looks up the array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  All calls share the one array and each rewrites what it reads, so
 * calls in sequence are independent, but calls that can overlap on the GPU
 * (different streams, or several threads) race on it and must be serialised by
 * the caller. */
int cattn_forward_noalloc(int variant, const cattn_problem_t *p, const void *q, const void *k,
                          const void *v, const float *b, const float *eps, const float *tau,
                          void *out, float *row_mass, float *row_max_score,
                          cattn_stream_t stream);

/* The forward of q, k, v held in HOST memory, with the outputs written back
 * to host memory: the computation of cattn_forward (the same maps, pages and
 * sections as above) plus the data movement, pipelined over `chunks` chunks
 * of the batch.  Batch entries are independent problems, so chunk c (batch
 * entries [B*c/n, B*(c+1)/n), n = min(chunks, B, 64)) is one cattn_forward
 * call on its slice, and its results equal those of that call bit for bit.
 * Chunk c+1 is copied in on `copy_in` while chunk c runs on `compute` and
 * chunk c-1 is copied out on `copy_out`.
 *
 * q_host, k_host, v_host: host [B,h,Tq,dk], [B,hkv,Tk,dk], [B,hkv,Tk,dv];
 * out_host [B,h,Tq,dv]; row_mass_host, row_max_host: host fp32 [B,h,Tq] or
 * NULL.  Page-locked host memory lets the copies overlap the computation;
 * pageable memory gives the same results with the copies serialised by the
 * CUDA runtime.  b, eps, tau: DEVICE fp32 [h], as for cattn_forward.
 * q_dev, k_dev, v_dev, out_dev: device staging buffers of the full shapes
 * above (16-byte aligned); row_mass_dev / row_max_dev: device fp32 [B,h,Tq],
 * NULL exactly when the host telemetry pointer is NULL.  workspace: at least
 * cattn_forward_host_workspace_bytes() bytes (the workspace of the largest
 * chunk; the chunks share it).  The caller owns every buffer; nothing is
 * allocated per call.
 *
 * Asynchronous: the call returns once everything is enqueued; the host
 * outputs are complete when `copy_out` (or `compute`, which is made to wait
 * for the last copy out) has drained, and no host input may change before
 * `copy_in` has.  Work the caller enqueued earlier on `compute` finishes
 * before the copies touch the staging buffers.  The three streams may be the
 * same stream (then nothing overlaps).  The first call on a device creates
 * the library's pool of 130 CUDA events for that device, kept until exit;
 * make it before any stream capture.  Calls from several host threads are
 * enqueued one at a time.
 *
 * Errors: as cattn_forward, checked for every chunk size before anything is
 * enqueued; CATTN_ERR_INVALID_ARG also for chunks < 1, a NULL host pointer,
 * mismatched telemetry pointers, or CATTN_FLAG_NORMS_READY (the key norms
 * are computed per chunk).  A CUDA error while enqueuing returns
 * CATTN_ERR_CUDA with the chunks before it already enqueued. */
size_t cattn_forward_host_workspace_bytes(int variant, const cattn_problem_t *p, int chunks);
int cattn_forward_host(int variant, const cattn_problem_t *p, const void *q_host,
                       const void *k_host, const void *v_host, const float *b, const float *eps,
                       const float *tau, void *out_host, float *row_mass_host,
                       float *row_max_host, void *q_dev, void *k_dev, void *v_dev, void *out_dev,
                       float *row_mass_dev, float *row_max_dev, void *workspace,
                       size_t workspace_bytes, int chunks, cattn_stream_t compute,
                       cattn_stream_t copy_in, cattn_stream_t copy_out);

/* tau* of the s^tau map, per query head, from one pass over the softmax
 * scores ("s^tau: a focal-length knob for attention", the closed-form
 * paragraph): tau*_i = Cov(s, ln phi(s)) / Var(ln phi(s)) over the scores
 * s = scale * q.k of every allowed (query row, key) pair of query head i,
 * pooled over the batch, with phi(s) = softplus(s) + eps_i.  It is the
 * least-squares slope that makes tau * ln phi(s) + C fit s, i.e. the tau for
 * which the s^tau map tracks the softmax map on these scores.
 *
 * The scores come from the same tensor-core S = Q K^T as the forward (bf16
 * only; dk in {64, 128}; p->dv and v are not used).  Causal masking as in the
 * forward.  eps: device fp32 [h] (> 0, not checked).  tau_star: device fp32
 * [h] output (NaN for a head with fewer than two scores).  moments: optional
 * device fp64 [h][6] output: n, sum s, sum g, sum s g, sum g^2 with
 * g = ln phi(s) - g0, and g0 = ln(ln 2 + eps_i) (the sums are taken from fp32
 * partial sums of each thread's scores in a work unit, added in fp64).
 * workspace: cattn_tau_star_workspace_bytes(p) bytes, 256-byte aligned,
 * contents need not be initialised.  Asynchronous on `stream`. */
size_t cattn_tau_star_workspace_bytes(const cattn_problem_t *p);
int cattn_tau_star(const cattn_problem_t *p, const void *q, const void *k, const float *eps,
                   float *tau_star, double *moments, void *workspace, size_t workspace_bytes,
                   cattn_stream_t stream);

/* Per-row statistics of the attention map, by a second pass over the scores
 * that takes the row normaliser from the forward: for every (b, i, t) the
 * normalised entropy -sum_j w_j ln w_j / ln n over the n allowed keys (0 when
 * n = 1; "The Kernel Between the Roles", section "The run"), the fraction of
 * allowed keys with w_j < 1e-6, and the sum of the ten largest w_j (the
 * sparsity and top-10 concentration of "s^tau: a focal-length knob for
 * attention").  The weights are the forward's: Yat kappa / (M + 1e-9),
 * softmax exp(s - lse), s^tau phi^tau / sum phi^tau.
 *
 * Arguments as cattn_forward, minus v and out: row_mass is the row_mass
 * output of cattn_forward for the same problem and inputs (device fp32
 * [B, h, Tq]); entropy, frac_small, top10 are device fp32 [B, h, Tq]
 * outputs, any of which may be NULL.  bf16 only, dk in {64, 128} (p->dv is
 * not used), Yat with yat_m <= 1.  workspace: cattn_row_stats_workspace_bytes
 * bytes (the Yat key norms are recomputed into it), 256-byte aligned.
 * Asynchronous on `stream`. */
size_t cattn_row_stats_workspace_bytes(int variant, const cattn_problem_t *p);
int cattn_row_stats(int variant, const cattn_problem_t *p, const void *q, const void *k,
                    const float *b, const float *eps, const float *tau, const float *row_mass,
                    float *entropy, float *frac_small, float *top10, void *workspace,
                    size_t workspace_bytes, cattn_stream_t stream);

/* Backward of cattn_forward: the gradients of L = sum(dout * out) with
 * respect to q, k, v and the per-head map parameters, for the forward of the
 * same problem whose out and row_mass are passed in.
 *
 * Per query row t the forward's weights are w_tj = f_tj / Z_t; they are
 * recomputed from the scores and row_mass (softmax, s^tau: log Z; Yat: the
 * library sums its own kappas for Z).  With D_t = sum_j w_tj dW_tj (= dout_t .
 * out_t) and dW_tj = dout_t . v_j:
 *   dv_j = sum_t w_tj dout_t
 *   softmax  dS_tj = w_tj (dW_tj - D_t); dq = scale dS k, dk = scale dS^T q
 *   s^tau    dS_tj = w_tj (dW_tj - D_t) tau sigma(s_tj) / phi(s_tj), same
 *            products; dtau = sum w (dW - D) ln phi, deps = sum w (dW - D) tau / phi
 *   Yat      g = (dW - D) / Z, a = 2m g (q.k + b)^{2m-1} / den,
 *            e = -g kappa / den, den = max(|q - k|^2, 0) + eps;
 *            dq_t = sum_j (a - 2 e [|q-k|^2 > 0]) k_j + 2 q_t sum_j e [..],
 *            dk_j symmetrically; db = sum a, deps = sum e
 * (the chain rule through the maps of "Softmax-Free Attention in JAX/Flax
 * NNX", section "One module, two compatibility functions", and "s^tau: a
 * focal-length knob for attention", core formula).  The sums over query
 * heads sharing a kv head (h > hkv) are taken inside the library.
 *
 *   q, k, v, out  the forward's inputs and output (layouts as above)
 *   dout          [B, h, Tq, dv], the element type of q: dL/d out
 *   row_mass      [B, h, Tq] fp32: the forward's row_mass output
 *   dq, dk, dv    shaped and typed like q, k, v; written, never read
 *   db, deps, dtau  fp32 [h] or NULL: the parameter gradients the map has
 *                 (Yat: db, deps; s^tau: deps, dtau; the others untouched)
 * Widths as for the forward (the tensor cores for bf16 (64, 64), (128, 128),
 * (128, 64); the CUDA cores otherwise); yat_m in {0, 1, 2, 3}; anything else
 * is CATTN_ERR_UNSUPPORTED.  A problem with no query rows writes zeros.  The
 * kernels' accumulation order is fixed: repeated calls give identical bits
 * for dq, dk and dv (the fp64 parameter sums use atomics).
 * cattn_backward_workspace_bytes: bytes needed (0 if the problem is
 * unsupported), 256-byte aligned; the workspace must be 256-byte aligned. */
size_t cattn_backward_workspace_bytes(int variant, const cattn_problem_t *p);
int cattn_backward(int variant, const cattn_problem_t *p, const void *q, const void *k,
                   const void *v, const void *out, const void *dout, const float *b,
                   const float *eps, const float *tau, const float *row_mass, void *dq, void *dk,
                   void *dv, float *db, float *deps, float *dtau, void *workspace,
                   size_t workspace_bytes, cattn_stream_t stream);

/* Synchronises `stream`, then reports (and clears) the device-side status
 * word the kernels set when a bounded wait gives up: CATTN_ERR_TIMEOUT if
 * any kernel since the last check did so, CATTN_ERR_CUDA if the stream
 * reports an error, else CATTN_OK. */
int cattn_check_status(cattn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CATTN_H */
