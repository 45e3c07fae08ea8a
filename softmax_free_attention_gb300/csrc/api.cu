// api.cu -- the C ABI declared in include/cattn.h: argument validation,
// workspace layout, TMA descriptor encoding and kernel dispatch.  Nothing here
// allocates device memory or synchronises (cattn_check_status excepted).
#include <cudaTypedefs.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <chrono>
#include <mutex>

#include "cattn.h"
#include "bwd.h"
#include "kernels.h"

namespace cattn {

// Generations of the key-norm maximum: distinct over the process's calls
// (a word whose generation differs from the call's is replaced, whatever its
// value), never 0, and seeded with the seconds since the epoch so that a
// workspace another process used is unlikely to hold the current one.
unsigned int next_norm_generation() {
  static std::atomic<unsigned int> g{(unsigned int)std::chrono::duration_cast<std::chrono::seconds>(
                                         std::chrono::system_clock::now().time_since_epoch())
                                         .count()};
  unsigned int v = g.fetch_add(1u) + 1u;
  while (v == 0u) v = g.fetch_add(1u) + 1u;
  return v;
}

}  // namespace cattn

namespace {

using namespace cattn;

constexpr int kTile = 128;  // the key-norm vector is padded to a multiple of this

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int tk_pad(const cattn_problem_t *p) { return (p->Tk + kTile - 1) / kTile * kTile; }

bool is_empty(const cattn_problem_t *p) { return p->B == 0 || p->h == 0 || p->Tq == 0; }

// Workspace layout of the bf16 (tensor-core) path, each part 256-byte aligned:
//   ctrl       256 B: the persistent schedule's unit ticket and (Yat) the
//              count of rows listed for the near-key pass (both zeroed by
//              each forward: by the key-norm kernel when the forward takes
//              the norms, else by a memset; the one-launch Yat forward reads
//              neither), then at byte 8 (Yat) the largest key norm as a
//              64-bit (generation << 32 | fp32 bits) word, which needs no
//              zeroing (launch_row_sqnorm_bf16)
//   nk         Yat only: squared k row norms [B*hkv, Tk_pad], fp32 (the
//              query norms are taken in-kernel from the Q tiles)
//   near       Yat only: the rows listed for the near-key pass, (batch*head,
//              row) uint32 pairs, room for every row once per key split
//   part_o     key splits only: unnormalised partial outputs
//              [n_splits, B*h, Tq, dv] fp32
//   part_stat  key splits only: per-row [n_splits, B*h, Tq, 4] fp32
// The fp32 path (kind::tf32 on the tensor cores, three passes) has its own
// layout (ws_tf32).  bf16 with widths the tensor-core kernel has no tiles for
// (the CUDA-core kernel) needs none.
size_t ws_nk_bytes(const cattn_problem_t *p) {
  return align256((size_t)p->B * p->hkv * tk_pad(p) * sizeof(float));
}

struct WsLayout {
  size_t ctrl, nk, near, part_o, part_stat, total;
  size_t near_cap;
  TcSchedule sched;
};

// the control block's words: the unit ticket, the near-key count, and (a
// 64-bit word at byte 8) the largest key norm with its generation
constexpr int kCtrlTicket = 0, kCtrlNearCount = 1, kCtrlNkMax = 2;

// Workspace of the fp32 path, each part 256-byte aligned: the control block
// (the near-key count), the hi / lo parts of q and k in their own layouts and
// of v transposed [B*hkv, dv, Tk_pad], then (Yat) |k|^2 [B*hkv, Tk_pad] and
// the near-key list.
struct WsTf32 {
  size_t ctrl, qh, ql, kh, kl, vth, vtl, nk, near, total;
  size_t near_cap;
};

WsTf32 ws_tf32(int variant, const cattn_problem_t *p) {
  WsTf32 w;
  memset(&w, 0, sizeof(w));
  const size_t nq = (size_t)p->B * p->h * p->Tq * p->dk * 4;
  const size_t nk = (size_t)p->B * p->hkv * p->Tk * p->dk * 4;
  const size_t nvt = (size_t)p->B * p->hkv * p->dv * tk_pad(p) * 4;
  size_t off = 256;
  w.qh = off;
  off += align256(nq);
  w.ql = off;
  off += align256(nq);
  w.kh = off;
  off += align256(nk);
  w.kl = off;
  off += align256(nk);
  w.vth = off;
  off += align256(nvt);
  w.vtl = off;
  off += align256(nvt);
  if (variant == CATTN_YAT) {
    w.nk = off;
    off += ws_nk_bytes(p);
    w.near = off;
    w.near_cap = (size_t)p->B * p->h * p->Tq;
    off += align256(w.near_cap * 8);
  }
  w.total = off;
  return w;
}

WsLayout ws_layout(int variant, const cattn_problem_t *p) {
  WsLayout w;
  memset(&w, 0, sizeof(w));
  if (p->dtype != CATTN_BF16 || !fwd_tc_supported(p->dk, p->dv)) return w;
  w.sched = tc_schedule(p->B, p->h, p->Tq, p->Tk, p->causal);
  size_t off = 0;
  w.ctrl = off;
  off += 256;
  if (variant == CATTN_YAT) {
    w.nk = off;
    off += ws_nk_bytes(p);
    w.near = off;
    w.near_cap = (size_t)w.sched.n_splits * p->B * p->h * p->Tq;
    off += align256(w.near_cap * 8);
  }
  if (w.sched.n_splits > 1) {
    const size_t rows = (size_t)w.sched.n_splits * p->B * p->h * p->Tq;
    w.part_o = off;
    off += align256(rows * p->dv * sizeof(float));
    w.part_stat = off;
    off += align256(rows * 4 * sizeof(float));
  }
  w.total = off;
  return w;
}

size_t forward_ws_bytes(int variant, const cattn_problem_t *p) {
  return p->dtype == CATTN_F32 ? ws_tf32(variant, p).total : ws_layout(variant, p).total;
}

int check_problem(int variant, const cattn_problem_t *p) {
  if (!p) return CATTN_ERR_INVALID_ARG;
  if (variant != CATTN_SOFTMAX && variant != CATTN_YAT && variant != CATTN_STAU)
    return CATTN_ERR_INVALID_ARG;
  if (p->dtype != CATTN_F32 && p->dtype != CATTN_BF16) return CATTN_ERR_INVALID_ARG;
  if (p->B < 0 || p->h < 0 || p->hkv < 1 || p->Tq < 0 || p->dk < 1 || p->dv < 1)
    return CATTN_ERR_INVALID_ARG;
  if (p->Tk < 1) return CATTN_ERR_SHAPE;
  if (p->h % p->hkv != 0) return CATTN_ERR_SHAPE;
  if (p->causal && p->Tq != p->Tk) return CATTN_ERR_SHAPE;
  if (variant != CATTN_YAT && !(p->scale > 0.f && p->scale < 3.0e38f)) return CATTN_ERR_INVALID_ARG;
  if (p->flags & ~(CATTN_FLAG_NORMS_READY | CATTN_FLAG_TEST_STALL)) return CATTN_ERR_INVALID_ARG;
  if (p->yat_m < 0 || p->yat_m > 3) return CATTN_ERR_INVALID_ARG;
  // every (dk, dv) in {32, 64, 128}^2: the tensor-core kernel for bf16 with
  // (64, 64), (128, 128), (128, 64), the CUDA-core kernel otherwise
  if (!fwd_simt_supported(p->dk, p->dv)) return CATTN_ERR_UNSUPPORTED;
  // every index the kernels form stays inside int32 per head and size_t overall
  if ((long long)p->Tq * p->dk > (1ll << 31) || (long long)p->Tk * p->dk > (1ll << 31) ||
      (long long)p->Tk * p->dv > (1ll << 31))
    return CATTN_ERR_UNSUPPORTED;
  if ((long long)p->B * p->h > (1ll << 24)) return CATTN_ERR_UNSUPPORTED;
  // the persistent schedule numbers its units with 32-bit ints
  if (p->dtype == CATTN_BF16 && tc_schedule(p->B, p->h, p->Tq, p->Tk, p->causal).n_units > (1ll << 30))
    return CATTN_ERR_UNSUPPORTED;
  return CATTN_OK;
}

int map_cuda(cudaError_t e) { return e == cudaSuccess ? CATTN_OK : CATTN_ERR_CUDA; }

// bf16 with widths the tensor-core kernel has tiles for
bool on_tensor_cores(const cattn_problem_t *p) {
  return p->dtype == CATTN_BF16 && fwd_tc_supported(p->dk, p->dv);
}

// The library is built for sm_103a only.
int check_device() {
  int dev = 0, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CATTN_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess)
    return CATTN_ERR_CUDA;
  if (cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return CATTN_ERR_CUDA;
  if (major != 10 || minor != 3) return CATTN_ERR_UNSUPPORTED;
  return CATTN_OK;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// A 3-D tiled tensor map [outer, rows, inner] of 2- or 4-byte elements with
// boxes of (128 bytes of inner) x box_rows x 1 and 128-byte swizzle (the
// shared-memory layout the tcgen05 descriptors describe); reads past the
// extents are zeros.  Encoded maps are kept in a small cache keyed by (base
// address, element size, extents, box rows): a map holds nothing but those
// values, so an entry stays valid for any buffer later found at the same
// address with the same shape, and repeated calls on the same tensors skip
// the driver's encode.
struct MapKey {
  uintptr_t base;
  int esize, inner, rows, outer, box_rows;
  bool operator==(const MapKey &o) const {
    return base == o.base && esize == o.esize && inner == o.inner && rows == o.rows &&
           outer == o.outer && box_rows == o.box_rows;
  }
};
constexpr int kMapCache = 64;
struct MapCache {
  std::mutex mu;
  MapKey key[kMapCache];
  CUtensorMap map[kMapCache];
  int used = 0, next = 0;
};
MapCache &map_cache() {
  static MapCache c;
  return c;
}

int encode_3d(CUtensorMap *map, const void *base, int esize, int inner, int rows, int outer,
              int box_rows) {
  const MapKey k{reinterpret_cast<uintptr_t>(base), esize, inner, rows, outer, box_rows};
  MapCache &c = map_cache();
  {
    std::lock_guard<std::mutex> lock(c.mu);
    for (int i = 0; i < c.used; ++i)
      if (c.key[i] == k) {
        *map = c.map[i];
        return CATTN_OK;
      }
  }
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return CATTN_ERR_CUDA;
  cuuint64_t dims[3] = {(cuuint64_t)inner, (cuuint64_t)rows, (cuuint64_t)outer};
  cuuint64_t strides[2] = {(cuuint64_t)inner * esize, (cuuint64_t)rows * inner * esize};
  cuuint32_t box[3] = {(cuuint32_t)(128 / esize), (cuuint32_t)box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, esize == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                  3, const_cast<void *>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return CATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(c.mu);
  const int slot = c.used < kMapCache ? c.used++ : (c.next++ % kMapCache);
  c.key[slot] = k;
  c.map[slot] = *map;
  return CATTN_OK;
}

// fp32 [outer, rows, inner] with boxes of 32 x box_rows x 1 (128-byte rows).
int encode_f32_3d(CUtensorMap *map, const void *base, int inner, int rows, int outer,
                  int box_rows) {
  return encode_3d(map, base, 4, inner, rows, outer, box_rows);
}

// bf16 [BH, T, d] with boxes of 64 x box_rows x 1.  Rows past T read as zeros.
int encode_bf16_3d(CUtensorMap *map, const void *base, int d, int T, int BH, int box_rows) {
  return encode_3d(map, base, 2, d, T, BH, box_rows);
}

}  // namespace

extern "C" {

int cattn_version(void) { return 100; }

const char *cattn_error_string(int status) {
  switch (status) {
    case CATTN_OK: return "ok";
    case CATTN_ERR_INVALID_ARG: return "invalid argument";
    case CATTN_ERR_SHAPE: return "inconsistent shape";
    case CATTN_ERR_UNSUPPORTED: return "unsupported configuration";
    case CATTN_ERR_CUDA: return "CUDA error";
    case CATTN_ERR_TIMEOUT: return "kernel wait timed out";
    case CATTN_ERR_SCRATCH_LIMIT: return "problem exceeds the fixed scratch of cattn_forward_noalloc";
    default: return "unknown status";
  }
}

size_t cattn_workspace_bytes(int variant, const cattn_problem_t *p) {
  if (check_problem(variant, p) != CATTN_OK) return 0;
  return forward_ws_bytes(variant, p);
}

int cattn_validate(int variant, const cattn_problem_t *p, const void *q, const void *k,
                   const void *v, const float *b, const float *eps, const float *tau,
                   const void *out, const void *workspace, size_t workspace_bytes) {
  int rc = check_problem(variant, p);
  if (rc != CATTN_OK) return rc;
  if (is_empty(p)) return CATTN_OK;
  if (!q || !k || !v || !out) return CATTN_ERR_INVALID_ARG;
  if (variant == CATTN_YAT && (!b || !eps)) return CATTN_ERR_INVALID_ARG;
  if (variant == CATTN_STAU && (!eps || !tau)) return CATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out))
    return CATTN_ERR_UNSUPPORTED;
  const size_t need = forward_ws_bytes(variant, p);
  if (need > 0) {
    if (!workspace) return CATTN_ERR_INVALID_ARG;
    if (workspace_bytes < need) return CATTN_ERR_SHAPE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CATTN_ERR_UNSUPPORTED;
  }
  return CATTN_OK;
}

int cattn_key_norms(const cattn_problem_t *p, const void *k, void *workspace,
                    size_t workspace_bytes, cattn_stream_t stream) {
  int rc = check_problem(CATTN_YAT, p);
  if (rc != CATTN_OK) return rc;
  if (p->dtype != CATTN_BF16) return CATTN_ERR_UNSUPPORTED;
  if (is_empty(p) || !on_tensor_cores(p)) return CATTN_OK;  // the CUDA-core path needs no norms
  if (!k || !workspace) return CATTN_ERR_INVALID_ARG;
  if (!aligned16(k) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return CATTN_ERR_UNSUPPORTED;
  const WsLayout w = ws_layout(CATTN_YAT, p);
  if (workspace_bytes < w.total) return CATTN_ERR_SHAPE;
  rc = check_device();
  if (rc != CATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  float *nk = reinterpret_cast<float *>(static_cast<char *>(workspace) + w.nk);
  unsigned long long *nk_max = reinterpret_cast<unsigned long long *>(
      reinterpret_cast<unsigned int *>(static_cast<char *>(workspace) + w.ctrl) + kCtrlNkMax);
  return map_cuda(launch_row_sqnorm_bf16(k, nk, p->B * p->hkv, p->Tk, tk_pad(p), p->dk, nk_max,
                                         next_norm_generation(), nullptr, 0, s));
}

}  // extern "C"

namespace {

// The forward of cattn_forward and cattn_forward_entropy (row_entropy NULL
// for the former).
int forward_impl(int variant, const cattn_problem_t *p, const void *q, const void *k,
                 const void *v, const float *b, const float *eps, const float *tau, void *out,
                 float *row_mass, float *row_max_score, float *row_entropy, void *workspace,
                 size_t workspace_bytes, cattn_stream_t stream) {
  int rc = cattn_validate(variant, p, q, k, v, b, eps, tau, out, workspace, workspace_bytes);
  if (rc != CATTN_OK) return rc;
  if (is_empty(p)) return CATTN_OK;
  rc = check_device();
  if (rc != CATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);

  FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  fp.q = q;
  fp.k = k;
  fp.v = v;
  fp.out = out;
  fp.out_align32 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
  fp.row_mass = row_mass;
  fp.row_max = row_max_score;
  fp.row_entropy = row_entropy;
  fp.b = b;
  fp.eps = eps;
  fp.tau = tau;
  fp.yat_m = p->yat_m > 1 ? p->yat_m : 1;
  fp.B = p->B;
  fp.h = p->h;
  fp.hkv = p->hkv;
  fp.Tq = p->Tq;
  fp.Tk = p->Tk;
  fp.Tk_pad = tk_pad(p);
  fp.causal = p->causal ? 1 : 0;
  fp.scale = p->scale;
  fp.n_qtiles = (p->Tq + kTcQueryTile - 1) / kTcQueryTile;
  fp.n_pairs = (fp.n_qtiles + 1) / 2;  // two query tiles per work unit
  fp.n_kv_tiles = (p->Tk + kTcKeyTile - 1) / kTcKeyTile;
  fp.test_stall = (p->flags & CATTN_FLAG_TEST_STALL) ? 1 : 0;

  if (p->dtype == CATTN_F32) {
    // fp32: split q, k, v into tf32 hi / lo parts, then the three-pass
    // tensor-core forward, then (Yat) the near-key pass
    const WsTf32 w = ws_tf32(variant, p);
    char *ws = static_cast<char *>(workspace);
    Tf32Split sp;
    sp.qh = reinterpret_cast<float *>(ws + w.qh);
    sp.ql = reinterpret_cast<float *>(ws + w.ql);
    sp.kh = reinterpret_cast<float *>(ws + w.kh);
    sp.kl = reinterpret_cast<float *>(ws + w.kl);
    sp.vth = reinterpret_cast<float *>(ws + w.vth);
    sp.vtl = reinterpret_cast<float *>(ws + w.vtl);
    sp.nk = variant == CATTN_YAT ? reinterpret_cast<float *>(ws + w.nk) : nullptr;
    fp.nk = sp.nk;
    if (variant == CATTN_YAT) {
      fp.near_count = reinterpret_cast<unsigned int *>(ws + w.ctrl) + kCtrlNearCount;
      fp.near_rows = reinterpret_cast<uint2 *>(ws + w.near);
      fp.near_cap = (unsigned int)(w.near_cap < 0xffffffffu ? w.near_cap : 0xffffffffu);
    }
    Tf32Maps m;
    const int BH = p->B * p->h, BHK = p->B * p->hkv;
    if ((rc = encode_f32_3d(&m.qh, sp.qh, p->dk, p->Tq, BH, 128)) != CATTN_OK) return rc;
    if ((rc = encode_f32_3d(&m.ql, sp.ql, p->dk, p->Tq, BH, 128)) != CATTN_OK) return rc;
    if ((rc = encode_f32_3d(&m.kh, sp.kh, p->dk, p->Tk, BHK, 32)) != CATTN_OK) return rc;
    if ((rc = encode_f32_3d(&m.kl, sp.kl, p->dk, p->Tk, BHK, 32)) != CATTN_OK) return rc;
    if ((rc = encode_f32_3d(&m.vh, sp.vth, fp.Tk_pad, p->dv, BHK, p->dv)) != CATTN_OK) return rc;
    if ((rc = encode_f32_3d(&m.vl, sp.vtl, fp.Tk_pad, p->dv, BHK, p->dv)) != CATTN_OK) return rc;
    // (the split pass also zeroes the near-key count)
    if ((rc = map_cuda(launch_split_tf32(fp, sp, variant, p->dk, p->dv, s))) != CATTN_OK) return rc;
    if ((rc = map_cuda(launch_fwd_tf32(variant, p->dk, p->dv, fp, m, s))) != CATTN_OK) return rc;
    if (variant == CATTN_YAT)
      return map_cuda(launch_near_fix_f32(p->dk, p->dv, fp.yat_m, fp, s));
    return CATTN_OK;
  }
  if (!on_tensor_cores(p))
    return map_cuda(launch_fwd_simt(variant, p->dtype == CATTN_BF16, p->dk, p->dv, fp, s));

  const WsLayout w = ws_layout(variant, p);
  char *ws = static_cast<char *>(workspace);
  fp.n_splits = w.sched.n_splits;
  fp.kv_per_split = w.sched.kv_per_split;
  fp.head_group = w.sched.head_group;
  fp.n_units = (int)w.sched.n_units;
  fp.tile_counter = reinterpret_cast<unsigned int *>(ws + w.ctrl) + kCtrlTicket;
  if (w.sched.n_splits > 1) {
    fp.part_o = reinterpret_cast<float *>(ws + w.part_o);
    fp.part_stat = reinterpret_cast<float *>(ws + w.part_stat);
  }
  // the forward takes the key norms itself unless the caller marked them ready
  const bool own_norms = variant == CATTN_YAT && !(p->flags & CATTN_FLAG_NORMS_READY);
  unsigned int *ctrl = reinterpret_cast<unsigned int *>(ws + w.ctrl);
  const unsigned int gen = own_norms ? next_norm_generation() : 0u;
  if (variant == CATTN_YAT) {
    fp.nk = reinterpret_cast<const float *>(ws + w.nk);
    fp.nk_max = reinterpret_cast<const unsigned long long *>(ctrl + kCtrlNkMax);
    fp.nk_gen = gen;
    fp.near_count = reinterpret_cast<unsigned int *>(ws + w.ctrl) + kCtrlNearCount;
    fp.near_rows = reinterpret_cast<uint2 *>(ws + w.near);
    fp.near_cap = (unsigned int)(w.near_cap < 0xffffffffu ? w.near_cap : 0xffffffffu);
  }
  CUtensorMap tq, tk, tv;
  if ((rc = encode_bf16_3d(&tq, q, p->dk, p->Tq, p->B * p->h, kTcQueryTile)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&tk, k, p->dk, p->Tk, p->B * p->hkv, kTcKeyTile)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&tv, v, p->dv, p->Tk, p->B * p->hkv, kTcKeyTile)) != CATTN_OK) return rc;
  // the unit ticket and the near-key count start at zero: the key-norm
  // kernel zeroes them when this call takes the norms (its maximum carries
  // this call's generation and needs no zeroing), a memset otherwise;
  // softmax and s^tau with no more units than CTAs read neither
  const int grid = tc_grid_size(w.sched.n_units);
  if (grid < 0) return CATTN_ERR_CUDA;
  const bool ticket = w.sched.n_units > grid;
  // a Yat problem whose units all run in one wave with short rows (no key
  // split, key tiles x dk <= 256: up to 512 keys at dk 64, 256 at dk 128;
  // exponent 1, no entropy) is one launch: the fused kernel takes each key
  // tile's norms from shared memory and recomputes its near-key rows itself,
  // and reads no control word.  (The map warps' norm work grows with the
  // tiles and dk: at 1024 keys and dk 128 the one launch measured 28% slower
  // than the key-norm kernel and the fused kernel.)
  fp.inline_norms = own_norms && !ticket && w.sched.n_splits == 1 &&
                    fp.n_kv_tiles * p->dk <= 256 && fp.yat_m == 1 && row_entropy == nullptr;
  if (fp.inline_norms) {
    // nothing before the kernel
  } else if (own_norms) {
    if ((rc = map_cuda(launch_row_sqnorm_bf16(
             k, reinterpret_cast<float *>(ws + w.nk), p->B * p->hkv, p->Tk, tk_pad(p), p->dk,
             reinterpret_cast<unsigned long long *>(ctrl + kCtrlNkMax), gen, ctrl, 2, s))) !=
        CATTN_OK)
      return rc;
  } else if ((variant == CATTN_YAT || ticket) &&
             (rc = map_cuda(cudaMemsetAsync(ctrl, 0, 2 * sizeof(unsigned int), s))) != CATTN_OK) {
    return rc;
  }
  return map_cuda(launch_fwd_tc(variant, p->dk, p->dv, fp, tq, tk, tv, s));
}

}  // namespace

extern "C" {

int cattn_forward(int variant, const cattn_problem_t *p, const void *q, const void *k,
                  const void *v, const float *b, const float *eps, const float *tau, void *out,
                  float *row_mass, float *row_max_score, void *workspace,
                  size_t workspace_bytes, cattn_stream_t stream) {
  return forward_impl(variant, p, q, k, v, b, eps, tau, out, row_mass, row_max_score, nullptr,
                      workspace, workspace_bytes, stream);
}

int cattn_forward_entropy(int variant, const cattn_problem_t *p, const void *q, const void *k,
                          const void *v, const float *b, const float *eps, const float *tau,
                          void *out, float *row_mass, float *row_max_score, float *row_entropy,
                          void *workspace, size_t workspace_bytes, cattn_stream_t stream) {
  int rc = check_problem(variant, p);
  if (rc != CATTN_OK) return rc;
  if (!on_tensor_cores(p) || p->yat_m > 1) return CATTN_ERR_UNSUPPORTED;
  if (is_empty(p)) return CATTN_OK;
  if (!row_entropy) return CATTN_ERR_INVALID_ARG;
  return forward_impl(variant, p, q, k, v, b, eps, tau, out, row_mass, row_max_score, row_entropy,
                      workspace, workspace_bytes, stream);
}

// The tau* pass reads no V: its problem is checked as an s^tau problem whose
// value width equals the key width.
cattn_problem_t tau_problem(const cattn_problem_t *p) {
  cattn_problem_t q = *p;
  q.dv = q.dk;
  return q;
}

size_t tau_ws_bytes(const cattn_problem_t *p) {
  return 256 + align256((size_t)p->h * 6 * sizeof(double));
}

size_t cattn_tau_star_workspace_bytes(const cattn_problem_t *p) {
  if (!p) return 0;
  const cattn_problem_t tp = tau_problem(p);
  if (check_problem(CATTN_STAU, &tp) != CATTN_OK || !on_tensor_cores(&tp)) return 0;
  return tau_ws_bytes(&tp);
}

int cattn_tau_star(const cattn_problem_t *p, const void *q, const void *k, const float *eps,
                   float *tau_star, double *moments, void *workspace, size_t workspace_bytes,
                   cattn_stream_t stream) {
  if (!p) return CATTN_ERR_INVALID_ARG;
  const cattn_problem_t tp = tau_problem(p);
  int rc = check_problem(CATTN_STAU, &tp);
  if (rc != CATTN_OK) return rc;
  if (!on_tensor_cores(&tp)) return CATTN_ERR_UNSUPPORTED;
  if (tp.h == 0) return CATTN_OK;
  if (!eps || !tau_star || !workspace) return CATTN_ERR_INVALID_ARG;
  if (!is_empty(&tp) && (!q || !k)) return CATTN_ERR_INVALID_ARG;
  if (!is_empty(&tp) && (!aligned16(q) || !aligned16(k))) return CATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return CATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < tau_ws_bytes(&tp)) return CATTN_ERR_SHAPE;
  rc = check_device();
  if (rc != CATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  double *acc = reinterpret_cast<double *>(ws + 256);
  // the ticket and the moments start at zero
  if ((rc = map_cuda(cudaMemsetAsync(ws, 0, tau_ws_bytes(&tp), s))) != CATTN_OK) return rc;
  if (!is_empty(&tp)) {
    const TcSchedule sched = tc_schedule(tp.B, tp.h, tp.Tq, tp.Tk, tp.causal);
    FwdParams fp;
    memset(&fp, 0, sizeof(fp));
    fp.q = q;
    fp.k = k;
    fp.eps = eps;
    fp.B = tp.B;
    fp.h = tp.h;
    fp.hkv = tp.hkv;
    fp.Tq = tp.Tq;
    fp.Tk = tp.Tk;
    fp.Tk_pad = tk_pad(&tp);
    fp.causal = tp.causal ? 1 : 0;
    fp.scale = tp.scale;
    fp.n_qtiles = (tp.Tq + kTcQueryTile - 1) / kTcQueryTile;
    fp.n_pairs = (fp.n_qtiles + 1) / 2;
    fp.n_kv_tiles = (tp.Tk + kTcKeyTile - 1) / kTcKeyTile;
    fp.n_splits = sched.n_splits;
    fp.kv_per_split = sched.kv_per_split;
    fp.head_group = sched.head_group;
    fp.n_units = (int)sched.n_units;
    fp.tile_counter = reinterpret_cast<unsigned int *>(ws);
    fp.moments = acc;
    CUtensorMap tq, tk;
    if ((rc = encode_bf16_3d(&tq, q, tp.dk, tp.Tq, tp.B * tp.h, kTcQueryTile)) != CATTN_OK) return rc;
    if ((rc = encode_bf16_3d(&tk, k, tp.dk, tp.Tk, tp.B * tp.hkv, kTcKeyTile)) != CATTN_OK) return rc;
    // the pass reads no V; the K map stands in for the unused V map
    if ((rc = map_cuda(launch_fwd_tc(kTau, tp.dk, tp.dk, fp, tq, tk, tk, s))) != CATTN_OK) return rc;
  }
  return map_cuda(launch_tau_finalize(acc, eps, tp.h, tau_star, moments, s));
}

// The row statistics pass has no key splits (its per-row results need every
// key of the row in one unit): the workspace is the ticket plus, for Yat, the
// key norms.
size_t stats_ws_bytes(int variant, const cattn_problem_t *p) {
  return 256 + (variant == CATTN_YAT ? ws_nk_bytes(p) : 0);
}

size_t cattn_row_stats_workspace_bytes(int variant, const cattn_problem_t *p) {
  if (!p) return 0;
  const cattn_problem_t tp = tau_problem(p);
  if (check_problem(variant, &tp) != CATTN_OK || !on_tensor_cores(&tp) || tp.yat_m > 1) return 0;
  return stats_ws_bytes(variant, &tp);
}

int cattn_row_stats(int variant, const cattn_problem_t *p, const void *q, const void *k,
                    const float *b, const float *eps, const float *tau, const float *row_mass,
                    float *entropy, float *frac_small, float *top10, void *workspace,
                    size_t workspace_bytes, cattn_stream_t stream) {
  if (!p) return CATTN_ERR_INVALID_ARG;
  const cattn_problem_t tp = tau_problem(p);
  int rc = check_problem(variant, &tp);
  if (rc != CATTN_OK) return rc;
  if (!on_tensor_cores(&tp) || tp.yat_m > 1) return CATTN_ERR_UNSUPPORTED;
  if (is_empty(&tp)) return CATTN_OK;
  if (!q || !k || !row_mass || !workspace) return CATTN_ERR_INVALID_ARG;
  if (variant == CATTN_YAT && (!b || !eps)) return CATTN_ERR_INVALID_ARG;
  if (variant == CATTN_STAU && (!eps || !tau)) return CATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k) || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
    return CATTN_ERR_UNSUPPORTED;
  if (workspace_bytes < stats_ws_bytes(variant, &tp)) return CATTN_ERR_SHAPE;
  rc = check_device();
  if (rc != CATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  char *ws = static_cast<char *>(workspace);
  FwdParams fp;
  memset(&fp, 0, sizeof(fp));
  fp.q = q;
  fp.k = k;
  fp.b = b;
  fp.eps = eps;
  fp.tau = tau;
  fp.yat_m = 1;
  fp.B = tp.B;
  fp.h = tp.h;
  fp.hkv = tp.hkv;
  fp.Tq = tp.Tq;
  fp.Tk = tp.Tk;
  fp.Tk_pad = tk_pad(&tp);
  fp.causal = tp.causal ? 1 : 0;
  fp.scale = tp.scale;
  fp.n_qtiles = (tp.Tq + kTcQueryTile - 1) / kTcQueryTile;
  fp.n_pairs = (fp.n_qtiles + 1) / 2;
  fp.n_kv_tiles = (tp.Tk + kTcKeyTile - 1) / kTcKeyTile;
  fp.n_splits = 1;
  fp.kv_per_split = fp.n_kv_tiles;
  fp.head_group = 16;
  fp.n_units = tp.B * tp.h * fp.n_pairs;
  fp.tile_counter = reinterpret_cast<unsigned int *>(ws);
  fp.norm_in = row_mass;
  fp.st_entropy = entropy;
  fp.st_small = frac_small;
  fp.st_top10 = top10;
  CUtensorMap tq, tk;
  if ((rc = encode_bf16_3d(&tq, q, tp.dk, tp.Tq, tp.B * tp.h, kTcQueryTile)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&tk, k, tp.dk, tp.Tk, tp.B * tp.hkv, kTcKeyTile)) != CATTN_OK) return rc;
  if (variant == CATTN_YAT) {
    // the key norms and their maximum (64-bit word at byte 8, this call's
    // generation) into this workspace; the norm kernel zeroes the ticket
    fp.nk = reinterpret_cast<const float *>(ws + 256);
    unsigned long long *nk_max = reinterpret_cast<unsigned long long *>(ws + 8);
    fp.nk_max = nk_max;
    fp.nk_gen = next_norm_generation();
    if ((rc = map_cuda(launch_row_sqnorm_bf16(k, reinterpret_cast<float *>(ws + 256), tp.B * tp.hkv,
                                              tp.Tk, tk_pad(&tp), tp.dk, nk_max, fp.nk_gen,
                                              fp.tile_counter, 1, s))) != CATTN_OK)
      return rc;
  } else if ((rc = map_cuda(cudaMemsetAsync(fp.tile_counter, 0, sizeof(unsigned int), s))) !=
             CATTN_OK) {
    return rc;
  }
  return map_cuda(launch_row_stats_tc(variant, tp.dk, fp, tq, tk, s));
}

}  // extern "C"

namespace {

// Backward workspace, each part 256-byte aligned:
//   dpar   [h][2] fp64 per-head parameter gradient sums (zeroed by each call),
//          then (Yat) the largest key norm as a 64-bit generation-tagged word
//   aux    three planes [B*h, Tq_pad] of floats: D, normaliser, |q|^2 per
//          query row (room for four)
//   nk     Yat only: squared k row norms [B*hkv, Tk_pad]
struct BwdWs {
  size_t dpar, nkmax, aux, nk, total;
};

int tq_pad(const cattn_problem_t *p) { return (p->Tq + kTile - 1) / kTile * kTile; }

// bf16 with widths the tensor-core backward has tiles for
bool bwd_on_tensor_cores(const cattn_problem_t *p) {
  return p->dtype == CATTN_BF16 && bwd_tc_supported(p->dk, p->dv);
}

BwdWs bwd_ws(int variant, const cattn_problem_t *p) {
  BwdWs w;
  memset(&w, 0, sizeof(w));
  w.dpar = 0;
  w.nkmax = (size_t)p->h * 2 * sizeof(double);
  size_t off = align256(w.nkmax + sizeof(unsigned long long));
  w.aux = off;
  if (!bwd_on_tensor_cores(p)) {  // the CUDA-core path: the rows' D and (Yat) Z
    off += align256((size_t)2 * p->B * p->h * p->Tq * sizeof(float));
    w.total = off;
    return w;
  }
  off += align256((size_t)p->B * p->h * tq_pad(p) * 16);
  if (variant == CATTN_YAT) {
    w.nk = off;
    off += ws_nk_bytes(p);
  }
  w.total = off;
  return w;
}

int check_bwd_problem(int variant, const cattn_problem_t *p) {
  int rc = check_problem(variant, p);
  if (rc != CATTN_OK) return rc;
  if (!fwd_simt_supported(p->dk, p->dv)) return CATTN_ERR_UNSUPPORTED;
  return CATTN_OK;
}

}  // namespace

extern "C" {

size_t cattn_backward_workspace_bytes(int variant, const cattn_problem_t *p) {
  if (check_bwd_problem(variant, p) != CATTN_OK) return 0;
  return bwd_ws(variant, p).total;
}

int cattn_backward(int variant, const cattn_problem_t *p, const void *q, const void *k,
                   const void *v, const void *out, const void *dout, const float *b,
                   const float *eps, const float *tau, const float *row_mass, void *dq, void *dk,
                   void *dv, float *db, float *deps, float *dtau, void *workspace,
                   size_t workspace_bytes, cattn_stream_t stream) {
  int rc = check_bwd_problem(variant, p);
  if (rc != CATTN_OK) return rc;
  const bool empty = is_empty(p);
  // dk and dv are written even without query rows (as zeros); dq has no
  // elements then
  const bool kv_empty = p->B == 0 || p->hkv == 0;
  if ((!kv_empty && (!dk || !dv)) || (!empty && !dq)) return CATTN_ERR_INVALID_ARG;
  if (!aligned16(dq) || !aligned16(dk) || !aligned16(dv)) return CATTN_ERR_UNSUPPORTED;
  if (!empty) {
    if (!q || !k || !v || !out || !dout || !row_mass || !workspace) return CATTN_ERR_INVALID_ARG;
    if (variant == CATTN_YAT && (!b || !eps)) return CATTN_ERR_INVALID_ARG;
    if (variant == CATTN_STAU && (!eps || !tau)) return CATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(dout) ||
        (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return CATTN_ERR_UNSUPPORTED;
    if (workspace_bytes < bwd_ws(variant, p).total) return CATTN_ERR_SHAPE;
  }
  rc = check_device();
  if (rc != CATTN_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (empty) {
    // no query rows: every gradient is zero
    const size_t es = p->dtype == CATTN_F32 ? 4 : 2;
    const size_t kbytes = (size_t)p->B * p->hkv * p->Tk * p->dk * es;
    const size_t vbytes = (size_t)p->B * p->hkv * p->Tk * p->dv * es;
    if (!kv_empty && (rc = map_cuda(cudaMemsetAsync(dk, 0, kbytes, s))) != CATTN_OK) return rc;
    if (!kv_empty && (rc = map_cuda(cudaMemsetAsync(dv, 0, vbytes, s))) != CATTN_OK) return rc;
    for (float *g : {db, deps, dtau})
      if (g && (rc = map_cuda(cudaMemsetAsync(g, 0, (size_t)p->h * sizeof(float), s))) != CATTN_OK)
        return rc;
    return CATTN_OK;
  }
  const BwdWs w = bwd_ws(variant, p);
  char *ws = static_cast<char *>(workspace);
  if (!bwd_on_tensor_cores(p)) {
    BwdSimtParams sp;
    memset(&sp, 0, sizeof(sp));
    sp.q = q;
    sp.k = k;
    sp.v = v;
    sp.dout = dout;
    sp.row_mass = row_mass;
    sp.b = b;
    sp.eps = eps;
    sp.tau = tau;
    sp.dq = dq;
    sp.dk = dk;
    sp.dv = dv;
    sp.Dbuf = reinterpret_cast<float *>(ws + w.aux);
    sp.dpar = reinterpret_cast<double *>(ws + w.dpar);
    sp.B = p->B;
    sp.h = p->h;
    sp.hkv = p->hkv;
    sp.Tq = p->Tq;
    sp.Tk = p->Tk;
    sp.causal = p->causal ? 1 : 0;
    sp.scale = p->scale;
    if ((rc = map_cuda(cudaMemsetAsync(ws, 0, w.aux, s))) != CATTN_OK) return rc;
    if ((rc = map_cuda(launch_bwd_simt(variant, p->dtype == CATTN_BF16, p->dk, p->dv,
                                       p->yat_m > 1 ? p->yat_m : 1, sp, s))) != CATTN_OK)
      return rc;
    return map_cuda(launch_bwd_param_finalize(variant, sp.dpar, p->h, db, deps, dtau, s));
  }
  BwdParams bp;
  memset(&bp, 0, sizeof(bp));
  bp.aux = reinterpret_cast<const float *>(ws + w.aux);
  bp.aux_w = reinterpret_cast<float *>(ws + w.aux);
  bp.aux_plane = (size_t)p->B * p->h * tq_pad(p);
  bp.b = b;
  bp.eps = eps;
  bp.tau = tau;
  bp.dq = dq;
  bp.dk = dk;
  bp.dv = dv;
  bp.dpar = reinterpret_cast<double *>(ws + w.dpar);
  bp.B = p->B;
  bp.h = p->h;
  bp.hkv = p->hkv;
  bp.Tq = p->Tq;
  bp.Tk = p->Tk;
  bp.Tq_pad = tq_pad(p);
  bp.Tk_pad = tk_pad(p);
  bp.causal = p->causal ? 1 : 0;
  bp.scale = p->scale;
  bp.n_q64 = (p->Tq + 63) / 64;
  bp.n_q128 = (p->Tq + 127) / 128;
  bp.n_k64 = (p->Tk + 63) / 64;
  bp.n_k128 = (p->Tk + 127) / 128;
  // the parameter sums and the key-norm maximum start at zero
  if ((rc = map_cuda(cudaMemsetAsync(ws, 0, w.aux, s))) != CATTN_OK) return rc;
  if (variant == CATTN_YAT) {
    bp.nk = reinterpret_cast<const float *>(ws + w.nk);
    unsigned long long *nk_max = reinterpret_cast<unsigned long long *>(ws + w.nkmax);
    if ((rc = map_cuda(launch_row_sqnorm_bf16(k, reinterpret_cast<float *>(ws + w.nk),
                                              p->B * p->hkv, p->Tk, tk_pad(p), p->dk, nk_max,
                                              next_norm_generation(), nullptr, 0, s))) != CATTN_OK)
      return rc;
  }
  if ((rc = map_cuda(launch_bwd_prep(variant, p->dk, p->dv, bp, q, out, dout, row_mass, s))) !=
      CATTN_OK)
    return rc;
  BwdMaps m;
  const int BH = p->B * p->h, BHK = p->B * p->hkv, dk_ = p->dk, dv_ = p->dv;
  if ((rc = encode_bf16_3d(&m.q128, q, dk_, p->Tq, BH, 128)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.do128, dout, dv_, p->Tq, BH, 128)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.k128, k, dk_, p->Tk, BHK, 128)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.v128, v, dv_, p->Tk, BHK, 128)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.q64, q, dk_, p->Tq, BH, 64)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.do64, dout, dv_, p->Tq, BH, 64)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.k64, k, dk_, p->Tk, BHK, 64)) != CATTN_OK) return rc;
  if ((rc = encode_bf16_3d(&m.v64, v, dv_, p->Tk, BHK, 64)) != CATTN_OK) return rc;
  if ((rc = map_cuda(launch_bwd_tc(variant, dk_, dv_, p->yat_m > 1 ? p->yat_m : 1, bp, m, s))) !=
      CATTN_OK)
    return rc;
  return map_cuda(launch_bwd_param_finalize(variant, bp.dpar, p->h, db, deps, dtau, s));
}

int cattn_check_status(cattn_stream_t stream) {
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return CATTN_ERR_CUDA;
  unsigned int status = 0, bstatus = 0, tstatus = 0;
  if (read_and_clear_status(&status) != cudaSuccess) return CATTN_ERR_CUDA;
  if (read_and_clear_bwd_status(&bstatus) != cudaSuccess) return CATTN_ERR_CUDA;
  if (read_and_clear_tf32_status(&tstatus) != cudaSuccess) return CATTN_ERR_CUDA;
  return (status | bstatus | tstatus) ? CATTN_ERR_TIMEOUT : CATTN_OK;
}

}  // extern "C"
