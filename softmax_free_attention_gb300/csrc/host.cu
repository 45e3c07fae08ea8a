// host.cu -- the forward of host-resident q, k, v, pipelined over chunks of
// the batch.
//
// The same computation as cattn_forward (every batch entry is an independent
// attention problem, so a chunk of the batch is one cattn_forward call on its
// slice); what this file adds is the data movement around it.  Chunk i+1 is
// copied to the device on one stream while chunk i is computed on a second
// and chunk i-1 is copied back on a third, ordered by events:
//
//   copy_in :  H2D q,k,v[0]  H2D [1]       H2D [2]  ...
//   compute :           fwd [0]      fwd [1]      fwd [2] ...
//   copy_out:                  D2H [0]      D2H [1]  ...
//
// Nothing here allocates device memory: the caller passes full-size device
// staging buffers and one workspace that fits the largest chunk (the chunks
// run one after another on the compute stream, so they can share it).  The
// events come from a pool made once per device and reused under a mutex:
// cudaStreamWaitEvent takes the event's state at the time of the call, so a
// later call may record the same event again.
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>

#include "cattn.h"

namespace {

constexpr int kMaxChunks = 64;

struct EventPool {
  cudaEvent_t in[kMaxChunks], done[kMaxChunks], start, end;
};

std::mutex g_host_mu;  // guards the event pools and every enqueue sequence below

int elem_bytes(const cattn_problem_t *p) { return p->dtype == CATTN_BF16 ? 2 : 4; }

int chunk_count(const cattn_problem_t *p, int chunks) {
  int n = chunks < p->B ? chunks : p->B;
  if (n > kMaxChunks) n = kMaxChunks;
  return n < 1 ? 1 : n;
}

// The two chunk sizes that occur (edges B*i/n): floor and ceil of B/n.
void chunk_problems(const cattn_problem_t *p, int n, cattn_problem_t *lo, cattn_problem_t *hi) {
  *lo = *p;
  *hi = *p;
  lo->B = p->B / n;
  hi->B = (p->B + n - 1) / n;
}

// The pool of the current device, made on first use (caller holds g_host_mu).
int device_pool(EventPool **out) {
  static std::map<int, EventPool> pools;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CATTN_ERR_CUDA;
  auto it = pools.find(dev);
  if (it == pools.end()) {
    EventPool ep;
    const unsigned fl = cudaEventDisableTiming;
    for (int i = 0; i < kMaxChunks; ++i) {
      if (cudaEventCreateWithFlags(&ep.in[i], fl) != cudaSuccess ||
          cudaEventCreateWithFlags(&ep.done[i], fl) != cudaSuccess)
        return CATTN_ERR_CUDA;
    }
    if (cudaEventCreateWithFlags(&ep.start, fl) != cudaSuccess ||
        cudaEventCreateWithFlags(&ep.end, fl) != cudaSuccess)
      return CATTN_ERR_CUDA;
    it = pools.emplace(dev, ep).first;
  }
  *out = &it->second;
  return CATTN_OK;
}

int cuda_ok(cudaError_t e) { return e == cudaSuccess ? CATTN_OK : CATTN_ERR_CUDA; }

}  // namespace

extern "C" {

size_t cattn_forward_host_workspace_bytes(int variant, const cattn_problem_t *p, int chunks) {
  if (!p || p->B < 0 || chunks < 1) return 0;
  if (p->B == 0) return 0;
  cattn_problem_t lo, hi;
  chunk_problems(p, chunk_count(p, chunks), &lo, &hi);
  const size_t a = lo.B > 0 ? cattn_workspace_bytes(variant, &lo) : 0;
  const size_t b = cattn_workspace_bytes(variant, &hi);
  return a > b ? a : b;
}

int cattn_forward_host(int variant, const cattn_problem_t *p, const void *q_host,
                       const void *k_host, const void *v_host, const float *b, const float *eps,
                       const float *tau, void *out_host, float *row_mass_host,
                       float *row_max_host, void *q_dev, void *k_dev, void *v_dev, void *out_dev,
                       float *row_mass_dev, float *row_max_dev, void *workspace,
                       size_t workspace_bytes, int chunks, cattn_stream_t compute,
                       cattn_stream_t copy_in, cattn_stream_t copy_out) {
  if (!p || chunks < 1) return CATTN_ERR_INVALID_ARG;
  if (p->flags & CATTN_FLAG_NORMS_READY) return CATTN_ERR_INVALID_ARG;  // norms are per chunk
  if ((row_mass_host == nullptr) != (row_mass_dev == nullptr) ||
      (row_max_host == nullptr) != (row_max_dev == nullptr))
    return CATTN_ERR_INVALID_ARG;
  if (p->B == 0 || p->h == 0 || p->Tq == 0)  // nothing to do, once the problem is valid
    return cattn_validate(variant, p, q_dev, k_dev, v_dev, b, eps, tau, out_dev, workspace,
                          workspace_bytes);
  if (!q_host || !k_host || !v_host || !out_host) return CATTN_ERR_INVALID_ARG;
  // each chunk size against the shapes, the device pointers and the
  // workspace (chunk offsets keep 16-byte alignment: a batch entry of q, k,
  // v or out spans a multiple of 64 bytes)
  const int n = chunk_count(p, chunks);
  cattn_problem_t lo, hi;
  chunk_problems(p, n, &lo, &hi);
  int rc = CATTN_OK;
  for (const cattn_problem_t *c : {&lo, &hi}) {
    if (c->B == 0) continue;
    rc = cattn_validate(variant, c, q_dev, k_dev, v_dev, b, eps, tau, out_dev, workspace,
                        workspace_bytes);
    if (rc != CATTN_OK) return rc;
  }

  cudaStream_t sc = reinterpret_cast<cudaStream_t>(compute);
  cudaStream_t si = reinterpret_cast<cudaStream_t>(copy_in);
  cudaStream_t so = reinterpret_cast<cudaStream_t>(copy_out);
  const size_t es = (size_t)elem_bytes(p);
  // bytes per batch entry of each tensor
  const size_t bq = (size_t)p->h * p->Tq * p->dk * es;
  const size_t bk = (size_t)p->hkv * p->Tk * p->dk * es;
  const size_t bv = (size_t)p->hkv * p->Tk * p->dv * es;
  const size_t bo = (size_t)p->h * p->Tq * p->dv * es;
  const size_t bt = (size_t)p->h * p->Tq * sizeof(float);
  auto at = [](const void *base, size_t off) {
    return static_cast<const char *>(base) + off;
  };
  auto atw = [](void *base, size_t off) { return static_cast<char *>(base) + off; };

  std::lock_guard<std::mutex> lock(g_host_mu);
  EventPool *ep = nullptr;
  if ((rc = device_pool(&ep)) != CATTN_OK) return rc;
  // the staging buffers may still be in use by earlier work on the compute stream
  if ((rc = cuda_ok(cudaEventRecord(ep->start, sc))) != CATTN_OK) return rc;
  if ((rc = cuda_ok(cudaStreamWaitEvent(si, ep->start, 0))) != CATTN_OK) return rc;
  if ((rc = cuda_ok(cudaStreamWaitEvent(so, ep->start, 0))) != CATTN_OK) return rc;
  for (int i = 0; i < n; ++i) {
    const int a = (int)((long long)p->B * i / n), z = (int)((long long)p->B * (i + 1) / n);
    if (a == z) continue;
    const size_t nb = (size_t)(z - a);
    cattn_problem_t c = *p;
    c.B = z - a;
    const cudaMemcpyKind h2d = cudaMemcpyHostToDevice, d2h = cudaMemcpyDeviceToHost;
    if ((rc = cuda_ok(cudaMemcpyAsync(atw(q_dev, a * bq), at(q_host, a * bq), nb * bq, h2d, si))) ||
        (rc = cuda_ok(cudaMemcpyAsync(atw(k_dev, a * bk), at(k_host, a * bk), nb * bk, h2d, si))) ||
        (rc = cuda_ok(cudaMemcpyAsync(atw(v_dev, a * bv), at(v_host, a * bv), nb * bv, h2d, si))) ||
        (rc = cuda_ok(cudaEventRecord(ep->in[i], si))) ||
        (rc = cuda_ok(cudaStreamWaitEvent(sc, ep->in[i], 0))))
      return rc;
    rc = cattn_forward(variant, &c, at(q_dev, a * bq), at(k_dev, a * bk), at(v_dev, a * bv), b,
                       eps, tau, atw(out_dev, a * bo),
                       row_mass_dev ? row_mass_dev + (size_t)a * p->h * p->Tq : nullptr,
                       row_max_dev ? row_max_dev + (size_t)a * p->h * p->Tq : nullptr, workspace,
                       workspace_bytes, compute);
    if (rc != CATTN_OK) return rc;
    if ((rc = cuda_ok(cudaEventRecord(ep->done[i], sc))) ||
        (rc = cuda_ok(cudaStreamWaitEvent(so, ep->done[i], 0))) ||
        (rc = cuda_ok(cudaMemcpyAsync(atw(out_host, a * bo), at(out_dev, a * bo), nb * bo, d2h,
                                      so))))
      return rc;
    if (row_mass_dev &&
        (rc = cuda_ok(cudaMemcpyAsync(atw(row_mass_host, a * bt), at(row_mass_dev, a * bt),
                                      nb * bt, d2h, so))))
      return rc;
    if (row_max_dev &&
        (rc = cuda_ok(cudaMemcpyAsync(atw(row_max_host, a * bt), at(row_max_dev, a * bt),
                                      nb * bt, d2h, so))))
      return rc;
  }
  // later work on the compute stream comes after the last copy out
  if ((rc = cuda_ok(cudaEventRecord(ep->end, so))) != CATTN_OK) return rc;
  return cuda_ok(cudaStreamWaitEvent(sc, ep->end, 0));
}

}  // extern "C"
