// noalloc.cu -- cattn_forward_noalloc: the forward for callers that cannot
// allocate device memory.
//
// Some callers must not allocate device memory on the call path: a plug-in
// inside a host engine that plans all device memory up front and forbids
// allocations after start-up, or a latency-critical loop where the implicit
// synchronisation of cudaMalloc is unacceptable.  cattn_forward asks them for
// a workspace (the work-unit ticket, the fp32 squared row norms of the bf16
// Yat map, the partials of a key split); this entry point supplies it from a
// fixed array in device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU on which the
// library's module is loaded holds its kScratchBytes until the process exits.
// Host code may only refer to it through the address cudaGetSymbolAddress
// returns (its name in host code is a host-side stand-in, not a device
// address); that address is looked up once per device, on the first call made
// with that device current.
#include <stdint.h>

#include <mutex>

#include "cattn.h"
#include "kernels.h"

static constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices];

// Device address of the scratch array on the current device.
int scratch_address(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return CATTN_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return CATTN_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void *addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return CATTN_ERR_CUDA;
    g_scratch_addr[dev] = addr;
  }
  *out = g_scratch_addr[dev];
  return CATTN_OK;
}

}  // namespace

extern "C" {

int cattn_forward_noalloc(int variant, const cattn_problem_t *p, const void *q, const void *k,
                          const void *v, const float *b, const float *eps, const float *tau,
                          void *out, float *row_mass, float *row_max_score,
                          cattn_stream_t stream) {
  if (p == nullptr) return CATTN_ERR_INVALID_ARG;
  // the shared array can never hold norms the caller computed
  if (p->flags & CATTN_FLAG_NORMS_READY) return CATTN_ERR_INVALID_ARG;
  const size_t need = cattn_workspace_bytes(variant, p);
  if (need == 0)  // no scratch needed (or an invalid problem, which cattn_forward reports)
    return cattn_forward(variant, p, q, k, v, b, eps, tau, out, row_mass, row_max_score, nullptr,
                         0, stream);
  if (need > kScratchBytes) return CATTN_ERR_SCRATCH_LIMIT;
  void *scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != CATTN_OK) return rc;
  // cattn_forward zeroes the ticket and rewrites every norm and partial it
  // reads (padding included), so stale contents from an earlier call never
  // leak into this one
  return cattn_forward(variant, p, q, k, v, b, eps, tau, out, row_mass, row_max_score, scratch,
                       kScratchBytes, stream);
}

}  // extern "C"
