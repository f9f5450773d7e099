// dion3_select_rows_noalloc: the row selection of dion3_select_rows for
// callers that cannot hand the library a workspace.
//
// Some callers are not allowed to allocate device memory at the point where
// they step the optimizer: a host program whose memory pool is owned by
// another framework (a caching allocator that must not be bypassed), code with
// a fixed device-memory budget decided up front, or a thin binding over the C
// ABI that has no allocator of its own.  This entry point needs no workspace:
// the per-row l1 norms and sums of squares live in one file-scope device array
// that is part of the library image, so every GPU that loads the library holds
// it (2 x kNoAllocMaxRows floats = 8 MiB) until the process exits.
//
// The scratch array is shared by every call on a device and keeps whatever the
// last call left there.  Nothing in it has to start at zero: each call writes
// every element it later reads.  Two calls whose work overlaps on the GPU (on
// different streams, or from different host threads without ordering) race on
// the array and may return wrong rows; order them on one stream.
//
// Set-up: the first call on each device, with that device current, asks the
// CUDA runtime for the array's device address (cudaGetSymbolAddress) and keeps
// it; make that first call before any stream capture begins.  The kept
// address belongs to the module loaded in the device's context: after a
// cudaDeviceReset it is stale, so this entry point must not be called on that
// device again in the same process.  No call
// allocates: there is no cudaMalloc, cudaFree or allocating library routine on
// this path.
//
// The kernels are the ones dion3_select_rows launches (accumulate + row norms,
// then the radix top-k), unchanged; only the place of their scratch differs.
#include "../../include/dion3.h"
#include "internal.h"

#include <cstdio>
#include <mutex>

namespace dion3 {
namespace {

// Largest batch x rows (row norms per call) the static scratch can hold.
constexpr long long kNoAllocMaxRows = 1LL << 20;

// l1 norms in [0, kNoAllocMaxRows), sums of squares in [kNoAllocMaxRows, 2x).
static __device__ __align__(256) float g_select_scratch[2 * kNoAllocMaxRows];

dion3_status reject(dion3_status st, const char* msg) {
  set_last_error_message(msg);
  return st;
}

dion3_status cuda_reject(const char* what, cudaError_t e) {
  char buf[256];
  snprintf(buf, sizeof buf, "%s: %s", what, cudaGetErrorString(e));
  set_last_error_message(buf);
  return DION3_ERR_CUDA;
}

// Device address of g_select_scratch on the current device, resolved once per
// device (host code must not use the symbol itself as an address).
float* scratch_address(cudaError_t* err) {
  static std::mutex mu;
  static float* addr[64] = {nullptr};
  int dev = 0;
  *err = cudaGetDevice(&dev);
  if (*err != cudaSuccess) return nullptr;
  if (dev < 0 || dev >= 64) {
    *err = cudaErrorInvalidDevice;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    *err = cudaGetSymbolAddress(&p, g_select_scratch);
    if (*err != cudaSuccess) return nullptr;
    addr[dev] = static_cast<float*>(p);
  }
  return addr[dev];
}

}  // namespace
}  // namespace dion3

using namespace dion3;

extern "C" {

dion3_status dion3_select_rows_noalloc(int32_t rows, int32_t cols, int32_t batch, float* const* momentum,
                                       const void* const* grads, int32_t grad_dtype, int32_t k,
                                       int32_t* idx_out, float* fro2_out, dion3_stream_t stream) {
  if (rows < 1 || cols < 1 || batch < 1 || k < 1 || k > rows)
    return reject(DION3_ERR_INVALID_ARG, "need rows, cols, batch >= 1 and 1 <= k <= rows");
  if (static_cast<long long>(batch) * rows > kNoAllocMaxRows)
    return reject(DION3_ERR_INVALID_ARG,
                  "batch * rows exceeds the static scratch of dion3_select_rows_noalloc (1048576 rows)");
  if (batch > 65535) return reject(DION3_ERR_INVALID_ARG, "batch > 65535");
  if (momentum == nullptr || idx_out == nullptr)
    return reject(DION3_ERR_INVALID_ARG, "momentum and idx_out must not be NULL");
  if (grads != nullptr && grad_dtype != DION3_F32 && grad_dtype != DION3_BF16)
    return reject(DION3_ERR_INVALID_ARG, "grad_dtype must be DION3_F32 or DION3_BF16");
  for (int b = 0; b < batch; ++b) {
    if (momentum[b] == nullptr || (reinterpret_cast<uintptr_t>(momentum[b]) & 15u))
      return reject(DION3_ERR_INVALID_ARG, "a momentum pointer is NULL or not 16-byte aligned");
    if (grads != nullptr && (grads[b] == nullptr || (reinterpret_cast<uintptr_t>(grads[b]) & 15u)))
      return reject(DION3_ERR_INVALID_ARG, "a gradient pointer is NULL or not 16-byte aligned");
  }
  cudaError_t e = cudaSuccess;
  float* scratch = scratch_address(&e);
  if (scratch == nullptr) return cuda_reject("cudaGetSymbolAddress of the static scratch", e);
  float* l1 = scratch;
  float* sq = scratch + kNoAllocMaxRows;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const bool vec = cols % 8 == 0;
  for (int b0 = 0; b0 < batch; b0 += kMaxBatchPerLaunch) {
    const int nb = batch - b0 < kMaxBatchPerLaunch ? batch - b0 : kMaxBatchPerLaunch;
    AccumArgs a{};
    a.rows = rows;
    a.cols = cols;
    a.batch = nb;
    a.grad_dtype = grad_dtype;
    for (int i = 0; i < nb; ++i) {
      a.M[i] = momentum[b0 + i];
      a.G[i] = grads ? grads[b0 + i] : nullptr;
    }
    a.l1 = l1 + static_cast<size_t>(b0) * rows;
    a.sq = sq + static_cast<size_t>(b0) * rows;
    if ((e = launch_accum_rownorm(a, vec, s)) != cudaSuccess) return cuda_reject("accum_rownorm launch", e);
  }
  TopkArgs t{};
  t.rows = rows;
  t.k = k;
  t.batch = batch;
  t.l1 = l1;
  t.sq = sq;
  t.idx = idx_out;
  t.fro2 = fro2_out;
  if ((e = launch_topk(t, s)) != cudaSuccess) return cuda_reject("topk launch", e);
  set_last_error_message("");
  return DION3_OK;
}

}  // extern "C"
