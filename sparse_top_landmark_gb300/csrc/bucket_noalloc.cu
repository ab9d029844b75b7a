// mita_bucket_noalloc: the bucket step for callers that cannot allocate
// device memory.
//
// Some callers cannot call cudaMalloc (or let this library call it for them):
// code running while a custom allocator owns all device memory, real-time
// loops that forbid allocation after start-up, or hosts where the CUDA
// memory pool is disabled.  This entry point does the same stable grouping as
// mita_bucket, but its per-chunk counters live in a fixed, file-scope device
// array instead of the library's workspace cache, so it never allocates.
//
// Limits and sharing rules:
//   * The array holds kNoAllocScratchInts int32 counters (4 MiB).  A call
//     needs B*H*(ceil(N*s/4096)+1)*m of them; larger calls are rejected with
//     MITA_ERR_UNSUPPORTED before anything runs.
//   * Every GPU that loads this library's module keeps the 4 MiB until the
//     process exits.
//   * All calls share the one array, and it keeps whatever the last call
//     left there.  Each call writes every counter it uses before reading it.  Calls
//     whose executions overlap on the GPU (different streams, no ordering
//     between them) race on the array and give wrong results: order them.
//   * The first call in a CUDA context (a device's primary context, or any
//     other context the caller makes current) looks up the array's device
//     address there (cudaGetSymbolAddress) and caches it under that context.
//     Make that first call before any stream capture begins; after a
//     cudaDeviceReset the device gets a new context, and the next call looks
//     the address up again (so it, too, should come before any capture).
//   * Route values outside [0, m) are skipped, as in mita_bucket, but are not
//     recorded in the status word read by mita_get_last_device_error (that
//     word needs a one-time allocation).
#include "mita.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>
#include <utility>
#include <vector>

#include "common.cuh"
#include "kernels.h"

namespace mita {
namespace {

constexpr size_t kNoAllocScratchInts = size_t(1) << 20;   // 4 MiB of int32

static __device__ __align__(256) int g_bucket_scratch[kNoAllocScratchInts];

// The array's address in each CUDA context the entry point has run in.  A
// module is loaded per context, so the address belongs to the context, not to
// the device ordinal.  The driver's cuCtxGetCurrent is looked up through the
// runtime (the library does not link libcuda directly).
std::mutex g_na_mu;
std::vector<std::pair<CUcontext, void*>> g_na_ptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
bool g_ctx_looked_up = false;

bool current_context(CUcontext* ctx) {
  if (!g_ctx_looked_up) {
    g_ctx_looked_up = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 4000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(fn);
    cudaGetLastError();
  }
  return g_ctx_current && g_ctx_current(ctx) == CUDA_SUCCESS && *ctx != nullptr;
}

}  // namespace
}  // namespace mita

extern "C" int mita_bucket_noalloc(const int32_t* route_idx, int B, int H, int N, int m, int s,
                                   int32_t* bucket_off, int32_t* bucket_qidx,
                                   mita_stream_t stream) {
  using namespace mita;
  if (B < 1 || H < 1 || N < 1 || m < 1 || m > N || s < 1 || s > m)
    return report_error(MITA_ERR_INVALID_ARG, "mita_bucket_noalloc: invalid B, H, N, m or s");
  if (s > kMaxRouteS || (long long)B * H * N * s >= (1LL << 31))
    return report_error(MITA_ERR_UNSUPPORTED, "mita_bucket_noalloc: s or B*H*N*s too large");
  if (!route_idx || !bucket_off || !bucket_qidx)
    return report_error(MITA_ERR_INVALID_ARG, "mita_bucket_noalloc: NULL argument");
  const size_t need = bucket_ws_bytes(B * H, N * s, m);
  if (need > kNoAllocScratchInts * sizeof(int))
    return report_error(MITA_ERR_UNSUPPORTED,
                        "mita_bucket_noalloc: B*H*(ceil(N*s/4096)+1)*m exceeds the 1048576 counters "
                        "(4 MiB) of its static scratch; use mita_bucket");

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return report_error(MITA_ERR_CUDA, "mita_bucket_noalloc: no current CUDA device");
  }
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lk(g_na_mu);
    // No context is current yet on a thread whose first runtime call this is;
    // cudaGetSymbolAddress then makes the device's primary context current.
    CUcontext ctx = nullptr;
    const bool had_ctx = current_context(&ctx);
    if (had_ctx)
      for (const auto& e : g_na_ptr)
        if (e.first == ctx) scratch = e.second;
    if (scratch == nullptr) {
      void* p = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&p, g_bucket_scratch);
      if (e != cudaSuccess || p == nullptr) {
        cudaGetLastError();
        return report_error(MITA_ERR_CUDA, "mita_bucket_noalloc: cudaGetSymbolAddress failed");
      }
      if (!had_ctx && !current_context(&ctx)) {
        cudaGetLastError();
        return report_error(MITA_ERR_CUDA, "mita_bucket_noalloc: no current CUDA context");
      }
      bool known = false;
      for (auto& c : g_na_ptr)
        if (c.first == ctx) { c.second = p; known = true; }
      if (!known) g_na_ptr.emplace_back(ctx, p);
      scratch = p;
    }
  }
  const cudaError_t e =
      launch_bucket(route_idx, B * H, N, m, scratch, bucket_off, bucket_qidx, nullptr, stream,
                    false, s);
  return e == cudaSuccess ? MITA_OK
                          : report_error(MITA_ERR_CUDA, "mita_bucket_noalloc: launch failed");
}
