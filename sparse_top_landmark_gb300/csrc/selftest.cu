// mita_check_bounded_wait: makes the kernels' bounded waits run out, on purpose
// and safely, so a test can see the failure path work.
//
// Every wait inside this library's kernels (on an mbarrier completed by a TMA
// copy, an MMA or another warp) gives up after about 2^31 SM cycles (~1 s),
// sets the timeout bit of the device status word and lets the kernel return,
// so a lost arrival can never hang the GPU.  The probe kernel below waits, with
// the same two helpers the kernels use (the whole-warp wait of the MMA issuers
// and the single-thread wait of the softmax threads), on an mbarrier that
// nothing ever arrives on.  Both waits must give up and flag the timeout; the
// context stays usable.
#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace mita {
namespace {
using namespace sm100;

__global__ void __launch_bounds__(64) bounded_wait_probe_kernel(int* status, int* result) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // one arrival would complete phase 0; none ever comes
    fence_mbar_init();
  }
  __syncthreads();
  const int warp = threadIdx.x >> 5;
  bool done = true;
  if (warp == 0) done = mbar_wait_warp(&bar, 0);
  else if (threadIdx.x == 32) done = mbar_wait(&bar, 0);
  if (!done) flag_error(status, kDevErrTimeout);
  if ((threadIdx.x & 31) == 0) result[warp] = done ? 0 : 1;
}

}  // namespace
}  // namespace mita

namespace mita {
cudaError_t launch_bounded_wait_probe(int* status, int* gave_up, cudaStream_t st) {
  bounded_wait_probe_kernel<<<1, 64, 0, st>>>(status, gave_up);
  count_launch();
  return cudaGetLastError();
}
}  // namespace mita
