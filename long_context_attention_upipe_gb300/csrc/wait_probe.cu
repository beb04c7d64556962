// A one-thread kernel around the bounded wait every warp-specialised kernel of the library uses:
// it waits on an mbarrier that nothing arrives at (or, as a control, one it has arrived at
// itself), so the wait's timeout path (give up after the limit, raise the error word, return)
// can be exercised on the GPU without breaking any real kernel.
#include "internal.h"
#include "tc_common.cuh"

namespace upipe {

namespace {

__global__ void k_wait_probe(TableHeader* h, int arrive, uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    h->error = 0;
    abort_flag = 0;
    tc::mbar_init(&bar, 1);
    tc::fence_mbar_init();
    if (arrive) tc::mbar_arrive(&bar);
    tc::mbar_wait(&bar, 0, &abort_flag, &h->error, limit_ns);  // on timeout: error word = DEVICE_TIMEOUT
  }
}

}  // namespace

cudaError_t launch_wait_probe(void* header, int arrive, cudaStream_t st) {
  k_wait_probe<<<1, 32, 0, st>>>(reinterpret_cast<TableHeader*>(header), arrive, wait_limit_ns());
  note_launch();
  return cudaGetLastError();
}

}  // namespace upipe
