// Failure-detection self-test: a one-CTA kernel waits on an mbarrier that
// nothing arrives on, with the same bounded-wait rule as the decode kernel
// (give up after a number of SM clocks, record kErrWaitTimeout in the pool's
// device error word, return).  The host then reads the word through
// mkv_check_device_errors, which reports MKV_ERR_DEVICE_CHECK and clears it;
// the context stays usable.  Nothing here faults, traps or spins unbounded.
#include <cuda_runtime.h>

#include <cstdint>

#include "mkv_internal.h"

namespace mkv {
namespace {

__global__ void __launch_bounds__(32) mkv_wait_probe_kernel(int* err, long long limit_cycles) {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t addr = static_cast<uint32_t>(__cvta_generic_to_shared(&bar));
  if (threadIdx.x == 0) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(addr) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncwarp();
  if (threadIdx.x != 0) return;
  // phase 0 never completes: no thread arrives and no copy is counted on it
  const long long t0 = clock64();
  for (;;) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], 0;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(addr)
        : "memory");
    if (done) return;
    if (clock64() - t0 > limit_cycles) {
      atomicOr(err, kErrWaitTimeout);
      return;
    }
  }
}

}  // namespace

cudaError_t launch_wait_probe(int* err, long long limit_cycles, cudaStream_t s) {
  mkv_wait_probe_kernel<<<1, 32, 0, s>>>(err, limit_cycles);
  return cudaGetLastError();
}

}  // namespace mkv
