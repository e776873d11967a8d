// Library-wide C entry points that are not tied to one kernel, and the
// self-test of the bounded wait that every kernel of the library uses.
#include "kvp_common.cuh"

extern "C" const char* kvp_status_string(int status) {
  switch (status) {
    case KVP_OK: return "ok";
    case KVP_ERR_INVALID: return "invalid argument";
    case KVP_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
    case KVP_ERR_CAPACITY: return "page pool, page table or reserve too small";
    case KVP_ERR_CUDA: return "CUDA runtime or launch error";
    case KVP_ERR_TIMEOUT: return "device-side wait gave up";
    case KVP_ERR_UNSUPPORTED: return "unsupported shape";
    case KVP_ERR_WORKSPACE: return "workspace missing or too small";
    case KVP_ERR_BOUNDS: return "page id or count out of range";
    default: return "unknown status";
  }
}

extern "C" int kvp_version(void) { return 100; }

namespace kvp {
namespace {

// One warp waits, with the library's mbar_wait, on an mbarrier that nothing
// arrives on: the wait gives up after limit_ns, the kernel records
// KVP_ERR_TIMEOUT and returns. No copy or tensor-core operation is in flight.
__global__ void __launch_bounds__(32) selftest_wait_kernel(uint64_t limit_ns, int32_t* status,
                                                            uint32_t* waited_us) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
  }
  __syncwarp();
  const uint64_t t0 = globaltimer_ns();
  const bool ok = mbar_wait(&bar, 0, nullptr, nullptr, limit_ns);
  const uint64_t t1 = globaltimer_ns();
  if (threadIdx.x == 0) {
    if (!ok) record_error(status, KVP_ERR_TIMEOUT);
    if (waited_us != nullptr) *waited_us = static_cast<uint32_t>((t1 - t0) / 1000);
  }
}

}  // namespace
}  // namespace kvp

extern "C" kvp_status kvp_selftest_wait(uint64_t limit_ns, int32_t* status, uint32_t* waited_us, void* stream) {
  if (status == nullptr || limit_ns > 10000000000ull) return KVP_ERR_INVALID;
  kvp::selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(limit_ns, status, waited_us);
  return cudaGetLastError() == cudaSuccess ? KVP_OK : KVP_ERR_CUDA;
}
