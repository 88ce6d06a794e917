// selftest.cu — a device check of the bounded waits that every pipeline of the library relies on.
//
// Each kernel of the library waits on mbarriers through mbar_wait_bounded (ptx.cuh): after
// kSpinLimitNs (2 s) without the phase completing it gives up, sets its reason bit in the status
// word, raises the CTA's abort flag and returns false, and every other waiting role of the CTA
// then leaves at its next check of that flag. Exit drains use mbar_wait_timeout with a shorter
// limit. In the forward these paths run only when something has already gone wrong, so a normal
// run never exercises them. This kernel makes them run out on purpose, on a barrier that nothing
// arrives on (no fault, no trap: the waits themselves end), so that a test can check that the GPU
// comes back with the right status bits and stays usable.
#include <cuda_runtime.h>

#include "internal.h"
#include "moe_ffn.h"
#include "ptx.cuh"

using namespace moe;

namespace {

constexpr unsigned long long kDrainLimitNs = 1000000ull;  // 1 ms

// One CTA of one warp; lane 0 does all the waiting, in order:
//   1. mbar_wait_bounded on a barrier with no arrivals: gives up after kSpinLimitNs with
//      kStatusWaitFull set and the abort flag raised;
//   2. mbar_wait_bounded again, now with the flag raised: leaves through the flag without setting
//      its own bit (kStatusWaitEmpty);
//   3. mbar_wait_timeout with a 1 ms limit: gives up with kStatusDrain set.
// rec[2i] = nanoseconds wait i took, rec[2i + 1] = what it returned (1 = phase completed).
__global__ void __launch_bounds__(32) wait_expiry_kernel(unsigned int* status, unsigned long long* rec) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  fence_barrier_init();
  abort_flag = 0;
  volatile int* abort = &abort_flag;

  unsigned long long t0 = global_ns();
  bool ok = mbar_wait_bounded(&bar, 0, abort, status, kStatusWaitFull);
  rec[0] = global_ns() - t0;
  rec[1] = ok ? 1ull : 0ull;

  t0 = global_ns();
  ok = mbar_wait_bounded(&bar, 0, abort, status, kStatusWaitEmpty);
  rec[2] = global_ns() - t0;
  rec[3] = ok ? 1ull : 0ull;

  t0 = global_ns();
  ok = mbar_wait_timeout(&bar, 0, kDrainLimitNs, status);
  rec[4] = global_ns() - t0;
  rec[5] = ok ? 1ull : 0ull;
}

}  // namespace

extern "C" int moe_ffn_selftest_wait_expiry(uint32_t* status_word, unsigned long long* record, void* stream) {
  if (!status_word || !record) return MOE_FFN_EINVAL;
  int device = 0, major = 0, minor = 0;
  if (cudaGetDevice(&device) != cudaSuccess ||
      cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess)
    return MOE_FFN_ECUDA;
  if (major != 10 || minor != 3) return MOE_FFN_EARCH;
  wait_expiry_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(reinterpret_cast<unsigned int*>(status_word), record);
  return cudaGetLastError() == cudaSuccess ? MOE_FFN_OK : MOE_FFN_ECUDA;
}
