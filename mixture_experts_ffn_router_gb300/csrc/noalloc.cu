// noalloc.cu — the router logits of the block through an entry point that allocates nothing.
//
// Some callers cannot allocate device memory when they call in: code running under a CUDA memory
// pool or allocator they do not own, plugins given only a stream and a few buffers, real-time
// paths where an allocation (and the synchronisation cudaMalloc can imply) is not allowed. Those
// callers cannot provide the workspace that moe_ffn_init needs. This file gives them one entry
// point, moe_ffn_router_logits_noalloc, whose scratch lives in a fixed array in device memory
// that the library reserves at load time.
//
// The scratch: g_router_scratch below, kNoAllocScratchBytes (about 2.6 MB) of device memory on
// every GPU the process uses with this library, held until the process exits. It holds the split
// router matrix (3 x 128 x 2816 bf16), the partial logits of up to kNoAllocMaxTokens tokens and a
// few control words. The array keeps what the last call left there. Each call first clears its
// status word (an asynchronous memset on the caller's stream, which allocates nothing); every
// other byte a call reads there is written earlier by the same call. All calls share the one
// array, so two calls whose GPU work overlaps in time (different streams, or different host
// threads) corrupt each other's results.
//
// Failure: the tensor-core router's waits are bounded; one that gives up sets the status word and
// the kernel writes no partial sums. The finishing kernel reads the word and then writes NaN to
// every logit of the call instead of logits made from stale partial sums, so a failed call can
// never pass for a good one.
#include <cuda_runtime.h>

#include <mutex>

#include "internal.h"
#include "moe_ffn.h"
#include "ptx.cuh"

namespace moe {
// Defined in moe_ffn.cu.
bool encode_bf16_tensor_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows);
}  // namespace moe

using namespace moe;

namespace {

constexpr int kNoAllocMaxTokens = 1024;
constexpr size_t kWsplitBytes = static_cast<size_t>(3) * E * H * 2;
constexpr size_t kPartBytes = static_cast<size_t>(kNoAllocMaxTokens) * E * 4;
constexpr size_t kHistBytes = static_cast<size_t>((kNoAllocMaxTokens + kScatterTok - 1) / kScatterTok) * E * 4;
constexpr size_t kCtrlBytes = 256;  // done counter and status word
constexpr size_t kNoAllocScratchBytes = kWsplitBytes + kPartBytes + kHistBytes + kCtrlBytes;

static __device__ __align__(256) uint8_t g_router_scratch[kNoAllocScratchBytes];

struct DeviceSetup {
  bool ready;
  uint8_t* scratch;       // device address of g_router_scratch on this device
  CUtensorMap map_wsplit; // TMA map of the split matrix inside the scratch
};

constexpr int kMaxDevices = 64;
DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// One warp per token: logits = partial sum * (1 / rms(x)) * router_scale, with the RMS taken as
// in the top-k kernel (fp32, eps inside the square root).
// If the status word is set (a bounded wait of the router gave up), every logit is NaN.
__global__ void __launch_bounds__(256) finish_logits_kernel(const uint16_t* x, const float* part, int T,
                                                            float eps, float scale, const unsigned int* status,
                                                            float* logits) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + warp;
  pdl_wait();
  if (t >= T) return;
  if (*reinterpret_cast<const volatile unsigned int*>(status) != 0u) {
#pragma unroll
    for (int j = 0; j < 4; ++j) logits[static_cast<size_t>(t) * E + lane + 32 * j] = __int_as_float(0x7fc00000);
    return;
  }
  const uint4* xr = reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * H);
  float ss = 0.0f;
#pragma unroll
  for (int c = 0; c < 11; ++c) {
    const uint4 v = xr[lane + 32 * c];
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = __uint_as_float(w4[j] << 16), b = __uint_as_float(w4[j] & 0xFFFF0000u);
      ss = fmaf(a, a, ss);
      ss = fmaf(b, b, ss);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
  const float inv = 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int e = lane + 32 * j;
    logits[static_cast<size_t>(t) * E + e] = part[static_cast<size_t>(t) * E + e] * inv * scale;
  }
}

// First use on the current device: look up the scratch array's device address and build the TMA
// map over it. Returns a status code.
int setup_current_device(DeviceSetup** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_FFN_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return MOE_FFN_EINVAL;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  DeviceSetup& s = g_setup[dev];
  if (!s.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return MOE_FFN_ECUDA;
    if (major != 10 || minor != 3) return MOE_FFN_EARCH;
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_router_scratch) != cudaSuccess || ptr == nullptr) return MOE_FFN_ECUDA;
    if (router_set_smem_limit() != cudaSuccess) return MOE_FFN_ECUDA;
    s.scratch = static_cast<uint8_t*>(ptr);
    if (!encode_bf16_tensor_map(&s.map_wsplit, s.scratch, 3 * E, H, 128)) return MOE_FFN_ECUDA;
    s.ready = true;
  }
  *out = &s;
  return MOE_FFN_OK;
}

}  // namespace

extern "C" int moe_ffn_router_logits_noalloc(const void* x, int T, const float* router_w,
                                             const float* router_norm_w, float router_scale, float eps,
                                             float* logits, void* stream) {
  if (T < 0 || !(eps > 0.0f) || !(router_scale > 0.0f)) return MOE_FFN_EINVAL;
  if (T > kNoAllocMaxTokens) return MOE_FFN_ETOOBIG;
  if (T == 0) return MOE_FFN_OK;
  if (!x || !router_w || !router_norm_w || !logits) return MOE_FFN_EINVAL;
  const void* ptrs[] = {x, router_w, router_norm_w, logits};
  for (const void* p : ptrs)
    if ((reinterpret_cast<uintptr_t>(p) & 15u) != 0) return MOE_FFN_EALIGN;
  DeviceSetup* dev = nullptr;
  const int rc = setup_current_device(&dev);
  if (rc != MOE_FFN_OK) return rc;

  uint8_t* sc = dev->scratch;
  Buffers b = {};
  b.wsplit = reinterpret_cast<uint16_t*>(sc);
  b.logits_part = reinterpret_cast<float*>(sc + kWsplitBytes);
  b.hist = reinterpret_cast<int32_t*>(sc + kWsplitBytes + kPartBytes);
  b.done_ctr = reinterpret_cast<int32_t*>(sc + kWsplitBytes + kPartBytes + kHistBytes);
  b.status = reinterpret_cast<unsigned int*>(sc + kWsplitBytes + kPartBytes + kHistBytes + 16);

  RouteParams p = {};
  p.x = static_cast<const uint16_t*>(x);
  p.router_w = router_w;
  p.router_norm_w = router_norm_w;
  p.T = T;
  p.ks = 1;  // one split: the partial buffer holds exactly T x 128 sums
  p.eps = eps;
  p.router_scale = router_scale;

  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // The status word starts every call at zero (the array keeps the last call's contents).
  if (cudaMemsetAsync(b.status, 0, sizeof(unsigned int), s) != cudaSuccess) return MOE_FFN_ECUDA;
  if (launch_router_prep(p, b, s) != cudaSuccess) return MOE_FFN_ECUDA;
  if (launch_router_logits(dev->map_wsplit, p, b, s) != cudaSuccess) return MOE_FFN_ECUDA;
  if (launch_pdl(finish_logits_kernel, dim3((T + 7) / 8), dim3(256), 0, s, p.x,
                 static_cast<const float*>(b.logits_part), T, eps, router_scale,
                 static_cast<const unsigned int*>(b.status), logits) != cudaSuccess)
    return MOE_FFN_ECUDA;
  return MOE_FFN_OK;
}
