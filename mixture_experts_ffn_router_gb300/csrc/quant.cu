// quant.cu — int8 (per-channel symmetric) and MXFP4 quantisation of expert weights on the device.
//
// "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 — where every rank weighted the
// wrong experts", section "Can it run on a smaller box?": the experts are stored as int8 with one
// scale per output channel (row) and symmetric range. The rule, fixed so that any implementation
// gives the same bits: scale = max |w| / 127 in fp32 (correctly rounded division), q = w / scale in
// fp32 (correctly rounded) rounded to nearest with ties to even, clamped to [-127, 127]; a row of
// zeros gets scale 0 and q 0. int8 values are exact in bf16, so the grouped GEMMs widen q to bf16
// and apply the scale to the fp32 accumulator.
#include <cuda_bf16.h>

#include "internal.h"
#include "moe_ffn.h"

namespace moe {

namespace {

constexpr int kQuantWarps = 8;

// One warp per row; each lane handles 8 consecutive columns at a time.
__global__ void __launch_bounds__(kQuantWarps * 32)
    quantize_int8_kernel(const uint16_t* w, long long rows, int cols, int8_t* q, float* scale) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const long long row = static_cast<long long>(blockIdx.x) * kQuantWarps + warp;
  if (row >= rows) return;
  const uint16_t* wr = w + row * cols;
  float amax = 0.0f;
  for (int c = lane * 8; c < cols; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(wr + c);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] << 16)));
      amax = fmaxf(amax, fabsf(__uint_as_float(w4[j] & 0xFFFF0000u)));
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const float s = __fdiv_rn(amax, 127.0f);
  if (lane == 0) scale[row] = s;
  int8_t* qr = q + row * cols;
  for (int c = lane * 8; c < cols; c += 256) {
    const uint4 v = *reinterpret_cast<const uint4*>(wr + c);
    const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
    uint32_t packed[2] = {0u, 0u};
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const float x = __uint_as_float(j & 1 ? (w4[j >> 1] & 0xFFFF0000u) : (w4[j >> 1] << 16));
      float r = 0.0f;
      if (s > 0.0f) r = fminf(fmaxf(rintf(__fdiv_rn(x, s)), -127.0f), 127.0f);
      packed[j >> 2] |= (static_cast<uint32_t>(static_cast<int>(r)) & 0xFFu) << (8 * (j & 3));
    }
    *reinterpret_cast<uint2*>(qr + c) = make_uint2(packed[0], packed[1]);
  }
}

}  // namespace

}  // namespace moe

extern "C" int moe_ffn_quantize_int8(const void* w, long long rows, int cols, int8_t* q, float* scale,
                                     void* stream) {
  if (!w || !q || !scale || rows < 0 || cols < 8 || cols % 8 != 0) return MOE_FFN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) != 0 || (reinterpret_cast<uintptr_t>(q) & 15u) != 0 ||
      (reinterpret_cast<uintptr_t>(scale) & 3u) != 0)
    return MOE_FFN_EALIGN;
  if (rows == 0) return MOE_FFN_OK;
  const long long blocks = (rows + moe::kQuantWarps - 1) / moe::kQuantWarps;
  if (blocks > 0x7FFFFFFFLL) return MOE_FFN_EINVAL;
  moe::quantize_int8_kernel<<<static_cast<unsigned>(blocks), moe::kQuantWarps * 32, 0,
                              static_cast<cudaStream_t>(stream)>>>(static_cast<const uint16_t*>(w), rows, cols, q,
                                                                   scale);
  return cudaGetLastError() == cudaSuccess ? MOE_FFN_OK : MOE_FFN_ECUDA;
}

namespace moe {

namespace {

constexpr int kF4Threads = 256;

// E2M1 magnitude code of a (the element over its block scale, a >= 0): the nearest of 0, 0.5, 1,
// 1.5, 2, 3, 4, 6 with midpoints going to the even code, magnitudes above 6 saturating to 6.
__device__ __forceinline__ uint32_t e2m1_magnitude_code(float a) {
  if (a <= 0.25f) return 0;
  if (a < 0.75f) return 1;
  if (a <= 1.25f) return 2;
  if (a < 1.75f) return 3;
  if (a <= 2.5f) return 4;
  if (a < 3.5f) return 5;
  if (a <= 5.0f) return 6;
  return 7;
}

// One thread per block of 32 elements: the block's largest magnitude gives the shared exponent
// floor(log2 amax) - 2 (ilogbf), every element is scaled by 2^-exponent (exact wherever the
// rounding decision depends on it) and rounded to E2M1.
__global__ void __launch_bounds__(kF4Threads)
    quantize_mxfp4_kernel(const uint16_t* w, long long rows, int cols, uint8_t* codes, uint8_t* scales) {
  const int nb = cols / 32;
  const long long blk = static_cast<long long>(blockIdx.x) * kF4Threads + threadIdx.x;
  if (blk >= rows * nb) return;
  const long long r = blk / nb;
  const int b = static_cast<int>(blk - r * nb);
  const uint16_t* src = w + r * cols + b * 32;
  float v[32];
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint4 q = *reinterpret_cast<const uint4*>(src + 8 * p);
    const uint32_t q4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      v[8 * p + 2 * j] = __uint_as_float(q4[j] << 16);
      v[8 * p + 2 * j + 1] = __uint_as_float(q4[j] & 0xFFFF0000u);
    }
  }
  float amax = 0.0f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(v[j]));
  uint32_t out[4] = {0u, 0u, 0u, 0u};
  uint8_t sbyte = 0;
  if (amax > 0.0f) {
    int se = ilogbf(amax) - 2;
    se = se < -127 ? -127 : (se > 127 ? 127 : se);
    sbyte = static_cast<uint8_t>(se + 127);
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float a = ldexpf(v[j], -se);
      uint32_t c = e2m1_magnitude_code(fabsf(a));
      if (c != 0 && a < 0.0f) c |= 8u;
      out[j >> 3] |= c << (4 * (j & 7));
    }
  }
  *reinterpret_cast<uint4*>(codes + r * (cols / 2) + b * 16) = make_uint4(out[0], out[1], out[2], out[3]);
  scales[r * nb + b] = sbyte;
}

}  // namespace

}  // namespace moe

extern "C" int moe_ffn_quantize_mxfp4(const void* w, long long rows, int cols, uint8_t* codes, uint8_t* scales,
                                      void* stream) {
  if (!w || !codes || !scales || rows < 0 || cols < 32 || cols % 32 != 0) return MOE_FFN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(w) & 15u) != 0 || (reinterpret_cast<uintptr_t>(codes) & 15u) != 0)
    return MOE_FFN_EALIGN;
  if (rows == 0) return MOE_FFN_OK;
  const long long nblk = rows * (cols / 32);
  const long long grid = (nblk + moe::kF4Threads - 1) / moe::kF4Threads;
  if (grid > 0x7FFFFFFFLL) return MOE_FFN_EINVAL;
  moe::quantize_mxfp4_kernel<<<static_cast<unsigned>(grid), moe::kF4Threads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint16_t*>(w), rows, cols, codes, scales);
  return cudaGetLastError() == cudaSuccess ? MOE_FFN_OK : MOE_FFN_ECUDA;
}
