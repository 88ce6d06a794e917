// router.cu — the router projection on the tensor cores, at fp32 accuracy.
//
// "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 — where every rank weighted the
// wrong experts", section "The architecture": the router normalises its input with its own
// RMSNorm, scales it and projects it to one logit per expert before an fp32 softmax and the top-8
// choice. The choice must be taken on fp32-accurate logits, so the projection cannot simply run
// in bf16. Two kernels compute, for a tile of tokens and a slice of the hidden dimension,
//
//     part[t][e] = sum_h x[t,h] * W'[e,h],   W'[e,h] = W_r[e,h] * (1 + router_norm_w[h])
//
// (the RMS factor and the scalar scale are applied after the split sum, in the top-k kernel):
//   * router_prep_kernel forms W' in fp32 and splits it into three bf16 matrices hi + mid + lo
//     that add back to W' exactly (each residual has at most 8 significant bits left);
//   * router_tc_kernel multiplies: x is bf16, so every bf16 x bf16 product is exact in fp32; each
//     64-wide chunk of h is summed on the tensor cores (3 parts x 64 products) into its own TMEM
//     accumulator, and the chunk sums are added in fp32 registers, so the tensor core's own
//     accumulation spans only the 192 products of one chunk.
// MMA: M = 128 experts (A = a W' part, K-major, by TMA), N = 64 tokens (B = x rows, K-major,
// staged by the producer warp). Warp 0 loads, warp 1 issues the MMAs, warps 2..5 add chunk sums.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kThreadsR = 192;
constexpr int kTile = 128 * 64 * 2;              // one 128-row x 64-element bf16 tile, 16 KB
constexpr int kBTile = kRouterN * 64 * 2;        // x tile, 8 KB
constexpr int kStageR = 3 * kTile + kBTile;      // hi, mid, lo, x
constexpr int kStagesR = 3;
constexpr int kAccR = 4;                         // rotating chunk accumulators in TMEM
constexpr int kSmemR = 1024 + kStagesR * kStageR + 256;
constexpr uint32_t kIdescR = idesc_bf16_f32(128, kRouterN);
static_assert(kBTile % 1024 == 0, "x tile alignment");

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// One CTA per expert row: W'[e] = W_r[e] * (1 + router_norm_w), split into bf16 hi, mid, lo.
__global__ void __launch_bounds__(256) router_prep_kernel(RouteParams p, Buffers b) {
  const int e = blockIdx.x;
  pdl_wait();
  for (int h = threadIdx.x; h < H; h += 256) {
    const float w = p.router_w[static_cast<size_t>(e) * H + h] * (1.0f + p.router_norm_w[h]);
    const float hi = bf16_round(w);
    const float r1 = w - hi;  // exact: hi is w rounded to 8 significant bits
    const float mid = bf16_round(r1);
    const float lo = r1 - mid;  // exact, and representable in bf16
    b.wsplit[(0 * E + e) * static_cast<size_t>(H) + h] = f32_to_bf16_rn(hi);
    b.wsplit[(1 * E + e) * static_cast<size_t>(H) + h] = f32_to_bf16_rn(mid);
    b.wsplit[(2 * E + e) * static_cast<size_t>(H) + h] = f32_to_bf16_rn(lo);
  }
  pdl_launch_dependents();
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__global__ void __launch_bounds__(kThreadsR, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap map_w, RouteParams p, Buffers b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStagesR * kStageR);
  uint64_t* empty_bar = full_bar + kStagesR;
  uint64_t* accf_bar = empty_bar + kStagesR;
  uint64_t* acce_bar = accf_bar + kAccR;
  uint64_t* final_bar = acce_bar + kAccR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kRouterN;
  const int ks = blockIdx.y;
  const int cps = (H / 64) / p.ks;  // chunks per split
  const int c_begin = ks * cps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesR; ++s) {
      mbar_init(&full_bar[s], 2);  // the TMA byte count + the x stores
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < kAccR; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], 4);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kAccR * kRouterN);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *b.done_ctr = 0;
  // The per-chunk expert counts that the top-k kernel accumulates start from zero.
  if (blockIdx.y == 0 && threadIdx.x >= 64)
    for (int c = blockIdx.x; c < (p.T + kScatterTok - 1) / kScatterTok; c += gridDim.x)
      b.hist[c * E + threadIdx.x - 64] = 0;

  if (warp == 0) {
    // ---------------- producer: TMA for the three W' parts, plain loads for the x rows
    const uint64_t pol = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;
    for (int ci = 0; ci < cps; ++ci) {
      int got = 1;
      if (lane == 0) got = mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, b.status, kStatusWaitEmpty);
      if (!__shfl_sync(0xffffffffu, got, 0)) break;
      uint8_t* st = smem + stage * kStageR;
      const int k0 = (c_begin + ci) * 64;
      if (lane == 0) {
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        mbar_arrive_expect_tx(&full_bar[stage], 3 * kTile);
#pragma unroll
        for (int part = 0; part < 3; ++part) tma_load_2d(st + part * kTile, &map_w, &full_bar[stage], k0, part * E, pol);
      }
      // x rows t0..t0+63, 16-byte chunks into the 128-byte-swizzled K-major tile; rows past T are 0.
#pragma unroll
      for (int i = 0; i < (kRouterN * 8) / 32; ++i) {
        const int idx = lane + 32 * i, r = idx >> 3, cc = idx & 7;
        const int t = t0 + r;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (t < p.T) v = __ldg(reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H + k0 + cc * 8));
        *reinterpret_cast<uint4*>(st + 3 * kTile + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(&full_bar[stage]);
      if (++stage == kStagesR) {
        stage = 0;
        phase ^= 1u;
      }
    }
    if (lane == 0)
      for (int s2 = 0; s2 < kStagesR; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&full_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer: one accumulator per chunk, rotating through kAccR buffers
    if (lane == 0) {
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      for (int ci = 0; ci < cps; ++ci) {
        if (!mbar_wait_bounded(&acce_bar[acc], acc_phase ^ 1u, abort_flag, b.status, kStatusWaitAccEmpty)) break;
        if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, b.status, kStatusWaitFull)) break;
        fence_proxy_async_smem();
        tc_fence_after();
        const uint32_t sa = smem_u32(smem + stage * kStageR);
        const uint64_t bdesc = smem_desc_sw128(sa + 3 * kTile);
        const uint32_t d = tmem_base + acc * kRouterN;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint64_t adesc = smem_desc_sw128(sa + part * kTile);
#pragma unroll
          for (int k = 0; k < 4; ++k) umma_bf16(d, adesc + 2u * k, bdesc + 2u * k, kIdescR, (part | k) != 0 ? 1u : 0u);
        }
        umma_commit(&empty_bar[stage]);
        umma_commit(&accf_bar[acc]);
        if (++stage == kStagesR) {
          stage = 0;
          phase ^= 1u;
        }
        if (++acc == kAccR) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      umma_commit(final_bar);
      mbar_wait_timeout(final_bar, 0, kSpinLimitNs);
    }
    __syncwarp();
  } else {
    // ---------------- warps 2..5: add the chunk sums (TMEM lane = expert) in fp32
    const int q = warp & 3;
    float z[kRouterN];
#pragma unroll
    for (int j = 0; j < kRouterN; ++j) z[j] = 0.0f;
    int acc = 0;
    uint32_t acc_phase = 0;
    bool ok = true;
    for (int ci = 0; ci < cps; ++ci) {
      int got = 1;
      if (lane == 0) got = mbar_wait_bounded(&accf_bar[acc], acc_phase, abort_flag, b.status, kStatusWaitAccFull);
      if (!__shfl_sync(0xffffffffu, got, 0)) {
        ok = false;
        break;
      }
      tc_fence_after();
#pragma unroll
      for (int g = 0; g < kRouterN / 32; ++g) {
        float v[32];
        tmem_ld32(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * kRouterN + g * 32, v);
#pragma unroll
        for (int j = 0; j < 32; ++j) z[g * 32 + j] += v[j];
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[acc]);
      if (++acc == kAccR) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
    if (ok) {
      const int e = q * 32 + lane;
#pragma unroll
      for (int j = 0; j < kRouterN; ++j) {
        const int t = t0 + j;
        if (t < p.T) b.logits_part[(static_cast<size_t>(ks) * p.T + t) * E + e] = z[j];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kAccR * kRouterN);
  }
}

}  // namespace

cudaError_t router_set_smem_limit() {
  return cudaFuncSetAttribute(router_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemR);
}

cudaError_t launch_router_prep(const RouteParams& p, const Buffers& b, cudaStream_t s) {
  return launch_pdl(router_prep_kernel, dim3(E), dim3(256), 0, s, p, b);
}

cudaError_t launch_router_logits(const CUtensorMap& map_w, const RouteParams& p, const Buffers& b, cudaStream_t s) {
  dim3 grid((p.T + kRouterN - 1) / kRouterN, p.ks);
  return launch_pdl(router_tc_kernel, grid, dim3(kThreadsR), static_cast<size_t>(kSmemR), s, map_w, p, b);
}

}  // namespace moe
