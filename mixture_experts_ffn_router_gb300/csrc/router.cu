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
// Batches of more than kRouteSmallT tokens use these two kernels; smaller ones take the same sums in
// fp32 on CUDA cores inside the small-batch routing kernel (route.cu), with no fold kernel.
// MMA: M = 128 experts (A = a W' part, K-major, by TMA), N = 128 tokens (B = x rows, K-major,
// staged by the producer warp). Warp 0 loads, warp 1 issues the MMAs, the other warps add chunk
// sums: with 128-token tiles sixteen of them, four per TMEM lane quarter taking a quarter of the
// token columns each (router logits 10.4 vs 11.9 us at T = 256 and 18.2 vs 18.8 us at T = 4096
// against two per quarter); with 64-token tiles eight, two per quarter.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {


constexpr int kTile = 128 * 64 * 2;              // one 128-row x 64-element bf16 tile, 16 KB
constexpr int kStagesR = 3;
constexpr int kAccR = 4;                         // rotating chunk accumulators in TMEM

// N = tokens per CTA: kRouterN, or 64 for decode-sized batches (a narrower MMA and epilogue).
template <int N>
struct RCfg {
  static constexpr int kEpiWarps = N >= 128 ? 16 : 8;  // chunk-sum warps: four | two per TMEM lane quarter
  static constexpr int kThreads = (2 + kEpiWarps) * 32;
  static constexpr int kBTile = N * 64 * 2;      // x tile
  static constexpr int kStage = 3 * kTile + kBTile;  // hi, mid, lo, x
  static constexpr int kSmem = 1024 + kStagesR * kStage + 256;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(128, N);
  static_assert(kBTile % 1024 == 0, "x tile alignment");
  static_assert(kAccR * N <= 512, "TMEM columns");
};
constexpr int kRouterSmallN = 64;

__device__ __forceinline__ float bf16_round(float v) { return __bfloat162float(__float2bfloat16_rn(v)); }

// One CTA per expert row: W'[e] = W_r[e] * (1 + router_norm_w), split into bf16 hi, mid, lo.
// 352 threads, 8 consecutive elements each (two 16-byte loads, three 16-byte stores).
constexpr int kPrepThreads = H / 8;

__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16_rn(lo)) | (static_cast<uint32_t>(f32_to_bf16_rn(hi)) << 16);
}

__global__ void __launch_bounds__(kPrepThreads) router_prep_kernel(RouteParams p, Buffers b) {
  const int e = blockIdx.x;
  const int h0 = threadIdx.x * 8;
  pdl_wait();
  pdl_launch_dependents();
  const float4 w0 = *reinterpret_cast<const float4*>(p.router_w + static_cast<size_t>(e) * H + h0);
  const float4 w1 = *reinterpret_cast<const float4*>(p.router_w + static_cast<size_t>(e) * H + h0 + 4);
  const float4 g0 = *reinterpret_cast<const float4*>(p.router_norm_w + h0);
  const float4 g1 = *reinterpret_cast<const float4*>(p.router_norm_w + h0 + 4);
  const float wv[8] = {w0.x * (1.0f + g0.x), w0.y * (1.0f + g0.y), w0.z * (1.0f + g0.z), w0.w * (1.0f + g0.w),
                       w1.x * (1.0f + g1.x), w1.y * (1.0f + g1.y), w1.z * (1.0f + g1.z), w1.w * (1.0f + g1.w)};
  float hi[8], mid[8], lo[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) {
    hi[u] = bf16_round(wv[u]);
    const float r1 = wv[u] - hi[u];  // exact: hi is w rounded to 8 significant bits
    mid[u] = bf16_round(r1);
    lo[u] = r1 - mid[u];             // exact, and representable in bf16
  }
  uint4* dst = reinterpret_cast<uint4*>(b.wsplit + static_cast<size_t>(e) * H + h0);
  const size_t part = static_cast<size_t>(E) * H / 8;  // one part, in 16-byte units
  dst[0] = make_uint4(pack2(hi[0], hi[1]), pack2(hi[2], hi[3]), pack2(hi[4], hi[5]), pack2(hi[6], hi[7]));
  dst[part] = make_uint4(pack2(mid[0], mid[1]), pack2(mid[2], mid[3]), pack2(mid[4], mid[5]), pack2(mid[6], mid[7]));
  dst[2 * part] = make_uint4(pack2(lo[0], lo[1]), pack2(lo[2], lo[3]), pack2(lo[4], lo[5]), pack2(lo[6], lo[7]));
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 16-byte cp.async; bytes past src_bytes (0 or 16) are written as zeros.
__device__ __forceinline__ void cp_async16_zfill(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

template <int N>
__global__ void __launch_bounds__(RCfg<N>::kThreads, 1)
    router_tc_kernel(const __grid_constant__ CUtensorMap map_w, RouteParams p, Buffers b) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kStagesR * RCfg<N>::kStage);
  uint64_t* empty_bar = full_bar + kStagesR;
  uint64_t* accf_bar = empty_bar + kStagesR;
  uint64_t* acce_bar = accf_bar + kAccR;
  uint64_t* final_bar = acce_bar + kAccR;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * N;
  const int ks = blockIdx.y;
  const int cps = (H / 64) / p.ks;  // chunks per split
  const int c_begin = ks * cps;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStagesR; ++s) {
      mbar_init(&full_bar[s], 1 + 32);  // the TMA byte count + the producer lanes' x copies
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < kAccR; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], RCfg<N>::kEpiWarps);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&map_w);
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, kAccR * N);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  pdl_wait();
  pdl_launch_dependents();
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0) *b.done_ctr = 0;
  // The per-chunk expert counts that the top-k kernel accumulates start from zero.
  if (blockIdx.y == 0 && threadIdx.x >= 64 && threadIdx.x < 64 + E)
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
      uint8_t* st = smem + stage * RCfg<N>::kStage;
      const int k0 = (c_begin + ci) * 64;
      if (lane == 0) {
        armed |= 1u << stage;
        armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
        mbar_arrive_expect_tx(&full_bar[stage], 3 * kTile);
#pragma unroll
        for (int part = 0; part < 3; ++part) tma_load_2d(st + part * kTile, &map_w, &full_bar[stage], k0, part * E, pol);
      }
      // x rows t0..t0+N-1, 16-byte chunks copied asynchronously into the 128-byte-swizzled K-major
      // tile (rows past T are zero-filled); each lane's arrival fires when its copies have landed.
      const uint32_t xs = smem_u32(st + 3 * kTile);
#pragma unroll
      for (int i = 0; i < (N * 8) / 32; ++i) {
        const int idx = lane + 32 * i, r = idx >> 3, cc = idx & 7;
        const int t = t0 + r;
        const uint16_t* src = p.x + static_cast<size_t>(t < p.T ? t : 0) * H + k0 + cc * 8;
        cp_async16_zfill(xs + r * 128 + ((cc ^ (r & 7)) << 4), src, t < p.T ? 16u : 0u);
      }
      cp_async_arrive_noinc(&full_bar[stage]);
      if (++stage == kStagesR) {
        stage = 0;
        phase ^= 1u;
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    if (lane == 0)
      for (int s2 = 0; s2 < kStagesR; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&full_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs, b.status);
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
        const uint32_t sa = smem_u32(smem + stage * RCfg<N>::kStage);
        const uint64_t bdesc = smem_desc_sw128(sa + 3 * kTile);
        const uint32_t d = tmem_base + acc * N;
#pragma unroll
        for (int part = 0; part < 3; ++part) {
          const uint64_t adesc = smem_desc_sw128(sa + part * kTile);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            umma_bf16(d, adesc + 2u * k, bdesc + 2u * k, RCfg<N>::kIdesc, (part | k) != 0 ? 1u : 0u);
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
      mbar_wait_timeout(final_bar, 0, kSpinLimitNs, b.status);
    }
    __syncwarp();
  } else {
    // ---------------- warps 2..: add the chunk sums (TMEM lane = expert) in fp32. The warps of a
    // lane quarter share its N token columns, each with all its TMEM loads of a chunk in flight
    // before one wait (one dependent wait per chunk instead of one per 32 columns).
    const int q = warp & 3;
    const int hf = (warp - 2) >> 2;
    constexpr int NH = N / (RCfg<N>::kEpiWarps / 4);
    float z[NH];
#pragma unroll
    for (int j = 0; j < NH; ++j) z[j] = 0.0f;
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
      uint32_t r[NH / 32][32];
#pragma unroll
      for (int g = 0; g < NH / 32; ++g)
        tmem_ld32_nowait(tmem_base + (static_cast<uint32_t>(q * 32) << 16) + acc * N + hf * NH + g * 32, r[g]);
      tmem_wait_ld();
#pragma unroll
      for (int g = 0; g < NH / 32; ++g) {
        reg_fence32(r[g]);
#pragma unroll
        for (int j = 0; j < 32; ++j) z[g * 32 + j] += __uint_as_float(r[g][j]);
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
      for (int j = 0; j < NH; ++j) {
        const int t = t0 + hf * NH + j;
        if (t < p.T) b.logits_part[(static_cast<size_t>(ks) * p.T + t) * E + e] = z[j];
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kAccR * N);
  }
}

}  // namespace

cudaError_t router_set_smem_limit() {
  const cudaError_t e = cudaFuncSetAttribute(router_tc_kernel<kRouterN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             RCfg<kRouterN>::kSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(router_tc_kernel<kRouterSmallN>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              RCfg<kRouterSmallN>::kSmem);
}

cudaError_t launch_router_prep(const RouteParams& p, const Buffers& b, cudaStream_t s) {
  return launch_pdl(router_prep_kernel, dim3(E), dim3(kPrepThreads), 0, s, p, b);
}

cudaError_t launch_router_logits(const CUtensorMap& map_w, const RouteParams& p, const Buffers& b, cudaStream_t s) {
  if (p.T <= kRouterSmallN)
    return launch_pdl(router_tc_kernel<kRouterSmallN>, dim3(1, p.ks), dim3(RCfg<kRouterSmallN>::kThreads),
                      static_cast<size_t>(RCfg<kRouterSmallN>::kSmem), s, map_w, p, b);
  dim3 grid((p.T + kRouterN - 1) / kRouterN, p.ks);
  return launch_pdl(router_tc_kernel<kRouterN>, grid, dim3(RCfg<kRouterN>::kThreads), static_cast<size_t>(RCfg<kRouterN>::kSmem), s,
                    map_w, p, b);
}

}  // namespace moe
