// gemm.cu — the two grouped GEMMs of the block on the 5th-generation tensor cores (tcgen05).
//
// "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 — where every rank weighted the
// wrong experts", section "The architecture": each expert holds a fused gate_up projection
// [128, 1408, 2816] (rows 0..703 gate, 704..1407 up) and a down projection [128, 2816, 704]; a
// token's 8 experts each compute down(gelu_tanh(gate x) * up x), and the shared MLP (width 2112)
// computes the same on every token. Instead of the pages' dense "compute all 128 experts and
// mask" form, the slots are sorted by expert and each expert multiplies only its own tokens.
//
// Layout ("swap AB"): the weight rows are the MMA's M side (128 rows per tile) and the tokens its
// N side (BN per tile), so a decode step with a handful of tokens per expert still streams every
// weight tile exactly once at full tile height. Work items are (token tile, 128-row weight tile)
// pairs; the token tiles of the experts come from a device-side list built by the top-k kernel,
// the shared MLP is one more group over all T tokens. Each CTA is persistent and takes every
// gridDim-th item, so the result does not depend on timing: every output element is written by
// exactly one CTA, with a fixed K order.
//
// Warp roles (192 threads): warp 0 loads A (weights, 2-D TMA boxes) and B (token rows, TMA
// gather4 by row index) into a ring of shared-memory stages; warp 1 issues tcgen05.mma into one of
// two TMEM accumulators; warps 2..5 drain the other accumulator (tcgen05.ld) and run the epilogue.
//
// gate_up epilogue: the A tile holds, per 32-row TMEM quarter, 16 gate rows then the 16 up rows of
// the same features, so one warp sees gate and up of a feature in lanes l and l+16 and forms
// h = gelu_tanh(gate) * up with one shuffle; h is stored bf16 in sorted-slot order.
// down epilogue: y[slot] = w_slot * acc (fp32, sorted-slot order); the shared MLP writes d.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                 // bf16 elements per 128-byte swizzled row
constexpr int kABytes = kBM * kBK * 2;  // 16 KB
constexpr int kThreads = 192;
constexpr int kSmemBudget = 196608;

template <int BN, bool GATE_UP>
struct Cfg {
  static constexpr int kBBytes = BN * kBK * 2;
  static constexpr int kStageBytes = kABytes + kBBytes;
  static constexpr int kStagesRaw = kSmemBudget / kStageBytes;
  static constexpr int kStages = kStagesRaw > 10 ? 10 : kStagesRaw;
  static constexpr int kTmemCols = 2 * BN < 32 ? 32 : 2 * BN;
  static constexpr int kMtExp = GATE_UP ? I / 64 : H / kBM;       // 11 | 22 weight tiles per expert
  static constexpr int kMtDense = GATE_UP ? D / 64 : H / kBM;     // 33 | 22
  static constexpr int kKbExp = GATE_UP ? H / kBK : I / kBK;      // 44 | 11
  static constexpr int kKbDense = GATE_UP ? H / kBK : D / kBK;    // 44 | 33
  static constexpr int kBarBytes = 256;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kBarBytes + BN * 4;
  static constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, BN);
  static_assert(kStageBytes % 1024 == 0, "stage buffers must stay 1024-byte aligned");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
};

struct Item {
  int dense;
  int e;
  int row0;
  int rows;
  int m;
};

// Items: the shared-MLP group first (its items are the longest for the down GEMM), then the
// experts' token tiles, each followed by its weight tiles in order.
template <int BN, bool GATE_UP>
__device__ __forceinline__ Item decode_item(int i, int n_dense_items, const int4* tiles, int T) {
  using C = Cfg<BN, GATE_UP>;
  Item it;
  if (i < n_dense_items) {
    const int j = i / C::kMtDense;
    it.dense = 1;
    it.e = E;
    it.m = i - j * C::kMtDense;
    it.row0 = j * BN;
    it.rows = min(BN, T - j * BN);
  } else {
    const int i2 = i - n_dense_items;
    const int j = i2 / C::kMtExp;
    const int4 tt = tiles[j];
    it.dense = 0;
    it.e = tt.x;
    it.row0 = tt.y;
    it.rows = tt.z;
    it.m = i2 - j * C::kMtExp;
  }
  return it;
}

template <int BN, bool GATE_UP>
__global__ void __launch_bounds__(kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a_exp, const __grid_constant__ CUtensorMap map_a_d0,
                        const __grid_constant__ CUtensorMap map_a_d1, const __grid_constant__ CUtensorMap map_b_exp,
                        const __grid_constant__ CUtensorMap map_b_dense, Buffers b, int T, int full_layer) {
  using C = Cfg<BN, GATE_UP>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + C::kStages * C::kStageBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* accf_bar = empty_bar + C::kStages;  // [2] accumulator ready
  uint64_t* acce_bar = accf_bar + 2;            // [2] accumulator drained
  uint64_t* final_bar = acce_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* idx_s = reinterpret_cast<int*>(smem + C::kStages * C::kStageBytes + C::kBarBytes);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], 4);
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&map_a_exp);
    prefetch_tmap(&map_b_exp);
    if (full_layer) {
      prefetch_tmap(&map_a_d0);
      if (GATE_UP) prefetch_tmap(&map_a_d1);
      prefetch_tmap(&map_b_dense);
    }
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Everything below reads what earlier kernels of the forward wrote.
  pdl_wait();
  const int n_tiles = *reinterpret_cast<volatile int*>(b.n_exp_tiles);
  const int n_dense_tiles = full_layer ? (T + BN - 1) / BN : 0;
  const int n_dense_items = n_dense_tiles * C::kMtDense;
  const int total = n_dense_items + n_tiles * C::kMtExp;

  if (warp == 0) {
    // ---------------- producer: TMA loads into the stage ring
    const uint64_t pol_w = policy_evict_first();
    const uint64_t pol_x = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;  // stages this warp armed, and the parity of the last arm
    bool ok = true;
    for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
      const Item it = decode_item<BN, GATE_UP>(i, n_dense_items, b.exp_tiles, T);
      // Source rows of the B operand for the token columns of this tile.
      for (int j = lane; j < BN; j += 32) {
        const int jj = min(j, it.rows - 1);
        int r;
        if (GATE_UP)
          r = it.dense ? it.row0 + jj : b.perm[it.row0 + jj];
        else
          r = it.row0 + jj;
        const int lim = GATE_UP ? T : (it.dense ? T : T * K);
        if (r < 0 || r >= lim) {
          atomicOr(b.status, kStatusBadIndex);
          r = 0;
        }
        idx_s[j] = r;
      }
      __syncwarp();
      const int n_g4 = (it.rows + 3) >> 2;  // only the valid rows are loaded
      const uint32_t tx_bytes = kABytes + n_g4 * 512;
      const int nkb = it.dense ? C::kKbDense : C::kKbExp;
      for (int kb = 0; kb < nkb; ++kb) {
        int got = 1;
        if (lane == 0) got = mbar_wait_bounded(&empty_bar[stage], phase ^ 1u, abort_flag, b.status, kStatusWaitEmpty);
        got = __shfl_sync(0xffffffffu, got, 0);
        if (!got) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* a_dst = stages + stage * C::kStageBytes;
          uint8_t* b_dst = a_dst + kABytes;
          armed |= 1u << stage;
          armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
          mbar_arrive_expect_tx(&full_bar[stage], tx_bytes);
          const int k0 = kb * kBK;
          if (GATE_UP) {
            const CUtensorMap* mg = it.dense ? &map_a_d0 : &map_a_exp;
            const CUtensorMap* mu = it.dense ? &map_a_d1 : &map_a_exp;
            const int gbase = it.dense ? it.m * 64 : it.e * (2 * I) + it.m * 64;
            const int ubase = it.dense ? it.m * 64 : it.e * (2 * I) + I + it.m * 64;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              tma_load_2d(a_dst + (2 * q) * 2048, mg, &full_bar[stage], k0, gbase + 16 * q, pol_w);
              tma_load_2d(a_dst + (2 * q + 1) * 2048, mu, &full_bar[stage], k0, ubase + 16 * q, pol_w);
            }
          } else {
            const CUtensorMap* ma = it.dense ? &map_a_d0 : &map_a_exp;
            const int arow = it.dense ? it.m * kBM : it.e * H + it.m * kBM;
            tma_load_2d(a_dst, ma, &full_bar[stage], k0, arow, pol_w);
          }
          const CUtensorMap* mb = it.dense ? &map_b_dense : &map_b_exp;
          for (int g = 0; g < n_g4; ++g) {
            const int jj = 4 * g;
            const int r0 = idx_s[jj];
            const int r1 = idx_s[min(jj + 1, it.rows - 1)];
            const int r2 = idx_s[min(jj + 2, it.rows - 1)];
            const int r3 = idx_s[min(jj + 3, it.rows - 1)];
            tma_gather4(b_dst + g * 512, mb, &full_bar[stage], k0, r0, r1, r2, r3, pol_x);
          }
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
      __syncwarp();
    }
    // Before the CTA can exit, every TMA load this warp issued must have landed.
    if (lane == 0)
      for (int s2 = 0; s2 < C::kStages; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&full_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs);
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer (one thread)
    if (lane == 0) {
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      bool ok = true;
      for (int i = blockIdx.x; i < total && ok; i += gridDim.x) {
        const int nkb = (i < n_dense_items) ? C::kKbDense : C::kKbExp;
        if (!mbar_wait_bounded(&acce_bar[acc], acc_phase ^ 1u, abort_flag, b.status, kStatusWaitAccEmpty)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, b.status, kStatusWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a_addr = smem_u32(stages + stage * C::kStageBytes);
          const uint64_t a_desc = smem_desc_sw128(a_addr);
          const uint64_t b_desc = smem_desc_sw128(a_addr + kABytes);
#pragma unroll
          for (int k = 0; k < kBK / 16; ++k)
            umma_bf16(d_tmem, a_desc + 2u * k, b_desc + 2u * k, C::kIdesc, (kb | k) != 0 ? 1u : 0u);
          umma_commit(&empty_bar[stage]);
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&accf_bar[acc]);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs issued above complete before this barrier's phase does.
      umma_commit(final_bar);
      mbar_wait_timeout(final_bar, 0, kSpinLimitNs);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2..5; TMEM lane quarter = warp % 4
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = blockIdx.x; i < total; i += gridDim.x) {
      const Item it = decode_item<BN, GATE_UP>(i, n_dense_items, b.exp_tiles, T);
      int got = 1;
      if (lane == 0) got = mbar_wait_bounded(&accf_bar[acc], acc_phase, abort_flag, b.status, kStatusWaitAccFull);
      got = __shfl_sync(0xffffffffu, got, 0);
      if (!got) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * BN);
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        if (c * 32 >= it.rows) break;
        float v[32];
        tmem_ld32(t_row + c * 32, v);
        if (GATE_UP) {
          // lanes 0..15: gate of feature f, lanes 16..31: up of the same feature
          const int f = it.m * 64 + 16 * q + (lane & 15);
          const bool is_gate = lane < 16;
          uint16_t* dst = it.dense ? b.h_dense : b.h;
          const int ld = it.dense ? D : I;
#pragma unroll
          for (int pr = 0; pr < 16; ++pr) {
            const float send = is_gate ? v[2 * pr + 1] : v[2 * pr];
            const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
            const float g = is_gate ? v[2 * pr] : recv;
            const float u = is_gate ? recv : v[2 * pr + 1];
            const int col = c * 32 + 2 * pr + (is_gate ? 0 : 1);
            if (col < it.rows) dst[static_cast<size_t>(it.row0 + col) * ld + f] = f32_to_bf16_rn(gelu_tanh_approx(g) * u);
          }
        } else {
          const int f = it.m * kBM + 32 * q + lane;
          if (it.dense) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = c * 32 + j;
              if (col < it.rows) b.d[static_cast<size_t>(it.row0 + col) * H + f] = v[j];
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int col = c * 32 + j;
              if (col < it.rows) {
                const int pos = it.row0 + col;
                b.y[static_cast<size_t>(pos) * H + f] = v[j] * b.w_sorted[pos];
              }
            }
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&acce_bar[acc]);
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  tc_fence_before();
  __syncthreads();
  pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, bool GATE_UP>
cudaError_t launch_t(const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid, cudaStream_t s) {
  using C = Cfg<BN, GATE_UP>;
  grouped_gemm_kernel<BN, GATE_UP><<<grid, kThreads, C::kSmem, s>>>(m.a_exp, m.a_dense0, m.a_dense1, m.b_exp,
                                                                    m.b_dense, b, T, full_layer);
  return cudaGetLastError();
}

template <int BN, bool GATE_UP>
cudaError_t set_limit() {
  using C = Cfg<BN, GATE_UP>;
  return cudaFuncSetAttribute(grouped_gemm_kernel<BN, GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              C::kSmem);
}

}  // namespace

cudaError_t gemm_set_smem_limits() {
  cudaError_t e;
  if ((e = set_limit<32, true>()) != cudaSuccess) return e;
  if ((e = set_limit<64, true>()) != cudaSuccess) return e;
  if ((e = set_limit<128, true>()) != cudaSuccess) return e;
  if ((e = set_limit<256, true>()) != cudaSuccess) return e;
  if ((e = set_limit<32, false>()) != cudaSuccess) return e;
  if ((e = set_limit<64, false>()) != cudaSuccess) return e;
  if ((e = set_limit<128, false>()) != cudaSuccess) return e;
  return set_limit<256, false>();
}

cudaError_t launch_gate_up(int bn, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                           cudaStream_t s) {
  switch (bn) {
    case 32: return launch_t<32, true>(m, b, T, full_layer, grid, s);
    case 64: return launch_t<64, true>(m, b, T, full_layer, grid, s);
    case 128: return launch_t<128, true>(m, b, T, full_layer, grid, s);
    case 256: return launch_t<256, true>(m, b, T, full_layer, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_down(int bn, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                        cudaStream_t s) {
  switch (bn) {
    case 32: return launch_t<32, false>(m, b, T, full_layer, grid, s);
    case 64: return launch_t<64, false>(m, b, T, full_layer, grid, s);
    case 128: return launch_t<128, false>(m, b, T, full_layer, grid, s);
    case 256: return launch_t<256, false>(m, b, T, full_layer, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
