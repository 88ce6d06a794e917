// gemm_pair.cu — the grouped down GEMM of the block for prefill-sized batches, on SM pairs
// (tcgen05.mma cta_group::2).
//
// What it computes is the same as the down GEMM of gemm.cu ("Porting a 128-expert MoE (Gemma-4
// 26B-A4B) to AWS Inferentia2 — where every rank weighted the wrong experts", section "The
// architecture": each expert's down projection [128, 2816, 704] of h, scaled by the slot's router
// weight, and the shared MLP's down projection [2816, 2112]).
//
// Why SM pairs: an M = 128 MMA reads its A and B operands from one SM's shared memory at every K
// step, 96 bytes per tensor cycle at N = 256, and the TMA loads write another 96 bytes per cycle
// into the same memory; together they exceed what shared memory delivers. A cluster of two CTAs
// on two SMs computes an M = 256 tile instead: each SM holds its 128 weight rows and half of the
// token rows, each half of B is read once for both SMs, and each SM loads half of B.
// (The gate_up GEMM stays on single SMs: its expert token rows are gathered with cp.async, and
// handing the peer's gathered rows to the leader's MMA costs more than the pair saves.)
//
// Layout of one work item (a token tile of up to 256 slots and a pair of 128-row weight tiles):
//   * rank r of the pair holds weight tile 2m + r: 128 rows of the hidden dimension;
//   * with an MMA width w (the tile's token rows rounded up to 16), rank r holds token rows
//     [r w/2, (r + 1) w/2) of the tile; the accumulator column j is token row j in both CTAs;
//   * each CTA's 128 accumulator rows sit in its own TMEM (two buffers of 256 columns).
// The leader (rank 0) issues the MMAs and commits to the barriers of both CTAs; both CTAs' TMA
// loads are counted on the leader's stage barrier. Both CTAs walk the same static list of items
// (cluster c takes every (gridDim/2)-th).
// Every output element is written by one CTA with a fixed K order, so results are reproducible.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kPBN = 256;                        // token rows per tile (the MMA's N)
constexpr int kPRows = 128;                      // weight rows per CTA (M = 256 per pair)
constexpr int kPBK = 64;                         // bf16 elements per 128-byte swizzled row
constexpr int kPAChunk = kPRows * kPBK * 2;      // 16 KB: this CTA's weight rows of one K chunk
constexpr int kPBChunk = (kPBN / 2) * kPBK * 2;  // 16 KB: this CTA's token rows of one K chunk
constexpr int kPStage = kPAChunk + kPBChunk;     // 32 KB
constexpr int kPStages = 6;
constexpr int kPTmemCols = 2 * kPBN;             // two accumulators of 256 columns
constexpr int kPThreads = 6 * 32;                // producer, MMA, four epilogue warps
constexpr int kPTiles = H / kPRows;              // 22 weight tiles per expert and for the shared MLP
constexpr int kPMt = kPTiles / 2;                // 11 pair items per token tile
constexpr int kPChunksExp = I / kPBK;            // 11 K chunks
constexpr int kPChunksDense = D / kPBK;          // 33
constexpr int kPXchgBytes = 4 * 32 * 32 * 4;     // a 32 x 32 output chunk per epilogue warp
constexpr int kPSmem = 1024 + kPStages * kPStage + kPXchgBytes + 512;
static_assert(kPTiles % 2 == 0, "weight tiles come in pairs");
static_assert(kPSmem <= 231424, "shared memory");

struct PItem {
  int dense;
  int e;
  int row0;
  int rows;
  int m;
  int nt;
};

// The same item order as gemm.cu: the shared-MLP group first, then the experts in id order, the
// token tile fastest within a group.
__device__ __forceinline__ PItem pair_item(int i, int n_dense_tiles, const int4* tiles, const int* tile_off, int T) {
  PItem it;
  const int n_dense_items = n_dense_tiles * kPMt;
  if (i < n_dense_items) {
    const int m = i / n_dense_tiles;
    const int j = i - m * n_dense_tiles;
    it.dense = 1;
    it.e = E;
    it.m = m;
    it.row0 = j * kPBN;
    it.rows = min(kPBN, T - j * kPBN);
    it.nt = n_dense_tiles;
  } else {
    const int i2 = i - n_dense_items;
    int lo = 0, hi = E - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (tile_off[mid] * kPMt <= i2)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int first = tile_off[lo];
    const int nt = tile_off[lo + 1] - first;
    const int local = i2 - first * kPMt;
    const int m = local / nt;
    const int j = local - m * nt;
    const int4 tt = tiles[first + j];
    it.dense = 0;
    it.e = tt.x;
    it.row0 = tt.y;
    it.rows = tt.z;
    it.m = m;
    it.nt = nt;
  }
  return it;
}

__device__ __forceinline__ bool pwarp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                           unsigned int* status, uint32_t why) {
  int got = 1;
  if ((threadIdx.x & 31) == 0) got = mbar_wait_bounded_cluster(bar, parity, abort_flag, status, why);
  return __shfl_sync(0xffffffffu, got, 0) != 0;
}

__global__ void __launch_bounds__(kPThreads, 1)
    down_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a_exp, const __grid_constant__ CUtensorMap map_a_dense,
                          const __grid_constant__ CUtensorMap map_b_exp, const __grid_constant__ CUtensorMap map_b_dense,
                          Buffers b, int T, int full_layer) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* xchg = smem + kPStages * kPStage;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(smem + kPStages * kPStage + kPXchgBytes);  // leader's
  uint64_t* empty_bar = full_bar + kPStages;  // both CTAs: the leader's MMAs are done with the stage
  uint64_t* accf_bar = empty_bar + kPStages;  // [2] both CTAs: accumulator ready
  uint64_t* acce_bar = accf_bar + 2;          // [2] leader: accumulator drained in both CTAs
  uint64_t* final_bar = acce_bar + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  const int cluster = static_cast<int>(blockIdx.x >> 1), n_clusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kPStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], 8);  // four epilogue warps in each CTA
    }
    mbar_init(final_bar, 1);
    *abort_flag = 0;
    fence_barrier_init_cluster();
    prefetch_tmap(&map_a_exp);
    prefetch_tmap(&map_b_exp);
    if (full_layer) {
      prefetch_tmap(&map_a_dense);
      prefetch_tmap(&map_b_dense);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, kPTmemCols);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers are initialised and the TMEM allocation is done before either CTA signals
  // the other.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  pdl_wait();
  const int n_tiles = *reinterpret_cast<volatile int*>(b.n_exp_tiles);
  const int n_dense_tiles = full_layer ? (T + kPBN - 1) / kPBN : 0;
  __shared__ int tile_off_s[E + 1];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) tile_off_s[e] = b.tile_off[e];
  __syncthreads();
  const int total = (n_dense_tiles + n_tiles) * kPMt;
  // The leader's stage and drained barriers, as shared::cluster addresses.
  const uint32_t full_leader0 = mapa_shared(smem_u32(&full_bar[0]), 0);
  const uint32_t acce_leader0 = mapa_shared(smem_u32(&acce_bar[0]), 0);

  if (warp == 0) {
    // ---------------- producer (both CTAs): this CTA's weight rows and token rows, by TMA
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;
    bool ok = true;
    for (int i = cluster; i < total && ok; i += n_clusters) {
      const PItem it = pair_item(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const int nch = it.dense ? kPChunksDense : kPChunksExp;
      const int half = min(kPBN, (it.rows + 15) & ~15) >> 1;
      const int tile = it.m * 2 + static_cast<int>(rank);
      const uint64_t pol_w = it.nt > 2 ? pol_keep : pol_once;
      const CUtensorMap* ma = it.dense ? &map_a_dense : &map_a_exp;
      const CUtensorMap* mb = it.dense ? &map_b_dense : &map_b_exp;
      const int arow = it.dense ? tile * kPRows : it.e * H + tile * kPRows;
      for (int c0 = 0; c0 < nch; ++c0) {
        if (!pwarp_wait(&empty_bar[stage], phase ^ 1u, abort_flag, b.status, kStatusWaitEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          uint8_t* st = stages + stage * kPStage;
          const uint32_t fb = full_leader0 + 8u * static_cast<uint32_t>(stage);
          if (leader) {
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            mbar_arrive_expect_tx(&full_bar[stage], 2 * kPStage);  // both CTAs' rows
          }
          const int k0 = c0 * kPBK;
          tma_load_2d_pair(st, ma, fb, k0, arow, pol_w);
          tma_load_2d_pair(st + kPAChunk, mb, fb, k0, it.row0 + static_cast<int>(rank) * half, pol_keep);
        }
        __syncwarp();
        if (++stage == kPStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // The leader's stage barriers count both CTAs' loads: wait for the last ones before exit.
    if (lane == 0 && leader)
      for (int s2 = 0; s2 < kPStages; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&full_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs, b.status);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader): M = 256 over the pair
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      for (int i = cluster; i < total && ok; i += n_clusters) {
        const PItem it = pair_item(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
        const int nch = it.dense ? kPChunksDense : kPChunksExp;
        const uint32_t idesc = idesc_bf16_f32(2 * kPRows, min(kPBN, (it.rows + 15) & ~15));
        if (!mbar_wait_bounded_cluster(&acce_bar[acc], acc_phase ^ 1u, abort_flag, b.status, kStatusWaitAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kPBN);
        for (int c0 = 0; c0 < nch; ++c0) {
          if (!mbar_wait_bounded_cluster(&full_bar[stage], phase, abort_flag, b.status, kStatusWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(stages + stage * kPStage);
          const uint64_t a_desc = smem_desc_sw128(st);
          const uint64_t b_desc = smem_desc_sw128(st + kPAChunk);
#pragma unroll
          for (int k = 0; k < kPBK / 16; ++k)
            umma_bf16_pair(d_tmem, a_desc + 2u * k, b_desc + 2u * k, idesc, (c0 | k) != 0 ? 1u : 0u);
          umma_commit_pair(&empty_bar[stage], 3);
          if (++stage == kPStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&accf_bar[acc], 3);
        acc ^= 1;
        if (acc == 0) acc_phase ^= 1u;
      }
      // All MMAs issued above complete before this barrier's phase does.
      umma_commit_pair(final_bar, 1);
      mbar_wait_timeout(final_bar, 0, kSpinLimitNs, b.status);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps 2..5 (both CTAs): TMEM lane quarter = warp % 4
    const int q = warp & 3;
    int acc = 0;
    uint32_t acc_phase = 0;
    for (int i = cluster; i < total; i += n_clusters) {
      const PItem it = pair_item(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const int tile = it.m * 2 + static_cast<int>(rank);
      if (!pwarp_wait(&accf_bar[acc], acc_phase, abort_flag, b.status, kStatusWaitAccFull)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + static_cast<uint32_t>(acc * kPBN);
      const int f0 = tile * kPRows + 32 * q;
      uint8_t* stg = xchg + q * 4096;
#pragma unroll 1
      for (int c = 0; c < kPBN / 32; ++c) {
        if (c * 32 >= it.rows) break;
        float v[32];
        tmem_ld32(t_row + c * 32, v);
        // The warp's 32 features x 32 token columns go through shared memory so that the global
        // stores are 16-byte vectors along the feature dimension.
        if (it.dense) {
          float* sd = reinterpret_cast<float*>(stg);  // [32 tokens][32 features]
#pragma unroll
          for (int j = 0; j < 32; ++j) sd[j * 32 + lane] = v[j];
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int idx = lane + 32 * u, r = idx >> 3, c4 = idx & 7;
            const int col = c * 32 + r;
            if (col < it.rows)
              *reinterpret_cast<float4*>(b.d + static_cast<size_t>(it.row0 + col) * H + f0 + 4 * c4) =
                  *reinterpret_cast<const float4*>(sd + r * 32 + 4 * c4);
          }
          __syncwarp();
        } else {
          // The router weights of this chunk's 32 slots: one coalesced load, then broadcast.
          const int my_col = c * 32 + lane;
          const float w_mine = my_col < it.rows ? __ldg(b.w_sorted + it.row0 + my_col) : 0.0f;
          uint16_t* sy = reinterpret_cast<uint16_t*>(stg);  // [32 slots][32 features] bf16
#pragma unroll
          for (int j = 0; j < 32; ++j) sy[j * 32 + lane] = f32_to_bf16_rn(v[j] * __shfl_sync(0xffffffffu, w_mine, j));
          __syncwarp();
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int idx = lane + 32 * u, r = idx >> 2, c8 = idx & 3;
            const int col = c * 32 + r;
            if (col < it.rows)
              *reinterpret_cast<uint4*>(b.y + static_cast<size_t>(it.row0 + col) * H + f0 + 8 * c8) =
                  *reinterpret_cast<const uint4*>(sy + r * 32 + 8 * c8);
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&acce_bar[acc]);
        else
          mbar_arrive_cluster(acce_leader0 + 8u * static_cast<uint32_t>(acc));
      }
      acc ^= 1;
      if (acc == 0) acc_phase ^= 1u;
    }
  }

  // Both CTAs stay until the leader's last MMA (which reads this CTA's shared memory and writes its
  // TMEM) has completed and every arrival on the other CTA's barriers has been made.
  tc_fence_before();
  __syncthreads();
  // The combine launches when this GEMM ends (its CTAs waiting beside the GEMM slowed it).
  pdl_launch_dependents();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, kPTmemCols);
  }
}

}  // namespace

cudaError_t gemm_pair_set_smem_limits() {
  return cudaFuncSetAttribute(down_gemm_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kPSmem);
}

// How many two-CTA clusters of the kernel can be resident at once on the current device (SMs pair
// up within a GPC, so this can be less than half the SMs); 0 if the query fails.
int gemm_pair_max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kPThreads);
  cfg.dynamicSmemBytes = kPSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, down_gemm_pair_kernel, &cfg) == cudaSuccess ? n : 0;
}

// grid: an even number of CTAs (one cluster per SM pair), at most twice gemm_pair_max_clusters().
// The maps: A = down / dense down weights (128-row boxes), B = h / h_dense (128-row boxes).
cudaError_t launch_down_pair(const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid, cudaStream_t s) {
  return launch_pdl_pair(down_gemm_pair_kernel, dim3(grid), dim3(kPThreads), kPSmem, s, m.a_exp, m.a_dense0, m.b_exp,
                         m.b_dense, b, T, full_layer);
}

}  // namespace moe
