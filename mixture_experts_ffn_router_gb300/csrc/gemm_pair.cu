// gemm_pair.cu — the two grouped GEMMs of the block for prefill-sized batches (token tiles of 256),
// on SM pairs (tcgen05.mma cta_group::2).
//
// What they compute is the same as the GEMMs of gemm.cu ("Porting a 128-expert MoE (Gemma-4
// 26B-A4B) to AWS Inferentia2 — where every rank weighted the wrong experts", section "The
// architecture"): gate_up forms h = gelu_tanh(gate x) * up x for each expert's tokens ([128, 1408,
// 2816], rows 0..703 gate, 704..1407 up) and for the shared MLP ([2112, 2816] gate and up); down
// forms y = w_slot * down(h) for the experts ([128, 2816, 704]) and d = down(h) for the shared MLP.
//
// Why SM pairs: an M = 128 MMA reads its A and B operands from one SM's shared memory at every K
// step, 96 bytes per tensor cycle at N = 256, and the TMA loads write more into the same memory. A
// cluster of two CTAs on two SMs computes an M = 256 tile instead: each SM holds its weight rows
// and half of the token rows, and each half of B is read once for both SMs.
//
// What bounds these GEMMs is the operand traffic from L2 into shared memory: one full-width M = 256
// item moves 1 byte per 128 FLOP, and at prefill the gate_up GEMM moved ~3.6 GB per launch at
// ~11 TB/s whether it ran on single SMs with two weight tiles per item or on pairs with one. So
// gate_up gives each CTA two weight tiles that share its half of the token rows: the gate rows of
// 128 features (tile 0) and the up rows of the same features (tile 1), two MMAs per K step into
// two accumulators. That cuts the bytes per FLOP by a quarter (2.9 GB per launch at T = 4096), and
// gate and up of a feature land in the same TMEM lane, so the epilogue forms gelu_tanh(g) * u with
// no hand-over. The two accumulators fill TMEM (2 x 256 columns), so they are single-buffered and
// drained by eight epilogue warps. down keeps one tile per CTA (its K = 704 is too short to hide a
// single-buffered epilogue) and double-buffers its accumulator; even so, one item's 11 K chunks
// take about as long as draining the accumulator with one warp per TMEM lane quarter, so down also
// drains with eight warps, two per quarter taking half the token columns each (T = 4096: 181 vs
// 198 us; sixteen warps: 189 us).
//
// Layout of one work item (a token tile of up to 256 slots and the pair's weight rows):
//   * gate_up: rank r holds features f = 256 m + 128 r .. + 127 (gate rows in tile 0, up rows in
//     tile 1, 128-row TMA boxes); 704 = 2.75 x 256 and 2112 = 8.25 x 256, so the last item of a
//     token tile has features past the end: their rows are read (inside the weight tensor, or
//     zero-filled past its end) and multiplied but not stored;
//   * down: rank r holds weight tile 2m + r: 128 rows of the hidden dimension;
//   * with an MMA width w (the tile's token rows rounded up to 16), rank r holds token rows
//     [r w/2, (r + 1) w/2) of the tile; the accumulator column j is token row j in both CTAs;
//   * each CTA's 128 accumulator rows sit in its own TMEM.
// The token rows are contiguous boxes: the shared MLP's n1 / h_dense in token order, the experts'
// gate_up input in sorted-slot order (a copy of n2 that the gate_up GEMM's epilogue warps write
// before their first accumulator is ready, while the shared-MLP items run) and their h.
//
// The leader (rank 0) issues the MMAs and commits to the barriers of both CTAs; both CTAs' TMA
// loads are counted on the leader's stage barrier. gate_up's work items are handed out dynamically: the
// leader's producer claims the next item from a global counter and publishes it in both CTAs'
// item rings (a store to the peer's shared memory and a remote arrive); the roles of both CTAs read
// the sequence from their own ring and release each slot on the leader's barrier. Which pair
// computes an item varies from run to run, but each item is computed whole by one pair in a fixed
// K order and every output element is written by one CTA, so the results do not.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kPBN = 256;                        // token rows per tile (the MMA's N)
constexpr int kPRows = 128;                      // weight rows per CTA and weight tile (M = 256 per pair)
constexpr int kPBK = 64;                         // bf16 elements per 128-byte swizzled row
constexpr int kPAChunk = kPRows * kPBK * 2;      // 16 KB: one weight tile of one K chunk
constexpr int kPBChunk = (kPBN / 2) * kPBK * 2;  // 16 KB: this CTA's token rows of one K chunk
constexpr int kPItemSlots = 8;

template <bool GATE_UP>
struct PCfg {
  static constexpr int MA = GATE_UP ? 2 : 1;                             // weight tiles per CTA
  static constexpr int kStage = MA * kPAChunk + kPBChunk;                // 48 | 32 KB
  static constexpr int kStages = GATE_UP ? 4 : 6;
  static constexpr int kNAcc = GATE_UP ? 1 : 2;                          // accumulator sets (buffers)
  static constexpr int kEpiWarps = 8;  // two per TMEM lane quarter, half the token columns each
  static constexpr int kThreads = (2 + kEpiWarps) * 32;                  // producer, MMA, epilogue
  // Item-slot consumers, all counted on the leader's release barrier: the leader's MMA thread and
  // epilogue warps, the peer's producer and epilogue warps.
  static constexpr int kItemConsumers = 2 + 2 * kEpiWarps;
  static constexpr int kFeat = GATE_UP ? 2 * kPRows : 0;                 // gate_up: features per item
  static constexpr int kMtExp = GATE_UP ? (I + kFeat - 1) / kFeat : H / (2 * kPRows);    // 3 | 11
  static constexpr int kMtDense = GATE_UP ? (D + kFeat - 1) / kFeat : H / (2 * kPRows);  // 9 | 11
  static constexpr int kChunksExp = GATE_UP ? H / kPBK : I / kPBK;      // 44 | 11 K chunks
  static constexpr int kChunksDense = GATE_UP ? H / kPBK : D / kPBK;    // 44 | 33
  static constexpr int kXchgBytes = kEpiWarps * 32 * 32 * 2;  // staging: 32 x 32 bf16 per warp
  static constexpr int kBarBytes = 512;
  static constexpr int kBarNeed = 8 * (2 * kStages + 2 * kNAcc + 1 + 2 * kPItemSlots) + 8 + 4 * kPItemSlots;
  static constexpr int kSmem = 1024 + kStages * kStage + kXchgBytes + kBarBytes;
  static constexpr int kTmemCols = 512;                                  // gate + up | two buffers
  static_assert(kStage % 1024 == 0, "operand tiles must stay 1024-byte aligned");
  static_assert(kBarNeed <= kBarBytes, "barrier area");
  static_assert(kSmem <= 231424, "shared memory");
  static_assert(kNAcc * MA * kPBN == kTmemCols, "TMEM columns");
};

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
template <bool GATE_UP>
__device__ __forceinline__ PItem pair_item(int i, int n_dense_tiles, const int4* tiles, const int* tile_off, int T) {
  using C = PCfg<GATE_UP>;
  PItem it;
  const int n_dense_items = n_dense_tiles * C::kMtDense;
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
      if (tile_off[mid] * C::kMtExp <= i2)
        lo = mid;
      else
        hi = mid - 1;
    }
    const int first = tile_off[lo];
    const int nt = tile_off[lo + 1] - first;
    const int local = i2 - first * C::kMtExp;
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

__device__ __forceinline__ void st_shared_cluster_u32(uint32_t cluster_addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(cluster_addr), "r"(v) : "memory");
}

// One consumer (a single thread) takes the next item from its CTA's ring and releases the slot on
// the leader's barrier: its index, -1 at the end, -2 if it gave up.
__device__ __forceinline__ int pair_next_item(uint64_t* itemf, const volatile int* item_s, uint32_t iteme_leader0,
                                              bool leader, uint64_t* iteme_local, int& slot, uint32_t& par,
                                              volatile int* abort_flag, unsigned int* status) {
  int i = -2;
  if (mbar_wait_bounded_cluster(&itemf[slot], par, abort_flag, status, kStatusWaitItem)) {
    i = item_s[slot];
    if (leader)
      mbar_arrive(&iteme_local[slot]);
    else
      mbar_arrive_cluster(iteme_leader0 + 8u * static_cast<uint32_t>(slot));
  }
  if (++slot == kPItemSlots) {
    slot = 0;
    par ^= 1u;
  }
  return i;
}

__device__ __forceinline__ int pair_warp_next_item(uint64_t* itemf, const volatile int* item_s, uint32_t iteme_leader0,
                                                   bool leader, uint64_t* iteme_local, int& slot, uint32_t& par,
                                                   volatile int* abort_flag, unsigned int* status) {
  int i = -2;
  if ((threadIdx.x & 31) == 0) {
    i = pair_next_item(itemf, item_s, iteme_leader0, leader, iteme_local, slot, par, abort_flag, status);
  } else if (++slot == kPItemSlots) {
    slot = 0;
    par ^= 1u;
  }
  return __shfl_sync(0xffffffffu, i, 0);
}

template <bool GATE_UP>
__global__ void __launch_bounds__(PCfg<GATE_UP>::kThreads, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a_exp, const __grid_constant__ CUtensorMap map_a_d0,
                             const __grid_constant__ CUtensorMap map_a_d1, const __grid_constant__ CUtensorMap map_b_exp,
                             const __grid_constant__ CUtensorMap map_b_dense, Buffers b, PermIn pin, int T,
                             int full_layer) {
  using C = PCfg<GATE_UP>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* xchg = smem + kStages * C::kStage;
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(xchg + C::kXchgBytes);  // leader's
  uint64_t* empty_bar = full_bar + kStages;    // both CTAs: the leader's MMAs are done with the stage
  uint64_t* accf_bar = empty_bar + kStages;    // [kNAcc] both CTAs: accumulator ready
  uint64_t* acce_bar = accf_bar + C::kNAcc;    // [kNAcc] leader: accumulator drained in both CTAs
  uint64_t* final_bar = acce_bar + C::kNAcc;
  uint64_t* itemf_bar = final_bar + 1;         // [kPItemSlots] both CTAs: the item is published
  uint64_t* iteme_bar = itemf_bar + kPItemSlots;  // [kPItemSlots] leader: every consumer has read it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(iteme_bar + kPItemSlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  volatile int* item_s = reinterpret_cast<volatile int*>(tmem_slot + 2);  // [kPItemSlots]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  // down: a static schedule (cluster c takes items c, c + clusters, ...), measured faster than the
  // dynamic one for its short items (200 vs 215 us at T = 4096).
  const int cluster = static_cast<int>(blockIdx.x >> 1), n_clusters = static_cast<int>(gridDim.x >> 1);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < C::kNAcc; ++a) {
      mbar_init(&accf_bar[a], 1);
      mbar_init(&acce_bar[a], 2 * C::kEpiWarps);  // the epilogue warps of both CTAs
    }
    mbar_init(final_bar, 1);
    for (int k = 0; k < kPItemSlots; ++k) {
      mbar_init(&itemf_bar[k], 1);
      mbar_init(&iteme_bar[k], C::kItemConsumers);
    }
    *abort_flag = 0;
    fence_barrier_init_cluster();
    prefetch_tmap(&map_a_exp);
    prefetch_tmap(&map_b_exp);
    if (full_layer) {
      prefetch_tmap(&map_a_d0);
      if (GATE_UP) prefetch_tmap(&map_a_d1);
      prefetch_tmap(&map_b_dense);
    }
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_slot, C::kTmemCols);
    tmem_relinquish_pair();
  }
  // Both CTAs' barriers are initialised and the TMEM allocation is done before either CTA signals
  // the other.
  tc_fence_before();
  cluster_sync_all();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  // Everything below reads what earlier kernels of the forward wrote.
  pdl_wait();
  // gate_up: dependents may launch now (the down GEMM runs nothing before its own wait that reads
  // this grid's results). The down GEMM's dependent is the combine, one CTA per token: thousands of
  // them waiting beside the GEMM's CTAs slowed it, so those launch when it ends.
  if (GATE_UP) pdl_launch_dependents();
  const int n_tiles = *reinterpret_cast<volatile int*>(b.n_exp_tiles);
  const int n_dense_tiles = full_layer ? (T + kPBN - 1) / kPBN : 0;
  __shared__ int tile_off_s[E + 1];
  for (int e = threadIdx.x; e <= E; e += blockDim.x) tile_off_s[e] = b.tile_off[e];
  __syncthreads();
  const int n_dense_items = n_dense_tiles * C::kMtDense;
  const int total = n_dense_items + n_tiles * C::kMtExp;
  // The leader's stage, drained and release barriers, as shared::cluster addresses.
  const uint32_t full_leader0 = mapa_shared(smem_u32(&full_bar[0]), 0);
  const uint32_t acce_leader0 = mapa_shared(smem_u32(&acce_bar[0]), 0);
  const uint32_t iteme_leader0 = mapa_shared(smem_u32(&iteme_bar[0]), 0);

  if (warp == 0) {
    // ---------------- producer (both CTAs): this CTA's weight rows and token rows, by TMA. The
    // leader's producer also claims the items and publishes them to both CTAs.
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int* sched = b.sched + (GATE_UP ? 0 : 1);
    const uint32_t itemf_peer0 = mapa_shared(smem_u32(&itemf_bar[0]), 1);
    const uint32_t item_peer0 = mapa_shared(smem_u32(const_cast<int*>(&item_s[0])), 1);
    int stage = 0;
    uint32_t phase = 0;
    uint32_t armed = 0, armed_par = 0;
    bool ok = true;
    int slot = 0;
    uint32_t slot_par = 0;
    int next = 0;
    bool have_next = false;
    bool copied = !GATE_UP;  // gate_up: the sorted copy of n2 is complete (seen once)
    int i_static = cluster;
    while (ok) {
      int i = -2;
      if (!GATE_UP) {
        i = i_static < total ? i_static : -1;
        i_static += n_clusters;
      } else if (leader) {
        if (lane == 0) {
          if (!have_next) next = atomicAdd(sched, 1);
          have_next = false;
          if (mbar_wait_bounded_cluster(&iteme_bar[slot], slot_par ^ 1u, abort_flag, b.status, kStatusWaitItem)) {
            i = next < total ? next : -1;
            item_s[slot] = i;
            st_shared_cluster_u32(item_peer0 + 4u * static_cast<uint32_t>(slot), static_cast<uint32_t>(i));
            mbar_arrive(&itemf_bar[slot]);
            mbar_arrive_cluster(itemf_peer0 + 8u * static_cast<uint32_t>(slot));
          }
        }
        i = __shfl_sync(0xffffffffu, i, 0);
        if (++slot == kPItemSlots) {
          slot = 0;
          slot_par ^= 1u;
        }
      } else {
        i = pair_warp_next_item(itemf_bar, item_s, iteme_leader0, false, iteme_bar, slot, slot_par, abort_flag,
                                b.status);
      }
      if (i < 0) break;
      const PItem it = pair_item<GATE_UP>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      if (!copied && !it.dense) {
        // The expert rows are the sorted copy of n2 that the epilogue warps of every CTA write
        // first: wait for all of them, then order the TMA reads after their (generic) stores.
        int got = 1;
        if (lane == 0)
          got = counter_wait_bounded(b.sched + 2, static_cast<int>(gridDim.x) * C::kEpiWarps, abort_flag, b.status,
                                     kStatusWaitCopy);
        if (!__shfl_sync(0xffffffffu, got, 0)) break;
        fence_proxy_async_global();
        copied = true;
      }
      const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
      const uint64_t pol_w = it.nt > 2 ? pol_keep : pol_once;
      const CUtensorMap* mb = it.dense ? &map_b_dense : &map_b_exp;
      const int brow = it.row0 + static_cast<int>(rank) * (min(kPBN, (it.rows + 15) & ~15) >> 1);
      const CUtensorMap* ma0 = it.dense ? &map_a_d0 : &map_a_exp;
      const CUtensorMap* ma1 = GATE_UP && it.dense ? &map_a_d1 : ma0;
      int arow0, arow1 = 0;
      if (GATE_UP) {
        // This CTA's 128 features; past the last feature the rows are read but not stored.
        const int f = it.m * C::kFeat + static_cast<int>(rank) * kPRows;
        arow0 = it.dense ? f : it.e * (2 * I) + f;
        arow1 = it.dense ? f : it.e * (2 * I) + I + f;
      } else {
        const int tile = it.m * 2 + static_cast<int>(rank);
        arow0 = it.dense ? tile * kPRows : it.e * H + tile * kPRows;
      }
      for (int c0 = 0; c0 < nch; ++c0) {
        if (!pwarp_wait(&empty_bar[stage], phase ^ 1u, abort_flag, b.status, kStatusWaitEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (GATE_UP && leader && !have_next && c0 + kStages >= nch) {
            next = atomicAdd(sched, 1);
            have_next = true;
          }
          uint8_t* st = stages + stage * C::kStage;
          const uint32_t fb = full_leader0 + 8u * static_cast<uint32_t>(stage);
          if (leader) {
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            mbar_arrive_expect_tx(&full_bar[stage], 2 * C::kStage);  // both CTAs' rows
          }
          const int k0 = c0 * kPBK;
          tma_load_2d_pair(st, ma0, fb, k0, arow0, pol_w);
          if (GATE_UP) tma_load_2d_pair(st + kPAChunk, ma1, fb, k0, arow1, pol_w);
          tma_load_2d_pair(st + C::MA * kPAChunk, mb, fb, k0, brow, pol_keep);
        }
        __syncwarp();
        if (++stage == kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // The leader's stage barriers count both CTAs' loads: wait for the last ones before exit.
    if (lane == 0 && leader)
      for (int s2 = 0; s2 < kStages; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&full_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs, b.status);
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0 && leader) {
      // ---------------- MMA issuer (leader): M = 256 over the pair, one MMA per weight tile
      int stage = 0, acc = 0;
      uint32_t phase = 0, acc_phase = 0;
      bool ok = true;
      int slot = 0;
      uint32_t slot_par = 0;
      int i_static = cluster;
      while (ok) {
        int i;
        if (GATE_UP) {
          i = pair_next_item(itemf_bar, item_s, iteme_leader0, true, iteme_bar, slot, slot_par, abort_flag, b.status);
        } else {
          i = i_static < total ? i_static : -1;
          i_static += n_clusters;
        }
        if (i < 0) break;
        const PItem it = pair_item<GATE_UP>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
        const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
        const uint32_t idesc = idesc_bf16_f32(2 * kPRows, min(kPBN, (it.rows + 15) & ~15));
        if (!mbar_wait_bounded_cluster(&acce_bar[acc], acc_phase ^ 1u, abort_flag, b.status, kStatusWaitAccEmpty))
          break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * C::MA * kPBN);
        for (int c0 = 0; c0 < nch; ++c0) {
          if (!mbar_wait_bounded_cluster(&full_bar[stage], phase, abort_flag, b.status, kStatusWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = smem_u32(stages + stage * C::kStage);
          const uint64_t b_desc = smem_desc_sw128(st + C::MA * kPAChunk);
#pragma unroll
          for (int k = 0; k < kPBK / 16; ++k)
#pragma unroll
            for (int a = 0; a < C::MA; ++a)
              umma_bf16_pair(d_tmem + static_cast<uint32_t>(a * kPBN), smem_desc_sw128(st + a * kPAChunk) + 2u * k,
                             b_desc + 2u * k, idesc, (c0 | k) != 0 ? 1u : 0u);
          umma_commit_pair(&empty_bar[stage], 3);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit_pair(&accf_bar[acc], 3);
        if (++acc == C::kNAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued above complete before this barrier's phase does.
      umma_commit_pair(final_bar, 1);
      mbar_wait_timeout(final_bar, 0, kSpinLimitNs, b.status);
    }
    __syncwarp();
  } else {
    // ---------------- epilogue warps (both CTAs): TMEM lane quarter q = warp % 4. gate_up: the two
    // warps of a quarter take half of the token columns each (down likewise).
    const int q = warp & 3;
    const int chalf = (warp - 2) >> 2;             // which share of the token columns
    constexpr int kColChunks = kPBN / 32 / (C::kEpiWarps / 4);  // 32-column chunks per warp
    if (GATE_UP) {
      // First, before any accumulator is ready: the experts' input in sorted-slot order. Warp w of
      // the grid takes tokens w, w + warps, ...: n2 = x / RMS(x) * (1 + pre_feedforward_layernorm_2)
      // (x itself in the experts-only mode), formed with the top-k kernel's arithmetic (same RMS
      // order and roundings), stored at the token's 8 sorted positions in the y buffer (which the
      // down GEMM overwrites only after this grid has ended). The producers wait for every warp's
      // count before their first expert item; the shared-MLP items, which read n1, run meanwhile.
      const int S = T * K;
      const int nw = static_cast<int>(gridDim.x) * C::kEpiWarps;
      for (int t = static_cast<int>(blockIdx.x) * C::kEpiWarps + (warp - 2); t < T; t += nw) {
        uint4 o[11];
        const uint4* xr = reinterpret_cast<const uint4*>(pin.x + static_cast<size_t>(t) * H);
#pragma unroll
        for (int c = 0; c < 11; ++c) o[c] = __ldg(xr + lane + 32 * c);
        const int4 pa = __ldcg(reinterpret_cast<const int4*>(b.slot_pos + static_cast<size_t>(t) * K));
        const int4 pb = __ldcg(reinterpret_cast<const int4*>(b.slot_pos + static_cast<size_t>(t) * K + 4));
        if (pin.w2) {
          float ss = 0.0f;
#pragma unroll
          for (int c = 0; c < 11; ++c) {
            const uint32_t w4[4] = {o[c].x, o[c].y, o[c].z, o[c].w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = __uint_as_float(w4[j] << 16), hi = __uint_as_float(w4[j] & 0xFFFF0000u);
              ss = fmaf(lo, lo, ss);
              ss = fmaf(hi, hi, ss);
            }
          }
#pragma unroll
          for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
          const float inv = 1.0f / sqrtf(ss / static_cast<float>(H) + pin.eps);
#pragma unroll
          for (int c = 0; c < 11; ++c) {
            const float4 wa = __ldg(reinterpret_cast<const float4*>(pin.w2) + 2 * (lane + 32 * c));
            const float4 wb = __ldg(reinterpret_cast<const float4*>(pin.w2) + 2 * (lane + 32 * c) + 1);
            const float g2[8] = {1.0f + wa.x, 1.0f + wa.y, 1.0f + wa.z, 1.0f + wa.w,
                                 1.0f + wb.x, 1.0f + wb.y, 1.0f + wb.z, 1.0f + wb.w};
            const uint32_t w4[4] = {o[c].x, o[c].y, o[c].z, o[c].w};
            uint32_t o2[4];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const float lo = __uint_as_float(w4[j] << 16) * inv, hi = __uint_as_float(w4[j] & 0xFFFF0000u) * inv;
              o2[j] = static_cast<uint32_t>(f32_to_bf16_rn(lo * g2[2 * j])) |
                      (static_cast<uint32_t>(f32_to_bf16_rn(hi * g2[2 * j + 1])) << 16);
            }
            o[c] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
          }
        }
        const int pos[K] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
        // An expert-parallel shard computes only its experts: the other slots need no copy.
        int ex[K] = {0, 0, 0, 0, 0, 0, 0, 0};
        if (pin.e_lo > 0 || pin.e_hi < E) {
          const int4 ea = __ldcg(reinterpret_cast<const int4*>(b.topk_idx + static_cast<size_t>(t) * K));
          const int4 eb = __ldcg(reinterpret_cast<const int4*>(b.topk_idx + static_cast<size_t>(t) * K + 4));
          ex[0] = ea.x; ex[1] = ea.y; ex[2] = ea.z; ex[3] = ea.w;
          ex[4] = eb.x; ex[5] = eb.y; ex[6] = eb.z; ex[7] = eb.w;
        } else {
#pragma unroll
          for (int k = 0; k < K; ++k) ex[k] = pin.e_lo;
        }
#pragma unroll
        for (int k = 0; k < K; ++k) {
          if (ex[k] < pin.e_lo || ex[k] >= pin.e_hi) continue;
          if (pos[k] < 0 || pos[k] >= S) {
            if (lane == 0) atomicOr(b.status, kStatusBadIndex);
            continue;
          }
          uint4* dst = reinterpret_cast<uint4*>(b.n2s + static_cast<size_t>(pos[k]) * H);
#pragma unroll
          for (int c = 0; c < 11; ++c) dst[lane + 32 * c] = o[c];
        }
      }
      fence_proxy_async_global();
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd(b.sched + 2, 1);
    }
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t slot_par = 0;
    int i_static = cluster;
    for (;;) {
      int i;
      if (GATE_UP) {
        i = pair_warp_next_item(itemf_bar, item_s, iteme_leader0, leader, iteme_bar, slot, slot_par, abort_flag,
                                b.status);
      } else {
        i = i_static < total ? i_static : -1;
        i_static += n_clusters;
      }
      if (i < 0) break;
      const PItem it = pair_item<GATE_UP>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      if (!pwarp_wait(&accf_bar[acc], acc_phase, abort_flag, b.status, kStatusWaitAccFull)) break;
      tc_fence_after();
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * C::MA * kPBN);
      if (GATE_UP) {
        // Features f .. f + 31 (one per lane): gate in columns [0, 256), up in [256, 512).
        const int f = it.m * C::kFeat + static_cast<int>(rank) * kPRows + 32 * q;
        const int nfeat = it.dense ? D : I;
        uint16_t* hs = reinterpret_cast<uint16_t*>(xchg) + (warp - 2) * (32 * 32);  // [32 columns][32 features]
        uint16_t* dst = it.dense ? b.h_dense : b.h;
        const int ld = it.dense ? D : I;
#pragma unroll 1
        for (int c = chalf * (kPBN / 64); c < (chalf + 1) * (kPBN / 64); ++c) {
          if (f >= nfeat || c * 32 >= it.rows) break;
          uint32_t g[32], u[32];
          tmem_ld32_nowait(t_row + c * 32, g);
          tmem_ld32_nowait(t_row + kPBN + c * 32, u);
          tmem_wait_ld();
          reg_fence32(g);
          reg_fence32(u);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            hs[j * 32 + lane] = f32_to_bf16_rn(gelu_tanh_approx(__uint_as_float(g[j])) * __uint_as_float(u[j]));
          __syncwarp();
#pragma unroll
          for (int u4 = 0; u4 < 4; ++u4) {
            const int idx = lane + 32 * u4, r = idx >> 2, c8 = idx & 3;
            const int col = c * 32 + r;
            if (col < it.rows)
              *reinterpret_cast<uint4*>(dst + static_cast<size_t>(it.row0 + col) * ld + f + 8 * c8) =
                  *reinterpret_cast<const uint4*>(hs + r * 32 + 8 * c8);
          }
          __syncwarp();
        }
      } else {
        const int f0 = (it.m * 2 + static_cast<int>(rank)) * kPRows + 32 * q;
        uint8_t* stg = xchg + (warp - 2) * 2048;
#pragma unroll 1
        for (int c = chalf * kColChunks; c < (chalf + 1) * kColChunks; ++c) {
          if (c * 32 >= it.rows) break;
          float v[32];
          tmem_ld32(t_row + c * 32, v);
          // The warp's 32 features x 32 token columns go through shared memory so that the global
          // stores are 16-byte vectors along the feature dimension.
          if (it.dense) {
            uint16_t* sd = reinterpret_cast<uint16_t*>(stg);  // [32 tokens][32 features] bf16
#pragma unroll
            for (int j = 0; j < 32; ++j) sd[j * 32 + lane] = f32_to_bf16_rn(v[j]);
            __syncwarp();
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const int idx = lane + 32 * u, r = idx >> 2, c8 = idx & 3;
              const int col = c * 32 + r;
              if (col < it.rows)
                *reinterpret_cast<uint4*>(b.d + static_cast<size_t>(it.row0 + col) * H + f0 + 8 * c8) =
                    *reinterpret_cast<const uint4*>(sd + r * 32 + 8 * c8);
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
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (leader)
          mbar_arrive(&acce_bar[acc]);
        else
          mbar_arrive_cluster(acce_leader0 + 8u * static_cast<uint32_t>(acc));
      }
      if (++acc == C::kNAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  }

  // Both CTAs stay until the leader's last MMA (which reads this CTA's shared memory and writes its
  // TMEM) has completed and every arrival on the other CTA's barriers has been made.
  tc_fence_before();
  __syncthreads();
  if (!GATE_UP) pdl_launch_dependents();
  cluster_sync_all();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, C::kTmemCols);
  }
}

template <bool GATE_UP>
cudaError_t set_pair_limit() {
  return cudaFuncSetAttribute(grouped_gemm_pair_kernel<GATE_UP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              PCfg<GATE_UP>::kSmem);
}

template <bool GATE_UP>
int max_clusters() {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(PCfg<GATE_UP>::kThreads);
  cfg.dynamicSmemBytes = PCfg<GATE_UP>::kSmem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<GATE_UP>, &cfg) == cudaSuccess ? n : 0;
}

}  // namespace

cudaError_t gemm_pair_set_smem_limits() {
  const cudaError_t e = set_pair_limit<true>();
  return e != cudaSuccess ? e : set_pair_limit<false>();
}

// How many two-CTA clusters of the pair GEMMs can be resident at once on the current device (SMs
// pair up within a GPC, so this can be less than half the SMs); 0 if the query fails.
int gemm_pair_max_clusters() {
  const int a = max_clusters<true>(), b = max_clusters<false>();
  return a < b ? a : b;
}

// grid: an even number of CTAs (one cluster per SM pair), at most twice gemm_pair_max_clusters().
// gate_up maps: A = gate_up rows / dense gate / dense up (128-row boxes), B = the sorted copy of n2 /
// n1 (128-row boxes). down maps: A = down / dense down (128-row boxes), B = h / h_dense (128-row
// boxes).
// gate_up also writes the sorted copy of n2 (pin: its inputs); every CTA must be resident at once,
// so grid is at most twice the resident-cluster count.
cudaError_t launch_gate_up_pair(const GemmMaps& m, const Buffers& b, const PermIn& pin, int T, int full_layer,
                                int grid, cudaStream_t s) {
  return launch_pdl_pair(grouped_gemm_pair_kernel<true>, dim3(grid), dim3(PCfg<true>::kThreads), PCfg<true>::kSmem, s,
                         m.a_exp, m.a_dense0, m.a_dense1, m.b_exp, m.b_dense, b, pin, T, full_layer);
}

cudaError_t launch_down_pair(const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid, cudaStream_t s) {
  const PermIn none = {nullptr, nullptr, 0.0f, 0, 0};
  return launch_pdl_pair(grouped_gemm_pair_kernel<false>, dim3(grid), dim3(PCfg<false>::kThreads), PCfg<false>::kSmem,
                         s, m.a_exp, m.a_dense0, m.a_dense1, m.b_exp, m.b_dense, b, none, T, full_layer);
}

}  // namespace moe
