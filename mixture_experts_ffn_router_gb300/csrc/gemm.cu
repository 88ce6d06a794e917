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
// pairs (or, for the widest token tiles, a token tile and two weight tiles); the token tiles of
// the experts come from a device-side list built by the top-k kernel, the shared MLP is one more
// group over all T tokens. CTAs are persistent and claim items one at a time from a global
// counter, so a CTA that drew short items takes more of them; every output element is written by
// exactly one CTA with a fixed K order, so results are bitwise reproducible.
//
// Operand loading. A (weights): 2-D TMA boxes of 64 K-elements (one 128-byte swizzled row) by 64
// (gate_up: gate rows, then up rows) or 128 (down) rows. B (tokens): when the token rows are
// contiguous in memory (the shared MLP's n1 / h_dense, the experts' h in sorted-slot order) one
// 2-D TMA box of BN rows; for the experts' gate_up input the rows are gathered by token index from
// n2 with cp.async by four gather warps, which write the same 128-byte-swizzled layout TMA would.
// A stage holds KC consecutive K chunks of 64 of both operands (KC = 2 for narrow token tiles, so
// each weight row is fetched 256 bytes at a time); one ring, so the MMA thread waits and commits
// once per stage. The MMA of a tile is only as wide as its token rows (rounded up to 16), which the
// producer passes to the MMA thread with each stage.
//
// Warp roles: warp 0 loads A, and B when it is a box; warp 1 issues the MMAs (one thread); warps
// 2..5 run the epilogue, warp w reading TMEM lanes 32*(w%4).. ; gate_up only: warps 6..9 gather B.
// Two TMEM accumulators let the epilogue of one item overlap the main loop of the next.
//
// gate_up epilogue: TMEM lanes 0..63 hold gate, 64..127 up, of features f0..f0+63. The warps of
// quarters q and q+2 hold gate and up of the same 32 features; each hands half of its columns to
// the other through shared memory, and each then forms h = gelu_tanh(gate) * up for 16 columns.
// down epilogue: y[slot] = w_slot * acc (bf16, sorted-slot order); the shared MLP writes d (bf16).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kBM = 128;
constexpr int kBK = 64;                    // bf16 elements per 128-byte swizzled row
constexpr int kAChunk = kBM * kBK * 2;     // 16 KB of A per K chunk
constexpr int kRingBudget = 204800;       // shared memory for the stage ring

// MA = weight tiles per work item: 1, or 2 (an M = 256 item: two 128-row weight tiles share each
// K chunk of the token tile, which cuts the operand bytes per FLOP from (1/128 + 1/BN) to
// (1/256 + 1/BN) of the row bytes).
//
// QW: the experts' weight format, 0 bf16, 1 int8 (kWInt8), 2 MXFP4 (kWFp4). With a converted
// format (CVT) the A operand of every MMA comes from tensor memory: a producer warp streams the
// weight rows by TMA into a ring of their own (kRawSlots slots of 128 rows x 128 bytes, 128-byte
// swizzle: two int8 K chunks, four MXFP4 K chunks, or one bf16 K chunk of the shared MLP); eight
// converter warps, two groups of four taking alternate K chunks, widen each chunk to bf16 (or copy
// it) into a ring of kASlots A chunks in TMEM; the stages in shared memory hold only B; two MMA
// issuers take alternate K chunks into partial accumulators. int8 rows are scaled in the
// epilogue (one scale per row), MXFP4 blocks in the widening (one scale per 32 weights).
constexpr int kWBf16 = 0, kWInt8 = 1, kWFp4 = 2;

template <int BN, bool GATE_UP, int MA, int QW = kWBf16>
struct Cfg {
  static constexpr bool CVT = QW != kWBf16;
  static constexpr bool F4 = QW == kWFp4;
  static constexpr int kExpChunksPerSlot = F4 ? 4 : 2;           // K chunks in a weight-row slot (CVT)
  static constexpr int KC = (BN <= 64 && !CVT) ? 2 : 1;
  static constexpr int kAStage = CVT ? 0 : MA * kAChunk;            // A bytes of one K chunk in a stage
  static constexpr int kBChunk = BN * kBK * 2;
  static constexpr int kChunkBytes = kAStage + kBChunk;
  static constexpr int kStageBytes = KC * kChunkBytes;
  static constexpr int kRawSlots = CVT ? (BN <= 32 ? 10 : 8) : 0;   // weight-row ring (CVT)
  static constexpr int kRawSlotBytes = kBM * 128;                  // 128 rows of 128 bytes
  static constexpr int kStagesRaw = (kRingBudget - kRawSlots * kRawSlotBytes) / kStageBytes;
  static constexpr int kStageCap = CVT ? 16 : 8;
  static constexpr int kStages = kStagesRaw > kStageCap ? kStageCap : kStagesRaw;
  static constexpr int kEpiWarps = 4 * MA;                         // one per TMEM lane quarter and tile
  static constexpr int kGatherWarps = GATE_UP ? 4 : 0;
  static constexpr int kGatherWarp0 = 2 + kEpiWarps;
  static constexpr int kConvWarps = CVT ? 8 : 0;                    // converters to bf16 (CVT)
  static constexpr int kConvWarp0 = kGatherWarp0 + kGatherWarps;
  static constexpr int kRawWarp = kConvWarp0 + kConvWarps;         // the weight-row producer (CVT)
  static constexpr int kMma2Warp = kRawWarp + 1;                   // the second MMA issuer (CVT)
  static constexpr int kIssuers = CVT ? 2 : 1;
  static constexpr int kThreads = (kRawWarp + (CVT ? 2 : 0)) * 32;
  static constexpr int kFullArrivals = 1 + kGatherWarps * 32;
  static constexpr int kItemConsumers = kIssuers + kEpiWarps + kGatherWarps + kConvWarps + (CVT ? 1 : 0);
  static constexpr int kAccCols = MA * BN;                         // TMEM columns of one accumulator set
  static constexpr int kNAcc = 2 * kAccCols <= 512 ? 2 : 1;        // double-buffered where it fits
  static constexpr int kACol0 = kNAcc * kIssuers * kAccCols;       // CVT: first TMEM column of the A ring
  static constexpr int kASlots = CVT ? (512 - kACol0) / 32 : 0;     // CVT: A chunks (128 x 64 bf16 = 32 columns)
  static constexpr int kTmemColsRaw = CVT ? 512 : kNAcc * kAccCols;
  static constexpr int kTmemCols = kTmemColsRaw < 32 ? 32 : kTmemColsRaw;
  static constexpr int kTilesExp = GATE_UP ? I / 64 : H / kBM;     // 11 | 22 weight tiles per expert
  static constexpr int kTilesDense = GATE_UP ? D / 64 : H / kBM;   // 33 | 22
  static constexpr int kMtExp = (kTilesExp + MA - 1) / MA;         // items per token tile
  static constexpr int kMtDense = (kTilesDense + MA - 1) / MA;
  static constexpr int kChunksExp = GATE_UP ? H / kBK : I / kBK;   // 44 | 11 K chunks
  static constexpr int kChunksDense = GATE_UP ? H / kBK : D / kBK; // 44 | 33
  // gate_up: the gate/up hand-over [warps][16][32] fp32; down: a 32x32 output chunk per warp.
  static constexpr int kXchgBytes = kEpiWarps * (GATE_UP ? 16 * 32 * 4 : 32 * 32 * 4);
  static constexpr int kBarBytes = CVT ? 1024 : 512;
  static constexpr int kBarNeed = 8 * (2 * kStages + 5 + 2 * 8 + 2 * kRawSlots + 2 * kASlots) + 8 + 4 * kStages + 4 * 8;
  static constexpr int kSmem = 1024 + kStages * kStageBytes + kRawSlots * kRawSlotBytes + kXchgBytes + kBarBytes;
  static_assert(kChunkBytes % 1024 == 0, "operand tiles must stay 1024-byte aligned");
  static_assert(BN % 32 == 0 && BN >= 32 && BN <= 256, "BN");
  static_assert(MA == 1 || MA == 2, "MA");
  static_assert(kTmemColsRaw <= 512 && (kTmemCols & (kTmemCols - 1)) == 0, "TMEM columns");
  static_assert(kStages >= 2, "stages");
  static_assert(!CVT || (MA == 1 && KC == 1), "converted weights: one weight tile per item, one K chunk per stage");
  static_assert(!CVT || kConvWarps == 8, "two groups of four converter warps, one per TMEM lane quarter");
  static_assert(!CVT || kASlots >= 4, "TMEM A ring");
  static_assert(kBarNeed <= kBarBytes, "barrier area");
  static_assert(kSmem <= 231424, "shared memory");
};

struct Item {
  int dense;
  int e;
  int row0;
  int rows;
  int m;
  int nt;  // token tiles of the item's group (expert or shared MLP)
};

// Items: the shared-MLP group first (its items are the longest for the down GEMM), then the experts
// in id order. Within a group the token tiles of one weight tile are consecutive (token tile
// fastest), so CTAs working at the same time share that weight tile through L2; an expert's items
// span [11 or 22] x (its token tiles), located with a binary search over tile_off.
template <int BN, bool GATE_UP, int MA>
__device__ __forceinline__ Item decode_item(int i, int n_dense_tiles, const int4* tiles, const int* tile_off,
                                            int T) {
  using C = Cfg<BN, GATE_UP, MA>;
  Item it;
  const int n_dense_items = n_dense_tiles * C::kMtDense;
  if (i < n_dense_items) {
    const int m = i / n_dense_tiles;
    const int j = i - m * n_dense_tiles;
    it.dense = 1;
    it.e = E;
    it.m = m;
    it.row0 = j * BN;
    it.rows = min(BN, T - j * BN);
    it.nt = n_dense_tiles;
  } else {
    const int i2 = i - n_dense_items;
    int lo = 0, hi = E - 1;  // the last expert whose items start at or before i2
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

__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ void named_bar_sync(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// Work items are handed out dynamically: the producer warp claims the next item index from a
// global counter and publishes it in a ring of kItemSlots slots in shared memory; the MMA thread,
// the epilogue warps and the gather warps read the same sequence from the ring. -1 ends the
// sequence. Which CTA computes an item varies from run to run, but each item is still computed
// whole by one CTA in a fixed order, so the results do not.
constexpr int kItemSlots = 8;

// One consumer (a single thread) takes the next item: its index, -1 at the end, -2 if it gave up.
__device__ __forceinline__ int next_item(uint64_t* itemf, uint64_t* iteme, const volatile int* item_s, int& slot,
                                         uint32_t& par, volatile int* abort_flag, unsigned int* status) {
  int i = -2;
  if (mbar_wait_bounded(&itemf[slot], par, abort_flag, status, kStatusWaitItem)) {
    i = item_s[slot];
    mbar_arrive(&iteme[slot]);
  }
  if (++slot == kItemSlots) {
    slot = 0;
    par ^= 1u;
  }
  return i;
}

// The same for a whole warp: lane 0 takes the item, the index is broadcast.
__device__ __forceinline__ int warp_next_item(uint64_t* itemf, uint64_t* iteme, const volatile int* item_s,
                                              int& slot, uint32_t& par, volatile int* abort_flag,
                                              unsigned int* status) {
  int i = -2;
  if ((threadIdx.x & 31) == 0) {
    i = next_item(itemf, iteme, item_s, slot, par, abort_flag, status);
  } else if (++slot == kItemSlots) {
    slot = 0;
    par ^= 1u;
  }
  return __shfl_sync(0xffffffffu, i, 0);
}

// Lane 0 waits, the result is broadcast, so the warp stays converged.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          unsigned int* status, uint32_t why) {
  int got = 1;
  if ((threadIdx.x & 31) == 0) got = mbar_wait_bounded(bar, parity, abort_flag, status, why);
  return __shfl_sync(0xffffffffu, got, 0) != 0;
}

template <int BN, bool GATE_UP, int MA, int QW>
__global__ void __launch_bounds__(Cfg<BN, GATE_UP, MA, QW>::kThreads, 1)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap map_a_exp, const __grid_constant__ CUtensorMap map_a_d0,
                        const __grid_constant__ CUtensorMap map_a_d1, const __grid_constant__ CUtensorMap map_b_exp,
                        const __grid_constant__ CUtensorMap map_b_dense, Buffers b, int T, int full_layer,
                        const __grid_constant__ CUtensorMap map_q, const void* q_scale) {
  using C = Cfg<BN, GATE_UP, MA, QW>;
  constexpr bool CVT = C::CVT;
  constexpr bool F4 = C::F4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stages = smem;
  uint8_t* raw_ring = smem + C::kStages * C::kStageBytes;  // CVT: weight-row slots
  uint8_t* after_rings = raw_ring + C::kRawSlots * C::kRawSlotBytes;
  float* xchg = reinterpret_cast<float*>(after_rings);
  uint64_t* full_bar = reinterpret_cast<uint64_t*>(after_rings + C::kXchgBytes);
  uint64_t* empty_bar = full_bar + C::kStages;
  uint64_t* accf_bar = empty_bar + C::kStages;  // [kNAcc] accumulator ready
  uint64_t* acce_bar = accf_bar + 2;            // [kNAcc] accumulator drained
  uint64_t* final_bar = acce_bar + 2;
  uint64_t* itemf_bar = final_bar + 1;          // [kItemSlots] item published
  uint64_t* iteme_bar = itemf_bar + kItemSlots; // [kItemSlots] item read by every consumer
  uint64_t* rawf_bar = iteme_bar + kItemSlots;      // [kRawSlots] CVT: a weight slot has landed
  uint64_t* rawe_bar = rawf_bar + C::kRawSlots;     // [kRawSlots] CVT: the converters are done with it
  uint64_t* af_bar = rawe_bar + C::kRawSlots;       // [kASlots] CVT: an A chunk is in TMEM
  uint64_t* ae_bar = af_bar + C::kASlots;           // [kASlots] CVT: the MMAs are done with it
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(ae_bar + C::kASlots);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* width_s = reinterpret_cast<int*>(tmem_slot + 2);  // [kStages] MMA width of each stage
  volatile int* item_s = reinterpret_cast<volatile int*>(width_s + C::kStages);  // [kItemSlots] item ring

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < C::kStages; ++s) {
      mbar_init(&full_bar[s], C::kFullArrivals);
      mbar_init(&empty_bar[s], 1);
    }
    for (int a = 0; a < C::kNAcc; ++a) {
      mbar_init(&accf_bar[a], C::kIssuers);
      mbar_init(&acce_bar[a], C::kEpiWarps);
    }
    mbar_init(final_bar, C::kIssuers);
    for (int k = 0; k < kItemSlots; ++k) {
      mbar_init(&itemf_bar[k], 1);
      mbar_init(&iteme_bar[k], C::kItemConsumers);
    }
    for (int r = 0; r < C::kRawSlots; ++r) {
      mbar_init(&rawf_bar[r], 1);
      mbar_init(&rawe_bar[r], C::kConvWarps);  // one arrival per warp (two for a slot read by one group)
    }
    for (int a = 0; a < C::kASlots; ++a) {
      mbar_init(&af_bar[a], C::kConvWarps / 2);
      mbar_init(&ae_bar[a], 1);
    }
    *abort_flag = 0;
    fence_barrier_init();
    prefetch_tmap(&map_a_exp);
    if (!GATE_UP) prefetch_tmap(&map_b_exp);
    if (CVT) prefetch_tmap(&map_q);
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

  // The down GEMM's tile list was written two kernels back, by a kernel that had completed before
  // gate_up passed its own dependency wait and let this grid launch, and its weights are inputs.
  // So its producer claims its first item and issues that item's first weight stages before the
  // wait, while gate_up's last items still run; the token rows (gate_up's output) follow after it.
  // Token tiles of at most 64 only: at T = 64 the forward ends 1.1 us earlier (the first weight
  // load moves from 1.6 us after gate_up's end to 11 us before it), at T = 1 1.7 us earlier; with
  // tiles of 128 (T = 1024) the down GEMM ended 6 us later.
  constexpr bool kPreload = !GATE_UP && !CVT && BN <= 64;
  // Each role decodes items with a binary search over the experts' first tiles; keep them on chip.
  __shared__ int tile_off_s[E + 1];
  int n_tiles = 0;
  auto load_tiles = [&]() {
    n_tiles = *reinterpret_cast<volatile int*>(b.n_exp_tiles);
    for (int e = threadIdx.x; e <= E; e += blockDim.x) tile_off_s[e] = b.tile_off[e];
    __syncthreads();
  };
  if (kPreload) load_tiles();
  const int n_dense_tiles = full_layer ? (T + BN - 1) / BN : 0;
  const int n_dense_items = n_dense_tiles * C::kMtDense;
  // The producer's item claimed before the wait (-2: none) and its stages armed there.
  int pre_item = -2, pre_stages = 0;
  if (kPreload && warp == 0) {
    if (lane == 0) {
      const int total0 = n_dense_items + n_tiles * C::kMtExp;
      const int i0 = atomicAdd(b.sched + 1, 1);
      pre_item = i0 < total0 ? i0 : -1;
      item_s[0] = pre_item;  // slot 0 of the item ring is free at the start
      mbar_arrive(&itemf_bar[0]);
      if (pre_item >= 0) {
        const Item it = decode_item<BN, GATE_UP, MA>(pre_item, n_dense_tiles, b.exp_tiles, tile_off_s, T);
        const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
        const int width = min(BN, (it.rows + 15) & ~15);
        const int na = min(MA, (it.dense ? C::kTilesDense : C::kTilesExp) - it.m * MA);
        const uint64_t pol_w = (it.nt > 2 && !(it.dense && BN <= 64)) ? policy_evict_last() : policy_evict_first();
        const CUtensorMap* mp = it.dense ? &map_a_d0 : &map_a_exp;
        pre_stages = min((nch + C::KC - 1) / C::KC, C::kStages);
        for (int s2 = 0; s2 < pre_stages; ++s2) {
          const int c0 = s2 * C::KC, nck = min(C::KC, nch - c0);
          uint8_t* st = stages + s2 * C::kStageBytes;
          width_s[s2] = width | (na << 16);
          mbar_expect_tx(&full_bar[s2], nck * na * kAChunk);
          for (int cc = 0; cc < nck; ++cc)
            for (int a = 0; a < na; ++a) {
              const int tile = it.m * MA + a;
              tma_load_2d(st + cc * C::kChunkBytes + a * kAChunk, mp, &full_bar[s2], (c0 + cc) * kBK,
                          it.dense ? tile * kBM : it.e * H + tile * kBM, pol_w);
            }
        }
      }
    }
    pre_item = __shfl_sync(0xffffffffu, pre_item, 0);
    pre_stages = __shfl_sync(0xffffffffu, pre_stages, 0);
  }

  // Everything below reads what earlier kernels of the forward wrote.
  pdl_wait();
  // Dependents may launch now (they run nothing before their own wait that reads this grid's
  // results, and everything before this grid is complete) -- except those of the down GEMM above
  // small batches: its dependent is the combine, one CTA per token, and thousands of combine CTAs
  // waiting beside the GEMM's CTAs slowed it (T = 256: 289.4 vs 286.8 us per layer; T = 4096:
  // 613.5 vs 595.7 us). Those launch when the GEMM ends.
  const bool early_dependents = GATE_UP || T <= kEarlyCombineT;
  if (early_dependents) pdl_launch_dependents();
  if (!kPreload) load_tiles();
  const int total = n_dense_items + n_tiles * C::kMtExp;

  if (warp == 0) {
    // ---------------- producer: TMA loads of A, and of B when its rows are contiguous
    // Weight tiles that at least two more token tiles of the same group read again are kept in L2
    // (evict_last); the rest stream through (evict_first). Keeping tiles with one re-read was
    // measured slower: the lines stay protected in L2 long after their last use. So was keeping
    // the shared MLP's tiles at 64-token tiles (T <= 256: up to four token tiles, read at nearly
    // the same time anyway): the 30-layer stack at T = 256 took 8.51 vs 8.23 ms.
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    const uint64_t pol_x = pol_keep;
    int stage = 0;
    uint32_t phase = 0;
    // stages this warp armed, and the parity of the last arm
    uint32_t armed = (1u << pre_stages) - 1u, armed_par = 0;
    bool ok = true;
    int* sched = b.sched + (GATE_UP ? 0 : 1);
    int slot = pre_item != -2 ? 1 : 0;  // the item claimed before the wait took slot 0
    uint32_t slot_par = 0;
    // The next item is claimed one ring's depth of stages before the current one is fully issued:
    // late enough that a CTA busy with a long item does not hold on to work an idle CTA could
    // take, early enough that the atomic's round trip overlaps the loads still to come.
    int next = 0;
    bool have_next = false;
    // Converted weights: the weight-row producer's ring holds 20 (int8) or 40 (MXFP4) K chunks, far
    // more than this warp's stage ring runs ahead of the MMAs, so each item is claimed and published
    // when the one before it starts (-3: none published ahead).
    int pub_next = -3;
    while (ok) {
      int i = -2;
      const bool preloaded = pre_item != -2;  // the item claimed (and published) before the wait
      if (preloaded) {
        i = pre_item;
        pre_item = -2;
      } else if (pub_next != -3) {
        i = pub_next;
        pub_next = -3;
      } else {
        if (lane == 0) {
          if (!have_next) next = atomicAdd(sched, 1);
          have_next = false;
          if (mbar_wait_bounded(&iteme_bar[slot], slot_par ^ 1u, abort_flag, b.status, kStatusWaitItem)) {
            i = next < total ? next : -1;
            item_s[slot] = i;
            mbar_arrive(&itemf_bar[slot]);
          }
        }
        i = __shfl_sync(0xffffffffu, i, 0);
        if (++slot == kItemSlots) {
          slot = 0;
          slot_par ^= 1u;
        }
      }
      if (i < 0) break;
      if (CVT) {
        int n2 = -2;
        if (lane == 0) {
          const int nx = atomicAdd(sched, 1);
          if (mbar_wait_bounded(&iteme_bar[slot], slot_par ^ 1u, abort_flag, b.status, kStatusWaitItem)) {
            n2 = nx < total ? nx : -1;
            item_s[slot] = n2;
            mbar_arrive(&itemf_bar[slot]);
          }
        }
        n2 = __shfl_sync(0xffffffffu, n2, 0);
        if (++slot == kItemSlots) {
          slot = 0;
          slot_par ^= 1u;
        }
        if (n2 == -2) break;  // gave up waiting (the status word says why)
        pub_next = n2;
      }
      const Item it = decode_item<BN, GATE_UP, MA>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
      const bool b_tma = !GATE_UP || it.dense;
      const int width = min(BN, (it.rows + 15) & ~15);
      const int n_tiles_raw = it.dense ? C::kTilesDense : C::kTilesExp;
      const int na = min(MA, n_tiles_raw - it.m * MA);  // weight tiles of this item
      const uint64_t pol_w = (it.nt > 2 && !(it.dense && BN <= 64)) ? pol_keep : pol_once;
      // gate_up with two tiles: tile 0 holds the gate rows and tile 1 the up rows of 128 features
      // ("paired"); otherwise each tile holds the gate and up rows of 64 features ("stacked").
      const bool paired = GATE_UP && MA == 2 && na == 2;
      // Converted weights: every A chunk reaches tensor memory through the converter warps, not by TMA.
      const bool a_tma = !CVT;
      for (int c0 = 0; c0 < nch; c0 += C::KC) {
        // A stage armed before the wait holds its weight rows already: only its token rows remain.
        const bool pre_st = preloaded && c0 / C::KC < pre_stages;
        if (!pre_st && !warp_wait(&empty_bar[stage], phase ^ 1u, abort_flag, b.status, kStatusWaitEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (!CVT && !have_next && c0 + C::kStages * C::KC >= nch) {
            next = atomicAdd(sched, 1);
            have_next = true;
          }
          const int nck = min(C::KC, nch - c0);
          uint8_t* st = stages + stage * C::kStageBytes;
          if (pre_st) {
            mbar_arrive_expect_tx(&full_bar[stage], nck * (b_tma ? C::kBChunk : 0));
          } else {
            armed |= 1u << stage;
            armed_par = (armed_par & ~(1u << stage)) | (phase << stage);
            width_s[stage] = width | (na << 16);
            mbar_arrive_expect_tx(&full_bar[stage], nck * ((a_tma ? na * kAChunk : 0) + (b_tma ? C::kBChunk : 0)));
          }
          for (int cc = 0; cc < nck; ++cc) {
            uint8_t* a_dst = st + cc * C::kChunkBytes;
            const int k0 = (c0 + cc) * kBK;
            if (paired && !pre_st) {
              const CUtensorMap* mg = it.dense ? &map_a_d0 : &map_a_exp;
              const CUtensorMap* mu = it.dense ? &map_a_d1 : &map_a_exp;
              const int f0 = it.m * 128;
              const int grow = it.dense ? f0 : it.e * (2 * I) + f0;
              const int urow = it.dense ? f0 : it.e * (2 * I) + I + f0;
              tma_load_2d(a_dst, mg, &full_bar[stage], k0, grow, pol_w);
              tma_load_2d(a_dst + kAChunk / 2, mg, &full_bar[stage], k0, grow + 64, pol_w);
              tma_load_2d(a_dst + kAChunk, mu, &full_bar[stage], k0, urow, pol_w);
              tma_load_2d(a_dst + kAChunk + kAChunk / 2, mu, &full_bar[stage], k0, urow + 64, pol_w);
            }
            for (int a = 0; a < (paired || !a_tma || pre_st ? 0 : na); ++a) {
              const int tile = it.m * MA + a;
              if (GATE_UP) {
                const CUtensorMap* mg = it.dense ? &map_a_d0 : &map_a_exp;
                const CUtensorMap* mu = it.dense ? &map_a_d1 : &map_a_exp;
                const int grow = it.dense ? tile * 64 : it.e * (2 * I) + tile * 64;
                const int urow = it.dense ? tile * 64 : it.e * (2 * I) + I + tile * 64;
                tma_load_2d(a_dst + a * kAChunk, mg, &full_bar[stage], k0, grow, pol_w);
                tma_load_2d(a_dst + a * kAChunk + kAChunk / 2, mu, &full_bar[stage], k0, urow, pol_w);
              } else {
                const CUtensorMap* mp = it.dense ? &map_a_d0 : &map_a_exp;
                const int arow = it.dense ? tile * kBM : it.e * H + tile * kBM;
                tma_load_2d(a_dst + a * kAChunk, mp, &full_bar[stage], k0, arow, pol_w);
              }
            }
            if (b_tma) {
              const CUtensorMap* mb = it.dense ? &map_b_dense : &map_b_exp;
              tma_load_2d(a_dst + C::kAStage, mb, &full_bar[stage], k0, it.row0, pol_x);
            }
          }
        }
        __syncwarp();
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    // Before the CTA can exit, every TMA load this warp issued must have landed.
    if (lane == 0)
      for (int s2 = 0; s2 < C::kStages; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&full_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs, b.status);
    __syncwarp();
  } else if (warp == 1 || (CVT && warp == C::kMma2Warp)) {
    // ---------------- MMA issuer (one thread; CVT: two, issuer j taking the item's K chunks with
    // index parity j, each into its own partial accumulator, which the epilogue adds in that order)
    if (lane == 0) {
      const int mi = warp == 1 ? 0 : 1;
      int stage = 0;
      uint32_t phase = 0;
      int acc = 0;
      uint32_t acc_phase = 0;
      int aslot = 0;  // CVT: TMEM A ring
      uint32_t aphase = 0;
      bool ok = true;
      int slot = 0;
      uint32_t slot_par = 0;
      while (ok) {
        const int i = next_item(itemf_bar, iteme_bar, item_s, slot, slot_par, abort_flag, b.status);
        if (i < 0) break;
        const int nch = (i < n_dense_items) ? C::kChunksDense : C::kChunksExp;
        if (!mbar_wait_bounded(&acce_bar[acc], acc_phase ^ 1u, abort_flag, b.status, kStatusWaitAccEmpty)) break;
        tc_fence_after();
        const uint32_t d_tmem =
            tmem_base + static_cast<uint32_t>((acc * C::kIssuers + mi) * C::kAccCols);
        uint32_t idesc = 0;
        int na = 1;
        bool first = true;  // this issuer's first chunk of the item
        for (int c0 = 0; c0 < nch; c0 += C::KC) {
          const bool mine = C::kIssuers == 1 || (c0 & 1) == mi;
          if (mine) {
            if (!mbar_wait_bounded(&full_bar[stage], phase, abort_flag, b.status, kStatusWaitFull)) {
              ok = false;
              break;
            }
            if (CVT && !mbar_wait_bounded(&af_bar[aslot], aphase, abort_flag, b.status, kStatusWaitFull)) {
              ok = false;
              break;
            }
            // The gathered B rows were written by cp.async (generic proxy); the MMA reads them
            // through the async proxy.
            if (GATE_UP || CVT) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            tc_fence_after();
            // The MMA is only as wide as the tile's token rows (rounded up to the MMA's step of 16).
            if (first) {
              const int ws = width_s[stage];
              idesc = idesc_bf16_f32(kBM, ws & 0xFFFF);
              na = ws >> 16;
            }
            const int nck = min(C::KC, nch - c0);
            const uint32_t st = smem_u32(stages + stage * C::kStageBytes);
            for (int cc = 0; cc < nck; ++cc) {
              const uint64_t b_desc = smem_desc_sw128(st + cc * C::kChunkBytes + C::kAStage);
              if constexpr (CVT) {
                const uint32_t a_tm = tmem_base + static_cast<uint32_t>(C::kACol0 + aslot * 32);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                  umma_bf16_ta(d_tmem, a_tm + 8u * k, b_desc + 2u * k, idesc, (first && k == 0) ? 0u : 1u);
              } else {
#pragma unroll
                for (int a = 0; a < MA; ++a) {
                  if (a >= na) break;
                  const uint64_t a_desc = smem_desc_sw128(st + cc * C::kChunkBytes + a * kAChunk);
#pragma unroll
                  for (int k = 0; k < kBK / 16; ++k)
                    umma_bf16(d_tmem + static_cast<uint32_t>(a * BN), a_desc + 2u * k, b_desc + 2u * k, idesc,
                              (c0 | cc | k) != 0 ? 1u : 0u);
                }
              }
            }
            first = false;
            umma_commit(&empty_bar[stage]);
            if (CVT) umma_commit(&ae_bar[aslot]);
          }
          if (CVT && ++aslot == C::kASlots) {
            aslot = 0;
            aphase ^= 1u;
          }
          if (++stage == C::kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&accf_bar[acc]);
        if (++acc == C::kNAcc) {
          acc = 0;
          acc_phase ^= 1u;
        }
      }
      // All MMAs issued above complete before this barrier's phase does.
      umma_commit(final_bar);
      mbar_wait_timeout(final_bar, 0, kSpinLimitNs, b.status);
    }
    __syncwarp();
  } else if (warp < C::kGatherWarp0) {
    // ---------------- epilogue warps 2..; TMEM lane quarter = warp % 4, weight tile (warp - 2) / 4
    const int q = warp & 3;
    const int ta = (warp - 2) >> 2;
    float* xw = xchg + (ta * 4) * (GATE_UP ? 512 : 1024);  // this tile's four hand-over slots
    int acc = 0;
    uint32_t acc_phase = 0;
    int slot = 0;
    uint32_t slot_par = 0;
    for (;;) {
      const int i = warp_next_item(itemf_bar, iteme_bar, item_s, slot, slot_par, abort_flag, b.status);
      if (i < 0) break;
      const Item it = decode_item<BN, GATE_UP, MA>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const int tile = it.m * MA + ta;
      const int n_tiles_raw = it.dense ? C::kTilesDense : C::kTilesExp;
      const bool has_tile = tile < n_tiles_raw;
      const bool paired = GATE_UP && MA == 2 && it.m * MA + 1 < n_tiles_raw;
      if (!warp_wait(&accf_bar[acc], acc_phase, abort_flag, b.status, kStatusWaitAccFull)) break;
      tc_fence_after();
      if (paired) {
        // Gate (tile 0) and up (tile 1) of features f + lane sit in this warp's own TMEM lanes;
        // the two warps of a lane quarter split the token columns.
        const int f = it.m * 128 + 32 * q;
        const uint32_t t_g = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * C::kIssuers * C::kAccCols);
        uint16_t* hs = reinterpret_cast<uint16_t*>(xw + q * 512);  // [32 columns][32 features] bf16
        uint16_t* dst = it.dense ? b.h_dense : b.h;
        const int ld = it.dense ? D : I;
#pragma unroll 1
        for (int c = ta * (BN / 64); c < (ta + 1) * (BN / 64); ++c) {
          if (c * 32 >= it.rows) break;
          uint32_t g[32], u[32];
          tmem_ld32_nowait(t_g + c * 32, g);
          tmem_ld32_nowait(t_g + BN + c * 32, u);
          tmem_wait_ld();
          reg_fence32(g);
          reg_fence32(u);
#pragma unroll
          for (int j = 0; j < 32; ++j)
            hs[j * 32 + lane] = f32_to_bf16_rn(gelu_tanh_approx(__uint_as_float(g[j])) * __uint_as_float(u[j]));
          __syncwarp();
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int idx = lane + 32 * i, r = idx >> 2, c8 = idx & 3;
            const int col = c * 32 + r;
            if (col < it.rows)
              *reinterpret_cast<uint4*>(dst + static_cast<size_t>(it.row0 + col) * ld + f + 8 * c8) =
                  *reinterpret_cast<const uint4*>(hs + r * 32 + 8 * c8);
          }
          __syncwarp();
        }
      }
      const uint32_t t_row = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * C::kIssuers * C::kAccCols + ta * BN);
      // CVT: this lane's weight row's scale (gate_up: lanes 0..63 gate rows, 64..127 up rows).
      float row_scale = 1.0f;
      if (CVT && !F4 && !it.dense && has_tile) {
        const size_t row = GATE_UP ? static_cast<size_t>(it.e) * (2 * I) + (q < 2 ? 0 : I) + tile * 64 + 32 * (q & 1) + lane
                                   : static_cast<size_t>(it.e) * H + tile * kBM + 32 * q + lane;
        row_scale = __ldg(static_cast<const float*>(q_scale) + row);
      }
#pragma unroll 1
      for (int c = 0; c < BN / 32; ++c) {
        if (paired || !has_tile || c * 32 >= it.rows) break;
        float v[32];
        tmem_ld32(t_row + c * 32, v);
        if (CVT) {
          // The second issuer's partial sum (the item's odd K chunks), added in a fixed order.
#pragma unroll
          for (int hf = 0; hf < 2; ++hf) {
            float v2[16];
            tmem_ld16(t_row + static_cast<uint32_t>(C::kAccCols + c * 32 + 16 * hf), v2);
#pragma unroll
            for (int j = 0; j < 16; ++j) v[16 * hf + j] += v2[j];
          }
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] *= row_scale;
        }
        if (GATE_UP) {
          // q 0/1: gate of features f0+32(q&1)+lane; q 2/3: up of the same features.
          const bool gate_holder = q < 2;
          const int pairbar = 1 + (q & 1) + 2 * ta;
          float* mine = xw + q * 512;
          const float* theirs = xw + (q ^ 2) * 512;
          // The gate holder hands over columns 16..31 and finishes 0..15; the up holder the reverse.
#pragma unroll
          for (int j = 0; j < 16; ++j) mine[j * 32 + lane] = gate_holder ? v[16 + j] : v[j];
          named_bar_sync(pairbar, 64);
          uint16_t* dst = it.dense ? b.h_dense : b.h;
          const int ld = it.dense ? D : I;
          const int keep = gate_holder ? 0 : 16;
          float hv[16];
#pragma unroll
          for (int j = 0; j < 16; ++j) {
            const float other = theirs[j * 32 + lane];
            const float own = gate_holder ? v[j] : v[16 + j];
            const float g = gate_holder ? own : other;
            const float u = gate_holder ? other : own;
            hv[j] = gelu_tanh_approx(g) * u;
          }
          named_bar_sync(pairbar, 64);
          // h of 16 token columns x the warp's 32 features goes through shared memory (the warp's
          // own hand-over slot, free again) so that the global stores are 16-byte vectors.
          uint16_t* hs = reinterpret_cast<uint16_t*>(mine);  // [16 columns][32 features]
#pragma unroll
          for (int j = 0; j < 16; ++j) hs[j * 32 + lane] = f32_to_bf16_rn(hv[j]);
          __syncwarp();
          const int f0 = tile * 64 + 32 * (q & 1);
#pragma unroll
          for (int i = 0; i < 2; ++i) {
            const int idx = lane + 32 * i, r = idx >> 2, c8 = idx & 3;
            const int col = c * 32 + keep + r;
            if (col < it.rows)
              *reinterpret_cast<uint4*>(dst + static_cast<size_t>(it.row0 + col) * ld + f0 + 8 * c8) =
                  *reinterpret_cast<const uint4*>(hs + r * 32 + 8 * c8);
          }
          __syncwarp();
        } else {
          // The warp's 32 features x 32 token columns go through shared memory so that the global
          // stores are 16-byte vectors along the feature dimension.
          const int f0 = tile * kBM + 32 * q;
          uint8_t* stg = reinterpret_cast<uint8_t*>(xw) + q * 4096;
          if (it.dense) {
            uint16_t* sd = reinterpret_cast<uint16_t*>(stg);  // [32 tokens][32 features] bf16
#pragma unroll
            for (int j = 0; j < 32; ++j) sd[j * 32 + lane] = f32_to_bf16_rn(v[j]);
            __syncwarp();
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const int idx = lane + 32 * i, r = idx >> 2, c8 = idx & 3;
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
            for (int i = 0; i < 4; ++i) {
              const int idx = lane + 32 * i, r = idx >> 2, c8 = idx & 3;
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
      if (lane == 0) mbar_arrive(&acce_bar[acc]);
      if (++acc == C::kNAcc) {
        acc = 0;
        acc_phase ^= 1u;
      }
    }
  } else if (warp < C::kConvWarp0) {
    // ---------------- gather warps (gate_up only): expert token rows of n2 by cp.async
    const int g = threadIdx.x - C::kGatherWarp0 * 32;  // 0..127
    const int chunk16 = g & 7;               // which 16 bytes of the 128-byte row
    const int rbase = g >> 3;                // rows rbase, rbase+16, ...
    int stage = 0;
    uint32_t phase = 0;
    bool ok = true;
    int slot = 0;
    uint32_t slot_par = 0;
    while (ok) {
      const int i = warp_next_item(itemf_bar, iteme_bar, item_s, slot, slot_par, abort_flag, b.status);
      if (i < 0) break;
      const Item it = decode_item<BN, GATE_UP, MA>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
      int src[BN / 16];
#pragma unroll
      for (int r = 0; r < BN / 16; ++r) {
        const int j = rbase + 16 * r;
        int t = -1;
        if (!it.dense && j < it.rows) {
          t = b.perm[it.row0 + j];
          if (t < 0 || t >= T) {
            atomicOr(b.status, kStatusBadIndex);
            t = 0;
          }
        }
        src[r] = t;
      }
      for (int c0 = 0; c0 < nch; c0 += C::KC) {
        if (!warp_wait(&empty_bar[stage], phase ^ 1u, abort_flag, b.status, kStatusWaitEmpty)) {
          ok = false;
          break;
        }
        if (!it.dense) {
          const int nck = min(C::KC, nch - c0);
          const uint32_t st = smem_u32(stages + stage * C::kStageBytes);
          for (int cc = 0; cc < nck; ++cc) {
            const uint32_t b_dst = st + cc * C::kChunkBytes + C::kAStage;
            const int k0 = (c0 + cc) * kBK;
#pragma unroll
            for (int r = 0; r < BN / 16; ++r) {
              const int j = rbase + 16 * r;
              if (src[r] >= 0) {
                const uint16_t* s = b.n2 + static_cast<size_t>(src[r]) * H + k0 + chunk16 * 8;
                cp_async16(b_dst + j * 128 + ((chunk16 ^ (j & 7)) << 4), s);
              }
            }
          }
        }
        cp_async_arrive_noinc(&full_bar[stage]);
        if (++stage == C::kStages) {
          stage = 0;
          phase ^= 1u;
        }
      }
    }
    cp_async_wait_all();
  } else if (warp < C::kRawWarp) {
    // ---------------- converters (CVT): weight rows from the raw ring into the TMEM A ring. Group g
    // (warps 4g..4g+3 of the eight) takes the item's K chunks with index parity g, so two chunks are
    // in flight; each warp covers the TMEM lane quarter it may access (warp % 4), one weight row per
    // lane, the chunk's 64 K elements per row. A raw slot holds cps chunks of every row (int8 2,
    // MXFP4 4, the shared MLP's bf16 1); each warp releases it after the last of its chunks there.
    const int grp = (warp - C::kConvWarp0) >> 2;
    const int q = warp & 3;
    const int row = 32 * q + lane;
    const int sw = row & 7;
    const uint32_t t_lane = tmem_base + (static_cast<uint32_t>(32 * q) << 16) + static_cast<uint32_t>(C::kACol0);
    int r = 0, as = 0;
    uint32_t rphase = 0, aphase = 0;
    bool ok = true;
    int slot = 0;
    uint32_t slot_par = 0;
    while (ok) {
      const int i = warp_next_item(itemf_bar, iteme_bar, item_s, slot, slot_par, abort_flag, b.status);
      if (i < 0) break;
      const Item it = decode_item<BN, GATE_UP, MA>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
      const bool cvt = !it.dense;  // the experts' converted rows; the shared MLP's rows are bf16
      const int cps = cvt ? C::kExpChunksPerSlot : 1;
      // MXFP4: this row's E8M0 scales, two per K chunk (blocks of 32).
      const uint8_t* srow = nullptr;
      if (F4 && cvt) {
        const size_t grow = GATE_UP ? static_cast<size_t>(it.e) * (2 * I) + (row < 64 ? 0 : I) + it.m * 64 + (row & 63)
                                    : static_cast<size_t>(it.e) * H + it.m * kBM + row;
        srow = static_cast<const uint8_t*>(q_scale) + grow * (GATE_UP ? H / 32 : I / 32);
      }
      // The scales of this group's next chunk are loaded one chunk ahead.
      uint32_t sc_next = 0;
      if (F4 && cvt && grp < nch) sc_next = __ldg(reinterpret_cast<const unsigned short*>(srow + 2 * grp));
      for (int c = 0; c < nch; ++c) {
        const int slot_lo = c - c % cps;
        const int slot_hi = min(slot_lo + cps, nch);
        const int j = c - slot_lo;  // chunk within the slot
        if ((c & 1) == grp) {
          const uint32_t sc2 = sc_next;
          if (F4 && cvt && c + 2 < nch) sc_next = __ldg(reinterpret_cast<const unsigned short*>(srow + 2 * (c + 2)));
          if (!warp_wait(&ae_bar[as], aphase ^ 1u, abort_flag, b.status, kStatusWaitEmpty) ||
              !warp_wait(&rawf_bar[r], rphase, abort_flag, b.status, kStatusWaitFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint8_t* src = raw_ring + r * C::kRawSlotBytes + row * 128;
          uint32_t o[32];
          if (cvt && !F4) {
            // 16 int8 per piece, widened exactly: with u = q + 128 (the byte with its top bit
            // flipped), the fp32 word 0x4B000000 | u is 2^23 + u, so subtracting 2^23 + 128 gives q;
            // |q| < 256 leaves the low 16 bits zero, so the high halves are the bf16 values.
#pragma unroll
            for (int p = 0; p < 4; ++p) {
              const uint4 v = *reinterpret_cast<const uint4*>(src + (((4 * j + p) ^ sw) << 4));
              const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {
                const uint32_t wx = w4[jj >> 1] ^ 0x80808080u;
                const uint32_t k0 = (jj & 1) * 2;
                const float q0 = __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | k0)) - 8388736.0f;
                const float q1 = __uint_as_float(__byte_perm(wx, 0x4B000000u, 0x7540u | (k0 + 1))) - 8388736.0f;
                o[8 * p + jj] = __byte_perm(__float_as_uint(q0), __float_as_uint(q1), 0x7632u);
              }
            }
          } else if (cvt) {
            // 64 E2M1 codes (32 bytes), four per 16-bit half word. For each block scale 2^(e - 127)
            // the eight scaled bf16 values (0 and 0.5, 1, 1.5, 2, 3, 4, 6 times the scale: their
            // bf16 bits plus (e - 127) << 7, exact for e in 2..252) are split into a table of high
            // bytes and one of low bytes; each code's 3-bit magnitude selects from both by
            // byte_perm, the sign goes to the top bit of the high byte, and two more byte_perms
            // interleave the bytes into bf16 pairs.
            uint32_t thx[2], thy[2], tlx[2], tly[2];
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const int off = static_cast<int>((sc2 >> (8 * hf)) & 0xFFu) - 127;
              const uint32_t o1 = static_cast<uint32_t>(off) << 7;   // added to one 16-bit value
              const uint32_t o2 = o1 * 0x10001u;                       // added to both halves
              const uint32_t A = 0x3F000000u + (o1 << 16);             // values 0 (kept 0) and 0.5
              const uint32_t Bv = 0x3FC03F80u + o2;                    // 1, 1.5
              const uint32_t Cv = 0x40404000u + o2;                    // 2, 3
              const uint32_t Dv = 0x40C04080u + o2;                    // 4, 6
              thx[hf] = __byte_perm(A, Bv, 0x7531u);
              tlx[hf] = __byte_perm(A, Bv, 0x6420u);
              thy[hf] = __byte_perm(Cv, Dv, 0x7531u);
              tly[hf] = __byte_perm(Cv, Dv, 0x6420u);
            }
#pragma unroll
            for (int p = 0; p < 2; ++p) {
              const uint4 v = *reinterpret_cast<const uint4*>(src + (((2 * j + p) ^ sw) << 4));
              const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
              for (int jj = 0; jj < 8; ++jj) {  // 16-bit halves of the piece: four codes each
                const uint32_t h = w4[jj >> 1] >> (16 * (jj & 1));
                const uint32_t sel = h & 0x7777u;
                const uint32_t sgn = __byte_perm(0u, 0x80u, (h >> 1) & 0x4444u);  // 0x80 in byte k if code k < 0
                const uint32_t hb = __byte_perm(thx[p], thy[p], sel) | sgn;
                const uint32_t lb = __byte_perm(tlx[p], tly[p], sel);
                const int oi = 16 * p + 2 * jj;  // output word: elements 2 oi, 2 oi + 1
                o[oi] = __byte_perm(lb, hb, 0x5140u);
                o[oi + 1] = __byte_perm(lb, hb, 0x7362u);
              }
            }
          } else {
            // bf16 rows: two K elements per 32-bit word already, the lower K in the low half.
#pragma unroll
            for (int p = 0; p < 8; ++p) {
              const uint4 v = *reinterpret_cast<const uint4*>(src + ((p ^ sw) << 4));
              o[4 * p] = v.x;
              o[4 * p + 1] = v.y;
              o[4 * p + 2] = v.z;
              o[4 * p + 3] = v.w;
            }
          }
          tmem_st32(t_lane + static_cast<uint32_t>(as * 32), o);
          tmem_wait_st();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&af_bar[as]);
            // Release the slot after this warp's last chunk in it; a slot with a single chunk is
            // read by one group only, which then counts for both.
            if (c + 2 >= slot_hi) mbar_arrive_n(&rawe_bar[r], slot_hi - slot_lo >= 2 ? 1u : 2u);
          }
        }
        if (++as == C::kASlots) {
          as = 0;
          aphase ^= 1u;
        }
        if (c + 1 == slot_hi && ++r == C::kRawSlots) {
          r = 0;
          rphase ^= 1u;
        }
      }
    }
  } else {
    // ---------------- weight-row producer (CVT): the experts' rows (128 bytes of each per slot: two
    // int8 or four MXFP4 K chunks) and the shared MLP's bf16 rows (one K chunk per slot)
    const uint64_t pol_once = policy_evict_first();
    const uint64_t pol_keep = policy_evict_last();
    int r = 0;
    uint32_t rphase = 0;
    uint32_t armed = 0, armed_par = 0;
    bool ok = true;
    int slot = 0;
    uint32_t slot_par = 0;
    while (ok) {
      const int i = warp_next_item(itemf_bar, iteme_bar, item_s, slot, slot_par, abort_flag, b.status);
      if (i < 0) break;
      const Item it = decode_item<BN, GATE_UP, MA>(i, n_dense_tiles, b.exp_tiles, tile_off_s, T);
      const uint64_t pol = it.nt > 2 ? pol_keep : pol_once;
      const int nch = it.dense ? C::kChunksDense : C::kChunksExp;
      const int nslots = it.dense ? nch : (nch + C::kExpChunksPerSlot - 1) / C::kExpChunksPerSlot;
      for (int sidx = 0; sidx < nslots; ++sidx) {
        if (!warp_wait(&rawe_bar[r], rphase ^ 1u, abort_flag, b.status, kStatusWaitEmpty)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          armed |= 1u << r;
          armed_par = (armed_par & ~(1u << r)) | (rphase << r);
          mbar_arrive_expect_tx(&rawf_bar[r], C::kRawSlotBytes);
          uint8_t* dst = raw_ring + r * C::kRawSlotBytes;
          if (it.dense) {
            const int k0 = sidx * kBK;
            if (GATE_UP) {
              tma_load_2d(dst, &map_a_d0, &rawf_bar[r], k0, it.m * 64, pol);
              tma_load_2d(dst + 64 * 128, &map_a_d1, &rawf_bar[r], k0, it.m * 64, pol);
            } else {
              tma_load_2d(dst, &map_a_d0, &rawf_bar[r], k0, it.m * kBM, pol);
            }
          } else {
            const int x0 = sidx * 128;  // 128 bytes of each row: 2 int8 or 4 MXFP4 K chunks
            if (GATE_UP) {
              tma_load_2d(dst, &map_q, &rawf_bar[r], x0, it.e * (2 * I) + it.m * 64, pol);
              tma_load_2d(dst + 64 * 128, &map_q, &rawf_bar[r], x0, it.e * (2 * I) + I + it.m * 64, pol);
            } else {
              tma_load_2d(dst, &map_q, &rawf_bar[r], x0, it.e * H + it.m * kBM, pol);
            }
          }
        }
        __syncwarp();
        if (++r == C::kRawSlots) {
          r = 0;
          rphase ^= 1u;
        }
      }
    }
    // Every load issued above must have landed before the CTA exits.
    if (lane == 0)
      for (int s2 = 0; s2 < C::kRawSlots; ++s2)
        if (armed & (1u << s2)) mbar_wait_timeout(&rawf_bar[s2], (armed_par >> s2) & 1u, kSpinLimitNs, b.status);
    __syncwarp();
  }

  tc_fence_before();
  __syncthreads();
  if (!early_dependents) pdl_launch_dependents();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, C::kTmemCols);
  }
}

template <int BN, bool GATE_UP, int MA, int QW = kWBf16>
cudaError_t launch_t(const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid, cudaStream_t s) {
  using C = Cfg<BN, GATE_UP, MA, QW>;
  return launch_pdl(grouped_gemm_kernel<BN, GATE_UP, MA, QW>, dim3(grid), dim3(C::kThreads), C::kSmem, s, m.a_exp,
                    m.a_dense0, m.a_dense1, m.b_exp, m.b_dense, b, T, full_layer, m.a_q, m.q_scale);
}

template <int BN, bool GATE_UP, int MA, int QW = kWBf16>
cudaError_t set_limit() {
  using C = Cfg<BN, GATE_UP, MA, QW>;
  return cudaFuncSetAttribute(grouped_gemm_kernel<BN, GATE_UP, MA, QW>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmem);
}

}  // namespace

// Weight tiles per work item of the gate_up GEMM: two for wide token tiles (T above 512), where
// the operand traffic per FLOP and the epilogue's gate/up hand-over cost more than the longer
// items do; one for decode-sized T, where the weight stream is the bound and more, shorter items
// balance better over the SMs. (Two tiles per item were measured slower for the down GEMM, whose
// short K leaves a single-buffered accumulator's epilogue exposed.)
int gate_up_tiles_per_item(int bn, int T) { return bn == 256 || (bn == 128 && T > 512) ? 2 : 1; }

cudaError_t gemm_set_smem_limits() {
  cudaError_t e;
  if ((e = set_limit<32, true, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<64, true, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<128, true, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<128, true, 2>()) != cudaSuccess) return e;
  if ((e = set_limit<256, true, 2>()) != cudaSuccess) return e;
  if ((e = set_limit<32, false, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<64, false, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<128, false, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<256, false, 1>()) != cudaSuccess) return e;
  if ((e = set_limit<32, true, 1, kWInt8>()) != cudaSuccess) return e;
  if ((e = set_limit<64, true, 1, kWInt8>()) != cudaSuccess) return e;
  if ((e = set_limit<32, false, 1, kWInt8>()) != cudaSuccess) return e;
  if ((e = set_limit<64, false, 1, kWInt8>()) != cudaSuccess) return e;
  if ((e = set_limit<32, true, 1, kWFp4>()) != cudaSuccess) return e;
  if ((e = set_limit<64, true, 1, kWFp4>()) != cudaSuccess) return e;
  if ((e = set_limit<32, false, 1, kWFp4>()) != cudaSuccess) return e;
  return set_limit<64, false, 1, kWFp4>();
}

// Converted experts (token tiles of 32 or 64): m.a_q maps the int8 rows or MXFP4 codes, m.q_scale holds
// the int8 row scales or the MXFP4 block scales.
cudaError_t launch_gate_up_cvt(int bn, bool fp4, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                              cudaStream_t s) {
  switch (bn * 2 + (fp4 ? 1 : 0)) {
    case 64: return launch_t<32, true, 1, kWInt8>(m, b, T, full_layer, grid, s);
    case 128: return launch_t<64, true, 1, kWInt8>(m, b, T, full_layer, grid, s);
    case 65: return launch_t<32, true, 1, kWFp4>(m, b, T, full_layer, grid, s);
    case 129: return launch_t<64, true, 1, kWFp4>(m, b, T, full_layer, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_down_cvt(int bn, bool fp4, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                           cudaStream_t s) {
  switch (bn * 2 + (fp4 ? 1 : 0)) {
    case 64: return launch_t<32, false, 1, kWInt8>(m, b, T, full_layer, grid, s);
    case 128: return launch_t<64, false, 1, kWInt8>(m, b, T, full_layer, grid, s);
    case 65: return launch_t<32, false, 1, kWFp4>(m, b, T, full_layer, grid, s);
    case 129: return launch_t<64, false, 1, kWFp4>(m, b, T, full_layer, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_gate_up(int bn, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                           cudaStream_t s) {
  switch (bn) {
    case 32: return launch_t<32, true, 1>(m, b, T, full_layer, grid, s);
    case 64: return launch_t<64, true, 1>(m, b, T, full_layer, grid, s);
    case 128: return gate_up_tiles_per_item(bn, T) == 2 ? launch_t<128, true, 2>(m, b, T, full_layer, grid, s)
                                                        : launch_t<128, true, 1>(m, b, T, full_layer, grid, s);
    case 256: return launch_t<256, true, 2>(m, b, T, full_layer, grid, s);  // two tiles per item
    default: return cudaErrorInvalidValue;
  }
}

cudaError_t launch_down(int bn, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                        cudaStream_t s) {
  switch (bn) {
    case 32: return launch_t<32, false, 1>(m, b, T, full_layer, grid, s);
    case 64: return launch_t<64, false, 1>(m, b, T, full_layer, grid, s);
    case 128: return launch_t<128, false, 1>(m, b, T, full_layer, grid, s);
    case 256: return launch_t<256, false, 1>(m, b, T, full_layer, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace moe
