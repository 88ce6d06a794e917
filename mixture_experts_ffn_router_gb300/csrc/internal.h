// internal.h — declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstdint>

namespace moe {

constexpr int H = 2816;   // hidden
constexpr int E = 128;    // experts
constexpr int K = 8;      // experts per token
constexpr int I = 704;    // expert intermediate width
constexpr int D = 2112;   // shared-MLP intermediate width

// Router kernel: 128 tokens per CTA (the MMA's N), the hidden dimension split into `ks` parts.
constexpr int kRouterN = 128;
// Token-scatter kernel: 256 tokens per CTA (8 warps of 32).
constexpr int kScatterTok = 256;
// Combine kernel: one CTA per token, 352 threads x 8 features.
constexpr int kCombineThreads = 352;

// Device pointers of one forward's intermediates, carved from the caller's workspace.
struct Buffers {
  float* logits_part;   // [ks, T, 128]
  float* logits;        // [Tm, 128]
  int32_t* topk_idx;    // [Tm, 8]
  float* topk_w;        // [Tm, 8]
  float* gap;           // [Tm]
  int32_t* hist;        // [kMaxRouteBlocks, 128] expert counts per 256-token chunk
  int32_t* base;        // [kMaxRouteBlocks, 128] first sorted position of each (chunk, expert)
  int32_t* counts;      // [128]
  int32_t* offsets;     // [129]
  int32_t* n_exp_tiles; // [1]
  int32_t* done_ctr;    // [1]
  int32_t* sched;       // [3] work-item counters of the gate_up and down GEMMs, and the count of
                        // warps that finished the sorted copy of n2 (all zeroed by top-k)
  int32_t* small_ctr;   // [8] tickets of the small-batch routing kernel (zero between forwards)
  int4* exp_tiles;      // [max_tiles] (expert, first sorted row, rows, 0), grouped by expert
  int32_t* tile_off;    // [129] index of each expert's first token tile in exp_tiles
  int32_t* perm;        // [S]
  float* w_sorted;      // [S]
  int32_t* slot_pos;    // [Tm, 8]
  uint16_t* n1;         // [Tm, 2816]
  uint16_t* n2;         // [Tm, 2816]
  uint16_t* h;          // [S, 704]
  uint16_t* h_dense;    // [Tm, 2112]
  uint16_t* y;          // [S, 2816] bf16
  uint16_t* n2s;        // [S, 2816] bf16: n2 rows in sorted-slot order (T > kPairGateUpT), aliases y
  uint16_t* d;          // [Tm, 2816] bf16
  unsigned int* status; // [1]
  uint16_t* wsplit;     // [3, 128, 2816] bf16: W_r * (1 + router_norm_w) as hi + mid + lo
  int max_tiles;
};

constexpr int kMaxRouteBlocks = 256;  // 256-token chunks: 65536 tokens at most

struct RouteParams {
  const uint16_t* x;
  const float* router_w;
  const float* router_norm_w;
  const float* per_expert_scale;
  const float* pre_ff_ln;
  const float* pre_ff_ln_2;
  int T;
  int ks;               // K splits of the router projection
  int tpw;              // tokens per warp in the top-k kernel
  int bn;               // token-tile width of the grouped GEMMs
  int full_layer;
  int write_n2;         // the top-k kernel writes n2 (token order); else the gate_up GEMM writes n2s
  int e_lo, e_hi;       // the experts whose token tiles the GEMMs compute: [0, 128), or a shard's
  float eps;
  float router_scale;
};

struct CombineParams {
  const uint16_t* x;
  const float* post_ff_ln_1;
  const float* post_ff_ln_2;
  const float* post_ff_ln;
  float layer_scalar;
  uint16_t* out;
  int T;
  int full_layer;
  float eps;
};

// The end of an expert-parallel shard forward: the fp32 sum of each token's weighted expert
// outputs over the experts [e_lo, e_hi), and optionally the shared-MLP output widened to fp32.
struct ShardParams {
  int T;
  int e_lo, e_hi;
  float* moe_out;    // [T, 2816]
  float* dense_out;  // [T, 2816] or NULL
};

// Maps of one grouped GEMM launch. For gate_up: a_exp = gate_up rows, a_dense0/1 = dense gate/up,
// b_dense = n1 (BN-row boxes; the experts' rows are gathered with cp.async, b_exp is unused). For
// down: a_exp = down rows, a_dense0 = dense down, b_exp = h, b_dense = h_dense (BN-row boxes).
struct GemmMaps {
  CUtensorMap a_exp, a_dense0, a_dense1, b_exp, b_dense;
  CUtensorMap a_q;         // converted expert weights: int8 rows, or packed MXFP4 codes
  const void* q_scale;     // int8: fp32 row scales; MXFP4: E8M0 block scales [rows, K / 32]
};

// Launches a kernel with programmatic dependent launch: its CTAs may start while the previous
// kernel on the stream finishes; every kernel here calls griddepcontrol.wait before it touches
// memory the previous kernels write or read.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                              Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// The same for kernels that run as clusters of two CTAs (SM pairs); grid.x must be even.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_pair(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                   Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}

// Kernel slots of one forward (events, breakdown): 0 router prep, 1 router logits, 2 top-k,
// 3 scatter, 4 gate_up, 5 down, 6 combine.
constexpr int kKernelsPerForward = 7;
// Above kPairGateUpT tokens (token tiles of 256) the gate_up GEMM runs on SM pairs and takes its
// expert rows from a copy of n2 in sorted-slot order, loaded by TMA boxes, instead of gathering them
// by token index; it writes that copy itself before its first expert item. From 1025 tokens (tiles
// of 256) up to kPairGateUpT it stays on single SMs with gathered token rows, where the copy's cost
// is not yet repaid. Layer time, uniform routing, single SMs vs pairs: T = 1500 372.5 vs 384.3 us,
// 2048 402.9 vs 415.2, 2560 448.1 vs 456.0, 3072 474.8 vs 479.3, 4096 636.0 vs 621.6.
constexpr int kPairGateUpT = 3072;
// Batches of at most kRouteSmallT tokens take the router's sums on CUDA cores, with the top-k and
// the counting sort in the same kernel (route_small_kernel).
constexpr int kRouteSmallT = 64;
// Largest batch for which the down GEMM lets the combine kernel launch before it ends.
constexpr int kEarlyCombineT = 64;
cudaError_t launch_route_small(const RouteParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_router_prep(const RouteParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_router_logits(const CUtensorMap& map_w, const RouteParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_route_topk(const RouteParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_route_scatter(const RouteParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_combine(const CombineParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_combine_shard(const ShardParams& p, const Buffers& b, cudaStream_t s);
cudaError_t launch_finish(const CombineParams& p, const float* moe_sum, const float* dense, cudaStream_t s);

// Grouped GEMMs (gemm.cu). `grid` CTAs persistent over the device-side tile list.
cudaError_t launch_gate_up(int bn, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                           cudaStream_t s);
cudaError_t launch_down(int bn, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                        cudaStream_t s);
cudaError_t gemm_set_smem_limits();
int gate_up_tiles_per_item(int bn, int T);
cudaError_t launch_gate_up_cvt(int bn, bool fp4, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                              cudaStream_t s);
cudaError_t launch_down_cvt(int bn, bool fp4, const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid,
                           cudaStream_t s);
// The inputs of the sorted copy of n2 that the SM-pair gate_up GEMM writes: the layer input, the
// expert branch's pre-norm weight (NULL in the experts-only mode, where n2 = x) and epsilon.
struct PermIn {
  const uint16_t* x;
  const float* w2;
  float eps;
  int e_lo, e_hi;  // only the slots of these experts are copied (a shard's range, or all)
};

// SM-pair (cta_group::2) gate_up and down GEMMs for token tiles of 256 (gemm_pair.cu).
cudaError_t gemm_pair_set_smem_limits();
int gemm_pair_max_clusters();
cudaError_t launch_gate_up_pair(const GemmMaps& m, const Buffers& b, const PermIn& pin, int T, int full_layer, int grid,
                                cudaStream_t s);
cudaError_t launch_down_pair(const GemmMaps& m, const Buffers& b, int T, int full_layer, int grid, cudaStream_t s);
cudaError_t router_set_smem_limit();

}  // namespace moe
