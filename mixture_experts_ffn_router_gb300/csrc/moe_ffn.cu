// moe_ffn.cu — host side of the library: the C ABI of include/moe_ffn.h, workspace layout,
// TMA tensor maps and the launch sequence of one forward.
//
// One forward of T tokens queues seven kernels on the caller's stream (programmatic dependent
// launch, so each one's launch and prologue overlap the previous one's tail), in this order:
//   0 router prep     W_r * (1 + router_norm_w) split into three bf16 parts
//   1 router logits   fp32-accurate partial projections on the tensor cores ("The
//                     architecture": own RMSNorm, a scale, softmax over 128 experts in fp32)
//   2 top-k           RMS of x, the pre-norms, softmax, top-8, renormalise, per_expert_scale,
//                     expert counts per 256-token chunk -> offsets, bases and the token-tile list
//   3 scatter         stable counting-sort scatter of the 8T slots by expert
//   4 gate_up GEMM    tcgen05 grouped GEMM, h = gelu_tanh(gate) * up (experts + shared MLP)
//   5 down GEMM       tcgen05 grouped GEMM, y = w * down(h) (experts), d = down(h) (shared MLP)
//   6 combine         per token: sum of its 8 y rows, the post-norms, residual, layer_scalar
// Nothing is read back to the host; the GEMMs size their work from device-side counts.
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "moe_ffn.h"
#include "internal.h"

using namespace moe;

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn lookup_encode() {
  void* p = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return reinterpret_cast<EncodeTiledFn>(p);
  return nullptr;
}

// The driver's tensor-map encoder, looked up once. A function-local static with an initialiser is
// initialised exactly once even when several host threads get here first at the same time
// (moe_ffn_init and the allocation-free entry point may run on different threads).
EncodeTiledFn get_encode() {
  static const EncodeTiledFn fn = lookup_encode();
  return fn;
}

// bf16 matrix [rows, cols] row-major, boxes of 64 columns x box_rows rows, 128-byte swizzle.
bool encode_bf16(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// int8 matrix [rows, cols] row-major, boxes of 128 columns (bytes) x box_rows rows, 128-byte swizzle.
bool encode_u8(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t es[2] = {1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(ptr), dims, strides, box, es,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Split of the router projection over the hidden dimension (a divisor of its 44 chunks of 64):
// the largest that keeps the router grid within one wave of a 152-SM part (one CTA per SM: its
// stage ring takes most of the shared memory), at most 22 (two chunks per CTA). 44 single-chunk
// splits were slower overall: the top-k kernel then adds 44 partial sums per logit (layer at
// T = 256: 285.8 vs 283.6 us). A fixed rule, so the workspace size does not depend on the device.
constexpr int kRouterWave = 152;
int choose_ks(int T) {
  static const int opts[] = {22, 11, 4, 2, 1};
  const int tiles = (T + kRouterN - 1) / kRouterN;
  for (int o : opts)
    if (tiles * o <= kRouterWave) return o;
  return 1;
}
constexpr size_t kPartRowsSmall = static_cast<size_t>(kRouterWave) * kRouterN;  // max ks * T where ks > 1

// Tokens per warp of the top-k kernel: one (its expert counts go to 256-token chunks, so the
// number of CTAs is not bounded).
int choose_tpw(int T) {
  (void)T;
  return 1;
}

// Token tile of the bf16 GEMMs: 64 tokens with two K chunks per stage up to T = 256 (more weight
// bytes in flight per SM than 128-token tiles: at T = 128 gate_up 159 vs 172 us; layer at T = 256
// 278.1 vs 283.6 us, the 30-layer stack 8.23 vs 8.48 ms), 128 up to 1024 (two weight tiles per
// gate_up item above 512), then 256.
int choose_bn(int T) {
  if (T <= 32) return 32;
  if (T <= 256) return 64;
  if (T <= 1024) return 128;
  return 256;
}

struct Layout {
  size_t logits_part, logits, topk_idx, topk_w, gap, hist, base, counts, offsets, tile_off, n_exp_tiles, done_ctr, sched, small_ctr,
      exp_tiles,
      perm, w_sorted, slot_pos, n1, n2, h, h_dense, y, d, status, wsplit, total;
  int max_tiles;
};

Layout make_layout(const moe_ffn_config& c) {
  const size_t Tm = static_cast<size_t>(c.max_tokens);
  const size_t S = Tm * K;
  Layout L;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes, 256);
    return at;
  };
  const size_t part_rows = Tm > kPartRowsSmall ? Tm : kPartRowsSmall;
  L.max_tiles = static_cast<int>(S / 32 + E);
  L.logits_part = take(part_rows * E * 4);
  L.logits = take(Tm * E * 4);
  L.topk_idx = take(Tm * K * 4);
  L.topk_w = take(Tm * K * 4);
  L.gap = take(Tm * 4);
  L.hist = take(static_cast<size_t>(kMaxRouteBlocks) * E * 4);
  L.base = take(static_cast<size_t>(kMaxRouteBlocks) * E * 4);
  L.counts = take(E * 4);
  L.offsets = take((E + 1) * 4);
  L.tile_off = take((E + 1) * 4);
  L.n_exp_tiles = take(4);
  L.done_ctr = take(4);
  L.sched = take(12);
  L.small_ctr = take(32);
  L.status = take(4);
  L.exp_tiles = take(static_cast<size_t>(L.max_tiles) * 16);
  L.perm = take(S * 4);
  L.w_sorted = take(S * 4);
  L.slot_pos = take(S * 4);
  L.n1 = take(c.mode == MOE_FFN_FULL_LAYER ? Tm * H * 2 : 0);
  L.n2 = take(Tm * H * 2);
  L.h = take(S * I * 2);
  L.h_dense = take(c.mode == MOE_FFN_FULL_LAYER ? Tm * D * 2 : 0);
  L.y = take(S * H * 2);
  L.d = take(c.mode == MOE_FFN_FULL_LAYER ? Tm * H * 2 : 0);
  L.wsplit = take(static_cast<size_t>(3) * E * H * 2);
  L.total = o;
  return L;
}

bool config_ok(const moe_ffn_config* c) {
  return c && c->hidden == H && c->n_experts == E && c->top_k == K && c->moe_inter == I && c->dense_inter == D &&
         (c->mode == MOE_FFN_MOE_ONLY || c->mode == MOE_FFN_FULL_LAYER) && c->max_tokens >= 1 &&
         c->max_tokens <= MOE_FFN_MAX_TOKENS_LIMIT && c->eps > 0.0f && c->router_scale > 0.0f;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace moe {
bool encode_bf16_tensor_map(CUtensorMap* map, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  return encode_bf16(map, ptr, rows, cols, box_rows);
}
}  // namespace moe

struct moe_ffn_ctx {
  moe_ffn_config cfg;
  int device;
  int num_sms;
  int pair_clusters;  // two-CTA clusters of the SM-pair GEMMs resident at once (0: do not use them)
  uint8_t* ws;
  size_t ws_bytes;
  Buffers buf;
  // token-operand maps, one per token-tile width (box rows = BN): n1, h, h_dense
  CUtensorMap map_n1[4], map_h[4], map_hd[4];
  // the experts' gate_up input in sorted-slot order (the y buffer), 128-row boxes (SM pairs: half
  // a token tile per CTA)
  CUtensorMap map_n2s_half;
  CUtensorMap map_wsplit;  // the router's split matrix, boxes of 64 x 128 rows
  // weight maps, re-encoded when the weight pointers change
  const void* cached_gate_up;
  const void* cached_down;
  const void* cached_dense_gate;
  const void* cached_dense_up;
  const void* cached_dense_down;
  const void* cached_gate_up_q;
  const void* cached_down_q;
  const void* cached_gate_up_f4;
  const void* cached_down_f4;
  bool cached_valid;
  CUtensorMap map_gate_up_q, map_down_q;  // converted experts: int8 rows or packed MXFP4 codes
  CUtensorMap map_gate_up, map_down, map_dense_gate, map_dense_up, map_dense_down;
  // gate_up weights in 128-row boxes for the SM-pair GEMM (a CTA's 128 gate rows, then its up rows)
  CUtensorMap map_gate_up_pair, map_dense_gate_pair, map_dense_up_pair;
  cudaEvent_t ev_start[kKernelsPerForward];
  cudaEvent_t ev_stop[kKernelsPerForward];
  int last_T;
};

extern "C" {

const char* moe_ffn_status_string(int status) {
  switch (status) {
    case MOE_FFN_OK: return "ok";
    case MOE_FFN_EINVAL: return "invalid argument";
    case MOE_FFN_EALIGN: return "device pointer not 16-byte aligned";
    case MOE_FFN_ETOOBIG: return "size above the context's limit";
    case MOE_FFN_EARCH: return "device is not sm_103 (GB300)";
    case MOE_FFN_ECUDA: return "CUDA call failed";
    case MOE_FFN_EDEVICE: return "a kernel reported a bounded-wait timeout or a bad index";
    default: return "unknown status";
  }
}

size_t moe_ffn_workspace_bytes(const moe_ffn_config* cfg) {
  if (!config_ok(cfg)) return 0;
  return make_layout(*cfg).total;
}

int moe_ffn_init(moe_ffn_ctx** out, const moe_ffn_config* cfg, void* workspace, size_t workspace_bytes,
                 int device) {
  if (!out) return MOE_FFN_EINVAL;
  *out = nullptr;
  if (!config_ok(cfg) || !workspace) return MOE_FFN_EINVAL;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return MOE_FFN_EALIGN;
  const Layout L = make_layout(*cfg);
  if (workspace_bytes < L.total) return MOE_FFN_ETOOBIG;
  if (cudaSetDevice(device) != cudaSuccess) return MOE_FFN_ECUDA;
  int major = 0, minor = 0, sms = 0;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess)
    return MOE_FFN_ECUDA;
  if (major != 10 || minor != 3) return MOE_FFN_EARCH;
  if (!get_encode()) return MOE_FFN_ECUDA;
  if (gemm_set_smem_limits() != cudaSuccess || gemm_pair_set_smem_limits() != cudaSuccess ||
      router_set_smem_limit() != cudaSuccess)
    return MOE_FFN_ECUDA;
  const int pair_clusters = gemm_pair_max_clusters();

  moe_ffn_ctx* c = new (std::nothrow) moe_ffn_ctx();
  if (!c) return MOE_FFN_ECUDA;
  c->cfg = *cfg;
  c->device = device;
  c->num_sms = sms;
  c->pair_clusters = pair_clusters < sms / 2 ? pair_clusters : sms / 2;
  c->ws = static_cast<uint8_t*>(workspace);
  c->ws_bytes = workspace_bytes;
  uint8_t* w = c->ws;
  Buffers& b = c->buf;
  b.logits_part = reinterpret_cast<float*>(w + L.logits_part);
  b.logits = reinterpret_cast<float*>(w + L.logits);
  b.topk_idx = reinterpret_cast<int32_t*>(w + L.topk_idx);
  b.topk_w = reinterpret_cast<float*>(w + L.topk_w);
  b.gap = reinterpret_cast<float*>(w + L.gap);
  b.hist = reinterpret_cast<int32_t*>(w + L.hist);
  b.base = reinterpret_cast<int32_t*>(w + L.base);
  b.counts = reinterpret_cast<int32_t*>(w + L.counts);
  b.offsets = reinterpret_cast<int32_t*>(w + L.offsets);
  b.tile_off = reinterpret_cast<int32_t*>(w + L.tile_off);
  b.n_exp_tiles = reinterpret_cast<int32_t*>(w + L.n_exp_tiles);
  b.done_ctr = reinterpret_cast<int32_t*>(w + L.done_ctr);
  b.sched = reinterpret_cast<int32_t*>(w + L.sched);
  b.small_ctr = reinterpret_cast<int32_t*>(w + L.small_ctr);
  b.status = reinterpret_cast<unsigned int*>(w + L.status);
  b.exp_tiles = reinterpret_cast<int4*>(w + L.exp_tiles);
  b.perm = reinterpret_cast<int32_t*>(w + L.perm);
  b.w_sorted = reinterpret_cast<float*>(w + L.w_sorted);
  b.slot_pos = reinterpret_cast<int32_t*>(w + L.slot_pos);
  b.n1 = cfg->mode == MOE_FFN_FULL_LAYER ? reinterpret_cast<uint16_t*>(w + L.n1) : nullptr;
  b.n2 = reinterpret_cast<uint16_t*>(w + L.n2);
  b.h = reinterpret_cast<uint16_t*>(w + L.h);
  b.h_dense = cfg->mode == MOE_FFN_FULL_LAYER ? reinterpret_cast<uint16_t*>(w + L.h_dense) : nullptr;
  b.y = reinterpret_cast<uint16_t*>(w + L.y);
  b.n2s = b.y;  // written and read by the SM-pair gate_up GEMM, then overwritten by the down GEMM
  b.d = cfg->mode == MOE_FFN_FULL_LAYER ? reinterpret_cast<uint16_t*>(w + L.d) : nullptr;
  b.wsplit = reinterpret_cast<uint16_t*>(w + L.wsplit);
  b.max_tiles = L.max_tiles;

  const uint64_t Tm = static_cast<uint64_t>(cfg->max_tokens);
  bool ok = encode_bf16(&c->map_wsplit, b.wsplit, 3 * E, H, 128) && encode_bf16(&c->map_n2s_half, b.n2s, Tm * K, H, 128);
  for (int k = 0; k < 4; ++k) {
    const uint32_t bn = 32u << k;
    ok = ok && encode_bf16(&c->map_h[k], b.h, Tm * K, I, bn);
    if (cfg->mode == MOE_FFN_FULL_LAYER)
      ok = ok && encode_bf16(&c->map_n1[k], b.n1, Tm, H, bn) && encode_bf16(&c->map_hd[k], b.h_dense, Tm, D, bn);
    else {
      c->map_n1[k] = c->map_h[k];
      c->map_hd[k] = c->map_h[k];
    }
  }
  // The small control words start at zero; the kernels keep them consistent afterwards.
  if (!ok || cudaMemset(w + L.hist, 0, L.exp_tiles - L.hist) != cudaSuccess ||
      cudaDeviceSynchronize() != cudaSuccess) {
    delete c;
    return MOE_FFN_ECUDA;
  }
  *out = c;
  return MOE_FFN_OK;
}

void moe_ffn_destroy(moe_ffn_ctx* ctx) { delete ctx; }

static int prepare_weights(moe_ffn_ctx* c, const moe_ffn_weights* w) {
  const bool full = c->cfg.mode == MOE_FFN_FULL_LAYER;
  // int8 experts: all four fields, or none; likewise MXFP4; not both.
  const bool q8 = w->gate_up_q || w->gate_up_scale || w->down_q || w->down_scale;
  const bool f4 = w->gate_up_f4 || w->gate_up_f4s || w->down_f4 || w->down_f4s;
  if (q8 && f4) return MOE_FFN_EINVAL;
  if (q8) {
    if (!w->gate_up_q || !w->gate_up_scale || !w->down_q || !w->down_scale) return MOE_FFN_EINVAL;
    if (!aligned16(w->gate_up_q) || !aligned16(w->down_q) || !aligned16(w->gate_up_scale) ||
        !aligned16(w->down_scale))
      return MOE_FFN_EALIGN;
  }
  if (f4) {
    if (!w->gate_up_f4 || !w->gate_up_f4s || !w->down_f4 || !w->down_f4s) return MOE_FFN_EINVAL;
    if (!aligned16(w->gate_up_f4) || !aligned16(w->down_f4) || !aligned16(w->gate_up_f4s) ||
        !aligned16(w->down_f4s))
      return MOE_FFN_EALIGN;
  }
  const bool cvt = q8 || f4;
  if (!w->router_w || !w->router_norm_w || !w->per_expert_scale || (!cvt && (!w->gate_up || !w->down)))
    return MOE_FFN_EINVAL;
  if (full && (!w->dense_gate || !w->dense_up || !w->dense_down || !w->pre_ff_ln || !w->pre_ff_ln_2 ||
               !w->post_ff_ln_1 || !w->post_ff_ln_2 || !w->post_ff_ln))
    return MOE_FFN_EINVAL;
  const void* gu = f4 ? static_cast<const void*>(w->gate_up_f4)
                      : q8 ? static_cast<const void*>(w->gate_up_q) : static_cast<const void*>(w->gate_up);
  const void* dn = f4 ? static_cast<const void*>(w->down_f4)
                      : q8 ? static_cast<const void*>(w->down_q) : static_cast<const void*>(w->down);
  const void* ps[] = {w->router_w, w->router_norm_w, w->per_expert_scale, gu, dn};
  for (const void* p : ps)
    if (!aligned16(p)) return MOE_FFN_EALIGN;
  if (full) {
    const void* pf[] = {w->dense_gate, w->dense_up, w->dense_down, w->pre_ff_ln, w->pre_ff_ln_2,
                        w->post_ff_ln_1, w->post_ff_ln_2, w->post_ff_ln};
    for (const void* p : pf)
      if (!aligned16(p)) return MOE_FFN_EALIGN;
  }
  const bool same = c->cached_gate_up == w->gate_up && c->cached_down == w->down &&
                    c->cached_gate_up_q == w->gate_up_q && c->cached_down_q == w->down_q &&
                    c->cached_gate_up_f4 == w->gate_up_f4 && c->cached_down_f4 == w->down_f4 &&
                    (!full || (c->cached_dense_gate == w->dense_gate && c->cached_dense_up == w->dense_up &&
                               c->cached_dense_down == w->dense_down));
  if (same && c->cached_valid) return MOE_FFN_OK;
  // With converted experts the bf16 expert maps are never read by a kernel; they are encoded over
  // the converted arrays (as bf16 of fewer columns) only so that every map handed to a kernel is
  // valid. The converted rows are read as bytes: int8 K bytes per row, MXFP4 K / 2.
  const uint64_t kb_gu = f4 ? H / 2 : H, kb_dn = f4 ? I / 2 : I;
  bool ok = cvt ? encode_u8(&c->map_gate_up_q, gu, static_cast<uint64_t>(E) * 2 * I, kb_gu, 64) &&
                      encode_u8(&c->map_down_q, dn, static_cast<uint64_t>(E) * H, kb_dn, 128) &&
                      encode_bf16(&c->map_gate_up, gu, static_cast<uint64_t>(E) * 2 * I, kb_gu / 2, 64) &&
                      encode_bf16(&c->map_down, dn, static_cast<uint64_t>(E) * H, kb_dn / 2, 128)
                : encode_bf16(&c->map_gate_up, w->gate_up, static_cast<uint64_t>(E) * 2 * I, H, 64) &&
                      encode_bf16(&c->map_down, w->down, static_cast<uint64_t>(E) * H, I, 128);
  if (!cvt) {
    c->map_gate_up_q = c->map_gate_up;
    c->map_down_q = c->map_down;
    ok = ok && encode_bf16(&c->map_gate_up_pair, w->gate_up, static_cast<uint64_t>(E) * 2 * I, H, 128);
  } else {
    c->map_gate_up_pair = c->map_gate_up;
  }
  if (full)
    ok = ok && encode_bf16(&c->map_dense_gate, w->dense_gate, D, H, 64) &&
         encode_bf16(&c->map_dense_up, w->dense_up, D, H, 64) &&
         encode_bf16(&c->map_dense_down, w->dense_down, H, D, 128) &&
         encode_bf16(&c->map_dense_gate_pair, w->dense_gate, D, H, 128) &&
         encode_bf16(&c->map_dense_up_pair, w->dense_up, D, H, 128);
  else {
    c->map_dense_gate = c->map_gate_up;
    c->map_dense_up = c->map_gate_up;
    c->map_dense_down = c->map_down;
    c->map_dense_gate_pair = c->map_gate_up_pair;
    c->map_dense_up_pair = c->map_gate_up_pair;
  }
  if (!ok) {
    c->cached_valid = false;
    return MOE_FFN_ECUDA;
  }
  c->cached_valid = true;
  c->cached_gate_up_q = w->gate_up_q;
  c->cached_down_q = w->down_q;
  c->cached_gate_up_f4 = w->gate_up_f4;
  c->cached_down_f4 = w->down_f4;
  c->cached_gate_up = w->gate_up;
  c->cached_down = w->down;
  c->cached_dense_gate = w->dense_gate;
  c->cached_dense_up = w->dense_up;
  c->cached_dense_down = w->dense_down;
  return MOE_FFN_OK;
}

// An expert-parallel shard of one forward: the experts [e_lo, e_hi) only, the shared MLP if
// with_dense, and the fp32 partial outputs instead of the block's output.
struct Shard {
  int e_lo, e_hi;
  bool with_dense;
  float* moe_out;
  float* dense_out;
};

static bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  const uint8_t* pa = static_cast<const uint8_t*>(a);
  const uint8_t* pb = static_cast<const uint8_t*>(b);
  return pa < pb + nb && pb < pa + na;
}

// The launch sequence of one forward (sh == NULL) or of one shard of it. Arguments are checked.
static int run_forward(moe_ffn_ctx* c, const void* x, int T, const moe_ffn_weights* w, void* out, void* stream,
                       const Shard* sh) {
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_FFN_ECUDA;
  if (cur != c->device && cudaSetDevice(c->device) != cudaSuccess) return MOE_FFN_ECUDA;
  int rc = prepare_weights(c, w);
  if (rc != MOE_FFN_OK) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const bool full = c->cfg.mode == MOE_FFN_FULL_LAYER;
  // The GEMMs run the shared-MLP group in the full layer, except in a shard that leaves it out.
  const int gemm_full = full && (!sh || sh->with_dense) ? 1 : 0;

  RouteParams rp;
  rp.x = static_cast<const uint16_t*>(x);
  rp.router_w = w->router_w;
  rp.router_norm_w = w->router_norm_w;
  rp.per_expert_scale = w->per_expert_scale;
  rp.pre_ff_ln = w->pre_ff_ln;
  rp.pre_ff_ln_2 = w->pre_ff_ln_2;
  rp.T = T;
  rp.ks = T <= kRouteSmallT ? 1 : choose_ks(T);
  rp.tpw = choose_tpw(T);
  // Converted experts (int8 or MXFP4) run the GEMM variants with A in tensor memory, built for
  // token tiles of 32 (small batches, deeper rings) or 64.
  const bool f4 = w->gate_up_f4 != nullptr;
  const bool cvt = w->gate_up_q != nullptr || f4;
  rp.bn = cvt ? (T <= 128 ? 32 : 64) : choose_bn(T);
  rp.full_layer = full ? 1 : 0;
  // Token tiles of 256 on SM pairs (above kPairGateUpT tokens): the gate_up GEMM writes and reads
  // the sorted copy of n2.
  const bool perm_rows = !cvt && rp.bn == 256 && c->pair_clusters > 0 && T > kPairGateUpT;
  rp.write_n2 = perm_rows ? 0 : 1;
  rp.e_lo = sh ? sh->e_lo : 0;
  rp.e_hi = sh ? sh->e_hi : E;
  rp.eps = c->cfg.eps;
  rp.router_scale = c->cfg.router_scale;

  CombineParams cp;
  cp.x = rp.x;
  cp.post_ff_ln_1 = w->post_ff_ln_1;
  cp.post_ff_ln_2 = w->post_ff_ln_2;
  cp.post_ff_ln = w->post_ff_ln;
  cp.layer_scalar = w->layer_scalar;
  cp.out = static_cast<uint16_t*>(out);
  cp.T = T;
  cp.full_layer = rp.full_layer;
  cp.eps = c->cfg.eps;

  const int bk = rp.bn == 32 ? 0 : rp.bn == 64 ? 1 : rp.bn == 128 ? 2 : 3;
  GemmMaps gu, dn;
  gu.a_exp = c->map_gate_up;
  gu.a_dense0 = c->map_dense_gate;
  gu.a_dense1 = c->map_dense_up;
  gu.b_exp = c->map_n1[bk];  // unused: the experts' gate_up rows are gathered with cp.async
  gu.b_dense = c->map_n1[bk];
  dn.a_exp = c->map_down;
  dn.a_dense0 = c->map_dense_down;
  dn.a_dense1 = c->map_dense_down;
  dn.b_exp = c->map_h[bk];
  dn.b_dense = c->map_hd[bk];
  gu.a_q = c->map_gate_up_q;
  gu.q_scale = f4 ? static_cast<const void*>(w->gate_up_f4s) : static_cast<const void*>(w->gate_up_scale);
  dn.a_q = c->map_down_q;
  dn.q_scale = f4 ? static_cast<const void*>(w->down_f4s) : static_cast<const void*>(w->down_scale);

  // Persistent GEMM grids: at most one CTA per SM, and no more than an upper bound of the items.
  const int S = T * K;
  const int bn = rp.bn;
  const int ub_tiles = (S < E ? S : E) + S / bn;
  const int nd = gemm_full ? (T + bn - 1) / bn : 0;
  const int ma = cvt ? 1 : gate_up_tiles_per_item(bn, T);
  const long items_gu = static_cast<long>(ub_tiles) * ((I / 64 + ma - 1) / ma) +
                        static_cast<long>(nd) * ((D / 64 + ma - 1) / ma);
  const long items_dn = static_cast<long>(ub_tiles) * (H / 128) + static_cast<long>(nd) * (H / 128);
  const int grid_gu = static_cast<int>(items_gu < c->num_sms ? items_gu : c->num_sms);
  int grid_dn = static_cast<int>(items_dn < c->num_sms ? items_dn : c->num_sms);
  // For token tiles of 256 (T above 1024) the down GEMM runs on SM pairs, and above kPairGateUpT
  // tokens the gate_up GEMM too: M = 256 per pair of CTAs, half of each token tile in each CTA, so
  // their B maps are the ones with 128-row boxes.
  const bool pairs = bn == 256 && c->pair_clusters > 0 && !cvt;
  const bool pairs_gu = perm_rows;
  int grid_gu_launch = grid_gu;
  if (pairs) {
    grid_dn = 2 * c->pair_clusters;
    dn.b_exp = c->map_h[2];
    dn.b_dense = c->map_hd[2];
  }
  if (pairs_gu) {
    grid_gu_launch = 2 * c->pair_clusters;
    gu.a_exp = c->map_gate_up_pair;
    gu.a_dense0 = c->map_dense_gate_pair;
    gu.a_dense1 = c->map_dense_up_pair;
    gu.b_exp = c->map_n2s_half;
    gu.b_dense = c->map_n1[2];
  }

  PermIn pin;
  pin.x = rp.x;
  pin.w2 = full ? w->pre_ff_ln_2 : nullptr;
  pin.eps = c->cfg.eps;
  pin.e_lo = rp.e_lo;
  pin.e_hi = rp.e_hi;
  ShardParams spar;
  spar.T = T;
  spar.e_lo = rp.e_lo;
  spar.e_hi = rp.e_hi;
  spar.moe_out = sh ? sh->moe_out : nullptr;
  spar.dense_out = sh ? sh->dense_out : nullptr;
  cudaError_t e = cudaSuccess;
  for (int k = 0; k < kKernelsPerForward && e == cudaSuccess; ++k) {
    if (c->ev_start[k]) e = cudaEventRecord(c->ev_start[k], s);
    if (e != cudaSuccess) break;
    switch (k) {
      // Small batches: no fold kernel; the router's sums on CUDA cores, the top-k and the counting
      // sort in the same kernel (slot 1), so slots 0, 2 and 3 launch nothing.
      case 0: e = T <= kRouteSmallT ? cudaSuccess : launch_router_prep(rp, c->buf, s); break;
      case 1:
        e = T <= kRouteSmallT ? launch_route_small(rp, c->buf, s) : launch_router_logits(c->map_wsplit, rp, c->buf, s);
        break;
      case 2: e = T <= kRouteSmallT ? cudaSuccess : launch_route_topk(rp, c->buf, s); break;
      case 3: e = T <= kRouteSmallT ? cudaSuccess : launch_route_scatter(rp, c->buf, s); break;
      case 4:
        e = cvt     ? launch_gate_up_cvt(bn, f4, gu, c->buf, T, gemm_full, grid_gu, s)
            : pairs_gu ? launch_gate_up_pair(gu, c->buf, pin, T, gemm_full, grid_gu_launch, s)
                    : launch_gate_up(bn, gu, c->buf, T, gemm_full, grid_gu, s);
        break;
      case 5:
        e = cvt     ? launch_down_cvt(bn, f4, dn, c->buf, T, gemm_full, grid_dn, s)
            : pairs ? launch_down_pair(dn, c->buf, T, gemm_full, grid_dn, s)
                    : launch_down(bn, dn, c->buf, T, gemm_full, grid_dn, s);
        break;
      case 6: e = sh ? launch_combine_shard(spar, c->buf, s) : launch_combine(cp, c->buf, s); break;
    }
    if (e == cudaSuccess && c->ev_stop[k]) e = cudaEventRecord(c->ev_stop[k], s);
  }
  if (e != cudaSuccess) return MOE_FFN_ECUDA;
  c->last_T = T;
  return MOE_FFN_OK;
}

int moe_ffn_forward(moe_ffn_ctx* c, const void* x, int T, const moe_ffn_weights* w, void* out, void* stream) {
  if (!c || !w) return MOE_FFN_EINVAL;
  if (T < 0) return MOE_FFN_EINVAL;
  if (T > c->cfg.max_tokens) return MOE_FFN_ETOOBIG;
  if (T == 0) return MOE_FFN_OK;
  if (!x || !out) return MOE_FFN_EINVAL;
  if (!aligned16(x) || !aligned16(out)) return MOE_FFN_EALIGN;
  const size_t io_bytes = static_cast<size_t>(T) * H * 2;
  if (overlaps(out, io_bytes, x, io_bytes) || overlaps(out, io_bytes, c->ws, c->ws_bytes)) return MOE_FFN_EINVAL;
  return run_forward(c, x, T, w, out, stream, nullptr);
}

int moe_ffn_forward_shard(moe_ffn_ctx* c, const void* x, int T, const moe_ffn_weights* w, int expert_begin,
                          int expert_end, int with_dense, float* moe_partial, float* dense_out, void* stream) {
  if (!c || !w) return MOE_FFN_EINVAL;
  if (T < 0 || expert_begin < 0 || expert_end > E || expert_begin > expert_end) return MOE_FFN_EINVAL;
  const bool full = c->cfg.mode == MOE_FFN_FULL_LAYER;
  if (with_dense && !full) return MOE_FFN_EINVAL;
  if (T > c->cfg.max_tokens) return MOE_FFN_ETOOBIG;
  if (T == 0) return MOE_FFN_OK;
  if (!x || !moe_partial || (with_dense && !dense_out)) return MOE_FFN_EINVAL;
  if (!aligned16(x) || !aligned16(moe_partial) || (with_dense && !aligned16(dense_out))) return MOE_FFN_EALIGN;
  const size_t f_bytes = static_cast<size_t>(T) * H * 4, x_bytes = static_cast<size_t>(T) * H * 2;
  if (overlaps(moe_partial, f_bytes, x, x_bytes) || overlaps(moe_partial, f_bytes, c->ws, c->ws_bytes))
    return MOE_FFN_EINVAL;
  if (with_dense && (overlaps(dense_out, f_bytes, x, x_bytes) || overlaps(dense_out, f_bytes, c->ws, c->ws_bytes) ||
                     overlaps(dense_out, f_bytes, moe_partial, f_bytes)))
    return MOE_FFN_EINVAL;
  Shard sh;
  sh.e_lo = expert_begin;
  sh.e_hi = expert_end;
  sh.with_dense = with_dense != 0;
  sh.moe_out = moe_partial;
  sh.dense_out = with_dense ? dense_out : nullptr;
  return run_forward(c, x, T, w, nullptr, stream, &sh);
}

int moe_ffn_finish_shards(moe_ffn_ctx* c, const void* x, int T, const moe_ffn_weights* w, const float* moe_sum,
                          const float* dense, void* out, void* stream) {
  if (!c || !w) return MOE_FFN_EINVAL;
  if (T < 0) return MOE_FFN_EINVAL;
  if (T > c->cfg.max_tokens) return MOE_FFN_ETOOBIG;
  if (T == 0) return MOE_FFN_OK;
  const bool full = c->cfg.mode == MOE_FFN_FULL_LAYER;
  if (!moe_sum || !out || (full && (!x || !dense || !w->post_ff_ln_1 || !w->post_ff_ln_2 || !w->post_ff_ln)))
    return MOE_FFN_EINVAL;
  if (!aligned16(moe_sum) || !aligned16(out) || (full && (!aligned16(x) || !aligned16(dense))) ||
      (full && (!aligned16(w->post_ff_ln_1) || !aligned16(w->post_ff_ln_2) || !aligned16(w->post_ff_ln))))
    return MOE_FFN_EALIGN;
  const size_t io_bytes = static_cast<size_t>(T) * H * 2, f_bytes = static_cast<size_t>(T) * H * 4;
  if (overlaps(out, io_bytes, moe_sum, f_bytes) || (full && (overlaps(out, io_bytes, x, io_bytes) ||
                                                             overlaps(out, io_bytes, dense, f_bytes))))
    return MOE_FFN_EINVAL;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess) return MOE_FFN_ECUDA;
  if (cur != c->device && cudaSetDevice(c->device) != cudaSuccess) return MOE_FFN_ECUDA;
  CombineParams cp;
  cp.x = static_cast<const uint16_t*>(x);
  cp.post_ff_ln_1 = w->post_ff_ln_1;
  cp.post_ff_ln_2 = w->post_ff_ln_2;
  cp.post_ff_ln = w->post_ff_ln;
  cp.layer_scalar = w->layer_scalar;
  cp.out = static_cast<uint16_t*>(out);
  cp.T = T;
  cp.full_layer = full ? 1 : 0;
  cp.eps = c->cfg.eps;
  return launch_finish(cp, moe_sum, full ? dense : nullptr, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_FFN_OK
             : MOE_FFN_ECUDA;
}

int moe_ffn_workspace_view(const moe_ffn_ctx* c, moe_ffn_views* v) {
  if (!c || !v) return MOE_FFN_EINVAL;
  const Buffers& b = c->buf;
  v->logits = b.logits;
  v->topk_idx = b.topk_idx;
  v->topk_w = b.topk_w;
  v->gap = b.gap;
  v->counts = b.counts;
  v->offsets = b.offsets;
  v->perm = b.perm;
  v->w_sorted = b.w_sorted;
  v->slot_pos = b.slot_pos;
  v->n1 = b.n1;
  v->n2 = b.n2;
  v->h = b.h;
  v->h_dense = b.h_dense;
  v->y = b.y;
  v->d = b.d;
  v->T = c->last_T;
  return MOE_FFN_OK;
}

int moe_ffn_device_status(moe_ffn_ctx* c, void* stream, uint32_t* word) {
  if (!c) return MOE_FFN_EINVAL;
  if (cudaSetDevice(c->device) != cudaSuccess) return MOE_FFN_ECUDA;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_FFN_ECUDA;
  uint32_t v = 0;
  if (cudaMemcpy(&v, c->buf.status, 4, cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_FFN_ECUDA;
  if (v != 0 && cudaMemset(c->buf.status, 0, 4) != cudaSuccess) return MOE_FFN_ECUDA;
  if (word) *word = v;
  return v ? MOE_FFN_EDEVICE : MOE_FFN_OK;
}

int moe_ffn_set_kernel_events(moe_ffn_ctx* c, int kernel, void* start, void* stop) {
  if (!c || kernel < 0 || kernel >= kKernelsPerForward) return MOE_FFN_EINVAL;
  if ((start == nullptr) != (stop == nullptr)) return MOE_FFN_EINVAL;
  c->ev_start[kernel] = static_cast<cudaEvent_t>(start);
  c->ev_stop[kernel] = static_cast<cudaEvent_t>(stop);
  return MOE_FFN_OK;
}

// The kernel slots a forward of T tokens launches, in launch order (see moe_ffn_set_kernel_events).
static int slots_of(int T, int* slots) {
  if (T == 0) return 0;
  int n = 0;
  for (int k = 0; k < kKernelsPerForward; ++k)
    if (T > kRouteSmallT || (k != 0 && k != 2 && k != 3)) slots[n++] = k;
  return n;
}

int moe_ffn_kernels_per_forward(const moe_ffn_ctx* c, int T) {
  if (!c || T < 0) return MOE_FFN_EINVAL;
  int slots[kKernelsPerForward];
  return slots_of(T, slots);
}

int moe_ffn_kernel_slots(const moe_ffn_ctx* c, int T, int* slots, int n_slots) {
  if (!c || T < 0 || !slots || n_slots < kKernelsPerForward) return MOE_FFN_EINVAL;
  return slots_of(T, slots);
}

}  // extern "C"
