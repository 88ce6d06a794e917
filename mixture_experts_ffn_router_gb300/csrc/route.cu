// route.cu — the CUDA-core kernels of the block: top-k with the pre-norms, the counting-sort
// scatter of token slots by expert, and the combine with the post-norms.
//
// What they compute follows "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 —
// where every rank weighted the wrong experts", section "The architecture: a dual-path FFN nobody
// warned me about": the router normalises its input with its own RMSNorm, multiplies by a scale
// and per-expert weights, takes a softmax over 128 experts in fp32, keeps the top 8, renormalises
// them to sum 1 and multiplies by per_expert_scale; the expert outputs are gathered back to their
// tokens and, with the shared MLP, pass through the feed-forward norms, the residual add and
// layer_scalar ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", §4.6).
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace moe {

namespace {

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16_rn(lo)) | (static_cast<uint32_t>(f32_to_bf16_rn(hi)) << 16);
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// An unsigned key with the order of the fp32 values (finite; -0 taken as +0), so that a warp
// maximum of keys is the maximum logit.
__device__ __forceinline__ uint32_t order_key(float v) {
  const uint32_t u = __float_as_uint(v == 0.0f ? 0.0f : v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The fp32 value of an order key (the inverse of order_key; -0 comes back as +0).
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// v[j] for a j known at run time, without local memory.
__device__ __forceinline__ float pick4(const float (&v)[4], int j) {
  return j == 0 ? v[0] : j == 1 ? v[1] : j == 2 ? v[2] : v[3];
}

// The routing of NT tokens by one warp, from their raw router sums. Lane l holds z[u][j], token
// u's sum over the hidden dimension for expert l + 32 j, and inv[u], the token's 1 / RMS. Logits
// are z * inv * router_scale (stored to rows[u] unless it is NULL); then an fp32 softmax over the
// 128 experts; the top 8 by logit, ties to the lower expert id, and the 9th for the gap; the 8
// probabilities renormalised to sum 1 and multiplied by per_expert_scale (pes, 128 values).
// Lanes 0..7 get the lane-th selected expert in ascending id (e_out) and its weight (w_out); every
// lane gets the 8th-minus-9th logit gap. The tokens' steps are interleaved for NT > 1; each
// token's arithmetic is the same for every NT.
template <int NT>
__device__ __forceinline__ void route_tokens(const float (&z)[NT][4], const float (&inv)[NT], float router_scale,
                                             float* const (&rows)[NT], const float* pes, int lane, int (&e_out)[NT],
                                             float (&w_out)[NT], float (&gap)[NT]) {
  constexpr unsigned kAll = 0xffffffffu;
  float lg[NT][4], pr[NT][4], zsum[NT];
  uint32_t mk[NT];
#pragma unroll
  for (int u = 0; u < NT; ++u) {
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      lg[u][j] = z[u][j] * inv[u] * router_scale;
      if (rows[u]) rows[u][lane + 32 * j] = lg[u][j];
    }
    mk[u] = order_key(fmaxf(fmaxf(lg[u][0], lg[u][1]), fmaxf(lg[u][2], lg[u][3])));
  }
  // The largest logit (the warp maximum of the keys), then exp(logit - max) and their sum in a
  // fixed butterfly order.
#pragma unroll
  for (int u = 0; u < NT; ++u) mk[u] = __reduce_max_sync(kAll, mk[u]);
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    const float m = key_value(mk[u]);
    zsum[u] = 0.0f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      pr[u][j] = expf(lg[u][j] - m);
      zsum[u] += pr[u][j];
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
#pragma unroll
    for (int u = 0; u < NT; ++u) zsum[u] += __shfl_xor_sync(kAll, zsum[u], o);
#pragma unroll
  for (int u = 0; u < NT; ++u)
#pragma unroll
    for (int j = 0; j < 4; ++j) pr[u][j] = pr[u][j] / zsum[u];

  // Top-8 (and the 9th for the gap) by repeated warp arg-max. Each round: the lane's best untaken
  // logit (the lower j, so the lower id, on equal values), the warp maximum of their keys, then the
  // lowest expert id among the lanes holding it.
  unsigned taken[NT];
  int sel_e[NT][K];
  float sel_p[NT][K];
  float l8[NT], l9[NT];
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    taken[u] = 0u;
    l8[u] = 0.0f;
    l9[u] = 0.0f;
  }
#pragma unroll
  for (int r = 0; r < K + 1; ++r) {
    uint32_t key[NT];
    int bj[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      bj[u] = -1;
      float bl = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (!(taken[u] & (1u << j)) && (bj[u] < 0 || lg[u][j] > bl)) {
          bj[u] = j;
          bl = lg[u][j];
        }
      key[u] = bj[u] < 0 ? 0u : order_key(bl);
    }
    uint32_t kmax[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) kmax[u] = __reduce_max_sync(kAll, key[u]);
    int ew[NT];
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      const uint32_t mine =
          (bj[u] >= 0 && key[u] == kmax[u]) ? static_cast<uint32_t>(lane + 32 * bj[u]) : 0xffffffffu;
      ew[u] = static_cast<int>(__reduce_min_sync(kAll, mine));
    }
#pragma unroll
    for (int u = 0; u < NT; ++u) {
      const int wlane = ew[u] & 31, wj = ew[u] >> 5;
      const float lw = __shfl_sync(kAll, pick4(lg[u], wj), wlane);
      const float pw = __shfl_sync(kAll, pick4(pr[u], wj), wlane);
      if (wlane == lane) taken[u] |= 1u << wj;
      if (r < K) {
        sel_e[u][r] = ew[u];
        sel_p[u][r] = pw;
      }
      if (r == K - 1) l8[u] = lw;
      if (r == K) l9[u] = lw;
    }
  }
#pragma unroll
  for (int u = 0; u < NT; ++u) {
    // Ascending expert id (odd-even transposition sort, identical in every lane).
#pragma unroll
    for (int pass = 0; pass < K; ++pass) {
#pragma unroll
      for (int j = (pass & 1); j + 1 < K; j += 2) {
        if (sel_e[u][j] > sel_e[u][j + 1]) {
          const int te = sel_e[u][j];
          sel_e[u][j] = sel_e[u][j + 1];
          sel_e[u][j + 1] = te;
          const float tp = sel_p[u][j];
          sel_p[u][j] = sel_p[u][j + 1];
          sel_p[u][j + 1] = tp;
        }
      }
    }
    float psum = 0.0f;
#pragma unroll
    for (int j = 0; j < K; ++j) psum += sel_p[u][j];
    int e = sel_e[u][0];
    float pp = sel_p[u][0];
#pragma unroll
    for (int j = 1; j < K; ++j)
      if (lane == j) {
        e = sel_e[u][j];
        pp = sel_p[u][j];
      }
    e_out[u] = e;
    w_out[u] = lane < K ? (pp / psum) * pes[e] : 0.0f;
    gap[u] = l8[u] - l9[u];
  }
}

// Warp 0 of the CTA that builds a forward's schedule. From the slot counts cnt[j] of the experts
// lane * 4 + j: the experts' first sorted positions (an exclusive scan) and, for the experts
// [e_lo, e_hi) this forward computes, their first token tiles (tiles of bn rows). Both scans go to
// scan_s / tscan_s [129] and to the buffers; the tile count is published (0, with a status bit, if
// it exceeds the list) and the GEMMs' work counters are reset.
__device__ __forceinline__ void expert_scan(const int (&cnt)[4], const RouteParams& p, const Buffers& b, int* scan_s,
                                            int* tscan_s, int lane) {
  int nt[4];
  int cs = 0, ts = 0;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ee = lane * 4 + j;
    nt[j] = (ee >= p.e_lo && ee < p.e_hi) ? (cnt[j] + p.bn - 1) / p.bn : 0;
    cs += cnt[j];
    ts += nt[j];
  }
  int ci = cs, ti = ts;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int a = __shfl_up_sync(0xffffffffu, ci, o);
    const int c = __shfl_up_sync(0xffffffffu, ti, o);
    if (lane >= o) {
      ci += a;
      ti += c;
    }
  }
  int cex = ci - cs, tex = ti - ts;
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const int ee = lane * 4 + j;
    scan_s[ee] = cex;
    tscan_s[ee] = tex;
    b.counts[ee] = cnt[j];
    b.offsets[ee] = cex;
    b.tile_off[ee] = tex;
    cex += cnt[j];
    tex += nt[j];
  }
  if (lane == 31) {
    scan_s[E] = cex;
    tscan_s[E] = tex;
    b.offsets[E] = cex;
    b.tile_off[E] = tex;
    if (tex > b.max_tiles) atomicOr(b.status, kStatusBadSchedule);
    *b.n_exp_tiles = tex <= b.max_tiles ? tex : 0;
    b.sched[0] = 0;  // the GEMMs of this forward claim their work items from these counters
    b.sched[1] = 0;
    b.sched[2] = 0;  // warps done with the sorted copy of n2 (SM-pair gate_up)
  }
}

// Expert e's token tiles (expert, first sorted row, rows, 0) from the scans above.
__device__ __forceinline__ void expert_tiles(int e, const RouteParams& p, const Buffers& b, const int* scan_s,
                                             const int* tscan_s) {
  if (tscan_s[E] > b.max_tiles) return;
  const int cnt = scan_s[e + 1] - scan_s[e];
  const int nt = tscan_s[e + 1] - tscan_s[e];
  for (int j = 0; j < nt; ++j) {
    const int rows = min(p.bn, cnt - j * p.bn);
    b.exp_tiles[tscan_s[e] + j] = make_int4(e, scan_s[e] + j * p.bn, rows, 0);
  }
}

// One 16-byte chunk (8 features) of a pre-norm row: x * inv_rms * (1 + w), the weights given as
// two float4 halves already holding 1 + w.
__device__ __forceinline__ uint4 norm_chunk(uint4 xc, float inv, float4 a0, float4 a1) {
  const float g[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
  const uint32_t w4[4] = {xc.x, xc.y, xc.z, xc.w};
  uint32_t o[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = bf16_lo(w4[j]) * inv, hi = bf16_hi(w4[j]) * inv;
    o[j] = pack_bf16(lo * g[2 * j], hi * g[2 * j + 1]);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// 1 / RMS of one token row held by a warp (lane l: 16-byte chunks l + 32 c): lane sums in chunk
// order, then a butterfly, so every kernel that takes it gets the same bits.
__device__ __forceinline__ float token_inv_rms(const uint4 (&xr)[11], float eps) {
  float ss = 0.0f;
#pragma unroll
  for (int c = 0; c < 11; ++c) {
    const uint32_t w4[4] = {xr[c].x, xr[c].y, xr[c].z, xr[c].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float a = bf16_lo(w4[j]), bb = bf16_hi(w4[j]);
      ss = fmaf(a, a, ss);
      ss = fmaf(bb, bb, ss);
    }
  }
  ss = warp_sum(ss);
  return 1.0f / sqrtf(ss / static_cast<float>(H) + eps);
}

// ------------------------------------------------------------------------------------------
// K2: one warp per token. RMS of x; logits = rms * scale * sum of the partials; fp32 softmax;
// top-8 by logit with the 9th for the gap; renormalise, times per_expert_scale; slots listed in
// ascending expert id. Each CTA counts its slots per expert and takes a finish ticket, then writes
// its tokens' expert-branch inputs (the two pre-norms in the full layer, else a copy of x); the
// last CTA to finish turns the counts into expert offsets, per-CTA base positions and the grouped
// GEMMs' token-tile list.
__global__ void __launch_bounds__(256, 4) route_topk_kernel(RouteParams p, Buffers b) {
  __shared__ int hist_s[E];
  __shared__ int part_s[2][E];
  __shared__ int scan_s[E + 1];
  __shared__ int tscan_s[E + 1];
  __shared__ float pes_s[E];
  // 1 + pre_feedforward_layernorm and 1 + pre_feedforward_layernorm_2 (full layer), so that the
  // norm loop below reads no global memory between its stores. Column group q = lane + 32 c (8
  // columns) is stored as two float4 halves at g_s[v][c][half][lane]: a warp's 16-byte loads
  // then hit consecutive addresses (a plain [H] layout puts lanes 32 bytes apart, two-way bank
  // conflicts).
  __shared__ float4 g_s[2][11][2][32];
  __shared__ float inv_s[kScatterTok];  // 1 / RMS of the CTA's tokens (8 tpw <= 256)
  __shared__ int is_last;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid < E) hist_s[tid] = 0;
  // Weights only, so they may be read before the wait for the router's partial sums: this grid
  // starts only after every router CTA has passed its own wait, so all earlier work on the
  // stream is complete. L2-coherent loads, so no line cached by an earlier kernel is seen.
  if (tid < E) pes_s[tid] = __ldcg(p.per_expert_scale + tid);
  if (p.full_layer)
    for (int i = tid; i < H / 4; i += 256) {
      const float4 a = __ldcg(reinterpret_cast<const float4*>(p.pre_ff_ln) + i);
      const float4 c = __ldcg(reinterpret_cast<const float4*>(p.pre_ff_ln_2) + i);
      const int q = i >> 1, hf = i & 1;  // float4 i holds columns 4i..4i+3 of group q
      g_s[0][q >> 5][hf][q & 31] = make_float4(1.0f + a.x, 1.0f + a.y, 1.0f + a.z, 1.0f + a.w);
      g_s[1][q >> 5][hf][q & 31] = make_float4(1.0f + c.x, 1.0f + c.y, 1.0f + c.z, 1.0f + c.w);
    }
  pdl_wait();
  // Dependents may launch now: they run nothing before their own wait that reads this grid's
  // results, and everything before this grid is complete.
  pdl_launch_dependents();
  __syncthreads();

  const int tb = 8 * p.tpw;
  for (int i = 0; i < p.tpw; ++i) {
    const int t = blockIdx.x * tb + warp * p.tpw + i;
    if (t >= p.T) break;
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H);
    float inv;
    {
      uint4 xv[11];
#pragma unroll
      for (int c = 0; c < 11; ++c) xv[c] = __ldg(xr + lane + 32 * c);
      inv = token_inv_rms(xv, p.eps);
    }

    if (lane == 0) inv_s[warp * p.tpw + i] = inv;

    // Logits: expert e = lane + 32 j. The partial sums of the lane's 4 experts are added in
    // ascending split order, loaded 8 splits (32 loads) at a time, the last group predicated.
    float z[1][4] = {{0.0f, 0.0f, 0.0f, 0.0f}};
    {
      const float* pp = b.logits_part + static_cast<size_t>(t) * E + lane;
      const size_t stride = static_cast<size_t>(p.T) * E;
      for (int s = 0; s < p.ks; s += 8) {
        float a[8][4];
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j) a[u][j] = s + u < p.ks ? pp[(s + u) * stride + 32 * j] : 0.0f;
#pragma unroll
        for (int u = 0; u < 8; ++u)
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (s + u < p.ks) z[0][j] += a[u][j];
      }
    }
    const float invs[1] = {inv};
    float* const rows[1] = {b.logits + static_cast<size_t>(t) * E};
    int sel[1];
    float wsel[1], gap[1];
    route_tokens<1>(z, invs, p.router_scale, rows, pes_s, lane, sel, wsel, gap);
    if (lane < K) {
      b.topk_idx[static_cast<size_t>(t) * K + lane] = sel[0];
      b.topk_w[static_cast<size_t>(t) * K + lane] = wsel[0];
      atomicAdd(&hist_s[sel[0]], 1);
    }
    if (lane == 0) b.gap[t] = gap[0];
  }

  // Per-CTA counts, then the last CTA to arrive builds the offsets, bases and tile list.
  __syncthreads();
  // Counts per 256-token chunk (the scatter kernel's unit); integer adds, so the totals do not
  // depend on the order in which CTAs arrive.
  if (tid < E && hist_s[tid] != 0) atomicAdd(b.hist + ((blockIdx.x * tb) / kScatterTok) * E + tid, hist_s[tid]);
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(b.done_ctr, 1);
    is_last = (ticket == static_cast<int>(gridDim.x) - 1);
  }

  __syncthreads();
  // The last CTA builds the schedule first, so that it does not wait behind its own row stores.
  if (is_last) {
    __threadfence();

    const int nb = (p.T + kScatterTok - 1) / kScatterTok;  // chunks
    const int e = tid & (E - 1), half = tid >> 7;
    const int bmid = (nb + 1) / 2;
    const int blo = half ? bmid : 0, bhi = half ? nb : bmid;
    // Eight chunks' counts in flight at a time; the first eight stay in registers for the base
    // positions below (all of them up to T = 4096).
    int c8[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) c8[u] = blo + u < bhi ? __ldcg(b.hist + (blo + u) * E + e) : 0;
    {
      int s = 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) s += c8[u];
      for (int b0 = blo + 8; b0 < bhi; b0 += 8) {
        int d8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) d8[u] = b0 + u < bhi ? __ldcg(b.hist + (b0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u) s += d8[u];
      }
      part_s[half][e] = s;
    }
    __syncthreads();
    if (warp == 0) {
      // Exclusive scans over the 128 experts of the counts and of the token-tile counts (tiles only
      // for the experts this forward computes: all of them, or a shard's range).
      int cnt[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) cnt[j] = part_s[0][lane * 4 + j] + part_s[1][lane * 4 + j];
      expert_scan(cnt, p, b, scan_s, tscan_s, lane);
    }
    __syncthreads();
    {
      // Base position of each (CTA, expert): the expert's offset plus the slots of earlier CTAs.
      int run = scan_s[e] + (half ? part_s[0][e] : 0);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (blo + u < bhi) {
          b.base[(blo + u) * E + e] = run;
          run += c8[u];
        }
      for (int b0 = blo + 8; b0 < bhi; b0 += 8) {
        int d8[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) d8[u] = b0 + u < bhi ? __ldcg(b.hist + (b0 + u) * E + e) : 0;
#pragma unroll
        for (int u = 0; u < 8; ++u)
          if (b0 + u < bhi) {
            b.base[(b0 + u) * E + e] = run;
            run += d8[u];
          }
      }
    }
    if (half == 0) expert_tiles(e, p, b, scan_s, tscan_s);
  }

  // The normalised rows are written only now: the routing above never waits behind these stores
  // (46 MB at T = 4096), and the last CTA's scan above overlaps the other CTAs' writes.
  for (int i = 0; i < p.tpw; ++i) {
    const int t = blockIdx.x * tb + warp * p.tpw + i;
    if (t >= p.T) break;
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H);
    const float inv = inv_s[warp * p.tpw + i];
    // Expert-branch input n2 and dense-branch input n1 (n2 only where the gate_up GEMM gathers
    // its rows by token index; above kPairGateUpT tokens the SM-pair gate_up GEMM writes them itself,
    // in sorted-slot order).
    uint4* n2r = reinterpret_cast<uint4*>(b.n2 + static_cast<size_t>(t) * H);
    if (p.full_layer) {
      uint4* n1r = reinterpret_cast<uint4*>(b.n1 + static_cast<size_t>(t) * H);
#pragma unroll
      for (int c = 0; c < 11; ++c) {
        // x again, read-only (this warp read the row above), so the row does not stay in
        // registers; the weights come from shared memory, so no load waits for a store.
        const uint4 xc = __ldg(xr + lane + 32 * c);
        n1r[lane + 32 * c] = norm_chunk(xc, inv, g_s[0][c][0][lane], g_s[0][c][1][lane]);
        if (p.write_n2) n2r[lane + 32 * c] = norm_chunk(xc, inv, g_s[1][c][0][lane], g_s[1][c][1][lane]);
      }
    } else if (p.write_n2) {
#pragma unroll
      for (int c = 0; c < 11; ++c) n2r[lane + 32 * c] = __ldg(xr + lane + 32 * c);
    }
  }
}

// One pre-norm row of token t, written by one warp: n1 (which = 0) or n2 (which = 1) in the full
// layer; in the experts-only mode n2 = x (which = 0) and nothing for which = 1.
__device__ __forceinline__ void write_norm_row(const RouteParams& p, const Buffers& b, int t, int which, int lane) {
  const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H);
  if (!p.full_layer) {
    if (which == 0 && p.write_n2) {
      uint4* n2r = reinterpret_cast<uint4*>(b.n2 + static_cast<size_t>(t) * H);
#pragma unroll
      for (int c = 0; c < 11; ++c) n2r[lane + 32 * c] = __ldg(xr + lane + 32 * c);
    }
    return;
  }
  if (which == 1 && !p.write_n2) return;
  const float4* wr = reinterpret_cast<const float4*>(which ? p.pre_ff_ln_2 : p.pre_ff_ln);
  uint4 xv[11];
  float4 w[11][2];
#pragma unroll
  for (int c = 0; c < 11; ++c) {
    xv[c] = __ldg(xr + lane + 32 * c);
    w[c][0] = __ldg(wr + 2 * (lane + 32 * c));
    w[c][1] = __ldg(wr + 2 * (lane + 32 * c) + 1);
  }
  const float inv = token_inv_rms(xv, p.eps);
  uint4* out = reinterpret_cast<uint4*>((which ? b.n2 : b.n1) + static_cast<size_t>(t) * H);
#pragma unroll
  for (int c = 0; c < 11; ++c) {
    const float4 a0 = w[c][0], a1 = w[c][1];
    out[lane + 32 * c] = norm_chunk(xv[c], inv, make_float4(1.0f + a0.x, 1.0f + a0.y, 1.0f + a0.z, 1.0f + a0.w),
                                    make_float4(1.0f + a1.x, 1.0f + a1.y, 1.0f + a1.z, 1.0f + a1.w));
  }
}

// ------------------------------------------------------------------------------------------
// Small batches (T <= kRouteSmallT): the routing front end in one kernel, three phases chained by
// tickets rather than by kernel boundaries.
//   1. CTA (x, g) forms W'[e] = W_r[e] * (1 + router_norm_w) in fp32 for the four experts
//      e = 4x .. 4x + 3 and the raw router sums of tokens 16g .. 16g + 15, two per warp, both rows
//      loaded before any sum starts. Lane l sums h = 8 (l + 32 k) .. + 7 for k = 0..10 in that
//      order and a butterfly adds the 32 lane sums, so every sum has one fixed order. Each CTA
//      then draws a ticket of its token group. The group's 32 pre-norm rows (n1 and n2 of 16
//      tokens) are written by the 31 CTAs that are not last, one row per ticket (two for the
//      ticket before the last): one row per CTA keeps the stores coalesced and spread over SMs.
//   2. The last CTA of the group routes its 16 tokens, two per warp (route_tokens on the sums,
//      with the RMS each warp took from its rows in phase 1), and writes the routing results.
//   3. The last group to finish phase 2 lists the slots by expert. A stable counting sort: the
//      rank of token t within expert e is the number of tokens below t that chose e, counted from
//      a 64-bit token mask per expert; then the expert offsets and the token-tile list.
// A ticket counter is reset by the CTA that draws its last ticket, so every counter is zero again
// when the kernel ends (the context starts them at zero).
constexpr int kSmallTok = 16;  // tokens per CTA: two per warp
constexpr int kSmallExp = 4;   // experts per CTA
constexpr int kSmallFinal = 4; // small_ctr index of the phase-3 ticket (0..3: token groups)
static_assert(kRouteSmallT <= 64 && kRouteSmallT <= 4 * kSmallTok, "token masks and group tickets");
static_assert(E / kSmallExp == 2 * kSmallTok, "one row job (n1 or n2 of a token) per CTA of a group");

__global__ void __launch_bounds__(256) route_small_kernel(RouteParams p, Buffers b) {
  // W' of expert ee, column group q (8 columns) as two float4 halves at wp[ee][half][q], so that
  // lanes reading groups q = lane + 32 k hit consecutive 16-byte words. Phase 3 reuses the space
  // for the experts' token masks.
  __shared__ float4 wp[kSmallExp][2][H / 8];
  __shared__ int ticket_s;
  __shared__ float pes_s[E];
  __shared__ int scan_s[E + 1];
  __shared__ int tscan_s[E + 1];
  __shared__ int role_s;
  unsigned long long* mask_s = reinterpret_cast<unsigned long long*>(&wp[0][0][0]);  // [128], phase 3
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int e0 = blockIdx.x * kSmallExp, g = blockIdx.y;
  pdl_wait();
  pdl_launch_dependents();
  const int t0 = g * kSmallTok + 2 * warp;
  const int nt = t0 >= p.T ? 0 : (t0 + 1 < p.T ? 2 : 1);
  // The token rows first (their latency overlaps the fold), then W' of the CTA's experts and
  // per_expert_scale.
  uint4 xv[2][11];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    const uint4* xr = reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(u < nt ? t0 + u : 0) * H);
#pragma unroll
    for (int k = 0; k < 11; ++k) xv[u][k] = u < nt ? xr[lane + 32 * k] : make_uint4(0u, 0u, 0u, 0u);
  }
  {
    const float4* gr = reinterpret_cast<const float4*>(p.router_norm_w);
    for (int i = tid; i < H / 4; i += 256) {
      const float4 gv = gr[i];
#pragma unroll
      for (int ee = 0; ee < kSmallExp; ++ee) {
        const float4 w = reinterpret_cast<const float4*>(p.router_w + static_cast<size_t>(e0 + ee) * H)[i];
        wp[ee][i & 1][i >> 1] =
            make_float4(w.x * (1.0f + gv.x), w.y * (1.0f + gv.y), w.z * (1.0f + gv.z), w.w * (1.0f + gv.w));
      }
    }
  }
  if (tid < E) pes_s[tid] = p.per_expert_scale[tid];
  __syncthreads();
  {
    float acc[2][kSmallExp];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int ee = 0; ee < kSmallExp; ++ee) acc[u][ee] = 0.0f;
#pragma unroll
    for (int k = 0; k < 11; ++k) {
#pragma unroll
      for (int ee = 0; ee < kSmallExp; ++ee) {
        const float4 w0 = wp[ee][0][lane + 32 * k], w1 = wp[ee][1][lane + 32 * k];
        const float wv[8] = {w0.x, w0.y, w0.z, w0.w, w1.x, w1.y, w1.z, w1.w};
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const uint32_t x4[4] = {xv[u][k].x, xv[u][k].y, xv[u][k].z, xv[u][k].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            acc[u][ee] = fmaf(bf16_lo(x4[j]), wv[2 * j], acc[u][ee]);
            acc[u][ee] = fmaf(bf16_hi(x4[j]), wv[2 * j + 1], acc[u][ee]);
          }
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int ee = 0; ee < kSmallExp; ++ee) {
        acc[u][ee] = warp_sum(acc[u][ee]);
        if (lane == u * kSmallExp + ee && u < nt) b.logits_part[static_cast<size_t>(t0 + u) * E + e0 + ee] = acc[u][ee];
      }
  }
  // Ticket of the token group: its last CTA goes on to phase 2.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(b.small_ctr + g, 1);
    ticket_s = ticket;
    role_s = ticket == static_cast<int>(gridDim.x) - 1;
    if (role_s) b.small_ctr[g] = 0;  // every CTA of the group has drawn its ticket
  }
  // 1 / RMS of the two tokens (phase 2 takes it from here).
  float inv[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) inv[u] = token_inv_rms(xv[u], p.eps);
  __syncthreads();
  if (!role_s) {
    // Row jobs: job j is row j & 1 (n1, n2) of token 16 g + j / 2; ticket k takes job k, and the
    // ticket before the last also job 31.
    const int ticket = ticket_s;
    const int job = warp == 0 ? ticket : (warp == 1 && ticket == static_cast<int>(gridDim.x) - 2) ? ticket + 1 : -1;
    if (job >= 0) {
      const int t = g * kSmallTok + (job >> 1);
      if (t < p.T) write_norm_row(p, b, t, job & 1, lane);
    }
    return;
  }
  __threadfence();

  // Phase 2: the group's sums (stored by 32 CTAs: L2-coherent loads), the routing.
  {
    float z[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int j = 0; j < 4; ++j)
        z[u][j] = u < nt ? 0.0f + __ldcg(b.logits_part + static_cast<size_t>(t0 + u) * E + lane + 32 * j) : 0.0f;
    float* const rows[2] = {nt > 0 ? b.logits + static_cast<size_t>(t0) * E : nullptr,
                            nt > 1 ? b.logits + static_cast<size_t>(t0 + 1) * E : nullptr};
    int sel[2];
    float wsel[2], gap[2];
    route_tokens<2>(z, inv, p.router_scale, rows, pes_s, lane, sel, wsel, gap);
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (u < nt) {
        if (lane < K) {
          b.topk_idx[static_cast<size_t>(t0 + u) * K + lane] = sel[u];
          b.topk_w[static_cast<size_t>(t0 + u) * K + lane] = wsel[u];
        }
        if (lane == 0) b.gap[t0 + u] = gap[u];
      }
  }
  // Ticket of phase 3.
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    const int ticket = atomicAdd(b.small_ctr + kSmallFinal, 1);
    role_s = ticket == static_cast<int>(gridDim.y) - 1;
    if (role_s) b.small_ctr[kSmallFinal] = 0;
  }
  __syncthreads();
  if (!role_s) return;
  __threadfence();

  // Phase 3: slot s = 8 t + k, two per thread (S <= 512).
  if (tid < E) mask_s[tid] = 0ull;
  __syncthreads();
  const int S = p.T * K;
  int se[2];
  float sw[2];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int sl = tid + 256 * i;
    se[i] = -1;
    sw[i] = 0.0f;
    if (sl < S) {
      se[i] = __ldcg(b.topk_idx + sl);
      sw[i] = __ldcg(b.topk_w + sl);
      if (se[i] < 0 || se[i] >= E) {
        atomicOr(b.status, kStatusBadIndex);
        se[i] = -1;
      } else {
        atomicOr(&mask_s[se[i]], 1ull << (sl >> 3));
      }
    }
  }
  __syncthreads();
  if (warp == 0) {
    int cnt[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) cnt[j] = __popcll(mask_s[lane * 4 + j]);
    expert_scan(cnt, p, b, scan_s, tscan_s, lane);
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int sl = tid + 256 * i;
    if (se[i] < 0) continue;
    const int t = sl >> 3;
    const int pos = scan_s[se[i]] + __popcll(mask_s[se[i]] & ((1ull << t) - 1ull));
    b.perm[pos] = t;
    b.w_sorted[pos] = sw[i];
    b.slot_pos[sl] = pos;
  }
  if (tid < E) expert_tiles(tid, p, b, scan_s, tscan_s);
}

// ------------------------------------------------------------------------------------------
// K3: stable scatter of the slots. A CTA takes 256 consecutive tokens (8 warps of 32); a slot's
// rank inside its expert is the number of earlier tokens of the CTA that chose the same expert
// (from per-warp bit masks), on top of the base the top-k kernel computed for the CTA.
__global__ void __launch_bounds__(256) route_scatter_kernel(RouteParams p, Buffers b) {
  __shared__ uint32_t mask_s[8][E];
  __shared__ int pre_s[8][E];
  __shared__ int base_s[E];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  for (int i = tid; i < 8 * E; i += 256) (&mask_s[0][0])[i] = 0u;
  pdl_wait();
  pdl_launch_dependents();
  const int b0 = blockIdx.x;
  const int t = b0 * kScatterTok + warp * 32 + lane;
  const bool valid = t < p.T;
  // Every load this CTA needs is issued here, so that it waits for memory once: the token's expert
  // ids and weights (16-byte vectors) and the CTA's base positions.
  int4 ia = make_int4(0, 0, 0, 0), ib = ia;
  float4 wa = make_float4(0.0f, 0.0f, 0.0f, 0.0f), wb = wa;
  if (valid) {
    ia = *reinterpret_cast<const int4*>(b.topk_idx + static_cast<size_t>(t) * K);
    ib = *reinterpret_cast<const int4*>(b.topk_idx + static_cast<size_t>(t) * K + 4);
    wa = *reinterpret_cast<const float4*>(b.topk_w + static_cast<size_t>(t) * K);
    wb = *reinterpret_cast<const float4*>(b.topk_w + static_cast<size_t>(t) * K + 4);
  }
  if (tid < E) base_s[tid] = b.base[b0 * E + tid];
  __syncthreads();
  int ids[K] = {ia.x, ia.y, ia.z, ia.w, ib.x, ib.y, ib.z, ib.w};
  const float ws[K] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (valid) {
      if (ids[k] < 0 || ids[k] >= E) {
        atomicOr(b.status, kStatusBadIndex);
        ids[k] = -1;
      } else {
        atomicOr(&mask_s[warp][ids[k]], 1u << lane);
      }
    }
  }
  __syncthreads();
  if (tid < E) {
    int run = 0;
#pragma unroll
    for (int w = 0; w < 8; ++w) {
      pre_s[w][tid] = run;
      run += __popc(mask_s[w][tid]);
    }
  }
  __syncthreads();
  if (!valid) return;
  const uint32_t lt = (1u << lane) - 1u;
  const int S = p.T * K;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const int e = ids[k];
    if (e < 0) continue;
    const int pos = base_s[e] + pre_s[warp][e] + __popc(mask_s[warp][e] & lt);
    if (pos < 0 || pos >= S) {
      atomicOr(b.status, kStatusBadIndex);
      continue;
    }
    b.perm[pos] = t;
    b.w_sorted[pos] = ws[k];
    b.slot_pos[static_cast<size_t>(t) * K + k] = pos;
  }
}

// ------------------------------------------------------------------------------------------
// K6: one CTA per token. The expert branch is the sum of the token's 8 weighted expert outputs
// in ascending expert id; in the full layer it is normalised by post_feedforward_layernorm_2, the
// shared-MLP output by post_feedforward_layernorm_1, their sum by post_feedforward_layernorm, the
// residual is added and the result multiplied by layer_scalar.
// Sum over the CTA of one or two values per thread; every thread gets the totals.
__device__ __forceinline__ float2 block_sum2(float2 v, float2* red) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v.x = warp_sum(v.x);
  v.y = warp_sum(v.y);
  __syncthreads();  // red may still be read by the previous reduction
  if (lane == 0) red[warp] = v;
  __syncthreads();
  float2 s = make_float2(0.0f, 0.0f);
#pragma unroll
  for (int w = 0; w < kCombineThreads / 32; ++w) {
    s.x += red[w].x;
    s.y += red[w].y;
  }
  return s;
}

// The block's output for 8 features f..f+7 of one token (a CTA per token, kCombineThreads threads
// of 8 features): in the full layer, RMSNorm(d; post_feedforward_layernorm_1) +
// RMSNorm(moe; post_feedforward_layernorm_2), normalised by post_feedforward_layernorm, plus the
// residual x, times layer_scalar; in the experts-only mode the expert sum itself. bf16.
__device__ __forceinline__ uint4 block_output(const CombineParams& p, const float (&dv)[8], const float (&moe)[8],
                                              const uint4 xv, int f, float2* red) {
  if (!p.full_layer)
    return make_uint4(pack_bf16(moe[0], moe[1]), pack_bf16(moe[2], moe[3]), pack_bf16(moe[4], moe[5]),
                      pack_bf16(moe[6], moe[7]));
  float sd = 0.0f, sm = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sd = fmaf(dv[j], dv[j], sd);
    sm = fmaf(moe[j], moe[j], sm);
  }
  const float2 r = block_sum2(make_float2(sd, sm), red);
  const float inv_d = 1.0f / sqrtf(r.x / static_cast<float>(H) + p.eps);
  const float inv_m = 1.0f / sqrtf(r.y / static_cast<float>(H) + p.eps);
  const float4 g1a = *reinterpret_cast<const float4*>(p.post_ff_ln_1 + f);
  const float4 g1b = *reinterpret_cast<const float4*>(p.post_ff_ln_1 + f + 4);
  const float4 g2a = *reinterpret_cast<const float4*>(p.post_ff_ln_2 + f);
  const float4 g2b = *reinterpret_cast<const float4*>(p.post_ff_ln_2 + f + 4);
  const float g1[8] = {g1a.x, g1a.y, g1a.z, g1a.w, g1b.x, g1b.y, g1b.z, g1b.w};
  const float g2[8] = {g2a.x, g2a.y, g2a.z, g2a.w, g2b.x, g2b.y, g2b.z, g2b.w};
  float sv[8];
  float ss = 0.0f;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    sv[j] = dv[j] * inv_d * (1.0f + g1[j]) + moe[j] * inv_m * (1.0f + g2[j]);
    ss = fmaf(sv[j], sv[j], ss);
  }
  const float inv_s = 1.0f / sqrtf(block_sum2(make_float2(ss, 0.0f), red).x / static_cast<float>(H) + p.eps);
  const float4 g3a = *reinterpret_cast<const float4*>(p.post_ff_ln + f);
  const float4 g3b = *reinterpret_cast<const float4*>(p.post_ff_ln + f + 4);
  const float g3[8] = {g3a.x, g3a.y, g3a.z, g3a.w, g3b.x, g3b.y, g3b.z, g3b.w};
  const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
  uint32_t ow[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float lo = (bf16_lo(xw[j]) + sv[2 * j] * inv_s * (1.0f + g3[2 * j])) * p.layer_scalar;
    const float hi = (bf16_hi(xw[j]) + sv[2 * j + 1] * inv_s * (1.0f + g3[2 * j + 1])) * p.layer_scalar;
    ow[j] = pack_bf16(lo, hi);
  }
  return make_uint4(ow[0], ow[1], ow[2], ow[3]);
}

// One CTA per token, 8 features per thread. Every load that does not depend on another is issued
// before the first use: the token's 8 slot positions, then its 8 rows of y, d and x, so the CTA
// waits for memory about twice (positions, then rows) rather than once per load.
__global__ void __launch_bounds__(kCombineThreads, 3) combine_kernel(CombineParams p, Buffers b) {
  __shared__ float2 red[kCombineThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  const int f = tid * 8;
  pdl_wait();
  pdl_launch_dependents();
  const int4 pa = *reinterpret_cast<const int4*>(b.slot_pos + static_cast<size_t>(t) * K);
  const int4 pb = *reinterpret_cast<const int4*>(b.slot_pos + static_cast<size_t>(t) * K + 4);
  float dv[8];
  uint4 xv = make_uint4(0u, 0u, 0u, 0u);
  if (p.full_layer) {
    const uint4 dd = __ldcs(reinterpret_cast<const uint4*>(b.d + static_cast<size_t>(t) * H + f));
    const uint32_t d4[4] = {dd.x, dd.y, dd.z, dd.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      dv[2 * j] = bf16_lo(d4[j]);
      dv[2 * j + 1] = bf16_hi(d4[j]);
    }
    xv = *reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H + f);
  }
  int pos[K] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
  const int n_slots = p.T * K;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (pos[k] < 0 || pos[k] >= n_slots) {
      if (tid == 0) atomicOr(b.status, kStatusBadIndex);
      pos[k] = 0;
    }
  }
  uint4 yv[K];
#pragma unroll
  for (int k = 0; k < K; ++k) yv[k] = __ldcs(reinterpret_cast<const uint4*>(b.y + static_cast<size_t>(pos[k]) * H + f));
  // The 8 expert outputs in ascending expert id (the order of the token's slots).
  float moe[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) moe[j] = 0.0f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    const uint32_t w4[4] = {yv[k].x, yv[k].y, yv[k].z, yv[k].w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      moe[2 * j] += bf16_lo(w4[j]);
      moe[2 * j + 1] += bf16_hi(w4[j]);
    }
  }
  *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * H + f) = block_output(p, dv, moe, xv, f, red);
}

// ------------------------------------------------------------------------------------------
// Expert-parallel shards ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2", section
// "The traceable trick": each rank owns a contiguous group of experts and the ranks' expert
// outputs are summed). A shard forward ends with combine_shard_kernel: per token, the sum of its
// weighted expert outputs over the slots whose expert lies in [e_lo, e_hi), in ascending expert
// id, in fp32 (the block's expert branch before post_feedforward_layernorm_2, which is not linear,
// so the ranks add these partials before it); and, on the rank that ran the shared MLP, its
// output d widened to fp32. finish_kernel then takes the summed partials and d and applies the
// rest of the block with the combine's own arithmetic (block_output).
__global__ void __launch_bounds__(kCombineThreads, 3) combine_shard_kernel(ShardParams p, Buffers b) {
  const int t = blockIdx.x, tid = threadIdx.x;
  const int f = tid * 8;
  pdl_wait();
  pdl_launch_dependents();
  const int4 pa = *reinterpret_cast<const int4*>(b.slot_pos + static_cast<size_t>(t) * K);
  const int4 pb = *reinterpret_cast<const int4*>(b.slot_pos + static_cast<size_t>(t) * K + 4);
  const int4 ea = *reinterpret_cast<const int4*>(b.topk_idx + static_cast<size_t>(t) * K);
  const int4 eb = *reinterpret_cast<const int4*>(b.topk_idx + static_cast<size_t>(t) * K + 4);
  const int pos[K] = {pa.x, pa.y, pa.z, pa.w, pb.x, pb.y, pb.z, pb.w};
  const int ex[K] = {ea.x, ea.y, ea.z, ea.w, eb.x, eb.y, eb.z, eb.w};
  const int n_slots = p.T * K;
  float moe[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) moe[j] = 0.0f;
#pragma unroll
  for (int k = 0; k < K; ++k) {
    if (ex[k] < p.e_lo || ex[k] >= p.e_hi) continue;
    if (pos[k] < 0 || pos[k] >= n_slots) {
      if (tid == 0) atomicOr(b.status, kStatusBadIndex);
      continue;
    }
    const uint4 yv = __ldcs(reinterpret_cast<const uint4*>(b.y + static_cast<size_t>(pos[k]) * H + f));
    const uint32_t w4[4] = {yv.x, yv.y, yv.z, yv.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      moe[2 * j] += bf16_lo(w4[j]);
      moe[2 * j + 1] += bf16_hi(w4[j]);
    }
  }
  float4* mo = reinterpret_cast<float4*>(p.moe_out + static_cast<size_t>(t) * H + f);
  mo[0] = make_float4(moe[0], moe[1], moe[2], moe[3]);
  mo[1] = make_float4(moe[4], moe[5], moe[6], moe[7]);
  if (p.dense_out) {
    const uint4 dd = __ldcs(reinterpret_cast<const uint4*>(b.d + static_cast<size_t>(t) * H + f));
    float4* dof = reinterpret_cast<float4*>(p.dense_out + static_cast<size_t>(t) * H + f);
    dof[0] = make_float4(bf16_lo(dd.x), bf16_hi(dd.x), bf16_lo(dd.y), bf16_hi(dd.y));
    dof[1] = make_float4(bf16_lo(dd.z), bf16_hi(dd.z), bf16_lo(dd.w), bf16_hi(dd.w));
  }
}

__global__ void __launch_bounds__(kCombineThreads, 3) finish_kernel(CombineParams p, const float* moe_sum,
                                                                    const float* dense) {
  __shared__ float2 red[kCombineThreads / 32];
  const int t = blockIdx.x, tid = threadIdx.x;
  const int f = tid * 8;
  pdl_wait();
  pdl_launch_dependents();
  const float4* mi = reinterpret_cast<const float4*>(moe_sum + static_cast<size_t>(t) * H + f);
  const float4 m0 = mi[0], m1 = mi[1];
  const float moe[8] = {m0.x, m0.y, m0.z, m0.w, m1.x, m1.y, m1.z, m1.w};
  float dv[8] = {0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f, 0.0f};
  uint4 xv = make_uint4(0u, 0u, 0u, 0u);
  if (p.full_layer) {
    const float4* di = reinterpret_cast<const float4*>(dense + static_cast<size_t>(t) * H + f);
    const float4 d0 = di[0], d1 = di[1];
    dv[0] = d0.x; dv[1] = d0.y; dv[2] = d0.z; dv[3] = d0.w;
    dv[4] = d1.x; dv[5] = d1.y; dv[6] = d1.z; dv[7] = d1.w;
    xv = *reinterpret_cast<const uint4*>(p.x + static_cast<size_t>(t) * H + f);
  }
  *reinterpret_cast<uint4*>(p.out + static_cast<size_t>(t) * H + f) = block_output(p, dv, moe, xv, f, red);
}

}  // namespace

cudaError_t launch_combine_shard(const ShardParams& p, const Buffers& b, cudaStream_t s) {
  return launch_pdl(combine_shard_kernel, dim3(p.T), dim3(kCombineThreads), 0, s, p, b);
}

cudaError_t launch_finish(const CombineParams& p, const float* moe_sum, const float* dense, cudaStream_t s) {
  return launch_pdl(finish_kernel, dim3(p.T), dim3(kCombineThreads), 0, s, p, moe_sum, dense);
}

cudaError_t launch_route_topk(const RouteParams& p, const Buffers& b, cudaStream_t s) {
  const int tb = 8 * p.tpw;
  return launch_pdl(route_topk_kernel, dim3((p.T + tb - 1) / tb), dim3(256), 0, s, p, b);
}

cudaError_t launch_route_small(const RouteParams& p, const Buffers& b, cudaStream_t s) {
  if (p.T < 1 || p.T > kRouteSmallT) return cudaErrorInvalidValue;
  return launch_pdl(route_small_kernel, dim3(E / kSmallExp, (p.T + kSmallTok - 1) / kSmallTok), dim3(256), 0, s, p, b);
}

cudaError_t launch_route_scatter(const RouteParams& p, const Buffers& b, cudaStream_t s) {
  return launch_pdl(route_scatter_kernel, dim3((p.T + kScatterTok - 1) / kScatterTok), dim3(256), 0, s, p, b);
}

cudaError_t launch_combine(const CombineParams& p, const Buffers& b, cudaStream_t s) {
  return launch_pdl(combine_kernel, dim3(p.T), dim3(kCombineThreads), 0, s, p, b);
}

}  // namespace moe
