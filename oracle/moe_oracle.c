/*
 * moe_oracle.c — the oracle (test infrastructure only; see moe_oracle.h for sources and
 * precision). Plain loops, one token at a time, in the order the pages describe the block:
 *
 *   residual x
 *   ├─ dense:  pre_feedforward_layernorm   → shared MLP (D)        → post_feedforward_layernorm_1
 *   └─ expert: pre_feedforward_layernorm_2 → router → K of E experts → post_feedforward_layernorm_2
 *   hidden = dense + expert → post_feedforward_layernorm → + residual → × layer_scalar
 *
 * ([MoE] "The architecture: a dual-path FFN nobody warned me about"; [Port] §4.6 for layer_scalar.)
 * Built with -ffp-contract=off so that no multiply-add is fused and x86 and Arm hosts give the
 * same bits.
 */
#include "moe_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the upper half of an IEEE fp32 word, so widening is exact. */
static float bf16_to_f32(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

/* [Port] §4.5: 0.5*x*(1+tanh(0.7978845608*(x + 0.044715*x^3))). */
double moe_oracle_gelu_tanh(double x) {
  return 0.5 * x * (1.0 + tanh(0.7978845608 * (x + 0.044715 * x * x * x)));
}

/* Gemma RMSNorm (x / rms(x) * (1 + w)), fp64. */
void moe_oracle_rmsnorm(const double* v, const float* w, int n, double eps, double* out) {
  double ss = 0.0;
  for (int i = 0; i < n; ++i) ss += v[i] * v[i];
  double inv = 1.0 / sqrt(ss / (double)n + eps);
  for (int i = 0; i < n; ++i) out[i] = v[i] * inv * (1.0 + (double)w[i]);
}

/* The router of one token, fp32 ([MoE] "The architecture": its own RMSNorm + a scale, then
 * softmax over the experts in fp32 → top-K → renormalise → × per_expert_scale).
 * xin: the router's input vector [H] in fp32. Writes logits[E], probs[E], the K selected experts
 * in ascending id with their renormalised and scaled weights, and the K-th/(K+1)-th logit gap. */
static void route_one(const moe_oracle_dims* d, const float* xin, const moe_oracle_weights* w,
                      float* r, float* logits, float* probs, int32_t* idx, float* wren,
                      float* wfin, float* gap) {
  const int H = d->hidden, E = d->n_experts, K = d->top_k;

  /* RMSNorm of the router input, then the scalar scale. */
  float ss = 0.0f;
  for (int h = 0; h < H; ++h) ss += xin[h] * xin[h];
  float inv = 1.0f / sqrtf(ss / (float)H + d->eps);
  for (int h = 0; h < H; ++h) r[h] = xin[h] * inv * (1.0f + w->router_norm_w[h]) * d->router_scale;

  /* Projection to one logit per expert. */
  for (int e = 0; e < E; ++e) {
    const float* row = w->router_w + (size_t)e * H;
    float acc = 0.0f;
    for (int h = 0; h < H; ++h) acc += r[h] * row[h];
    logits[e] = acc;
  }

  /* Softmax with the maximum subtracted. */
  float m = logits[0];
  for (int e = 1; e < E; ++e)
    if (logits[e] > m) m = logits[e];
  float z = 0.0f;
  for (int e = 0; e < E; ++e) {
    probs[e] = expf(logits[e] - m);
    z += probs[e];
  }
  for (int e = 0; e < E; ++e) probs[e] = probs[e] / z;

  /* Top-K by logit (softmax is monotone in the logit), larger first, lower id first on equal
   * logits: K+1 rounds of arg-max over the experts not yet taken. */
  int taken[1024];
  int order[1025];
  for (int e = 0; e < E; ++e) taken[e] = 0;
  int rounds = (K < E) ? K + 1 : K;
  for (int j = 0; j < rounds; ++j) {
    int best = -1;
    for (int e = 0; e < E; ++e) {
      if (taken[e]) continue;
      if (best < 0 || logits[e] > logits[best]) best = e; /* '>' keeps the lower id on ties */
    }
    taken[best] = 1;
    order[j] = best;
  }
  *gap = (K < E) ? logits[order[K - 1]] - logits[order[K]] : 0.0f;

  /* The selected set, listed in ascending expert id. */
  int n = 0;
  for (int e = 0; e < E; ++e) {
    int sel = 0;
    for (int j = 0; j < K; ++j)
      if (order[j] == e) sel = 1;
    if (sel) idx[n++] = e;
  }

  /* Renormalise the selected probabilities to sum 1, then multiply by per_expert_scale. */
  float s = 0.0f;
  for (int j = 0; j < K; ++j) s += probs[idx[j]];
  for (int j = 0; j < K; ++j) {
    wren[j] = probs[idx[j]] / s;
    wfin[j] = wren[j] * w->per_expert_scale[idx[j]];
  }
}

/* The E2M1 magnitudes, by the 3-bit magnitude code. */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

/* Element (row, col) of an expert weight matrix with `cols` columns: the bf16 value; or, when the
 * int8 form is given, q * scale of the row (exact in fp64: q has 8 bits, scale 24); or, when the
 * MXFP4 form is given, the E2M1 value of its code times its block's power-of-two scale (exact). */
static double expert_weight(const uint16_t* bf, const int8_t* q, const float* scale, const uint8_t* f4,
                            const uint8_t* f4s, size_t row, size_t col, size_t cols) {
  if (f4) {
    const uint8_t byte = f4[row * (cols / 2) + col / 2];
    const int code = (col & 1) ? (byte >> 4) : (byte & 15);
    const double mag = kE2M1[code & 7];
    const int e = (int)f4s[row * (cols / 32) + col / 32] - 127;
    return ldexp((code & 8) ? -mag : mag, e);
  }
  if (q) return (double)q[row * cols + col] * (double)scale[row];
  return (double)bf16_to_f32(bf[row * cols + col]);
}

/* One expert's MLP on input v[H] ([MoE] "The architecture": fused gate_up [E,2I,H], down [E,H,I];
 * [Lab] gelu_pytorch_tanh): hvec = gelu_tanh(gate·v) * (up·v), y = down·hvec. With the int8 form
 * ([MoE] "Can it run on a smaller box?": per-channel symmetric int8 experts) each weight is
 * q * scale of its output row. */
static void expert_mlp(const moe_oracle_dims* d, const moe_oracle_weights* w, int e,
                       const double* v, double* hvec, double* y) {
  const int H = d->hidden, I = d->moe_inter;
  const size_t g0 = (size_t)e * 2 * I;  /* first gate_up row of expert e */
  for (int i = 0; i < I; ++i) {
    double g = 0.0, u = 0.0;
    for (int h = 0; h < H; ++h) {
      g += expert_weight(w->gate_up, w->gate_up_q, w->gate_up_scale, w->gate_up_f4, w->gate_up_f4s, g0 + i, h, H) * v[h];
      u += expert_weight(w->gate_up, w->gate_up_q, w->gate_up_scale, w->gate_up_f4, w->gate_up_f4s, g0 + I + i, h, H) * v[h];
    }
    hvec[i] = moe_oracle_gelu_tanh(g) * u;
  }
  const size_t d0 = (size_t)e * H;  /* first down row of expert e */
  for (int h = 0; h < H; ++h) {
    double acc = 0.0;
    for (int i = 0; i < I; ++i) acc += expert_weight(w->down, w->down_q, w->down_scale, w->down_f4, w->down_f4s, d0 + h, i, I) * hvec[i];
    y[h] = acc;
  }
}

/* The shared dense MLP ([MoE] "The architecture": mlp (2112)), same gating as the experts. */
static void dense_mlp(const moe_oracle_dims* d, const moe_oracle_weights* w, const double* v,
                      double* hvec, double* y) {
  const int H = d->hidden, D = d->dense_inter;
  for (int i = 0; i < D; ++i) {
    double g = 0.0, u = 0.0;
    for (int h = 0; h < H; ++h) {
      g += (double)bf16_to_f32(w->dense_gate[(size_t)i * H + h]) * v[h];
      u += (double)bf16_to_f32(w->dense_up[(size_t)i * H + h]) * v[h];
    }
    hvec[i] = moe_oracle_gelu_tanh(g) * u;
  }
  for (int h = 0; h < H; ++h) {
    double acc = 0.0;
    for (int i = 0; i < D; ++i) acc += (double)bf16_to_f32(w->dense_down[(size_t)h * D + i]) * hvec[i];
    y[h] = acc;
  }
}

static int dims_ok(const moe_oracle_dims* d) {
  if (!d) return 0;
  if (d->hidden < 1 || d->n_experts < 1 || d->n_experts > 1024) return 0;
  if (d->top_k < 1 || d->top_k > d->n_experts) return 0;
  if (d->moe_inter < 1) return 0;
  if (d->full_layer && d->dense_inter < 1) return 0;
  if (!(d->eps > 0.0f)) return 0;
  return 1;
}

int moe_oracle_forward(const moe_oracle_dims* d, int T, const uint16_t* x,
                       const moe_oracle_weights* w, const moe_oracle_outputs* o, int masked_dense) {
  if (!dims_ok(d) || T < 0 || !w || !o || (T > 0 && !x)) return -1;
  if ((!w->gate_up && !(w->gate_up_q && w->gate_up_scale) && !(w->gate_up_f4 && w->gate_up_f4s)) ||
      (!w->down && !(w->down_q && w->down_scale) && !(w->down_f4 && w->down_f4s)))
    return -1;
  if ((w->gate_up_f4 && d->hidden % 32 != 0) || (w->down_f4 && d->moe_inter % 32 != 0)) return -1;
  const int H = d->hidden, E = d->n_experts, K = d->top_k, I = d->moe_inter;
  const int D = d->full_layer ? d->dense_inter : 1;
  int bad = 0;

#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
  for (int t = 0; t < T; ++t) {
    double* xd = malloc(sizeof(double) * H);
    double* n1 = malloc(sizeof(double) * H);
    double* n2 = malloc(sizeof(double) * H);
    double* moe = malloc(sizeof(double) * H);
    double* y = malloc(sizeof(double) * H);
    double* dn = malloc(sizeof(double) * H);
    double* hv = malloc(sizeof(double) * (I > D ? I : D));
    float* xin = malloc(sizeof(float) * H);
    float* r = malloc(sizeof(float) * H);
    float* logits = malloc(sizeof(float) * E);
    float* probs = malloc(sizeof(float) * E);
    int32_t* idx = malloc(sizeof(int32_t) * K);
    float* wren = malloc(sizeof(float) * K);
    float* wfin = malloc(sizeof(float) * K);
    if (!xd || !n1 || !n2 || !moe || !y || !dn || !hv || !xin || !r || !logits || !probs || !idx ||
        !wren || !wfin) {
      bad |= 1;
    } else {
      for (int h = 0; h < H; ++h) xd[h] = (double)bf16_to_f32(x[(size_t)t * H + h]);

      /* Branch inputs: the two pre-norms in the full layer; raw x for the experts otherwise. */
      if (d->full_layer) {
        moe_oracle_rmsnorm(xd, w->pre_ff_ln, H, (double)d->eps, n1);
        moe_oracle_rmsnorm(xd, w->pre_ff_ln_2, H, (double)d->eps, n2);
      } else {
        for (int h = 0; h < H; ++h) n2[h] = xd[h];
      }

      /* Router input: the layer input x, or (alternative reading) pre_feedforward_layernorm_2(x). */
      for (int h = 0; h < H; ++h)
        xin[h] = (d->full_layer && d->router_reads_pre2) ? (float)n2[h] : (float)xd[h];
      float gap;
      route_one(d, xin, w, r, logits, probs, idx, wren, wfin, &gap);

      /* Expert branch: sum over experts in ascending id, starting from +0. */
      for (int h = 0; h < H; ++h) moe[h] = 0.0;
      if (!masked_dense) {
        for (int k = 0; k < K; ++k) {
          expert_mlp(d, w, idx[k], n2, hv, y);
          if (o->h_slot)
            for (int i = 0; i < I; ++i) o->h_slot[((size_t)t * K + k) * I + i] = hv[i];
          for (int h = 0; h < H; ++h) {
            double c = (double)wfin[k] * y[h];
            moe[h] += c;
            if (o->y_slot) o->y_slot[((size_t)t * K + k) * H + h] = c;
          }
        }
      } else {
        /* Every expert, weighted by its router weight or by 0 when it is not selected: a
         * non-selected expert adds 0 * y = ±0, which leaves the running sum unchanged. */
        int k = 0;
        for (int e = 0; e < E; ++e) {
          double we = 0.0;
          int is_sel = (k < K && idx[k] == e);
          if (is_sel) we = (double)wfin[k];
          expert_mlp(d, w, e, n2, hv, y);
          if (is_sel && o->h_slot)
            for (int i = 0; i < I; ++i) o->h_slot[((size_t)t * K + k) * I + i] = hv[i];
          for (int h = 0; h < H; ++h) {
            double c = we * y[h];
            moe[h] += c;
            if (is_sel && o->y_slot) o->y_slot[((size_t)t * K + k) * H + h] = c;
          }
          if (is_sel) ++k;
        }
      }

      if (d->full_layer) {
        dense_mlp(d, w, n1, hv, dn);
        if (o->h_dense)
          for (int i = 0; i < D; ++i) o->h_dense[(size_t)t * D + i] = hv[i];
        if (o->dense)
          for (int h = 0; h < H; ++h) o->dense[(size_t)t * H + h] = dn[h];
        if (o->moe)
          for (int h = 0; h < H; ++h) o->moe[(size_t)t * H + h] = moe[h];
        /* post_feedforward_layernorm_1 on the dense branch, _2 on the expert branch, add, then
         * post_feedforward_layernorm, + residual, × layer_scalar. */
        moe_oracle_rmsnorm(dn, w->post_ff_ln_1, H, (double)d->eps, dn);
        moe_oracle_rmsnorm(moe, w->post_ff_ln_2, H, (double)d->eps, moe);
        for (int h = 0; h < H; ++h) y[h] = dn[h] + moe[h];
        moe_oracle_rmsnorm(y, w->post_ff_ln, H, (double)d->eps, y);
        if (o->out)
          for (int h = 0; h < H; ++h)
            o->out[(size_t)t * H + h] = (xd[h] + y[h]) * (double)w->layer_scalar;
      } else {
        if (o->moe)
          for (int h = 0; h < H; ++h) o->moe[(size_t)t * H + h] = moe[h];
        if (o->out)
          for (int h = 0; h < H; ++h) o->out[(size_t)t * H + h] = moe[h];
      }

      if (o->logits) memcpy(o->logits + (size_t)t * E, logits, sizeof(float) * E);
      if (o->probs) memcpy(o->probs + (size_t)t * E, probs, sizeof(float) * E);
      if (o->topk_idx) memcpy(o->topk_idx + (size_t)t * K, idx, sizeof(int32_t) * K);
      if (o->topk_w_renorm) memcpy(o->topk_w_renorm + (size_t)t * K, wren, sizeof(float) * K);
      if (o->topk_w) memcpy(o->topk_w + (size_t)t * K, wfin, sizeof(float) * K);
      if (o->gap) o->gap[t] = gap;
    }
    free(xd); free(n1); free(n2); free(moe); free(y); free(dn); free(hv);
    free(xin); free(r); free(logits); free(probs); free(idx); free(wren); free(wfin);
  }
  return bad ? -1 : 0;
}

int moe_oracle_route(const moe_oracle_dims* d, int T, const uint16_t* x, const moe_oracle_weights* w,
                     const moe_oracle_outputs* o) {
  if (!dims_ok(d) || T < 0 || !w || !o || (T > 0 && !x)) return -1;
  const int H = d->hidden, E = d->n_experts, K = d->top_k;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : bad)
  for (int t = 0; t < T; ++t) {
    double* xd = malloc(sizeof(double) * H);
    double* n2 = malloc(sizeof(double) * H);
    float* xin = malloc(sizeof(float) * H);
    float* r = malloc(sizeof(float) * H);
    float* logits = malloc(sizeof(float) * E);
    float* probs = malloc(sizeof(float) * E);
    int32_t* idx = malloc(sizeof(int32_t) * K);
    float* wren = malloc(sizeof(float) * K);
    float* wfin = malloc(sizeof(float) * K);
    if (!xd || !n2 || !xin || !r || !logits || !probs || !idx || !wren || !wfin) {
      bad |= 1;
    } else {
      for (int h = 0; h < H; ++h) xd[h] = (double)bf16_to_f32(x[(size_t)t * H + h]);
      if (d->full_layer && d->router_reads_pre2) moe_oracle_rmsnorm(xd, w->pre_ff_ln_2, H, (double)d->eps, n2);
      for (int h = 0; h < H; ++h)
        xin[h] = (d->full_layer && d->router_reads_pre2) ? (float)n2[h] : (float)xd[h];
      float gap;
      route_one(d, xin, w, r, logits, probs, idx, wren, wfin, &gap);
      if (o->logits) memcpy(o->logits + (size_t)t * E, logits, sizeof(float) * E);
      if (o->probs) memcpy(o->probs + (size_t)t * E, probs, sizeof(float) * E);
      if (o->topk_idx) memcpy(o->topk_idx + (size_t)t * K, idx, sizeof(int32_t) * K);
      if (o->topk_w_renorm) memcpy(o->topk_w_renorm + (size_t)t * K, wren, sizeof(float) * K);
      if (o->topk_w) memcpy(o->topk_w + (size_t)t * K, wfin, sizeof(float) * K);
      if (o->gap) o->gap[t] = gap;
    }
    free(xd); free(n2); free(xin); free(r); free(logits); free(probs); free(idx); free(wren); free(wfin);
  }
  return bad ? -1 : 0;
}

/* Per-channel symmetric int8 ([MoE] "Can it run on a smaller box?"): one fp32 scale per row,
 * max|w| / 127; each element w / scale rounded to nearest (ties to even) and clamped to ±127. */
int moe_oracle_quantize_int8(const uint16_t* w, long long rows, int cols, int8_t* q, float* scale) {
  if (!w || !q || !scale || rows < 0 || cols < 1) return -1;
  for (long long r = 0; r < rows; ++r) {
    const uint16_t* wr = w + (size_t)r * cols;
    float amax = 0.0f;
    for (int c = 0; c < cols; ++c) {
      const float a = fabsf(bf16_to_f32(wr[c]));
      if (a > amax) amax = a;
    }
    const float s = amax / 127.0f;
    scale[r] = s;
    for (int c = 0; c < cols; ++c) {
      float v = 0.0f;
      if (s > 0.0f) {
        v = rintf(bf16_to_f32(wr[c]) / s);
        if (v > 127.0f) v = 127.0f;
        if (v < -127.0f) v = -127.0f;
      }
      q[(size_t)r * cols + c] = (int8_t)v;
    }
  }
  return 0;
}

/* E2M1 code of v (the element already divided by its block scale): the nearest of the E2M1
 * magnitudes, ties to the even code (the one whose mantissa bit, bit 0 of the code, is 0),
 * magnitudes above 6 saturated to 6; the sign in bit 3, zero as +0. */
static int e2m1_code(double v) {
  const double a = fabs(v);
  int best = 0;
  for (int k = 1; k < 8; ++k) {
    const double dk = fabs(a - kE2M1[k]), db = fabs(a - kE2M1[best]);
    if (dk < db || (dk == db && (k & 1) == 0)) best = k;
  }
  if (a > 6.0) best = 7;
  return (best != 0 && v < 0) ? (best | 8) : best;
}

/* MXFP4 ([MoE] "The fp4 rabbit hole": 32 fp4 values share one scale), read as the OCP
 * Microscaling v1.0 conversion: per block of 32 consecutive elements of a row, a power-of-two
 * scale from the block's largest magnitude, then every element rounded to E2M1. */
int moe_oracle_quantize_mxfp4(const uint16_t* w, long long rows, int cols, uint8_t* codes, uint8_t* scales) {
  if (!w || !codes || !scales || rows < 0 || cols < 32 || cols % 32 != 0) return -1;
  const int nb = cols / 32;
  for (long long r = 0; r < rows; ++r) {
    const uint16_t* wr = w + (size_t)r * cols;
    for (int b = 0; b < nb; ++b) {
      /* 1. the block's largest magnitude */
      double amax = 0.0;
      for (int j = 0; j < 32; ++j) {
        const double a = fabs((double)bf16_to_f32(wr[b * 32 + j]));
        if (a > amax) amax = a;
      }
      /* 2. the shared exponent floor(log2 amax) - emax(E2M1) = ... - 2, in the E8M0 range */
      int se = 0;
      uint8_t sbyte = 0;
      if (amax > 0.0) {
        int ex;
        frexp(amax, &ex); /* amax = m * 2^ex, m in [0.5, 1): floor(log2 amax) = ex - 1 */
        se = (ex - 1) - 2;
        if (se < -127) se = -127;
        if (se > 127) se = 127;
        sbyte = (uint8_t)(se + 127);
      }
      scales[(size_t)r * nb + b] = sbyte;
      /* 3. every element divided by the scale 2^se and rounded to E2M1 */
      for (int j = 0; j < 32; j += 2) {
        int c0 = 0, c1 = 0;
        if (amax > 0.0) {
          c0 = e2m1_code(ldexp((double)bf16_to_f32(wr[b * 32 + j]), -se));
          c1 = e2m1_code(ldexp((double)bf16_to_f32(wr[b * 32 + j + 1]), -se));
        }
        codes[(size_t)r * (cols / 2) + (b * 32 + j) / 2] = (uint8_t)(c0 | (c1 << 4));
      }
    }
  }
  return 0;
}

/* Slots sorted by (expert, token): the gather that precedes each expert's MLP and the scatter
 * back ([MoE] "The architecture": the experts' sparse gather/scatter loop), as a counting sort. */
int moe_oracle_permute(int T, int K, int E, const int32_t* topk_idx, const float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* perm, float* w_sorted,
                       int32_t* slot_pos) {
  if (T < 0 || K < 1 || E < 1 || (T > 0 && !topk_idx) || !counts || !offsets) return -1;
  for (int e = 0; e < E; ++e) counts[e] = 0;
  for (long s = 0; s < (long)T * K; ++s) {
    int e = topk_idx[s];
    if (e < 0 || e >= E) return -1;
    counts[e] += 1;
  }
  offsets[0] = 0;
  for (int e = 0; e < E; ++e) offsets[e + 1] = offsets[e] + counts[e];
  int32_t* next = malloc(sizeof(int32_t) * E);
  if (!next) return -1;
  for (int e = 0; e < E; ++e) next[e] = offsets[e];
  /* Tokens ascending, so within one expert the tokens ascend. */
  for (int t = 0; t < T; ++t) {
    for (int k = 0; k < K; ++k) {
      int e = topk_idx[(size_t)t * K + k];
      int pos = next[e]++;
      if (perm) perm[pos] = t;
      if (w_sorted && topk_w) w_sorted[pos] = topk_w[(size_t)t * K + k];
      if (slot_pos) slot_pos[(size_t)t * K + k] = pos;
    }
  }
  free(next);
  return 0;
}

void moe_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int moe_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
