/*
 * moe_oracle.h — the oracle: a plain, slow CPU implementation of the Gemma-4 26B-A4B dual-path
 * feed-forward block, used as test infrastructure only (tests, the smoke check and the CPU
 * baseline of the benchmark). It shares no code, header or table with the CUDA path and is never
 * part of the product path.
 *
 * Sources, by page and section:
 *   [MoE]   "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2 — where every rank
 *           weighted the wrong experts", section "The architecture: a dual-path FFN nobody warned
 *           me about" (layer diagram, router steps, expert shapes) and section "The traceable
 *           trick: compute all experts, mask to top-8" (the sparse == dense-masked identity).
 *   [Port]  "Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", §4.5 (the tanh form of GELU)
 *           and §4.6 (hidden_states *= layer_scalar, a per-layer buffer).
 *   [Lab]   "Lab 008 — Raw lab detail", "The model under test" (hidden 2816, 128 experts,
 *           moe_intermediate 704, hidden_activation gelu_pytorch_tanh).
 *
 * Precision. The router (its RMSNorm, the projection, the softmax, the top-k choice and the
 * renormalisation) runs in fp32, because [MoE] fixes the softmax at fp32 and the choice of experts
 * must be taken in that precision. Everything after the router (the pre- and post-norms, the
 * expert and shared MLPs, the weighted sum, the residual and layer_scalar) runs in fp64. bf16
 * inputs are widened exactly.
 *
 * Pins. Every function declared here is checked against facts that do not come from the oracle
 * (closed forms, library routines, the sparse == dense-masked identity, an independent float64
 * brute force, the OCP MX rules): tests/test_oracle_pins.py, test_oracle_int8.py and
 * test_oracle_fp4.py; tests/test_oracle_mutants.py checks that those pins fail on plausible
 * mistakes planted in copies of moe_oracle.c. Agreement with the published checkpoint's own
 * activations is parity unpinned: the pages print none and no checkpoint is at hand.
 *
 * Dimensions are arguments, so the same code runs the real shapes and tiny brute-force shapes.
 * All arrays are dense row-major host memory. Tokens are independent and each token is computed
 * serially, so results do not depend on the number of threads.
 */
#ifndef MOE_ORACLE_H
#define MOE_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct moe_oracle_dims {
  int hidden;             /* H */
  int n_experts;          /* E */
  int top_k;              /* K, 1 <= K <= E */
  int moe_inter;          /* I */
  int dense_inter;        /* D (read only when full_layer) */
  int full_layer;         /* 0: router + experts only, out = expert sum; 1: whole layer */
  int router_reads_pre2;  /* 0: the router normalises the layer input x (default reading);
                             1: the router reads pre_feedforward_layernorm_2(x) (alternative) */
  float eps;              /* RMSNorm epsilon */
  float router_scale;     /* scalar on the router's normed input */
} moe_oracle_dims;

typedef struct moe_oracle_weights {
  const float* router_w;          /* [E, H] */
  const float* router_norm_w;     /* [H] */
  const float* per_expert_scale;  /* [E] */
  const uint16_t* gate_up;        /* [E, 2I, H] bf16; rows 0..I-1 gate, I..2I-1 up */
  const uint16_t* down;           /* [E, H, I] bf16 */
  const uint16_t* dense_gate;     /* [D, H] bf16 */
  const uint16_t* dense_up;       /* [D, H] bf16 */
  const uint16_t* dense_down;     /* [H, D] bf16 */
  const float* pre_ff_ln;         /* [H] */
  const float* pre_ff_ln_2;       /* [H] */
  const float* post_ff_ln_1;      /* [H] */
  const float* post_ff_ln_2;      /* [H] */
  const float* post_ff_ln;        /* [H] */
  float layer_scalar;
  /* Optional int8 form of the expert weights ([MoE] "Can it run on a smaller box?": per-channel
   * symmetric int8 experts). When gate_up_q is set, expert weight (row, col) of gate_up is
   * gate_up_q[row, col] * gate_up_scale[row] and gate_up may be NULL; likewise for down. */
  const int8_t* gate_up_q;        /* [E * 2I, H] */
  const float* gate_up_scale;     /* [E * 2I] */
  const int8_t* down_q;           /* [E * H, I] */
  const float* down_scale;        /* [E * H] */
  /* Optional MXFP4 form of the expert weights (the microscaling fp4 format [MoE] "The fp4 rabbit
   * hole" names: blocks of 32 consecutive elements of a row share one scale). When gate_up_f4 is
   * set, expert weight (row, col) of gate_up is e2m1(code) * 2^(gate_up_f4s[row, col / 32] - 127),
   * code = the low nibble of byte gate_up_f4[row, col / 2] for even col, the high nibble for odd
   * col (bit 3 the sign, bits 2..0 the magnitude index into {0, 0.5, 1, 1.5, 2, 3, 4, 6}); gate_up
   * and gate_up_q may then be NULL. Likewise for down. */
  const uint8_t* gate_up_f4;      /* [E * 2I, H / 2] */
  const uint8_t* gate_up_f4s;     /* [E * 2I, H / 32] */
  const uint8_t* down_f4;         /* [E * H, I / 2] */
  const uint8_t* down_f4s;        /* [E * H, I / 32] */
} moe_oracle_weights;

/* Every field may be NULL (not written). Slot (t, k): token t's k-th selected expert, k in
 * ascending expert id. */
typedef struct moe_oracle_outputs {
  double* out;          /* [T, H] block output */
  double* moe;          /* [T, H] expert branch: sum of w_k * y_k before post_feedforward_layernorm_2 */
  double* dense;        /* [T, H] shared MLP output before post_feedforward_layernorm_1 */
  double* h_slot;       /* [T, K, I] gelu_tanh(gate) * up of each slot */
  double* y_slot;       /* [T, K, H] w_k * down(h) of each slot */
  double* h_dense;      /* [T, D] shared MLP activation */
  float* logits;        /* [T, E] router logits */
  float* probs;         /* [T, E] softmax of the logits */
  int32_t* topk_idx;    /* [T, K] selected experts, ascending id */
  float* topk_w_renorm; /* [T, K] renormalised weights (sum 1), same order */
  float* topk_w;        /* [T, K] renormalised weights times per_expert_scale */
  float* gap;           /* [T] K-th largest logit minus (K+1)-th largest (0 if K == E) */
} moe_oracle_outputs;

/* GELU, tanh form ([Port] §4.5). */
double moe_oracle_gelu_tanh(double x);

/* Gemma RMSNorm in fp64: out = v / sqrt(mean(v^2) + eps) * (1 + w). out may equal v. */
void moe_oracle_rmsnorm(const double* v, const float* w, int n, double eps, double* out);

/* The block for T tokens. x: [T, H] bf16. masked_dense = 0 runs the sparse form (only the K
 * selected experts); masked_dense = 1 runs every expert with weight 0 off the top-K ([MoE], "The
 * traceable trick"), which must give the same bits. Returns 0, or -1 on bad arguments. */
int moe_oracle_forward(const moe_oracle_dims* d, int T, const uint16_t* x,
                       const moe_oracle_weights* w, const moe_oracle_outputs* o, int masked_dense);

/* Only the router of the block for T tokens: fills the logits, probs, topk_idx, topk_w_renorm,
 * topk_w and gap fields of *o (the others are ignored), exactly as moe_oracle_forward would.
 * Returns 0, or -1 on bad arguments. */
int moe_oracle_route(const moe_oracle_dims* d, int T, const uint16_t* x, const moe_oracle_weights* w,
                     const moe_oracle_outputs* o);

/* Per-channel symmetric int8 quantisation of a bf16 matrix [rows, cols] (one channel per row):
 * scale[r] = max_c |w[r, c]| / 127 (fp32), q[r, c] = w[r, c] / scale[r] (fp32) rounded to nearest,
 * ties to even, clamped to [-127, 127]; an all-zero row gets scale 0 and q 0. Returns 0, or -1 on
 * bad arguments. */
int moe_oracle_quantize_int8(const uint16_t* w, long long rows, int cols, int8_t* q, float* scale);

/* MXFP4 quantisation of a bf16 matrix [rows, cols] (cols a multiple of 32), after the OCP
 * Microscaling Formats (MX) v1.0 conversion: for each block of 32 consecutive elements of a row,
 * amax = max |w|; if amax > 0 the shared exponent is floor(log2 amax) - 2 (2 = the largest exponent
 * of E2M1), clamped to [-127, 127], and the block scale X = 2^that; each element w / X is rounded to
 * the nearest E2M1 value (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6; ties to the even code), and
 * magnitudes above 6 saturate to 6. A value that rounds to zero is stored as code 0 (+0). An
 * all-zero block gets scale byte 0 and codes 0. scales[r, b] = shared exponent + 127 (E8M0);
 * codes[r, c / 2] holds element c in its low nibble (even c) or high nibble (odd c). Returns 0,
 * or -1 on bad arguments. */
int moe_oracle_quantize_mxfp4(const uint16_t* w, long long rows, int cols, uint8_t* codes, uint8_t* scales);

/* Stable counting sort of the T*K slots by expert: counts[E], offsets[E+1] (exclusive prefix sum,
 * offsets[E] = T*K), perm[T*K] (token of each sorted slot; within one expert tokens ascend),
 * w_sorted[T*K] (topk_w of each sorted slot; may be NULL with topk_w NULL), slot_pos[T*K] (sorted
 * position of slot (t, k)). Returns 0, or -1 on an expert id out of range. */
int moe_oracle_permute(int T, int K, int E, const int32_t* topk_idx, const float* topk_w,
                       int32_t* counts, int32_t* offsets, int32_t* perm, float* w_sorted,
                       int32_t* slot_pos);

/* OpenMP thread control for timing: set (n <= 0 leaves it) and query. */
void moe_oracle_set_threads(int n);
int moe_oracle_max_threads(void);

#ifdef __cplusplus
}
#endif

#endif /* MOE_ORACLE_H */
