/*
 * moe_ffn.h — C ABI of the Gemma-4 26B-A4B sparse MoE feed-forward block on one GB300 (sm_103a).
 *
 * What the block computes is defined by the blog post "Porting a 128-expert MoE (Gemma-4 26B-A4B)
 * to AWS Inferentia2 — where every rank weighted the wrong experts", section "The architecture: a
 * dual-path FFN nobody warned me about": from the post-attention residual x, a dense branch
 * (pre_feedforward_layernorm -> shared MLP of width 2112 -> post_feedforward_layernorm_1) and an
 * expert branch (pre_feedforward_layernorm_2 -> router -> 128 experts of width 704 ->
 * post_feedforward_layernorm_2) are added, normalised by post_feedforward_layernorm, added to the
 * residual and multiplied by layer_scalar. The router has its own RMSNorm, a scale and a
 * per-expert scale; it takes an fp32 softmax over the 128 experts, keeps the top 8, renormalises
 * them to sum 1 and multiplies by per_expert_scale. The experts hold a fused gate_up projection
 * [128,1408,2816] and a down projection [128,2816,704]. The activation is the tanh form of GELU
 * ("Porting Gemma-4 (2B / 4B / 12B) to AWS Inferentia2", §4.5; "Lab 008 — Raw lab detail",
 * "The model under test": hidden_activation=gelu_pytorch_tanh). layer_scalar is a per-layer
 * buffer that weight loaders that copy parameters only silently drop (same page, §4.6), so here it
 * is a required field of the weights with no default.
 *
 * Conventions for every entry point:
 *   - Return value: an int status (MOE_FFN_OK or a negative MOE_FFN_E* code). No entry point
 *     aborts, throws or prints; moe_ffn_status_string() names a code.
 *   - "device pointer" means memory of the CUDA device the context was created on; "host pointer"
 *     means ordinary process memory. Every pointer is borrowed: the library never frees memory it
 *     did not allocate, and the caller keeps each buffer alive while work that uses it is queued.
 *   - A stream argument is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     moe_ffn_forward only enqueues work on that stream: it does not synchronise the host, does
 *     not allocate device memory and does not read anything back to the host.
 *   - Tensors are dense and row-major (last index fastest); bf16 is IEEE bfloat16 stored as 16-bit
 *     words. Every device pointer must be 16-byte aligned (MOE_FFN_EALIGN otherwise).
 *   - There is no CPU fallback: without an sm_103 device the calls fail with MOE_FFN_EARCH or
 *     MOE_FFN_ECUDA.
 */
#ifndef MOE_FFN_H
#define MOE_FFN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
#define MOE_FFN_OK 0
#define MOE_FFN_EINVAL (-1)   /* a NULL pointer, a size out of range or a dimension other than the model's */
#define MOE_FFN_EALIGN (-2)   /* a device pointer not 16-byte aligned */
#define MOE_FFN_ETOOBIG (-3)  /* T above the context's max_tokens, or a workspace smaller than required */
#define MOE_FFN_EARCH (-4)    /* the device is not compute capability 10.3 (sm_103) */
#define MOE_FFN_ECUDA (-5)    /* a CUDA runtime or driver call failed */
#define MOE_FFN_EDEVICE (-6)  /* a kernel gave up a bounded wait or found a bad index and set the status word */

/* Bits of the device status word (moe_ffn_device_status): which bounded wait gave up, or which
 * check rejected an index. Several can be set at once. */
#define MOE_FFN_STATUS_WAIT_FULL 0x1u       /* the MMA issuer gave up waiting for a filled stage */
#define MOE_FFN_STATUS_WAIT_EMPTY 0x2u      /* a producer gave up waiting for a free stage */
#define MOE_FFN_STATUS_WAIT_ACC_FULL 0x4u   /* an epilogue gave up waiting for an accumulator */
#define MOE_FFN_STATUS_WAIT_ACC_EMPTY 0x8u  /* the MMA issuer gave up waiting for a drained accumulator */
#define MOE_FFN_STATUS_BAD_INDEX 0x10u      /* an index read from the workspace was out of range */
#define MOE_FFN_STATUS_BAD_SCHEDULE 0x20u   /* a tile list larger than its buffer */
#define MOE_FFN_STATUS_DRAIN 0x40u          /* an exit drain gave up waiting for work in flight */
#define MOE_FFN_STATUS_WAIT_ITEM 0x80u      /* a GEMM role gave up waiting for its next work item */
#define MOE_FFN_STATUS_WAIT_COPY 0x100u     /* a GEMM producer gave up waiting for the sorted copy of
                                               its token rows (forwards above 3072 tokens) */

/* Modes. */
#define MOE_FFN_MOE_ONLY 0    /* router + experts only: out = sum of the 8 weighted expert outputs */
#define MOE_FFN_FULL_LAYER 1  /* the whole dual-path feed-forward layer with norms, residual, layer_scalar */

/* Model dimensions of Gemma-4 26B-A4B ("Lab 008 — Raw lab detail", "The model under test";
 * top-8 and the gate_up/down shapes from the 26B-A4B post, "The architecture"). The kernels are
 * built for exactly these; moe_ffn_init rejects any other value with MOE_FFN_EINVAL. */
#define MOE_FFN_HIDDEN 2816
#define MOE_FFN_N_EXPERTS 128
#define MOE_FFN_TOP_K 8
#define MOE_FFN_MOE_INTER 704
#define MOE_FFN_DENSE_INTER 2112
#define MOE_FFN_MAX_TOKENS_LIMIT 65536

typedef struct moe_ffn_config {
  int hidden;          /* must be 2816 */
  int n_experts;       /* must be 128 */
  int top_k;           /* must be 8 */
  int moe_inter;       /* must be 704 */
  int dense_inter;     /* must be 2112 */
  int mode;            /* MOE_FFN_MOE_ONLY or MOE_FFN_FULL_LAYER */
  int max_tokens;      /* the largest T a forward call on this context may pass, 1..65536 */
  float eps;           /* RMSNorm epsilon for all six norms, > 0 (1e-6 for this model) */
  float router_scale;  /* scalar applied to the router's normed input, > 0 (2816^-1/2) */
} moe_ffn_config;

/* Weights of one layer. Every pointer is a DEVICE pointer, borrowed. RMSNorm weights are in the
 * Gemma form: a norm multiplies by (1 + w). In MOE_FFN_MOE_ONLY mode the dense and norm fields
 * other than router_norm_w are ignored and may be NULL; layer_scalar is still read and ignored. */
typedef struct moe_ffn_weights {
  const float* router_w;          /* [128, 2816] fp32: router projection, row e gives expert e's logit */
  const float* router_norm_w;     /* [2816] fp32: the router's own RMSNorm weight */
  const float* per_expert_scale;  /* [128] fp32 */
  const uint16_t* gate_up;        /* [128, 1408, 2816] bf16: rows 0..703 gate, rows 704..1407 up */
  const uint16_t* down;           /* [128, 2816, 704] bf16 */
  const uint16_t* dense_gate;     /* [2112, 2816] bf16 (FULL_LAYER) */
  const uint16_t* dense_up;       /* [2112, 2816] bf16 (FULL_LAYER) */
  const uint16_t* dense_down;     /* [2816, 2112] bf16 (FULL_LAYER) */
  const float* pre_ff_ln;         /* [2816] fp32: pre_feedforward_layernorm (dense branch input) */
  const float* pre_ff_ln_2;       /* [2816] fp32: pre_feedforward_layernorm_2 (expert branch input) */
  const float* post_ff_ln_1;      /* [2816] fp32: post_feedforward_layernorm_1 (dense branch output) */
  const float* post_ff_ln_2;      /* [2816] fp32: post_feedforward_layernorm_2 (expert branch output) */
  const float* post_ff_ln;        /* [2816] fp32: post_feedforward_layernorm (after the sum) */
  float layer_scalar;             /* required; multiplies (residual + normed sum) */
  /* Optional int8 experts ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2",
   * section "Can it run on a smaller box?": per-channel symmetric int8). When gate_up_q is not
   * NULL, all four fields must be set; the experts' weights are then q[row, col] * scale[row] and
   * gate_up / down are not read (the shared MLP stays bf16). moe_ffn_quantize_int8 makes them. */
  const int8_t* gate_up_q;        /* [128 * 1408, 2816] int8 */
  const float* gate_up_scale;     /* [128 * 1408] fp32, one per row */
  const int8_t* down_q;           /* [128 * 2816, 704] int8 */
  const float* down_scale;        /* [128 * 2816] fp32, one per row */
  /* Optional MXFP4 experts (the microscaling fp4 format of the same post, section "The fp4 rabbit
   * hole": blocks of 32 consecutive elements of a row share one power-of-two scale). When
   * gate_up_f4 is not NULL, all four fields must be set and the int8 fields must be NULL; expert
   * weight (row, col) is then e2m1(code) * 2^(scale byte - 127), where the code is the low nibble
   * of byte [row, col / 2] for even col and the high nibble for odd col (bit 3 the sign, bits 2..0
   * index the magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) and the scale byte is [row, col / 32] (E8M0).
   * gate_up / down are not read (the shared MLP stays bf16). moe_ffn_quantize_mxfp4 makes them.
   * The forward applies a block's scale exactly for scale bytes 2..252 (what the quantiser gives
   * any block whose largest magnitude is at least 2^-123) and reads all-zero blocks as zero. */
  const uint8_t* gate_up_f4;      /* [128 * 1408, 1408] packed E2M1 codes */
  const uint8_t* gate_up_f4s;     /* [128 * 1408, 88] E8M0 block scales */
  const uint8_t* down_f4;         /* [128 * 2816, 352] packed E2M1 codes */
  const uint8_t* down_f4s;        /* [128 * 2816, 22] E8M0 block scales */
} moe_ffn_weights;

/* Device views into the workspace, filled by moe_ffn_workspace_view. Contents are those of the
 * last forward queued on the context and are valid once that forward has completed, until the
 * next forward. S = 8*T slots; slot (t, k) is token t's k-th selected expert, k ascending in
 * expert id. */
typedef struct moe_ffn_views {
  const float* logits;        /* [T, 128] fp32 router logits */
  const int32_t* topk_idx;    /* [T, 8] selected experts, ascending expert id */
  const float* topk_w;        /* [T, 8] renormalised weights times per_expert_scale, same order */
  const float* gap;           /* [T] 8th-largest minus 9th-largest logit */
  const int32_t* counts;      /* [128] slots per expert */
  const int32_t* offsets;     /* [129] exclusive prefix sum of counts; offsets[128] = S */
  const int32_t* perm;        /* [S] token of each slot in expert-major, token-ascending order */
  const float* w_sorted;      /* [S] the weight of each sorted slot */
  const int32_t* slot_pos;    /* [T, 8] sorted position of slot (t, k) */
  const uint16_t* n1;         /* [T, 2816] bf16 pre_feedforward_layernorm(x) (FULL_LAYER) */
  const uint16_t* n2;         /* [T, 2816] bf16 expert input: pre_feedforward_layernorm_2(x), or x
                               (forwards of at most 3072 tokens or with converted experts; larger
                               ones write it in sorted-slot order into the y buffer instead, which the
                               down GEMM then overwrites) */
  const uint16_t* h;          /* [S, 704] bf16 gelu_tanh(gate) * up per sorted slot */
  const uint16_t* h_dense;    /* [T, 2112] bf16 shared-MLP activation (FULL_LAYER) */
  const uint16_t* y;          /* [S, 2816] bf16 weighted expert output per sorted slot */
  const uint16_t* d;          /* [T, 2816] bf16 shared-MLP output (FULL_LAYER) */
  int T;                      /* tokens of that forward */
} moe_ffn_views;

typedef struct moe_ffn_ctx moe_ffn_ctx;

/* Bytes of device workspace a context with this config needs (0 if the config is invalid). */
size_t moe_ffn_workspace_bytes(const moe_ffn_config* cfg);

/* Creates a context on CUDA device `device` (which this call makes current). `workspace` is a
 * device pointer to at least moe_ffn_workspace_bytes(cfg) bytes, 256-byte aligned, that the
 * context uses for its intermediates; the caller owns it. Several contexts may share one workspace
 * if their forwards never overlap in time (e.g. all on one stream). Fails with MOE_FFN_EARCH on a
 * device other than sm_103. On failure *ctx is set to NULL. */
int moe_ffn_init(moe_ffn_ctx** ctx, const moe_ffn_config* cfg, void* workspace,
                 size_t workspace_bytes, int device);

/* Queues one forward of the block on `stream`: out = block(x) for T tokens, the block being the
 * dual-path layer of "Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS Inferentia2", section "The
 * architecture: a dual-path FFN nobody warned me about" (described at the top of this file). Each
 * expert multiplies only the tokens routed to it; the result equals the post's "compute all
 * experts, mask to top-8" form (section "The traceable trick") up to rounding.
 *   x   device pointer, [T, 2816] bf16, the layer input (the post-attention residual).
 *   T   0..max_tokens; T = 0 queues nothing and returns MOE_FFN_OK.
 *   w   host pointer to a weights struct whose fields are device pointers; the struct is read
 *       during the call, the tensors it names are read by the queued kernels.
 *   out device pointer, [T, 2816] bf16; must not overlap x or the workspace.
 * The result is deterministic: the same inputs give bitwise-equal outputs. Errors found while
 * queueing are returned; errors found by the kernels set the device status word (see
 * moe_ffn_device_status). */
int moe_ffn_forward(moe_ffn_ctx* ctx, const void* x, int T, const moe_ffn_weights* w, void* out,
                    void* stream);

/* Expert-parallel shard of one forward ("Porting a 128-expert MoE (Gemma-4 26B-A4B) to AWS
 * Inferentia2", section "The traceable trick: compute all experts, mask to top-8": each rank owns a
 * contiguous group of experts, e.g. 16 of 128 on 8 ranks, and the ranks' expert outputs are summed
 * by an all-reduce). Every rank computes the router and the top-8 choice for all T tokens (the
 * router weights are replicated, so all ranks choose the same experts without an exchange), then
 * runs the grouped GEMMs over the experts [expert_begin, expert_end) only, and writes
 *   moe_partial  device pointer, [T, 2816] fp32: for each token, the sum over its selected experts
 *                in the range, in ascending expert id, of (routing weight x expert output), each
 *                term rounded to bf16 as in moe_ffn_forward; 0 where none is in the range. This is
 *                the expert branch before post_feedforward_layernorm_2, which is not linear, so
 *                the ranks exchange and add these partials (an all-reduce sum) before it;
 *   dense_out    with with_dense != 0 (FULL_LAYER only): device pointer, [T, 2816] fp32, the shared
 *                MLP's output before post_feedforward_layernorm_1 (bf16 values widened); one rank
 *                runs it. With with_dense == 0 it is not read and may be NULL.
 * x, T and w are as for moe_ffn_forward (w must hold every field moe_ffn_forward needs). 0 <=
 * expert_begin <= expert_end <= 128 (an empty range writes zeros). The outputs must not overlap x,
 * each other or the workspace. Asynchronous on `stream`; the same errors as moe_ffn_forward, and
 * MOE_FFN_EINVAL for a bad range or with_dense in MOE_FFN_MOE_ONLY mode. The workspace views hold
 * this shard's routing (all experts) afterwards. */
int moe_ffn_forward_shard(moe_ffn_ctx* ctx, const void* x, int T, const moe_ffn_weights* w, int expert_begin,
                          int expert_end, int with_dense, float* moe_partial, float* dense_out, void* stream);

/* The rest of the block after the shards' exchange: out = (x + RMSNorm(RMSNorm(dense;
 * post_feedforward_layernorm_1) + RMSNorm(moe_sum; post_feedforward_layernorm_2);
 * post_feedforward_layernorm)) x layer_scalar in FULL_LAYER mode (the same arithmetic as the end of
 * moe_ffn_forward), out = moe_sum rounded to bf16 in MOE_FFN_MOE_ONLY mode.
 *   moe_sum  device pointer, [T, 2816] fp32: the sum over all shards of moe_partial;
 *   dense    device pointer, [T, 2816] fp32: the dense_out of the rank that ran the shared MLP
 *            (FULL_LAYER; ignored and may be NULL in MOE_ONLY mode);
 *   x        device pointer, [T, 2816] bf16, the layer input (FULL_LAYER);
 *   out      device pointer, [T, 2816] bf16; must not overlap x, moe_sum or dense.
 * Reads the norm weights and layer_scalar of w. Asynchronous on `stream`. */
int moe_ffn_finish_shards(moe_ffn_ctx* ctx, const void* x, int T, const moe_ffn_weights* w, const float* moe_sum,
                          const float* dense, void* out, void* stream);

/* Fills *views with device pointers into the workspace (see moe_ffn_views). */
int moe_ffn_workspace_view(const moe_ffn_ctx* ctx, moe_ffn_views* views);

/* Synchronises `stream`, reads the device status word and clears it. Returns MOE_FFN_EDEVICE if a
 * kernel gave up a bounded wait or rejected an index since the last call, MOE_FFN_ECUDA if the
 * stream reported a CUDA error, else MOE_FFN_OK. *word (if not NULL) receives the raw status bits
 * (MOE_FFN_STATUS_*). */
int moe_ffn_device_status(moe_ffn_ctx* ctx, void* stream, uint32_t* word);

/* Profiling hook: from now on every forward records `start` (a cudaEvent_t as void*) on its stream
 * right before the launch of kernel slot `kernel` and `stop` right after it. NULL events turn the
 * hook off. Slots (0..6): 0 router matrix split, 1 router logits, 2 top-k and pre-norms,
 * 3 permutation (counting-sort scatter), 4 gate_up grouped GEMM, 5 down grouped GEMM, 6 combine and
 * post-norms. Forwards of at most 64 tokens run the whole routing front end (router sums on CUDA
 * cores, top-k, pre-norms, counting sort) as one kernel in slot 1 and launch nothing at slots 0, 2
 * and 3, whose events are then recorded back to back (moe_ffn_kernel_slots). */
int moe_ffn_set_kernel_events(moe_ffn_ctx* ctx, int kernel, void* start, void* stop);

/* Number of kernels one forward of T tokens launches on the device (0 for T = 0; 4 for T <= 64,
 * else 7). */
int moe_ffn_kernels_per_forward(const moe_ffn_ctx* ctx, int T);

/* The kernel slots (see moe_ffn_set_kernel_events) one forward of T tokens launches, in launch
 * order, written to slots[0..n-1]; returns n (or MOE_FFN_EINVAL: NULL ctx or slots, T < 0, or
 * n_slots below 7). Host only. */
int moe_ffn_kernel_slots(const moe_ffn_ctx* ctx, int T, int* slots, int n_slots);

/* The block's fp32 router logits, [T, 128], for callers that cannot allocate device memory (code
 * running under a memory pool or allocator it does not own, a plugin handed only a stream and its
 * buffers, a real-time path where an allocation is not allowed). The pages have no counterpart to
 * this entry point; it exists for such callers only.
 *   x             device pointer, [T, 2816] bf16, the layer input;
 *   T             0..1024 tokens (above 1024: MOE_FFN_ETOOBIG, nothing queued; 0: no-op);
 *   router_w      device pointer, [128, 2816] fp32; router_norm_w: device pointer, [2816] fp32;
 *   router_scale  the scalar on the normed input (2816^-1/2), eps: the RMSNorm epsilon (1e-6);
 *   logits        device pointer, [T, 128] fp32, written with the same logits moe_ffn_forward
 *                 computes for the same x and weights (up to fp32 summation order);
 *   stream        cudaStream_t as void*; the work is queued there, the host is not synchronised.
 * It allocates nothing: its scratch is one array of about 2.6 MB in device memory that the library
 * reserves on each GPU it runs on, held until the process exits. Every call shares that array, so
 * calls whose GPU work overlaps in time (other streams, other host threads) race and corrupt each
 * other's results. The array keeps the last call's contents: each call clears its status word
 * first (an asynchronous memset on `stream`), and every other byte it reads there it has written
 * itself. Calls queued back to back on one stream are ordered and do not race. It runs on the
 * calling thread's current CUDA device. The first call on a device looks up the array's device
 * address and builds a TMA descriptor over it; make that first call before any stream capture.
 * All pointers must be 16-byte aligned (MOE_FFN_EALIGN).
 * Failure: if one of the router's bounded device waits gives up (MOE_FFN_STATUS_* above), that
 * call writes NaN to all T x 128 logits; the return value only covers errors found while queueing. */
int moe_ffn_router_logits_noalloc(const void* x, int T, const float* router_w, const float* router_norm_w,
                                  float router_scale, float eps, float* logits, void* stream);

/* Per-channel symmetric int8 quantisation of a bf16 matrix [rows, cols] on the device (the int8
 * experts of the 26B-A4B post, section "Can it run on a smaller box?"), one channel per row: scale[r] = max_c |w[r, c]| / 127 in fp32, q[r, c] = w[r, c] / scale[r] in fp32 rounded
 * to nearest (ties to even) and clamped to [-127, 127]; an all-zero row gets scale 0 and q 0. All
 * pointers are device pointers; w and q 16-byte aligned, cols a multiple of 8. Asynchronous on
 * `stream`. Returns MOE_FFN_EINVAL / MOE_FFN_EALIGN on bad arguments, MOE_FFN_ECUDA if the launch
 * fails. */
int moe_ffn_quantize_int8(const void* w, long long rows, int cols, int8_t* q, float* scale, void* stream);

/* MXFP4 quantisation of a bf16 matrix [rows, cols] on the device (the microscaling fp4 experts of
 * the 26B-A4B post, section "The fp4 rabbit hole"), after the OCP Microscaling Formats (MX) v1.0
 * conversion: for each block of 32 consecutive elements of a row, amax = max |w|;
 * if amax > 0 the shared exponent is floor(log2 amax) - 2, clamped to [-127, 127], and every
 * element w / 2^exponent is rounded to the nearest E2M1 magnitude (0, 0.5, 1, 1.5, 2, 3, 4, 6; ties
 * to the even code; above 6 saturates to 6) with its sign; a value that rounds to zero is +0 (code
 * 0). An all-zero block gets scale byte 0 and codes 0. codes[r, c / 2] holds element c in its low
 * (even c) or high (odd c) nibble; scales[r, c / 32] = exponent + 127. All pointers are device
 * pointers; w and codes 16-byte aligned, cols a multiple of 32. Asynchronous on `stream`. Returns
 * MOE_FFN_EINVAL / MOE_FFN_EALIGN on bad arguments, MOE_FFN_ECUDA if the launch fails. */
int moe_ffn_quantize_mxfp4(const void* w, long long rows, int cols, uint8_t* codes, uint8_t* scales,
                           void* stream);

/* Self-test of the bounded device waits behind MOE_FFN_EDEVICE (failure detection); the pages have
 * no counterpart. Queues on `stream` one kernel of one CTA that waits on an mbarrier nothing
 * arrives on, through the same helpers the forward's kernels wait with:
 *   wait 1, bounded: gives up after the 2 s limit, ORs MOE_FFN_STATUS_WAIT_FULL into
 *           *status_word and raises the CTA's abort flag;
 *   wait 2, bounded: leaves at once through the abort flag and sets nothing (its bit,
 *           MOE_FFN_STATUS_WAIT_EMPTY, stays clear);
 *   wait 3, exit drain with a 1 ms limit: gives up and ORs MOE_FFN_STATUS_DRAIN.
 * Nothing faults, traps or hangs; the kernel ends after about 2 s and the context stays usable.
 *   status_word  device pointer to one uint32 the caller has zeroed;
 *   record       device pointer to 6 uint64: record[2i] = nanoseconds wait i+1 took,
 *                record[2i+1] = 1 if its phase completed (0 expected for all three);
 *   stream       cudaStream_t as void*; the host is not synchronised.
 * Runs on the calling thread's current device. Returns MOE_FFN_EINVAL for a NULL pointer,
 * MOE_FFN_EARCH on a device other than sm_103, MOE_FFN_ECUDA if the launch fails. */
int moe_ffn_selftest_wait_expiry(uint32_t* status_word, unsigned long long* record, void* stream);

/* A static string naming a status code. */
const char* moe_ffn_status_string(int status);

/* Releases the host state of a context (it holds no device memory). Never frees the workspace or
 * any caller buffer. Safe on NULL. */
void moe_ffn_destroy(moe_ffn_ctx* ctx);

#ifdef __cplusplus
}
#endif

#endif /* MOE_FFN_H */
