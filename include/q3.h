/*
 * q3.h -- C ABI of the GB300 (sm_103a) forward of a dense Qwen3-style decoder.
 *
 * The forward is the token round of the Kipp engine's dense Qwen3 path:
 * RMSNorm (eps from the config, 1e-6 for the family), the seven per-layer
 * projections over BF16 or Q8_0 weights with FP32 accumulation, per-head q/k
 * RMSNorm and RoPE, GQA attention over a paged BF16 KV cache addressed through
 * 32-position block tables, SwiGLU, and full-vocabulary FP32 lm_head logits
 * with the greedy argmax.  It serves prefill rounds and batched decode.
 *
 * Sources on the Kipp pages:
 *  - "Kipp Model Support", section "The registry": 8 KV heads, head width
 *    128, vocabulary 151,936, RMS epsilon 1e-6, per-checkpoint dimensions,
 *    RoPE theta and embedding tying (tied: lm_head is the token embedding).
 *  - "Kipp Model Support", section "Quantization (Q8_0)": the seven
 *    projections in 32-weight blocks (fp16 scale + int8 quants); embedding,
 *    lm_head and norms stay BF16.
 *  - "Kipp Model Support", section "qwen3-0.6b-base": K and V are stored as
 *    BF16 (the KV storage contract).
 *  - "Kipp Roadmap", status v0.0.2: multi-session evaluation (kipp_eval_batch),
 *    paged KV through a per-session 32-position block table; status v0.0.3:
 *    one model-owned pool of 32-token blocks shared by sessions; status
 *    v0.0.4: activation scratch is one per model.
 *  - "Kipp Model Support", section "What the gates check": truncate/resume,
 *    batched evaluation; section "CUDA (NVIDIA H100 80GB ...)": weights are
 *    resident in device memory, stateless prefill and reset/reuse; a backend
 *    failure is fatal with no fallback ("Reproducing Kipp", section "Build";
 *    "Kipp Model Support", section "Backends").
 *
 * Conventions
 *  - Every pointer named *_dev is device memory on the model's device; every
 *    other pointer is host memory.
 *  - All calls are asynchronous on the model's CUDA stream except q3_sync,
 *    the create/destroy calls and the error queries.  Outputs are valid after
 *    q3_sync (or any later synchronisation of that stream).
 *  - Return value: Q3_OK (0) or a negative Q3_ERR_* code; q3_last_error()
 *    gives a message (thread-local).  A CUDA error or a failed device-side
 *    check poisons the model: every later call on it returns Q3_ERR_POISONED.
 *  - Calls on one model are not thread-safe; use one host thread per model.
 *  - Handles may be destroyed in any order: a model's memory is released
 *    when its handle and all its pools are destroyed, a pool's when its
 *    handle and all its sessions are.  A destroyed handle must not be used.
 */
#ifndef Q3_H
#define Q3_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define Q3_OK 0
#define Q3_ERR_INVALID_ARG (-1)
#define Q3_ERR_UNSUPPORTED_DEVICE (-2) /* not an sm_103 device */
#define Q3_ERR_OOM (-3)                /* device allocation failed */
#define Q3_ERR_POOL_EXHAUSTED (-4)     /* no free KV block */
#define Q3_ERR_CTX_OVERFLOW (-5)       /* round would pass the model's max_ctx */
#define Q3_ERR_CUDA (-6)               /* a CUDA call failed; model poisoned */
#define Q3_ERR_DEVICE_CHECK (-7)       /* a kernel's own check failed; model poisoned */
#define Q3_ERR_POISONED (-8)           /* an earlier error poisoned the model */

#define Q3_BF16 0
#define Q3_Q8_0 1
#define Q3_AFFINE4 2
#define Q3_KV_BLOCK 32       /* positions per KV block */
#define Q3_Q8_0_BLOCK 32     /* weights per Q8_0 block */
#define Q3_Q8_0_BYTES 34     /* bytes per canonical Q8_0 block */
#define Q3_AFFINE4_GROUP 32  /* weights per AFFINE4_GS32 group */
#define Q3_AFFINE4_BYTES 20  /* bytes per AFFINE4_GS32 group */

/* Device status-word bits (q3_sync reports them as Q3_ERR_DEVICE_CHECK). */
#define Q3_STATUS_TOKEN_RANGE 0x1   /* a token id outside [0, vocab) */
#define Q3_STATUS_BLOCK_RANGE 0x2   /* a block-table entry outside the pool */
#define Q3_STATUS_TIMEOUT 0x4       /* a bounded device wait ran out */
#define Q3_STATUS_F16_RANGE 0x8     /* a tensor-core activation beyond the fp16 range */

typedef struct q3_model q3_model;
typedef struct q3_pool q3_pool;
typedef struct q3_session q3_session;

/* Shape of the decoder.  head_dim must be 128, n_q_heads a multiple of
 * n_kv_heads (GQA group of at most 8), hidden, ffn, vocab and
 * n_q_heads*head_dim multiples of 128.  max_ctx bounds a session's length
 * (the RoPE table is built for it).  scheme: Q3_BF16, Q3_Q8_0 or Q3_AFFINE4
 * (the seven projections only).  tied: 1 when lm_head is the token embedding.
 * kv_scheme: Q3_BF16 (the K/V storage contract of "Kipp Model Support",
 * section "qwen3-0.6b-base") or Q3_Q8_0, the opt-in quantized cache of "Kipp
 * Roadmap", status v0.0.4: every position's K and V head rows (after the q/k
 * norm and RoPE) packed by the weights' Q8_0 rule -- blocks of 32 values,
 * d = absmax / 127 in FP32, stored as fp16(d), codes round-half-even(x / d)
 * clamped to [-127, 127] -- 136 bytes per head row against 256, about 1.9x
 * smaller.  Attention reads fp16(fp16 d * code) (each product rounded once);
 * a Q8_0-cache model runs prefill attention on the mma.sync kernel and
 * one-session decode on the per-operation path. */
typedef struct q3_config {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab, max_ctx;
    float rope_theta, rms_eps;
    int tied;
    int scheme;
    int kv_scheme;
} q3_config;

/* Device pointers of one layer.  Norm gains are bf16 [hidden] (attn_norm,
 * ffn_norm) or [head_dim] (q_norm, k_norm).  Projections are row-major
 * [out][in] (the nn.Linear layout): wq [n_q*d][hidden], wk and wv
 * [n_kv*d][hidden], wo [hidden][n_q*d], w_gate and w_up [ffn][hidden],
 * w_down [hidden][ffn].  With Q3_BF16 they are bf16; with Q3_Q8_0 they are
 * canonical Q8_0 blocks [out][in/32] of 34 bytes (little-endian fp16 scale,
 * then 32 int8 quants), as q3_quantize_q8_0 writes them; with Q3_AFFINE4
 * they are AFFINE4_GS32 groups [out][in/32] of 20 bytes, 4-byte aligned, as
 * q3_quantize_affine4 writes them. */
typedef struct q3_layer_weights {
    const void *attn_norm, *wq, *wk, *wv, *q_norm, *k_norm, *wo,
               *ffn_norm, *w_gate, *w_up, *w_down;
} q3_layer_weights;

/* embed: bf16 [vocab][hidden]; final_norm: bf16 [hidden]; lm_head: bf16
 * [vocab][hidden], or NULL when tied; layers: host array of n_layers. */
typedef struct q3_weights {
    const void* embed;
    const void* final_norm;
    const void* lm_head;
    const q3_layer_weights* layers;
} q3_weights;

/* Create a model on the current CUDA device.  The weights are borrowed: the
 * caller keeps them alive and unchanged until q3_model_destroy.  With Q3_Q8_0
 * the library derives its own device layout of the projections (an int8
 * plane and an fp16 scale plane, bit-equal to the canonical blocks) once,
 * here.  Rounds of more than one token run their projections on tcgen05
 * tensor cores with fp16 operands (kind::f16 takes A and B of one type and
 * fp16 activations keep 3 more mantissa bits than bf16): the library keeps
 * an fp16 copy of the BF16 projections and lm_head (exact except for
 * |w| < 2^-17, whose rounding is below 2^-25), or of the Q8_0 projections
 * dequantised once (d * q rounded to fp16; 2 bytes per weight of device
 * memory beside the 1.0625 of the planes).  With Q3_AFFINE4, rounds of more
 * than one token run their projections on the tensor cores over an fp16 copy
 * of the dequantised groups (scale * code + bias rounded to FP32, then to
 * fp16, as q3_affine4_to_f16 writes it), and one-token rounds on a 5.0-bit
 * matvec over lane-major planes derived here from the groups (the format's
 * bytes rearranged; see q3_op_matvec_affine4); the fused decode step takes
 * BF16 and Q8_0 only.  Weights beyond the fp16 range make creation fail with
 * Q3_ERR_INVALID_ARG; an activation beyond it is reported by q3_sync as
 * Q3_ERR_DEVICE_CHECK (Q3_STATUS_F16_RANGE).  max_round_tokens bounds the rows of one round (the activation
 * scratch, owned by the model, is sized for it; longer q3_session_eval rounds
 * are split into chunks of this size).  stream: a cudaStream_t, or NULL for
 * the legacy default stream.  Errors: Q3_ERR_INVALID_ARG (bad shape or NULL
 * weight), Q3_ERR_UNSUPPORTED_DEVICE, Q3_ERR_OOM, Q3_ERR_CUDA. */
int q3_model_create(const q3_config* cfg, const q3_weights* w, int max_round_tokens,
                    void* stream, q3_model** out);
void q3_model_destroy(q3_model* m);

/* A pool of n_blocks KV blocks of 32 positions for all layers, owned by the
 * library; up to max_sessions sessions draw from it.  One block holds, per
 * layer, K and V of every KV head: 32 * head_dim bf16 values each, or with
 * the Q8_0 cache a tile of 4,096 int8 codes ([32 positions][128]) followed
 * by 128 fp16 scales ([32 positions][4]).  Errors: Q3_ERR_INVALID_ARG,
 * Q3_ERR_OOM. */
int q3_pool_create(q3_model* m, int n_blocks, int max_sessions, q3_pool** out);
void q3_pool_destroy(q3_pool* p);

/* A session: a position counter and a block table in the pool.  Sessions of
 * one pool may be evaluated together with q3_eval_batch.
 * Errors: Q3_ERR_INVALID_ARG (pool full of sessions), Q3_ERR_OOM. */
int q3_session_create(q3_pool* p, q3_session** out);
void q3_session_destroy(q3_session* s);   /* returns its blocks to the pool */

/* Fix which pool blocks back the session's first n*32 positions, in order
 * (block i holds positions [32 i, 32 i + 32)); later positions draw free
 * blocks as usual.  Only on an empty session (position 0); the ids must be
 * free and in range.  Errors: Q3_ERR_INVALID_ARG. */
int q3_session_set_block_table(q3_session* s, const int32_t* phys_ids, int n);

/* One round of n tokens appended to the session at its current position
 * (prefill when n > 1, a decode step when n == 1).  tokens_dev: int32 [n]
 * device.  logits_dev: float [vocab] device, receives the FP32 logits of the
 * round's last token.  argmax_dev: int32 [1] device or NULL, receives the
 * greedy token (lowest index on ties).  Both may be the tokens_dev of a later
 * call.  Token ids outside [0, vocab) are reported by q3_sync as
 * Q3_ERR_DEVICE_CHECK.  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CTX_OVERFLOW,
 * Q3_ERR_POOL_EXHAUSTED, Q3_ERR_CUDA, Q3_ERR_POISONED. */
int q3_session_eval(q3_session* s, const int32_t* tokens_dev, int n,
                    float* logits_dev, int32_t* argmax_dev);

/* One round of n tokens for one session, returning the logits of its last
 * n_logits rows (1 <= n_logits <= n; n_logits == n scores every prompt row)
 * ("Kipp Roadmap", status v0.0.2: multi-logit evaluation, kipp_session_eval_n).
 * logits_dev: f32 [n_logits][vocab], row i the logits after token
 * n - n_logits + i; argmax_dev: int32 [n_logits] or NULL.  Rounds longer
 * than max_round_tokens are split as in q3_session_eval; the result does not
 * depend on the split.  n_logits == 1 is q3_session_eval.  Asynchronous on
 * the model's stream.  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CTX_OVERFLOW,
 * Q3_ERR_POOL_EXHAUSTED, Q3_ERR_CUDA, Q3_ERR_POISONED. */
int q3_session_eval_n(q3_session* s, const int32_t* tokens_dev, int n, int n_logits, float* logits_dev,
                      int32_t* argmax_dev);

/* One round over ns distinct sessions of one pool ("Kipp Roadmap", status
 * v0.0.2, kipp_eval_batch): session i appends n[i] tokens.  tokens_dev:
 * int32 device, the rounds concatenated in session order (sum n[i] tokens,
 * at most max_round_tokens).  n: host int [ns].  logits_dev: float
 * [ns][vocab] device, the last row of each session's round.  argmax_dev:
 * int32 [ns] device or NULL.  Errors as q3_session_eval. */
int q3_eval_batch(q3_session* const* sessions, int ns, const int32_t* tokens_dev,
                  const int* n, float* logits_dev, int32_t* argmax_dev);

/* Forget positions >= n_pos (truncate/resume); 0 <= n_pos <= position.
 * Blocks past the new end return to the pool unless fixed by
 * q3_session_set_block_table.  If the block holding position n_pos is
 * shared (published, or attached by other sessions), it is first copied to
 * a block of the session's own, asynchronously on the model's stream.
 * Errors: Q3_ERR_INVALID_ARG, Q3_ERR_POOL_EXHAUSTED (no block for that
 * copy), Q3_ERR_CUDA. */
int q3_session_truncate(q3_session* s, int n_pos);
/* Back to position 0 (reset/reuse). */
int q3_session_reset(q3_session* s);
int q3_session_pos(const q3_session* s);

/* Content-addressed prefix sharing over a pool ("Kipp Roadmap", status
 * v0.0.3: a content-addressed 32-token block pool, publish-at-finish,
 * memcmp-verified).  A published block is addressed by the block before it
 * in its chain and its 32 tokens; a lookup hashes that key (64-bit FNV-1a)
 * into one of 2^hash_bits buckets and accepts a candidate only if the
 * previous block and the tokens compare equal, so a collision never shares
 * a block.  The pool keeps each published block until it needs the room:
 * with no free block, the least recently published or attached block that
 * no session holds and no published block follows is reused.
 *
 * q3_pool_enable_prefix: once per pool; hash_bits in [0, 24].
 * q3_session_publish: tokens (host, int32 [n], n == the session's position)
 *   are the tokens the session evaluated; its full blocks become shared,
 *   and where an equal chain is already published the session switches to
 *   it and frees its own blocks.  *n_published: blocks newly published.
 *   Not for sessions with a table fixed by q3_session_set_block_table.
 * q3_session_attach_prefix: on an empty session, attach the longest
 *   published chain matching the leading full blocks of tokens (host, int32
 *   [n]), leaving at least one token to evaluate; the session's position
 *   becomes *n_attached (a multiple of 32) and the caller evaluates
 *   tokens[*n_attached .. n).
 * A round never writes a shared block (Q3_ERR_INVALID_ARG if it would).
 * Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CTX_OVERFLOW. */
int q3_pool_enable_prefix(q3_pool* p, int hash_bits);
int q3_session_publish(q3_session* s, const int32_t* tokens, int n, int* n_published);
int q3_session_attach_prefix(q3_session* s, const int32_t* tokens, int n, int* n_attached);

/* Wait for the model's stream; read and clear the device status word.
 * Errors: Q3_ERR_CUDA, Q3_ERR_DEVICE_CHECK (both poison), Q3_ERR_POISONED. */
int q3_sync(q3_model* m);

/* Pack bf16 weights into canonical Q8_0 blocks on the device (the format of
 * "Kipp Model Support", section "Quantization (Q8_0)"): per block of 32,
 * d = absmax/127 in FP32, stored as fp16(d) round-to-nearest-even; quants
 * are round-half-even(w/d) against the FP32 d, clamped to [-127, 127]; an
 * all-zero block has scale 0 and zero quants.  w_dev: bf16 [n]; blocks_dev:
 * [n/32][34] bytes; n a multiple of 32.  Asynchronous on stream (a
 * cudaStream_t or NULL).  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CUDA. */
int q3_quantize_q8_0(const void* w_dev, int64_t n, void* blocks_dev, void* stream);

/* Pack bf16 weights into AFFINE4_GS32 groups on the device ("Kipp Model
 * Support", section "Quantization (AFFINE4_GS32)": 32 weights, 4-bit codes,
 * an fp16 scale and an fp16 bias, 5.0 bits per weight).  A weight is
 * scale * code + bias, code in [0, 15].  Per group: bias = fp16(min),
 * scale = fp16((max - min) / 15) with the FP32 subtraction and division
 * correctly rounded; code = round-half-even((w - bias) / scale) in FP32
 * against the stored scale and bias, clamped to [0, 15]; a zero scale gives
 * zero codes.  Record: 16 code bytes (weight 2i in the low nibble of byte i,
 * weight 2i + 1 in the high nibble), then the scale, then the bias, fp16
 * little-endian.  w_dev: bf16 [n], 16-byte aligned; groups_dev: [n/32][20]
 * bytes, 4-byte aligned; n a multiple of 32.  Asynchronous on stream.
 * Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CUDA. */
int q3_quantize_affine4(const void* w_dev, int64_t n, void* groups_dev, void* stream);

/* The fp16 copy the model keeps of AFFINE4_GS32 projections: out[i] =
 * fp16_rne(fp32_rne(scale * code + bias)) (one fused multiply-add, then the
 * fp16 rounding), with scale, bias and code those of weight i's group.
 * groups_dev: [n/32][20] bytes, 4-byte aligned; out_dev: fp16 [n], 16-byte
 * aligned; n a multiple of 32.  Asynchronous on stream.
 * Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CUDA. */
int q3_affine4_to_f16(const void* groups_dev, int64_t n, void* out_dev, void* stream);

/* Operator entry points, for per-kernel gates like the pages' operator tests
 * ("Reproducing Kipp", section "Model-backed CPU and Metal gates":
 * kipp_test_metal --metal-operators; "Kipp Roadmap", status v0.0.4: the
 * first operator test of the flash prefill kernel).  They run one kernel of
 * the forward on caller buffers, asynchronously on stream.
 *
 * q3_op_matmul: y[n][m] = sum_k w[m][k] * x[n][k] on the tcgen05 GEMM
 * (the operand type of the prefill path, see q3_model_create).
 * w_dev: fp16 [M][K]; x_dev: fp16 [N][K] with at least round_up(N, 256)
 * rows allocated (rows past N are read but their products discarded);
 * y_dev: f32 [N][M].  M a multiple of 128, K a multiple of 64, 1 <= N.
 * block_n: token-tile width (32, 64, 96, 128, 144, 160, 176, 192 or 256), or 0 for the
 * width the prefill planner would pick; no split-K.  Pointers 16-byte
 * aligned.  Synchronous: returns once the kernel has finished on stream (it
 * allocates and frees a status word).  Errors: Q3_ERR_INVALID_ARG,
 * Q3_ERR_OOM, Q3_ERR_CUDA, Q3_ERR_DEVICE_CHECK (a bounded device wait ran
 * out; the message gives the status bits). */
int q3_op_matmul(const void* w_dev, const void* x_dev, int M, int N, int K, float* y_dev,
                 int block_n, void* stream);

/* q3_op_gemm: one projection GEMM of a prefill round with the round's
 * epilogue and split-K ("Kipp Roadmap", status v0.0.6: layer projections of
 * prefill on the tensor units), on caller buffers.  With d[n][m] =
 * sum_k w[m][k] * x[n][k]:
 *   Q3_OP_STORE:  out f32 [N][M] = d                   (QKV, lm_head rows)
 *   Q3_OP_ADD:    out f32 [N][M] += d                  (O and down: the residual)
 *   Q3_OP_SWIGLU: out fp16 [N][M] = fp16(silu(g) * u), g = the product with
 *                 w (gate), u = the product with w2 (up), silu(z) = z / (1 + e^-z)
 * w_dev, w2_dev: fp16 [M][K] (w2_dev only for Q3_OP_SWIGLU); x_dev: fp16
 * [N][K] with at least round_up(N, 256) rows allocated.  M a multiple of 128
 * (of 64 for Q3_OP_SWIGLU), K of 64, 1 <= N.  block_n as q3_op_matmul (0:
 * the planner's width); k_splits: 1..8 K splits (at most K/64; > 1 sums FP32
 * partials in split order in a second kernel, as a round does), or 0 for the
 * planner's choice.  Pointers 16-byte aligned.  Synchronous: allocates a
 * status word and the split workspace for the call and returns once the
 * kernels have finished.  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_OOM,
 * Q3_ERR_CUDA, Q3_ERR_DEVICE_CHECK (a bounded wait ran out, or an fp16
 * SwiGLU output beyond the fp16 range). */
#define Q3_OP_STORE 0
#define Q3_OP_ADD 1
#define Q3_OP_SWIGLU 2
int q3_op_gemm(const void* w_dev, const void* w2_dev, const void* x_dev, int M, int N, int K, int epi,
               void* out_dev, int block_n, int k_splits, void* stream);

/* q3_gemm_plan: the token-tile width (*block_n) and K-split count
 * (*k_splits) that a model's rounds use for a projection GEMM of M output
 * rows, N token rows and K inputs (the model's 32 Mi-float split workspace).
 * Host only: no CUDA call, no GPU needed.  In a prefill round of the BF16
 * cache, a QKV plan with k_splits == 1 applies the q/k head norm, RoPE and
 * the K/V append in the GEMM's epilogue; a split plan leaves them to the
 * separate kernel.  M a multiple of 128, K of 64, 1 <= N; M, N and K at
 * most 262,144; block_n and k_splits non-NULL.  Errors: Q3_ERR_INVALID_ARG. */
int q3_gemm_plan(int M, int N, int K, int* block_n, int* k_splits);

/* q3_attention_plan: the number of splits per (row, KV head) (*n_splits)
 * that the decode attention of batched and per-operation rounds uses for T
 * rows whose longest context is max_ctx positions, with n_kv_heads KV heads.
 * One 32-position block per warp (four warps a CTA) while the split CTAs fit
 * in about one wave of three per SM, else 2, 4 or 8 blocks per warp; at most
 * 128 splits and one per block; a round of 8 x 152 (row, KV head) units or
 * more takes none.  Host only: no CUDA call, no GPU needed.  1 <= n_kv_heads
 * <= 64, 1 <= T <= 65,536, 1 <= max_ctx <= 2^24; n_splits non-NULL.
 * Errors: Q3_ERR_INVALID_ARG. */
int q3_attention_plan(int n_kv_heads, int T, int max_ctx, int* n_splits);

/* q3_op_matvec: y[m] = sum_k w[m][k] * x[k] on the decode GEMV.  With
 * scales_dev == NULL, w_dev is bf16 [M][K]; otherwise w_dev is the int8
 * quant plane [M][K] and scales_dev the fp16 scale plane [M][K/32] of Q8_0
 * weights.  x_dev: f32 [K]; y_dev: f32 [M].  M a multiple of 8, K of 256;
 * pointers 16-byte aligned.
 * Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CUDA. */
int q3_op_matvec(const void* w_dev, const void* scales_dev, const float* x_dev, int M, int K,
                 float* y_dev, void* stream);

/* q3_op_matvec_affine4: y[m] = sum_k w[m][k] * x[k] on the 5.0-bit matvec
 * of one-token rounds over AFFINE4_GS32 weights ("Kipp Model Support",
 * section "Quantization (AFFINE4_GS32)"), with w[m][k] = scale * code + bias
 * of its group.  groups_dev: canonical 20-byte groups [M][K/32], 4-byte
 * aligned (as q3_quantize_affine4 writes them); x_dev: f32 [K]; y_dev: f32
 * [M].  M a multiple of 8, K of 128 (at most 32,768).  The call derives the
 * matvec's lane-major planes (allocated and freed here) and returns once the
 * kernel has finished.  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_OOM, Q3_ERR_CUDA,
 * Q3_ERR_DEVICE_CHECK (an activation beyond the fp16 range). */
int q3_op_matvec_affine4(const void* groups_dev, const float* x_dev, int M, int K, float* y_dev,
                         void* stream);

/* q3_op_prefill_attention: the causal GQA attention of one session's
 * prefill round over its paged K/V ("Kipp Roadmap", status v0.0.3:
 * flash-attention prefill kernel; "Kipp Model Support", section
 * "qwen3-0.6b-base": BF16 K/V in 32-position blocks).  Row t (position
 * pos0 + t) of head h: out[t][h] = sum_j softmax_j(q[t][h] . K[j][h / G] /
 * sqrt(128)) V[j][h / G] over positions j <= pos0 + t, G = n_q / n_kv.
 * q_dev: fp16 [T][n_q][128] (normed, rotated); kv_dev: bf16
 * [n_blocks][2][n_kv][32][128] (K then V of each block, the layout of one
 * layer of a pool); table_dev: int32 [n_table] physical block of each 32
 * positions, n_table >= ceil((pos0 + T) / 32); out_dev: fp16 [T][n_q * 128].
 * use_tc selects the tcgen05 kernel (1) or the mma.sync kernel (0).
 * Pointers 16-byte aligned.  Synchronous: returns once the kernel has
 * finished on stream (it allocates and frees a small metadata buffer).
 * Errors: Q3_ERR_INVALID_ARG, Q3_ERR_OOM, Q3_ERR_CUDA, Q3_ERR_DEVICE_CHECK (a
 * table entry outside [0, n_blocks) or a bounded wait that ran out; the
 * message gives the status bits). */
int q3_op_prefill_attention(const void* q_dev, const void* kv_dev, const int32_t* table_dev, int n_table,
                            int n_blocks, int pos0, int T, int n_q, int n_kv, void* out_dev, int use_tc,
                            void* stream);

/* Split-K matmul that allocates nothing (the Kipp pages have no counterpart;
 * this entry point serves callers that cannot call cudaMalloc where they need
 * the product: a host framework that owns all device memory through its own
 * allocator, a plug-in that may not grow its footprint, a latency-critical
 * loop that cannot afford cudaMalloc's implicit synchronisation).
 * y[n][m] = sum_k w[m][k] * x[n][k], the same tcgen05 GEMM as q3_op_matmul
 * with K split over k_splits CTAs; the split partial sums live in a fixed
 * scratch array of Q3_NOALLOC_SCRATCH_FLOATS floats (8 MiB) compiled into the
 * library, which every GPU that loads the library holds until exit.
 * w_dev: fp16 [M][K]; x_dev: fp16 [N][K] with at least round_up(N, 256)
 * rows allocated; y_dev: f32 [N][M]; M a multiple of 128, K of 64, 1 <= N,
 * 2 <= k_splits <= min(8, K/64), and k_splits * N * M must not exceed
 * Q3_NOALLOC_SCRATCH_FLOATS (else Q3_ERR_INVALID_ARG, nothing launched).
 * The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress) with that device current; that lookup loads the
 * library's device code for this entry point, which is when the driver
 * commits the scratch's memory on the device, so make the first call (a
 * warm-up) outside any latency-critical region and before any stream
 * capture.  All calls share the scratch: calls whose kernels may overlap on
 * the GPU race on it, so order them on one stream.  The caller must pass
 * buffers of the stated sizes: the library cannot check an allocation's
 * extent, and a short x_dev or y_dev is read or written past its end.
 * Synchronous: the call reads its device status word back into a host
 * variable and waits for the stream, so it returns once the kernels have
 * finished.  Allocates no device or host memory.  Errors (the message from
 * q3_noalloc_last_error): Q3_ERR_INVALID_ARG, Q3_ERR_CUDA,
 * Q3_ERR_DEVICE_CHECK (a bounded device wait ran out; the output is then
 * not valid). */
#define Q3_NOALLOC_SCRATCH_FLOATS (2 * 1024 * 1024)
int q3_op_matmul_splitk_noalloc(const void* w_dev, const void* x_dev, int M, int N, int K,
                                int k_splits, float* y_dev, void* stream);
const char* q3_noalloc_last_error(void);

/* Fused decode step.  A one-session decode round (q3_session_eval with
 * n == 1) runs as ONE persistent kernel -- embedding, every layer's
 * projections, q/k norm + RoPE + KV append, attention, SwiGLU, final norm,
 * lm_head and argmax -- instead of one launch per operation.  It computes
 * what the per-operation path computes ("Kipp Model Support", section
 * "qwen3-0.6b-base"; "Kipp Roadmap", status v0.0.4) with the same FP32
 * accumulation; only summation order differs.  On by default wherever the
 * shapes allow it.  q3_model_set_fused_decode(m, 0) selects the
 * per-operation path (for comparison); on = 1 where the shapes do not
 * allow it returns Q3_ERR_INVALID_ARG.  q3_model_fused_decode returns 1 when
 * the fused step is in use, 0 otherwise. */
int q3_model_set_fused_decode(q3_model* m, int on);
int q3_model_fused_decode(const q3_model* m);

/* Prefill attention on the tcgen05 tensor cores.  Rounds with more than one
 * row per session (prefill, chunked prefill, mixed rounds) run their causal
 * GQA attention ("Kipp Roadmap", status v0.0.3: flash-attention prefill
 * kernel) with scores and outputs accumulated in tensor memory; the result
 * equals the mma.sync kernel's up to summation order.  On by default where
 * the shapes allow it (query heads a multiple of KV heads, at most 128 query
 * heads per KV head).  q3_model_set_prefill_tc(m, 0) selects the mma.sync
 * kernel (for comparison); on = 1 where unsupported returns
 * Q3_ERR_INVALID_ARG.  q3_model_prefill_tc returns 1 when the tcgen05
 * kernel is in use, 0 otherwise. */
int q3_model_set_prefill_tc(q3_model* m, int on);
int q3_model_prefill_tc(const q3_model* m);

/* Bytes one position's K and V take in one layer of the cache: 2 * n_kv *
 * 256 (BF16) or 2 * n_kv * 136 (Q8_0); -1 for a NULL model. */
int q3_model_kv_bytes_per_position(const q3_model* m);

/* q3_op_kv_pack_q8_0: the Q8_0 cache writers' packing on caller rows
 * (operator gate of the cache writers, "Kipp Roadmap", status v0.0.4).
 * rows_dev: f32 [n_rows][128], 16-byte aligned; out_dev: [n_rows][136]
 * bytes, each row four canonical Q8_0 blocks of 34 bytes (little-endian
 * fp16 scale, then 32 int8 codes), by the rule q3_config's kv_scheme states.
 * Asynchronous on stream.  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CUDA. */
int q3_op_kv_pack_q8_0(const float* rows_dev, int n_rows, void* out_dev, void* stream);

/* Message of the last error on this host thread ("" if none). */
const char* q3_last_error(void);

/* Number of kernel launches this model has issued (for launch accounting). */
int64_t q3_model_launch_count(const q3_model* m);

/* Per-kernel timing for measurement (no counterpart on the pages beyond
 * their isolated matmul instrument, "Kipp Roadmap", status v0.0.5).  While
 * on, every kernel launch of the model's rounds is bracketed by CUDA events
 * on the model's stream, which serialises the launches (no programmatic
 * overlap), so a profiled round runs slower than an unprofiled one.
 * q3_model_profile_read synchronises the stream and returns, for kernel
 * class cls, the summed device time in ms and the launch count since the
 * last reset.  Errors: Q3_ERR_INVALID_ARG, Q3_ERR_CUDA. */
#define Q3_K_GEMV 0      /* decode matvec (projections, lm_head) */
#define Q3_K_GEMM 1      /* tcgen05 GEMM and its split-K reduce */
#define Q3_K_ATTN 2      /* attention and split combine */
#define Q3_K_ROPE 3      /* the separate q/k norm + RoPE + KV append kernel (prefill rounds with
                            the Q8_0 cache, a split-K QKV plan or one token; otherwise it runs
                            in the QKV GEMM's epilogue, timed as Q3_K_GEMM) */
#define Q3_K_NORM 4      /* embedding and RMSNorm */
#define Q3_K_OTHER 5     /* argmax, Q8_0 dequantisation */
#define Q3_K_STEP 6      /* fused one-kernel decode step */
#define Q3_K_CLASSES 7
int q3_model_profile(q3_model* m, int on);
int q3_model_profile_reset(q3_model* m);
int q3_model_profile_read(q3_model* m, int cls, double* total_ms, int64_t* launches);

#ifdef __cplusplus
}
#endif
#endif
