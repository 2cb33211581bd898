/*
 * q3_oracle.h -- plain CPU oracle for the token-round forward of a dense
 * Qwen3-style decoder.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline leg use this library.  It shares no code, header, table or
 * helper with the CUDA path under qwen3_dense_decoder_gb300/csrc.
 *
 * What it follows (Kipp pages):
 *  - "Kipp Model Support", section "The registry": dense Qwen3 decoders,
 *    8 KV heads, head width 128, RMS epsilon 1e-6, per-checkpoint RoPE theta
 *    and embedding tying.
 *  - "Kipp Model Support", section "qwen3-0.6b-base": K/V are stored in BF16
 *    (the "storage contract"); attention width may exceed the hidden width.
 *  - "Kipp Model Support", section "Quantization (Q8_0)": the seven per-layer
 *    projections in 32-weight blocks of fp16 scale + int8 quants; embedding,
 *    lm_head and all norms stay BF16.
 *  - "Kipp Model Support", section "Quantization (AFFINE4_GS32)": 32-weight
 *    groups of 4-bit codes with an fp16 scale and an fp16 bias, 5.0 bits per
 *    weight (the same seven projections; the rest stays BF16).
 *  - "Kipp Roadmap", status v0.0.2: paged KV through a per-session
 *    32-position block table, bitwise equal to the contiguous layout;
 *    batched evaluation equal to isolated evaluation.
 *  - "Kipp Roadmap", status v0.0.4: an opt-in Q8_0 KV cache, about 1.9x
 *    smaller than BF16, gated for tolerance and placement invariance.
 *  - "Reproducing Kipp", section "Model-backed CPU and Metal gates": cached
 *    decode must equal recomputation; the CPU oracle is FP32.
 * The layer math itself is not printed on the pages; the oracle takes the
 * plain reading of a standard dense Qwen3 decoder (pre-norm RMSNorm blocks,
 * per-head q/k RMSNorm before rotate-half RoPE, causal GQA softmax attention,
 * SwiGLU FFN, no biases).
 *
 * Precision: activations are stored in FP32; every dot product, mean square
 * and softmax sum accumulates in FP64 and is rounded to FP32 when stored;
 * RoPE angles and their cos/sin are evaluated in FP64.
 */
#ifndef Q3_ORACLE_H
#define Q3_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_BF16 = 0, ORC_Q8_0 = 1, ORC_AFFINE4 = 2 };
enum { ORC_BLOCK = 32 };          /* KV positions per block; weights per Q8_0 block / AFFINE4 group */
enum { ORC_Q8_0_BYTES = 34 };     /* fp16 scale + 32 int8 quants */
enum { ORC_AFFINE4_BYTES = 20 };  /* 16 bytes of 4-bit codes + fp16 scale + fp16 bias */

typedef struct orc_cfg {
    int n_layers, hidden, n_q_heads, n_kv_heads, head_dim, ffn, vocab;
    int tied;     /* 1: lm_head is the token embedding */
    int scheme;   /* ORC_BF16, ORC_Q8_0 or ORC_AFFINE4 (the seven projections only) */
    double rope_theta, rms_eps;
    int kv_quant; /* ORC_BF16: K/V stored as bf16; ORC_Q8_0: as Q8_0 blocks */
} orc_cfg;

/* Per-layer weights, host memory, row-major [out][in].  BF16 tensors are
 * uint16 bit patterns.  With ORC_Q8_0 the seven projections point at
 * canonical blocks: [out][in/32] records of 34 bytes (little-endian fp16
 * scale, then 32 int8 quants).  With ORC_AFFINE4 they point at [out][in/32]
 * groups of 20 bytes (16 code bytes, then little-endian fp16 scale and bias). */
typedef struct orc_layer {
    const uint16_t *attn_norm, *q_norm, *k_norm, *ffn_norm;
    const void *wq, *wk, *wv, *wo, *wg, *wu, *wd;
} orc_layer;

typedef struct orc_model orc_model;
typedef struct orc_pool orc_pool;
typedef struct orc_session orc_session;

/* ---- scalar conversions ---- */
float    orc_bf16_to_f32(uint16_t b);
uint16_t orc_f32_to_bf16(float f);              /* round to nearest even */
float    orc_f16_to_f32(uint16_t h);
uint16_t orc_f32_to_f16(float f);               /* round to nearest even */

/* ---- Q8_0 ---- */
/* w: n floats (n % 32 == 0) -> n/32 canonical blocks. */
void orc_q8_0_pack(const float* w, long n, uint8_t* blocks);
void orc_q8_0_unpack(const uint8_t* blocks, long n, float* w);

/* ---- AFFINE4_GS32 ---- */
/* w: n floats (n % 32 == 0) -> n/32 groups of 20 bytes. */
void orc_affine4_pack(const float* w, long n, uint8_t* groups);
void orc_affine4_unpack(const uint8_t* groups, long n, float* w);

/* ---- components (exported so the tests can pin each one) ---- */
void  orc_rmsnorm(const float* x, const uint16_t* gain, int n, double eps, float* y);
void  orc_rope(float* v, int head_dim, int pos, double theta);       /* in place */
float orc_silu(float z);
/* y[t][o] = sum_i W[o][i] * x[t][i]; W bf16 (scheme 0), Q8_0 blocks (1) or
 * AFFINE4 groups (2). */
void  orc_matmul(const void* W, int scheme, int n_out, int n_in,
                 const float* x, int n_tok, float* y, int n_threads);
/* One query row of GQA attention over ctx cached positions.
 * q: [n_q][d] f32; K, V: [ctx][n_kv][d] bf16; o: [n_q][d]. */
void  orc_gqa_attend(const float* q, const uint16_t* K, const uint16_t* V,
                     int ctx, int n_q, int n_kv, int d, float* o);

/* Bytes one position's K and V take in one layer's cache: 2 n_kv d (bf16)
 * or 2 n_kv (d/32) 34 (Q8_0 blocks). */
long  orc_kv_bytes_per_position(const orc_cfg* c);

/* ---- model / KV / sessions ---- */
orc_model* orc_model_create(const orc_cfg* cfg, const uint16_t* embed,
                            const uint16_t* final_norm, const uint16_t* lm_head,
                            const orc_layer* layers, int n_threads);
void orc_model_free(orc_model* m);

/* A pool of 32-position KV blocks shared by paged sessions. */
orc_pool* orc_pool_create(orc_model* m, int n_blocks);
void orc_pool_free(orc_pool* p);

/* pool == NULL: contiguous per-session KV of max_ctx positions.
 * pool != NULL: paged KV; blocks come from the pool in order unless a
 * table is set with orc_session_set_block_table. */
orc_session* orc_session_create(orc_model* m, orc_pool* pool, int max_ctx);
void orc_session_free(orc_session* s);
int  orc_session_set_block_table(orc_session* s, const int32_t* ids, int n);
int  orc_session_pos(const orc_session* s);
int  orc_session_truncate(orc_session* s, int n_pos);

/* Content-addressed prefix sharing over a pool ("Kipp Roadmap", status
 * v0.0.3: a content-addressed 32-token block pool, publish-at-finish,
 * memcmp-verified).  enable: an index of 2^hash_bits buckets (0..24; few
 * buckets force hash collisions, which the token comparison resolves).
 * publish: the session's full blocks become shareable; returns how many
 * were newly published.  attach_prefix: at position 0, take the longest
 * published chain matching the prompt's leading full blocks, leaving at
 * least one token to evaluate; returns the positions attached. */
int  orc_pool_enable_prefix(orc_pool* p, int hash_bits);
/* blocks no session holds and the index does not keep */
int  orc_pool_free_blocks(const orc_pool* p);
int  orc_session_publish(orc_session* s);
int  orc_session_attach_prefix(orc_session* s, const int32_t* tokens, int n);

/* One round of n tokens appended at the session's position.  logits_last:
 * [vocab] logits of the round's last token (may be NULL).  logits_all:
 * [n][vocab] logits of every row (may be NULL).  Returns 0 or -1. */
int orc_eval(orc_session* s, const int32_t* tokens, int n,
             float* logits_last, float* logits_all);

/* The same round, returning the logits of the listed rows only: rows are
 * indices into the round, increasing; logits: [n_rows][vocab].  n_rows == 0
 * appends the positions (their K/V stored) and computes no logits.
 * Returns 0 or -1. */
int orc_eval_rows(orc_session* s, const int32_t* tokens, int n, const int* rows,
                  int n_rows, float* logits);

/* One round over several sessions, processed layer by layer over all rows
 * at once.  logits: [ns][vocab], the last row of each session's round. */
int orc_eval_batch(orc_session* const* s, const int32_t* const* tokens,
                   const int* n, int ns, float* logits);

/* argmax with the lowest index on ties */
int orc_argmax(const float* v, int n);

#ifdef __cplusplus
}
#endif
#endif
