/*
 * q3_oracle.c -- plain CPU oracle for the token-round forward of a dense
 * Qwen3-style decoder.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the bench's CPU-baseline leg call it; the CUDA path never does.
 *
 * Sources (Kipp pages): "Kipp Model Support" (sections "The registry",
 * "What the gates check", "qwen3-0.6b-base", "Quantization (Q8_0)",
 * "Quantization (AFFINE4_GS32)"),
 * "Kipp Roadmap" (status v0.0.2: paged KV and batched evaluation; status
 * v0.0.4: the Q8_0 KV cache), and
 * "Reproducing Kipp" (section "Model-backed CPU and Metal gates").  Where the
 * pages leave the layer math open, the oracle takes the plain reading of a
 * standard dense Qwen3 decoder; each such reading is marked "reading".
 *
 * Every function is written to be checked by eye: one output at a time, in
 * logical order, FP64 accumulators, FP32 storage.  Threads only split the
 * list of independent outputs; each output is computed the same way whatever
 * the thread count, so results do not depend on it.
 */
#include "q3_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------ */
/* scalar conversions                                                  */
/* ------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of the float with the same value. */
float orc_bf16_to_f32(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* Round a float to the nearest bf16, ties to the even pattern.  Adding
 * 0x7fff (+1 when the kept part is odd) to the bits carries into the kept
 * half exactly when the dropped half is above the tie, or at the tie with an
 * odd kept half. */
uint16_t orc_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7fffffffu) > 0x7f800000u)         /* NaN: keep it a quiet NaN */
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7fffu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
float orc_f16_to_f32(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 0x1f, m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* (1 + m/1024) * 2^(e-15) */
    return (float)(sign ? -v : v);
}

/* Nearest binary16, ties to even (the default rounding mode of nearbyint). */
uint16_t orc_f32_to_f16(float f)
{
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    double a = fabs((double)f);
    if (isnan(f))
        return sign | 0x7e00;
    if (isinf(f))
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {                     /* subnormal range, quantum 2^-24 */
        double r = nearbyint(a * ldexp(1.0, 24));  /* exact scaling, then round */
        return sign | (uint16_t)r;                 /* r == 1024 encodes 2^-14 */
    }
    int e;
    frexp(a, &e);                                  /* a = f * 2^e, f in [0.5, 1) */
    double r = nearbyint(ldexp(a, 11 - e));        /* 11 significant bits: [1024, 2048] */
    int E = e - 1 + 15;
    if (r == 2048.0) { r = 1024.0; E += 1; }
    if (E >= 31)
        return sign | 0x7c00;                      /* overflow to infinity */
    return (uint16_t)(sign | (E << 10) | ((int)r - 1024));
}

int orc_argmax(const float* v, int n)
{
    int best = 0;
    for (int i = 1; i < n; i++)
        if (v[i] > v[best]) best = i;              /* strict: lowest index wins ties */
    return best;
}

/* ------------------------------------------------------------------ */
/* Q8_0 ("Kipp Model Support", section "Quantization (Q8_0)")          */
/* ------------------------------------------------------------------ */

/* Reading: per block of 32 weights, d = absmax/127 in FP32; the stored
 * scale is fp16(d); quants are round-half-even(w/d) against the FP32 d,
 * clamped to [-127, 127]; an all-zero block has d = 0 and zero quants. */
void orc_q8_0_pack(const float* w, long n, uint8_t* blocks)
{
    for (long b = 0; b < n / ORC_BLOCK; b++) {
        const float* x = w + b * ORC_BLOCK;
        uint8_t* out = blocks + b * ORC_Q8_0_BYTES;
        float amax = 0.0f;
        for (int i = 0; i < ORC_BLOCK; i++)
            if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
        float d = amax / 127.0f;
        uint16_t dh = orc_f32_to_f16(d);
        out[0] = (uint8_t)(dh & 0xff);
        out[1] = (uint8_t)(dh >> 8);
        for (int i = 0; i < ORC_BLOCK; i++) {
            int q = 0;
            if (d != 0.0f) {
                float r = nearbyintf(x[i] / d);
                if (r > 127.0f) r = 127.0f;
                if (r < -127.0f) r = -127.0f;
                q = (int)r;
            }
            out[2 + i] = (uint8_t)(int8_t)q;
        }
    }
}

/* w = f32(fp16 scale) * q; the product is exact in FP32 (11 x 8 bits). */
void orc_q8_0_unpack(const uint8_t* blocks, long n, float* w)
{
    for (long b = 0; b < n / ORC_BLOCK; b++) {
        const uint8_t* in = blocks + b * ORC_Q8_0_BYTES;
        float d = orc_f16_to_f32((uint16_t)(in[0] | (in[1] << 8)));
        for (int i = 0; i < ORC_BLOCK; i++)
            w[b * ORC_BLOCK + i] = d * (float)(int8_t)in[2 + i];
    }
}

/* ------------------------------------------------------------------ */
/* AFFINE4_GS32 ("Kipp Model Support", section                         */
/* "Quantization (AFFINE4_GS32)")                                       */
/* ------------------------------------------------------------------ */

/* The pages fix the group (32 weights), the parts (4-bit codes, an fp16 scale
 * and an fp16 bias) and the size (5.0 bits per weight, so 20 bytes a group).
 * Readings for the rest:
 *  - a weight is scale * q + bias with the code q in [0, 15] (affine: the
 *    bias is the value of code 0);
 *  - record layout: the 16 code bytes, weight 2i in the low nibble of byte i
 *    and weight 2i + 1 in its high nibble, then the scale, then the bias,
 *    each fp16 little-endian;
 *  - quantizer: bias = fp16(min), scale = fp16((max - min) / 15) with the
 *    subtraction and the division in FP32; each code rounds
 *    (w - bias) / scale, computed in FP32 against the stored (fp16) scale
 *    and bias, to the nearest integer, ties to even, clamped to [0, 15]; a
 *    stored scale of zero (a constant group, or a range below half the
 *    smallest fp16 step) gives all codes zero. */
void orc_affine4_pack(const float* w, long n, uint8_t* groups)
{
    for (long g = 0; g < n / ORC_BLOCK; g++) {
        const float* x = w + g * ORC_BLOCK;
        uint8_t* out = groups + g * ORC_AFFINE4_BYTES;
        float lo = x[0], hi = x[0];
        for (int i = 1; i < ORC_BLOCK; i++) {
            if (x[i] < lo) lo = x[i];
            if (x[i] > hi) hi = x[i];
        }
        float range = hi - lo;
        uint16_t sh = orc_f32_to_f16(range / 15.0f);
        uint16_t bh = orc_f32_to_f16(lo);
        float scale = orc_f16_to_f32(sh), bias = orc_f16_to_f32(bh);
        memset(out, 0, 16);
        for (int i = 0; i < ORC_BLOCK; i++) {
            int q = 0;
            if (scale != 0.0f) {
                float diff = x[i] - bias;
                float r = nearbyintf(diff / scale);
                if (r < 0.0f) r = 0.0f;
                if (r > 15.0f) r = 15.0f;
                q = (int)r;
            }
            out[i / 2] |= (uint8_t)(i % 2 ? q << 4 : q);
        }
        out[16] = (uint8_t)(sh & 0xff);
        out[17] = (uint8_t)(sh >> 8);
        out[18] = (uint8_t)(bh & 0xff);
        out[19] = (uint8_t)(bh >> 8);
    }
}

/* w = scale * q + bias rounded once to FP32.  In FP64 the product of an fp16
 * scale and a 4-bit code and its sum with an fp16 bias are exact (they span
 * at most 2^-24 .. 2^21, 45 bits), so one rounding follows. */
void orc_affine4_unpack(const uint8_t* groups, long n, float* w)
{
    for (long g = 0; g < n / ORC_BLOCK; g++) {
        const uint8_t* in = groups + g * ORC_AFFINE4_BYTES;
        double scale = orc_f16_to_f32((uint16_t)(in[16] | (in[17] << 8)));
        double bias = orc_f16_to_f32((uint16_t)(in[18] | (in[19] << 8)));
        for (int i = 0; i < ORC_BLOCK; i++) {
            int q = i % 2 ? in[i / 2] >> 4 : in[i / 2] & 0xf;
            w[g * ORC_BLOCK + i] = (float)(scale * q + bias);
        }
    }
}

/* ------------------------------------------------------------------ */
/* threads: split [0, n) into contiguous ranges, one per thread         */
/* ------------------------------------------------------------------ */

typedef void (*range_fn)(void* ctx, long i0, long i1);
typedef struct { range_fn fn; void* ctx; long i0, i1; } range_job;

static void* range_main(void* a)
{
    range_job* j = (range_job*)a;
    j->fn(j->ctx, j->i0, j->i1);
    return NULL;
}

static void parallel_for(long n, int n_threads, range_fn fn, void* ctx)
{
    if (n_threads < 1) n_threads = 1;
    if (n_threads > n) n_threads = (int)(n > 0 ? n : 1);
    if (n_threads == 1) { fn(ctx, 0, n); return; }
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * n_threads);
    range_job* jobs = (range_job*)malloc(sizeof(range_job) * n_threads);
    for (int k = 0; k < n_threads; k++) {
        jobs[k].fn = fn; jobs[k].ctx = ctx;
        jobs[k].i0 = n * k / n_threads;
        jobs[k].i1 = n * (k + 1) / n_threads;
        pthread_create(&th[k], NULL, range_main, &jobs[k]);
    }
    for (int k = 0; k < n_threads; k++) pthread_join(th[k], NULL);
    free(th);
    free(jobs);
}

/* ------------------------------------------------------------------ */
/* components                                                          */
/* ------------------------------------------------------------------ */

/* RMSNorm (reading): y = x / sqrt(mean(x^2) + eps) * g, eps inside the root,
 * the gain multiplies as stored (not 1 + g). */
void orc_rmsnorm(const float* x, const uint16_t* gain, int n, double eps, float* y)
{
    double ss = 0.0;
    for (int i = 0; i < n; i++) ss += (double)x[i] * (double)x[i];
    double r = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; i++)
        y[i] = (float)((double)x[i] * r * (double)orc_bf16_to_f32(gain[i]));
}

/* RoPE (reading: rotate-half pairing).  For i < d/2 the pair (v[i],
 * v[i + d/2]) turns by the angle pos * theta^(-2i/d):
 *   v[i]       <- v[i] cos a - v[i+d/2] sin a
 *   v[i + d/2] <- v[i+d/2] cos a + v[i] sin a
 * pos is the absolute 0-based position in the session. */
void orc_rope(float* v, int head_dim, int pos, double theta)
{
    int half = head_dim / 2;
    for (int i = 0; i < half; i++) {
        double inv_freq = pow(theta, -(2.0 * i) / head_dim);
        double a = (double)pos * inv_freq;
        double c = cos(a), s = sin(a);
        double x1 = v[i], x2 = v[i + half];
        v[i] = (float)(x1 * c - x2 * s);
        v[i + half] = (float)(x2 * c + x1 * s);
    }
}

/* SiLU(z) = z / (1 + e^-z) */
float orc_silu(float z)
{
    return (float)((double)z / (1.0 + exp(-(double)z)));
}

typedef struct {
    const void* W; int scheme, n_out, n_in;
    const float* x; int n_tok; float* y;
} matmul_job;

static void matmul_rows(void* a, long o0, long o1)
{
    matmul_job* j = (matmul_job*)a;
    double* w = (double*)malloc(sizeof(double) * j->n_in);
    float* wq = (float*)malloc(sizeof(float) * j->n_in);
    for (long o = o0; o < o1; o++) {
        if (j->scheme == ORC_BF16) {
            const uint16_t* row = (const uint16_t*)j->W + o * (long)j->n_in;
            for (int i = 0; i < j->n_in; i++) w[i] = orc_bf16_to_f32(row[i]);
        } else if (j->scheme == ORC_Q8_0) {
            const uint8_t* row = (const uint8_t*)j->W
                               + o * (long)(j->n_in / ORC_BLOCK) * ORC_Q8_0_BYTES;
            orc_q8_0_unpack(row, j->n_in, wq);
            for (int i = 0; i < j->n_in; i++) w[i] = wq[i];
        } else {
            const uint8_t* row = (const uint8_t*)j->W
                               + o * (long)(j->n_in / ORC_BLOCK) * ORC_AFFINE4_BYTES;
            orc_affine4_unpack(row, j->n_in, wq);
            for (int i = 0; i < j->n_in; i++) w[i] = wq[i];
        }
        for (int t = 0; t < j->n_tok; t++) {
            const float* xt = j->x + (long)t * j->n_in;
            double acc = 0.0;
            for (int i = 0; i < j->n_in; i++) acc += w[i] * (double)xt[i];
            j->y[(long)t * j->n_out + o] = (float)acc;
        }
    }
    free(w);
    free(wq);
}

/* y[t][o] = sum_i W[o][i] x[t][i], W row-major [n_out][n_in] (nn.Linear). */
void orc_matmul(const void* W, int scheme, int n_out, int n_in,
                const float* x, int n_tok, float* y, int n_threads)
{
    matmul_job j = { W, scheme, n_out, n_in, x, n_tok, y };
    parallel_for(n_out, n_threads, matmul_rows, &j);
}

/* Causal softmax attention of one query row over ctx cached positions
 * (reading: scale 1/sqrt(d), the max subtracted before exp, contiguous GQA
 * grouping: query head h reads KV head h / (n_q / n_kv)). */
static void gqa_attend_f32(const float* q, const float* K, const float* V,
                           int ctx, int n_q, int n_kv, int d, float* o);

void orc_gqa_attend(const float* q, const uint16_t* K, const uint16_t* V,
                    int ctx, int n_q, int n_kv, int d, float* o)
{
    long n = (long)ctx * n_kv * d;
    float* Kf = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
    float* Vf = (float*)malloc(sizeof(float) * (n > 0 ? n : 1));
    for (long i = 0; i < n; i++) {
        Kf[i] = orc_bf16_to_f32(K[i]);
        Vf[i] = orc_bf16_to_f32(V[i]);
    }
    gqa_attend_f32(q, Kf, Vf, ctx, n_q, n_kv, d, o);
    free(Kf);
    free(Vf);
}

/* The same over K and V already in FP32 (exact bf16 or Q8_0 values). */
static void gqa_attend_f32(const float* q, const float* K, const float* V,
                           int ctx, int n_q, int n_kv, int d, float* o)
{
    int group = n_q / n_kv;
    double scale = 1.0 / sqrt((double)d);
    double* s = (double*)malloc(sizeof(double) * (ctx > 0 ? ctx : 1));
    for (int h = 0; h < n_q; h++) {
        int kvh = h / group;
        const float* qh = q + (long)h * d;
        double mx = -INFINITY;
        for (int j = 0; j < ctx; j++) {
            const float* kj = K + ((long)j * n_kv + kvh) * d;
            double dot = 0.0;
            for (int i = 0; i < d; i++) dot += (double)qh[i] * kj[i];
            s[j] = dot * scale;
            if (s[j] > mx) mx = s[j];
        }
        double z = 0.0;
        for (int j = 0; j < ctx; j++) { s[j] = exp(s[j] - mx); z += s[j]; }
        for (int i = 0; i < d; i++) {
            double acc = 0.0;
            for (int j = 0; j < ctx; j++)
                acc += s[j] * V[((long)j * n_kv + kvh) * d + i];
            o[(long)h * d + i] = (float)(acc / z);
        }
    }
    free(s);
}

/* ------------------------------------------------------------------ */
/* model, KV storage, sessions                                         */
/* ------------------------------------------------------------------ */

struct orc_model {
    orc_cfg c;
    const uint16_t *embed, *final_norm, *lm_head;
    orc_layer* layers;
    int n_threads;
};

struct orc_pool {
    orc_model* m;
    int n_blocks;
    uint8_t *k, *v;         /* [L][n_blocks][32] K (V) rows of kv_row_bytes */
    int* ref;               /* holders of each block: sessions, +1 while published */
    /* content-addressed prefix index (orc_pool_enable_prefix) */
    int prefix_on;
    unsigned hash_mask;     /* buckets - 1 */
    int* bucket;            /* [buckets] first published block of the bucket, or -1 */
    int* next;              /* [n_blocks] next published block in the same bucket */
    int* parent;            /* [n_blocks] the published block before it (-1: first) */
    int* children;          /* [n_blocks] published blocks whose parent it is */
    long* stamp;            /* [n_blocks] last publish or attach, for eviction */
    int32_t* btok;          /* [n_blocks][32] the tokens of a published block */
    unsigned char* published;
    long clock;
};

struct orc_session {
    orc_model* m;
    orc_pool* pool;         /* NULL: contiguous */
    int max_ctx, pos;
    uint8_t *k, *v;         /* contiguous: [L][max_ctx] K (V) rows of kv_row_bytes */
    int32_t* table;         /* paged: block id per 32 positions */
    int n_table, n_given;   /* blocks taken; entries given by the caller */
    int32_t* toks;          /* [max_ctx] the token at each position */
};

orc_model* orc_model_create(const orc_cfg* cfg, const uint16_t* embed,
                            const uint16_t* final_norm, const uint16_t* lm_head,
                            const orc_layer* layers, int n_threads)
{
    if (cfg->n_q_heads % cfg->n_kv_heads || cfg->head_dim % 2 ||
        (cfg->kv_quant != ORC_BF16 && cfg->kv_quant != ORC_Q8_0) ||
        (cfg->kv_quant == ORC_Q8_0 && cfg->head_dim % ORC_BLOCK) ||
        (cfg->scheme != ORC_BF16 && cfg->scheme != ORC_Q8_0 && cfg->scheme != ORC_AFFINE4) ||
        (cfg->scheme != ORC_BF16 && (cfg->hidden % ORC_BLOCK || cfg->ffn % ORC_BLOCK ||
                                     (cfg->n_q_heads * cfg->head_dim) % ORC_BLOCK)))
        return NULL;
    orc_model* m = (orc_model*)calloc(1, sizeof(orc_model));
    m->c = *cfg;
    m->embed = embed;
    m->final_norm = final_norm;
    m->lm_head = cfg->tied ? embed : lm_head;
    m->layers = (orc_layer*)malloc(sizeof(orc_layer) * cfg->n_layers);
    memcpy(m->layers, layers, sizeof(orc_layer) * cfg->n_layers);
    m->n_threads = n_threads > 0 ? n_threads : 1;
    return m;
}

void orc_model_free(orc_model* m)
{
    if (!m) return;
    free(m->layers);
    free(m);
}

static long kv_row(const orc_cfg* c) { return (long)c->n_kv_heads * c->head_dim; }

/* Bytes of one position's K (or V) row: bf16 values, or Q8_0 blocks of 32
 * consecutive values (a head row of d values is d/32 whole blocks). */
static long kv_row_bytes(const orc_cfg* c)
{
    return c->kv_quant == ORC_Q8_0 ? kv_row(c) / ORC_BLOCK * ORC_Q8_0_BYTES : kv_row(c) * 2;
}

long orc_kv_bytes_per_position(const orc_cfg* c) { return 2 * kv_row_bytes(c); }

orc_pool* orc_pool_create(orc_model* m, int n_blocks)
{
    orc_pool* p = (orc_pool*)calloc(1, sizeof(orc_pool));
    long n = (long)m->c.n_layers * n_blocks * ORC_BLOCK * kv_row_bytes(&m->c);
    p->m = m;
    p->n_blocks = n_blocks;
    p->k = (uint8_t*)calloc(n, 1);
    p->v = (uint8_t*)calloc(n, 1);
    p->ref = (int*)calloc(n_blocks, sizeof(int));
    if (!p->k || !p->v || !p->ref) { orc_pool_free(p); return NULL; }
    return p;
}

void orc_pool_free(orc_pool* p)
{
    if (!p) return;
    free(p->k); free(p->v); free(p->ref);
    free(p->bucket); free(p->next); free(p->parent); free(p->children); free(p->stamp);
    free(p->btok); free(p->published);
    free(p);
}

/* ---- content-addressed prefix sharing ("Kipp Roadmap", status v0.0.3) ---- */

/* Readings (the pages name the parts, not the rules):
 *  - a published block is addressed by its content: the block before it in
 *    the chain (its parent, -1 for a prompt's first block) and its 32
 *    tokens; a lookup hashes that key (64-bit FNV-1a over the parent id and
 *    the tokens, little-endian) to a bucket and accepts a candidate only if
 *    its parent is equal and its tokens compare equal (memcmp), so a hash
 *    collision never shares a block;
 *  - only full blocks are published, when a session says it is finished
 *    with them (orc_session_publish); an equal block published earlier is
 *    shared in place of the session's own copy;
 *  - the index holds one reference to each published block, so it outlives
 *    its session; when the pool has no free block, the published block held
 *    by the index alone, with no published successor, that was published or
 *    attached longest ago is evicted;
 *  - a session writes only blocks that it alone holds: attaching stops on a
 *    block boundary, and a truncation into a shared block copies it first. */
int orc_pool_enable_prefix(orc_pool* p, int hash_bits)
{
    if (!p || hash_bits < 0 || hash_bits > 24 || p->prefix_on) return -1;
    int nb = 1 << hash_bits, n = p->n_blocks;
    p->bucket = (int*)malloc(sizeof(int) * nb);
    p->next = (int*)malloc(sizeof(int) * n);
    p->parent = (int*)malloc(sizeof(int) * n);
    p->children = (int*)calloc(n, sizeof(int));
    p->stamp = (long*)calloc(n, sizeof(long));
    p->btok = (int32_t*)calloc((size_t)n * ORC_BLOCK, sizeof(int32_t));
    p->published = (unsigned char*)calloc(n, 1);
    if (!p->bucket || !p->next || !p->parent || !p->children || !p->stamp || !p->btok ||
        !p->published)
        return -1;
    for (int i = 0; i < nb; i++) p->bucket[i] = -1;
    for (int i = 0; i < n; i++) p->next[i] = p->parent[i] = -1;
    p->hash_mask = (unsigned)nb - 1;
    p->prefix_on = 1;
    return 0;
}

int orc_pool_free_blocks(const orc_pool* p)
{
    int n = 0;
    for (int b = 0; b < p->n_blocks; b++) n += p->ref[b] == 0;
    return n;
}

static uint64_t block_hash(int parent, const int32_t* t)
{
    uint64_t h = 14695981039346656037ull;              /* FNV-1a offset basis */
    uint32_t words[1 + ORC_BLOCK];
    words[0] = (uint32_t)parent;
    for (int i = 0; i < ORC_BLOCK; i++) words[1 + i] = (uint32_t)t[i];
    for (int w = 0; w < 1 + ORC_BLOCK; w++)
        for (int b = 0; b < 4; b++) {
            h ^= (words[w] >> (8 * b)) & 0xffu;
            h *= 1099511628211ull;                     /* FNV-1a 64-bit prime */
        }
    return h;
}

static int find_published(orc_pool* p, int parent, const int32_t* t)
{
    for (int b = p->bucket[block_hash(parent, t) & p->hash_mask]; b >= 0; b = p->next[b])
        if (p->parent[b] == parent && memcmp(p->btok + (long)b * ORC_BLOCK, t,
                                             sizeof(int32_t) * ORC_BLOCK) == 0)
            return b;
    return -1;
}

static void index_insert(orc_pool* p, int b, int parent, const int32_t* t)
{
    unsigned h = (unsigned)(block_hash(parent, t) & p->hash_mask);
    memcpy(p->btok + (long)b * ORC_BLOCK, t, sizeof(int32_t) * ORC_BLOCK);
    p->parent[b] = parent;
    p->next[b] = p->bucket[h];
    p->bucket[h] = b;
    p->published[b] = 1;
    p->stamp[b] = ++p->clock;
    p->ref[b]++;
    if (parent >= 0) p->children[parent]++;
}

static void index_remove(orc_pool* p, int b)
{
    unsigned h = (unsigned)(block_hash(p->parent[b], p->btok + (long)b * ORC_BLOCK) & p->hash_mask);
    int* link = &p->bucket[h];
    while (*link != b) link = &p->next[*link];
    *link = p->next[b];
    if (p->parent[b] >= 0) p->children[p->parent[b]]--;
    p->next[b] = p->parent[b] = -1;
    p->published[b] = 0;
    p->ref[b]--;
}

/* a block someone else may read: published, or held by more than one */
static int shared_block(const orc_pool* p, int b)
{
    return p->ref[b] > 1 || (p->prefix_on && p->published[b]);
}

/* the lowest free block, evicting a published block when none is free */
static int take_block(orc_pool* p)
{
    for (int b = 0; b < p->n_blocks; b++)
        if (p->ref[b] == 0) { p->ref[b] = 1; return b; }
    if (!p->prefix_on) return -1;
    int best = -1;
    for (int b = 0; b < p->n_blocks; b++)
        if (p->published[b] && p->ref[b] == 1 && p->children[b] == 0 &&
            (best < 0 || p->stamp[b] < p->stamp[best]))
            best = b;
    if (best < 0) return -1;
    index_remove(p, best);
    p->ref[best] = 1;
    return best;
}

orc_session* orc_session_create(orc_model* m, orc_pool* pool, int max_ctx)
{
    orc_session* s = (orc_session*)calloc(1, sizeof(orc_session));
    s->m = m;
    s->pool = pool;
    s->max_ctx = max_ctx;
    if (!pool) {
        long n = (long)m->c.n_layers * max_ctx * kv_row_bytes(&m->c);
        s->k = (uint8_t*)calloc(n, 1);
        s->v = (uint8_t*)calloc(n, 1);
        if (!s->k || !s->v) { orc_session_free(s); return NULL; }
    } else {
        s->table = (int32_t*)calloc((max_ctx + ORC_BLOCK - 1) / ORC_BLOCK, sizeof(int32_t));
    }
    s->toks = (int32_t*)calloc(max_ctx > 0 ? max_ctx : 1, sizeof(int32_t));
    if (!s->toks || (pool && !s->table)) { orc_session_free(s); return NULL; }
    return s;
}

static void release_blocks(orc_session* s, int from)
{
    for (int b = from; b < s->n_table; b++) s->pool->ref[s->table[b]]--;
    s->n_table = from;
    if (s->n_given > from) s->n_given = from;
}

void orc_session_free(orc_session* s)
{
    if (!s) return;
    if (s->pool && s->table) release_blocks(s, 0);
    free(s->k); free(s->v); free(s->table); free(s->toks); free(s);
}

/* The caller fixes which pool blocks back the session's positions, in
 * order: block i holds positions [32 i, 32 i + 32). */
int orc_session_set_block_table(orc_session* s, const int32_t* ids, int n)
{
    if (!s->pool || s->pos != 0 || n < 0 || n > (s->max_ctx + ORC_BLOCK - 1) / ORC_BLOCK) return -1;
    release_blocks(s, 0);
    for (int i = 0; i < n; i++) {
        int dup = 0;
        for (int j = 0; j < i; j++) dup |= ids[j] == ids[i];
        if (ids[i] < 0 || ids[i] >= s->pool->n_blocks || s->pool->ref[ids[i]] || dup) return -1;
    }
    for (int i = 0; i < n; i++) {
        s->pool->ref[ids[i]] = 1;
        s->table[i] = ids[i];
    }
    s->n_table = n;
    s->n_given = n;
    return 0;
}

int orc_session_pos(const orc_session* s) { return s->pos; }

/* Forget positions >= n_pos.  Paged: blocks wholly past the new end go back
 * to the pool (those the caller fixed stay); a shared block that still holds
 * kept positions and would be written next is first copied to a block of the
 * session's own. */
int orc_session_truncate(orc_session* s, int n_pos)
{
    if (n_pos < 0 || n_pos > s->pos) return -1;
    if (s->pool) {
        orc_pool* p = s->pool;
        int keep = (n_pos + ORC_BLOCK - 1) / ORC_BLOCK;
        if (keep < s->n_given) keep = s->n_given < s->n_table ? s->n_given : s->n_table;
        if (keep < s->n_table) release_blocks(s, keep);
        int last = n_pos / ORC_BLOCK;                  /* the block position n_pos falls in */
        if (n_pos % ORC_BLOCK && last < s->n_table && shared_block(p, s->table[last])) {
            int b = s->table[last], nb = take_block(p);
            if (nb < 0) return -1;
            const orc_cfg* c = &s->m->c;
            long blk = ORC_BLOCK * kv_row_bytes(c);
            for (int l = 0; l < c->n_layers; l++) {
                memcpy(p->k + ((long)l * p->n_blocks + nb) * blk, p->k + ((long)l * p->n_blocks + b) * blk, blk);
                memcpy(p->v + ((long)l * p->n_blocks + nb) * blk, p->v + ((long)l * p->n_blocks + b) * blk, blk);
            }
            p->ref[b]--;
            s->table[last] = nb;
        }
    }
    s->pos = n_pos;
    return 0;
}

/* make room for positions [0, end): take the lowest free pool blocks */
static int reserve(orc_session* s, int end)
{
    if (end > s->max_ctx) return -1;
    if (!s->pool) return 0;
    int need = (end + ORC_BLOCK - 1) / ORC_BLOCK;
    while (s->n_table < need) {
        int b = take_block(s->pool);
        if (b < 0) return -1;
        s->table[s->n_table++] = b;
    }
    return 0;
}

/* Publish the session's full blocks: each becomes content-addressed, or is
 * swapped for an equal block published earlier (same chain, same tokens,
 * so the same K/V bits).  Returns the number of blocks newly published. */
int orc_session_publish(orc_session* s)
{
    orc_pool* p = s->pool;
    if (!p || !p->prefix_on || s->n_given) return -1;
    int parent = -1, count = 0;
    for (int i = 0; i < s->pos / ORC_BLOCK; i++) {
        int b = s->table[i];
        const int32_t* t = s->toks + (long)i * ORC_BLOCK;
        if (!p->published[b]) {
            int e = find_published(p, parent, t);
            if (e >= 0) {
                p->ref[e]++;
                p->ref[b]--;
                s->table[i] = e;
                b = e;
            } else {
                index_insert(p, b, parent, t);
                count++;
            }
        }
        parent = b;
    }
    return count;
}

/* Before a session's first round: attach the longest chain of published
 * blocks that matches the prompt's leading full blocks, keeping at least one
 * token of the prompt to evaluate.  Returns the positions attached (a
 * multiple of 32, and the session's new position). */
int orc_session_attach_prefix(orc_session* s, const int32_t* tokens, int n)
{
    orc_pool* p = s->pool;
    if (!p || !p->prefix_on || s->pos != 0 || s->n_given || n < 1 || n > s->max_ctx) return -1;
    release_blocks(s, 0);
    int parent = -1, i = 0;
    for (; i < (n - 1) / ORC_BLOCK; i++) {
        int e = find_published(p, parent, tokens + (long)i * ORC_BLOCK);
        if (e < 0) break;
        p->ref[e]++;
        p->stamp[e] = ++p->clock;
        s->table[i] = e;
        parent = e;
    }
    s->n_table = i;
    s->pos = i * ORC_BLOCK;
    memcpy(s->toks, tokens, sizeof(int32_t) * (size_t)s->pos);
    return s->pos;
}

/* address of the K (or V) row of position p in layer l */
static uint8_t* kv_slot(orc_session* s, int l, int p, int is_v)
{
    const orc_cfg* c = &s->m->c;
    if (!s->pool) {
        uint8_t* base = is_v ? s->v : s->k;
        return base + ((long)l * s->max_ctx + p) * kv_row_bytes(c);
    }
    uint8_t* base = is_v ? s->pool->v : s->pool->k;
    long blk = s->table[p / ORC_BLOCK];
    return base + (((long)l * s->pool->n_blocks + blk) * ORC_BLOCK + p % ORC_BLOCK) * kv_row_bytes(c);
}

/* store one position's K (or V) row: rounded to bf16, or packed to Q8_0
 * blocks straight from FP32 (reading: the quantizer of the weights) */
static void kv_store(const orc_cfg* c, const float* row, uint8_t* slot)
{
    if (c->kv_quant == ORC_Q8_0) {
        orc_q8_0_pack(row, kv_row(c), slot);
        return;
    }
    for (long i = 0; i < kv_row(c); i++) {
        uint16_t b = orc_f32_to_bf16(row[i]);
        slot[2 * i] = (uint8_t)(b & 0xff);
        slot[2 * i + 1] = (uint8_t)(b >> 8);
    }
}

/* read it back as FP32 values (exact: bf16 widening, or fp16 scale times quant) */
static void kv_load(const orc_cfg* c, const uint8_t* slot, float* row)
{
    if (c->kv_quant == ORC_Q8_0) {
        orc_q8_0_unpack(slot, kv_row(c), row);
        return;
    }
    for (long i = 0; i < kv_row(c); i++)
        row[i] = orc_bf16_to_f32((uint16_t)(slot[2 * i] | (slot[2 * i + 1] << 8)));
}

/* ---- one round over a set of rows (one or more sessions) ---- */

typedef struct {
    orc_session* const* S;
    const int* row_sess;     /* session of each row */
    const int* row_pos;      /* absolute position of each row */
    const float* q;          /* [T][n_q d] */
    float* att;              /* [T][n_q d] */
    int layer;
} attn_job;

static void attn_rows(void* a, long t0, long t1)
{
    attn_job* j = (attn_job*)a;
    for (long t = t0; t < t1; t++) {
        orc_session* s = j->S[j->row_sess[t]];
        const orc_cfg* c = &s->m->c;
        int ctx = j->row_pos[t] + 1;               /* causal: positions 0..pos */
        long kvr = kv_row(c);
        float* K = (float*)malloc(sizeof(float) * ctx * kvr);
        float* V = (float*)malloc(sizeof(float) * ctx * kvr);
        for (int p = 0; p < ctx; p++) {            /* gather through the layout */
            kv_load(c, kv_slot(s, j->layer, p, 0), K + p * kvr);
            kv_load(c, kv_slot(s, j->layer, p, 1), V + p * kvr);
        }
        long qw = (long)c->n_q_heads * c->head_dim;
        gqa_attend_f32(j->q + t * qw, K, V, ctx, c->n_q_heads, c->n_kv_heads,
                       c->head_dim, j->att + t * qw);
        free(K);
        free(V);
    }
}

/* One round over the sessions' rows (row t of the round: session row_sess[t],
 * rows of a session consecutive and in order).  sel: the rows whose logits
 * are wanted, increasing, n_sel of them; out: [n_sel][vocab].  With no row
 * wanted (n_sel == 0) nothing reads the last layer past its K/V store, so
 * the round stops there: the positions are appended with the same K/V. */
static int eval_rows(orc_session* const* S, const int32_t* const* toks, const int* n,
                     int ns, const int* sel, int n_sel, float* out)
{
    orc_model* m = S[0]->m;
    const orc_cfg* c = &m->c;
    const int H = c->hidden, F = c->ffn, d = c->head_dim;
    const int QW = c->n_q_heads * d, KW = c->n_kv_heads * d;
    int T = 0;
    for (int b = 0; b < ns; b++) {
        if (S[b]->m != m || n[b] < 1) return -1;
        for (int i = 0; i < n[b]; i++)
            if (toks[b][i] < 0 || toks[b][i] >= c->vocab) return -1;
        if (reserve(S[b], S[b]->pos + n[b])) return -1;
        if (S[b]->pool)
            for (int i = S[b]->pos / ORC_BLOCK; i <= (S[b]->pos + n[b] - 1) / ORC_BLOCK; i++)
                if (shared_block(S[b]->pool, S[b]->table[i])) return -1;
        T += n[b];
    }
    int* row_sess = (int*)malloc(sizeof(int) * T);
    int* row_pos = (int*)malloc(sizeof(int) * T);
    int* row_tok = (int*)malloc(sizeof(int) * T);
    for (int b = 0, t = 0; b < ns; b++)
        for (int i = 0; i < n[b]; i++, t++) {
            row_sess[t] = b;
            row_pos[t] = S[b]->pos + i;
            row_tok[t] = toks[b][i];
        }

    float* x = (float*)malloc(sizeof(float) * (long)T * H);
    float* h = (float*)malloc(sizeof(float) * (long)T * H);
    float* y = (float*)malloc(sizeof(float) * (long)T * H);
    float* q = (float*)malloc(sizeof(float) * (long)T * QW);
    float* k = (float*)malloc(sizeof(float) * (long)T * KW);
    float* v = (float*)malloc(sizeof(float) * (long)T * KW);
    float* att = (float*)malloc(sizeof(float) * (long)T * QW);
    float* g = (float*)malloc(sizeof(float) * (long)T * F);
    float* u = (float*)malloc(sizeof(float) * (long)T * F);

    /* token embedding: x = f32(E[token]) */
    for (int t = 0; t < T; t++)
        for (int i = 0; i < H; i++)
            x[(long)t * H + i] = orc_bf16_to_f32(m->embed[(long)row_tok[t] * H + i]);

    for (int l = 0; l < c->n_layers; l++) {
        const orc_layer* W = &m->layers[l];
        /* attention block */
        for (int t = 0; t < T; t++)
            orc_rmsnorm(x + (long)t * H, W->attn_norm, H, c->rms_eps, h + (long)t * H);
        orc_matmul(W->wq, c->scheme, QW, H, h, T, q, m->n_threads);
        orc_matmul(W->wk, c->scheme, KW, H, h, T, k, m->n_threads);
        orc_matmul(W->wv, c->scheme, KW, H, h, T, v, m->n_threads);
        for (int t = 0; t < T; t++) {
            for (int hh = 0; hh < c->n_q_heads; hh++) {   /* q-norm, then RoPE */
                float* qh = q + (long)t * QW + (long)hh * d;
                orc_rmsnorm(qh, W->q_norm, d, c->rms_eps, qh);
                orc_rope(qh, d, row_pos[t], c->rope_theta);
            }
            for (int hh = 0; hh < c->n_kv_heads; hh++) {  /* k-norm, then RoPE */
                float* kh = k + (long)t * KW + (long)hh * d;
                orc_rmsnorm(kh, W->k_norm, d, c->rms_eps, kh);
                orc_rope(kh, d, row_pos[t], c->rope_theta);
            }
            /* store K and V: rounded to bf16 (the KV storage contract) or
             * packed to Q8_0 (the opt-in quantized cache) */
            kv_store(c, k + (long)t * KW, kv_slot(S[row_sess[t]], l, row_pos[t], 0));
            kv_store(c, v + (long)t * KW, kv_slot(S[row_sess[t]], l, row_pos[t], 1));
        }
        if (n_sel == 0 && l == c->n_layers - 1) break;   /* no logits: nothing reads on */
        attn_job aj = { S, row_sess, row_pos, q, att, l };
        parallel_for(T, m->n_threads, attn_rows, &aj);
        orc_matmul(W->wo, c->scheme, H, QW, att, T, y, m->n_threads);
        for (long i = 0; i < (long)T * H; i++) x[i] = x[i] + y[i];

        /* FFN block: x += down(silu(gate(h)) * up(h)) */
        for (int t = 0; t < T; t++)
            orc_rmsnorm(x + (long)t * H, W->ffn_norm, H, c->rms_eps, h + (long)t * H);
        orc_matmul(W->wg, c->scheme, F, H, h, T, g, m->n_threads);
        orc_matmul(W->wu, c->scheme, F, H, h, T, u, m->n_threads);
        for (long i = 0; i < (long)T * F; i++)
            g[i] = (float)((double)orc_silu(g[i]) * (double)u[i]);
        orc_matmul(W->wd, c->scheme, H, F, g, T, y, m->n_threads);
        for (long i = 0; i < (long)T * H; i++) x[i] = x[i] + y[i];
    }

    /* final norm and lm_head on the requested rows */
    if (n_sel > 0) {
        for (int i = 0; i < n_sel; i++)
            orc_rmsnorm(x + (long)sel[i] * H, m->final_norm, H, c->rms_eps, h + (long)i * H);
        orc_matmul(m->lm_head, ORC_BF16, c->vocab, H, h, n_sel, out, m->n_threads);
    }
    for (int b = 0; b < ns; b++) {
        memcpy(S[b]->toks + S[b]->pos, toks[b], sizeof(int32_t) * (size_t)n[b]);
        S[b]->pos += n[b];
    }

    free(x); free(h); free(y); free(q); free(k); free(v); free(att); free(g); free(u);
    free(row_sess); free(row_pos); free(row_tok);
    return 0;
}

int orc_eval(orc_session* s, const int32_t* tokens, int n, float* logits_last,
             float* logits_all)
{
    if (n < 1) return -1;
    int* sel = (int*)malloc(sizeof(int) * (size_t)n);
    int n_sel = 0;
    if (logits_all)
        for (int t = 0; t < n; t++) sel[n_sel++] = t;
    else if (logits_last)
        sel[n_sel++] = n - 1;
    float* out = logits_all ? logits_all : logits_last;
    int rc = eval_rows(&s, &tokens, &n, 1, sel, n_sel, out);
    if (rc == 0 && logits_all && logits_last)
        memcpy(logits_last, logits_all + (long)(n - 1) * s->m->c.vocab,
               sizeof(float) * s->m->c.vocab);
    free(sel);
    return rc;
}

int orc_eval_rows(orc_session* s, const int32_t* tokens, int n, const int* rows,
                  int n_rows, float* logits)
{
    if (n < 1 || n_rows < 0 || (n_rows > 0 && !logits)) return -1;
    for (int i = 0; i < n_rows; i++)
        if (rows[i] < 0 || rows[i] >= n || (i > 0 && rows[i] <= rows[i - 1])) return -1;
    return eval_rows(&s, &tokens, &n, 1, rows, n_rows, logits);
}

int orc_eval_batch(orc_session* const* s, const int32_t* const* tokens,
                   const int* n, int ns, float* logits)
{
    if (ns < 1) return -1;
    for (int a = 0; a < ns; a++) {
        if (n[a] < 1) return -1;
        for (int b = 0; b < a; b++)
            if (s[a] == s[b]) return -1;
    }
    int* sel = (int*)malloc(sizeof(int) * (size_t)ns);
    for (int b = 0, t = 0; b < ns; b++) {
        t += n[b];
        sel[b] = t - 1;                 /* the last row of each session's round */
    }
    int rc = eval_rows(s, tokens, n, ns, logits ? sel : NULL, logits ? ns : 0, logits);
    free(sel);
    return rc;
}
