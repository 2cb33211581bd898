// k_decode.cu -- the one-token decode round of one session as one persistent
// kernel.
//
// A decode step streams every projection, the KV context and the lm_head
// once ("Kipp Roadmap", status v0.0.4: split-K decode matvec; "Kipp Model
// Support", section "qwen3-0.6b-base": BF16 K/V, RMSNorm before attention
// and MLP, q/k head norms, RoPE, SwiGLU, greedy argmax).  On GB300 the bytes
// are ~1.2 ms of HBM time at batch 1, so what decides the step time is how
// much of that time HBM is kept busy.  Launching one kernel per operation
// leaves HBM idle at every boundary (drain, launch, ramp).  This kernel
// runs the whole step with one CTA per SM:
//  - a producer warp walks the same stage sequence as the consumers and
//    streams this CTA's share of every stage -- weight rows, and the KV
//    blocks of its attention unit -- into a ring of shared-memory slots with
//    bulk copies (evict-first in L2).  Weights and earlier KV do not depend
//    on this step's activations, so the producer runs ahead across stage
//    boundaries and HBM keeps streaming while the consumers wait at a
//    barrier;
//  - 16 consumer warps compute each stage from the ring: matvec tiles with
//    the activation row staged in shared memory (RMS-normalised on the way
//    in for QKV, gate/up and the lm_head), attention units with the per-head
//    q/k RMSNorm, RoPE and the KV append fused in, and the epilogues
//    (store, residual add, SwiGLU, greedy argmax);
//  - stages that need the previous stage's output of other CTAs (5 per
//    layer) are separated by a grid barrier: a monotonic global counter,
//    release-add then acquire-spin, bounded in time.  The launch is
//    cooperative, so all CTAs are resident.
// Row partials are summed in a fixed order (lanes, then warp segments in
// order), attention splits merge in split order, so results do not depend
// on scheduling.  Every wait is bounded: on timeout the kernel records
// Q3_STATUS_TIMEOUT, unwinds, and waits (bounded) for its copies in flight.
#include "common.cuh"
#include "kernels.h"
#include "attn_block.cuh"

namespace q3 {

namespace {

typedef __nv_bfloat16 bf16;

constexpr int NCW = 16;                    // consumer warps
constexpr int NCT = NCW * 32;              // consumer threads
constexpr int PRODUCER = NCW;              // warp index of the producer
constexpr int EPILOGUE = NCW + 1;          // warp index of the epilogue warp
constexpr int THREADS = NCT + 64;          // + producer and epilogue warps
constexpr int SLOT = 40 * 1024;            // bytes per ring slot
constexpr int RED = 64;                    // row partials per slot (rows x warp segments)
constexpr int D = 128, KVB = 32;
constexpr int KSTR = D + 8;                // staged K/V/q row stride (bf16): 272 bytes, conflict-free ldmatrix
constexpr int KT_BYTES = KVB * KSTR * 2;
constexpr int VT_BYTES = KVB * KSTR * 2;
constexpr int BLK_BYTES = KT_BYTES + VT_BYTES;
constexpr int BLKS_PER_SLOT = 2;
constexpr int CONS_BAR = 1;                // named barrier of the consumer warps
constexpr int MIN_SLOTS = 3, MAX_SLOTS = 8;
constexpr int XCPL = 5;
constexpr int MAX_OWN = 64;                // residual rows a CTA owns (H / grid, rounded up)                    // activation chunks a lane keeps in registers (bf16 tiles)

static_assert(BLKS_PER_SLOT * BLK_BYTES <= SLOT, "two KV blocks per slot");

enum StageKind { ST_QKV, ST_O, ST_GU, ST_DOWN, ST_LM };

__host__ __device__ inline int row_bytes(int K, bool q8) { return q8 ? K + K / 16 : 2 * K; }

// rows per ring slot: the largest power of two (<= the consumer warps) whose
// rows fit in a slot (a gate/up pair tile holds half gate rows, half up rows)
__host__ __device__ inline int tile_rows(int K, bool q8) {
    int nr = 1;
    while (nr < NCW && 2 * nr * row_bytes(K, q8) <= SLOT) nr *= 2;
    return nr;
}

// Attention scratch (floats) inside the activation area: q heads, the new
// K/V row, per-warp partials, split maxima/weights, and the partial outputs
// (per warp, or all splits of the KV head while the last split CTA merges).
struct AttScratch {
    int sq, snew, pm, pl, sml, sw, po, total;
};

__host__ __device__ inline AttScratch att_scratch(int G, int ns) {
    AttScratch a;
    int o = 0;
    a.sq = o; o += 16 * KSTR / 2;                 // bf16 [16][KSTR]: q hi / lo rows
    a.snew = o; o += D;
    a.pm = o; o += 4 * G;
    a.pl = o; o += 4 * G;
    a.sml = o; o += 2 * G * ns;
    a.sw = o; o += G * ns;
    o = (o + 3) & ~3;
    a.po = o; o += (4 * G * D > G * ns * D ? 4 * G * D : G * ns * D);
    a.total = o;
    return a;
}

// floats of the activation / attention scratch area
__host__ __device__ inline int sx_floats(int H, int F, int n_q, int n_kv, int n_splits) {
    int k = H > n_q * D ? H : n_q * D;
    k = k > F ? k : F;
    const int att = att_scratch(n_q / n_kv, n_splits).total;
    k = k > att ? k : att;
    return (k + 3) & ~3;
}

// per-layer pointer table in shared memory: 7 weight planes, 7 Q8_0 scale
// planes, then the attention, q, k and FFN norm gains
constexpr int WP_N = 18, WP_ATTN_NORM = 14, WP_Q_NORM = 15, WP_K_NORM = 16, WP_FFN_NORM = 17;

struct Layout {
    size_t sx, red, bars, misc, ptrs, total;
};

__host__ __device__ inline Layout make_layout(int n_slots, int sxf, int n_layers) {
    Layout L;
    L.sx = (size_t)n_slots * SLOT;
    L.red = L.sx + (size_t)sxf * 4;
    L.bars = L.red + (size_t)n_slots * RED * 4;
    L.misc = L.bars + (size_t)(3 * n_slots) * 8;
    L.ptrs = L.misc + (size_t)(3 * NCW + 4 + MAX_OWN) * 4;
    L.ptrs = (L.ptrs + 15) & ~(size_t)15;
    L.total = L.ptrs + (size_t)n_layers * WP_N * 8;   // per layer: weight planes, scale planes, norm gains
    return L;
}

struct Smem {
    uint8_t* ring;
    float* sx;          // activation row, or attention scratch
    float* red;         // [n_slots][RED]
    uint64_t* full;     // [n_slots] tile landed (tx bytes)
    uint64_t* empty;    // [n_slots] tile consumed: NCW readers + the epilogue warp
    uint64_t* redf;     // [n_slots] all NCW row partials written
    float* ss;          // [NCW]
    float* bv;          // [NCW]
    int* bi;            // [NCW]
    volatile int* abort;
    int* ticket;
    float* xres;        // [MAX_OWN] the CTA's residual rows (epilogue warp only)
    const void** wp;    // [n_layers][14]: the layer's 7 weight planes, then their 7 scale planes
    int n_slots;
};

// ---------------------------------------------------------------- small helpers
Q3_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

Q3_DEV bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

Q3_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

Q3_DEV float dot8(uint4 w, float4 a, float4 b) {
    float s = bf16lo(w.x) * a.x;
    s = fmaf(bf16hi(w.x), a.y, s);
    s = fmaf(bf16lo(w.y), a.z, s);
    s = fmaf(bf16hi(w.y), a.w, s);
    s = fmaf(bf16lo(w.z), b.x, s);
    s = fmaf(bf16hi(w.z), b.y, s);
    s = fmaf(bf16lo(w.w), b.z, s);
    s = fmaf(bf16hi(w.w), b.w, s);
    return s;
}

Q3_DEV float dot4_i8(uint32_t q, float4 a) {
    const uint32_t f = q ^ 0x80808080u;
    float s = i8_byte(f, 0x7650) * a.x;
    s = fmaf(i8_byte(f, 0x7651), a.y, s);
    s = fmaf(i8_byte(f, 0x7652), a.z, s);
    s = fmaf(i8_byte(f, 0x7653), a.w, s);
    return s;
}

Q3_DEV uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// bulk copy global -> shared with an L2 cache policy (16-byte aligned, size a
// multiple of 16)
Q3_DEV void bulk_load_hint(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol) : "memory");
}

Q3_DEV unsigned long long ld_acquire_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

Q3_DEV void consumer_sync() { named_bar(CONS_BAR, NCT); }

// Bounded mbarrier wait that also gives up as soon as the CTA is aborting.
Q3_DEV bool wait_bar(uint64_t* bar, uint32_t parity, const Smem& sm, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*sm.abort) return false;
        if (global_ns() - t0 > Q3_WAIT_LIMIT_NS) {
            set_status(status, Q3_STATUS_TIMEOUT);
            *sm.abort = 1;
            return false;
        }
    }
}

// Grid barrier among the consumer warps of all CTAs.  After a matvec stage
// (by_epilogue) this CTA's arrival is the epilogue warp's: it releases the
// stage's outputs as soon as it has written them; after the attention stage
// the consumers' thread 0 releases theirs.  Returns false, the same on every
// consumer thread, when the step is aborting.
Q3_DEV bool grid_sync(const DecodeArgs& p, const Smem& sm, unsigned long long target, bool by_epilogue) {
    consumer_sync();
    if (threadIdx.x == 0 && !*sm.abort) {
        if (!by_epilogue) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" :: "l"(p.bar) : "memory");
        const uint64_t t0 = global_ns();
        for (uint32_t n = 1; ld_acquire_u64(p.bar) < target; ++n) {
            if ((n & 63) == 0 && global_ns() - t0 > Q3_WAIT_LIMIT_NS) {
                set_status(p.status, Q3_STATUS_TIMEOUT);
                *sm.abort = 1;
                break;
            }
        }
    }
    return named_bar_and(CONS_BAR, NCT, *sm.abort == 0);
}

// ---------------------------------------------------------------- stages
// One matvec stage: rows of up to three tensors stacked (QKV), or gate/up
// row pairs; this CTA owns the row (pair) range [r0, r1).
struct WStage {
    const uint8_t* w[3];
    const __half* sc[3];
    int rows[3];
    int K, pair, q8, nr, per, r0, r1;
};

Q3_DEV WStage weight_stage(const DecodeArgs& p, const Smem& sm, int l, int kind) {
    WStage s{};
    const int qw = p.n_q * D, kvw = p.n_kv * D;
    int M;
    if (kind == ST_LM) {
        s.w[0] = reinterpret_cast<const uint8_t*>(p.lm_head);
        s.rows[0] = p.V;
        s.K = p.H;
        M = p.V;
    } else {
        const void* const* lp = sm.wp + (size_t)l * WP_N;
        s.q8 = p.q8;
        auto set = [&](int i, int proj, int rows) {
            s.w[i] = static_cast<const uint8_t*>(lp[proj]);
            s.sc[i] = static_cast<const __half*>(lp[7 + proj]);
            s.rows[i] = rows;
        };
        switch (kind) {
        case ST_QKV: set(0, 0, qw); set(1, 1, kvw); set(2, 2, kvw); s.K = p.H; M = qw + 2 * kvw; break;
        case ST_O: set(0, 3, p.H); s.K = qw; M = p.H; break;
        case ST_GU: set(0, 4, p.F); set(1, 5, p.F); s.K = p.H; s.pair = 1; M = p.F; break;
        default: set(0, 6, p.H); s.K = p.F; M = p.H; break;
        }
    }
    s.nr = tile_rows(s.K, s.q8);
    s.per = s.pair ? s.nr / 2 : s.nr;
    s.r0 = (int)((long long)blockIdx.x * M / gridDim.x);
    s.r1 = (int)((long long)(blockIdx.x + 1) * M / gridDim.x);
    return s;
}

// This CTA's attention unit: KV head kvh, split `split` of the context's
// 32-position blocks [b0, b1).
struct Unit {
    int kvh, split, b0, b1, nblk, ctx, pos;
    bool active;
};

Q3_DEV Unit attention_unit(const DecodeArgs& p) {
    Unit u;
    u.pos = p.row_pos[0];
    u.ctx = u.pos + 1;
    u.nblk = (u.ctx + KVB - 1) / KVB;
    u.active = (int)blockIdx.x < p.n_kv * p.n_splits;
    u.kvh = blockIdx.x / p.n_splits;
    u.split = blockIdx.x % p.n_splits;
    const int bps = (u.nblk + p.n_splits - 1) / p.n_splits;
    u.b0 = u.split * bps;
    u.b1 = min(u.b0 + bps, u.nblk);
    if (!u.active || u.b1 < u.b0) u.b1 = u.b0;
    return u;
}

Q3_DEV const bf16* kv_block(const DecodeArgs& p, int l, int phys, int kvh) {
    return p.kv + (size_t)l * p.layer_kv + ((size_t)phys * 2 * p.n_kv + kvh) * (KVB * D);
}

// ---------------------------------------------------------------- producer
Q3_DEV bool acquire_slot(const Smem& sm, int slot, uint32_t use, int lane, int* status) {
    bool ok = true;
    if (lane == 0 && use > 0) ok = wait_bar(&sm.empty[slot], (use - 1) & 1, sm, status);
    return __shfl_sync(0xffffffffu, ok, 0);
}

template <bool Q8>
Q3_DEV bool produce_weights(const WStage& s, const Smem& sm, uint32_t& it, int lane, int* status,
                            uint64_t pol) {
    const size_t qb = Q8 ? (size_t)s.K : (size_t)s.K * 2;   // quant (or bf16) bytes per row
    const size_t sb = Q8 ? (size_t)s.K / 16 : 0;            // fp16 scale bytes per row
    for (int a = s.r0; a < s.r1; a += s.per) {
        const int b = min(a + s.per, s.r1), n = b - a;
        const int slot = it % sm.n_slots;
        if (!acquire_slot(sm, slot, it / sm.n_slots, lane, status)) return false;
        if (lane == 0) {
            uint8_t* dst = sm.ring + (size_t)slot * SLOT;
            uint8_t* dsc = dst + (size_t)s.nr * qb;            // scale rows follow the quant rows
            mbar_arrive_expect_tx(&sm.full[slot], (uint32_t)((size_t)n * (qb + sb) * (s.pair ? 2 : 1)));
            if (s.pair) {
                for (int t = 0; t < 2; ++t) {
                    bulk_load_hint(dst + (size_t)t * s.per * qb, s.w[t] + (size_t)a * qb,
                                   (uint32_t)(n * qb), &sm.full[slot], pol);
                    if (Q8)
                        bulk_load_hint(dsc + (size_t)t * s.per * sb,
                                       reinterpret_cast<const uint8_t*>(s.sc[t]) + (size_t)a * sb,
                                       (uint32_t)(n * sb), &sm.full[slot], pol);
                }
            } else {
                int r = a, base = 0;
                for (int t = 0; t < 3 && r < b; ++t) {
                    const int e = min(b, base + s.rows[t]);
                    if (r < e) {
                        bulk_load_hint(dst + (size_t)(r - a) * qb, s.w[t] + (size_t)(r - base) * qb,
                                       (uint32_t)((e - r) * qb), &sm.full[slot], pol);
                        if (Q8)
                            bulk_load_hint(dsc + (size_t)(r - a) * sb,
                                           reinterpret_cast<const uint8_t*>(s.sc[t]) + (size_t)(r - base) * sb,
                                           (uint32_t)((e - r) * sb), &sm.full[slot], pol);
                        r = e;
                    }
                    base += s.rows[t];
                }
            }
        }
        __syncwarp();
        ++it;
    }
    return true;
}

// KV blocks of the attention unit, two per slot: K and V rows padded to KSTR
// (one 256-byte copy per row; lane l copies row l of both).
Q3_DEV bool produce_attention(const DecodeArgs& p, int l, const Unit& u, const int* table,
                              const Smem& sm, uint32_t& it, int lane) {
    for (int b = u.b0; b < u.b1; b += BLKS_PER_SLOT) {
        const int nb = min(BLKS_PER_SLOT, u.b1 - b);
        const int slot = it % sm.n_slots;
        if (!acquire_slot(sm, slot, it / sm.n_slots, lane, p.status)) return false;
        int phys[BLKS_PER_SLOT];
        uint32_t bytes = 0;
#pragma unroll
        for (int j = 0; j < BLKS_PER_SLOT; ++j) {
            phys[j] = j < nb ? table[b + j] : -1;
            if (phys[j] >= p.n_blocks) phys[j] = -1;
            if (phys[j] >= 0) bytes += 2 * KVB * D * 2;   // 64 rows of 256 bytes
        }
        if (lane == 0) mbar_arrive_expect_tx(&sm.full[slot], bytes);
        __syncwarp();
        uint8_t* dst = sm.ring + (size_t)slot * SLOT;
#pragma unroll
        for (int j = 0; j < BLKS_PER_SLOT; ++j) {
            if (phys[j] < 0) continue;
            const bf16* Kb = kv_block(p, l, phys[j], u.kvh);
            const bf16* Vb = Kb + (size_t)p.n_kv * KVB * D;
            bulk_load(dst + j * BLK_BYTES + lane * KSTR * 2, Kb + lane * D, D * 2, &sm.full[slot]);
            bulk_load(dst + j * BLK_BYTES + KT_BYTES + lane * KSTR * 2, Vb + lane * D, D * 2, &sm.full[slot]);
        }
        __syncwarp();
        ++it;
    }
    return true;
}

template <bool Q8>
Q3_DEV void producer(const DecodeArgs& p, const Unit& u, const int* table, const Smem& sm, int lane) {
    const uint64_t pol = policy_evict_first();
    uint32_t it = 0;
    bool ok = true;
    for (int l = 0; l < p.n_layers && ok; ++l) {
        ok = produce_weights<Q8>(weight_stage(p, sm, l, ST_QKV), sm, it, lane, p.status, pol) &&
             produce_attention(p, l, u, table, sm, it, lane) &&
             produce_weights<Q8>(weight_stage(p, sm, l, ST_O), sm, it, lane, p.status, pol) &&
             produce_weights<Q8>(weight_stage(p, sm, l, ST_GU), sm, it, lane, p.status, pol) &&
             produce_weights<Q8>(weight_stage(p, sm, l, ST_DOWN), sm, it, lane, p.status, pol);
    }
    if (ok) produce_weights<false>(weight_stage(p, sm, 0, ST_LM), sm, it, lane, p.status, pol);
    // copies still in flight must land before the CTA may exit
    if (lane == 0) {
        for (int s = 0; s < sm.n_slots; ++s)
            if (it > (uint32_t)s) mbar_wait(&sm.full[s], ((it - 1 - s) / sm.n_slots) & 1, p.status);
    }
}

// ---------------------------------------------------------------- consumers
// Stage the activation row (f32, or the bf16 embedding row) into shared
// memory, RMS-normalised with `gain` when given.
// Rows with a gain (the hidden width, at most 4 NCT GAIN_IT) fetch the gain in
// the same pass as the row, held in registers until the scale is known.
constexpr int GAIN_IT = 3;

Q3_DEV void stage_x(const Smem& sm, const float* src, const bf16* src16, int K, const bf16* gain,
                    float eps) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    float ss = 0.f;
    if (gain) {
        uint2 gr[GAIN_IT];
#pragma unroll
        for (int k = 0; k < GAIN_IT; ++k) {
            const int i = (tid + k * NCT) * 4;
            if (i < K) {
                float4 v;
                if (src16) {
                    const uint2 w = *reinterpret_cast<const uint2*>(src16 + i);
                    v = make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
                } else {
                    v = __ldcg(reinterpret_cast<const float4*>(src + i));
                }
                gr[k] = *reinterpret_cast<const uint2*>(gain + i);
                *reinterpret_cast<float4*>(sm.sx + i) = v;
                ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
            }
        }
        ss = warp_sum(ss);
        if (lane == 0) sm.ss[warp] = ss;
        consumer_sync();
        float t = 0.f;
        for (int w = 0; w < NCW; ++w) t += sm.ss[w];
        const float scl = 1.0f / sqrtf(t / (float)K + eps);
#pragma unroll
        for (int k = 0; k < GAIN_IT; ++k) {
            const int i = (tid + k * NCT) * 4;
            if (i < K) {
                float4 v = *reinterpret_cast<const float4*>(sm.sx + i);
                v.x = v.x * scl * bf16lo(gr[k].x);
                v.y = v.y * scl * bf16hi(gr[k].x);
                v.z = v.z * scl * bf16lo(gr[k].y);
                v.w = v.w * scl * bf16hi(gr[k].y);
                *reinterpret_cast<float4*>(sm.sx + i) = v;
            }
        }
    } else {
        for (int i = tid * 4; i < K; i += NCT * 4) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(src + i));
            *reinterpret_cast<float4*>(sm.sx + i) = v;
        }
    }
    consumer_sync();
}

// The epilogue of one tile, once every warp's segment sums are in: rows add
// their S segment sums in segment order; store, residual add, SwiGLU of a
// gate/up pair, or store plus greedy-argmax tracking.
Q3_DEV void tile_epilogue(const WStage& s, int kind, const float* red, int S, int a, int nvalid, int lane,
                          float* out, float* xres, float& best, int& best_i) {
    for (int rho = lane; rho < nvalid; rho += 32) {
        const int row = a + rho;
        float v = 0.f;
        for (int q = 0; q < S; ++q) v += red[rho * S + q];
        if (s.pair) {
            float u = 0.f;
            for (int q = 0; q < S; ++q) u += red[(rho + s.per) * S + q];
            __stcg(out + row, silu(v) * u);
        } else if (kind == ST_O || kind == ST_DOWN) {
            // the residual row lives in shared memory; global memory gets a copy
            const float x = xres[row - s.r0] + v;
            xres[row - s.r0] = x;
            __stcg(out + row, x);
        } else {
            __stcg(out + row, v);
            if (kind == ST_LM && better(v, row, best, best_i)) { best = v; best_i = row; }
        }
    }
}

// A consumer warp hands a tile back: its segment sums are posted, the slot
// released on its side.
Q3_DEV void tile_finish(const Smem& sm, int slot, int lane) {
    __syncwarp();
    if (lane == 0) {
        mbar_arrive(&sm.redf[slot]);
        mbar_arrive(&sm.empty[slot]);
    }
}

// BF16 matvec tiles.  A tile holds nr rows; warp w takes row w / S and the
// (w % S)-th of S = NCW / nr contiguous segments of the row's 16-byte chunks
// (at most 32 XCPL per segment).  The lane's activation chunks (c0 + lane +
// 32 j) are loaded into registers once per stage, so the inner loop only
// reads weights: XCPL independent 8-term dot products per lane and tile.
Q3_DEV void consume_bf16(const WStage& s, const Smem& sm, uint32_t& it, int warp, int lane,
                         const DecodeArgs& p) {
    const int nr = s.nr, S = NCW / nr;
    const int row = warp / S, seg = warp % S;
    const int nch = s.K / 8;
    const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
    const size_t qb = (size_t)s.K * 2;
    float4 xa[XCPL], xb[XCPL];
#pragma unroll
    for (int j = 0; j < XCPL; ++j) {
        const int c = c0 + lane + 32 * j;
        xa[j] = c < c1 ? *reinterpret_cast<const float4*>(sm.sx + c * 8) : make_float4(0.f, 0.f, 0.f, 0.f);
        xb[j] = c < c1 ? *reinterpret_cast<const float4*>(sm.sx + c * 8 + 4) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    for (int a = s.r0; a < s.r1; a += s.per) {
        const int nvalid = min(s.per, s.r1 - a);
        const int slot = it % sm.n_slots;
        const uint32_t use = it / sm.n_slots;
        ++it;
        if (!wait_bar(&sm.full[slot], use & 1, sm, p.status)) return;
        const bool rv = s.pair ? (row % s.per) < nvalid : row < nvalid;
        float acc = 0.f;
        if (rv) {
            const uint8_t* trow = sm.ring + (size_t)slot * SLOT + (size_t)row * qb;
            float part[XCPL];
#pragma unroll
            for (int j = 0; j < XCPL; ++j) {
                const int c = c0 + lane + 32 * j;
                part[j] = c < c1 ? dot8(*reinterpret_cast<const uint4*>(trow + (size_t)c * 16), xa[j], xb[j]) : 0.f;
            }
#pragma unroll
            for (int j = 0; j < XCPL; ++j) acc += part[j];
        }
        acc = warp_sum(acc);
        if (lane == 0) sm.red[slot * RED + row * S + seg] = acc;
        tile_finish(sm, slot, lane);
    }
}

// Q8_0 matvec tiles (int8 quant rows, then their fp16 scale rows).  The tile
// is split into nr / RB row groups of RB rows; the S = NCW / groups warps of a
// group each take one contiguous segment of the 16-quant chunks, so one
// activation load (from shared memory) serves RB rows.
Q3_DEV void consume_q8(const WStage& s, const Smem& sm, uint32_t& it, int warp, int lane,
                       const DecodeArgs& p) {
    const int nr = s.nr, RB = nr < 4 ? nr : 4, G = nr / RB, S = NCW / G;
    const int grp = warp / S, seg = warp % S;
    const int nch = s.K / 16;
    const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
    const size_t qb = (size_t)s.K, sb = (size_t)s.K / 16;
    for (int a = s.r0; a < s.r1; a += s.per) {
        const int nvalid = min(s.per, s.r1 - a);
        const int slot = it % sm.n_slots;
        const uint32_t use = it / sm.n_slots;
        ++it;
        if (!wait_bar(&sm.full[slot], use & 1, sm, p.status)) return;
        const uint8_t* tile = sm.ring + (size_t)slot * SLOT;
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        bool rv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int rho = grp * RB + i;
            rv[i] = i < RB && (s.pair ? (rho % s.per) < nvalid : rho < nvalid);
        }
        const uint8_t* trow = tile + (size_t)(grp * RB) * qb;
        for (int c = c0 + lane; c < c1; c += 32) {
            const float4* h = reinterpret_cast<const float4*>(sm.sx + c * 16);
            const float4 h0 = h[0], h1 = h[1], h2 = h[2], h3 = h[3];
            const uint8_t* tsc = tile + (size_t)nr * qb + (size_t)(grp * RB) * sb + (c >> 1) * 2;
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (rv[i]) {
                    const uint4 q = *reinterpret_cast<const uint4*>(trow + i * qb + c * 16);
                    const float d = dot4_i8(q.x, h0) + dot4_i8(q.y, h1) + dot4_i8(q.z, h2) + dot4_i8(q.w, h3);
                    acc[i] = fmaf(__half2float(*reinterpret_cast<const __half*>(tsc + i * sb)), d, acc[i]);
                }
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if (i < RB) {
                const float v = warp_sum(acc[i]);
                if (lane == 0) sm.red[slot * RED + (grp * RB + i) * S + seg] = v;
            }
        }
        tile_finish(sm, slot, lane);
    }
}

template <bool Q8>
Q3_DEV void consume_weights(const WStage& s, const Smem& sm, uint32_t& it, int warp, int lane,
                            const DecodeArgs& p) {
    if (Q8) consume_q8(s, sm, it, warp, lane, p);
    else consume_bf16(s, sm, it, warp, lane, p);
}

// ---------------------------------------------------------------- attention on tensor cores
constexpr int ATT_DQ = 4;                  // warps per block: each takes 128 / ATT_DQ output dims
constexpr int ATT_DT = D / 8 / ATT_DQ;     // dimension tiles of 8 per warp
static_assert(KSTR == ATT_KSTR, "staged rows of the shared block routine");
using AttWarp = AttAcc<ATT_DT>;

// The attention unit of this CTA: q heads of its KV head normed, rotated and
// split into bf16 high/low rows; the new K/V appended (by the unit holding
// the last block) and patched into its staged tile; blocks attended on
// tensor cores by groups of ATT_DQ warps (block j of each round of 4, one
// quarter of the output dimensions each);
// then merged: block lanes in order, then splits in order by the last split
// CTA of the KV head, which first stages every split's partials in shared
// memory.
Q3_DEV void consume_attention(const DecodeArgs& p, int l, const Unit& u, const int* table, const Smem& sm,
                              uint32_t& it, int warp, int lane) {
    const int G = p.n_q / p.n_kv, ns = p.n_splits, tid = threadIdx.x;
    constexpr int BR = 2 * BLKS_PER_SLOT;                      // blocks per round (2 slots)
    const AttScratch A = att_scratch(G, ns);
    bf16* sqa = reinterpret_cast<bf16*>(sm.sx + A.sq);         // [16][KSTR]
    bf16* snew = reinterpret_cast<bf16*>(sm.sx + A.snew);      // [2][D]
    float* pm = sm.sx + A.pm;                                  // [BR][G]
    float* pl = sm.sx + A.pl;                                  // [BR][G]
    float* sml = sm.sx + A.sml;                                // [G][ns][2]
    float* sw = sm.sx + A.sw;                                  // [G][ns]
    float* po = sm.sx + A.po;                                  // [BR][G][D], then [G][ns][D]
    const int last_blk = u.nblk - 1;
    const bool mine = u.active && u.b0 <= last_blk && last_blk < u.b1;
    const float2* rope_row = p.rope + (size_t)u.pos * (D / 2);
    const void* const* lp = sm.wp + (size_t)l * WP_N;
    const bf16* q_gain = static_cast<const bf16*>(lp[WP_Q_NORM]);
    const bf16* k_gain = static_cast<const bf16*>(lp[WP_K_NORM]);
    const float qscale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    if (u.active) {
        if (warp < G) {
            const float4 v = __ldcg(reinterpret_cast<const float4*>(p.qkv + (u.kvh * G + warp) * D + lane * 4));
            float y[4] = {v.x, v.y, v.z, v.w};
            head_norm_rope(y, q_gain, rope_row, p.eps, lane);
            float hi[4], lo[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float q = y[e] * qscale;
                hi[e] = __bfloat162float(__float2bfloat16_rn(q));
                lo[e] = q - hi[e];
            }
            *reinterpret_cast<uint2*>(sqa + (2 * warp) * KSTR + lane * 4) =
                make_uint2(pack_bf16(hi[0], hi[1]), pack_bf16(hi[2], hi[3]));
            *reinterpret_cast<uint2*>(sqa + (2 * warp + 1) * KSTR + lane * 4) =
                make_uint2(pack_bf16(lo[0], lo[1]), pack_bf16(lo[2], lo[3]));
        } else if (mine && warp < G + 2) {
            const bool is_k = warp == G;
            const float4 v = __ldcg(reinterpret_cast<const float4*>(
                p.qkv + (p.n_q + (is_k ? 0 : p.n_kv) + u.kvh) * D + lane * 4));
            float y[4] = {v.x, v.y, v.z, v.w};
            if (is_k) head_norm_rope(y, k_gain, rope_row, p.eps, lane);
            const uint2 packed = make_uint2(pack_bf16(y[0], y[1]), pack_bf16(y[2], y[3]));
            *reinterpret_cast<uint2*>(snew + (is_k ? 0 : D) + lane * 4) = packed;
            const int phys = table[last_blk];
            if (phys >= 0 && phys < p.n_blocks) {
                bf16* dst = const_cast<bf16*>(kv_block(p, l, phys, u.kvh)) +
                            (is_k ? 0 : (size_t)p.n_kv * KVB * D) + (size_t)(u.pos % KVB) * D + lane * 4;
                *reinterpret_cast<uint2*>(dst) = packed;
            } else if (lane == 0) {
                set_status(p.status, Q3_STATUS_BLOCK_RANGE);
            }
        } else if (warp >= G + 2) {
            // rows of the 16-row q operand past the G heads are zero
            for (int i = (warp - G - 2) * 32 + lane; i < (16 - 2 * G) * (D / 8); i += (NCW - G - 2) * 32)
                *reinterpret_cast<uint4*>(sqa + (2 * G + i / (D / 8)) * KSTR + (i % (D / 8)) * 8) =
                    make_uint4(0u, 0u, 0u, 0u);
        }
    }
    consumer_sync();

    // warp w: block j = w / ATT_DQ of each round, dimension quarter dq = w % ATT_DQ
    const int j = warp / ATT_DQ, dq = warp % ATT_DQ;
    const bool worker = j < BR;
    AttWarp st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int dt = 0; dt < ATT_DT; ++dt) st.o[dt][0] = st.o[dt][1] = st.o[dt][2] = st.o[dt][3] = 0.f;
    const int new_r = u.pos % KVB;
    for (int b = u.b0, k = 0; b < u.b1; b += BLKS_PER_SLOT, ++k) {
        const int slot = it % sm.n_slots;
        const uint32_t use = it / sm.n_slots;
        ++it;
        if (!wait_bar(&sm.full[slot], use & 1, sm, p.status)) break;
        // slot k of the unit holds blocks b, b + 1: in a round of BR blocks it
        // is slot k % (BR / 2), served by block lanes j = 2 (k % (BR / 2)) + {0, 1}
        const int blk = b + (j % BLKS_PER_SLOT);
        if (worker && j / BLKS_PER_SLOT == k % (BR / BLKS_PER_SLOT) && blk < u.b1) {
            const int phys = table[blk];
            if (phys >= 0 && phys < p.n_blocks) {
                uint8_t* kt = sm.ring + (size_t)slot * SLOT + (j % BLKS_PER_SLOT) * BLK_BYTES;
                uint8_t* vt = kt + KT_BYTES;
                if (blk == last_blk) {
                    // this step's K/V row replaces the stale one in the tile
                    if (dq == 0) {
                        const int kv = lane >> 4, c = lane & 15;
                        *reinterpret_cast<uint4*>(const_cast<uint8_t*>(tile_chunk(kv ? vt : kt, new_r, c))) =
                            *reinterpret_cast<const uint4*>(snew + kv * D + c * 8);
                    }
                    named_bar(2 + j, ATT_DQ * 32);
                }
                attend_block_tc<ATT_DT>(kt, vt, sqa, min(KVB, u.ctx - blk * KVB), dq * ATT_DT, lane, st);
            } else if (lane == 0 && dq == 0) {
                set_status(p.status, Q3_STATUS_BLOCK_RANGE);
            }
        }
        __syncwarp();
        if (lane == 0) {
            mbar_arrive(&sm.redf[slot]);                     // keeps the slot's phases in step
            mbar_arrive(&sm.empty[slot]);
        }
    }
    // per-warp partials: rows g (head g / 2) and g + 8 (head 4 + g / 2); the
    // two parts of a head are summed across lanes g, g ^ 1
    if (worker && u.active) {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int dt = 0; dt < ATT_DT; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.o[dt][e] += __shfl_xor_sync(0xffffffffu, st.o[dt][e], 4);
        if ((g & 1) == 0) {
#pragma unroll
            for (int hr = 0; hr < 2; ++hr) {
                const int h = hr * 4 + g / 2;
                if (h < G) {
                    if (dq == 0 && tig == 0) { pm[j * G + h] = st.m[hr]; pl[j * G + h] = st.l[hr]; }
#pragma unroll
                    for (int dt = 0; dt < ATT_DT; ++dt)
                        *reinterpret_cast<float2*>(po + (j * G + h) * D + dq * (D / ATT_DQ) + dt * 8 + 2 * tig) =
                            make_float2(st.o[dt][2 * hr], st.o[dt][2 * hr + 1]);
                }
            }
        }
    }
    consumer_sync();

    // block lanes of each head, in order: this split's partial
    if (u.active) {
        for (int i = tid; i < G * D; i += NCT) {
            const int hg = i / D, d = i % D;
            float M = -INFINITY;
            for (int jj = 0; jj < BR; ++jj) M = fmaxf(M, pm[jj * G + hg]);
            float Lx = 0.f, O = 0.f;
            if (M != -INFINITY) {
                for (int jj = 0; jj < BR; ++jj) {
                    const float mj = pm[jj * G + hg];
                    const float e = mj == -INFINITY ? 0.f : exp2f(mj - M);
                    Lx = fmaf(pl[jj * G + hg], e, Lx);
                    O = fmaf(po[(jj * G + hg) * D + d], e, O);
                }
            }
            const int head = u.kvh * G + hg;
            if (ns == 1) {
                __stcg(p.att + head * D + d, O / Lx);
            } else {
                __stcg(p.part_o + ((size_t)head * ns + u.split) * D + d, O);
                if (d == 0) {
                    __stcg(p.part_ml + ((size_t)head * ns + u.split) * 2 + 0, M);
                    __stcg(p.part_ml + ((size_t)head * ns + u.split) * 2 + 1, Lx);
                }
            }
        }
    }
    if (ns == 1) return;
    // the last split CTA of this KV head merges every split in order: one
    // acquire-release ticket per CTA publishes its partials and, for the last,
    // makes every other split's visible
    consumer_sync();
    if (tid == 0) {
        int t = -1;
        if (u.active)
            asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(t) : "l"(p.counters + u.kvh) : "memory");
        *sm.ticket = t;
    }
    consumer_sync();
    if (*sm.ticket != ns - 1) return;
    // the G heads of this KV head hold contiguous partials: [G][ns][2] and
    // [G][ns][D] from head kvh * G; fetch them all at once
    {
        const float4* src = reinterpret_cast<const float4*>(p.part_o + (size_t)u.kvh * G * ns * D);
        float4* dst = reinterpret_cast<float4*>(po);
        const int n4 = G * ns * D / 4;
        for (int i = tid; i < n4; i += NCT) dst[i] = __ldcg(src + i);
        const float* ml = p.part_ml + (size_t)u.kvh * G * ns * 2;
        for (int i = tid; i < 2 * G * ns; i += NCT) sml[i] = __ldcg(ml + i);
    }
    consumer_sync();
    if (tid < G) {
        float M = -INFINITY;
        for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, sml[2 * (tid * ns + sp)]);
        float Lx = 0.f;
        for (int sp = 0; sp < ns; ++sp) {
            const float ms = sml[2 * (tid * ns + sp)];
            const float e = ms == -INFINITY ? 0.f : exp2f(ms - M);
            sw[tid * ns + sp] = e;
            Lx = fmaf(sml[2 * (tid * ns + sp) + 1], e, Lx);
        }
        pl[tid] = Lx;
    }
    consumer_sync();
    for (int i = tid; i < G * D; i += NCT) {
        const int hg = i / D, d = i % D;
        const float* pg = po + (size_t)hg * ns * D + d;
        float O = 0.f;
        for (int sp = 0; sp < ns; ++sp) O = fmaf(pg[(size_t)sp * D], sw[hg * ns + sp], O);
        __stcg(p.att + (u.kvh * G + hg) * D + d, O / pl[hg]);
    }
    if (tid == 0) p.counters[u.kvh] = 0;
}

Q3_DEV int checked_token(const DecodeArgs& p) {
    const int tok = p.token[0];
    return (tok < 0 || tok >= p.V) ? 0 : tok;
}

template <bool Q8>
Q3_DEV void consumer(const DecodeArgs& p, const Unit& u, const int* table, const Smem& sm, int warp,
                     int lane) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && (p.token[0] < 0 || p.token[0] >= p.V))
        set_status(p.status, Q3_STATUS_TOKEN_RANGE);
    const bf16* erow = p.embed + (size_t)checked_token(p) * p.H;
    uint32_t it = 0;
    unsigned long long target = p.bar_base;
    const int qw = p.n_q * D;
    for (int l = 0; l < p.n_layers; ++l) {
        const void* const* lp = sm.wp + (size_t)l * WP_N;
        stage_x(sm, p.x, l == 0 ? erow : nullptr, p.H, static_cast<const bf16*>(lp[WP_ATTN_NORM]), p.eps);
        consume_weights<Q8>(weight_stage(p, sm, l, ST_QKV), sm, it, warp, lane, p);
        if (!grid_sync(p, sm, target += gridDim.x, true)) return;
        consume_attention(p, l, u, table, sm, it, warp, lane);
        if (!grid_sync(p, sm, target += gridDim.x, false)) return;
        stage_x(sm, p.att, nullptr, qw, nullptr, p.eps);
        consume_weights<Q8>(weight_stage(p, sm, l, ST_O), sm, it, warp, lane, p);
        if (!grid_sync(p, sm, target += gridDim.x, true)) return;
        stage_x(sm, p.x, nullptr, p.H, static_cast<const bf16*>(lp[WP_FFN_NORM]), p.eps);
        consume_weights<Q8>(weight_stage(p, sm, l, ST_GU), sm, it, warp, lane, p);
        if (!grid_sync(p, sm, target += gridDim.x, true)) return;
        stage_x(sm, p.ffn, nullptr, p.F, nullptr, p.eps);
        consume_weights<Q8>(weight_stage(p, sm, l, ST_DOWN), sm, it, warp, lane, p);
        if (!grid_sync(p, sm, target += gridDim.x, true)) return;
    }
    stage_x(sm, p.x, nullptr, p.H, p.final_norm, p.eps);
    consume_weights<false>(weight_stage(p, sm, 0, ST_LM), sm, it, warp, lane, p);
}

// The epilogue warp: for every matvec tile, once the consumer warps' segment
// sums are in, the rows' sums and outputs; then it releases the slot.  It
// owns this CTA's residual rows (written first with the embedding row) and
// the lm_head argmax: its partial per CTA, merged by the last CTA.
Q3_DEV bool epilogue_stage(const DecodeArgs& p, const WStage& s, int kind, const Smem& sm, uint32_t& it,
                           int lane, float* out, float& best, int& best_i) {
    const int S = NCW / (s.q8 ? s.nr / (s.nr < 4 ? s.nr : 4) : s.nr);
    for (int a = s.r0; a < s.r1; a += s.per) {
        const int nvalid = min(s.per, s.r1 - a);
        const int slot = it % sm.n_slots;
        const uint32_t use = it / sm.n_slots;
        ++it;
        if (!wait_bar(&sm.redf[slot], use & 1, sm, p.status)) return false;
        tile_epilogue(s, kind, sm.red + slot * RED, S, a, nvalid, lane, out, sm.xres, best, best_i);
        __syncwarp();
        if (lane == 0) mbar_arrive(&sm.empty[slot]);
    }
    return true;
}

Q3_DEV void epilogue(const DecodeArgs& p, const Unit& u, const Smem& sm, int lane) {
    const bf16* erow = p.embed + (size_t)checked_token(p) * p.H;
    {
        const WStage so = weight_stage(p, sm, 0, ST_O);
        for (int r = so.r0 + lane; r < so.r1; r += 32) {
            const float x = __bfloat162float(erow[r]);
            sm.xres[r - so.r0] = x;
            __stcg(p.x + r, x);
        }
    }
    uint32_t it = 0;
    float best = -INFINITY;
    int best_i = 0x7fffffff;
    bool ok = true;
    // a matvec stage's outputs are written: this CTA's grid-barrier arrival
    auto closed = [&]() {
        __syncwarp();
        if (lane == 0) asm volatile("red.release.gpu.global.add.u64 [%0], 1;" :: "l"(p.bar) : "memory");
    };
    for (int l = 0; l < p.n_layers && ok; ++l) {
        ok = epilogue_stage(p, weight_stage(p, sm, l, ST_QKV), ST_QKV, sm, it, lane, p.qkv, best, best_i);
        if (!ok) break;
        closed();
        // attention slots: nothing to finish, only the slot release
        for (int b = u.b0; b < u.b1 && ok; b += BLKS_PER_SLOT) {
            const int slot = it % sm.n_slots;
            const uint32_t use = it / sm.n_slots;
            ++it;
            ok = wait_bar(&sm.full[slot], use & 1, sm, p.status);
            __syncwarp();
            if (ok && lane == 0) mbar_arrive(&sm.empty[slot]);
        }
        ok = ok && epilogue_stage(p, weight_stage(p, sm, l, ST_O), ST_O, sm, it, lane, p.x, best, best_i);
        if (!ok) break;
        closed();
        ok = epilogue_stage(p, weight_stage(p, sm, l, ST_GU), ST_GU, sm, it, lane, p.ffn, best, best_i);
        if (!ok) break;
        closed();
        ok = epilogue_stage(p, weight_stage(p, sm, l, ST_DOWN), ST_DOWN, sm, it, lane, p.x, best, best_i);
        if (!ok) break;
        closed();
    }
    if (!ok) return;
    if (!epilogue_stage(p, weight_stage(p, sm, 0, ST_LM), ST_LM, sm, it, lane, p.logits, best, best_i)) return;
    if (!p.argmax_out) return;

    // this CTA's argmax partial, then the last CTA to finish merges them all
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (better(ov, oi, best, best_i)) { best = ov; best_i = oi; }
    }
    int ticket = 0;
    if (lane == 0) {
        p.am_val[blockIdx.x] = best;
        p.am_idx[blockIdx.x] = best_i;
        __threadfence();
        ticket = atomicAdd(p.am_counter, 1);
    }
    ticket = __shfl_sync(0xffffffffu, ticket, 0);
    if (ticket != (int)gridDim.x - 1) return;
    __threadfence();
    best = -INFINITY;
    best_i = 0x7fffffff;
    for (int b = lane; b < (int)gridDim.x; b += 32) {
        const float bv = __ldcg(p.am_val + b);
        const int bi = __ldcg(p.am_idx + b);
        if (better(bv, bi, best, best_i)) { best = bv; best_i = bi; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
        if (better(ov, oi, best, best_i)) { best = ov; best_i = oi; }
    }
    if (lane == 0) {
        *p.argmax_out = best_i == 0x7fffffff ? 0 : best_i;
        *p.am_counter = 0;
    }
}

template <bool Q8>
__global__ void __launch_bounds__(THREADS, 1) decode_step_kernel(const DecodeArgs p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const Layout lay = make_layout(p.n_slots, sx_floats(p.H, p.F, p.n_q, p.n_kv, p.n_splits), p.n_layers);
    Smem sm;
    sm.n_slots = p.n_slots;
    sm.ring = smem;
    sm.sx = reinterpret_cast<float*>(smem + lay.sx);
    sm.red = reinterpret_cast<float*>(smem + lay.red);
    sm.full = reinterpret_cast<uint64_t*>(smem + lay.bars);
    sm.empty = sm.full + p.n_slots;
    sm.redf = sm.empty + p.n_slots;
    sm.ss = reinterpret_cast<float*>(smem + lay.misc);
    sm.bv = sm.ss + NCW;
    sm.bi = reinterpret_cast<int*>(sm.bv + NCW);
    sm.abort = reinterpret_cast<volatile int*>(sm.bi + NCW);
    sm.ticket = const_cast<int*>(sm.abort) + 1;
    sm.xres = reinterpret_cast<float*>(sm.ticket + 3);
    sm.wp = reinterpret_cast<const void**>(smem + lay.ptrs);
    // the per-layer weight and gain pointers, read on every stage by producer, consumers and epilogue
    for (int i = threadIdx.x; i < p.n_layers * WP_N; i += blockDim.x) {
        const DecodeLayer& L = p.layers[i / WP_N];
        const int k = i % WP_N;
        const void* v = k < 7 ? L.w[k] : k < 14 ? static_cast<const void*>(L.sc[k - 7])
                      : k == WP_ATTN_NORM ? static_cast<const void*>(L.attn_norm)
                      : k == WP_Q_NORM ? static_cast<const void*>(L.q_norm)
                      : k == WP_K_NORM ? static_cast<const void*>(L.k_norm)
                      : static_cast<const void*>(L.ffn_norm);
        sm.wp[i] = v;
    }

    if (threadIdx.x == 0) {
        for (int s = 0; s < p.n_slots; ++s) {
            mbar_init(&sm.full[s], 1);
            mbar_init(&sm.empty[s], NCW + 1);
            mbar_init(&sm.redf[s], NCW);
        }
        *sm.abort = 0;
        fence_barrier_init();
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const Unit u = attention_unit(p);
    const int* table = p.tables + (size_t)p.row_slot[0] * p.max_blocks;
    if (warp == PRODUCER) producer<Q8>(p, u, table, sm, lane);
    else if (warp == EPILOGUE) epilogue(p, u, sm, lane);
    else consumer<Q8>(p, u, table, sm, warp, lane);
}

}  // namespace

int decode_step_slot_bytes() { return SLOT; }

int decode_step_barriers(int n_layers) { return 5 * n_layers; }

size_t decode_step_smem(int H, int F, int n_q, int n_kv, int q8, int n_slots, int n_splits, int grid,
                        int n_layers)
{
    if (n_kv < 1 || n_q % n_kv || n_q / n_kv > NCW / BLKS_PER_SLOT) return 0;
    if (grid < 1 || (H + grid - 1) / grid > MAX_OWN) return 0;
    if (n_slots < MIN_SLOTS || n_slots > MAX_SLOTS || n_splits < 1) return 0;
    const int qw = n_q * D;
    const int align = q8 ? 256 : 8;
    if (H % align || qw % align || F % align || H % 8) return 0;
    if (H > 4 * NCT * GAIN_IT) return 0;                         // the normalised row's gain in registers
    // one row of every matvec (and a gate/up pair of rows) must fit a slot
    if (tile_rows(H, q8) < 2 || row_bytes(H, false) > SLOT || row_bytes(qw, q8) > SLOT ||
        row_bytes(F, q8) > SLOT)
        return 0;
    // bf16 tiles: a warp's segment of a row must fit its lanes' activation registers
    for (int K : {H, qw, F}) {
        if (q8 && K != H) continue;
        const int S = NCW / tile_rows(K, false);
        if ((K / 8 + S - 1) / S > 32 * XCPL) return 0;
    }
    return make_layout(n_slots, sx_floats(H, F, n_q, n_kv, n_splits), n_layers).total;
}

cudaError_t decode_step_prepare(size_t smem)
{
    cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(decode_step_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem);
    if (e != cudaSuccess) return e;
    int n0 = 0, n1 = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n0, decode_step_kernel<false>, THREADS, smem);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n1, decode_step_kernel<true>, THREADS, smem);
    if (e != cudaSuccess) return e;
    return (n0 >= 1 && n1 >= 1) ? cudaSuccess : cudaErrorInvalidConfiguration;
}

cudaError_t launch_decode_step(const Launch& L, const DecodeArgs& a, int grid, size_t smem)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return a.q8 ? cudaLaunchKernelEx(&cfg, decode_step_kernel<true>, a)
                : cudaLaunchKernelEx(&cfg, decode_step_kernel<false>, a);
}

}  // namespace q3
