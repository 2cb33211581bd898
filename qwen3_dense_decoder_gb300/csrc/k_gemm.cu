// k_gemm.cu -- tcgen05/TMEM tensor-core GEMM fed by TMA (sm_103a).
//
// Computes the token-round projections of the decoder ("Kipp Model Support",
// section "Quantization (Q8_0)": the seven per-layer projection tensors;
// "Kipp Roadmap", status v0.0.6: BF16 layer projections of prefill on the
// tensor units, with activations kept wider than BF16) as D = W * X^T with
// FP32 accumulation: the weight matrix W [out][in] is the MMA's A operand
// (128 output features per tile, TMEM lanes) and the round's token rows X
// [tokens][in] are the B operand (BN tokens per tile, TMEM columns).  Both
// operands are K-major fp16 tiles of 64 elements (one 128-byte swizzle row)
// staged by TMA into a STAGES-deep ring: kind::f16 wants A and B of one
// type, and fp16 activations carry 3 more mantissa bits than bf16 ones, so
// the weights enter as an fp16 copy of the bf16 tensors (exact except for
// |w| < 2^-17).
//
// Persistent and warp-specialised: one CTA per SM walks its share of the
// (token tile, weight tile, K split) units.  Warp 0 lane 0 issues TMA loads
// into a STAGES-deep ring, warp 1 lane 0 issues tcgen05.mma into one of two
// TMEM accumulators and owns the TMEM allocation, and warps 2..5 drain the
// other accumulator (warp w reads TMEM lanes 32 (w % 4)..+31) through the
// fused epilogue: plain store, residual add, or SwiGLU of a paired gate/up
// tile.  The epilogue of one unit therefore overlaps the main loop of the
// next.  Consecutive units of a CTA share the weight tile, which is read
// from HBM once and then hit in L2.  Split-K writes FP32 partials that
// gemm_splitk_reduce sums in split order.
//
// A second instantiation (gemm_tc_kernel<BN, true>) carries the QKV head
// epilogue of prefill rounds: each 128-row tile is one head, which it
// RMS-normalises and rotates (q and k heads) and writes as fp16 q rows or as
// BF16 K/V rows of the paged pool ("Kipp Model Support", section "The
// registry": RMS epsilon and RoPE theta; section "qwen3-0.6b-base": K/V
// rounded to BF16 on store; "Kipp Roadmap", status v0.0.2: 32-position
// block tables).  The layer math the pages do not print follows the standard
// dense Qwen3 decoder: q/k norm over each 128-wide head with gains shared by
// the heads, then RoPE in rotate-half pairs (i, i + 64).  It is a separate
// kernel so that the generic epilogues keep their register allocation.
#include <cuda.h>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int A_BYTES = BM * BK * 2;

template <int BN>
struct GemmCfg {
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    // as many stages as fit beside the SwiGLU exchange buffer, at most 8
    static constexpr int STAGES_RAW = (192 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr uint32_t ACC_COLS = BN < 32 ? 32 : BN;     // one accumulator
    // two accumulators, allocated as a power of two of at least 32 columns
    static constexpr uint32_t TMEM_COLS = 2 * ACC_COLS <= 64 ? 64 : 2 * ACC_COLS <= 128 ? 128
                                        : 2 * ACC_COLS <= 256 ? 256 : 512;
    static constexpr int XCH_BYTES = 32 * 128 * 4;                // SwiGLU exchange, 32 columns
    static constexpr int SMEM = STAGES * STAGE_BYTES + XCH_BYTES + 1024 /*align*/ + 512 /*barriers*/;
};

constexpr int GEMM_THREADS = 192;     // producer, MMA issuer, 4 epilogue warps
constexpr int BAR_EPI = 1;            // named barrier of the epilogue warps

Q3_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

// EPI_QKV_ROPE epilogue.  A tile is one head (m-tile hh, q heads, then k
// heads, then v heads) of BN tokens; each 32-token chunk goes through the
// exchange buffer.  Epilogue warp ew takes tokens ew, ew + 4, ... of a chunk
// (8, two at a time: half-warp h the token ew + 4 (2 i + h)), and lane g of a
// half-warp holds features [4 g, 4 g + 4) and their rotate-half partners
// [64 + 4 g, + 4): the RMSNorm reduces over 16 lanes and RoPE needs no
// exchange.  The GEMM streams its operands through L2, where a load waits
// microseconds: before the accumulator wait, lane l looks up the position
// (K/V heads: also the pool block) of the warp's tokens l and l + 32 of the
// tile, and each chunk's (cos, sin) rows are requested two chunks ahead.
struct QkvRows {
    int pos_a, pos_b, blk_a, blk_b;
    uint2 g_lo, g_hi;                           // the lane's gain values (q/k heads)
};

Q3_DEV QkvRows qkv_rope_rows(const RopeArgs& a, int hh, int tile_n0, int lim, int ew, int lane) {
    QkvRows r{0, 0, 0, 0, make_uint2(0u, 0u), make_uint2(0u, 0u)};
    const bool is_q = hh < a.n_q, is_k = !is_q && hh < a.n_q + a.n_kv;
    if (is_q || is_k) {
        const __nv_bfloat16* gain = is_q ? a.q_gain : a.k_gain;
        r.g_lo = *reinterpret_cast<const uint2*>(gain + (lane & 15) * 4);
        r.g_hi = *reinterpret_cast<const uint2*>(gain + 64 + (lane & 15) * 4);
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int idx = lane + 32 * h;                      // chunk idx / 8, token ew + 4 (idx % 8)
        const int t = tile_n0 + (idx >> 3) * 32 + ew + 4 * (idx & 7);
        int pos = 0, blk = 0;
        if (t < lim) {
            pos = a.row_pos[t];
            if (!is_q) blk = a.tables[(size_t)a.row_slot[t] * a.max_blocks + pos / 32];
        }
        (h ? r.pos_b : r.pos_a) = pos;
        (h ? r.blk_b : r.blk_a) = blk;
    }
    return r;
}

// the position or pool block of token k (0..7) of chunk c of the warp (k may differ by lane)
Q3_DEV int qkv_row_pos(const QkvRows& r, int c, int k) {
    return __shfl_sync(0xffffffffu, c < 4 ? r.pos_a : r.pos_b, (c & 3) * 8 + k);
}
Q3_DEV int qkv_row_blk(const QkvRows& r, int c, int k) {
    return __shfl_sync(0xffffffffu, c < 4 ? r.blk_a : r.blk_b, (c & 3) * 8 + k);
}

// The (cos, sin) pairs of frequencies [4 g, 4 g + 4) for the lane's 4 tokens
// of chunk c (cs[2 i], cs[2 i + 1]: token 2 i + h); a half-warp reads a
// 512-byte table row whole.  Tokens past the tile's end have position 0: a
// valid row, unused.
Q3_DEV void qkv_cs_load(const RopeArgs& a, const QkvRows& r, int c, int lane, float4 (&cs)[8]) {
    const int h = lane >> 4, g = lane & 15;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float4* row = reinterpret_cast<const float4*>(a.rope + (size_t)qkv_row_pos(r, c, 2 * i + h) * 64);
        cs[2 * i] = row[2 * g];
        cs[2 * i + 1] = row[2 * g + 1];
    }
}

Q3_DEV uint2 pack_f16x4(const float (&v)[4], bool& bad) {
    __half2 lo, hi;
    lo.x = to_f16(v[0], bad); lo.y = to_f16(v[1], bad);
    hi.x = to_f16(v[2], bad); hi.y = to_f16(v[3], bad);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}
Q3_DEV uint2 pack_bf16x4(const float (&v)[4]) {
    const __nv_bfloat162 lo = __floats2bfloat162_rn(v[0], v[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(v[2], v[3]);
    return make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
}

// Chunk c (tokens n0 ..) of head hh, staged in xch [token][128 features].
// All tokens are computed (columns past the tile's end hold zeros) and only
// the stores are predicated, so the 4 iterations' reductions interleave.
Q3_DEV void qkv_rope_chunk(const RopeArgs& a, int hh, int c, int n0, int lim, const float* xch, int ew, int lane,
                           const QkvRows& r, const float4 (&cs)[8], bool& bad) {
    const bool is_q = hh < a.n_q, is_k = !is_q && hh < a.n_q + a.n_kv;
    const int h = lane >> 4, g = lane & 15;
    float x1[4][4], x2[4][4];                   // features [4 g, + 4) and [64 + 4 g, + 4) of token 2 i + h
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float* src = xch + (ew + 4 * (2 * i + h)) * 128 + 4 * g;
        const float4 u = *reinterpret_cast<const float4*>(src);
        const float4 v = *reinterpret_cast<const float4*>(src + 64);
        x1[i][0] = u.x; x1[i][1] = u.y; x1[i][2] = u.z; x1[i][3] = u.w;
        x2[i][0] = v.x; x2[i][1] = v.y; x2[i][2] = v.z; x2[i][3] = v.w;
    }
    if (is_q || is_k) {
        const float g1[4] = {bf16lo(r.g_lo.x), bf16hi(r.g_lo.x), bf16lo(r.g_lo.y), bf16hi(r.g_lo.y)};
        const float g2[4] = {bf16lo(r.g_hi.x), bf16hi(r.g_hi.x), bf16lo(r.g_hi.y), bf16hi(r.g_hi.y)};
        float ss[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            ss[i] = 0.f;
#pragma unroll
            for (int e = 0; e < 4; ++e) ss[i] += x1[i][e] * x1[i][e] + x2[i][e] * x2[i][e];
        }
#pragma unroll
        for (int o = 8; o > 0; o >>= 1)
#pragma unroll
            for (int i = 0; i < 4; ++i) ss[i] += __shfl_xor_sync(0xffffffffu, ss[i], o);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float rr = 1.0f / sqrtf(ss[i] / 128.0f + a.eps);
            const float cv[4][2] = {{cs[2 * i].x, cs[2 * i].y}, {cs[2 * i].z, cs[2 * i].w},
                                    {cs[2 * i + 1].x, cs[2 * i + 1].y}, {cs[2 * i + 1].z, cs[2 * i + 1].w}};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float y1 = x1[i][e] * rr * g1[e], y2 = x2[i][e] * rr * g2[e];
                x1[i][e] = y1 * cv[e][0] - y2 * cv[e][1];     // first half: x1 cos - x2 sin
                x2[i][e] = y2 * cv[e][0] + y1 * cv[e][1];     // second half: x2 cos + x1 sin
            }
        }
    }
    const int kvh = is_k ? hh - a.n_q : hh - a.n_q - a.n_kv;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int k = 2 * i + h, t = n0 + ew + 4 * k;
        if (is_q) {
            if (t < lim) {
                __half* dst = a.q_out16 + ((size_t)t * a.n_q + hh) * 128 + 4 * g;
                *reinterpret_cast<uint2*>(dst) = pack_f16x4(x1[i], bad);
                *reinterpret_cast<uint2*>(dst + 64) = pack_f16x4(x2[i], bad);
            }
            continue;
        }
        const int pos = qkv_row_pos(r, c, k), blk = qkv_row_blk(r, c, k);
        if (t >= lim) continue;
        if (blk < 0 || blk >= a.n_blocks) {
            if (g == 0) set_status(a.status, Q3_STATUS_BLOCK_RANGE);
            continue;
        }
        __nv_bfloat16* dst = a.kv_layer + (((size_t)blk * 2 + (is_k ? 0 : 1)) * a.n_kv + kvh) * (32 * 128) +
                             (size_t)(pos % 32) * 128 + 4 * g;
        *reinterpret_cast<uint2*>(dst) = pack_bf16x4(x1[i]);
        *reinterpret_cast<uint2*>(dst + 64) = pack_bf16x4(x2[i]);
    }
}
Q3_DEV void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}
Q3_DEV float silu_fast(float g) { return __fdividef(g, 1.0f + __expf(-g)); }

struct Unit {
    int nt, mt, split, kb0, kb1;
};

Q3_DEV Unit decode_unit(const GemmArgs& p, int u, int n_tiles)
{
    Unit w;
    const int m_tiles = p.M / BM;
    w.nt = u % n_tiles;
    const int rest = u / n_tiles;
    w.mt = rest % m_tiles;
    w.split = rest / m_tiles;
    const int kb_total = p.K / BK;
    w.kb0 = w.split * kb_total / p.k_splits;
    w.kb1 = (w.split + 1) * kb_total / p.k_splits;
    return w;
}

template <int BN, bool QKV>
__global__ void __launch_bounds__(GEMM_THREADS, 1)
gemm_tc_kernel(const __grid_constant__ CUtensorMap ta0, const __grid_constant__ CUtensorMap ta1,
               const __grid_constant__ CUtensorMap ta2, const __grid_constant__ CUtensorMap tb,
               const GemmArgs p)
{
    using C = GemmCfg<BN>;
    constexpr int STAGES = C::STAGES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~uintptr_t(1023));
    uint8_t* sa = smem;
    uint8_t* sb = smem + STAGES * A_BYTES;
    float* xch = reinterpret_cast<float*>(sb + STAGES * C::B_BYTES);
    uint64_t* full = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(xch) + C::XCH_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;       // accumulator ready, one per TMEM buffer
    uint64_t* tempty = tfull + 2;           // accumulator drained
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BN - 1) / BN;
    const int units = n_tiles * (p.M / BM) * p.k_splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 4);       // one arrival per epilogue warp
        }
        fence_barrier_init();
        prefetch_tmap(&ta0);
        prefetch_tmap(&tb);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    // the weight tile (A) of stage s for k-block kb of unit w
    auto load_a = [&](int s, const Unit& w, int kb) {
        const int kc = kb * BK;
        uint8_t* a_dst = sa + s * A_BYTES;
        if (p.pair) {
            tma_load_2d(a_dst, &ta0, &full[s], kc, w.mt * 64);
            tma_load_2d(a_dst + A_BYTES / 2, &ta1, &full[s], kc, w.mt * 64);
        } else if (w.mt < p.a_tiles0) {
            tma_load_2d(a_dst, &ta0, &full[s], kc, w.mt * BM);
        } else if (w.mt < p.a_tiles1) {
            tma_load_2d(a_dst, &ta1, &full[s], kc, (w.mt - p.a_tiles0) * BM);
        } else {
            tma_load_2d(a_dst, &ta2, &full[s], kc, (w.mt - p.a_tiles1) * BM);
        }
    };
    // Weights do not depend on the previous kernel: with early_a the first
    // ring stages' weight tiles are requested before the dependency wait
    // (their stage barriers expect the token tiles' bytes too, requested
    // after it).
    int pre = 0;
    if (p.early_a && warp == 0 && lane == 0) {
        for (int u = blockIdx.x; u < units && pre < STAGES; u += gridDim.x) {
            const Unit w = decode_unit(p, u, n_tiles);
            for (int kb = w.kb0; kb < w.kb1 && pre < STAGES; ++kb, ++pre) {
                mbar_arrive_expect_tx(&full[pre], C::STAGE_BYTES);
                load_a(pre, w, kb);
            }
        }
    }

    // the token rows (B) are written by the previous kernel
    grid_dep_wait();

    if (warp == 0) {
        // ---------------- TMA producer
        if (lane == 0) {
            int it = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x) {
                const Unit w = decode_unit(p, u, n_tiles);
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t use = it / STAGES;
                    if (it < pre) {                        // weights already requested
                        tma_load_2d(sb + s * C::B_BYTES, &tb, &full[s], kb * BK, w.nt * BN);
                        continue;
                    }
                    if (it >= STAGES && !mbar_wait(&empty[s], (use & 1) ^ 1, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
                    const int kc = kb * BK;
                    uint8_t* a_dst = sa + s * A_BYTES;
                    if (p.pair) {
                        tma_load_2d(a_dst, &ta0, &full[s], kc, w.mt * 64);
                        tma_load_2d(a_dst + A_BYTES / 2, &ta1, &full[s], kc, w.mt * 64);
                    } else if (w.mt < p.a_tiles0) {
                        tma_load_2d(a_dst, &ta0, &full[s], kc, w.mt * BM);
                    } else if (w.mt < p.a_tiles1) {
                        tma_load_2d(a_dst, &ta1, &full[s], kc, (w.mt - p.a_tiles0) * BM);
                    } else {
                        tma_load_2d(a_dst, &ta2, &full[s], kc, (w.mt - p.a_tiles1) * BM);
                    }
                    tma_load_2d(sb + s * C::B_BYTES, &tb, &full[s], kc, w.nt * BN);
                }
            }
        }
    } else if (warp == 1) {
        // ---------------- MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
            int it = 0, local = 0;
            bool ok = true;
            for (int u = blockIdx.x; u < units && ok; u += gridDim.x, ++local) {
                const Unit w = decode_unit(p, u, n_tiles);
                const int ab = local & 1;
                const uint32_t use_ab = local >> 1;
                if (local >= 2 && !mbar_wait(&tempty[ab], (use_ab - 1) & 1, p.status)) break;
                tc_fence_after();
                const uint32_t d = tmem + ab * C::ACC_COLS;
                for (int kb = w.kb0; kb < w.kb1; ++kb, ++it) {
                    const int s = it % STAGES;
                    const uint32_t use = it / STAGES;
                    if (!mbar_wait(&full[s], use & 1, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sa + s * A_BYTES);
                    const uint32_t b_base = smem_u32(sb + s * C::B_BYTES);
#pragma unroll
                    for (int k = 0; k < BK / 16; ++k) {
                        // advancing 16 elements (32 bytes) along K inside the swizzle row
                        tc_mma_f16(d, smem_desc_sw128(a_base + k * 32), smem_desc_sw128(b_base + k * 32),
                                   idesc, (kb > w.kb0 || k > 0) ? 1u : 0u);
                    }
                    tc_commit(&empty[s]);
                }
                tc_commit(&tfull[ab]);
            }
        }
    } else if constexpr (QKV) {
        // ---------------- epilogue (EPI_QKV_ROPE): warps 2..5
        constexpr int NCH = (BN + 31) / 32;
        const RopeArgs& a = p.rope;
        const int q = warp & 3, row = q * 32 + lane, ew = warp - 2;
        bool range_bad = false;
        int local = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
            const Unit w = decode_unit(p, u, n_tiles);
            const int ab = local & 1;
            const uint32_t use_ab = local >> 1;
            const int lim = min(p.N, w.nt * BN + BN);       // this tile's last column + 1
            const bool qk = w.mt < a.n_q + a.n_kv;
            const QkvRows rows = qkv_rope_rows(a, w.mt, w.nt * BN, lim, ew, lane);
            // chunks c, c + 1 and c + 2 in flight; the loop stays rolled (an
            // unrolled tile overflows the instruction cache)
            float4 cs0[8], cs1[8], cs2[8];
            if (qk) {
                qkv_cs_load(a, rows, 0, lane, cs0);
                if (NCH > 1) qkv_cs_load(a, rows, 1, lane, cs1);
            }
            if (!named_bar_and(BAR_EPI, 128, mbar_wait(&tfull[ab], use_ab & 1, p.status))) break;
            tc_fence_after();
            const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + ab * C::ACC_COLS;
#pragma unroll 1
            for (int c = 0; c < NCH; ++c) {
                if (qk && c + 2 < NCH) qkv_cs_load(a, rows, c + 2, lane, cs2);
                uint32_t r[32];
                if (BN - c * 32 >= 32) {
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                } else {
                    tmem_ld_32x32b_x16(t_row + c * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
#pragma unroll
                    for (int j = 16; j < 32; ++j) r[j] = 0u;
                }
                tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) xch[j * 128 + row] = __uint_as_float(r[j]);
                named_bar(BAR_EPI, 128);
                qkv_rope_chunk(a, w.mt, c, w.nt * BN + c * 32, lim, xch, ew, lane, rows, cs0, range_bad);
                named_bar(BAR_EPI, 128);
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    cs0[k] = cs1[k];
                    cs1[k] = cs2[k];
                }
            }
            // this accumulator may be overwritten by the unit after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
        }
        if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
    } else {
        // ---------------- epilogue: TMEM -> registers -> global, warps 2..5
        const int q = warp & 3;                         // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;                  // D row = TMEM lane
        const bool swiglu = (p.epi == EPI_SWIGLU_F16 || p.epi == EPI_SWIGLU_F32) && p.k_splits == 1;
        bool range_bad = false;
        int local = 0;
        for (int u = blockIdx.x; u < units; u += gridDim.x, ++local) {
            const Unit w = decode_unit(p, u, n_tiles);
            const int ab = local & 1;
            const uint32_t use_ab = local >> 1;
            if (!named_bar_and(BAR_EPI, 128, mbar_wait(&tfull[ab], use_ab & 1, p.status))) break;
            tc_fence_after();
            const uint32_t t_row = tmem + ((uint32_t)(q * 32) << 16) + ab * C::ACC_COLS;
            // 32 columns at a time; a tile width of 16 mod 32 ends with 16
#pragma unroll 1
            for (int c = 0; c < (BN + 31) / 32; ++c) {
                uint32_t r[32];
                if (BN - c * 32 >= 32) {
                    tmem_ld_32x32b_x32(t_row + c * 32, r);
                } else {
                    tmem_ld_32x32b_x16(t_row + c * 32, *reinterpret_cast<uint32_t(*)[16]>(r));
#pragma unroll
                    for (int j = 16; j < 32; ++j) r[j] = 0u;
                }
                tmem_ld_wait();
                const int n0 = w.nt * BN + c * 32;
                const int lim = min(p.N, w.nt * BN + BN);   // this tile's last column + 1
                if (p.k_splits > 1) {
                    float* ws = p.ws + (size_t)w.split * p.N * p.M;
                    const int m = w.mt * BM + row;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n0 + j < lim) ws[(size_t)(n0 + j) * p.M + m] = __uint_as_float(r[j]);
                } else if (swiglu) {
                    // rows 0..63 hold the gate and rows 64..127 the up projection of
                    // the same 64 features: every thread posts its 32 columns, then
                    // computes 16 columns of one feature (all four warps share the work)
#pragma unroll
                    for (int j = 0; j < 32; ++j) xch[j * 128 + row] = __uint_as_float(r[j]);
                    named_bar(BAR_EPI, 128);
                    const int fr = row & 63;                    // feature row
                    const int jh = (row >> 6) * 16;             // column half
                    const int f = w.mt * 64 + fr;
#pragma unroll
                    for (int jj = 0; jj < 16; ++jj) {
                        const int j = jh + jj;
                        if (n0 + j < lim) {
                            const float v = silu_fast(xch[j * 128 + fr]) * xch[j * 128 + 64 + fr];
                            if (p.epi == EPI_SWIGLU_F16)
                                reinterpret_cast<__half*>(p.out)[(size_t)(n0 + j) * p.ldo + f] =
                                    to_f16(v, range_bad);
                            else
                                reinterpret_cast<float*>(p.out)[(size_t)(n0 + j) * p.ldo + f] = v;
                        }
                    }
                    named_bar(BAR_EPI, 128);
                } else if (p.epi == EPI_ADD_F32) {
                    // residual add: all 32 loads are issued before any store
                    const int m = w.mt * BM + row;
                    float* out = reinterpret_cast<float*>(p.out);
                    float old[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        old[j] = n0 + j < lim ? out[(size_t)(n0 + j) * p.ldo + m] : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j)
                        if (n0 + j < lim) out[(size_t)(n0 + j) * p.ldo + m] = old[j] + __uint_as_float(r[j]);
                } else {
                    const int m = w.mt * BM + row;
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        if (n0 + j < lim) {
                            const size_t o = (size_t)(n0 + j) * p.ldo + m;
                            const float v = __uint_as_float(r[j]);
                            if (p.epi == EPI_STORE_F32)
                                reinterpret_cast<float*>(p.out)[o] = v;
                            else
                                reinterpret_cast<__half*>(p.out)[o] = to_f16(v, range_bad);
                        }
                    }
                }
            }
            // this accumulator may be overwritten by the unit after next
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[ab]);
        }
        if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
    }

    // the next kernel may start its prologue while this grid drains
    grid_dep_launch();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, C::TMEM_COLS);
    }
}

// Sum the split-K partials in split order and apply the epilogue.
__global__ void gemm_splitk_reduce_kernel(const GemmArgs p)
{
    grid_dep_wait();
    const int m_out = p.pair ? p.M / 2 : p.M;
    const size_t total = (size_t)p.N * m_out;
    const size_t slab = (size_t)p.N * p.M;
    bool range_bad = false;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int n = (int)(i / m_out), f = (int)(i % m_out);
        if (p.pair) {
            const int m_g = (f / 64) * BM + (f % 64), m_u = m_g + 64;
            float g = 0.f, u = 0.f;
            for (int s = 0; s < p.k_splits; ++s) {
                g += p.ws[s * slab + (size_t)n * p.M + m_g];
                u += p.ws[s * slab + (size_t)n * p.M + m_u];
            }
            const float v = silu(g) * u;
            if (p.epi == EPI_SWIGLU_F16)
                reinterpret_cast<__half*>(p.out)[(size_t)n * p.ldo + f] = to_f16(v, range_bad);
            else
                reinterpret_cast<float*>(p.out)[(size_t)n * p.ldo + f] = v;
        } else {
            float acc = 0.f;
            for (int s = 0; s < p.k_splits; ++s) acc += p.ws[s * slab + (size_t)n * p.M + f];
            const size_t o = (size_t)n * p.ldo + f;
            if (p.epi == EPI_STORE_F32)
                reinterpret_cast<float*>(p.out)[o] = acc;
            else if (p.epi == EPI_ADD_F32)
                reinterpret_cast<float*>(p.out)[o] += acc;
            else
                reinterpret_cast<__half*>(p.out)[o] = to_f16(acc, range_bad);
        }
    }
    if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
}
// Split-K finish of a residual-add GEMM fused with the RMSNorm that follows
// it (batched decode rounds: O, then the FFN norm; down, then the next
// layer's attention norm).  One CTA per token row: the partials summed in
// split order and added to the residual row (the values gemm_splitk_reduce
// would store), the row written back, then its RMSNorm with gain g as fp16.
constexpr int ADDNORM_THREADS = 256, ADDNORM_VEC = 5;

__global__ void __launch_bounds__(ADDNORM_THREADS) gemm_splitk_add_norm_kernel(const GemmArgs p,
                                                                               const __nv_bfloat16* g,
                                                                               float eps, __half* h)
{
    __shared__ float red[ADDNORM_THREADS / 32];
    __shared__ float s_scale;
    grid_dep_wait();
    const int n = blockIdx.x, H = p.M;
    const size_t slab = (size_t)p.N * p.M;
    float* x = reinterpret_cast<float*>(p.out) + (size_t)n * p.ldo;
    const float* w0 = p.ws + (size_t)n * p.M;
    float4 v[ADDNORM_VEC];
#pragma unroll
    for (int k = 0; k < ADDNORM_VEC; ++k) v[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    // four splits' loads in flight at a time, added in split order
    for (int s0 = 0; s0 < p.k_splits; s0 += 4) {
        float4 t[4][ADDNORM_VEC];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int k = 0; k < ADDNORM_VEC; ++k) {
                const int i = (threadIdx.x + k * ADDNORM_THREADS) * 4;
                t[j][k] = s0 + j < p.k_splits && i < H
                              ? __ldcg(reinterpret_cast<const float4*>(w0 + (size_t)(s0 + j) * slab + i))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
        for (int j = 0; j < 4; ++j)
            if (s0 + j < p.k_splits) {
#pragma unroll
                for (int k = 0; k < ADDNORM_VEC; ++k) {
                    v[k].x += t[j][k].x; v[k].y += t[j][k].y; v[k].z += t[j][k].z; v[k].w += t[j][k].w;
                }
            }
    }
    float ss = 0.f;
#pragma unroll
    for (int k = 0; k < ADDNORM_VEC; ++k) {
        const int i = (threadIdx.x + k * ADDNORM_THREADS) * 4;
        if (i < H) {
            const float4 o = *reinterpret_cast<const float4*>(x + i);
            v[k] = make_float4(o.x + v[k].x, o.y + v[k].y, o.z + v[k].z, o.w + v[k].w);
            *reinterpret_cast<float4*>(x + i) = v[k];
            ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
        }
    }
    grid_dep_launch();
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < ADDNORM_THREADS / 32; ++w) t += red[w];
        s_scale = 1.0f / sqrtf(t / (float)H + eps);
    }
    __syncthreads();
    const float sc = s_scale;
    __half* hr = h + (size_t)n * H;
    bool bad = false;
#pragma unroll
    for (int k = 0; k < ADDNORM_VEC; ++k) {
        const int i = (threadIdx.x + k * ADDNORM_THREADS) * 4;
        if (i < H) {
            const uint2 gg = *reinterpret_cast<const uint2*>(g + i);
            __half2 lo, hi;
            lo.x = to_f16(v[k].x * sc * bf16lo(gg.x), bad);
            lo.y = to_f16(v[k].y * sc * bf16hi(gg.x), bad);
            hi.x = to_f16(v[k].z * sc * bf16lo(gg.y), bad);
            hi.y = to_f16(v[k].w * sc * bf16hi(gg.y), bad);
            uint2 o;
            o.x = *reinterpret_cast<const uint32_t*>(&lo);
            o.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(hr + i) = o;
        }
    }
    if (bad) set_status(p.status, Q3_STATUS_F16_RANGE);
}

template <int BN, bool QKV>
cudaError_t launch_bn(const Launch& L, const CUtensorMap& a0, const CUtensorMap& a1,
                      const CUtensorMap& a2, const CUtensorMap& b, const GemmArgs& g)
{
    using C = GemmCfg<BN>;
    static std::atomic<unsigned long long> attr_done{0};
    if (cudaError_t e = allow_smem_per_device(gemm_tc_kernel<BN, QKV>, C::SMEM, attr_done)) return e;
    const int n_tiles = (g.N + BN - 1) / BN;
    const int units = n_tiles * (g.M / BM) * g.k_splits;
    const int grid = units < 152 ? units : 152;          // persistent: one CTA per SM
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(GEMM_THREADS);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN, QKV>, a0, a1, a2, b, g);
}

}  // namespace

int gemm_block_n(int N)
{
    if (N <= 32) return 32;
    if (N <= 64) return 64;
    if (N <= 128) return 128;
    return 256;
}

bool gemm_block_n_supported(int bn)
{
    return bn == 32 || bn == 64 || bn == 96 || bn == 128 || bn == 144 || bn == 160 || bn == 176 || bn == 192 ||
           bn == 256;
}

cudaError_t launch_gemm(const Launch& L, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& a2, const CUtensorMap& b, int bn, const GemmArgs& g)
{
    // the fused head epilogue needs whole tiles in one pass, one 128-row head
    // per m-tile (q, then k, then v heads), and every buffer it reads or writes
    if (g.epi == EPI_QKV_ROPE) {
        const RopeArgs& r = g.rope;
        if (g.k_splits != 1 || g.pair || r.n_q < 1 || r.n_kv < 1 || g.M != (r.n_q + 2 * r.n_kv) * BM ||
            !r.row_pos || !r.row_slot || !r.tables || !r.rope || !r.q_gain || !r.k_gain || !r.kv_layer ||
            !r.q_out16 || !r.status || r.kvq_layer || r.n_blocks < 1 || r.max_blocks < 1)
            return cudaErrorInvalidValue;
    }
    if (g.epi == EPI_QKV_ROPE) {
        switch (bn) {
        case 32: return launch_bn<32, true>(L, a0, a1, a2, b, g);
        case 64: return launch_bn<64, true>(L, a0, a1, a2, b, g);
        case 96: return launch_bn<96, true>(L, a0, a1, a2, b, g);
        case 128: return launch_bn<128, true>(L, a0, a1, a2, b, g);
        case 144: return launch_bn<144, true>(L, a0, a1, a2, b, g);
        case 160: return launch_bn<160, true>(L, a0, a1, a2, b, g);
        case 176: return launch_bn<176, true>(L, a0, a1, a2, b, g);
        case 192: return launch_bn<192, true>(L, a0, a1, a2, b, g);
        case 256: return launch_bn<256, true>(L, a0, a1, a2, b, g);
        default: return cudaErrorInvalidValue;
        }
    }
    switch (bn) {
    case 32: return launch_bn<32, false>(L, a0, a1, a2, b, g);
    case 64: return launch_bn<64, false>(L, a0, a1, a2, b, g);
    case 96: return launch_bn<96, false>(L, a0, a1, a2, b, g);
    case 128: return launch_bn<128, false>(L, a0, a1, a2, b, g);
    case 144: return launch_bn<144, false>(L, a0, a1, a2, b, g);
    case 160: return launch_bn<160, false>(L, a0, a1, a2, b, g);
    case 176: return launch_bn<176, false>(L, a0, a1, a2, b, g);
    case 192: return launch_bn<192, false>(L, a0, a1, a2, b, g);
    case 256: return launch_bn<256, false>(L, a0, a1, a2, b, g);
    default: return cudaErrorInvalidValue;
    }
}


cudaError_t launch_gemm_splitk_reduce(const Launch& L, const GemmArgs& g)
{
    const int m_out = g.pair ? g.M / 2 : g.M;
    const size_t total = (size_t)g.N * m_out;
    int blocks = (int)((total + 255) / 256);
    if (blocks > 152 * 16) blocks = 152 * 16;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(blocks);
    cfg.blockDim = dim3(256);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, gemm_splitk_reduce_kernel, g);
}

bool gemm_add_norm_ok(const GemmArgs& g)
{
    return g.k_splits > 1 && !g.pair && g.epi == EPI_ADD_F32 && g.M % 4 == 0 && g.ldo % 4 == 0 &&
           g.M <= ADDNORM_THREADS * 4 * ADDNORM_VEC;
}

cudaError_t launch_gemm_splitk_add_norm(const Launch& L, const GemmArgs& g, const __nv_bfloat16* gain, float eps,
                                        __half* h)
{
    if (!gemm_add_norm_ok(g)) return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(g.N);
    cfg.blockDim = dim3(ADDNORM_THREADS);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, gemm_splitk_add_norm_kernel, g, gain, eps, h);
}

}  // namespace q3
