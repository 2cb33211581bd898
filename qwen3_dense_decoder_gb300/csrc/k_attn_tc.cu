// k_attn_tc.cu -- causal GQA attention of prefill rounds on the tcgen05
// tensor cores, scores and outputs accumulated in tensor memory.
//
// Rows of a prefill round attend to every earlier position of their session
// and to the rows before them in the round ("Kipp Roadmap", status v0.0.3:
// flash-attention prefill kernel; status v0.0.6: long-context prefill
// attention is the next lever; "Kipp Model Support", section
// "qwen3-0.6b-base": K/V stored as BF16, 32-position blocks).
//
// Work item: R = 128 / G consecutive positions of one session for all G query
// heads of one KV head, packed as the 128 rows of one MMA tile (row
// r = position index r / G, head r % G), so the heads of a group share every
// K/V tile.  The session's paged K/V is walked in tiles of 128 positions
// (four blocks through the block table) with an online softmax:
//   S  = Q K^T        tcgen05.mma, A = Q (tensor memory), B = K tile (shared
//                     memory), FP32 accumulator in tensor memory
//   P  = exp2(S - m)  softmax warps, two threads per row (64 columns each),
//                     P written back over its own S columns
//   O += P V          tcgen05.mma, A = P (tensor memory), B = V tile read
//                     MN-major from shared memory, FP32 accumulator in TMEM
// Operands are BF16, so the K/V tiles feed the products exactly as stored,
// straight from the bulk tensor copies.  Q (fp16) and P enter as high/low
// BF16 pairs: Q = hi + lo exactly, P to about 16 bits, each product being two
// MMAs into the same accumulator.
// The running maximum is raised lazily: O and the row sum are rescaled only
// when a row maximum grows by more than 2^8, and the final O / l is the same
// quantity.
//
// K and V pass through three-stage rings; Q has one tensor-memory buffer,
// released for the next item once the item's last scores have been computed.
//
// Roles (one CTA per SM, items from a host-built per-CTA list):
//   warp 0       lane 0 issues every MMA and owns the tensor-memory columns
//   warps 1, 2   lane 0 fetches the K (warp 1) or V (warp 2) blocks of each
//                tile with TMA (blocks past the item's last position, or
//                outside the pool, are read at a negative row and land as
//                zeros); a K stage is free again once its scores are done, a
//                V stage once its PV is
//   warps 4..11  softmax and output: warp w reads TMEM lanes 32 (w % 4) ..
//                + 32 and columns 64 ((w - 4) / 4) .. + 64 of its row, so two
//                warps share each row (maxima exchanged through shared memory)
//   warps 12..15 Q: warp w loads the rows of TMEM lanes 32 (w % 4) .. + 32 of
//                the next item ahead of time and stores their high/low parts
//                once the buffer is free
// Tensor memory (512 columns): S[2] at 0 / 128 (P high at +0, low at +64,
// over S), O at 256, Q high at 384, low at 448.
// K/V rows past a row's position are finite (the pool is zeroed when it is
// made, and only finite BF16 values are stored), so P = 0 there contributes
// nothing.  Every wait is bounded; a timeout sets the status word and the CTA
// winds down without touching its remaining items.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int BN = 128;                      // key positions per K/V tile
constexpr int ATOM = 128 * 128;              // one 128-row x 64-column bf16 swizzle atom (bytes)
constexpr int TILE = 2 * ATOM;               // 128 rows x 128 bf16 (32 KB)
constexpr int NSOFT = 8;                     // softmax warps (two per TMEM lane quadrant)
constexpr int SOFT0 = 4, QL0 = SOFT0 + NSOFT;
constexpr int NQL = 4;                       // Q warps (one per TMEM lane quadrant)
constexpr int THREADS = (QL0 + NQL) * 32;
constexpr int TMEM_COLS = 512;
constexpr uint32_t T_S = 0, T_O = 256, T_Q = 384;
constexpr float LAZY = 8.0f;                 // log2 growth of a row maximum tolerated before rescaling

constexpr int NST = 3;                       // K/V ring stages

struct alignas(1024) TcSmem {
    uint8_t k[NST][TILE];
    uint8_t v[NST][TILE];
    uint64_t q_full, q_free, k_load[NST], k_free[NST], v_load[NST], v_free[NST], s_full[2], p_full[2], pv_done[2];
    uint64_t o_free, drain, pair[4];
    float xch[2][128];                       // [column half][row] maxima, then row sums
    uint32_t tmem;
    int abort;
};
constexpr size_t SMEM_BYTES = sizeof(TcSmem) + 1024;

// Instruction descriptors: bf16 A/B (format 1 at [7,10) and [10,13)), FP32
// accumulator, M = 128, N = 128.  S: B K-major.  PV: B (V, positions x dims)
// MN-major (bit 16).
constexpr uint32_t IDESC_S = idesc_f16_f32(128, 128) | (1u << 7) | (1u << 10);
constexpr uint32_t IDESC_PV = IDESC_S | (1u << 16);

// MN-major 128-byte-swizzled operand: rows of 64 MN elements (128 bytes),
// 8-row groups 1024 bytes apart along K (stride offset), 64-element MN blocks
// `lbo` bytes apart (leading offset).
Q3_DEV uint64_t smem_desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// D[tmem] (+)= A[tmem] * B[smem], kind::f16
Q3_DEV void tc_mma_f16_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t bdesc, uint32_t idesc,
                          uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

Q3_DEV void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                   "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                 : "r"(taddr));
}

Q3_DEV void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
                    "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
                    "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}
Q3_DEV void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// x as a high/low pair of bf16: hi = bf16(x), lo = bf16(x - hi)
Q3_DEV void split_bf16(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const float2 hf = __bfloat1622float2(h);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - hf.x, x1 - hf.y);
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

// Bounded mbarrier wait shared by all roles of the CTA: gives up when another
// role has aborted or Q3_WAIT_LIMIT_NS passes (then sets the timeout status).
Q3_DEV bool wait_bar(uint64_t* bar, uint32_t parity, TcSmem& sm, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (*(volatile int*)&sm.abort) return false;
        if (global_ns() - t0 > Q3_WAIT_LIMIT_NS) {
            set_status(status, Q3_STATUS_TIMEOUT);
            *(volatile int*)&sm.abort = 1;
            return false;
        }
    }
}

struct Item {
    int row0, nrows, pos0, pos_last, n_kt, kvh;
    const int* table;
};

Q3_DEV Item item_of(const PrefillAttnArgs& p, int k) {
    Item it;
    const int code = p.sched_items[k];
    const int tile = code / p.n_kv;
    it.kvh = code % p.n_kv;
    it.row0 = p.tile_row0[tile];
    it.nrows = p.tile_rows[tile];
    it.pos0 = p.row_pos[it.row0];
    it.pos_last = it.pos0 + it.nrows - 1;
    it.n_kt = it.pos_last / BN + 1;
    it.table = p.tables + (size_t)p.row_slot[it.row0] * p.max_blocks;
    return it;
}

// ---------------------------------------------------------------- MMA issuer
Q3_DEV void mma_role(const PrefillAttnArgs& p, TcSmem& sm, uint32_t tmem, int i0, int i1) {
    uint32_t g = 0;                                  // K/V tiles issued so far by this CTA
    // S = (Q_hi + Q_lo) K^T: 16 dims a step, the high part's 8 steps, then the low part's
    auto issue_s = [&](uint32_t gt) -> bool {
        const int b = gt & 1, st = gt % NST;
        if (!wait_bar(&sm.k_load[st], (gt / NST) & 1, sm, p.status)) return false;
        tc_fence_after();
        const uint32_t ka = smem_u32(sm.k[st]);
#pragma unroll
        for (int part = 0; part < 2; ++part)
#pragma unroll
            for (int s = 0; s < D / 16; ++s) {
                const uint32_t off = (s >> 2) * ATOM + (s & 3) * 32;
                tc_mma_f16_ts(tmem + T_S + b * 128, tmem + T_Q + part * 64 + s * 8, smem_desc_sw128(ka + off),
                              IDESC_S, (part > 0 || s > 0) ? 1u : 0u);
            }
        tc_commit(&sm.s_full[b]);
        tc_commit(&sm.k_free[st]);
        return true;
    };
    bool ok = true;
    if (i0 < i1) {
        const Item it0 = item_of(p, i0);
        ok = wait_bar(&sm.q_full, 0, sm, p.status) && issue_s(0);
        if (ok && it0.n_kt == 1) tc_commit(&sm.q_free);
    }
    for (int k = i0, local = 0; k < i1 && ok; ++k, ++local) {
        const Item it = item_of(p, k);
        for (int t = 0; t < it.n_kt; ++t, ++g) {
            // scores of the item's next tile run while the softmax works on this one;
            // after the item's last scores its Q buffer is free for the next item
            if (t + 1 < it.n_kt) {
                if (!(ok = issue_s(g + 1))) break;
                if (t + 2 == it.n_kt) tc_commit(&sm.q_free);
            }
            // O of the previous item read out before this item's first PV overwrites it
            if (t == 0 && local > 0 && !(ok = wait_bar(&sm.o_free, (local - 1) & 1, sm, p.status))) break;
            const int b = g & 1, st = g % NST;
            if (!(ok = wait_bar(&sm.p_full[b], (g >> 1) & 1, sm, p.status))) break;
            if (!(ok = wait_bar(&sm.v_load[st], (g / NST) & 1, sm, p.status))) break;
            tc_fence_after();
            // O += (P_hi + P_lo) V, 16 positions a step; P lies over S[b]
            const uint32_t va = smem_u32(sm.v[st]);
#pragma unroll
            for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int s = 0; s < BN / 16; ++s)
                    tc_mma_f16_ts(tmem + T_O, tmem + T_S + b * 128 + part * 64 + s * 8,
                                  smem_desc_sw128_mn(va + s * 2048, ATOM), IDESC_PV,
                                  (t > 0 || part > 0 || s > 0) ? 1u : 0u);
            tc_commit(&sm.pv_done[b]);
            tc_commit(&sm.v_free[st]);
        }
        if (!ok) break;
        // the next item's first scores (g is its first tile)
        if (k + 1 < i1) {
            const int nl = local + 1;
            const Item nx = item_of(p, k + 1);
            ok = wait_bar(&sm.q_full, nl & 1, sm, p.status) && issue_s(g);
            if (ok && nx.n_kt == 1) tc_commit(&sm.q_free);
        }
    }
    // nothing of this CTA's may still run on the tensor cores at deallocation
    tc_commit(&sm.drain);
    mbar_wait(&sm.drain, 0, p.status);
}

// ---------------------------------------------------------------- K/V loaders
// One thread fetches the K (which = 0) or V (which = 1) blocks of each tile,
// up to NST tiles ahead: per block two 64-column boxes of 32 positions into
// their 128-byte-swizzled places.  The tile's block-table entries are read
// before the stage is waited for.  A block past the item's last position (or
// whose table entry is outside the pool) is read at row -32, wholly outside
// the tensor, and lands as zeros.
Q3_DEV void load_role(const PrefillAttnArgs& p, const CUtensorMap* tkv, TcSmem& sm, int i0, int i1, int which) {
    uint64_t* ld = which ? sm.v_load : sm.k_load;
    uint64_t* fr = which ? sm.v_free : sm.k_free;
    uint32_t g = 0;
    for (int k = i0; k < i1; ++k) {
        const Item it = item_of(p, k);
        for (int t = 0; t < it.n_kt; ++t, ++g) {
            const int b = g % NST;
            int row[BN / 32];
#pragma unroll
            for (int j = 0; j < BN / 32; ++j) {
                const int kp = t * BN + 32 * j;
                row[j] = -32;
                if (kp <= it.pos_last) {
                    const int ph = it.table[kp >> 5];
                    if (ph >= 0 && ph < p.n_blocks)
                        row[j] = p.kv_row0 + ((ph * 2 + which) * p.n_kv + it.kvh) * 32;
                    else if (which == 0)
                        set_status(p.status, Q3_STATUS_BLOCK_RANGE);
                }
            }
            if (g >= NST && !wait_bar(&fr[b], (g / NST - 1) & 1, sm, p.status)) return;
            uint8_t* dst = which ? sm.v[b] : sm.k[b];
            mbar_arrive_expect_tx(&ld[b], TILE);
#pragma unroll
            for (int j = 0; j < BN / 32; ++j) {
                tma_load_2d(dst + j * 32 * 128, tkv, &ld[b], 0, row[j]);
                tma_load_2d(dst + ATOM + j * 32 * 128, tkv, &ld[b], 64, row[j]);
            }
        }
    }
}

// ---------------------------------------------------------------- Q
// Warp w holds TMEM lanes 32 (w % 4) .. + 32: lane l's row r is position
// index r / G, head r % G of the item (padding rows repeat row 0).  The next
// item's rows are loaded while the current item's scores still read the
// buffer; once the last of them is done the high and low parts are stored.
Q3_DEV void q_role(const PrefillAttnArgs& p, TcSmem& sm, uint32_t tmem, int i0, int i1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, row = quad * 32 + lane;
    const int G = p.n_q / p.n_kv, R = 128 / G;
    const int qw = p.n_q * D;
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    for (int k = i0, local = 0; k < i1; ++k, ++local) {
        const Item it = item_of(p, k);
        int ir = row / G, hh = row % G;
        if (ir >= R) ir = hh = 0;
        const int src_row = it.row0 + min(ir, it.nrows - 1);
        const uint4* src = reinterpret_cast<const uint4*>(p.q + (size_t)src_row * qw + (it.kvh * G + hh) * D);
        uint4 qv[D / 8];
#pragma unroll
        for (int c = 0; c < D / 8; ++c) qv[c] = __ldcg(src + c);
        if (local >= 1 && !wait_bar(&sm.q_free, (local - 1) & 1, sm, p.status)) return;
        tc_fence_after();
#pragma unroll
        for (int c = 0; c < 4; ++c) {                      // 32 dims (16 columns) at a time
            uint32_t hi[16], lo[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const uint4 w = qv[c * 4 + e / 4];
                const uint32_t h2 = (&w.x)[e & 3];
                const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
                split_bf16(f.x, f.y, hi[e], lo[e]);
            }
            tmem_st_32x32b_x16(tl + T_Q + c * 16, hi);
            tmem_st_32x32b_x16(tl + T_Q + 64 + c * 16, lo);
        }
        tmem_st_wait();
        tc_fence_before();
        mbar_arrive(&sm.q_full);
    }
}

// ---------------------------------------------------------------- softmax + output
Q3_DEV float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}


// the two warps of a TMEM lane quadrant meet on the quadrant's mbarrier
// (bounded, so a partner that gave up cannot leave this warp waiting); n
// counts the meetings so far
Q3_DEV bool pair_sync(TcSmem& sm, int quad, uint32_t& n, int* status) {
    mbar_arrive(&sm.pair[quad]);
    const bool ok = wait_bar(&sm.pair[quad], n & 1, sm, status);
    ++n;
    return ok;
}

Q3_DEV void softmax_role(const PrefillAttnArgs& p, TcSmem& sm, uint32_t tmem, int i0, int i1) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, half = (warp - SOFT0) >> 2;
    const int row = quad * 32 + lane;
    const int c0 = half * 64;                                     // this warp's 64 columns
    const int G = p.n_q / p.n_kv, R = 128 / G;
    const int qw = p.n_q * D;
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);     // this warp's TMEM lanes
    const float scale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    uint32_t g = 0, npair = 0;
    for (int k = i0, local = 0; k < i1; ++k, ++local) {
        const Item it = item_of(p, k);
        const int ir = row / G, hh = row % G;
        const bool valid = ir < R && ir < it.nrows;
        const int qp = it.pos0 + min(ir, it.nrows - 1);
        float m_used = -INFINITY, l = 0.f;
        for (int t = 0; t < it.n_kt; ++t, ++g) {
            const int b = g & 1;
            if (!wait_bar(&sm.s_full[b], (g >> 1) & 1, sm, p.status)) return;
            tc_fence_after();
            uint32_t v[2][32];
            tmem_ld_32x32b_x32(tl + T_S + b * 128 + c0, v[0]);
            tmem_ld_32x32b_x32(tl + T_S + b * 128 + c0 + 32, v[1]);
            tmem_ld_wait();
            // raw scores are scaled by a positive constant: their maximum scales with them
            const int kb = t * BN + c0;
            const bool need_mask = kb + 63 > it.pos0;
            float mx = -INFINITY;
            if (need_mask) {
#pragma unroll
                for (int e = 0; e < 64; ++e)
                    if (kb + e > qp) v[e >> 5][e & 31] = __float_as_uint(-INFINITY);
            }
#pragma unroll
            for (int e = 0; e < 64; ++e) mx = fmaxf(mx, __uint_as_float(v[e >> 5][e & 31]));
            if (!pair_sync(sm, quad, npair, p.status)) return;   // the partner has read the last exchange
            sm.xch[half][row] = mx * scale;
            if (!pair_sync(sm, quad, npair, p.status)) return;
            const float m_new = fmaxf(m_used, fmaxf(sm.xch[0][row], sm.xch[1][row]));
            if (t == 0) {
                m_used = m_new;
            } else if (__any_sync(0xffffffffu, m_new > m_used + LAZY)) {
                // raise the maximum: O (complete up to the previous tile) and l rescale;
                // both warps of the rows take the same decision from the same values
                const float alpha = ex2(m_used - m_new);
                const uint32_t gp = g - 1;
                if (!wait_bar(&sm.pv_done[gp & 1], (gp >> 1) & 1, sm, p.status)) return;
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < 4; ++c) {                   // 16 columns at a time: S stays in registers
                    uint32_t o[16];
                    tmem_ld_32x32b_x16(tl + T_O + c0 + c * 16, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
                    tmem_st_32x32b_x16(tl + T_O + c0 + c * 16, o);
                }
                tmem_st_wait();
                l *= alpha;
                m_used = m_new;
            }
            // P over S[b]: both warps of the row read their S columns before the
            // maxima were exchanged, and the PV two tiles back that read P there
            // ran before these scores (the tensor cores keep issue order)
            float sum = 0.f;
#pragma unroll
            for (int hq = 0; hq < 2; ++hq) {
                uint32_t ph[16], pl[16];
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const float p0 = ex2(fmaf(__uint_as_float(v[hq][2 * e]), scale, -m_used));
                    const float p1 = ex2(fmaf(__uint_as_float(v[hq][2 * e + 1]), scale, -m_used));
                    sum += p0 + p1;
                    split_bf16(p0, p1, ph[e], pl[e]);
                }
                tmem_st_32x32b_x16(tl + T_S + b * 128 + c0 / 2 + 16 * hq, ph);
                tmem_st_32x32b_x16(tl + T_S + b * 128 + 64 + c0 / 2 + 16 * hq, pl);
            }
            tmem_st_wait();
            l += sum;
            tc_fence_before();
            mbar_arrive(&sm.p_full[b]);
        }
        // the item's O is complete once the PV of its last tile is; the row
        // sum is the two halves'
        if (!pair_sync(sm, quad, npair, p.status)) return;
        sm.xch[half][row] = l;
        {
            const uint32_t gl = g - 1;
            if (!wait_bar(&sm.pv_done[gl & 1], (gl >> 1) & 1, sm, p.status)) return;
            tc_fence_after();
        }
        if (!pair_sync(sm, quad, npair, p.status)) return;
        const float inv = 1.0f / (sm.xch[0][row] + sm.xch[1][row]);
        bool bad = false;
        __half* dst = p.out + (size_t)(it.row0 + min(ir, it.nrows - 1)) * qw + (it.kvh * G + hh) * D + c0;
#pragma unroll 1
        for (int c = 0; c < 2; ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tl + T_O + c0 + c * 32, o);
            tmem_ld_wait();
            if (valid) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    uint4 w;
                    uint32_t* wp = &w.x;
#pragma unroll
                    for (int f = 0; f < 4; ++f) {
                        __half2 h2;
                        h2.x = to_f16(__uint_as_float(o[8 * e + 2 * f]) * inv, bad);
                        h2.y = to_f16(__uint_as_float(o[8 * e + 2 * f + 1]) * inv, bad);
                        wp[f] = *reinterpret_cast<uint32_t*>(&h2);
                    }
                    *reinterpret_cast<uint4*>(dst + c * 32 + e * 8) = w;
                }
            }
        }
        if (bad) set_status(p.status, Q3_STATUS_F16_RANGE);
        tc_fence_before();
        mbar_arrive(&sm.o_free);
    }
}

__global__ void __launch_bounds__(THREADS, 1) prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap tkv,
                                                                      const PrefillAttnArgs p)
{
    extern __shared__ uint8_t smem_raw[];
    TcSmem& sm = *reinterpret_cast<TcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(&sm.q_full, NQL * 32);
        mbar_init(&sm.q_free, 1);
        for (int b = 0; b < NST; ++b) {
            mbar_init(&sm.k_load[b], 1);
            mbar_init(&sm.k_free[b], 1);
            mbar_init(&sm.v_load[b], 1);
            mbar_init(&sm.v_free[b], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&sm.s_full[b], 1);
            mbar_init(&sm.p_full[b], NSOFT * 32);
            mbar_init(&sm.pv_done[b], 1);
        }
        mbar_init(&sm.o_free, NSOFT * 32);
        for (int i = 0; i < 4; ++i) mbar_init(&sm.pair[i], 64);
        mbar_init(&sm.drain, 1);
        sm.abort = 0;
        fence_barrier_init();
        prefetch_tmap(&tkv);
    }
    if (warp == 0) {
        tmem_alloc(&sm.tmem, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sm.tmem;

    grid_dep_wait();
    const int i0 = p.sched_start[blockIdx.x], i1 = p.sched_start[blockIdx.x + 1];
    if (warp == 0) {
        if ((threadIdx.x & 31) == 0) mma_role(p, sm, tmem, i0, i1);
        __syncwarp();
    } else if (warp == 1 || warp == 2) {
        if ((threadIdx.x & 31) == 0) load_role(p, &tkv, sm, i0, i1, warp - 1);
        __syncwarp();
    } else if (warp >= SOFT0 && warp < SOFT0 + NSOFT) {
        softmax_role(p, sm, tmem, i0, i1);
    } else if (warp >= QL0) {
        q_role(p, sm, tmem, i0, i1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
    grid_dep_launch();
}

}  // namespace

int prefill_tc_rows(int n_q, int n_kv)
{
    if (n_kv < 1 || n_q % n_kv) return 0;
    const int G = n_q / n_kv;
    return G <= 128 ? 128 / G : 0;
}

size_t prefill_tc_smem() { return SMEM_BYTES; }

cudaError_t launch_prefill_attention_tc(const Launch& L, const CUtensorMap& tkv, const PrefillAttnArgs& a, int grid)
{
    if (prefill_tc_rows(a.n_q, a.n_kv) < 1 || grid < 1) return cudaErrorInvalidValue;
    static std::atomic<unsigned long long> attr_done{0};
    if (cudaError_t e = allow_smem_per_device(prefill_attn_tc_kernel, (int)SMEM_BYTES, attr_done)) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, prefill_attn_tc_kernel, tkv, a);
}

}  // namespace q3
