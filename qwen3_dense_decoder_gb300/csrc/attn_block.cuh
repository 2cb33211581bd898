// attn_block.cuh -- one 32-position block of GQA decode attention on
// mma.sync tensor cores, shared by the fused decode step and the batched
// decode attention kernel.
//
// Scores q . k / sqrt(128) over a paged BF16 K/V block ("Kipp Model
// Support", section "qwen3-0.6b-base": K/V stored as BF16), online softmax
// in base 2 (log2(e) folded into q), O += P V.  q and P enter the BF16
// products as high/low BF16 pairs (row 2h the high part of head h, row
// 2h + 1 the remainder), so both products keep about 16 bits while K and V
// are used exactly as stored.  With the opt-in Q8_0 cache the staged tiles
// hold fp16(scale * code) and the products run in fp16, q and P as fp16
// high/low pairs (about 22 bits).
#pragma once

#include "common.cuh"

namespace q3 {

constexpr int ATT_KSTR = 128 + 8;          // staged K/V/q row stride (bf16): 272 bytes, conflict-free ldmatrix

Q3_DEV void ldsm_x4(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
Q3_DEV void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]) : "r"(smem_u32(p)));
}
// D = A (16 x 16, row) * B (16 x 8, col) + D, bf16 inputs, fp32 accumulate
Q3_DEV void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                     uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                 "{%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
Q3_DEV uint32_t pack_bf16(float lo, float hi) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// the same with fp16 inputs
Q3_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0,
                    uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                 "{%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
Q3_DEV uint32_t pack_h2(float lo, float hi) {
    const __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t*>(&v);
}
// operand type of the block products: bf16 (the BF16 cache) or fp16 (Q8_0 cache)
template <bool F16>
Q3_DEV void mma_kv(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, uint32_t b0, uint32_t b1) {
    if (F16) mma_f16(d, a0, a1, a2, a3, b0, b1);
    else mma_bf16(d, a0, a1, a2, a3, b0, b1);
}
template <bool F16>
Q3_DEV float round_op(float x) {
    return F16 ? __half2float(__float2half_rn(x)) : __bfloat162float(__float2bfloat16_rn(x));
}
template <bool F16>
Q3_DEV uint32_t pack_op(float lo, float hi) {
    return F16 ? pack_h2(lo, hi) : pack_bf16(lo, hi);
}

// Online-softmax state of one warp over its blocks: the warp holds S and O
// rows g = lane / 4 and g + 8 of the 16-row operands, row r standing for
// query head r / 2 (even r: the bf16 high part of q or p, odd r: the
// remainder), so q . k and p . v are exact to about 16 bits while K and V
// stay the stored BF16.  NDT dimension tiles of 8 from tile dt0.
template <int NDT>
struct AttAcc {
    float m[2], l[2];
    float o[NDT][4];
};

// Address of 16-byte chunk c (0..15, 8 dims each) of row r of a staged K/V
// tile (rows of ATT_KSTR bf16).
Q3_DEV const uint8_t* tile_chunk(const uint8_t* t, int r, int c) {
    return t + r * (ATT_KSTR * 2) + c * 16;
}

// The two halves of one 32-position block for the G query heads of the KV
// head (rows 2h, 2h+1 of sqa, rows of ATT_KSTR elements).  attend_qk: S =
// q K^T on 4 x 8 mma (positions x dims), masked to n_pos, the online-softmax
// update (running maximum and sum, O rescaled) and P as high/low pairs in
// the A-fragment registers pa.  attend_pv: O += P V for output dimension
// tiles [dt0, dt0 + NDT).  Kept apart so a caller may reuse one staged tile
// for K and then V.
template <int NDT, bool F16>
Q3_DEV void attend_qk(const uint8_t* kt, const uint16_t* sqa, int n_pos, int lane, AttAcc<NDT>& w,
                      uint32_t (&pa)[4][2]) {
    const int g = lane >> 2, tig = lane & 3;
    float sacc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
    const int mi = lane >> 3, r8 = lane & 7;
#pragma unroll
    for (int kk = 0; kk < 128 / 16; ++kk) {
        uint32_t a[4];
        // A: matrices (rows 0-7, k 0-7), (rows 8-15, k 0-7), (rows 0-7, k 8-15), (rows 8-15, k 8-15)
        ldsm_x4(a, sqa + ((mi & 1) * 8 + r8) * ATT_KSTR + kk * 16 + (mi >> 1) * 8);
#pragma unroll
        for (int nh = 0; nh < 2; ++nh) {
            uint32_t b[4];
            // B: positions 16 nh + (0-7 | 8-15) x dims (0-7 | 8-15) of this k step
            ldsm_x4(b, tile_chunk(kt, nh * 16 + (mi >> 1) * 8 + r8, kk * 2 + (mi & 1)));
            mma_kv<F16>(sacc[2 * nh], a[0], a[1], a[2], a[3], b[0], b[1]);
            mma_kv<F16>(sacc[2 * nh + 1], a[0], a[1], a[2], a[3], b[2], b[3]);
        }
    }
    // rows 2h and 2h + 1 hold the two parts of head h: add them (lanes g ^ 1)
    float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            float v = sacc[nt][e] + __shfl_xor_sync(0xffffffffu, sacc[nt][e], 4);
            const int pos = nt * 8 + 2 * tig + (e & 1);
            v = pos < n_pos ? v : -INFINITY;
            sacc[nt][e] = v;
            mx[e >> 1] = fmaxf(mx[e >> 1], v);
        }
    }
    float alpha[2], sum[2] = {0.f, 0.f};
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 1));
        mx[h] = fmaxf(mx[h], __shfl_xor_sync(0xffffffffu, mx[h], 2));
        const float m_new = fmaxf(w.m[h], mx[h]);
        alpha[h] = exp2f(w.m[h] - m_new);          // 0 on the first block (m = -inf)
        w.m[h] = m_new;
    }
    // P and its split: even rows take the high part, odd rows the rest
    const bool hi_row = (g & 1) == 0;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
        float pv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            pv[e] = exp2f(sacc[nt][e] - w.m[e >> 1]);
            sum[e >> 1] += pv[e];
        }
#pragma unroll
        for (int hp = 0; hp < 2; ++hp) {
            const float x0 = pv[2 * hp], x1 = pv[2 * hp + 1];
            const float h0 = round_op<F16>(x0);
            const float h1 = round_op<F16>(x1);
            pa[nt][hp] = hi_row ? pack_op<F16>(h0, h1) : pack_op<F16>(x0 - h0, x1 - h1);
        }
    }
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 1);
        sum[h] += __shfl_xor_sync(0xffffffffu, sum[h], 2);
        w.l[h] = w.l[h] * alpha[h] + sum[h];
    }
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) {
        w.o[dt][0] *= alpha[0]; w.o[dt][1] *= alpha[0];
        w.o[dt][2] *= alpha[1]; w.o[dt][3] *= alpha[1];
    }
}

template <int NDT, bool F16>
Q3_DEV void attend_pv(const uint8_t* vt, int dt0, int lane, AttAcc<NDT>& w, const uint32_t (&pa)[4][2]) {
    const int mi = lane >> 3, r8 = lane & 7;
    // O += P V: k = positions (2 steps of 16), n = this warp's dimension tiles
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) {
        uint32_t b[4];
        // V^T: matrices of positions (0-7 | 8-15 | 16-23 | 24-31) x dims 8 (dt0 + dt)
        ldsm_x4_t(b, tile_chunk(vt, mi * 8 + r8, dt0 + dt));
        mma_kv<F16>(w.o[dt], pa[0][0], pa[0][1], pa[1][0], pa[1][1], b[0], b[1]);
        mma_kv<F16>(w.o[dt], pa[2][0], pa[2][1], pa[3][0], pa[3][1], b[2], b[3]);
    }
}

// One whole block: attend_qk on kt, then attend_pv on vt.
template <int NDT, bool F16 = false>
Q3_DEV void attend_block_tc(const uint8_t* kt, const uint8_t* vt, const void* sqa, int n_pos, int dt0,
                            int lane, AttAcc<NDT>& w) {
    uint32_t pa[4][2];
    attend_qk<NDT, F16>(kt, static_cast<const uint16_t*>(sqa), n_pos, lane, w, pa);
    attend_pv<NDT, F16>(vt, dt0, lane, w, pa);
}


}  // namespace q3
