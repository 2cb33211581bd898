// k_attn.cu -- causal GQA attention over the paged BF16 KV cache.
//
// Every token row t of a round attends to positions [0, pos_t] of its own
// session ("Kipp Roadmap", status v0.0.2: paged KV through a per-session
// 32-position block table, bitwise equal to the contiguous layout; "Kipp
// Model Support", section "qwen3-0.6b-base": K/V stored as BF16).  Scores
// are q.k / sqrt(128); the softmax subtracts the running maximum (online
// softmax, base-2 exponentials with log2(e) folded into q).
//
// One CTA handles one (row, KV head, split): the G query heads that share the
// KV head (contiguous GQA grouping, query head h reads KV head h / G) read
// each K/V block once.  A split is a contiguous range of logical blocks whose
// bounds depend only on the context length, never on which physical blocks
// back it, so paged and contiguous layouts give identical bits.  Each of the
// four warps takes blocks round-robin and stages a block's K and V tiles in
// shared memory with cp.async (one memory latency per block), then attends
// the block on mma.sync tensor cores (q and P as BF16 high/low pairs, K and V
// as stored; the routine the fused decode step uses).
// Warps merge in warp order; splits merge in split order, done by whichever
// split CTA of the (row, KV head) finishes last (an atomic ticket, no
// waiting), so the result does not depend on scheduling.
//
// With the opt-in Q8_0 cache ("Kipp Roadmap", status v0.0.4) a warp copies
// the block's raw Q8_0 tiles (codes and fp16 scales, 4,352 bytes each for K
// and V, two copy groups) and expands them in shared memory into an fp16
// tile of scale * code (each product rounded once to fp16): K first for the
// scores and softmax, then V into the same tile for O += P V, with the next
// block's raw copies issued as soon as the raw buffer is free, so they
// overlap the products.  One tile per warp keeps three CTAs on an SM.  The
// new position's K/V are packed by the same rule as every other row.
//
// Decode rounds (each row the single new token of its session) fuse the
// per-head q/k RMSNorm, RoPE and the K/V append of that token: the new K/V
// row goes to the cache and straight into the staged tile, so tiles of
// earlier positions can be fetched before the projections of this round
// have landed (they are issued ahead of the programmatic-launch wait).
#include "attn_block.cuh"
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int KV_BLOCK = 32;
constexpr int AWARPS = 4;
constexpr int K_STRIDE = ATT_KSTR;     // bf16 per staged K/V row: 272 bytes, conflict-free ldmatrix
constexpr int K_TILE = KV_BLOCK * K_STRIDE;
constexpr int V_TILE = KV_BLOCK * K_STRIDE;
constexpr int NDT = D / 8;             // a warp attends all 16 dimension tiles of its blocks

template <int G, bool KQ>
struct AttnSmem {
    static constexpr size_t q_bytes = (size_t)16 * K_STRIDE * 2;     // q high/low rows (bf16 or fp16)
    static constexpr size_t k_bytes = (size_t)AWARPS * K_TILE * 2;
    static constexpr size_t v_bytes = KQ ? 0 : (size_t)AWARPS * V_TILE * 2;   // Q8_0: V reuses the K tile
    static constexpr size_t new_bytes = 2 * D * 2;                  // new K and V row (bf16 or fp16)
    static constexpr size_t misc_bytes = 2 * AWARPS * G * sizeof(float) + 16;
    static constexpr size_t raw_bytes = KQ ? (size_t)AWARPS * 2 * KVQ_TILE : 0;   // Q8_0 K and V tiles
    static constexpr size_t total = q_bytes + k_bytes + v_bytes + new_bytes + misc_bytes + raw_bytes;
};

// stage one 32-position K or V tile: 32 rows of 256 bytes, 16-byte pieces,
// 16 per lane, as one copy group
Q3_DEV void stage_tile(__nv_bfloat16* t, const __nv_bfloat16* src, int lane) {
#pragma unroll
    for (int i = 0; i < 16; ++i) {
        const int piece = i * 32 + lane;          // 512 pieces: row = piece / 16, col16 = piece % 16
        const int row = piece >> 4, c = piece & 15;
        cp_async_16(t + row * K_STRIDE + c * 8, src + row * D + c * 8);
    }
    cp_async_commit();
}

// stage the raw Q8_0 K and V tiles of one block: 272 16-byte pieces each,
// K and V as two copy groups (K can be expanded while V is in flight)
Q3_DEV void stage_block_q8(uint8_t* raw, const uint8_t* Kq, const uint8_t* Vq, int lane) {
    for (int i = lane; i < KVQ_TILE / 16; i += 32) cp_async_16(raw + i * 16, Kq + i * 16);
    cp_async_commit();
    for (int i = lane; i < KVQ_TILE / 16; i += 32) cp_async_16(raw + KVQ_TILE + i * 16, Vq + i * 16);
    cp_async_commit();
}

// expand one staged Q8_0 tile into an fp16 tile of scale * code (rows of
// K_STRIDE halves); lane l takes values [4l, 4l + 4) of every row
Q3_DEV void expand_q8(__nv_bfloat16* tile, const uint8_t* raw, int lane) {
#pragma unroll 4
    for (int r = 0; r < 32; ++r) {
        const uint32_t w = *reinterpret_cast<const uint32_t*>(raw + r * 128 + lane * 4);
        const __half d = *reinterpret_cast<const __half*>(raw + KVQ_CODES + (r * 4 + (lane >> 3)) * 2);
        *reinterpret_cast<uint2*>(tile + r * K_STRIDE + lane * 4) = kvq_dequant4(w, d);
    }
}

// head g's q (lane: dims [4 lane, 4 lane + 4)), scaled, as rows 2g (high
// part) and 2g + 1 (remainder) of the 16-row tensor-core operand, in the
// operand type of the block products (bf16, or fp16 for the Q8_0 cache)
template <bool F16>
Q3_DEV void store_q_split(__nv_bfloat16* sqa, int g, const float (&y)[4], float scale, int lane) {
    float hi[4], lo[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float q = y[e] * scale;
        hi[e] = round_op<F16>(q);
        lo[e] = q - hi[e];
    }
    *reinterpret_cast<uint2*>(sqa + (2 * g) * K_STRIDE + lane * 4) =
        make_uint2(pack_op<F16>(hi[0], hi[1]), pack_op<F16>(hi[2], hi[3]));
    *reinterpret_cast<uint2*>(sqa + (2 * g + 1) * K_STRIDE + lane * 4) =
        make_uint2(pack_op<F16>(lo[0], lo[1]), pack_op<F16>(lo[2], lo[3]));
}

template <int G, bool FUSED, bool KQ>
__global__ void __launch_bounds__(AWARPS * 32, 3) attn_kernel(const AttnArgs p)
{
    using S = AttnSmem<G, KQ>;
    extern __shared__ __align__(16) uint8_t smem[];
    __nv_bfloat16* sqa = reinterpret_cast<__nv_bfloat16*>(smem);                  // [16][K_STRIDE]
    __nv_bfloat16* kt_all = reinterpret_cast<__nv_bfloat16*>(smem + S::q_bytes);
    __nv_bfloat16* vt_all = reinterpret_cast<__nv_bfloat16*>(smem + S::q_bytes + S::k_bytes);
    __nv_bfloat16* snew = reinterpret_cast<__nv_bfloat16*>(smem + S::q_bytes + S::k_bytes + S::v_bytes);
    float* s_m = reinterpret_cast<float*>(smem + S::q_bytes + S::k_bytes + S::v_bytes + S::new_bytes);
    float* s_l = s_m + AWARPS * G;
    float* s_o = reinterpret_cast<float*>(kt_all);     // [AWARPS][G][D], reuses the K tiles at the end
    uint8_t* raw_all = smem + S::q_bytes + S::k_bytes + S::v_bytes + S::new_bytes + S::misc_bytes;
    __shared__ int s_ticket;

    const int split = blockIdx.x, kvh = blockIdx.y;
    const int t = p.row_order ? p.row_order[blockIdx.z] : (int)blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __nv_bfloat16* kt = kt_all + warp * K_TILE;
    __nv_bfloat16* vt = KQ ? kt : vt_all + warp * V_TILE;
    uint8_t* raw = raw_all + (size_t)warp * 2 * KVQ_TILE;     // (Q8_0 cache only)

    // Row metadata and block tables were uploaded before the round began, so
    // they may be read before the programmatic-launch wait.
    const int pos = p.row_pos[t];
    const int ctx = pos + 1;
    const int* table = p.tables + (size_t)p.row_slot[t] * p.max_blocks;
    const int nblk = (ctx + KV_BLOCK - 1) / KV_BLOCK;
    const int bps = (nblk + p.n_splits - 1) / p.n_splits;
    const int ns = (nblk + bps - 1) / bps;              // splits of this row that hold blocks
    const int b0 = split * bps;
    const int b1 = min(b0 + bps, nblk);
    const size_t head_elems = (size_t)KV_BLOCK * D;
    const int last_blk = nblk - 1;

    // issue the copies of block b's K/V (bf16 tiles, or raw Q8_0 tiles)
    auto stage = [&](int b) -> bool {
        const int phys = table[b];
        if (phys < 0 || phys >= p.n_blocks) return false;
        if (KQ) {
            const uint8_t* Kq = p.kvq_layer + ((size_t)phys * 2 * p.n_kv + kvh) * KVQ_TILE;
            stage_block_q8(raw, Kq, Kq + (size_t)p.n_kv * KVQ_TILE, lane);
        } else {
            const __nv_bfloat16* Kb = p.kv_layer + ((size_t)phys * 2 * p.n_kv + kvh) * head_elems;
            stage_tile(kt, Kb, lane);
            stage_tile(vt, Kb + (size_t)p.n_kv * head_elems, lane);
        }
        return true;
    };
    // BF16 cache: the next block's K copy once this block's scores are done,
    // its V copy once P V is done (each a copy group; false: nothing issued)
    auto stage_next_k = [&](int bn) -> bool {
        if (bn >= b1) return false;
        const int phys = table[bn];
        if (phys < 0 || phys >= p.n_blocks) return false;
        stage_tile(kt, p.kv_layer + ((size_t)phys * 2 * p.n_kv + kvh) * head_elems, lane);
        return true;
    };
    auto stage_next_v = [&](int bn) {
        const int phys = table[bn];
        stage_tile(vt, p.kv_layer + ((size_t)phys * 2 * p.n_kv + kvh) * head_elems + (size_t)p.n_kv * head_elems,
                   lane);
    };

    int b = b0 + warp;
    bool staged = false;
    if (FUSED && b < b1) staged = stage(b);   // K/V of earlier rounds do not depend on this round's kernels

    if (threadIdx.x == 0)
        issue_l2_prefetch(p.next, blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z),
                          gridDim.x * gridDim.y * gridDim.z);
    // the grid is sized for the round's longest context: splits past a
    // shorter row's blocks have nothing to do
    if (split >= ns) return;
    // the next kernel may now be scheduled into the SM space this grid leaves
    grid_dep_launch();
    grid_dep_wait();

    const float qscale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    if (FUSED) {
        const int n_heads = p.n_q + 2 * p.n_kv;
        const size_t row0 = (size_t)t * n_heads * D;
        const float2* rope_row = p.rope + (size_t)pos * (D / 2);
        // four projections of this row's head h: stored, or the QKV GEMM's
        // split-K partials summed in split order (the values its reduce stores)
        auto head4 = [&](int h) -> float4 {
            const size_t o = row0 + (size_t)h * D + lane * 4;
            if (p.qkv_splits <= 1) return *reinterpret_cast<const float4*>(p.qkv + o);
            const size_t slab = (size_t)p.T * n_heads * D;
            float4 s = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int sp = 0; sp < p.qkv_splits; ++sp) {
                const float4 w = __ldcg(reinterpret_cast<const float4*>(p.qkv_ws + sp * slab + o));
                s.x += w.x; s.y += w.y; s.z += w.z; s.w += w.w;
            }
            return s;
        };
        for (int g = warp; g < G; g += AWARPS) {
            const float4 v = head4(kvh * G + g);
            float y[4] = {v.x, v.y, v.z, v.w};
            head_norm_rope(y, p.q_gain, rope_row, p.eps, lane);
            store_q_split<KQ>(sqa, g, y, qscale, lane);
        }
        const bool mine = b0 <= last_blk && last_blk < b1;   // this split holds the new position
        if (mine && warp >= AWARPS - 2) {
            const bool is_k = warp == AWARPS - 2;
            const float4 v = head4(p.n_q + (is_k ? 0 : p.n_kv) + kvh);
            float y[4] = {v.x, v.y, v.z, v.w};
            if (is_k) head_norm_rope(y, p.k_gain, rope_row, p.eps, lane);
            const int phys = table[last_blk];
            const bool in_pool = phys >= 0 && phys < p.n_blocks;
            if (KQ) {
                // packed by the cache's Q8_0 rule; the tile gets the values the cache holds
                uint32_t codes;
                __half scale;
                float deq[4];
                kvq_pack(y, codes, scale, deq);
                *reinterpret_cast<uint2*>(snew + (is_k ? 0 : D) + lane * 4) =
                    make_uint2(pack_h2(deq[0], deq[1]), pack_h2(deq[2], deq[3]));
                if (in_pool)
                    kvq_store(p.kvq_layer + (((size_t)phys * 2 + (is_k ? 0 : 1)) * p.n_kv + kvh) * KVQ_TILE,
                              pos % KV_BLOCK, codes, scale, lane);
            } else {
                const __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
                const __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
                uint2 packed;
                packed.x = *reinterpret_cast<const uint32_t*>(&lo);
                packed.y = *reinterpret_cast<const uint32_t*>(&hi);
                *reinterpret_cast<uint2*>(snew + (is_k ? 0 : D) + lane * 4) = packed;
                if (in_pool) {
                    __nv_bfloat16* dst = p.kv_layer +
                        (((size_t)phys * 2 + (is_k ? 0 : 1)) * p.n_kv + kvh) * head_elems +
                        (size_t)(pos % KV_BLOCK) * D + lane * 4;
                    *reinterpret_cast<uint2*>(dst) = packed;
                }
            }
            if (!in_pool && lane == 0) set_status(p.status, Q3_STATUS_BLOCK_RANGE);
        }
    } else {
        for (int g = warp; g < G; g += AWARPS) {
            const float4 v = *reinterpret_cast<const float4*>(p.q + ((size_t)t * p.n_q + kvh * G + g) * D + lane * 4);
            float y[4] = {v.x, v.y, v.z, v.w};
            store_q_split<KQ>(sqa, g, y, qscale, lane);
        }
    }
    // rows of the 16-row q operand past the G heads are zero
    for (int i = threadIdx.x; i < (16 - 2 * G) * (D / 8); i += AWARPS * 32)
        *reinterpret_cast<uint4*>(sqa + (2 * G + i / (D / 8)) * K_STRIDE + (i % (D / 8)) * 8) = make_uint4(0, 0, 0, 0);
    __syncthreads();

    AttAcc<NDT> st;
    st.m[0] = st.m[1] = -INFINITY;
    st.l[0] = st.l[1] = 0.f;
#pragma unroll
    for (int dt = 0; dt < NDT; ++dt) st.o[dt][0] = st.o[dt][1] = st.o[dt][2] = st.o[dt][3] = 0.f;

    for (; b < b1; b += AWARPS) {
        if (!staged && !stage(b)) {
            if (lane == 0) set_status(p.status, Q3_STATUS_BLOCK_RANGE);
            continue;
        }
        staged = false;
        const int n_pos = min(KV_BLOCK, ctx - b * KV_BLOCK);
        const bool new_row = FUSED && b == last_blk;     // the new position: its K/V came from above
        const int r_new = pos % KV_BLOCK;
        if (KQ) {
            uint32_t pa[4][2];
            cp_async_wait_all_but(1);                      // K landed; V may still be in flight
            __syncwarp();
            expand_q8(kt, raw, lane);
            __syncwarp();
            if (new_row) {
                *reinterpret_cast<uint2*>(kt + r_new * K_STRIDE + lane * 4) =
                    *reinterpret_cast<const uint2*>(snew + lane * 4);
                __syncwarp();
            }
            attend_qk<NDT, true>(reinterpret_cast<const uint8_t*>(kt), reinterpret_cast<const uint16_t*>(sqa),
                                 n_pos, lane, st, pa);
            cp_async_wait_all();
            __syncwarp();                                  // every lane is done reading K
            expand_q8(kt, raw + KVQ_TILE, lane);
            __syncwarp();
            if (new_row) {
                *reinterpret_cast<uint2*>(kt + r_new * K_STRIDE + lane * 4) =
                    *reinterpret_cast<const uint2*>(snew + D + lane * 4);
                __syncwarp();
            }
            // the raw buffer is free: the next block's copies overlap this block's P V
            if (b + AWARPS < b1) staged = stage(b + AWARPS);
            attend_pv<NDT, true>(reinterpret_cast<const uint8_t*>(kt), 0, lane, st, pa);
            __syncwarp();      // the tile is rewritten by the next block's expansion
            continue;
        }
        // BF16: K and V landed as two groups (K first); the next block's K
        // copy overlaps this block's P V, its V copy the next block's scores
        uint32_t pa[4][2];
        cp_async_wait_all_but(1);                          // K landed
        __syncwarp();
        if (new_row) {
            *reinterpret_cast<uint2*>(kt + r_new * K_STRIDE + lane * 4) =
                *reinterpret_cast<const uint2*>(snew + lane * 4);
            __syncwarp();
        }
        attend_qk<NDT, false>(reinterpret_cast<const uint8_t*>(kt), reinterpret_cast<const uint16_t*>(sqa),
                              n_pos, lane, st, pa);
        __syncwarp();                                      // every lane is done reading K
        const bool next = stage_next_k(b + AWARPS);
        if (next) cp_async_wait_all_but(1);                // V landed (the next K may be in flight)
        else cp_async_wait_all();
        __syncwarp();
        if (new_row) {
            *reinterpret_cast<uint2*>(vt + r_new * K_STRIDE + lane * 4) =
                *reinterpret_cast<const uint2*>(snew + D + lane * 4);
            __syncwarp();
        }
        attend_pv<NDT, false>(reinterpret_cast<const uint8_t*>(vt), 0, lane, st, pa);
        __syncwarp();                                      // every lane is done reading V
        if (next) {
            stage_next_v(b + AWARPS);
            staged = true;
        }
    }
    cp_async_wait_all();
    __syncthreads();       // the K tiles become the warp-merge buffer

    // rows 2h and 2h + 1 of the accumulator hold the high and low parts of
    // head h (rows g and g + 8 of lane g = lane / 4): head h of this warp is
    // their sum, kept by the lanes of even g
    {
        const int g = lane >> 2, tig = lane & 3;
#pragma unroll
        for (int dt = 0; dt < NDT; ++dt)
#pragma unroll
            for (int e = 0; e < 4; ++e) st.o[dt][e] += __shfl_xor_sync(0xffffffffu, st.o[dt][e], 4);
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int h = half * 4 + (g >> 1);
            if ((g & 1) == 0 && h < G) {
                if (tig == 0) { s_m[warp * G + h] = st.m[half]; s_l[warp * G + h] = st.l[half]; }
#pragma unroll
                for (int dt = 0; dt < NDT; ++dt)
                    *reinterpret_cast<float2*>(s_o + (warp * G + h) * D + dt * 8 + 2 * tig) =
                        make_float2(st.o[dt][2 * half], st.o[dt][2 * half + 1]);
            }
        }
    }
    __syncthreads();

    // merge the warps in order; thread d owns output dimension d
    const int d = threadIdx.x;
    bool range_bad = false;
    float Mg[G], Lg[G], Og[G];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
        for (int w = 0; w < AWARPS; ++w) M = fmaxf(M, s_m[w * G + g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < AWARPS; ++w) {
                const float e = exp2f(s_m[w * G + g] - M);   // 0 for a warp with no block
                L = fmaf(s_l[w * G + g], e, L);
                O = fmaf(s_o[(w * G + g) * D + d], e, O);
            }
        }
        Mg[g] = M; Lg[g] = L; Og[g] = O;
    }
    const size_t row0 = (size_t)t * p.n_q + kvh * G;
    if (ns == 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float v = Og[g] / Lg[g];
            if (p.out_f16) reinterpret_cast<__half*>(p.out)[(row0 + g) * D + d] = to_f16(v, range_bad);
            else reinterpret_cast<float*>(p.out)[(row0 + g) * D + d] = v;
        }
    } else {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            p.part_o[((row0 + g) * p.n_splits + split) * D + d] = Og[g];
            if (d == 0) {
                p.part_ml[((row0 + g) * p.n_splits + split) * 2 + 0] = Mg[g];
                p.part_ml[((row0 + g) * p.n_splits + split) * 2 + 1] = Lg[g];
            }
        }
        // the last split CTA of this (row, KV head) merges its ns splits in order
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) s_ticket = atomicAdd(p.counters + (size_t)t * p.n_kv + kvh, 1);
        __syncthreads();
        if (s_ticket == ns - 1) {
            __threadfence();
            // split maxima and sums of all G heads, fetched in parallel; the
            // staging area is free (the warp merge above is done)
            float* s_ml = s_o + AWARPS * G * D;              // [G][n_splits][2]
            float* s_w = s_ml + 2 * G * p.n_splits;          // [G][n_splits]
            for (int i = threadIdx.x; i < G * ns; i += AWARPS * 32) {
                const int g = i / ns, sp = i % ns;
                const float* ml = p.part_ml + ((row0 + g) * p.n_splits + sp) * 2;
                s_ml[2 * (g * p.n_splits + sp)] = __ldcg(ml);
                s_ml[2 * (g * p.n_splits + sp) + 1] = __ldcg(ml + 1);
            }
            __syncthreads();
            if (threadIdx.x < G) {
                const int g = threadIdx.x;
                float M = -INFINITY;
                for (int sp = 0; sp < ns; ++sp) M = fmaxf(M, s_ml[2 * (g * p.n_splits + sp)]);
                float L = 0.f;
                for (int sp = 0; sp < ns; ++sp) {
                    const float ms = s_ml[2 * (g * p.n_splits + sp)];
                    const float e = ms == -INFINITY ? 0.f : exp2f(ms - M);
                    s_w[g * p.n_splits + sp] = e;
                    L = fmaf(s_ml[2 * (g * p.n_splits + sp) + 1], e, L);
                }
                s_m[g] = L;                                  // reuse: the merged denominator
            }
            __syncthreads();
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float* po = p.part_o + (row0 + g) * p.n_splits * D + d;
                float O = 0.f;
#pragma unroll 8
                for (int sp = 0; sp < ns; ++sp) O = fmaf(__ldcg(po + (size_t)sp * D), s_w[g * p.n_splits + sp], O);
                const float v = O / s_m[g];
                if (p.out_f16) reinterpret_cast<__half*>(p.out)[(row0 + g) * D + d] = to_f16(v, range_bad);
                else reinterpret_cast<float*>(p.out)[(row0 + g) * D + d] = v;
            }
            if (threadIdx.x == 0) p.counters[(size_t)t * p.n_kv + kvh] = 0;
        }
    }
    if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
}

template <int G, bool FUSED, bool KQ>
cudaError_t launch_g(const Launch& L, const AttnArgs& a)
{
    const size_t smem = AttnSmem<G, KQ>::total;
    static std::atomic<unsigned long long> attr_done{0};
    if (cudaError_t e = allow_smem_per_device(attn_kernel<G, FUSED, KQ>, (int)smem, attr_done)) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.n_splits, a.n_kv, a.T);
    cfg.blockDim = dim3(AWARPS * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, attn_kernel<G, FUSED, KQ>, a);
}

template <bool FUSED, bool KQ>
cudaError_t launch_fused(const Launch& L, const AttnArgs& a)
{
    switch (a.n_q / a.n_kv) {
    case 1: return launch_g<1, FUSED, KQ>(L, a);
    case 2: return launch_g<2, FUSED, KQ>(L, a);
    case 3: return launch_g<3, FUSED, KQ>(L, a);
    case 4: return launch_g<4, FUSED, KQ>(L, a);
    case 5: return launch_g<5, FUSED, KQ>(L, a);
    case 6: return launch_g<6, FUSED, KQ>(L, a);
    case 7: return launch_g<7, FUSED, KQ>(L, a);
    case 8: return launch_g<8, FUSED, KQ>(L, a);
    default: return cudaErrorInvalidValue;
    }
}

}  // namespace

#ifndef Q3_ATTN_BLOCKS_PER_WARP
#define Q3_ATTN_BLOCKS_PER_WARP 1
#endif
int attention_blocks_per_cta() { return Q3_ATTN_BLOCKS_PER_WARP * AWARPS; }

int attention_max_splits() { return 128; }

cudaError_t launch_attention(const Launch& L, const AttnArgs& a, bool fused)
{
    if (a.kvq_layer)
        return fused ? launch_fused<true, true>(L, a) : launch_fused<false, true>(L, a);
    return fused ? launch_fused<true, false>(L, a) : launch_fused<false, false>(L, a);
}

}  // namespace q3
