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
// each K/V block once.  The split covers a contiguous range of logical
// blocks whose bounds depend only on the context length, never on which
// physical blocks back it, so paged and contiguous layouts give identical
// bits.  Within a block, lane j scores position j; the values are then
// accumulated with each lane owning 4 of the 128 output dimensions.  Warps
// of the CTA take blocks round-robin and are merged in warp order; splits
// are merged by attn_combine in split order.
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int KV_BLOCK = 32;
constexpr int AWARPS = 4;

Q3_DEV float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}
Q3_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

template <int G>
__global__ void __launch_bounds__(AWARPS * 32) attn_split_kernel(const AttnArgs p)
{
    __shared__ __align__(16) float sq[G][D];
    __shared__ float s_m[AWARPS][G], s_l[AWARPS][G];
    __shared__ __align__(16) float s_o[AWARPS][G][D];

    const int split = blockIdx.x, kvh = blockIdx.y, t = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    grid_dep_wait();

    const int ctx = p.row_pos[t] + 1;
    const int slot = p.row_slot[t];
    const int nblk = (ctx + KV_BLOCK - 1) / KV_BLOCK;
    const int bps = (nblk + p.n_splits - 1) / p.n_splits;
    const int b0 = split * bps;
    const int b1 = min(b0 + bps, nblk);

    // q of the G heads, scaled by log2(e) / sqrt(128)
    const float qscale = 1.4426950408889634f * 0.08838834764831845f;
    for (int i = threadIdx.x; i < G * D; i += AWARPS * 32)
        sq[i / D][i % D] = p.q[((size_t)t * p.n_q + kvh * G + i / D) * D + i % D] * qscale;
    __syncthreads();

    float m[G], l[G], o[G][4];
#pragma unroll
    for (int g = 0; g < G; ++g) {
        m[g] = -INFINITY;
        l[g] = 0.f;
        o[g][0] = o[g][1] = o[g][2] = o[g][3] = 0.f;
    }

    const int* table = p.tables + (size_t)slot * p.max_blocks;
    const size_t head_elems = (size_t)KV_BLOCK * D;
    for (int b = b0 + warp; b < b1; b += AWARPS) {
        const int phys = table[b];
        if (phys < 0 || phys >= p.n_blocks) {
            if (lane == 0) set_status(p.status, Q3_STATUS_BLOCK_RANGE);
            continue;
        }
        const __nv_bfloat16* Kb = p.kv_layer + ((size_t)phys * 2 * p.n_kv + kvh) * head_elems;
        const __nv_bfloat16* Vb = Kb + (size_t)p.n_kv * head_elems;
        const bool valid = b * KV_BLOCK + lane < ctx;

        // scores: lane j <- position b*32 + j
        float s[G];
#pragma unroll
        for (int g = 0; g < G; ++g) s[g] = 0.f;
        const uint4* krow = reinterpret_cast<const uint4*>(Kb + (size_t)lane * D);
#pragma unroll 4
        for (int c = 0; c < D / 8; ++c) {
            const uint4 kw = __ldg(krow + c);
            const float k8[8] = {bf16lo(kw.x), bf16hi(kw.x), bf16lo(kw.y), bf16hi(kw.y),
                                 bf16lo(kw.z), bf16hi(kw.z), bf16lo(kw.w), bf16hi(kw.w)};
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float4 qa = *reinterpret_cast<const float4*>(&sq[g][c * 8]);
                const float4 qb = *reinterpret_cast<const float4*>(&sq[g][c * 8 + 4]);
                s[g] = fmaf(k8[0], qa.x, s[g]);
                s[g] = fmaf(k8[1], qa.y, s[g]);
                s[g] = fmaf(k8[2], qa.z, s[g]);
                s[g] = fmaf(k8[3], qa.w, s[g]);
                s[g] = fmaf(k8[4], qb.x, s[g]);
                s[g] = fmaf(k8[5], qb.y, s[g]);
                s[g] = fmaf(k8[6], qb.z, s[g]);
                s[g] = fmaf(k8[7], qb.w, s[g]);
            }
        }
        float pr[G];
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float sg = valid ? s[g] : -INFINITY;
            const float m_new = fmaxf(m[g], warp_max(sg));
            const float alpha = exp2f(m[g] - m_new);      // 0 on the first block (m = -inf)
            pr[g] = valid ? exp2f(sg - m_new) : 0.f;
            l[g] = l[g] * alpha + warp_sum(pr[g]);
            o[g][0] *= alpha; o[g][1] *= alpha; o[g][2] *= alpha; o[g][3] *= alpha;
            m[g] = m_new;
        }
        // values: lane owns dims [4 lane, 4 lane + 4)
        const int nvalid = min(KV_BLOCK, ctx - b * KV_BLOCK);
        for (int j = 0; j < nvalid; ++j) {
            const uint2 vw = __ldg(reinterpret_cast<const uint2*>(Vb + (size_t)j * D) + lane);
            const float v0 = bf16lo(vw.x), v1 = bf16hi(vw.x), v2 = bf16lo(vw.y), v3 = bf16hi(vw.y);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float pj = __shfl_sync(0xffffffffu, pr[g], j);
                o[g][0] = fmaf(pj, v0, o[g][0]);
                o[g][1] = fmaf(pj, v1, o[g][1]);
                o[g][2] = fmaf(pj, v2, o[g][2]);
                o[g][3] = fmaf(pj, v3, o[g][3]);
            }
        }
    }

#pragma unroll
    for (int g = 0; g < G; ++g) {
        if (lane == 0) { s_m[warp][g] = m[g]; s_l[warp][g] = l[g]; }
        *reinterpret_cast<float4*>(&s_o[warp][g][lane * 4]) = make_float4(o[g][0], o[g][1], o[g][2], o[g][3]);
    }
    __syncthreads();

    // merge the warps in order; thread d owns output dimension d
    const int d = threadIdx.x;
    bool range_bad = false;
    for (int g = 0; g < G; ++g) {
        float M = -INFINITY;
        for (int w = 0; w < AWARPS; ++w) M = fmaxf(M, s_m[w][g]);
        float L = 0.f, O = 0.f;
        if (M != -INFINITY) {
            for (int w = 0; w < AWARPS; ++w) {
                const float e = exp2f(s_m[w][g] - M);   // 0 for a warp with no block
                L = fmaf(s_l[w][g], e, L);
                O = fmaf(s_o[w][g][d], e, O);
            }
        }
        const int hq = kvh * G + g;
        const size_t row = (size_t)t * p.n_q + hq;
        if (p.n_splits == 1) {
            const float v = O / L;
            if (p.out_f16) reinterpret_cast<__half*>(p.out)[row * D + d] = to_f16(v, range_bad);
            else reinterpret_cast<float*>(p.out)[row * D + d] = v;
        } else {
            p.part_o[(row * p.n_splits + split) * D + d] = O;
            if (d == 0) {
                p.part_ml[(row * p.n_splits + split) * 2 + 0] = M;
                p.part_ml[(row * p.n_splits + split) * 2 + 1] = L;
            }
        }
    }
    if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
    grid_dep_launch();
}

// Merge split partials in split order: o = sum_s O_s 2^(m_s - M) / sum_s l_s 2^(m_s - M).
__global__ void __launch_bounds__(D) attn_combine_kernel(const AttnArgs p)
{
    grid_dep_wait();
    const size_t row = blockIdx.x;        // t * n_q + head
    const int d = threadIdx.x;
    const float* ml = p.part_ml + row * p.n_splits * 2;
    float M = -INFINITY;
    for (int s = 0; s < p.n_splits; ++s) M = fmaxf(M, ml[2 * s]);
    float L = 0.f, O = 0.f;
    for (int s = 0; s < p.n_splits; ++s) {
        const float e = ml[2 * s] == -INFINITY ? 0.f : exp2f(ml[2 * s] - M);
        L = fmaf(ml[2 * s + 1], e, L);
        O = fmaf(p.part_o[(row * p.n_splits + s) * D + d], e, O);
    }
    const float v = O / L;
    bool range_bad = false;
    if (p.out_f16) reinterpret_cast<__half*>(p.out)[row * D + d] = to_f16(v, range_bad);
    else reinterpret_cast<float*>(p.out)[row * D + d] = v;
    if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
    grid_dep_launch();
}

template <typename K, typename A>
cudaError_t launch_ex(const Launch& L, K kern, dim3 grid, dim3 block, const A& args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, kern, args);
}

}  // namespace

cudaError_t launch_attention(const Launch& L, const AttnArgs& a)
{
    const int G = a.n_q / a.n_kv;
    const dim3 grid(a.n_splits, a.n_kv, a.T), block(AWARPS * 32);
    cudaError_t e;
    switch (G) {
    case 1: e = launch_ex(L, attn_split_kernel<1>, grid, block, a); break;
    case 2: e = launch_ex(L, attn_split_kernel<2>, grid, block, a); break;
    case 3: e = launch_ex(L, attn_split_kernel<3>, grid, block, a); break;
    case 4: e = launch_ex(L, attn_split_kernel<4>, grid, block, a); break;
    case 5: e = launch_ex(L, attn_split_kernel<5>, grid, block, a); break;
    case 6: e = launch_ex(L, attn_split_kernel<6>, grid, block, a); break;
    case 7: e = launch_ex(L, attn_split_kernel<7>, grid, block, a); break;
    case 8: e = launch_ex(L, attn_split_kernel<8>, grid, block, a); break;
    default: return cudaErrorInvalidValue;
    }
    if (e != cudaSuccess || a.n_splits == 1) return e;
    return launch_ex(L, attn_combine_kernel, dim3(a.T * a.n_q), dim3(D), a);
}

}  // namespace q3
