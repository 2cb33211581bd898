// k_gemv.cu -- HBM-streaming matrix-vector product for one-token rounds.
//
// A decode step of one session multiplies every projection and the lm_head
// by a single activation row ("Kipp Roadmap", status v0.0.4: the split-K
// decode matvec and its partial buffer; "Kipp Model Support", section
// "Quantization (Q8_0)": Q8_0 decode).  The work is a pure weight stream, so
// the kernel is shaped by HBM:
//  - each warp owns a segment of one weight row and has up to 8 16-byte
//    loads per lane of it in flight at once (8 bf16, or 16 int8 quants of
//    half a Q8_0 block, per load; non-allocating in L1); a longer segment
//    (K > 16384 at 8 warps per row) streams in further passes;
//  - the first segment's loads are issued before the programmatic-launch
//    wait, so they overlap the previous kernel's tail, and each next
//    segment's loads are issued before the current one is reduced;
//  - the grid is sized so every CTA handles the same number of row groups.
// The FP32 activation row is staged once per CTA in shared memory, RMS-
// normalised on the way in when a gain is given (the norm before QKV,
// gate/up and lm_head).  A row split over S warps of a CTA is summed in
// warp order, so results are deterministic.  Epilogues: store, residual add,
// SwiGLU of a gate/up row pair, and the greedy argmax of the lm_head.  Q8_0
// dequantisation happens in registers: fp16 scale times the block's int8
// dot product.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int CPL = 8;              // 16-byte loads per lane per row segment
constexpr int CTAS_PER_SM = 4;      // register budget of __launch_bounds__(THREADS, 4)

Q3_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

Q3_DEV float dot8_bf16(uint4 w, const float* h) {
    const float4 a = *reinterpret_cast<const float4*>(h);
    const float4 b = *reinterpret_cast<const float4*>(h + 4);
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

Q3_DEV float dot16_i8(uint4 q, const float* h) {
    const float4* hv = reinterpret_cast<const float4*>(h);
    float s = dot4_i8(q.x, hv[0]);
    s += dot4_i8(q.y, hv[1]);
    s += dot4_i8(q.z, hv[2]);
    s += dot4_i8(q.w, hv[3]);
    return s;
}

Q3_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

Q3_DEV bool better(float v, int i, float bv, int bi) { return v > bv || (v == bv && i < bi); }

// The weight row segment a warp streams for row group grp.
struct Seg {
    const uint4* row;       // 16-byte chunks of the row
    const __half* scales;   // Q8_0 scale row (else null)
    int c0, c1;             // chunk range
};

template <int SCHEME>
Q3_DEV Seg locate(const GemvArgs& p, int grp, int slot, int seg, int S, int R)
{
    int t, lr;
    if (p.pair) {
        t = slot & 1;                                  // 0: gate, 1: up
        lr = grp * (R / 2) + (slot >> 1);
    } else {
        lr = grp * R + slot;
        t = 0;
        if (lr >= p.rows[0]) { lr -= p.rows[0]; t = 1; }
        if (t == 1 && lr >= p.rows[1]) { lr -= p.rows[1]; t = 2; }
    }
    const void* w = t == 0 ? p.w[0] : (t == 1 ? p.w[1] : p.w[2]);
    const __half* sc = t == 0 ? p.scales[0] : (t == 1 ? p.scales[1] : p.scales[2]);
    constexpr int per_chunk = SCHEME == Q3_BF16 ? 8 : 16;
    const int nch = p.K / per_chunk;
    Seg s;
    s.row = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(w) +
                                           (size_t)lr * p.K * (SCHEME == Q3_BF16 ? 2 : 1));
    s.scales = SCHEME == Q3_BF16 ? nullptr : sc + (size_t)lr * (p.K / 32);
    s.c0 = seg * nch / S;
    s.c1 = (seg + 1) * nch / S;
    return s;
}

template <int SCHEME>
Q3_DEV void issue(const Seg& s, int lane, uint4 (&v)[CPL], float (&sc)[CPL])
{
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
        const int c = s.c0 + lane + 32 * u;
        if (c < s.c1) {
            v[u] = ldg_nc_v4(s.row + c);
            if (SCHEME != Q3_BF16) sc[u] = __half2float(s.scales[c >> 1]);
        }
    }
}

template <int SCHEME>
Q3_DEV float consume(const Seg& s, int lane, const uint4 (&v)[CPL], const float (&sc)[CPL],
                     const float* h)
{
    float acc = 0.f;
#pragma unroll
    for (int u = 0; u < CPL; ++u) {
        const int c = s.c0 + lane + 32 * u;
        if (c < s.c1) {
            if (SCHEME == Q3_BF16) acc += dot8_bf16(v[u], h + (size_t)c * 8);
            else acc = fmaf(sc[u], dot16_i8(v[u], h + (size_t)c * 16), acc);
        }
    }
    return acc;
}

template <int SCHEME>
__global__ void __launch_bounds__(THREADS, CTAS_PER_SM) gemv_kernel(const GemvArgs p)
{
    extern __shared__ float smem[];
    float* h = smem;                       // [K]
    float* red = smem + p.K;               // [WARPS]
    __shared__ float s_scale;
    __shared__ float s_bv[WARPS];
    __shared__ int s_bi[WARPS];
    __shared__ int s_ticket;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.warps_per_row;
    const int R = WARPS / S;               // row slots per group
    const int slot = warp / S, seg = warp % S;
    const int total_rows = p.rows[0] + (p.n_tensors > 1 ? p.rows[1] : 0) +
                           (p.n_tensors > 2 ? p.rows[2] : 0);
    const int n_groups = p.pair ? p.rows[0] / (R / 2) : total_rows / R;

    // Weights do not depend on earlier kernels: start streaming them first.
    uint4 v[CPL];
    float sc[CPL];
    int grp = blockIdx.x;
    Seg cur{};
    if (grp < n_groups) {
        cur = locate<SCHEME>(p, grp, slot, seg, S, R);
        issue<SCHEME>(cur, lane, v, sc);
    }
    if (threadIdx.x == 0) issue_l2_prefetch(p.next, blockIdx.x, gridDim.x);
    grid_dep_wait();

    // stage the activation row, RMS-normalised when a gain is given
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < p.K; i += THREADS * 4) {
        const float4 x = *reinterpret_cast<const float4*>(p.x + i);
        *reinterpret_cast<float4*>(h + i) = x;
        ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
    }
    if (p.norm_gain) {
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float t = 0.f;
            for (int w = 0; w < WARPS; ++w) t += red[w];
            s_scale = 1.0f / sqrtf(t / (float)p.K + p.eps);
        }
        __syncthreads();
        const float scl = s_scale;
        for (int i = threadIdx.x; i < p.K; i += THREADS)
            h[i] = h[i] * scl * __bfloat162float(p.norm_gain[i]);
    }
    __syncthreads();

    float best = -INFINITY;
    int best_i = 0x7fffffff;
    for (; grp < n_groups; grp += gridDim.x) {
        float acc = consume<SCHEME>(cur, lane, v, sc, h);
        // a segment longer than one pass (32 lanes x CPL loads) takes more passes
        for (Seg rest = cur; (rest.c0 += 32 * CPL) < rest.c1;) {
            issue<SCHEME>(rest, lane, v, sc);
            acc += consume<SCHEME>(rest, lane, v, sc, h);
        }
        const int nxt = grp + gridDim.x;
        if (nxt < n_groups) {                     // next segment's loads go out before the reduction
            cur = locate<SCHEME>(p, nxt, slot, seg, S, R);
            issue<SCHEME>(cur, lane, v, sc);
        }
        acc = warp_sum(acc);
        if (S == 1 && !p.pair) {
            if (lane == 0) {
                const int r = grp * R + slot;
                if (p.epi == EPI_ADD_F32) p.out[r] += acc;
                else p.out[r] = acc;
                if (better(acc, r, best, best_i)) { best = acc; best_i = r; }
            }
            continue;
        }
        if (lane == 0) red[warp] = acc;
        __syncthreads();
        if (p.pair) {
            if (threadIdx.x < R / 2) {
                float g = 0.f, u = 0.f;
                for (int s = 0; s < S; ++s) {
                    g += red[(2 * threadIdx.x) * S + s];
                    u += red[(2 * threadIdx.x + 1) * S + s];
                }
                p.out[grp * (R / 2) + threadIdx.x] = silu(g) * u;
            }
        } else if (threadIdx.x < R) {
            float a = 0.f;
            for (int s = 0; s < S; ++s) a += red[threadIdx.x * S + s];
            const int r = grp * R + threadIdx.x;
            if (p.epi == EPI_ADD_F32) p.out[r] += a;
            else p.out[r] = a;
            if (better(a, r, best, best_i)) { best = a; best_i = r; }
        }
        __syncthreads();
    }

    if (p.argmax_out) {
        // CTA partial, then the last CTA to finish merges all partials
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, best_i, o);
            if (better(ov, oi, best, best_i)) { best = ov; best_i = oi; }
        }
        if (lane == 0) { s_bv[warp] = best; s_bi[warp] = best_i; }
        __syncthreads();
        if (threadIdx.x == 0) {
            for (int w = 1; w < WARPS; ++w)
                if (better(s_bv[w], s_bi[w], s_bv[0], s_bi[0])) { s_bv[0] = s_bv[w]; s_bi[0] = s_bi[w]; }
            p.am_val[blockIdx.x] = s_bv[0];
            p.am_idx[blockIdx.x] = s_bi[0];
            __threadfence();
            s_ticket = atomicAdd(p.am_counter, 1);
        }
        __syncthreads();
        if (s_ticket == (int)gridDim.x - 1) {
            __threadfence();
            best = -INFINITY;
            best_i = 0x7fffffff;
            for (int b = threadIdx.x; b < (int)gridDim.x; b += THREADS) {
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
            __syncthreads();
            if (lane == 0) { s_bv[warp] = best; s_bi[warp] = best_i; }
            __syncthreads();
            if (threadIdx.x == 0) {
                for (int w = 1; w < WARPS; ++w)
                    if (better(s_bv[w], s_bi[w], s_bv[0], s_bi[0])) { s_bv[0] = s_bv[w]; s_bi[0] = s_bi[w]; }
                *p.argmax_out = s_bi[0] == 0x7fffffff ? 0 : s_bi[0];
                *p.am_counter = 0;
            }
        }
    }
    // the next kernel may be scheduled once every CTA is past its stream
    grid_dep_launch();
}

size_t gemv_smem(int K) { return (size_t)K * sizeof(float) + WARPS * sizeof(float); }

int ctas_per_sm(int K)
{
    const size_t smem = gemv_smem(K) + 1024;
    int n = (int)((220 * 1024) / smem);
    return n < 1 ? 1 : (n > CTAS_PER_SM ? CTAS_PER_SM : n);
}

}  // namespace

int gemv_warps_per_row(int rows, int K, int scheme, int pair)
{
    const int nch = K / (scheme == Q3_BF16 ? 8 : 16);
    int S = 1;
    while (S < WARPS && (nch + S - 1) / S > 32 * CPL) S *= 2;
    // split rows further while the machine would be under-filled
    const int C = 152 * ctas_per_sm(K);
    while (S < WARPS && (rows * S) / WARPS < C && nch / (2 * S) >= 64) S *= 2;
    if (pair && S > 4) S = 4;
    return S;
}

int gemv_max_grid() { return 152 * CTAS_PER_SM; }

cudaError_t launch_gemv(const Launch& L, int scheme, const GemvArgs& a)
{
    const int R = WARPS / a.warps_per_row;
    const int total = a.rows[0] + (a.n_tensors > 1 ? a.rows[1] : 0) + (a.n_tensors > 2 ? a.rows[2] : 0);
    const int n_groups = a.pair ? a.rows[0] / (R / 2) : total / R;
    const size_t smem = gemv_smem(a.K);
    // every CTA takes the same number of groups (the last round may be short)
    const int C = 152 * ctas_per_sm(a.K);
    const int iters = (n_groups + C - 1) / C;
    const int grid = (n_groups + iters - 1) / iters;
    auto kern = scheme == Q3_Q8_0 ? gemv_kernel<Q3_Q8_0> : gemv_kernel<Q3_BF16>;
    // the largest dynamic shared memory allowed so far, per device and scheme
    static std::mutex attr_mu;
    static size_t attr_set[64][2] = {};
    if (smem > 48 * 1024) {
        int dev = 0;
        if (cudaError_t e = cudaGetDevice(&dev)) return e;
        std::lock_guard<std::mutex> lock(attr_mu);
        size_t* have = (dev >= 0 && dev < 64) ? &attr_set[dev][scheme == Q3_Q8_0] : nullptr;
        if (!have || *have < smem) {
            cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 (int)smem);
            if (e != cudaSuccess) return e;
            if (have) *have = smem;
        }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(THREADS);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

}  // namespace q3
