// k_gemv.cu -- HBM-streaming matrix-vector product for one-token rounds.
//
// A decode step of one session multiplies every projection and the lm_head
// by a single activation row ("Kipp Roadmap", status v0.0.4: the split-K
// decode matvec and its partial buffer; "Kipp Model Support", section
// "Quantization (Q8_0)": Q8_0 decode).  The work is a pure weight stream, so
// the kernel is built around HBM: each warp reads weight rows with 16-byte
// non-allocating loads (8 bf16, or 16 int8 quants of a Q8_0 block half),
// UNROLL loads in flight per lane, and multiplies them against the FP32
// activation row staged once per CTA in shared memory, optionally RMS-
// normalised on the way in (the norm before QKV, gate/up and lm_head).
// A row may be split over up to 8 warps of the CTA (split-K); the partial
// sums meet in shared memory and are added in warp order, so results are
// deterministic.  Epilogues: store, residual add, and SwiGLU of a gate/up
// row pair.  Q8_0 dequantisation happens in registers: fp16 scale times the
// block's int8 dot product.
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int UNROLL = 4;

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
    float s = (float)(int8_t)(q & 0xff) * a.x;
    s = fmaf((float)(int8_t)((q >> 8) & 0xff), a.y, s);
    s = fmaf((float)(int8_t)((q >> 16) & 0xff), a.z, s);
    s = fmaf((float)(int8_t)(q >> 24), a.w, s);
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

// Weight row `lr` of tensor `t`, as seen by this warp.
template <int SCHEME>
Q3_DEV float row_dot(const GemvArgs& p, int t, int lr, int seg, int S, int lane, const float* h)
{
    float acc = 0.f;
    if (SCHEME == Q3_BF16) {
        const uint4* wrow = reinterpret_cast<const uint4*>(
            static_cast<const __nv_bfloat16*>(p.w[t]) + (size_t)lr * p.K);
        const int nch = p.K / 8;
        const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
        for (int c = c0 + lane; c < c1; c += 32 * UNROLL) {
            uint4 v[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                if (c + 32 * u < c1) v[u] = ldg_nc_v4(wrow + c + 32 * u);
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                if (c + 32 * u < c1) acc += dot8_bf16(v[u], h + (size_t)(c + 32 * u) * 8);
        }
    } else {
        const uint4* qrow = reinterpret_cast<const uint4*>(
            static_cast<const int8_t*>(p.w[t]) + (size_t)lr * p.K);
        const __half* srow = p.scales[t] + (size_t)lr * (p.K / 32);
        const int nch = p.K / 16;
        const int c0 = seg * nch / S, c1 = (seg + 1) * nch / S;
        for (int c = c0 + lane; c < c1; c += 32 * UNROLL) {
            uint4 v[UNROLL];
            float sc[UNROLL];
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                if (c + 32 * u < c1) {
                    v[u] = ldg_nc_v4(qrow + c + 32 * u);
                    sc[u] = __half2float(srow[(c + 32 * u) >> 1]);
                }
#pragma unroll
            for (int u = 0; u < UNROLL; ++u)
                if (c + 32 * u < c1)
                    acc = fmaf(sc[u], dot16_i8(v[u], h + (size_t)(c + 32 * u) * 16), acc);
        }
    }
    return warp_sum(acc);
}

template <int SCHEME>
__global__ void __launch_bounds__(THREADS) gemv_kernel(const GemvArgs p)
{
    extern __shared__ float smem[];
    float* h = smem;                       // [K]
    float* red = smem + p.K;               // [WARPS]
    __shared__ float s_scale;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.warps_per_row;
    const int R = WARPS / S;               // row slots per group
    const int slot = warp / S, seg = warp % S;
    const int total_rows = p.rows[0] + (p.n_tensors > 1 ? p.rows[1] : 0) +
                           (p.n_tensors > 2 ? p.rows[2] : 0);
    const int n_groups = p.pair ? p.rows[0] / (R / 2) : total_rows / R;

    grid_dep_wait();

    // stage the activation row, RMS-normalised when a gain is given
    float ss = 0.f;
    for (int i = threadIdx.x * 4; i < p.K; i += THREADS * 4) {
        const float4 v = *reinterpret_cast<const float4*>(p.x + i);
        *reinterpret_cast<float4*>(h + i) = v;
        ss += v.x * v.x + v.y * v.y + v.z * v.z + v.w * v.w;
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
        const float sc = s_scale;
        for (int i = threadIdx.x; i < p.K; i += THREADS)
            h[i] = h[i] * sc * __bfloat162float(p.norm_gain[i]);
    }
    __syncthreads();

    for (int grp = blockIdx.x; grp < n_groups; grp += gridDim.x) {
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
        const float v = row_dot<SCHEME>(p, t, lr, seg, S, lane, h);
        if (S == 1 && !p.pair) {
            if (lane == 0) {
                const int r = grp * R + slot;
                if (p.epi == EPI_ADD_F32) p.out[r] += v;
                else p.out[r] = v;
            }
            continue;
        }
        if (lane == 0) red[warp] = v;
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
            float acc = 0.f;
            for (int s = 0; s < S; ++s) acc += red[threadIdx.x * S + s];
            const int r = grp * R + threadIdx.x;
            if (p.epi == EPI_ADD_F32) p.out[r] += acc;
            else p.out[r] = acc;
        }
        __syncthreads();
    }
    grid_dep_launch();
}

}  // namespace

int gemv_warps_per_row(int rows, int K)
{
    // enough row groups to cover every SM several times; a row never splits
    // below 1024 elements per warp
    int S = 1;
    while (S < WARPS && (rows * S) / WARPS < 152 * 6 && K / (2 * S) >= 1024) S *= 2;
    return S;
}

cudaError_t launch_gemv(const Launch& L, int scheme, const GemvArgs& a)
{
    const int R = WARPS / a.warps_per_row;
    const int total = a.rows[0] + (a.n_tensors > 1 ? a.rows[1] : 0) + (a.n_tensors > 2 ? a.rows[2] : 0);
    const int n_groups = a.pair ? a.rows[0] / (R / 2) : total / R;
    const size_t smem = (size_t)a.K * sizeof(float) + WARPS * sizeof(float);
    int per_sm = (int)((200 * 1024) / (smem + 1024));
    if (per_sm > 2048 / THREADS) per_sm = 2048 / THREADS;
    if (per_sm < 1) per_sm = 1;
    int grid = n_groups < 152 * per_sm ? n_groups : 152 * per_sm;
    auto kern = scheme == Q3_Q8_0 ? gemv_kernel<Q3_Q8_0> : gemv_kernel<Q3_BF16>;
    static size_t attr_set[2] = {0, 0};
    if (smem > 48 * 1024 && attr_set[scheme] < smem) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
        attr_set[scheme] = smem;
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
