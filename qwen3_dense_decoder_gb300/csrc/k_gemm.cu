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
// Roles in a 128-thread CTA: warp 0 lane 0 issues TMA loads, warp 1 lane 0
// issues tcgen05.mma and owns the TMEM allocation, and all four warps drain
// the accumulator (warp w reads TMEM lanes 32w..32w+31) through the fused
// epilogue: plain store, residual add, or SwiGLU of a paired gate/up tile.
// Split-K writes FP32 partials that gemm_splitk_reduce sums in split order.
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
    // as many stages as fit in ~200 KB, at most 8
    static constexpr int STAGES_RAW = (200 * 1024) / STAGE_BYTES;
    static constexpr int STAGES = STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr uint32_t TMEM_COLS = BN < 32 ? 32 : BN;
    static constexpr int SMEM = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

Q3_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

template <int BN>
__global__ void __launch_bounds__(128, 1)
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
    uint64_t* full = reinterpret_cast<uint64_t*>(sb + STAGES * C::B_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* accum = empty + STAGES;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(accum + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int n_tiles = (p.N + BN - 1) / BN;
    const int m_tiles = p.M / BM;
    int bid = blockIdx.x;
    const int nt = bid % n_tiles;
    bid /= n_tiles;
    const int mt = bid % m_tiles;
    const int split = bid / m_tiles;
    const int kb_total = p.K / BK;
    const int kb0 = split * kb_total / p.k_splits;
    const int kb1 = (split + 1) * kb_total / p.k_splits;
    const int nkb = kb1 - kb0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(accum, 1);
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

    // The token rows (B) are written by the previous kernel.
    grid_dep_wait();

    if (warp == 0 && lane == 0) {
        // ---------------- TMA producer
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            const uint32_t use = i / STAGES;
            if (i >= STAGES && !mbar_wait(&empty[s], (use & 1) ^ 1, p.status)) break;
            mbar_arrive_expect_tx(&full[s], C::STAGE_BYTES);
            const int kc = (kb0 + i) * BK;
            uint8_t* a_dst = sa + s * A_BYTES;
            if (p.pair) {
                tma_load_2d(a_dst, &ta0, &full[s], kc, mt * 64);
                tma_load_2d(a_dst + A_BYTES / 2, &ta1, &full[s], kc, mt * 64);
            } else if (mt < p.a_tiles0) {
                tma_load_2d(a_dst, &ta0, &full[s], kc, mt * BM);
            } else if (mt < p.a_tiles1) {
                tma_load_2d(a_dst, &ta1, &full[s], kc, (mt - p.a_tiles0) * BM);
            } else {
                tma_load_2d(a_dst, &ta2, &full[s], kc, (mt - p.a_tiles1) * BM);
            }
            tma_load_2d(sb + s * C::B_BYTES, &tb, &full[s], kc, nt * BN);
        }
    } else if (warp == 1 && lane == 0) {
        // ---------------- MMA issuer
        constexpr uint32_t idesc = idesc_f16_f32(BM, BN);
        for (int i = 0; i < nkb; ++i) {
            const int s = i % STAGES;
            const uint32_t use = i / STAGES;
            if (!mbar_wait(&full[s], use & 1, p.status)) break;
            tc_fence_after();
            const uint32_t a_base = smem_u32(sa + s * A_BYTES);
            const uint32_t b_base = smem_u32(sb + s * C::B_BYTES);
#pragma unroll
            for (int k = 0; k < BK / 16; ++k) {
                // advancing 16 elements (32 bytes) along K inside the swizzle row
                tc_mma_f16(tmem, smem_desc_sw128(a_base + k * 32), smem_desc_sw128(b_base + k * 32),
                           idesc, (i > 0 || k > 0) ? 1u : 0u);
            }
            tc_commit(&empty[s]);
        }
        tc_commit(accum);
    }
    __syncwarp();

    // The next kernel may start its prologue while this epilogue drains.
    grid_dep_launch();

    // ---------------- epilogue: all four warps
    // CTA-uniform: a failed (timed-out) wait anywhere skips every TMEM read
    const bool have = __syncthreads_and(mbar_wait(accum, 0, p.status)) != 0;
    tc_fence_after();
    const int row = warp * 32 + lane;                      // D row = TMEM lane
    const uint32_t t_row = tmem + ((uint32_t)(warp * 32) << 16);
    float* xch = reinterpret_cast<float*>(smem);           // SwiGLU exchange (ring is idle now)
    const bool swiglu = (p.epi == EPI_SWIGLU_F16 || p.epi == EPI_SWIGLU_F32) && p.k_splits == 1;
    bool range_bad = false;

#pragma unroll 1
    for (int c = 0; c < BN / 32; ++c) {
        if (!have) break;
        uint32_t r[32];
        tmem_ld_32x32b_x32(t_row + c * 32, r);
        tmem_ld_wait();
        const int n0 = nt * BN + c * 32;
        if (p.k_splits > 1) {
            float* ws = p.ws + (size_t)split * p.N * p.M;
            const int m = mt * BM + row;
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (n0 + j < p.N) ws[(size_t)(n0 + j) * p.M + m] = __uint_as_float(r[j]);
        } else if (swiglu) {
            // rows 64..127 hold the up projection of the features of rows 0..63
            if (warp >= 2) {
#pragma unroll
                for (int j = 0; j < 32; ++j) xch[j * 64 + (row - 64)] = __uint_as_float(r[j]);
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
            if (warp < 2) {
                const int f = mt * 64 + row;
#pragma unroll
                for (int j = 0; j < 32; ++j) {
                    if (n0 + j < p.N) {
                        const float g = __uint_as_float(r[j]);
                        const float v = silu(g) * xch[j * 64 + row];
                        if (p.epi == EPI_SWIGLU_F16)
                            reinterpret_cast<__half*>(p.out)[(size_t)(n0 + j) * p.ldo + f] =
                                to_f16(v, range_bad);
                        else
                            reinterpret_cast<float*>(p.out)[(size_t)(n0 + j) * p.ldo + f] = v;
                    }
                }
            }
            asm volatile("bar.sync 1, 128;" ::: "memory");
        } else {
            const int m = mt * BM + row;
#pragma unroll
            for (int j = 0; j < 32; ++j) {
                if (n0 + j < p.N) {
                    const size_t o = (size_t)(n0 + j) * p.ldo + m;
                    const float v = __uint_as_float(r[j]);
                    if (p.epi == EPI_STORE_F32)
                        reinterpret_cast<float*>(p.out)[o] = v;
                    else if (p.epi == EPI_ADD_F32)
                        reinterpret_cast<float*>(p.out)[o] += v;
                    else
                        reinterpret_cast<__half*>(p.out)[o] = to_f16(v, range_bad);
                }
            }
        }
    }

    if (range_bad) set_status(p.status, Q3_STATUS_F16_RANGE);
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

template <int BN>
cudaError_t launch_bn(const Launch& L, const CUtensorMap& a0, const CUtensorMap& a1,
                      const CUtensorMap& a2, const CUtensorMap& b, const GemmArgs& g)
{
    using C = GemmCfg<BN>;
    static bool attr_done = false;
    if (!attr_done) {
        cudaError_t e = cudaFuncSetAttribute(gemm_tc_kernel<BN>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM);
        if (e != cudaSuccess) return e;
        attr_done = true;
    }
    const int n_tiles = (g.N + BN - 1) / BN;
    const int grid = n_tiles * (g.M / BM) * g.k_splits;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(128);
    cfg.dynamicSmemBytes = C::SMEM;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, gemm_tc_kernel<BN>, a0, a1, a2, b, g);
}

}  // namespace

int gemm_block_n(int N)
{
    if (N <= 32) return 32;
    if (N <= 64) return 64;
    if (N <= 128) return 128;
    return 256;
}

cudaError_t launch_gemm(const Launch& L, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& a2, const CUtensorMap& b, int bn, const GemmArgs& g)
{
    switch (bn) {
    case 32: return launch_bn<32>(L, a0, a1, a2, b, g);
    case 64: return launch_bn<64>(L, a0, a1, a2, b, g);
    case 128: return launch_bn<128>(L, a0, a1, a2, b, g);
    case 256: return launch_bn<256>(L, a0, a1, a2, b, g);
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

}  // namespace q3
