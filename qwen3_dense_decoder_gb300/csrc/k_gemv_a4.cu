// k_gemv_a4.cu -- one-token matvec over AFFINE4_GS32 weights at 5.0 bits a
// weight ("Kipp Model Support", section "Quantization (AFFINE4_GS32)": 32
// weights a group, 4-bit codes, an fp16 scale and an fp16 bias; "Kipp
// Roadmap", "Delivered since": dedicated affine4 decode paths).
//
// A decode step streams every weight once, so the kernel reads the format's
// bytes and nothing more: 16 bytes of codes and 4 bytes of (scale, bias) per
// group.  At the HBM rate an SM must retire about 34 weights a cycle, so the
// work per weight has to stay well under the SM's issue budget.  The
// products run on mma.sync m16n8k16 (fp16 in, FP32 accumulate):
//  - B (16 x 8) is eight weight rows by 16 codes.  A lane's four fp16 pairs
//    come from one 32-bit word of the derived code plane:
//    (w >> 4j) & 0x000F000F | 0x64006400 is the pair 1024 + q, one HSUB2
//    leaves q exactly, and one HFMA2 with the row's (scale, bias) gives the
//    weight fp16(scale * q + bias) rounded once -- the same values as the
//    fp16 copy the tensor-core path of wider rounds reads;
//  - A (16 x 16) holds the activation rounded to fp16 in row 0 (rows 1..15
//    zero), so row 0 of D accumulates y over the whole K segment with no
//    per-group work at all.
// The derived planes (built once at model creation from the 20-byte groups)
// are lane-major so every load is a coalesced vector:
//  - codes: [rows / 8][K / 128][32 lanes][4 groups] 32-bit words; lane
//    (n = lane / 4, t = lane % 4) holds row n's codes at k = 2t, 2t + 1,
//    2t + 8, 2t + 9, 16 + 2t, 17 + 2t, 24 + 2t, 25 + 2t of the group: fp16
//    pair j low halves in bits 4j .. 4j + 3, high halves in bits 16 + 4j ..;
//  - (scale, bias): [rows / 8][K / 128][8 rows][4 groups] fp16 pairs; lane
//    (n, t) loads row n's 16 bytes (the four lanes of a row share them).
// Rows of one output are split over S warps of a CTA and summed in warp
// order; epilogues as the BF16 matvec (store, residual add, SwiGLU pairs).
#include <mutex>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int THREADS = 256;
constexpr int WARPS = THREADS / 32;
constexpr int CTAS_PER_SM = 3;
constexpr int BPL = 2;              // 4-group blocks a warp keeps in flight

Q3_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

Q3_DEV float silu(float g) { return g / (1.0f + expf(-g)); }

Q3_DEV void mma_f16(float (&d)[4], uint32_t a0, uint32_t a2, uint32_t b0, uint32_t b1) {
    // rows 8..15 of A are zero (a1 = a3 = 0)
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                 "{%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
                 : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
}

// fp16 pair j of a code word as weights: fp16(scale * q + bias), one rounding
Q3_DEV uint32_t weight_pair(uint32_t w, int j, __half2 sc, __half2 bi) {
    const uint32_t v = ((w >> (4 * j)) & 0x000F000Fu) | 0x64006400u;
    const __half2 q = __hsub2(*reinterpret_cast<const __half2*>(&v), __half2half2(__ushort_as_half(0x6400)));
    const __half2 h = __hfma2(q, sc, bi);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// A unit is one 8-row tile of one tensor; tile index -> (tensor, row tile)
struct A4Tile {
    const uint4* codes;     // the tile's code blocks [K/128][32 lanes] uint4
    const uint4* sb;        // the tile's (scale, bias) blocks [K/128][8 rows] uint4
};

Q3_DEV A4Tile locate_a4(const GemvArgs& p, int tile) {
    int t = 0;
    if (p.pair) {
        t = tile & 1;
        tile >>= 1;
    } else {
        if (tile >= p.rows[0] / 8) { tile -= p.rows[0] / 8; t = 1; }
        if (t == 1 && tile >= p.rows[1] / 8) { tile -= p.rows[1] / 8; t = 2; }
    }
    const size_t nb = (size_t)p.K / 128;
    A4Tile a;
    a.codes = static_cast<const uint4*>(p.w[t]) + (size_t)tile * nb * 32;
    a.sb = reinterpret_cast<const uint4*>(p.scales[t]) + (size_t)tile * nb * 8;
    return a;
}

__global__ void __launch_bounds__(THREADS, CTAS_PER_SM) gemv_a4_kernel(const GemvArgs p)
{
    extern __shared__ __align__(16) uint8_t smem[];
    const int G = p.K / 32;
    uint2* xf = reinterpret_cast<uint2*>(smem);                       // [G][2 ksteps][4 t]
    float* red = reinterpret_cast<float*>(xf + (size_t)G * 8);        // [WARPS][8] row partials
    __shared__ float s_scale;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int S = p.warps_per_row;
    const int R = WARPS / S;                     // tiles per unit
    const int slot = warp / S, seg = warp % S;
    const int n_tiles = p.pair ? 2 * (p.rows[0] / 8)
                               : (p.rows[0] + (p.n_tensors > 1 ? p.rows[1] : 0) +
                                  (p.n_tensors > 2 ? p.rows[2] : 0)) / 8;
    const int n_units = n_tiles / R;
    const int nb = p.K / 128;
    const int b0 = seg * nb / S, b1 = (seg + 1) * nb / S;
    const int t = lane & 3, n = lane >> 2;

    // Slot u of the in-flight ring holds block b0 + u + k BPL of the current
    // unit; a slot consumed at block b reloads block b + BPL, or, past the
    // segment, block b0 + u of the next unit, which is where that unit's
    // loop expects it.
    int unit = blockIdx.x;
    uint4 cw[BPL], sbw[BPL];
    auto load = [&](const A4Tile& a, int b, int u) {
        cw[u] = ldg_nc_v4(a.codes + (size_t)b * 32 + lane);
        sbw[u] = ldg_nc_v4(a.sb + (size_t)b * 8 + n);
    };
    A4Tile cur{};
    if (unit < n_units) {
        cur = locate_a4(p, unit * R + slot);
#pragma unroll
        for (int u = 0; u < BPL; ++u)
            if (b0 + u < b1) load(cur, b0 + u, u);
    }
    if (threadIdx.x == 0) issue_l2_prefetch(p.next, blockIdx.x, gridDim.x);
    grid_dep_wait();

    // the activation (RMS-normalised when a gain is given), rounded to fp16,
    // in the A-fragment order: entry (g, kstep j, t) holds the values at
    // k = 32 g + 16 j + {2t, 2t + 1} and {+8, +9}
    float scl = 1.0f;
    if (p.norm_gain) {
        float ss = 0.f;
        for (int i = threadIdx.x * 4; i < p.K; i += THREADS * 4) {
            const float4 x = *reinterpret_cast<const float4*>(p.x + i);
            ss += x.x * x.x + x.y * x.y + x.z * x.z + x.w * x.w;
        }
        ss = warp_sum(ss);
        if (lane == 0) red[warp] = ss;
        __syncthreads();
        if (threadIdx.x == 0) {
            float tot = 0.f;
            for (int w = 0; w < WARPS; ++w) tot += red[w];
            s_scale = 1.0f / sqrtf(tot / (float)p.K + p.eps);
        }
        __syncthreads();
        scl = s_scale;
    }
    {
        uint32_t* xw = reinterpret_cast<uint32_t*>(xf);
        bool bad = false;
        for (int k = threadIdx.x * 4; k < p.K; k += THREADS * 4) {
            float4 x = *reinterpret_cast<const float4*>(p.x + k);
            if (p.norm_gain) {
                const uint2 gg = *reinterpret_cast<const uint2*>(p.norm_gain + k);
                x.x = x.x * scl * bf16lo(gg.x);
                x.y = x.y * scl * bf16hi(gg.x);
                x.z = x.z * scl * bf16lo(gg.y);
                x.w = x.w * scl * bf16hi(gg.y);
            }
            bad |= fabsf(x.x) > 65504.f || fabsf(x.y) > 65504.f || fabsf(x.z) > 65504.f || fabsf(x.w) > 65504.f;
            // value k = 32 g + 16 j + r: pair (r & 7) / 2 of k step j, half r / 8 of the entry
            const int g = k >> 5, j = (k >> 4) & 1, r = k & 15;
            const int tt = (r & 7) >> 1, e = r >> 3;
            const __half2 h0 = __floats2half2_rn(x.x, x.y), h1 = __floats2half2_rn(x.z, x.w);
            const int base = (g * 2 + j) * 4 + tt;
            xw[base * 2 + e] = *reinterpret_cast<const uint32_t*>(&h0);
            xw[(base + 1) * 2 + e] = *reinterpret_cast<const uint32_t*>(&h1);
        }
        if (bad) set_status(p.status, Q3_STATUS_F16_RANGE);
    }
    __syncthreads();

    for (; unit < n_units; unit += gridDim.x) {
        const bool more = unit + (int)gridDim.x < n_units;
        const A4Tile nxt = more ? locate_a4(p, (unit + gridDim.x) * R + slot) : cur;
        float d[4] = {0.f, 0.f, 0.f, 0.f};       // row 0 of D: lanes 0..3 hold rows 2t, 2t + 1
        for (int blk0 = b0; blk0 < b1; blk0 += BPL) {
#pragma unroll
            for (int u = 0; u < BPL; ++u) {
                const int b = blk0 + u;
                if (b >= b1) break;
                const uint4 c = cw[u], sv = sbw[u];
                if (b + BPL < b1) load(cur, b + BPL, u);
                else if (more) load(nxt, b0 + u, u);
                const uint32_t wq[4] = {c.x, c.y, c.z, c.w};
                const uint32_t sq[4] = {sv.x, sv.y, sv.z, sv.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int g = b * 4 + q;
                    const __half2 sb2 = *reinterpret_cast<const __half2*>(&sq[q]);
                    const __half2 sc = __low2half2(sb2), bi = __high2half2(sb2);
#pragma unroll
                    for (int j = 0; j < 2; ++j) {
                        uint2 a = make_uint2(0u, 0u);
                        if (lane < 4) a = xf[(g * 2 + j) * 4 + t];
                        mma_f16(d, a.x, a.y, weight_pair(wq[q], 2 * j, sc, bi),
                                weight_pair(wq[q], 2 * j + 1, sc, bi));
                    }
                }
            }
        }
        // rows of the tile: lane t (< 4) holds rows 2t, 2t + 1; warps of a tile sum in order
        if (lane < 4) {
            red[warp * 8 + 2 * t] = d[0];
            red[warp * 8 + 2 * t + 1] = d[1];
        }
        __syncthreads();
        const int tile0 = unit * R;
        if (p.pair) {
            // slots 2i (gate) and 2i + 1 (up) cover the same rows
            for (int i = threadIdx.x; i < (R / 2) * 8; i += THREADS) {
                const int pr = i >> 3, r = i & 7;
                float gv = 0.f, uv = 0.f;
                for (int s2 = 0; s2 < S; ++s2) {
                    gv += red[((2 * pr) * S + s2) * 8 + r];
                    uv += red[((2 * pr + 1) * S + s2) * 8 + r];
                }
                p.out[((tile0 >> 1) + pr) * 8 + r] = silu(gv) * uv;
            }
        } else {
            for (int i = threadIdx.x; i < R * 8; i += THREADS) {
                const int sl = i >> 3, r = i & 7;
                float a = 0.f;
                for (int s2 = 0; s2 < S; ++s2) a += red[(sl * S + s2) * 8 + r];
                const int row = (tile0 + sl) * 8 + r;
                if (p.epi == EPI_ADD_F32) p.out[row] += a;
                else p.out[row] = a;
            }
        }
        __syncthreads();
        cur = nxt;
    }
    grid_dep_launch();
}

size_t gemv_a4_smem(int K)
{
    return (size_t)(K / 32) * 8 * 8 + WARPS * 8 * 4;
}

// Derived planes from canonical 20-byte groups [rows][K/32] (16 code bytes:
// weight 2i in the low nibble of byte i, 2i + 1 in the high nibble; then
// the fp16 scale and bias).  One thread per (tile, 4-group block, lane).
__global__ void a4_planes_kernel(const uint8_t* groups, int rows, int K, uint4* codes, uint32_t* sb)
{
    const int nb = K / 128, G = K / 32;
    const size_t total = (size_t)(rows / 8) * nb * 32;
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < total;
         i += (size_t)gridDim.x * blockDim.x) {
        const int lane = (int)(i & 31);
        const size_t tb = i >> 5;                 // tile * nb + block
        const int blk = (int)(tb % nb);
        const size_t tile = tb / nb;
        const int n = lane >> 2, t = lane & 3;
        const int row = (int)(tile * 8) + n;
        uint32_t out[4];
        for (int q = 0; q < 4; ++q) {
            const uint8_t* rec = groups + ((size_t)row * G + blk * 4 + q) * 20;
            // fp16 pair j of the word: (k_lo, k_hi) = (2t, 2t+1), (2t+8, 2t+9), (16+2t, 17+2t), (24+2t, 25+2t)
            const int klo[4] = {2 * t, 2 * t + 8, 16 + 2 * t, 24 + 2 * t};
            uint32_t w = 0;
            for (int j = 0; j < 4; ++j) {
                const int k0 = klo[j], k1 = klo[j] + 1;
                const uint32_t c0 = (rec[k0 >> 1] >> ((k0 & 1) * 4)) & 0xF;
                const uint32_t c1 = (rec[k1 >> 1] >> ((k1 & 1) * 4)) & 0xF;
                w |= c0 << (4 * j);
                w |= c1 << (16 + 4 * j);
            }
            out[q] = w;
        }
        codes[i] = make_uint4(out[0], out[1], out[2], out[3]);
        // word `lane` of the (scale, bias) block: 4 n + q is group q of row n (lane t = q)
        {
            const uint8_t* rec = groups + ((size_t)row * G + blk * 4 + t) * 20;
            sb[tb * 32 + lane] = (uint32_t)rec[16] | ((uint32_t)rec[17] << 8) | ((uint32_t)rec[18] << 16) |
                                 ((uint32_t)rec[19] << 24);
        }
    }
}

}  // namespace

int gemv_a4_warps_per_tile(int rows, int K, int pair)
{
    // split each tile's K over more warps while the CTAs would not fill the machine
    const int nb = K / 128;
    int S = 1;
    const int C = 152 * CTAS_PER_SM;
    const int tiles = (pair ? 2 : 1) * rows / 8;
    while (S < WARPS && tiles * S / WARPS < C && nb / (2 * S) >= 2) S *= 2;
    // a unit of WARPS / S tiles must divide the tiles (an even number of them in pair mode)
    while (S < WARPS && tiles % (WARPS / S)) S *= 2;
    if (pair && S > 4) S = 4;          // a unit holds gate and up tiles of the same rows
    return S;
}

cudaError_t launch_a4_planes(cudaStream_t s, const uint8_t* groups, int rows, int K, void* codes, void* sb)
{
    const size_t total = (size_t)(rows / 8) * (K / 128) * 32;
    int grid = (int)((total + 255) / 256);
    if (grid > 152 * 32) grid = 152 * 32;
    a4_planes_kernel<<<grid, 256, 0, s>>>(groups, rows, K, static_cast<uint4*>(codes), static_cast<uint32_t*>(sb));
    return cudaGetLastError();
}

cudaError_t launch_gemv_a4(const Launch& L, const GemvArgs& a)
{
    const int R = WARPS / a.warps_per_row;
    const int n_tiles = a.pair ? 2 * (a.rows[0] / 8)
                               : (a.rows[0] + (a.n_tensors > 1 ? a.rows[1] : 0) +
                                  (a.n_tensors > 2 ? a.rows[2] : 0)) / 8;
    const int n_units = n_tiles / R;
    if (n_units < 1 || n_tiles % R) return cudaErrorInvalidValue;
    const size_t smem = gemv_a4_smem(a.K);
    int grid = std::min(n_units, 152 * CTAS_PER_SM);
    const int iters = (n_units + grid - 1) / grid;
    grid = (n_units + iters - 1) / iters;
    static std::atomic<unsigned long long> attr_done{0};
    if (smem > 48 * 1024)
        if (cudaError_t e = allow_smem_per_device(gemv_a4_kernel, (int)gemv_a4_smem(32768), attr_done)) return e;
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
    return cudaLaunchKernelEx(&cfg, gemv_a4_kernel, a);
}

}  // namespace q3
