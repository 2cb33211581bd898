// k_misc.cu -- the small kernels of the round: token embedding, RMSNorm to
// bf16 rows, the fused per-head q/k RMSNorm + RoPE + paged KV append, the
// vocabulary argmax, and the Q8_0 format kernels.
//
// Sources (Kipp pages): "Kipp Model Support", section "The registry" (RMS
// epsilon, RoPE theta, embedding tying), section "qwen3-0.6b-base" (K/V
// rounded to BF16 on store), section "Quantization (Q8_0)" (32-weight blocks
// of fp16 scale + int8 quants); "Kipp Roadmap", status v0.0.2 (32-position
// block tables).  Layer math not printed on the pages follows the standard
// dense Qwen3 decoder: RMSNorm x / sqrt(mean(x^2) + eps) * g; q/k norm over
// each 128-wide head with gains shared by the heads, before RoPE; RoPE in
// rotate-half pairs (i, i + 64) with angle pos * theta^(-2i/128).
#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;

Q3_DEV float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
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

// ---------------------------------------------------------------- embedding
struct EmbedArgs {
    const int32_t* tokens;
    const __nv_bfloat16* E;
    int H, vocab;
    float* x;
    int* status;
};

__global__ void __launch_bounds__(256) embed_kernel(const EmbedArgs a)
{
    grid_dep_launch();
    grid_dep_wait();
    const int t = blockIdx.x;
    int tok = a.tokens[t];
    if (tok < 0 || tok >= a.vocab) {
        if (threadIdx.x == 0) set_status(a.status, Q3_STATUS_TOKEN_RANGE);
        tok = 0;
    }
    const uint4* src = reinterpret_cast<const uint4*>(a.E + (size_t)tok * a.H);
    float* dst = a.x + (size_t)t * a.H;
    for (int c = threadIdx.x; c < a.H / 8; c += blockDim.x) {
        const uint4 w = __ldg(src + c);
        float4* o = reinterpret_cast<float4*>(dst + c * 8);
        o[0] = make_float4(bf16lo(w.x), bf16hi(w.x), bf16lo(w.y), bf16hi(w.y));
        o[1] = make_float4(bf16lo(w.z), bf16hi(w.z), bf16lo(w.w), bf16hi(w.w));
    }
}

// ---------------------------------------------------------------- RMSNorm -> fp16
struct NormArgs {
    const float* x;
    const int* rows;
    int H;
    const __nv_bfloat16* g;
    float eps;
    __half* h;
    int* status;
};

// The row stays in registers between the two passes (rows up to NORM_MAX
// floats; wider rows re-read it); gains and outputs move 4 values at a time.
constexpr int NORM_THREADS = 256;
constexpr int NORM_VEC = 8;                          // float4 per thread held in registers
constexpr int NORM_MAX = NORM_THREADS * 4 * NORM_VEC;

__global__ void __launch_bounds__(NORM_THREADS) rmsnorm_f16_kernel(const NormArgs a)
{
    __shared__ float red[NORM_THREADS / 32];
    __shared__ float s_scale;
    grid_dep_wait();
    const int r = blockIdx.x;
    const int src = a.rows ? a.rows[r] : r;
    const float* x = a.x + (size_t)src * a.H;
    const bool held = a.H <= NORM_MAX;
    float4 v[NORM_VEC];
    float ss = 0.f;
    if (held) {
#pragma unroll
        for (int k = 0; k < NORM_VEC; ++k) {
            const int i = (threadIdx.x + k * NORM_THREADS) * 4;
            v[k] = i < a.H ? *reinterpret_cast<const float4*>(x + i) : make_float4(0.f, 0.f, 0.f, 0.f);
            ss += v[k].x * v[k].x + v[k].y * v[k].y + v[k].z * v[k].z + v[k].w * v[k].w;
        }
    } else {
        for (int i = threadIdx.x * 4; i < a.H; i += NORM_THREADS * 4) {
            const float4 w = *reinterpret_cast<const float4*>(x + i);
            ss += w.x * w.x + w.y * w.y + w.z * w.z + w.w * w.w;
        }
    }
    grid_dep_launch();
    ss = warp_sum(ss);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ss;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < NORM_THREADS / 32; ++w) t += red[w];
        s_scale = 1.0f / sqrtf(t / (float)a.H + a.eps);
    }
    __syncthreads();
    const float sc = s_scale;
    __half* h = a.h + (size_t)r * a.H;
    bool bad = false;
    auto put = [&](int i, float4 w) {
        const uint2 gg = *reinterpret_cast<const uint2*>(a.g + i);
        __half2 lo, hi;
        lo.x = to_f16(w.x * sc * bf16lo(gg.x), bad);
        lo.y = to_f16(w.y * sc * bf16hi(gg.x), bad);
        hi.x = to_f16(w.z * sc * bf16lo(gg.y), bad);
        hi.y = to_f16(w.w * sc * bf16hi(gg.y), bad);
        uint2 o;
        o.x = *reinterpret_cast<const uint32_t*>(&lo);
        o.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(h + i) = o;
    };
    if (held) {
#pragma unroll
        for (int k = 0; k < NORM_VEC; ++k) {
            const int i = (threadIdx.x + k * NORM_THREADS) * 4;
            if (i < a.H) put(i, v[k]);
        }
    } else {
        for (int i = threadIdx.x * 4; i < a.H; i += NORM_THREADS * 4)
            put(i, *reinterpret_cast<const float4*>(x + i));
    }
    if (bad) set_status(a.status, Q3_STATUS_F16_RANGE);
}

// ---------------------------------------------------------------- q/k norm + RoPE + KV append
// One warp per head of one row; lane l holds elements [4l, 4l + 4).  The
// rotate-half partner of element i < 64 is i + 64, held by lane l ^ 16.
__global__ void __launch_bounds__(128) qk_norm_rope_append_kernel(const RopeArgs a)
{
    grid_dep_wait();
    const int t = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int hh = blockIdx.y * 4 + warp;                // q heads, then k heads, then v heads
    const int n_heads = a.n_q + 2 * a.n_kv;
    if (hh >= n_heads) return;
    const int ld = n_heads * D;
    const int pos = a.row_pos[t];
    const float4 v = *reinterpret_cast<const float4*>(a.qkv + (size_t)t * ld + hh * D + lane * 4);
    float y[4] = {v.x, v.y, v.z, v.w};

    const bool is_q = hh < a.n_q, is_k = !is_q && hh < a.n_q + a.n_kv;
    if (is_q || is_k) {
        // gain (4 bf16) and the (cos, sin) pairs of the lane's 4 frequencies, as vector loads
        const uint2 gg = *reinterpret_cast<const uint2*>((is_q ? a.q_gain : a.k_gain) + lane * 4);
        const float4* csv = reinterpret_cast<const float4*>(a.rope + (size_t)pos * (D / 2) + (lane & 15) * 4);
        const float4 c01 = csv[0], c23 = csv[1];
        const float2 cs[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w), make_float2(c23.x, c23.y),
                              make_float2(c23.z, c23.w)};
        const float gf[4] = {bf16lo(gg.x), bf16hi(gg.x), bf16lo(gg.y), bf16hi(gg.y)};
        const float ss = warp_sum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
        const float r = 1.0f / sqrtf(ss / (float)D + a.eps);
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = y[e] * r * gf[e];
        float out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const float z = __shfl_xor_sync(0xffffffffu, y[e], 16);
            const float2 c = cs[e];
            out[e] = lane < 16 ? y[e] * c.x - z * c.y      // first half: x1 cos - x2 sin
                               : y[e] * c.x + z * c.y;     // second half: x2 cos + x1 sin
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) y[e] = out[e];
    }
    if (is_q) {
        const size_t o = ((size_t)t * a.n_q + hh) * D + lane * 4;
        if (a.q_out)
            *reinterpret_cast<float4*>(a.q_out + o) = make_float4(y[0], y[1], y[2], y[3]);
        if (a.q_out16) {
            bool bad = false;
            __half2 lo, hi;
            lo.x = to_f16(y[0], bad); lo.y = to_f16(y[1], bad);
            hi.x = to_f16(y[2], bad); hi.y = to_f16(y[3], bad);
            uint2 packed;
            packed.x = *reinterpret_cast<const uint32_t*>(&lo);
            packed.y = *reinterpret_cast<const uint32_t*>(&hi);
            *reinterpret_cast<uint2*>(a.q_out16 + o) = packed;
            if (bad) set_status(a.status, Q3_STATUS_F16_RANGE);
        }
        return;
    }
    const int slot = a.row_slot[t];
    const int blk = a.tables[(size_t)slot * a.max_blocks + pos / 32];
    if (blk < 0 || blk >= a.n_blocks) {
        if (lane == 0) set_status(a.status, Q3_STATUS_BLOCK_RANGE);
        return;
    }
    const int kvh = is_k ? hh - a.n_q : hh - a.n_q - a.n_kv;
    if (a.kvq_layer) {
        uint32_t codes;
        __half scale;
        float deq[4];
        kvq_pack(y, codes, scale, deq);
        kvq_store(a.kvq_layer + (((size_t)blk * 2 + (is_k ? 0 : 1)) * a.n_kv + kvh) * KVQ_TILE, pos % 32,
                  codes, scale, lane);
        return;
    }
    __nv_bfloat16* dst = a.kv_layer +
        (((size_t)blk * 2 + (is_k ? 0 : 1)) * a.n_kv + kvh) * (32 * D) + (size_t)(pos % 32) * D + lane * 4;
    const __nv_bfloat162 lo = __floats2bfloat162_rn(y[0], y[1]);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(y[2], y[3]);
    uint2 packed;
    packed.x = *reinterpret_cast<const uint32_t*>(&lo);
    packed.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(dst) = packed;
}

// ---------------------------------------------------------------- argmax
struct ArgmaxArgs {
    const float* logits;
    int V;
    int32_t* out;
};

// Greedy token: the largest logit, the lowest index on ties.
__global__ void __launch_bounds__(1024) argmax_kernel(const ArgmaxArgs a)
{
    __shared__ float sv[32];
    __shared__ int si[32];
    grid_dep_wait();
    const float* x = a.logits + (size_t)blockIdx.x * a.V;
    float best = -INFINITY;
    int bi = 0x7fffffff;
    auto take = [&](float v, int i) {
        if (v > best) { best = v; bi = i; }      // ascending i per thread: first max kept
    };
    int tail = 0;
    if ((a.V & 3) == 0 && (reinterpret_cast<uintptr_t>(x) & 15) == 0) {
        // 16-byte loads, four in flight per thread (the row is one CTA's)
        const float4* x4 = reinterpret_cast<const float4*>(x);
        const int n4 = a.V / 4, T = blockDim.x;
        int c = threadIdx.x;
        for (; c + 3 * T < n4; c += 4 * T) {
            float4 v[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) v[u] = __ldcg(x4 + c + u * T);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int i = 4 * (c + u * T);
                take(v[u].x, i); take(v[u].y, i + 1); take(v[u].z, i + 2); take(v[u].w, i + 3);
            }
        }
        for (; c < n4; c += T) {
            const float4 v = __ldcg(x4 + c);
            take(v.x, 4 * c); take(v.y, 4 * c + 1); take(v.z, 4 * c + 2); take(v.w, 4 * c + 3);
        }
        tail = a.V;
    }
    for (int i = tail + threadIdx.x; i < a.V; i += blockDim.x) take(x[i], i);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
    }
    if ((threadIdx.x & 31) == 0) { sv[threadIdx.x >> 5] = best; si[threadIdx.x >> 5] = bi; }
    __syncthreads();
    if (threadIdx.x < 32) {
        best = sv[threadIdx.x];
        bi = si[threadIdx.x];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, best, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (ov > best || (ov == best && oi < bi)) { best = ov; bi = oi; }
        }
        if (threadIdx.x == 0) a.out[blockIdx.x] = bi == 0x7fffffff ? 0 : bi;
    }
    grid_dep_launch();
}

// ---------------------------------------------------------------- Q8_0
// canonical block: bytes 0-1 little-endian fp16 scale, bytes 2-33 int8 quants
__global__ void q8_split_kernel(const uint8_t* blocks, int64_t nblocks, int8_t* qs, __half* scales)
{
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        const uint8_t* in = blocks + b * Q3_Q8_0_BYTES;
        const uint16_t bits = (uint16_t)(in[0] | (in[1] << 8));
        scales[b] = __ushort_as_half(bits);
        int8_t* o = qs + b * 32;
        for (int i = 0; i < 32; ++i) o[i] = (int8_t)in[2 + i];
    }
}

struct Q8DeqArgs {
    const int8_t* qs;
    const __half* scales;
    int64_t n;
    __half* w;
};

// fp16(fp16 scale * quant) for the tensor-core prefill path (|d q| <= 127 d
// never leaves the fp16 range; the product is rounded to 11 bits)
__global__ void q8_to_f16_kernel(const Q8DeqArgs a)
{
    grid_dep_wait();
    for (int64_t i = (blockIdx.x * (int64_t)blockDim.x + threadIdx.x) * 8; i < a.n;
         i += (int64_t)gridDim.x * blockDim.x * 8) {
        const float d = __half2float(a.scales[i / 32]);
        const uint2 q = *reinterpret_cast<const uint2*>(a.qs + i);
        __half out[8];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            out[e] = __float2half_rn(d * (float)(int8_t)((q.x >> (8 * e)) & 0xff));
            out[4 + e] = __float2half_rn(d * (float)(int8_t)((q.y >> (8 * e)) & 0xff));
        }
        *reinterpret_cast<uint4*>(a.w + i) = *reinterpret_cast<const uint4*>(out);
    }
    grid_dep_launch();
}

// fp16 copy of bf16 weights (exact for 2^-17 <= |w| <= 65504 and 0)
__global__ void bf16_to_f16_kernel(const __nv_bfloat16* w, int64_t n, __half* out,
                                   unsigned long long* inexact, unsigned long long* overflow)
{
    unsigned long long n_inexact = 0, n_over = 0;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const float v = __bfloat162float(w[i]);
        const __half h = __float2half_rn(v);
        out[i] = h;
        const float back = __half2float(h);
        if (!(fabsf(v) <= 65504.0f)) ++n_over;
        else if (back != v) ++n_inexact;
    }
    if (n_inexact) atomicAdd(inexact, n_inexact);
    if (n_over) atomicAdd(overflow, n_over);
}

// Per block of 32: d = absmax / 127 (FP32, correctly rounded), scale =
// fp16(d) round-to-nearest-even, q = round-half-even(w / d) clamped to
// [-127, 127]; an all-zero block gets scale 0 and zero quants.
__global__ void quantize_q8_0_kernel(const __nv_bfloat16* w, int64_t nblocks, uint8_t* blocks)
{
    for (int64_t b = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; b < nblocks;
         b += (int64_t)gridDim.x * blockDim.x) {
        float x[32];
        float amax = 0.f;
        for (int i = 0; i < 32; ++i) {
            x[i] = __bfloat162float(w[b * 32 + i]);
            amax = fmaxf(amax, fabsf(x[i]));
        }
        const float d = __fdiv_rn(amax, 127.0f);
        // the 34-byte record as 17 little-endian 16-bit words (2-byte aligned)
        uint16_t* out = reinterpret_cast<uint16_t*>(blocks + b * Q3_Q8_0_BYTES);
        out[0] = __half_as_ushort(__float2half_rn(d));
        for (int i = 0; i < 32; i += 2) {
            int q0 = 0, q1 = 0;
            if (d != 0.f) {
                q0 = __float2int_rn(__fdiv_rn(x[i], d));
                q1 = __float2int_rn(__fdiv_rn(x[i + 1], d));
                q0 = q0 > 127 ? 127 : (q0 < -127 ? -127 : q0);
                q1 = q1 > 127 ? 127 : (q1 < -127 ? -127 : q1);
            }
            out[1 + i / 2] = (uint16_t)((uint8_t)(int8_t)q0 | ((uint16_t)(uint8_t)(int8_t)q1 << 8));
        }
    }
}

// ---------------------------------------------------------------- AFFINE4_GS32
// 20-byte group: 16 code bytes (weight 2i in the low nibble of byte i, weight
// 2i + 1 in the high nibble), then fp16 scale and fp16 bias, little-endian;
// a weight is scale * code + bias.  As five little-endian words, weight i's
// code sits in word i / 8 at bit 4 (i % 8), and word 4 holds scale | bias << 16.

// Per group of 32: bias = fp16(min), scale = fp16((max - min) / 15) (FP32,
// correctly rounded), code = round-half-even((w - bias) / scale) in FP32
// against the stored scale and bias, clamped to [0, 15]; a zero scale gives
// zero codes.  One thread per group.
__global__ void quantize_affine4_kernel(const __nv_bfloat16* w, int64_t ngroups, uint8_t* groups)
{
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < ngroups;
         g += (int64_t)gridDim.x * blockDim.x) {
        float x[32];
        const uint4* src = reinterpret_cast<const uint4*>(w + g * 32);
#pragma unroll
        for (int v = 0; v < 4; ++v) {
            const uint4 u = src[v];
            const uint32_t wd[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                x[8 * v + 2 * e] = __uint_as_float(wd[e] << 16);
                x[8 * v + 2 * e + 1] = __uint_as_float(wd[e] & 0xffff0000u);
            }
        }
        float lo = x[0], hi = x[0];
#pragma unroll
        for (int i = 1; i < 32; ++i) {
            if (x[i] < lo) lo = x[i];
            if (x[i] > hi) hi = x[i];
        }
        const __half sh = __float2half_rn(__fdiv_rn(__fsub_rn(hi, lo), 15.0f));
        const __half bh = __float2half_rn(lo);
        const float scale = __half2float(sh), bias = __half2float(bh);
        uint32_t out[5] = {0u, 0u, 0u, 0u,
                           (uint32_t)__half_as_ushort(sh) | ((uint32_t)__half_as_ushort(bh) << 16)};
        if (scale != 0.f) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                int q = __float2int_rn(__fdiv_rn(__fsub_rn(x[i], bias), scale));
                q = q < 0 ? 0 : (q > 15 ? 15 : q);
                out[i / 8] |= (uint32_t)q << (4 * (i % 8));
            }
        }
        uint32_t* dst = reinterpret_cast<uint32_t*>(groups + g * Q3_AFFINE4_BYTES);
#pragma unroll
        for (int k = 0; k < 5; ++k) dst[k] = out[k];
    }
}

// fp16(fma(scale, code, bias)) for the tensor-core path; one thread per group.
__global__ void affine4_to_f16_kernel(const uint8_t* groups, int64_t ngroups, __half* w,
                                      unsigned long long* overflow)
{
    unsigned long long n_over = 0;
    for (int64_t g = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; g < ngroups;
         g += (int64_t)gridDim.x * blockDim.x) {
        const uint32_t* in = reinterpret_cast<const uint32_t*>(groups + g * Q3_AFFINE4_BYTES);
        const uint32_t sb = in[4];
        const float scale = __half2float(__ushort_as_half((unsigned short)(sb & 0xffffu)));
        const float bias = __half2float(__ushort_as_half((unsigned short)(sb >> 16)));
        uint4* dst = reinterpret_cast<uint4*>(w + g * 32);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t c = in[k];
            uint32_t h[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float v0 = __fmaf_rn(scale, (float)((c >> (8 * e)) & 0xfu), bias);
                const float v1 = __fmaf_rn(scale, (float)((c >> (8 * e + 4)) & 0xfu), bias);
                if (!(fabsf(v0) <= 65504.0f)) ++n_over;
                if (!(fabsf(v1) <= 65504.0f)) ++n_over;
                h[e] = (uint32_t)__half_as_ushort(__float2half_rn(v0)) |
                       ((uint32_t)__half_as_ushort(__float2half_rn(v1)) << 16);
            }
            dst[k] = make_uint4(h[0], h[1], h[2], h[3]);
        }
    }
    if (n_over && overflow) atomicAdd(overflow, n_over);
}

}  // namespace

cudaError_t launch_embed(const Launch& L, const int32_t* tokens, int T, const __nv_bfloat16* E,
                         int H, int vocab, float* x, int* status)
{
    return launch_ex(L, embed_kernel, dim3(T), dim3(256), EmbedArgs{tokens, E, H, vocab, x, status});
}

cudaError_t launch_rmsnorm_f16(const Launch& L, const float* x, const int* rows, int n, int H,
                               const __nv_bfloat16* g, float eps, __half* h, int* status)
{
    return launch_ex(L, rmsnorm_f16_kernel, dim3(n), dim3(256), NormArgs{x, rows, H, g, eps, h, status});
}

cudaError_t launch_qk_norm_rope_append(const Launch& L, const RopeArgs& a)
{
    const int heads = a.n_q + 2 * a.n_kv;
    return launch_ex(L, qk_norm_rope_append_kernel, dim3(a.T, (heads + 3) / 4), dim3(128), a);
}

// Q8_0 K/V packing of caller rows (operator gate of the cache writers): one
// warp per 128-value row, written as 4 canonical blocks of 34 bytes.
__global__ void __launch_bounds__(128) kv_pack_q8_kernel(const float* rows, int n, uint8_t* out)
{
    const int r = blockIdx.x * 4 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
    if (r >= n) return;
    const float4 v = *reinterpret_cast<const float4*>(rows + (size_t)r * 128 + lane * 4);
    const float y[4] = {v.x, v.y, v.z, v.w};
    uint32_t codes;
    __half scale;
    float deq[4];
    kvq_pack(y, codes, scale, deq);
    uint8_t* blk = out + (size_t)r * 136 + (lane >> 3) * 34;
    if ((lane & 7) == 0) {
        const unsigned short sb = __half_as_ushort(scale);
        blk[0] = (uint8_t)(sb & 0xff);
        blk[1] = (uint8_t)(sb >> 8);
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) blk[2 + (lane & 7) * 4 + e] = (uint8_t)(codes >> (8 * e));
}

cudaError_t launch_kv_pack_q8(cudaStream_t s, const float* rows, int n, uint8_t* out)
{
    kv_pack_q8_kernel<<<(n + 3) / 4, 128, 0, s>>>(rows, n, out);
    return cudaGetLastError();
}

cudaError_t launch_argmax(const Launch& L, const float* logits, int rows, int V, int32_t* out)
{
    return launch_ex(L, argmax_kernel, dim3(rows), dim3(1024), ArgmaxArgs{logits, V, out});
}

cudaError_t launch_q8_split(cudaStream_t s, const uint8_t* blocks, int64_t nblocks, int8_t* qs,
                            __half* scales)
{
    int grid = (int)((nblocks + 255) / 256);
    if (grid > 152 * 32) grid = 152 * 32;
    q8_split_kernel<<<grid, 256, 0, s>>>(blocks, nblocks, qs, scales);
    return cudaGetLastError();
}

cudaError_t launch_q8_to_f16(const Launch& L, const int8_t* qs, const __half* scales, int64_t n,
                             __half* w)
{
    int64_t grid = (n / 8 + 255) / 256;
    if (grid > 152 * 32) grid = 152 * 32;
    return launch_ex(L, q8_to_f16_kernel, dim3((unsigned)grid), dim3(256), Q8DeqArgs{qs, scales, n, w});
}

cudaError_t launch_bf16_to_f16(cudaStream_t s, const __nv_bfloat16* w, int64_t n, __half* out,
                               unsigned long long* inexact, unsigned long long* overflow)
{
    int64_t grid = (n + 255) / 256;
    if (grid > 152 * 32) grid = 152 * 32;
    if (grid < 1) grid = 1;
    bf16_to_f16_kernel<<<(unsigned)grid, 256, 0, s>>>(w, n, out, inexact, overflow);
    return cudaGetLastError();
}

cudaError_t launch_quantize_affine4(cudaStream_t s, const __nv_bfloat16* w, int64_t n, uint8_t* groups)
{
    const int64_t ng = n / 32;
    int grid = (int)((ng + 255) / 256);
    if (grid > 152 * 32) grid = 152 * 32;
    if (grid < 1) grid = 1;
    quantize_affine4_kernel<<<grid, 256, 0, s>>>(w, ng, groups);
    return cudaGetLastError();
}

cudaError_t launch_affine4_to_f16(cudaStream_t s, const uint8_t* groups, int64_t n, __half* w,
                                  unsigned long long* overflow)
{
    const int64_t ng = n / 32;
    int grid = (int)((ng + 255) / 256);
    if (grid > 152 * 32) grid = 152 * 32;
    if (grid < 1) grid = 1;
    affine4_to_f16_kernel<<<grid, 256, 0, s>>>(groups, ng, w, overflow);
    return cudaGetLastError();
}

cudaError_t launch_quantize_q8_0(cudaStream_t s, const __nv_bfloat16* w, int64_t n, uint8_t* blocks)
{
    const int64_t nb = n / 32;
    int grid = (int)((nb + 255) / 256);
    if (grid > 152 * 32) grid = 152 * 32;
    if (grid < 1) grid = 1;
    quantize_q8_0_kernel<<<grid, 256, 0, s>>>(w, nb, blocks);
    return cudaGetLastError();
}

}  // namespace q3
