// k_attn_prefill.cu -- causal GQA attention of prefill rounds on tensor cores.
//
// Rows of a prefill round attend to every earlier position of their session
// and to the rows before them in the round ("Kipp Roadmap", status v0.0.3:
// flash-attention prefill kernel; status v0.0.6: long-context prefill
// attention is the next lever; "Kipp Model Support", section
// "qwen3-0.6b-base": K/V stored as BF16).  Flash-style tiling: a CTA owns 64
// query rows of one session for up to four query heads of one KV head (four
// warps of 16 rows per head) and walks the session's paged K/V in tiles of
// 64 positions (two 32-position blocks through the block table), keeping the
// online-softmax row maximum and sum and the 16 x 128 output accumulator in
// registers; the heads of the group share each staged K/V tile.
//
// Products run on mma.sync m16n8k16 with fp16 operands and FP32
// accumulation: Q arrives in fp16; K/V tiles are copied as stored (BF16)
// with cp.async into a double buffer and converted once per CTA into fp16
// shared-memory tiles (exact for the ranges of normed, rotated K and of V;
// fp16 keeps 3 more mantissa bits than bf16 for Q and P).  Shared-memory
// tiles use an XOR swizzle of 16-byte chunks so ldmatrix reads are
// conflict-free.  With the opt-in Q8_0 cache ("Kipp Roadmap", status v0.0.4)
// the raw Q8_0 tiles (codes and fp16 scales) are copied instead and the
// conversion writes fp16(scale * code), each product rounded once.
// Scores are scaled by log2(e)/sqrt(128) and exponentiated
// in base 2; positions after a query's own position are masked.  Positions a
// block does not hold read zeros, never stale shared memory.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"

namespace q3 {

namespace {

constexpr int D = 128;
constexpr int BM = 64;                 // query rows per CTA
constexpr int BN = 64;                 // key positions per tile
constexpr int TILE_BYTES = BM * D * 2; // 16 KB (64 rows x 256 bytes)

// byte offset of 16-byte chunk c of row r in a swizzled 64 x 128 fp16 tile
Q3_DEV uint32_t swz(int r, int c) { return (uint32_t)(r * 256 + ((c ^ (r & 7)) << 4)); }

Q3_DEV void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
Q3_DEV void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
Q3_DEV void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                     uint32_t b0, uint32_t b1) {
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
Q3_DEV uint32_t pack_f16(float lo, float hi) {
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&h);
}
// 8 bf16 (one 16-byte chunk) -> 8 fp16
Q3_DEV uint4 bf16x8_to_f16x8(uint4 w) {
    uint4 o;
    o.x = pack_f16(bf16lo(w.x), bf16hi(w.x));
    o.y = pack_f16(bf16lo(w.y), bf16hi(w.y));
    o.z = pack_f16(bf16lo(w.z), bf16hi(w.z));
    o.w = pack_f16(bf16lo(w.w), bf16hi(w.w));
    return o;
}

// One CTA per (64-row query tile of one session, KV head, group of HPC query
// heads of that KV head): the heads of a group share each K/V tile, fetched
// and converted once for all of them.  Warp w takes query head w / 4 of the
// group and rows 16 (w % 4) .. + 16 of the tile.
template <int HPC>
__global__ void __launch_bounds__(HPC * 4 * 32, 1) prefill_attn_kernel(const PrefillAttnArgs p)
{
    constexpr int NT = HPC * 4 * 32;
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t* sQ = smem;                                   // [HPC] fp16 swizzled 64 x 128 tiles
    uint8_t* sK = smem + HPC * TILE_BYTES;
    uint8_t* sV = sK + TILE_BYTES;
    uint8_t* bKV = sV + TILE_BYTES;                       // [2 buffers][K, V] bf16, linear

    __shared__ int s_item;
    const int G = p.n_q / p.n_kv;
    const int Z = G / HPC;                                // head groups per KV head
    const int n_items = p.n_tiles * p.n_kv * Z;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hg = warp >> 2, rg = warp & 3;
    const int g = lane >> 2, tq = lane & 3;

    grid_dep_wait();

    // Persistent CTAs take (tile, KV head, head group) items from a queue in
    // order: tiles come longest context first, so the longest items start
    // first.  Each CTA's final draw lands past the end; the last of those
    // resets the queue for the next launch.
    for (;;) {
    __syncthreads();
    if (tid == 0) {
        const int it = atomicAdd(p.work_counter, 1);
        if (it == n_items + (int)gridDim.x - 1) *p.work_counter = 0;
        s_item = it;
    }
    __syncthreads();
    const int item = s_item;
    if (item >= n_items) break;
    const int tile = item / (p.n_kv * Z);
    const int kvh = (item / Z) % p.n_kv;
    const int head0 = kvh * G + (item % Z) * HPC;         // first query head of the group
    const int h = head0 + hg;

    const int row0 = p.tile_row0[tile];
    const int nrows = p.tile_rows[tile];
    const int pos0 = p.row_pos[row0];
    const int pos_last = pos0 + nrows - 1;
    const int* table = p.tables + (size_t)p.row_slot[row0] * p.max_blocks;
    const int nblk = (pos_last + 32) / 32;                // blocks holding positions 0..pos_last
    const int n_kt = (pos_last + BN) / BN;
    const int qw = p.n_q * D;

    // ---- Q tiles of the G heads (rows past the round repeat its last row)
    for (int i = tid; i < HPC * BM * 16; i += NT) {
        const int hh = i / (BM * 16), r = (i >> 4) % BM, c = i & 15;
        const int src_row = row0 + min(r, nrows - 1);
        cp_async_16(sQ + hh * TILE_BYTES + swz(r, c), p.q + (size_t)src_row * qw + (head0 + hh) * D + c * 8);
    }
    cp_async_commit();

    // ---- K/V tile kt -> staging buffer buf (bf16, linear rows of 256 bytes)
    auto issue_kv = [&](int kt, int buf) {
        uint8_t* dstK = bKV + (size_t)buf * 2 * TILE_BYTES;
        uint8_t* dstV = dstK + TILE_BYTES;
        if (p.kvq_layer) {
            // raw Q8_0 tiles of the two blocks: block j at j * KVQ_TILE
            for (int i = tid; i < 2 * (KVQ_TILE / 16); i += NT) {
                const int j = i / (KVQ_TILE / 16), piece = i % (KVQ_TILE / 16);
                const int b = 2 * kt + j;
                if (b >= nblk) continue;
                const int phys = table[b];
                if (phys < 0 || phys >= p.n_blocks) {
                    if (piece == 0) set_status(p.status, Q3_STATUS_BLOCK_RANGE);
                    continue;
                }
                const uint8_t* Kq = p.kvq_layer + ((size_t)phys * 2 * p.n_kv + kvh) * KVQ_TILE;
                const uint8_t* Vq = Kq + (size_t)p.n_kv * KVQ_TILE;
                cp_async_16(dstK + j * KVQ_TILE + piece * 16, Kq + piece * 16);
                cp_async_16(dstV + j * KVQ_TILE + piece * 16, Vq + piece * 16);
            }
            cp_async_commit();
            return;
        }
        for (int i = tid; i < BN * 16; i += NT) {
            const int r = i >> 4, c = i & 15;
            const int b = 2 * kt + (r >> 5);
            if (b >= nblk) continue;
            const int phys = table[b];
            if (phys < 0 || phys >= p.n_blocks) {
                if (c == 0 && (r & 31) == 0) set_status(p.status, Q3_STATUS_BLOCK_RANGE);
                continue;
            }
            const __nv_bfloat16* Kb = p.kv_layer + ((size_t)phys * 2 * p.n_kv + kvh) * (32 * D);
            const __nv_bfloat16* Vb = Kb + (size_t)p.n_kv * (32 * D);
            cp_async_16(dstK + r * 256 + c * 16, Kb + (r & 31) * D + c * 8);
            cp_async_16(dstV + r * 256 + c * 16, Vb + (r & 31) * D + c * 8);
        }
        cp_async_commit();
    };
    issue_kv(0, 0);

    float o[16][4];
#pragma unroll
    for (int n = 0; n < 16; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
    float m_r[2] = {-INFINITY, -INFINITY}, l_r[2] = {0.f, 0.f};
    const int qr0 = rg * 16 + g;                          // this thread's two query rows
    const int qp[2] = {pos0 + min(qr0, nrows - 1), pos0 + min(qr0 + 8, nrows - 1)};
    const int qp_min = pos0 + min(rg * 16, nrows - 1);    // the warp's first query position
    const float scale = 1.4426950408889634f * 0.08838834764831845f;   // log2(e) / sqrt(128)
    const uint32_t qbase = smem_u32(sQ + hg * TILE_BYTES);

    for (int kt = 0; kt < n_kt; ++kt) {
        if (kt + 1 < n_kt) {
            issue_kv(kt + 1, (kt + 1) & 1);
            cp_async_wait_all_but(1);
        } else {
            cp_async_wait_all();
        }
        __syncthreads();
        // convert the staged tile to fp16 (rows of absent blocks become zeros)
        {
            const uint8_t* srcK = bKV + (size_t)(kt & 1) * 2 * TILE_BYTES;
            const uint8_t* srcV = srcK + TILE_BYTES;
            for (int i = tid; i < BN * 16; i += NT) {
                const int r = i >> 4, c = i & 15;
                const bool present = 2 * kt + (r >> 5) < nblk;
                uint4 k = make_uint4(0, 0, 0, 0), v = make_uint4(0, 0, 0, 0);
                if (present && p.kvq_layer) {
                    // 8 codes of row r at dims 8c.., scale of their 32-dim block c / 4
                    const int off = (r >> 5) * KVQ_TILE, rr = r & 31;
                    const uint2 ck = *reinterpret_cast<const uint2*>(srcK + off + rr * 128 + c * 8);
                    const uint2 cv = *reinterpret_cast<const uint2*>(srcV + off + rr * 128 + c * 8);
                    const __half dk = *reinterpret_cast<const __half*>(srcK + off + KVQ_CODES + (rr * 4 + c / 4) * 2);
                    const __half dv = *reinterpret_cast<const __half*>(srcV + off + KVQ_CODES + (rr * 4 + c / 4) * 2);
                    const uint2 k0 = kvq_dequant4(ck.x, dk), k1 = kvq_dequant4(ck.y, dk);
                    const uint2 v0 = kvq_dequant4(cv.x, dv), v1 = kvq_dequant4(cv.y, dv);
                    k = make_uint4(k0.x, k0.y, k1.x, k1.y);
                    v = make_uint4(v0.x, v0.y, v1.x, v1.y);
                } else if (present) {
                    k = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(srcK + r * 256 + c * 16));
                    v = bf16x8_to_f16x8(*reinterpret_cast<const uint4*>(srcV + r * 256 + c * 16));
                }
                *reinterpret_cast<uint4*>(sK + swz(r, c)) = k;
                *reinterpret_cast<uint4*>(sV + swz(r, c)) = v;
            }
        }
        __syncthreads();

        // ---- S = Q K^T (16 x 64 per warp)
        float s[8][4];
#pragma unroll
        for (int n = 0; n < 8; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
        const uint32_t kbase = smem_u32(sK);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4(qbase + swz(rg * 16 + (lane & 15), 2 * kk + (lane >> 4)), a0, a1, a2, a3);
#pragma unroll
            for (int np = 0; np < 4; ++np) {
                const int r = 16 * np + (lane & 7) + ((lane >> 4) & 1) * 8;
                uint32_t b0, b1, b2, b3;
                ldsm_x4(kbase + swz(r, 2 * kk + ((lane >> 3) & 1)), b0, b1, b2, b3);
                mma16816(s[2 * np], a0, a1, a2, a3, b0, b1);
                mma16816(s[2 * np + 1], a0, a1, a2, a3, b2, b3);
            }
        }

        // ---- causal mask (only tiles reaching past the warp's first row) and online softmax
        const bool masked = kt * BN + BN - 1 > qp_min;
        float mx[2] = {m_r[0], m_r[1]};
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int kp = kt * BN + n * 8 + 2 * tq + (e & 1);
                const int ri = e >> 1;
                const float v = (!masked || kp <= qp[ri]) ? s[n][e] * scale : -INFINITY;
                s[n][e] = v;
                mx[ri] = fmaxf(mx[ri], v);
            }
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 1));
            mx[ri] = fmaxf(mx[ri], __shfl_xor_sync(0xffffffffu, mx[ri], 2));
        }
        float alpha[2], rs[2] = {0.f, 0.f};
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) alpha[ri] = exp2f(m_r[ri] - mx[ri]);   // 0 when m_r = -inf
#pragma unroll
        for (int n = 0; n < 8; ++n) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const float pv = exp2f(s[n][e] - mx[e >> 1]);
                s[n][e] = pv;
                rs[e >> 1] += pv;
            }
        }
#pragma unroll
        for (int ri = 0; ri < 2; ++ri) {
            rs[ri] += __shfl_xor_sync(0xffffffffu, rs[ri], 1);
            rs[ri] += __shfl_xor_sync(0xffffffffu, rs[ri], 2);
            l_r[ri] = l_r[ri] * alpha[ri] + rs[ri];
            m_r[ri] = mx[ri];
        }
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            o[n][0] *= alpha[0]; o[n][1] *= alpha[0];
            o[n][2] *= alpha[1]; o[n][3] *= alpha[1];
        }

        // ---- O += P V
        const uint32_t vbase = smem_u32(sV);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const uint32_t a0 = pack_f16(s[2 * kk][0], s[2 * kk][1]);
            const uint32_t a1 = pack_f16(s[2 * kk][2], s[2 * kk][3]);
            const uint32_t a2 = pack_f16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
            const uint32_t a3 = pack_f16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
            const int r = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
            for (int dp = 0; dp < 8; ++dp) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(vbase + swz(r, 2 * dp + (lane >> 4)), b0, b1, b2, b3);
                mma16816(o[2 * dp], a0, a1, a2, a3, b0, b1);
                mma16816(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        __syncthreads();       // sK / sV are rewritten by the next tile's conversion
    }

    // ---- normalise and store fp16
    bool bad = false;
#pragma unroll
    for (int ri = 0; ri < 2; ++ri) {
        const int qr = qr0 + 8 * ri;
        if (qr >= nrows) continue;
        const float inv = 1.0f / l_r[ri];
        __half* dst = p.out + (size_t)(row0 + qr) * qw + h * D;
#pragma unroll
        for (int n = 0; n < 16; ++n) {
            __half2 v;
            v.x = to_f16(o[n][2 * ri] * inv, bad);
            v.y = to_f16(o[n][2 * ri + 1] * inv, bad);
            *reinterpret_cast<__half2*>(dst + n * 8 + 2 * tq) = v;
        }
    }
    if (bad) set_status(p.status, Q3_STATUS_F16_RANGE);
    }   // items
    grid_dep_launch();
}

template <int HPC>
cudaError_t launch_prefill_g(const Launch& L, const PrefillAttnArgs& a)
{
    const size_t smem = (size_t)(HPC + 2) * TILE_BYTES + 2 * 2 * TILE_BYTES;   // Q x HPC, K, V fp16 + staged K/V
    static std::atomic<unsigned long long> attr_done{0};
    if (cudaError_t e = allow_smem_per_device(prefill_attn_kernel<HPC>, (int)smem, attr_done)) return e;
    // resident CTAs per SM and SMs of the current device (asked on every launch:
    // cheap beside the kernel, and right on any device)
    int dev = 0, per_sm = 0, n_sm = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, prefill_attn_kernel<HPC>, HPC * 4 * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    const int items = a.n_tiles * a.n_q / HPC;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(std::min(items, per_sm * n_sm));
    cfg.blockDim = dim3(HPC * 4 * 32);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = L.pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (L.counter) ++*L.counter;
    return cudaLaunchKernelEx(&cfg, prefill_attn_kernel<HPC>, a);
}

}  // namespace

// Heads per CTA: the largest of 4, 3, 2, 1 dividing the group size (16
// warps at most, for the registers the accumulators need).
cudaError_t launch_prefill_attention(const Launch& L, const PrefillAttnArgs& a)
{
    const int G = a.n_q / a.n_kv;
    if (G < 1 || a.n_q % a.n_kv) return cudaErrorInvalidValue;
    if (G % 4 == 0) return launch_prefill_g<4>(L, a);
    if (G % 3 == 0) return launch_prefill_g<3>(L, a);
    if (G % 2 == 0) return launch_prefill_g<2>(L, a);
    return launch_prefill_g<1>(L, a);
}

}  // namespace q3
