// common.cuh -- device helpers shared by the sm_103a kernels: bf16/fp16
// conversions, vector loads, the bounded mbarrier wait, TMA and tcgen05
// (TMEM) inline PTX.  Host-visible launch declarations live in kernels.h.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/q3.h"
#include "kernels.h"

#define Q3_DEV __device__ __forceinline__

// A bounded device wait gives up after this many nanoseconds of global time,
// sets Q3_STATUS_TIMEOUT in the status word and lets the kernel unwind.
#ifndef Q3_WAIT_LIMIT_NS
#define Q3_WAIT_LIMIT_NS 2000000000ull
#endif

namespace q3 {

Q3_DEV uint32_t smem_u32_early(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

Q3_DEV float bf16_bits_to_f32(uint32_t b16) { return __uint_as_float(b16 << 16); }
Q3_DEV float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
Q3_DEV float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
// The four signed bytes of q as exact floats without the int-to-float unit:
// with the sign bit flipped a byte b becomes b + 128 in [0, 255], and the
// word 0x4B000000 | (b + 128) is the float 2^23 + 128 + b exactly, so one
// byte permute and one subtraction give b (the same value as a conversion).
Q3_DEV float i8_byte(uint32_t flipped, uint32_t sel) {
    return __uint_as_float(__byte_perm(flipped, 0x4B000000u, sel)) - 8388736.0f;
}

Q3_DEV uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

Q3_DEV uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

Q3_DEV void set_status(int* status, int bits) { atomicOr(status, bits); }

// ---------------------------------------------------------------- cp.async
Q3_DEV void cp_async_16(void* smem_dst, const void* gmem_src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"(smem_u32_early(smem_dst)), "l"(gmem_src) : "memory");
}
Q3_DEV void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
Q3_DEV void cp_async_wait_all() { asm volatile("cp.async.wait_group 0;" ::: "memory"); }
// wait until at most one committed group is still in flight
Q3_DEV void cp_async_wait_all_but(int) { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// ---------------------------------------------------------------- per-head q/k norm + RoPE
// One warp holds one 128-wide head, lane l elements [4l, 4l + 4).  RMSNorm
// over the head with the shared gain, then rotate-half RoPE: element i < 64
// pairs with i + 64 (lane l ^ 16); angle pos * theta^(-2i/128) from the
// (cos, sin) table row of the position.
Q3_DEV float warp_allsum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// The same, from the lane's gain (4 bf16) and (cos, sin) pairs already loaded
Q3_DEV void head_norm_rope_loaded(float (&y)[4], uint2 g4, float4 c01, float4 c23, float eps, int lane) {
    const float gv[4] = {bf16lo(g4.x), bf16hi(g4.x), bf16lo(g4.y), bf16hi(g4.y)};
    const float2 cv[4] = {make_float2(c01.x, c01.y), make_float2(c01.z, c01.w), make_float2(c23.x, c23.y),
                          make_float2(c23.z, c23.w)};
    const float ss = warp_allsum(y[0] * y[0] + y[1] * y[1] + y[2] * y[2] + y[3] * y[3]);
    const float r = 1.0f / sqrtf(ss / 128.0f + eps);
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = y[e] * r * gv[e];
    float out[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const float z = __shfl_xor_sync(0xffffffffu, y[e], 16);
        const float2 c = cv[e];
        out[e] = lane < 16 ? y[e] * c.x - z * c.y      // first half: x1 cos - x2 sin
                           : y[e] * c.x + z * c.y;     // second half: x2 cos + x1 sin
    }
#pragma unroll
    for (int e = 0; e < 4; ++e) y[e] = out[e];
}

Q3_DEV void head_norm_rope(float (&y)[4], const __nv_bfloat16* gain, const float2* rope_row,
                           float eps, int lane) {
    // gain and cos/sin loads go out before the reduction that precedes their use
    const uint2 g4 = *reinterpret_cast<const uint2*>(gain + lane * 4);
    const float4* cs = reinterpret_cast<const float4*>(rope_row + (lane & 15) * 4);
    head_norm_rope_loaded(y, g4, cs[0], cs[1], eps, lane);
}

// ---------------------------------------------------------------- Q8_0 K/V rows
// The opt-in Q8_0 K/V cache ("Kipp Roadmap", status v0.0.4: an opt-in Q8_0 KV
// cache, about 1.9x smaller than BF16) packs each position's 128-wide head
// row with the weights' Q8_0 rule ("Kipp Model Support", section
// "Quantization (Q8_0)"): blocks of 32 consecutive values, d = absmax / 127
// in FP32 (correctly rounded), stored as fp16(d); codes round-half-even(x / d)
// against the FP32 d, clamped to [-127, 127]; an all-zero block has d = 0.
// The pool's tile layout (KVQ_CODES, KVQ_TILE) is in kernels.h.

// One head row held by a warp, lane l values [4l, 4l + 4): block b is lanes
// 8b .. 8b + 7.  Returns the lane's four codes (bytes, value 4l + i in byte
// i), its block's fp16 scale, and the values the cache then holds (fp16
// scale times code, exact in FP32).
Q3_DEV void kvq_pack(const float (&y)[4], uint32_t& codes, __half& scale, float (&deq)[4]) {
    float am = fmaxf(fmaxf(fabsf(y[0]), fabsf(y[1])), fmaxf(fabsf(y[2]), fabsf(y[3])));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 1));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 2));
    am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, 4));
    const float d = __fdiv_rn(am, 127.0f);
    scale = __float2half_rn(d);
    const float ds = __half2float(scale);
    codes = 0;
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        int q = 0;
        if (d != 0.0f) q = (int)fminf(fmaxf(rintf(__fdiv_rn(y[e], d)), -127.0f), 127.0f);
        codes |= (uint32_t)(q & 0xff) << (8 * e);
        deq[e] = ds * (float)q;
    }
}

// Store a packed row at position r of a pool tile (lane l: codes of values
// [4l, 4l + 4); lane 8b: the scale of block b).
Q3_DEV void kvq_store(uint8_t* tile, int r, uint32_t codes, __half scale, int lane) {
    *reinterpret_cast<uint32_t*>(tile + r * 128 + lane * 4) = codes;
    if ((lane & 7) == 0) *reinterpret_cast<__half*>(tile + KVQ_CODES + (r * 4 + (lane >> 3)) * 2) = scale;
}

// Four codes (bytes of w) times the fp16 scale d, each product rounded once to
// fp16 (the tensor-core operand type): two fp16 pairs.  A byte b becomes
// 1024 + (b ^ 0x80) as the fp16 0x64 << 8 | (b ^ 0x80), exactly; subtracting
// 1152 leaves the signed code, and the multiply rounds the exact product.
Q3_DEV uint2 kvq_dequant4(uint32_t w, __half d) {
    const uint32_t f = w ^ 0x80808080u;
    const uint32_t lo = __byte_perm(f, 0x64646464u, 0x5140);      // bytes 0, 1
    const uint32_t hi = __byte_perm(f, 0x64646464u, 0x5342);      // bytes 2, 3
    const __half2 bias = __half2half2(__ushort_as_half((unsigned short)0x6480));   // 1152
    const __half2 dd = __half2half2(d);
    __half2 a = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&lo), bias), dd);
    __half2 b = __hmul2(__hsub2(*reinterpret_cast<const __half2*>(&hi), bias), dd);
    return make_uint2(*reinterpret_cast<uint32_t*>(&a), *reinterpret_cast<uint32_t*>(&b));
}

// ---------------------------------------------------------------- PDL
// Programmatic dependent launch: a kernel may start while its predecessor
// drains; it must call grid_dep_wait() before touching what the predecessor
// writes.  Both are no-ops when the launch did not opt in.
Q3_DEV void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
Q3_DEV void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- mbarrier
Q3_DEV uint32_t smem_u32(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

Q3_DEV void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count));
}

Q3_DEV void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

Q3_DEV void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}

Q3_DEV void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}

Q3_DEV bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete.  Returns false (and
// sets the timeout status bit) when Q3_WAIT_LIMIT_NS passes first.
Q3_DEV bool mbar_wait(uint64_t* bar, uint32_t parity, int* status) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > Q3_WAIT_LIMIT_NS) {
            set_status(status, Q3_STATUS_TIMEOUT);
            return false;
        }
    }
}

// ---------------------------------------------------------------- TMA
Q3_DEV void tma_load_2d(void* dst, const void* tmap, uint64_t* bar, int c0, int c1) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];"
        :: "r"(smem_u32(dst)), "l"(tmap), "r"(smem_u32(bar)), "r"(c0), "r"(c1)
        : "memory");
}

// 1-D bulk copy global -> shared completing on an mbarrier (16-byte aligned
// addresses, size a multiple of 16)
Q3_DEV void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        :: "r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}

// asynchronous prefetch of a contiguous global range into L2 (16-byte
// aligned, size a multiple of 16)
Q3_DEV void prefetch_l2(const void* src, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(src), "r"(bytes) : "memory");
}

// This CTA's share of an L2 prefetch: each range is cut into n_ctas equal
// 16-byte-aligned slices.
Q3_DEV void issue_l2_prefetch(const L2Prefetch& pf, int cta, int n_ctas) {
#pragma unroll
    for (int i = 0; i < 3; ++i) {
        if (!pf.bytes[i]) continue;
        const uint64_t slice = ((pf.bytes[i] + n_ctas - 1) / n_ctas + 15) & ~uint64_t(15);
        const uint64_t off = slice * cta;
        if (off >= pf.bytes[i]) continue;
        const uint64_t n = min(slice, pf.bytes[i] - off) & ~uint64_t(15);
        if (n) prefetch_l2(static_cast<const uint8_t*>(pf.ptr[i]) + off, (uint32_t)n);
    }
}

// named barrier over a subset of the CTA's warps
Q3_DEV void named_bar(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// named barrier that also ANDs a predicate over the participating threads
Q3_DEV bool named_bar_and(int id, int threads, bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\t"
                 "setp.ne.u32 p, %1, 0;\n\t"
                 "barrier.cta.red.and.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred), "r"(id), "r"(threads) : "memory");
    return r != 0;
}

Q3_DEV void prefetch_tmap(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}

// ---------------------------------------------------------------- tcgen05
Q3_DEV void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
}
Q3_DEV void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
Q3_DEV void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;"
                 :: "r"(taddr), "r"(ncols) : "memory");
}
Q3_DEV void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
Q3_DEV void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, kind::f16 (16-bit inputs, f32 accumulate).
Q3_DEV void tc_mma_f16(uint32_t tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                       uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
                 : "memory");
}

// Arrive on an mbarrier once every tcgen05 op issued so far by this thread
// has completed.
Q3_DEV void tc_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

// 32 lanes x 32 consecutive 32-bit columns: thread i of the warp gets row
// (lane base + i), columns [col, col + 32).
Q3_DEV void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
          "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
          "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]),
          "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]),
          "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
Q3_DEV void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Shared-memory matrix descriptor of a K-major operand tile stored with the
// 128-byte swizzle (rows of 64 16-bit elements, 8-row groups 1024 bytes apart), as TMA
// writes it with CU_TENSOR_MAP_SWIZZLE_128B.  Bits: start address >> 4
// [0,14), leading offset >> 4 [16,30) (unused for this layout, 1), stride
// offset >> 4 [32,46) = 1024 >> 4, version 1 [46,48), swizzle mode 2
// (128-byte) [61,64).
Q3_DEV uint64_t smem_desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor of kind::f16 with fp16 A and B (both K-major, A/B
// format field 0 at [7,10) and [10,13)) and an f32 accumulator (D format 1
// at [4,6)), for an M x N tile: N >> 3 at [17,23), M >> 4 at [24,29).
__host__ __device__ constexpr uint32_t idesc_f16_f32(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// fp16 of an activation; |v| beyond the fp16 range is reported (the caller
// ORs the flag into the status word once) rather than silently saturated.
Q3_DEV __half to_f16(float v, bool& out_of_range) {
    out_of_range |= !(fabsf(v) <= 65504.0f);
    return __float2half_rn(v);
}

}  // namespace q3
