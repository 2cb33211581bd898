// kernels.h -- host-side launch interface of the sm_103a kernels.
// Every launcher is asynchronous on the given stream and returns the CUDA
// launch status.  Shapes are validated by the runtime before these calls.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace q3 {

// ---------------------------------------------------------------- Q8_0 K/V cache layout
// With the opt-in Q8_0 cache a (block, K or V, KV head) tile of the pool is
// KVQ_TILE bytes: the codes [32 positions][128] int8, then the scales
// [32 positions][4] fp16 (one per 32 values of a head row) -- 136 bytes per
// position and head against 256 in BF16.
constexpr int KVQ_CODES = 32 * 128;
constexpr int KVQ_TILE = KVQ_CODES + 32 * 4 * 2;

// ---------------------------------------------------------------- kernel attributes
// A kernel that takes more than 48 KB of dynamic shared memory must be
// allowed it on every device it launches on.  `done` keeps one bit per
// device id (ids 0..63) so the attribute is set once per device; devices
// past 63 set it on every launch.
template <typename Kernel>
cudaError_t allow_smem_per_device(Kernel* kernel, int bytes, std::atomic<unsigned long long>& done)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long bit = (dev >= 0 && dev < 64) ? 1ull << dev : 0ull;
    if (bit && (done.load(std::memory_order_acquire) & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess && bit) done.fetch_or(bit, std::memory_order_acq_rel);
    return e;
}

// ---------------------------------------------------------------- launch
// How a kernel is launched: stream, and whether it may start early under
// programmatic dependent launch.
struct Launch {
    cudaStream_t stream;
    bool pdl;
    int64_t* counter;   // incremented per launch
};

// ---------------------------------------------------------------- GEMM
// D[M x N] = A[M x K] * B[N x K]^T on tcgen05 tensor cores.  A is the
// weight matrix (fp16, row-major [out][in]); B holds N token rows (fp16
// [rows][K]).  Output element (n, m) goes to out[n * ldo + m].
enum Epi : int {
    EPI_STORE_F32 = 0,   // out = acc (f32)
    EPI_ADD_F32 = 1,     // out += acc (f32 residual)
    EPI_STORE_F16 = 2,   // out = fp16(acc)
    EPI_SWIGLU_F16 = 3,  // paired gate/up tile: out[n][f] = fp16(silu(g) * u)
    EPI_SWIGLU_F32 = 4,
    EPI_QKV_ROPE = 5,    // QKV tiles, one head each (q, then k, then v heads): the q/k head
                         // RMSNorm and RoPE, q as fp16 into rope.q_out16, K and V as bf16 into the
                         // pool through the block table (rope; the BF16 cache)
};

struct RopeArgs {
    const float* qkv;          // [T][n_q*128 + 2*n_kv*128]
    int T, n_q, n_kv;
    const __nv_bfloat16* q_gain;
    const __nv_bfloat16* k_gain;
    float eps;
    const float2* rope;        // [max_ctx][64] (cos, sin)
    const int* row_pos;        // [T]
    const int* row_slot;       // [T] session slot
    const int* tables;         // [slots][max_blocks]
    int max_blocks;
    __nv_bfloat16* kv_layer;   // pool base of this layer: [n_blocks][2][n_kv][32][128]
    uint8_t* kvq_layer;        // Q8_0 cache: pool base of this layer, [n_blocks][2][n_kv] tiles of
                               // KVQ_TILE bytes (null: the BF16 cache at kv_layer)
    int64_t layer_stride;      // elements between layers (unused by the kernel)
    int n_blocks;
    float* q_out;              // [T][n_q*128] f32, or null
    __half* q_out16;           // [T][n_q*128] fp16, or null
    int* status;
};


struct GemmArgs {
    int M, N, K;          // M multiple of 128; K multiple of 64
    int a_tiles0, a_tiles1;  // plain mode: 128-row tiles [0,t0) from map a0, [t0,t1) from a1, rest a2
    int pair;             // 1: tile t takes rows [64 t, 64 t + 64) of a0 (gate) then of a1 (up)
    int k_splits;         // > 1: partial sums to ws, then gemm_splitk_reduce
    int epi;
    void* out;
    int ldo;
    float* ws;
    int early_a;          // request the first stages' weight tiles before the dependency wait
                          // (helps short GEMMs, whose ring ramp is a large part of the launch)
    RopeArgs rope;        // EPI_QKV_ROPE: the rows' positions, slots, tables, gains and outputs
    int* status;
};

// Box shapes a tensor map must have for the GEMM: weights 64 (K) x 128
// rows (64 rows in pair mode); activations 64 x BN.
int gemm_block_n(int N);          // smallest tile width covering N token rows
bool gemm_block_n_supported(int bn);   // 32, 64, 96, 128, 144, 160, 176, 192 or 256
cudaError_t launch_gemm(const Launch& L, const CUtensorMap& a0, const CUtensorMap& a1,
                        const CUtensorMap& a2, const CUtensorMap& b, int bn,
                        const GemmArgs& g);
cudaError_t launch_gemm_splitk_reduce(const Launch& L, const GemmArgs& g);
// Split-K finish of a residual-add GEMM (plain rows, EPI_ADD_F32, M <= 5120)
// fused with the RMSNorm of the updated rows: out[n] += sum of the partials
// in split order, then h[n] = fp16(RMSNorm(out[n]) * gain), one CTA a row.
bool gemm_add_norm_ok(const GemmArgs& g);
cudaError_t launch_gemm_splitk_add_norm(const Launch& L, const GemmArgs& g, const __nv_bfloat16* gain, float eps,
                                        __half* h);

// Weights the next launch will stream: up to three contiguous ranges that a
// kernel prefetches into L2 (a capped prefix, split over its CTAs) so HBM
// stays busy across the kernel boundary.
struct L2Prefetch {
    const void* ptr[3];
    uint64_t bytes[3];
};

// ---------------------------------------------------------------- GEMV
// One token row: y[r] = sum_k W[r][k] * h[k], with h = x (or RMSNorm(x) * g
// when norm_gain is set).  BF16 weights or Q8_0 planes (int8 quants +
// fp16 scales per 32).
struct GemvArgs {
    const void* w[3];          // weight planes (bf16, or int8 quants for Q8_0)
    const __half* scales[3];   // Q8_0 scale planes [rows][K/32] (else null)
    int rows[3];               // rows per tensor (plain mode stacks them)
    int n_tensors;
    int pair;                  // w[0] = gate, w[1] = up, output F = rows[0] features
    int K;
    int warps_per_row;         // 1, 2, 4 or 8
    const float* x;            // [K]
    const __nv_bfloat16* norm_gain;  // null: no norm
    float eps;
    int epi;                   // EPI_STORE_F32, EPI_ADD_F32, EPI_SWIGLU_F32
    float* out;
    int* status;
    // optional greedy argmax of the outputs (lowest index on ties): per-CTA
    // partials, merged by the last CTA to finish (ticket counter kept at 0)
    int32_t* argmax_out;
    float* am_val;             // [grid]
    int* am_idx;               // [grid]
    int* am_counter;
    L2Prefetch next;           // weights of the next launch (bytes 0: none)
};
cudaError_t launch_gemv(const Launch& L, int scheme, const GemvArgs& a);
// AFFINE4_GS32 matvec (w: lane-major code planes, scales: (scale, bias)
// planes, as launch_a4_planes derives them; rows multiples of 8, K of 128)
cudaError_t launch_gemv_a4(const Launch& L, const GemvArgs& a);
int gemv_a4_warps_per_tile(int rows, int K, int pair);
// canonical 20-byte groups [rows][K/32] -> the matvec's code and (scale, bias) planes
// (codes: rows * K / 2 bytes; sb: rows * K / 32 * 4 bytes)
cudaError_t launch_a4_planes(cudaStream_t s, const uint8_t* groups, int rows, int K, void* codes, void* sb);
// segments per row: a power of two, preferably with at most 8 loads per lane
int gemv_warps_per_row(int rows, int K, int scheme, int pair);
int gemv_max_grid();

// ---------------------------------------------------------------- elementwise
cudaError_t launch_embed(const Launch& L, const int32_t* tokens, int T, const __nv_bfloat16* E,
                         int H, int vocab, float* x, int* status);
// h[r] = fp16(RMSNorm(x[rows[r]]) * g) for r < n (rows null: r itself)
cudaError_t launch_rmsnorm_f16(const Launch& L, const float* x, const int* rows, int n, int H,
                               const __nv_bfloat16* g, float eps, __half* h, int* status);

cudaError_t launch_qk_norm_rope_append(const Launch& L, const RopeArgs& a);

struct AttnArgs {
    const float* q;            // [T][n_q][128], normed and rotated (unfused rounds)
    const float* qkv;          // [T][(n_q + 2 n_kv) 128] raw projections (fused decode rounds)
    const float* qkv_ws;       // or, with qkv_splits > 1, the QKV GEMM's split-K partials
    int qkv_splits;            // ([split][T][(n_q + 2 n_kv) 128]), summed here in split order
    const __nv_bfloat16* q_gain;
    const __nv_bfloat16* k_gain;
    const float2* rope;        // [max_ctx][64] (cos, sin)
    float eps;
    int T, n_q, n_kv;
    const int* row_pos;
    const int* row_slot;
    const int* row_order;      // [T] row of grid z-index z (longest context first), or null: row z
    const int* tables;
    int max_blocks;
    __nv_bfloat16* kv_layer;   // pool slab of this layer; written by the fused append
    uint8_t* kvq_layer;        // Q8_0 cache: the layer's tiles instead (null: BF16 cache)
    int n_blocks;
    int n_splits;
    float* part_ml;            // [T][n_q][n_splits][2]
    float* part_o;             // [T][n_q][n_splits][128]
    int* counters;             // [T][n_kv], zero between calls (the last split CTA resets it)
    L2Prefetch next;           // weights of the next launch
    void* out;                 // [T][n_q*128], f32 or fp16
    int out_f16;
    int* status;
};
// Prefill attention on tensor cores (mma.sync, fp16): query tiles of 64 rows
// of one session, one query head per CTA, 64-position K/V tiles.
struct PrefillAttnArgs {
    const __half* q;           // [T][n_q][128] normed, rotated (fp16)
    int T, n_q, n_kv;
    const int* row_pos;
    const int* row_slot;
    const int* tile_row0;      // [n_tiles] first row of each 64-row query tile, longest context first
    const int* tile_rows;      // [n_tiles] rows in the tile (<= 64)
    int n_tiles;
    int* work_counter;         // work queue position, zero between launches (the kernel resets it)
    const int* sched_start;    // tcgen05 kernel: [grid + 1] first item of each CTA
    const int* sched_items;    // tcgen05 kernel: items (tile * n_kv + KV head), per CTA in order
    int kv_row0;               // tcgen05 kernel: row of this layer's first K row in the pool's
                               // tensor map (rows of 128 bf16: [layer][block][K/V][n_kv][32])
    const int* tables;
    int max_blocks;
    const __nv_bfloat16* kv_layer;
    const uint8_t* kvq_layer;  // Q8_0 cache (mma.sync kernel only): the layer's tiles (null: BF16)
    int n_blocks;
    __half* out;               // [T][n_q * 128] fp16
    int* status;
};
cudaError_t launch_prefill_attention(const Launch& L, const PrefillAttnArgs& a);
// tcgen05 variant: query tiles of prefill_tc_rows() positions carry all query
// heads of a KV head; CTA c takes items sched_start[c] .. sched_start[c + 1].
int prefill_tc_rows(int n_q, int n_kv);
size_t prefill_tc_smem();
cudaError_t launch_prefill_attention_tc(const Launch& L, const CUtensorMap& tkv, const PrefillAttnArgs& a, int grid);

// fused: every row is the single new token of its session; q/k norm, RoPE
// and the K/V append of that token happen inside the attention kernel.
cudaError_t launch_attention(const Launch& L, const AttnArgs& a, bool fused);
// blocks of context each split CTA should take, and the most splits a row may use
int attention_blocks_per_cta();
int attention_max_splits();

// ---------------------------------------------------------------- fused decode step
// The whole one-token round of one session in one persistent kernel: one CTA
// per SM, a producer warp streaming weight and KV tiles into a shared-memory
// ring with bulk copies, and consumer warps computing every stage (QKV, q/k
// norm + RoPE + KV append + attention, O, gate/up + SwiGLU, down, lm_head +
// argmax), separated by grid-wide barriers.
struct DecodeLayer {
    const __nv_bfloat16* attn_norm;
    const __nv_bfloat16* q_norm;
    const __nv_bfloat16* k_norm;
    const __nv_bfloat16* ffn_norm;
    const void* w[7];          // wq, wk, wv, wo, w_gate, w_up, w_down: bf16, or Q8_0 int8 quants
    const __half* sc[7];       // Q8_0 fp16 scale planes [rows][K/32] (null for bf16)
};

struct DecodeArgs {
    int n_layers, H, F, V, n_q, n_kv;
    float eps;
    int q8;                    // projections are Q8_0 planes (the lm_head is bf16 either way)
    const DecodeLayer* layers; // device [n_layers]
    const __nv_bfloat16* embed;
    const __nv_bfloat16* final_norm;
    const __nv_bfloat16* lm_head;
    const float2* rope;        // [max_ctx][64] (cos, sin)
    const int32_t* token;      // [1]
    const int* row_pos;        // [1] position of the new token
    const int* row_slot;       // [1] session slot
    const int* tables;
    int max_blocks;
    __nv_bfloat16* kv;         // pool base: [n_layers][n_blocks][2][n_kv][32][128]
    int64_t layer_kv;          // elements per layer
    int n_blocks;
    int n_splits;              // attention splits per KV head (n_kv * n_splits <= grid)
    float* x;                  // [H] residual
    float* qkv;                // [(n_q + 2 n_kv) 128]
    float* att;                // [n_q 128]
    float* ffn;                // [F]
    float* part_ml;            // [n_q][n_splits][2]
    float* part_o;             // [n_q][n_splits][128]
    int* counters;             // [n_kv], zero between calls
    float* logits;             // [V]
    int32_t* argmax_out;       // [1] or null
    float* am_val;             // [grid]
    int* am_idx;               // [grid]
    int* am_counter;           // zero between calls
    unsigned long long* bar;   // grid barrier counter (monotonic across launches)
    unsigned long long bar_base;   // its value when this launch starts
    int n_slots;               // ring depth
    int* status;
};
// Shared memory of the fused step for these dimensions and ring depth; 0 if
// the shapes are outside what the kernel handles.
size_t decode_step_smem(int H, int F, int n_q, int n_kv, int q8, int n_slots, int n_splits, int grid,
                        int n_layers);
int decode_step_slot_bytes();
// Grid barriers one launch performs (each adds grid to *bar).
int decode_step_barriers(int n_layers);
cudaError_t decode_step_prepare(size_t smem);
cudaError_t launch_decode_step(const Launch& L, const DecodeArgs& a, int grid, size_t smem);

cudaError_t launch_argmax(const Launch& L, const float* logits, int rows, int V, int32_t* out);

// Q8_0 K/V rows: n rows of 128 floats packed into canonical Q8_0 blocks (4 x
// 34 bytes a row: fp16 scale, then 32 codes), by the cache writers' rule.
cudaError_t launch_kv_pack_q8(cudaStream_t s, const float* rows, int n, uint8_t* out);

// Q8_0: canonical blocks -> (int8 plane, fp16 scale plane); planes -> fp16
// tensor-core operand; bf16 -> canonical blocks.
cudaError_t launch_q8_split(cudaStream_t s, const uint8_t* blocks, int64_t nblocks, int8_t* qs,
                            __half* scales);
cudaError_t launch_q8_to_f16(const Launch& L, const int8_t* qs, const __half* scales, int64_t n,
                             __half* w);
// fp16 copy of bf16 weights for the tensor-core path; counts values that do
// not convert exactly (|w| < 2^-17, rounded) in *inexact and values beyond
// the fp16 range in *overflow.
cudaError_t launch_bf16_to_f16(cudaStream_t s, const __nv_bfloat16* w, int64_t n, __half* out,
                               unsigned long long* inexact, unsigned long long* overflow);
cudaError_t launch_quantize_q8_0(cudaStream_t s, const __nv_bfloat16* w, int64_t n, uint8_t* blocks);
// AFFINE4_GS32: bf16 -> 20-byte groups; groups -> fp16 tensor-core operand,
// counting values beyond the fp16 range in *overflow (may be NULL).
cudaError_t launch_quantize_affine4(cudaStream_t s, const __nv_bfloat16* w, int64_t n, uint8_t* groups);
cudaError_t launch_affine4_to_f16(cudaStream_t s, const uint8_t* groups, int64_t n, __half* w,
                                  unsigned long long* overflow);

}  // namespace q3
