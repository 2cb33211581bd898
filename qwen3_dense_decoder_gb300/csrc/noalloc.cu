// noalloc.cu -- a split-K tensor-core matmul that allocates no device memory.
//
// Some callers cannot call cudaMalloc at the point where they need a matmul:
// a host framework that owns all device memory through its own allocator and
// forbids outside allocations, a plug-in that runs inside someone else's
// process and may not grow its footprint, or a latency-critical loop where
// cudaMalloc's implicit device synchronisation is not acceptable.  For them,
// q3_op_matmul_splitk_noalloc runs the same tcgen05 GEMM as q3_op_matmul with
// its K dimension split across CTAs, and keeps the split partial sums in a
// fixed scratch array that is part of the library image instead of a
// cudaMalloc'ed workspace.
//
// The scratch is a file-scope __device__ array of Q3_NOALLOC_SCRATCH_FLOATS
// floats (8 MiB).  Every GPU that loads the library holds it until the
// process exits.  Host code cannot use the array's name as a device address
// (it is a host-side stand-in), so the first call on each device looks the
// address up with cudaGetSymbolAddress while that device is current and
// caches it.  That first call also loads this file's device code, which is
// when the driver commits the array's memory on that device: make it outside
// any latency-critical region.  All calls share the one array: two calls
// whose kernels overlap on the GPU (different streams, no ordering between
// them) race on it.  Each call reads the status word of its bounded waits
// back into a host variable and waits for the stream, so it returns only
// once its kernels have finished and reports a wait that ran out.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cstdio>
#include <mutex>

#include "../../include/q3.h"
#include "common.cuh"
#include "kernels.h"

// the fixed scratch (file scope; host code must not take its name as a device
// address, see device_scratch below) and the status word of the bounded waits
static __device__ __align__(256) float q3_noalloc_scratch[Q3_NOALLOC_SCRATCH_FLOATS];
static __device__ __align__(256) int q3_noalloc_status;

namespace {

constexpr int kMaxDevices = 64;

struct DeviceScratch {
    float* scratch = nullptr;
    int* status = nullptr;
};

std::mutex g_mu;
DeviceScratch g_dev[kMaxDevices];

thread_local char g_msg[256];

int noalloc_fail(int code, const char* msg)
{
    snprintf(g_msg, sizeof g_msg, "%s", msg);
    return code;
}

// Device addresses of the scratch array and status word on the current
// device, looked up once per device.
bool device_scratch(DeviceScratch* out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceScratch& d = g_dev[dev];
    if (!d.scratch) {
        void* s = nullptr;
        void* st = nullptr;
        if (cudaGetSymbolAddress(&s, q3_noalloc_scratch) != cudaSuccess) return false;
        if (cudaGetSymbolAddress(&st, q3_noalloc_status) != cudaSuccess) return false;
        d.scratch = static_cast<float*>(s);
        d.status = static_cast<int*>(st);
    }
    *out = d;
    return true;
}

bool tmap_f16_2d(CUtensorMap* m, const void* ptr, uint64_t rows, uint64_t cols, uint32_t box_rows)
{
    // the driver's encoder, resolved once and thread-safely (a function-local static)
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = []() -> PFN_cuTensorMapEncodeTiled_v12000 {
        cudaDriverEntryPointQueryResult q;
        void* p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 2};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t elem[2] = {1, 1};
    return fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, elem,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

extern "C" {

const char* q3_noalloc_last_error(void) { return g_msg; }

int q3_op_matmul_splitk_noalloc(const void* w_dev, const void* x_dev, int M, int N, int K,
                                int k_splits, float* y_dev, void* stream)
{
    using namespace q3;
    if (!w_dev || !x_dev || !y_dev || M < 128 || M % 128 || K < 64 || K % 64 || N < 1 ||
        (reinterpret_cast<uintptr_t>(w_dev) & 15) || (reinterpret_cast<uintptr_t>(x_dev) & 15))
        return noalloc_fail(Q3_ERR_INVALID_ARG, "matmul_splitk_noalloc: bad argument");
    if (k_splits < 2 || k_splits > 8 || K / 64 < k_splits)
        return noalloc_fail(Q3_ERR_INVALID_ARG,
                            "matmul_splitk_noalloc: k_splits must be in [2, 8] and at most K/64");
    if ((long long)k_splits * N * M > (long long)Q3_NOALLOC_SCRATCH_FLOATS)
        return noalloc_fail(Q3_ERR_INVALID_ARG,
                            "matmul_splitk_noalloc: k_splits * N * M exceeds the fixed scratch "
                            "(Q3_NOALLOC_SCRATCH_FLOATS floats)");
    DeviceScratch d;
    if (!device_scratch(&d))
        return noalloc_fail(Q3_ERR_CUDA, "matmul_splitk_noalloc: scratch address lookup failed");
    const int bn = gemm_block_n(N);
    CUtensorMap a, b;
    if (!tmap_f16_2d(&a, w_dev, M, K, 128) || !tmap_f16_2d(&b, x_dev, (N + 255) / 256 * 256, K, bn))
        return noalloc_fail(Q3_ERR_CUDA, "matmul_splitk_noalloc: tensor map encoding failed");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the status word must start at zero; the partials are fully overwritten
    if (cudaMemsetAsync(d.status, 0, sizeof(int), s) != cudaSuccess)
        return noalloc_fail(Q3_ERR_CUDA, "matmul_splitk_noalloc: status clear failed");
    GemmArgs g{};
    g.M = M; g.N = N; g.K = K;
    g.a_tiles0 = g.a_tiles1 = M / 128;
    g.k_splits = k_splits;
    g.epi = EPI_STORE_F32;
    g.out = y_dev; g.ldo = M;
    g.ws = d.scratch;
    g.status = d.status;
    Launch L{s, false, nullptr};
    cudaError_t e = launch_gemm(L, a, a, a, b, bn, g);
    if (e == cudaSuccess) e = launch_gemm_splitk_reduce(L, g);
    // the status word comes back to a host int on this stack (no allocation):
    // a bounded wait that ran out leaves partial sums behind, so it is an error
    int word = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&word, d.status, sizeof(int), cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return noalloc_fail(Q3_ERR_CUDA, cudaGetErrorString(e));
    if (word) {
        snprintf(g_msg, sizeof g_msg, "matmul_splitk_noalloc: device status 0x%x (a bounded wait ran out)",
                 word);
        return Q3_ERR_DEVICE_CHECK;
    }
    return Q3_OK;
}

}  // extern "C"
