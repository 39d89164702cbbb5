// Allocation-free entry point: momentum, Nesterov direction and Frobenius
// normalisation of ONE matrix, with its scratch in a fixed static device array.
//
// Some callers cannot call cudaMalloc at the point where they run this step:
// frameworks whose device memory all belongs to their own pool or arena (a
// foreign allocation would break their accounting or fragment it), code that
// runs where an allocation would synchronise the device or is forbidden (a
// latency-critical loop, a host callback), and embedded users whose memory
// budget is fixed when the library is loaded.  For them this entry point keeps
// its scratch -- one partial sum of u^2 per 64 x 64 tile plus the resulting
// scale -- in the file-scope array below instead of a handle's arena.
//
// Limits and sharing:
//   * at most kNoallocMaxTiles = 65536 tiles of 64 x 64 (e.g. 16384 x 16384);
//     larger matrices are rejected with MUON_ERR_SHAPE;
//   * the array (65536 + 64 floats, about 256 KB) exists once per GPU that
//     loads the library and stays allocated until the process exits;
//   * every call uses the same array and leaves its contents behind.  Each
//     call writes every partial sum it later reads and the scale it uses, so
//     nothing has to start at zero; but two calls whose work overlaps on the
//     GPU (different streams, or different host threads) race on the array and
//     produce wrong results.  Order such calls on one stream.
//   * in host code `g_noalloc_scratch` names a host-side stand-in, not a device
//     address: the device address is fetched with cudaGetSymbolAddress on the
//     first call made while a device is current, and again whenever that
//     device's current context has changed since (for instance after
//     cudaDeviceReset, which unloads the module that holds the array).  Make
//     the first call on a device, and the first call after a reset, outside
//     any stream capture.
//   * momentum, x0 and (for fp32 gradients) grad must not overlap; identical
//     pointers are rejected with MUON_ERR_ARG.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdio>
#include <mutex>

#include "../../include/muon.h"
#include "ptx_sm103.cuh"

namespace {

constexpr int kNoallocTile = 64;
constexpr int kNoallocMaxTiles = 65536;
constexpr int kScaleSlot = kNoallocMaxTiles;   // scale s = 1 / (||u||_F + 1e-7)
constexpr int kMaxDevices = 64;

static __device__ __align__(256) float g_noalloc_scratch[kNoallocMaxTiles + 64];

std::mutex g_setup_mu;
float* g_scratch_dev[kMaxDevices] = {};
CUcontext g_scratch_ctx[kMaxDevices] = {};  // context the address was looked up in

typedef CUresult (*PFN_ctxGetCurrent)(CUcontext*);

// cuCtxGetCurrent through the runtime's driver entry point (no link against libcuda)
CUcontext current_context() {
    static PFN_ctxGetCurrent fn = nullptr;
    if (fn == nullptr) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        fn = reinterpret_cast<PFN_ctxGetCurrent>(p);
    }
    CUcontext c = nullptr;
    return fn(&c) == CUDA_SUCCESS ? c : nullptr;
}

// momentum buffer and Nesterov direction of one element (lerp or mul/add form)
__device__ __forceinline__ float na_momentum(float g, float& b, float mu, int lerp_form, int nesterov) {
    if (lerp_form) {
        b = fmaf(1.f - mu, g - b, b);
        return nesterov ? fmaf(mu, b - g, g) : b;
    }
    b = fmaf(mu, b, g);
    return nesterov ? fmaf(mu, b, g) : b;
}

struct NaParams {
    const void* grad;
    float* mom;
    float* x0;
    float* scratch;  // device address of g_noalloc_scratch
    int64_t rows, cols;
    int32_t tiles_c;
    float mu;
    int32_t grad_f32, lerp_form, nesterov;
};

// One 64 x 64 tile per block: updates the momentum, writes u into x0 and the
// tile's sum of u^2 into scratch[tile].
__global__ void __launch_bounds__(256) k_na_momentum(const NaParams p) {
    __shared__ float red[8];
    const int tile = blockIdx.x;
    const int64_t r0 = (int64_t)(tile / p.tiles_c) * kNoallocTile, c0 = (int64_t)(tile % p.tiles_c) * kNoallocTile;
    float sumsq = 0.f;
    for (int e = threadIdx.x; e < kNoallocTile * kNoallocTile; e += 256) {
        const int64_t r = r0 + e / kNoallocTile, c = c0 + e % kNoallocTile;
        if (r >= p.rows || c >= p.cols) continue;
        const int64_t i = r * p.cols + c;
        const float g = p.grad_f32 ? static_cast<const float*>(p.grad)[i]
                                   : muon::bf2f(static_cast<const uint16_t*>(p.grad)[i]);
        float b = p.mom[i];
        const float u = na_momentum(g, b, p.mu, p.lerp_form, p.nesterov);
        p.mom[i] = b;
        p.x0[i] = u;
        sumsq = fmaf(u, u, sumsq);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sumsq += __shfl_xor_sync(0xffffffffu, sumsq, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = sumsq;
    __syncthreads();
    if (threadIdx.x == 0) {
        float t = 0.f;
        for (int w = 0; w < 8; ++w) t += red[w];
        p.scratch[tile] = t;
    }
}

// Sums the tiles' partial sums in a fixed order and stores the scale.
__global__ void __launch_bounds__(256) k_na_norm(float* scratch, int ntiles) {
    __shared__ float red[256];
    float s = 0.f;
    for (int t = threadIdx.x; t < ntiles; t += 256) s += scratch[t];
    red[threadIdx.x] = s;
    __syncthreads();
    for (int w = 128; w > 0; w >>= 1) {
        if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
        __syncthreads();
    }
    if (threadIdx.x == 0) scratch[kScaleSlot] = 1.f / (sqrtf(red[0]) + 1e-7f);
}

__global__ void __launch_bounds__(256) k_na_scale(float* x0, int64_t n, const float* scratch) {
    const float s = scratch[kScaleSlot];
    for (int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x; i < n; i += (int64_t)gridDim.x * 256) x0[i] *= s;
}

}  // namespace

extern "C" int muon_nesterov_normalize_noalloc(const void* grad, int32_t grad_dtype, float* momentum, float* x0,
                                               int64_t rows, int64_t cols, float mu, int32_t lerp_form,
                                               int32_t nesterov, void* stream) {
    if (grad == nullptr || momentum == nullptr || x0 == nullptr) return MUON_ERR_ARG;
    if (grad_dtype != MUON_GRAD_BF16 && grad_dtype != MUON_GRAD_F32) return MUON_ERR_ARG;
    // the three buffers are read and written element by element in one pass: they must not alias
    if (static_cast<const void*>(momentum) == static_cast<const void*>(x0)) return MUON_ERR_ARG;
    if (grad_dtype == MUON_GRAD_F32 && (grad == static_cast<const void*>(momentum) || grad == static_cast<const void*>(x0)))
        return MUON_ERR_ARG;
    if (rows < 1 || cols < 1) return MUON_ERR_SHAPE;
    // reject sizes beyond the scratch before any product that could overflow
    const int64_t max_side = (int64_t)kNoallocTile * kNoallocMaxTiles;
    if (rows > max_side || cols > max_side) return MUON_ERR_SHAPE;
    const int64_t tiles_r = (rows + kNoallocTile - 1) / kNoallocTile;
    const int64_t tiles_c = (cols + kNoallocTile - 1) / kNoallocTile;
    if (tiles_r > kNoallocMaxTiles / tiles_c) {
        fprintf(stderr,
                "muon_nesterov_normalize_noalloc: %lld x %lld needs more than %d tiles of 64 x 64 (the static "
                "scratch's limit)\n",
                (long long)rows, (long long)cols, kNoallocMaxTiles);
        return MUON_ERR_SHAPE;
    }
    // an error left over from the caller's earlier work is not this call's: report it as such
    if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MUON_ERR_CUDA;
    float* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lk(g_setup_mu);
        const CUcontext ctx = current_context();
        if (g_scratch_dev[dev] == nullptr || ctx != g_scratch_ctx[dev]) {
            void* ptr = nullptr;
            if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
                cudaGetLastError();
                return MUON_ERR_CUDA;
            }
            g_scratch_dev[dev] = static_cast<float*>(ptr);
            g_scratch_ctx[dev] = ctx;
        }
        scratch = g_scratch_dev[dev];
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    NaParams p;
    p.grad = grad;
    p.mom = momentum;
    p.x0 = x0;
    p.scratch = scratch;
    p.rows = rows;
    p.cols = cols;
    p.tiles_c = (int32_t)tiles_c;
    p.mu = mu;
    p.grad_f32 = grad_dtype == MUON_GRAD_F32;
    p.lerp_form = lerp_form;
    p.nesterov = nesterov;
    const int ntiles = (int)(tiles_r * tiles_c);
    k_na_momentum<<<ntiles, 256, 0, s>>>(p);
    if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;
    k_na_norm<<<1, 256, 0, s>>>(scratch, ntiles);
    if (cudaGetLastError() != cudaSuccess) return MUON_ERR_CUDA;
    const int64_t n = rows * cols;
    int64_t blocks = (n + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    k_na_scale<<<(unsigned)blocks, 256, 0, s>>>(x0, n, scratch);
    return cudaGetLastError() == cudaSuccess ? MUON_OK : MUON_ERR_CUDA;
}
