// CUDA-core Newton-Schulz products: a slow debugging engine (MUON_GEMM_SIMT).
//
// Computes the same three products and epilogues as the tcgen05 kernels but
// naively: full m x m results (no triangle, no mirror), plain global loads,
// fp32 accumulation in registers.  It exists to cross-check the tensor-core
// path (descriptors, swizzles, symmetric tiles) on the device; it is never timed.
#include "muon_internal.h"
#include "ptx_sm103.cuh"

namespace muon {

template <int MODE>
__global__ void __launch_bounds__(256) k_ns_gemm_simt(const __grid_constant__ GemmParams p, int gslot) {
    const GemmGroup& G = p.grp[gslot];
    const int idx = blockIdx.y;
    const int M = G.m;
    const int N = (MODE == MODE_UPDATE) ? G.n : G.m;
    const int K = (MODE == MODE_GRAM) ? G.n : G.m;
    const int tiles_n = (N + 63) / 64;
    const int ti = blockIdx.x / tiles_n, tj = blockIdx.x % tiles_n;
    if (ti * 64 >= M) return;

    const int ldl = (MODE == MODE_GRAM) ? G.ldx : G.lda;
    const int ldr = (MODE == MODE_POLY) ? G.lda : G.ldx;
    const uint16_t* L = G.opl16 + (int64_t)idx * ((MODE == MODE_GRAM) ? G.x_stride : G.a_stride);
    const uint16_t* R = G.opr16 + (int64_t)idx * ((MODE == MODE_POLY) ? G.a_stride : G.x_stride);

    // operands: bf16 in the first iteration, fp16 after
    auto dec = [&](uint16_t b) { return p.f16 ? h2f(b) : bf2f(b); };
    auto enc = [&](float x) { return p.f16 ? f2h(x) : f2bf(x); };
    __shared__ float sl[16][65];
    __shared__ float sr[16][65];
    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int e = threadIdx.x; e < 16 * 64; e += 256) {
            const int kk = e & 15, ii = e >> 4;
            const int i = ti * 64 + ii, k = k0 + kk;
            sl[kk][ii] = (i < M && k < K) ? dec(L[(int64_t)i * ldl + k]) : 0.f;
            const int j = tj * 64 + ii;
            float r = 0.f;
            if (j < N && k < K) {
                if (MODE == MODE_GRAM)
                    r = dec(R[(int64_t)j * ldr + k]);  // X^T[k][j] = X[j][k]
                else
                    r = dec(R[(int64_t)k * ldr + j]);  // A[k][j] (poly), X[k][j] (update)
            }
            sr[kk][ii] = r;
        }
        __syncthreads();
#pragma unroll
        for (int kk = 0; kk < 16; ++kk) {
            float a[4], b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = sl[kk][ty * 4 + q];
                b[q] = sr[kk][tx * 4 + q];
            }
#pragma unroll
            for (int r = 0; r < 4; ++r)
#pragma unroll
                for (int c = 0; c < 4; ++c) acc[r][c] = fmaf(a[r], b[c], acc[r][c]);
        }
        __syncthreads();
    }

    // stored iterate X / c (c = ||X0||): see the tensor-core kernels
    const float cs = p.iter_scale[G.sub0 + idx];
    const float c2 = cs * cs;
    const float s = p.first ? p.norm_scale[G.sub0 + idx] / cs : 1.f;
#pragma unroll
    for (int r = 0; r < 4; ++r) {
        const int i = ti * 64 + ty * 4 + r;
        if (i >= M) continue;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
            const int j = tj * 64 + tx * 4 + c;
            if (j >= N) continue;
            if (MODE == MODE_GRAM) {
                G.out16[(int64_t)idx * G.a_stride + (int64_t)i * G.lda + j] = enc(acc[r][c] * (s * s));
            } else if (MODE == MODE_POLY) {
                const float a = dec(G.a16[(int64_t)idx * G.a_stride + (int64_t)i * G.lda + j]);
                float v = fmaf(p.cb, a, (p.cc * c2) * acc[r][c]);
                if (p.f16) v = c2 * v + (i == j ? p.ca : 0.f);  // later iterations: P' = a I + P, unscaled
                G.out16[(int64_t)idx * G.a_stride + (int64_t)i * G.lda + j] = enc(v);
            } else {
                const int64_t off = (int64_t)idx * G.x_stride + (int64_t)i * G.ldx + j;
                // the first update reads u as hi + lo (bf16) for its a X term; later ones
                // find a on the diagonal of P.  The next iterate is fp16.
                if (p.f16) {
                    G.x16_out[off] = f2h(acc[r][c]);
                } else {
                    const float x = bf2f(R[(int64_t)i * ldr + j]) + bf2f(G.xlo_in[off]);
                    G.x16_out[off] = f2h(s * fmaf(p.ca, x, c2 * acc[r][c]));
                }
            }
        }
    }
}

// Row sums of O^2 per 256-column tile, in the layout the tensor-core update writes.
__global__ void __launch_bounds__(256) k_rowsq_simt(const __grid_constant__ GemmParams p, int gslot) {
    const GemmGroup& G = p.grp[gslot];
    const int idx = blockIdx.y;
    const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (e >= (int64_t)G.m * G.ntile_n) return;
    const int row = (int)(e / G.ntile_n), t = (int)(e % G.ntile_n);
    const uint16_t* o = G.x16_out + (int64_t)idx * G.x_stride + (int64_t)row * G.ldx;
    float s = 0.f;
    for (int j = t * kBNUpd; j < min(G.n, (t + 1) * kBNUpd); ++j) {
        const float v = h2f(o[j]);  // O is fp16
        s = fmaf(v, v, s);
    }
    float* out = G.rowsq + (int64_t)idx * G.ntile_n * 2 * G.m;  // [tile, half][row] layout
    out[(int64_t)(t * 2) * G.m + row] = s;
    out[(int64_t)(t * 2 + 1) * G.m + row] = 0.f;
}

template <int MODE>
cudaError_t launch_ns_gemm_simt(const GemmParams& p, int gslot, int count, cudaStream_t stream) {
    const GemmGroup& G = p.grp[gslot];
    const int N = (MODE == MODE_UPDATE) ? G.n : G.m;
    dim3 grid(((G.m + 63) / 64) * ((N + 63) / 64), count);
    k_ns_gemm_simt<MODE><<<grid, 256, 0, stream>>>(p, gslot);
    cudaError_t e = cudaGetLastError();
    if (e == cudaSuccess && MODE == MODE_UPDATE && p.want_rowsq) {
        dim3 g2((unsigned)(((int64_t)G.m * G.ntile_n + 255) / 256), count);
        k_rowsq_simt<<<g2, 256, 0, stream>>>(p, gslot);
        e = cudaGetLastError();
    }
    return e;
}

template cudaError_t launch_ns_gemm_simt<MODE_GRAM>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_ns_gemm_simt<MODE_POLY>(const GemmParams&, int, int, cudaStream_t);
template cudaError_t launch_ns_gemm_simt<MODE_UPDATE>(const GemmParams&, int, int, cudaStream_t);

}  // namespace muon
