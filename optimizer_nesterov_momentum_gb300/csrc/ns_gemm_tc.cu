// Grouped Newton-Schulz GEMMs on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel template serves the three products of an iteration
// (the quintic map of the Muon orthogonalisation, "modded-nanogpt 50B-token"
// write-up, section "Muon from the source", grouped as X <- a X + (b A + c A^2) X):
//
//   MODE_GRAM    A = sc * X X^T           (sc = s^2 on the first iteration, s = 1/(||u||+eps))
//   MODE_POLY    P = b A + c A A          (A symmetric, so A A = sum_k A[i,k] A[j,k])
//   MODE_UPDATE  X' = s1 (a X + P X)      (s1 = s on the first iteration)
//
// A and P are symmetric: GRAM and POLY only compute tiles on and above the
// diagonal and store each tile twice (itself and its mirror).  The left
// operand is always K-major (rows of X, A or P); the right operand is K-major
// for GRAM / POLY (rows again, thanks to the symmetry) and MN-major for
// UPDATE (X[k, j] with j contiguous), selected in the instruction descriptor.
//
// Warp roles (192 threads, one CTA per SM, persistent over a tile list):
//   warp 0     TMA producer (one thread): 128 B-swizzled tiles into a ring of
//              shared-memory stages, completion tracked by mbarriers
//   warp 1     TMEM allocator + MMA issuer (one thread): tcgen05.mma M=128,
//              N=128/256, K=16 into a double-buffered TMEM accumulator
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (warp w owns TMEM lanes
//              32*(w%4)..+31), combine in fp32, round to bf16, store
// Every wait is bounded (2 s); on a timeout the kernel sets the status word,
// lets copies and MMAs in flight finish, frees TMEM and returns.
#include "muon_internal.h"
#include "ptx_sm103.cuh"

namespace muon {

template <int MODE>
struct TcCfg {
    static constexpr int BN = (MODE == MODE_UPDATE) ? kBNUpd : kBNSym;
    static constexpr int STAGES = (MODE == MODE_UPDATE) ? 4 : 6;
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr bool B_MN = (MODE == MODE_UPDATE);
    static constexpr uint32_t IDESC = make_idesc_bf16(kBM, BN, B_MN);
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 /*align*/ + 256 /*barriers*/;
};

__device__ __forceinline__ void store_bf16_row32(uint16_t* dst, const float (&v)[32], int nvalid) {
    if (nvalid >= 32) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w;
            w.x = pack_bf2(v[8 * q + 0], v[8 * q + 1]);
            w.y = pack_bf2(v[8 * q + 2], v[8 * q + 3]);
            w.z = pack_bf2(v[8 * q + 4], v[8 * q + 5]);
            w.w = pack_bf2(v[8 * q + 6], v[8 * q + 7]);
            d4[q] = w;
        }
    } else {
        for (int e = 0; e < nvalid; ++e) dst[e] = f2bf(v[e]);
    }
}

__device__ __forceinline__ void load_bf16_row32(const uint16_t* src, float (&v)[32], int nvalid) {
    if (nvalid >= 32) {
        const uint4* s4 = reinterpret_cast<const uint4*>(src);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w = s4[q];
            uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                v[8 * q + 2 * h] = __uint_as_float(ws[h] << 16);
                v[8 * q + 2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
            }
        }
    } else {
        for (int e = 0; e < 32; ++e) v[e] = (e < nvalid) ? bf2f(src[e]) : 0.f;
    }
}

template <int MODE>
__global__ void __launch_bounds__(192, 1) k_ns_gemm_tc(const __grid_constant__ GemmParams p) {
    using C = TcCfg<MODE>;
    constexpr int BN = C::BN;
    constexpr int STAGES = C::STAGES;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::A_BYTES;
    uint64_t* full = reinterpret_cast<uint64_t*>(sB + STAGES * C::B_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;   // [2] accumulator ready
    uint64_t* tempty = tfull + 2;       // [2] accumulator drained
    uint64_t* mma_done = tempty + 2;    // abort path only
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 4);
        }
        mbar_init(mma_done, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int g = 0; g < p.ngroups; ++g) {
                tma_prefetch_desc(&p.map_a[g]);
                if (MODE == MODE_UPDATE) tma_prefetch_desc(&p.map_b[g]);
            }
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[STAGES];
            bool issued[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) issued[s] = false;
            bool ok = true;
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                const int4 tile = p.tiles[t];
                const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
                const int K = (MODE == MODE_GRAM) ? p.grp[g].n : p.grp[g].m;
                const int nkb = (K + kBK - 1) / kBK;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                    uint8_t* a_dst = sA + stage * C::A_BYTES;
                    uint8_t* b_dst = sB + stage * C::B_BYTES;
                    if (MODE == MODE_UPDATE) {
                        tma_load_3d(a_dst, &p.map_a[g], &full[stage], kb * kBK, ti * kBM, idx);
#pragma unroll
                        for (int c = 0; c < BN / 64; ++c)
                            tma_load_3d(b_dst + c * (64 * kBK * 2), &p.map_b[g], &full[stage], tj * BN + c * 64,
                                        kb * kBK, idx);
                    } else {
                        tma_load_3d(a_dst, &p.map_a[g], &full[stage], kb * kBK, ti * kBM, idx);
                        tma_load_3d(b_dst, &p.map_a[g], &full[stage], kb * kBK, tj * BN, idx);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok) {
                // let every copy already issued land before the CTA can exit
#pragma unroll
                for (int s = 0; s < STAGES; ++s)
                    if (issued[s]) mbar_wait_drain(&full[s], issued_phase[s], 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            bool any = false;
            const uint32_t a_base = smem_u32(sA);
            const uint32_t b_base = smem_u32(sB);
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                const int4 tile = p.tiles[t];
                const int g = tile.x;
                const int K = (MODE == MODE_GRAM) ? p.grp[g].n : p.grp[g].m;
                const int nkb = (K + kBK - 1) / kBK;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_st = a_base + stage * C::A_BYTES;
                    const uint32_t b_st = b_base + stage * C::B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t adesc = make_sdesc_sw128(a_st + kk * 32, 16, 1024);
                        uint64_t bdesc;
                        if (C::B_MN)
                            bdesc = make_sdesc_sw128(b_st + kk * (16 * 128), 64 * kBK * 2, 1024);
                        else
                            bdesc = make_sdesc_sw128(b_st + kk * 32, 16, 1024);
                        umma_bf16(d_tmem, adesc, bdesc, C::IDESC, (kb | kk) != 0 ? 1u : 0u);
                        any = true;
                    }
                    umma_commit(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                // wait for the MMAs in flight before TMEM is released
                umma_commit(mma_done);
                mbar_wait_drain(mma_done, 0, 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int r_in_tile = quad * 32 + lane;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
            const int4 tile = p.tiles[t];
            const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
            const GemmGroup& G = p.grp[g];
            const bool got = mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const int row = ti * kBM + r_in_tile;
            const uint32_t t_acc = tmem_base + lane_off + (uint32_t)(acc * BN);
            if (MODE == MODE_UPDATE) {
                const bool row_ok = row < G.m;
                const float s1 = p.first ? p.norm_scale[G.sub0 + idx] : 1.f;
                const int64_t xoff = (int64_t)idx * G.x_stride + (int64_t)row * G.ldx;
                float sumsq = 0.f;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_load_32x32(t_acc + c * 32, v);
                    const int col0 = tj * BN + c * 32;
                    const int nvalid = min(32, G.n - col0);
                    if (row_ok && nvalid > 0) {
                        float x[32];
                        const float* xin = G.x32_in + xoff + col0;
                        if (nvalid >= 32) {
#pragma unroll
                            for (int q = 0; q < 8; ++q) {
                                float4 f = reinterpret_cast<const float4*>(xin)[q];
                                x[4 * q] = f.x;
                                x[4 * q + 1] = f.y;
                                x[4 * q + 2] = f.z;
                                x[4 * q + 3] = f.w;
                            }
                        } else {
                            for (int e = 0; e < 32; ++e) x[e] = (e < nvalid) ? xin[e] : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = s1 * fmaf(p.ca, x[e], v[e]);
                        if (G.x32_out != nullptr) {
                            float* xo = G.x32_out + xoff + col0;
                            if (nvalid >= 32) {
#pragma unroll
                                for (int q = 0; q < 8; ++q)
                                    reinterpret_cast<float4*>(xo)[q] =
                                        make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
                            } else {
                                for (int e = 0; e < nvalid; ++e) xo[e] = v[e];
                            }
                        }
                        store_bf16_row32(G.x16_out + xoff + col0, v, nvalid);
                        if (p.want_rowsq) {
                            for (int e = 0; e < 32; ++e) {
                                if (e < nvalid) {
                                    const float ob = bf2f(f2bf(v[e]));
                                    sumsq = fmaf(ob, ob, sumsq);
                                }
                            }
                        }
                    }
                }
                if (p.want_rowsq && row_ok)
                    G.rowsq[((int64_t)idx * G.m + row) * G.ntile_n + tj] = sumsq;
            } else {
                const bool row_ok = row < G.m;
                float sc = 1.f;
                if (MODE == MODE_GRAM && p.first) {
                    const float s = p.norm_scale[G.sub0 + idx];
                    sc = s * s;
                }
                uint16_t* out = G.out16 + (int64_t)idx * G.a_stride;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    float v[32];
                    tmem_load_32x32(t_acc + c * 32, v);
                    const int col0 = tj * BN + c * 32;
                    const int nvalid = min(32, G.m - col0);
                    if (MODE == MODE_POLY) {
                        float a[32];
                        if (row_ok && nvalid > 0)
                            load_bf16_row32(G.a16 + (int64_t)idx * G.a_stride + (int64_t)row * G.lda + col0, a,
                                            nvalid);
                        else
#pragma unroll
                            for (int e = 0; e < 32; ++e) a[e] = 0.f;
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = fmaf(p.cb, a[e], p.cc * v[e]);
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= sc;
                    }
                    if (row_ok && nvalid > 0) store_bf16_row32(out + (int64_t)row * G.lda + col0, v, nvalid);
                    if (ti != tj && row_ok) {
                        for (int e = 0; e < 32; ++e)
                            if (e < nvalid) out[(int64_t)(col0 + e) * G.lda + row] = f2bf(v[e]);
                    }
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

cudaError_t ns_gemm_tc_configure() {
    cudaError_t e = cudaFuncSetAttribute(k_ns_gemm_tc<MODE_GRAM>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         TcCfg<MODE_GRAM>::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_ns_gemm_tc<MODE_POLY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcCfg<MODE_POLY>::SMEM_BYTES);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_ns_gemm_tc<MODE_UPDATE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 TcCfg<MODE_UPDATE>::SMEM_BYTES);
    return e;
}

template <int MODE>
cudaError_t launch_ns_gemm_tc(const GemmParams& p, int num_sms, cudaStream_t stream) {
    using C = TcCfg<MODE>;
    if (p.ntiles <= 0) return cudaSuccess;
    const int grid = p.ntiles < num_sms ? p.ntiles : num_sms;
    k_ns_gemm_tc<MODE><<<grid, 192, C::SMEM_BYTES, stream>>>(p);
    return cudaGetLastError();
}

template cudaError_t launch_ns_gemm_tc<MODE_GRAM>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_POLY>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_UPDATE>(const GemmParams&, int, cudaStream_t);

}  // namespace muon
