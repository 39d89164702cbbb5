// Elementwise stages of the step (HBM-bound; 128-bit accesses, 64 x 64 tiles).
//
//   k_momentum    S1 + S2 + S3 + S4 partials: momentum buffer update (lerp form
//                 of the FixMuonLR record, or the mul/add form of the
//                 "modded-nanogpt 50B-token" write-up), Nesterov direction u,
//                 u written in the wide orientation (through shared memory for
//                 tall matrices) as a bf16 hi + lo pair, per-tile partial sums
//                 of u^2
//   k_norm_scale  S4: s = 1 / (||u||_F + 1e-7) per matrix (fixed-order reduction);
//                 flags a matrix whose ||u|| is not finite
//   k_col_sumsq   S8 for column lanes: per (64-row slab, column) sums of O^2
//   k_lane_stats  S8 + S9 factors: r from the update epilogue's row sums (or the
//                 column sums), v <- lerp(v, r, 1 - beta2),
//                 q = 1/sqrt(max(v, 1e-10)), norm-preserving gamma, lane factor
//                 lr * lr_mul * gamma * q (plain Muon: lr * lr_mul * max(1, R/C)^0.5)
//   k_apply       S10: p <- p * (1 - lr*lr_mul*wd*wd_mul) - lane_factor * O,
//                 O read in the wide orientation and written back in the
//                 caller's orientation
// Reductions are two-stage with a fixed order, so results are reproducible.
//
// Failure handling.  A fatal bit in the status word (a bounded wait that gave
// up, or an SM pair without a shared TMEM allocation) makes k_momentum,
// k_lane_stats and k_apply return without writing, so neither the caller's
// parameters nor the optimizer state take in what a failed Newton-Schulz
// launch left behind; this holds for every step until muon_sync_status clears
// the word.  A momentum element whose new value is not finite keeps its old
// value and makes u non-finite; k_norm_scale then flags the matrix, and its
// second moment and parameters are left as they were for that step.
#include <algorithm>

#include "muon_internal.h"
#include "ptx_sm103.cuh"

namespace muon {

// Sum over the block (up to 32 warps; red holds one float per warp).
__device__ __forceinline__ float block_sum_256(float v, float* red) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    __syncthreads();
    if (l == 0) red[w] = v;
    __syncthreads();
    float t = 0.f;
    if (w == 0) {
        t = (l < (int)(blockDim.x >> 5)) ? red[l] : 0.f;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
        if (l == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

template <bool GRAD_F32>
__device__ __forceinline__ void load_grad8(const void* base, int64_t off, float (&g)[8]) {
    if (GRAD_F32) {
        const float4* s = reinterpret_cast<const float4*>(static_cast<const float*>(base) + off);
        const float4 a = s[0], b = s[1];
        g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
        g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
    } else {
        const uint4 w = *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(base) + off);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            g[2 * h] = __uint_as_float(ws[h] << 16);
            g[2 * h + 1] = __uint_as_float(ws[h] & 0xFFFF0000u);
        }
    }
}

template <bool GRAD_F32>
__device__ __forceinline__ float load_grad1(const void* base, int64_t off) {
    if (GRAD_F32) return static_cast<const float*>(base)[off];
    return bf2f(static_cast<const uint16_t*>(base)[off]);
}

__device__ __forceinline__ void store8_f32(float* dst, const float (&v)[8]) {
    reinterpret_cast<float4*>(dst)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4*>(dst)[1] = make_float4(v[4], v[5], v[6], v[7]);
}

__device__ __forceinline__ void load8_f32(const float* src, float (&v)[8]) {
    const float4 a = reinterpret_cast<const float4*>(src)[0];
    const float4 b = reinterpret_cast<const float4*>(src)[1];
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

__device__ __forceinline__ void store8_bf16(uint16_t* dst, const float (&v)[8]) {
    uint4 w;
    w.x = pack_bf2(v[0], v[1]);
    w.y = pack_bf2(v[2], v[3]);
    w.z = pack_bf2(v[4], v[5]);
    w.w = pack_bf2(v[6], v[7]);
    *reinterpret_cast<uint4*>(dst) = w;
}

// u as two bf16 halves: hi = bf16(u), lo = bf16(u - hi); hi + lo keeps ~16 mantissa bits
__device__ __forceinline__ void store8_hilo(uint16_t* hi, uint16_t* lo, const float (&v)[8]) {
    float l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) l[e] = v[e] - bf2f(f2bf(v[e]));
    store8_bf16(hi, v);
    store8_bf16(lo, l);
}

__device__ __forceinline__ void store1_hilo(uint16_t* hi, uint16_t* lo, float v) {
    const uint16_t h = f2bf(v);
    *hi = h;
    *lo = f2bf(v - bf2f(h));
}

// eight fp16 values (the Newton-Schulz output O)
__device__ __forceinline__ void load8_f16(const uint16_t* src, float (&v)[8]) {
    const uint4 w = *reinterpret_cast<const uint4*>(src);
    const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
        v[2 * h] = h2f((uint16_t)(ws[h] & 0xFFFFu));
        v[2 * h + 1] = h2f((uint16_t)(ws[h] >> 16));
    }
}

// momentum and Nesterov direction of one element.  A new buffer value that is
// not finite (a non-finite gradient, or an overflow) is not stored: the element
// keeps its old value and the direction is NaN, which flags the matrix.
__device__ __forceinline__ float momentum_elem(float g, float& b, float mu, int lerp_form, int nesterov) {
    float bn, u;
    if (lerp_form) {
        bn = fmaf(1.f - mu, g - b, b);          // buf.lerp_(g, 1 - mu)
        u = nesterov ? fmaf(mu, bn - g, g)      // lerp(g, buf, mu)
                     : bn;
    } else {
        bn = fmaf(mu, b, g);                    // buf.mul_(mu).add_(g)
        u = nesterov ? fmaf(mu, bn, g) : bn;    // g + mu * buf
    }
    const bool ok = isfinite(bn);
    b = ok ? bn : b;
    return ok ? u : __int_as_float(0x7fc00000);
}

template <int CAP, bool GRAD_F32>
__global__ void __launch_bounds__(256, 6) k_momentum(const __grid_constant__ ElemParams<CAP> p) {
    __shared__ float su[kTile][kTile + 1];
    __shared__ float red[8];
    // the tile list and the descriptors are written once, at create: they are read before the
    // wait for the previous kernel; the status word after it
    const int4 tile = p.tiles[blockIdx.x];
    const SubDesc d = p.subs[tile.x];
    grid_dep_wait();
    grid_dep_launch();
    const int fatal = *p.status & kStatusFatal;
    if (fatal) return;  // an earlier step failed: leave the momentum as it is (uniform over the block)
    const int r0 = tile.y, c0 = tile.z;
    const float mu = p.hp[HP_MU];
    const int tr = threadIdx.x >> 3, tc = threadIdx.x & 7;
    const void* gbase = p.ptr.grad[d.parent];
    float sumsq = 0.f;

#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int rl = pass * 32 + tr, cl = tc * 8;
        const int r = r0 + rl, c = c0 + cl;
        float u[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) u[e] = 0.f;
        if (r < d.rows && c < d.cols) {
            const int64_t goff = d.grad_off + (int64_t)r * d.ld + c;
            float* bptr = d.mom + (int64_t)r * d.ld_mom + c;
            if (d.vec) {
                float g[8], b[8];
                load_grad8<GRAD_F32>(gbase, goff, g);
                load8_f32(bptr, b);
#pragma unroll
                for (int e = 0; e < 8; ++e) u[e] = momentum_elem(g[e], b[e], mu, p.lerp_form, p.nesterov);
                store8_f32(bptr, b);
            } else {
                for (int e = 0; e < 8 && c + e < d.cols; ++e) {
                    float b = bptr[e];
                    u[e] = momentum_elem(load_grad1<GRAD_F32>(gbase, goff + e), b, mu, p.lerp_form, p.nesterov);
                    bptr[e] = b;
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) sumsq = fmaf(u[e], u[e], sumsq);
            if (!d.transposed) {
                const int64_t xo = (int64_t)r * d.ldx + c;
                if (d.vec) {
                    store8_hilo(d.u16 + xo, d.ulo16 + xo, u);
                } else {
                    for (int e = 0; e < 8 && c + e < d.cols; ++e) store1_hilo(d.u16 + xo + e, d.ulo16 + xo + e, u[e]);
                }
            }
        }
        if (d.transposed) {
#pragma unroll
            for (int e = 0; e < 8; ++e) su[cl + e][rl] = u[e];
        }
    }

    if (d.transposed) {
        __syncthreads();
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int i = pass * 32 + tr;         // wide row (caller column) within the tile
            const int wr = c0 + i, wc = r0 + tc * 8;
            if (wr < d.cols && wc < d.rows) {
                float v[8];
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = su[i][tc * 8 + e];
                const int64_t xo = (int64_t)wr * d.ldx + wc;
                if (wc + 8 <= d.rows) {
                    store8_hilo(d.u16 + xo, d.ulo16 + xo, v);
                } else {
                    for (int e = 0; e < 8 && wc + e < d.rows; ++e) store1_hilo(d.u16 + xo + e, d.ulo16 + xo + e, v[e]);
                }
            }
        }
    }
    const float total = block_sum_256(sumsq, red);
    if (threadIdx.x == 0) p.norm_part[blockIdx.x] = total;
}

__global__ void __launch_bounds__(256) k_norm_scale(const __grid_constant__ NormParams p) {
    __shared__ float red[8];
    const SubDesc& d = p.subs[blockIdx.x];
    grid_dep_wait();
    grid_dep_launch();
    float s = 0.f;
    for (int t = threadIdx.x; t < d.k1_ntiles; t += 256) s += p.norm_part[d.k1_tile0 + t];
    const float total = block_sum_256(s, red);
    if (threadIdx.x == 0) {
        const float norm = sqrtf(total);
        const float sc = 1.f / (norm + kNormEps);
        p.norm_scale[blockIdx.x] = sc;
        // ||X0|| = ||u|| s: the Newton-Schulz kernels keep their iterate divided by it
        p.iter_scale[blockIdx.x] = norm > 0.f ? norm * sc : 1.f;
        // a non-finite direction: this matrix's second moment and parameters are left alone
        const int bad = isfinite(total) ? 0 : 1;
        *d.skip = bad;
        if (bad) atomicOr(p.status, STATUS_NONFINITE);
    }
}

// Per (sub, 64-row slab): sums over the slab's rows of O^2 for every column of
// the wide orientation (subs whose NorMuon lanes are its columns).
__global__ void __launch_bounds__(256) k_col_sumsq(const __grid_constant__ ColSumParams p) {
    const int2 w = p.work[blockIdx.x];
    const SubDesc& d = p.subs[w.x];
    grid_dep_wait();
    grid_dep_launch();
    const int r0 = w.y * kTile, r1 = min(r0 + kTile, d.m);
    float* out = d.colsq + (int64_t)w.y * d.n;
    for (int j0 = threadIdx.x * 8; j0 < d.n; j0 += 256 * 8) {
        float acc[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] = 0.f;
        if (j0 + 8 <= d.n) {
            for (int r = r0; r < r1; ++r) {
                float o[8];
                load8_f16(d.o16 + (int64_t)r * d.ldx + j0, o);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] = fmaf(o[e], o[e], acc[e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) out[j0 + e] = acc[e];
        } else {
            for (int r = r0; r < r1; ++r)
                for (int e = 0; e < 8 && j0 + e < d.n; ++e) {
                    const float o = h2f(d.o16[(int64_t)r * d.ldx + j0 + e]);
                    acc[e] = fmaf(o, o, acc[e]);
                }
            for (int e = 0; e < 8 && j0 + e < d.n; ++e) out[j0 + e] = acc[e];
        }
    }
}

constexpr int kLaneThreads = 1024;  // one block per matrix, one thread per lane up to 1024 lanes

__global__ void __launch_bounds__(kLaneThreads) k_lane_stats(const __grid_constant__ LaneParams p) {
    __shared__ float red[32];
    const SubDesc& d = p.subs[blockIdx.x];
    grid_dep_wait();
    grid_dep_launch();
    // a failed step (fatal status) or a non-finite direction: the second moment stays as it is
    if ((*p.status & kStatusFatal) || *d.skip) return;
    const float eff = p.hp[HP_LR] * d.lr_mul;
    const float cs = p.iter_scale[blockIdx.x];  // O = cs * (the stored output)
    const int nl = d.lane_cols ? d.n : d.m;     // lanes
    if (!p.normuon) {
        const float f = eff * d.shape_scale * cs;
        for (int i = threadIdx.x; i < nl; i += kLaneThreads) d.lane[i] = f;
        return;
    }
    const float beta2 = p.hp[HP_BETA2];
    const float inv_len = 1.f / (float)(d.lane_cols ? d.m : d.n);  // the mean runs across the lanes' length
    float before = 0.f, after = 0.f;
    // v <- lerp(v, r, 1 - beta2) and the lane's rsqrt, given the lane's sum of O^2 (stored scale)
    auto lane_update = [&](int i, float rs) {
        rs *= cs * cs;
        const float r = rs * inv_len;
        const float v0 = d.v[i];
        const float v1 = fmaf(1.f - beta2, r - v0, v0);  // v.lerp_(r, 1 - beta2)
        d.v[i] = v1;
        const float q = 1.f / sqrtf(fmaxf(v1, kVFloor));
        d.lane[i] = q;
        before += rs;
        after = fmaf(rs, q * q, after);
    };
    // one thread per lane; the partial sums are stored part-major ([part][lane]), so neighbouring
    // threads read neighbouring words, and each lane adds its parts in a fixed order
    const int nparts = d.lane_cols ? (d.m + kTile - 1) / kTile : 2 * d.ntile_n;
    const float* parts = d.lane_cols ? d.colsq : d.rowsq;
    for (int i = threadIdx.x; i < nl; i += kLaneThreads) {
        float rs = 0.f;
#pragma unroll 4
        for (int t = 0; t < nparts; ++t) rs += parts[(int64_t)t * nl + i];
        lane_update(i, rs);
    }
    const float sb = block_sum_256(before, red);
    const float sa = block_sum_256(after, red);
    const float gamma = p.norm_preserve ? sqrtf(sb) / fmaxf(sqrtf(sa), kVFloor) : 1.f;
    const float f = eff * gamma * cs;
    for (int i = threadIdx.x; i < nl; i += kLaneThreads) d.lane[i] *= f;
}

template <int CAP>
__global__ void __launch_bounds__(256, 5) k_apply(const __grid_constant__ ElemParams<CAP> p) {
    __shared__ float so[kTile][kTile + 1];
    // Everything a block needs before its data loads sits on a chain of dependent loads
    // (tile -> matrix descriptor -> parameter pointer).  The tile list and the descriptors are
    // written once, at create, so they are read before the wait for the previous kernel.  The
    // status word, the hyper-parameters and the skip flag are loaded alongside the data, and
    // tested only once the data loads are in flight, so they add no latency of their own.
    const int4 tile = p.tiles[blockIdx.x];
    const SubDesc d = p.subs[tile.x];
    grid_dep_wait();
    grid_dep_launch();
    const int fatal = *p.status & kStatusFatal;  // a Newton-Schulz launch failed: keep the parameters
    const float lr = p.hp[HP_LR], wd = p.hp[HP_WD];
    const int r0 = tile.y, c0 = tile.z;
    const int tr = threadIdx.x >> 3, tc = threadIdx.x & 7;
    float* P = p.ptr.param[d.parent] + d.grad_off;
    // lanes along the caller's columns (rows of a transposed matrix's wide orientation, or the
    // wide columns of an untransposed one), else along its rows
    const bool per_col = d.transposed != d.lane_cols;

    // loads of both row passes first; the lane factors are per column (the same eight for both
    // passes) or per row (one per pass)
    float pv[2][8], o[2][8], fcol[8], frow[2] = {0.f, 0.f};
    bool act[2];
#pragma unroll
    for (int e = 0; e < 8; ++e) fcol[e] = 0.f;
    if (per_col && c0 + tc * 8 < d.cols && r0 + tr < d.rows)
        for (int e = 0; e < 8; ++e) fcol[e] = (c0 + tc * 8 + e < d.cols) ? d.lane[c0 + tc * 8 + e] : 0.f;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        const int r = r0 + pass * 32 + tr, c = c0 + tc * 8;
        act[pass] = r < d.rows && c < d.cols;
#pragma unroll
        for (int e = 0; e < 8; ++e) pv[pass][e] = o[pass][e] = 0.f;
        if (act[pass]) {
            const float* pp = P + (int64_t)r * d.ld + c;
            if (d.vec) {
                load8_f32(pp, pv[pass]);
            } else {
                for (int e = 0; e < 8 && c + e < d.cols; ++e) pv[pass][e] = pp[e];
            }
            if (!d.transposed) {
                const uint16_t* src = d.o16 + (int64_t)r * d.ldx + c;
                if (d.vec)
                    load8_f16(src, o[pass]);
                else
                    for (int e = 0; e < 8 && c + e < d.cols; ++e) o[pass][e] = h2f(src[e]);
            }
            if (!per_col) frow[pass] = d.lane[r];
        }
    }
    const int skip = *d.skip;  // this matrix's direction was not finite
    if (fatal || skip) return;  // uniform over the block, before any barrier or store

    if (d.transposed) {
        // O is stored in the wide orientation: stage its tile transposed through shared memory
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int i = pass * 32 + tr;
            const int wr = c0 + i, wc = r0 + tc * 8;
            float v[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) v[e] = 0.f;
            if (wr < d.cols && wc < d.rows) {
                const uint16_t* src = d.o16 + (int64_t)wr * d.ldx + wc;
                if (wc + 8 <= d.rows)
                    load8_f16(src, v);
                else
                    for (int e = 0; e < 8 && wc + e < d.rows; ++e) v[e] = h2f(src[e]);
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) so[i][tc * 8 + e] = v[e];
        }
        __syncthreads();
#pragma unroll
        for (int pass = 0; pass < 2; ++pass) {
            const int rl = pass * 32 + tr, cl = tc * 8;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[pass][e] = so[cl + e][rl];
        }
    }

    const float decay = 1.f - lr * d.lr_mul * wd * d.wd_mul;
#pragma unroll
    for (int pass = 0; pass < 2; ++pass) {
        if (!act[pass]) continue;
        const int r = r0 + pass * 32 + tr, c = c0 + tc * 8;
        float* pp = P + (int64_t)r * d.ld + c;
        float out[8];
#pragma unroll
        for (int e = 0; e < 8; ++e) out[e] = fmaf(-(per_col ? fcol[e] : frow[pass]), o[pass][e], pv[pass][e] * decay);
        if (d.vec) {
            store8_f32(pp, out);
        } else {
            for (int e = 0; e < 8 && c + e < d.cols; ++e) pp[e] = out[e];
        }
    }
}

// u = hi + lo of one matrix into a dense fp32 m x n array (state access)
// O = c * (the stored fp16 output), dense fp32 m x n
__global__ void k_scale_f16(float* dst, const uint16_t* src, const float* c, int m, int n, int ld) {
    const int64_t total = (int64_t)m * n;
    const float cs = *c;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / n, j = e % n;
        dst[e] = cs * h2f(src[i * ld + j]);
    }
}

cudaError_t launch_scale_f16(float* dst, const uint16_t* src, const float* c, int m, int n, int ld, cudaStream_t s) {
    const int64_t total = (int64_t)m * n;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    k_scale_f16<<<blocks, 256, 0, s>>>(dst, src, c, m, n, ld);
    return cudaGetLastError();
}

__global__ void k_combine_hilo(float* dst, const uint16_t* hi, const uint16_t* lo, int m, int n, int ld) {
    const int64_t total = (int64_t)m * n;
    for (int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; e < total; e += (int64_t)gridDim.x * blockDim.x) {
        const int64_t i = e / n, j = e % n;
        dst[e] = bf2f(hi[i * ld + j]) + bf2f(lo[i * ld + j]);
    }
}

cudaError_t launch_combine_hilo(float* dst, const uint16_t* hi, const uint16_t* lo, int m, int n, int ld,
                                cudaStream_t s) {
    const int64_t total = (int64_t)m * n;
    const int blocks = (int)std::min<int64_t>((total + 255) / 256, 4096);
    k_combine_hilo<<<blocks, 256, 0, s>>>(dst, hi, lo, m, n, ld);
    return cudaGetLastError();
}

__global__ void k_set_hparams(float* hp, float lr, float mu, float beta2, float wd) {
    hp[HP_LR] = lr;
    hp[HP_MU] = mu;
    hp[HP_BETA2] = beta2;
    hp[HP_WD] = wd;
}

// Installs a schedule (by value) and its starting step.
__global__ void k_schedule_set(DevSchedule* dst, DevSchedule val) { *dst = val; }

// Start of a scheduled step: lr and mu of step s into the device scalars, then
// s <- s + 1.  Evaluated in double, stored as fp32.
__global__ void k_schedule_advance(float* hp, DevSchedule* sc) {
    const int64_t s = sc->step;
    double mult;
    if (s <= sc->cooldown_start)
        mult = 1.0;
    else if (s >= sc->cooldown_end)
        mult = (double)sc->lr_floor;
    else
        mult = (double)sc->lr_floor + (1.0 - (double)sc->lr_floor) * ((double)(sc->cooldown_end - s) /
                                                                      (double)(sc->cooldown_end - sc->cooldown_start));
    const double frac = sc->momentum_warmup == 0 ? 1.0 : fmin((double)s / (double)sc->momentum_warmup, 1.0);
    hp[HP_LR] = (float)((double)sc->lr_base * mult);
    hp[HP_MU] = (float)((double)sc->momentum_start + ((double)sc->momentum_end - (double)sc->momentum_start) * frac);
    sc->step = s + 1;
}

// ------------------------------------------------------------------ launchers
// overlap: launched with programmatic stream serialization (see launch_kernel)
template <int CAP>
cudaError_t launch_momentum(const ElemParams<CAP>& p, bool grad_f32, bool overlap, cudaStream_t s) {
    if (p.ntiles <= 0) return cudaSuccess;
    if (grad_f32) return launch_kernel(k_momentum<CAP, true>, dim3(p.ntiles), dim3(256), 0, s, overlap, p);
    return launch_kernel(k_momentum<CAP, false>, dim3(p.ntiles), dim3(256), 0, s, overlap, p);
}

template <int CAP>
cudaError_t launch_apply(const ElemParams<CAP>& p, bool overlap, cudaStream_t s) {
    if (p.ntiles <= 0) return cudaSuccess;
    return launch_kernel(k_apply<CAP>, dim3(p.ntiles), dim3(256), 0, s, overlap, p);
}

cudaError_t launch_norm_scale(const NormParams& p, bool overlap, cudaStream_t s) {
    if (p.nsubs <= 0) return cudaSuccess;
    return launch_kernel(k_norm_scale, dim3(p.nsubs), dim3(256), 0, s, overlap, p);
}

cudaError_t launch_col_sumsq(const ColSumParams& p, bool overlap, cudaStream_t s) {
    if (p.nwork <= 0) return cudaSuccess;
    return launch_kernel(k_col_sumsq, dim3(p.nwork), dim3(256), 0, s, overlap, p);
}

cudaError_t launch_lane_stats(const LaneParams& p, bool overlap, cudaStream_t s) {
    if (p.nsubs <= 0) return cudaSuccess;
    return launch_kernel(k_lane_stats, dim3(p.nsubs), dim3(kLaneThreads), 0, s, overlap, p);
}

cudaError_t launch_set_hparams(float* hp, float lr, float mu, float beta2, float wd, cudaStream_t s) {
    k_set_hparams<<<1, 1, 0, s>>>(hp, lr, mu, beta2, wd);
    return cudaGetLastError();
}

cudaError_t launch_schedule_set(DevSchedule* dst, const DevSchedule& val, cudaStream_t s) {
    k_schedule_set<<<1, 1, 0, s>>>(dst, val);
    return cudaGetLastError();
}

cudaError_t launch_schedule_advance(float* hp, DevSchedule* sc, cudaStream_t s) {
    k_schedule_advance<<<1, 1, 0, s>>>(hp, sc);
    return cudaGetLastError();
}

#define MUON_INSTANTIATE_CAP(CAP)                                                           \
    template cudaError_t launch_momentum<CAP>(const ElemParams<CAP>&, bool, bool, cudaStream_t); \
    template cudaError_t launch_apply<CAP>(const ElemParams<CAP>&, bool, cudaStream_t);
MUON_INSTANTIATE_CAP(64)
MUON_INSTANTIATE_CAP(256)
MUON_INSTANTIATE_CAP(1024)

}  // namespace muon
