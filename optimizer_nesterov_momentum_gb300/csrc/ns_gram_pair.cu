// The Gram product of the Newton-Schulz iteration on SM pairs ("modded-nanogpt
// 50B-token" write-up, section "Muon from the source"):
//
//   A = sc * X X^T      (sc = (s / c)^2 on the first iteration, else 1)
//
// with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) issued by CTA 0 of a
// two-CTA cluster.  A pair tile is the 256 x 256 block (I, J), J >= I, of the
// symmetric result.  CTA r stages rows 256 I + 128 r .. + 127 of X (the left
// operand's half) and rows 256 J + 128 r .. + 127 (the right operand's half,
// both K-major), so an off-diagonal tile stages 32 KB per SM per 64-deep
// k-block and a diagonal tile, whose two halves are the same rows, 16 KB.
// CTA r's TMEM receives rows 128 r .. + 127 of the tile.
//
// The epilogue works warp by warp: warp (quad, half) owns TMEM lanes
// 32 quad .. + 31 and columns 32 half .. + 31 of each 64-column chunk, i.e.
// four 32 x 32 blocks per tile.  It stores each block, and for an
// off-diagonal tile (I < J) also its transpose at (J, I), from its own ring of
// shared-memory slots; a diagonal tile is computed whole (both triangles) and
// stored once.  No barrier spans warps.
//
// Warp 0: TMA producer (both CTAs), warp 1: pair-wide TMEM allocation (both)
// and the MMA issuer (CTA 0), warps 2-9: epilogue (both).  All mbarrier waits
// are bounded (2 s) and raise the status word.
#include "muon_internal.h"
#include "pair_sm103.cuh"
#include "ptx_sm103.cuh"

namespace muon {
namespace {

constexpr int kSymThreads = 320;
constexpr int kSymRows = kBM * kBK * 2;  // 16 KB: 128 operand rows x 64
constexpr int kSymStage = 2 * kSymRows;  // left half | right half
constexpr int kBlk = 32 * 32 * 2;        // one 32 x 32 16-bit block (64-byte rows, 64-byte swizzle)
constexpr int kEpiWarps = 8;
constexpr uint32_t kNoTmem = 0xFFFFFFFFu;

constexpr int kGramStages = 6;
constexpr int kOutSlots = 2;  // per warp: blocks and mirrors in flight
constexpr int kGramSmem = kGramStages * kSymStage + kEpiWarps * kOutSlots * kBlk + 1024 + 512;
static_assert(kGramSmem <= 232448, "shared memory budget");

}  // namespace

using namespace pair;

template <bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSymThreads, 1)
    k_ns_gram_pair(const __grid_constant__ GemmParams p) {
    constexpr int STAGES = kGramStages;
    constexpr uint32_t IDESC = make_idesc_16bit(256, 256, /*b_mn_major=*/false, F16);

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sS = smem;                                   // STAGES x (left | right)
    uint8_t* sO = sS + STAGES * kSymStage;                // per warp kOutSlots blocks
    uint64_t* full = reinterpret_cast<uint64_t*>(sO + kEpiWarps * kOutSlots * kBlk);  // CTA 0's are used
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;   // [2]
    uint64_t* tempty = tfull + 2;       // [2] CTA 0's: 8 warps of each CTA arrive
    uint64_t* mma_done = tempty + 2;    // abort path only
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_done + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* pair_ok = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pr = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * kEpiWarps);
        }
        mbar_init(mma_done, 1);
        *tmem_slot = kNoTmem;
        *abort_flag = 0;
        *pair_ok = 0;
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, 512);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    cluster_sync_all();  // barriers initialised and the allocation written in both CTAs
    tc_fence_after();
    if (threadIdx.x == 32) {
        const uint32_t mine = *tmem_slot;
        const uint32_t peer = ld_cluster_u32(cluster_addr(tmem_slot, rank ^ 1u));
        const int ok = (mine != kNoTmem && mine == peer) ? 1 : 0;
        *pair_ok = ok;
        if (!ok) {
            *abort_flag = 1;
            atomicOr(p.status, STATUS_PAIR);
        }
    }
    __syncthreads();
    const bool run = *pair_ok != 0;
    const uint32_t tbase = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ operand producer (both CTAs)
        if (lane == 0 && run) {
            for (int g = 0; g < p.ngroups; ++g) tma_prefetch_desc(&p.map_a[g]);
            const uint32_t full0 = cluster_addr(&full[0], 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            for (int t = pr; t < p.ntiles && ok; t += npairs) {
                const int4 tile = p.tiles[t];
                const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
                const int K = p.grp[g].n;
                const int nkb = (K + kBK - 1) / kBK;
                const bool diag = ti == tj;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(&full[stage], diag ? 2 * kSymRows : 2 * kSymStage);
                    const uint32_t bar = full0 + (uint32_t)(stage * 8);
                    uint8_t* dst = sS + stage * kSymStage;
                    tma_load_3d_pair(dst, &p.map_a[g], bar, kb * kBK, ti * 256 + (int)rank * kBM, idx);
                    if (!diag) tma_load_3d_pair(dst + kSymRows, &p.map_a[g], bar, kb * kBK, tj * 256 + (int)rank * kBM, idx);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer (CTA 0)
        if (lane == 0 && run && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true, any = false;
            const uint32_t s_base = smem_u32(sS);
            for (int t = pr; t < p.ntiles && ok; t += npairs) {
                const int4 tile = p.tiles[t];
                const int K = p.grp[tile.x].n;
                const int nkb = (K + kBK - 1) / kBK;
                const bool diag = tile.z == tile.w;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tbase + (uint32_t)(acc * 256);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_st = s_base + stage * kSymStage;
                    const uint32_t b_st = diag ? a_st : a_st + kSymRows;  // a diagonal tile's halves are the same rows
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t adesc = make_sdesc_sw128(a_st + kk * 32, 16, 1024);
                        const uint64_t bdesc = make_sdesc_sw128(b_st + kk * 32, 16, 1024);
                        umma_f16_pair(d_tmem, adesc, bdesc, IDESC, (kb | kk) != 0 ? 1u : 0u);
                        any = true;
                    }
                    umma_commit_pair(&empty[stage]);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && any) {
                umma_commit_pair(mma_done);
                mbar_wait_drain(mma_done, 0, 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int ew = warp - 2;
        const int quad = warp & 3;
        const int half = ew >> 2;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint8_t* wout = sO + ew * (kOutSlots * kBlk);
        const uint32_t tempty0 = cluster_addr(&tempty[0], 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        int nout = 0;  // output slots used so far (one bulk group each)
        for (int t = pr; run && t < p.ntiles; t += npairs) {
            const int4 tile = p.tiles[t];
            const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
            const GemmGroup& G = p.grp[g];
            const bool diag = ti == tj;
            const int row0 = ti * 256 + (int)rank * kBM + quad * 32;  // this warp's first row
            mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
            tc_fence_after();
            uint32_t raw[2][32];
            const uint32_t t_acc = tbase + (uint32_t)(acc * 256) + lane_off + (uint32_t)(half * 32);
            float scale = 1.f;
            if (p.first) {
                const float s = p.norm_scale[G.sub0 + idx] / p.iter_scale[G.sub0 + idx];
                scale = s * s;
            }
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if ((c & 1) == 0) {
                    // two chunks in flight at once; after the last two the accumulator is in
                    // registers and goes back to the MMA before the stores
                    tmem_load_32x32_async(t_acc + c * 64, raw[0]);
                    tmem_load_32x32_async(t_acc + (c + 1) * 64, raw[1]);
                    tmem_wait_loads();
                    if (c == 2) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster(tempty0 + (uint32_t)(acc * 8));
                    }
                }
                const int col0 = tj * 256 + c * 64 + half * 32;  // this block's first column
                uint16_t b[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) b[e] = f2x<F16>(scale * __uint_as_float(raw[c & 1][e]));

                // this block at (row0, col0)
                {
                    uint8_t* slot = wout + (nout % kOutSlots) * kBlk;
                    if (nout >= kOutSlots && lane == 0) bulk_wait_read<kOutSlots - 1>();
                    __syncwarp();
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        uint4 w;
                        w.x = (uint32_t)b[8 * jj + 0] | ((uint32_t)b[8 * jj + 1] << 16);
                        w.y = (uint32_t)b[8 * jj + 2] | ((uint32_t)b[8 * jj + 3] << 16);
                        w.z = (uint32_t)b[8 * jj + 4] | ((uint32_t)b[8 * jj + 5] << 16);
                        w.w = (uint32_t)b[8 * jj + 6] | ((uint32_t)b[8 * jj + 7] << 16);
                        *reinterpret_cast<uint4*>(slot + sw64((uint32_t)lane, (uint32_t)jj)) = w;
                    }
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&p.map_out[g], slot, col0, row0, idx);
                        bulk_commit();
                    }
                    ++nout;
                }
                if (!diag) {
                    // its transpose at (col0, row0): element (lane, e) goes to row e, column lane
                    uint8_t* slot = wout + (nout % kOutSlots) * kBlk;
                    if (nout >= kOutSlots && lane == 0) bulk_wait_read<kOutSlots - 1>();
                    __syncwarp();
                    const uint32_t cj = (uint32_t)lane >> 3, cb2 = ((uint32_t)lane & 7u) * 2u;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        *reinterpret_cast<uint16_t*>(slot + sw64((uint32_t)e, cj) + cb2) = b[e];
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        tma_store_3d(&p.map_out[g], slot, row0, col0, idx);
                        bulk_commit();
                    }
                    ++nout;
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (lane == 0) bulk_wait<0>();
    }

    if (*abort_flag && run) {
        // copies of the peer may still be landing in this CTA's stages (they are
        // counted on CTA 0's barriers): give them time before the CTA can exit
        const uint64_t t0 = global_timer_ns();
        while (global_timer_ns() - t0 < 2000000ull) {
        }
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync_all();  // no MMA, copy or remote arrival of the pair is still in flight
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if (tbase != kNoTmem) tmem_dealloc_pair(tbase, 512);
    }
}

cudaError_t ns_gram_pair_configure() {
    cudaError_t e = cudaFuncSetAttribute(k_ns_gram_pair<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGramSmem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_ns_gram_pair<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kGramSmem);
    return e;
}

// p.tiles: 256 x 256 tiles {group slot, index, tile row I, tile column J >= I} (units of 256).
template <bool F16>
cudaError_t launch_ns_gram_pair(const GemmParams& p, int num_sms, cudaStream_t stream) {
    if (p.ntiles <= 0) return cudaSuccess;
    const int pairs = p.ntiles < num_sms / 2 ? p.ntiles : num_sms / 2;
    k_ns_gram_pair<F16><<<2 * pairs, kSymThreads, kGramSmem, stream>>>(p);
    return cudaGetLastError();
}

template cudaError_t launch_ns_gram_pair<false>(const GemmParams&, int, cudaStream_t);
template cudaError_t launch_ns_gram_pair<true>(const GemmParams&, int, cudaStream_t);

}  // namespace muon
