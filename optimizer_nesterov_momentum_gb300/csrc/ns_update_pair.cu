// Newton-Schulz update on SM pairs ("modded-nanogpt 50B-token" write-up, section
// "Muon from the source": X <- a X + (b A + c A^2) X), on tcgen05.mma.cta_group::2:
//   first iteration   X1 = s (a u + P0 u_hi), u read as its bf16 hi + lo pair
//   later iterations  X' = P' X, with a I folded into P' = a I + b A + c A^2 by
//                     the polynomial kernel
//
// The two CTAs of a cluster share one 256 x 256 output tile: CTA r holds rows
// 128 r .. 128 r + 127 of the tile's left operand (P' rows, K-major) and
// columns 128 r .. 128 r + 127 of its right operand (X rows, MN-major), and its
// own TMEM receives its 128 rows of the product.  The MMA, issued by CTA 0
// (M = 256, N = 256, K = 16), reads both CTAs' shared memory.  Each SM thus
// stages 32 KB per 64 of depth for the same 4.2 MFLOP that a one-SM 128 x 256
// tile stages 48 KB for: the update's mainloop is bound by how fast shared
// memory fills, so this is 1.5x the math per staged byte.
//
// The same kernel computes the Gram pairs' m x m products T = A P' and
// Q = P'' P'.  A symmetric operand (P', A, P'') is stored as its upper block
// triangle (GemmGroup.sym_l / sym_r): a left-operand k-block left of the
// diagonal comes from the mirror block as MN-major boxes, a right-operand
// k-block below it as K-major boxes, and the MMA's instruction descriptor
// takes the matching major-ness per k-block.  The producer runs one copy loop
// per layout run of a tile (at most three).
//
// Warp roles (320 threads per CTA, one CTA per SM):
//   warp 0     TMA producer (both CTAs): loads its own halves into its own
//              stage ring; every copy signals CTA 0's "full" mbarrier, which
//              CTA 0's producer armed with the bytes of both halves
//   warp 1     TMEM: one pair-wide 512-column allocation, made together by
//              warp 1 of both CTAs (the accumulator is double-buffered); CTA
//              0's lane 0 issues the MMAs and commits stage releases and
//              "accumulator full" to both CTAs' mbarriers at once (multicast
//              commit)
//   warps 2-9  epilogue (both CTAs): drain this CTA's 128 accumulator rows
//              into registers and release the accumulator on CTA 0's mbarrier,
//              then round to fp16 (the first iteration first adds a u, from
//              32 x 32 blocks of u's hi and lo halves each warp TMA-loads two
//              chunks ahead), stage and TMA-store warp by warp (each warp its
//              own 32 x 32 blocks, no barrier across warps); NorMuon row sums
//              on the last iteration
// Every mbarrier wait is bounded (2 s) and raises the status word on expiry.
// The allocation is checked before use: both CTAs must see the same TMEM
// address, else the kernel reports the mismatch in the status word and does
// no work.
#include <type_traits>

#include "muon_internal.h"
#include "pair_sm103.cuh"
#include "ptx_sm103.cuh"

namespace muon {
namespace {

constexpr int kPairThreads = 320;
constexpr int kWarpSlot = 32 * 32 * 2;   // one warp's 32 x 32 16-bit block (64-byte rows, 64-byte swizzle)
constexpr int kWarpSlots = 2;            // output staging slots per epilogue warp
constexpr int kPairEpiWarps = 8;
constexpr int kPairOutBytes = kPairEpiWarps * kWarpSlots * kWarpSlot;
constexpr uint32_t kNoTmem = 0xFFFFFFFFu;

// HILO: the first iteration, X1 = (s / c)(a u + c^2 (P / c^2) u_hi) with u a bf16
// hi + lo pair: bf16 operands, and each warp reads its 32 x 32 blocks of u's hi and
// lo halves for the a u term (two chunks ahead, by TMA).  Otherwise the folded
// fp16 update, which reads nothing.
//
// A stage holds one BK-deep k-block: this CTA's 128 rows of P' as BK / 64 K-major
// boxes of 128 x 64, and its 128 columns of X as two MN-major boxes of BK x 64.  The
// folded update takes 128-deep k-blocks: every copy is then a 16 KB box, which the
// copy engine moves faster per byte than the 8 KB boxes of 64-deep ones.  The first
// iteration keeps 64-deep k-blocks, because its epilogue input ring leaves room for
// only 128 KB of stages.
template <bool HILO>
struct UpdPairCfg {
    static constexpr int BK = HILO ? 64 : 128;
    static constexpr int A_BYTES = kBM * BK * 2;
    static constexpr int B_BYTES = 128 * BK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = HILO ? 4 : 3;
    static constexpr int IN_WARP = HILO ? 2 * 2 * kWarpSlot : 0;  // two chunks in flight, hi and lo
    static constexpr int SMEM = STAGES * STAGE + kPairOutBytes + kPairEpiWarps * IN_WARP + 1024 + 512;
    static_assert(SMEM <= 232448, "shared memory budget");
    // by operand major-ness: P' (or another left operand) K-major and X MN-major, except
    // where a symmetric operand's k-block comes from its mirror (GemmGroup.sym_l / sym_r)
    static constexpr uint32_t IDESC_KM = make_idesc_16bit_ab(256, 256, false, true, /*fp16=*/!HILO);
    static constexpr uint32_t IDESC_MM = make_idesc_16bit_ab(256, 256, true, true, !HILO);
    static constexpr uint32_t IDESC_KK = make_idesc_16bit_ab(256, 256, false, false, !HILO);
    static constexpr uint32_t IDESC_MK = make_idesc_16bit_ab(256, 256, true, false, !HILO);
};

}  // namespace

using namespace pair;

template <bool HILO>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    k_ns_update_pair(const __grid_constant__ GemmParams p) {
    using C = UpdPairCfg<HILO>;
    constexpr int kPairStages = C::STAGES;
    constexpr int BK = C::BK;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = sA + kPairStages * C::A_BYTES;
    uint8_t* sO = sB + kPairStages * C::B_BYTES;
    uint8_t* sI = sO + kPairOutBytes;  // HILO: per warp two chunks of (hi | lo) blocks
    uint64_t* full = reinterpret_cast<uint64_t*>(sI + kPairEpiWarps * C::IN_WARP);  // CTA 0's are used
    uint64_t* empty = full + kPairStages;
    uint64_t* tfull = empty + kPairStages;  // [2]
    uint64_t* tempty = tfull + 2;           // [2] CTA 0's are used: 8 warps of each CTA arrive
    uint64_t* mma_done = tempty + 2;        // abort path only
    uint64_t* in_full = mma_done + 1;       // HILO: [kPairEpiWarps][2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(in_full + 2 * kPairEpiWarps);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* pair_ok = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_rank();
    const bool leader = rank == 0;
    const int pair = (int)(blockIdx.x >> 1), npairs = (int)(gridDim.x >> 1);

    if (threadIdx.x == 0) {
        for (int s = 0; s < kPairStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], 2 * kPairEpiWarps);
        }
        mbar_init(mma_done, 1);
        for (int i = 0; i < 2 * kPairEpiWarps; ++i) mbar_init(&in_full[i], 1);
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
    // everything above touches only this pair's shared memory and TMEM, and may overlap the
    // previous kernel's last tiles; global memory only from here on
    grid_dep_wait();
    grid_dep_launch();
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
    const uint32_t tacc[2] = {tbase, tbase + 256u};
    bool mma_any = false;

    if (warp == 0) {
        // ------------------------------------------------------------ operand producer
        if (lane == 0 && run) {
            for (int g = 0; g < p.ngroups; ++g) {
                tma_prefetch_desc(&p.map_a[g]);
                tma_prefetch_desc(&p.map_b[g]);
                if (p.grp[g].sym_l) tma_prefetch_desc(&p.map_al[g]);
                if (p.grp[g].sym_r) tma_prefetch_desc(&p.map_bk[g]);
            }
            const uint32_t full0 = cluster_addr(&full[0], 0);  // CTA 0's full barriers
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = pair < p.ntiles ? p.tiles[pair] : make_int4(0, 0, 0, 0);
            for (int t = pair; t < p.ntiles && ok; t += npairs) {
                const int4 tile = tile_nx;
                if (t + npairs < p.ntiles) tile_nx = p.tiles[t + npairs];
                const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
                const int nkb = (p.grp[g].m + BK - 1) / BK;
                const int row0 = ti * 2 * kBM + (int)rank * kBM;
                const int col0 = tj * 256 + (int)rank * 128;
                const bool syl = p.grp[g].sym_l != 0, syr = p.grp[g].sym_r != 0;
                // k-blocks kb0 .. kb1 - 1 with one operand layout throughout: the left operand from
                // its mirror (LMN) or its own rows, the right one from its mirror (RK) or as usual.
                // A loop per layout keeps each one's body minimal.
                auto produce = [&](auto lmn, auto rk, int kb0, int kb1) {
                    constexpr bool LMN = decltype(lmn)::value, RK = decltype(rk)::value;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
                            ok = false;
                            return;
                        }
                        if (leader) mbar_arrive_expect_tx(&full[stage], 2 * C::STAGE);
                        const uint32_t bar = full0 + (uint32_t)(stage * 8);
                        uint8_t* da = sA + stage * C::A_BYTES;
                        uint8_t* db = sB + stage * C::B_BYTES;
                        if (LMN) {
                            // a symmetric left operand left of the diagonal: the mirror block's
                            // columns row0 .. + 127 of rows kb, two MN-major boxes of BK x 64
                            tma_load_3d_pair(da, &p.map_al[g], bar, row0, kb * BK, idx);
                            tma_load_3d_pair(da + BK * 128, &p.map_al[g], bar, row0 + 64, kb * BK, idx);
                        } else {
#pragma unroll
                            for (int ks = 0; ks < BK / 64; ++ks)
                                tma_load_3d_pair(da + ks * (kBM * 128), &p.map_a[g], bar, kb * BK + ks * 64, row0, idx);
                        }
                        if (RK) {
                            // a symmetric right operand below the diagonal: the mirror block's rows
                            // col0 .. + 127 of columns kb, BK / 64 K-major boxes of 128 x 64
#pragma unroll
                            for (int ks = 0; ks < BK / 64; ++ks)
                                tma_load_3d_pair(db + ks * (128 * 128), &p.map_bk[g], bar, kb * BK + ks * 64, col0, idx);
                        } else {
                            tma_load_3d_pair(db, &p.map_b[g], bar, col0, kb * BK, idx);
                            tma_load_3d_pair(db + BK * 128, &p.map_b[g], bar, col0 + 64, kb * BK, idx);
                        }
                        if (++stage == kPairStages) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                };
                using F_ = std::false_type;
                using T_ = std::true_type;
                if (!syl && !syr) {
                    produce(F_{}, F_{}, 0, nkb);
                } else {
                    // left mirrored for k in blocks K < I, right for K > J: at most three runs
                    const int a_end = syl ? min(nkb, ti * (256 / BK)) : 0;
                    const int b_beg = syr ? min(nkb, (tj + 1) * (256 / BK)) : nkb;
                    if (a_end <= b_beg) {
                        produce(T_{}, F_{}, 0, a_end);
                        if (ok) produce(F_{}, F_{}, a_end, b_beg);
                        if (ok) produce(F_{}, T_{}, b_beg, nkb);
                    } else {
                        produce(T_{}, F_{}, 0, b_beg);
                        if (ok) produce(T_{}, T_{}, b_beg, a_end);
                        if (ok) produce(F_{}, T_{}, a_end, nkb);
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
            bool ok = true;
            const uint32_t a_base = smem_u32(sA);
            const uint32_t b_base = smem_u32(sB);
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = pair < p.ntiles ? p.tiles[pair] : make_int4(0, 0, 0, 0);
            for (int t = pair; t < p.ntiles && ok; t += npairs) {
                const int4 tile = tile_nx;
                if (t + npairs < p.ntiles) tile_nx = p.tiles[t + npairs];
                const int nkb = (p.grp[tile.x].m + BK - 1) / BK;
                const bool syl = p.grp[tile.x].sym_l != 0, syr = p.grp[tile.x].sym_r != 0;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // the stage's descriptors; a 16-deep step adds to the start-address field
                    // (16-byte units): 32 bytes along a 64-wide K-major box (16 KB to the next
                    // box), 16 rows of 128 bytes along an MN-major operand (BK rows per 64-column
                    // box).  Left K-major and right MN-major, except for a symmetric operand's
                    // mirrored k-blocks.
                    const int kblk = (kb * BK) >> 8;
                    const bool a_mn = syl && kblk < tile.z;
                    const bool b_mn = !(syr && kblk > tile.w);
                    const uint64_t ad = make_sdesc_sw128(a_base + stage * C::A_BYTES, a_mn ? BK * 128 : 16, 1024);
                    const uint64_t bd = make_sdesc_sw128(b_base + stage * C::B_BYTES, b_mn ? BK * 128 : 16, 1024);
                    const uint32_t idesc =
                        a_mn ? (b_mn ? C::IDESC_MM : C::IDESC_MK) : (b_mn ? C::IDESC_KM : C::IDESC_KK);
#pragma unroll
                    for (int kk = 0; kk < BK / 16; ++kk) {
                        const uint64_t kmaj = (uint64_t)((kk >> 2) * (kBM * 128 / 16) + (kk & 3) * 2);
                        const uint64_t mnmaj = (uint64_t)(kk * 128);
                        umma_f16_pair(tacc[acc], ad + (a_mn ? mnmaj : kmaj), bd + (b_mn ? mnmaj : kmaj), idesc,
                                      (kb | kk) != 0 ? 1u : 0u);
                    }
                    mma_any = true;
                    umma_commit_pair(&empty[stage]);
                    if (++stage == kPairStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                umma_commit_pair(&tfull[acc]);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            if (!ok && mma_any) {
                // the MMAs in flight read both CTAs' stages and write both TMEMs
                umma_commit_pair(mma_done);
                mbar_wait_drain(mma_done, 0, 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue (both CTAs)
        // Each warp drains its 32 TMEM lanes x 32 columns of every 64-column chunk and
        // stores that 32 x 32 block itself from a ring of private staging slots: no
        // barrier across warps.
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        uint8_t* wst = sO + (warp - 2) * (kWarpSlots * kWarpSlot);
        uint8_t* win = sI + (warp - 2) * C::IN_WARP;  // HILO: slot c holds hi | lo of a chunk
        uint64_t* ibar = &in_full[2 * (warp - 2)];
        const uint32_t tempty0 = cluster_addr(&tempty[0], 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        int wchunk = 0;  // chunks this warp has staged
        uint32_t in_phase[2] = {0u, 0u};
        bool in_pending[2] = {false, false};
        if (HILO && lane == 0)
            for (int g = 0; g < p.ngroups; ++g) {
                tma_prefetch_desc(&p.map_ein[g]);
                tma_prefetch_desc(&p.map_ein2[g]);
            }
        // the tile list is read one tile ahead: no role waits on global memory between tiles
        int4 tile_nx = pair < p.ntiles ? p.tiles[pair] : make_int4(0, 0, 0, 0);
        for (int t = pair; run && t < p.ntiles; t += npairs) {
            const int4 tile = tile_nx;
            if (t + npairs < p.ntiles) tile_nx = p.tiles[t + npairs];
            const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
            const GemmGroup& G = p.grp[g];
            const int row0 = ti * 2 * kBM + (int)rank * kBM + quad * 32;  // this warp's first row
            auto load_in = [&](int c, int sl) {  // u's hi and lo blocks of chunk c (HILO, lane 0)
                mbar_arrive_expect_tx(&ibar[sl], 2 * kWarpSlot);
                const int col = tj * 256 + c * 64 + half * 32;
                tma_load_3d(win + sl * 2 * kWarpSlot, &p.map_ein[g], &ibar[sl], col, row0, idx);
                tma_load_3d(win + sl * 2 * kWarpSlot + kWarpSlot, &p.map_ein2[g], &ibar[sl], col, row0, idx);
                in_pending[sl] = true;
            };
            if (HILO && lane == 0) {
                load_in(0, 0);  // before the accumulator is ready
                load_in(1, 1);
            }
            mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
            tc_fence_after();
            const uint32_t t_acc = tacc[acc] + lane_off + (uint32_t)(half * 32);
            float sumsq = 0.f;
            float scale = 1.f, c2 = 1.f;
            if (HILO) {
                // the first iteration: X1 / c = (s / c)(a u + c^2 (P0 / c^2) u_hi)
                const float cs = p.iter_scale[G.sub0 + idx];
                scale = p.norm_scale[G.sub0 + idx] / cs;
                c2 = cs * cs;
            }
            // LB chunks in flight per TMEM wait (all four for the folded update); after the
            // last wait the accumulator is in registers and goes back to the MMA
            constexpr int LB = HILO ? 2 : 4;
            uint32_t raw[LB][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                if (c % LB == 0) {
#pragma unroll
                    for (int i = 0; i < LB; ++i) tmem_load_32x32_async(t_acc + (c + i) * 64, raw[i]);
                    tmem_wait_loads();
                    if (c + LB == 4) {
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0) mbar_arrive_cluster_relaxed(tempty0 + (uint32_t)(acc * 8));
                    }
                }
                const uint32_t* r32 = raw[c % LB];
                uint32_t ow[4][4];
                if (HILO) {
                    const int sl = c & 1;
                    mbar_wait(&ibar[sl], in_phase[sl], abort_flag, p.status);
                    in_phase[sl] ^= 1u;
                    in_pending[sl] = false;
                    uint4 hw[4], lw[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        hw[jj] = *reinterpret_cast<const uint4*>(win + sl * 2 * kWarpSlot + sw64((uint32_t)lane, (uint32_t)jj));
                        lw[jj] = *reinterpret_cast<const uint4*>(win + sl * 2 * kWarpSlot + kWarpSlot +
                                                                 sw64((uint32_t)lane, (uint32_t)jj));
                    }
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t hs[4] = {hw[jj].x, hw[jj].y, hw[jj].z, hw[jj].w};
                        const uint32_t ls[4] = {lw[jj].x, lw[jj].y, lw[jj].z, lw[jj].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float x0 = __uint_as_float(hs[h] << 16) + __uint_as_float(ls[h] << 16);
                            const float x1 = __uint_as_float(hs[h] & 0xFFFF0000u) + __uint_as_float(ls[h] & 0xFFFF0000u);
                            const float y0 = scale * fmaf(p.ca, x0, c2 * __uint_as_float(r32[8 * jj + 2 * h]));
                            const float y1 = scale * fmaf(p.ca, x1, c2 * __uint_as_float(r32[8 * jj + 2 * h + 1]));
                            const __half2 hv = __floats2half2_rn(y0, y1);
                            ow[jj][h] = *reinterpret_cast<const uint32_t*>(&hv);
                            if (p.want_rowsq) {
                                const float2 o = __half22float2(hv);
                                sumsq = fmaf(o.x, o.x, sumsq);
                                sumsq = fmaf(o.y, o.y, sumsq);
                            }
                        }
                    }
                    // the slot goes back to the copy engine only after every lane has used what it
                    // read and ordered those reads before the async proxy's write
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && c + 2 < 4) load_in(c + 2, sl);
                } else {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const __half2 hv = __floats2half2_rn(__uint_as_float(r32[8 * jj + 2 * h]),
                                                                 __uint_as_float(r32[8 * jj + 2 * h + 1]));
                            ow[jj][h] = *reinterpret_cast<const uint32_t*>(&hv);
                            if (p.want_rowsq) {
                                const float2 o = __half22float2(hv);
                                sumsq = fmaf(o.x, o.x, sumsq);
                                sumsq = fmaf(o.y, o.y, sumsq);
                            }
                        }
                    }
                }
                uint8_t* slot = wst + (wchunk % kWarpSlots) * kWarpSlot;
                // the store issued kWarpSlots chunks ago read this slot: it must be done with it
                if (wchunk >= kWarpSlots && lane == 0) bulk_wait_read<kWarpSlots - 1>();
                __syncwarp();
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    *reinterpret_cast<uint4*>(slot + sw64((uint32_t)lane, (uint32_t)jj)) =
                        make_uint4(ow[jj][0], ow[jj][1], ow[jj][2], ow[jj][3]);
                fence_async_smem();
                __syncwarp();
                if (lane == 0) {
                    tma_store_3d(&p.map_out[g], slot, tj * 256 + c * 64 + half * 32, row0, idx);
                    bulk_commit();
                }
                ++wchunk;
            }
            if (p.want_rowsq && G.rowsq != nullptr) {
                const int row = row0 + lane;
                if (row < G.m)  // part-major: [matrix][256-column tile, half][row]
                    G.rowsq[((int64_t)idx * G.ntile_n * 2 + tj * 2 + half) * G.m + row] = sumsq;
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (HILO && lane == 0) {
            // input copies of an aborted run still in flight must land before the CTA exits
#pragma unroll
            for (int sl = 0; sl < 2; ++sl)
                if (in_pending[sl]) mbar_wait_drain(&ibar[sl], in_phase[sl], 100000000ull);
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

cudaError_t ns_update_pair_configure() {
    cudaError_t e = cudaFuncSetAttribute(k_ns_update_pair<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         UpdPairCfg<false>::SMEM);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(k_ns_update_pair<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 UpdPairCfg<true>::SMEM);
    return e;
}

// p.tiles: 256 x 256 tiles {group slot, index, tile row (of 256), tile column (of 256)}.
// hilo: the first iteration (bf16 operands, u read as hi + lo for the a u term).
cudaError_t launch_ns_update_pair(const GemmParams& p, bool hilo, int num_sms, bool overlap, cudaStream_t stream) {
    if (p.ntiles <= 0) return cudaSuccess;
    const int pairs = p.ntiles < num_sms / 2 ? p.ntiles : num_sms / 2;
    if (hilo)
        return launch_kernel(k_ns_update_pair<true>, dim3(2 * pairs), dim3(kPairThreads), UpdPairCfg<true>::SMEM, stream,
                             overlap, p);
    return launch_kernel(k_ns_update_pair<false>, dim3(2 * pairs), dim3(kPairThreads), UpdPairCfg<false>::SMEM, stream,
                         overlap, p);
}

}  // namespace muon
