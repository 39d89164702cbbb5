// The two symmetric products of the Newton-Schulz iteration on SM pairs
// ("modded-nanogpt 50B-token" write-up, section "Muon from the source",
// grouped as X <- a X + (b A + c A^2) X):
//
//   MODE_GRAM   A = sc * X X^T        (sc = (s / c)^2 on the first iteration, else 1)
//   MODE_POLY   P = b A + c A A       (A symmetric, so A A = A A^T: the same product
//                                      as the Gram with A's rows for X's; from the
//                                      second iteration on the epilogue adds a to
//                                      the diagonal: P' = a I + P)
// A Gram launch may also carry plain products C = L R for some of its groups
// (GemmGroup.b_mn: L and R symmetric polynomials in one Gram matrix, so they commute and
// C is symmetric; the Gram-space product A <- T P' rides along with the Gram matrices of
// the other groups): those tiles take an MN-major right operand and K = m.
//
// with tcgen05.mma.cta_group::2 (M = 256, N = 256, K = 16) issued by CTA 0 of a
// two-CTA cluster.  A pair tile is the 256 x 256 block (I, J), J >= I, of the
// symmetric result.  CTA r stages rows 256 I + 128 r .. + 127 of the operand
// (the left operand's half, K-major) and the right operand's half: for the
// Gram, rows 256 J + 128 r .. + 127 of X (K-major); for the polynomial,
// columns 256 J + 128 r .. + 127 of A (MN-major: A is symmetric, so its
// columns are its rows; the tensor cores read either layout at the same
// rate).  An off-diagonal tile stages 32 KB per SM per 64-deep k-block;
// a diagonal Gram tile, whose two halves are the same rows, 16 KB.  CTA r's
// TMEM receives rows 128 r .. + 127 of the tile.
//
// Storage of the symmetric results: the upper block triangle only.  A result is
// stored as its 256 x 256 blocks (I, J) with J >= I (a diagonal block whole, both
// triangles); nothing is written below.  Every SM-pair product that reads such a
// matrix (the polynomial here, the update kernel's products) takes a k-block that
// lies below the diagonal from the mirror block above it, loaded in the other
// layout: a left operand's rows 256 I + .. for k in block K < I are the columns
// 256 I + .. of rows k, an MN-major box; a right operand's columns 256 J + .. for k
// in block K > J are the rows 256 J + .. of columns k, a K-major box.  The tensor
// cores take either layout per k-block (instruction-descriptor major-ness bits), so
// a consumer reads exactly the bytes it read from a full matrix, and the producer
// stores a third fewer (six of nine blocks of a 768-wide matrix).
//
// The epilogue works warp by warp: warp (quad, half) owns TMEM lanes
// 32 quad .. + 31 and columns 32 half .. + 31 of each 64-column chunk, i.e.
// four 32 x 32 blocks per tile, and stores each block from its own ring of
// shared-memory slots.  The polynomial's b A term comes from A's own 32 x 32
// blocks (block (I, J) is stored), which each warp TMA-loads two blocks ahead
// into a private two-slot ring.  No barrier spans warps.
//
// Warp 0: TMA producer (both CTAs), warp 1: pair-wide TMEM allocation (both)
// and the MMA issuer (CTA 0), warps 2-9: epilogue (both).  All mbarrier waits
// are bounded (2 s) and raise the status word.
#include <type_traits>

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
constexpr int kOutSlots = 2;  // per warp: output blocks in flight

template <int MODE>
struct SymPairCfg {
    static constexpr bool POLY = MODE == MODE_POLY;
    static constexpr bool MNB = MODE == MODE_POLY;  // right operand MN-major (columns of a symmetric matrix)
    // the polynomial gives up one stage for its per-warp input ring (two 32 x 32 blocks of A)
    static constexpr int STAGES = POLY ? 5 : 6;
    static constexpr int IN_SLOTS = POLY ? 2 : 0;
    static constexpr int SMEM = STAGES * kSymStage + kEpiWarps * (kOutSlots + IN_SLOTS) * kBlk + 1024 + 512;
    static_assert(SMEM <= 232448, "shared memory budget");
};

}  // namespace

using namespace pair;

template <int MODE, bool F16>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kSymThreads, 1)
    k_ns_sym_pair(const __grid_constant__ GemmParams p) {
    using C = SymPairCfg<MODE>;
    constexpr int STAGES = C::STAGES;
    // Instruction descriptors by operand major-ness.  The Gram's operands are K-major; the
    // polynomial's right operand is MN-major (columns of the symmetric A), and so is that of
    // a Gram launch's groups with b_mn set.  A symmetric operand's k-blocks below the
    // diagonal come from its mirror blocks in the other major-ness (GemmGroup.sym_l / sym_r).
    constexpr uint32_t IDESC_KK = make_idesc_16bit_ab(256, 256, false, false, F16);
    constexpr uint32_t IDESC_KM = make_idesc_16bit_ab(256, 256, false, true, F16);
    constexpr uint32_t IDESC_MK = make_idesc_16bit_ab(256, 256, true, false, F16);
    constexpr uint32_t IDESC_MM = make_idesc_16bit_ab(256, 256, true, true, F16);
    // the polynomial of the second and later iterations adds a to the diagonal of P
    constexpr bool FOLD = C::POLY && F16;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sS = smem;                                   // STAGES x (left | right)
    uint8_t* sO = sS + STAGES * kSymStage;                // per warp kOutSlots blocks
    uint8_t* sI = sO + kEpiWarps * kOutSlots * kBlk;      // POLY: per warp IN_SLOTS blocks of A
    uint64_t* full = reinterpret_cast<uint64_t*>(sI + kEpiWarps * C::IN_SLOTS * kBlk);  // CTA 0's are used
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;   // [2]
    uint64_t* tempty = tfull + 2;       // [2] CTA 0's: 8 warps of each CTA arrive
    uint64_t* mma_done = tempty + 2;    // abort path only
    uint64_t* in_full = mma_done + 1;   // POLY: [kEpiWarps][2]
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(in_full + 2 * kEpiWarps);
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
        for (int i = 0; i < 2 * kEpiWarps; ++i) mbar_init(&in_full[i], 1);
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

    if (warp == 0) {
        // ------------------------------------------------------------ operand producer (both CTAs)
        if (lane == 0 && run) {
            for (int g = 0; g < p.ngroups; ++g) {
                tma_prefetch_desc(&p.map_a[g]);
                if (C::MNB || p.grp[g].b_mn) tma_prefetch_desc(&p.map_b[g]);
                if (p.grp[g].sym_l) tma_prefetch_desc(&p.map_al[g]);
                if (p.grp[g].sym_r) tma_prefetch_desc(&p.map_bk[g]);
            }
            const uint32_t full0 = cluster_addr(&full[0], 0);
            int stage = 0;
            uint32_t phase = 0;
            bool ok = true;
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = pr < p.ntiles ? p.tiles[pr] : make_int4(0, 0, 0, 0);
            for (int t = pr; t < p.ntiles && ok; t += npairs) {
                const int4 tile = tile_nx;
                if (t + npairs < p.ntiles) tile_nx = p.tiles[t + npairs];
                const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
                const bool mnb = C::MNB || p.grp[g].b_mn;
                const bool syl = p.grp[g].sym_l != 0, syr = p.grp[g].sym_r != 0;
                const int K = mnb ? p.grp[g].m : p.grp[g].n;
                const int nkb = (K + kBK - 1) / kBK;
                const bool diag = !mnb && ti == tj;  // a diagonal Gram tile stages one set of rows
                // k-blocks kb0 .. kb1 - 1 with one operand layout throughout: the left operand from
                // its mirror (LMN, MN-major) or its own rows; the right operand from its mirror
                // (RK, K-major) or as usual.  A loop per layout keeps each one's body minimal.
                auto produce = [&](auto lmn, auto rk, auto mnbv, auto diagv, int kb0, int kb1) {
                    constexpr bool LMN = decltype(lmn)::value, RK = decltype(rk)::value;
                    constexpr bool MN = decltype(mnbv)::value, DIAG = decltype(diagv)::value;
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
                            ok = false;
                            return;
                        }
                        if (leader) mbar_arrive_expect_tx(&full[stage], DIAG ? 2 * kSymRows : 2 * kSymStage);
                        const uint32_t bar = full0 + (uint32_t)(stage * 8);
                        uint8_t* dst = sS + stage * kSymStage;
                        if (LMN) {
                            // rows 256 I + 128 r .. + 127 of a symmetric left operand, k-block left
                            // of the diagonal: its mirror, rows kb of columns 256 I + 128 r .., as
                            // two MN-major 64-column boxes
                            const int col = ti * 256 + (int)rank * kBM;
                            tma_load_3d_pair(dst, &p.map_al[g], bar, col, kb * kBK, idx);
                            tma_load_3d_pair(dst + 64 * kBK * 2, &p.map_al[g], bar, col + 64, kb * kBK, idx);
                        } else {
                            tma_load_3d_pair(dst, &p.map_a[g], bar, kb * kBK, ti * 256 + (int)rank * kBM, idx);
                        }
                        if (RK) {
                            // a symmetric right operand's k-block below the diagonal: its mirror,
                            // the K-major rows 256 J + 128 r .. + 127
                            tma_load_3d_pair(dst + kSymRows, &p.map_bk[g], bar, kb * kBK, tj * 256 + (int)rank * 128,
                                             idx);
                        } else if (MN) {
                            // columns 256 J + 128 r .. + 127 of the right operand for k-block rows
                            // kb: two 64-column boxes
                            const int col = tj * 256 + (int)rank * 128;
                            tma_load_3d_pair(dst + kSymRows, &p.map_b[g], bar, col, kb * kBK, idx);
                            tma_load_3d_pair(dst + kSymRows + 64 * kBK * 2, &p.map_b[g], bar, col + 64, kb * kBK, idx);
                        } else if (!DIAG) {
                            tma_load_3d_pair(dst + kSymRows, &p.map_a[g], bar, kb * kBK, tj * 256 + (int)rank * kBM,
                                             idx);
                        }
                        if (++stage == STAGES) {
                            stage = 0;
                            phase ^= 1u;
                        }
                    }
                };
                using F_ = std::false_type;
                using T_ = std::true_type;
                if (mnb) {
                    // J >= I: the left operand's mirrored k-blocks (block K < I) all come before the
                    // right operand's (block K > J)
                    const int a_end = syl ? min(nkb, ti * (256 / kBK)) : 0;
                    const int b_beg = syr ? min(nkb, (tj + 1) * (256 / kBK)) : nkb;
                    produce(T_{}, F_{}, T_{}, F_{}, 0, a_end);
                    if (ok) produce(F_{}, F_{}, T_{}, F_{}, a_end, b_beg);
                    if (ok) produce(F_{}, T_{}, T_{}, F_{}, b_beg, nkb);
                } else if (diag) {
                    produce(F_{}, F_{}, F_{}, T_{}, 0, nkb);
                } else {
                    produce(F_{}, F_{}, F_{}, F_{}, 0, nkb);
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
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = pr < p.ntiles ? p.tiles[pr] : make_int4(0, 0, 0, 0);
            for (int t = pr; t < p.ntiles && ok; t += npairs) {
                const int4 tile = tile_nx;
                if (t + npairs < p.ntiles) tile_nx = p.tiles[t + npairs];
                const bool mnb = C::MNB || p.grp[tile.x].b_mn;
                const bool syl = p.grp[tile.x].sym_l != 0, syr = p.grp[tile.x].sym_r != 0;
                const int K = mnb ? p.grp[tile.x].m : p.grp[tile.x].n;
                const int nkb = (K + kBK - 1) / kBK;
                const bool diag = !mnb && tile.z == tile.w;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tbase + (uint32_t)(acc * 256);
                // Stages are taken two at a time: both waits first, then eight MMAs back to
                // back.  A wait between every four MMAs leaves the tensor pipe idle for part of
                // each k-block; eight in a row keep it busy.
                for (int kb = 0; kb < nkb; kb += 2) {
                    const int nst = kb + 1 < nkb ? 2 : 1;
                    int st1 = stage + 1;
                    uint32_t ph1 = phase;
                    if (st1 == STAGES) {
                        st1 = 0;
                        ph1 ^= 1u;
                    }
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status) ||
                        (nst == 2 && !mbar_wait(&full[st1], ph1, abort_flag, p.status))) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        if (h < nst) {
                            const int st = h ? st1 : stage;
                            const uint32_t a_st = s_base + st * kSymStage;
                            const uint32_t b_st = diag ? a_st : a_st + kSymRows;  // a diagonal tile's halves are the same rows
                            const int kblk = (kb + h) >> 2;
                            const bool a_mn = syl && kblk < tile.z;
                            const bool b_mn = mnb && !(syr && kblk > tile.w);
                            // the stage's descriptors; a 16-deep step adds to the start-address field
                            // (16-byte units): 32 bytes along a K-major operand, 16 rows of 128 bytes
                            // along an MN-major one (8 KB between its 64-column boxes)
                            const uint64_t ad = a_mn ? make_sdesc_sw128(a_st, 64 * kBK * 2, 1024)
                                                     : make_sdesc_sw128(a_st, 16, 1024);
                            const uint64_t bd = b_mn ? make_sdesc_sw128(b_st, 64 * kBK * 2, 1024)
                                                     : make_sdesc_sw128(b_st, 16, 1024);
                            const uint64_t a_step = a_mn ? 128 : 2, b_step = b_mn ? 128 : 2;
                            const uint32_t idesc = a_mn ? (b_mn ? IDESC_MM : IDESC_MK) : (b_mn ? IDESC_KM : IDESC_KK);
#pragma unroll
                            for (int kk = 0; kk < kBK / 16; ++kk)
                                umma_f16_pair(d_tmem, ad + a_step * (uint64_t)kk, bd + b_step * (uint64_t)kk, idesc,
                                              (kb | h | kk) != 0 ? 1u : 0u);
                            any = true;
                            umma_commit_pair(&empty[st]);
                        }
                    }
                    stage = st1;
                    phase = ph1;
                    if (nst == 2 && ++stage == STAGES) {
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
        uint8_t* win = sI + ew * (C::IN_SLOTS * kBlk);  // POLY: slot c & 1 holds A's block of chunk c
        uint64_t* ibar = &in_full[2 * ew];
        const uint32_t tempty0 = cluster_addr(&tempty[0], 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        int nout = 0;  // output slots used so far (one bulk group each)
        uint32_t in_phase[2] = {0u, 0u};
        bool in_pending[2] = {false, false};
        if (C::POLY && lane == 0)
            for (int g = 0; g < p.ngroups; ++g) tma_prefetch_desc(&p.map_ein[g]);
        // the tile list is read one tile ahead: no role waits on global memory between tiles
        int4 tile_nx = pr < p.ntiles ? p.tiles[pr] : make_int4(0, 0, 0, 0);
        for (int t = pr; run && t < p.ntiles; t += npairs) {
            const int4 tile = tile_nx;
            if (t + npairs < p.ntiles) tile_nx = p.tiles[t + npairs];
            const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
            const GemmGroup& G = p.grp[g];
            const int row0 = ti * 256 + (int)rank * kBM + quad * 32;  // this warp's first row
            // POLY: A's block of chunk c at (row0, this warp's columns of chunk c), lane 0 issues
            auto load_in = [&](int c, int sl) {
                mbar_arrive_expect_tx(&ibar[sl], kBlk);
                tma_load_3d(win + sl * kBlk, &p.map_ein[g], &ibar[sl], tj * 256 + c * 64 + half * 32, row0, idx);
                in_pending[sl] = true;
            };
            if (C::POLY && lane == 0) {
                load_in(0, 0);  // before the accumulator is ready
                load_in(1, 1);
            }
            mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
            tc_fence_after();
            uint32_t raw[2][32];
            const uint32_t t_acc = tbase + (uint32_t)(acc * 256) + lane_off + (uint32_t)(half * 32);
            // the iterate is stored as X / c (c = ||X0||): the first Gram scales u u^T by (s / c)^2;
            // A A carries a factor c^2 against the stored A / c^2
            const float cs = p.iter_scale[G.sub0 + idx];
            const float c2 = cs * cs;
            float scale = 1.f;
            if (!C::POLY && p.first) {
                const float s = p.norm_scale[G.sub0 + idx] / cs;
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
                        if (lane == 0) mbar_arrive_cluster_relaxed(tempty0 + (uint32_t)(acc * 8));
                    }
                }
                const int col0 = tj * 256 + c * 64 + half * 32;  // this block's first column
                float v[32];
                if (C::POLY) {
                    // P / c^2 = b (A / c^2) + c c^2 (A / c^2)^2 ; from the second iteration on
                    // P' = a I + c^2 (P / c^2), stored unscaled
                    const int sl = c & 1;
                    mbar_wait(&ibar[sl], in_phase[sl], abort_flag, p.status);
                    in_phase[sl] ^= 1u;
                    in_pending[sl] = false;
                    uint4 aw[4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        aw[jj] = *reinterpret_cast<const uint4*>(win + sl * kBlk + sw64((uint32_t)lane, (uint32_t)jj));
                    const int dcol = row0 + lane - col0;  // this lane's diagonal element, if in the block
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const uint32_t ws[4] = {aw[jj].x, aw[jj].y, aw[jj].z, aw[jj].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const int e = 8 * jj + 2 * h;
                            const float a0 = x2f<F16>((uint16_t)(ws[h] & 0xFFFFu));
                            const float a1 = x2f<F16>((uint16_t)(ws[h] >> 16));
                            float p0 = fmaf(p.cb, a0, (p.cc * c2) * __uint_as_float(raw[c & 1][e]));
                            float p1 = fmaf(p.cb, a1, (p.cc * c2) * __uint_as_float(raw[c & 1][e + 1]));
                            if (FOLD) {
                                p0 = c2 * p0 + (e == dcol ? p.ca : 0.f);
                                p1 = c2 * p1 + (e + 1 == dcol ? p.ca : 0.f);
                            }
                            v[e] = p0;
                            v[e + 1] = p1;
                        }
                    }
                    // The slot goes back to the copy engine only after every lane has used what it
                    // read (the loads are complete) and ordered those reads before the async
                    // proxy's write: otherwise, under heavy shared-memory traffic, the next block's
                    // copy could land before a lane's read of this one is served.
                    fence_async_smem();
                    __syncwarp();
                    if (lane == 0 && c + 2 < 4) load_in(c + 2, sl);
                } else {
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = scale * __uint_as_float(raw[c & 1][e]);
                }
                uint16_t b[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) b[e] = f2x<F16>(v[e]);

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
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (C::POLY && lane == 0) {
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

template <int MODE, bool F16>
static cudaError_t configure_sym() {
    return cudaFuncSetAttribute(k_ns_sym_pair<MODE, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SymPairCfg<MODE>::SMEM);
}

cudaError_t ns_gram_pair_configure() {
    cudaError_t e = configure_sym<MODE_GRAM, false>();
    if (e == cudaSuccess) e = configure_sym<MODE_GRAM, true>();
    if (e == cudaSuccess) e = configure_sym<MODE_POLY, false>();
    if (e == cudaSuccess) e = configure_sym<MODE_POLY, true>();
    return e;
}

// p.tiles: 256 x 256 tiles {group slot, index, tile row I, tile column J >= I} (units of 256).
// MODE_GRAM: p.map_a = 128-row boxes of the iterate (K = n); MODE_POLY: of A (K = m), with
// p.map_b = A's 64 x 64 boxes (the MN-major right operand) and p.map_ein = A's 32 x 32 boxes
// for the b A term; groups with b_mn set: p.map_a = 128-row boxes of L, p.map_b = 64 x 64
// boxes of R (K = m).  p.map_out: 32 x 32 boxes of the result.
template <int MODE, bool F16>
cudaError_t launch_ns_sym_pair(const GemmParams& p, int num_sms, bool overlap, cudaStream_t stream) {
    if (p.ntiles <= 0) return cudaSuccess;
    const int pairs = p.ntiles < num_sms / 2 ? p.ntiles : num_sms / 2;
    return launch_kernel(k_ns_sym_pair<MODE, F16>, dim3(2 * pairs), dim3(kSymThreads), SymPairCfg<MODE>::SMEM, stream,
                         overlap, p);
}

template cudaError_t launch_ns_sym_pair<MODE_GRAM, false>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_sym_pair<MODE_GRAM, true>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_sym_pair<MODE_POLY, false>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_sym_pair<MODE_POLY, true>(const GemmParams&, int, bool, cudaStream_t);

}  // namespace muon
