// Grouped Newton-Schulz GEMMs on the 5th-generation tensor cores (tcgen05).
//
// One persistent kernel template serves the three products of an iteration
// (the quintic map of the Muon orthogonalisation, "modded-nanogpt 50B-token"
// write-up, section "Muon from the source", grouped as X <- a X + (b A + c A^2) X):
//
//   MODE_GRAM    A = sc * X X^T           (sc = s^2 on the first iteration, s = 1/(||u||+eps))
//   MODE_POLY    P = b A + c A A          (A symmetric, so A A = sum_k A[i,k] A[j,k])
//   MODE_UPDATE  X' = s (a X + P X)       on the first iteration
//                X' = P X                 on later ones, whose POLY adds a to the
//                                         diagonal of P: a X + P X = (a I + P) X
//                                         (these run on SM pairs, ns_update_pair.cu,
//                                         where the shapes tile by 256)
//
// A and P are symmetric: GRAM and POLY compute 128 x 256 tiles that reach the
// diagonal or lie above it, and store every 128 x 128 block above the
// diagonal twice (itself and its mirror) and the diagonal block once; the
// 64-column chunks of a tile that fall below the diagonal are neither
// staged nor stored.  The left
// operand is always K-major (rows of X, A or P); the right operand is K-major
// for GRAM / POLY (rows again, thanks to the symmetry) and MN-major for
// UPDATE (X[k, j] with j contiguous), selected in the instruction descriptor.
//
// Warp roles (352 threads, one CTA per SM, persistent over a tile list):
//   warp 0     TMA producer (one thread): 128 B-swizzled operand tiles into a
//              ring of shared-memory stages, completion tracked by mbarriers
//   warp 1     TMEM allocator + MMA issuer (one thread): tcgen05.mma M=128,
//              N=128/256, K=16 into a double-buffered TMEM accumulator
//   warps 2-9  epilogue: tcgen05.ld of the accumulator (warp w reads TMEM lanes
//              32*(w%4)..+31; warps 2-5 take the first half of every column
//              chunk, warps 6-9 the second), combine in fp32, round, write
//              swizzled shared-memory staging tiles; one thread issues TMA
//              bulk stores
//   warp 10    epilogue loader (one thread, POLY and the first UPDATE):
//              TMA-loads the tiles the epilogue combines with (A for POLY; the
//              hi and lo halves of u for the first UPDATE) into an input ring
//              whose slots come back as soon as every epilogue thread has read
//              its part into registers; results go to a separate output
//              staging area that the bulk stores read from
// Precision: the first iteration runs on the Nesterov direction u, held as a
// bf16 pair u = hi + lo (about 16 mantissa bits): hi is the tensor-core
// operand of the Gram and the update, and the first update rebuilds u from
// both halves for its a*X term.  Its result and every later X, A and P are
// fp16, stored divided by a per-matrix scale (X / c, A / c^2, P / c^2 with
// c = ||X0|| <= 1) that keeps them near unit size whatever the gradient's norm;
// the folded P' = a I + P of the later iterations is stored unscaled.
// Every wait is bounded (2 s); on a timeout the kernel sets the status word,
// lets copies and MMAs in flight finish, frees TMEM and returns.  After an
// abort no role re-arms an mbarrier whose copy might still be in flight: the
// producer's stages come back only through MMA commits (which follow landed
// copies), and the epilogue loader stops issuing as soon as it sees the abort
// flag (the epilogue may then release input slots without waiting for them);
// both drain the copies they issued before the CTA exits.
#include "muon_internal.h"
#include "ptx_sm103.cuh"

namespace muon {

// F16: operands and results in fp16 (the iterations after the first); otherwise
// bf16 operands (the first iteration, on the Nesterov direction u).
template <int MODE, bool F16>
struct TcCfg {
    static constexpr bool UPD = (MODE == MODE_UPDATE);
    static constexpr bool SYM = !UPD;
    // from the second iteration on, the a X term rides on the tensor cores: POLY adds a
    // to the diagonal of P and UPDATE is the plain product, with no epilogue input
    static constexpr bool FOLD = F16;
    static constexpr int BN = UPD ? kBNUpd : kBNSym;
    // the mainloop is bound by stages in flight against load latency: four where the
    // epilogue's staging leaves room (the Gram and the folded update have no input)
    static constexpr int STAGES = (MODE == MODE_GRAM || (UPD && FOLD)) ? 4 : 3;
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int TMEM_COLS = 2 * BN;
    static constexpr bool B_MN = UPD;
    static constexpr uint32_t IDESC = make_idesc_16bit(kBM, BN, B_MN, F16);
    static constexpr uint32_t IDESC_N128 = make_idesc_16bit(kBM, 128, B_MN, F16);  // right half of a tile
    // epilogue: column chunks; an input ring (TMA-loaded operands of the
    // combine) and a double-buffered output staging area (read by TMA stores).
    // The first update reads u as a bf16 hi | lo pair (32 columns per chunk);
    // later updates read nothing (64 columns).  Updates write fp16.
    static constexpr bool HILO_IN = UPD && !FOLD;
    static constexpr int CHUNK = HILO_IN ? 32 : 64;      // columns per chunk
    static constexpr int NCHUNK = BN / CHUNK;
    static constexpr bool HAS_EIN = (MODE == MODE_POLY) || HILO_IN;
    static constexpr int HALF_BYTES = kBM * 32 * 2;                                     // 128 x 32, 16-bit
    static constexpr int ISLOTS = HILO_IN ? 3 : (HAS_EIN ? 1 : 0);
    static constexpr int IN_BYTES = kBM * 64 * 2;        // u hi | lo (32 columns) / A (64 columns)
    static constexpr int OSLOTS = (MODE == MODE_GRAM) ? 1 : 2;
    static constexpr int OUT_BYTES = UPD ? kBM * 64 * 2 : 2 * kBM * 64 * 2;           // X' / out | mirror
    static constexpr int SMEM_BYTES =
        STAGES * STAGE_BYTES + ISLOTS * IN_BYTES + OSLOTS * OUT_BYTES + 1024 /*align*/ + 512;
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
    static_assert(!HAS_EIN || ISLOTS >= 1, "an epilogue with inputs needs an input slot");
    static_assert(OSLOTS >= 1 && OSLOTS <= 2, "two output-buffer mbarriers are reserved");
};

// Operand sharing in the symmetric products.  The rows of tile (ti, tj) are
// rows of the operand too, so a tile whose rows lie inside its own 256-column
// block needs fewer bytes:
//   SYM_FULL   rows outside the block: 128 left rows + 256 right rows per k-block
//   SYM_LEFT   ti == 2 tj: the left operand is the first half of the right one
//   SYM_RIGHT  ti == 2 tj + 1: only the right half of the tile is live (the left
//              half lies below the diagonal), and it is the 128 x 128 product of
//              those same rows with themselves: one 128-row load, N = 128, into
//              TMEM columns 128..255
enum { SYM_FULL = 0, SYM_LEFT = 1, SYM_RIGHT = 2 };
__device__ __forceinline__ int sym_tile_kind(int ti, int tj) {
    return ti == 2 * tj ? SYM_LEFT : (ti == 2 * tj + 1 ? SYM_RIGHT : SYM_FULL);
}

// A 64-column chunk of a symmetric tile is live unless its 128-column block
// lies left of (below) the diagonal block of the tile's rows.
__device__ __forceinline__ bool sym_chunk_live(int ti, int tj, int c) {
    return ((tj * kBNSym + c * 64) >> 7) >= ti;
}

constexpr int kThreads = 352;
constexpr int kEpiThreads = 256;  // warps 2-9
constexpr int kLoaderWarp = 10;
constexpr int kStoreThread = 64;  // warp 2, lane 0: issues and tracks the bulk stores

template <int MODE, bool F16>
__global__ void __launch_bounds__(kThreads, 1) k_ns_gemm_tc(const __grid_constant__ GemmParams p) {
    using C = TcCfg<MODE, F16>;
    constexpr int BN = C::BN;
    constexpr int STAGES = C::STAGES;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * C::A_BYTES;
    uint8_t* sI = sB + STAGES * C::B_BYTES;     // ISLOTS x IN_BYTES: epilogue inputs
    uint8_t* sO = sI + C::ISLOTS * C::IN_BYTES;  // OSLOTS x OUT_BYTES: epilogue outputs
    uint64_t* full = reinterpret_cast<uint64_t*>(sO + C::OSLOTS * C::OUT_BYTES);
    uint64_t* empty = full + STAGES;
    uint64_t* tfull = empty + STAGES;      // [2] accumulator ready
    uint64_t* tempty = tfull + 2;          // [2] accumulator drained
    uint64_t* ein_full = tempty + 2;       // [ISLOTS] epilogue input landed
    uint64_t* ein_empty = ein_full + 4;    // [ISLOTS] input read by every epilogue thread
    uint64_t* mma_done = ein_empty + 4;    // abort path only
    uint64_t* obuf_free = mma_done + 1;    // [OSLOTS] output staging buffer read by its bulk store
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(obuf_free + 2);
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
            mbar_init(&tempty[a], kEpiThreads / 32);
        }
        for (int s = 0; s < C::ISLOTS; ++s) {
            mbar_init(&ein_full[s], 1);
            mbar_init(&ein_empty[s], kEpiThreads);
        }
        mbar_init(mma_done, 1);
        for (int b = 0; b < C::OSLOTS; ++b) mbar_init(&obuf_free[b], 1);
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
    // everything above touches only this CTA's shared memory and TMEM, and may overlap the
    // previous kernel's last tiles; global memory only from here on
    grid_dep_wait();
    grid_dep_launch();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------------------ operand producer
        if (lane == 0) {
            for (int g = 0; g < p.ngroups; ++g) {
                tma_prefetch_desc(&p.map_a[g]);
                tma_prefetch_desc(&p.map_b[g]);
            }
            int stage = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[STAGES];
            bool issued[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) issued[s] = false;
            bool ok = true;
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = blockIdx.x < p.ntiles ? p.tiles[blockIdx.x] : make_int4(0, 0, 0, 0);
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                const int4 tile = tile_nx;
                if (t + gridDim.x < p.ntiles) tile_nx = p.tiles[t + gridDim.x];
                const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
                const int K = (MODE == MODE_GRAM) ? p.grp[g].n : p.grp[g].m;
                const int nkb = (K + kBK - 1) / kBK;
                const int kind = C::SYM ? sym_tile_kind(ti, tj) : SYM_FULL;
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    uint8_t* a_dst = sA + stage * C::A_BYTES;
                    uint8_t* b_dst = sB + stage * C::B_BYTES;
                    if (C::B_MN) {
                        mbar_arrive_expect_tx(&full[stage], C::STAGE_BYTES);
                        tma_load_3d(a_dst, &p.map_a[g], &full[stage], kb * kBK, ti * kBM, idx);
#pragma unroll
                        for (int c = 0; c < BN / 64; ++c)
                            tma_load_3d(b_dst + c * (64 * kBK * 2), &p.map_b[g], &full[stage], tj * BN + c * 64,
                                        kb * kBK, idx);
                    } else if (kind == SYM_RIGHT) {
                        // the tile's own 128 rows only, in the left-operand slot
                        mbar_arrive_expect_tx(&full[stage], C::A_BYTES);
                        tma_load_3d(a_dst, &p.map_a[g], &full[stage], kb * kBK, tj * BN + kBM, idx);
                    } else {
                        mbar_arrive_expect_tx(&full[stage], kind == SYM_LEFT ? C::B_BYTES : C::STAGE_BYTES);
                        if (kind == SYM_FULL) tma_load_3d(a_dst, &p.map_a[g], &full[stage], kb * kBK, ti * kBM, idx);
                        // the right operand's 256 rows in one box
                        tma_load_3d(b_dst, &p.map_b[g], &full[stage], kb * kBK, tj * BN, idx);
                    }
                    issued[stage] = true;
                    issued_phase[stage] = phase;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok || *abort_flag) {
                // after an abort the MMA may not have consumed the last copies: let every
                // copy already issued land before the CTA can exit
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
            // test only: wait on an mbarrier nothing arrives on (mma_done is armed only on the
            // abort path, which needs any == true) until the bounded wait gives up
            if (p.debug_stall) ok = mbar_wait(mma_done, 0u, abort_flag, p.status);
            const uint32_t a_base = smem_u32(sA);
            const uint32_t b_base = smem_u32(sB);
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = blockIdx.x < p.ntiles ? p.tiles[blockIdx.x] : make_int4(0, 0, 0, 0);
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                const int4 tile = tile_nx;
                if (t + gridDim.x < p.ntiles) tile_nx = p.tiles[t + gridDim.x];
                const int g = tile.x;
                const int K = (MODE == MODE_GRAM) ? p.grp[g].n : p.grp[g].m;
                const int nkb = (K + kBK - 1) / kBK;
                const int kind = C::SYM ? sym_tile_kind(tile.z, tile.w) : SYM_FULL;
                const uint32_t idesc = kind == SYM_RIGHT ? C::IDESC_N128 : C::IDESC;
                if (!mbar_wait(&tempty[acc], acc_phase ^ 1u, abort_flag, p.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                // SYM_RIGHT accumulates only the tile's right half: TMEM columns 128..255
                const uint32_t d_tmem = tmem_base + (uint32_t)(acc * BN) + (kind == SYM_RIGHT ? 128u : 0u);
                for (int kb = 0; kb < nkb; ++kb) {
                    if (!mbar_wait(&full[stage], phase, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    // SYM_LEFT: the left operand is the first 128 rows of the right one;
                    // SYM_RIGHT: both operands are the 128 rows in the left slot
                    const uint32_t a_st = kind == SYM_LEFT ? b_base + stage * C::B_BYTES : a_base + stage * C::A_BYTES;
                    const uint32_t b_st = kind == SYM_RIGHT ? a_base + stage * C::A_BYTES : b_base + stage * C::B_BYTES;
#pragma unroll
                    for (int kk = 0; kk < kBK / 16; ++kk) {
                        const uint64_t adesc = make_sdesc_sw128(a_st + kk * 32, 16, 1024);
                        const uint64_t bdesc = C::B_MN ? make_sdesc_sw128(b_st + kk * (16 * 128), 64 * kBK * 2, 1024)
                                                       : make_sdesc_sw128(b_st + kk * 32, 16, 1024);
                        umma_bf16(d_tmem, adesc, bdesc, idesc, (kb | kk) != 0 ? 1u : 0u);
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
    } else if (warp == kLoaderWarp) {
        // ------------------------------------------------------------ epilogue loader
        if (C::HAS_EIN && lane == 0) {
            for (int g = 0; g < p.ngroups; ++g) {
                tma_prefetch_desc(&p.map_ein[g]);
                if (C::HILO_IN) tma_prefetch_desc(&p.map_ein2[g]);
            }
            int slot = 0;
            uint32_t phase = 0;
            uint32_t issued_phase[C::ISLOTS > 0 ? C::ISLOTS : 1];
            bool issued[C::ISLOTS > 0 ? C::ISLOTS : 1];
#pragma unroll
            for (int s = 0; s < C::ISLOTS; ++s) issued[s] = false;
            bool ok = true;
            // the tile list is read one tile ahead: no role waits on global memory between tiles
            int4 tile_nx = blockIdx.x < p.ntiles ? p.tiles[blockIdx.x] : make_int4(0, 0, 0, 0);
            for (int t = blockIdx.x; t < p.ntiles && ok; t += gridDim.x) {
                const int4 tile = tile_nx;
                if (t + gridDim.x < p.ntiles) tile_nx = p.tiles[t + gridDim.x];
                const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
                for (int c = 0; c < C::NCHUNK; ++c) {
                    if (C::SYM && !sym_chunk_live(ti, tj, c)) continue;
                    if (!mbar_wait(&ein_empty[slot], phase ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    // after an abort the epilogue hands slots back without waiting for their
                    // copies: re-arming one could overlap a copy still landing, so stop here
                    if (*abort_flag) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(&ein_full[slot], C::IN_BYTES);
                    uint8_t* dst = sI + slot * C::IN_BYTES;
                    tma_load_3d(dst, &p.map_ein[g], &ein_full[slot], tj * BN + c * C::CHUNK, ti * kBM, idx);
                    if (C::HILO_IN)
                        tma_load_3d(dst + C::HALF_BYTES, &p.map_ein2[g], &ein_full[slot], tj * BN + c * C::CHUNK,
                                    ti * kBM, idx);
                    issued[slot] = true;
                    issued_phase[slot] = phase;
                    if (++slot == C::ISLOTS) {
                        slot = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!ok || *abort_flag) {
                // every slot's last copy must have landed before the CTA can exit
#pragma unroll
                for (int s = 0; s < C::ISLOTS; ++s)
                    if (issued[s]) mbar_wait_drain(&ein_full[s], issued_phase[s], 100000000ull);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ epilogue
        const int quad = warp & 3;
        const int half = (warp - 2) >> 2;                  // which half of each column chunk
        const uint32_t r = (uint32_t)(quad * 32 + lane);  // row within the tile = TMEM lane
        const uint32_t lane_off = (uint32_t)(quad * 32) << 16;
        const bool store_thread = threadIdx.x == kStoreThread;
        int acc = 0;
        uint32_t acc_phase = 0;
        int islot = 0;       // input ring position
        uint32_t iphase = 0;
        int ochunk = 0;      // chunks staged so far (output buffer = ochunk % OSLOTS)
        // The epilogue never leaves its loops early: after an abort every wait returns
        // at once and the remaining tiles run through on scratch data, so all epilogue
        // threads always meet at the same named barriers.  Each thread waits on the
        // mbarriers itself; the one barrier per chunk orders the staging writes before
        // the store thread's bulk stores.
        // the tile list is read one tile ahead: no role waits on global memory between tiles
        int4 tile_nx = blockIdx.x < p.ntiles ? p.tiles[blockIdx.x] : make_int4(0, 0, 0, 0);
        for (int t = blockIdx.x; t < p.ntiles; t += gridDim.x) {
            const int4 tile = tile_nx;
            if (t + gridDim.x < p.ntiles) tile_nx = p.tiles[t + gridDim.x];
            const int g = tile.x, idx = tile.y, ti = tile.z, tj = tile.w;
            const GemmGroup& G = p.grp[g];
            mbar_wait(&tfull[acc], acc_phase, abort_flag, p.status);
            tc_fence_after();
            const uint32_t t_acc = tmem_base + lane_off + (uint32_t)(acc * BN);
            // the iterate is stored as X / c (c = ||X0||): the first Gram scales u u^T by
            // (s / c)^2, the first update u by s / c; A A and P X carry a factor c^2
            const float cs = p.iter_scale[G.sub0 + idx];
            const float c2 = cs * cs;
            float scale = 1.f;
            if (p.first && MODE != MODE_POLY) {
                const float s = p.norm_scale[G.sub0 + idx] / cs;
                scale = (MODE == MODE_GRAM) ? s * s : s;
            }
            float sumsq = 0.f;
            for (int c = 0; c < C::NCHUNK; ++c) {
                if (C::SYM && !sym_chunk_live(ti, tj, c)) continue;  // below the diagonal: nothing to do
                uint8_t* ein = sI + islot * C::IN_BYTES;
                const int ob = ochunk % C::OSLOTS;
                uint8_t* obuf = sO + ob * C::OUT_BYTES;
                const int col0 = tj * BN + c * C::CHUNK;
                const bool mirror = C::SYM && (col0 >> 7) > ti;  // strictly above the diagonal block
                // the bulk store that last read this output buffer must be done with it
                auto wait_obuf = [&]() {
                    if (ochunk >= C::OSLOTS)
                        mbar_wait(&obuf_free[ob], (uint32_t)((ochunk / C::OSLOTS - 1) & 1), abort_flag, p.status);
                };
                if (C::HILO_IN) {
                    // first update: X0 = s u with u as a bf16 hi | lo pair; X1 in fp16
                    float v[16];
                    tmem_load_32x16(t_acc + c * 32 + half * 16, v);
                    // inputs: hi and lo halves of u, rows of 64 bytes, 64-byte swizzle
                    mbar_wait(&ein_full[islot], iphase, abort_flag, p.status);
                    uint4 hw[2], lw[2];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const uint32_t j = (uint32_t)(half * 2 + jj);
                        hw[jj] = *reinterpret_cast<const uint4*>(ein + sw64(r, j));
                        lw[jj] = *reinterpret_cast<const uint4*>(ein + C::HALF_BYTES + sw64(r, j));
                    }
                    mbar_arrive(&ein_empty[islot]);  // this thread is done with the input slot
                    uint32_t ow[2][4];
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const uint32_t hs[4] = {hw[jj].x, hw[jj].y, hw[jj].z, hw[jj].w};
                        const uint32_t ls[4] = {lw[jj].x, lw[jj].y, lw[jj].z, lw[jj].w};
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const float x0 = __uint_as_float(hs[h] << 16) + __uint_as_float(ls[h] << 16);
                            const float x1 = __uint_as_float(hs[h] & 0xFFFF0000u) + __uint_as_float(ls[h] & 0xFFFF0000u);
                            const uint16_t b0 = f2h(scale * fmaf(p.ca, x0, c2 * v[8 * jj + 2 * h]));
                            const uint16_t b1 = f2h(scale * fmaf(p.ca, x1, c2 * v[8 * jj + 2 * h + 1]));
                            ow[jj][h] = (uint32_t)b0 | ((uint32_t)b1 << 16);
                            if (p.want_rowsq) {
                                const float o0 = h2f(b0), o1 = h2f(b1);
                                sumsq = fmaf(o0, o0, sumsq);
                                sumsq = fmaf(o1, o1, sumsq);
                            }
                        }
                    }
                    wait_obuf();
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj)
                        *reinterpret_cast<uint4*>(obuf + sw64(r, (uint32_t)(half * 2 + jj))) =
                            make_uint4(ow[jj][0], ow[jj][1], ow[jj][2], ow[jj][3]);
                } else if (MODE == MODE_UPDATE) {
                    // later updates: X' / c = P' (X / c) with P' = a I + P, no input;
                    // fp16 out, 64-column chunks, 128-byte swizzle
                    float v[32];
                    tmem_load_32x32(t_acc + c * 64 + half * 32, v);
                    uint32_t ow[4][4];
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
#pragma unroll
                        for (int h = 0; h < 4; ++h) {
                            const uint16_t b0 = f2h(v[8 * jj + 2 * h]);
                            const uint16_t b1 = f2h(v[8 * jj + 2 * h + 1]);
                            ow[jj][h] = (uint32_t)b0 | ((uint32_t)b1 << 16);
                            if (p.want_rowsq) {
                                const float o0 = h2f(b0), o1 = h2f(b1);
                                sumsq = fmaf(o0, o0, sumsq);
                                sumsq = fmaf(o1, o1, sumsq);
                            }
                        }
                    }
                    wait_obuf();
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj)
                        *reinterpret_cast<uint4*>(obuf + sw128(r, (uint32_t)(half * 4 + jj))) =
                            make_uint4(ow[jj][0], ow[jj][1], ow[jj][2], ow[jj][3]);
                } else {
                    float v[32];
                    tmem_load_32x32(t_acc + c * 64 + half * 32, v);
                    if (MODE == MODE_POLY) {
                        mbar_wait(&ein_full[islot], iphase, abort_flag, p.status);
                        uint4 aw[4];
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj)
                            aw[jj] = *reinterpret_cast<const uint4*>(ein + sw128(r, (uint32_t)(half * 4 + jj)));
                        mbar_arrive(&ein_empty[islot]);  // this thread is done with the input slot
#pragma unroll
                        for (int jj = 0; jj < 4; ++jj) {
                            const uint32_t ws[4] = {aw[jj].x, aw[jj].y, aw[jj].z, aw[jj].w};
#pragma unroll
                            for (int h = 0; h < 4; ++h) {
                                const float lo = x2f<F16>((uint16_t)(ws[h] & 0xFFFFu)), hi = x2f<F16>((uint16_t)(ws[h] >> 16));
                                v[8 * jj + 2 * h] = fmaf(p.cb, lo, (p.cc * c2) * v[8 * jj + 2 * h]);
                                v[8 * jj + 2 * h + 1] = fmaf(p.cb, hi, (p.cc * c2) * v[8 * jj + 2 * h + 1]);
                            }
                        }
                        if (C::FOLD) {
                            // P' = a I + P, stored unscaled (P' multiplies X / c into X' / c);
                            // c <= 1, so it stays near a in size
                            const int dcol = ti * kBM + (int)r - (col0 + half * 32);
#pragma unroll
                            for (int e = 0; e < 32; ++e) v[e] = c2 * v[e] + (e == dcol ? p.ca : 0.f);
                        }
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] *= scale;
                    }
                    uint16_t b[32];
#pragma unroll
                    for (int e = 0; e < 32; ++e) b[e] = f2x<F16>(v[e]);
                    wait_obuf();
                    uint8_t* eout = obuf;                  // 128 x 64 bf16, 128-byte swizzle
                    uint8_t* emir = obuf + kBM * 64 * 2;  // transposed chunk: two 64 x 64 boxes
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        uint4 w;
                        w.x = (uint32_t)b[8 * jj + 0] | ((uint32_t)b[8 * jj + 1] << 16);
                        w.y = (uint32_t)b[8 * jj + 2] | ((uint32_t)b[8 * jj + 3] << 16);
                        w.z = (uint32_t)b[8 * jj + 4] | ((uint32_t)b[8 * jj + 5] << 16);
                        w.w = (uint32_t)b[8 * jj + 6] | ((uint32_t)b[8 * jj + 7] << 16);
                        *reinterpret_cast<uint4*>(eout + sw128(r, (uint32_t)(half * 4 + jj))) = w;
                    }
                    if (mirror) {
                        // element (r, e) of this chunk goes to row e, column r of the transposed
                        // chunk, stored as two 64 x 64 boxes (columns r / 64)
                        uint8_t* mbox = emir + (r >> 6) * (64 * 128);
                        const uint32_t rc = r & 63u;
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const uint32_t me = (uint32_t)(half * 32 + e);
                            *reinterpret_cast<uint16_t*>(mbox + sw128(me, rc >> 3) + (rc & 7u) * 2) = b[e];
                        }
                    }
                }
                fence_async_smem();
                named_barrier(1, kEpiThreads);
                if (store_thread) {
                    if (MODE == MODE_UPDATE) {
                        if (col0 < G.n) tma_store_3d(&p.map_out[g], obuf, col0, ti * kBM, idx);
                    } else if (col0 < G.m) {
                        tma_store_3d(&p.map_out[g], obuf, col0, ti * kBM, idx);
                        if (mirror) {
                            uint8_t* emir = obuf + kBM * 64 * 2;
                            tma_store_3d(&p.map_out2[g], emir, ti * kBM, col0, idx);
                            if (ti * kBM + 64 < G.m) tma_store_3d(&p.map_out2[g], emir + 64 * 128, ti * kBM + 64, col0, idx);
                        }
                    }
                    bulk_commit();
                    // once the store of chunk ochunk - (OSLOTS - 1) has read its buffer, chunk
                    // ochunk + 1 (which uses that buffer) may be staged
                    if (ochunk >= C::OSLOTS - 1) {
                        bulk_wait_read<C::OSLOTS - 1>();
                        mbar_arrive(&obuf_free[(ochunk - (C::OSLOTS - 1)) % C::OSLOTS]);
                    }
                }
                ++ochunk;
                if (C::HAS_EIN && ++islot == C::ISLOTS) {
                    islot = 0;
                    iphase ^= 1u;
                }
            }
            if (MODE == MODE_UPDATE && p.want_rowsq) {
                const int row = ti * kBM + (int)r;
                if (row < G.m)  // part-major: [matrix][256-column tile, half][row]
                    G.rowsq[((int64_t)idx * G.ntile_n * 2 + tj * 2 + half) * G.m + row] = sumsq;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (store_thread) bulk_wait<0>();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        tmem_dealloc(tmem_base, C::TMEM_COLS);
    }
}

template <int MODE, bool F16>
static cudaError_t configure_one() {
    return cudaFuncSetAttribute(k_ns_gemm_tc<MODE, F16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                TcCfg<MODE, F16>::SMEM_BYTES);
}

cudaError_t ns_gemm_tc_configure() {
    cudaError_t e = configure_one<MODE_GRAM, false>();
    if (e == cudaSuccess) e = configure_one<MODE_GRAM, true>();
    if (e == cudaSuccess) e = configure_one<MODE_POLY, false>();
    if (e == cudaSuccess) e = configure_one<MODE_POLY, true>();
    if (e == cudaSuccess) e = configure_one<MODE_UPDATE, false>();
    if (e == cudaSuccess) e = configure_one<MODE_UPDATE, true>();
    return e;
}

template <int MODE, bool F16>
cudaError_t launch_ns_gemm_tc(const GemmParams& p, int num_sms, bool overlap, cudaStream_t stream) {
    using C = TcCfg<MODE, F16>;
    if (p.ntiles <= 0) return cudaSuccess;
    const int grid = p.ntiles < num_sms ? p.ntiles : num_sms;
    return launch_kernel(k_ns_gemm_tc<MODE, F16>, dim3(grid), dim3(kThreads), C::SMEM_BYTES, stream, overlap, p);
}

template cudaError_t launch_ns_gemm_tc<MODE_GRAM, false>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_GRAM, true>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_POLY, false>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_POLY, true>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_UPDATE, false>(const GemmParams&, int, bool, cudaStream_t);
template cudaError_t launch_ns_gemm_tc<MODE_UPDATE, true>(const GemmParams&, int, bool, cudaStream_t);

}  // namespace muon
