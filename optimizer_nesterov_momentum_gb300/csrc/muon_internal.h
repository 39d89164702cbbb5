// Internal types shared by the host runtime (muon_runtime.cu) and the kernels.
//
// Layout of the device state for one handle:
//   * momentum arena: one dense fp32 [rows x cols] block per parameter (S1).
//   * per split matrix ("sub"), in the wide orientation m x n (m <= n):
//       u16 / ulo16 Nesterov direction as a pair of bf16 arrays, u = hi + lo (S2)
//       x16         Newton-Schulz iterate after the first iteration, fp16 (the
//                   tensor-core operand), stored as X / c with c = ||X0|| so that
//                   small inputs stay inside fp16's range (A and P likewise as
//                   A / c^2, P / c^2); two buffers used in turn (S5-S7)
//       a16 / p16   A = X X^T and P = b A + c A A, m x m: bf16 in the first
//                   iteration (on u), fp16 after (S5, S6); from the second
//                   iteration on p16 holds P' = a I + P, unscaled
//       rowsq       per (256-column tile, column half, row) sums of O^2 from the
//                   last iteration (S8), part-major so that one thread per row
//                   reads (and the epilogue writes) neighbouring words
//       colsq       column lanes only: per (64-row slab, column) sums of O^2
//       v           second moment, fp32, one per lane (S8): [m] when the lanes are
//                   the rows of the wide orientation (the default), [n] when they
//                   are its columns
//       lane        per-lane update factor lr*lr_mul*gamma/sqrt(v) (S9)
//   Matrices with the same (m, n) form a group and sit back to back in each
//   arena, so one 3-D TMA descriptor (n, m, count) covers a whole group.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace muon {

constexpr int kMaxGroupsPerLaunch = 8;
constexpr int kTile = 64;            // edge of the elementwise tiles (K1 / K5)
constexpr int kBM = 128;             // Newton-Schulz tile rows (TMEM lanes)
constexpr int kBK = 64;              // k-block: 64 bf16 = one 128-byte swizzle row
constexpr int kBNSym = 256;          // Gram / polynomial tile columns
constexpr int kBNUpd = 256;          // update tile columns
constexpr float kNormEps = 1e-7f;
constexpr float kVFloor = 1e-10f;

// device hyper-parameter slots (muon_set_hparams)
enum { HP_LR = 0, HP_MU = 1, HP_BETA2 = 2, HP_WD = 3, HP_COUNT = 4 };

// Device copy of a step schedule (see muon_schedule in muon.h) and its counter.
struct DevSchedule {
    int64_t step;             // schedule index of the next step
    int64_t cooldown_start, cooldown_end, momentum_warmup;
    float lr_base, lr_floor, momentum_start, momentum_end;
};

// bits of the device status word.  TIMEOUT and PAIR are fatal: once either is
// raised the write-back, the second-moment update and the momentum update of
// every later step are skipped until muon_sync_status clears the word.
// NONFINITE records that some matrix had a non-finite update direction; only
// that matrix's step was skipped (per-matrix flag, rewritten every step).
enum { STATUS_TIMEOUT = 1, STATUS_PAIR = 2, STATUS_NONFINITE = 4 };  // PAIR: an SM pair did not get one shared TMEM allocation
constexpr int kStatusFatal = STATUS_TIMEOUT | STATUS_PAIR;

// NorMuon lanes (muon_config.normuon_lanes)
enum { LANES_SHORT_SIDE = 0, LANES_ROWS = 1, LANES_COLS = 2 };

enum GemmMode { MODE_GRAM = 0, MODE_POLY = 1, MODE_UPDATE = 2 };

struct SubDesc {
    // caller-side addressing (original orientation, rows x cols)
    int64_t grad_off;    // element offset of (0, 0) in the parent's grad / param
    int64_t ld;          // caller row stride (elements)
    float* mom;          // momentum of this sub, row stride ld_mom
    int64_t ld_mom;
    int32_t rows, cols;
    int32_t parent;
    int32_t transposed;  // rows > cols: worked on as its transpose
    int32_t vec;         // 8-wide vector access is legal (cols, ld, offsets multiples of 8)
    int32_t m, n;        // wide shape
    int32_t ldx;         // row stride of the wide arenas
    int32_t ntile_n;     // 256-column tiles per row (2 rowsq entries each)
    int32_t k1_tile0, k1_ntiles;  // range of this sub's elementwise tiles
    float lr_mul, wd_mul, shape_scale;
    int32_t lane_cols;   // NorMuon lanes are the columns of the wide orientation (n lanes), else its rows (m)
    int32_t colsq_tile0; // lane_cols: first (sub, slab) entry of this sub in the column-sum work list
    // wide-orientation arenas of this sub
    uint16_t* u16;        // hi half of u (bf16(u))
    uint16_t* ulo16;      // lo half of u (bf16(u - hi))
    const uint16_t* o16;  // final Newton-Schulz output (fp16), m x n, row stride ldx
    float* rowsq;         // (ntile_n x 2) x m, part-major
    float* colsq;         // lane_cols: ceil(m / 64) x n
    float* v;             // one per lane
    float* lane;          // one per lane
    int* skip;            // per-sub flag: this step's direction was not finite (written by k_norm_scale)
};

// Per-launch pointer table of the caller's buffers (kernel parameter; CAP
// entries so the parameter block stays small for small models).
template <int CAP>
struct PtrTable {
    const void* grad[CAP];
    float* param[CAP];
};

template <int CAP>
struct ElemParams {
    PtrTable<CAP> ptr;
    const SubDesc* subs;
    const int4* tiles;       // {sub, row0, col0, 0} over the original orientation
    int32_t ntiles;
    const float* hp;         // HP_* slots
    float* norm_part;        // one partial sum of u^2 per tile
    int32_t nesterov, lerp_form;
    const int* status;       // device status word: a fatal bit skips the kernel's writes
};

struct GemmGroup {
    int32_t m, n, ldx, lda;
    int32_t ntile_n;
    int32_t b_mn;            // SM-pair Gram launch: this group's tiles are plain products L R of two
                             // symmetric m x m matrices (right operand MN-major, K = m), not X X^T
    // SM-pair kernels: the left (sym_l) or right (sym_r) operand is a symmetric m x m matrix
    // stored as its upper block triangle (256 x 256 blocks (I, J) with J >= I; the SM-pair
    // symmetric products store nothing below).  A k-block below the diagonal is read from
    // the mirror block through the operand's other view (map_al / map_bk) and fed to the
    // tensor cores in the other major-ness.
    int32_t sym_l, sym_r;
    int32_t sub0;            // sub index of the group's first matrix (subs are group-ordered)
    int64_t x_stride;        // elements between matrices in x / u arenas (m * ldx)
    int64_t a_stride;        // elements between matrices in a / p arenas (m * lda)
    const uint16_t* xlo_in;  // first update: lo half of u read by the a*X term (hi: opr16); else nullptr
    uint16_t* xlo_out;       // unused (kept zero)
    uint16_t* x16_out;       // update: the next iterate / final O (fp16)
    const uint16_t* a16;     // poly epilogue: A (also simt operand)
    uint16_t* out16;         // gram: A, poly: P
    float* rowsq;            // update, last iteration: per-row sums of O^2 ([ntile_n * 2][m] per matrix)
    const uint16_t* opl16;   // simt: left operand base (gram: X, poly: A, update: P)
    const uint16_t* opr16;   // simt: right operand base (gram: X, poly: A, update: X)
};

struct GemmParams {
    CUtensorMap map_a[kMaxGroupsPerLaunch];     // left operand (K-major)
    CUtensorMap map_b[kMaxGroupsPerLaunch];     // right operand: 256-row K-major box (gram / poly), MN-major X (update)
    CUtensorMap map_ein[kMaxGroupsPerLaunch];   // epilogue input: poly A tile, first update hi half of u
    CUtensorMap map_ein2[kMaxGroupsPerLaunch];  // epilogue input: first update lo half of u
    CUtensorMap map_out[kMaxGroupsPerLaunch];   // gram/poly: A / P tile; update: X' tile
    CUtensorMap map_out2[kMaxGroupsPerLaunch];  // one-SM gram/poly: mirrored tile (the SM-pair kernels store none)
    CUtensorMap map_al[kMaxGroupsPerLaunch];    // sym_l: the left operand's MN-major boxes (64 columns)
    CUtensorMap map_bk[kMaxGroupsPerLaunch];    // sym_r: the right operand's K-major boxes (128 rows x 64)
    GemmGroup grp[kMaxGroupsPerLaunch];
    const int4* tiles;       // {group slot, index in group, tile row, tile col}
    int32_t ntiles;
    int32_t ngroups;
    const float* norm_scale; // s per sub (first iteration), else nullptr
    const float* iter_scale; // c per sub: X, A, P are stored as X / c, A / c^2, P / c^2
    float ca, cb, cc;        // (a, b, c) of this iteration
    int32_t first, last, want_rowsq;
    int32_t f16;             // operands and results fp16 (iterations after the first); else bf16
    int32_t pair;            // update on SM pairs: tiles are 256 x 256 (tile row and column in units of 256)
    int32_t debug_stall;     // test only (muon_debug_inject_stall): the MMA issuer first waits on an
                             // mbarrier that nothing arrives on, until its bounded wait gives up
    int* status;
};

struct LaneParams {
    const SubDesc* subs;
    int32_t nsubs;
    const float* hp;
    int32_t normuon, norm_preserve;
    const float* iter_scale;  // c per sub: the stored iterate is X / c
    const int* status;
};

struct NormParams {
    const SubDesc* subs;
    int32_t nsubs;
    const float* norm_part;
    float* norm_scale;
    float* iter_scale;        // c = ||u|| s = ||X0|| per sub (1 when u = 0)
    int* status;
};

// Column sums of O^2 for subs whose NorMuon lanes are the wide columns: one
// block per (sub, 64-row slab).
struct ColSumParams {
    const SubDesc* subs;
    const int2* work;         // {sub, slab}
    int32_t nwork;
};

// Launches kernel<<<grid, block, smem, s>>>(args...).  With `overlap` the launch carries
// programmatic stream serialization: its CTAs may be scheduled while the stream's
// previous kernel is still finishing, so the kernel must call grid_dep_wait() before it
// touches memory that earlier work wrote or reads.  Every kernel of the Muon step does.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                 bool overlap, const Args&... args) {
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr.val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cfg.attrs = &attr;
    cfg.numAttrs = overlap ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

}  // namespace muon
