// Host runtime behind include/muon.h: validates shapes, builds the execution
// plan (matrix groups, tile work lists, arenas, TMA descriptors) once at
// muon_create, and replays a fixed launch sequence on every muon_step:
//
//   k_momentum -> k_norm_scale -> ns_steps x (gram -> poly -> update) -> k_lane_stats -> k_apply
//
// muon_step allocates nothing and never synchronises the host, so a caller
// can capture it in a CUDA graph.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "../../include/muon.h"
#include "muon_internal.h"

namespace muon {
// kernels (elementwise.cu, ns_gemm_tc.cu, ns_gemm_simt.cu)
template <int CAP>
cudaError_t launch_momentum(const ElemParams<CAP>&, bool, bool, cudaStream_t);
template <int CAP>
cudaError_t launch_apply(const ElemParams<CAP>&, bool, cudaStream_t);
cudaError_t launch_norm_scale(const NormParams&, bool, cudaStream_t);
cudaError_t launch_lane_stats(const LaneParams&, bool, cudaStream_t);
cudaError_t launch_col_sumsq(const ColSumParams&, bool, cudaStream_t);
cudaError_t launch_set_hparams(float*, float, float, float, float, cudaStream_t);
cudaError_t launch_schedule_set(DevSchedule*, const DevSchedule&, cudaStream_t);
cudaError_t launch_schedule_advance(float*, DevSchedule*, cudaStream_t);
cudaError_t launch_combine_hilo(float*, const uint16_t*, const uint16_t*, int, int, int, cudaStream_t);
cudaError_t launch_scale_f16(float*, const uint16_t*, const float*, int, int, int, cudaStream_t);
cudaError_t ns_gemm_tc_configure();
cudaError_t ns_update_pair_configure();
cudaError_t launch_ns_update_pair(const GemmParams&, bool, int, bool, cudaStream_t);
cudaError_t ns_gram_pair_configure();
template <int MODE, bool F16>
cudaError_t launch_ns_sym_pair(const GemmParams&, int, bool, cudaStream_t);
template <int MODE, bool F16>
cudaError_t launch_ns_gemm_tc(const GemmParams&, int, bool, cudaStream_t);
template <int MODE>
cudaError_t launch_ns_gemm_simt(const GemmParams&, int, int, cudaStream_t);
}  // namespace muon

using namespace muon;

namespace {

constexpr float kDefaultCoeffs[3] = {3.4445f, -4.7750f, 2.0315f};

thread_local std::string g_create_error;

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

struct Group {
    int32_t m = 0, n = 0;
    int32_t count = 0;
    int32_t ldx = 0, lda = 0, ntile_n = 0;
    int32_t sub0 = 0;
    // device arenas (count matrices back to back); u and X are hi + lo bf16 pairs
    uint16_t* u16 = nullptr;
    uint16_t* ulo16 = nullptr;
    uint16_t* x16[2] = {nullptr, nullptr};
    uint16_t* a16 = nullptr;
    uint16_t* p16 = nullptr;
    // Gram-pair iterations (muon_config.ns_form): the second polynomial of a pair and
    // T = A P', whose buffer then holds Q = P'' P'
    int32_t gs = 0;
    int32_t final_buf = 0;  // the iterate buffer that ends up holding the last output
    uint16_t* pb16 = nullptr;
    uint16_t* t16 = nullptr;
    float* rowsq = nullptr;
    float* v = nullptr;
    float* lane = nullptr;
    float* colsq = nullptr;   // column lanes: per matrix ceil(m / 64) x n
    int32_t lane_stride = 0;  // floats per matrix in v / lane: m, or n when some matrix has column lanes
    // TMA descriptors: bf16 operand boxes (64 x 128, 64 x 64), 32 x 128 boxes of
    // the iterate's hi and lo halves for the update epilogue, mirror boxes of A / P
    CUtensorMap map_u_k, map_u_mn, map_x_k[2], map_x_mn[2], map_a_k, map_p_k;
    CUtensorMap map_x_mn128[2];  // X as MN-major boxes 128 rows deep (the SM-pair folded update's 128-deep k-blocks)
    // Gram-pair groups: P as the MN-major right operand of the plain products, the
    // second polynomial and T (or Q) as 128-row K-major left operands, and their stores
    CUtensorMap map_p_mn, map_p_mn128, map_pb_k, map_pb_w32, map_t_k, map_t_w32;
    // MN-major 64 x 128 boxes of A and of the second polynomial: the SM-pair update kernel's
    // left operand below the diagonal (T = A P', Q = P'' P'; see GemmGroup.sym_l); 64 x 64
    // boxes of T: the left operand of A <- T P' below the diagonal
    CUtensorMap map_a_mn128, map_pb_mn128, map_t_mn;
    CUtensorMap map_u_k256, map_x_k256[2], map_a_k256;  // 64 x 256 boxes: right operand of gram / poly
    CUtensorMap map_a_mn;      // 64 x 64 boxes of A: the MN-major right operand of the SM-pair polynomial
    CUtensorMap map_u_hi, map_u_lo, map_x_o32[2], map_a_mir, map_p_mir;
    CUtensorMap map_x_w32[2];  // 32 x 32 boxes, 64-byte swizzle: stores of the SM-pair update's warps
    CUtensorMap map_a_w32;     // the same for A (SM-pair Gram stores, SM-pair polynomial's b A input)
    CUtensorMap map_p_w32;     // and for P (SM-pair polynomial stores)
    CUtensorMap map_u_hi_w32, map_u_lo_w32;  // and for u's halves (first SM-pair update)
};

struct Chunk {        // up to kMaxGroupsPerLaunch groups per GEMM launch
    // Every tile list below is followed by the same tiles with the matrix order reversed
    // within each cost class (at offset off + n): successive GEMM launches alternate
    // between the two orders, so that each starts on the matrices its predecessor wrote
    // last, which are the ones most likely still in L2.
    int32_t ng = 0;
    int32_t gi[kMaxGroupsPerLaunch] = {};  // the chunk's groups (indices into muon_s::groups)
    int32_t gram_off = 0, gram_n = 0;
    int32_t poly_off = 0, poly_n = 0;
    int32_t upd_off = 0, upd_n = 0;
    int32_t pair_off = 0, pair_n = 0;  // 256 x 256 update tiles for SM pairs (0: chunk not eligible)
    int32_t spg_off = 0, spg_n = 0;    // 256 x 256 Gram tiles (J >= I) for SM pairs
    // Gram-pair chunks: the update tiles of the standard-form groups together with the m x m
    // tiles on or above the diagonal of the Gram-pair groups (the first half of a pair computes
    // the symmetric T = A P' in the update launch), and the full m x m tiles of the Gram-pair
    // groups alone (Q = P'' P')
    int32_t pair_t_off = 0, pair_t_n = 0;
    int32_t pair_q_off = 0, pair_q_n = 0;
    // The launch of Q also takes the first update tiles of the standard-form groups (they
    // depend only on their own polynomial, which precedes it) when that fills its last wave
    // of SM pairs and saves one in the update launch after it: q_fill[sl] of group slot sl's
    // tiles move.  pair_qx: the Q tiles and those; pair_ux: every update tile but those.
    int32_t q_fill[kMaxGroupsPerLaunch] = {};
    int32_t q_fill_n = 0;
    int32_t pair_qx_off = 0, pair_qx_n = 0;
    int32_t pair_ux_off = 0, pair_ux_n = 0;
};

// One Newton-Schulz launch of the step, in order.
struct Launch {
    int32_t stage;  // MUON_STAGE_*
    int32_t mode;   // GemmMode
    int32_t chunk;
    int32_t it;     // Newton-Schulz iteration
    int32_t pair;   // SM-pair kernels
    int32_t f16;    // fp16 operands (iterations after the first)
};

typedef CUresult (*PFN_encodeTiled)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                    const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                    CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

}  // namespace

struct muon_s {
    bool alive = true;
    int device = 0;
    int num_sms = 0;
    muon_config cfg{};
    std::vector<float> coeffs;          // ns_steps * 3
    std::vector<muon_shape> shapes;
    std::vector<float> lr_mul, wd_mul;
    std::vector<SubDesc> subs;          // group-ordered
    std::vector<int32_t> sub_parent_q;  // split index of each sub
    std::vector<Group> groups;
    std::vector<Chunk> chunks;
    std::vector<int64_t> mom_off;       // per parent, offset into momentum arena (floats)
    int32_t n_elem_tiles = 0;
    int32_t n_colwork = 0;              // (sub, slab) blocks of k_col_sumsq (column lanes only)
    bool stall_next = false;            // muon_debug_inject_stall: the next step's first one-SM polynomial stalls
    int stall_chunk = -1;               // the launch chunk whose polynomial runs on one SM per tile
    // device memory
    void* arena = nullptr;
    size_t arena_bytes = 0;
    float* hp = nullptr;
    int* status = nullptr;
    DevSchedule* sched = nullptr;  // step schedule + counter (zero at create)
    bool schedule_on = false;      // muon_step starts with the schedule kernel
    float* norm_scale = nullptr;
    float* iter_scale = nullptr;   // c = ||X0|| per sub
    float* norm_part = nullptr;
    float* momentum = nullptr;
    SubDesc* d_subs = nullptr;
    int* skip = nullptr;               // per sub: this step's direction was not finite
    int2* d_colwork = nullptr;
    int4* d_elem_tiles = nullptr;
    int4* d_gemm_tiles = nullptr;
    // the Newton-Schulz launches of one step and their pre-built parameter blocks
    std::vector<Launch> plan;
    std::vector<GemmParams> gparams;
    // algorithmic work of one step per stage (muon_stage_work)
    int64_t work_flops[MUON_NUM_STAGES] = {};
    int64_t work_bytes[MUON_NUM_STAGES] = {};
    int32_t work_launches[MUON_NUM_STAGES] = {};
    std::string last_error;
    // profiling: one event before every launch plus one at the end
    bool profiling = false;
    std::vector<cudaEvent_t> events;
    std::vector<int> event_stage;  // stage of the launch that follows event k
    int n_recorded = 0;
};

namespace {

std::mutex g_handles_mu;
std::set<muon_s*> g_handles;

int fail(muon_s* h, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    if (h)
        h->last_error = buf;
    else
        g_create_error = buf;
    return code;
}

int check_handle(muon_s* h) {
    if (h == nullptr) return fail(nullptr, MUON_ERR_ARG, "null handle");
    std::lock_guard<std::mutex> lk(g_handles_mu);
    if (g_handles.find(h) == g_handles.end()) return fail(nullptr, MUON_ERR_ARG, "unknown handle");
    if (!h->alive) return fail(h, MUON_ERR_DESTROYED, "handle was destroyed");
    return MUON_OK;
}

#define MUON_CUDA(h, call)                                                                              \
    do {                                                                                               \
        cudaError_t e_ = (call);                                                                       \
        if (e_ != cudaSuccess) return fail((h), MUON_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

PFN_encodeTiled get_encode_fn() {
    static PFN_encodeTiled fn = nullptr;
    if (fn) return fn;
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    fn = reinterpret_cast<PFN_encodeTiled>(p);
    return fn;
}

// 3-D tensor map over `count` matrices of rows x cols (row stride ld elements,
// matrices back to back), box {box_cols, box_rows, 1}.
bool encode_3d(PFN_encodeTiled enc, CUtensorMap* map, CUtensorMapDataType dtype, int esize, void* base, int64_t cols,
               int64_t rows, int64_t count, int64_t ld, uint32_t box_cols, uint32_t box_rows,
               CUtensorMapSwizzle swz) {
    cuuint64_t dims[3] = {(cuuint64_t)cols, (cuuint64_t)rows, (cuuint64_t)count};
    cuuint64_t strides[2] = {(cuuint64_t)(ld * esize), (cuuint64_t)(ld * esize * rows)};
    cuuint32_t box[3] = {box_cols, box_rows, 1};
    cuuint32_t estr[3] = {1, 1, 1};
    CUresult r = enc(map, dtype, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                     CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_bf16_3d(PFN_encodeTiled enc, CUtensorMap* map, void* base, int64_t cols, int64_t rows, int64_t count,
                    int64_t ld, uint32_t box_rows) {
    return encode_3d(enc, map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, base, cols, rows, count, ld, 64, box_rows,
                     CU_TENSOR_MAP_SWIZZLE_128B);
}

template <int CAP>
void fill_ptrs(PtrTable<CAP>& t, float* const* params, const void* const* grads, int n) {
    for (int i = 0; i < n; ++i) {
        t.param[i] = params[i];
        t.grad[i] = grads[i];
    }
}

template <int CAP>
cudaError_t run_elem(muon_s* h, float* const* params, const void* const* grads, bool apply, bool overlap,
                     cudaStream_t s) {
    ElemParams<CAP> ep;
    memset(&ep, 0, sizeof(ep));
    fill_ptrs<CAP>(ep.ptr, params, grads, (int)h->shapes.size());
    ep.subs = h->d_subs;
    ep.tiles = h->d_elem_tiles;
    ep.ntiles = h->n_elem_tiles;
    ep.hp = h->hp;
    ep.norm_part = h->norm_part;
    ep.nesterov = h->cfg.nesterov;
    ep.lerp_form = h->cfg.lerp_form;
    ep.status = h->status;
    if (apply) return launch_apply<CAP>(ep, overlap, s);
    return launch_momentum<CAP>(ep, h->cfg.grad_dtype == MUON_GRAD_F32, overlap, s);
}

cudaError_t run_elem_any(muon_s* h, float* const* params, const void* const* grads, bool apply, bool overlap,
                         cudaStream_t s) {
    const size_t n = h->shapes.size();
    if (n <= 64) return run_elem<64>(h, params, grads, apply, overlap, s);
    if (n <= 256) return run_elem<256>(h, params, grads, apply, overlap, s);
    return run_elem<1024>(h, params, grads, apply, overlap, s);
}

// What a group does in one Newton-Schulz iteration.  Standard form (the write-ups'
// order of operations): A = X X^T, P' = a I + b A + c A^2 (the first iteration keeps a
// out of P and adds a u in the update), X <- P' X.  Gram-pair groups run the first
// iteration in the standard form and then take the rest two at a time in Gram space:
// with A_k = X_k X_k^T and P'_k a polynomial in A_k, X_{k+1} = P'_k X_k gives
// A_{k+1} = P'_k A_k P'_k = (A_k P'_k) P'_k and X_{k+2} = (P'_{k+1} P'_k) X_k, so a pair
// of iterations forms one Gram matrix and one update instead of two of each, for three
// m x m products.  Two of them ride along with launches the other groups make anyway:
// T = A_k P'_k with the first half's updates (on the update kernel, the m x m tiles on or
// above the diagonal: T is symmetric, its computed asymmetry is at the level of P''s
// rounding, and it is read as its upper block triangle like A and P'), A_{k+1} = T P'_k
// with the second half's Gram matrices (symmetric tiles).  Q = P'_{k+1} P'_k has a launch
// of its own on the update kernel: it is symmetric only in exact arithmetic (the computed
// P' and P'' commute up to the error of A_{k+1}), and storing its upper triangle mirrored
// measurably raised the error of the output, where the full product keeps it at the
// standard form's level.  A single iteration left at the end runs in the standard form.
enum GroupOp { OP_NONE, OP_GRAM, OP_POLY, OP_POLY_B, OP_PLAIN_A, OP_PROD_Q, OP_UPD, OP_UPD_T, OP_UPD_Q };
enum Phase { PH_GRAM, PH_POLY, PH_PLAIN, PH_UPDATE, PH_COUNT };

GroupOp group_op(const Group& g, int it, int steps, int phase) {
    int kind = 0;  // 0: standard, 1: first of a Gram pair, 2: second of a pair
    if (g.gs && it > 0) {
        const int pos = (it - 1) % 2;
        kind = pos == 1 ? 2 : (it + 1 < steps ? 1 : 0);
    }
    switch (phase) {
        case PH_GRAM: return kind == 2 ? OP_PLAIN_A : OP_GRAM;
        case PH_POLY: return kind == 2 ? OP_POLY_B : OP_POLY;
        case PH_PLAIN: return kind == 2 ? OP_PROD_Q : OP_NONE;
        default: return kind == 1 ? OP_UPD_T : (kind == 2 ? OP_UPD_Q : OP_UPD);
    }
}

// The iterate buffer that holds the last output: the first iteration writes buffer 0
// and every later update flips it.
int final_buffer(const Group& g, int steps) {
    int cur = 0;
    for (int it = 1; it < steps; ++it) {
        const GroupOp op = group_op(g, it, steps, PH_UPDATE);
        if (op == OP_UPD || op == OP_UPD_Q) cur ^= 1;
    }
    return cur;
}

int launches_per_step(const muon_s* h) {
    // k_momentum, k_norm_scale, k_lane_stats, k_apply + the Newton-Schulz products
    // (+ k_schedule_advance while a schedule is installed)
    const int sched = h->schedule_on ? 1 : 0;
    const int colsum = h->n_colwork > 0 ? 1 : 0;  // k_col_sumsq for column lanes
    if (h->cfg.gemm_engine == MUON_GEMM_TCGEN05) return sched + colsum + 4 + (int)h->plan.size();
    const int per_iter = 3 * (int)h->groups.size();
    const int rowsq = h->cfg.normuon ? (int)h->groups.size() : 0;  // extra pass after the last update
    return sched + colsum + 4 + per_iter * h->cfg.ns_steps + rowsq;
}

cudaError_t mark(muon_s* h, int stage, cudaStream_t s) {
    if (!h->profiling) return cudaSuccess;
    if (h->n_recorded >= (int)h->events.size()) return cudaErrorInvalidValue;
    h->event_stage[h->n_recorded] = stage;
    return cudaEventRecord(h->events[h->n_recorded++], s);
}

}  // namespace

// ===================================================================== C ABI
extern "C" {

void muon_config_default(muon_config* cfg) {
    if (!cfg) return;
    memset(cfg, 0, sizeof(*cfg));
    cfg->lr = 0.02f;
    cfg->momentum = 0.95f;
    cfg->beta2 = 0.95f;
    cfg->weight_decay = 0.f;
    cfg->ns_steps = 5;
    cfg->nesterov = 1;
    cfg->lerp_form = 1;
    cfg->normuon = 1;
    cfg->norm_preserve = 1;
    cfg->grad_dtype = MUON_GRAD_BF16;
    cfg->gemm_engine = MUON_GEMM_TCGEN05;
    cfg->normuon_lanes = MUON_LANES_SHORT_SIDE;
    cfg->ns_form = MUON_NS_GRAM_PAIRS;
    cfg->launch_overlap = 1;
}

const char* muon_error_string(int code) {
    switch (code) {
        case MUON_OK: return "ok";
        case MUON_ERR_ARG: return "invalid argument";
        case MUON_ERR_ALIGN: return "pointer not 16-byte aligned";
        case MUON_ERR_SHAPE: return "unsupported or inconsistent shape";
        case MUON_ERR_CUDA: return "CUDA error";
        case MUON_ERR_TIMEOUT: return "device wait timed out";
        case MUON_ERR_DESTROYED: return "handle destroyed";
        case MUON_ERR_NOMEM: return "out of device memory";
        case MUON_ERR_UNSUPPORTED: return "device is not sm_103";
        case MUON_ERR_NONFINITE: return "a matrix's update direction was not finite; its step was skipped";
        default: return "unknown error";
    }
}

const char* muon_last_error(muon_handle h) {
    if (h == nullptr) return g_create_error.c_str();
    std::lock_guard<std::mutex> lk(g_handles_mu);
    if (g_handles.find(h) == g_handles.end()) return "unknown handle";
    return h->last_error.c_str();
}

int muon_create(const muon_shape* shapes, int32_t n_mats, const muon_config* cfg_in, int32_t device,
                muon_handle* out) {
    g_create_error.clear();
    if (out == nullptr) return fail(nullptr, MUON_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (shapes == nullptr || n_mats <= 0) return fail(nullptr, MUON_ERR_ARG, "need at least one shape");
    if (n_mats > MUON_MAX_MATRICES) return fail(nullptr, MUON_ERR_ARG, "too many matrices (max %d)", MUON_MAX_MATRICES);
    muon_config cfg;
    if (cfg_in)
        cfg = *cfg_in;
    else
        muon_config_default(&cfg);
    if (cfg.ns_steps < 1 || cfg.ns_steps > MUON_MAX_NS_STEPS)
        return fail(nullptr, MUON_ERR_ARG, "ns_steps must be in [1, %d]", MUON_MAX_NS_STEPS);
    if (cfg.grad_dtype != MUON_GRAD_BF16 && cfg.grad_dtype != MUON_GRAD_F32)
        return fail(nullptr, MUON_ERR_ARG, "bad grad_dtype");
    if (cfg.gemm_engine != MUON_GEMM_TCGEN05 && cfg.gemm_engine != MUON_GEMM_SIMT)
        return fail(nullptr, MUON_ERR_ARG, "bad gemm_engine");
    if (cfg.normuon_lanes != MUON_LANES_SHORT_SIDE && cfg.normuon_lanes != MUON_LANES_ROWS &&
        cfg.normuon_lanes != MUON_LANES_COLS)
        return fail(nullptr, MUON_ERR_ARG, "bad normuon_lanes");
    if (cfg.ns_form != MUON_NS_STANDARD && cfg.ns_form != MUON_NS_GRAM_PAIRS)
        return fail(nullptr, MUON_ERR_ARG, "bad ns_form");
    if (cfg.launch_overlap != 0 && cfg.launch_overlap != 1)
        return fail(nullptr, MUON_ERR_ARG, "launch_overlap must be 0 or 1");

    // ---- shapes -> split matrices (host-only validation first)
    struct Pending {
        int parent, q;
        int64_t rows, cols, ld, off, mom_off_in_parent, ld_mom;
    };
    std::vector<Pending> pend;
    std::vector<int64_t> mom_off(n_mats);
    int64_t mom_total = 0;
    for (int i = 0; i < n_mats; ++i) {
        const muon_shape& s = shapes[i];
        const int64_t ld = s.ld == 0 ? s.cols : s.ld;
        const int split = s.split <= 0 ? 1 : s.split;
        if (s.rows < 1 || s.cols < 1) return fail(nullptr, MUON_ERR_SHAPE, "shape %d: rows and cols must be >= 1", i);
        if (s.rows > (1 << 20) || s.cols > (1 << 20))
            return fail(nullptr, MUON_ERR_SHAPE, "shape %d: dimensions above 2^20 are not supported", i);
        if (ld < s.cols) return fail(nullptr, MUON_ERR_SHAPE, "shape %d: ld < cols", i);
        if (s.cols % split) return fail(nullptr, MUON_ERR_SHAPE, "shape %d: cols not divisible by split", i);
        if (s.flags != MUON_SPLIT_CONTIGUOUS && s.flags != MUON_SPLIT_COLUMNS)
            return fail(nullptr, MUON_ERR_ARG, "shape %d: bad flags", i);
        if (split > 1 && s.flags == MUON_SPLIT_CONTIGUOUS && ld != s.cols)
            return fail(nullptr, MUON_ERR_SHAPE, "shape %d: a contiguous split needs ld == cols", i);
        mom_off[i] = mom_total;
        mom_total += round_up(s.rows * s.cols, 64);
        const int64_t cs = s.cols / split;
        for (int q = 0; q < split; ++q) {
            Pending p;
            p.parent = i;
            p.q = q;
            p.rows = s.rows;
            p.cols = cs;
            if (split == 1) {
                p.ld = ld;
                p.off = 0;
                p.mom_off_in_parent = 0;
                p.ld_mom = s.cols;
            } else if (s.flags == MUON_SPLIT_CONTIGUOUS) {
                p.ld = cs;
                p.off = (int64_t)q * s.rows * cs;
                p.mom_off_in_parent = p.off;
                p.ld_mom = cs;
            } else {
                p.ld = ld;
                p.off = (int64_t)q * cs;
                p.mom_off_in_parent = (int64_t)q * cs;
                p.ld_mom = s.cols;
            }
            pend.push_back(p);
        }
    }

    // ---- device checks
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || ndev == 0)
        return fail(nullptr, MUON_ERR_CUDA, "no CUDA device");
    if (device < 0 || device >= ndev) return fail(nullptr, MUON_ERR_ARG, "bad device %d", device);
    if (cudaSetDevice(device) != cudaSuccess) return fail(nullptr, MUON_ERR_CUDA, "cudaSetDevice failed");
    cudaDeviceProp prop;
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
        return fail(nullptr, MUON_ERR_CUDA, "cudaGetDeviceProperties failed");
    if (!(prop.major == 10 && prop.minor == 3))
        return fail(nullptr, MUON_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                    device, prop.major, prop.minor);
    PFN_encodeTiled enc = get_encode_fn();
    if (!enc) return fail(nullptr, MUON_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");

    muon_s* h = new muon_s();
    h->device = device;
    h->num_sms = prop.multiProcessorCount;
    h->cfg = cfg;
    h->cfg.lr_mul = h->cfg.wd_mul = h->cfg.ns_coeffs = nullptr;
    h->shapes.assign(shapes, shapes + n_mats);
    h->mom_off = mom_off;
    for (int i = 0; i < n_mats; ++i) {
        h->lr_mul.push_back(cfg.lr_mul ? cfg.lr_mul[i] : 1.f);
        h->wd_mul.push_back(cfg.wd_mul ? cfg.wd_mul[i] : 1.f);
    }
    for (int it = 0; it < cfg.ns_steps; ++it)
        for (int k = 0; k < 3; ++k) h->coeffs.push_back(cfg.ns_coeffs ? cfg.ns_coeffs[3 * it + k] : kDefaultCoeffs[k]);

    // ---- groups by wide shape, in order of first appearance
    std::map<std::pair<int, int>, int> gid;
    std::vector<int> sub_group(pend.size());
    for (size_t k = 0; k < pend.size(); ++k) {
        const int m = (int)std::min(pend[k].rows, pend[k].cols), n = (int)std::max(pend[k].rows, pend[k].cols);
        auto key = std::make_pair(m, n);
        auto it = gid.find(key);
        if (it == gid.end()) {
            Group g;
            g.m = m;
            g.n = n;
            g.ldx = (int)round_up(n, 8);
            g.lda = (int)round_up(m, 8);
            g.ntile_n = (n + kBNUpd - 1) / kBNUpd;
            it = gid.emplace(key, (int)h->groups.size()).first;
            h->groups.push_back(g);
        }
        sub_group[k] = it->second;
    }
    // wide groups that tile by 256 take their iterations in Gram pairs (n >= 2m: a pair then
    // saves more than its three m x m products cost)
    for (Group& g : h->groups)
        g.gs = cfg.ns_form == MUON_NS_GRAM_PAIRS && cfg.gemm_engine == MUON_GEMM_TCGEN05 && cfg.ns_steps >= 3 &&
               g.m % 256 == 0 && g.n % 256 == 0 && g.n >= 2 * g.m;
    std::vector<size_t> order(pend.size());
    for (size_t k = 0; k < order.size(); ++k) order[k] = k;
    std::stable_sort(order.begin(), order.end(), [&](size_t a, size_t b) { return sub_group[a] < sub_group[b]; });

    // ---- arena layout
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += (bytes + 255) / 256 * 256;
        return o;
    };
    const int nsubs = (int)pend.size();
    const size_t o_hp = take(sizeof(float) * HP_COUNT);
    const size_t o_status = take(sizeof(int));
    const size_t o_sched = take(sizeof(DevSchedule));
    const size_t o_norm_scale = take(sizeof(float) * nsubs);
    const size_t o_iter_scale = take(sizeof(float) * nsubs);
    const size_t o_skip = take(sizeof(int) * nsubs);
    // NorMuon lanes of each sub: the rows of its wide orientation, or its columns
    // (the caller's rows of a tall matrix under MUON_LANES_ROWS, the caller's
    // columns of a wide or square one under MUON_LANES_COLS)
    std::vector<int> sub_lane_cols(nsubs, 0);
    for (int sidx = 0; sidx < nsubs; ++sidx) {
        const Pending& pd = pend[order[sidx]];
        const bool tr = pd.rows > pd.cols;
        sub_lane_cols[sidx] = cfg.normuon && ((cfg.normuon_lanes == MUON_LANES_ROWS && tr) ||
                                              (cfg.normuon_lanes == MUON_LANES_COLS && !tr));
    }
    // elementwise tiles
    std::vector<int4> elem_tiles;
    std::vector<int32_t> k1_tile0(nsubs), k1_ntiles(nsubs);
    for (int sidx = 0; sidx < nsubs; ++sidx) {
        const Pending& pd = pend[order[sidx]];
        k1_tile0[sidx] = (int32_t)elem_tiles.size();
        for (int64_t r0 = 0; r0 < pd.rows; r0 += kTile)
            for (int64_t c0 = 0; c0 < pd.cols; c0 += kTile) elem_tiles.push_back(make_int4(sidx, (int)r0, (int)c0, 0));
        k1_ntiles[sidx] = (int32_t)elem_tiles.size() - k1_tile0[sidx];
    }
    if (elem_tiles.size() > (size_t)0x7fffffff / 2) {
        delete h;
        return fail(nullptr, MUON_ERR_SHAPE, "too many elementwise tiles");
    }
    h->n_elem_tiles = (int32_t)elem_tiles.size();
    const size_t o_norm_part = take(sizeof(float) * elem_tiles.size());
    const size_t o_mom = take(sizeof(float) * (size_t)mom_total);
    std::vector<size_t> go_ulo, go_u16, go_x16[2], go_a16, go_p16, go_pb16, go_t16, go_rowsq, go_v, go_lane, go_colsq;
    for (auto& g : h->groups) {
        g.count = 0;
        g.lane_stride = g.m;
    }
    std::vector<int> group_cols(h->groups.size(), 0);  // some matrix of the group has column lanes
    for (int sidx = 0; sidx < nsubs; ++sidx) {
        Group& g = h->groups[sub_group[order[sidx]]];
        g.count++;
        if (sub_lane_cols[sidx]) {
            g.lane_stride = g.n;
            group_cols[sub_group[order[sidx]]] = 1;
        }
    }
    {
        int s0 = 0;
        for (auto& g : h->groups) {
            g.sub0 = s0;
            s0 += g.count;
        }
    }
    for (auto& g : h->groups) {
        const size_t xe = (size_t)g.count * g.m * g.ldx, ae = (size_t)g.count * g.m * g.lda;
        go_ulo.push_back(take(xe * 2));
        go_u16.push_back(take(xe * 2));
        for (int b = 0; b < 2; ++b) {
            go_x16[b].push_back(take(xe * 2));
        }
        go_a16.push_back(take(ae * 2));
        go_p16.push_back(take(ae * 2));
        go_pb16.push_back(g.gs ? take(ae * 2) : 0);
        go_t16.push_back(g.gs ? take(ae * 2) : 0);
        go_rowsq.push_back(take((size_t)g.count * g.m * g.ntile_n * 2 * 4));
        go_v.push_back(take((size_t)g.count * g.lane_stride * 4));
        go_lane.push_back(take((size_t)g.count * g.lane_stride * 4));
    }
    for (size_t gi = 0; gi < h->groups.size(); ++gi) {
        const Group& g = h->groups[gi];
        go_colsq.push_back(group_cols[gi] ? take((size_t)g.count * ((g.m + kTile - 1) / kTile) * g.n * 4) : 0);
    }
    // k_col_sumsq work list: one block per (sub, 64-row slab) of the subs with column lanes
    std::vector<int2> colwork;
    std::vector<int32_t> colwork0(nsubs, 0);
    for (int sidx = 0; sidx < nsubs; ++sidx) {
        colwork0[sidx] = (int32_t)colwork.size();
        if (!sub_lane_cols[sidx]) continue;
        const Group& g = h->groups[sub_group[order[sidx]]];
        for (int slab = 0; slab < (g.m + kTile - 1) / kTile; ++slab) colwork.push_back(make_int2(sidx, slab));
    }
    h->n_colwork = (int32_t)colwork.size();
    const size_t o_colwork = take(sizeof(int2) * std::max<size_t>(colwork.size(), 1));
    const size_t o_subs = take(sizeof(SubDesc) * nsubs);
    const size_t o_etiles = take(sizeof(int4) * elem_tiles.size());

    // GEMM tile lists, per chunk of groups.  Groups whose m and n are multiples of 256 run
    // the Gram and the update on SM pairs; they are chunked apart from the others so that
    // one group of another shape does not take its chunk-mates off the pair kernels.
    std::vector<int4> gemm_tiles;
    std::vector<std::vector<int>> chunk_groups;
    for (int fit = 1; fit >= 0; --fit) {
        std::vector<int> gs;
        for (int gi = 0; gi < (int)h->groups.size(); ++gi) {
            const Group& g = h->groups[gi];
            if ((g.m % 256 == 0 && g.n % 256 == 0) == (fit == 1)) gs.push_back(gi);
        }
        for (size_t i = 0; i < gs.size(); i += kMaxGroupsPerLaunch)
            chunk_groups.emplace_back(gs.begin() + i, gs.begin() + std::min(gs.size(), i + kMaxGroupsPerLaunch));
    }
    for (const std::vector<int>& cg : chunk_groups) {
        Chunk ch;
        ch.ng = (int32_t)cg.size();
        for (int sl = 0; sl < ch.ng; ++sl) ch.gi[sl] = cg[(size_t)sl];
        struct T {
            int4 t;
            int64_t cost;
        };
        auto emit = [&](std::vector<T>& v, int32_t& o, int32_t& n) {
            std::stable_sort(v.begin(), v.end(), [](const T& a, const T& b) { return a.cost > b.cost; });
            o = (int32_t)gemm_tiles.size();
            for (auto& x : v) gemm_tiles.push_back(x.t);
            n = (int32_t)v.size();
            for (size_t i = 0; i < v.size();) {  // the reversed copy, cost classes kept in order
                size_t j = i;
                while (j < v.size() && v[j].cost == v[i].cost) ++j;
                for (size_t k = j; k > i; --k) gemm_tiles.push_back(v[k - 1].t);
                i = j;
            }
        };
        std::vector<T> gram, poly, upd;
        for (int sl = 0; sl < ch.ng; ++sl) {
            const Group& g = h->groups[ch.gi[sl]];
            const int tm = (g.m + kBM - 1) / kBM;
            const int tn = (g.n + kBNUpd - 1) / kBNUpd;
            const int ts = (g.m + kBNSym - 1) / kBNSym;  // 256-column blocks of A / P
            for (int idx = 0; idx < g.count; ++idx) {
                // symmetric 128 x 256 tiles that reach the diagonal or lie above it
                for (int ti = 0; ti < tm; ++ti)
                    for (int tj = 0; tj < ts; ++tj) {
                        if ((tj * kBNSym + kBNSym - 1) / kBM < ti) continue;
                        gram.push_back({make_int4(sl, idx, ti, tj), (int64_t)g.n});
                        poly.push_back({make_int4(sl, idx, ti, tj), (int64_t)g.m});
                    }
                for (int ti = 0; ti < tm; ++ti)
                    for (int tj = 0; tj < tn; ++tj) upd.push_back({make_int4(sl, idx, ti, tj), (int64_t)g.m});
            }
        }
        emit(gram, ch.gram_off, ch.gram_n);
        emit(poly, ch.poly_off, ch.poly_n);
        emit(upd, ch.upd_off, ch.upd_n);
        // the Gram and the updates run on SM pairs when every group of the chunk tiles
        // exactly into 256 x 256 pair tiles
        bool pair_fit = true;
        for (int sl = 0; sl < ch.ng; ++sl) {
            const Group& g = h->groups[ch.gi[sl]];
            pair_fit = pair_fit && g.m % 256 == 0 && g.n % 256 == 0;
        }
        if (pair_fit) {
            // which: 0 every group, 1 the standard-form groups, 2 the Gram-pair groups
            auto member = [&](int sl, int which) {
                const bool gs = h->groups[ch.gi[sl]].gs != 0;
                return which == 0 || (which == 1 && !gs) || (which == 2 && gs);
            };
            // square: the Gram-pair groups' tiles cover their m x m products; upper: only the
            // blocks on or above the diagonal of those (T = A P', symmetric, is stored as its
            // upper block triangle; Q is a full product)
            auto upd_list = [&](int which, bool square, bool upper, int32_t& o, int32_t& n) {
                std::vector<T> pr;
                for (int sl = 0; sl < ch.ng; ++sl) {
                    if (!member(sl, which)) continue;
                    const Group& g = h->groups[ch.gi[sl]];
                    const int cols = square && g.gs ? g.m : g.n;
                    for (int idx = 0; idx < g.count; ++idx)
                        for (int ti = 0; ti < g.m / 256; ++ti)
                            for (int tj = (upper && square && g.gs) ? ti : 0; tj < cols / 256; ++tj)
                                pr.push_back({make_int4(sl, idx, ti, tj), (int64_t)g.m});
                }
                emit(pr, o, n);
            };
            auto sym_list = [&](int which, int32_t& o, int32_t& n) {
                std::vector<T> sg;
                for (int sl = 0; sl < ch.ng; ++sl) {
                    if (!member(sl, which)) continue;
                    const Group& g = h->groups[ch.gi[sl]];
                    for (int idx = 0; idx < g.count; ++idx)
                        for (int ti = 0; ti < g.m / 256; ++ti)
                            for (int tj = ti; tj < g.m / 256; ++tj)
                                sg.push_back({make_int4(sl, idx, ti, tj), (int64_t)g.n});
                }
                emit(sg, o, n);
            };
            upd_list(0, false, false, ch.pair_off, ch.pair_n);
            sym_list(0, ch.spg_off, ch.spg_n);
            bool any_gs = false;
            for (int sl = 0; sl < ch.ng; ++sl) any_gs = any_gs || member(sl, 2);
            if (any_gs) {
                upd_list(0, true, true, ch.pair_t_off, ch.pair_t_n);
                upd_list(2, true, false, ch.pair_q_off, ch.pair_q_n);
                // Q's launch and the update launch after it hold tiles of one size when every
                // group has the same m; then move s standard update tiles, the fewest that
                // minimise the two launches' waves over the SM pairs
                std::vector<T> std_t, gs_t, q_t;
                bool one_m = true;
                for (int sl = 0; sl < ch.ng; ++sl) {
                    const Group& g = h->groups[ch.gi[sl]];
                    one_m = one_m && g.m == h->groups[ch.gi[0]].m;
                    for (int idx = 0; idx < g.count; ++idx)
                        for (int ti = 0; ti < g.m / 256; ++ti) {
                            for (int tj = 0; tj < g.n / 256; ++tj)
                                (g.gs ? gs_t : std_t).push_back({make_int4(sl, idx, ti, tj), (int64_t)g.m});
                            if (g.gs)
                                for (int tj = 0; tj < g.m / 256; ++tj)
                                    q_t.push_back({make_int4(sl, idx, ti, tj), (int64_t)g.m});
                        }
                }
                const int64_t P = std::max(1, h->num_sms / 2);
                const int64_t nq = (int64_t)q_t.size(), nu = (int64_t)(std_t.size() + gs_t.size());
                auto waves = [&](int64_t x) { return (x + P - 1) / P; };
                int64_t best = 0;
                if (one_m)
                    for (int64_t sft = 1; sft <= std::min<int64_t>((int64_t)std_t.size(), P - 1); ++sft)
                        if (waves(nq + sft) + waves(nu - sft) < waves(nq + best) + waves(nu - best)) best = sft;
                if (best > 0) {
                    ch.q_fill_n = (int32_t)best;
                    std::vector<T> qx(q_t), ux(gs_t);
                    for (size_t i = 0; i < std_t.size(); ++i) {
                        if ((int64_t)i < best) {
                            qx.push_back(std_t[i]);
                            ch.q_fill[std_t[i].t.x]++;
                        } else {
                            ux.push_back(std_t[i]);
                        }
                    }
                    emit(qx, ch.pair_qx_off, ch.pair_qx_n);
                    emit(ux, ch.pair_ux_off, ch.pair_ux_n);
                }
            }
        }
        h->chunks.push_back(ch);
    }
    const size_t o_gtiles = take(sizeof(int4) * std::max<size_t>(gemm_tiles.size(), 1));

    h->arena_bytes = off;
    if (cudaMalloc(&h->arena, off) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return fail(nullptr, MUON_ERR_NOMEM, "cudaMalloc of %zu bytes failed", off);
    }
    char* base = static_cast<char*>(h->arena);
    if (cudaMemset(h->arena, 0, off) != cudaSuccess) {
        cudaFree(h->arena);
        delete h;
        return fail(nullptr, MUON_ERR_CUDA, "cudaMemset failed");
    }
    h->hp = reinterpret_cast<float*>(base + o_hp);
    h->status = reinterpret_cast<int*>(base + o_status);
    h->sched = reinterpret_cast<DevSchedule*>(base + o_sched);
    h->norm_scale = reinterpret_cast<float*>(base + o_norm_scale);
    h->iter_scale = reinterpret_cast<float*>(base + o_iter_scale);
    h->skip = reinterpret_cast<int*>(base + o_skip);
    h->d_colwork = reinterpret_cast<int2*>(base + o_colwork);
    h->norm_part = reinterpret_cast<float*>(base + o_norm_part);
    h->momentum = reinterpret_cast<float*>(base + o_mom);
    h->d_subs = reinterpret_cast<SubDesc*>(base + o_subs);
    h->d_elem_tiles = reinterpret_cast<int4*>(base + o_etiles);
    h->d_gemm_tiles = reinterpret_cast<int4*>(base + o_gtiles);
    for (size_t gi = 0; gi < h->groups.size(); ++gi) {
        Group& g = h->groups[gi];
        g.ulo16 = reinterpret_cast<uint16_t*>(base + go_ulo[gi]);
        g.u16 = reinterpret_cast<uint16_t*>(base + go_u16[gi]);
        for (int b = 0; b < 2; ++b) {
            g.x16[b] = reinterpret_cast<uint16_t*>(base + go_x16[b][gi]);
        }
        g.a16 = reinterpret_cast<uint16_t*>(base + go_a16[gi]);
        g.p16 = reinterpret_cast<uint16_t*>(base + go_p16[gi]);
        g.pb16 = g.gs ? reinterpret_cast<uint16_t*>(base + go_pb16[gi]) : nullptr;
        g.t16 = g.gs ? reinterpret_cast<uint16_t*>(base + go_t16[gi]) : nullptr;
        g.final_buf = final_buffer(g, cfg.ns_steps);
        g.rowsq = reinterpret_cast<float*>(base + go_rowsq[gi]);
        g.v = reinterpret_cast<float*>(base + go_v[gi]);
        g.lane = reinterpret_cast<float*>(base + go_lane[gi]);
        g.colsq = group_cols[gi] ? reinterpret_cast<float*>(base + go_colsq[gi]) : nullptr;
        bool ok = encode_bf16_3d(enc, &g.map_u_k, g.u16, g.n, g.m, g.count, g.ldx, kBM) &&
                  encode_bf16_3d(enc, &g.map_u_mn, g.u16, g.n, g.m, g.count, g.ldx, 64) &&
                  encode_bf16_3d(enc, &g.map_a_k, g.a16, g.m, g.m, g.count, g.lda, kBM) &&
                  encode_bf16_3d(enc, &g.map_p_k, g.p16, g.m, g.m, g.count, g.lda, kBM) &&
                  encode_bf16_3d(enc, &g.map_u_k256, g.u16, g.n, g.m, g.count, g.ldx, 2 * kBM) &&
                  encode_bf16_3d(enc, &g.map_a_k256, g.a16, g.m, g.m, g.count, g.lda, 2 * kBM) &&
                  encode_bf16_3d(enc, &g.map_a_mn, g.a16, g.m, g.m, g.count, g.lda, 64);
        for (int b = 0; b < 2 && ok; ++b)
            ok = encode_bf16_3d(enc, &g.map_x_k[b], g.x16[b], g.n, g.m, g.count, g.ldx, kBM) &&
                 encode_bf16_3d(enc, &g.map_x_k256[b], g.x16[b], g.n, g.m, g.count, g.ldx, 2 * kBM) &&
                 encode_bf16_3d(enc, &g.map_x_mn[b], g.x16[b], g.n, g.m, g.count, g.ldx, 64) &&
                 encode_bf16_3d(enc, &g.map_x_mn128[b], g.x16[b], g.n, g.m, g.count, g.ldx, 128) &&
                 encode_3d(enc, &g.map_x_o32[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.x16[b], g.n, g.m, g.count,
                           g.ldx, 32, kBM, CU_TENSOR_MAP_SWIZZLE_64B) &&
                 encode_3d(enc, &g.map_x_w32[b], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.x16[b], g.n, g.m, g.count,
                           g.ldx, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
        ok = ok &&
             encode_3d(enc, &g.map_a_w32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.a16, g.m, g.m, g.count, g.lda, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_3d(enc, &g.map_p_w32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.p16, g.m, g.m, g.count, g.lda, 32, 32,
                       CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_3d(enc, &g.map_u_hi_w32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.u16, g.n, g.m, g.count, g.ldx, 32,
                       32, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_3d(enc, &g.map_u_lo_w32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.ulo16, g.n, g.m, g.count, g.ldx, 32,
                       32, CU_TENSOR_MAP_SWIZZLE_64B);
        ok = ok &&
             encode_3d(enc, &g.map_u_hi, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.u16, g.n, g.m, g.count, g.ldx, 32, kBM,
                       CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_3d(enc, &g.map_u_lo, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.ulo16, g.n, g.m, g.count, g.ldx, 32,
                       kBM, CU_TENSOR_MAP_SWIZZLE_64B) &&
             encode_bf16_3d(enc, &g.map_a_mir, g.a16, g.m, g.m, g.count, g.lda, 64) &&
             encode_bf16_3d(enc, &g.map_p_mir, g.p16, g.m, g.m, g.count, g.lda, 64) &&
             encode_bf16_3d(enc, &g.map_p_mn, g.p16, g.m, g.m, g.count, g.lda, 64) &&
             encode_bf16_3d(enc, &g.map_p_mn128, g.p16, g.m, g.m, g.count, g.lda, 128);
        if (ok && g.gs)
            ok = encode_bf16_3d(enc, &g.map_a_mn128, g.a16, g.m, g.m, g.count, g.lda, 128) &&
                 encode_bf16_3d(enc, &g.map_t_mn, g.t16, g.m, g.m, g.count, g.lda, 64) &&
                 encode_bf16_3d(enc, &g.map_pb_mn128, g.pb16, g.m, g.m, g.count, g.lda, 128) &&
                 encode_bf16_3d(enc, &g.map_pb_k, g.pb16, g.m, g.m, g.count, g.lda, kBM) &&
                 encode_bf16_3d(enc, &g.map_t_k, g.t16, g.m, g.m, g.count, g.lda, kBM) &&
                 encode_3d(enc, &g.map_pb_w32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.pb16, g.m, g.m, g.count, g.lda,
                           32, 32, CU_TENSOR_MAP_SWIZZLE_64B) &&
                 encode_3d(enc, &g.map_t_w32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, g.t16, g.m, g.m, g.count, g.lda,
                           32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
        if (!ok) {
            cudaFree(h->arena);
            delete h;
            return fail(nullptr, MUON_ERR_CUDA, "cuTensorMapEncodeTiled rejected a descriptor");
        }
    }

    // ---- sub descriptors (group order)
    std::vector<int> idx_in_group(h->groups.size(), 0);
    for (int sidx = 0; sidx < nsubs; ++sidx) {
        const Pending& pd = pend[order[sidx]];
        Group& g = h->groups[sub_group[order[sidx]]];
        const int gi = idx_in_group[sub_group[order[sidx]]]++;
        SubDesc d;
        memset(&d, 0, sizeof(d));
        d.grad_off = pd.off;
        d.ld = pd.ld;
        d.mom = h->momentum + h->mom_off[pd.parent] + pd.mom_off_in_parent;
        d.ld_mom = pd.ld_mom;
        d.rows = (int32_t)pd.rows;
        d.cols = (int32_t)pd.cols;
        d.parent = pd.parent;
        d.transposed = pd.rows > pd.cols ? 1 : 0;
        d.vec = (pd.cols % 8 == 0 && pd.ld % 8 == 0 && pd.off % 8 == 0 && pd.ld_mom % 8 == 0 &&
                 (h->mom_off[pd.parent] + pd.mom_off_in_parent) % 8 == 0)
                    ? 1
                    : 0;
        d.m = g.m;
        d.n = g.n;
        d.ldx = g.ldx;
        d.ntile_n = g.ntile_n;
        d.k1_tile0 = k1_tile0[sidx];
        d.k1_ntiles = k1_ntiles[sidx];
        d.lr_mul = h->lr_mul[pd.parent];
        d.wd_mul = h->wd_mul[pd.parent];
        d.shape_scale = (float)std::sqrt(std::max(1.0, (double)pd.rows / (double)pd.cols));
        const int64_t xo = (int64_t)gi * g.m * g.ldx;
        d.u16 = g.u16 + xo;
        d.ulo16 = g.ulo16 + xo;
        d.o16 = g.x16[g.final_buf] + xo;
        d.rowsq = g.rowsq + (int64_t)gi * g.m * g.ntile_n * 2;
        d.v = g.v + (int64_t)gi * g.lane_stride;
        d.lane = g.lane + (int64_t)gi * g.lane_stride;
        d.lane_cols = sub_lane_cols[sidx];
        d.colsq_tile0 = colwork0[sidx];
        d.colsq = g.colsq ? g.colsq + (int64_t)gi * ((g.m + kTile - 1) / kTile) * g.n : nullptr;
        d.skip = h->skip + sidx;
        h->subs.push_back(d);
        h->sub_parent_q.push_back(pd.q);
    }

    // ---- upload descriptors and tiles, default hyper-parameters
    bool ok = cudaMemcpy(h->d_subs, h->subs.data(), sizeof(SubDesc) * nsubs, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(h->d_elem_tiles, elem_tiles.data(), sizeof(int4) * elem_tiles.size(),
                         cudaMemcpyHostToDevice) == cudaSuccess &&
              (colwork.empty() || cudaMemcpy(h->d_colwork, colwork.data(), sizeof(int2) * colwork.size(),
                                             cudaMemcpyHostToDevice) == cudaSuccess) &&
              (gemm_tiles.empty() || cudaMemcpy(h->d_gemm_tiles, gemm_tiles.data(), sizeof(int4) * gemm_tiles.size(),
                                                cudaMemcpyHostToDevice) == cudaSuccess);
    float hpv[HP_COUNT] = {cfg.lr, cfg.momentum, cfg.beta2, cfg.weight_decay};
    ok = ok && cudaMemcpy(h->hp, hpv, sizeof(hpv), cudaMemcpyHostToDevice) == cudaSuccess;
    ok = ok && ns_gemm_tc_configure() == cudaSuccess && ns_update_pair_configure() == cudaSuccess &&
         ns_gram_pair_configure() == cudaSuccess;
    if (!ok) {
        cudaFree(h->arena);
        delete h;
        return fail(nullptr, MUON_ERR_CUDA, "upload / kernel configuration failed");
    }

    // ---- the Newton-Schulz launch plan: per iteration the Gram, polynomial, plain-product
    // and update phases, each one launch per chunk whose groups have work in that phase
    {
        const int steps = cfg.ns_steps;
        std::vector<int> cur(h->groups.size(), 0);      // iterate buffer holding the current X (after the first iteration)
        std::vector<int> nlaunch(h->chunks.size(), 0);  // per chunk: launches so far (alternating tile order)
        // frac: the share of the group's tiles this launch computes
        auto add_work = [&](int stage, const Group& g, GroupOp op, bool first, bool pairs, double frac) {
            const double m = g.m, n = g.n;
            // a symmetric result: the SM-pair kernels write its upper block triangle (256 x 256
            // blocks), the one-SM kernels the whole matrix
            const double nb = std::ceil(m / 256.0);
            const double sym_out = pairs ? 2 * 256.0 * 256.0 * nb * (nb + 1) / 2 : 2 * m * m;
            double fl = 0, by = 0;
            switch (op) {
                case OP_GRAM: fl = m * (m + 1) * n; by = 2 * m * n + sym_out; break;
                case OP_POLY:
                case OP_POLY_B: fl = m * m * (m + 1); by = 2 * m * m + sym_out; break;
                case OP_PLAIN_A: fl = m * m * (m + 1); by = 4 * m * m + sym_out; break;
                // on the update kernel: Q as a full product, T (symmetric) as its upper block triangle
                case OP_UPD_T:
                    fl = pairs ? 2 * m * m * m * (nb + 1) / (2 * nb) : 2 * m * m * m;
                    by = 4 * m * m + sym_out;
                    break;
                case OP_PROD_Q: fl = 2 * m * m * m; by = 6 * m * m; break;
                case OP_UPD: fl = 2 * m * m * n; by = 2 * m * m + (first ? 6 : 4) * m * n; break;
                case OP_UPD_Q: fl = 2 * m * m * n; by = 2 * m * m + 4 * m * n; break;
                default: break;
            }
            h->work_flops[stage] += (int64_t)(fl * g.count * frac);
            h->work_bytes[stage] += (int64_t)(by * g.count * frac);
        };
        for (int it = 0; it < steps; ++it) {
            const bool first = it == 0, last = it == steps - 1;
            for (int ph = 0; ph < PH_COUNT; ++ph) {
                for (int c = 0; c < (int)h->chunks.size(); ++c) {
                    const Chunk& ch = h->chunks[c];
                    const bool pairs = ch.spg_n > 0;  // the chunk tiles by 256: SM-pair kernels
                    GemmParams gp;
                    memset(&gp, 0, sizeof(gp));
                    gp.ngroups = ch.ng;
                    gp.norm_scale = h->norm_scale;
                    gp.iter_scale = h->iter_scale;
                    gp.ca = h->coeffs[3 * it + 0];
                    gp.cb = h->coeffs[3 * it + 1];
                    gp.cc = h->coeffs[3 * it + 2];
                    gp.first = first;
                    gp.last = last;
                    gp.f16 = it > 0;
                    // this iteration's launch of Q = P'' P' (a Gram-pair chunk's second iteration of
                    // a pair); it may carry standard-form update tiles (Chunk.q_fill)
                    bool q_launch = false;
                    for (int sl = 0; sl < ch.ng; ++sl)
                        q_launch = q_launch || group_op(h->groups[ch.gi[sl]], it, steps, PH_PLAIN) == OP_PROD_Q;
                    const bool q_fill = pairs && q_launch && ch.q_fill_n > 0;
                    gp.want_rowsq = (ph == PH_UPDATE || (ph == PH_PLAIN && q_fill)) && last && cfg.normuon;
                    gp.status = h->status;
                    gp.pair = pairs ? 1 : 0;
                    int n_in = 0, n_in_gs = 0, n_gs = 0;
                    GroupOp ops[kMaxGroupsPerLaunch];
                    for (int sl = 0; sl < ch.ng; ++sl) {
                        const Group& g = h->groups[ch.gi[sl]];
                        const int cb = cur[ch.gi[sl]], nb = first ? 0 : cur[ch.gi[sl]] ^ 1;
                        GemmGroup& G = gp.grp[sl];
                        G.m = g.m;
                        G.n = g.n;
                        G.ldx = g.ldx;
                        G.lda = g.lda;
                        G.ntile_n = g.ntile_n;
                        G.sub0 = g.sub0;
                        G.x_stride = (int64_t)g.m * g.ldx;
                        G.a_stride = (int64_t)g.m * g.lda;
                        G.a16 = g.a16;
                        G.rowsq = g.rowsq;
                        const uint16_t* xin16 = first ? g.u16 : g.x16[cb];
                        GroupOp op = group_op(g, it, steps, ph);
                        if (ph == PH_PLAIN && q_fill && op == OP_NONE && ch.q_fill[sl] > 0 &&
                            group_op(g, it, steps, PH_UPDATE) == OP_UPD)
                            op = OP_UPD;  // some of its update tiles ride along with Q
                        ops[sl] = op;
                        n_gs += g.gs ? 1 : 0;
                        // every slot carries valid descriptors (the kernels prefetch all of them);
                        // the group's own operation below replaces them
                        gp.map_a[sl] = g.map_a_k;
                        gp.map_b[sl] = g.map_a_mn;
                        gp.map_ein[sl] = g.map_a_w32;
                        gp.map_ein2[sl] = g.map_a_w32;
                        gp.map_out[sl] = g.map_a_w32;
                        gp.map_out2[sl] = g.map_a_mir;
                        gp.map_al[sl] = g.map_a_mn;
                        gp.map_bk[sl] = g.map_a_k;
                        if (op == OP_NONE) continue;
                        ++n_in;
                        n_in_gs += g.gs ? 1 : 0;
                        switch (op) {
                            case OP_GRAM:
                                gp.map_a[sl] = first ? g.map_u_k : g.map_x_k[cb];
                                gp.map_b[sl] = first ? g.map_u_k256 : g.map_x_k256[cb];
                                gp.map_out[sl] = pairs ? g.map_a_w32 : g.map_a_k;
                                gp.map_out2[sl] = g.map_a_mir;
                                G.out16 = g.a16;
                                G.opl16 = xin16;
                                G.opr16 = xin16;
                                break;
                            case OP_POLY:
                            case OP_POLY_B:  // the second polynomial of a Gram pair keeps the first one's P
                                gp.map_a[sl] = g.map_a_k;
                                gp.map_b[sl] = pairs ? g.map_a_mn : g.map_a_k256;
                                gp.map_ein[sl] = pairs ? g.map_a_w32 : g.map_a_k;
                                gp.map_out[sl] = op == OP_POLY_B ? g.map_pb_w32 : (pairs ? g.map_p_w32 : g.map_p_k);
                                gp.map_out2[sl] = g.map_p_mir;
                                G.out16 = op == OP_POLY_B ? g.pb16 : g.p16;
                                G.opl16 = g.a16;
                                G.opr16 = g.a16;
                                // on SM pairs A is stored as its upper block triangle: A's rows below
                                // the diagonal come from its columns, its columns from its rows
                                G.sym_l = G.sym_r = pairs ? 1 : 0;
                                gp.map_al[sl] = g.map_a_mn;
                                gp.map_bk[sl] = g.map_a_k;
                                break;
                            case OP_PLAIN_A:  // A <- T P', in the Gram launch
                                gp.map_a[sl] = g.map_t_k;
                                gp.map_b[sl] = g.map_p_mn;
                                gp.map_out[sl] = g.map_a_w32;
                                G.b_mn = 1;
                                G.out16 = g.a16;
                                G.opl16 = g.t16;
                                G.opr16 = g.p16;
                                // T and P' as their upper block triangles
                                G.sym_l = G.sym_r = 1;
                                gp.map_al[sl] = g.map_t_mn;
                                gp.map_bk[sl] = g.map_p_k;
                                break;
                            case OP_PROD_Q:  // Q = P'' P', full m x m tiles on the update kernel (into T's buffer)
                                gp.map_a[sl] = g.map_pb_k;
                                gp.map_b[sl] = g.map_p_mn128;
                                gp.map_out[sl] = g.map_t_w32;
                                G.x16_out = g.t16;
                                G.opl16 = g.pb16;
                                G.opr16 = g.p16;
                                G.rowsq = nullptr;  // Q is not an output: no row sums
                                G.sym_l = G.sym_r = 1;  // P'' and P' as their upper block triangles
                                gp.map_al[sl] = g.map_pb_mn128;
                                gp.map_bk[sl] = g.map_p_k;
                                break;
                            case OP_UPD:
                                gp.map_a[sl] = g.map_p_k;
                                // the folded update on SM pairs takes 128-deep k-blocks (16 KB boxes of X)
                                gp.map_b[sl] = first ? g.map_u_mn : (pairs ? g.map_x_mn128[cb] : g.map_x_mn[cb]);
                                // first update: u hi | lo in 32-column boxes, X1 out in 32-column boxes;
                                // later updates (a on the diagonal of P): no input, X' out in 64-column boxes
                                gp.map_ein[sl] = pairs ? g.map_u_hi_w32 : g.map_u_hi;
                                gp.map_ein2[sl] = pairs ? g.map_u_lo_w32 : g.map_u_lo;
                                gp.map_out[sl] = pairs ? g.map_x_w32[nb] : (first ? g.map_x_o32[nb] : g.map_x_k[nb]);
                                G.xlo_in = first ? g.ulo16 : nullptr;  // the first update reads u as hi + lo
                                G.x16_out = g.x16[nb];
                                G.opl16 = g.p16;
                                G.opr16 = xin16;
                                // on SM pairs P' is stored as its upper block triangle (the first
                                // update takes 64-deep k-blocks, later ones 128-deep)
                                G.sym_l = pairs ? 1 : 0;
                                gp.map_al[sl] = first ? g.map_p_mn : g.map_p_mn128;
                                break;
                            case OP_UPD_T:  // T = A P', full m x m tiles in the update launch
                                gp.map_a[sl] = g.map_a_k;
                                gp.map_b[sl] = g.map_p_mn128;
                                gp.map_out[sl] = g.map_t_w32;
                                G.x16_out = g.t16;
                                G.opl16 = g.a16;
                                G.opr16 = g.p16;
                                G.sym_l = G.sym_r = 1;  // A and P' as their upper block triangles
                                gp.map_al[sl] = g.map_a_mn128;
                                gp.map_bk[sl] = g.map_p_k;
                                break;
                            case OP_UPD_Q:  // X_{k+2} = Q X_k
                                gp.map_a[sl] = g.map_t_k;
                                gp.map_b[sl] = g.map_x_mn128[cb];
                                gp.map_out[sl] = g.map_x_w32[nb];
                                G.x16_out = g.x16[nb];
                                G.opl16 = g.t16;
                                G.opr16 = xin16;
                                break;
                            default: break;
                        }
                    }
                    if (n_in == 0) continue;
                    // the tile list of the groups that take part: every group of the chunk, or the
                    // Gram-pair groups alone (their own product Q)
                    const bool all_in = n_in == ch.ng;
                    bool has_t = false;
                    for (int sl = 0; sl < ch.ng; ++sl) has_t = has_t || ops[sl] == OP_UPD_T;
                    if (!all_in && !(n_in == n_gs && n_in_gs == n_gs) && !(ph == PH_PLAIN && q_fill)) {
                        cudaFree(h->arena);
                        delete h;
                        return fail(nullptr, MUON_ERR_CUDA, "internal error: launch plan group set");
                    }
                    const bool rev = (nlaunch[c]++ & 1) != 0;
                    auto pick = [&](int32_t off, int32_t n) {
                        gp.tiles = h->d_gemm_tiles + off + (rev ? n : 0);
                        gp.ntiles = n;
                    };
                    // the Gram-pair product Q runs on the update kernel
                    int mode = ph == PH_GRAM ? MODE_GRAM : (ph == PH_POLY ? MODE_POLY : MODE_UPDATE);
                    if (pairs) {
                        if (ph == PH_PLAIN && q_fill)
                            pick(ch.pair_qx_off, ch.pair_qx_n);
                        else if (ph == PH_PLAIN)
                            pick(ch.pair_q_off, ch.pair_q_n);
                        else if (mode == MODE_UPDATE && q_fill)
                            pick(ch.pair_ux_off, ch.pair_ux_n);
                        else if (mode == MODE_UPDATE)
                            pick(has_t ? ch.pair_t_off : ch.pair_off, has_t ? ch.pair_t_n : ch.pair_n);
                        else
                            pick(ch.spg_off, ch.spg_n);
                    } else {
                        pick(mode == MODE_GRAM ? ch.gram_off : (mode == MODE_POLY ? ch.poly_off : ch.upd_off),
                             mode == MODE_GRAM ? ch.gram_n : (mode == MODE_POLY ? ch.poly_n : ch.upd_n));
                    }
                    const int stage = ph == PH_PLAIN ? MUON_STAGE_PRODUCT
                                                     : (mode == MODE_GRAM ? MUON_STAGE_GRAM
                                                                          : (mode == MODE_POLY ? MUON_STAGE_POLY
                                                                                               : MUON_STAGE_UPDATE));
                    for (int sl = 0; sl < ch.ng; ++sl) {
                        if (ops[sl] == OP_NONE) continue;
                        const Group& g = h->groups[ch.gi[sl]];
                        double frac = 1.0;
                        if (q_fill && ops[sl] == OP_UPD) {
                            const double moved = (double)ch.q_fill[sl] / ((double)g.count * (g.m / 256) * (g.n / 256));
                            frac = ph == PH_PLAIN ? moved : 1.0 - moved;
                        }
                        add_work(stage, g, ops[sl], first, pairs, frac);
                    }
                    h->work_launches[stage]++;
                    h->plan.push_back(Launch{stage, mode, c, it, pairs ? 1 : 0, it > 0 ? 1 : 0});
                    h->gparams.push_back(gp);
                }
            }
            // groups that updated their iterate now hold it in the other buffer
            for (size_t gi = 0; gi < h->groups.size(); ++gi) {
                const GroupOp op = group_op(h->groups[gi], it, steps, PH_UPDATE);
                if (op == OP_UPD || op == OP_UPD_Q) cur[gi] = first ? 0 : cur[gi] ^ 1;
            }
        }
        for (size_t gi = 0; gi < h->groups.size(); ++gi)
            if (cur[gi] != h->groups[gi].final_buf) {
                cudaFree(h->arena);
                delete h;
                return fail(nullptr, MUON_ERR_CUDA, "internal error: iterate buffer bookkeeping");
            }
        // the elementwise stages' algorithmic bytes: momentum reads g and the buffer and writes
        // the buffer and u's hi and lo halves; apply reads O (fp16) and p and writes p
        int64_t elems = 0;
        for (const muon_shape& sh : h->shapes) elems += sh.rows * sh.cols;
        h->work_bytes[MUON_STAGE_MOMENTUM] = elems * ((cfg.grad_dtype == MUON_GRAD_BF16 ? 2 : 4) + 4 + 4 + 2 + 2);
        h->work_bytes[MUON_STAGE_APPLY] = elems * (2 + 4 + 4);
        h->work_launches[MUON_STAGE_MOMENTUM] = 1;
        h->work_launches[MUON_STAGE_NORM] = 1;
        h->work_launches[MUON_STAGE_LANE] = 1 + (h->n_colwork > 0 ? 1 : 0);
        h->work_launches[MUON_STAGE_APPLY] = 1;
    }

    {
        std::lock_guard<std::mutex> lk(g_handles_mu);
        g_handles.insert(h);
    }
    *out = h;
    return MUON_OK;
}

int muon_step(muon_handle h, float* const* params, const void* const* grads, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (params == nullptr || grads == nullptr) return fail(h, MUON_ERR_ARG, "params / grads array is NULL");
    const int n = (int)h->shapes.size();
    for (int i = 0; i < n; ++i) {
        if (params[i] == nullptr || grads[i] == nullptr) return fail(h, MUON_ERR_ARG, "matrix %d: NULL pointer", i);
        if ((reinterpret_cast<uintptr_t>(params[i]) | reinterpret_cast<uintptr_t>(grads[i])) & 15u)
            return fail(h, MUON_ERR_ALIGN, "matrix %d: pointer not 16-byte aligned", i);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_CUDA(h, cudaSetDevice(h->device));
    h->n_recorded = 0;
    // Every launch after the step's first one may overlap the previous kernel's last tiles
    // (muon_config.launch_overlap): its CTAs start on SMs that kernel no longer fills, set
    // up their shared memory and TMEM, and wait in the kernel for its results.  The first
    // launch keeps plain stream order behind the caller's work.
    const bool ov = h->cfg.launch_overlap != 0;
    MUON_CUDA(h, mark(h, MUON_STAGE_MOMENTUM, s));
    if (h->schedule_on) MUON_CUDA(h, launch_schedule_advance(h->hp, h->sched, s));
    MUON_CUDA(h, run_elem_any(h, params, grads, false, ov && h->schedule_on, s));
    NormParams np{h->d_subs, (int32_t)h->subs.size(), h->norm_part, h->norm_scale, h->iter_scale, h->status};
    MUON_CUDA(h, mark(h, MUON_STAGE_NORM, s));
    MUON_CUDA(h, launch_norm_scale(np, ov, s));
    for (size_t k = 0; k < h->plan.size(); ++k) {
        const Launch& L = h->plan[k];
        const GemmParams* gpp = &h->gparams[k];
        GemmParams stalled;
        if (h->stall_next && L.it == 0 && L.chunk == h->stall_chunk && L.mode == MODE_POLY &&
            h->cfg.gemm_engine == MUON_GEMM_TCGEN05) {
            // test only (muon_debug_inject_stall): this launch's MMA issuers wait on an
            // mbarrier that nothing arrives on until their bounded wait gives up
            stalled = *gpp;
            stalled.debug_stall = 1;
            gpp = &stalled;
            h->stall_next = false;
        }
        const GemmParams& gp = *gpp;
        MUON_CUDA(h, mark(h, L.stage, s));
        if (h->cfg.gemm_engine == MUON_GEMM_TCGEN05) {
            // the first iteration works on bf16 u; later ones on the fp16 iterate
            const bool f16 = L.f16 != 0;
            cudaError_t e = cudaSuccess;
            switch (L.mode) {
                case MODE_GRAM:
                    e = L.pair ? (f16 ? launch_ns_sym_pair<MODE_GRAM, true>(gp, h->num_sms, ov, s)
                                      : launch_ns_sym_pair<MODE_GRAM, false>(gp, h->num_sms, ov, s))
                               : (f16 ? launch_ns_gemm_tc<MODE_GRAM, true>(gp, h->num_sms, ov, s)
                                      : launch_ns_gemm_tc<MODE_GRAM, false>(gp, h->num_sms, ov, s));
                    break;
                case MODE_POLY:
                    e = L.pair ? (f16 ? launch_ns_sym_pair<MODE_POLY, true>(gp, h->num_sms, ov, s)
                                      : launch_ns_sym_pair<MODE_POLY, false>(gp, h->num_sms, ov, s))
                               : (f16 ? launch_ns_gemm_tc<MODE_POLY, true>(gp, h->num_sms, ov, s)
                                      : launch_ns_gemm_tc<MODE_POLY, false>(gp, h->num_sms, ov, s));
                    break;
                default:
                    e = L.pair ? launch_ns_update_pair(gp, !f16, h->num_sms, ov, s)
                               : (f16 ? launch_ns_gemm_tc<MODE_UPDATE, true>(gp, h->num_sms, ov, s)
                                      : launch_ns_gemm_tc<MODE_UPDATE, false>(gp, h->num_sms, ov, s));
                    break;
            }
            MUON_CUDA(h, e);
        } else {
            for (int sl = 0; sl < gp.ngroups; ++sl) {
                const int cnt = h->groups[h->chunks[L.chunk].gi[sl]].count;
                if (L.mode == MODE_GRAM) MUON_CUDA(h, launch_ns_gemm_simt<MODE_GRAM>(gp, sl, cnt, s));
                if (L.mode == MODE_POLY) MUON_CUDA(h, launch_ns_gemm_simt<MODE_POLY>(gp, sl, cnt, s));
                if (L.mode == MODE_UPDATE) MUON_CUDA(h, launch_ns_gemm_simt<MODE_UPDATE>(gp, sl, cnt, s));
            }
        }
    }
    LaneParams lp{h->d_subs, (int32_t)h->subs.size(), h->hp, h->cfg.normuon, h->cfg.norm_preserve, h->iter_scale,
                  h->status};
    MUON_CUDA(h, mark(h, MUON_STAGE_LANE, s));
    if (h->n_colwork > 0) {
        ColSumParams cp{h->d_subs, h->d_colwork, h->n_colwork};
        MUON_CUDA(h, launch_col_sumsq(cp, ov, s));
    }
    MUON_CUDA(h, launch_lane_stats(lp, ov, s));
    MUON_CUDA(h, mark(h, MUON_STAGE_APPLY, s));
    MUON_CUDA(h, run_elem_any(h, params, grads, true, ov, s));
    MUON_CUDA(h, mark(h, -1, s));
    return MUON_OK;
}

int muon_reset(muon_handle h, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_CUDA(h, cudaSetDevice(h->device));
    int64_t mom_floats = 0;
    for (size_t i = 0; i < h->shapes.size(); ++i) mom_floats += round_up(h->shapes[i].rows * h->shapes[i].cols, 64);
    MUON_CUDA(h, cudaMemsetAsync(h->momentum, 0, sizeof(float) * (size_t)mom_floats, s));
    for (const Group& g : h->groups)
        MUON_CUDA(h, cudaMemsetAsync(g.v, 0, sizeof(float) * (size_t)g.count * g.lane_stride, s));
    MUON_CUDA(h, cudaMemsetAsync(&h->sched->step, 0, sizeof(int64_t), s));
    return MUON_OK;
}

int muon_set_schedule(muon_handle h, const muon_schedule* sched, int64_t start_step, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (start_step < 0) return fail(h, MUON_ERR_ARG, "start_step must be >= 0");
    DevSchedule d;
    memset(&d, 0, sizeof(d));
    d.step = start_step;
    if (sched) {
        const muon_schedule& q = *sched;
        if (!std::isfinite(q.lr_base) || q.lr_base < 0.f || !std::isfinite(q.lr_floor) || q.lr_floor < 0.f)
            return fail(h, MUON_ERR_ARG, "lr_base and lr_floor must be finite and >= 0");
        if (q.cooldown_start < -1 || q.cooldown_end <= q.cooldown_start)
            return fail(h, MUON_ERR_ARG, "need -1 <= cooldown_start < cooldown_end");
        if (q.momentum_warmup < 0) return fail(h, MUON_ERR_ARG, "momentum_warmup must be >= 0");
        if (!std::isfinite(q.momentum_start) || !std::isfinite(q.momentum_end))
            return fail(h, MUON_ERR_ARG, "momentum_start / momentum_end must be finite");
        d.cooldown_start = q.cooldown_start;
        d.cooldown_end = q.cooldown_end;
        d.momentum_warmup = q.momentum_warmup;
        d.lr_base = q.lr_base;
        d.lr_floor = q.lr_floor;
        d.momentum_start = q.momentum_start;
        d.momentum_end = q.momentum_end;
    }
    MUON_CUDA(h, cudaSetDevice(h->device));
    MUON_CUDA(h, launch_schedule_set(h->sched, d, static_cast<cudaStream_t>(stream)));
    h->schedule_on = sched != nullptr;
    return MUON_OK;
}

int muon_get_step(muon_handle h, int64_t* step, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!step) return fail(h, MUON_ERR_ARG, "step is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_CUDA(h, cudaSetDevice(h->device));
    MUON_CUDA(h, cudaStreamSynchronize(s));
    MUON_CUDA(h, cudaMemcpy(step, &h->sched->step, sizeof(int64_t), cudaMemcpyDeviceToHost));
    return MUON_OK;
}

int muon_set_hparams(muon_handle h, float lr, float momentum, float beta2, float weight_decay, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    MUON_CUDA(h, cudaSetDevice(h->device));
    MUON_CUDA(h, launch_set_hparams(h->hp, lr, momentum, beta2, weight_decay, static_cast<cudaStream_t>(stream)));
    h->cfg.lr = lr;
    h->cfg.momentum = momentum;
    h->cfg.beta2 = beta2;
    h->cfg.weight_decay = weight_decay;
    return MUON_OK;
}

int muon_sync_status(muon_handle h, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    MUON_CUDA(h, cudaSetDevice(h->device));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_CUDA(h, cudaStreamSynchronize(s));
    int st = 0;
    MUON_CUDA(h, cudaMemcpy(&st, h->status, sizeof(int), cudaMemcpyDeviceToHost));
    if (st != 0) {
        MUON_CUDA(h, cudaMemset(h->status, 0, sizeof(int)));
        if (st & STATUS_TIMEOUT)
            return fail(h, MUON_ERR_TIMEOUT,
                        "a kernel's bounded wait gave up; the parameters and the second moment were left unchanged "
                        "from that step on");
        if (st & STATUS_PAIR) return fail(h, MUON_ERR_CUDA, "an SM pair did not get one shared TMEM allocation");
        if (st & STATUS_NONFINITE)
            return fail(h, MUON_ERR_NONFINITE,
                        "a matrix's update direction was not finite; that matrix's step was skipped");
    }
    return MUON_OK;
}

int muon_destroy(muon_handle h) {
    int rc = check_handle(h);
    if (rc) return rc;
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    if (h->arena) cudaFree(h->arena);
    h->arena = nullptr;
    for (cudaEvent_t e : h->events) cudaEventDestroy(e);
    h->events.clear();
    h->profiling = false;
    h->alive = false;  // the host object stays as a tombstone so stale handles are recognised
    h->gparams.clear();
    h->gparams.shrink_to_fit();
    h->plan.clear();
    return MUON_OK;
}

int muon_num_matrices(muon_handle h, int32_t* out) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!out) return fail(h, MUON_ERR_ARG, "out is NULL");
    *out = (int32_t)h->subs.size();
    return MUON_OK;
}

int muon_matrix_info(muon_handle h, int32_t index, int64_t out[8]) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!out || index < 0 || index >= (int32_t)h->subs.size()) return fail(h, MUON_ERR_ARG, "bad index");
    const SubDesc& d = h->subs[index];
    out[0] = d.parent;
    out[1] = h->sub_parent_q[index];
    out[2] = d.rows;
    out[3] = d.cols;
    out[4] = d.transposed;
    out[5] = d.m;
    out[6] = d.n;
    out[7] = d.lane_cols ? d.n : d.m;
    return MUON_OK;
}

int muon_workspace_bytes(muon_handle h, int64_t* out) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!out) return fail(h, MUON_ERR_ARG, "out is NULL");
    *out = (int64_t)h->arena_bytes;
    return MUON_OK;
}

int muon_launch_count(muon_handle h, int32_t* out) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!out) return fail(h, MUON_ERR_ARG, "out is NULL");
    *out = launches_per_step(h);
    return MUON_OK;
}

int muon_stage_work(muon_handle h, int64_t* flops, int64_t* bytes, int32_t* launches) {
    int rc = check_handle(h);
    if (rc) return rc;
    for (int k = 0; k < MUON_NUM_STAGES; ++k) {
        if (flops) flops[k] = h->work_flops[k];
        if (bytes) bytes[k] = h->work_bytes[k];
        if (launches) launches[k] = h->work_launches[k];
    }
    return MUON_OK;
}

int muon_set_profiling(muon_handle h, int32_t enable) {
    int rc = check_handle(h);
    if (rc) return rc;
    MUON_CUDA(h, cudaSetDevice(h->device));
    if (enable && h->events.empty()) {
        const int n = 4 + (int)h->plan.size() + 1;
        h->events.resize(n);
        h->event_stage.assign(n, -1);
        for (int k = 0; k < n; ++k) MUON_CUDA(h, cudaEventCreate(&h->events[k]));
    }
    h->profiling = enable != 0;
    h->n_recorded = 0;
    return MUON_OK;
}

int muon_get_stage_times(muon_handle h, float* out) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!out) return fail(h, MUON_ERR_ARG, "out is NULL");
    for (int k = 0; k < MUON_NUM_STAGES; ++k) out[k] = 0.f;
    if (h->n_recorded < 2) return fail(h, MUON_ERR_ARG, "no profiled step recorded");
    MUON_CUDA(h, cudaSetDevice(h->device));
    MUON_CUDA(h, cudaEventSynchronize(h->events[h->n_recorded - 1]));
    for (int k = 0; k + 1 < h->n_recorded; ++k) {
        float ms = 0.f;
        MUON_CUDA(h, cudaEventElapsedTime(&ms, h->events[k], h->events[k + 1]));
        const int st = h->event_stage[k];
        if (st >= 0 && st < MUON_NUM_STAGES) out[st] += ms;
    }
    return MUON_OK;
}

int muon_get_state(muon_handle h, int32_t which, int32_t index, void* dst, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!dst) return fail(h, MUON_ERR_ARG, "dst is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_CUDA(h, cudaSetDevice(h->device));
    if (which == MUON_STATE_MOMENTUM) {
        if (index < 0 || index >= (int32_t)h->shapes.size()) return fail(h, MUON_ERR_ARG, "bad parameter index");
        const muon_shape& sh = h->shapes[index];
        MUON_CUDA(h, cudaMemcpyAsync(dst, h->momentum + h->mom_off[index], sizeof(float) * sh.rows * sh.cols,
                                     cudaMemcpyDefault, s));
        return MUON_OK;
    }
    if (index < 0 || index >= (int32_t)h->subs.size()) return fail(h, MUON_ERR_ARG, "bad matrix index");
    const SubDesc& d = h->subs[index];
    if (which == MUON_STATE_SECOND_MOMENT) {
        MUON_CUDA(h, cudaMemcpyAsync(dst, d.v, sizeof(float) * (d.lane_cols ? d.n : d.m), cudaMemcpyDefault, s));
    } else if (which == MUON_STATE_ORTHO || which == MUON_STATE_DIRECTION) {
        // both are rebuilt on the device: O = c * (stored fp16 output), u = hi + lo
        cudaPointerAttributes attr;
        if (cudaPointerGetAttributes(&attr, dst) != cudaSuccess ||
            (attr.type != cudaMemoryTypeDevice && attr.type != cudaMemoryTypeManaged)) {
            cudaGetLastError();
            return fail(h, MUON_ERR_ARG, "MUON_STATE_ORTHO / MUON_STATE_DIRECTION need a device destination");
        }
        if (which == MUON_STATE_ORTHO)
            MUON_CUDA(h, launch_scale_f16(static_cast<float*>(dst), d.o16, h->iter_scale + index, d.m, d.n, d.ldx, s));
        else
            MUON_CUDA(h, launch_combine_hilo(static_cast<float*>(dst), d.u16, d.ulo16, d.m, d.n, d.ldx, s));
    } else {
        return fail(h, MUON_ERR_ARG, "bad state selector %d", which);
    }
    return MUON_OK;
}

int muon_set_state(muon_handle h, int32_t which, int32_t index, const void* src, void* stream) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (!src) return fail(h, MUON_ERR_ARG, "src is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    MUON_CUDA(h, cudaSetDevice(h->device));
    if (which == MUON_STATE_MOMENTUM) {
        if (index < 0 || index >= (int32_t)h->shapes.size()) return fail(h, MUON_ERR_ARG, "bad parameter index");
        const muon_shape& sh = h->shapes[index];
        MUON_CUDA(h, cudaMemcpyAsync(h->momentum + h->mom_off[index], src, sizeof(float) * sh.rows * sh.cols,
                                     cudaMemcpyDefault, s));
        return MUON_OK;
    }
    if (which == MUON_STATE_SECOND_MOMENT) {
        if (index < 0 || index >= (int32_t)h->subs.size()) return fail(h, MUON_ERR_ARG, "bad matrix index");
        const SubDesc& d = h->subs[index];
        MUON_CUDA(h, cudaMemcpyAsync(d.v, src, sizeof(float) * (d.lane_cols ? d.n : d.m), cudaMemcpyDefault, s));
        return MUON_OK;
    }
    return fail(h, MUON_ERR_ARG, "state %d cannot be written", which);
}

int muon_debug_inject_stall(muon_handle h) {
    int rc = check_handle(h);
    if (rc) return rc;
    if (h->cfg.gemm_engine != MUON_GEMM_TCGEN05)
        return fail(h, MUON_ERR_ARG, "the stall is injected into a tensor-core kernel (gemm_engine TCGEN05 only)");
    // the stall goes into the one-SM polynomial kernel: a chunk of groups that do not tile by 256
    h->stall_chunk = -1;
    for (int c = 0; c < (int)h->chunks.size() && h->stall_chunk < 0; ++c)
        if (h->chunks[c].spg_n == 0) h->stall_chunk = c;
    if (h->stall_chunk < 0)
        return fail(h, MUON_ERR_ARG, "no matrix of this handle runs the one-SM polynomial (every shape tiles by 256)");
    h->stall_next = true;
    return MUON_OK;
}

}  // extern "C"
