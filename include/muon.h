/*
 * muon.h -- C ABI of the GB300 (sm_103a) Muon / NorMuon optimizer step.
 *
 * One call, muon_step(), applies one optimizer step to a list of 2-D fp32
 * parameter matrices given their gradients:
 *
 *   S1  momentum        buf <- lerp(buf, g, 1 - mu)            (or buf <- mu*buf + g)
 *   S2  Nesterov        u   <- lerp(g, buf, mu)                (or u <- g + mu*buf; or u <- buf)
 *   S3  split + orient  a bank [R, C] with split = k is viewed as k matrices
 *                       [R, C/k]; each matrix is worked on in its wide
 *                       orientation (transposed when R > C)
 *   S4  normalise       X0 = u / (||u||_F + 1e-7)
 *   S5-S7 Newton-Schulz ns_steps times: A = X X^T; P = b A + c A A; X <- a X + P X
 *   S8  second moment   r_i = mean_j O_ij^2 over the long side; v <- lerp(v, r, 1 - beta2)
 *   S9  lane scale      O'_ij = O_ij / sqrt(max(v_i, 1e-10)), rescaled to ||O||_F
 *   S10 write-back      p <- p * (1 - lr*lr_mul*wd*wd_mul) - lr*lr_mul*O'
 *                       (plain Muon: no S8/S9, update scaled by lr*lr_mul*max(1, R/C)^0.5)
 *
 * Sources (web pages on the modded-nanogpt speedrun):
 *   - "modded-nanogpt 50B-token 长时程训练实验解析：Muon vs Adam 与数据复用策略的实证对比",
 *     section "从源码看 Muon 的分布式正交化实现" (Muon from the source): S1 (mul/add form),
 *     S2, S3 (transpose to the short side), S4, S5-S7 (coefficients (3.4445, -4.7750,
 *     2.0315), bf16 iteration), S10 (max(1, rows/cols)^0.5, p.add_(g, alpha=-lr));
 *     section "优化器三件套": Muon(lr=0.02, momentum=0.95), Nesterov on by default.
 *   - the 2025-10-27 FixMuonLR record write-up: S1 lerp form and reset() (change 2,
 *     momentum buffer moved to the group), S3 bank view as 4 matrices (change 2,
 *     attention reshape), S8/S9 NorMuon second_momentum_buffer (background; change 2),
 *     per-matrix lr_mul / wd_mul with c_fc.lr_mul = 2.0 (change 1).
 *
 * Threading and streams.  A handle may be used from one host thread at a time.
 * Every call that takes a stream only enqueues work on it (no host
 * synchronisation, no allocation) unless stated otherwise.  Streams are passed
 * as `void*` holding a cudaStream_t (NULL = the legacy default stream).
 *
 * Errors.  Functions return MUON_OK (0) or a negative muon_status.  The text
 * of the last error of a handle is available from muon_last_error(); errors
 * raised before a handle exists go to muon_last_error(NULL).  Errors detected
 * on the device are recorded in a device status word and reported by
 * muon_sync_status():
 *   - a bounded wait that gave up (MUON_ERR_TIMEOUT), or an SM pair that did not
 *     get one shared TMEM allocation (MUON_ERR_CUDA), is fatal: from the step in
 *     which it happened until muon_sync_status clears the word, every step leaves
 *     the parameters, the momentum and the second moment as they were (the
 *     failed step itself has already folded its gradient into the momentum);
 *   - a matrix whose update direction is not finite (a NaN or infinite gradient
 *     element, or an overflow) is reported as MUON_ERR_NONFINITE: only that
 *     matrix's step is skipped (its parameters and second moment stay as they
 *     were), and a momentum element whose new value would not be finite keeps
 *     its previous value.  Later steps run normally.
 * None of the pages specifies failure handling; the pages' only stability
 * advice concerns spikes in the gradient norm.
 */
#ifndef MUON_GB300_H
#define MUON_GB300_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct muon_s* muon_handle;

typedef enum {
    MUON_OK = 0,
    MUON_ERR_ARG = -1,         /* invalid argument (NULL pointer, bad count, bad enum, ...) */
    MUON_ERR_ALIGN = -2,       /* a parameter / gradient pointer is not 16-byte aligned */
    MUON_ERR_SHAPE = -3,       /* unsupported or inconsistent shape */
    MUON_ERR_CUDA = -4,        /* a CUDA runtime / driver call failed (text in muon_last_error) */
    MUON_ERR_TIMEOUT = -5,     /* a kernel's bounded wait gave up (device status word) */
    MUON_ERR_DESTROYED = -6,   /* the handle was destroyed */
    MUON_ERR_NOMEM = -7,       /* device allocation failed in muon_create */
    MUON_ERR_UNSUPPORTED = -8, /* the current device is not an sm_103 GPU */
    MUON_ERR_NONFINITE = -9    /* a matrix's update direction was not finite; its step was skipped */
} muon_status;

typedef enum { MUON_GRAD_BF16 = 0, MUON_GRAD_F32 = 1 } muon_grad_dtype;

/* muon_shape.flags */
#define MUON_SPLIT_CONTIGUOUS 0  /* bank split = view of contiguous [R, C] as [split, R, C/split] */
#define MUON_SPLIT_COLUMNS 1     /* bank split = column blocks [:, q*C/split : (q+1)*C/split] */

/* Newton-Schulz gemm engine (muon_config.gemm_engine) */
#define MUON_GEMM_TCGEN05 0      /* tcgen05 / TMEM / TMA grouped kernels (the product path) */
#define MUON_GEMM_SIMT 1         /* plain CUDA-core kernels; a slow debugging cross-check */

/* NorMuon lanes (muon_config.normuon_lanes): which rows or columns of a matrix
 * each get one second-moment entry.  The FixMuonLR record write-up (background
 * and change 2) has NorMuon average the squared update along the longer
 * dimension and scale each remaining lane by an rsqrt; it also says the early
 * attention reshape makes NorMuon act per column (per output dimension).
 * SHORT_SIDE is the first statement taken literally and is the default. */
#define MUON_LANES_SHORT_SIDE 0  /* one lane per row of the short side (mean over the long side) */
#define MUON_LANES_ROWS 1        /* one lane per row of the matrix as stored (mean over its columns) */
#define MUON_LANES_COLS 2        /* one lane per column of the matrix as stored (mean over its rows) */

/* Order of the Newton-Schulz work (muon_config.ns_form).  The iteration of the
 * "modded-nanogpt 50B-token" write-up (section "Muon from the source") is
 * X <- a X + (b A + c A^2) X with A = X X^T.  STANDARD computes exactly that every
 * iteration.  GRAM_PAIRS gives the same result in exact arithmetic for matrices whose
 * sides tile by 256 with n >= 2m: after the first iteration it takes iterations two
 * at a time, forming A_k = X_k X_k^T once, the pair's second Gram matrix as
 * A_{k+1} = (A_k P_k) P_k with P_k = a I + b A_k + c A_k^2, and the pair's output as
 * X_{k+2} = (P_{k+1} P_k) X_k: one m x n Gram matrix and one update per pair instead
 * of two of each, for three m x m products.  A single iteration left at the end, and
 * every other matrix, runs in the standard form.  Rounding differs from STANDARD at
 * the level of the 16-bit operands; every pair restarts from a freshly formed Gram
 * matrix, which keeps the error at the standard form's level. */
#define MUON_NS_STANDARD 0
#define MUON_NS_GRAM_PAIRS 1

#define MUON_MAX_MATRICES 1024   /* parameter matrices per handle */
#define MUON_MAX_NS_STEPS 16

/* One parameter matrix as the caller stores it: row-major fp32 params and
 * row-major gradients (bf16 or fp32, see muon_config.grad_dtype) of shape
 * rows x cols with row stride ld elements (ld = 0 means ld = cols).  With
 * split > 1 the matrix is a bank viewed as `split` matrices (flags select how);
 * a contiguous split needs ld == cols. */
typedef struct {
    int64_t rows;
    int64_t cols;
    int64_t ld;
    int32_t split;
    int32_t flags;
} muon_shape;

typedef struct {
    float lr;              /* base learning rate (device scalar; see muon_set_hparams) */
    float momentum;        /* mu (device scalar) */
    float beta2;           /* NorMuon second-moment decay (device scalar) */
    float weight_decay;    /* decoupled weight decay (device scalar) */
    int32_t ns_steps;      /* Newton-Schulz iterations, 1..MUON_MAX_NS_STEPS */
    int32_t nesterov;      /* 1: Nesterov direction (default) */
    int32_t lerp_form;     /* 1: buf.lerp_(g, 1-mu) (default); 0: buf = mu*buf + g */
    int32_t normuon;       /* 1: NorMuon lane scaling (S8/S9); 0: plain Muon */
    int32_t norm_preserve; /* 1: rescale O' to ||O||_F (default) */
    int32_t grad_dtype;    /* muon_grad_dtype */
    int32_t gemm_engine;   /* MUON_GEMM_TCGEN05 (default) or MUON_GEMM_SIMT */
    const float* lr_mul;   /* host array [n_mats] or NULL (all 1.0); copied at create */
    const float* wd_mul;   /* host array [n_mats] or NULL (all 1.0); copied at create */
    const float* ns_coeffs;/* host array [ns_steps * 3] of (a, b, c) per iteration, or NULL
                              for (3.4445, -4.7750, 2.0315) every iteration; copied */
    int32_t normuon_lanes; /* MUON_LANES_*: the second moment's lanes (NorMuon only) */
    int32_t ns_form;       /* MUON_NS_*: order of the Newton-Schulz products */
    int32_t launch_overlap;/* 1: every launch of a step after its first may begin while the previous
                              kernel finishes (programmatic dependent launch: the next kernel's CTAs
                              take the SMs the previous one no longer fills, set up their shared
                              memory and tensor memory, and wait in the kernel for its results);
                              0: plain stream order.  Results are identical either way. */
} muon_config;

/* Fills *cfg with: lr 0.02, momentum 0.95, beta2 0.95, weight_decay 0, ns_steps 5,
 * nesterov 1, lerp_form 1, normuon 1, norm_preserve 1, grad_dtype BF16,
 * gemm_engine TCGEN05, NULL arrays, normuon_lanes MUON_LANES_SHORT_SIDE,
 * ns_form MUON_NS_GRAM_PAIRS, launch_overlap 1.  Layout: 88 bytes (84 used), ns_form at
 * offset 76, launch_overlap at offset 80. */
void muon_config_default(muon_config* cfg);

/* Builds the execution plan for `n_mats` matrices on CUDA device `device`:
 * validates shapes, groups the (split) matrices by their wide shape, allocates
 * and zeroes all optimizer state (momentum: fp32, one per parameter; second
 * moment: fp32, one per lane) and the Newton-Schulz workspace, and encodes the
 * TMA descriptors.  This is the only call that allocates device memory.
 * Synchronous.  On success *out owns everything until muon_destroy. */
int muon_create(const muon_shape* shapes, int32_t n_mats, const muon_config* cfg,
                int32_t device, muon_handle* out);

/* One optimizer step.  params[i] (fp32, device, updated in place) and grads[i]
 * (device, read only) follow shapes[i] of muon_create; both 16-byte aligned.
 * The pointer arrays themselves are host arrays read during the call.
 * Enqueues all work on `stream`: no allocation, no host synchronisation, so it
 * can be captured in a CUDA graph (a captured graph keeps the pointers it was
 * captured with).  The caller keeps the buffers alive until the work is done. */
int muon_step(muon_handle h, float* const* params, const void* const* grads, void* stream);

/* Zeroes the momentum and second-moment buffers and the schedule's step
 * counter on `stream` (the reset() the FixMuonLR record adds to clear state
 * dirtied by warm-up / graph capture). */
int muon_reset(muon_handle h, void* stream);

/* Sets the device-resident scalars read by later steps (stream-ordered, so a
 * captured step graph follows schedule updates made between replays). */
int muon_set_hparams(muon_handle h, float lr, float momentum, float beta2,
                     float weight_decay, void* stream);

/* Step-indexed schedules evaluated on the device.
 *
 * Learning rate (FlexAttention record write-up, hyper-parameter table: a
 * constant phase and a linear warmdown to 0; FixMuonLR write-up, change 3: a
 * linear cool-down to an absolute floor that stays flat through the
 * extension steps):  lr(s) = lr_base * m(s), with m(s) = 1 for
 * s <= cooldown_start, lr_floor for s >= cooldown_end, and the straight line
 * between them in between.
 * Momentum (FlexAttention record write-up, section on the optimizer split):
 * mu(s) = momentum_start + (momentum_end - momentum_start) * min(s / momentum_warmup, 1)
 * (momentum_end throughout when momentum_warmup == 0).
 * s counts steps from 0.  Layout: 40 bytes, offsets 0, 4, 8, 16, 24, 28, 32. */
typedef struct {
    float lr_base;           /* lr at multiplier 1 */
    float lr_floor;          /* multiplier from cooldown_end on (0: decay to zero), >= 0 */
    int64_t cooldown_start;  /* last step at multiplier 1 (>= -1) */
    int64_t cooldown_end;    /* first step at lr_floor (> cooldown_start) */
    float momentum_start;    /* mu at step 0 */
    float momentum_end;      /* mu from step momentum_warmup on */
    int64_t momentum_warmup; /* steps of linear warm-up (>= 0) */
} muon_schedule;

/* Installs `sched` (copied) and sets the device step counter to `start_step`
 * (>= 0; e.g. when resuming), both stream-ordered on `stream`.  From then on
 * every muon_step first runs one single-thread kernel that writes lr(s) and
 * mu(s) into the device scalars (overriding muon_set_hparams for those two)
 * and advances s, so a graph captured after this call follows the schedule on
 * every replay with no host call.  sched == NULL removes the schedule (later
 * steps launch no schedule kernel; graphs captured before keep theirs).
 * muon_reset sets s back to 0.  MUON_ERR_ARG for a non-finite or negative
 * lr_base / lr_floor, cooldown_end <= cooldown_start, cooldown_start < -1,
 * momentum_warmup < 0 or start_step < 0. */
int muon_set_schedule(muon_handle h, const muon_schedule* sched, int64_t start_step, void* stream);

/* Synchronises `stream` and reads the device step counter: the schedule index
 * the next muon_step will use (0 when no schedule was ever installed). */
int muon_get_step(muon_handle h, int64_t* step, void* stream);

/* Synchronises `stream`, reads and clears the device status word (see
 * "Errors" above).  Returns MUON_OK, MUON_ERR_TIMEOUT, MUON_ERR_CUDA or
 * MUON_ERR_NONFINITE (in that order of precedence when several were raised). */
int muon_sync_status(muon_handle h, void* stream);

/* Releases all device memory of the handle.  Synchronises the device. */
int muon_destroy(muon_handle h);

const char* muon_error_string(int code);
const char* muon_last_error(muon_handle h);

/* ---- introspection and state access (checkpointing, tests) -------------- */

/* Number of matrices after bank splits. */
int muon_num_matrices(muon_handle h, int32_t* out);

/* Describes split matrix `index`: out[0] = parent parameter index, out[1] =
 * split index, out[2] = rows, out[3] = cols (as stored), out[4] = 1 if it is
 * worked on transposed, out[5] = m = min(rows, cols), out[6] = n = max(rows, cols),
 * out[7] = number of NorMuon lanes (the length of its second moment). */
int muon_matrix_info(muon_handle h, int32_t index, int64_t out[8]);

/* Bytes of device memory owned by the handle. */
int muon_workspace_bytes(muon_handle h, int64_t* out);

/* Number of kernel launches one muon_step enqueues. */
int muon_launch_count(muon_handle h, int32_t* out);

/* The work one muon_step does per stage, as planned at create time: flops[k]
 * the algorithmic flops of stage k (symmetric products counted once per
 * element of their upper triangle: m(m+1)n for a Gram matrix, m^2(m+1) for an
 * m x m product; 2 m^2 n for an update), bytes[k] its algorithmic DRAM bytes
 * (each operand read once, each result written once, at its stored width),
 * launches[k] its kernel launches.  Host arrays of MUON_NUM_STAGES entries;
 * any of them may be NULL. */
int muon_stage_work(muon_handle h, int64_t* flops, int64_t* bytes, int32_t* launches);

/* ---- stage timing (benchmarks) -------------------------------------------- */

/* Stages of one step. */
#define MUON_STAGE_MOMENTUM 0    /* S1-S3 + norm partials (k_momentum) */
#define MUON_STAGE_NORM 1        /* S4 scale per matrix (k_norm_scale) */
#define MUON_STAGE_GRAM 2        /* S5, all iterations summed */
#define MUON_STAGE_POLY 3        /* S6, all iterations summed */
#define MUON_STAGE_UPDATE 4      /* S7, all iterations summed */
#define MUON_STAGE_LANE 5        /* S8 + S9 factors (k_lane_stats) */
#define MUON_STAGE_APPLY 6       /* S10 (k_apply) */
#define MUON_STAGE_PRODUCT 7     /* MUON_NS_GRAM_PAIRS: each pair's product P_{k+1} P_k (its other
                                    two m x m products run inside the Gram and update launches) */
#define MUON_NUM_STAGES 8

/* enable != 0: every later muon_step records CUDA events around each launch
 * on its stream (creates the events on first use; no device allocation). */
int muon_set_profiling(muon_handle h, int32_t enable);

/* Per-stage device time (ms) of the most recent profiled step, summed over
 * that stage's launches: out[MUON_NUM_STAGES].  Waits for the step's events. */
int muon_get_stage_times(muon_handle h, float* out);

#define MUON_STATE_MOMENTUM 0      /* per parameter i: fp32 rows x cols, row-major, dense */
#define MUON_STATE_SECOND_MOMENT 1 /* per split matrix: fp32, one per NorMuon lane (muon_matrix_info out[7]);
                                      lanes in the order of the rows or columns they stand for */
#define MUON_STATE_ORTHO 2         /* per split matrix: last Newton-Schulz output O, wide
                                      orientation m x n, fp32, DEVICE destination only
                                      (rebuilt on the device from its scaled fp16 copy) */
#define MUON_STATE_DIRECTION 3     /* per split matrix: last Nesterov direction u, wide
                                      orientation m x n, fp32, DEVICE destination only
                                      (rebuilt on the device from its bf16 hi + lo pair) */

/* Copies one state array into `dst` (host or device memory; cudaMemcpyDefault)
 * on `stream`.  Layouts as listed above. */
int muon_get_state(muon_handle h, int32_t which, int32_t index, void* dst, void* stream);

/* Overwrites one state array (MOMENTUM or SECOND_MOMENT) from `src`. */
int muon_set_state(muon_handle h, int32_t which, int32_t index, const void* src, void* stream);

/* ---- test support ----------------------------------------------------------
 *
 * For failure-handling tests only; no part of the optimizer step uses it.
 * Makes the next muon_step's first one-SM polynomial launch (a tcgen05 kernel
 * that serves the matrices whose sides are not multiples of 256) wait on an
 * mbarrier that nothing arrives on, so that its bounded wait gives up after
 * about 2 s: the kernel then sets the status word, lets the copies it issued
 * land, frees its TMEM and returns, and the step leaves the parameters and
 * second moment unchanged (see "Errors").  One-shot.  MUON_ERR_ARG when
 * gemm_engine is not MUON_GEMM_TCGEN05 or when every matrix of the handle
 * tiles by 256 (no one-SM polynomial runs). */
int muon_debug_inject_stall(muon_handle h);

/* ---- allocation-free entry point ------------------------------------------
 *
 * No counterpart on the pages: this call exists for callers that cannot call
 * cudaMalloc where they run the step -- frameworks whose device memory belongs
 * to their own pool or arena, code where an allocation would synchronise the
 * device or is not allowed (a latency-critical loop, a host callback), and
 * users with a device-memory budget fixed at load time.
 *
 * For ONE matrix, dense row-major rows x cols: updates `momentum` (fp32, in
 * place) with the gradient `grad` (bf16 or fp32 per grad_dtype) exactly as
 * muon_step does (lerp or mul/add form), forms the Nesterov direction u and
 * writes x0 = u / (||u||_F + 1e-7) (fp32) -- steps S1, S2 and S4 in the
 * matrix's own orientation.  All pointers are device pointers.  Work is
 * enqueued on `stream`; nothing is allocated.
 *
 * Scratch: the per-tile partial sums of u^2 and the scale live in one static
 * device array of MUON_NOALLOC_MAX_TILES + 64 floats (about 256 KB) that every
 * GPU loading the library holds until the process exits.  Matrices needing
 * more than MUON_NOALLOC_MAX_TILES tiles of 64 x 64 are rejected with
 * MUON_ERR_SHAPE.  All calls share the array; calls whose work overlaps on
 * the GPU race, so order them on one stream.  The first call on a device looks
 * up the array's device address (cudaGetSymbolAddress) with that device
 * current, and looks it up again when the device's current context has
 * changed (after cudaDeviceReset the array may sit elsewhere); make the first
 * call, and the first call after a reset, before any stream capture.
 * momentum, x0 and grad must not overlap (identical pointers: MUON_ERR_ARG).
 * A CUDA error pending from earlier work of the caller is returned as
 * MUON_ERR_CUDA before anything is enqueued.  Returns MUON_OK, MUON_ERR_ARG,
 * MUON_ERR_SHAPE or MUON_ERR_CUDA. */
#define MUON_NOALLOC_MAX_TILES 65536
int muon_nesterov_normalize_noalloc(const void* grad, int32_t grad_dtype, float* momentum, float* x0,
                                    int64_t rows, int64_t cols, float mu, int32_t lerp_form,
                                    int32_t nesterov, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* MUON_GB300_H */
