/*
 * muon_adam.h -- C ABI of the fused Adam step for the parameters Muon does
 * not take: the token embedding, the output head and scalar parameters.
 *
 * Sources:
 *   - "modded-nanogpt 50B-token 长时程训练实验解析：Muon vs Adam 与数据复用策略的实证对比",
 *     section "优化器三件套" (the optimizer trio): the embedding (lr 0.3) and
 *     the head (lr 0.002) are trained by the library Adam with betas
 *     (0.9, 0.95), fused, weight decay 0, next to Muon on the body; one WSD
 *     schedule scales every optimizer's learning rate.
 *   - "modded-nanogpt 的 FlexAttention 记录解析", section "优化器分工": the same
 *     split with lr 0.6 / 0.008 and a scalar group at lr 0.04.
 * The pages pass only lr and betas, so the rest is the library default
 * (eps 1e-8, no AMSGrad, an L2 term g + wd*p that is 0 there).  Per element,
 * with the shared step counter t starting at 1:
 *
 *   g <- g + wd * p
 *   m <- beta1 m + (1 - beta1) g
 *   v <- beta2 v + (1 - beta2) g^2
 *   p <- p - lr * s * (m / (1 - beta1^t)) / (sqrt(v / (1 - beta2^t)) + eps)
 *
 * where s is the step's learning-rate multiplier (muon_adam_set_lr_scale or a
 * schedule).  m and v are fp32, owned by the handle.
 *
 * Streams, threading and errors follow muon.h: calls enqueue on `stream`
 * unless stated otherwise, a handle is used from one host thread at a time,
 * and functions return MUON_OK or a negative muon_status.
 */
#ifndef MUON_ADAM_GB300_H
#define MUON_ADAM_GB300_H

#include <stdint.h>

#include "muon.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct muon_adam_s* muon_adam_handle;

#define MUON_ADAM_MAX_TENSORS 1024

/* One tensor of the group: numel contiguous elements (fp32 parameters,
 * gradients of muon_adam_config.grad_dtype).  16 bytes. */
typedef struct {
    int64_t numel;       /* >= 1 */
    float lr;            /* base learning rate of this tensor (finite, >= 0) */
    float weight_decay;  /* L2 coefficient (finite; 0 on the pages) */
} muon_adam_tensor;

/* 16 bytes. */
typedef struct {
    float beta1;         /* in [0, 1) */
    float beta2;         /* in [0, 1) */
    float eps;           /* finite, >= 0 */
    int32_t grad_dtype;  /* muon_grad_dtype */
} muon_adam_config;

/* Fills *cfg with beta1 0.9, beta2 0.95, eps 1e-8, grad_dtype BF16. */
void muon_adam_config_default(muon_adam_config* cfg);

/* Builds the work list for `n` tensors on CUDA device `device`, allocates and
 * zeroes m, v and the step counter.  The only allocating call; synchronous.
 * MUON_ERR_ARG for bad counts / values, MUON_ERR_UNSUPPORTED when the device
 * is not sm_103, MUON_ERR_NOMEM when the allocation fails. */
int muon_adam_create(const muon_adam_tensor* tensors, int32_t n, const muon_adam_config* cfg, int32_t device,
                     muon_adam_handle* out);

/* One Adam step over every tensor: params[i] (fp32, device, in place) and
 * grads[i] (device, read only), both 16-byte aligned (MUON_ERR_ALIGN
 * otherwise).  Two kernel launches (one thread that advances t and the
 * schedule, then the fused update); no allocation and no host
 * synchronisation, so it can be captured in a CUDA graph. */
int muon_adam_step(muon_adam_handle h, float* const* params, const void* const* grads, void* stream);

/* Zeroes m, v, the step counter t and the schedule's step index. */
int muon_adam_reset(muon_adam_handle h, void* stream);

/* Learning-rate multiplier used while no schedule is installed (default 1),
 * a device scalar written in stream order. */
int muon_adam_set_lr_scale(muon_adam_handle h, float scale, void* stream);

/* Installs a step schedule for the multiplier: s = lr_base * m(step) with the
 * curve of muon_set_schedule (muon.h); its momentum fields are not used.
 * The schedule index starts at `start_step` and advances on the device with
 * every step.  sched == NULL returns to the muon_adam_set_lr_scale value.
 * Argument rules as muon_set_schedule. */
int muon_adam_set_schedule(muon_adam_handle h, const muon_schedule* sched, int64_t start_step, void* stream);

/* Synchronises `stream` and reads t, the number of steps since create/reset. */
int muon_adam_get_step(muon_adam_handle h, int64_t* t, void* stream);

/* Sets t (>= 0) in stream order, e.g. with muon_adam_set_state when resuming
 * from a checkpoint: the next step then runs as step t + 1. */
int muon_adam_set_step(muon_adam_handle h, int64_t t, void* stream);

/* Device-to-device copy of tensor `index`'s first (which = 0) or second
 * (which = 1) moment, numel floats, to / from `dst` / `src` on `stream`. */
int muon_adam_get_state(muon_adam_handle h, int32_t which, int32_t index, float* dst, void* stream);
int muon_adam_set_state(muon_adam_handle h, int32_t which, int32_t index, const float* src, void* stream);

/* Kernel launches one step enqueues (2). */
int muon_adam_launch_count(muon_adam_handle h, int32_t* out);

/* Text of the handle's last error (NULL: the last muon_adam_create failure). */
const char* muon_adam_last_error(muon_adam_handle h);

/* Frees everything the handle owns (synchronises its device). */
int muon_adam_destroy(muon_adam_handle h);

#ifdef __cplusplus
}
#endif

#endif
