// Fused Adam for the embedding, head and scalar groups (include/muon_adam.h).
//
// The pages train these tensors with the library Adam, betas (0.9, 0.95)
// ("modded-nanogpt 50B-token ..." section "优化器三件套"; "modded-nanogpt 的
// FlexAttention 记录解析" section "优化器分工").  One step is two launches:
//
//   k_adam_prologue  one thread: t <- t + 1, the bias corrections of step t,
//                    the step's lr multiplier (a device schedule or a scalar)
//   k_adam           every element of every tensor once: 4096-element work
//                    units, one per CTA, 16 elements per thread as four
//                    16-byte vectors, all loads issued before any arithmetic
//
// The update reads g (2 or 4 bytes), p, m, v and writes p, m, v: 26 bytes per
// element with bf16 gradients, so the kernel is bound by HBM bandwidth.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <vector>

#include "../../include/muon_adam.h"
#include "muon_internal.h"
#include "ptx_sm103.cuh"

namespace muon {

constexpr int kAdamThreads = 256;
constexpr int kAdamUnit = 4096;                                   // elements per CTA
constexpr int kAdamVecs = kAdamUnit / 4 / kAdamThreads;           // 16-byte vectors per thread

struct AdamDev {
    int64_t t;            // steps taken since create / reset
    float lr_scale;       // multiplier while no schedule is installed
    float step_scale;     // multiplier of the running step (prologue output)
    float inv_bc1;        // 1 / (1 - beta1^t)
    float inv_sqrt_bc2;   // 1 / sqrt(1 - beta2^t)
    int32_t sched_on;
    int32_t pad;
    DevSchedule sched;    // lr curve and its step index (momentum fields unused)
};

struct AdamUnit {
    int64_t start;        // first element within the tensor (a multiple of kAdamUnit)
    int32_t tensor;
    int32_t count;        // elements in this unit, 1..kAdamUnit
};

template <int CAP>
struct AdamParams {
    const AdamUnit* units;
    float* m;
    float* v;
    const int64_t* off;   // per tensor: first element of its m / v slice (a multiple of 4)
    const float* lr;
    const float* wd;
    const AdamDev* dev;
    float beta1, omb1, beta2, omb2, eps;
    float* p[CAP];
    const void* g[CAP];
};

__global__ void k_adam_prologue(AdamDev* d, double beta1, double beta2) {
    const int64_t t = d->t + 1;
    d->t = t;
    d->inv_bc1 = (float)(1.0 / (1.0 - pow(beta1, (double)t)));
    d->inv_sqrt_bc2 = (float)(1.0 / sqrt(1.0 - pow(beta2, (double)t)));
    float s = d->lr_scale;
    if (d->sched_on) {
        const DevSchedule& sc = d->sched;
        const int64_t st = sc.step;
        double mult;
        if (st <= sc.cooldown_start)
            mult = 1.0;
        else if (st >= sc.cooldown_end)
            mult = (double)sc.lr_floor;
        else
            mult = (double)sc.lr_floor + (1.0 - (double)sc.lr_floor) * ((double)(sc.cooldown_end - st) /
                                                                        (double)(sc.cooldown_end - sc.cooldown_start));
        s = (float)((double)sc.lr_base * mult);
        d->sched.step = st + 1;
    }
    d->step_scale = s;
}

__global__ void k_adam_set_sched(AdamDev* d, DevSchedule val, int32_t on) {
    d->sched = val;
    d->sched_on = on;
}

__global__ void k_adam_set_scale(AdamDev* d, float scale) { d->lr_scale = scale; }

__global__ void k_adam_set_t(AdamDev* d, int64_t t) { d->t = t; }

template <bool GRAD_F32>
__device__ __forceinline__ float4 load_grad4(const void* g, int64_t e) {
    if (GRAD_F32) return __ldg(reinterpret_cast<const float4*>(static_cast<const float*>(g) + e));
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(g) + e));
    return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u), __uint_as_float(w.y << 16),
                       __uint_as_float(w.y & 0xFFFF0000u));
}

template <bool GRAD_F32>
__device__ __forceinline__ float load_grad1(const void* g, int64_t e) {
    if (GRAD_F32) return static_cast<const float*>(g)[e];
    return bf2f(static_cast<const uint16_t*>(g)[e]);
}

struct AdamCoef {
    float beta1, omb1, beta2, omb2, eps, wd, step, inv_sqrt_bc2;
    bool l2;
};

__device__ __forceinline__ void adam_elem(float& p, float& m, float& v, float g, const AdamCoef& c) {
    if (c.l2) g = fmaf(c.wd, p, g);
    m = fmaf(c.beta1, m, c.omb1 * g);
    v = fmaf(c.beta2, v, (c.omb2 * g) * g);
    const float denom = fmaf(sqrtf(v), c.inv_sqrt_bc2, c.eps);
    p = fmaf(-c.step, m / denom, p);
}

template <int CAP, bool GRAD_F32>
__global__ void __launch_bounds__(kAdamThreads) k_adam(const __grid_constant__ AdamParams<CAP> a) {
    const AdamUnit u = a.units[blockIdx.x];
    const int ti = u.tensor;
    float* p = a.p[ti] + u.start;
    const void* g = a.g[ti];
    float* m = a.m + a.off[ti] + u.start;
    float* v = a.v + a.off[ti] + u.start;
    AdamCoef c;
    c.beta1 = a.beta1;
    c.omb1 = a.omb1;
    c.beta2 = a.beta2;
    c.omb2 = a.omb2;
    c.eps = a.eps;
    c.wd = a.wd[ti];
    c.l2 = c.wd != 0.f;
    c.step = a.lr[ti] * a.dev->step_scale * a.dev->inv_bc1;
    c.inv_sqrt_bc2 = a.dev->inv_sqrt_bc2;

    const int nvec = u.count >> 2;
    float4 pv[kAdamVecs], mv[kAdamVecs], vv[kAdamVecs], gv[kAdamVecs];
#pragma unroll
    for (int k = 0; k < kAdamVecs; ++k) {
        const int vi = threadIdx.x + k * kAdamThreads;
        if (vi < nvec) {
            pv[k] = *reinterpret_cast<const float4*>(p + 4 * vi);
            mv[k] = *reinterpret_cast<const float4*>(m + 4 * vi);
            vv[k] = *reinterpret_cast<const float4*>(v + 4 * vi);
            gv[k] = load_grad4<GRAD_F32>(g, u.start + 4 * vi);
        }
    }
#pragma unroll
    for (int k = 0; k < kAdamVecs; ++k) {
        const int vi = threadIdx.x + k * kAdamThreads;
        if (vi < nvec) {
            adam_elem(pv[k].x, mv[k].x, vv[k].x, gv[k].x, c);
            adam_elem(pv[k].y, mv[k].y, vv[k].y, gv[k].y, c);
            adam_elem(pv[k].z, mv[k].z, vv[k].z, gv[k].z, c);
            adam_elem(pv[k].w, mv[k].w, vv[k].w, gv[k].w, c);
            *reinterpret_cast<float4*>(p + 4 * vi) = pv[k];
            *reinterpret_cast<float4*>(m + 4 * vi) = mv[k];
            *reinterpret_cast<float4*>(v + 4 * vi) = vv[k];
        }
    }
    // last 1-3 elements of a tensor whose size is not a multiple of 4
    const int tail = u.count & 3;
    if ((int)threadIdx.x < tail) {
        const int e = 4 * nvec + threadIdx.x;
        float pe = p[e], me = m[e], ve = v[e];
        adam_elem(pe, me, ve, load_grad1<GRAD_F32>(g, u.start + e), c);
        p[e] = pe;
        m[e] = me;
        v[e] = ve;
    }
}

}  // namespace muon

using namespace muon;

struct muon_adam_s {
    bool alive = true;
    int device = 0;
    muon_adam_config cfg{};
    std::vector<muon_adam_tensor> tensors;
    std::vector<int64_t> off;       // host copy of the m / v offsets
    void* arena = nullptr;
    AdamDev* dev = nullptr;
    float* m = nullptr;
    float* v = nullptr;
    int64_t* d_off = nullptr;
    float* d_lr = nullptr;
    float* d_wd = nullptr;
    AdamUnit* d_units = nullptr;
    int64_t nunits = 0;
    int64_t state_floats = 0;
    std::string last_error;
};

namespace {

std::mutex g_adam_mu;
std::set<muon_adam_s*> g_adam_handles;
std::string g_adam_create_error;

int adam_fail(muon_adam_s* h, int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    if (h)
        h->last_error = buf;
    else
        g_adam_create_error = buf;
    return code;
}

int adam_check(muon_adam_s* h) {
    if (h == nullptr) return adam_fail(nullptr, MUON_ERR_ARG, "null handle");
    std::lock_guard<std::mutex> lk(g_adam_mu);
    if (g_adam_handles.find(h) == g_adam_handles.end()) return adam_fail(nullptr, MUON_ERR_ARG, "unknown handle");
    if (!h->alive) return adam_fail(h, MUON_ERR_DESTROYED, "handle was destroyed");
    return MUON_OK;
}

#define ADAM_CUDA(h, call)                                                                                \
    do {                                                                                                  \
        cudaError_t e_ = (call);                                                                          \
        if (e_ != cudaSuccess) return adam_fail((h), MUON_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

template <int CAP>
int adam_launch(muon_adam_s* h, float* const* params, const void* const* grads, cudaStream_t s) {
    AdamParams<CAP> a;
    a.units = h->d_units;
    a.m = h->m;
    a.v = h->v;
    a.off = h->d_off;
    a.lr = h->d_lr;
    a.wd = h->d_wd;
    a.dev = h->dev;
    a.beta1 = h->cfg.beta1;
    a.omb1 = (float)(1.0 - (double)h->cfg.beta1);
    a.beta2 = h->cfg.beta2;
    a.omb2 = (float)(1.0 - (double)h->cfg.beta2);
    a.eps = h->cfg.eps;
    const int n = (int)h->tensors.size();
    for (int i = 0; i < CAP; ++i) {
        a.p[i] = i < n ? params[i] : nullptr;
        a.g[i] = i < n ? grads[i] : nullptr;
    }
    const dim3 grid((unsigned)h->nunits);
    if (h->cfg.grad_dtype == MUON_GRAD_F32)
        k_adam<CAP, true><<<grid, kAdamThreads, 0, s>>>(a);
    else
        k_adam<CAP, false><<<grid, kAdamThreads, 0, s>>>(a);
    ADAM_CUDA(h, cudaGetLastError());
    return MUON_OK;
}

bool finite_nonneg(float x) { return std::isfinite(x) && x >= 0.f; }

}  // namespace

extern "C" {

void muon_adam_config_default(muon_adam_config* cfg) {
    if (!cfg) return;
    cfg->beta1 = 0.9f;
    cfg->beta2 = 0.95f;
    cfg->eps = 1e-8f;
    cfg->grad_dtype = MUON_GRAD_BF16;
}

int muon_adam_create(const muon_adam_tensor* tensors, int32_t n, const muon_adam_config* cfg, int32_t device,
                     muon_adam_handle* out) {
    if (!out) return adam_fail(nullptr, MUON_ERR_ARG, "out is NULL");
    *out = nullptr;
    if (!tensors || !cfg) return adam_fail(nullptr, MUON_ERR_ARG, "tensors / cfg is NULL");
    if (n < 1 || n > MUON_ADAM_MAX_TENSORS)
        return adam_fail(nullptr, MUON_ERR_ARG, "tensor count %d outside 1..%d", n, MUON_ADAM_MAX_TENSORS);
    if (!(cfg->beta1 >= 0.f && cfg->beta1 < 1.f) || !(cfg->beta2 >= 0.f && cfg->beta2 < 1.f))
        return adam_fail(nullptr, MUON_ERR_ARG, "betas must lie in [0, 1)");
    if (!finite_nonneg(cfg->eps)) return adam_fail(nullptr, MUON_ERR_ARG, "eps must be finite and >= 0");
    if (cfg->grad_dtype != MUON_GRAD_BF16 && cfg->grad_dtype != MUON_GRAD_F32)
        return adam_fail(nullptr, MUON_ERR_ARG, "unknown grad_dtype %d", cfg->grad_dtype);
    for (int i = 0; i < n; ++i) {
        const muon_adam_tensor& t = tensors[i];
        if (t.numel < 1) return adam_fail(nullptr, MUON_ERR_SHAPE, "tensor %d: numel %lld < 1", i, (long long)t.numel);
        if (!finite_nonneg(t.lr)) return adam_fail(nullptr, MUON_ERR_ARG, "tensor %d: lr must be finite and >= 0", i);
        if (!std::isfinite(t.weight_decay)) return adam_fail(nullptr, MUON_ERR_ARG, "tensor %d: weight_decay not finite", i);
    }
    cudaDeviceProp prop;
    if (cudaSetDevice(device) != cudaSuccess) return adam_fail(nullptr, MUON_ERR_CUDA, "no CUDA device %d", device);
    if (cudaGetDeviceProperties(&prop, device) != cudaSuccess)
        return adam_fail(nullptr, MUON_ERR_CUDA, "cudaGetDeviceProperties failed");
    if (!(prop.major == 10 && prop.minor == 3))
        return adam_fail(nullptr, MUON_ERR_UNSUPPORTED, "device %d is sm_%d%d; this library is built for sm_103a",
                         device, prop.major, prop.minor);

    muon_adam_s* h = new muon_adam_s;
    h->device = device;
    h->cfg = *cfg;
    h->tensors.assign(tensors, tensors + n);
    std::vector<AdamUnit> units;
    int64_t floats = 0;
    for (int i = 0; i < n; ++i) {
        h->off.push_back(floats);
        floats += (tensors[i].numel + 3) / 4 * 4;
        for (int64_t st = 0; st < tensors[i].numel; st += kAdamUnit) {
            AdamUnit u;
            u.start = st;
            u.tensor = i;
            u.count = (int32_t)std::min<int64_t>(kAdamUnit, tensors[i].numel - st);
            units.push_back(u);
        }
    }
    if (units.size() > 0x7fffffffull) {
        delete h;
        return adam_fail(nullptr, MUON_ERR_SHAPE, "too many elements");
    }
    h->nunits = (int64_t)units.size();
    h->state_floats = floats;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off += (bytes + 255) / 256 * 256;
        return o;
    };
    const size_t o_dev = take(sizeof(AdamDev));
    const size_t o_off = take(sizeof(int64_t) * n);
    const size_t o_lr = take(sizeof(float) * n);
    const size_t o_wd = take(sizeof(float) * n);
    const size_t o_units = take(sizeof(AdamUnit) * units.size());
    const size_t o_m = take(sizeof(float) * (size_t)floats);
    const size_t o_v = take(sizeof(float) * (size_t)floats);
    if (cudaMalloc(&h->arena, off) != cudaSuccess) {
        cudaGetLastError();
        delete h;
        return adam_fail(nullptr, MUON_ERR_NOMEM, "cudaMalloc of %zu bytes failed", off);
    }
    char* base = static_cast<char*>(h->arena);
    h->dev = reinterpret_cast<AdamDev*>(base + o_dev);
    h->d_off = reinterpret_cast<int64_t*>(base + o_off);
    h->d_lr = reinterpret_cast<float*>(base + o_lr);
    h->d_wd = reinterpret_cast<float*>(base + o_wd);
    h->d_units = reinterpret_cast<AdamUnit*>(base + o_units);
    h->m = reinterpret_cast<float*>(base + o_m);
    h->v = reinterpret_cast<float*>(base + o_v);
    std::vector<float> lr(n), wd(n);
    for (int i = 0; i < n; ++i) {
        lr[i] = tensors[i].lr;
        wd[i] = tensors[i].weight_decay;
    }
    AdamDev d0;
    memset(&d0, 0, sizeof(d0));
    d0.lr_scale = 1.f;
    bool ok = cudaMemset(h->arena, 0, off) == cudaSuccess &&
              cudaMemcpy(h->dev, &d0, sizeof(d0), cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(h->d_off, h->off.data(), sizeof(int64_t) * n, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(h->d_lr, lr.data(), sizeof(float) * n, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(h->d_wd, wd.data(), sizeof(float) * n, cudaMemcpyHostToDevice) == cudaSuccess &&
              cudaMemcpy(h->d_units, units.data(), sizeof(AdamUnit) * units.size(), cudaMemcpyHostToDevice) ==
                  cudaSuccess;
    if (!ok) {
        cudaFree(h->arena);
        delete h;
        return adam_fail(nullptr, MUON_ERR_CUDA, "initialising the Adam state failed");
    }
    {
        std::lock_guard<std::mutex> lk(g_adam_mu);
        g_adam_handles.insert(h);
    }
    *out = h;
    return MUON_OK;
}

int muon_adam_step(muon_adam_handle h, float* const* params, const void* const* grads, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (!params || !grads) return adam_fail(h, MUON_ERR_ARG, "params / grads array is NULL");
    const int n = (int)h->tensors.size();
    for (int i = 0; i < n; ++i) {
        if (!params[i] || !grads[i]) return adam_fail(h, MUON_ERR_ARG, "tensor %d: NULL pointer", i);
        if ((reinterpret_cast<uintptr_t>(params[i]) | reinterpret_cast<uintptr_t>(grads[i])) & 15u)
            return adam_fail(h, MUON_ERR_ALIGN, "tensor %d: pointer not 16-byte aligned", i);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ADAM_CUDA(h, cudaSetDevice(h->device));
    k_adam_prologue<<<1, 1, 0, s>>>(h->dev, (double)h->cfg.beta1, (double)h->cfg.beta2);
    ADAM_CUDA(h, cudaGetLastError());
    return n <= 16 ? adam_launch<16>(h, params, grads, s) : adam_launch<MUON_ADAM_MAX_TENSORS>(h, params, grads, s);
}

int muon_adam_reset(muon_adam_handle h, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    ADAM_CUDA(h, cudaSetDevice(h->device));
    ADAM_CUDA(h, cudaMemsetAsync(h->m, 0, sizeof(float) * (size_t)h->state_floats, s));
    ADAM_CUDA(h, cudaMemsetAsync(h->v, 0, sizeof(float) * (size_t)h->state_floats, s));
    ADAM_CUDA(h, cudaMemsetAsync(&h->dev->t, 0, sizeof(int64_t), s));
    ADAM_CUDA(h, cudaMemsetAsync(&h->dev->sched.step, 0, sizeof(int64_t), s));
    return MUON_OK;
}

int muon_adam_set_lr_scale(muon_adam_handle h, float scale, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (!finite_nonneg(scale)) return adam_fail(h, MUON_ERR_ARG, "scale must be finite and >= 0");
    ADAM_CUDA(h, cudaSetDevice(h->device));
    k_adam_set_scale<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(h->dev, scale);
    ADAM_CUDA(h, cudaGetLastError());
    return MUON_OK;
}

int muon_adam_set_schedule(muon_adam_handle h, const muon_schedule* sched, int64_t start_step, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (start_step < 0) return adam_fail(h, MUON_ERR_ARG, "start_step must be >= 0");
    DevSchedule d;
    memset(&d, 0, sizeof(d));
    d.step = start_step;
    if (sched) {
        const muon_schedule& q = *sched;
        if (!finite_nonneg(q.lr_base) || !finite_nonneg(q.lr_floor))
            return adam_fail(h, MUON_ERR_ARG, "lr_base and lr_floor must be finite and >= 0");
        if (q.cooldown_start < -1 || q.cooldown_end <= q.cooldown_start)
            return adam_fail(h, MUON_ERR_ARG, "need -1 <= cooldown_start < cooldown_end");
        d.cooldown_start = q.cooldown_start;
        d.cooldown_end = q.cooldown_end;
        d.lr_base = q.lr_base;
        d.lr_floor = q.lr_floor;
    }
    ADAM_CUDA(h, cudaSetDevice(h->device));
    k_adam_set_sched<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(h->dev, d, sched ? 1 : 0);
    ADAM_CUDA(h, cudaGetLastError());
    return MUON_OK;
}

int muon_adam_get_step(muon_adam_handle h, int64_t* t, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (!t) return adam_fail(h, MUON_ERR_ARG, "t is NULL");
    ADAM_CUDA(h, cudaSetDevice(h->device));
    ADAM_CUDA(h, cudaStreamSynchronize(static_cast<cudaStream_t>(stream)));
    ADAM_CUDA(h, cudaMemcpy(t, &h->dev->t, sizeof(int64_t), cudaMemcpyDeviceToHost));
    return MUON_OK;
}

int muon_adam_set_step(muon_adam_handle h, int64_t t, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (t < 0) return adam_fail(h, MUON_ERR_ARG, "t must be >= 0");
    ADAM_CUDA(h, cudaSetDevice(h->device));
    k_adam_set_t<<<1, 1, 0, static_cast<cudaStream_t>(stream)>>>(h->dev, t);
    ADAM_CUDA(h, cudaGetLastError());
    return MUON_OK;
}

static int adam_state_copy(muon_adam_s* h, int32_t which, int32_t index, float* dst, const float* src, void* stream) {
    if (which != 0 && which != 1) return adam_fail(h, MUON_ERR_ARG, "which must be 0 (m) or 1 (v)");
    if (index < 0 || index >= (int32_t)h->tensors.size()) return adam_fail(h, MUON_ERR_ARG, "bad tensor index %d", index);
    float* state = (which == 0 ? h->m : h->v) + h->off[index];
    const size_t bytes = sizeof(float) * (size_t)h->tensors[index].numel;
    ADAM_CUDA(h, cudaSetDevice(h->device));
    if (dst)
        ADAM_CUDA(h, cudaMemcpyAsync(dst, state, bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
    else
        ADAM_CUDA(h, cudaMemcpyAsync(state, src, bytes, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)));
    return MUON_OK;
}

int muon_adam_get_state(muon_adam_handle h, int32_t which, int32_t index, float* dst, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (!dst) return adam_fail(h, MUON_ERR_ARG, "dst is NULL");
    return adam_state_copy(h, which, index, dst, nullptr, stream);
}

int muon_adam_set_state(muon_adam_handle h, int32_t which, int32_t index, const float* src, void* stream) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (!src) return adam_fail(h, MUON_ERR_ARG, "src is NULL");
    return adam_state_copy(h, which, index, nullptr, src, stream);
}

int muon_adam_launch_count(muon_adam_handle h, int32_t* out) {
    int rc = adam_check(h);
    if (rc) return rc;
    if (!out) return adam_fail(h, MUON_ERR_ARG, "out is NULL");
    *out = 2;
    return MUON_OK;
}

const char* muon_adam_last_error(muon_adam_handle h) {
    if (h == nullptr) return g_adam_create_error.c_str();
    std::lock_guard<std::mutex> lk(g_adam_mu);
    if (g_adam_handles.find(h) == g_adam_handles.end()) return "unknown handle";
    return h->last_error.c_str();
}

int muon_adam_destroy(muon_adam_handle h) {
    int rc = adam_check(h);
    if (rc) return rc;
    cudaSetDevice(h->device);
    cudaDeviceSynchronize();
    cudaFree(h->arena);
    {
        std::lock_guard<std::mutex> lk(g_adam_mu);
        g_adam_handles.erase(h);
    }
    delete h;
    return MUON_OK;
}

}  // extern "C"
