// C ABI of the per-unit FSDP cycle (declared in include/fsdp_unit.h).
//
// A unit owns five slabs of length plan.slab_len (fp32 master, fp32 gradient
// shard, fp32 m, fp32 v, bf16 shadow); rank k's arena is
// [arena_base[k], arena_base[k] + arena_len[k]) of each.  Pads are zero from
// creation and stay zero: the gather and reduce-scatter never touch them and
// AdamW maps (p, g, m, v) = 0 to 0.
//
// The bf16 shadow equals RNE(master) whenever anything reads it.  AdamW
// stores it only when the unit gathers from it; otherwise the unit marks it
// stale, and the next read (a gather from it, a state export) first runs one
// cast pass over the slab.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdio>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "fsdp_unit.h"
#include "kernels.hpp"
#include "plan.hpp"

using fsdp::Plan;
using fsdp::Tile;

namespace {

thread_local std::string g_last_error;

int fail(int code, const std::string& why) {
    g_last_error = why;
    return code;
}

int cuda_fail(cudaError_t e, const char* what) {
    return fail(FSDP_E_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

struct ProfRecord {
    int kind;
    cudaEvent_t start;
    cudaEvent_t stop;
};

class DeviceGuard {
public:
    explicit DeviceGuard(int device) : device_(device) {
        if (cudaGetDevice(&prev_) != cudaSuccess) prev_ = -1;
        if (prev_ != device_) ok_ = cudaSetDevice(device_) == cudaSuccess;
    }
    ~DeviceGuard() {
        if (prev_ >= 0 && prev_ != device_) cudaSetDevice(prev_);
    }
    bool ok() const { return ok_; }

private:
    int device_;
    int prev_ = -1;
    bool ok_ = true;
};

bool aligned32(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 31u) == 0; }
bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

namespace fsdp {
// The calling thread's failure reason for fsdp_last_error, for the entry
// points defined outside this file.
int record_error(int code, const std::string& why) { return fail(code, why); }
}  // namespace fsdp

struct fsdp_unit {
    int device = 0;
    Plan plan;
    int nparams = 0;
    int grad_dtype = FSDP_DTYPE_F32;
    int raf = 1;
    int replicas = 1;
    int reduce_dtype = FSDP_DTYPE_F32;
    int gather_source = FSDP_GATHER_FROM_MASTER;
    int fuse = 0;
    fsdp_allocator allocator{nullptr, nullptr, nullptr};   // alloc == nullptr: cudaMalloc / cudaFree
    // device-step mode (CUDA-graph replay of AdamW): constants of steps
    // step_base+1 .. step_base+step_count live in step_table; step_counter
    // counts the steps taken on the device since the table was made
    bool device_steps = false;
    fsdp::AdamWConsts* step_table = nullptr;
    int64_t step_table_cap = 0;
    int64_t step_count = 0;
    int64_t step_base = 0;
    int64_t* step_counter = nullptr;
    int32_t* step_status = nullptr;
    int32_t* kstatus = nullptr;   // FSDP_KSTATUS_* bits raised by kernels
    unsigned long long wait_ns = 0;   // bound of the staged kernels' waits (0: their 10 s default)
    int withhold_next = 0;            // one-shot test of the give-up path (fsdp_unit_set_wait_limit)
    bool needs_reload = false;        // a kernel gave up: state incomplete until fsdp_load_params
    bool broken = false;              // a drain wait ran out too: only destroy is accepted
    float* master = nullptr;
    float* grad = nullptr;
    float* m = nullptr;
    float* v = nullptr;
    uint16_t* shadow = nullptr;
    Tile* tiles = nullptr;
    int64_t ntiles = 0;
    Tile* load_tiles = nullptr;
    int64_t nload_tiles = 0;
    fsdp::ParamSrc* param_src = nullptr;
    int64_t t = 0;
    bool loaded = false;
    mutable bool shadow_valid = true;   // the shadow slab holds RNE(master)
    bool profiling = false;
    std::vector<ProfRecord> prof;
};

namespace {

// Device memory of a unit: from the caller's allocator when one was given,
// else cudaMalloc.  The buffers are read with 32-byte vector accesses, so a
// caller's block must be aligned to 256 bytes; a misaligned one is handed
// back at once.  Returns FSDP_OK or an error code (set via fail()).
int dev_alloc(fsdp_unit* u, void** p, size_t bytes) {
    if (bytes == 0) bytes = 32;
    *p = nullptr;
    if (u->allocator.alloc != nullptr) {
        void* q = u->allocator.alloc(bytes, u->allocator.ctx);
        if (q == nullptr) return fail(FSDP_E_OOM, "the caller's allocator returned NULL");
        if ((reinterpret_cast<uintptr_t>(q) & 255u) != 0) {
            u->allocator.free(q, u->allocator.ctx);
            return fail(FSDP_E_ALIGN, "the caller's allocator returned a block not aligned to 256 bytes");
        }
        *p = q;
        return FSDP_OK;
    }
    cudaError_t e = cudaMalloc(p, bytes);
    if (e != cudaSuccess) {
        cudaGetLastError();
        *p = nullptr;
        return fail(e == cudaErrorMemoryAllocation ? FSDP_E_OOM : FSDP_E_CUDA,
                    std::string("cudaMalloc: ") + cudaGetErrorString(e));
    }
    return FSDP_OK;
}

void dev_free(fsdp_unit* u, void* p) {
    if (p == nullptr) return;
    if (u->allocator.alloc != nullptr) u->allocator.free(p, u->allocator.ctx);
    else cudaFree(p);
}

void free_unit(fsdp_unit* u) {
    for (void* p : {static_cast<void*>(u->master), static_cast<void*>(u->grad),
                    static_cast<void*>(u->m), static_cast<void*>(u->v),
                    static_cast<void*>(u->shadow), static_cast<void*>(u->tiles),
                    static_cast<void*>(u->load_tiles), static_cast<void*>(u->param_src),
                    static_cast<void*>(u->step_table), static_cast<void*>(u->step_counter),
                    static_cast<void*>(u->step_status), static_cast<void*>(u->kstatus)}) {
        dev_free(u, p);
    }
    for (auto& r : u->prof) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    u->prof.clear();
}

// Launch `fn` bracketed by profiler events when profiling is on.
template <typename F>
int profiled_launch(fsdp_unit* u, int kind, cudaStream_t st, const char* what, F&& fn) {
    ProfRecord rec{kind, nullptr, nullptr};
    bool timed = u->profiling;
    if (timed) {   // launches recorded into a CUDA graph are not timed
        cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
        if (cudaStreamIsCapturing(st, &cs) != cudaSuccess || cs != cudaStreamCaptureStatusNone) {
            cudaGetLastError();
            timed = false;
        }
    }
    if (timed) {
        if (cudaEventCreate(&rec.start) != cudaSuccess) return fail(FSDP_E_CUDA, "cudaEventCreate failed");
        if (cudaEventCreate(&rec.stop) != cudaSuccess) {
            cudaEventDestroy(rec.start);
            return fail(FSDP_E_CUDA, "cudaEventCreate failed");
        }
        cudaEventRecord(rec.start, st);
    }
    cudaError_t e = fn();
    if (e != cudaSuccess) {
        if (rec.start) cudaEventDestroy(rec.start);
        if (rec.stop) cudaEventDestroy(rec.stop);
        return cuda_fail(e, what);
    }
    if (timed) {
        cudaEventRecord(rec.stop, st);
        u->prof.push_back(rec);
    }
    return FSDP_OK;
}

float* state_f32(const fsdp_unit* u, int which) {
    switch (which) {
        case FSDP_STATE_PARAM: return u->master;
        case FSDP_STATE_GRAD: return u->grad;
        case FSDP_STATE_EXP_AVG: return u->m;
        case FSDP_STATE_EXP_AVG_SQ: return u->v;
        default: return nullptr;
    }
}

// base pointer and element size of a state, or nullptr for a bad `which`
char* state_base(const fsdp_unit* u, int which, size_t* esz) {
    if (which == FSDP_STATE_SHADOW) {
        *esz = 2;
        return reinterpret_cast<char*>(u->shadow);
    }
    *esz = 4;
    return reinterpret_cast<char*>(state_f32(u, which));
}

int check_unit(const fsdp_unit* u, bool need_loaded) {
    if (u == nullptr) return fail(FSDP_E_INVALID_ARG, "unit is null");
    if (need_loaded && !u->loaded) return fail(FSDP_E_STATE, "fsdp_load_params has not been called");
    return FSDP_OK;
}

int check_hp(const fsdp_adamw_hp* hp) {
    if (hp == nullptr) return fail(FSDP_E_INVALID_ARG, "hp is null");
    auto fin = [](double x) { return std::isfinite(x); };
    if (!fin(hp->lr) || !fin(hp->beta1) || !fin(hp->beta2) || !fin(hp->eps) || !fin(hp->weight_decay))
        return fail(FSDP_E_INVALID_ARG, "AdamW hyper-parameters must be finite");
    if (hp->lr < 0 || hp->eps < 0 || hp->weight_decay < 0)
        return fail(FSDP_E_INVALID_ARG, "lr, eps and weight_decay must be >= 0");
    if (!(hp->beta1 >= 0 && hp->beta1 < 1) || !(hp->beta2 >= 0 && hp->beta2 < 1))
        return fail(FSDP_E_INVALID_ARG, "betas must be in [0, 1)");
    return FSDP_OK;
}

// Gradient buffers must be 16-byte aligned; *narrow is set when one of them
// is not 32-byte aligned (the kernels then use 16-byte loads).
int check_grads(const fsdp_unit* u, const void* const* grads, int* narrow) {
    if (grads == nullptr) return fail(FSDP_E_INVALID_ARG, "grads array is null");
    *narrow = 0;
    for (int r = 0; r < u->plan.N * u->replicas; ++r) {
        if (grads[r] == nullptr) return fail(FSDP_E_INVALID_ARG, "a gradient pointer is null");
        if (!aligned16(grads[r])) return fail(FSDP_E_ALIGN, "a gradient buffer is not 16-byte aligned");
        if (!aligned32(grads[r])) *narrow = 1;
    }
    return FSDP_OK;
}

// The gathered output is written in 16-byte groups at 8-element boundaries.
int check_out(const uint16_t* out) {
    if (out == nullptr) return fail(FSDP_E_INVALID_ARG, "output buffer is null");
    if (!aligned16(out)) return fail(FSDP_E_ALIGN, "output buffer is not 16-byte aligned");
    return FSDP_OK;
}

// Hot-path calls are refused after a kernel gave up (see fsdp_kernel_status).
int check_usable(const fsdp_unit* u) {
    if (u->broken)
        return fail(FSDP_E_STATE, "a kernel's copies may have landed after it ended (FSDP_KSTATUS_DRAIN_TIMEOUT); "
                                  "destroy the unit");
    if (u->needs_reload)
        return fail(FSDP_E_STATE, "a kernel gave up waiting (FSDP_KSTATUS_WAIT_TIMEOUT) and left the state "
                                  "incomplete; reload it with fsdp_load_params");
    return FSDP_OK;
}

// The staged kernels' wait bound and the one-shot give-up test, into `a`.
void wait_args(fsdp_unit* u, fsdp::ReduceArgs* a) {
    a->wait_ns = u->wait_ns;
    a->withhold = u->withhold_next;
    u->withhold_next = 0;
}

fsdp::AdamWConsts adamw_consts(const fsdp_adamw_hp* hp, int64_t t) {
    const double bc1 = 1.0 - std::pow(hp->beta1, static_cast<double>(t));
    const double bc2 = 1.0 - std::pow(hp->beta2, static_cast<double>(t));
    fsdp::AdamWConsts c;
    c.decay = static_cast<float>(1.0 - hp->lr * hp->weight_decay);
    c.b1 = static_cast<float>(hp->beta1);
    c.c1 = static_cast<float>(1.0 - hp->beta1);
    c.b2 = static_cast<float>(hp->beta2);
    c.c2 = static_cast<float>(1.0 - hp->beta2);
    c.bc2 = static_cast<float>(bc2);
    c.step = static_cast<float>(hp->lr / bc1);
    c.eps = static_cast<float>(hp->eps);
    return c;
}

// Recompute the whole shadow slab from the master if AdamW left it stale.
int ensure_shadow(const fsdp_unit* u, cudaStream_t st) {
    if (u->shadow_valid) return FSDP_OK;
    cudaError_t e = fsdp::launch_cast_range(u->master, u->shadow, 0, u->plan.slab_len, st);
    if (e != cudaSuccess) return cuda_fail(e, "shadow refresh");
    u->shadow_valid = true;
    return FSDP_OK;
}

fsdp::StepSource step_source(const fsdp_unit* u, const fsdp_adamw_hp* hp) {
    fsdp::StepSource s{};
    s.write_shadow = u->gather_source == FSDP_GATHER_FROM_SHADOW ? 1 : 0;
    if (u->device_steps) {
        s.table = u->step_table;
        s.counter = u->step_counter;
        s.count = u->step_count;
        s.status = u->step_status;
    } else {
        s.c = adamw_consts(hp, u->t + 1);
    }
    return s;
}

// After an AdamW launch in device-step mode: advance the device counter.
int advance_device_step(fsdp_unit* u, cudaStream_t st) {
    if (!u->device_steps) return FSDP_OK;
    cudaError_t e = fsdp::launch_advance_step(u->step_counter, u->step_count, st);
    return e == cudaSuccess ? FSDP_OK : cuda_fail(e, "step-counter launch");
}

// overlap: the stream's previous kernel is this step's first gather, which
// writes the same bytes to `out` and touches nothing else this one does.
int enqueue_gather(fsdp_unit* u, uint16_t* out, cudaStream_t st, bool overlap = false) {
    if (u->gather_source == FSDP_GATHER_FROM_SHADOW) {
        int rc = ensure_shadow(u, st);
        if (rc) return rc;
    }
    return profiled_launch(u, FSDP_KERNEL_GATHER, st, "gather launch", [&] {
        if (u->gather_source == FSDP_GATHER_FROM_SHADOW)
            return fsdp::launch_gather_shadow(u->tiles, u->ntiles, u->shadow, out, st, overlap);
        return fsdp::launch_gather(u->tiles, u->ntiles, u->master, out, st, overlap);
    });
}

int check_rs_options(const fsdp_rs_options* opt) {
    if (opt == nullptr) return FSDP_OK;
    if (!std::isfinite(opt->inv_scale) || opt->inv_scale < 0)
        return fail(FSDP_E_INVALID_ARG, "inv_scale must be finite and >= 0");
    if (opt->found_nonfinite_dev != nullptr && (reinterpret_cast<uintptr_t>(opt->found_nonfinite_dev) & 3u))
        return fail(FSDP_E_ALIGN, "found_nonfinite_dev is not 4-byte aligned");
    return FSDP_OK;
}

// overlap: the stream's previous kernels are this step's gathers, which touch
// neither the gradients nor the gradient shard (only the register-staged
// kernels take it; the shared-memory staged ones wait at their start).
int enqueue_reduce_scatter(fsdp_unit* u, const void* const* grads, int narrow, const fsdp_rs_options* opt,
                           cudaStream_t st, bool overlap = false) {
    fsdp::ReduceArgs a{};
    a.overlap = overlap ? 1 : 0;
    a.F = u->plan.N;
    a.groups = u->replicas;
    a.bf16_reduce = u->reduce_dtype == FSDP_DTYPE_BF16 ? 1 : 0;
    a.inv_scale = 1.0f;
    a.narrow = narrow;
    wait_args(u, &a);
    if (opt != nullptr) {
        if (opt->inv_scale != 0.0 && opt->inv_scale != 1.0) {
            a.scale = 1;
            a.inv_scale = static_cast<float>(opt->inv_scale);
        }
        a.accumulate = opt->accumulate ? 1 : 0;
        a.found = opt->found_nonfinite_dev;
        if (a.found != nullptr) {
            cudaError_t e = cudaMemsetAsync(a.found, 0, sizeof(int32_t), st);
            if (e != cudaSuccess) return cuda_fail(e, "clearing the found-non-finite flag");
        }
    }
    return profiled_launch(u, FSDP_KERNEL_REDUCE_SCATTER, st, "reduce-scatter launch", [&] {
        return fsdp::launch_reduce_scatter(u->tiles, u->ntiles, grads, u->grad_dtype, a, u->grad, u->kstatus, st);
    });
}

int enqueue_reduce_adamw(fsdp_unit* u, const void* const* grads, int narrow, const fsdp_adamw_hp* hp,
                         cudaStream_t st) {
    fsdp::ReduceArgs a{};
    a.F = u->plan.N;
    a.groups = u->replicas;
    a.bf16_reduce = u->reduce_dtype == FSDP_DTYPE_BF16 ? 1 : 0;
    a.inv_scale = 1.0f;
    a.narrow = narrow;
    wait_args(u, &a);
    const fsdp::StepSource c = step_source(u, hp);
    // a step that is skipped on the device (used-up step table) leaves the
    // shadow as it was, so a stale one is refreshed before a storing launch
    int rc = c.write_shadow ? ensure_shadow(u, st) : FSDP_OK;
    if (rc == FSDP_OK)
        rc = profiled_launch(u, FSDP_KERNEL_REDUCE_ADAMW, st, "fused reduce-scatter + AdamW launch", [&] {
            return fsdp::launch_reduce_adamw(u->tiles, u->ntiles, grads, u->grad_dtype, a, u->grad, u->master,
                                             u->m, u->v, u->shadow, c, u->kstatus, st);
        });
    if (rc == FSDP_OK) u->shadow_valid = c.write_shadow != 0;
    if (rc == FSDP_OK) rc = advance_device_step(u, st);
    if (rc == FSDP_OK) u->t += 1;
    return rc;
}

int enqueue_adamw(fsdp_unit* u, const fsdp_adamw_hp* hp, cudaStream_t st) {
    const fsdp::StepSource c = step_source(u, hp);
    int rc = c.write_shadow ? ensure_shadow(u, st) : FSDP_OK;
    if (rc == FSDP_OK)
        rc = profiled_launch(u, FSDP_KERNEL_ADAMW, st, "AdamW launch", [&] {
            return fsdp::launch_adamw(u->plan.slab_len / 8, u->master, u->grad, u->m, u->v, u->shadow, c, st);
        });
    if (rc == FSDP_OK) u->shadow_valid = c.write_shadow != 0;
    if (rc == FSDP_OK) rc = advance_device_step(u, st);
    if (rc == FSDP_OK) u->t += 1;
    return rc;
}

}  // namespace

extern "C" {

const char* fsdp_strerror(int code) {
    switch (code) {
        case FSDP_OK: return "ok";
        case FSDP_E_INVALID_ARG: return "invalid argument";
        case FSDP_E_OOM: return "out of memory";
        case FSDP_E_CUDA: return "CUDA error";
        case FSDP_E_STATE: return "invalid state";
        case FSDP_E_ALIGN: return "misaligned buffer";
        case FSDP_E_CAPACITY: return "output array too small";
        default: return "unknown error";
    }
}

const char* fsdp_last_error(void) { return g_last_error.c_str(); }

int fsdp_kernel_status(fsdp_unit* u, int32_t* flags, void* stream) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (flags == nullptr) return fail(FSDP_E_INVALID_ARG, "flags is null");
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, u->kstatus, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(u->kstatus, 0, sizeof(int32_t), st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the kernel status word");
    *flags = v;
    if (v & FSDP_KSTATUS_WAIT_TIMEOUT) u->needs_reload = true;
    if (v & FSDP_KSTATUS_DRAIN_TIMEOUT) u->broken = true;
    return FSDP_OK;
}

int fsdp_unit_set_wait_limit(fsdp_unit* u, double seconds, int withhold_next) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (!(seconds >= 1e-6 && seconds <= 60.0)) return fail(FSDP_E_INVALID_ARG, "seconds must be in [1e-6, 60]");
    if (withhold_next < 0 || withhold_next > 2) return fail(FSDP_E_INVALID_ARG, "withhold_next must be 0, 1 or 2");
    u->wait_ns = static_cast<unsigned long long>(seconds * 1e9);
    u->withhold_next = withhold_next;
    return FSDP_OK;
}

int fsdp_selftest_bounded_wait(double limit_seconds, int32_t* timed_out, void* stream) {
    if (timed_out == nullptr) return fail(FSDP_E_INVALID_ARG, "timed_out is null");
    if (!(limit_seconds >= 1e-3 && limit_seconds <= 10.0))
        return fail(FSDP_E_INVALID_ARG, "limit_seconds must be in [1e-3, 10]");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int32_t* word = nullptr;
    cudaError_t e = cudaMalloc(reinterpret_cast<void**>(&word), sizeof(int32_t));
    if (e != cudaSuccess) return cuda_fail(e, "self-test status word");
    int32_t v = 0;
    e = cudaMemsetAsync(word, 0, sizeof(int32_t), st);
    if (e == cudaSuccess)
        e = fsdp::launch_wait_selftest(word, static_cast<unsigned long long>(limit_seconds * 1e9), st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&v, word, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(word);
    if (e != cudaSuccess) return cuda_fail(e, "bounded-wait self-test");
    *timed_out = (v & FSDP_KSTATUS_WAIT_TIMEOUT) ? 1 : 0;
    return FSDP_OK;
}

int fsdp_host_device_pointer(const void* host, void** dev) {
    if (host == nullptr || dev == nullptr) return fail(FSDP_E_INVALID_ARG, "host/dev is null");
    *dev = nullptr;
    cudaPointerAttributes attr;
    cudaError_t e = cudaPointerGetAttributes(&attr, host);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeHost) {
        cudaGetLastError();
        return fail(FSDP_E_INVALID_ARG, "not pinned host memory known to CUDA");
    }
    void* d = nullptr;
    e = cudaHostGetDevicePointer(&d, const_cast<void*>(host), 0);
    if (e != cudaSuccess || d == nullptr) {
        cudaGetLastError();
        return fail(FSDP_E_INVALID_ARG, std::string("no device mapping: ") + cudaGetErrorString(e));
    }
    *dev = d;
    return FSDP_OK;
}

int fsdp_plan_layout(int nparams, const int* ndims, const int64_t* dims, int layout, int num_ranks,
                     int64_t* numel, int64_t* nsegs, fsdp_segment* segs, int64_t cap) {
    Plan plan;
    std::string err;
    int rc = fsdp::build_plan(nparams, ndims, dims, layout, num_ranks, &plan, &err);
    if (rc != FSDP_OK) return fail(rc, err);
    const int64_t n = static_cast<int64_t>(plan.segs.size());
    if (numel) *numel = plan.P;
    if (nsegs) *nsegs = n;
    if (segs) {
        if (cap < n) return fail(FSDP_E_CAPACITY, "segment array too small");
        std::memcpy(segs, plan.segs.data(), sizeof(fsdp_segment) * static_cast<size_t>(n));
    }
    return FSDP_OK;
}

int fsdp_unit_create(int nparams, const int* ndims, const int64_t* dims,
                     const fsdp_unit_config* cfg, fsdp_unit** out) {
    return fsdp_unit_create_with_allocator(nparams, ndims, dims, cfg, nullptr, out);
}

int fsdp_unit_create_with_allocator(int nparams, const int* ndims, const int64_t* dims,
                                    const fsdp_unit_config* cfg, const fsdp_allocator* alloc,
                                    fsdp_unit** out) {
    if (out == nullptr || cfg == nullptr) return fail(FSDP_E_INVALID_ARG, "cfg/out is null");
    *out = nullptr;
    if (alloc != nullptr && (alloc->alloc == nullptr || alloc->free == nullptr))
        return fail(FSDP_E_INVALID_ARG, "an allocator needs both alloc and free");
    if (cfg->grad_dtype != FSDP_DTYPE_F32 && cfg->grad_dtype != FSDP_DTYPE_BF16)
        return fail(FSDP_E_INVALID_ARG, "grad_dtype must be FSDP_DTYPE_F32 or FSDP_DTYPE_BF16");
    if (cfg->reduce_dtype != FSDP_DTYPE_F32 && cfg->reduce_dtype != FSDP_DTYPE_BF16)
        return fail(FSDP_E_INVALID_ARG, "reduce_dtype must be FSDP_DTYPE_F32 or FSDP_DTYPE_BF16");
    if (cfg->gather_source != FSDP_GATHER_FROM_MASTER && cfg->gather_source != FSDP_GATHER_FROM_SHADOW)
        return fail(FSDP_E_INVALID_ARG, "gather_source must be FSDP_GATHER_FROM_MASTER or _FROM_SHADOW");
    if (cfg->num_ranks < 1 || cfg->num_ranks > fsdp::kMaxRanks)
        return fail(FSDP_E_INVALID_ARG, "num_ranks must be in [1, 1024]");
    const int replicas = cfg->replicas == 0 ? 1 : cfg->replicas;
    if (replicas < 1 || replicas > fsdp::kMaxRanks / cfg->num_ranks)
        return fail(FSDP_E_INVALID_ARG, "replicas must be >= 1 with num_ranks * replicas <= 1024");
    if (replicas > 1 && cfg->reduce_dtype == FSDP_DTYPE_BF16)
        return fail(FSDP_E_INVALID_ARG, "bf16 reduction is supported with replicas == 1 only");
    Plan plan;
    std::string err;
    int rc = fsdp::build_plan(nparams, ndims, dims, cfg->layout, cfg->num_ranks, &plan, &err);
    if (rc != FSDP_OK) return fail(rc, err);

    fsdp_unit* u = new (std::nothrow) fsdp_unit;
    if (u == nullptr) return fail(FSDP_E_OOM, "host allocation failed");
    if (cudaGetDevice(&u->device) != cudaSuccess) {
        delete u;
        return fail(FSDP_E_CUDA, "no CUDA device");
    }
    u->plan = std::move(plan);
    u->nparams = nparams;
    u->grad_dtype = cfg->grad_dtype;
    u->raf = cfg->reshard_after_forward ? 1 : 0;
    u->replicas = replicas;
    u->reduce_dtype = cfg->reduce_dtype;
    u->gather_source = cfg->gather_source;
    u->fuse = cfg->fuse_reduce_adamw ? 1 : 0;
    if (alloc != nullptr) u->allocator = *alloc;

    std::vector<Tile> tiles, load_tiles;
    fsdp::build_tiles(u->plan, &tiles);
    fsdp::build_load_tiles(u->plan, &load_tiles);
    u->ntiles = static_cast<int64_t>(tiles.size());
    u->nload_tiles = static_cast<int64_t>(load_tiles.size());

    const size_t S = static_cast<size_t>(u->plan.slab_len);
    struct Alloc {
        void** p;
        size_t bytes;
    } allocs[] = {
        {reinterpret_cast<void**>(&u->master), S * 4},
        {reinterpret_cast<void**>(&u->grad), S * 4},
        {reinterpret_cast<void**>(&u->m), S * 4},
        {reinterpret_cast<void**>(&u->v), S * 4},
        {reinterpret_cast<void**>(&u->shadow), S * 2},
        {reinterpret_cast<void**>(&u->tiles), tiles.size() * sizeof(Tile)},
        {reinterpret_cast<void**>(&u->load_tiles), load_tiles.size() * sizeof(Tile)},
        {reinterpret_cast<void**>(&u->param_src), static_cast<size_t>(nparams) * sizeof(fsdp::ParamSrc)},
        {reinterpret_cast<void**>(&u->kstatus), 32},
    };
    for (auto& a : allocs) {
        rc = dev_alloc(u, a.p, a.bytes);
        if (rc != FSDP_OK) {   // the reason is already recorded
            free_unit(u);
            delete u;
            return rc;
        }
    }
    cudaError_t e = cudaSuccess;
    for (int i = 0; i < 5 && e == cudaSuccess; ++i) e = cudaMemset(*allocs[i].p, 0, allocs[i].bytes);
    if (e == cudaSuccess) e = cudaMemset(u->kstatus, 0, 32);
    if (e == cudaSuccess && !tiles.empty())
        e = cudaMemcpy(u->tiles, tiles.data(), tiles.size() * sizeof(Tile), cudaMemcpyHostToDevice);
    if (e == cudaSuccess && !load_tiles.empty())
        e = cudaMemcpy(u->load_tiles, load_tiles.data(), load_tiles.size() * sizeof(Tile),
                       cudaMemcpyHostToDevice);
    if (e != cudaSuccess) {
        free_unit(u);
        delete u;
        return cuda_fail(e, "unit set-up");
    }
    *out = u;
    return FSDP_OK;
}

int fsdp_unit_destroy(fsdp_unit* u) {
    if (u == nullptr) return FSDP_OK;
    DeviceGuard dg(u->device);
    cudaDeviceSynchronize();
    free_unit(u);
    delete u;
    return FSDP_OK;
}

int fsdp_load_params(fsdp_unit* u, const float* const* params, void* stream) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (u->broken) return check_usable(u);
    if (params == nullptr) return fail(FSDP_E_INVALID_ARG, "params array is null");
    std::vector<fsdp::ParamSrc> src(u->nparams);
    for (int p = 0; p < u->nparams; ++p) {
        const fsdp::ParamInfo& pi = u->plan.params[p];
        if (pi.numel > 0 && params[p] == nullptr)
            return fail(FSDP_E_INVALID_ARG, "a parameter pointer is null");
        if ((reinterpret_cast<uintptr_t>(params[p]) & 3u) != 0)
            return fail(FSDP_E_ALIGN, "a parameter buffer is not 4-byte aligned");
        src[p] = fsdp::ParamSrc{params[p], pi.offset};
    }
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t S = static_cast<size_t>(u->plan.slab_len);
    cudaError_t e = cudaMemcpyAsync(u->param_src, src.data(), src.size() * sizeof(fsdp::ParamSrc),
                                    cudaMemcpyHostToDevice, st);
    // pageable source: the copy has been staged when cudaMemcpyAsync returns
    if (e == cudaSuccess) e = cudaMemsetAsync(u->master, 0, S * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(u->grad, 0, S * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(u->m, 0, S * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(u->v, 0, S * 4, st);
    if (e == cudaSuccess) e = cudaMemsetAsync(u->shadow, 0, S * 2, st);
    if (e != cudaSuccess) return cuda_fail(e, "load set-up");
    rc = profiled_launch(u, FSDP_KERNEL_SHARD_IN, st, "shard-in launch", [&] {
        return fsdp::launch_shard_in(u->load_tiles, u->nload_tiles, u->param_src, u->master, u->shadow, st);
    });
    if (rc) return rc;
    u->t = 0;
    u->device_steps = false;
    u->loaded = true;
    u->needs_reload = false;
    u->shadow_valid = true;   // shard-in writes RNE(master)
    return FSDP_OK;
}

int fsdp_allgather(fsdp_unit* u, uint16_t* out, void* stream) {
    int rc = check_unit(u, true);
    if (rc == FSDP_OK) rc = check_usable(u);
    if (rc == FSDP_OK) rc = check_out(out);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    return enqueue_gather(u, out, static_cast<cudaStream_t>(stream));
}

int fsdp_reduce_scatter(fsdp_unit* u, const void* const* grads, void* stream) {
    int narrow = 0;
    int rc = check_unit(u, true);
    if (rc == FSDP_OK) rc = check_usable(u);
    if (rc == FSDP_OK) rc = check_grads(u, grads, &narrow);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    return enqueue_reduce_scatter(u, grads, narrow, nullptr, static_cast<cudaStream_t>(stream));
}

int fsdp_reduce_scatter_ex(fsdp_unit* u, const void* const* grads, const fsdp_rs_options* opt,
                           void* stream) {
    int narrow = 0;
    int rc = check_unit(u, true);
    if (rc == FSDP_OK) rc = check_usable(u);
    if (rc == FSDP_OK) rc = check_grads(u, grads, &narrow);
    if (rc == FSDP_OK) rc = check_rs_options(opt);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    return enqueue_reduce_scatter(u, grads, narrow, opt, static_cast<cudaStream_t>(stream));
}

int fsdp_zero_grad(fsdp_unit* u, void* stream) {
    int rc = check_unit(u, true);
    if (rc == FSDP_OK) rc = check_usable(u);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaError_t e = cudaMemsetAsync(u->grad, 0, static_cast<size_t>(u->plan.slab_len) * 4,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FSDP_OK : cuda_fail(e, "zeroing the gradient shards");
}

int fsdp_adamw_step(fsdp_unit* u, const fsdp_adamw_hp* hp, void* stream) {
    int rc = check_unit(u, true);
    if (rc == FSDP_OK) rc = check_usable(u);
    if (rc == FSDP_OK) rc = check_hp(hp);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    return enqueue_adamw(u, hp, static_cast<cudaStream_t>(stream));
}

int fsdp_step(fsdp_unit* u, const void* const* grads, uint16_t* out, const fsdp_adamw_hp* hp,
              void* stream) {
    int narrow = 0;
    int rc = check_unit(u, true);
    if (rc == FSDP_OK) rc = check_usable(u);
    if (rc == FSDP_OK) rc = check_out(out);
    if (rc == FSDP_OK) rc = check_grads(u, grads, &narrow);
    if (rc == FSDP_OK) rc = check_hp(hp);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the first gather waits for everything before it in the stream; the
    // second gather and the reduce-scatter may start beside the kernel before
    // them (each completes after it), and AdamW waits for all three
    rc = enqueue_gather(u, out, st);                       // forward
    if (rc == FSDP_OK && u->raf) rc = enqueue_gather(u, out, st, true);   // backward re-gather
    if (rc == FSDP_OK && u->fuse) return enqueue_reduce_adamw(u, grads, narrow, hp, st);
    if (rc == FSDP_OK) rc = enqueue_reduce_scatter(u, grads, narrow, nullptr, st, true);
    if (rc == FSDP_OK) rc = enqueue_adamw(u, hp, st);
    return rc;
}

static int copy_state(const fsdp_unit* u, int which, int rank, void* ext, bool to_unit, void* stream) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (rank < 0 || rank >= u->plan.N) return fail(FSDP_E_INVALID_ARG, "rank out of range");
    size_t esz = 0;
    char* base = state_base(u, which, &esz);
    if (base == nullptr) return fail(FSDP_E_INVALID_ARG, "unknown state");
    if (ext == nullptr && u->plan.shard_len[rank] > 0) return fail(FSDP_E_INVALID_ARG, "buffer is null");
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (which == FSDP_STATE_SHADOW) {   // read: refresh a stale shadow; write: start from a fresh one
        rc = ensure_shadow(u, st);
        if (rc) return rc;
    }
    const int64_t abase = u->plan.arena_base[rank];
    for (int64_t i = u->plan.rank_first_seg[rank]; i < u->plan.rank_first_seg[rank + 1]; ++i) {
        const fsdp_segment& s = u->plan.segs[i];
        char* dev = base + static_cast<size_t>(abase + s.arena_off) * esz;
        char* host = static_cast<char*>(ext) + static_cast<size_t>(s.shard_off) * esz;
        cudaError_t e = to_unit ? cudaMemcpyAsync(dev, host, s.len * esz, cudaMemcpyDefault, st)
                                : cudaMemcpyAsync(host, dev, s.len * esz, cudaMemcpyDefault, st);
        if (e != cudaSuccess) return cuda_fail(e, "state copy");
    }
    if (to_unit && which == FSDP_STATE_PARAM) {   // keep shadow == RNE(master)
        cudaError_t e = fsdp::launch_cast_range(u->master, u->shadow, abase, u->plan.arena_len[rank], st);
        if (e != cudaSuccess) return cuda_fail(e, "shadow refresh");
    }
    return FSDP_OK;
}

int fsdp_get_state(const fsdp_unit* u, int which, int rank, void* dst, void* stream) {
    return copy_state(u, which, rank, dst, false, stream);
}

int fsdp_set_state(fsdp_unit* u, int which, int rank, const void* src, void* stream) {
    return copy_state(u, which, rank, const_cast<void*>(src), true, stream);
}

int fsdp_read_global(const fsdp_unit* u, int which, int64_t begin, int64_t count, void* dst,
                     void* stream) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (begin < 0 || count < 0 || begin + count > u->plan.P)
        return fail(FSDP_E_INVALID_ARG, "range outside the unit");
    size_t esz = 0;
    char* base = state_base(u, which, &esz);
    if (base == nullptr) return fail(FSDP_E_INVALID_ARG, "unknown state");
    if (count > 0 && dst == nullptr) return fail(FSDP_E_INVALID_ARG, "dst is null");
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (which == FSDP_STATE_SHADOW) {
        rc = ensure_shadow(u, st);
        if (rc) return rc;
    }
    const int64_t end = begin + count;
    for (const fsdp_segment& s : u->plan.segs) {
        const int64_t a = s.global_off > begin ? s.global_off : begin;
        const int64_t b = s.global_off + s.len < end ? s.global_off + s.len : end;
        if (b <= a) continue;
        const int64_t slab = u->plan.arena_base[s.rank] + s.arena_off + (a - s.global_off);
        cudaError_t e = cudaMemcpyAsync(static_cast<char*>(dst) + static_cast<size_t>(a - begin) * esz,
                                        base + static_cast<size_t>(slab) * esz,
                                        static_cast<size_t>(b - a) * esz, cudaMemcpyDefault, st);
        if (e != cudaSuccess) return cuda_fail(e, "state copy");
    }
    return FSDP_OK;
}

int fsdp_read_arena(const fsdp_unit* u, int which, int rank, void* dst, int64_t* arena_len, void* stream) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (rank < 0 || rank >= u->plan.N) return fail(FSDP_E_INVALID_ARG, "rank out of range");
    size_t esz = 0;
    char* base = state_base(u, which, &esz);
    if (base == nullptr) return fail(FSDP_E_INVALID_ARG, "unknown state");
    const int64_t n = u->plan.arena_len[rank];
    if (arena_len) *arena_len = n;
    if (dst == nullptr) return FSDP_OK;   // size query
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    if (which == FSDP_STATE_SHADOW) {
        rc = ensure_shadow(u, static_cast<cudaStream_t>(stream));
        if (rc) return rc;
    }
    cudaError_t e = cudaMemcpyAsync(dst, base + static_cast<size_t>(u->plan.arena_base[rank]) * esz,
                                    static_cast<size_t>(n) * esz, cudaMemcpyDefault,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? FSDP_OK : cuda_fail(e, "arena copy");
}

int fsdp_get_step_count(const fsdp_unit* u, int64_t* t) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (t == nullptr) return fail(FSDP_E_INVALID_ARG, "t is null");
    *t = u->t;
    return FSDP_OK;
}

int fsdp_set_step_count(fsdp_unit* u, int64_t t) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (t < 0) return fail(FSDP_E_INVALID_ARG, "step count must be >= 0");
    if (u->device_steps) return fail(FSDP_E_STATE, "device-step mode is on; turn it off first");
    u->t = t;
    return FSDP_OK;
}

int fsdp_unit_set_step_options(fsdp_unit* u, int gather_source, int fuse_reduce_adamw) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (gather_source != FSDP_GATHER_FROM_MASTER && gather_source != FSDP_GATHER_FROM_SHADOW)
        return fail(FSDP_E_INVALID_ARG, "gather_source must be FSDP_GATHER_FROM_MASTER or _FROM_SHADOW");
    u->gather_source = gather_source;
    u->fuse = fuse_reduce_adamw ? 1 : 0;
    return FSDP_OK;
}

int fsdp_adamw_device_steps(fsdp_unit* u, const fsdp_adamw_hp* hp, int64_t count, void* stream) {
    int rc = check_unit(u, true);
    if (rc) return rc;
    if (count < 0) return fail(FSDP_E_INVALID_ARG, "count must be >= 0");
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (count == 0) {   // leave the mode; the host step count takes the device's
        if (u->device_steps) {
            int64_t taken = 0;
            cudaError_t e = cudaMemcpyAsync(&taken, u->step_counter, sizeof(int64_t), cudaMemcpyDeviceToHost, st);
            if (e == cudaSuccess) e = cudaStreamSynchronize(st);
            if (e != cudaSuccess) return cuda_fail(e, "reading the device step counter");
            u->t = u->step_base + taken;
            u->device_steps = false;
        }
        return FSDP_OK;
    }
    rc = check_hp(hp);
    if (rc) return rc;
    if (count > (int64_t(1) << 24)) return fail(FSDP_E_INVALID_ARG, "count must be <= 2^24 steps");
    if (u->device_steps) {
        rc = fsdp_adamw_device_steps(u, nullptr, 0, stream);   // fold in the steps taken so far
        if (rc) return rc;
    }
    std::vector<fsdp::AdamWConsts> table(static_cast<size_t>(count));
    for (int64_t i = 0; i < count; ++i) table[static_cast<size_t>(i)] = adamw_consts(hp, u->t + 1 + i);
    if (u->step_counter == nullptr) {
        rc = dev_alloc(u, reinterpret_cast<void**>(&u->step_counter), 64);
        if (rc) return rc;
    }
    if (u->step_status == nullptr) {
        rc = dev_alloc(u, reinterpret_cast<void**>(&u->step_status), 64);
        if (rc) return rc;
    }
    if (u->step_table_cap < count) {
        cudaStreamSynchronize(st);   // the old table may still be in use
        dev_free(u, u->step_table);
        u->step_table = nullptr;
        u->step_table_cap = 0;
        rc = dev_alloc(u, reinterpret_cast<void**>(&u->step_table), sizeof(fsdp::AdamWConsts) * static_cast<size_t>(count));
        if (rc) return rc;
        u->step_table_cap = count;
    }
    cudaError_t e = cudaSuccess;
    if (e == cudaSuccess)
        e = cudaMemcpyAsync(u->step_table, table.data(), sizeof(fsdp::AdamWConsts) * table.size(),
                            cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);   // `table` is a host temporary
    if (e == cudaSuccess) e = cudaMemsetAsync(u->step_counter, 0, sizeof(int64_t), st);
    if (e == cudaSuccess) e = cudaMemsetAsync(u->step_status, 0, sizeof(int32_t), st);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return fail(e == cudaErrorMemoryAllocation ? FSDP_E_OOM : FSDP_E_CUDA,
                    std::string("device-step set-up: ") + cudaGetErrorString(e));
    }
    u->step_count = count;
    u->step_base = u->t;
    u->device_steps = true;
    return FSDP_OK;
}

int fsdp_adamw_device_status(fsdp_unit* u, int64_t* step, int32_t* exhausted, void* stream) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (!u->device_steps) {
        if (step) *step = u->t;
        if (exhausted) *exhausted = 0;
        return FSDP_OK;
    }
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int64_t taken = 0;
    int32_t status = 0;
    cudaError_t e = cudaMemcpyAsync(&taken, u->step_counter, sizeof(int64_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaMemcpyAsync(&status, u->step_status, sizeof(int32_t), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device step counter");
    if (step) *step = u->step_base + taken;
    if (exhausted) *exhausted = status;
    return FSDP_OK;
}

int fsdp_unit_info(const fsdp_unit* u, int64_t* numel, fsdp_unit_config* cfg) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (numel) *numel = u->plan.P;
    if (cfg) {
        cfg->layout = u->plan.layout;
        cfg->num_ranks = u->plan.N;
        cfg->grad_dtype = u->grad_dtype;
        cfg->reshard_after_forward = u->raf;
        cfg->replicas = u->replicas;
        cfg->reduce_dtype = u->reduce_dtype;
        cfg->gather_source = u->gather_source;
        cfg->fuse_reduce_adamw = u->fuse;
    }
    return FSDP_OK;
}

int fsdp_unit_segments(const fsdp_unit* u, fsdp_segment* segs, int64_t cap, int64_t* nsegs) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    const int64_t n = static_cast<int64_t>(u->plan.segs.size());
    if (nsegs) *nsegs = n;
    if (segs) {
        if (cap < n) return fail(FSDP_E_CAPACITY, "segment array too small");
        std::memcpy(segs, u->plan.segs.data(), sizeof(fsdp_segment) * static_cast<size_t>(n));
    }
    return FSDP_OK;
}

int fsdp_memory_report(const fsdp_unit* u, int rank, int64_t* param_bytes, int64_t* grad_bytes,
                       int64_t* adam_bytes, int64_t* shadow_bytes, int64_t* pad_bytes) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (rank < 0 || rank >= u->plan.N) return fail(FSDP_E_INVALID_ARG, "rank out of range");
    const int64_t n = u->plan.shard_len[rank];
    const int64_t pads = u->plan.arena_len[rank] - n;
    if (param_bytes) *param_bytes = 4 * n;
    if (grad_bytes) *grad_bytes = 4 * n;
    if (adam_bytes) *adam_bytes = 8 * n;
    if (shadow_bytes) *shadow_bytes = 2 * n;
    if (pad_bytes) *pad_bytes = pads * (4 + 4 + 8 + 2);
    return FSDP_OK;
}

int fsdp_profile_enable(fsdp_unit* u, int on) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    u->profiling = on != 0;
    return FSDP_OK;
}

int fsdp_profile_read(fsdp_unit* u, int kernel, double* total_ms, int64_t* launches) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    if (kernel < 0 || kernel >= FSDP_KERNEL_COUNT) return fail(FSDP_E_INVALID_ARG, "unknown kernel");
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    double sum = 0.0;
    int64_t n = 0;
    for (const ProfRecord& r : u->prof) {
        if (r.kind != kernel) continue;
        cudaError_t e = cudaEventSynchronize(r.stop);
        float ms = 0.f;
        if (e == cudaSuccess) e = cudaEventElapsedTime(&ms, r.start, r.stop);
        if (e != cudaSuccess) return cuda_fail(e, "profiler event");
        sum += ms;
        ++n;
    }
    if (total_ms) *total_ms = sum;
    if (launches) *launches = n;
    return FSDP_OK;
}

int fsdp_profile_reset(fsdp_unit* u) {
    int rc = check_unit(u, false);
    if (rc) return rc;
    DeviceGuard dg(u->device);
    if (!dg.ok()) return fail(FSDP_E_CUDA, "cannot select the unit's device");
    for (auto& r : u->prof) {
        cudaEventSynchronize(r.stop);
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    u->prof.clear();
    return FSDP_OK;
}

}  // extern "C"
