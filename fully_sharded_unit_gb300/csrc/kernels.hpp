// Launchers for the per-unit kernels (host side).  Every launcher enqueues
// one kernel on `stream` and returns the launch status.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "plan.hpp"

namespace fsdp {

// fp32 constants of one AdamW step, formed on the host.
struct AdamWConsts {
    float decay;   // 1 - lr*wd
    float b1, c1;  // beta1, 1 - beta1
    float b2, c2;  // beta2, 1 - beta2
    float bc2;     // 1 - beta2^t
    float step;    // lr / (1 - beta1^t)
    float eps;
};

// Where AdamW takes one step's constants from: the host-formed `c`, or (for
// CUDA-graph replay) entry *counter of a device table of consecutive steps.
struct StepSource {
    AdamWConsts c;
    const AdamWConsts* table;   // null: use c
    const int64_t* counter;     // device: steps taken since the table was made
    int64_t count;              // table length
    int32_t* status;            // device: set to 1 when a step finds the table used up
    int write_shadow;           // 1: also store the bf16 shadow RNE(p) of every updated element
};

struct ParamSrc {
    const float* ptr;   // parameter's first element
    int64_t offset;     // its FlatParameter offset
};

// Reduce-scatter arguments beyond the tile table and the gradient pointers.
struct ReduceArgs {
    int F;              // ranks per sharding group (the unit's N)
    int groups;         // replication groups R >= 1; W = F*R gradients
    int bf16_reduce;    // 1: bf16 arithmetic (requires groups == 1)
    float inv_scale;    // multiplier applied when `scale` is set
    int scale;
    int accumulate;     // add into the existing gradient shard
    int32_t* found;     // set to 1 when a written value is not finite; may be null
    int narrow;         // 1: some gradient buffer is only 16-byte aligned (16-byte loads)
    unsigned long long wait_ns;   // bound of each wait in the staged kernels (0: 10 s)
    int overlap;        // register-staged kernels: may run beside the previous kernel
                        // (touches nothing it touches; completes after it)
    int withhold;       // test of the give-up path: CTA 0 of a staged kernel arms its
                        // first stage's barrier but issues none of that stage's copies;
                        // 1: the drain skips that stage, 2: the drain waits for it too
                        // (and runs out: no copy is in flight, nothing lands late)
};

cudaError_t launch_shard_in(const Tile* tiles, int64_t ntiles, const ParamSrc* params,
                            float* master, uint16_t* shadow, cudaStream_t st);

// overlap: the kernel touches nothing the stream's previous kernel touches,
// so it may run beside it (it still completes after it); see pdl_begin.
cudaError_t launch_gather(const Tile* tiles, int64_t ntiles, const float* master,
                          uint16_t* out, cudaStream_t st, bool overlap = false);

// The gather from the bf16 shadow shards (a copy; the cast was done by AdamW
// or shard-in).
cudaError_t launch_gather_shadow(const Tile* tiles, int64_t ntiles, const uint16_t* shadow,
                                 uint16_t* out, cudaStream_t st, bool overlap = false);

// grads: W = a.F * a.groups pointers (fp32 or bf16 per grad_dtype), each P elements.
// kstatus: the unit's device status word (FSDP_KSTATUS_* bits).
cudaError_t launch_reduce_scatter(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                  int grad_dtype, const ReduceArgs& a, float* gshard, int32_t* kstatus,
                                  cudaStream_t st);

// shadow[i] = RNE_bf16(master[i]) for i in [begin, begin + n); begin and n
// multiples of 8.
cudaError_t launch_cast_range(const float* master, uint16_t* shadow, int64_t begin, int64_t n, cudaStream_t st);

// Fused reduce-scatter (no unscale / accumulation / flag) and AdamW over the
// unit's segments; a.F * a.groups gradient pointers.
// kstatus: the unit's device status word (FSDP_KSTATUS_* bits raised by
// kernels whose bounded waits run out).
cudaError_t launch_reduce_adamw(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                int grad_dtype, const ReduceArgs& a, float* gshard, float* p, float* m,
                                float* v, uint16_t* shadow, const StepSource& c, int32_t* kstatus,
                                cudaStream_t st);

// One CTA waiting up to limit_ns on a barrier nothing completes; raises
// FSDP_KSTATUS_WAIT_TIMEOUT in *status.
cudaError_t launch_wait_selftest(int32_t* status, unsigned long long limit_ns, cudaStream_t st);

// n8: number of 8-element groups in the slab (slab length / 8).
cudaError_t launch_adamw(int64_t n8, float* p, const float* g, float* m, float* v,
                         uint16_t* shadow, const StepSource& c, cudaStream_t st);

// One thread: ++*counter unless the table is used up (device-step mode).
cudaError_t launch_advance_step(int64_t* counter, int64_t count, cudaStream_t st);

}  // namespace fsdp
