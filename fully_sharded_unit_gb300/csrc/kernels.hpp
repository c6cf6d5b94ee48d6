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

struct ParamSrc {
    const float* ptr;   // parameter's first element
    int64_t offset;     // its FlatParameter offset
};

struct LaunchShape {
    int grid;    // CTAs
    int block;   // threads per CTA
};

// Grid sizes: CTAs resident at once on the whole GPU (SMs x occupancy),
// capped by the available work.
struct KernelGrids {
    LaunchShape gather;
    LaunchShape reduce_small;   // N <= 64
    LaunchShape reduce_large;   // N <= 1024
    LaunchShape adamw;
    LaunchShape shard_in;
};

cudaError_t query_grids(int device, int grad_dtype, KernelGrids* out);

cudaError_t launch_shard_in(const Tile* tiles, int64_t ntiles, const ParamSrc* params,
                            float* master, uint16_t* shadow, LaunchShape ls, cudaStream_t st);

cudaError_t launch_gather(const Tile* tiles, int64_t ntiles, const float* master,
                          uint16_t* out, LaunchShape ls, cudaStream_t st);

// grads: N pointers (fp32 or bf16 per grad_dtype), each P elements.
cudaError_t launch_reduce_scatter(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                  int N, int grad_dtype, float* gshard, LaunchShape small,
                                  LaunchShape large, cudaStream_t st);

// n8: number of 8-element groups in the slab (slab length / 8).
cudaError_t launch_adamw(int64_t n8, float* p, const float* g, float* m, float* v,
                         uint16_t* shadow, const AdamWConsts& c, LaunchShape ls, cudaStream_t st);

}  // namespace fsdp
