// Per-unit FSDP kernels for sm_103a: shard-in, gather+cast, reduce-scatter,
// AdamW.  All four are HBM-bandwidth bound streaming passes; none is a
// contraction, so no tensor cores are involved.
//
// Memory access: an 8-element group is one 256-bit fp32 access
// (ld/st .v8.f32) or one 128-bit bf16 access (.v4.b32).  Segment-driven
// kernels walk a tile table (see plan.hpp): a tile never spans two segments,
// and because arena slots are congruent to global indices modulo 32 elements,
// a group that is aligned in the unsharded buffer is aligned in the arena.
// Each tile has at most 7 unaligned head and 7 tail elements, done scalar.
//
// Numerics: every floating-point operation is an explicitly rounded
// intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so nothing is
// contracted into FMAs and the results equal a sequential IEEE evaluation of
// the same expression; the fp32 -> bf16 cast is the round-to-nearest-even
// conversion instruction.  Denormals are not flushed (no fast-math).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "kernels.hpp"

namespace fsdp {
namespace {

constexpr int kBlock = 256;
constexpr int kGroupsPerThread = static_cast<int>(kTile / (8 * kBlock));   // 4
static_assert(kTile == 8 * kBlock * kGroupsPerThread, "a tile is one pass of the CTA");

struct F8 {
    float v[8];
};

// Read-only input streamed once: bypass L1.
__device__ __forceinline__ F8 ld8_ro(const float* p) {
    F8 r;
    asm("ld.global.nc.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]), "=f"(r.v[5]),
          "=f"(r.v[6]), "=f"(r.v[7])
        : "l"(p));
    return r;
}

// Input that the same thread overwrites afterwards (coherent path).
__device__ __forceinline__ F8 ld8_rw(const float* p) {
    F8 r;
    asm("ld.global.L1::no_allocate.v8.f32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3]), "=f"(r.v[4]), "=f"(r.v[5]),
          "=f"(r.v[6]), "=f"(r.v[7])
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st8(float* p, const F8& r) {
    asm volatile("st.global.L1::no_allocate.v8.f32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(p),
                 "f"(r.v[0]), "f"(r.v[1]), "f"(r.v[2]), "f"(r.v[3]), "f"(r.v[4]), "f"(r.v[5]),
                 "f"(r.v[6]), "f"(r.v[7]));
}

// 8 bf16 values (read-only input)
__device__ __forceinline__ uint4 ld8bf_ro(const uint16_t* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ void st8bf(uint16_t* p, uint4 r) {
    asm volatile("st.global.L1::no_allocate.v4.b32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(r.x),
                 "r"(r.y), "r"(r.z), "r"(r.w));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);   // round to nearest even
    return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
    __nv_bfloat16 h = __float2bfloat16_rn(x);
    return *reinterpret_cast<uint16_t*>(&h);
}

__device__ __forceinline__ uint4 pack8(const F8& r) {
    return make_uint4(pack_bf16x2(r.v[0], r.v[1]), pack_bf16x2(r.v[2], r.v[3]),
                      pack_bf16x2(r.v[4], r.v[5]), pack_bf16x2(r.v[6], r.v[7]));
}

__device__ __forceinline__ float bf16_to_f32(uint32_t h) { return __uint_as_float(h << 16); }

// bf16 pair (packed in a 32-bit word, low half first) widened exactly
__device__ __forceinline__ void widen2(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}

// Split of a tile into an unaligned head, 8-element groups and a tail.
struct TileSplit {
    int head;   // elements before the first 8-aligned global index
    int nvec;   // 8-element groups
    int tail;   // elements after the last group
};

__device__ __forceinline__ TileSplit split_tile(int64_t g, int len) {
    TileSplit t;
    t.head = static_cast<int>((8 - (g & 7)) & 7);
    if (t.head > len) t.head = len;
    t.nvec = (len - t.head) >> 3;
    t.tail = len - t.head - 8 * t.nvec;
    return t;
}

// ---------------------------------------------------------------- shard-in

__global__ void __launch_bounds__(kBlock) shard_in_kernel(const Tile* __restrict__ tiles,
                                                          int64_t ntiles,
                                                          const ParamSrc* __restrict__ params,
                                                          float* __restrict__ master,
                                                          uint16_t* __restrict__ shadow) {
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const ParamSrc ps = params[tl.aux];
        const float* src = ps.ptr + (tl.g - ps.offset);
        for (int j = threadIdx.x; j < tl.len; j += kBlock) {
            float x = src[j];
            master[tl.s + j] = x;
            shadow[tl.s + j] = to_bf16(x);
        }
    }
}

// ---------------------------------------------------------------- gather + cast

__global__ void __launch_bounds__(kBlock) gather_cast_kernel(const Tile* __restrict__ tiles,
                                                             int64_t ntiles,
                                                             const float* __restrict__ master,
                                                             uint16_t* __restrict__ out) {
    const int tid = threadIdx.x;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const TileSplit sp = split_tile(tl.g, tl.len);
        if (tid < sp.head) {
            out[tl.g + tid] = to_bf16(master[tl.s + tid]);
        } else if (tid >= 8 && tid < 8 + sp.tail) {
            const int j = sp.head + 8 * sp.nvec + (tid - 8);
            out[tl.g + j] = to_bf16(master[tl.s + j]);
        }
        const float* src = master + tl.s + sp.head;
        uint16_t* dst = out + tl.g + sp.head;
        F8 r[kGroupsPerThread];
#pragma unroll
        for (int u = 0; u < kGroupsPerThread; ++u) {
            const int v = tid + u * kBlock;
            if (v < sp.nvec) r[u] = ld8_ro(src + 8 * v);
        }
#pragma unroll
        for (int u = 0; u < kGroupsPerThread; ++u) {
            const int v = tid + u * kBlock;
            if (v < sp.nvec) st8bf(dst + 8 * v, pack8(r[u]));
        }
    }
}

// ---------------------------------------------------------------- reduce-scatter

template <int NMAX>
struct GradPtrs {
    const void* p[NMAX];
};

// Ranks are folded in batches of kBatch loads in flight per group.
constexpr int kBatch = 8;

template <typename GT>
struct GradIO;

template <>
struct GradIO<float> {
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return static_cast<const float*>(base)[i];
    }
    struct Group {
        F8 f;
    };
    static __device__ __forceinline__ Group load8(const void* base, int64_t i) {
        return Group{ld8_ro(static_cast<const float*>(base) + i)};
    }
    static __device__ __forceinline__ void widen(const Group& g, F8& out) { out = g.f; }
};

template <>
struct GradIO<uint16_t> {
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return bf16_to_f32(static_cast<const uint16_t*>(base)[i]);
    }
    struct Group {
        uint4 w;
    };
    static __device__ __forceinline__ Group load8(const void* base, int64_t i) {
        return Group{ld8bf_ro(static_cast<const uint16_t*>(base) + i)};
    }
    static __device__ __forceinline__ void widen(const Group& g, F8& out) {
        widen2(g.w.x, out.v[0], out.v[1]);
        widen2(g.w.y, out.v[2], out.v[3]);
        widen2(g.w.z, out.v[4], out.v[5]);
        widen2(g.w.w, out.v[6], out.v[7]);
    }
};

template <typename GT, int NMAX>
__global__ void __launch_bounds__(kBlock) reduce_scatter_kernel(const Tile* __restrict__ tiles,
                                                                int64_t ntiles, GradPtrs<NMAX> gp,
                                                                int N, float* __restrict__ gshard) {
    using IO = GradIO<GT>;
    const int tid = threadIdx.x;
    const float fN = static_cast<float>(N);
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const TileSplit sp = split_tile(tl.g, tl.len);
        // scalar head and tail
        int j = -1;
        if (tid < sp.head) j = tid;
        else if (tid >= 8 && tid < 8 + sp.tail) j = sp.head + 8 * sp.nvec + (tid - 8);
        if (j >= 0) {
            float acc = IO::load1(gp.p[0], tl.g + j);
            for (int r = 1; r < N; ++r) acc = __fadd_rn(acc, IO::load1(gp.p[r], tl.g + j));
            gshard[tl.s + j] = __fdiv_rn(acc, fN);
        }
        // 8-element groups: fold ranks 0..N-1 in order, kBatch loads in flight
        const int64_t g0 = tl.g + sp.head;
        float* dst = gshard + tl.s + sp.head;
        for (int v = tid; v < sp.nvec; v += kBlock) {
            const int64_t gi = g0 + 8 * static_cast<int64_t>(v);
            F8 acc;
            for (int r0 = 0; r0 < N; r0 += kBatch) {
                typename IO::Group x[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (r0 + b < N) x[b] = IO::load8(gp.p[r0 + b], gi);
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    if (r0 + b < N) {
                        F8 w;
                        IO::widen(x[b], w);
                        if (r0 + b == 0) {
                            acc = w;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) acc.v[e] = __fadd_rn(acc.v[e], w.v[e]);
                        }
                    }
                }
            }
#pragma unroll
            for (int e = 0; e < 8; ++e) acc.v[e] = __fdiv_rn(acc.v[e], fN);
            st8(dst + 8 * v, acc);
        }
    }
}

// ---------------------------------------------------------------- AdamW

__device__ __forceinline__ void adamw_elem(float& p, float g, float& m, float& v,
                                           const AdamWConsts& c) {
    const float pd = __fmul_rn(p, c.decay);
    m = __fadd_rn(__fmul_rn(c.b1, m), __fmul_rn(c.c1, g));
    v = __fadd_rn(__fmul_rn(c.b2, v), __fmul_rn(c.c2, __fmul_rn(g, g)));
    const float denom = __fadd_rn(__fsqrt_rn(__fdiv_rn(v, c.bc2)), c.eps);
    p = __fsub_rn(pd, __fmul_rn(c.step, __fdiv_rn(m, denom)));
}

__global__ void __launch_bounds__(kBlock) adamw_kernel(int64_t n8, float* __restrict__ p,
                                                       const float* __restrict__ g,
                                                       float* __restrict__ m,
                                                       float* __restrict__ v,
                                                       uint16_t* __restrict__ shadow,
                                                       AdamWConsts c) {
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n8; i += stride) {
        F8 P = ld8_rw(p + 8 * i);
        F8 G = ld8_ro(g + 8 * i);
        F8 M = ld8_rw(m + 8 * i);
        F8 V = ld8_rw(v + 8 * i);
#pragma unroll
        for (int e = 0; e < 8; ++e) adamw_elem(P.v[e], G.v[e], M.v[e], V.v[e], c);
        st8(p + 8 * i, P);
        st8(m + 8 * i, M);
        st8(v + 8 * i, V);
        st8bf(shadow + 8 * i, pack8(P));
    }
}

template <typename K>
int resident_ctas(K kernel, int device, int sms) {
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kBlock, 0) != cudaSuccess ||
        per_sm < 1)
        per_sm = 1;
    (void)device;
    return per_sm * sms;
}

int capped(int grid, int64_t work) {
    if (work < 1) return 1;
    return static_cast<int>(work < grid ? work : grid);
}

}  // namespace

cudaError_t query_grids(int device, int grad_dtype, KernelGrids* out) {
    int sms = 0;
    cudaError_t e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device);
    if (e != cudaSuccess) return e;
    out->gather = {resident_ctas(gather_cast_kernel, device, sms), kBlock};
    if (grad_dtype == FSDP_DTYPE_BF16) {
        out->reduce_small = {resident_ctas(reduce_scatter_kernel<uint16_t, 64>, device, sms), kBlock};
        out->reduce_large = {resident_ctas(reduce_scatter_kernel<uint16_t, kMaxRanks>, device, sms), kBlock};
    } else {
        out->reduce_small = {resident_ctas(reduce_scatter_kernel<float, 64>, device, sms), kBlock};
        out->reduce_large = {resident_ctas(reduce_scatter_kernel<float, kMaxRanks>, device, sms), kBlock};
    }
    out->adamw = {resident_ctas(adamw_kernel, device, sms), kBlock};
    out->shard_in = {resident_ctas(shard_in_kernel, device, sms), kBlock};
    return cudaGetLastError();
}

cudaError_t launch_shard_in(const Tile* tiles, int64_t ntiles, const ParamSrc* params,
                            float* master, uint16_t* shadow, LaunchShape ls, cudaStream_t st) {
    if (ntiles == 0) return cudaSuccess;
    shard_in_kernel<<<capped(ls.grid, ntiles), kBlock, 0, st>>>(tiles, ntiles, params, master, shadow);
    return cudaGetLastError();
}

cudaError_t launch_gather(const Tile* tiles, int64_t ntiles, const float* master, uint16_t* out,
                          LaunchShape ls, cudaStream_t st) {
    if (ntiles == 0) return cudaSuccess;
    gather_cast_kernel<<<capped(ls.grid, ntiles), kBlock, 0, st>>>(tiles, ntiles, master, out);
    return cudaGetLastError();
}

template <typename GT, int NMAX>
static cudaError_t launch_rs_t(const Tile* tiles, int64_t ntiles, const void* const* grads, int N,
                               float* gshard, LaunchShape ls, cudaStream_t st) {
    GradPtrs<NMAX> gp;
    for (int r = 0; r < NMAX; ++r) gp.p[r] = r < N ? grads[r] : nullptr;
    reduce_scatter_kernel<GT, NMAX><<<capped(ls.grid, ntiles), kBlock, 0, st>>>(tiles, ntiles, gp, N, gshard);
    return cudaGetLastError();
}

cudaError_t launch_reduce_scatter(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                  int N, int grad_dtype, float* gshard, LaunchShape small,
                                  LaunchShape large, cudaStream_t st) {
    if (ntiles == 0) return cudaSuccess;
    if (grad_dtype == FSDP_DTYPE_BF16) {
        return N <= 64 ? launch_rs_t<uint16_t, 64>(tiles, ntiles, grads, N, gshard, small, st)
                       : launch_rs_t<uint16_t, kMaxRanks>(tiles, ntiles, grads, N, gshard, large, st);
    }
    return N <= 64 ? launch_rs_t<float, 64>(tiles, ntiles, grads, N, gshard, small, st)
                   : launch_rs_t<float, kMaxRanks>(tiles, ntiles, grads, N, gshard, large, st);
}

cudaError_t launch_adamw(int64_t n8, float* p, const float* g, float* m, float* v,
                         uint16_t* shadow, const AdamWConsts& c, LaunchShape ls, cudaStream_t st) {
    if (n8 == 0) return cudaSuccess;
    const int64_t blocks_needed = (n8 + kBlock - 1) / kBlock;
    adamw_kernel<<<capped(ls.grid, blocks_needed), kBlock, 0, st>>>(n8, p, g, m, v, shadow, c);
    return cudaGetLastError();
}

}  // namespace fsdp
