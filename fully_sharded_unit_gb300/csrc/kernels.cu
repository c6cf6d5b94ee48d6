// Per-unit FSDP kernels for sm_103a: shard-in, gather+cast (from the fp32
// master or the bf16 shadow), reduce-scatter, AdamW, the fused reduce-scatter
// + AdamW (staged in shared memory by bulk asynchronous copies, or in
// registers for wide units), a range cast, the device step counter and a
// bounded-wait self-test.  All are HBM-bandwidth bound streaming passes; none
// is a contraction, so no tensor cores are involved.
//
// Memory access: an 8-element group is one 256-bit fp32 access
// (ld/st .v8.f32) or one 128-bit bf16 access (.v4.b32); the plain
// bf16-gradient reduce-scatter reads 16-element groups, one 256-bit access
// per rank; the staged fused kernel moves whole chunk rows with cp.async.bulk.
// Gradient buffers that are only 16-byte aligned take the NARROW instances of
// the register-staged reductions: fp32 groups load as two 128-bit halves and
// the plain bf16 reduce-scatter falls back to 8-element (128-bit) groups.
// Segment-driven kernels walk a tile table (see plan.hpp): a tile never spans
// two segments, and because arena slots are congruent to global indices
// modulo 32 elements, a group that is aligned in the unsharded buffer is
// aligned in the arena.  Each tile has at most A-1 unaligned head and A-1
// tail elements (A = 8 or 16), done scalar.
//
// Launch: every kernel is launched with programmatic stream serialization
// and starts with griddepcontrol.wait (pdl_enter), so the next kernel's CTAs
// are scheduled during the previous kernel's last wave while the stream order
// of every memory access stays the same (the staged fused kernel waits but
// does not release its successor early).  Inside a unit step the second
// gather and the reduce-scatter, which share no memory with the kernel
// before them, may instead start at once and wait only before exiting
// (pdl_begin / pdl_leave with `overlap`).
//
// Numerics: every floating-point operation is an explicitly rounded
// intrinsic (__fadd_rn, __fmul_rn, __fdiv_rn, __fsqrt_rn), so nothing is
// contracted into FMAs and the results equal a sequential IEEE evaluation of
// the same expression; the fp32 -> bf16 cast is the round-to-nearest-even
// conversion instruction.  Denormals are not flushed (no fast-math).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <type_traits>

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

// The same eight values as two 128-bit accesses, for buffers that are only
// 16-byte aligned.
__device__ __forceinline__ F8 ld8_ro_narrow(const float* p) {
    F8 r;
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
        : "=f"(r.v[0]), "=f"(r.v[1]), "=f"(r.v[2]), "=f"(r.v[3])
        : "l"(p));
    asm("ld.global.nc.L1::no_allocate.v4.f32 {%0,%1,%2,%3}, [%4];"
        : "=f"(r.v[4]), "=f"(r.v[5]), "=f"(r.v[6]), "=f"(r.v[7])
        : "l"(p + 4));
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

// 16 bf16 values (read-only input), one 32-byte access
struct U8 {
    uint32_t w[8];
};

__device__ __forceinline__ U8 ld16bf_ro(const uint16_t* p) {
    U8 r;
    asm("ld.global.nc.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
        : "=r"(r.w[0]), "=r"(r.w[1]), "=r"(r.w[2]), "=r"(r.w[3]), "=r"(r.w[4]), "=r"(r.w[5]),
          "=r"(r.w[6]), "=r"(r.w[7])
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

// Programmatic dependent launch.  Every kernel is launched with programmatic
// stream serialization, so its grid may be scheduled while the previous
// kernel of the stream is still running; it waits here, before touching any
// memory, until that kernel has completed and its writes are visible, so the
// stream order of all reads and writes is unchanged.  Having waited, it lets
// the next kernel's grid be scheduled in turn: its CTAs take the SMs that
// this grid's last wave leaves idle and start the moment this grid ends.
__device__ __forceinline__ void pdl_enter() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// The same for a kernel that touches nothing its predecessor writes or reads
// (inside fsdp_step: the second gather after the first, the reduce-scatter
// after the gathers).  With `overlap` it lets its successor be scheduled at
// once and starts its work beside the predecessor's last wave, and waits for
// the predecessor only before exiting (pdl_leave): it still completes after
// it, so a kernel that waits on this one also finds every earlier one done.
// Every block of the predecessor has already been scheduled when this grid
// starts (it starts only once they have all released it), so the waiting
// blocks cannot keep the predecessor from finishing.
__device__ __forceinline__ void pdl_begin(bool overlap) {
    if (!overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ void pdl_leave(bool overlap) {
    if (overlap) asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Correctly rounded (RNE) addition of two bf16 pairs.  It equals the fp32 sum
// rounded once to bf16: the exact sum of two bf16 values rounded to fp32 and
// then to bf16 cannot differ from it rounded straight to bf16, because fp32
// carries at least 2*8+2 significant bits (double rounding is innocuous).
__device__ __forceinline__ uint32_t add_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("add.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// bf16 partial sums of 8 elements, 4 packed pairs, folded in one rank order.
struct B8 {
    uint32_t w[4];
};

// Split of a tile into an unaligned head, 8-element groups and a tail.
struct TileSplit {
    int head;   // elements before the first 8-aligned global index
    int nvec;   // 8-element groups
    int tail;   // elements after the last group
};

// A-element groups (A = 8, or 16 for the bf16-gradient reduce-scatter).
template <int A = 8>
__device__ __forceinline__ TileSplit split_tile(int64_t g, int len) {
    TileSplit t;
    t.head = static_cast<int>((A - (g & (A - 1))) & (A - 1));
    if (t.head > len) t.head = len;
    t.nvec = (len - t.head) / A;
    t.tail = len - t.head - A * t.nvec;
    return t;
}

// ---------------------------------------------------------------- shard-in

__global__ void __launch_bounds__(kBlock) shard_in_kernel(const Tile* __restrict__ tiles,
                                                          int64_t ntiles,
                                                          const ParamSrc* __restrict__ params,
                                                          float* __restrict__ master,
                                                          uint16_t* __restrict__ shadow) {
    pdl_enter();
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
                                                             uint16_t* __restrict__ out, int overlap) {
    pdl_begin(overlap);
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
    pdl_leave(overlap);
}

// ---------------------------------------------------------------- gather from the shadow

__global__ void __launch_bounds__(kBlock) gather_shadow_kernel(const Tile* __restrict__ tiles,
                                                               int64_t ntiles,
                                                               const uint16_t* __restrict__ shadow,
                                                               uint16_t* __restrict__ out, int overlap) {
    pdl_begin(overlap);
    const int tid = threadIdx.x;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const TileSplit sp = split_tile(tl.g, tl.len);
        if (tid < sp.head) {
            out[tl.g + tid] = shadow[tl.s + tid];
        } else if (tid >= 8 && tid < 8 + sp.tail) {
            const int j = sp.head + 8 * sp.nvec + (tid - 8);
            out[tl.g + j] = shadow[tl.s + j];
        }
        const uint16_t* src = shadow + tl.s + sp.head;
        uint16_t* dst = out + tl.g + sp.head;
        uint4 r[kGroupsPerThread];
#pragma unroll
        for (int u = 0; u < kGroupsPerThread; ++u) {
            const int v = tid + u * kBlock;
            if (v < sp.nvec) r[u] = ld8bf_ro(src + 8 * v);
        }
#pragma unroll
        for (int u = 0; u < kGroupsPerThread; ++u) {
            const int v = tid + u * kBlock;
            if (v < sp.nvec) st8bf(dst + 8 * v, r[u]);
        }
    }
    pdl_leave(overlap);
}

// ---------------------------------------------------------------- range cast

__global__ void __launch_bounds__(kBlock) cast_range_kernel(const float* __restrict__ master,
                                                            uint16_t* __restrict__ shadow,
                                                            int64_t n8) {
    pdl_enter();
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kBlock;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * kBlock + threadIdx.x; i < n8; i += stride)
        st8bf(shadow + 8 * i, pack8(ld8_ro(master + 8 * i)));
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
    // NARROW: the gradient buffers may be only 16-byte aligned
    template <bool NARROW>
    static __device__ __forceinline__ Group load8(const void* base, int64_t i) {
        if constexpr (NARROW) return Group{ld8_ro_narrow(static_cast<const float*>(base) + i)};
        else return Group{ld8_ro(static_cast<const float*>(base) + i)};
    }
    static __device__ __forceinline__ void widen(const Group& g, F8& out) { out = g.f; }
    // the group rounded to bf16 pairs (RNE), for the bf16 reduction
    static __device__ __forceinline__ B8 pack(const Group& g) {
        return B8{{pack_bf16x2(g.f.v[0], g.f.v[1]), pack_bf16x2(g.f.v[2], g.f.v[3]),
                   pack_bf16x2(g.f.v[4], g.f.v[5]), pack_bf16x2(g.f.v[6], g.f.v[7])}};
    }
};

template <>
struct GradIO<uint16_t> {
    static __device__ __forceinline__ float load1(const void* base, int64_t i) {
        return bf16_to_f32(static_cast<const uint16_t*>(base)[i]);
    }
    struct Group {
        uint4 w;
    };
    // one 16-byte access: needs 16-byte alignment either way
    template <bool NARROW>
    static __device__ __forceinline__ Group load8(const void* base, int64_t i) {
        return Group{ld8bf_ro(static_cast<const uint16_t*>(base) + i)};
    }
    static __device__ __forceinline__ void widen(const Group& g, F8& out) {
        widen2(g.w.x, out.v[0], out.v[1]);
        widen2(g.w.y, out.v[2], out.v[3]);
        widen2(g.w.z, out.v[4], out.v[5]);
        widen2(g.w.w, out.v[6], out.v[7]);
    }
    static __device__ __forceinline__ B8 pack(const Group& g) { return B8{{g.w.x, g.w.y, g.w.z, g.w.w}}; }
};

// fp32 value rounded to bf16 (RNE) and widened back: one bf16 rounding.
__device__ __forceinline__ float round_bf16(float x) {
    return __bfloat162float(__float2bfloat16_rn(x));
}

__device__ __forceinline__ bool not_finite(float x) {
    return (__float_as_uint(x) & 0x7F800000u) == 0x7F800000u;
}

// One element: group-wise left folds, the fold over groups, the division by W.
template <typename GT, int NMAX, bool BF16>
__device__ __forceinline__ float reduce1(const GradPtrs<NMAX>& gp, const ReduceArgs& a, int groups,
                                         float fW, int64_t i) {
    using IO = GradIO<GT>;
    if (BF16) {
        // bf16 gradients are already bf16; only fp32 inputs need the rounding
        constexpr bool round_in = !std::is_same<GT, uint16_t>::value;
        float acc = IO::load1(gp.p[0], i);
        if (round_in) acc = round_bf16(acc);
        for (int r = 1; r < a.F; ++r) {
            float x = IO::load1(gp.p[r], i);
            if (round_in) x = round_bf16(x);
            acc = round_bf16(__fadd_rn(acc, x));
        }
        return round_bf16(__fdiv_rn(acc, fW));
    }
    float tot = 0.f;
    for (int grp = 0; grp < groups; ++grp) {
        const int base = grp * a.F;
        float acc = IO::load1(gp.p[base], i);
        for (int r = 1; r < a.F; ++r) acc = __fadd_rn(acc, IO::load1(gp.p[base + r], i));
        tot = grp == 0 ? acc : __fadd_rn(tot, acc);
    }
    return __fdiv_rn(tot, fW);
}

// bf16 reduction of one aligned group (reduce_dtype bf16, one group: the host
// rejects it with replicas): inputs rounded to bf16 (exact for bf16
// gradients), the rank-order partial sums kept as packed bf16 pairs, then
// the quotient by F rounded to bf16.  Same values as rounding every fp32
// partial sum (see add_bf16x2).
template <int W>
struct BGroup {
    uint32_t w[W];
};

template <int W>
__device__ __forceinline__ void finish_bf16(const BGroup<W>& acc, float fW, F8* out) {
#pragma unroll
    for (int q = 0; q < W; ++q) {
        F8& o = out[q / 4];
        widen2(acc.w[q], o.v[2 * (q % 4)], o.v[2 * (q % 4) + 1]);
    }
#pragma unroll
    for (int h = 0; h < W / 4; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) out[h].v[e] = round_bf16(__fdiv_rn(out[h].v[e], fW));
}

// Eight consecutive elements (an aligned group), same order of operations.
// NARROW: 16-byte instead of 32-byte fp32 gradient loads.
template <typename GT, int NMAX, bool BF16, bool NARROW = false>
__device__ __forceinline__ F8 reduce8(const GradPtrs<NMAX>& gp, const ReduceArgs& a, int groups,
                                      float fW, int64_t gi) {
    using IO = GradIO<GT>;
    F8 tot;
    if constexpr (BF16) {
        BGroup<4> acc;
        for (int r0 = 0; r0 < a.F; r0 += kBatch) {
            typename IO::Group x[kBatch];
#pragma unroll
            for (int b = 0; b < kBatch; ++b)
                if (r0 + b < a.F) x[b] = IO::template load8<NARROW>(gp.p[r0 + b], gi);
#pragma unroll
            for (int b = 0; b < kBatch; ++b) {
                if (r0 + b < a.F) {
                    const B8 w = IO::pack(x[b]);
#pragma unroll
                    for (int q = 0; q < 4; ++q) acc.w[q] = r0 + b == 0 ? w.w[q] : add_bf16x2(acc.w[q], w.w[q]);
                }
            }
        }
        finish_bf16<4>(acc, fW, &tot);
        return tot;
    } else {
        for (int grp = 0; grp < groups; ++grp) {
            const int base = grp * a.F;
            F8 acc;
            for (int r0 = 0; r0 < a.F; r0 += kBatch) {
                typename IO::Group x[kBatch];
#pragma unroll
                for (int b = 0; b < kBatch; ++b)
                    if (r0 + b < a.F) x[b] = IO::template load8<NARROW>(gp.p[base + r0 + b], gi);
#pragma unroll
                for (int b = 0; b < kBatch; ++b) {
                    if (r0 + b < a.F) {
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
            if (grp == 0) {
                tot = acc;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) tot.v[e] = __fadd_rn(tot.v[e], acc.v[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) tot.v[e] = __fdiv_rn(tot.v[e], fW);
        return tot;
    }
}

// Ranks folded per batch in the 16-wide path: 4 x 32 bytes in flight per
// thread, as many bytes as the 8-wide path's 8 x 16, in half the registers.
constexpr int kBatch16 = 4;

// Sixteen consecutive bf16-gradient elements (one 32-byte load per rank), same
// order of operations as reduce8.
template <int NMAX, bool BF16>
__device__ __forceinline__ void reduce16(const GradPtrs<NMAX>& gp, const ReduceArgs& a, int groups,
                                         float fW, int64_t gi, F8& out0, F8& out1) {
    if constexpr (BF16) {
        BGroup<8> acc;
        for (int r0 = 0; r0 < a.F; r0 += kBatch16) {
            U8 x[kBatch16];
#pragma unroll
            for (int b = 0; b < kBatch16; ++b)
                if (r0 + b < a.F) x[b] = ld16bf_ro(static_cast<const uint16_t*>(gp.p[r0 + b]) + gi);
#pragma unroll
            for (int b = 0; b < kBatch16; ++b) {
                if (r0 + b < a.F) {
#pragma unroll
                    for (int q = 0; q < 8; ++q)
                        acc.w[q] = r0 + b == 0 ? x[b].w[q] : add_bf16x2(acc.w[q], x[b].w[q]);
                }
            }
        }
        F8 o[2];
        finish_bf16<8>(acc, fW, o);
        out0 = o[0];
        out1 = o[1];
        return;
    } else {
        F8 t0, t1;
        for (int grp = 0; grp < groups; ++grp) {
            const int base = grp * a.F;
            F8 a0, a1;
            for (int r0 = 0; r0 < a.F; r0 += kBatch16) {
                U8 x[kBatch16];
#pragma unroll
                for (int b = 0; b < kBatch16; ++b)
                    if (r0 + b < a.F) x[b] = ld16bf_ro(static_cast<const uint16_t*>(gp.p[base + r0 + b]) + gi);
#pragma unroll
                for (int b = 0; b < kBatch16; ++b) {
                    if (r0 + b < a.F) {
                        F8 w0, w1;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            widen2(x[b].w[q], w0.v[2 * q], w0.v[2 * q + 1]);
                            widen2(x[b].w[4 + q], w1.v[2 * q], w1.v[2 * q + 1]);
                        }
                        if (r0 + b == 0) {
                            a0 = w0;
                            a1 = w1;
                        } else {
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                a0.v[e] = __fadd_rn(a0.v[e], w0.v[e]);
                                a1.v[e] = __fadd_rn(a1.v[e], w1.v[e]);
                            }
                        }
                    }
                }
            }
            if (grp == 0) {
                t0 = a0;
                t1 = a1;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) {
                    t0.v[e] = __fadd_rn(t0.v[e], a0.v[e]);
                    t1.v[e] = __fadd_rn(t1.v[e], a1.v[e]);
                }
            }
        }
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            t0.v[e] = __fdiv_rn(t0.v[e], fW);
            t1.v[e] = __fdiv_rn(t1.v[e], fW);
        }
        out0 = t0;
        out1 = t1;
    }
}

// Optional unscale / accumulation / non-finite check of eight results.
__device__ __forceinline__ void post8(F8& x, const float* dst, bool post, const ReduceArgs& a,
                                      bool check, bool& bad) {
    if (post) {
        F8 old;
        if (a.accumulate) old = ld8_rw(dst);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            if (a.scale) x.v[e] = __fmul_rn(x.v[e], a.inv_scale);
            if (a.accumulate) x.v[e] = __fadd_rn(old.v[e], x.v[e]);
        }
    }
    if (check) {
#pragma unroll
        for (int e = 0; e < 8; ++e) bad |= not_finite(x.v[e]);
    }
}

// EXT = false compiles the plain reduce-scatter (one group, no unscale, no
// accumulation, no flag) with the fewest registers; EXT = true adds hybrid
// groups and the post-reduction options.  NARROW = true serves gradient
// buffers that are only 16-byte aligned: 16-byte loads throughout.
template <typename GT, int NMAX, bool BF16, bool EXT, bool NARROW>
__global__ void __launch_bounds__(kBlock) reduce_scatter_kernel(const Tile* __restrict__ tiles,
                                                                int64_t ntiles, GradPtrs<NMAX> gp,
                                                                ReduceArgs a, float* __restrict__ gshard) {
    pdl_begin(a.overlap != 0);
    const int tid = threadIdx.x;
    const int groups = EXT ? a.groups : 1;
    const float fW = static_cast<float>(a.F * groups);
    const bool post = EXT && (a.scale || a.accumulate);
    int32_t* const found = EXT ? a.found : nullptr;
    // bf16 gradients, plain reduce-scatter: 16-element groups, one 32-byte
    // load per rank (measured 7.46 TB/s against 7.24 TB/s with 16-byte loads
    // on the minGPT unit).  The extended one keeps 8-element groups: its
    // separate per-group and total accumulators make the 16-wide form need
    // 128 registers (2 CTAs per SM), the 8-wide one 78 (3 CTAs per SM), which
    // measured 9.44 ms against 9.73 ms for two replication groups and 6.10 ms
    // against 6.53 ms per accumulated micro-batch.
    constexpr int A = (std::is_same<GT, uint16_t>::value && !EXT && !NARROW) ? 16 : 8;
    bool bad = false;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const TileSplit sp = split_tile<A>(tl.g, tl.len);
        // scalar head and tail
        int j = -1;
        if (tid < sp.head) j = tid;
        else if (tid >= A && tid < A + sp.tail) j = sp.head + A * sp.nvec + (tid - A);
        if (j >= 0) {
            float x = reduce1<GT, NMAX, BF16>(gp, a, groups, fW, tl.g + j);
            if (post && a.scale) x = __fmul_rn(x, a.inv_scale);
            if (post && a.accumulate) x = __fadd_rn(gshard[tl.s + j], x);
            if (found != nullptr) bad |= not_finite(x);
            gshard[tl.s + j] = x;
        }
        // A-element groups
        const int64_t g0 = tl.g + sp.head;
        float* dst = gshard + tl.s + sp.head;
        for (int v = tid; v < sp.nvec; v += kBlock) {
            float* d = dst + A * v;
            if constexpr (A == 16) {
                F8 x0, x1;
                reduce16<NMAX, BF16>(gp, a, groups, fW, g0 + 16 * static_cast<int64_t>(v), x0, x1);
                post8(x0, d, post, a, found != nullptr, bad);
                post8(x1, d + 8, post, a, found != nullptr, bad);
                st8(d, x0);
                st8(d + 8, x1);
            } else {
                F8 x = reduce8<GT, NMAX, BF16, NARROW>(gp, a, groups, fW, g0 + 8 * static_cast<int64_t>(v));
                post8(x, d, post, a, found != nullptr, bad);
                st8(d, x);
            }
        }
    }
    if (found != nullptr) {   // uniform across the CTA
        if (__syncthreads_or(bad) && tid == 0) *found = 1;
    }
    pdl_leave(a.overlap != 0);
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

// This step's constants.  Device-step mode reads entry *counter of the table
// (the counter only changes in launch_advance_step, which runs after this
// kernel on the same stream); a used-up table skips the update and raises
// the status word instead.
__device__ __forceinline__ bool step_constants(const StepSource& src, AdamWConsts& c) {
    if (src.table == nullptr) {
        c = src.c;
        return true;
    }
    const int64_t i = *src.counter;
    if (i >= src.count) {
        if (blockIdx.x == 0 && threadIdx.x == 0) *src.status = 1;
        return false;
    }
    c = src.table[i];
    return true;
}

__global__ void advance_step_kernel(int64_t* counter, int64_t count) {
    pdl_enter();
    if (*counter < count) *counter += 1;
}

__global__ void __launch_bounds__(kBlock) adamw_kernel(int64_t n8, float* __restrict__ p,
                                                       const float* __restrict__ g,
                                                       float* __restrict__ m,
                                                       float* __restrict__ v,
                                                       uint16_t* __restrict__ shadow,
                                                       StepSource src) {
    pdl_enter();
    AdamWConsts c;
    if (!step_constants(src, c)) return;   // uniform over the grid
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
        if (src.write_shadow) st8bf(shadow + 8 * i, pack8(P));
    }
}

// ---------------------------------------------------------------- fused reduce-scatter + AdamW

// One pass per element of the unit: the reduce-scatter result (any group
// count, fp32 or bf16 reduction; no unscale, accumulation or flag) is written
// to the gradient shard and used by the AdamW update without being read back
// from HBM.  Two phases per tile: phase 1 reduces the thread's 8-element
// groups into shared memory (and writes the gradient shard), phase 2 runs
// AdamW on the same groups reading G back from shared memory.  A thread reads
// only the slots it wrote, so no barrier is needed.  Registers are capped so
// that 3 CTAs fit per SM with bf16 gradients (2 with fp32, whose reduction
// alone needs ~120): measured on the minGPT unit, the capped kernel took
// 12.35 ms against 13.24 ms uncapped.  Same operation sequence as the two
// separate kernels, so the results are identical; only segment elements are
// touched (pads stay zero, which AdamW would preserve anyway).
template <typename GT, int NMAX, bool BF16, bool HYBRID, bool NARROW>
__global__ void __launch_bounds__(kBlock, sizeof(GT) == 2 ? 3 : 2) reduce_adamw_kernel(const Tile* __restrict__ tiles,
                                                              int64_t ntiles, GradPtrs<NMAX> gp,
                                                              ReduceArgs a, float* __restrict__ gshard,
                                                              float* __restrict__ p, float* __restrict__ m,
                                                              float* __restrict__ v,
                                                              uint16_t* __restrict__ shadow, StepSource src) {
    pdl_enter();
    AdamWConsts c;
    if (!step_constants(src, c)) return;   // uniform over the grid
    __shared__ __align__(16) float gsm[kTile];
    const int tid = threadIdx.x;
    const int groups = HYBRID ? a.groups : 1;
    const float fW = static_cast<float>(a.F * groups);
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const TileSplit sp = split_tile(tl.g, tl.len);
        int j = -1;
        if (tid < sp.head) j = tid;
        else if (tid >= 8 && tid < 8 + sp.tail) j = sp.head + 8 * sp.nvec + (tid - 8);
        const int64_t g0 = tl.g + sp.head;
        const int64_t s0 = tl.s + sp.head;
        // phase 1: reduce
        float xj = 0.f;
        if (j >= 0) {
            xj = reduce1<GT, NMAX, BF16>(gp, a, groups, fW, tl.g + j);
            gshard[tl.s + j] = xj;
        }
#pragma unroll 1
        for (int vi = tid; vi < sp.nvec; vi += kBlock) {
            const F8 G = reduce8<GT, NMAX, BF16, NARROW>(gp, a, groups, fW, g0 + 8 * static_cast<int64_t>(vi));
            st8(gshard + s0 + 8 * static_cast<int64_t>(vi), G);
            float4* slot = reinterpret_cast<float4*>(gsm + 8 * vi);
            slot[0] = make_float4(G.v[0], G.v[1], G.v[2], G.v[3]);
            slot[1] = make_float4(G.v[4], G.v[5], G.v[6], G.v[7]);
        }
        // phase 2: AdamW on the same elements, G from shared memory
        if (j >= 0) {
            const int64_t s = tl.s + j;
            float pp = p[s], mm = m[s], vv = v[s];
            adamw_elem(pp, xj, mm, vv, c);
            p[s] = pp;
            m[s] = mm;
            v[s] = vv;
            if (src.write_shadow) shadow[s] = to_bf16(pp);
        }
#pragma unroll 1
        for (int vi = tid; vi < sp.nvec; vi += kBlock) {
            const int64_t s = s0 + 8 * static_cast<int64_t>(vi);
            F8 P = ld8_rw(p + s);
            F8 M = ld8_rw(m + s);
            F8 V = ld8_rw(v + s);
            const float4* slot = reinterpret_cast<const float4*>(gsm + 8 * vi);
            const float4 lo = slot[0], hi = slot[1];
            const float G[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) adamw_elem(P.v[e], G[e], M.v[e], V.v[e], c);
            st8(p + s, P);
            st8(m + s, M);
            st8(v + s, V);
            if (src.write_shadow) st8bf(shadow + s, pack8(P));
        }
    }
}

// ---------------------------------------------------------------- fused reduce-scatter + AdamW, bulk-copy staged

// The fused reduce-scatter + AdamW with its inputs staged in shared memory.
// A CTA takes one tile and streams it in chunks of CH elements through a
// ring of kStages stages.  A stage holds the chunk's W gradient rows and its
// p, m, v; one thread brings them in with bulk asynchronous copies
// (cp.async.bulk, the tensor-memory accelerator's untiled form) counted by the
// stage's mbarrier, and all threads fold, update and store from shared
// memory.  The loads in flight live in shared memory instead of registers:
// about 60 registers and no spills against 80 with spills for the
// register-staged kernel; on the minGPT unit (bf16 gradients, W = 8) 7.12 TB/s
// against 6.74, and 7.24 against 6.46 TB/s with two replication groups
// (W = 16).  Measured over chunk x stages at W = 8: 2048 x 2 (115 KB, 2 CTAs
// per SM) and 1024 x 3 (86 KB, 2 per SM) within 0.4 %; 512-element chunks
// (1 KB copies) and 2048 x 3 (1 CTA per SM) 10-35 % slower; one CTA per tile
// beats 2 or 4 tiles per CTA and a persistent grid.  So two stages of at most
// 56 KB, the chunk the largest of 2048, 1024, 512 elements that fits: up to
// W x gradient bytes = 100 (bf16 gradients with W <= 50, fp32 with W <= 25);
// wider units take reduce_adamw_kernel.
constexpr int kStages = 2;
// A stage holds at most this many bytes (2 CTAs of 2 stages fit an SM); the
// chunk is the largest of 2048, 1024 and 512 elements that fits.
constexpr int kStageMaxBytes = 57344;
__host__ __device__ constexpr int chunk_for(int elem_bytes) {   // stage bytes per chunk element
    return 2048 * elem_bytes <= kStageMaxBytes ? 2048
         : 1024 * elem_bytes <= kStageMaxBytes ? 1024
         : 512 * elem_bytes <= kStageMaxBytes ? 512 : 0;
}
// A wait on a stage gives up after ReduceArgs::wait_ns (this default when 0):
// the kernel then raises bit FSDP_KSTATUS_WAIT_TIMEOUT of the unit's status
// word, waits (again bounded) for its own copies in flight, raising
// FSDP_KSTATUS_DRAIN_TIMEOUT if one of those waits runs out too, and returns.
constexpr unsigned long long kWaitLimitNs = 10000000000ull;

__device__ __forceinline__ unsigned long long wait_limit(const ReduceArgs& a) {
    return a.wait_ns != 0 ? a.wait_ns : kWaitLimitNs;
}

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Wait for the barrier phase with the given parity; false if it has not
// completed within limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity,
                                          unsigned long long limit_ns = kWaitLimitNs) {
    const uint32_t addr = smem_addr(bar);
    unsigned long long t0 = 0;
    for (uint32_t i = 0;; ++i) {
        uint32_t done;
        asm volatile(
            "{ .reg .pred p; mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2; selp.u32 %0, 1, 0, p; }"
            : "=r"(done)
            : "r"(addr), "r"(parity)
            : "memory");
        if (done) return true;
        if (i == 0) t0 = global_ns();
        else if ((i & 63) == 0 && global_ns() - t0 > limit_ns) return false;
    }
}

// Layout of one stage: W gradient rows of CH GT, then p, m, v (fp32).
template <typename GT, int CH>
__device__ __forceinline__ size_t stage_bytes(int W) {
    return static_cast<size_t>(CH) * (W * sizeof(GT) + 12);
}

// The aligned body of a tile: [ga, gb), multiples of 16 elements.
struct Body {
    int64_t ga;   // global index of the first body element
    int64_t sa;   // its arena slot
    int64_t n;    // body elements (multiple of 16)
    int head;     // elements before ga
    int tail;     // elements after the body
};

__device__ __forceinline__ Body tile_body(const Tile& tl) {
    Body b;
    const int64_t ga = (tl.g + 15) & ~int64_t(15);
    const int64_t ge = tl.g + tl.len;
    int64_t gb = ge & ~int64_t(15);
    if (gb < ga) gb = ga;
    if (ga >= ge) {
        b.ga = ge;
        b.n = 0;
        b.head = tl.len;
        b.tail = 0;
    } else {
        b.ga = ga;
        b.n = gb - ga;
        b.head = static_cast<int>(ga - tl.g);
        b.tail = static_cast<int>(ge - gb);
    }
    b.sa = tl.s + (b.ga - tl.g);
    return b;
}

// Four consecutive reduced gradients from a stage, same operation order as
// reduce8 (fp32 fold within each group, then across groups, then / W; or
// the bf16 fold).
template <typename GT, bool BF16, int CH>
__device__ __forceinline__ void reduce4_smem(const unsigned char* rows, int F, int groups, float fW, int e,
                                             float out[4]) {
    if constexpr (BF16) {
        uint32_t acc[2];
        for (int r = 0; r < F; ++r) {
            uint32_t w[2];
            if constexpr (sizeof(GT) == 2) {
                const uint2 q = *reinterpret_cast<const uint2*>(rows + (static_cast<size_t>(r) * CH + e) * 2);
                w[0] = q.x;
                w[1] = q.y;
            } else {
                const float4 q = *reinterpret_cast<const float4*>(rows + (static_cast<size_t>(r) * CH + e) * 4);
                w[0] = pack_bf16x2(q.x, q.y);
                w[1] = pack_bf16x2(q.z, q.w);
            }
            acc[0] = r == 0 ? w[0] : add_bf16x2(acc[0], w[0]);
            acc[1] = r == 0 ? w[1] : add_bf16x2(acc[1], w[1]);
        }
        widen2(acc[0], out[0], out[1]);
        widen2(acc[1], out[2], out[3]);
#pragma unroll
        for (int k = 0; k < 4; ++k) out[k] = round_bf16(__fdiv_rn(out[k], fW));
    } else {
        float tot[4];
        for (int grp = 0; grp < groups; ++grp) {
            float acc[4];
            for (int r = 0; r < F; ++r) {
                const int row = grp * F + r;
                float x[4];
                if constexpr (sizeof(GT) == 2) {
                    const uint2 q = *reinterpret_cast<const uint2*>(rows + (static_cast<size_t>(row) * CH + e) * 2);
                    widen2(q.x, x[0], x[1]);
                    widen2(q.y, x[2], x[3]);
                } else {
                    const float4 q = *reinterpret_cast<const float4*>(rows + (static_cast<size_t>(row) * CH + e) * 4);
                    x[0] = q.x;
                    x[1] = q.y;
                    x[2] = q.z;
                    x[3] = q.w;
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) acc[k] = r == 0 ? x[k] : __fadd_rn(acc[k], x[k]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) tot[k] = grp == 0 ? acc[k] : __fadd_rn(tot[k], acc[k]);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) out[k] = __fdiv_rn(tot[k], fW);
    }
}

template <typename GT, int NMAX, bool BF16, bool HYBRID, int CH>
__global__ void __launch_bounds__(kBlock) reduce_adamw_bulk_kernel(const Tile* __restrict__ tiles,
                                                                   int64_t ntiles, GradPtrs<NMAX> gp,
                                                                   ReduceArgs a, float* __restrict__ gshard,
                                                                   float* __restrict__ p, float* __restrict__ m,
                                                                   float* __restrict__ v,
                                                                   uint16_t* __restrict__ shadow, StepSource src,
                                                                   int32_t* wait_status) {
    // Waits for the previous kernel like pdl_enter, but does not let the next
    // kernel's CTAs be scheduled before this grid ends: those early CTAs,
    // parked beside this kernel's last wave, cost 0.23 ms per launch on the
    // minGPT unit (27.94 against 27.47 ms per fused two-unit step).
    asm volatile("griddepcontrol.wait;" ::: "memory");
    AdamWConsts c;
    if (!step_constants(src, c)) return;   // uniform over the grid
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    unsigned char* ring = smem + 128;
    const int tid = threadIdx.x;
    const int groups = HYBRID ? a.groups : 1;
    const int W = a.F * groups;
    const float fW = static_cast<float>(W);
    const size_t sbytes = stage_bytes<GT, CH>(W);
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    // producer state (thread 0): the next chunk to bring in
    int64_t pt = blockIdx.x;   // its tile
    int64_t pc = 0;            // its chunk within the tile
    Body pb{};
    bool pb_valid = false;
    uint32_t issued = 0, consumed = 0;
    uint32_t withheld = 0xFFFFFFFFu;   // the stage armed without copies (a.withhold), if any
    const unsigned long long limit = wait_limit(a);
    auto top_up = [&]() {
        while (issued - consumed < static_cast<uint32_t>(kStages) && pt < ntiles) {
            if (!pb_valid) {
                pb = tile_body(tiles[pt]);
                pb_valid = true;
            }
            const int64_t nch = (pb.n + CH - 1) / CH;
            if (pc >= nch) {
                pt += gridDim.x;
                pc = 0;
                pb_valid = false;
                continue;
            }
            const int64_t off = pc * CH;
            const uint32_t n = static_cast<uint32_t>(pb.n - off < CH ? pb.n - off : CH);
            const int s = static_cast<int>(issued % kStages);
            unsigned char* st = ring + s * sbytes;
            mbar_expect_tx(&full[s], n * static_cast<uint32_t>(W * sizeof(GT) + 12));
            if (a.withhold != 0 && blockIdx.x == 0 && issued == 0) {
                withheld = issued;   // nothing will complete this stage: its wait runs out
            } else {
                for (int r = 0; r < W; ++r)
                    bulk_g2s(st + static_cast<size_t>(r) * CH * sizeof(GT),
                             static_cast<const GT*>(gp.p[r]) + pb.ga + off, n * sizeof(GT), &full[s]);
                unsigned char* pmv = st + static_cast<size_t>(W) * CH * sizeof(GT);
                bulk_g2s(pmv, p + pb.sa + off, n * 4, &full[s]);
                bulk_g2s(pmv + CH * 4, m + pb.sa + off, n * 4, &full[s]);
                bulk_g2s(pmv + 2 * CH * 4, v + pb.sa + off, n * 4, &full[s]);
            }
            ++issued;
            ++pc;
        }
    };

    bool ok = true;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const Body b = tile_body(tl);
        // unaligned head and tail, straight from global memory
        int j = -1;
        if (tid < b.head) j = tid;
        else if (tid >= 16 && tid < 16 + b.tail) j = b.head + static_cast<int>(b.n) + (tid - 16);
        if (j >= 0) {
            const float xj = reduce1<GT, NMAX, BF16>(gp, a, groups, fW, tl.g + j);
            const int64_t s = tl.s + j;
            gshard[s] = xj;
            float pp = p[s], mm = m[s], vv = v[s];
            adamw_elem(pp, xj, mm, vv, c);
            p[s] = pp;
            m[s] = mm;
            v[s] = vv;
            if (src.write_shadow) shadow[s] = to_bf16(pp);
        }
        const int64_t nch = (b.n + CH - 1) / CH;
        for (int64_t ch = 0; ch < nch; ++ch) {
            if (tid == 0) top_up();
            const int s = static_cast<int>(consumed % kStages);
            const uint32_t parity = (consumed / kStages) & 1u;
            const bool got = mbar_wait(&full[s], parity, limit);
            const int64_t off = ch * CH;
            const int64_t n = b.n - off < CH ? b.n - off : CH;
            for (int e = tid * 4; got && e < n; e += 4 * kBlock) {
                const unsigned char* st = ring + s * sbytes;
                float G[4];
                reduce4_smem<GT, BF16, CH>(st, a.F, groups, fW, e, G);
                const float* pmv = reinterpret_cast<const float*>(st + static_cast<size_t>(W) * CH * sizeof(GT));
                float4 P = *reinterpret_cast<const float4*>(pmv + e);
                float4 M = *reinterpret_cast<const float4*>(pmv + CH + e);
                float4 V = *reinterpret_cast<const float4*>(pmv + 2 * CH + e);
                adamw_elem(P.x, G[0], M.x, V.x, c);
                adamw_elem(P.y, G[1], M.y, V.y, c);
                adamw_elem(P.z, G[2], M.z, V.z, c);
                adamw_elem(P.w, G[3], M.w, V.w, c);
                const int64_t so = b.sa + off + e;
                *reinterpret_cast<float4*>(gshard + so) = make_float4(G[0], G[1], G[2], G[3]);
                *reinterpret_cast<float4*>(p + so) = P;
                *reinterpret_cast<float4*>(m + so) = M;
                *reinterpret_cast<float4*>(v + so) = V;
                if (src.write_shadow)
                    *reinterpret_cast<uint2*>(shadow + so) = make_uint2(pack_bf16x2(P.x, P.y), pack_bf16x2(P.z, P.w));
            }
            ++consumed;
            ok = __syncthreads_and(got) != 0;
            if (!ok) break;
        }
        if (!ok) break;
    }
    if (!ok) {
        // a copy did not arrive in time: report, wait (bounded) for the copies
        // this CTA still has in flight, and leave; a drain wait that runs out
        // too means copies may still land in this SM's shared memory
        if (tid == 0) {
            atomicOr(wait_status, FSDP_KSTATUS_WAIT_TIMEOUT);
            for (uint32_t q = consumed - 1; q < issued; ++q) {
                if (q == withheld && a.withhold == 1) continue;   // armed, but no copy was issued
                if (!mbar_wait(&full[q % kStages], (q / kStages) & 1u, limit))
                    atomicOr(wait_status, FSDP_KSTATUS_DRAIN_TIMEOUT);
            }
        }
        __syncthreads();
    }
}

// ---------------------------------------------------------------- reduce-scatter, bulk-copy staged

// The extended reduce-scatter (hybrid groups, unscale, accumulation, flag)
// with its inputs staged in shared memory the same way as
// reduce_adamw_bulk_kernel: a stage holds the chunk's W gradient rows and,
// when accumulating, the old gradient shard; the fold, unscale, accumulation
// and non-finite check run from shared memory in the same order as
// reduce_scatter_kernel (same bits).  Measured on the minGPT unit: two
// replication groups (W = 16) 9.18 ms against 9.44 ms register-staged; an
// accumulated micro-batch the same (6.10 ms).  The plain reduce-scatter stays
// register-staged: staged, it was 1 % slower with bf16 gradients (5.03
// against 4.98 ms) and 2 % slower with fp32 ones (GPT-2-Large, 0.114 against
// 0.111 ms).
template <typename GT, int NMAX, bool BF16, int CH, int S>
__global__ void __launch_bounds__(kBlock) reduce_scatter_bulk_kernel(const Tile* __restrict__ tiles,
                                                                     int64_t ntiles, GradPtrs<NMAX> gp,
                                                                     ReduceArgs a, float* __restrict__ gshard,
                                                                     int32_t* kstatus) {
    asm volatile("griddepcontrol.wait;" ::: "memory");   // no early release (see the fused kernel)
    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem);
    unsigned char* ring = smem + 128;
    const int tid = threadIdx.x;
    const int groups = a.groups;
    const int W = a.F * groups;
    const float fW = static_cast<float>(W);
    const bool acc = a.accumulate != 0;
    const size_t rows_bytes = static_cast<size_t>(CH) * W * sizeof(GT);
    const size_t sbytes = rows_bytes + (acc ? static_cast<size_t>(CH) * 4 : 0);
    const uint32_t elem_bytes = static_cast<uint32_t>(W * sizeof(GT) + (acc ? 4 : 0));
    if (tid == 0) {
        for (int s = 0; s < S; ++s) mbar_init(&full[s], 1);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();

    int64_t pt = blockIdx.x;
    int64_t pc = 0;
    Body pb{};
    bool pb_valid = false;
    uint32_t issued = 0, consumed = 0;
    uint32_t withheld = 0xFFFFFFFFu;   // the stage armed without copies (a.withhold), if any
    const unsigned long long limit = wait_limit(a);
    auto top_up = [&]() {
        while (issued - consumed < static_cast<uint32_t>(S) && pt < ntiles) {
            if (!pb_valid) {
                pb = tile_body(tiles[pt]);
                pb_valid = true;
            }
            const int64_t nch = (pb.n + CH - 1) / CH;
            if (pc >= nch) {
                pt += gridDim.x;
                pc = 0;
                pb_valid = false;
                continue;
            }
            const int64_t off = pc * CH;
            const uint32_t n = static_cast<uint32_t>(pb.n - off < CH ? pb.n - off : CH);
            const int s = static_cast<int>(issued % S);
            unsigned char* st = ring + s * sbytes;
            mbar_expect_tx(&full[s], n * elem_bytes);
            if (a.withhold != 0 && blockIdx.x == 0 && issued == 0) {
                withheld = issued;   // nothing will complete this stage: its wait runs out
            } else {
                for (int r = 0; r < W; ++r)
                    bulk_g2s(st + static_cast<size_t>(r) * CH * sizeof(GT),
                             static_cast<const GT*>(gp.p[r]) + pb.ga + off, n * sizeof(GT), &full[s]);
                if (acc) bulk_g2s(st + rows_bytes, gshard + pb.sa + off, n * 4, &full[s]);
            }
            ++issued;
            ++pc;
        }
    };

    bool ok = true;
    bool bad = false;
    for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
        const Tile tl = tiles[t];
        const Body b = tile_body(tl);
        int j = -1;
        if (tid < b.head) j = tid;
        else if (tid >= 16 && tid < 16 + b.tail) j = b.head + static_cast<int>(b.n) + (tid - 16);
        if (j >= 0) {
            float x = reduce1<GT, NMAX, BF16>(gp, a, groups, fW, tl.g + j);
            if (a.scale) x = __fmul_rn(x, a.inv_scale);
            if (acc) x = __fadd_rn(gshard[tl.s + j], x);
            bad |= not_finite(x);
            gshard[tl.s + j] = x;
        }
        const int64_t nch = (b.n + CH - 1) / CH;
        for (int64_t ch = 0; ch < nch; ++ch) {
            if (tid == 0) top_up();
            const int s = static_cast<int>(consumed % S);
            const uint32_t parity = (consumed / S) & 1u;
            const bool got = mbar_wait(&full[s], parity, limit);
            const int64_t off = ch * CH;
            const int64_t n = b.n - off < CH ? b.n - off : CH;
            for (int e = tid * 4; got && e < n; e += 4 * kBlock) {
                const unsigned char* st = ring + s * sbytes;
                float G[4];
                reduce4_smem<GT, BF16, CH>(st, a.F, groups, fW, e, G);
                if (a.scale) {
#pragma unroll
                    for (int k = 0; k < 4; ++k) G[k] = __fmul_rn(G[k], a.inv_scale);
                }
                if (acc) {
                    const float4 o = *reinterpret_cast<const float4*>(st + rows_bytes + static_cast<size_t>(e) * 4);
                    G[0] = __fadd_rn(o.x, G[0]);
                    G[1] = __fadd_rn(o.y, G[1]);
                    G[2] = __fadd_rn(o.z, G[2]);
                    G[3] = __fadd_rn(o.w, G[3]);
                }
#pragma unroll
                for (int k = 0; k < 4; ++k) bad |= not_finite(G[k]);
                *reinterpret_cast<float4*>(gshard + b.sa + off + e) = make_float4(G[0], G[1], G[2], G[3]);
            }
            ++consumed;
            ok = __syncthreads_and(got) != 0;
            if (!ok) break;
        }
        if (!ok) break;
    }
    if (!ok && tid == 0) {
        atomicOr(kstatus, FSDP_KSTATUS_WAIT_TIMEOUT);
        for (uint32_t q = consumed - 1; q < issued; ++q) {
            if (q == withheld && a.withhold == 1) continue;   // armed, but no copy was issued
            if (!mbar_wait(&full[q % S], (q / S) & 1u, limit)) atomicOr(kstatus, FSDP_KSTATUS_DRAIN_TIMEOUT);
        }
    }
    if (__syncthreads_or(bad) && tid == 0 && a.found != nullptr) *a.found = 1;
}

// A bounded wait on a barrier that nothing completes: exercises the limit
// and the status path of mbar_wait without any copy in flight.
__global__ void wait_selftest_kernel(int32_t* status, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);   // expects one arrival, which never comes
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    const bool got = mbar_wait(&bar, 0, limit_ns);
    if (__syncthreads_and(got) == 0 && threadIdx.x == 0) atomicOr(status, FSDP_KSTATUS_WAIT_TIMEOUT);
}

// Grid policy: one CTA per tile (segment kernels) or per 256 groups of 8
// elements (flat kernels), launched in order, instead of a persistent grid
// that strides over the work.  Measured on GB300 with the minGPT unit, the
// AdamW pass moved 7.15 TB/s this way against 6.38 TB/s as a persistent
// grid-stride loop: short CTAs retire and start continuously, so loads,
// arithmetic and stores of different CTAs overlap instead of advancing in
// lockstep.  The kernels still loop, so any grid size is correct.
unsigned grid_for(int64_t work) {
    const int64_t cap = 0x7FFFFFFF;
    if (work < 1) return 1;
    return static_cast<unsigned>(work < cap ? work : cap);
}

// Launch `kernel` on `grid` CTAs of `block` threads with programmatic stream
// serialization (see pdl_enter).
// Raise `kernel`'s dynamic shared-memory limit to the staged kernels' most,
// once per kernel and device (the attribute belongs to the device's context).
// `done` is the caller's per-kernel array of flags; a benign race at worst
// repeats the idempotent call.
constexpr int kMaxDevices = 64;

template <typename... KArgs>
cudaError_t allow_staged_smem(void (*kernel)(KArgs...), int* done) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < kMaxDevices && done[dev]) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 128 + kStages * kStageMaxBytes);
    if (e == cudaSuccess && dev >= 0 && dev < kMaxDevices) done[dev] = 1;
    return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_smem(void (*kernel)(KArgs...), unsigned grid, unsigned block, size_t smem,
                            cudaStream_t st, Args... args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(block);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t st,
                       Args... args) {
    return launch_pdl_smem(kernel, grid, block, 0, st, args...);
}

}  // namespace

cudaError_t launch_shard_in(const Tile* tiles, int64_t ntiles, const ParamSrc* params,
                            float* master, uint16_t* shadow, cudaStream_t st) {
    if (ntiles == 0) return cudaSuccess;
    return launch_pdl(shard_in_kernel, grid_for(ntiles), kBlock, st, tiles, ntiles, params, master,
                      shadow);
}

cudaError_t launch_gather(const Tile* tiles, int64_t ntiles, const float* master, uint16_t* out, cudaStream_t st,
                          bool overlap) {
    if (ntiles == 0) return cudaSuccess;
    return launch_pdl(gather_cast_kernel, grid_for(ntiles), kBlock, st, tiles, ntiles, master, out,
                      overlap ? 1 : 0);
}

cudaError_t launch_gather_shadow(const Tile* tiles, int64_t ntiles, const uint16_t* shadow,
                                 uint16_t* out, cudaStream_t st, bool overlap) {
    if (ntiles == 0) return cudaSuccess;
    return launch_pdl(gather_shadow_kernel, grid_for(ntiles), kBlock, st, tiles, ntiles, shadow, out,
                      overlap ? 1 : 0);
}

cudaError_t launch_cast_range(const float* master, uint16_t* shadow, int64_t begin, int64_t n, cudaStream_t st) {
    const int64_t n8 = n / 8;
    if (n8 == 0) return cudaSuccess;
    return launch_pdl(cast_range_kernel, grid_for((n8 + kBlock - 1) / kBlock), kBlock, st, master + begin,
                      shadow + begin, n8);
}

// Stages and chunk of the staged reduce-scatter for `bpe` stage bytes per
// element.  Three CTAs per SM (each at most 75 KB) matter most: two stages of
// 2048 elements when they fit that budget, else three stages of 1024 when
// those do, else two stages of at most 56 KB as for the fused kernel.
// Measured on the minGPT unit (bf16 gradients, W = 8): accumulating (20 bytes
// per element) 5.88 ms with 3 x 1024 against 6.10 with 2 x 2048 (2 CTAs per
// SM); the flag or unscale alone (16 bytes) 5.04 ms with 2 x 2048 against
// 5.08 with 3 x 1024; two replication groups (32 bytes) 9.18 ms with
// 2 x 1024 against 10.70 with 3 x 1024 (2 CTAs per SM).
constexpr int kThreeCtaBytes = 76800;
struct StagePlan {
    int stages;
    int chunk;
};
constexpr StagePlan rs_plan(int bpe) {
    return 2 * 2048 * bpe <= kThreeCtaBytes   ? StagePlan{2, 2048}
           : 3 * 1024 * bpe <= kThreeCtaBytes ? StagePlan{3, 1024}
                                              : StagePlan{2, chunk_for(bpe)};
}

template <typename GT, int NMAX, bool BF16, int CH, int S>
static cudaError_t launch_rs_bulk(const Tile* tiles, int64_t ntiles, const GradPtrs<NMAX>& gp,
                                  const ReduceArgs& a, float* gshard, int32_t* kstatus, cudaStream_t st) {
    static int done[kMaxDevices] = {};
    cudaError_t e = allow_staged_smem(reduce_scatter_bulk_kernel<GT, NMAX, BF16, CH, S>, done);
    if (e != cudaSuccess) return e;
    const int W = a.F * a.groups;
    const size_t smem = 128 + static_cast<size_t>(S) * CH * (W * sizeof(GT) + (a.accumulate ? 4 : 0));
    return launch_pdl_smem(reduce_scatter_bulk_kernel<GT, NMAX, BF16, CH, S>, grid_for(ntiles), kBlock, smem, st,
                           tiles, ntiles, gp, a, gshard, kstatus);
}

template <typename GT, int NMAX, bool BF16, bool EXT>
static cudaError_t launch_rs_t(const Tile* tiles, int64_t ntiles, const void* const* grads,
                               const ReduceArgs& a, float* gshard, int32_t* kstatus, cudaStream_t st) {
    GradPtrs<NMAX> gp;
    const int W = a.F * a.groups;
    for (int r = 0; r < NMAX; ++r) gp.p[r] = r < W ? grads[r] : nullptr;
    if constexpr (NMAX <= 64) {
        if (EXT) {   // the plain form is faster register-staged
            const StagePlan sp = rs_plan(W * static_cast<int>(sizeof(GT)) + (a.accumulate ? 4 : 0));
            if (sp.stages == 3) return launch_rs_bulk<GT, NMAX, BF16, 1024, 3>(tiles, ntiles, gp, a, gshard, kstatus, st);
            if (sp.chunk == 2048) return launch_rs_bulk<GT, NMAX, BF16, 2048, 2>(tiles, ntiles, gp, a, gshard, kstatus, st);
            if (sp.chunk == 1024) return launch_rs_bulk<GT, NMAX, BF16, 1024, 2>(tiles, ntiles, gp, a, gshard, kstatus, st);
            if (sp.chunk == 512) return launch_rs_bulk<GT, NMAX, BF16, 512, 2>(tiles, ntiles, gp, a, gshard, kstatus, st);
        }
    }
    // 16-byte-aligned gradients: fp32 groups load as two 16-byte halves, and
    // the plain bf16 form drops from 16-wide (32-byte) to 8-wide groups; the
    // extended bf16 form already loads 16 bytes at a time
    if constexpr (std::is_same<GT, float>::value || !EXT) {
        if (a.narrow)
            return launch_pdl(reduce_scatter_kernel<GT, NMAX, BF16, EXT, true>, grid_for(ntiles), kBlock, st, tiles,
                              ntiles, gp, a, gshard);
    }
    return launch_pdl(reduce_scatter_kernel<GT, NMAX, BF16, EXT, false>, grid_for(ntiles), kBlock, st, tiles, ntiles,
                      gp, a, gshard);
}

template <typename GT, int NMAX, bool BF16>
static cudaError_t launch_rs_ext(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                 const ReduceArgs& a, float* gshard, int32_t* ks, cudaStream_t st) {
    const bool ext = a.groups > 1 || a.scale || a.accumulate || a.found != nullptr;
    return ext ? launch_rs_t<GT, NMAX, BF16, true>(tiles, ntiles, grads, a, gshard, ks, st)
               : launch_rs_t<GT, NMAX, BF16, false>(tiles, ntiles, grads, a, gshard, ks, st);
}

template <typename GT>
static cudaError_t launch_rs_dt(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                const ReduceArgs& a, float* gshard, int32_t* ks, cudaStream_t st) {
    const bool small = a.F * a.groups <= 64;
    if (a.bf16_reduce)
        return small ? launch_rs_ext<GT, 64, true>(tiles, ntiles, grads, a, gshard, ks, st)
                     : launch_rs_ext<GT, kMaxRanks, true>(tiles, ntiles, grads, a, gshard, ks, st);
    return small ? launch_rs_ext<GT, 64, false>(tiles, ntiles, grads, a, gshard, ks, st)
                 : launch_rs_ext<GT, kMaxRanks, false>(tiles, ntiles, grads, a, gshard, ks, st);
}

cudaError_t launch_reduce_scatter(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                  int grad_dtype, const ReduceArgs& a, float* gshard, int32_t* kstatus,
                                  cudaStream_t st) {
    if (ntiles == 0) return cudaSuccess;
    if (grad_dtype == FSDP_DTYPE_BF16)
        return launch_rs_dt<uint16_t>(tiles, ntiles, grads, a, gshard, kstatus, st);
    return launch_rs_dt<float>(tiles, ntiles, grads, a, gshard, kstatus, st);
}

// The staged kernel needs more than the default 48 KB of dynamic shared
// memory: raise the kernel's limit once per instantiation and device.
template <typename GT, int NMAX, bool BF16, bool HYBRID, int CH>
static cudaError_t bulk_smem_attr() {
    static int done[kMaxDevices] = {};
    return allow_staged_smem(reduce_adamw_bulk_kernel<GT, NMAX, BF16, HYBRID, CH>, done);
}

template <typename GT, int NMAX, bool BF16, bool HYBRID, int CH>
static cudaError_t launch_bulk(const Tile* tiles, int64_t ntiles, const GradPtrs<NMAX>& gp, const ReduceArgs& a,
                               float* gshard, float* p, float* m, float* v, uint16_t* shadow,
                               const StepSource& c, int32_t* kstatus, cudaStream_t st) {
    const int W = a.F * a.groups;
    const size_t smem = 128 + static_cast<size_t>(kStages) * CH * (W * sizeof(GT) + 12);
    cudaError_t e = bulk_smem_attr<GT, NMAX, BF16, HYBRID, CH>();
    if (e != cudaSuccess) return e;
    return launch_pdl_smem(reduce_adamw_bulk_kernel<GT, NMAX, BF16, HYBRID, CH>, grid_for(ntiles), kBlock, smem,
                           st, tiles, ntiles, gp, a, gshard, p, m, v, shadow, c, kstatus);
}

template <typename GT, int NMAX, bool BF16, bool HYBRID>
static cudaError_t launch_bulk_ch(int ch, const Tile* tiles, int64_t ntiles, const GradPtrs<NMAX>& gp,
                                  const ReduceArgs& a, float* gshard, float* p, float* m, float* v,
                                  uint16_t* shadow, const StepSource& c, int32_t* kstatus, cudaStream_t st) {
    if (ch == 2048)
        return launch_bulk<GT, NMAX, BF16, HYBRID, 2048>(tiles, ntiles, gp, a, gshard, p, m, v, shadow, c, kstatus, st);
    if (ch == 1024)
        return launch_bulk<GT, NMAX, BF16, HYBRID, 1024>(tiles, ntiles, gp, a, gshard, p, m, v, shadow, c, kstatus, st);
    return launch_bulk<GT, NMAX, BF16, HYBRID, 512>(tiles, ntiles, gp, a, gshard, p, m, v, shadow, c, kstatus, st);
}

template <typename GT, int NMAX, bool BF16>
static cudaError_t launch_ra_t(const Tile* tiles, int64_t ntiles, const void* const* grads,
                               const ReduceArgs& a, float* gshard, float* p, float* m, float* v,
                               uint16_t* shadow, const StepSource& c, int32_t* kstatus, cudaStream_t st) {
    GradPtrs<NMAX> gp;
    const int W = a.F * a.groups;
    for (int r = 0; r < NMAX; ++r) gp.p[r] = r < W ? grads[r] : nullptr;
    if constexpr (NMAX <= 64) {   // wider units never fit a stage
        const int ch = chunk_for(W * static_cast<int>(sizeof(GT)) + 12);
        if (ch > 0) {
            if (a.groups > 1)
                return launch_bulk_ch<GT, NMAX, BF16, true>(ch, tiles, ntiles, gp, a, gshard, p, m, v, shadow, c,
                                                            kstatus, st);
            return launch_bulk_ch<GT, NMAX, BF16, false>(ch, tiles, ntiles, gp, a, gshard, p, m, v, shadow, c,
                                                         kstatus, st);
        }
    }
    if constexpr (std::is_same<GT, float>::value) {   // 16-byte-aligned fp32 gradients
        if (a.narrow) {
            if (a.groups > 1)
                return launch_pdl(reduce_adamw_kernel<GT, NMAX, BF16, true, true>, grid_for(ntiles), kBlock, st,
                                  tiles, ntiles, gp, a, gshard, p, m, v, shadow, c);
            return launch_pdl(reduce_adamw_kernel<GT, NMAX, BF16, false, true>, grid_for(ntiles), kBlock, st,
                              tiles, ntiles, gp, a, gshard, p, m, v, shadow, c);
        }
    }
    if (a.groups > 1)
        return launch_pdl(reduce_adamw_kernel<GT, NMAX, BF16, true, false>, grid_for(ntiles), kBlock, st, tiles,
                          ntiles, gp, a, gshard, p, m, v, shadow, c);
    return launch_pdl(reduce_adamw_kernel<GT, NMAX, BF16, false, false>, grid_for(ntiles), kBlock, st, tiles,
                      ntiles, gp, a, gshard, p, m, v, shadow, c);
}

template <typename GT>
static cudaError_t launch_ra_dt(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                const ReduceArgs& a, float* gshard, float* p, float* m, float* v,
                                uint16_t* shadow, const StepSource& c, int32_t* ks, cudaStream_t st) {
    const bool small = a.F * a.groups <= 64;
    if (a.bf16_reduce)
        return small ? launch_ra_t<GT, 64, true>(tiles, ntiles, grads, a, gshard, p, m, v, shadow, c, ks, st)
                     : launch_ra_t<GT, kMaxRanks, true>(tiles, ntiles, grads, a, gshard, p, m, v, shadow, c, ks, st);
    return small ? launch_ra_t<GT, 64, false>(tiles, ntiles, grads, a, gshard, p, m, v, shadow, c, ks, st)
                 : launch_ra_t<GT, kMaxRanks, false>(tiles, ntiles, grads, a, gshard, p, m, v, shadow, c, ks, st);
}

cudaError_t launch_reduce_adamw(const Tile* tiles, int64_t ntiles, const void* const* grads,
                                int grad_dtype, const ReduceArgs& a, float* gshard, float* p, float* m,
                                float* v, uint16_t* shadow, const StepSource& c, int32_t* kstatus,
                                cudaStream_t st) {
    if (ntiles == 0) return cudaSuccess;
    if (grad_dtype == FSDP_DTYPE_BF16)
        return launch_ra_dt<uint16_t>(tiles, ntiles, grads, a, gshard, p, m, v, shadow, c, kstatus, st);
    return launch_ra_dt<float>(tiles, ntiles, grads, a, gshard, p, m, v, shadow, c, kstatus, st);
}

cudaError_t launch_wait_selftest(int32_t* status, unsigned long long limit_ns, cudaStream_t st) {
    return launch_pdl(wait_selftest_kernel, 1, 32, st, status, limit_ns);
}

cudaError_t launch_adamw(int64_t n8, float* p, const float* g, float* m, float* v,
                         uint16_t* shadow, const StepSource& c, cudaStream_t st) {
    if (n8 == 0) return cudaSuccess;
    return launch_pdl(adamw_kernel, grid_for((n8 + kBlock - 1) / kBlock), kBlock, st, n8, p, g, m, v, shadow,
                      c);
}

cudaError_t launch_advance_step(int64_t* counter, int64_t count, cudaStream_t st) {
    return launch_pdl(advance_step_kernel, 1, 1, st, counter, count);
}

}  // namespace fsdp
