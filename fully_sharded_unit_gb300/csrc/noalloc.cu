// fsdp_reduce_scatter_flat_noalloc: a reduce-scatter that allocates no device
// memory (declared in include/fsdp_unit.h).
//
// Every segment-driven kernel of this library walks a table of work tiles in
// device memory.  A unit allocates its table once, at creation, next to its
// shard arenas.  This entry point needs no unit: the caller passes the
// gradients and one output buffer, and the tile table lives in the file-scope
// device array below, which the CUDA runtime reserves on every device that
// loads the library, for the life of the process.  Host code cannot use the
// array's name as a device address (in host code it names a host-side stand-
// in), so the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and keeps it.
//
// The table is filled on the host into a static staging array and copied
// into the device array with cudaMemcpyAsync on the caller's stream (a
// pageable-source copy returns once the bytes are staged, so the staging
// array can be reused at once).  The copy and the kernel are stream-ordered,
// so calls on one stream follow each other correctly; calls that overlap on
// the GPU (different streams, no ordering between them) share the one table
// and race.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>
#include <string>

#include "fsdp_unit.h"
#include "kernels.hpp"
#include "plan.hpp"

namespace fsdp {
// Records the calling thread's failure reason for fsdp_last_error (api.cu).
int record_error(int code, const std::string& why);
}  // namespace fsdp

namespace {

int nofail(int code, const std::string& why) { return fsdp::record_error(code, why); }

constexpr int64_t kMaxTiles = FSDP_NOALLOC_MAX_TILES;
static_assert(kMaxTiles * static_cast<int64_t>(sizeof(fsdp::Tile)) == 786432, "768 KiB of scratch");

// The scratch: the tile table of the call in flight.
static __device__ __align__(256) fsdp::Tile g_noalloc_tiles[kMaxTiles];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;                          // guards the two arrays below
void* g_tiles_addr[kMaxDevices] = {};        // device address of g_noalloc_tiles, per device
fsdp::Tile g_staging[kMaxTiles];             // host staging of the table


// Tiles of the FLAT layout written straight to the unsharded output: rank k's
// elements [floor(kP/N), floor((k+1)P/N)) cut at multiples of kTile, each
// tile's output slot equal to its global index.  Returns the tile count; when
// `dst` is null only counts.
int64_t flat_tiles(int64_t P, int N, fsdp::Tile* dst) {
    int64_t n = 0;
    for (int k = 0; k < N; ++k) {
        const int64_t a = static_cast<int64_t>((static_cast<__int128>(k) * P) / N);
        const int64_t b = static_cast<int64_t>((static_cast<__int128>(k + 1) * P) / N);
        for (int64_t g = a; g < b;) {
            const int64_t next = (g / fsdp::kTile + 1) * fsdp::kTile;
            const int64_t len = (b < next ? b : next) - g;
            if (dst != nullptr) dst[n] = fsdp::Tile{g, g, static_cast<int32_t>(len), 0};
            ++n;
            g += len;
        }
    }
    return n;
}

}  // namespace

extern "C" {

int fsdp_reduce_scatter_flat_noalloc(const void* const* grads_dev, int num_ranks, int grad_dtype,
                                     int64_t numel, float* out_dev, void* stream) {
    if (num_ranks < 1 || num_ranks > fsdp::kMaxRanks)
        return nofail(FSDP_E_INVALID_ARG, "num_ranks must be in [1, 1024]");
    if (grad_dtype != FSDP_DTYPE_F32 && grad_dtype != FSDP_DTYPE_BF16)
        return nofail(FSDP_E_INVALID_ARG, "grad_dtype must be FSDP_DTYPE_F32 or FSDP_DTYPE_BF16");
    if (numel < 1) return nofail(FSDP_E_INVALID_ARG, "numel must be >= 1");
    if (grads_dev == nullptr || out_dev == nullptr)
        return nofail(FSDP_E_INVALID_ARG, "grads_dev and out_dev must be non-null");
    for (int r = 0; r < num_ranks; ++r) {
        if (grads_dev[r] == nullptr) return nofail(FSDP_E_INVALID_ARG, "a gradient pointer is null");
        if (reinterpret_cast<uintptr_t>(grads_dev[r]) & 31u)
            return nofail(FSDP_E_ALIGN, "a gradient buffer is not 32-byte aligned");
    }
    if (reinterpret_cast<uintptr_t>(out_dev) & 31u)
        return nofail(FSDP_E_ALIGN, "the output buffer is not 32-byte aligned");
    // the bound is checked before anything touches the device; a unit of
    // more than kMaxTiles whole tiles is rejected before the count loop
    if ((numel + fsdp::kTile - 1) / fsdp::kTile > kMaxTiles)
        return nofail(FSDP_E_INVALID_ARG, "numel " + std::to_string(numel) + " needs more than the " +
                                              std::to_string(kMaxTiles) + " work tiles the scratch holds");
    const int64_t ntiles = flat_tiles(numel, num_ranks, nullptr);
    if (ntiles > kMaxTiles)
        return nofail(FSDP_E_INVALID_ARG, "numel " + std::to_string(numel) + " at " + std::to_string(num_ranks) +
                                              " ranks needs " + std::to_string(ntiles) + " work tiles; the scratch holds " +
                                              std::to_string(kMaxTiles));

    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return nofail(FSDP_E_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices) return nofail(FSDP_E_CUDA, "device ordinal beyond 63");
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_tiles_addr[dev] == nullptr) {   // set-up, once per device, with that device current
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_tiles);
        if (e != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return nofail(FSDP_E_CUDA, std::string("cudaGetSymbolAddress of the scratch table: ") +
                                           cudaGetErrorString(e));
        }
        g_tiles_addr[dev] = p;
    }
    fsdp::Tile* tiles = static_cast<fsdp::Tile*>(g_tiles_addr[dev]);
    flat_tiles(numel, num_ranks, g_staging);
    // every tile the kernel reads is written by this copy: nothing to clear
    e = cudaMemcpyAsync(tiles, g_staging, static_cast<size_t>(ntiles) * sizeof(fsdp::Tile),
                        cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return nofail(FSDP_E_CUDA, std::string("tile table copy: ") + cudaGetErrorString(e));

    fsdp::ReduceArgs a{};
    a.F = num_ranks;
    a.groups = 1;
    a.inv_scale = 1.0f;
    // the plain reduce-scatter (no options) never touches a status word
    e = fsdp::launch_reduce_scatter(tiles, ntiles, grads_dev, grad_dtype, a, out_dev, nullptr, st);
    if (e != cudaSuccess) return nofail(FSDP_E_CUDA, std::string("reduce-scatter launch: ") + cudaGetErrorString(e));
    return FSDP_OK;
}

}  // extern "C"
