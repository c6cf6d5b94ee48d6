// Host-side layout planning: FLAT and DIM0 both become one table of
// segments (rank, global range, arena range) and the kernels' tile tables.
#pragma once

#include <cstdint>
#include <string>
#include <vector>

#include "fsdp_unit.h"

namespace fsdp {

// A rank's arena slot and the global index it holds agree modulo kAlign
// elements, so an 8-element group that is aligned in the unsharded buffer is
// aligned in the arena too (32-byte fp32 / 16-byte bf16 vector accesses).
constexpr int64_t kAlign = 32;

// Kernel work unit: tile boundaries sit at global multiples of kTile, so a
// tile never spans two segments and never crosses a kTile boundary.
constexpr int64_t kTile = 8192;

constexpr int kMaxRanks = 1024;
constexpr int kMaxDims = 8;

struct ParamInfo {
    int64_t numel = 0;
    int64_t rows = 0;      // dim-0 size (1 for a 0-d parameter)
    int64_t row_len = 0;   // elements per dim-0 row
    int64_t offset = 0;    // FlatParameter offset
};

struct Plan {
    int layout = 0;
    int N = 0;
    int64_t P = 0;
    std::vector<ParamInfo> params;
    std::vector<fsdp_segment> segs;     // rank-major, rank storage order
    std::vector<int64_t> rank_first_seg;  // N+1 entries: segs of rank k are [first[k], first[k+1])
    std::vector<int64_t> shard_len;     // per rank, owned elements
    std::vector<int64_t> layout_pad;    // per rank, padding the layout stores (FLAT_PADDED)
    std::vector<int64_t> arena_len;     // per rank, multiple of kAlign
    std::vector<int64_t> arena_base;    // per rank, offset in the slab (multiple of kAlign)
    int64_t slab_len = 0;               // sum of arena_len
};

// Work tile for the segment-driven kernels: `len` elements from global index
// `g` live at slab index `s`; `aux` is the parameter index (load tiles) or 0.
struct Tile {
    int64_t g;
    int64_t s;
    int32_t len;
    int32_t aux;
};
static_assert(sizeof(Tile) == 24, "Tile layout is shared with the kernels");

// Returns FSDP_OK or an FSDP_E_* code with a reason in *err.
int build_plan(int nparams, const int* ndims, const int64_t* dims, int layout, int N,
               Plan* out, std::string* err);

// Tiles over every segment (gather, reduce-scatter).
void build_tiles(const Plan& plan, std::vector<Tile>* tiles);

// Tiles over every segment, additionally cut at parameter boundaries, with
// aux = parameter index (shard-in from per-parameter buffers).
void build_load_tiles(const Plan& plan, std::vector<Tile>* tiles);

}  // namespace fsdp
