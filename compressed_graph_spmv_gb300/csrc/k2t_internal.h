// k2t_internal.h -- structures shared by the host builder (k2t_host.cpp) and
// the device side (k2t_device.cu).  Not part of the public ABI.
#pragma once

#include <cstdint>
#include <vector>

#include "../../include/k2t.h"

namespace k2t {

constexpr uint32_t kDirS = 256;        // directory sample period (section 3.2: S = 256)
constexpr uint32_t kMaxChunkCap = 512;
constexpr uint32_t kArenaAlign = 256;
constexpr uint32_t kBandChunkNodes = 16384;  // BANDED: nodes per thread block at most
// leaf_k 0 (automatic): 4x4 leaves when 2x2 leaves would average at least this
// many non-zeros (measured: 1.0-1.04 per 2x2 leaf favours 2x2, 2.1 favours 4x4)
constexpr double kAutoLeaf4Density = 1.75;
// Heavy plus-times outputs (more non-zeros than one fp32 sum may hold within
// the bound |y - y_ref| <= 1e-5 * sum|w x| + 1e-6): each is summed in 2^bits
// fp32 partial sums, a term going to the partial that a multiplicative hash
// of its leaf's first input run picks; or in an fp64 slot of two rows
// (bits = kHeavyFp64).  Its record (one uint32 per output, 0 for the others)
// is (first row << 5) | bits, rows of max_batch fp32 words.
constexpr uint32_t kDefaultHeavyTerms = 160;
constexpr uint32_t kHeavyHash = 2654435761u;
constexpr uint32_t kHeavyFp64 = 31u;
constexpr uint32_t kHeavyMaxBits = 22;
constexpr uint64_t kHeavyMaxRows = 1ull << 27;   // rows a record can address

#ifdef __CUDACC__
#define K2T_HD __host__ __device__
#else
#define K2T_HD
#endif

// Partial sum (of 2^bits, 1 <= bits <= 31) of a heavy output that the terms of
// a leaf whose first input (column for right products, row for left ones) is
// `in` go to: the top bits of run * kHeavyHash, run = in >> kHeavyRunBits.
// The inputs of one aligned run of 32 (a leaf never straddles two) share a
// partial, so the terms a warp meets close together in Z-order land on few
// partial sums, while the hash spreads the runs over all of them.  The builder
// counts the terms of every partial with this function, the kernels route
// with it.
constexpr uint32_t kHeavyRunBits = 5;
K2T_HD inline uint32_t heavy_partial(uint32_t in, uint32_t bits)
{
    return ((in >> kHeavyRunBits) * kHeavyHash) >> (32u - bits);
}

// Coordinates of a node's block, in units of the block side at its level.
// A frontier entry: (row, col) instead of the pages' Morton code; the two
// carry the same bits, but a pair needs no deinterleave at the leaves.
struct Coord { uint32_t r, c; };

// One launch of the level-synchronous engine.
struct LsStep {
    uint8_t kind;      // 0 expand, 1 leaf
    uint8_t level;     // level of the parents
    uint8_t src;       // 0xff: host-expanded top; else level whose buffer holds the codes
    uint8_t pad;
    uint32_t a;        // first node (index within its level)
    uint32_t count;    // nodes in the tile
    uint32_t src_base; // level index of slot 0 of the source buffer
    uint32_t dst_base; // level index of slot 0 of the destination buffer (= first child)
};

inline uint64_t align_up(uint64_t v, uint64_t a) { return (v + a - 1) / a * a; }

// Byte offsets of every part inside the device arena.
struct ArenaLayout {
    uint64_t sig_off[K2T_MAX_LEVELS];   // levels d0..l-1 (l-1 = L)
    uint64_t sig_bytes[K2T_MAX_LEVELS];
    uint64_t dir_off[K2T_MAX_LEVELS];   // levels d0..l-2
    uint64_t dir_bytes[K2T_MAX_LEVELS];
    uint64_t top_off, top_bytes;
    uint64_t cached_off, cached_bytes;
    uint64_t chunk_off, chunk_bytes;
    uint64_t bleaf_off, bleaf_bytes;    // BANDED: first leaf of each band-ordered node
    uint64_t bsig_off, bsig_bytes;      // BANDED: signatures in band order
    uint64_t bchunk_off, bchunk_bytes;  // BANDED: (band, first node, node count) per block
    uint64_t root_off, root_bytes;
    uint64_t buf_off[K2T_MAX_LEVELS];   // LEVELSYNC frontier buffers (levels d0+1..l-2)
    uint64_t buf_bytes;                 // per buffer
    uint64_t scan_off, scan_bytes;      // LEVELSYNC scan space (block sums + prefixes)
    uint64_t err_off, err_bytes;        // device error word
    uint64_t vec_off[2], vec_bytes;     // host-product x and y
    // heavy outputs of plus-times products, per direction (0 right, 1 left)
    uint64_t hdir_off[2], hdir_bytes[2];    // per output up to the last heavy one: its record
    uint64_t hlist_off[2], hlist_bytes[2];  // the heavy outputs, ascending
    uint64_t acc_off, acc_bytes;            // rows of the heavy sums, shared by both directions
    uint64_t total;
};

struct DeviceState;  // defined in k2t_device.cu

}  // namespace k2t

struct k2t_tree {
    k2t_opts opts;
    uint64_t n_rows = 0, n_cols = 0, nnz = 0;
    int dim_bits = 0, n_k4 = 0, levels = 0;
    int leaf_k4 = 0;       // 1: the leaf level holds 4x4 bitmaps (16-bit signatures)
    int d0 = 0;
    uint32_t engine = 0;   // resolved engine
    bool empty = false;    // nnz == 0: a product is only the fill
    std::vector<uint64_t> nodes;                  // N_d
    // Signatures: k = 2 levels hold 16 nibbles per word (node t at bits
    // 4*(t%16)); k = 4 levels (the n_k4 top levels, and the leaf level when
    // leaf_k4) hold 4 16-bit signatures per word.
    std::vector<std::vector<uint64_t>> sig;
    std::vector<std::vector<uint32_t>> dir;       // index d - d0, levels d0..l-2
    std::vector<k2t::Coord> top;                  // level d0
    std::vector<k2t::Coord> cached;               // level l-2 (k^2+F; banded: in band order)
    // BANDED: level l-2 regrouped by row band
    std::vector<uint32_t> bleaf;                  // first leaf of each node
    std::vector<uint64_t> bsig;                   // signatures, 16 nibbles per word
    std::vector<uint32_t> bchunks;                // per block: band, first node, count
    uint32_t band_shift = 0;                      // band of a node = node row >> band_shift
    // FUSED plan: per chunk, [root index, d_c, (start, count) for levels d0..l-1]
    std::vector<uint32_t> chunks;
    uint32_t chunk_stride = 0;
    uint64_t n_chunks = 0;
    std::vector<k2t::Coord> roots;                // top entries, then roots of split chunks
    // LEVELSYNC plan
    std::vector<k2t::LsStep> steps;
    uint64_t max_tile_nodes = 0;
    // Heavy plus-times outputs (more than opts.heavy_terms non-zeros),
    // per direction (0: rows, outputs of right products; 1: columns):
    std::vector<uint32_t> hlist[2];   // the outputs, ascending
    std::vector<uint32_t> hdir[2];    // record of every output below the last heavy one + padding
    uint64_t hrows[2] = {0, 0};       // accumulator rows of the direction
    uint64_t hparts[2] = {0, 0};      // fp32 partial sums of the direction
    uint64_t hfp64[2] = {0, 0};       // outputs of the direction summed in fp64 alone
    uint32_t hmax_part[2] = {0, 0};   // largest term count of one fp32 partial sum
    k2t::ArenaLayout layout{};
    k2t::DeviceState *dev = nullptr;
};

namespace k2t {
// implemented in k2t_host.cpp
uint64_t level_offset(const k2t_tree *t, int d, uint64_t node);  // first child of node (d0 <= d <= l-2)
uint32_t level_sig(const k2t_tree *t, int d, uint64_t node);
inline bool level_is_k4(const k2t_tree *t, int d) { return d < t->n_k4 || (t->leaf_k4 && d == t->levels - 1); }
void compute_layout(k2t_tree *t);
void level_directory(const k2t_tree *t, int d, std::vector<uint32_t> &dir, int nt);
// implemented in k2t_device.cu
void device_release(k2t_tree *t);
// A tree from the sorted distinct path keys of its cells (plain k = 2 levels;
// key of cell (r, c): r's bits at odd positions, c's at even ones), as
// k2t_build would make it from those cells with opts: the device-side
// product of two trees hands its result over this way.  Errors as
// k2t_build, EINVAL for keys out of order or past the padded side.
int build_from_sorted_keys(const uint64_t *keys, uint64_t m, uint64_t n_rows, uint64_t n_cols, const k2t_opts *opts,
                           k2t_tree **out);
}  // namespace k2t
