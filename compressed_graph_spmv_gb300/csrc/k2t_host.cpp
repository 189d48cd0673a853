// k2t_host.cpp -- host side of the k^2-tree library: construction, planning,
// workspace accounting, statistics and decoding.
//
// Construction (the host step of section 5.1 of "A GPU Engine for Sparse
// Matrix-Vector Products on k^2-Tree-Compressed Graphs"; the pages do not
// describe its algorithm, this one is ours): every cell gets a 64-bit path
// key, the child indices of its path from the root, two bits per k = 2
// level and four per k = 4 level.  Sorting the keys sorts every level into
// level order, because level order lists the children of consecutive nodes
// consecutively (section 3, notation of Algorithm 1).  The levels are then
// produced bottom-up by grouping equal key prefixes; a group's signature is
// the OR of 1 << (child digit) over its members.
//
// Planning (sections 3.2-3.5): the host expands the top of the tree down to
// the deepest level with at most 2^16 nodes, samples the child offsets of
// every level every 256 nodes (the directory), and plans either chunks of
// whole subtrees for the fused engine or the depth-first tile sequence of
// the level-synchronous engine, with the exact scratch each needs.
#include <algorithm>
#include <cstring>
#include <functional>
#include <new>
#include <stdexcept>
#include <thread>
#include <vector>

#include "k2t_internal.h"

namespace k2t {
namespace {

int thread_count(const k2t_opts &o)
{
    if (o.threads) return (int)o.threads;
    unsigned h = std::thread::hardware_concurrency();
    return h ? (int)h : 4;
}

void parallel_for(int nt, const std::function<void(int)> &fn)
{
    if (nt <= 1) { fn(0); return; }
    std::vector<std::thread> th;
    th.reserve((size_t)nt);
    for (int t = 0; t < nt; ++t) th.emplace_back(fn, t);
    for (auto &x : th) x.join();
}

inline int popc64(uint64_t v) { return __builtin_popcountll(v); }

// bit i of v -> bit 2i
inline uint64_t spread_bits(uint32_t v)
{
    uint64_t x = v;
    x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
    x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
    x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
    x = (x | (x << 2)) & 0x3333333333333333ull;
    x = (x | (x << 1)) & 0x5555555555555555ull;
    return x;
}

// Path key of cell (r, c): interleaved bits with the row bit first in every
// pair (quadrant b = 2*b1 + b0), except that each of the first n_k4 nibbles
// (and the last nibble, for 4x4 leaves) is reordered from (r1 c1 r0 c0) to the
// row-major k = 4 digit (r1 r0 c1 c0).
inline uint64_t k4_digit(uint64_t m, int sh)
{
    uint64_t nib = (m >> sh) & 15u;
    uint64_t dig = (nib & 9u) | ((nib & 4u) >> 1) | ((nib & 2u) << 1);
    return (m & ~(15ull << sh)) | (dig << sh);
}

inline uint64_t path_key(uint32_t r, uint32_t c, int dim_bits, int n_k4, int leaf_k4)
{
    uint64_t m = (spread_bits(r) << 1) | spread_bits(c);
    for (int i = 0; i < n_k4; ++i) m = k4_digit(m, 2 * dim_bits - 4 * (i + 1));
    if (leaf_k4) m = k4_digit(m, 0);
    return m;
}

// Block coordinates of a level-d node from its path prefix.
inline Coord prefix_coord(uint64_t prefix, int d, int n_k4)
{
    int k4 = std::min(d, n_k4);
    int bits = 4 * k4 + 2 * (d - k4);
    uint64_t r = 0, c = 0;
    int pos = bits;
    for (int i = 0; i < k4; ++i) {
        pos -= 4;
        uint64_t dig = (prefix >> pos) & 15u;
        r = (r << 2) | (dig >> 2);
        c = (c << 2) | (dig & 3u);
    }
    for (int i = k4; i < d; ++i) {
        pos -= 2;
        uint64_t dig = (prefix >> pos) & 3u;
        r = (r << 1) | (dig >> 1);
        c = (c << 1) | (dig & 1u);
    }
    return Coord{(uint32_t)r, (uint32_t)c};
}

void radix_sort(std::vector<uint64_t> &a, std::vector<uint64_t> &tmp, int bits, int nt)
{
    size_t n = a.size();
    if (n < 2) return;
    tmp.resize(n);
    std::vector<size_t> hist((size_t)nt * 256);
    for (int shift = 0; shift < bits; shift += 8) {
        std::fill(hist.begin(), hist.end(), 0);
        parallel_for(nt, [&](int t) {
            size_t lo = n * t / nt, hi = n * (t + 1) / nt;
            size_t *h = &hist[(size_t)t * 256];
            for (size_t i = lo; i < hi; ++i) h[(a[i] >> shift) & 255u]++;
        });
        int used = 0;
        for (int d = 0; d < 256 && used < 2; ++d) {
            size_t s = 0;
            for (int t = 0; t < nt; ++t) s += hist[(size_t)t * 256 + d];
            used += s != 0;
        }
        if (used <= 1) continue;
        size_t run = 0;
        for (int d = 0; d < 256; ++d)
            for (int t = 0; t < nt; ++t) {
                size_t c = hist[(size_t)t * 256 + d];
                hist[(size_t)t * 256 + d] = run;
                run += c;
            }
        parallel_for(nt, [&](int t) {
            size_t lo = n * t / nt, hi = n * (t + 1) / nt;
            size_t *h = &hist[(size_t)t * 256];
            for (size_t i = lo; i < hi; ++i) tmp[h[(a[i] >> shift) & 255u]++] = a[i];
        });
        a.swap(tmp);
    }
}

// Stable compaction of a sorted array to its distinct values (into out).
size_t unique_into(const uint64_t *in, size_t n, uint64_t *out, int nt)
{
    std::vector<size_t> cnt((size_t)nt + 1, 0);
    parallel_for(nt, [&](int t) {
        size_t lo = n * t / nt, hi = n * (t + 1) / nt, c = 0;
        for (size_t i = lo; i < hi; ++i) c += (i == 0 || in[i] != in[i - 1]);
        cnt[(size_t)t + 1] = c;
    });
    for (int t = 0; t < nt; ++t) cnt[(size_t)t + 1] += cnt[(size_t)t];
    parallel_for(nt, [&](int t) {
        size_t lo = n * t / nt, hi = n * (t + 1) / nt, w = cnt[(size_t)t];
        for (size_t i = lo; i < hi; ++i)
            if (i == 0 || in[i] != in[i - 1]) out[w++] = in[i];
    });
    return cnt[(size_t)nt];
}

// Group a sorted prefix array by (value >> s): out_prefix = value >> s of each
// group, out_sig = OR of 1 << (value & (2^s - 1)).
size_t group_level(const uint64_t *in, size_t n, int s, uint64_t *out_prefix, uint16_t *out_sig, int nt)
{
    std::vector<size_t> cnt((size_t)nt + 1, 0);
    parallel_for(nt, [&](int t) {
        size_t lo = n * t / nt, hi = n * (t + 1) / nt, c = 0;
        for (size_t i = lo; i < hi; ++i) c += (i == 0 || (in[i] >> s) != (in[i - 1] >> s));
        cnt[(size_t)t + 1] = c;
    });
    for (int t = 0; t < nt; ++t) cnt[(size_t)t + 1] += cnt[(size_t)t];
    const uint64_t mask = (1ull << s) - 1;
    parallel_for(nt, [&](int t) {
        size_t lo = n * t / nt, hi = n * (t + 1) / nt, w = cnt[(size_t)t];
        size_t i = lo;
        while (i < hi) {
            if (!(i == 0 || (in[i] >> s) != (in[i - 1] >> s))) { ++i; continue; }
            uint64_t p = in[i] >> s;
            uint32_t sg = 0;
            size_t j = i;
            while (j < n && (in[j] >> s) == p) { sg |= 1u << (in[j] & mask); ++j; }
            out_prefix[w] = p;
            out_sig[w] = (uint16_t)sg;
            ++w;
            i = j;
        }
    });
    return cnt[(size_t)nt];
}

void pack_level(k2t_tree *t, int d, const uint16_t *sg, size_t n, int nt)
{
    bool k4 = level_is_k4(t, d);
    size_t per = k4 ? 4 : 16;
    size_t words = (n + per - 1) / per;
    std::vector<uint64_t> &out = t->sig[(size_t)d];
    out.assign(words + 1, 0);  // one spare word keeps partial reads in bounds
    parallel_for(nt, [&](int th) {
        size_t lo = words * th / nt, hi = words * (th + 1) / nt;
        for (size_t w = lo; w < hi; ++w) {
            uint64_t v = 0;
            for (size_t k = 0; k < per; ++k) {
                size_t i = w * per + k;
                if (i >= n) break;
                v |= (uint64_t)sg[i] << (k4 ? 16 * k : 4 * k);
            }
            out[w] = v;
        }
    });
}

void build_directory(k2t_tree *t, int d, int nt)
{
    level_directory(t, d, t->dir[(size_t)(d - t->d0)], nt);
}

}  // namespace

// Directory of a k = 2 level d <= l-2: the first child of every 256-node
// block (level-relative), then the level's child total (section 3.2).
void level_directory(const k2t_tree *t, int d, std::vector<uint32_t> &dir, int nt)
{
    uint64_t n = t->nodes[(size_t)d];
    uint64_t blocks = (n + kDirS - 1) / kDirS;
    dir.assign(blocks + 1, 0);
    const std::vector<uint64_t> &w = t->sig[(size_t)d];
    std::vector<uint64_t> sums(blocks, 0);
    parallel_for(nt, [&](int th) {
        uint64_t lo = blocks * th / nt, hi = blocks * (th + 1) / nt;
        for (uint64_t b = lo; b < hi; ++b) {
            uint64_t s = 0;
            uint64_t w0 = b * (kDirS / 16), w1 = std::min<uint64_t>((b + 1) * (kDirS / 16), (n + 15) / 16);
            for (uint64_t k = w0; k < w1; ++k) s += (uint64_t)popc64(w[k]);
            sums[b] = s;
        }
    });
    uint64_t run = 0;
    for (uint64_t b = 0; b < blocks; ++b) { dir[b] = (uint32_t)run; run += sums[b]; }
    dir[blocks] = (uint32_t)run;
}

uint32_t level_sig(const k2t_tree *t, int d, uint64_t node)
{
    if (level_is_k4(t, d)) return (uint32_t)((t->sig[(size_t)d][node / 4] >> (16 * (node % 4))) & 0xffffu);
    return (uint32_t)((t->sig[(size_t)d][node / 16] >> (4 * (node % 16))) & 15u);
}

// First child of `node` at level d (d0 <= d <= l-2), from the directory sample
// of its block plus the popcount of the signatures before it (section 3.2).
uint64_t level_offset(const k2t_tree *t, int d, uint64_t node)
{
    const std::vector<uint32_t> &dir = t->dir[(size_t)(d - t->d0)];
    uint64_t blk = node / kDirS;
    uint64_t base = dir[blk];
    const std::vector<uint64_t> &w = t->sig[(size_t)d];
    uint64_t w0 = blk * (kDirS / 16), w1 = node / 16;
    for (uint64_t k = w0; k < w1; ++k) base += (uint64_t)popc64(w[k]);
    uint64_t rem = node % 16;
    if (rem) base += (uint64_t)popc64(w[w1] & ((1ull << (4 * rem)) - 1));
    return base;
}

namespace {

// leaves (level l-1) under the level-d node range [a, b)
uint64_t count_last(const k2t_tree *t, int d, uint64_t a, uint64_t b)
{
    for (int e = d; e < t->levels - 1; ++e) {
        a = level_offset(t, e, a);
        b = level_offset(t, e, b);
    }
    return b - a;
}

// Plans the chunks of a range of top nodes into its own lists (several run
// in parallel over parts of the top level, then join_fused_plans appends
// them in order); a chunk rooted below the top stores its roots in `roots`,
// indexed from 0 within the planner.
struct FusedPlanner {
    const k2t_tree *t;
    uint64_t cap;
    std::vector<uint32_t> chunks;
    std::vector<Coord> roots;
    uint64_t n_chunks = 0;

    void emit(int d, uint64_t a, uint64_t b, const Coord *coords, bool from_top)
    {
        std::vector<uint32_t> &ch = chunks;
        size_t base = ch.size();
        ch.resize(base + t->chunk_stride, 0);
        uint32_t *rec = &ch[base];
        if (from_top) {
            rec[0] = (uint32_t)a;
        } else {
            rec[0] = (uint32_t)roots.size();
            for (uint64_t i = a; i < b; ++i) roots.push_back(coords[i - a]);
        }
        rec[1] = (uint32_t)d;
        uint64_t s = a, e = b;
        for (int lv = d; lv < t->levels; ++lv) {
            rec[2 + 2 * (lv - t->d0)] = (uint32_t)s;
            rec[3 + 2 * (lv - t->d0)] = (uint32_t)(e - s);
            if (lv + 1 < t->levels) {
                s = level_offset(t, lv, s);
                e = level_offset(t, lv, e);
            }
        }
        n_chunks++;
    }

    // nodes [a, b) of level d are whole subtrees; coords[i - a] is node i's block
    void range(int d, uint64_t a, uint64_t b, const Coord *coords, bool from_top)
    {
        uint64_t i = a;
        while (i < b) {
            if (count_last(t, d, i, i + 1) > cap) {
                uint32_t s = level_sig(t, d, i);
                uint64_t c0 = level_offset(t, d, i);
                Coord kids[4];
                int f = 0;
                for (int q = 0; q < 4; ++q)
                    if (s & (1u << q))
                        kids[f++] = Coord{2 * coords[i - a].r + (uint32_t)(q >> 1), 2 * coords[i - a].c + (uint32_t)(q & 1)};
                range(d + 1, c0, c0 + (uint64_t)f, kids, false);
                ++i;
                continue;
            }
            uint64_t lo = i + 1, hi = b;
            while (lo < hi) {
                uint64_t mid = lo + (hi - lo + 1) / 2;
                if (count_last(t, d, i, mid) <= cap) lo = mid; else hi = mid - 1;
            }
            emit(d, i, lo, coords + (i - a), from_top);
            i = lo;
        }
    }
};

struct LsPlanner {
    k2t_tree *t;
    uint64_t m;
    std::vector<uint64_t> buf_need;  // per level: largest destination tile

    void leaf_steps(int d, uint64_t a, uint64_t b, uint8_t src, uint64_t src_base)
    {
        for (uint64_t i = a; i < b; i += m) {
            uint64_t j = std::min(b, i + m);
            LsStep s{1, (uint8_t)d, src, 0, (uint32_t)i, (uint32_t)(j - i), (uint32_t)src_base, 0};
            t->steps.push_back(s);
            t->max_tile_nodes = std::max<uint64_t>(t->max_tile_nodes, j - i);
        }
    }

    void range(int d, uint64_t a, uint64_t b, uint8_t src, uint64_t src_base)
    {
        if (d == t->levels - 2) { leaf_steps(d, a, b, src, src_base); return; }
        uint64_t i = a;
        while (i < b) {
            uint64_t ci = level_offset(t, d, i);
            uint64_t lo = i + 1, hi = b;
            while (lo < hi) {
                uint64_t mid = lo + (hi - lo + 1) / 2;
                if (level_offset(t, d, mid) - ci <= m) lo = mid; else hi = mid - 1;
            }
            uint64_t j = lo;
            uint64_t cj = level_offset(t, d, j);
            LsStep s{0, (uint8_t)d, src, 0, (uint32_t)i, (uint32_t)(j - i), (uint32_t)src_base, (uint32_t)ci};
            t->steps.push_back(s);
            t->max_tile_nodes = std::max<uint64_t>(t->max_tile_nodes, j - i);
            buf_need[(size_t)d + 1] = std::max(buf_need[(size_t)d + 1], cj - ci);
            range(d + 1, ci, cj, (uint8_t)(d + 1), ci);
            i = j;
        }
    }
};

// BANDED: regroup the last internal level into 2-D tiles of band_rows rows by
// band_cols columns, tiles ordered column band first (all row bands of one
// column band, then the next), level order inside a tile; each node keeps its
// first leaf and signature.  Thread blocks take tiles (cut into blocks of at
// most kBandChunkNodes nodes) in that order, so the blocks running at the same
// time share one column band of x (L2-resident) while each keeps its row band
// of y in shared memory.
void plan_bands(k2t_tree *t, int nt)
{
    const int d = t->levels - 2;
    const uint64_t n = t->nodes[(size_t)d];
    uint32_t shift = 0, cshift = 0;
    while ((4u << shift) < t->opts.band_rows) ++shift;   // a node covers 4 rows
    while ((4ull << cshift) < t->opts.band_cols) ++cshift;
    t->band_shift = shift;
    const uint64_t nrb = ((t->n_rows + 3) / 4 >> shift) + 1;
    const uint64_t ncb = ((t->n_cols + 3) / 4 >> cshift) + 1;
    const uint64_t ntiles = nrb * ncb;
    auto tile_of = [&](const Coord &p) -> uint64_t { return (uint64_t)(p.c >> cshift) * nrb + (p.r >> shift); };
    // first leaf of every node (level order): directory sample + popcount
    std::vector<uint32_t> off(n);
    parallel_for(nt, [&](int th) {
        uint64_t lo = n * th / nt, hi = n * (th + 1) / nt;
        if (lo >= hi) return;
        uint64_t o = level_offset(t, d, lo);
        for (uint64_t i = lo; i < hi; ++i) {
            off[i] = (uint32_t)o;
            o += (uint64_t)__builtin_popcount(level_sig(t, d, i));
        }
    });
    // stable counting sort by tile
    std::vector<uint64_t> cnt((size_t)nt * ntiles, 0);
    parallel_for(nt, [&](int th) {
        uint64_t lo = n * th / nt, hi = n * (th + 1) / nt;
        uint64_t *c = &cnt[(size_t)th * ntiles];
        for (uint64_t i = lo; i < hi; ++i) c[tile_of(t->cached[i])]++;
    });
    std::vector<uint64_t> tile_start(ntiles + 1, 0);
    uint64_t run = 0;
    for (uint64_t b = 0; b < ntiles; ++b) {
        tile_start[b] = run;
        for (int th = 0; th < nt; ++th) {
            uint64_t c = cnt[(size_t)th * ntiles + b];
            cnt[(size_t)th * ntiles + b] = run;
            run += c;
        }
    }
    tile_start[ntiles] = run;
    std::vector<Coord> bc(n);
    t->bleaf.assign(n, 0);
    std::vector<uint8_t> sg(n);
    parallel_for(nt, [&](int th) {
        uint64_t lo = n * th / nt, hi = n * (th + 1) / nt;
        uint64_t *c = &cnt[(size_t)th * ntiles];
        for (uint64_t i = lo; i < hi; ++i) {
            uint64_t dst = c[tile_of(t->cached[i])]++;
            bc[dst] = t->cached[i];
            t->bleaf[dst] = off[i];
            sg[dst] = (uint8_t)level_sig(t, d, i);
        }
    });
    t->cached.swap(bc);
    t->bsig.assign((n + 15) / 16 + 1, 0);
    for (uint64_t i = 0; i < n; ++i) t->bsig[i / 16] |= (uint64_t)sg[i] << (4 * (i % 16));
    t->bchunks.clear();
    for (uint64_t b = 0; b < ntiles; ++b)
        for (uint64_t s0 = tile_start[b]; s0 < tile_start[b + 1]; s0 += kBandChunkNodes) {
            uint64_t e = std::min<uint64_t>(tile_start[b + 1], s0 + kBandChunkNodes);
            t->bchunks.push_back((uint32_t)(b % nrb));  // row band
            t->bchunks.push_back((uint32_t)s0);
            t->bchunks.push_back((uint32_t)(e - s0));
        }
}

// Heavy plus-times outputs of one direction: those with more than `limit`
// non-zeros (counted over the input list: a repeated pair counts each time,
// so a count never falls short).  Fills the ascending list and the record of
// every output up to the last heavy one (0 for the others), which says where
// its terms are summed, in rows of max_batch fp32 words:
//   - mode 1: in an fp64 slot of two rows (record bits kHeavyFp64);
//   - mode 0: in 2^bits rows of fp32 partial sums, a term going to partial
//     heavy_partial(its leaf's first input, bits).  The builder counts
//     the terms every partial receives and raises bits until none holds more
//     than `limit`, so every fp32 sum the product forms, in whatever order
//     its atomics land, has at most `limit` terms.  An output whose inputs
//     still crowd one partial at kHeavyMaxBits (only possible for adversarial
//     or repeated input) is summed in its fp64 slot alone.
// out_ids/in_ids: the output and input index of every input pair.
void heavy_outputs(const uint32_t *out_ids, const uint32_t *in_ids, uint64_t nnz, uint64_t n, uint32_t limit,
                   uint32_t mode, int nt, k2t_tree *t, int dir)
{
    std::vector<uint32_t> &list = t->hlist[dir], &hdir = t->hdir[dir];
    list.clear();
    hdir.clear();
    t->hrows[dir] = t->hparts[dir] = t->hfp64[dir] = 0;
    t->hmax_part[dir] = 0;
    if (limit == 0xffffffffu || nnz <= limit) return;
    // saturating counts: a thread adds only below kSat, so nt racing adds stay below 2^32
    constexpr uint32_t kSat = 0xfffff000u;
    auto bump = [](uint32_t *p) {
        if (__atomic_load_n(p, __ATOMIC_RELAXED) < kSat) __atomic_fetch_add(p, 1u, __ATOMIC_RELAXED);
    };
    std::vector<uint32_t> cnt(n, 0);
    parallel_for(nt, [&](int th) {
        uint64_t lo = nnz * th / nt, hi = nnz * (th + 1) / nt;
        for (uint64_t i = lo; i < hi; ++i) bump(cnt.data() + out_ids[i]);
    });
    for (uint64_t i = 0; i < n; ++i)
        if (cnt[i] > limit) list.push_back((uint32_t)i);
    if (list.empty()) return;
    const size_t h = list.size();
    // records cover every output up to the last heavy one, plus room for the
    // 16-byte read of a 4x4 leaf's four outputs
    hdir.assign(((uint64_t)list.back() + 1 + 3) / 4 * 4 + 4, 0);
    std::vector<uint32_t> bits(h, kHeavyFp64);
    if (mode == 0) {
        // ids during the count: hdir[o] = id + 1
        for (size_t id = 0; id < h; ++id) hdir[list[id]] = (uint32_t)id + 1;
        // first guess: a mean of at most limit / 1.5 terms per partial
        for (size_t id = 0; id < h; ++id) {
            const double want = 1.5 * (double)cnt[list[id]] / (double)limit;
            uint32_t b = 1;
            while (b < kHeavyMaxBits && (double)(1u << b) < want) ++b;
            bits[id] = b;
        }
        std::vector<uint8_t> todo(h, 1);
        bool any = true;
        while (any) {
            // count the terms of every partial of the outputs still to check
            std::vector<uint64_t> base(h, 0);
            uint64_t total = 0;
            for (size_t id = 0; id < h; ++id)
                if (todo[id]) { base[id] = total; total += 1ull << bits[id]; }
            std::vector<uint32_t> pc(total, 0);
            parallel_for(nt, [&](int th) {
                uint64_t lo = nnz * th / nt, hi = nnz * (th + 1) / nt;
                for (uint64_t i = lo; i < hi; ++i) {
                    const uint32_t o = out_ids[i];
                    if (o >= hdir.size() || !hdir[o]) continue;
                    const size_t id = hdir[o] - 1;
                    if (!todo[id]) continue;
                    bump(pc.data() + base[id] + heavy_partial(in_ids[i], bits[id]));
                }
            });
            any = false;
            for (size_t id = 0; id < h; ++id) {
                if (!todo[id]) continue;
                uint32_t mx = 0;
                for (uint64_t q = 0; q < (1ull << bits[id]); ++q) mx = std::max(mx, pc[base[id] + q]);
                if (mx <= limit) {
                    todo[id] = 0;
                    t->hmax_part[dir] = std::max(t->hmax_part[dir], mx);
                } else if (bits[id] < kHeavyMaxBits) {
                    ++bits[id];
                    any = true;
                } else {
                    todo[id] = 0;
                    bits[id] = kHeavyFp64;
                }
            }
        }
    }
    // rows: the fp32 partial sums (2^bits, bits >= 1), or two rows (B doubles)
    // of fp64 slot; the first row of every output is even, so every slot is
    // 8-byte aligned
    uint64_t rows = 0;
    for (size_t id = 0; id < h; ++id) {
        const uint64_t parts = bits[id] == kHeavyFp64 ? 0 : (1ull << bits[id]);
        const uint64_t take = parts ? parts : 2;
        if (rows + take > kHeavyMaxRows) throw std::length_error("heavy partial sums");
        hdir[list[id]] = (uint32_t)(rows << 5) | bits[id];
        rows += take;
        t->hparts[dir] += parts;
        t->hfp64[dir] += parts ? 0 : 1;
    }
    t->hrows[dir] = rows;
}

}  // namespace

void compute_layout(k2t_tree *t)
{
    ArenaLayout &L = t->layout;
    L = ArenaLayout{};
    uint64_t off = 0;
    auto take = [&](uint64_t bytes) {
        uint64_t at = off;
        off = align_up(off + bytes, kArenaAlign);
        return at;
    };
    const int l = t->levels;
    const bool fused = t->engine == K2T_ENGINE_FUSED;
    const bool ls = t->engine == K2T_ENGINE_LEVELSYNC;
    const bool banded = t->engine == K2T_ENGINE_BANDED;
    const bool cached = t->engine == K2T_ENGINE_CACHED || banded;
    // the status word comes first: it is the arena's first 4 bytes (k2t.h)
    L.err_bytes = 64;
    L.err_off = take(L.err_bytes);
    if (!t->empty) {
        int first = cached ? l - 2 : t->d0;
        for (int d = first; d < l; ++d) {
            if (banded && d == l - 2) continue;  // signatures are kept in band order
            // nibble bytes (4x4 leaves: 2 bytes a node) plus 16 bytes of slack for vector loads
            L.sig_bytes[d] = (t->leaf_k4 && d == l - 1 ? 2 * t->nodes[(size_t)d] : (t->nodes[(size_t)d] + 1) / 2) + 16;
            L.sig_off[d] = take(L.sig_bytes[d]);
        }
        bool want_dir = (ls && t->opts.offsets == K2T_OFFSETS_DIRECTORY);
        for (int d = t->d0; d <= l - 2; ++d) {
            bool need = want_dir || (cached && !banded && d == l - 2);
            if (!need) continue;
            L.dir_bytes[d] = t->dir[(size_t)(d - t->d0)].size() * sizeof(uint32_t);
            L.dir_off[d] = take(L.dir_bytes[d]);
        }
        if (ls) {
            L.top_bytes = t->top.size() * sizeof(Coord) + 16;  // slack: bulk copies round up to 16 bytes
            L.top_off = take(L.top_bytes);
        }
        if (cached) {
            L.cached_bytes = t->cached.size() * sizeof(Coord) + 16;
            L.cached_off = take(L.cached_bytes);
        }
        if (banded) {
            L.bleaf_bytes = t->bleaf.size() * sizeof(uint32_t) + 16;
            L.bleaf_off = take(L.bleaf_bytes);
            L.bsig_bytes = (t->nodes[(size_t)l - 2] + 1) / 2 + 16;
            L.bsig_off = take(L.bsig_bytes);
            L.bchunk_bytes = t->bchunks.size() * sizeof(uint32_t);
            L.bchunk_off = take(L.bchunk_bytes);
        }
        if (fused) {
            L.chunk_bytes = t->chunks.size() * sizeof(uint32_t);
            L.chunk_off = take(L.chunk_bytes);
            L.root_bytes = t->roots.size() * sizeof(Coord) + 16;
            L.root_off = take(L.root_bytes);
        }
        if (ls) {
            // exact scratch: every level's buffer holds its largest tile
            uint64_t maxbuf = 0;
            for (const LsStep &s : t->steps)
                if (s.kind == 0) {
                    uint64_t need = level_offset(t, s.level, (uint64_t)s.a + s.count) - s.dst_base;
                    maxbuf = std::max(maxbuf, need);
                }
            L.buf_bytes = maxbuf * sizeof(Coord) + 16;
            for (int d = t->d0 + 1; d <= l - 2; ++d) L.buf_off[d] = take(L.buf_bytes);
            if (t->opts.offsets == K2T_OFFSETS_SCAN) {
                uint64_t blocks = (t->max_tile_nodes + kDirS - 1) / kDirS + 1;
                L.scan_bytes = 2 * blocks * sizeof(uint32_t);
                L.scan_off = take(L.scan_bytes);
            }
        }
    }
    if (!t->empty) {
        uint64_t rows = 0;
        for (int dd = 0; dd < 2; ++dd) {
            if (t->hlist[dd].empty()) continue;
            L.hdir_bytes[dd] = t->hdir[dd].size() * sizeof(uint32_t);
            L.hdir_off[dd] = take(L.hdir_bytes[dd]);
            L.hlist_bytes[dd] = t->hlist[dd].size() * sizeof(uint32_t);
            L.hlist_off[dd] = take(L.hlist_bytes[dd]);
            rows = std::max(rows, t->hrows[dd]);
        }
        if (rows) {
            L.acc_bytes = rows * (uint64_t)t->opts.max_batch * sizeof(float);
            L.acc_off = take(L.acc_bytes);
        }
    }
    if (t->opts.host_vectors) {
        uint64_t n = std::max(t->n_rows, t->n_cols);
        L.vec_bytes = n * (uint64_t)t->opts.max_batch * 4u;
        L.vec_off[0] = take(L.vec_bytes);
        L.vec_off[1] = take(L.vec_bytes);
    }
    L.total = off;
}

// Everything of a build once the sorted distinct path keys of the cells are
// known (keys[0..m), for dim_bits `bits` and the leaf side leaf_k4): heavy
// outputs (counted over the input list rows/cols of nnz pairs), the levels
// bottom-up with the cached and top coordinates, directories, plans and the
// arena layout.  keys and tmp are consumed.  Errors: K2T_ERANGE.
int finish_build(k2t_tree *t, const k2t_opts &o, int nt, std::vector<uint64_t> &keys, std::vector<uint64_t> &tmp,
                 size_t m, int bits, int leaf_k4, const uint32_t *rows, const uint32_t *cols, uint64_t nnz)
{
    const uint64_t n_rows = t->n_rows, n_cols = t->n_cols;
    t->opts.leaf_k = leaf_k4 ? 4u : 2u;
    t->dim_bits = bits;
    t->leaf_k4 = leaf_k4;
    t->levels = bits - t->n_k4 - leaf_k4;
    const int l = t->levels;
    heavy_outputs(rows, cols, nnz, n_rows, o.heavy_terms, o.heavy_mode, nt, t, 0);
    heavy_outputs(cols, rows, nnz, n_cols, o.heavy_terms, o.heavy_mode, nt, t, 1);
    for (int dd = 0; dd < 2; ++dd)
        if (t->hlist[dd].size() >= (1u << 28)) return K2T_ERANGE;

    t->nodes.assign((size_t)l, 0);
    t->sig.assign((size_t)l, std::vector<uint64_t>());
    t->nnz = m;

    if (m == 0) {
        t->empty = true;
        for (int dd = 0; dd < 2; ++dd) {
            t->hlist[dd].clear();
            t->hdir[dd].clear();
            t->hrows[dd] = t->hparts[dd] = t->hfp64[dd] = 0;
        }
        t->nodes[0] = 1;
        t->sig[0].assign(2, 0);
        for (int d = 1; d < l; ++d) t->sig[(size_t)d].assign(1, 0);
        t->d0 = 0;
    } else {
        std::vector<uint16_t> sg(m);
        bool have_top = false;
        uint64_t top_max = o.host_top_max_nodes;
        // cells -> leaves -> ... -> root
        uint64_t *cur = keys.data(), *nxt = tmp.data();
        size_t ncur = m;
        for (int d = l - 1; d >= 0; --d) {
            int s = level_is_k4(t, d) ? 4 : 2;
            size_t nn = group_level(cur, ncur, s, nxt, sg.data(), nt);
            if (nn >= (1ull << 32)) return K2T_ERANGE;
            t->nodes[(size_t)d] = nn;
            pack_level(t, d, sg.data(), nn, nt);
            if (d == l - 2 && (t->engine == K2T_ENGINE_CACHED || t->engine == K2T_ENGINE_BANDED)) {
                t->cached.resize(nn);
                parallel_for(nt, [&](int th) {
                    size_t lo = nn * th / nt, hi = nn * (th + 1) / nt;
                    for (size_t i = lo; i < hi; ++i) t->cached[i] = prefix_coord(nxt[i], d, t->n_k4);
                });
            }
            if (!have_top && d <= l - 2 && d >= t->n_k4 && (nn <= top_max || d == t->n_k4)) {
                have_top = true;
                t->d0 = d;
                t->top.resize(nn);
                for (size_t i = 0; i < nn; ++i) t->top[i] = prefix_coord(nxt[i], d, t->n_k4);
            }
            std::swap(cur, nxt);
            ncur = nn;
        }
    }
    std::vector<uint64_t>().swap(keys);
    std::vector<uint64_t>().swap(tmp);

    if (!t->empty) {
        t->dir.assign((size_t)(l - 1 - t->d0), std::vector<uint32_t>());
        for (int d = t->d0; d <= l - 2; ++d) build_directory(t, d, nt);
        if (t->engine == K2T_ENGINE_BANDED) plan_bands(t, nt);
        if (t->engine == K2T_ENGINE_FUSED) {
            // the top level cut into one part per thread, planned in
            // parallel and joined in order (a chunk never spans two parts);
            // roots below the top follow the top's coordinates
            t->chunk_stride = 2 + 2 * (uint32_t)(l - t->d0);
            t->roots = t->top;
            const uint64_t n0 = t->nodes[(size_t)t->d0];
            std::vector<FusedPlanner> parts((size_t)nt, FusedPlanner{t, o.chunk_cap, {}, {}, 0});
            parallel_for(nt, [&](int th) {
                const uint64_t lo = n0 * th / nt, hi = n0 * (th + 1) / nt;
                if (lo < hi) parts[(size_t)th].range(t->d0, lo, hi, t->top.data() + lo, true);
            });
            for (FusedPlanner &pp : parts) {
                const uint32_t shift = (uint32_t)t->roots.size();
                for (size_t c = 0; c < pp.n_chunks; ++c) {
                    uint32_t *rec = &pp.chunks[c * t->chunk_stride];
                    if ((int)rec[1] != t->d0) rec[0] += shift;
                }
                t->chunks.insert(t->chunks.end(), pp.chunks.begin(), pp.chunks.end());
                t->roots.insert(t->roots.end(), pp.roots.begin(), pp.roots.end());
                t->n_chunks += pp.n_chunks;
            }
        } else if (t->engine == K2T_ENGINE_LEVELSYNC) {
            LsPlanner p{t, o.tile_m, std::vector<uint64_t>((size_t)l + 1, 0)};
            p.range(t->d0, 0, t->nodes[(size_t)t->d0], 0xff, 0);
        }
    }
    compute_layout(t);
    return K2T_OK;
}

// Options with defaults filled in and checked for a matrix of n_rows x n_cols.
int normalize_opts(const k2t_opts *opts, uint64_t n_rows, uint64_t n_cols, k2t_opts &o)
{
    if (opts) o = *opts; else k2t_default_opts(&o);
    if (o.engine > K2T_ENGINE_BANDED || o.offsets > K2T_OFFSETS_SCAN) return K2T_EINVAL;
    if (o.band_rows < 16 || o.band_rows > 65536 || (o.band_rows & (o.band_rows - 1))) return K2T_EINVAL;
    if (o.band_cols && (o.band_cols < 16 || (o.band_cols & (o.band_cols - 1)))) return K2T_EINVAL;
    if (!o.band_cols) o.band_cols = 1u << 31;
    if (!o.heavy_terms) o.heavy_terms = kDefaultHeavyTerms;
    if (o.heavy_mode > 1) return K2T_EINVAL;
    if (o.leaf_k != 0 && o.leaf_k != 2 && o.leaf_k != 4) return K2T_EINVAL;
    if (o.chunk_cap < 4 || o.chunk_cap > kMaxChunkCap || o.tile_m < 4) return K2T_EINVAL;
    if (o.max_batch < 1 || o.max_batch > K2T_MAX_BATCH) return K2T_ERANGE;
    if (o.host_top_max_nodes < 1) return K2T_EINVAL;
    if (o.n_k4_levels > 15) return K2T_EINVAL;
    if (n_rows > (1ull << 32) || n_cols > (1ull << 32)) return K2T_ERANGE;
    if ((o.engine == K2T_ENGINE_CACHED || o.engine == K2T_ENGINE_BANDED) && !o.cache_last_internal) return K2T_EINVAL;
    // 4x4 leaves: the CACHED and FUSED engines
    const bool leaf4_ok = o.engine == K2T_ENGINE_AUTO || o.engine == K2T_ENGINE_CACHED || o.engine == K2T_ENGINE_FUSED;
    if (o.leaf_k == 4 && !leaf4_ok) return K2T_EINVAL;

    return K2T_OK;
}

// Bits 0, 2, 4, ... of x, packed (the inverse of spread_bits).
inline uint32_t compact_bits(uint64_t x)
{
    x &= 0x5555555555555555ull;
    x = (x | (x >> 1)) & 0x3333333333333333ull;
    x = (x | (x >> 2)) & 0x0F0F0F0F0F0F0F0Full;
    x = (x | (x >> 4)) & 0x00FF00FF00FF00FFull;
    x = (x | (x >> 8)) & 0x0000FFFF0000FFFFull;
    x = (x | (x >> 16)) & 0x00000000FFFFFFFFull;
    return (uint32_t)x;
}

int build_from_sorted_keys(const uint64_t *keys, uint64_t m, uint64_t n_rows, uint64_t n_cols, const k2t_opts *opts,
                           k2t_tree **out)
{
    if (!out) return K2T_EINVAL;
    *out = nullptr;
    if (n_rows == 0 || n_cols == 0 || (m && !keys)) return K2T_EINVAL;
    k2t_opts o;
    int rc = normalize_opts(opts, n_rows, n_cols, o);
    if (rc) return rc;
    if (o.n_k4_levels) return K2T_EINVAL;
    const bool leaf4_ok = o.engine == K2T_ENGINE_AUTO || o.engine == K2T_ENGINE_CACHED || o.engine == K2T_ENGINE_FUSED;
    uint64_t n = std::max(n_rows, n_cols);
    int bits0 = 0;
    while ((1ull << bits0) < n) ++bits0;
    bits0 = std::max(bits0, 2);
    const int nt = thread_count(o);
    try {
        // keys strictly increasing, inside the padded side
        std::vector<int> bad((size_t)nt, 0);
        const uint64_t lim = bits0 >= 32 ? ~0ull : (1ull << (2 * bits0));
        parallel_for(nt, [&](int th) {
            uint64_t lo = m * th / nt, hi = m * (th + 1) / nt;
            for (uint64_t i = lo; i < hi; ++i)
                if (keys[i] >= lim || (i && keys[i] <= keys[i - 1])) { bad[(size_t)th] = 1; break; }
        });
        for (int b : bad) if (b) return K2T_EINVAL;
        // the leaf side: 4x4 when chosen, or when 2x2 leaves would be dense
        bool four = o.leaf_k == 4;
        if (o.leaf_k == 0 && leaf4_ok && m > 0) {
            std::vector<uint64_t> part((size_t)nt, 0);
            parallel_for(nt, [&](int th) {
                uint64_t lo = m * th / nt, hi = m * (th + 1) / nt, c = 0;
                for (uint64_t i = lo; i < hi; ++i) c += (i == 0 || (keys[i] >> 2) != (keys[i - 1] >> 2)) ? 1 : 0;
                part[(size_t)th] = c;
            });
            uint64_t leaves = 0;
            for (uint64_t c : part) leaves += c;
            four = (double)m >= kAutoLeaf4Density * (double)leaves;
        }
        // the cells as pairs: the input list of the heavy outputs (and of a
        // 4x4-leaf build, which needs keys of another digit order)
        std::vector<uint32_t> rows, cols;
        if (four || o.heavy_terms != 0xffffffffu) {
            rows.resize(m);
            cols.resize(m);
            parallel_for(nt, [&](int th) {
                uint64_t lo = m * th / nt, hi = m * (th + 1) / nt;
                for (uint64_t i = lo; i < hi; ++i) {
                    rows[i] = compact_bits(keys[i] >> 1);
                    cols[i] = compact_bits(keys[i]);
                    if (rows[i] >= n_rows || cols[i] >= n_cols) { bad[(size_t)th] = 1; break; }
                }
            });
            for (int b : bad) if (b) return K2T_ERANGE;
        }
        if (four) return k2t_build(rows.data(), cols.data(), m, n_rows, n_cols, &o, out);
        k2t_tree *t = new (std::nothrow) k2t_tree;
        if (!t) return K2T_ENOMEM;
        try {
            t->opts = o;
            t->n_rows = n_rows;
            t->n_cols = n_cols;
            t->n_k4 = 0;
            t->engine = o.engine == K2T_ENGINE_AUTO ? (o.cache_last_internal ? K2T_ENGINE_CACHED : K2T_ENGINE_FUSED)
                                                    : o.engine;
            std::vector<uint64_t> kv(keys, keys + m), tmp(m);
            rc = finish_build(t, o, nt, kv, tmp, m, bits0, 0, rows.data(), cols.data(), rows.size());
        } catch (...) {
            delete t;
            throw;
        }
        if (rc) { delete t; return rc; }
        *out = t;
        return K2T_OK;
    } catch (const std::bad_alloc &) {
        return K2T_ENOMEM;
    } catch (const std::length_error &) {
        return K2T_ERANGE;
    }
}

}  // namespace k2t

using namespace k2t;

extern "C" {

void k2t_default_opts(k2t_opts *o)
{
    if (!o) return;
    std::memset(o, 0, sizeof(*o));
    o->n_k4_levels = 0;
    o->cache_last_internal = 0;
    o->engine = K2T_ENGINE_AUTO;
    o->offsets = K2T_OFFSETS_DIRECTORY;
    o->host_top_max_nodes = 1u << 16;
    o->chunk_cap = 256;
    o->tile_m = 1ull << 20;
    o->max_batch = 32;
    o->host_vectors = 0;
    o->use_graph = 1;
    o->threads = 0;
    o->band_rows = 4096;
    o->band_cols = 1u << 23;
    o->heavy_terms = kDefaultHeavyTerms;
    o->leaf_k = 0;
}

int k2t_build(const uint32_t *rows, const uint32_t *cols, uint64_t nnz,
              uint64_t n_rows, uint64_t n_cols, const k2t_opts *opts, k2t_tree **out)
{
    if (!out) return K2T_EINVAL;
    *out = nullptr;
    if (n_rows == 0 || n_cols == 0) return K2T_EINVAL;
    if (nnz && (!rows || !cols)) return K2T_EINVAL;
    k2t_opts o;
    int rc = normalize_opts(opts, n_rows, n_cols, o);
    if (rc) return rc;
    const bool leaf4_ok = o.engine == K2T_ENGINE_AUTO || o.engine == K2T_ENGINE_CACHED || o.engine == K2T_ENGINE_FUSED;
    k2t_tree *t = new (std::nothrow) k2t_tree;
    if (!t) return K2T_ENOMEM;
    try {
        t->opts = o;
        t->n_rows = n_rows;
        t->n_cols = n_cols;
        uint64_t n = std::max(n_rows, n_cols);
        int bits0 = 0;
        while ((1ull << bits0) < n) ++bits0;
        bits0 = std::max(bits0, 2);
        if (std::max(bits0, 2 * (int)o.n_k4_levels + 2 + (o.leaf_k == 4 ? 1 : 0)) > 32) { delete t; return K2T_ERANGE; }
        t->n_k4 = (int)o.n_k4_levels;
        const int nt = thread_count(o);
        t->engine = o.engine == K2T_ENGINE_AUTO
                        ? (o.cache_last_internal ? K2T_ENGINE_CACHED : K2T_ENGINE_FUSED)
                        : o.engine;

        // validate ids
        std::vector<int> bad((size_t)nt, 0);
        parallel_for(nt, [&](int th) {
            uint64_t lo = nnz * th / nt, hi = nnz * (th + 1) / nt;
            for (uint64_t i = lo; i < hi; ++i)
                if (rows[i] >= n_rows || cols[i] >= n_cols) { bad[(size_t)th] = 1; break; }
        });
        for (int b : bad) if (b) { delete t; return K2T_ERANGE; }

        // Sorted distinct path keys of the cells for a leaf side.  With
        // leaf_k 0 the side is chosen here: 4x4 leaves when the 2x2 leaves
        // would hold at least kAutoLeaf4Density non-zeros each on average
        // (the measured break-even of the two leaf sizes), 2x2 otherwise.
        std::vector<uint64_t> keys(nnz), tmp;
        int leaf_k4 = o.leaf_k == 4 ? 1 : 0, bits = 0;
        size_t m = 0;
        auto make_keys = [&](int l4) {
            bits = std::max(bits0, 2 * (int)o.n_k4_levels + 2 + l4);
            keys.resize(nnz);
            parallel_for(nt, [&](int th) {
                uint64_t lo = nnz * th / nt, hi = nnz * (th + 1) / nt;
                for (uint64_t i = lo; i < hi; ++i) keys[i] = path_key(rows[i], cols[i], bits, t->n_k4, l4);
            });
            radix_sort(keys, tmp, 2 * bits, nt);
            tmp.resize(keys.size());
            m = unique_into(keys.data(), keys.size(), tmp.data(), nt);
            keys.swap(tmp);
            keys.resize(m);
            tmp.resize(m);
        };
        make_keys(leaf_k4);
        if (o.leaf_k == 0 && leaf4_ok && m > 0 && 2 * (int)o.n_k4_levels + 3 <= 32) {
            // distinct 2x2 leaves: keys that differ above the leaf-cell digit
            std::vector<uint64_t> part((size_t)nt, 0);
            parallel_for(nt, [&](int th) {
                size_t lo = m * th / nt, hi = m * (th + 1) / nt;
                uint64_t c = 0;
                for (size_t i = lo; i < hi; ++i) c += (i == 0 || (keys[i] >> 2) != (keys[i - 1] >> 2)) ? 1 : 0;
                part[(size_t)th] = c;
            });
            uint64_t leaves = 0;
            for (uint64_t c : part) leaves += c;
            if ((double)m >= kAutoLeaf4Density * (double)leaves) {
                leaf_k4 = 1;
                make_keys(1);
            }
        }
        rc = finish_build(t, o, nt, keys, tmp, m, bits, leaf_k4, rows, cols, nnz);
        if (rc) { delete t; return rc; }
    } catch (const std::bad_alloc &) {
        delete t;
        return K2T_ENOMEM;
    } catch (const std::length_error &) {
        delete t;
        return K2T_ERANGE;
    }
    *out = t;
    return K2T_OK;
}

int k2t_workspace_bytes(const k2t_tree *t, uint64_t *bytes)
{
    if (!t || !bytes) return K2T_EINVAL;
    *bytes = t->layout.total;
    return K2T_OK;
}

int k2t_level_signatures(const k2t_tree *t, uint32_t level, uint8_t *out, uint64_t cap, uint64_t *written)
{
    if (!t || !written || level >= (uint32_t)t->levels) return K2T_EINVAL;
    uint64_t n = t->nodes[level];
    bool k4 = level_is_k4(t, (int)level);
    uint64_t need = k4 ? 2 * n : n;
    *written = need;
    if (!out || cap < need) return K2T_ERANGE;
    for (uint64_t i = 0; i < n; ++i) {
        uint32_t s = level_sig(t, (int)level, i);
        if (k4) { out[2 * i] = (uint8_t)(s & 0xff); out[2 * i + 1] = (uint8_t)(s >> 8); }
        else out[i] = (uint8_t)s;
    }
    return K2T_OK;
}

int k2t_decode(const k2t_tree *t, uint32_t *rows, uint32_t *cols, uint64_t cap, uint64_t *n_out)
{
    if (!t || !n_out) return K2T_EINVAL;
    *n_out = t->nnz;
    if (cap < t->nnz || (t->nnz && (!rows || !cols))) return K2T_ERANGE;
    if (t->empty) return K2T_OK;
    std::vector<Coord> cur(1, Coord{0, 0}), nxt;
    for (int d = 0; d < t->levels - 1; ++d) {
        int k = d < t->n_k4 ? 4 : 2;
        nxt.clear();
        nxt.reserve(t->nodes[(size_t)d + 1]);
        for (uint64_t i = 0; i < cur.size(); ++i) {
            uint32_t s = level_sig(t, d, i);
            for (int b = 0; b < k * k; ++b)
                if (s & (1u << b))
                    nxt.push_back(Coord{cur[i].r * (uint32_t)k + (uint32_t)(b / k), cur[i].c * (uint32_t)k + (uint32_t)(b % k)});
        }
        cur.swap(nxt);
    }
    uint64_t w = 0;
    const int d = t->levels - 1;
    const uint32_t k = t->leaf_k4 ? 4u : 2u;
    for (uint64_t i = 0; i < cur.size(); ++i) {
        uint32_t s = level_sig(t, d, i);
        for (uint32_t b = 0; b < k * k; ++b)
            if (s & (1u << b)) {
                rows[w] = k * cur[i].r + b / k;
                cols[w] = k * cur[i].c + b % k;
                ++w;
            }
    }
    return K2T_OK;
}

int k2t_stats_get(const k2t_tree *t, k2t_stats *s)
{
    if (!t || !s) return K2T_EINVAL;
    std::memset(s, 0, sizeof(*s));
    s->n_rows = t->n_rows;
    s->n_cols = t->n_cols;
    s->nnz = t->nnz;
    s->levels = (uint32_t)t->levels;
    s->n_k4_levels = (uint32_t)t->n_k4;
    s->dim_bits = (uint32_t)t->dim_bits;
    s->d0 = (uint32_t)t->d0;
    uint64_t bits = 0;
    for (int d = 0; d < t->levels; ++d) {
        s->level_nodes[d] = t->nodes[(size_t)d];
        int k = level_is_k4(t, d) ? 4 : 2;
        bits += t->nodes[(size_t)d] * (uint64_t)(k * k);
    }
    s->tree_bits = bits;
    const ArenaLayout &L = t->layout;
    for (int d = 0; d < t->levels - 1; ++d) s->t_bytes_device += L.sig_bytes[d];
    s->l_bytes_device = L.sig_bytes[t->levels - 1];
    for (int d = 0; d < t->levels; ++d) s->dir_bytes += L.dir_bytes[d];
    s->top_bytes = L.top_bytes;
    s->cached_bytes = L.cached_bytes + L.bleaf_bytes + L.bsig_bytes;
    s->plan_bytes = 0;
    s->plan_bytes = L.chunk_bytes + L.root_bytes + L.bchunk_bytes;
    uint64_t nbuf = 0;
    for (int d = 0; d < t->levels; ++d) nbuf += L.buf_off[d] ? 1 : 0;
    s->scratch_bytes = nbuf * L.buf_bytes + L.scan_bytes;
    s->vector_bytes = 2 * L.vec_bytes;
    s->workspace_bytes = L.total;
    s->n_chunks = t->n_chunks;
    s->n_steps = t->steps.size();
    s->engine = t->engine;
    s->offsets = t->opts.offsets;
    s->uploaded = t->dev != nullptr;
    s->heavy_rows = (uint32_t)t->hlist[0].size();
    s->heavy_cols = (uint32_t)t->hlist[1].size();
    uint64_t hb = L.acc_bytes;
    for (int dd = 0; dd < 2; ++dd) hb += L.hdir_bytes[dd] + L.hlist_bytes[dd];
    s->heavy_kib = (uint32_t)((hb + 1023) / 1024);
    s->leaf_k = t->leaf_k4 ? 4u : 2u;
    for (int dd = 0; dd < 2; ++dd) {
        s->heavy_partials[dd] = t->hparts[dd];
        s->heavy_fp64[dd] = (uint32_t)t->hfp64[dd];
        s->heavy_max_terms[dd] = t->hmax_part[dd];
    }
    return K2T_OK;
}

void k2t_free(k2t_tree *t)
{
    if (!t) return;
    device_release(t);
    delete t;
}

const char *k2t_strerror(int status)
{
    switch (status) {
    case K2T_OK: return "ok";
    case K2T_EINVAL: return "invalid argument";
    case K2T_ERANGE: return "value out of range";
    case K2T_ENOMEM: return "out of memory";
    case K2T_ECUDA: return "CUDA runtime error";
    case K2T_ESTATE: return "call out of order";
    case K2T_EDEVICE: return "device-side check failed";
    case K2T_ETIMEOUT: return "device-side wait ran out";
    default: return "unknown status";
    }
}

}  // extern "C"
