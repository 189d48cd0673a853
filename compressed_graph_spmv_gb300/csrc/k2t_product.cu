// k2t_product.cu -- Boolean product of two trees, C = A B, and the transitive
// closure by repeated squaring.
//
// "A GPU Engine for Sparse Matrix-Vector Products on k^2-Tree-Compressed
// Graphs" closes (section 7) on extending its level-synchronous traversal to
// products of two trees: a frontier of node pairs expands into matching
// quadrant sub-products, which gives Boolean A B, and repeated squaring the
// transitive closure, kept compressed.  This file builds that on the device:
//
//  * A frontier entry is a pair (a, b, i, j): node a of A and node b of B at
//    the same level d, a covering block (i, k) of A and b block (k, j) of B
//    (same k); together they contribute to block (i, j) of C.  The root pair
//    starts it.
//  * Expansion: quadrant (ar, ac) of a meets quadrant (br, bc) of b when
//    ac == br, giving the child pair (a's child, b's child, 2i + ar, 2j + bc).
//    A pair has at most 8 children.  Children are placed by an exclusive
//    prefix sum of the per-pair counts; child positions in each tree come
//    from its directory (section 3.2).
//  * At the last internal level the children are leaves: each matching pair
//    of 2x2 leaf bitmaps gives the 2x2 Boolean product of the two blocks,
//    one record (leaf row, leaf column, 4-bit bitmap) of C.
//  * The frontier is processed depth first in tiles: a tile of at most M/8
//    pairs has at most M children, so every level needs one buffer of M
//    pairs.
//  * C's cells stay on the device.  Whenever the record buffer fills, and at
//    the end, the records are merged into a sorted set of C's distinct leaves:
//    leaf path keys sorted with their products, repeats (several k reach one
//    block) OR-ed together (CUB radix sort and reduce-by-key).  The set then
//    expands into the sorted path keys of C's cells, which is the order the
//    builder packs levels in; only those keys go to the host, which packs the
//    levels without sorting.  The transitive closure keeps C's keys on the
//    device from one squaring to the next and forms C or C C there (merge of
//    two sorted key sets).
//
// Requirements: A is n x m and B is m x p with the same padded side and
// k = 2 on every level (no hybrid top, 2x2 leaves).  The trees need not be
// uploaded: the product copies what it reads (every level's signatures and
// directory) to its own device memory and frees it on return.
#include <algorithm>
#include <vector>

#include <cub/device/device_radix_sort.cuh>
#include <cub/device/device_reduce.cuh>
#include <cub/device/device_scan.cuh>
#include <cub/device/device_select.cuh>

#include "k2t_kernels.cuh"

namespace k2t {

struct Pair {
    uint32_t a, b;  // node of A, node of B (level-relative indices)
    uint32_t i, j;  // block row and column of C at this level
};

struct ProdLevel {
    const uint8_t *sig;   // nibble t at byte t/2, low nibble first
    const uint32_t *dir;  // first child per 256 nodes, then the level's total
    uint32_t n;           // nodes
};

constexpr int kProdThreads = 256;

// Child pairs of a pair: sum over the set quadrants (ar, ac) of a of the set
// quadrants of b in row ac.
__device__ __forceinline__ uint32_t pair_fanout(uint32_t sa, uint32_t sb)
{
    uint32_t c = 0;
#pragma unroll
    for (uint32_t qa = 0; qa < 4; ++qa)
        if ((sa >> qa) & 1u) c += (uint32_t)__popc(sb & (3u << (2u * (qa & 1u))));
    return c;
}

// 2x2 Boolean product: C_ij = OR_k A_ik AND B_kj with cell (r, c) of a leaf
// at bit 2r + c.
__device__ __forceinline__ uint32_t leaf_product(uint32_t la, uint32_t lb)
{
    uint32_t c = 0;
#pragma unroll
    for (uint32_t i = 0; i < 2; ++i)
#pragma unroll
        for (uint32_t j = 0; j < 2; ++j) {
            const uint32_t v = (((la >> (2u * i)) & (lb >> j)) | ((la >> (2u * i + 1u)) & (lb >> (2u + j)))) & 1u;
            c |= v << (2u * i + j);
        }
    return c;
}

// cnt[t] = child pairs of pair t (t < n).
__global__ void __launch_bounds__(kProdThreads) pair_count_kernel(ProdLevel la, ProdLevel lb, const Pair *p,
                                                                  uint32_t n, uint32_t *cnt)
{
    const uint32_t t = blockIdx.x * kProdThreads + threadIdx.x;
    if (t >= n) return;
    const Pair q = p[t];
    cnt[t] = pair_fanout(nibble_at(la.sig, q.a), nibble_at(lb.sig, q.b));
}

// Exclusive prefix sums of cnt within blocks of kProdThreads (pos), and the
// block totals (bsum); ls_scan_kernel then scans bsum.
__global__ void __launch_bounds__(kProdThreads) block_scan_kernel(const uint32_t *cnt, uint32_t n, uint32_t *pos,
                                                                  uint32_t *bsum)
{
    __shared__ uint32_t wsum[kProdThreads / 32];
    const uint32_t t = blockIdx.x * kProdThreads + threadIdx.x;
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t v = t < n ? cnt[t] : 0u;
    const uint32_t incl = warp_incl_scan(v);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    uint32_t before = 0, total = 0;
    for (uint32_t w = 0; w < kProdThreads / 32; ++w) {
        if (w < warp) before += wsum[w];
        total += wsum[w];
    }
    if (t < n) pos[t] = before + incl - v;
    if (threadIdx.x == 0) bsum[blockIdx.x] = total;
}

// Children of pair t written at dst[bpre[t / kProdThreads] + pos[t] ...], in
// quadrant order of a, then of b.
__global__ void __launch_bounds__(kProdThreads) pair_expand_kernel(ProdLevel la, ProdLevel lb, const Pair *p,
                                                                   uint32_t n, const uint32_t *pos,
                                                                   const uint32_t *bpre, Pair *dst)
{
    const uint32_t t = blockIdx.x * kProdThreads + threadIdx.x;
    if (t >= n) return;
    const Pair q = p[t];
    const uint32_t sa = nibble_at(la.sig, q.a), sb = nibble_at(lb.sig, q.b);
    if (!pair_fanout(sa, sb)) return;
    const uint32_t oa = dir_offset(la.sig, la.dir, la.n, q.a);
    const uint32_t ob = dir_offset(lb.sig, lb.dir, lb.n, q.b);
    Pair *o = dst + bpre[t / kProdThreads] + pos[t];
#pragma unroll
    for (uint32_t qa = 0; qa < 4; ++qa) {
        if (!((sa >> qa) & 1u)) continue;
        const uint32_t ar = qa >> 1, ac = qa & 1u;
        const uint32_t ca = oa + (uint32_t)__popc(sa & ((1u << qa) - 1u));
#pragma unroll
        for (uint32_t bc = 0; bc < 2; ++bc) {
            const uint32_t qb = 2u * ac + bc;
            if (!((sb >> qb) & 1u)) continue;
            const uint32_t cb = ob + (uint32_t)__popc(sb & ((1u << qb) - 1u));
            *o++ = Pair{ca, cb, 2u * q.i + ar, 2u * q.j + bc};
        }
    }
}

// Leaf step: every matching pair of leaves under pair t (last internal
// level) gives one record (leaf row, leaf column, 2x2 product) when the
// product is not empty.  A warp reserves its records with one atomic; the
// host guarantees room for 8 records per pair.
__global__ void __launch_bounds__(kProdThreads) pair_leaf_kernel(ProdLevel la, ProdLevel lb, const uint8_t *leafa,
                                                                 const uint8_t *leafb, const Pair *p, uint32_t n,
                                                                 uint32_t *rec, unsigned long long *count)
{
    const uint32_t t = blockIdx.x * kProdThreads + threadIdx.x;
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t sa = 0, sb = 0, oa = 0, ob = 0;
    Pair q{0, 0, 0, 0};
    if (t < n) {
        q = p[t];
        sa = nibble_at(la.sig, q.a);
        sb = nibble_at(lb.sig, q.b);
        if (pair_fanout(sa, sb)) {
            oa = dir_offset(la.sig, la.dir, la.n, q.a);
            ob = dir_offset(lb.sig, lb.dir, lb.n, q.b);
        } else {
            sa = 0;
        }
    }
    // pass 1: count this thread's non-empty products; pass 2: write them
    uint32_t mine = 0;
    for (int pass = 0; pass < 2; ++pass) {
        uint64_t at = 0;
        if (pass == 1) {
            const uint32_t incl = warp_incl_scan(mine);
            const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
            unsigned long long base = 0;
            if (lane == 31 && total) base = atomicAdd(count, (unsigned long long)total);
            base = __shfl_sync(0xffffffffu, base, 31);
            at = base + incl - mine;
        }
#pragma unroll
        for (uint32_t qa = 0; qa < 4; ++qa) {
            if (!((sa >> qa) & 1u)) continue;
            const uint32_t ac = qa & 1u;
            const uint32_t lam_a = nibble_at(leafa, oa + (uint32_t)__popc(sa & ((1u << qa) - 1u)));
#pragma unroll
            for (uint32_t bc = 0; bc < 2; ++bc) {
                const uint32_t qb = 2u * ac + bc;
                if (!((sb >> qb) & 1u)) continue;
                const uint32_t lam_b = nibble_at(leafb, ob + (uint32_t)__popc(sb & ((1u << qb) - 1u)));
                const uint32_t c = leaf_product(lam_a, lam_b);
                if (!c) continue;
                if (pass == 0) {
                    ++mine;
                } else {
                    uint32_t *r = rec + 3 * at++;
                    r[0] = 2u * q.i + (qa >> 1);
                    r[1] = 2u * q.j + bc;
                    r[2] = c;
                }
            }
        }
    }
}

// bit i of v -> bit 2i
__host__ __device__ __forceinline__ uint64_t spread2(uint32_t v)
{
    uint64_t x = v;
    x = (x | (x << 16)) & 0x0000FFFF0000FFFFull;
    x = (x | (x << 8)) & 0x00FF00FF00FF00FFull;
    x = (x | (x << 4)) & 0x0F0F0F0F0F0F0F0Full;
    x = (x | (x << 2)) & 0x3333333333333333ull;
    x = (x | (x << 1)) & 0x5555555555555555ull;
    return x;
}

// Path key of leaf block (lr, lc) (lr's bits at odd positions) and the 2x2
// product of each record, written at key[at + i], bits[at + i].
__global__ void __launch_bounds__(kProdThreads) record_keys_kernel(const uint32_t *rec, uint64_t n, uint64_t at,
                                                                   uint64_t *key, uint32_t *bits)
{
    const uint64_t i = (uint64_t)blockIdx.x * kProdThreads + threadIdx.x;
    if (i >= n) return;
    key[at + i] = (spread2(rec[3 * i]) << 1) | spread2(rec[3 * i + 1]);
    bits[at + i] = rec[3 * i + 2];
}

// cnt[i] = cells of distinct leaf i.
__global__ void __launch_bounds__(kProdThreads) leaf_count_kernel(const uint32_t *bits, uint64_t n, uint64_t *cnt)
{
    const uint64_t i = (uint64_t)blockIdx.x * kProdThreads + threadIdx.x;
    if (i < n) cnt[i] = (uint64_t)__popc(bits[i]);
}

// The cells of distinct leaf i as path keys (leaf key, then the cell digit
// 2r + c), in digit order, at cell[pos[i] ...]: sorted leaves give sorted
// cells.
__global__ void __launch_bounds__(kProdThreads) leaf_cells_kernel(const uint64_t *leaf, const uint32_t *bits,
                                                                  const uint64_t *pos, uint64_t n, uint64_t *cell)
{
    const uint64_t i = (uint64_t)blockIdx.x * kProdThreads + threadIdx.x;
    if (i >= n) return;
    const uint32_t b = bits[i];
    uint64_t o = pos[i];
#pragma unroll
    for (uint32_t q = 0; q < 4; ++q)
        if ((b >> q) & 1u) cell[o++] = (leaf[i] << 2) | q;
}

// Path keys of cells (r, c) given as pairs.
__global__ void __launch_bounds__(kProdThreads) cell_keys_kernel(const uint32_t *r, const uint32_t *c, uint64_t n,
                                                                 uint64_t *key)
{
    const uint64_t i = (uint64_t)blockIdx.x * kProdThreads + threadIdx.x;
    if (i < n) key[i] = (spread2(r[i]) << 1) | spread2(c[i]);
}

struct BitOr {
    __device__ __forceinline__ uint32_t operator()(uint32_t a, uint32_t b) const { return a | b; }
};

namespace {

inline unsigned grid_of(uint64_t n) { return (unsigned)((n + kProdThreads - 1) / kProdThreads); }

// One device allocation, freed with its owner.
struct DevMem {
    void *p = nullptr;
    DevMem() = default;
    DevMem(const DevMem &) = delete;
    DevMem &operator=(const DevMem &) = delete;
    ~DevMem() { if (p) cudaFree(p); }
    int alloc(size_t bytes)
    {
        if (p) { cudaFree(p); p = nullptr; }
        cudaError_t e = cudaMalloc(&p, bytes ? bytes : 16);
        if (e != cudaSuccess) { g_last_cuda = (int)e; p = nullptr; return K2T_ENOMEM; }
        return K2T_OK;
    }
    template <class T> T *as() const { return static_cast<T *>(p); }
    void swap(DevMem &o) { std::swap(p, o.p); }
};

// A sorted set of distinct leaves of C on the device: path keys and the OR of
// their 2x2 products.
struct LeafSet {
    DevMem key, bits;
    uint64_t n = 0;
};

// CUB's scratch for one call (queried, then allocated).
template <class F>
int cub_run(F &&f, cudaStream_t st)
{
    size_t bytes = 0;
    K2T_CUDA(f(nullptr, bytes));
    DevMem tmp;
    int rc = tmp.alloc(bytes);
    if (rc) return rc;
    K2T_CUDA(f(tmp.p, bytes));
    (void)st;
    return K2T_OK;
}

// Merge c records (device, 3 words each) into the set: their leaf keys and
// products with the set's entries, sorted by key (bits [0, key_bits)),
// repeats OR-ed together.
int absorb(LeafSet &s, const uint32_t *rec, uint64_t c, int key_bits, cudaStream_t st)
{
    if (!c) return K2T_OK;
    const uint64_t n = s.n + c;
    DevMem k0, b0, k1, b1, runs;
    int rc = k0.alloc(n * 8);
    if (!rc) rc = b0.alloc(n * 4);
    if (!rc) rc = k1.alloc(n * 8);
    if (!rc) rc = b1.alloc(n * 4);
    if (!rc) rc = runs.alloc(8);
    if (rc) return rc;
    if (s.n) {
        K2T_CUDA(cudaMemcpyAsync(k0.p, s.key.p, s.n * 8, cudaMemcpyDeviceToDevice, st));
        K2T_CUDA(cudaMemcpyAsync(b0.p, s.bits.p, s.n * 4, cudaMemcpyDeviceToDevice, st));
    }
    record_keys_kernel<<<grid_of(c), kProdThreads, 0, st>>>(rec, c, s.n, k0.as<uint64_t>(), b0.as<uint32_t>());
    K2T_CUDA(cudaGetLastError());
    const int64_t ni = (int64_t)n;
    rc = cub_run([&](void *t, size_t &b) {
        return cub::DeviceRadixSort::SortPairs(t, b, k0.as<uint64_t>(), k1.as<uint64_t>(), b0.as<uint32_t>(),
                                               b1.as<uint32_t>(), ni, 0, key_bits, st);
    }, st);
    if (rc) return rc;
    rc = cub_run([&](void *t, size_t &b) {
        return cub::DeviceReduce::ReduceByKey(t, b, k1.as<uint64_t>(), k0.as<uint64_t>(), b1.as<uint32_t>(),
                                              b0.as<uint32_t>(), runs.as<int64_t>(), BitOr(), ni, st);
    }, st);
    if (rc) return rc;
    int64_t m = 0;
    K2T_CUDA(cudaMemcpyAsync(&m, runs.p, 8, cudaMemcpyDeviceToHost, st));
    K2T_CUDA(cudaStreamSynchronize(st));
    s.key.swap(k0);
    s.bits.swap(b0);
    s.n = (uint64_t)m;
    return K2T_OK;
}

// The sorted path keys of the set's cells, on the device (*m of them).
int set_cells(const LeafSet &s, DevMem &cells, uint64_t *m, cudaStream_t st)
{
    *m = 0;
    if (!s.n) return cells.alloc(16);
    DevMem cnt, pos;
    int rc = cnt.alloc(s.n * 8);
    if (!rc) rc = pos.alloc(s.n * 8);
    if (rc) return rc;
    leaf_count_kernel<<<grid_of(s.n), kProdThreads, 0, st>>>(s.bits.as<uint32_t>(), s.n, cnt.as<uint64_t>());
    K2T_CUDA(cudaGetLastError());
    const int64_t ni = (int64_t)s.n;
    rc = cub_run([&](void *t, size_t &b) {
        return cub::DeviceScan::ExclusiveSum(t, b, cnt.as<uint64_t>(), pos.as<uint64_t>(), ni, st);
    }, st);
    if (rc) return rc;
    uint64_t last[2] = {0, 0};
    K2T_CUDA(cudaMemcpyAsync(&last[0], pos.as<uint64_t>() + s.n - 1, 8, cudaMemcpyDeviceToHost, st));
    K2T_CUDA(cudaMemcpyAsync(&last[1], cnt.as<uint64_t>() + s.n - 1, 8, cudaMemcpyDeviceToHost, st));
    K2T_CUDA(cudaStreamSynchronize(st));
    *m = last[0] + last[1];
    rc = cells.alloc(*m * 8);
    if (rc) return rc;
    leaf_cells_kernel<<<grid_of(s.n), kProdThreads, 0, st>>>(s.key.as<uint64_t>(), s.bits.as<uint32_t>(),
                                                              pos.as<uint64_t>(), s.n, cells.as<uint64_t>());
    K2T_CUDA(cudaGetLastError());
    return K2T_OK;
}

// out = the sorted union of two sorted key sets (device; *m keys).
int key_union(const uint64_t *a, uint64_t na, const uint64_t *b, uint64_t nb, int key_bits, DevMem &out, uint64_t *m,
              cudaStream_t st)
{
    const uint64_t n = na + nb;
    DevMem k0, k1, cnt;
    int rc = k0.alloc(n * 8);
    if (!rc) rc = k1.alloc(n * 8);
    if (!rc) rc = cnt.alloc(8);
    if (rc) return rc;
    if (na) K2T_CUDA(cudaMemcpyAsync(k0.p, a, na * 8, cudaMemcpyDeviceToDevice, st));
    if (nb) K2T_CUDA(cudaMemcpyAsync(k0.as<uint64_t>() + na, b, nb * 8, cudaMemcpyDeviceToDevice, st));
    const int64_t ni = (int64_t)n;
    rc = cub_run([&](void *t, size_t &bb) {
        return cub::DeviceRadixSort::SortKeys(t, bb, k0.as<uint64_t>(), k1.as<uint64_t>(), ni, 0, key_bits, st);
    }, st);
    if (rc) return rc;
    rc = cub_run([&](void *t, size_t &bb) {
        return cub::DeviceSelect::Unique(t, bb, k1.as<uint64_t>(), k0.as<uint64_t>(), cnt.as<int64_t>(), ni, st);
    }, st);
    if (rc) return rc;
    int64_t got = 0;
    K2T_CUDA(cudaMemcpyAsync(&got, cnt.p, 8, cudaMemcpyDeviceToHost, st));
    K2T_CUDA(cudaStreamSynchronize(st));
    out.swap(k0);
    *m = (uint64_t)got;
    return K2T_OK;
}

// Device keys -> host, then C's tree from them.
int tree_from_device_keys(const DevMem &cells, uint64_t m, uint64_t n_rows, uint64_t n_cols, const k2t_opts *opts,
                          cudaStream_t st, std::vector<uint64_t> &host, k2t_tree **out)
{
    host.resize(m);
    if (m) {
        K2T_CUDA(cudaMemcpyAsync(host.data(), cells.p, m * 8, cudaMemcpyDeviceToHost, st));
        K2T_CUDA(cudaStreamSynchronize(st));
    }
    return build_from_sorted_keys(host.data(), m, n_rows, n_cols, opts, out);
}

// One tree's levels on the device: signatures of levels 0..l-1 and
// directories of levels 0..l-2, in one allocation.
struct ProdTree {
    std::vector<ProdLevel> lv;
    void *mem = nullptr;
};

int upload_levels(const k2t_tree *t, ProdTree &pt, cudaStream_t st)
{
    const int l = t->levels;
    std::vector<std::vector<uint32_t>> dirs((size_t)l);
    uint64_t bytes = 0;
    std::vector<uint64_t> sig_off((size_t)l), dir_off((size_t)l);
    for (int d = 0; d < l; ++d) {
        sig_off[(size_t)d] = bytes;
        bytes = align_up(bytes + (t->nodes[(size_t)d] + 1) / 2 + 16, kArenaAlign);
        if (d <= l - 2) {
            level_directory(t, d, dirs[(size_t)d], 8);
            dir_off[(size_t)d] = bytes;
            bytes = align_up(bytes + dirs[(size_t)d].size() * sizeof(uint32_t), kArenaAlign);
        }
    }
    cudaError_t e = cudaMalloc(&pt.mem, bytes ? bytes : kArenaAlign);
    if (e != cudaSuccess) { g_last_cuda = (int)e; pt.mem = nullptr; return K2T_ENOMEM; }
    pt.lv.assign((size_t)l, ProdLevel{nullptr, nullptr, 0});
    char *base = static_cast<char *>(pt.mem);
    for (int d = 0; d < l; ++d) {
        ProdLevel &L = pt.lv[(size_t)d];
        L.n = (uint32_t)t->nodes[(size_t)d];
        L.sig = reinterpret_cast<const uint8_t *>(base + sig_off[(size_t)d]);
        K2T_CUDA(cudaMemsetAsync(base + sig_off[(size_t)d], 0, (t->nodes[(size_t)d] + 1) / 2 + 16, st));
        K2T_CUDA(cudaMemcpyAsync(base + sig_off[(size_t)d], t->sig[(size_t)d].data(), (t->nodes[(size_t)d] + 1) / 2,
                                 cudaMemcpyHostToDevice, st));
        if (d <= l - 2) {
            L.dir = reinterpret_cast<const uint32_t *>(base + dir_off[(size_t)d]);
            K2T_CUDA(cudaMemcpyAsync(base + dir_off[(size_t)d], dirs[(size_t)d].data(),
                                     dirs[(size_t)d].size() * sizeof(uint32_t), cudaMemcpyHostToDevice, st));
        }
    }
    // the host vectors must outlive the copies
    K2T_CUDA(cudaStreamSynchronize(st));
    return K2T_OK;
}

struct Product {
    const k2t_tree *a, *b;
    ProdTree ta, tb;
    cudaStream_t st = nullptr;
    uint32_t m = 0;                      // pairs per level buffer
    std::vector<Pair *> buf;             // per level 0..l-2
    uint32_t *cnt = nullptr, *pos = nullptr, *bsum = nullptr, *bpre = nullptr;
    uint32_t *rec = nullptr;             // records on the device
    uint64_t rec_cap = 0;
    unsigned long long *count = nullptr; // records written since the last drain
    void *scratch = nullptr;
    LeafSet set;                         // C's distinct leaves so far
    int key_bits = 64;                   // significant bits of a leaf key

    // merge the records written since the last drain into the leaf set
    int drain()
    {
        unsigned long long c = 0;
        K2T_CUDA(cudaMemcpyAsync(&c, count, sizeof(c), cudaMemcpyDeviceToHost, st));
        K2T_CUDA(cudaStreamSynchronize(st));
        if (c) {
            int rc = absorb(set, rec, (uint64_t)c, key_bits, st);
            if (rc) return rc;
            K2T_CUDA(cudaMemsetAsync(count, 0, sizeof(unsigned long long), st));
        }
        return K2T_OK;
    }

    // pairs p[0..n) of level d (n <= m)
    int process(int d, const Pair *p, uint32_t n)
    {
        const int l = a->levels;
        if (!n) return K2T_OK;
        if (d == l - 2) {
            unsigned long long c = 0;
            K2T_CUDA(cudaMemcpyAsync(&c, count, sizeof(c), cudaMemcpyDeviceToHost, st));
            K2T_CUDA(cudaStreamSynchronize(st));
            if (c + 8ull * n > rec_cap) {
                int rc = drain();
                if (rc) return rc;
            }
            pair_leaf_kernel<<<(n + kProdThreads - 1) / kProdThreads, kProdThreads, 0, st>>>(
                ta.lv[(size_t)d], tb.lv[(size_t)d], ta.lv[(size_t)l - 1].sig, tb.lv[(size_t)l - 1].sig, p, n, rec,
                count);
            K2T_CUDA(cudaGetLastError());
            return K2T_OK;
        }
        const uint32_t tile = m / 8;
        for (uint32_t s = 0; s < n; s += tile) {
            const uint32_t k = std::min(tile, n - s);
            const uint32_t blocks = (k + kProdThreads - 1) / kProdThreads;
            pair_count_kernel<<<blocks, kProdThreads, 0, st>>>(ta.lv[(size_t)d], tb.lv[(size_t)d], p + s, k, cnt);
            block_scan_kernel<<<blocks, kProdThreads, 0, st>>>(cnt, k, pos, bsum);
            ls_scan_kernel<<<1, 1024, 0, st>>>(bsum, blocks, bpre);
            pair_expand_kernel<<<blocks, kProdThreads, 0, st>>>(ta.lv[(size_t)d], tb.lv[(size_t)d], p + s, k, pos,
                                                                bpre, buf[(size_t)d + 1]);
            K2T_CUDA(cudaGetLastError());
            uint32_t total = 0;
            K2T_CUDA(cudaMemcpyAsync(&total, bpre + blocks, sizeof(total), cudaMemcpyDeviceToHost, st));
            K2T_CUDA(cudaStreamSynchronize(st));
            int rc = process(d + 1, buf[(size_t)d + 1], total);
            if (rc) return rc;
        }
        return K2T_OK;
    }

    ~Product()
    {
        if (scratch) cudaFree(scratch);
        if (ta.mem) cudaFree(ta.mem);
        if (tb.mem) cudaFree(tb.mem);
    }
};

bool plain_k2(const k2t_tree *t) { return t->n_k4 == 0 && !t->leaf_k4; }

// C = A B on the device: the pair descent, its records merged into C's leaf
// set, then the sorted path keys of C's cells (*m of them) in `cells`.
int run_product(const k2t_tree *a, const k2t_tree *b, cudaStream_t st, DevMem &cells, uint64_t *m)
{
    *m = 0;
    if (a->empty || b->empty) return cells.alloc(16);
    Product P;
    P.a = a;
    P.b = b;
    P.st = st;
    P.key_bits = std::max(2 * (a->dim_bits - 1), 1);
    int rc = upload_levels(a, P.ta, P.st);
    if (!rc) rc = upload_levels(b, P.tb, P.st);
    if (rc) return rc;
    const int l = a->levels;
    P.m = 1u << 20;
    P.rec_cap = 32ull * P.m;  // records between merges into the leaf set
    const uint32_t tile = P.m / 8;
    const uint32_t tblocks = (tile + kProdThreads - 1) / kProdThreads;
    uint64_t bytes = 0;
    std::vector<uint64_t> buf_off((size_t)l, 0);
    for (int d = 1; d <= l - 2; ++d) {
        buf_off[(size_t)d] = bytes;
        bytes = align_up(bytes + (uint64_t)P.m * sizeof(Pair), kArenaAlign);
    }
    const uint64_t root_off = bytes;
    bytes = align_up(bytes + sizeof(Pair), kArenaAlign);
    const uint64_t cnt_off = bytes;
    bytes = align_up(bytes + (uint64_t)tile * 4, kArenaAlign);
    const uint64_t pos_off = bytes;
    bytes = align_up(bytes + (uint64_t)tile * 4, kArenaAlign);
    const uint64_t bsum_off = bytes;
    bytes = align_up(bytes + (uint64_t)(tblocks + 1) * 4, kArenaAlign);
    const uint64_t bpre_off = bytes;
    bytes = align_up(bytes + (uint64_t)(tblocks + 1) * 4, kArenaAlign);
    const uint64_t count_off = bytes;
    bytes = align_up(bytes + 8, kArenaAlign);
    const uint64_t rec_off = bytes;
    bytes = align_up(bytes + P.rec_cap * 12, kArenaAlign);
    cudaError_t e = cudaMalloc(&P.scratch, bytes);
    if (e != cudaSuccess) { g_last_cuda = (int)e; P.scratch = nullptr; return K2T_ENOMEM; }
    char *base = static_cast<char *>(P.scratch);
    P.buf.assign((size_t)l, nullptr);
    for (int d = 1; d <= l - 2; ++d) P.buf[(size_t)d] = reinterpret_cast<Pair *>(base + buf_off[(size_t)d]);
    Pair *root = reinterpret_cast<Pair *>(base + root_off);
    P.cnt = reinterpret_cast<uint32_t *>(base + cnt_off);
    P.pos = reinterpret_cast<uint32_t *>(base + pos_off);
    P.bsum = reinterpret_cast<uint32_t *>(base + bsum_off);
    P.bpre = reinterpret_cast<uint32_t *>(base + bpre_off);
    P.count = reinterpret_cast<unsigned long long *>(base + count_off);
    P.rec = reinterpret_cast<uint32_t *>(base + rec_off);
    const Pair r0{0u, 0u, 0u, 0u};
    K2T_CUDA(cudaMemcpyAsync(root, &r0, sizeof(Pair), cudaMemcpyHostToDevice, P.st));
    K2T_CUDA(cudaMemsetAsync(P.count, 0, sizeof(unsigned long long), P.st));
    K2T_CUDA(cudaStreamSynchronize(P.st));
    rc = P.process(0, root, 1u);
    if (!rc) rc = P.drain();
    if (!rc) rc = set_cells(P.set, cells, m, st);
    return rc;
}

}  // namespace
}  // namespace k2t

using namespace k2t;

extern "C" {

int k2t_bool_product(const k2t_tree *a, const k2t_tree *b, const k2t_opts *opts, k2t_tree **out, void *stream)
{
    if (!a || !b || !out) return K2T_EINVAL;
    *out = nullptr;
    if (a->n_cols != b->n_rows || a->dim_bits != b->dim_bits || !plain_k2(a) || !plain_k2(b)) return K2T_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DevMem cells;
    uint64_t m = 0;
    int rc = run_product(a, b, st, cells, &m);
    if (rc) return rc;
    std::vector<uint64_t> host;
    return tree_from_device_keys(cells, m, a->n_rows, b->n_cols, opts, st, host, out);
}

int k2t_bool_closure(const k2t_tree *a, const k2t_opts *opts, uint32_t max_iters, k2t_tree **out, uint32_t *iters,
                     void *stream)
{
    if (!a || !out || !iters) return K2T_EINVAL;
    *out = nullptr;
    *iters = 0;
    if (a->n_rows != a->n_cols || !plain_k2(a)) return K2T_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // every squaring takes a tree with 2x2 leaves: an automatic leaf size
    // resolves to 2 here (an explicit 4 fails in the first squaring)
    k2t_opts wo;
    if (opts) wo = *opts; else k2t_default_opts(&wo);
    if (wo.leaf_k == 0) wo.leaf_k = 2;
    if (wo.leaf_k != 2) return K2T_EINVAL;
    // the trees between squarings only feed the next product: no heavy tables
    k2t_opts io = wo;
    io.heavy_terms = 0xffffffffu;
    // C <- A: its cells, in level order, are its sorted path keys
    std::vector<uint32_t> r(a->nnz), c(a->nnz);
    uint64_t got = 0;
    int rc = k2t_decode(a, r.data(), c.data(), a->nnz, &got);
    if (rc) return rc;
    const int key_bits = std::max(2 * a->dim_bits, 1);
    DevMem cur_keys;
    uint64_t m_cur = got;
    {
        DevMem dr, dc;
        rc = dr.alloc(got * 4);
        if (!rc) rc = dc.alloc(got * 4);
        if (!rc) rc = cur_keys.alloc(got * 8);
        if (rc) return rc;
        if (got) {
            K2T_CUDA(cudaMemcpyAsync(dr.p, r.data(), got * 4, cudaMemcpyHostToDevice, st));
            K2T_CUDA(cudaMemcpyAsync(dc.p, c.data(), got * 4, cudaMemcpyHostToDevice, st));
            cell_keys_kernel<<<grid_of(got), kProdThreads, 0, st>>>(dr.as<uint32_t>(), dc.as<uint32_t>(), got,
                                                                      cur_keys.as<uint64_t>());
            K2T_CUDA(cudaGetLastError());
        }
        K2T_CUDA(cudaStreamSynchronize(st));
    }
    std::vector<uint64_t> host;
    k2t_tree *cur = nullptr;
    rc = tree_from_device_keys(cur_keys, m_cur, a->n_rows, a->n_cols, &io, st, host, &cur);
    if (rc) return rc;
    for (uint32_t it = 0; it < max_iters; ++it) {
        DevMem sq;
        uint64_t m_sq = 0;
        rc = run_product(cur, cur, st, sq, &m_sq);
        if (rc) { k2t_free(cur); return rc; }
        *iters = it + 1;
        // C or C C, on the device
        DevMem nxt;
        uint64_t m_nxt = 0;
        rc = key_union(cur_keys.as<uint64_t>(), m_cur, sq.as<uint64_t>(), m_sq, key_bits, nxt, &m_nxt, st);
        if (rc) { k2t_free(cur); return rc; }
        if (m_nxt == m_cur) break;   // C stopped growing
        k2t_free(cur);
        cur = nullptr;
        cur_keys.swap(nxt);
        m_cur = m_nxt;
        if (it + 1 < max_iters) {
            rc = tree_from_device_keys(cur_keys, m_cur, a->n_rows, a->n_cols, &io, st, host, &cur);
            if (rc) return rc;
        }
    }
    if (cur) k2t_free(cur);
    // the result, with the caller's options
    return tree_from_device_keys(cur_keys, m_cur, a->n_rows, a->n_cols, &wo, st, host, out);
}

}  // extern "C"
