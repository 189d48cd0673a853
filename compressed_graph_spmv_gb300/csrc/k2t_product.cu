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
//    pairs.  The records of C, with repeats (several k reach one block), go to
//    the host, which builds C's tree with k2t_build (repeats collapse there).
//
// Requirements: A is n x m and B is m x p with the same padded side and
// k = 2 on every level (no hybrid top, 2x2 leaves).  The trees need not be
// uploaded: the product copies what it reads (every level's signatures and
// directory) to its own device memory and frees it on return.
#include <algorithm>
#include <vector>

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

namespace {

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
    std::vector<uint32_t> out;           // drained records (3 words each)

    int drain()
    {
        unsigned long long c = 0;
        K2T_CUDA(cudaMemcpyAsync(&c, count, sizeof(c), cudaMemcpyDeviceToHost, st));
        K2T_CUDA(cudaStreamSynchronize(st));
        if (c) {
            const size_t at = out.size();
            out.resize(at + 3 * (size_t)c);
            K2T_CUDA(cudaMemcpyAsync(out.data() + at, rec, 3 * (size_t)c * sizeof(uint32_t), cudaMemcpyDeviceToHost, st));
            K2T_CUDA(cudaMemsetAsync(count, 0, sizeof(unsigned long long), st));
            K2T_CUDA(cudaStreamSynchronize(st));
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

// Distinct cells of C from the records, then C's tree.
int build_from_records(const std::vector<uint32_t> &recs, uint64_t n_rows, uint64_t n_cols, const k2t_opts *opts,
                       k2t_tree **out)
{
    std::vector<uint32_t> rows, cols;
    const size_t nrec = recs.size() / 3;
    rows.reserve(nrec * 2);
    cols.reserve(nrec * 2);
    for (size_t r = 0; r < nrec; ++r) {
        const uint32_t lr = recs[3 * r], lc = recs[3 * r + 1], bits = recs[3 * r + 2];
        for (uint32_t b = 0; b < 4; ++b)
            if ((bits >> b) & 1u) {
                rows.push_back(2u * lr + (b >> 1));
                cols.push_back(2u * lc + (b & 1u));
            }
    }
    return k2t_build(rows.data(), cols.data(), rows.size(), n_rows, n_cols, opts, out);
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
    if (a->empty || b->empty) {
        std::vector<uint32_t> none;
        return build_from_records(none, a->n_rows, b->n_cols, opts, out);
    }
    Product P;
    P.a = a;
    P.b = b;
    P.st = static_cast<cudaStream_t>(stream);
    int rc = upload_levels(a, P.ta, P.st);
    if (!rc) rc = upload_levels(b, P.tb, P.st);
    if (rc) return rc;
    const int l = a->levels;
    P.m = 1u << 20;
    P.rec_cap = 8ull * P.m;  // a full level buffer of pairs has at most 8 leaf products each
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
    if (rc) return rc;
    return build_from_records(P.out, a->n_rows, b->n_cols, opts, out);
}

int k2t_bool_closure(const k2t_tree *a, const k2t_opts *opts, uint32_t max_iters, k2t_tree **out, uint32_t *iters,
                     void *stream)
{
    if (!a || !out || !iters) return K2T_EINVAL;
    *out = nullptr;
    *iters = 0;
    if (a->n_rows != a->n_cols || !plain_k2(a)) return K2T_EINVAL;
    // every squaring takes a tree with 2x2 leaves: an automatic leaf size
    // resolves to 2 here (an explicit 4 fails in the first squaring)
    k2t_opts wo;
    if (opts) wo = *opts; else k2t_default_opts(&wo);
    if (wo.leaf_k == 0) wo.leaf_k = 2;
    opts = &wo;
    // C <- A, rebuilt with the caller's options
    std::vector<uint32_t> r(a->nnz), c(a->nnz);
    uint64_t got = 0;
    int rc = k2t_decode(a, r.data(), c.data(), a->nnz, &got);
    if (rc) return rc;
    k2t_tree *cur = nullptr;
    rc = k2t_build(r.data(), c.data(), got, a->n_rows, a->n_cols, opts, &cur);
    if (rc) return rc;
    for (uint32_t it = 0; it < max_iters; ++it) {
        if (cur->dim_bits != a->dim_bits || !plain_k2(cur)) { k2t_free(cur); return K2T_EINVAL; }
        k2t_tree *sq = nullptr;
        rc = k2t_bool_product(cur, cur, opts, &sq, stream);
        if (rc) { k2t_free(cur); return rc; }
        *iters = it + 1;
        // C or C C
        std::vector<uint32_t> rr(cur->nnz + sq->nnz), cc(cur->nnz + sq->nnz);
        uint64_t n1 = 0, n2 = 0;
        rc = k2t_decode(cur, rr.data(), cc.data(), cur->nnz, &n1);
        if (!rc) rc = k2t_decode(sq, rr.data() + n1, cc.data() + n1, sq->nnz, &n2);
        k2t_free(sq);
        if (rc) { k2t_free(cur); return rc; }
        k2t_tree *nxt = nullptr;
        rc = k2t_build(rr.data(), cc.data(), n1 + n2, a->n_rows, a->n_cols, opts, &nxt);
        if (rc) { k2t_free(cur); return rc; }
        const bool done = nxt->nnz == cur->nnz;
        k2t_free(cur);
        cur = nxt;
        if (done) break;
    }
    *out = cur;
    return K2T_OK;
}

}  // extern "C"
