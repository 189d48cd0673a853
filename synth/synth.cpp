// synth.cpp -- seeded synthetic graph generators.
//
// These generators produce the inputs (COO edge lists) that both the library
// and the CPU oracle consume.  They hold none of the product's arithmetic:
// no tree, no Morton codes, no semiring.  Every random draw is a pure
// function of (seed, draw index), so the output is the same for any number
// of host threads and on any host architecture (integer arithmetic only;
// floating-point constants are compared as fixed-point integers).
//
// Random source: the SplitMix64 output function (Steele, Lea & Flood,
// "Fast splittable pseudorandom number generators", OOPSLA 2014) applied to a
// counter, i.e. hash(seed, index).
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <functional>
#include <cstdlib>
#include <thread>
#include <vector>

namespace {

inline uint64_t splitmix(uint64_t z)
{
    z += 0x9e3779b97f4a7c15ull;
    z = (z ^ (z >> 30)) * 0xbf58476d1ce4e5b9ull;
    z = (z ^ (z >> 27)) * 0x94d049bb133111ebull;
    return z ^ (z >> 31);
}

inline uint64_t draw(uint64_t seed, uint64_t stream, uint64_t index)
{
    return splitmix(splitmix(seed ^ (stream * 0xd1b54a32d192ed03ull)) + index * 0x9e3779b97f4a7c15ull);
}

// All hardware threads, or K2T_SYNTH_THREADS when set (the output does not
// depend on it; tests vary it to check that).
int nthreads()
{
    if (const char *e = std::getenv("K2T_SYNTH_THREADS")) {
        int v = std::atoi(e);
        if (v > 0) return v;
    }
    unsigned h = std::thread::hardware_concurrency();
    return h ? (int)h : 4;
}

void parallel_for(int nt, const std::function<void(int)> &fn)
{
    std::vector<std::thread> th;
    th.reserve(nt);
    for (int t = 0; t < nt; ++t) th.emplace_back(fn, t);
    for (auto &x : th) x.join();
}

// Stable LSD radix sort of 64-bit keys on their low `bits` bits, 8 bits per pass.
void radix_sort(std::vector<uint64_t> &a, int bits)
{
    size_t n = a.size();
    if (n < 2) return;
    std::vector<uint64_t> b(n);
    int nt = nthreads();
    std::vector<size_t> hist((size_t)nt * 256);
    for (int shift = 0; shift < bits; shift += 8) {
        std::fill(hist.begin(), hist.end(), 0);
        parallel_for(nt, [&](int t) {
            size_t lo = n * t / nt, hi = n * (t + 1) / nt;
            size_t *h = &hist[(size_t)t * 256];
            for (size_t i = lo; i < hi; ++i) h[(a[i] >> shift) & 255]++;
        });
        // skip a pass where every key has the same digit
        int nonzero = 0;
        for (int d = 0; d < 256; ++d) {
            size_t s = 0;
            for (int t = 0; t < nt; ++t) s += hist[(size_t)t * 256 + d];
            if (s) ++nonzero;
        }
        if (nonzero <= 1) continue;
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
            for (size_t i = lo; i < hi; ++i) b[h[(a[i] >> shift) & 255]++] = a[i];
        });
        a.swap(b);
    }
}

void unique_sorted(std::vector<uint64_t> &a)
{
    a.erase(std::unique(a.begin(), a.end()), a.end());
}

// Keep exactly `target` keys of a sorted unique array: those with the smallest
// hash(seed, key) (a uniform random subset), preserving sorted order.
void truncate_by_hash(std::vector<uint64_t> &a, uint64_t target, uint64_t seed)
{
    if (a.size() <= target) return;
    std::vector<uint64_t> h(a.size());
    int nt = nthreads();
    size_t n = a.size();
    parallel_for(nt, [&](int t) {
        size_t lo = n * t / nt, hi = n * (t + 1) / nt;
        for (size_t i = lo; i < hi; ++i) h[i] = draw(seed, 7, a[i]);
    });
    std::vector<uint64_t> hs(h);
    std::nth_element(hs.begin(), hs.begin() + (ptrdiff_t)(target - 1), hs.end());
    uint64_t thr = hs[target - 1];
    std::vector<uint64_t>().swap(hs);
    size_t w = 0, kept_eq = 0;
    size_t below = 0;
    for (size_t i = 0; i < n; ++i) below += h[i] < thr;
    size_t eq_budget = target - below;
    for (size_t i = 0; i < n; ++i) {
        if (h[i] < thr || (h[i] == thr && kept_eq < eq_budget)) {
            if (h[i] == thr) ++kept_eq;
            a[w++] = a[i];
        }
    }
    a.resize(w);
}

// Fixed-point (2^-32) thresholds of a probability vector.
struct Quad { uint64_t t0, t1, t2; };

Quad thresholds(double a, double b, double c)
{
    Quad q;
    q.t0 = (uint64_t)std::floor(a * 4294967296.0);
    q.t1 = (uint64_t)std::floor((a + b) * 4294967296.0);
    q.t2 = (uint64_t)std::floor((a + b + c) * 4294967296.0);
    return q;
}

// Sample `count` R-MAT edges with indices [first, first+count) into keys
// (row << scale | col), self-loops dropped, optionally with the reverse edge
// (as the canonical pair min/max when `undirected`).
void rmat_sample(std::vector<uint64_t> &out, uint64_t first, uint64_t count, int scale,
                 const Quad &q, uint64_t seed, bool undirected)
{
    int nt = nthreads();
    std::vector<std::vector<uint64_t>> part(nt);
    parallel_for(nt, [&](int t) {
        uint64_t lo = first + count * t / nt, hi = first + count * (t + 1) / nt;
        auto &p = part[t];
        p.reserve(hi - lo);
        for (uint64_t i = lo; i < hi; ++i) {
            uint64_t r = 0, c = 0, bits = 0;
            for (int lev = 0; lev < scale; ++lev) {
                if ((lev & 1) == 0) bits = draw(seed, 1, i * 32 + (uint64_t)(lev >> 1));
                uint64_t u = (lev & 1) ? (bits >> 32) : (bits & 0xffffffffull);
                int quad = u < q.t0 ? 0 : (u < q.t1 ? 1 : (u < q.t2 ? 2 : 3));
                r = (r << 1) | (uint64_t)(quad >> 1);
                c = (c << 1) | (uint64_t)(quad & 1);
            }
            if (r == c) continue;
            if (undirected && r > c) std::swap(r, c);
            p.push_back((r << scale) | c);
        }
    });
    size_t total = out.size();
    for (auto &p : part) total += p.size();
    out.reserve(total);
    for (auto &p : part) { out.insert(out.end(), p.begin(), p.end()); std::vector<uint64_t>().swap(p); }
}

} // namespace

struct SynthEdges {
    std::vector<uint64_t> keys;  // (row << shift) | col, sorted
    int shift;
};

extern "C" {

// Edge lists are returned through an opaque handle: query the size, copy the
// rows and columns out, then free it.
uint64_t synth_edges_size(void *h) { return static_cast<SynthEdges *>(h)->keys.size(); }

void synth_edges_copy(void *h, uint32_t *rows, uint32_t *cols)
{
    auto *e = static_cast<SynthEdges *>(h);
    uint64_t mask = (1ull << e->shift) - 1;
    size_t n = e->keys.size();
    int nt = nthreads();
    parallel_for(nt, [&](int t) {
        size_t lo = n * t / nt, hi = n * (t + 1) / nt;
        for (size_t i = lo; i < hi; ++i) {
            rows[i] = (uint32_t)(e->keys[i] >> e->shift);
            cols[i] = (uint32_t)(e->keys[i] & mask);
        }
    });
}

void synth_edges_free(void *h) { delete static_cast<SynthEdges *>(h); }

// R-MAT graph on 2^scale vertices with (a, b, c, 1-a-b-c) quadrant
// probabilities (a: top-left, b: top-right, c: bottom-left).  Samples are
// drawn in index order until the distinct non-loop edges reach `target`
// (directed) or target/2 distinct unordered pairs (symmetric), then exactly
// that many are kept, chosen by smallest hash(seed, edge).  Symmetric graphs
// add the reverse of every kept pair.  Output is sorted by (row, col).
void *synth_rmat(int scale, double a, double b, double c, uint64_t target, uint64_t seed, int symmetric)
{
    if (scale < 1 || scale > 31) return nullptr;
    Quad q = thresholds(a, b, c);
    uint64_t want = symmetric ? target / 2 : target;
    auto *res = new SynthEdges;
    res->shift = scale;
    std::vector<uint64_t> &keys = res->keys;
    uint64_t drawn = 0;
    uint64_t next = want + want / 8 + 1024;
    for (int round = 0; round < 64; ++round) {
        rmat_sample(keys, drawn, next, scale, q, seed, symmetric != 0);
        drawn += next;
        radix_sort(keys, 2 * scale);
        unique_sorted(keys);
        if (keys.size() >= want) break;
        double per = (double)keys.size() / (double)drawn;  // distinct yield per draw
        uint64_t short_by = want - keys.size();
        next = (uint64_t)((double)short_by / std::max(per * 0.5, 1e-3)) + 1024;
    }
    truncate_by_hash(keys, want, seed);
    uint64_t mask = (1ull << scale) - 1;
    if (symmetric) {
        size_t n0 = keys.size();
        keys.resize(2 * n0);
        for (size_t i = 0; i < n0; ++i) {
            uint64_t r = keys[i] >> scale, cc = keys[i] & mask;
            keys[n0 + i] = (cc << scale) | r;
        }
        radix_sort(keys, 2 * scale);
    }
    return res;
}

// Web-like locality graph on n vertices: every source draws a Poisson(lambda)
// out-degree (inversion against a CDF built by products and quotients);
// each target is src + U{-window..window} with probability local_frac, else
// U[0, n).  Out-of-range targets, self-loops and duplicates are dropped.
// Output sorted by (row, col).
void *synth_weblike(uint64_t n, double lambda, double local_frac, int64_t window, uint64_t seed)
{
    std::vector<uint64_t> cdf;
    // exp(-lambda) as 1 / sum_k lambda^k / k! (positive terms, basic operations
    // only, so every IEEE host computes the same bits without a libm call)
    double e = 0.0, term = 1.0;
    for (int k = 0; k < 400; ++k) { e += term; term = term * lambda / (double)(k + 1); }
    double p = 1.0 / e, s = 0.0;
    for (int k = 0; k < 1000 && s < 1.0; ++k) {
        if (k > 0) p = p * lambda / (double)k;
        s += p;
        cdf.push_back((uint64_t)std::min(9007199254740991.0, std::floor(s * 9007199254740992.0)));
        if (k > lambda && p < 1e-18) break;
    }
    uint64_t loc_thr = (uint64_t)std::floor(local_frac * 4294967296.0);
    uint64_t span = (uint64_t)(2 * window + 1);
    int nt = nthreads();
    std::vector<std::vector<uint64_t>> part(nt);
    parallel_for(nt, [&](int t) {
        uint64_t lo = n * t / nt, hi = n * (t + 1) / nt;
        auto &out = part[t];
        std::vector<uint64_t> tmp;
        for (uint64_t src = lo; src < hi; ++src) {
            uint64_t u = draw(seed, 2, src) >> 11;  // 53 bits
            int deg = 0;
            while (deg < (int)cdf.size() && u >= cdf[deg]) ++deg;
            tmp.clear();
            for (int k = 0; k < deg; ++k) {
                uint64_t r1 = draw(seed, 3, src * 4096 + (uint64_t)k);
                uint64_t r2 = draw(seed, 4, src * 4096 + (uint64_t)k);
                int64_t tgt;
                if ((r1 & 0xffffffffull) < loc_thr) {
                    int64_t off = (int64_t)(((r2 & 0xffffffffull) * span) >> 32) - window;
                    tgt = (int64_t)src + off;
                } else {
                    unsigned __int128 m = (unsigned __int128)r2 * n;
                    tgt = (int64_t)(uint64_t)(m >> 64);
                }
                if (tgt < 0 || (uint64_t)tgt >= n || (uint64_t)tgt == src) continue;
                tmp.push_back((uint64_t)tgt);
            }
            std::sort(tmp.begin(), tmp.end());
            tmp.erase(std::unique(tmp.begin(), tmp.end()), tmp.end());
            for (uint64_t v : tmp) out.push_back((src << 32) | v);
        }
    });
    auto *res = new SynthEdges;
    res->shift = 32;
    uint64_t total = 0;
    for (auto &pp : part) total += pp.size();
    res->keys.reserve(total);
    for (auto &pp : part) res->keys.insert(res->keys.end(), pp.begin(), pp.end());
    return res;
}

// Relabel vertex ids in place: first a uniform random permutation (Fisher-Yates
// over counter-based draws), then breadth-first order: a directed BFS over
// out-edges from the vertex of largest out-degree (ties: smallest id), visiting
// neighbours in increasing id; vertices never reached follow in increasing id.
// The final id of a vertex is its position in that order.
void synth_permute_bfs(uint64_t n, uint32_t *rows, uint32_t *cols, uint64_t nnz, uint64_t seed)
{
    std::vector<uint32_t> perm(n);
    for (uint64_t i = 0; i < n; ++i) perm[i] = (uint32_t)i;
    for (uint64_t i = n; i > 1; --i) {
        unsigned __int128 m = (unsigned __int128)draw(seed, 5, i) * i;
        uint64_t j = (uint64_t)(m >> 64);
        std::swap(perm[i - 1], perm[j]);
    }
    int nt = nthreads();
    parallel_for(nt, [&](int t) {
        uint64_t lo = nnz * t / nt, hi = nnz * (t + 1) / nt;
        for (uint64_t e = lo; e < hi; ++e) { rows[e] = perm[rows[e]]; cols[e] = perm[cols[e]]; }
    });
    std::vector<uint32_t>().swap(perm);
    // CSR by source (counting sort), neighbours sorted per row
    std::vector<uint64_t> ptr(n + 1, 0);
    for (uint64_t e = 0; e < nnz; ++e) ptr[rows[e] + 1]++;
    for (uint64_t v = 0; v < n; ++v) ptr[v + 1] += ptr[v];
    std::vector<uint32_t> adj(nnz);
    {
        std::vector<uint64_t> at(ptr.begin(), ptr.end() - 1);
        for (uint64_t e = 0; e < nnz; ++e) adj[at[rows[e]]++] = cols[e];
    }
    parallel_for(nt, [&](int t) {
        uint64_t lo = n * t / nt, hi = n * (t + 1) / nt;
        for (uint64_t v = lo; v < hi; ++v) std::sort(adj.begin() + (ptrdiff_t)ptr[v], adj.begin() + (ptrdiff_t)ptr[v + 1]);
    });
    uint64_t root = 0, best = 0;
    for (uint64_t v = 0; v < n; ++v) {
        uint64_t d = ptr[v + 1] - ptr[v];
        if (d > best) { best = d; root = v; }
    }
    const uint32_t NONE = 0xffffffffu;
    std::vector<uint32_t> order(n, NONE);  // new id of each vertex
    std::vector<uint32_t> queue;
    queue.reserve(n);
    uint64_t next_id = 0;
    if (n) {
        order[root] = (uint32_t)next_id++;
        queue.push_back((uint32_t)root);
        for (size_t h = 0; h < queue.size(); ++h) {
            uint32_t v = queue[h];
            for (uint64_t k = ptr[v]; k < ptr[v + 1]; ++k) {
                uint32_t u = adj[k];
                if (order[u] == NONE) { order[u] = (uint32_t)next_id++; queue.push_back(u); }
            }
        }
    }
    for (uint64_t v = 0; v < n; ++v)
        if (order[v] == NONE) order[v] = (uint32_t)next_id++;
    parallel_for(nt, [&](int t) {
        uint64_t lo = nnz * t / nt, hi = nnz * (t + 1) / nt;
        for (uint64_t e = lo; e < hi; ++e) { rows[e] = order[rows[e]]; cols[e] = order[cols[e]]; }
    });
}

} // extern "C"
