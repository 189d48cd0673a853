// k2t_device.cu -- sm_103a kernels and the device half of the C ABI.
//
// What a product computes follows Algorithm 1 of "A GPU Engine for Sparse
// Matrix-Vector Products on k^2-Tree-Compressed Graphs": y is filled with the
// semiring zero, the frontier of a cached level is expanded level by level
// (child j of node t at position off_t + j, off_t the exclusive prefix sum of
// the fan-outs), and the nodes of the last internal level visit their leaves
// in place, adding w (x) x_c to y_r for every set cell (r, c) with one atomic
// of the semiring (Table 1).  Left products swap the decoded coordinates
// (section 3.6); batches update B contiguous entries per cell (section 3.6).
//
// Three engines share the leaf step:
//   FUSED      one launch; each thread block takes a chunk of whole subtrees
//              and descends it level by level in shared memory, offsets from
//              block-wide scans of the fan-outs; no global scratch.
//   LEVELSYNC  the tiled descent of section 3.4: one launch per tile and
//              level, frontier codes in global buffers of at most M entries,
//              offsets from the directory or from a per-tile scan (3.2);
//              optionally replayed as one CUDA graph.
//   CACHED     the k^2+F configuration of section 3.5: one leaf kernel over
//              the cached coordinates of the last internal level.
//
// A frontier entry is the pair (row, col) of its block in units of the
// block side of its level, rather than the pages' 64-bit Morton code: the
// same information, one shift-or per coordinate per level, and nothing to
// deinterleave at the leaves.
#include <algorithm>

#include "k2t_kernels.cuh"

namespace k2t {

thread_local int g_last_cuda = 0;

// y <- 0bar: `words` 32-bit words set to `pattern` (Algorithm 1, line 1).
__global__ void __launch_bounds__(256) fill_kernel(uint32_t *y, uint64_t words, uint32_t pattern)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    const uint64_t head = (16u - ((uintptr_t)y & 15u)) / 4u % 4u;  // words before 16-byte alignment
    if (i < head && i < words) y[i] = pattern;
    uint64_t nvec = words > head ? (words - head) / 4 : 0;
    uint4 p4 = make_uint4(pattern, pattern, pattern, pattern);
    uint4 *v = reinterpret_cast<uint4 *>(y + head);
    for (uint64_t k = i; k < nvec; k += stride) v[k] = p4;
    uint64_t tail = head + nvec * 4;
    for (uint64_t k = tail + i; k < words; k += stride) y[k] = pattern;
}

// Heavy outputs of a plus-times product: output list[i] of vector k receives
// its sum, rounded to fp32 once: the 2^bits fp32 partial sums of its record
// (rows first .. first + 2^bits - 1 of acc) added in fp64, or, for bits
// kHeavyFp64, its fp64 slot (rows first, first + 1: B doubles).  The product
// sends every term of such an output there, so y holds the fill's zero;
// adding it keeps the result right even if it did not.
//  - B >= 8 dividing 32: a group of B lanes per output (32 / B outputs per
//    warp at once), lane k summing slice k down the partial rows, four rows
//    in flight;
//  - otherwise one warp per output, the lanes striding over its words.
__global__ void __launch_bounds__(256) heavy_finish_kernel(const float *acc, const uint32_t *hdir,
                                                           const uint32_t *list, uint32_t h, uint32_t B, float *y)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint64_t warps = (uint64_t)gridDim.x * (blockDim.x >> 5);
    const uint64_t gw = (uint64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (B >= 8u && 32u % B == 0) {
        const uint32_t per = 32u / B, sub = lane / B, k = lane % B;
        for (uint64_t id = gw * per + sub; id < (uint64_t)h + sub; id += warps * per) {
            if (id >= h) continue;
            const uint32_t o = __ldg(list + id);
            const uint32_t rec = __ldg(hdir + o);
            const uint32_t bits = rec & 31u;
            const uint64_t first = rec >> 5;
            const uint64_t parts = bits == kHeavyFp64 ? 0u : ((uint64_t)1 << bits);
            const float *a = acc + first * B + k;
            double s = 0.0;
            uint64_t p = 0;
            for (; p + 4 <= parts; p += 4)
                s += ((double)__ldg(a + p * B) + (double)__ldg(a + (p + 1) * B)) +
                     ((double)__ldg(a + (p + 2) * B) + (double)__ldg(a + (p + 3) * B));
            for (; p < parts; ++p) s += (double)__ldg(a + p * B);
            if (!parts) s = reinterpret_cast<const double *>(acc + first * B)[k];   // fp64 slot
            float *yo = y + (uint64_t)o * B + k;
            *yo = __double2float_rn(s + (double)*yo);
        }
        return;
    }
    for (uint64_t id = gw; id < h; id += warps) {
        const uint32_t o = __ldg(list + id);
        const uint32_t rec = __ldg(hdir + o);
        const uint32_t bits = rec & 31u;
        const uint64_t first = rec >> 5;
        const uint64_t parts = bits == kHeavyFp64 ? 0u : ((uint64_t)1 << bits);
        const double *a64 = reinterpret_cast<const double *>(acc + first * B);   // fp64 slot (parts == 0)
        float *yo = y + (uint64_t)o * B;
        const uint64_t words = parts * B;
        const float *a = acc + first * B;
        if (32u % B == 0) {
            // lane l always reads slice l % B: sum, then fold the lanes of one slice
            double s = 0.0;
            for (uint64_t e = lane; e < words; e += 32u) s += (double)a[e];
            for (uint32_t f = 16; f >= B; f >>= 1) s += __shfl_xor_sync(0xffffffffu, s, f);
            if (lane < B) yo[lane] = __double2float_rn(s + (parts ? 0.0 : a64[lane]) + (double)yo[lane]);
        } else {
            for (uint32_t k = 0; k < B; ++k) {
                double s = 0.0;
                for (uint64_t e = k + (uint64_t)lane * B; e < words; e += 32ull * B) s += (double)a[e];
#pragma unroll
                for (int f = 16; f > 0; f >>= 1) s += __shfl_xor_sync(0xffffffffu, s, f);
                if (lane == 0) yo[k] = __double2float_rn(s + (parts ? 0.0 : a64[k]) + (double)yo[k]);
            }
        }
    }
}

// Algorithm 1, lines 5-10, for one tile: the frontier entries of nodes
// [a, a+count) (read from src at index t - src_base) expand into their
// children's entries, written at dst[child - dst_base].
__global__ void __launch_bounds__(kWalkThreads)
ls_expand_kernel(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix, uint32_t a, uint32_t count,
                 const Coord *src, uint32_t src_base, Coord *dst, uint32_t dst_base, uint64_t dst_entries,
                 uint32_t *status)
{
    const uint32_t wid = blockIdx.x * (kWalkThreads / 32) + (threadIdx.x >> 5);
    uint32_t s, e, base;
    if (!tile_block(sig, dir, prefix, a, count, dst_base, wid, s, e, base)) return;
    warp_walk(sig, s, e, base, [&](uint32_t t, uint32_t sg, uint32_t pos) {
        if (!K2T_IN_RANGE((uint64_t)(pos - dst_base) + (uint32_t)__popc(sg) <= dst_entries, status)) return;
        const Coord p = src[t - src_base];
        Coord *o = dst + (pos - dst_base);
#pragma unroll
        for (int b = 0; b < 4; ++b)
            if (sg & (1u << b)) *o++ = child_of(p, b);
    });
}

// Scan offsets (section 3.2), first pass: fan-out total of every 256-node
// block of the tile [a, a+count).
__global__ void __launch_bounds__(kWalkThreads)
ls_block_sums_kernel(const uint8_t *sig, uint32_t a, uint32_t count, uint32_t *sums)
{
    const uint32_t wid = blockIdx.x * (kWalkThreads / 32) + (threadIdx.x >> 5);
    const uint32_t s = a + 256u * wid;
    if (s >= a + count) return;
    const uint32_t e = min(s + 256u, a + count);
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t t0 = s + 8u * lane;
    uint32_t v = t0 < e ? (uint32_t)__popc(load8(sig, t0, e)) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) sums[wid] = v;
}

// Second pass: exclusive prefix sums of the block totals, one thread block.
__global__ void __launch_bounds__(1024) ls_scan_kernel(const uint32_t *sums, uint32_t nblocks, uint32_t *prefix)
{
    __shared__ uint32_t wsum[32];
    const uint32_t tid = threadIdx.x, lane = tid & 31u, warp = tid >> 5;
    const uint32_t per = (nblocks + blockDim.x - 1) / blockDim.x;
    const uint32_t i0 = min(tid * per, nblocks), i1 = min(i0 + per, nblocks);
    uint32_t tot = 0;
    for (uint32_t i = i0; i < i1; ++i) tot += sums[i];
    uint32_t incl = warp_incl_scan(tot);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = lane < (blockDim.x >> 5) ? wsum[lane] : 0u;
        uint32_t vi = warp_incl_scan(v);
        wsum[lane] = vi - v;
    }
    __syncthreads();
    uint32_t run = wsum[warp] + incl - tot;
    for (uint32_t i = i0; i < i1; ++i) { prefix[i] = run; run += sums[i]; }
    // prefix[nblocks] = the tile's total (every thread whose run ends there
    // holds the same value)
    if (i1 == nblocks) prefix[nblocks] = run;
}

// Multi-source search, one level: new = y & ~visited (bits of the batch);
// visited |= new; frontier = new; dist[v][b] = level for every new bit b;
// the number of vertices with a new bit is added to *count.
__global__ void __launch_bounds__(256) msbfs_mark_kernel(const uint32_t *y, uint32_t *visited, uint32_t *frontier,
                                                         int32_t *dist, uint64_t n, uint32_t B, uint32_t mask,
                                                         int32_t level, unsigned long long *count)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    uint32_t found = 0;
    for (uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += stride) {
        const uint32_t nw = y[v] & ~visited[v] & mask;
        frontier[v] = nw;
        if (nw) {
            visited[v] |= nw;
            ++found;
            uint32_t rest = nw;
            while (rest) {
                const uint32_t b = (uint32_t)(__ffs(rest) - 1);
                rest &= rest - 1u;
                dist[v * B + b] = level;
            }
        }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) found += __shfl_xor_sync(0xffffffffu, found, o);
    if ((threadIdx.x & 31u) == 0 && found) atomicAdd(count, (unsigned long long)found);
}

// Level 0: dist = -1 everywhere, visited = frontier = the sources' bits.
__global__ void __launch_bounds__(256) msbfs_init_kernel(uint32_t *visited, uint32_t *frontier, int32_t *dist,
                                                         uint64_t n, uint32_t B)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n * B; i += stride) dist[i] = -1;
    for (uint64_t v = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; v < n; v += stride) {
        visited[v] = 0u;
        frontier[v] = 0u;
    }
}

__global__ void msbfs_seed_kernel(const uint32_t *src, uint32_t B, uint32_t *visited, uint32_t *frontier,
                                  int32_t *dist)
{
    // one thread seeds all sources in order (B <= 32), so repeated sources are safe
    if (threadIdx.x != 0 || blockIdx.x != 0) return;
    for (uint32_t b = 0; b < B; ++b) {
        const uint32_t s = src[b];
        visited[s] |= 1u << b;
        frontier[s] |= 1u << b;
        dist[(uint64_t)s * B + b] = 0;
    }
}

void device_release(k2t_tree *t)
{
    DeviceState *d = t->dev;
    if (!d) return;
    if (d->gexec) cudaGraphExecDestroy(d->gexec);
    if (d->graph) cudaGraphDestroy(d->graph);
    if (d->cap_stream) cudaStreamDestroy(d->cap_stream);
    if (d->owned && d->arena) cudaFree(d->arena);
    delete d;
    t->dev = nullptr;
}


namespace {

// Map a status word to a status code: bit 0 a wait that ran out, any other
// bit a failed device-side check.
int status_code(uint32_t w)
{
    if (!w) return K2T_OK;
    return (w & K2T_STATUS_WAIT_TIMEOUT) ? K2T_ETIMEOUT : K2T_EDEVICE;
}

// Wait for `st`, then read the tree's status word (with the work queued
// before it) and map it.
int read_status(const DeviceState *d, cudaStream_t st)
{
    uint32_t w = 0;
    K2T_CUDA(cudaMemcpyAsync(&w, d->err, sizeof(w), cudaMemcpyDeviceToHost, st));
    K2T_CUDA(cudaStreamSynchronize(st));
    return status_code(w);
}

LaunchFn pick(uint32_t engine, int semiring, int dir, int vw)
{
    if (semiring == K2T_PLUS_TIMES) return pick_plus_times(engine, dir, vw);
    if (semiring == K2T_BOOLEAN) return pick_boolean(engine, dir, vw);
    return pick_min_plus(engine, dir, vw);
}

// Queue a whole product (fill + engine) on `st`.
int enqueue_product(k2t_tree *t, int32_t dir, int32_t semiring, float w, const void *x, void *y, uint32_t B,
                    cudaStream_t st, cudaEvent_t marker)
{
    DeviceState *d = t->dev;
    const uint64_t n_out = dir == K2T_RIGHT ? t->n_rows : t->n_cols;
    const uint64_t words = semiring == K2T_BOOLEAN ? n_out : n_out * (uint64_t)B;
    const uint32_t pattern = semiring == K2T_MIN_PLUS ? 0x7f800000u : 0u;
    if (words) {
        uint64_t blocks = (words / 4 + 255) / 256 + 1;
        if (blocks > 152ull * 16) blocks = 152ull * 16;
        fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<uint32_t *>(y), words, pattern);
    }
    if (marker) cudaEventRecord(marker, st);
    if (t->empty) return K2T_OK;
    int vw = 1;
    if (semiring != K2T_BOOLEAN) {
        uintptr_t al = (uintptr_t)x | (uintptr_t)y;
        if (B % 4 == 0 && (al & 15u) == 0) vw = 4;
        else if (B % 2 == 0 && (al & 7u) == 0) vw = 2;
    }
    VecArgs va;
    va.x = x;
    va.y = y;
    va.B = B;
    va.w = w;
    va.mask = B >= 32 ? 0xffffffffu : ((1u << B) - 1u);
    va.n_out = n_out;
    va.n_in = dir == K2T_RIGHT ? t->n_cols : t->n_rows;
    va.status = d->err;
    const bool heavy = heavy_begin(t, d, dir, semiring, va, st);
    uint32_t engine = t->engine;
    if (engine == K2T_ENGINE_CACHED && t->leaf_k4) engine = kEngineCached4;
    pick(engine, semiring, dir, vw)(t, d, va, st);
    if (heavy) heavy_end(t, d, dir, va, st);
    return K2T_OK;
}

}  // namespace
}  // namespace k2t

using namespace k2t;

extern "C" {

int k2t_upload(k2t_tree *t, void *arena, uint64_t arena_bytes, void *stream)
{
    if (!t) return K2T_EINVAL;
    if (t->dev) return K2T_ESTATE;
    if (arena && ((uintptr_t)arena % kArenaAlign)) return K2T_EINVAL;
    const ArenaLayout &L = t->layout;
    if (arena && arena_bytes < L.total) return K2T_ENOMEM;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceState *d = new (std::nothrow) DeviceState;
    if (!d) return K2T_ENOMEM;
    cudaGetDevice(&d->device);
    if (!arena) {
        cudaError_t e = cudaMalloc(&d->arena, L.total ? L.total : kArenaAlign);
        if (e != cudaSuccess) { g_last_cuda = (int)e; delete d; return K2T_ENOMEM; }
        d->owned = true;
    } else {
        d->arena = arena;
    }
    t->dev = d;
    auto fail = [&](cudaError_t e) { g_last_cuda = (int)e; device_release(t); return K2T_ECUDA; };
    cudaError_t e = cudaMemsetAsync(d->arena, 0, L.total, st);
    if (e != cudaSuccess) return fail(e);
    const int l = t->levels;
    d->tree.levels = l;
    d->tree.d0 = t->d0;
    d->err = at<uint32_t>(d->arena, L.err_off);
    for (int lv = 0; lv < l; ++lv) {
        d->tree.lv[lv].n = (uint32_t)t->nodes[(size_t)lv];
        if (L.sig_bytes[lv]) {
            uint8_t *p = at<uint8_t>(d->arena, L.sig_off[lv]);
            d->tree.lv[lv].sig = p;
            uint64_t bytes = level_is_k4(t, lv) ? 2 * t->nodes[(size_t)lv] : (t->nodes[(size_t)lv] + 1) / 2;
            if (bytes && (e = cudaMemcpyAsync(p, t->sig[(size_t)lv].data(), bytes, cudaMemcpyHostToDevice, st)) != cudaSuccess)
                return fail(e);
        }
        if (L.dir_bytes[lv]) {
            uint32_t *p = at<uint32_t>(d->arena, L.dir_off[lv]);
            d->tree.lv[lv].dir = p;
            if ((e = cudaMemcpyAsync(p, t->dir[(size_t)(lv - t->d0)].data(), L.dir_bytes[lv], cudaMemcpyHostToDevice, st)) != cudaSuccess)
                return fail(e);
        }
        if (L.buf_off[lv]) d->buf[lv] = at<Coord>(d->arena, L.buf_off[lv]);
    }
    auto put = [&](uint64_t off, uint64_t bytes, const void *src) -> cudaError_t {
        if (!bytes) return cudaSuccess;
        return cudaMemcpyAsync(at<char>(d->arena, off), src, bytes, cudaMemcpyHostToDevice, st);
    };
    if (L.top_bytes) { d->top = at<Coord>(d->arena, L.top_off); if ((e = put(L.top_off, L.top_bytes, t->top.data()))) return fail(e); }
    if (L.cached_bytes) { d->cached = at<Coord>(d->arena, L.cached_off); if ((e = put(L.cached_off, t->cached.size() * sizeof(Coord), t->cached.data()))) return fail(e); }
    if (L.bleaf_bytes) { d->bleaf = at<uint32_t>(d->arena, L.bleaf_off); if ((e = put(L.bleaf_off, t->bleaf.size() * 4, t->bleaf.data()))) return fail(e); }
    if (L.bsig_bytes) { d->bsig = at<uint8_t>(d->arena, L.bsig_off); if ((e = put(L.bsig_off, (t->nodes[(size_t)t->levels - 2] + 1) / 2, t->bsig.data()))) return fail(e); }
    if (L.bchunk_bytes) { d->bchunks = at<uint32_t>(d->arena, L.bchunk_off); if ((e = put(L.bchunk_off, L.bchunk_bytes, t->bchunks.data()))) return fail(e); }
    if (L.chunk_bytes) { d->chunks = at<uint32_t>(d->arena, L.chunk_off); if ((e = put(L.chunk_off, L.chunk_bytes, t->chunks.data()))) return fail(e); }
    if (L.root_bytes) { d->roots = at<Coord>(d->arena, L.root_off); if ((e = put(L.root_off, L.root_bytes, t->roots.data()))) return fail(e); }
    if (L.scan_bytes) {
        d->scan_sums = at<uint32_t>(d->arena, L.scan_off);
        d->scan_prefix = d->scan_sums + L.scan_bytes / 8;
    }
    if (L.vec_bytes) { d->vec[0] = at<void>(d->arena, L.vec_off[0]); d->vec[1] = at<void>(d->arena, L.vec_off[1]); }
    for (int dd = 0; dd < 2; ++dd) {
        if (!L.hdir_bytes[dd]) continue;
        d->hdir[dd] = at<uint32_t>(d->arena, L.hdir_off[dd]);
        d->hlist[dd] = at<uint32_t>(d->arena, L.hlist_off[dd]);
        if ((e = put(L.hdir_off[dd], L.hdir_bytes[dd], t->hdir[dd].data()))) return fail(e);
        if ((e = put(L.hlist_off[dd], L.hlist_bytes[dd], t->hlist[dd].data()))) return fail(e);
    }
    if (L.acc_bytes) d->acc = at<float>(d->arena, L.acc_off);
    if ((e = cudaStreamSynchronize(st)) != cudaSuccess) return fail(e);
    return K2T_OK;
}

int k2t_spmv_marked(k2t_tree *t, int32_t dir, int32_t semiring, float w, const void *x, void *y, uint32_t B,
                    void *stream, void *event_after_fill)
{
    if (!t) return K2T_EINVAL;
    if (!t->dev) return K2T_ESTATE;
    if (dir != K2T_RIGHT && dir != K2T_LEFT) return K2T_EINVAL;
    if (semiring < K2T_PLUS_TIMES || semiring > K2T_MIN_PLUS) return K2T_EINVAL;
    if (!x || !y || B == 0) return K2T_EINVAL;
    if (B > K2T_MAX_BATCH) return K2T_ERANGE;
    if (semiring == K2T_PLUS_TIMES && t->dev->hdir[dir] && B > t->opts.max_batch) return K2T_ERANGE;
    if (((uintptr_t)x | (uintptr_t)y) & 3u) return K2T_EINVAL;
    const uint64_t n_in = dir == K2T_RIGHT ? t->n_cols : t->n_rows;
    const uint64_t n_out = dir == K2T_RIGHT ? t->n_rows : t->n_cols;
    const uint64_t esz = semiring == K2T_BOOLEAN ? 4u : 4u * (uint64_t)B;
    uintptr_t xa = (uintptr_t)x, ya = (uintptr_t)y;
    if (xa < ya + n_out * esz && ya < xa + n_in * esz) return K2T_EINVAL;
    int cur = -1;
    K2T_CUDA(cudaGetDevice(&cur));
    if (cur != t->dev->device) return K2T_ESTATE;   // the tree's arena lives on its own device
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceState *d = t->dev;
    const bool graph = t->engine == K2T_ENGINE_LEVELSYNC && t->opts.use_graph && !t->empty;
    if (!graph) {
        int rc = enqueue_product(t, dir, semiring, w, x, y, B, st, static_cast<cudaEvent_t>(event_after_fill));
        if (rc) return rc;
        K2T_CUDA(cudaGetLastError());
        return K2T_OK;
    }
    uint32_t wb;
    std::memcpy(&wb, &w, 4);
    GraphKey k;
    k.dir = dir; k.semiring = semiring; k.wbits = wb; k.B = B; k.x = x; k.y = y;
    const GraphKey &o = d->key;
    bool same = d->gexec && o.dir == k.dir && o.semiring == k.semiring && o.wbits == k.wbits && o.B == k.B &&
                o.x == k.x && o.y == k.y;
    if (!same) {
        if (d->gexec) { cudaGraphExecDestroy(d->gexec); d->gexec = nullptr; }
        if (d->graph) { cudaGraphDestroy(d->graph); d->graph = nullptr; }
        if (!d->cap_stream) K2T_CUDA(cudaStreamCreateWithFlags(&d->cap_stream, cudaStreamNonBlocking));
        K2T_CUDA(cudaStreamBeginCapture(d->cap_stream, cudaStreamCaptureModeThreadLocal));
        enqueue_product(t, dir, semiring, w, x, y, B, d->cap_stream, nullptr);
        cudaError_t e = cudaStreamEndCapture(d->cap_stream, &d->graph);
        if (e != cudaSuccess) { g_last_cuda = (int)e; d->graph = nullptr; return K2T_ECUDA; }
        K2T_CUDA(cudaGraphInstantiate(&d->gexec, d->graph, 0));
        d->key = k;
    }
    if (event_after_fill) K2T_CUDA(cudaEventRecord(static_cast<cudaEvent_t>(event_after_fill), st));
    K2T_CUDA(cudaGraphLaunch(d->gexec, st));
    return K2T_OK;
}

int k2t_spmv(k2t_tree *t, int32_t dir, int32_t semiring, float w, const void *x, void *y, uint32_t B, void *stream)
{
    return k2t_spmv_marked(t, dir, semiring, w, x, y, B, stream, nullptr);
}

int k2t_spmv_host(k2t_tree *t, int32_t dir, int32_t semiring, float w, const void *x_host, void *y_host, uint32_t B,
                  void *stream)
{
    if (!t || !x_host || !y_host || B == 0) return K2T_EINVAL;
    if (!t->dev) return K2T_ESTATE;
    if (!t->opts.host_vectors || !t->dev->vec[0]) return K2T_ESTATE;
    if (B > t->opts.max_batch) return K2T_ERANGE;
    const uint64_t n_in = dir == K2T_RIGHT ? t->n_cols : t->n_rows;
    const uint64_t n_out = dir == K2T_RIGHT ? t->n_rows : t->n_cols;
    const uint64_t esz = semiring == K2T_BOOLEAN ? 4u : 4u * (uint64_t)B;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    DeviceState *d = t->dev;
    K2T_CUDA(cudaMemcpyAsync(d->vec[0], x_host, n_in * esz, cudaMemcpyHostToDevice, st));
    int rc = k2t_spmv(t, dir, semiring, w, d->vec[0], d->vec[1], B, stream);
    if (rc) return rc;
    K2T_CUDA(cudaMemcpyAsync(y_host, d->vec[1], n_out * esz, cudaMemcpyDeviceToHost, st));
    return read_status(d, st);
}

uint64_t k2t_msbfs_work_bytes(const k2t_tree *t)
{
    if (!t) return 0;
    const uint64_t n = std::max(t->n_rows, t->n_cols);
    return align_up(3 * n * 4 + 32 * 4 + 16, kArenaAlign);  // frontier, visited, y, sources, counter
}

int k2t_msbfs(k2t_tree *t, int32_t dir, const uint32_t *sources, uint32_t B, int32_t *dist, void *work,
              uint32_t max_levels, uint32_t *levels, void *stream)
{
    if (!t || !sources || !dist || !work || !levels) return K2T_EINVAL;
    if (!t->dev) return K2T_ESTATE;
    if (t->n_rows != t->n_cols) return K2T_EINVAL;
    if (dir != K2T_RIGHT && dir != K2T_LEFT) return K2T_EINVAL;
    if (B == 0 || B > 32) return K2T_ERANGE;
    const uint64_t n = t->n_rows;
    for (uint32_t b = 0; b < B; ++b)
        if (sources[b] >= n) return K2T_ERANGE;
    if ((uintptr_t)work & 15u) return K2T_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t *frontier = static_cast<uint32_t *>(work);
    uint32_t *visited = frontier + n;
    uint32_t *y = visited + n;
    uint32_t *src = y + n;
    unsigned long long *count = reinterpret_cast<unsigned long long *>(
        static_cast<char *>(work) + align_up(3 * n * 4 + 32 * 4, 8));
    const uint32_t mask = B >= 32 ? 0xffffffffu : ((1u << B) - 1u);
    const unsigned grid = (unsigned)std::min<uint64_t>((n * B + 255) / 256 + 1, 152ull * 16);
    msbfs_init_kernel<<<grid, 256, 0, st>>>(visited, frontier, dist, n, B);
    K2T_CUDA(cudaMemcpyAsync(src, sources, B * sizeof(uint32_t), cudaMemcpyHostToDevice, st));
    msbfs_seed_kernel<<<1, 32, 0, st>>>(src, B, visited, frontier, dist);
    K2T_CUDA(cudaGetLastError());
    uint32_t lv = 0;
    unsigned long long found = 0;
    for (uint32_t level = 1; level <= max_levels; ++level) {
        int rc = k2t_spmv(t, dir, K2T_BOOLEAN, 1.0f, frontier, y, B, stream);
        if (rc) return rc;
        K2T_CUDA(cudaMemsetAsync(count, 0, sizeof(unsigned long long), st));
        msbfs_mark_kernel<<<grid, 256, 0, st>>>(y, visited, frontier, dist, n, B, mask, (int32_t)level, count);
        K2T_CUDA(cudaMemcpyAsync(&found, count, sizeof(found), cudaMemcpyDeviceToHost, st));
        if ((rc = read_status(t->dev, st))) return rc;
        lv = level;
        if (!found) break;
    }
    *levels = lv;
    return K2T_OK;
}

int k2t_status(k2t_tree *t, uint32_t *word, int32_t clear, void *stream)
{
    if (!t || !word) return K2T_EINVAL;
    if (!t->dev) return K2T_ESTATE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t w = 0;
    K2T_CUDA(cudaMemcpyAsync(&w, t->dev->err, sizeof(w), cudaMemcpyDeviceToHost, st));
    if (clear) K2T_CUDA(cudaMemsetAsync(t->dev->err, 0, sizeof(w), st));
    K2T_CUDA(cudaStreamSynchronize(st));
    *word = w;
    return K2T_OK;
}

int k2t_device_level(const k2t_tree *t, uint32_t level, const void **sig, const void **dir)
{
    if (!t || !sig || !dir || level >= (uint32_t)t->levels) return K2T_EINVAL;
    if (!t->dev) return K2T_ESTATE;
    *sig = t->dev->tree.lv[level].sig;
    *dir = t->dev->tree.lv[level].dir;
    return K2T_OK;
}

int k2t_last_cuda_error(void) { return g_last_cuda; }

}  // extern "C"
