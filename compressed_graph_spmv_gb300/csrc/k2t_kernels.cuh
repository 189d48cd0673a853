// k2t_kernels.cuh -- device structures, semiring arithmetic and the kernels
// templated on (semiring, direction, vector width), shared by k2t_device.cu
// and the per-semiring instantiation files.
#pragma once
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <new>

#include "k2t_internal.h"

namespace k2t {

struct DevLevel {
    const uint8_t *sig;   // nibble t at byte t/2, low nibble first
    const uint32_t *dir;  // directory samples (or null)
    uint32_t n;           // nodes
    uint32_t pad;
};

struct DevTree {
    DevLevel lv[K2T_MAX_LEVELS];
    int32_t levels;
    int32_t d0;
};

struct VecArgs {
    const void *x;
    void *y;
    uint32_t B;
    float w;
    uint32_t mask;  // Boolean: bits of the batch
};

__device__ __forceinline__ uint32_t nibble_at(const uint8_t *sig, uint32_t t)
{
    return (uint32_t)(__ldg(sig + (t >> 1)) >> ((t & 1u) * 4u)) & 15u;
}

// ---- semiring arithmetic ------------------------------------------------
// Total order of IEEE floats without NaN, -0 < +0, as a signed key.
__device__ __forceinline__ int32_t order_key(float v)
{
    uint32_t u = __float_as_uint(v);
    return (int32_t)(u ^ ((uint32_t)((int32_t)u >> 31) & 0x7fffffffu));
}

// min in that order, applied atomically: a value with the sign bit clear is
// smaller than the stored value exactly when its bits are smaller as a signed
// integer; a value with the sign bit set is smaller exactly when its bits are
// larger as an unsigned integer.  Each of the two atomics is therefore a
// correct min for any stored float, so concurrent updates commute.
__device__ __forceinline__ void atomic_min_total(float *p, float v)
{
    uint32_t u = __float_as_uint(v);
    if (u & 0x80000000u) atomicMax(reinterpret_cast<unsigned int *>(p), u);
    else atomicMin(reinterpret_cast<int *>(p), (int)u);
}

template <int SR> struct Fp32Sem;

template <> struct Fp32Sem<K2T_PLUS_TIMES> {
    static __device__ __forceinline__ float zero() { return 0.0f; }
    static __device__ __forceinline__ float contrib(float x, float w) { return w * x; }
    static __device__ __forceinline__ float plus(float a, float b) { return a + b; }
    static __device__ __forceinline__ bool skip(float) { return false; }
    static __device__ __forceinline__ void update(float *y, const float (&v)[1]) { atomicAdd(y, v[0]); }
    static __device__ __forceinline__ void update(float *y, const float (&v)[2])
    {
        atomicAdd(reinterpret_cast<float2 *>(y), make_float2(v[0], v[1]));
    }
    static __device__ __forceinline__ void update(float *y, const float (&v)[4])
    {
        atomicAdd(reinterpret_cast<float4 *>(y), make_float4(v[0], v[1], v[2], v[3]));
    }
};

template <> struct Fp32Sem<K2T_MIN_PLUS> {
    static __device__ __forceinline__ float zero() { return __uint_as_float(0x7f800000u); }
    static __device__ __forceinline__ float contrib(float x, float w) { return __fadd_rn(w, x); }
    static __device__ __forceinline__ float plus(float a, float b) { return order_key(b) < order_key(a) ? b : a; }
    // +inf never lowers a minimum that starts at +inf
    static __device__ __forceinline__ bool skip(float v) { return __float_as_uint(v) == 0x7f800000u; }
    template <int VW> static __device__ __forceinline__ void update(float *y, const float (&v)[VW])
    {
#pragma unroll
        for (int k = 0; k < VW; ++k)
            if (!skip(v[k])) atomic_min_total(y + k, v[k]);
    }
};

template <int VW> struct VecLoad;
template <> struct VecLoad<1> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[1]) { v[0] = __ldg(p); }
};
template <> struct VecLoad<2> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[2])
    {
        float2 t = __ldg(reinterpret_cast<const float2 *>(p));
        v[0] = t.x; v[1] = t.y;
    }
};
template <> struct VecLoad<4> {
    static __device__ __forceinline__ void load(const float *p, float (&v)[4])
    {
        float4 t = __ldg(reinterpret_cast<const float4 *>(p));
        v[0] = t.x; v[1] = t.y; v[2] = t.z; v[3] = t.w;
    }
};

// Cells of one leaf (a 2x2 block with origin (r, c), set cells in `lam`, bit
// 2*dr + dc).  The (up to) two cells that share an output are combined with
// the semiring's addition before the atomic, so a leaf issues at most two
// atomics per vector slice.
//   right: output r gets bits 0 (input c) and 1 (input c+1); output r+1 bits 2, 3
//   left:  output c gets bits 0 (input r) and 2 (input r+1); output c+1 bits 1, 3
template <int SR, int DIR, int VW>
__device__ __forceinline__ void leaf_cells(uint32_t lam, uint32_t r, uint32_t c, const VecArgs &a)
{
    const uint32_t in = DIR == K2T_RIGHT ? c : r;
    const uint32_t out = DIR == K2T_RIGHT ? r : c;
    const bool a0 = lam & 1u;
    const bool a1 = DIR == K2T_RIGHT ? (lam & 2u) : (lam & 4u);
    const bool b0 = DIR == K2T_RIGHT ? (lam & 4u) : (lam & 2u);
    const bool b1 = lam & 8u;
    if constexpr (SR == K2T_BOOLEAN) {
        const uint32_t *x = static_cast<const uint32_t *>(a.x);
        uint32_t *y = static_cast<uint32_t *>(a.y);
        uint32_t x0 = (a0 || b0) ? __ldg(x + in) : 0u;
        uint32_t x1 = (a1 || b1) ? __ldg(x + in + 1) : 0u;
        uint32_t v0 = ((a0 ? x0 : 0u) | (a1 ? x1 : 0u)) & a.mask;
        uint32_t v1 = ((b0 ? x0 : 0u) | (b1 ? x1 : 0u)) & a.mask;
        if (v0) atomicOr(y + out, v0);
        if (v1) atomicOr(y + out + 1, v1);
    } else {
        using S = Fp32Sem<SR>;
        const float *x = static_cast<const float *>(a.x);
        float *y = static_cast<float *>(a.y);
        const size_t B = a.B;
        const bool need0 = a0 || b0, need1 = a1 || b1;
        for (uint32_t k = 0; k < a.B; k += VW) {
            float x0[VW], x1[VW], v0[VW], v1[VW];
            if (need0) VecLoad<VW>::load(x + (size_t)in * B + k, x0);
            if (need1) VecLoad<VW>::load(x + (size_t)(in + 1) * B + k, x1);
#pragma unroll
            for (int q = 0; q < VW; ++q) {
                float c0 = need0 ? S::contrib(x0[q], a.w) : S::zero();
                float c1 = need1 ? S::contrib(x1[q], a.w) : S::zero();
                v0[q] = a0 ? (a1 ? S::plus(c0, c1) : c0) : c1;
                v1[q] = b0 ? (b1 ? S::plus(c0, c1) : c0) : c1;
            }
            if (a0 || a1) S::update(y + (size_t)out * B + k, v0);
            if (b0 || b1) S::update(y + (size_t)(out + 1) * B + k, v1);
        }
    }
}

// A node of the last internal level (block side 4, coordinates rc) with
// signature s: its f = popcount(s) leaves sit at positions off .. off+f-1 of
// the leaf level (Algorithm 1, lines 13-18).
template <int SR, int DIR, int VW>
__device__ __forceinline__ void visit_node(Coord rc, uint32_t s, uint32_t off, const uint8_t *leaf, const VecArgs &a)
{
    uint32_t j = off;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
        if (s & (1u << b)) {
            uint32_t lam = nibble_at(leaf, j);
            ++j;
            leaf_cells<SR, DIR, VW>(lam, 4u * rc.r + 2u * (uint32_t)(b >> 1), 4u * rc.c + 2u * (uint32_t)(b & 1), a);
        }
    }
}

__device__ __forceinline__ Coord child_of(Coord p, int b)
{
    return Coord{2u * p.r + (uint32_t)(b >> 1), 2u * p.c + (uint32_t)(b & 1)};
}

__device__ __forceinline__ uint32_t warp_incl_scan(uint32_t v)
{
    const uint32_t lane = threadIdx.x & 31u;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t t = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= (uint32_t)o) v += t;
    }
    return v;
}

}  // namespace k2t

namespace k2t {

// ---- kernels --------------------------------------------------------------
constexpr int kWalkThreads = 256;   // 8 warps, one 256-node block each
constexpr int kFusedThreads = 256;
constexpr int kFusedWarps = kFusedThreads / 32;

// Kernels without template parameters, defined in k2t_device.cu.
__global__ void fill_kernel(uint32_t *y, uint64_t words, uint32_t pattern);
__global__ void ls_expand_kernel(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix, uint32_t a,
                                 uint32_t count, const Coord *src, uint32_t src_base, Coord *dst, uint32_t dst_base);
__global__ void ls_block_sums_kernel(const uint8_t *sig, uint32_t a, uint32_t count, uint32_t *sums);
__global__ void ls_scan_kernel(const uint32_t *sums, uint32_t nblocks, uint32_t *prefix);

// Fan-outs of up to 8 consecutive nodes t0..t0+7 (those < e), packed as
// nibbles of one word.
__device__ __forceinline__ uint32_t load8(const uint8_t *sig, uint32_t t0, uint32_t e)
{
    uint32_t w = 0;
    if (t0 + 8 <= e && (t0 & 7u) == 0) {
        w = __ldg(reinterpret_cast<const uint32_t *>(sig + (t0 >> 1)));
    } else {
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k)
            if (t0 + k < e) w |= nibble_at(sig, t0 + k) << (4 * k);
    }
    return w;
}

// Set bits of the signatures of nodes [g, s) of one level, g <= s < g + 256,
// summed over the warp (all lanes get the total).
__device__ __forceinline__ uint32_t warp_popc_range(const uint8_t *sig, uint32_t g, uint32_t s)
{
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t t0 = g + 8u * lane;
    uint32_t v = t0 < s ? (uint32_t)__popc(load8(sig, t0, s)) : 0u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// One warp walks the consecutive nodes [s, e) (e - s <= 256) of a level:
// lane l takes nodes s + 8l .. s + 8l + 7; `base` is the first child of node
// s.  fn(t, sig_t, first_child_t) runs for every node, in order per lane.
template <class F>
__device__ __forceinline__ void warp_walk(const uint8_t *sig, uint32_t s, uint32_t e, uint32_t base, F &&fn)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t t0 = s + 8u * lane;
    const uint32_t w = t0 < e ? load8(sig, t0, e) : 0u;
    const uint32_t f = (uint32_t)__popc(w);
    uint32_t pos = base + warp_incl_scan(f) - f;
#pragma unroll
    for (uint32_t k = 0; k < 8; ++k) {
        if (t0 + k < e) {
            uint32_t sg = (w >> (4 * k)) & 15u;
            fn(t0 + k, sg, pos);
            pos += (uint32_t)__popc(sg);
        }
    }
}

// Range [s, e) and first-child base of the block a warp handles inside the
// tile of nodes [a, a + count) of a level.  Directory mode: blocks aligned to
// the directory's 256-node samples (the first may start mid-block).  Scan
// mode: blocks of 256 counted from a, with prefix[j] the fan-outs of the tile
// before block j and dst_base the first child of node a.
__device__ __forceinline__ bool tile_block(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix,
                                           uint32_t a, uint32_t count, uint32_t dst_base, uint32_t wid,
                                           uint32_t &s, uint32_t &e, uint32_t &base)
{
    const uint32_t end = a + count;
    if (prefix) {
        s = a + 256u * wid;
        if (s >= end) return false;
        e = min(s + 256u, end);
        base = dst_base + prefix[wid];
        return true;
    }
    const uint32_t g = a / kDirS + wid;
    const uint32_t gs = g * kDirS;
    if (gs >= end) return false;
    s = max(gs, a);
    e = min(gs + kDirS, end);
    base = __ldg(dir + g);
    if (s > gs) base += warp_popc_range(sig, gs, s);
    return true;
}

// Algorithm 1, lines 12-20, for one tile of the last internal level.
template <int SR, int DIR, int VW>
__global__ void __launch_bounds__(kWalkThreads)
ls_leaf_kernel(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix, uint32_t a, uint32_t count,
               const Coord *src, uint32_t src_base, uint32_t leaf_base, const uint8_t *leaf, VecArgs va)
{
    const uint32_t wid = blockIdx.x * (kWalkThreads / 32) + (threadIdx.x >> 5);
    uint32_t s, e, base;
    if (!tile_block(sig, dir, prefix, a, count, leaf_base, wid, s, e, base)) return;
    warp_walk(sig, s, e, base, [&](uint32_t t, uint32_t sg, uint32_t pos) {
        visit_node<SR, DIR, VW>(src[t - src_base], sg, pos, leaf, va);
    });
}

// k^2+F (section 3.5): every node of the last internal level takes its
// coordinates from the cache and its first leaf from the directory.
template <int SR, int DIR, int VW>
__global__ void __launch_bounds__(kWalkThreads)
cached_leaf_kernel(const uint8_t *sig, const uint32_t *dir, uint32_t n, const Coord *coords,
                   const uint8_t *leaf, VecArgs va)
{
    const uint32_t g = blockIdx.x * (kWalkThreads / 32) + (threadIdx.x >> 5);
    const uint32_t s = g * kDirS;
    if (s >= n) return;
    const uint32_t e = min(s + kDirS, n);
    warp_walk(sig, s, e, __ldg(dir + g), [&](uint32_t t, uint32_t sg, uint32_t pos) {
        visit_node<SR, DIR, VW>(coords[t], sg, pos, leaf, va);
    });
}

// Exclusive block-wide prefix sum over kFusedThreads threads.
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *wsum)
{
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t incl = warp_incl_scan(v);
    if (lane == 31) wsum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t t = lane < (uint32_t)kFusedWarps ? wsum[lane] : 0u;
        uint32_t ti = warp_incl_scan(t);
        if (lane < (uint32_t)kFusedWarps) wsum[lane] = ti - t;
    }
    __syncthreads();
    const uint32_t r = wsum[warp] + incl - v;
    __syncthreads();
    return r;
}

// FUSED engine: thread block k descends chunk k, a run of whole subtrees
// rooted at level d_c, down to the leaves.  The chunk record holds the
// index of its roots' coordinates and, for every level, the first node and
// the node count of the chunk there (planned once per tree on the host).
// Each level: a thread takes a contiguous run of parents, the block scans
// the run fan-outs, and children are written to the other shared buffer.
template <int SR, int DIR, int VW>
__global__ void __launch_bounds__(kFusedThreads)
fused_kernel(DevTree tr, const uint32_t *chunks, uint32_t stride, const Coord *roots, VecArgs va)
{
    extern __shared__ Coord fsm[];
    __shared__ uint32_t wsum[kFusedWarps];
    Coord *cur = fsm;
    Coord *nxt = fsm + kMaxChunkCap;
    const uint32_t *rec = chunks + (size_t)blockIdx.x * stride;
    const uint32_t rc = rec[0];
    const int dc = (int)rec[1];
    const uint32_t *rng = rec + 2;
    const int d0 = tr.d0, l = tr.levels;
    const uint32_t tid = threadIdx.x;
    {
        const uint32_t n = rng[2 * (dc - d0) + 1];
        for (uint32_t i = tid; i < n; i += kFusedThreads) cur[i] = roots[rc + i];
    }
    __syncthreads();
    for (int d = dc; d < l - 2; ++d) {
        const uint32_t s = rng[2 * (d - d0)], n = rng[2 * (d - d0) + 1];
        const uint8_t *sig = tr.lv[d].sig;
        const uint32_t per = (n + kFusedThreads - 1) / kFusedThreads;
        const uint32_t i0 = min(tid * per, n), i1 = min(i0 + per, n);
        uint32_t tot = 0;
        for (uint32_t i = i0; i < i1; ++i) tot += (uint32_t)__popc(nibble_at(sig, s + i));
        uint32_t pos = block_excl_scan(tot, wsum);
        for (uint32_t i = i0; i < i1; ++i) {
            const uint32_t sg = nibble_at(sig, s + i);
            const Coord p = cur[i];
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (sg & (1u << b)) nxt[pos++] = child_of(p, b);
        }
        __syncthreads();
        Coord *t = cur; cur = nxt; nxt = t;
    }
    {
        const int d = l - 2;
        const uint32_t s = rng[2 * (d - d0)], n = rng[2 * (d - d0) + 1];
        const uint32_t sl = rng[2 * (d + 1 - d0)];
        const uint8_t *sig = tr.lv[d].sig;
        const uint8_t *leaf = tr.lv[l - 1].sig;
        const uint32_t per = (n + kFusedThreads - 1) / kFusedThreads;
        const uint32_t i0 = min(tid * per, n), i1 = min(i0 + per, n);
        uint32_t tot = 0;
        for (uint32_t i = i0; i < i1; ++i) tot += (uint32_t)__popc(nibble_at(sig, s + i));
        uint32_t pos = sl + block_excl_scan(tot, wsum);
        for (uint32_t i = i0; i < i1; ++i) {
            const uint32_t sg = nibble_at(sig, s + i);
            visit_node<SR, DIR, VW>(cur[i], sg, pos, leaf, va);
            pos += (uint32_t)__popc(sg);
        }
    }
}

}  // namespace k2t

namespace k2t {

extern thread_local int g_last_cuda;

#define K2T_CUDA(call)                                   \
    do {                                                 \
        cudaError_t e_ = (call);                         \
        if (e_ != cudaSuccess) {                         \
            g_last_cuda = (int)e_;                       \
            return K2T_ECUDA;                            \
        }                                                \
    } while (0)

struct GraphKey {
    int32_t dir = -1, semiring = -1;
    uint32_t wbits = 0, B = 0;
    const void *x = nullptr;
    void *y = nullptr;
};

struct DeviceState {
    void *arena = nullptr;
    bool owned = false;
    int device = 0;
    DevTree tree{};
    const Coord *top = nullptr;
    const Coord *cached = nullptr;
    const uint32_t *chunks = nullptr;
    const Coord *roots = nullptr;
    Coord *buf[K2T_MAX_LEVELS] = {};
    uint32_t *scan_sums = nullptr;
    uint32_t *scan_prefix = nullptr;
    uint32_t *err = nullptr;
    void *vec[2] = {nullptr, nullptr};
    cudaStream_t cap_stream = nullptr;
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t gexec = nullptr;
    GraphKey key;
};

template <class T> inline T *at(void *arena, uint64_t off) { return reinterpret_cast<T *>(static_cast<char *>(arena) + off); }

inline int grid_for_blocks(uint64_t warps_needed)
{
    uint64_t per = kWalkThreads / 32;
    return (int)((warps_needed + per - 1) / per);
}

// ---- per-(semiring, direction, vector width) launch tables --------------
template <int SR, int DIR, int VW>
void launch_fused(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const size_t smem = 2 * kMaxChunkCap * sizeof(Coord);
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(fused_kernel<SR, DIR, VW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        configured = true;
    }
    fused_kernel<SR, DIR, VW><<<(unsigned)t->n_chunks, kFusedThreads, smem, st>>>(d->tree, d->chunks, t->chunk_stride,
                                                                                 d->roots, va);
}

template <int SR, int DIR, int VW>
void launch_cached(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const int l = t->levels;
    const uint32_t n = (uint32_t)t->nodes[(size_t)l - 2];
    const uint64_t blocks = (n + kDirS - 1) / kDirS;
    cached_leaf_kernel<SR, DIR, VW><<<grid_for_blocks(blocks), kWalkThreads, 0, st>>>(
        d->tree.lv[l - 2].sig, d->tree.lv[l - 2].dir, n, d->cached, d->tree.lv[l - 1].sig, va);
}

template <int SR, int DIR, int VW>
void launch_ls(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const bool scan = t->opts.offsets == K2T_OFFSETS_SCAN;
    const int l = t->levels;
    for (const LsStep &s : t->steps) {
        const int lv = s.level;
        const Coord *src = s.src == 0xff ? d->top : d->buf[s.src];
        const uint8_t *sig = d->tree.lv[lv].sig;
        const uint32_t *dir = d->tree.lv[lv].dir;
        const uint64_t blocks = scan ? (s.count + 255u) / 256u
                                     : ((uint64_t)s.a + s.count + kDirS - 1) / kDirS - s.a / kDirS;
        const uint32_t *prefix = nullptr;
        uint32_t base = s.dst_base;
        if (s.kind == 1) base = scan ? (uint32_t)level_offset(t, lv, s.a) : 0u;
        if (scan) {
            ls_block_sums_kernel<<<grid_for_blocks(blocks), kWalkThreads, 0, st>>>(sig, s.a, s.count, d->scan_sums);
            ls_scan_kernel<<<1, 1024, 0, st>>>(d->scan_sums, (uint32_t)blocks, d->scan_prefix);
            prefix = d->scan_prefix;
        }
        if (s.kind == 0) {
            ls_expand_kernel<<<grid_for_blocks(blocks), kWalkThreads, 0, st>>>(
                sig, dir, prefix, s.a, s.count, src, s.src_base, d->buf[lv + 1], s.dst_base);
        } else {
            ls_leaf_kernel<SR, DIR, VW><<<grid_for_blocks(blocks), kWalkThreads, 0, st>>>(
                sig, dir, prefix, s.a, s.count, src, s.src_base, base, d->tree.lv[l - 1].sig, va);
        }
    }
}

using LaunchFn = void (*)(const k2t_tree *, const DeviceState *, const VecArgs &, cudaStream_t);

template <int SR, int DIR, int VW>
LaunchFn pick_engine(uint32_t engine)
{
    switch (engine) {
    case K2T_ENGINE_FUSED: return launch_fused<SR, DIR, VW>;
    case K2T_ENGINE_CACHED: return launch_cached<SR, DIR, VW>;
    default: return launch_ls<SR, DIR, VW>;
    }
}

template <int SR, int DIR>
LaunchFn pick_vw(uint32_t engine, int vw)
{
    if constexpr (SR == K2T_BOOLEAN) {
        (void)vw;
        return pick_engine<SR, DIR, 1>(engine);
    } else {
        if (vw == 4) return pick_engine<SR, DIR, 4>(engine);
        if (vw == 2) return pick_engine<SR, DIR, 2>(engine);
        return pick_engine<SR, DIR, 1>(engine);
    }
}

// One instantiation file per semiring (k2t_sr_*.cu) defines these.
LaunchFn pick_plus_times(uint32_t engine, int dir, int vw);
LaunchFn pick_boolean(uint32_t engine, int dir, int vw);
LaunchFn pick_min_plus(uint32_t engine, int dir, int vw);

}  // namespace k2t
