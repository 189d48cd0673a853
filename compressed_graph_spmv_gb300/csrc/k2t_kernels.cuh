// k2t_kernels.cuh -- device structures, semiring arithmetic and the kernels
// templated on (semiring, direction, vector width), shared by k2t_device.cu
// and the per-semiring instantiation files.
#pragma once
#include <cuda_runtime.h>

#include <algorithm>

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
    uint32_t mask;   // Boolean: bits of the batch
    uint64_t n_out;  // entries (vertices) of y
    uint64_t n_in;   // entries (vertices) of x
    // Heavy plus-times outputs (null hdir: none in this product)
    const uint32_t *hdir;   // per output below hdir_len: its record, 0 if not heavy
    uint32_t hdir_len;
    float *acc;             // rows of B fp32 words: partial sums and fp64 slots of heavy outputs
    uint32_t *status;       // the tree's device status word (checked builds report into it)
};

// ---- checked build ---------------------------------------------------------
// Compiled with -DK2T_CHECKED (libk2t_checked.so), the kernels test the
// indexes they take from the tree and its plan against the bounds of what
// those address: outputs and inputs of every leaf against n_out and n_in,
// a chunk's level widths against the FUSED staging slots, expand positions
// against the LEVELSYNC frontier buffers.  A failed test sets
// K2T_STATUS_OUT_OF_RANGE in the status word and the access is skipped, so a
// planning or indexing fault shows up as K2T_EDEVICE instead of a memory
// fault.  In the product build the tests compile away.
#ifdef K2T_CHECKED
__device__ __forceinline__ bool in_range(bool ok, uint32_t *status)
{
    if (!ok && status) atomicOr(status, K2T_STATUS_OUT_OF_RANGE);
    return ok;
}
#define K2T_IN_RANGE(cond, status) ::k2t::in_range((cond), (status))
#else
#define K2T_IN_RANGE(cond, status) true
#endif

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

// Semiring updates of a shared-memory accumulator (one 32-bit word per entry).
__device__ __forceinline__ void smem_min_total(float *p, float v)
{
    uint32_t u = __float_as_uint(v);
    if (u & 0x80000000u) atomicMax(reinterpret_cast<unsigned int *>(p), u);
    else atomicMin(reinterpret_cast<int *>(p), (int)u);
}

template <int SR>
__device__ __forceinline__ void smem_update(uint32_t *w, uint32_t v)
{
    if constexpr (SR == K2T_PLUS_TIMES) atomicAdd(reinterpret_cast<float *>(w), __uint_as_float(v));
    else if constexpr (SR == K2T_BOOLEAN) atomicOr(w, v);
    else smem_min_total(reinterpret_cast<float *>(w), __uint_as_float(v));
}

// The same update applied once to y from a flushed accumulator word.
template <int SR>
__device__ __forceinline__ void global_update_word(uint32_t *y, uint32_t v)
{
    if constexpr (SR == K2T_PLUS_TIMES) atomicAdd(reinterpret_cast<float *>(y), __uint_as_float(v));
    else if constexpr (SR == K2T_BOOLEAN) atomicOr(y, v);
    else atomic_min_total(reinterpret_cast<float *>(y), __uint_as_float(v));
}

template <int SR>
__device__ __forceinline__ uint32_t zero_word()
{
    return SR == K2T_MIN_PLUS ? 0x7f800000u : 0u;
}

// An accumulator word that leaves y unchanged: +-0 (plus-times: y never holds
// -0), +inf (tropical), 0 (Boolean).
template <int SR>
__device__ __forceinline__ bool is_noop_word(uint32_t v)
{
    if constexpr (SR == K2T_PLUS_TIMES) return (v & 0x7fffffffu) == 0u;
    else if constexpr (SR == K2T_BOOLEAN) return v == 0u;
    else return v == 0x7f800000u;
}

// ---- heavy outputs (plus-times) ------------------------------------------------
// An output with more non-zeros than one fp32 sum can take within the bound
// is "heavy".  Its record (one word per output, built once per tree) names rows of
// the accumulator array acc (B fp32 words a row): 2^bits fp32 partial sums,
// each receiving at most heavy_terms terms; or, bits kHeavyFp64, an fp64 slot
// of two rows (B doubles), which then takes every term.  The records cover the
// outputs below hdir_len (the last heavy output, rounded up to a multiple of
// 4, plus 4): heavy_near(out) says whether a leaf with first output `out`
// may have a heavy output; heavy_word: the records of a 2x2 leaf's outputs
// out (even) and out + 1, read together (one 8-byte load), for such a leaf.
__device__ __forceinline__ uint32_t heavy_near(const VecArgs &va, uint32_t out)
{
    return out < va.hdir_len ? 1u : 0u;
}

__device__ __forceinline__ uint2 heavy_word(const VecArgs &va, uint32_t out)
{
    return __ldg(reinterpret_cast<const uint2 *>(va.hdir + out));
}

// fp64 slot (B doubles) of a heavy output summed in fp64 (bits kHeavyFp64).
__device__ __forceinline__ double *heavy_slot64(const VecArgs &va, uint32_t rec)
{
    return reinterpret_cast<double *>(va.acc + (size_t)(rec >> 5) * va.B);
}

// Where a heavy output (record rec, slice k) sums the terms of a leaf with
// first input `in`: the fp32 partial sum heavy_partial(in, bits), or (null
// p32, bits kHeavyFp64) its fp64 slot.
struct HeavyDst {
    float *p32;
    double *p64;
};

__device__ __forceinline__ HeavyDst heavy_dst(const VecArgs &va, uint32_t rec, uint32_t in, uint32_t k)
{
    const uint32_t bits = rec & 31u;
    if (bits == kHeavyFp64) return HeavyDst{nullptr, heavy_slot64(va, rec) + k};
    return HeavyDst{va.acc + ((size_t)(rec >> 5) + heavy_partial(in, bits)) * va.B + k, nullptr};
}

// Update a heavy output (record rec, slice k) with a leaf's contribution: v
// is the fp32 combination of its cells (one term of an fp32 partial sum); for
// an fp64 output the cells w*xa (when ua) and w*xb (when ub) are added in
// fp64, where the sum of two floats is exact.
template <int SR, int VW>
__device__ __forceinline__ void heavy_put(const VecArgs &va, uint32_t rec, uint32_t in, uint32_t k,
                                          const float (&v)[VW], const float (&xa)[VW], const float (&xb)[VW], bool ua,
                                          bool ub)
{
    const HeavyDst dst = heavy_dst(va, rec, in, k);
    if (dst.p32) {
        Fp32Sem<SR>::update(dst.p32, v);
        return;
    }
#pragma unroll
    for (int i = 0; i < VW; ++i)
        atomicAdd(dst.p64 + i, (ua ? (double)(va.w * xa[i]) : 0.0) + (ub ? (double)(va.w * xb[i]) : 0.0));
}

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
constexpr int kFusedThreads = 64;   // two warps: a block frees its slot once its two chunks are done
constexpr int kFusedWarps = kFusedThreads / 32;   // chunks per thread block (one per warp)

// Kernels without template parameters, defined in k2t_device.cu.
__global__ void fill_kernel(uint32_t *y, uint64_t words, uint32_t pattern);
__global__ void heavy_finish_kernel(const float *acc, const uint32_t *hdir, const uint32_t *list, uint32_t h,
                                    uint32_t B, float *y);
__global__ void ls_expand_kernel(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix, uint32_t a,
                                 uint32_t count, const Coord *src, uint32_t src_base, Coord *dst, uint32_t dst_base,
                                 uint64_t dst_entries, uint32_t *status);
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


// Leaves of U leaf blocks (origins r[u], c[u], cells lam[u]) with x entries
// already loaded (xo[u][0]: input r or c, xo[u][1]: the next one); one
// vector slice (B = 1 fp32, or a Boolean word).  hw[u] (plus-times): the
// heavy records of leaf u's outputs (heavy_word, loaded with its x entries),
// zero for outputs that are not heavy; outside a window heavy outputs go to
// their heavy sums.
template <int SR, int DIR, int U, class InOf>
__device__ __forceinline__ void leaf_apply1(const uint32_t (&lam)[U], const uint32_t (&out)[U], InOf &&in_of,
                                            const uint32_t (&xo)[U][2], const uint2 (&hw)[U], const VecArgs &va,
                                            uint32_t *win, uint32_t lo)
{
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t l = lam[u];
        if (!l) continue;
        const bool a0 = l & 1u;
        const bool a1 = DIR == K2T_RIGHT ? (l & 2u) : (l & 4u);
        const bool b0 = DIR == K2T_RIGHT ? (l & 4u) : (l & 2u);
        const bool b1 = l & 8u;
        if (!K2T_IN_RANGE(out[u] + ((b0 || b1) ? 1u : 0u) < va.n_out, va.status)) continue;
        if constexpr (SR == K2T_BOOLEAN) {
            uint32_t *y = static_cast<uint32_t *>(va.y);
            const uint32_t v0 = ((a0 ? xo[u][0] : 0u) | (a1 ? xo[u][1] : 0u)) & va.mask;
            const uint32_t v1 = ((b0 ? xo[u][0] : 0u) | (b1 ? xo[u][1] : 0u)) & va.mask;
            if (win) {
                if (v0) atomicOr(win + (out[u] - lo), v0);
                if (v1) atomicOr(win + (out[u] + 1 - lo), v1);
            } else {
                if (v0) atomicOr(y + out[u], v0);
                if (v1) atomicOr(y + out[u] + 1, v1);
            }
        } else {
            using S = Fp32Sem<SR>;
            float *y = static_cast<float *>(va.y);
            const float c0 = S::contrib(__uint_as_float(xo[u][0]), va.w);
            const float c1 = S::contrib(__uint_as_float(xo[u][1]), va.w);
            const uint2 h = hw[u];
            const float xa[1] = {__uint_as_float(xo[u][0])}, xb[1] = {__uint_as_float(xo[u][1])};
            if (a0 || a1) {
                const float v[1] = {a0 ? (a1 ? S::plus(c0, c1) : c0) : c1};
                if (h.x) heavy_put<SR, 1>(va, h.x, in_of(u), 0u, v, xa, xb, a0, a1);
                else if (!S::skip(v[0])) {
                    if (win) smem_update<SR>(win + (out[u] - lo), __float_as_uint(v[0]));
                    else S::update(y + out[u], v);
                }
            }
            if (b0 || b1) {
                const float v[1] = {b0 ? (b1 ? S::plus(c0, c1) : c0) : c1};
                if (h.y) heavy_put<SR, 1>(va, h.y, in_of(u), 0u, v, xa, xb, b0, b1);
                else if (!S::skip(v[0])) {
                    if (win) smem_update<SR>(win + (out[u] + 1 - lo), __float_as_uint(v[0]));
                    else S::update(y + out[u] + 1, v);
                }
            }
        }
    }
}

// ---- per-warp leaf stage -------------------------------------------------------
#ifndef K2T_LEAF_U
#define K2T_LEAF_U 4
#endif
#ifndef K2T_WARP_WINDOW
#define K2T_WARP_WINDOW 256
#endif
constexpr int kLeafU = K2T_LEAF_U;                  // leaves per lane per round (one vector slice)
constexpr int kBatchU = 2;                          // leaves per lane group per round (batches)
constexpr uint32_t kWarpWindow = K2T_WARP_WINDOW;   // words of a warp's output window

// Per-warp segmented scatter.  [mn, mx] bounds the warp's output coordinates
// in units of `unit` cells (4 or 8 for nodes of the last internal level with
// 2x2 or 4x4 leaves, 2 or 4 for leaves).  When the outputs fit the warp's
// window (kWarpWindow words), the window is cleared and returned; updates are
// then reduced there and each touched entry reaches y once
// (warp_window_flush).  Hub rows of power-law graphs then cost one global
// atomic per warp instead of one per non-zero.
//
// Window modes (wmode):
//   kWinF32     no heavy plus-times output among the window's outputs, so
//               leaves need no heavy lookups;
//   kWinShared  the span holds heavy outputs (or, BANDED, it may): heavy
//               outputs are routed per leaf to their partial sums and never
//               enter the window, whose sums stay within the fp32 term bound
//               of the outputs that do.
constexpr int kWinF32 = 0, kWinShared = 2;

// Heavy plus-times outputs among [lo, lo + span) (span <= kWarpWindow), over
// the warp: the lanes read the range's records (coalesced).
__device__ __forceinline__ bool warp_span_has_heavy(const VecArgs &va, uint32_t lo, uint32_t span)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t hi = (uint32_t)min((uint64_t)lo + span, (uint64_t)va.hdir_len);   // exclusive
    uint32_t any = 0u;
    for (uint32_t o = lo + lane; o < hi; o += 32u) any |= __ldg(va.hdir + o);
    return __any_sync(0xffffffffu, any != 0u);
}

template <int SR>
__device__ __forceinline__ uint32_t *warp_window_begin(uint32_t mn, uint32_t mx, uint32_t unit, uint32_t width,
                                                       uint32_t *mem, uint32_t &lo, uint32_t &span,
                                                       const VecArgs &va, int &wmode)
{
    const uint32_t lane = threadIdx.x & 31u;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    lo = unit * mn;
    span = 0;
    wmode = kWinF32;
    if (mn > mx) return nullptr;
    const uint64_t span64 = (uint64_t)unit * ((uint64_t)mx - mn + 1u);
    if (span64 * width > kWarpWindow) return nullptr;
    if (SR == K2T_PLUS_TIMES && va.hdir != nullptr && warp_span_has_heavy(va, lo, (uint32_t)span64))
        wmode = kWinShared;
    span = (uint32_t)span64;
    const uint32_t words = span * width;
    for (uint32_t i = lane; i < words; i += 32u) mem[i] = zero_word<SR>();
    __syncwarp();
    return mem;
}

template <int SR>
__device__ __forceinline__ void warp_window_flush(const uint32_t *win, uint32_t lo, uint32_t span, uint32_t width,
                                                  const VecArgs &va, int wmode)
{
    const uint32_t lane = threadIdx.x & 31u;
    __syncwarp();
    (void)wmode;
    uint32_t *y = static_cast<uint32_t *>(va.y) + (size_t)lo * width;
    const uint64_t limit = (va.n_out - lo) * width;
    for (uint32_t i = lane; i < span * width; i += 32u) {
        const uint32_t v = win[i];
        if (is_noop_word<SR>(v) || i >= limit) continue;
        global_update_word<SR>(y + i, v);
    }
}

// The VW-wide slice k of the two input rows of one leaf (origin r, c; cells
// lam) that its cells use: x0 from its first input, x1 from the next.
template <int SR, int DIR, int VW>
__device__ __forceinline__ void leaf_slice_load(uint32_t lam, uint32_t r, uint32_t c, uint32_t k, const VecArgs &va,
                                                float (&x0)[VW], float (&x1)[VW])
{
    const uint32_t in = DIR == K2T_RIGHT ? c : r;
    const bool u0 = DIR == K2T_RIGHT ? (lam & 5u) : (lam & 3u);    // cells on the first input
    const bool u1 = DIR == K2T_RIGHT ? (lam & 10u) : (lam & 12u);  // cells on the second
    const float *x = static_cast<const float *>(va.x);
    const size_t B = va.B;
    if (!K2T_IN_RANGE(in + (u1 ? 1u : 0u) < va.n_in, va.status)) return;
    if (u0) VecLoad<VW>::load(x + (size_t)in * B + k, x0);
    if (u1) VecLoad<VW>::load(x + (size_t)(in + 1) * B + k, x1);
}

// One VW-wide vector slice k of one leaf (origin r, c; cells lam) whose input
// slices x0, x1 are loaded (leaf_slice_load): combines per output, updates y
// or the window; outputs with a record in hv (heavy_word) go to their heavy
// sums.
template <int SR, int DIR, int VW>
__device__ __forceinline__ void leaf_slice(uint32_t lam, uint32_t r, uint32_t c, uint32_t k, uint2 hv,
                                           const float (&x0)[VW], const float (&x1)[VW], const VecArgs &va,
                                           uint32_t *win, uint32_t lo)
{
    using S = Fp32Sem<SR>;
    const uint32_t in = DIR == K2T_RIGHT ? c : r;
    const uint32_t out = DIR == K2T_RIGHT ? r : c;
    const bool a0 = lam & 1u;
    const bool a1 = DIR == K2T_RIGHT ? (lam & 2u) : (lam & 4u);
    const bool b0 = DIR == K2T_RIGHT ? (lam & 4u) : (lam & 2u);
    const bool b1 = lam & 8u;
    if (!K2T_IN_RANGE(out + ((b0 || b1) ? 1u : 0u) < va.n_out && in + ((a1 || b1) ? 1u : 0u) < va.n_in, va.status))
        return;
    float *y = static_cast<float *>(va.y);
    const size_t B = va.B;
    // One output's combined contribution from x0, x1 (cells u0 on input in,
    // u1 on in + 1), and its update of y or the window.
    auto combine = [&](bool u0, bool u1, float (&v)[VW]) {
#pragma unroll
        for (int q = 0; q < VW; ++q) {
            const float c0 = u0 ? S::contrib(x0[q], va.w) : S::zero();
            const float c1 = u1 ? S::contrib(x1[q], va.w) : S::zero();
            v[q] = u0 ? (u1 ? S::plus(c0, c1) : c0) : c1;
        }
    };
    auto put = [&](uint32_t o, bool u0, bool u1) {
        float v[VW];
        combine(u0, u1, v);
        if (win) {
#pragma unroll
            for (int q = 0; q < VW; ++q)
                if (!S::skip(v[q])) smem_update<SR>(win + (size_t)(o - lo) * B + k + q, __float_as_uint(v[q]));
        } else {
            S::update(y + (size_t)o * B + k, v);
        }
    };
    if (SR == K2T_PLUS_TIMES && (hv.x | hv.y)) {
        // a leaf with a heavy output: separate branch, so the fp32 path below
        // keeps its registers
        if (a0 || a1) {
            if (hv.x) {
                float v[VW];
                combine(a0, a1, v);
                heavy_put<SR, VW>(va, hv.x, in, k, v, x0, x1, a0, a1);
            } else {
                put(out, a0, a1);
            }
        }
        if (b0 || b1) {
            if (hv.y) {
                float v[VW];
                combine(b0, b1, v);
                heavy_put<SR, VW>(va, hv.y, in, k, v, x0, x1, b0, b1);
            } else {
                put(out + 1, b0, b1);
            }
        }
        return;
    }
    if (a0 || a1) put(out, a0, a1);
    if (b0 || b1) put(out + 1, b0, b1);
}

// Leaves [jb, je) of a warp.  leaf_at(j, lam, r, c, li) gives leaf j's cells,
// the origin of its 2x2 block and its index in the leaf level (for the heavy
// output flags).
//  - One vector slice (B = 1 fp32, or a Boolean word): leaves dealt round-
//    robin, kLeafU per lane per round; both input entries of a block come in
//    one 8-byte load together with the leaf signature.
//  - Batches (B > VW): G = B / VW adjacent lanes share a leaf, lane g owning
//    the VW-wide slice g of every vector row, so a row of x is one coalesced
//    load and a row of y one coalesced vector reduction (the pages' B
//    adjacent threads per node, section 3.6).
// Updates go to the window when there is one (wmode as warp_window_begin
// says), else to y; heavy plus-times outputs outside a window go to their
// partial sums.  out_min: no output of the warp's leaves is below it (0 when
// unknown); a warp whose outputs all lie past the last heavy one skips the
// heavy lookups.
template <int SR, int DIR, int VW, class LeafAt>
__device__ __forceinline__ void warp_leaf_rounds(uint32_t jb, uint32_t je, LeafAt &&leaf_at, const VecArgs &va,
                                                 uint32_t *win, uint32_t lo, int wmode, uint32_t out_min)
{
    const uint32_t lane = threadIdx.x & 31u;
    const bool heavy = SR == K2T_PLUS_TIMES && va.hdir != nullptr && out_min < va.hdir_len &&
                       (!win || wmode == kWinShared);
    if (SR == K2T_BOOLEAN || (VW == 1 && va.B == 1)) {
        constexpr int U = kLeafU;
        const uint32_t *x = static_cast<const uint32_t *>(va.x);
        const bool x8 = ((uintptr_t)x & 7u) == 0;
        for (uint32_t j0 = jb; j0 < je; j0 += 32u * U) {
            uint32_t lam[U], r[U], c[U], fl = 0u;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t j = j0 + 32u * u + lane;
                lam[u] = 0u;
                r[u] = 0u;
                c[u] = 0u;
                uint32_t li = 0u;
                if (j < je) {
                    leaf_at(j, lam[u], r[u], c[u], li);
                    if (heavy) fl |= heavy_near(va, DIR == K2T_RIGHT ? r[u] : c[u]) << u;
                }
            }
            uint32_t xo[U][2], out[U];
            uint2 hw[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t in = DIR == K2T_RIGHT ? c[u] : r[u];  // even
                out[u] = DIR == K2T_RIGHT ? r[u] : c[u];
                xo[u][0] = 0u;
                xo[u][1] = 0u;
                hw[u] = make_uint2(0u, 0u);
                if (lam[u]) {
                    if (x8 && in + 1u < va.n_in) {
                        const uint2 v = __ldg(reinterpret_cast<const uint2 *>(x + in));
                        xo[u][0] = v.x;
                        xo[u][1] = v.y;
                    } else {
                        xo[u][0] = __ldg(x + in);
                        if (in + 1u < va.n_in) xo[u][1] = __ldg(x + in + 1u);
                    }
                    if (SR == K2T_PLUS_TIMES && ((fl >> u) & 1u)) hw[u] = heavy_word(va, out[u]);
                }
            }
            // the input index of leaf u, looked up again (only leaves with a
            // heavy output outside a window need it)
            auto in_of = [&](int u) {
                uint32_t l2, r2, c2, li2;
                leaf_at(j0 + 32u * (uint32_t)u + lane, l2, r2, c2, li2);
                return DIR == K2T_RIGHT ? c2 : r2;
            };
            leaf_apply1<SR, DIR, U>(lam, out, in_of, xo, hw, va, win, lo);
        }
        return;
    }
    if constexpr (SR != K2T_BOOLEAN) {
        constexpr int U = kBatchU;
        const uint32_t G = va.B / VW;                    // lanes per leaf (B is a multiple of VW)
        const uint32_t per = G <= 32u ? 32u / G : 1u;    // leaves per lane-group round
        const uint32_t groups = G <= 32u ? G : 32u;      // lanes that own a slice per round
        const uint32_t slot = lane / groups, sub = lane % groups;
        const bool active = slot < per;
        for (uint32_t j0 = jb; j0 < je; j0 += per * U) {
            uint32_t lam[U], r[U], c[U];
            uint2 hv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t j = j0 + (uint32_t)u * per + slot;
                lam[u] = 0u;
                r[u] = 0u;
                c[u] = 0u;
                hv[u] = make_uint2(0u, 0u);
                uint32_t li = 0u;
                if (active && j < je) {
                    leaf_at(j, lam[u], r[u], c[u], li);
                    if (heavy && heavy_near(va, DIR == K2T_RIGHT ? r[u] : c[u]))
                        hv[u] = heavy_word(va, DIR == K2T_RIGHT ? r[u] : c[u]);
                }
            }
            // a group of G lanes covers the row; rows wider than 32 slices
            // loop.  Every gather of the round is issued before its updates.
            for (uint32_t k = sub * VW; k < va.B; k += groups * VW) {
                float x0[U][VW], x1[U][VW];
#pragma unroll
                for (int u = 0; u < U; ++u) leaf_slice_load<SR, DIR, VW>(lam[u], r[u], c[u], k, va, x0[u], x1[u]);
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (lam[u]) leaf_slice<SR, DIR, VW>(lam[u], r[u], c[u], k, hv[u], x0[u], x1[u], va, win, lo);
            }
        }
    }
}

// The nodes of one warp's block of the last internal level, within the tile
// [a, a + count): block g of the tile (directory mode: the 256-node block of
// the directory, clipped to the tile; scan mode, prefix != null: nodes
// a + 256 g ..., the tile's g-th block of 256).  Sets the block's first node
// blk, the tile-clipped range [s, e), the first leaf `base` of node s, and
// lane's 8 nibbles (nodes blk + 8 lane ..., those outside [s, e) cleared);
// false when the block lies past the tile.
__device__ __forceinline__ bool tile_warp_block(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix,
                                                uint32_t leaf_base, uint32_t a, uint32_t count, uint32_t g,
                                                uint32_t &blk, uint32_t &s, uint32_t &e, uint32_t &base,
                                                uint32_t &w)
{
    const uint32_t lane = threadIdx.x & 31u;
    const uint32_t end = a + count;
    if (prefix) {
        blk = a + kDirS * g;
        if (blk >= end) return false;
        s = blk;
        e = min(blk + kDirS, end);
        base = leaf_base + __ldg(prefix + g);
        const uint32_t t0 = blk + 8u * lane;
        w = t0 < e ? load8(sig, t0, e) : 0u;
        return true;
    }
    const uint32_t G = a / kDirS + g;
    blk = G * kDirS;
    if (blk >= end) return false;
    s = max(blk, a);
    e = min(blk + kDirS, end);
    const uint32_t t0 = blk + 8u * lane;
    w = 0u;
    uint32_t pre = 0u;   // fan-outs of the block's nodes before s (the tile's start)
    if (t0 < e) {
        const uint32_t word = __ldg(reinterpret_cast<const uint32_t *>(sig + blk / 2) + lane);
        const uint32_t lo = s > t0 ? min(s - t0, 8u) : 0u;          // nibbles before s
        const uint32_t hi = min(e - t0, 8u);                          // nibbles before e
        const uint32_t below_lo = lo == 8u ? 0xffffffffu : ((1u << (4u * lo)) - 1u);
        const uint32_t below_hi = hi == 8u ? 0xffffffffu : ((1u << (4u * hi)) - 1u);
        w = word & below_hi & ~below_lo;
        pre = (uint32_t)__popc(word & below_lo);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) pre += __shfl_xor_sync(0xffffffffu, pre, o);
    base = __ldg(dir + G) + pre;
    return true;
}

// Leaf step over a tile [a, a + count) of the last internal level whose
// coordinates are known (coords[i] = node a + i): the k^2+F engine (section
// 3.5) over the whole cached level, and the leaf tiles of the level-
// synchronous engine (section 3.4) over their frontier buffers.  One warp per
// 256-node block: the warp reads the block's signatures (one word of 8
// nibbles per lane), the first leaf from the directory (or the tile's scan),
// and the coordinates; a warp scan of the fan-outs turns the block into a
// list of its leaves (node, quadrant) in shared memory.  The lanes then take
// the leaves round-robin: leaf signature and the x entries of its two inputs
// are loaded together, then the combined updates are applied.  Every lane
// does the same work per leaf, whatever the fan-out of its node.
constexpr int kCachedWarps = 8;
constexpr uint32_t kLeafWords = 4 * kDirS / 8 + 1;   // words of 8 leaf nibbles covering one block's leaves

// Blocks per SM the kernel is compiled for: 5 for 4-wide batches (48
// registers, no spills; 5% faster than 4 blocks on the 300M-edge R-MAT at
// B = 16, and 3 or 4 leaves per lane group at 4 or 3 blocks are slower), 4
// otherwise (at 5 the single-vector path spills and runs 13% slower).
template <int VW> constexpr int cached_min_blocks() { return 4; }

template <int SR, int DIR, int VW>
__global__ void __launch_bounds__(32 * kCachedWarps, cached_min_blocks<VW>())
cached_block_kernel(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix, uint32_t leaf_base, uint32_t a,
                    uint32_t count, const Coord *coords, const uint8_t *leaf, VecArgs va)
{
    __shared__ Coord cs[kCachedWarps][kDirS];
    __shared__ uint16_t slots[kCachedWarps][4 * kDirS];
    __shared__ __align__(16) uint32_t wins[kCachedWarps][kWarpWindow];
    __shared__ uint32_t lsigs[kCachedWarps][kLeafWords];
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    uint32_t blk, s, e, base, w;
    if (!tile_warp_block(sig, dir, prefix, leaf_base, a, count, blockIdx.x * kCachedWarps + warp, blk, s, e, base, w))
        return;
    Coord *cw = cs[warp];
    uint16_t *sl = slots[warp];
    uint32_t *lw = lsigs[warp];
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (uint32_t q = 0; q < kDirS / 32; ++q) {
        const uint32_t i = 32u * q + lane;   // node blk + i
        if (blk + i >= s && blk + i < e) {
            const Coord p = coords[blk + i - a];
            cw[i] = p;
            const uint32_t o = DIR == K2T_RIGHT ? p.r : p.c;
            mn = min(mn, o);
            mx = max(mx, o);
        }
    }
    const uint32_t f = (uint32_t)__popc(w);
    const uint32_t incl = warp_incl_scan(f);
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    // the block's leaf signatures [base, base + total), as the words of 8
    // nibbles that hold them (coalesced; total <= 1024, so at most 129 words)
    const uint32_t lw0 = base >> 3, lsh = base & 7u;
    const uint32_t nlw = (lsh + total + 7u) >> 3;
    for (uint32_t k = lane; k < nlw; k += 32u) lw[k] = __ldg(reinterpret_cast<const uint32_t *>(leaf) + lw0 + k);
    uint32_t pos = incl - f;
    uint32_t rest = w;
    while (rest) {
        const uint32_t bit = (uint32_t)(__ffs(rest) - 1);  // 4*k + b
        rest &= rest - 1u;
        sl[pos++] = (uint16_t)(((8u * lane + bit / 4u) << 2) | (bit & 3u));
    }
    const uint32_t width = SR == K2T_BOOLEAN ? 1u : va.B;
    uint32_t lo, span;
    int wmode;
    uint32_t *win = warp_window_begin<SR>(mn, mx, 4u, width, wins[warp], lo, span, va, wmode);
    __syncwarp();
    warp_leaf_rounds<SR, DIR, VW>(0u, total, [&](uint32_t j, uint32_t &lam, uint32_t &r, uint32_t &c, uint32_t &li) {
        const uint32_t el = sl[j];
        const Coord p = cw[el >> 2];
        const uint32_t b = el & 3u;
        r = 4u * p.r + 2u * (b >> 1);
        c = 4u * p.c + 2u * (b & 1u);
        li = base + j;
        const uint32_t q = lsh + j;
        lam = (lw[q >> 3] >> (4u * (q & 7u))) & 15u;
    }, va, win, lo, wmode, lo);
    if (win) warp_window_flush<SR>(win, lo, span, width, va, wmode);
}

// ---- 4x4 leaves (leaf_k = 4) ------------------------------------------------------
#ifndef K2T_LEAF4_U
#define K2T_LEAF4_U 2
#endif
// The leaves the pages name as the next lever (section 5.6): a leaf is a 4x4
// bitmap (16-bit signature, cell (dr, dc) at bit 4*dr + dc).  Its four inputs
// are consecutive, so one vector load brings them; each of its (at most four)
// outputs sums its row segment (right) or column segment (left) in registers
// and updates y once.

// Cells of output q of a leaf as a 4-bit set over its inputs: right products
// take row q (bits 4q..4q+3), left products column q (bits q, q+4, q+8, q+12).
template <int DIR>
__device__ __forceinline__ uint32_t seg4(uint32_t lam, int q)
{
    if (DIR == K2T_RIGHT) return (lam >> (4 * q)) & 15u;
    const uint32_t v = (lam >> q) & 0x1111u;
    return (v | (v >> 3) | (v >> 6) | (v >> 9)) & 15u;
}

// Inputs a leaf reads: columns (right) or rows (left) holding a cell.
template <int DIR>
__device__ __forceinline__ uint32_t used4(uint32_t lam)
{
    if (DIR == K2T_RIGHT) return (lam | (lam >> 4) | (lam >> 8) | (lam >> 12)) & 15u;
    return (uint32_t)((lam & 0xfu) != 0) | ((uint32_t)((lam & 0xf0u) != 0) << 1) |
           ((uint32_t)((lam & 0xf00u) != 0) << 2) | ((uint32_t)((lam & 0xf000u) != 0) << 3);
}

// Records of the outputs out .. out + 3 of a 4x4 leaf (out a multiple of 4),
// one 16-byte load; 0 where an output is not heavy.
__device__ __forceinline__ uint4 heavy_word4(const VecArgs &va, uint32_t out)
{
    return __ldg(reinterpret_cast<const uint4 *>(va.hdir + out));
}

__device__ __forceinline__ uint32_t rec_at(const uint4 &h, int q)
{
    return q == 0 ? h.x : (q == 1 ? h.y : (q == 2 ? h.z : h.w));
}

// One vector slice (B = 1 fp32, or a Boolean word) of U leaves whose inputs
// xo[u][0..3] are loaded: every output with a cell gets its combined segment.
template <int SR, int DIR, int U, class InOf>
__device__ __forceinline__ void leaf4_apply1(const uint32_t (&lam)[U], const uint32_t (&out)[U], InOf &&in_of,
                                             const uint32_t (&xo)[U][4], uint32_t fl, const VecArgs &va,
                                             uint32_t *win, uint32_t lo)
{
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const uint32_t l = lam[u];
        if (!l) continue;
        if (!K2T_IN_RANGE(out[u] + 31u - (uint32_t)__clz(used4<DIR == K2T_RIGHT ? K2T_LEFT : K2T_RIGHT>(l)) < va.n_out,
                          va.status))
            continue;
        if constexpr (SR == K2T_BOOLEAN) {
            uint32_t *y = static_cast<uint32_t *>(va.y);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t s = seg4<DIR>(l, q);
                uint32_t v = 0u;
#pragma unroll
                for (int i = 0; i < 4; ++i) v |= ((s >> i) & 1u) ? xo[u][i] : 0u;
                v &= va.mask;
                if (!v) continue;
                if (win) atomicOr(win + (out[u] + q - lo), v);
                else atomicOr(y + out[u] + q, v);
            }
        } else {
            using S = Fp32Sem<SR>;
            float *y = static_cast<float *>(va.y);
            const uint4 h = SR == K2T_PLUS_TIMES && ((fl >> u) & 1u) ? heavy_word4(va, out[u]) : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t s = seg4<DIR>(l, q);
                if (!s) continue;
                HeavyDst hd{nullptr, nullptr};
                if (SR == K2T_PLUS_TIMES && rec_at(h, q)) {
                    hd = heavy_dst(va, rec_at(h, q), in_of(u), 0u);
                    if (!hd.p32) {
                        double d = 0.0;
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if ((s >> i) & 1u) d += (double)(va.w * __uint_as_float(xo[u][i]));
                        atomicAdd(hd.p64, d);
                        continue;
                    }
                }
                float v[1] = {S::zero()};
                bool any = false;
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    if ((s >> i) & 1u) {
                        const float c = S::contrib(__uint_as_float(xo[u][i]), va.w);
                        v[0] = any ? S::plus(v[0], c) : c;
                        any = true;
                    }
                if (hd.p32) {
                    S::update(hd.p32, v);
                    continue;
                }
                if (S::skip(v[0])) continue;
                if (win) smem_update<SR>(win + (out[u] + q - lo), __float_as_uint(v[0]));
                else S::update(y + out[u] + q, v);
            }
        }
    }
}

// One VW-wide slice k of one 4x4 leaf (origin r, c; cells lam) for batches.
template <int SR, int DIR, int VW>
__device__ __forceinline__ void leaf4_slice(uint32_t lam, uint32_t r, uint32_t c, uint32_t k, uint4 hv,
                                            const VecArgs &va, uint32_t *win, uint32_t lo)
{
    using S = Fp32Sem<SR>;
    const uint32_t in = DIR == K2T_RIGHT ? c : r;
    const uint32_t out = DIR == K2T_RIGHT ? r : c;
    const uint32_t use = used4<DIR>(lam);
    const float *x = static_cast<const float *>(va.x);
    float *y = static_cast<float *>(va.y);
    const size_t B = va.B;
    float xv[4][VW];
    if (!K2T_IN_RANGE(in + 31u - (uint32_t)__clz(use) < va.n_in &&
                          out + 31u - (uint32_t)__clz(used4<DIR == K2T_RIGHT ? K2T_LEFT : K2T_RIGHT>(lam)) < va.n_out,
                      va.status))
        return;
#pragma unroll
    for (int i = 0; i < 4; ++i)
        if ((use >> i) & 1u) VecLoad<VW>::load(x + (size_t)(in + i) * B + k, xv[i]);
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const uint32_t s = seg4<DIR>(lam, q);
        if (!s) continue;
        HeavyDst hd{nullptr, nullptr};
        if (SR == K2T_PLUS_TIMES && rec_at(hv, q)) {
            hd = heavy_dst(va, rec_at(hv, q), in, k);
            if (!hd.p32) {
#pragma unroll
                for (int e = 0; e < VW; ++e) {
                    double d = 0.0;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        if ((s >> i) & 1u) d += (double)(va.w * xv[i][e]);
                    atomicAdd(hd.p64 + e, d);
                }
                continue;
            }
        }
        float v[VW];
#pragma unroll
        for (int e = 0; e < VW; ++e) {
            bool any = false;
            v[e] = S::zero();
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if ((s >> i) & 1u) {
                    const float cv = S::contrib(xv[i][e], va.w);
                    v[e] = any ? S::plus(v[e], cv) : cv;
                    any = true;
                }
        }
        if (hd.p32) {
            S::update(hd.p32, v);
        } else if (win) {
#pragma unroll
            for (int e = 0; e < VW; ++e)
                if (!S::skip(v[e])) smem_update<SR>(win + (size_t)(out + q - lo) * B + k + e, __float_as_uint(v[e]));
        } else {
            S::update(y + (size_t)(out + q) * B + k, v);
        }
    }
}

// Leaves [jb, je) of a warp with 4x4 leaves; leaf_at(j, lam, r, c, li) as for
// warp_leaf_rounds (lam a 16-bit bitmap, (r, c) its block's origin).
//  - One vector slice: leaves dealt round-robin, four per lane per round; the
//    four inputs of a block come in one 16-byte load when x allows it.
//  - Batches: G = B/VW adjacent lanes share a leaf, each owning a VW slice.
template <int SR, int DIR, int VW, class LeafAt>
__device__ __forceinline__ void warp_leaf4_rounds(uint32_t jb, uint32_t je, LeafAt &&leaf_at, const VecArgs &va,
                                                  uint32_t *win, uint32_t lo, int wmode, uint32_t out_min)
{
    const uint32_t lane = threadIdx.x & 31u;
    const bool heavy = SR == K2T_PLUS_TIMES && va.hdir != nullptr && out_min < va.hdir_len &&
                       (!win || wmode == kWinShared);
    if (SR == K2T_BOOLEAN || (VW == 1 && va.B == 1)) {
        constexpr int U = K2T_LEAF4_U;
        const uint32_t *x = static_cast<const uint32_t *>(va.x);
        const bool x16 = ((uintptr_t)x & 15u) == 0;
        for (uint32_t j0 = jb; j0 < je; j0 += 32u * U) {
            uint32_t lam[U], r[U], c[U], fl = 0u;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t j = j0 + 32u * u + lane;
                lam[u] = 0u;
                r[u] = 0u;
                c[u] = 0u;
                uint32_t li = 0u;
                if (j < je) {
                    leaf_at(j, lam[u], r[u], c[u], li);
                    if (heavy) fl |= heavy_near(va, DIR == K2T_RIGHT ? r[u] : c[u]) << u;
                }
            }
            uint32_t xo[U][4], out[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t in = DIR == K2T_RIGHT ? c[u] : r[u];  // a multiple of 4
                out[u] = DIR == K2T_RIGHT ? r[u] : c[u];
#pragma unroll
                for (int i = 0; i < 4; ++i) xo[u][i] = 0u;
                if (lam[u]) {
                    if (x16 && in + 3u < va.n_in) {
                        const uint4 v = __ldg(reinterpret_cast<const uint4 *>(x + in));
                        xo[u][0] = v.x;
                        xo[u][1] = v.y;
                        xo[u][2] = v.z;
                        xo[u][3] = v.w;
                    } else {
#pragma unroll
                        for (int i = 0; i < 4; ++i)
                            if (in + (uint32_t)i < va.n_in) xo[u][i] = __ldg(x + in + i);
                    }
                }
            }
            auto in_of = [&](int u) {
                uint32_t l2, r2, c2, li2;
                leaf_at(j0 + 32u * (uint32_t)u + lane, l2, r2, c2, li2);
                return DIR == K2T_RIGHT ? c2 : r2;
            };
            leaf4_apply1<SR, DIR, U>(lam, out, in_of, xo, fl, va, win, lo);
        }
        return;
    }
    if constexpr (SR != K2T_BOOLEAN) {
        constexpr int U = kBatchU;
        const uint32_t G = va.B / VW;
        const uint32_t per = G <= 32u ? 32u / G : 1u;
        const uint32_t groups = G <= 32u ? G : 32u;
        const uint32_t slot = lane / groups, sub = lane % groups;
        const bool active = slot < per;
        for (uint32_t j0 = jb; j0 < je; j0 += per * U) {
            uint32_t lam[U], r[U], c[U];
            uint4 hv[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const uint32_t j = j0 + (uint32_t)u * per + slot;
                lam[u] = 0u;
                r[u] = 0u;
                c[u] = 0u;
                hv[u] = make_uint4(0u, 0u, 0u, 0u);
                uint32_t li = 0u;
                if (active && j < je) {
                    leaf_at(j, lam[u], r[u], c[u], li);
                    if (heavy && heavy_near(va, DIR == K2T_RIGHT ? r[u] : c[u]))
                        hv[u] = heavy_word4(va, DIR == K2T_RIGHT ? r[u] : c[u]);
                }
            }
            for (uint32_t k = sub * VW; k < va.B; k += groups * VW) {
#pragma unroll
                for (int u = 0; u < U; ++u)
                    if (lam[u]) leaf4_slice<SR, DIR, VW>(lam[u], r[u], c[u], k, hv[u], va, win, lo);
            }
        }
    }
}

// CACHED engine with 4x4 leaves: as cached_block_kernel (one warp per 256-node
// directory block of the last internal level, leaf list built by a warp scan,
// per-warp output window), with nodes covering 8x8 cells and 16-bit leaves.
#ifndef K2T_LEAF4_MINB
#define K2T_LEAF4_MINB 4
#endif
template <int SR, int DIR, int VW>
__global__ void __launch_bounds__(32 * kCachedWarps, K2T_LEAF4_MINB)
cached4_block_kernel(const uint8_t *sig, const uint32_t *dir, uint32_t n, const Coord *coords, const uint16_t *leaf,
                     VecArgs va)
{
    __shared__ Coord cs[kCachedWarps][kDirS];
    __shared__ uint16_t slots[kCachedWarps][4 * kDirS];
    __shared__ __align__(16) uint32_t wins[kCachedWarps][kWarpWindow];
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t g = blockIdx.x * kCachedWarps + warp;
    const uint32_t s = g * kDirS;
    if (s >= n) return;
    const uint32_t cnt = min(n - s, kDirS);
    Coord *cw = cs[warp];
    uint16_t *sl = slots[warp];
    uint32_t w = 0;
    if (8u * lane < cnt) {
        w = __ldg(reinterpret_cast<const uint32_t *>(sig + s / 2) + lane);
        if (8u * lane + 8u > cnt) w &= (1u << (4u * (cnt - 8u * lane))) - 1u;
    }
    const uint32_t base = __ldg(dir + g);
    uint32_t mn = 0xffffffffu, mx = 0u;
#pragma unroll
    for (uint32_t q = 0; q < kDirS / 32; ++q) {
        const uint32_t i = 32u * q + lane;
        if (i < cnt) {
            const Coord p = coords[s + i];
            cw[i] = p;
            const uint32_t o = DIR == K2T_RIGHT ? p.r : p.c;
            mn = min(mn, o);
            mx = max(mx, o);
        }
    }
    const uint32_t f = (uint32_t)__popc(w);
    const uint32_t incl = warp_incl_scan(f);
    const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
    uint32_t pos = incl - f;
    uint32_t rest = w;
    while (rest) {
        const uint32_t bit = (uint32_t)(__ffs(rest) - 1);  // 4*k + b
        rest &= rest - 1u;
        sl[pos++] = (uint16_t)(((8u * lane + bit / 4u) << 2) | (bit & 3u));
    }
    const uint32_t width = SR == K2T_BOOLEAN ? 1u : va.B;
    uint32_t lo, span;
    int wmode;
    uint32_t *win = warp_window_begin<SR>(mn, mx, 8u, width, wins[warp], lo, span, va, wmode);
    __syncwarp();
    warp_leaf4_rounds<SR, DIR, VW>(0u, total, [&](uint32_t j, uint32_t &lam, uint32_t &r, uint32_t &c, uint32_t &li) {
        const uint32_t e = sl[j];
        const Coord p = cw[e >> 2];
        const uint32_t b = e & 3u;
        r = 8u * p.r + 4u * (b >> 1);
        c = 8u * p.c + 4u * (b & 1u);
        li = base + j;
        lam = __ldg(leaf + li);
    }, va, win, lo, wmode, lo);
    if (win) warp_window_flush<SR>(win, lo, span, width, va, wmode);
}

// BANDED engine: the cached last internal level grouped by row band (band_rows
// rows each; level order inside a band), one thread block per block of at most
// kBandChunkNodes nodes of one band.  Warps take 256-node tiles: coordinates,
// first leaves and signatures are read coalesced, a warp scan turns a tile
// into a leaf list (node, quadrant, rank) in shared memory, and the lanes take
// the leaves round-robin.
//  - Right products: every output row of the block lies in its band, so the
//    block reduces y in a shared-memory window over the band (semiring shared
//    atomics) and adds each touched row to y once, consecutively.  The only
//    scattered access left per leaf is the gather of x.
//  - Left products: the inputs are the band's rows, a small contiguous slice
//    of x that stays in L1; the outputs (columns) are reduced straight into y.
constexpr int kBandWarps = 8;
constexpr uint32_t kBandWindow = 8192;  // words of the block's window
constexpr size_t kBandSmem = kBandWindow * 4 + kBandWarps * kDirS * (8 + 4 + 8);

template <int SR, int DIR, int VW>
__global__ void __launch_bounds__(32 * kBandWarps)
banded_kernel(const uint32_t *chunks, const Coord *coords, const uint32_t *bleaf, const uint8_t *bsig,
              const uint8_t *leaf, uint32_t band_rows, VecArgs va)
{
    // one dynamic buffer (more than 48 KB: opted in at launch)
    extern __shared__ __align__(16) uint8_t bsm[];
    uint32_t *win = reinterpret_cast<uint32_t *>(bsm);
    Coord (*cs)[kDirS] = reinterpret_cast<Coord (*)[kDirS]>(bsm + kBandWindow * 4);
    uint32_t (*lf)[kDirS] = reinterpret_cast<uint32_t (*)[kDirS]>(bsm + kBandWindow * 4 + kBandWarps * kDirS * 8);
    uint16_t (*slots)[4 * kDirS] =
        reinterpret_cast<uint16_t (*)[4 * kDirS]>(bsm + kBandWindow * 4 + kBandWarps * kDirS * 12);
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint32_t band = chunks[3 * blockIdx.x], s0 = chunks[3 * blockIdx.x + 1], cnt = chunks[3 * blockIdx.x + 2];
    const uint32_t width = SR == K2T_BOOLEAN ? 1u : va.B;
    const uint64_t band_lo = (uint64_t)band * band_rows;
    const uint64_t band_hi = min(band_lo + band_rows, (uint64_t)va.n_out);
    const bool windowed = DIR == K2T_RIGHT && band_hi > band_lo && (band_hi - band_lo) * width <= kBandWindow;
    const uint32_t words = windowed ? (uint32_t)((band_hi - band_lo) * width) : 0u;
    if (windowed) {
        for (uint32_t i = threadIdx.x; i < words; i += 32u * kBandWarps) win[i] = zero_word<SR>();
        __syncthreads();
    }
    Coord *cw = cs[warp];
    uint32_t *lw = lf[warp];
    uint16_t *sl = slots[warp];
    for (uint32_t t0 = 256u * warp; t0 < cnt; t0 += 256u * kBandWarps) {
        const uint32_t tn = min(cnt - t0, 256u);
        const uint32_t base = s0 + t0;
        uint32_t w = 0;
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k) {
            const uint32_t i = 8u * lane + k;
            if (i < tn) w |= nibble_at(bsig, base + i) << (4u * k);
        }
#pragma unroll
        for (uint32_t q = 0; q < kDirS / 32; ++q) {
            const uint32_t i = 32u * q + lane;
            if (i < tn) {
                cw[i] = coords[base + i];
                lw[i] = bleaf[base + i];
            }
        }
        const uint32_t f = (uint32_t)__popc(w);
        const uint32_t incl = warp_incl_scan(f);
        const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t pos = incl - f;
#pragma unroll
        for (uint32_t k = 0; k < 8; ++k) {
            const uint32_t sg = (w >> (4u * k)) & 15u;
            uint32_t rank = 0;
#pragma unroll
            for (uint32_t b = 0; b < 4; ++b)
                if (sg & (1u << b)) sl[pos++] = (uint16_t)(((8u * lane + k) << 4) | (b << 2) | rank++);
        }
        __syncwarp();
        warp_leaf_rounds<SR, DIR, VW>(0u, total, [&](uint32_t j, uint32_t &lam, uint32_t &r, uint32_t &c, uint32_t &li) {
            const uint32_t e = sl[j];
            const uint32_t node = e >> 4, b = (e >> 2) & 3u;
            const Coord p = cw[node];
            r = 4u * p.r + 2u * (b >> 1);
            c = 4u * p.c + 2u * (b & 1u);
            li = lw[node] + (e & 3u);
            lam = nibble_at(leaf, li);
        }, va, windowed ? win : nullptr, (uint32_t)band_lo, kWinShared, 0u);
        __syncwarp();
    }
    if (windowed) {
        __syncthreads();
        uint32_t *y = static_cast<uint32_t *>(va.y) + band_lo * width;
        for (uint32_t i = threadIdx.x; i < words; i += 32u * kBandWarps) {
            const uint32_t v = win[i];
            if (!is_noop_word<SR>(v)) global_update_word<SR>(y + i, v);
        }
    }
}

// ---- shared-memory staging with the bulk-copy (TMA) engine ------------------
// One thread arms an mbarrier with the total byte count and issues one
// cp.async.bulk per contiguous range; every thread then waits on the barrier.
// Each wait polls at most kWaitLimit times; a stage that does not complete
// sets bit 0 of the device status word and the block leaves without touching
// its outputs (after one more bounded wait for its copies).
constexpr uint32_t kWaitLimit = 1u << 24;
constexpr uint32_t kStatusStageTimeout = 1u;

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t *bar)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(smem_u32(bar)) : "memory");
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes) : "memory");
}

// dst (shared) and src (global) 16-byte aligned, bytes a multiple of 16
__device__ __forceinline__ void bulk_copy(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t phase)
{
    for (uint32_t i = 0; i < kWaitLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(phase)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// A staged copy of global bytes [lo, hi) of `base`, widened to 16-byte
// boundaries; returns the offset of byte lo inside the copy.
struct StagePlan {
    uint64_t lo16;
    uint32_t bytes;
    uint32_t shift;
};

__device__ __forceinline__ StagePlan stage_plan(uint64_t lo, uint64_t hi)
{
    StagePlan p;
    p.lo16 = lo & ~(uint64_t)15;
    uint64_t hi16 = (hi + 15) & ~(uint64_t)15;
    p.bytes = (uint32_t)(hi16 - p.lo16);
    p.shift = (uint32_t)(lo - p.lo16);
    return p;
}

// nibble k of a staged signature copy
__device__ __forceinline__ uint32_t snib(const uint8_t *sg, uint32_t k)
{
    return (uint32_t)(sg[k >> 1] >> ((k & 1u) * 4u)) & 15u;
}

// First child of `node` of a level from its directory: the sample of its
// 256-node block plus the fan-outs before it in the block (section 3.2).
// `n` is the level's node count; node == n gives the level's total.
__device__ __forceinline__ uint32_t dir_offset(const uint8_t *sig, const uint32_t *dir, uint32_t n, uint32_t node)
{
    if (node >= n) return __ldg(dir + (n + kDirS - 1) / kDirS);
    const uint32_t g = node / kDirS;
    uint32_t base = __ldg(dir + g);
    const uint64_t *w = reinterpret_cast<const uint64_t *>(sig);
    const uint32_t w0 = g * (kDirS / 16), w1 = node / 16;
    for (uint32_t k = w0; k < w1; ++k) base += (uint32_t)__popcll(__ldg(w + k));
    const uint32_t rem = node & 15u;
    if (rem) base += (uint32_t)__popcll(__ldg(w + w1) & ((1ull << (4 * rem)) - 1ull));
    return base;
}

// ---- FUSED engine ------------------------------------------------------------------
// One warp expands the parents at nibbles [nb, nb + n) of a staged level
// (parent i at nibble nb + i, coordinates cur[i]), one parent per lane per
// round: lanes read consecutive signatures and coordinates, a warp scan
// places the children, which go to nxt[0 ...] in level order.
__device__ __forceinline__ void warp_expand(const uint8_t *sg8, uint32_t nb, uint32_t n, const Coord *cur, Coord *nxt)
{
    const uint32_t lane = threadIdx.x & 31u;
    uint32_t start = 0;
    for (uint32_t i0 = 0; i0 < n; i0 += 32u) {
        const uint32_t i = i0 + lane;
        const uint32_t sg = i < n ? snib(sg8, nb + i) : 0u;
        const uint32_t f = (uint32_t)__popc(sg);
        const uint32_t incl = warp_incl_scan(f);
        uint32_t pos = start + incl - f;
        start += __shfl_sync(0xffffffffu, incl, 31);
        if (sg) {
            const Coord p = cur[i];
#pragma unroll
            for (int b = 0; b < 4; ++b)
                if (sg & (1u << b)) nxt[pos++] = child_of(p, b);
        }
    }
}

// Bytes of one level's staging slot in fused_kernel: the nibbles (or, for a
// 4x4 leaf level, the 16-bit signatures) of at most cap nodes, widened to
// 16-byte boundaries at both ends, with room for an 8-byte read past the end.
__host__ __device__ constexpr uint32_t fused_slot(uint32_t cap, bool wide)
{
    return ((wide ? 2u * cap : cap / 2u) + 48u + 15u) & ~15u;
}

// Header of a warp's shared memory in fused_kernel: its mbarrier (16 bytes)
// and the nibble (or element) offset of each staged level inside its slot.
__host__ __device__ constexpr uint32_t fused_header() { return (16u + 4u * K2T_MAX_LEVELS + 15u) & ~15u; }

// Shared memory of one warp of fused_kernel for a tree: the header, one
// staging slot per level from d0 (the leaf level's holds 2 bytes a leaf with
// 4x4 leaves) and two coordinate buffers of cap entries.  A multiple of 16.
inline uint32_t fused_warp_bytes(int levels, int d0, uint32_t cap, bool l4)
{
    return fused_header() + (uint32_t)(levels - 1 - d0) * fused_slot(cap, false) + fused_slot(cap, l4) + 16u * cap;
}

// FUSED engine: warp w of thread block k descends chunk 2k + w, a run of whole
// subtrees rooted at level d_c with at most `cap` leaves, from its roots to
// the leaves, alone: no block barrier, so narrow levels keep only their own
// warp busy.  The chunk record holds the index of its roots' coordinates and,
// for every level, the first node and the node count of the chunk there
// (planned once per tree on the host).  The warp stages the signatures of all
// its levels with one bulk copy per level on its own mbarrier, expands level
// by level in its shared memory down to the last internal level, then runs
// the leaf step over that level's nodes as the k^2+F kernel does over the
// cached level: a warp scan of the fan-outs lists the leaves (node, quadrant)
// and the lanes take them round-robin.  No global scratch.  L4: the leaf
// level holds 4x4 bitmaps (16-bit signatures, section 5.6).
template <int SR, int DIR, int VW, bool L4>
__global__ void __launch_bounds__(kFusedThreads, 16)
fused_kernel(DevTree tr, const uint32_t *chunks, uint32_t stride, const Coord *roots, uint32_t cap, uint64_t n_chunks,
             uint32_t wbytes, VecArgs va, uint32_t *status)
{
    extern __shared__ __align__(16) uint8_t fsm[];
    const uint32_t lane = threadIdx.x & 31u, warp = threadIdx.x >> 5;
    const uint64_t chunk = (uint64_t)blockIdx.x * kFusedWarps + warp;
    if (chunk >= n_chunks) return;
    const int d0 = tr.d0, l = tr.levels;
    uint8_t *wsm = fsm + (size_t)warp * wbytes;
    uint64_t *bar = reinterpret_cast<uint64_t *>(wsm);
    uint32_t *nbase = reinterpret_cast<uint32_t *>(wsm + 16);   // per level from d0
    uint8_t *stage = wsm + fused_header();
    const uint32_t slot = fused_slot(cap, false);
    Coord *cur = reinterpret_cast<Coord *>(stage + (size_t)(l - 1 - d0) * slot + fused_slot(cap, L4));
    Coord *nxt = cur + cap;

    const uint32_t *rec = chunks + chunk * stride;
    const uint32_t rc = rec[0];
    const int dc = (int)rec[1];
    const uint32_t *rng = rec + 2;
#ifdef K2T_CHECKED
    {
        bool fits = dc >= d0 && dc <= l - 2;
        for (int d = dc; fits && d < l; ++d) fits = rng[2 * (d - d0) + 1] <= cap;
        if (!K2T_IN_RANGE(fits, status)) return;
    }
#endif
    if (lane == 0) {
        // the byte range of every level of the chunk, widened to 16 bytes
        auto plan = [&](int d) {
            const uint32_t s = rng[2 * (d - d0)], n = rng[2 * (d - d0) + 1];
            if (L4 && d == l - 1) return stage_plan(2ull * s, 2ull * ((uint64_t)s + n));   // 2 bytes a leaf
            return stage_plan(s >> 1, ((uint64_t)s + n + 1) >> 1);                      // a nibble a node
        };
        uint32_t total = 0;
        for (int d = dc; d < l; ++d) {
            const StagePlan pl = plan(d);
            total += pl.bytes;
            nbase[d - d0] = L4 && d == l - 1 ? pl.shift / 2u : 2u * pl.shift + (rng[2 * (d - d0)] & 1u);
        }
        mbar_init(bar);
        mbar_expect_tx(bar, total);
        for (int d = dc; d < l; ++d) {
            const StagePlan pl = plan(d);
            bulk_copy(stage + (size_t)(d - d0) * slot, tr.lv[d].sig + pl.lo16, pl.bytes, bar);
        }
    }
    {
        const uint32_t n = rng[2 * (dc - d0) + 1];
        for (uint32_t i = lane; i < n; i += 32u) cur[i] = roots[rc + i];
    }
    __syncwarp();
    if (!mbar_wait(bar, 0)) {
        if (lane == 0) atomicOr(status, kStatusStageTimeout);
        mbar_wait(bar, 0);
        return;
    }
    // descent to the last internal level
    for (int d = dc; d < l - 2; ++d) {
        warp_expand(stage + (size_t)(d - d0) * slot, nbase[d - d0], rng[2 * (d - d0) + 1], cur, nxt);
        __syncwarp();
        Coord *t = cur;
        cur = nxt;
        nxt = t;
    }
    // leaf step over the chunk's nodes of the last internal level (cur)
    const uint32_t n2 = rng[2 * (l - 2 - d0) + 1];
    const uint32_t *sig2 = reinterpret_cast<const uint32_t *>(stage + (size_t)(l - 2 - d0) * slot);
    const uint32_t nb2 = nbase[l - 2 - d0];
    const uint8_t *lsig = stage + (size_t)(l - 1 - d0) * slot;
    const uint32_t lnb = nbase[l - 1 - d0];
    const uint32_t leaf0 = rng[2 * (l - 1 - d0)];   // the chunk's first leaf (level order)
    constexpr uint32_t unit = L4 ? 8u : 4u;         // cells a node covers per side
    uint32_t mn = 0xffffffffu, mx = 0u;
    for (uint32_t i = lane; i < n2; i += 32u) {
        const Coord p = cur[i];
        const uint32_t o = DIR == K2T_RIGHT ? p.r : p.c;
        mn = min(mn, o);
        mx = max(mx, o);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        mn = min(mn, __shfl_xor_sync(0xffffffffu, mn, o));
        mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    // the free buffer holds the leaf list of one 256-node round, then, when
    // there is room, the warp's output window
    uint16_t *sl = reinterpret_cast<uint16_t *>(nxt);
    const uint32_t sl_bytes = (2u * min(cap, 4u * kDirS) + 15u) & ~15u;
    const uint32_t width = SR == K2T_BOOLEAN ? 1u : va.B;
    uint32_t lo = unit * mn, span = 0u;
    int wmode = kWinF32;
    uint32_t *win = nullptr;
    if (8u * cap >= sl_bytes + 4u * kWarpWindow)
        win = warp_window_begin<SR>(mn, mx, unit, width,
                                    reinterpret_cast<uint32_t *>(reinterpret_cast<uint8_t *>(nxt) + sl_bytes), lo, span,
                                    va, wmode);
    const uint32_t out_min = unit * mn;
    uint32_t lj0 = 0;   // leaves of the chunk before this round
    for (uint32_t b0 = 0; b0 < n2; b0 += kDirS) {
        // lane's 8 nibbles: nodes b0 + 8 lane .. + 7 (those below n2)
        const uint32_t t0 = b0 + 8u * lane;
        uint32_t w = 0u;
        if (t0 < n2) {
            const uint32_t q = nb2 + t0;
            w = __funnelshift_r(sig2[q >> 3], sig2[(q >> 3) + 1], 4u * (q & 7u));
            if (n2 - t0 < 8u) w &= (1u << (4u * (n2 - t0))) - 1u;
        }
        const uint32_t f = (uint32_t)__popc(w);
        const uint32_t incl = warp_incl_scan(f);
        const uint32_t total = __shfl_sync(0xffffffffu, incl, 31);
        uint32_t pos = incl - f;
        uint32_t rest = w;
        while (rest) {
            const uint32_t bit = (uint32_t)(__ffs(rest) - 1);  // 4*k + b
            rest &= rest - 1u;
            sl[pos++] = (uint16_t)(((8u * lane + bit / 4u) << 2) | (bit & 3u));
        }
        __syncwarp();
        const Coord *cb = cur + b0;
        const uint32_t ljb = lj0;
        if constexpr (L4) {
            const uint16_t *ls16 = reinterpret_cast<const uint16_t *>(lsig) + lnb + ljb;
            warp_leaf4_rounds<SR, DIR, VW>(0u, total, [&](uint32_t j, uint32_t &lam, uint32_t &r, uint32_t &c, uint32_t &li) {
                const uint32_t el = sl[j];
                const Coord p = cb[el >> 2];
                const uint32_t b = el & 3u;
                r = 8u * p.r + 4u * (b >> 1);
                c = 8u * p.c + 4u * (b & 1u);
                li = leaf0 + ljb + j;
                lam = ls16[j];
            }, va, win, lo, wmode, out_min);
        } else {
            warp_leaf_rounds<SR, DIR, VW>(0u, total, [&](uint32_t j, uint32_t &lam, uint32_t &r, uint32_t &c, uint32_t &li) {
                const uint32_t el = sl[j];
                const Coord p = cb[el >> 2];
                const uint32_t b = el & 3u;
                r = 4u * p.r + 2u * (b >> 1);
                c = 4u * p.c + 2u * (b & 1u);
                li = leaf0 + ljb + j;
                lam = snib(lsig, lnb + ljb + j);
            }, va, win, lo, wmode, out_min);
        }
        lj0 += total;
        __syncwarp();
    }
    if (win) warp_window_flush<SR>(win, lo, span, width, va, wmode);
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
    const uint32_t *bchunks = nullptr;
    const uint32_t *bleaf = nullptr;
    const uint8_t *bsig = nullptr;
    Coord *buf[K2T_MAX_LEVELS] = {};
    uint32_t *scan_sums = nullptr;
    uint32_t *scan_prefix = nullptr;
    uint32_t *err = nullptr;
    void *vec[2] = {nullptr, nullptr};
    const uint32_t *hdir[2] = {nullptr, nullptr};   // heavy outputs, per direction (null: none)
    const uint32_t *hlist[2] = {nullptr, nullptr};
    float *acc = nullptr;
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
template <int SR, int DIR, int VW, bool L4>
void launch_fused_k(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const uint32_t wb = fused_warp_bytes(t->levels, t->d0, t->opts.chunk_cap, L4);
    const size_t smem = (size_t)wb * kFusedWarps;
    static size_t configured = 0;
    if (smem > configured) {
        cudaFuncSetAttribute(fused_kernel<SR, DIR, VW, L4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        configured = smem;
    }
    const uint64_t grid = (t->n_chunks + kFusedWarps - 1) / kFusedWarps;
    if (grid)
        fused_kernel<SR, DIR, VW, L4><<<(unsigned)grid, kFusedThreads, smem, st>>>(
            d->tree, d->chunks, t->chunk_stride, d->roots, t->opts.chunk_cap, t->n_chunks, wb, va, d->err);
}

template <int SR, int DIR, int VW>
void launch_fused(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    if (t->leaf_k4) launch_fused_k<SR, DIR, VW, true>(t, d, va, st);
    else launch_fused_k<SR, DIR, VW, false>(t, d, va, st);
}

// Leaf step over the tile [a, a + count) of the last internal level (coords
// index 0 = node a): directory mode (prefix null) or scan mode.
template <int SR, int DIR, int VW>
void launch_leaf_tile(const uint8_t *sig, const uint32_t *dir, const uint32_t *prefix, uint32_t leaf_base, uint32_t a,
                      uint32_t count, const Coord *coords, const uint8_t *leaf, const VecArgs &va, cudaStream_t st)
{
    const uint64_t blocks = prefix ? ((uint64_t)count + kDirS - 1) / kDirS
                                   : ((uint64_t)a + count + kDirS - 1) / kDirS - a / kDirS;
    const unsigned grid = (unsigned)((blocks + kCachedWarps - 1) / kCachedWarps);
    if (grid)
        cached_block_kernel<SR, DIR, VW><<<grid, 32 * kCachedWarps, 0, st>>>(sig, dir, prefix, leaf_base, a, count,
                                                                             coords, leaf, va);
}

template <int SR, int DIR, int VW>
void launch_cached(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const int l = t->levels;
    const uint32_t n = (uint32_t)t->nodes[(size_t)l - 2];
    launch_leaf_tile<SR, DIR, VW>(d->tree.lv[l - 2].sig, d->tree.lv[l - 2].dir, nullptr, 0u, 0u, n, d->cached,
                                  d->tree.lv[l - 1].sig, va, st);
}

template <int SR, int DIR, int VW>
void launch_cached4(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const int l = t->levels;
    const uint32_t n = (uint32_t)t->nodes[(size_t)l - 2];
    const uint32_t blocks = (n + kDirS - 1) / kDirS;
    const unsigned grid = (unsigned)((blocks + kCachedWarps - 1) / kCachedWarps);
    cached4_block_kernel<SR, DIR, VW><<<grid, 32 * kCachedWarps, 0, st>>>(
        d->tree.lv[l - 2].sig, d->tree.lv[l - 2].dir, n, d->cached,
        reinterpret_cast<const uint16_t *>(d->tree.lv[l - 1].sig), va);
}

template <int SR, int DIR, int VW>
void launch_banded(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    const int l = t->levels;
    const unsigned grid = (unsigned)(t->bchunks.size() / 3);
    if (!grid) return;
    static bool configured = false;
    if (!configured) {
        cudaFuncSetAttribute(banded_kernel<SR, DIR, VW>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kBandSmem);
        configured = true;
    }
    banded_kernel<SR, DIR, VW><<<grid, 32 * kBandWarps, kBandSmem, st>>>(d->bchunks, d->cached, d->bleaf, d->bsig,
                                                                          d->tree.lv[l - 1].sig, t->opts.band_rows, va);
}

// Scratch of one level-synchronous product: a frontier buffer per expanded
// level and, for scan offsets, the block sums and their prefixes.  k2t_spmv
// takes them from the tree's arena, k2t_spmv_noalloc from its static array.
struct LsBufs {
    Coord *buf[K2T_MAX_LEVELS];
    uint32_t *sums;
    uint32_t *prefix;
    uint64_t buf_entries;   // entries of each frontier buffer
};

// The planned launch sequence of the level-synchronous engine (section 3.4).
template <int SR, int DIR, int VW>
void run_ls(const k2t_tree *t, const DeviceState *d, const LsBufs &sb, const VecArgs &va, cudaStream_t st)
{
    const bool scan = t->opts.offsets == K2T_OFFSETS_SCAN;
    const int l = t->levels;
    for (const LsStep &s : t->steps) {
        const int lv = s.level;
        const Coord *src = s.src == 0xff ? d->top : sb.buf[s.src];
        const uint8_t *sig = d->tree.lv[lv].sig;
        const uint32_t *dir = d->tree.lv[lv].dir;
        const uint64_t blocks = scan ? (s.count + 255u) / 256u
                                     : ((uint64_t)s.a + s.count + kDirS - 1) / kDirS - s.a / kDirS;
        const uint32_t *prefix = nullptr;
        if (scan) {
            ls_block_sums_kernel<<<grid_for_blocks(blocks), kWalkThreads, 0, st>>>(sig, s.a, s.count, sb.sums);
            ls_scan_kernel<<<1, 1024, 0, st>>>(sb.sums, (uint32_t)blocks, sb.prefix);
            prefix = sb.prefix;
        }
        if (s.kind == 0) {
            ls_expand_kernel<<<grid_for_blocks(blocks), kWalkThreads, 0, st>>>(
                sig, dir, prefix, s.a, s.count, src, s.src_base, sb.buf[lv + 1], s.dst_base, sb.buf_entries, va.status);
        } else {
            const uint32_t base = scan ? (uint32_t)level_offset(t, lv, s.a) : 0u;
            launch_leaf_tile<SR, DIR, VW>(sig, scan ? nullptr : dir, prefix, base, s.a, s.count,
                                          src + (s.a - s.src_base), d->tree.lv[l - 1].sig, va, st);
        }
    }
}

template <int SR, int DIR, int VW>
void launch_ls(const k2t_tree *t, const DeviceState *d, const VecArgs &va, cudaStream_t st)
{
    LsBufs sb{};
    for (int lv = 0; lv < K2T_MAX_LEVELS; ++lv) sb.buf[lv] = d->buf[lv];
    sb.sums = d->scan_sums;
    sb.prefix = d->scan_prefix;
    sb.buf_entries = t->layout.buf_bytes / sizeof(Coord);
    run_ls<SR, DIR, VW>(t, d, sb, va, st);
}

using LaunchFn = void (*)(const k2t_tree *, const DeviceState *, const VecArgs &, cudaStream_t);

// Internal engine id: the CACHED engine on a tree with 4x4 leaves.
constexpr uint32_t kEngineCached4 = 100;

// Plus-times products of a direction with heavy outputs.  heavy_begin points
// va at the direction's tables and zeroes their sums for the B vectors
// (queued after the fill of y); heavy_end adds each output's sums in fp64 and
// rounds the total into y once (queued after the product).  Other semirings:
// va gets no tables.
inline bool heavy_begin(const k2t_tree *t, const DeviceState *d, int dir, int semiring, VecArgs &va, cudaStream_t st)
{
    va.hdir = nullptr;
    va.hdir_len = 0u;
    va.acc = nullptr;
    if (semiring != K2T_PLUS_TIMES || !d->hdir[dir]) return false;
    va.hdir = d->hdir[dir];
    va.hdir_len = (uint32_t)t->hdir[dir].size();
    va.acc = d->acc;
    const uint64_t words = t->hrows[dir] * va.B;
    const uint64_t blocks = std::min<uint64_t>((words / 4 + 255) / 256 + 1, 152ull * 8);
    fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(reinterpret_cast<uint32_t *>(d->acc), words, 0u);
    return true;
}

inline void heavy_end(const k2t_tree *t, const DeviceState *d, int dir, const VecArgs &va, cudaStream_t st)
{
    const uint32_t h = (uint32_t)t->hlist[dir].size();
    const uint64_t blocks = std::min<uint64_t>(((uint64_t)h + 7) / 8, 152ull * 32);
    heavy_finish_kernel<<<(unsigned)blocks, 256, 0, st>>>(d->acc, d->hdir[dir], d->hlist[dir], h, va.B,
                                                          static_cast<float *>(va.y));
}

template <int SR, int DIR, int VW>
LaunchFn pick_engine(uint32_t engine)
{
    switch (engine) {
    case K2T_ENGINE_FUSED: return launch_fused<SR, DIR, VW>;
    case K2T_ENGINE_CACHED: return launch_cached<SR, DIR, VW>;
    case K2T_ENGINE_BANDED: return launch_banded<SR, DIR, VW>;
    case kEngineCached4: return launch_cached4<SR, DIR, VW>;
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
