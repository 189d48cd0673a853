// k2t_static.cu -- a level-synchronous product that allocates nothing.
//
// Some callers cannot call cudaMalloc at product time: code that runs inside
// a framework owning all device memory through its own pool, code that must
// never synchronise the device (cudaMalloc can), and code working to a fixed
// device-memory budget committed before it starts.  k2t_spmv_noalloc serves
// them: it runs the tiled level-synchronous descent with its frontier buffers
// and scan space in one file-scope device array of kStaticScratchBytes,
// present on every GPU that loads this library until the process exits.  The
// caller still provides the tree's arena (to k2t_upload) and x and y.
//
// Host code must not pass the array's name to a kernel: on the host it is a
// stand-in, not a device address.  The first call on each device looks the
// address up with cudaGetSymbolAddress (with that device current) and keeps
// it; later calls reuse it.
//
// Every call shares the array.  Nothing in it has to start at zero (each
// frontier buffer and scan entry is written before it is read within one
// product), and calls whose work overlaps on the GPU race on it.
#include <mutex>

#include "k2t_kernels.cuh"

namespace k2t {

constexpr uint64_t kStaticScratchBytes = 64ull << 20;   // 64 MiB
constexpr int kStaticMaxDevices = 64;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

namespace {

std::mutex g_static_mutex;
void *g_static_ptr[kStaticMaxDevices] = {};

// Device address of the scratch array on device `dev`, which is current
// (looked up once per device).
int static_scratch(int dev, void **out)
{
    if (dev < 0 || dev >= kStaticMaxDevices) return K2T_ERANGE;
    std::lock_guard<std::mutex> lock(g_static_mutex);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || !p) { g_last_cuda = (int)e; return K2T_ECUDA; }
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return K2T_OK;
}

using StaticFn = void (*)(const k2t_tree *, const DeviceState *, const LsBufs &, const VecArgs &, cudaStream_t);

template <int SR, int DIR>
StaticFn pick_static_vw(int vw)
{
    if constexpr (SR == K2T_BOOLEAN) {
        (void)vw;
        return run_ls<SR, DIR, 1>;
    } else {
        if (vw == 4) return run_ls<SR, DIR, 4>;
        if (vw == 2) return run_ls<SR, DIR, 2>;
        return run_ls<SR, DIR, 1>;
    }
}

StaticFn pick_static(int semiring, int dir, int vw)
{
    if (semiring == K2T_PLUS_TIMES)
        return dir == K2T_RIGHT ? pick_static_vw<K2T_PLUS_TIMES, K2T_RIGHT>(vw) : pick_static_vw<K2T_PLUS_TIMES, K2T_LEFT>(vw);
    if (semiring == K2T_BOOLEAN)
        return dir == K2T_RIGHT ? pick_static_vw<K2T_BOOLEAN, K2T_RIGHT>(vw) : pick_static_vw<K2T_BOOLEAN, K2T_LEFT>(vw);
    return dir == K2T_RIGHT ? pick_static_vw<K2T_MIN_PLUS, K2T_RIGHT>(vw) : pick_static_vw<K2T_MIN_PLUS, K2T_LEFT>(vw);
}

}  // namespace
}  // namespace k2t

using namespace k2t;

extern "C" {

uint64_t k2t_noalloc_scratch_limit(void) { return kStaticScratchBytes; }

int k2t_spmv_noalloc(k2t_tree *t, int32_t dir, int32_t semiring, float w, const void *x, void *y, uint32_t B,
                     void *stream)
{
    if (!t) return K2T_EINVAL;
    if (!t->dev) return K2T_ESTATE;
    if (t->engine != K2T_ENGINE_LEVELSYNC) return K2T_ESTATE;
    if (dir != K2T_RIGHT && dir != K2T_LEFT) return K2T_EINVAL;
    if (semiring < K2T_PLUS_TIMES || semiring > K2T_MIN_PLUS) return K2T_EINVAL;
    if (!x || !y || B == 0) return K2T_EINVAL;
    if (B > K2T_MAX_BATCH) return K2T_ERANGE;
    if (semiring == K2T_PLUS_TIMES && t->dev->hdir[dir] && B > t->opts.max_batch) return K2T_ERANGE;
    if (((uintptr_t)x | (uintptr_t)y) & 3u) return K2T_EINVAL;
    const uint64_t n_in = dir == K2T_RIGHT ? t->n_cols : t->n_rows;
    const uint64_t n_out = dir == K2T_RIGHT ? t->n_rows : t->n_cols;
    const uint64_t esz = semiring == K2T_BOOLEAN ? 4u : 4u * (uint64_t)B;
    const uintptr_t xa = (uintptr_t)x, ya = (uintptr_t)y;
    if (xa < ya + n_out * esz && ya < xa + n_in * esz) return K2T_EINVAL;
    // the array used must be the one on the tree's device
    int cur = -1;
    cudaError_t ce = cudaGetDevice(&cur);
    if (ce != cudaSuccess) { g_last_cuda = (int)ce; return K2T_ECUDA; }
    if (cur != t->dev->device) return K2T_ESTATE;

    // scratch this tree needs: one frontier buffer per expanded level, plus
    // the scan space when offsets come from a scan
    const ArenaLayout &L = t->layout;
    const int l = t->levels;
    uint64_t need = 0;
    LsBufs sb{};
    sb.buf_entries = L.buf_bytes / sizeof(Coord);
    void *base = nullptr;
    int rc = static_scratch(cur, &base);
    if (rc) return rc;
    uint8_t *p = static_cast<uint8_t *>(base);
    for (int lv = t->d0 + 1; lv <= l - 2; ++lv) {
        if (!t->empty) sb.buf[lv] = reinterpret_cast<Coord *>(p + need);
        need += align_up(L.buf_bytes, kArenaAlign);
    }
    if (L.scan_bytes) {
        sb.sums = reinterpret_cast<uint32_t *>(p + need);
        sb.prefix = sb.sums + L.scan_bytes / 8;
        need += align_up(L.scan_bytes, kArenaAlign);
    }
    if (need > kStaticScratchBytes) return K2T_ERANGE;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const uint64_t words = semiring == K2T_BOOLEAN ? n_out : n_out * (uint64_t)B;
    const uint32_t pattern = semiring == K2T_MIN_PLUS ? 0x7f800000u : 0u;
    if (words) {
        uint64_t blocks = (words / 4 + 255) / 256 + 1;
        if (blocks > 152ull * 16) blocks = 152ull * 16;
        fill_kernel<<<(unsigned)blocks, 256, 0, st>>>(static_cast<uint32_t *>(y), words, pattern);
    }
    if (!t->empty) {
        int vw = 1;
        if (semiring != K2T_BOOLEAN) {
            const uintptr_t al = xa | ya;
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
        va.status = t->dev->err;
        va.n_in = n_in;
        const bool heavy = heavy_begin(t, t->dev, dir, semiring, va, st);
        pick_static(semiring, dir, vw)(t, t->dev, sb, va, st);
        if (heavy) heavy_end(t, t->dev, dir, va, st);
    }
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { g_last_cuda = (int)e; return K2T_ECUDA; }
    return K2T_OK;
}

}  // extern "C"
