// k2t_probe.cu -- memory-system ceilings for the access patterns of the leaf
// step, measured on the device the library runs on: instrumentation for the
// benchmark, built into its own libk2t_probe.so, outside the product
// library and its ABI (the microbenchmark of
// section 5.6 of "A GPU Engine for Sparse Matrix-Vector Products on
// k^2-Tree-Compressed Graphs": copy bandwidth and the rates of consecutive and
// scattered vector updates y_o += x_i, re-measured here with gathers added).
// Scattered indices come from a multiplicative hash of the operation index,
// so no index array is read.
#include <cuda_runtime.h>

#include <cstdint>

#include "../../../include/k2t.h"

namespace {

__device__ __forceinline__ uint64_t scramble(uint64_t i)
{
    i ^= i >> 31;
    i *= 0x9e3779b97f4a7c15ull;
    i ^= i >> 29;
    return i;
}

// y[i] = x[i] for n floats, float4 wide
__global__ void probe_copy(const float4 *x, float4 *y, uint64_t n4)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += stride) y[i] = x[i];
}

// m gathers x[h(i) mod n] (n a power of two); one write per thread keeps them live
__global__ void probe_gather(const float *x, float *y, uint64_t mask, uint64_t m, uint32_t pairs)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    const uint64_t t = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x;
    float acc = 0.0f;
    if (pairs) {
        for (uint64_t i = t; i < m; i += stride) {
            const float2 v = __ldg(reinterpret_cast<const float2 *>(x + (scramble(i) & mask & ~1ull)));
            acc += v.x + v.y;
        }
    } else {
        for (uint64_t i = t; i < m; i += stride) acc += __ldg(x + (scramble(i) & mask));
    }
    if (acc == 1.2345f) y[t & mask] = acc;
}

// m reductions y[o(i)] += 1, o(i) = i mod n (consecutive) or h(i) mod n (scattered)
__global__ void probe_red(float *y, uint64_t mask, uint64_t m, uint32_t scattered)
{
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < m; i += stride)
        atomicAdd(y + ((scattered ? scramble(i) : i) & mask), 1.0f);
}

// m shared-memory reductions per grid into a 2048-entry table per block, at
// hashed slots: fp32 (kind 5) or fp64 (kind 6) atomicAdd; the table is
// added to y once per block so the work stays live
template <class T>
__global__ void probe_smem_red(float *y, uint64_t m)
{
    __shared__ T tab[2048];
    for (uint32_t i = threadIdx.x; i < 2048; i += blockDim.x) tab[i] = (T)0;
    __syncthreads();
    const uint64_t stride = (uint64_t)gridDim.x * blockDim.x;
    for (uint64_t i = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; i < m; i += stride)
        atomicAdd(&tab[scramble(i) & 2047u], (T)1);
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(y + (blockIdx.x & 1023u), (float)tab[blockIdx.x & 2047u]);
}

}  // namespace

extern "C" {

K2T_API int k2t_probe(int32_t kind, const void *x, void *y, uint64_t n, uint64_t m, void *stream);

/* Launch one probe pass on `stream` (the caller times it):
 *   kind 0: copy n floats x -> y (n a multiple of 4)
 *   kind 1: m scattered 4-byte gathers from x[0..n)
 *   kind 2: m scattered 8-byte gathers (pairs) from x[0..n)
 *   kind 3: m consecutive reductions y[i mod n] += 1
 *   kind 4: m scattered reductions y[h(i) mod n] += 1
 *   kind 5: m fp32 shared-memory reductions at hashed slots of a 2048-entry
 *           table per block (y: at least 1024 floats)
 *   kind 6: the same with fp64 shared-memory reductions
 * n must be a power of two for kinds 1-4.  Returns K2T_OK or K2T_EINVAL /
 * K2T_ECUDA. */
int k2t_probe(int32_t kind, const void *x, void *y, uint64_t n, uint64_t m, void *stream)
{
    if (!y || n == 0 || (kind <= 2 && !x)) return K2T_EINVAL;
    if (kind != 0 && (n & (n - 1))) return K2T_EINVAL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const unsigned grid = (unsigned)(sms * 8), block = 256;
    switch (kind) {
    case 0:
        if (n % 4) return K2T_EINVAL;
        probe_copy<<<grid, block, 0, st>>>(static_cast<const float4 *>(x), static_cast<float4 *>(y), n / 4);
        break;
    case 1:
    case 2:
        probe_gather<<<grid, block, 0, st>>>(static_cast<const float *>(x), static_cast<float *>(y), n - 1, m,
                                             kind == 2);
        break;
    case 3:
    case 4:
        probe_red<<<grid, block, 0, st>>>(static_cast<float *>(y), n - 1, m, kind == 4);
        break;
    case 5:
        if (n < 1024) return K2T_EINVAL;
        probe_smem_red<float><<<grid, block, 0, st>>>(static_cast<float *>(y), m);
        break;
    case 6:
        if (n < 1024) return K2T_EINVAL;
        probe_smem_red<double><<<grid, block, 0, st>>>(static_cast<float *>(y), m);
        break;
    default:
        return K2T_EINVAL;
    }
    return cudaGetLastError() == cudaSuccess ? K2T_OK : K2T_ECUDA;
}

}  // extern "C"
