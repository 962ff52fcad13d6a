// pkv_blocks.cu — whole-block copies: inside the pool for copy-on-write ("The
// inference engine" (wpnews), "Paging turns variable sequences into block
// tables": copy-on-write restores separate ownership when a branch
// diverges), and between the pool and page-locked host memory for swapping a
// preempted sequence out and back in ("continuous batching server"
// (scalablesystem), "Preemption and Eviction: Recompute vs Swap").
//
// A block is every layer's K and V of 16 token positions (block_bytes, a
// multiple of 16). One launch moves a batch of blocks: grid.y walks the list,
// grid.x splits each block into 16-byte chunks, four independent 16-byte
// loads in flight per thread. The host side of a swap is read or written in
// place through its device-visible address (NVLink-C2C on Grace), so a batch
// of scattered pool blocks goes to one contiguous host buffer in one launch.
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 4;

__device__ __forceinline__ void copy_chunks(const uint4* __restrict__ src, uint4* __restrict__ dst, int64_t n16)
{
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    int64_t j = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; j + (kCopyUnroll - 1) * stride < n16; j += kCopyUnroll * stride) {
        uint4 v[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) v[u] = src[j + u * stride];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) dst[j + u * stride] = v[u];
    }
    for (; j < n16; j += stride) dst[j] = src[j];
}

// Pair i = (src block, dst block). Pairs whose blocks fall outside the pool are skipped and flagged.
__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(char* pool, int64_t block_bytes,
                                                                   const int32_t* __restrict__ pairs,
                                                                   int64_t num_blocks, int first,
                                                                   unsigned int* status)
{
    const int i = first + blockIdx.y;
    const int32_t s = __ldg(pairs + 2 * i), d = __ldg(pairs + 2 * i + 1);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, PKV_DEV_BAD_BLOCK);
        return;
    }
    copy_chunks(reinterpret_cast<const uint4*>(pool + (int64_t)s * block_bytes),
                reinterpret_cast<uint4*>(pool + (int64_t)d * block_bytes), block_bytes / 16);
}

// Block list entry i <-> host[i * block_bytes .. +block_bytes).
__global__ void __launch_bounds__(kCopyThreads) swap_blocks_kernel(char* pool, int64_t block_bytes,
                                                                   const int32_t* __restrict__ blocks,
                                                                   int64_t num_blocks, char* host, int to_host,
                                                                   int first, unsigned int* status)
{
    const int i = first + blockIdx.y;
    const int32_t b = __ldg(blocks + i);
    if (b < 0 || b >= num_blocks) {
        if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(status, PKV_DEV_BAD_BLOCK);
        return;
    }
    char* dev = pool + (int64_t)b * block_bytes;
    char* hst = host + (int64_t)i * block_bytes;
    if (to_host)
        copy_chunks(reinterpret_cast<const uint4*>(dev), reinterpret_cast<uint4*>(hst), block_bytes / 16);
    else
        copy_chunks(reinterpret_cast<const uint4*>(hst), reinterpret_cast<uint4*>(dev), block_bytes / 16);
}

// CTAs per block: enough for about four waves over the GPU in total, at most one per 4 KB.
int ctas_per_block(int n, int64_t block_bytes)
{
    int sms = 152;
    int dev = 0;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t want = ((int64_t)sms * 4 * 8 + n - 1) / n;  // 8 resident CTAs of 256 threads per SM
    const int64_t cap = std::max<int64_t>(1, block_bytes / 4096);
    return (int)std::max<int64_t>(1, std::min(want, cap));
}

constexpr int kMaxGridY = 65535;

}  // namespace

cudaError_t launch_copy_blocks(const PoolGeom& g, const int32_t* pairs, int n, unsigned int* status,
                               cudaStream_t stream)
{
    const int gx = ctas_per_block(n, g.block_bytes);
    for (int first = 0; first < n; first += kMaxGridY) {
        const int m = std::min(kMaxGridY, n - first);
        copy_blocks_kernel<<<dim3(gx, m), kCopyThreads, 0, stream>>>(const_cast<char*>(g.base), g.block_bytes, pairs,
                                                                      g.num_blocks, first, status);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_swap_blocks(const PoolGeom& g, const int32_t* blocks, int n, void* host, bool to_host,
                               unsigned int* status, cudaStream_t stream)
{
    const int gx = ctas_per_block(n, g.block_bytes);
    for (int first = 0; first < n; first += kMaxGridY) {
        const int m = std::min(kMaxGridY, n - first);
        swap_blocks_kernel<<<dim3(gx, m), kCopyThreads, 0, stream>>>(const_cast<char*>(g.base), g.block_bytes, blocks,
                                                                      g.num_blocks, static_cast<char*>(host),
                                                                      to_host ? 1 : 0, first, status);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace pkv
