// pkv_noalloc.cu — decode attention for callers that cannot allocate device
// memory. Its split-K scratch is a fixed array compiled into the library
// instead of a caller-provided workspace.
#include <cuda_runtime.h>

#include <atomic>

#include "pkv_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;  // 16 MiB per GPU, held until the process exits

// File-scope device array. In host code this name is only a stand-in: the
// device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
// Atomic so that two host threads making their first call on the same device at once do not race: both look
// the (same) address up and both store it.
std::atomic<void*> g_scratch_addr[kMaxDevices] = {};

// First call on a device: make it current and look the array's address up.
pkv_status scratch_for_device(int device, void** out)
{
    if (device < 0 || device >= kMaxDevices) return pkv::fail(PKV_E_INVALID, "device ordinal %d unsupported", device);
    void* cached = g_scratch_addr[device].load(std::memory_order_acquire);
    if (!cached) {
        int prev = -1;
        cudaError_t e = cudaGetDevice(&prev);
        if (e != cudaSuccess) return pkv::cuda_fail(e, "cudaGetDevice");
        if (prev != device && (e = cudaSetDevice(device)) != cudaSuccess) return pkv::cuda_fail(e, "cudaSetDevice");
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (prev != device) cudaSetDevice(prev);
        if (e != cudaSuccess || !p) return pkv::cuda_fail(e, "cudaGetSymbolAddress(decode scratch)");
        g_scratch_addr[device].store(p, std::memory_order_release);
        cached = p;
    }
    *out = cached;
    return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_decode_attn_noalloc(pkv_pool* pool, int32_t layer, const void* q,
                                              const int32_t* block_tables, int32_t max_blocks,
                                              const int32_t* ctx_lens, int32_t num_seqs, float scale, void* out,
                                              void* stream)
{
    if (!pool) return pkv::fail(PKV_E_INVALID, "pool is NULL");
    if (pool->host_only) return pkv::fail(PKV_E_INVALID, "pool has no device memory (host-only block manager)");
    if (num_seqs < 0 || max_blocks < 1) return pkv::fail(PKV_E_INVALID, "num_seqs < 0 or max_blocks < 1");
    const size_t need = pkv_decode_workspace_bytes(pool, num_seqs, max_blocks);
    if (need > kScratchBytes)
        return pkv::fail(PKV_E_INVALID,
                         "pkv_decode_attn_noalloc: %d rows with tables %d blocks wide need %zu bytes of scratch, "
                         "above the built-in %zu; use pkv_decode_attn with a workspace",
                         num_seqs, max_blocks, need, kScratchBytes);
    void* scratch = nullptr;
    if (pkv_status s = scratch_for_device(pool->device, &scratch)) return s;
    // pkv_decode_attn clears the scratch's per-(row, head) arrival counters on the stream (a memset, no
    // allocation) before its kernel; the partial outputs are written before they are read.
    return pkv_decode_attn(pool, layer, q, block_tables, max_blocks, ctx_lens, num_seqs, scale, out, scratch,
                           kScratchBytes, stream);
}
