// pkv_prefill.cu — chunked causal prefill attention over the paged pool.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <string>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

// 5-D TMA map over the pool for 2 KB boxes of one (block, layer, K|V, head)
// tile's 64-dim half: dims innermost first are
//   d (128), t (16, 256 B), K|V*H + head (2H, 4 KB), layer (L), block (N).
bool encode_kv_tmap(const PoolGeom& g, TensorMap128* out, std::string* err)
{
    static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
    if (!encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || !fn) {
            if (err) *err = "cuTensorMapEncodeTiled unavailable";
            return false;
        }
        encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    const cuuint64_t dims[5] = {(cuuint64_t)kHeadDim, (cuuint64_t)kBlockSize, (cuuint64_t)(2 * g.num_heads),
                                (cuuint64_t)g.num_layers, (cuuint64_t)g.num_blocks};
    const cuuint64_t strides[4] = {(cuuint64_t)kHeadDim * 2, (cuuint64_t)kTileBytes, (cuuint64_t)g.layer_bytes,
                                   (cuuint64_t)g.block_bytes};
    const cuuint32_t box[5] = {64, (cuuint32_t)kBlockSize, 1, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encode(reinterpret_cast<CUtensorMap*>(out->bytes), CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 5,
                        const_cast<char*>(g.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (err) *err = "cuTensorMapEncodeTiled failed";
        return false;
    }
    return true;
}

cudaError_t launch_prefill(const pkv_pool*, int, const void*, const int32_t*, const int32_t*, int, const int32_t*, int,
                           int, float, void*, cudaStream_t)
{
    return cudaErrorNotSupported;
}

}  // namespace pkv
