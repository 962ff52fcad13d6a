// pkv_internal.h — shared between libpkv's host code and its kernel launchers.
#pragma once
#include <cstdint>
#include <string>
#include <unordered_map>
#include <vector>

#include <cuda_runtime.h>

#include "pkv.h"

namespace pkv {

constexpr int kHeadDim = 128;
constexpr int kBlockSize = 16;
constexpr int kTileBytes = kBlockSize * kHeadDim * 2;  // one head of one block: 4,096 B
// 8-bit pools: a tile is the 16 x 128 INT8 codes followed by 16 FP32 scales (one per token row).
constexpr int kTileBytesI8 = kBlockSize * kHeadDim + 4 * kBlockSize;  // 2,112 B
// Decode split-K partition: large enough that a CTA's start-up (metadata loads,
// first copies) is a small part of its life, small enough that long rows still
// spread over the GPU. Measured on the batch-32 decode workloads (1,024 beat
// 512, 768 and 1,536 on 4 of 5 length draws).
constexpr int kDefaultPartition = 1024;
constexpr int kMaxPartition = 2048;         // pools whose decode is the one-head kernel (block ids in its lanes)
constexpr int kMaxPartitionTiles = 4096;    // grouped-head and 8-bit pools (block ids in shared memory)
constexpr int kMaxPartitionsPerRow = 4096;  // the decode kernel merges at most this many partitions of a row

struct Seq {
    std::vector<int32_t> table;
    int64_t len = 0;
    bool swapped = false;  // blocks given back; the contents live in a caller's host buffer
};

// One prefix-cache entry: the block holding a full block of tokens whose chained hash is the key.
struct CacheEntry {
    int32_t block;
    uint64_t last_use;
    int64_t depth;  // position of the block in its chain
};

// Geometry of the device pool in bytes, for the kernels.
struct PoolGeom {
    const char* base;
    int64_t num_blocks;
    int32_t num_layers;
    int32_t num_heads;    // K/V heads stored per layer
    int32_t num_q_heads;  // query heads (a multiple of num_heads)
    int32_t group;        // num_q_heads / num_heads: query head h reads K/V head h / group
    int32_t dtype;        // PKV_DTYPE_FP16 or PKV_DTYPE_INT8
    int64_t tile_bytes;   // one (block, layer, K/V, head) tile: kTileBytes or kTileBytesI8
    int64_t block_bytes;  // one block, all layers: L * 2 * H * tile_bytes
    int64_t layer_bytes;  // one layer of one block: 2 * H * tile_bytes
    int64_t kv_bytes;     // K half to V half: H * tile_bytes
};

// Split-K scratch of one decode launch, carved from the caller's workspace.
struct DecodeWs {
    float* o;                // [B][num_q_heads][parts][128] un-normalised partial outputs
    float* ml;               // [B][num_q_heads][parts][2] partial max and sum
    unsigned int* counters;  // [B][num_q_heads] arrival counters, zero between launches
    int parts;               // partial slots per (row, query head)
};

struct alignas(64) TensorMap128 {
    alignas(64) unsigned char bytes[128];
};

}  // namespace pkv

struct pkv_pool {
    pkv_pool_desc desc;
    int device = 0;
    bool host_only = false;  // created without device memory: block manager only
    int partition_tokens = pkv::kDefaultPartition;
    unsigned int* status_dev = nullptr;  // sticky device error word of this device
    pkv::PoolGeom geom{};
    pkv::TensorMap128 kv_tmap{};  // 5-D TMA map over the pool (prefill K/V tiles)
    bool kv_tmap_ok = false;
    pkv::TensorMap128 tile_tmap{};  // decode map: a whole 4 KB FP16 tile (grouped decode) or an 8-bit tile's codes
    bool tile_tmap_ok = false;
    std::vector<int32_t> ref;
    std::vector<int32_t> free_stack;  // back() is handed out next
    std::unordered_map<int64_t, pkv::Seq> seqs;
    std::unordered_map<uint64_t, pkv::CacheEntry> cache;  // prefix cache: chained hash -> block
    std::vector<char> cached;                              // [num_blocks] block is in the cache
    uint64_t clock = 0;
};

namespace pkv {

pkv_status fail(pkv_status s, const char* fmt, ...);
pkv_status cuda_fail(cudaError_t e, const char* what);

// pkv_kernels.cu
cudaError_t status_word(int device, unsigned int** out);
cudaError_t launch_kv_append(const PoolGeom& g, int layer, const void* k, const void* v, const int64_t* slots,
                             int num_tokens, unsigned int* status, cudaStream_t stream);
int decode_max_parts(int max_blocks, int partition_tokens);
// extra_parts: partial slots beyond the plain plan's (cascade decode needs one more per row).
size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int max_blocks, int partition_tokens,
                              int extra_parts = 0);
DecodeWs decode_ws(const PoolGeom& g, void* ws, int num_seqs, int max_blocks, int partition_tokens,
                   int extra_parts = 0);
// Zero the split-K counters of a decode workspace (they return to zero after every
// completed launch; this covers the first use and any launch that stopped early).
cudaError_t clear_decode_counters(const PoolGeom& g, int num_seqs, int max_blocks, int partition_tokens, void* ws,
                                  cudaStream_t stream, int extra_parts = 0);
// k_new/v_new/slots non-NULL: the decode rows' kv_append is done by the same kernel.
// group_start/group_blocks (num_groups > 0): skip each row's partitions inside its group's shared prefix
// (launch_decode_shared_prefix computed them).
cudaError_t launch_decode(const PoolGeom& g, int layer, const void* q, const int32_t* tables, int max_blocks,
                          const int32_t* ctx_lens, int num_seqs, float scale, void* out, const DecodeWs& ws,
                          int partition_tokens, const void* k_new, const void* v_new, const int64_t* slots,
                          unsigned int* status, cudaStream_t stream, const int32_t* group_start = nullptr,
                          const int32_t* group_blocks = nullptr, int num_groups = 0, int pdl = 0);
// pdl: 1 = launched with a programmatic dependency on the stream's previous kernel (the previous layer's
// decode in a decode-only pkv_step): its CTAs load lengths, tables and K/V tiles, then wait for that kernel;
// 2 = the same launch without the wait (after a kernel whose results it does not read: the prefill launch of
// a mixed pkv_step layer), so its CTAs run beside that kernel's.

// pkv_int8.cu: the 8-bit cache (quantising kv_append; decode that dequantises in its loaders).
cudaError_t launch_kv_append_i8(const PoolGeom& g, int layer, const void* k, const void* v, const int64_t* slots,
                                int num_tokens, unsigned int* status, cudaStream_t stream);
bool encode_i8_tmap(const PoolGeom& g, TensorMap128* out, std::string* err);
cudaError_t launch_decode_i8(const PoolGeom& g, const TensorMap128& i8_tmap, int layer, const void* q,
                             const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                             float scale, void* out, const DecodeWs& ws, int partition_tokens, const void* k_new,
                             const void* v_new, const int64_t* slots, unsigned int* status, cudaStream_t stream,
                             int pdl = 0, const int32_t* group_start = nullptr,
                             const int32_t* group_blocks = nullptr, int num_groups = 0);
// Cascade over an 8-bit pool: the partitions wholly inside each group's shared prefix, for every row of the
// group at once (merging, as launch_decode_shared_prefix, the rows whose partials it completes).
cudaError_t launch_decode_i8_shared_prefix(const PoolGeom& g, const TensorMap128& i8_tmap, int layer, const void* q,
                                           const int32_t* tables, int max_blocks, const int32_t* ctx_lens,
                                           const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                                           int max_group_rows, float scale, void* out, const DecodeWs& ws,
                                           int partition_tokens, unsigned int* status, cudaStream_t stream);

// pkv_decode_group.cu: decode attention for pools whose K/V heads serve groups of query heads.
bool encode_tile_tmap(const PoolGeom& g, TensorMap128* out, std::string* err);
int decode_group_slices(int group);
// Cascade: the partitions wholly inside each group's shared prefix, for every row of the group at once. The
// private keys' launch may run beside it (launched with pdl = 2): whichever partial of a row arrives last merges
// the row into out, so both launches know every row's partition plan (ctx_lens).
cudaError_t launch_decode_shared_prefix(const PoolGeom& g, const TensorMap128& kv_tmap, int layer, const void* q,
                                        const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                                        const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                                        int max_group_rows, float scale, void* out, const DecodeWs& ws,
                                        int partition_tokens, unsigned int* status, cudaStream_t stream);
// group_start/group_blocks (num_groups > 0): skip each row's keys inside its group's shared prefix
// (launch_decode_shared_prefix computed them).
cudaError_t launch_decode_group(const PoolGeom& g, const TensorMap128& kv_tmap, int layer, const void* q,
                                const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                                float scale, void* out, const DecodeWs& ws, int partition_tokens, const void* k_new,
                                const void* v_new, const int64_t* slots, unsigned int* status, cudaStream_t stream,
                                int pdl = 0, const int32_t* group_start = nullptr,
                                const int32_t* group_blocks = nullptr, int num_groups = 0);
// pkv_blocks.cu: whole-block copies inside the pool (copy-on-write) and to / from host memory (swap).
cudaError_t launch_copy_blocks(const PoolGeom& g, const int32_t* pairs, int n, unsigned int* status,
                               cudaStream_t stream);
cudaError_t launch_swap_blocks(const PoolGeom& g, const int32_t* blocks, int n, void* host, bool to_host,
                               unsigned int* status, cudaStream_t stream);

cudaError_t launch_wait_probe(uint64_t timeout_ns, unsigned int* status, cudaStream_t stream);

// pkv_prefill.cu
bool encode_kv_tmap(const PoolGeom& g, TensorMap128* out, std::string* err);
cudaError_t launch_prefill(const pkv_pool* pool, int layer, const void* q, const int32_t* q_start,
                           const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                           int max_q_len, float scale, void* out, cudaStream_t stream);

}  // namespace pkv
