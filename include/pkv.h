/*
 * pkv.h — C ABI of libpkv: a paged KV cache on one GB300 (sm_103a).
 *
 * The cache is one device allocation of FP16 blocks. A block holds the keys
 * and values of 16 token positions for every layer, laid out as
 *     [layer][2 (0 = K, 1 = V)][head][16 tokens][head_dim]
 * so element (block b, layer l, kv, head h, token t, dim d) sits at
 *     ((((b*L + l)*2 + kv)*H + h)*16 + t)*head_dim + d
 * ("llm-inference-batching" (faangrind), the KV pool listing; 524,288 B per
 * token and 8,388,608 B per block for 32 layers x 32 heads x 128 dims).
 * A sequence's block table maps its logical block i (positions 16i..16i+15)
 * to a physical block; position p lives at slot table[p/16]*16 + p%16
 * (same page, "block_table"; "continuous batching server" (scalablesystem),
 * "PagedAttention Block Table Lookup").
 *
 * Conventions for every call:
 *   - Ownership: the caller owns every device buffer (pool, q/k/v, tables,
 *     outputs, workspace); pointers are borrowed for the duration of the
 *     call. The library owns only the opaque pkv_pool host handle.
 *   - Asynchrony: kernel calls enqueue work on `stream` (a cudaStream_t,
 *     NULL = legacy default stream) and return without synchronising.
 *   - Errors: every call returns a pkv_status. Bad arguments are refused on
 *     the host before anything is launched (PKV_E_INVALID, with a message in
 *     pkv_last_error_string()). Inputs that live on the device (tables,
 *     lengths, slots) are bounds-checked by the kernels: a bad entry skips
 *     the access and sets a sticky per-device error word that
 *     pkv_get_status() reads. No C++ exception crosses this boundary.
 *   - Threads: a pool is not thread-safe; one scheduler thread owns it
 *     ("llm-inference-batching", step 3: one scheduler thread owns the GPU).
 *   - Supported geometry: head_dim 128, block_size 16, FP16 or 8-bit
 *     (PKV_DTYPE_INT8) elements, any number of layers (1..1024) and K/V heads
 *     (1..256). num_q_heads is a multiple of the K/V heads (grouped-query
 *     and multi-query attention: query head h reads K/V head
 *     h / (num_q_heads / num_heads)), at most 1,024.
 */
#ifndef PKV_H
#define PKV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pkv_status {
    PKV_OK = 0,
    PKV_E_INVALID = 1,  /* bad argument, refused before launch */
    PKV_E_NOMEM = 2,    /* free list cannot cover the request; nothing changed (caller preempts) */
    PKV_E_SHARED = 3,   /* a new token would be written into a block whose ref_count > 1 */
    PKV_E_DEVICE = 4,   /* CUDA error, or a kernel found a bad table entry / slot / length */
    PKV_E_TIMEOUT = 5   /* a kernel's bounded wait ran out; the kernel returned early */
} pkv_status;

/* Element types of a pool. PKV_DTYPE_INT8 is the 8-bit cache ("Inference
 * Infrastructure" (seeitflow), the KV cache arithmetic: 8 bits per element
 * halve the cache): each (block, layer, K/V, head) tile holds the 16 x 128
 * INT8 codes, token-major, then 16 FP32 scales, one per token row (2,112 B
 * instead of 4,096). Rule: scale = max|x| / 127 over the row's 128 FP16
 * values, code = round-half-even(x / scale) clamped to +-127, both in IEEE
 * single precision; attention reads code * scale. kv_append quantises,
 * decode attention dequantises in its loaders (tensor cores: codes become
 * FP16 exactly, the K scale multiplies the scores, the V scale folds into the
 * softmax weights, which are rounded to FP16). Prefill attention does the
 * same: each 128-key tile's codes arrive by TMA and become exact FP16 codes
 * in shared memory for the tensor cores; the row scales arrive beside them
 * and are applied in FP32 in the softmax (K scales to the scores, V scales to
 * the weights before their rounding to FP16), never to the operands. */
enum { PKV_DTYPE_FP16 = 0, PKV_DTYPE_INT8 = 1 };

/* Bits of the sticky device error word (pkv_get_status). */
enum {
    PKV_DEV_BAD_SLOT = 1u << 0,   /* kv_append: slot outside [0, num_blocks*16) */
    PKV_DEV_BAD_BLOCK = 1u << 1,  /* attention: block id outside [0, num_blocks) */
    PKV_DEV_BAD_CTX = 1u << 2,    /* attention: ctx_len < 1 or beyond the table width */
    PKV_DEV_BAD_QLEN = 1u << 3,   /* prefill: q_len < 1, > ctx_len, or beyond max_q_len */
    PKV_DEV_TIMEOUT = 1u << 4     /* a bounded wait on an mbarrier ran out */
};

/* ------------------------------------------------------------------ pool */

typedef struct pkv_pool_desc {
    int64_t num_blocks;   /* physical blocks in the pool (7,152 for a 60 GB pool) */
    int32_t num_layers;   /* 32 */
    int32_t num_heads;    /* K/V heads stored per layer: 32 for the MHA model, 8 for GQA */
    int32_t head_dim;     /* must be 128 */
    int32_t block_size;   /* must be 16 */
    int32_t dtype;        /* PKV_DTYPE_FP16 or PKV_DTYPE_INT8 */
    int32_t partition_tokens; /* decode split-K partition size in tokens; 0 = default 1024;
                                 a multiple of 64 in [64, 2048] for FP16 pools with one query
                                 head per K/V head, in [64, 4096] for grouped-head and 8-bit
                                 pools. Results depend only on a row's ctx_len and this value,
                                 never on the rest of the batch. */
    void* dev_base;       /* device pointer to the pool, 256-byte aligned; NULL makes a host-only
                             pool (block manager and step metadata only; kernel calls refused) */
    size_t bytes;         /* size of that allocation, >= pkv_pool_bytes(desc) */
    const int64_t* free_order; /* optional host array [num_blocks], a permutation: the order in
                                  which blocks are handed out. NULL = 0, 1, 2, ... */
    int32_t num_q_heads;  /* query heads; 0 = num_heads (MHA). A multiple of num_heads, at most
                             1,024: each K/V head serves G = num_q_heads / num_heads consecutive
                             query heads, query head h reading K/V head h / G (grouped-query
                             attention, "Inference Infrastructure" (seeitflow), the KV cache
                             arithmetic: 8 K/V heads, 131,072 B per token over 32 layers;
                             num_heads = 1 is multi-query attention). q and out of the attention
                             calls are [.., num_q_heads, 128]; k, v and the pool hold num_heads. */
} pkv_pool_desc;

typedef struct pkv_pool pkv_pool;

/* Bytes the pool needs: num_blocks * num_layers * 2 * num_heads * tile, tile =
 * block_size * head_dim * 2 = 4,096 B for FP16 ("llm-inference-batching", "KV
 * cache": 8,388,608 B per block for the 7B model) or 2,112 B for INT8.
 * Returns 0 for an invalid descriptor. */
size_t pkv_pool_bytes(const pkv_pool_desc* desc);

/* Validate desc, bind the pool to the current CUDA device and build its host handle.
 * The device memory is not touched. *out receives the handle. With dev_base NULL
 * no CUDA call is made and the handle serves the block manager only. */
pkv_status pkv_pool_create(const pkv_pool_desc* desc, pkv_pool** out);
pkv_status pkv_pool_destroy(pkv_pool* pool);

/* ---------------------------------------------------- block manager (host) */
/* A ref-counted allocator over the pool's blocks: a free list, one block
 * table per sequence and ref_count[block] ("llm-inference-batching", the KV
 * pool listing; "continuous batching server", "The KV Cache Block Manager";
 * "Serving LLMs" (sreshtalluri), "Paged KV memory"). Host only; no GPU work. */

/* Make seq_id (created on first use) own ceil(new_len/16) blocks and set its
 * length to new_len. New blocks come off the free list with ref_count 1.
 * PKV_E_NOMEM if the free list cannot cover it (nothing changes: the caller
 * preempts); PKV_E_INVALID if new_len is below the current length. */
pkv_status pkv_seq_grow(pkv_pool* pool, int64_t seq_id, int64_t new_len);

/* Point a new sequence dst_seq at the first n_blocks (full) blocks of src_seq
 * and raise their ref_count; dst's length becomes 16*n_blocks. Shared blocks
 * are read-only: a later write into one is refused with PKV_E_SHARED. */
pkv_status pkv_seq_share_prefix(pkv_pool* pool, int64_t dst_seq, int64_t src_seq, int64_t n_blocks);

/* Finished or cancelled sequence: drop one reference to each of its blocks;
 * a block whose ref_count reaches 0 returns to the free list. */
pkv_status pkv_seq_free(pkv_pool* pool, int64_t seq_id);

int64_t pkv_free_blocks(const pkv_pool* pool);                 /* -1 for a NULL pool */
int32_t pkv_ref_count(const pkv_pool* pool, int64_t block);     /* -1 if out of range */
int64_t pkv_seq_len(const pkv_pool* pool, int64_t seq_id);      /* -1 if unknown */

/* ------------------------------------------ copy-on-write, swap, prefix cache */

/* Parallel sampling: a new sequence dst_seq shares every block of src_seq,
 * the partly filled last block included (ref_count + 1 each), with src's
 * length ("The inference engine" (wpnews), "Paging turns variable sequences
 * into block tables": copy-on-write sharing for parallel sampling). */
pkv_status pkv_seq_fork(pkv_pool* pool, int64_t dst_seq, int64_t src_seq);

/* Copy-on-write ("The inference engine" (wpnews), "Paging turns variable
 * sequences into block tables": a branch that diverges gets its own copy).
 * Call after pkv_seq_grow and before the step that writes seq_id's last
 * num_new positions [len - num_new, len) (num_new = the row's q_len in
 * pkv_build_step). If a block holding one of those positions is also named
 * by another table (ref_count > 1), the first such block in table order is
 * replaced in seq_id's table by a free block (old ref_count - 1, new 1) and
 * *src_block / *dst_block name the copy the caller must make on the device
 * (pkv_copy_blocks: every layer) before the step; otherwise both are -1 and
 * nothing changes. One call handles one block: call again until it returns
 * -1 (after a fork only the partly filled last block is shared, so one call
 * suffices). Afterwards pkv_build_step does not refuse the row with
 * PKV_E_SHARED. PKV_E_NOMEM (nothing changes) if no block is free;
 * PKV_E_INVALID if num_new is negative or above the length. */
pkv_status pkv_seq_cow(pkv_pool* pool, int64_t seq_id, int64_t num_new, int32_t* src_block, int32_t* dst_block);

/* Preemption by swap ("continuous batching server", "Preemption and Eviction:
 * Recompute vs Swap"; the choice of victim and of swap over recompute is the
 * caller's). pkv_seq_swap_out writes seq_id's blocks (table order) to
 * blocks[0..*n_blocks) and releases them (ref_count - 1, free at 0); the
 * sequence keeps its length but has no blocks until pkv_seq_swap_in, which
 * takes ceil(len/16) fresh blocks off the free list (PKV_E_NOMEM: nothing
 * changes) and writes them to blocks. The caller moves the contents with
 * pkv_swap_blocks_out before anything else writes the released blocks (same
 * stream) and with pkv_swap_blocks_in before the sequence's next step. If
 * capacity < *n_blocks the call fails with PKV_E_INVALID, nothing changes,
 * and *n_blocks says how many are needed. A swapped-out sequence can only be
 * swapped in or freed. */
pkv_status pkv_seq_swap_out(pkv_pool* pool, int64_t seq_id, int32_t* blocks, int64_t capacity, int64_t* n_blocks);
pkv_status pkv_seq_swap_in(pkv_pool* pool, int64_t seq_id, int32_t* blocks, int64_t capacity, int64_t* n_blocks);

/* Chained prefix hashes of a token-id stream ("Serving LLMs" (sreshtalluri),
 * "Prefix caching": a block's hash covers the block and, through the chain,
 * every token before it). out[i] = FNV-1a-64 over the 8 little-endian bytes
 * of out[i-1] (0 for i = 0) followed by the 16 token ids of block i (4
 * little-endian bytes each). Only full blocks are hashed: returns
 * n_tokens / 16 (written to out, capacity >= that), -1 on a bad argument. */
int64_t pkv_block_hashes(const int32_t* tokens, int64_t n_tokens, uint64_t* out, int64_t capacity);

/* The pool's prefix cache: chained hash -> block. The cache holds one
 * reference to each cached block, so it outlives the sequences using it.
 *   pkv_prefix_register: cache seq_id's first n_hashes full blocks under
 *     hashes[0..n_hashes) (the hashes of its tokens); a hash already cached
 *     keeps its block, a block already cached under another hash is left out;
 *     *n_new = blocks added.
 *   pkv_prefix_match: the number of leading hashes that are cached (the walk
 *     stops at the first miss); -1 on a bad argument.
 *   pkv_seq_attach_prefix: create seq_id on the blocks of its longest cached
 *     prefix (ref_count + 1 each, length 16 * *n_attached); the caller then
 *     grows it and prefills only the rest of the prompt.
 *   pkv_prefix_evict: drop up to max_blocks entries whose block only the
 *     cache references, least recently used (registered or attached) first
 *     and, among equals, deeper chain positions first; those blocks return to
 *     the free list. Returns the number evicted, -1 on a bad argument. */
pkv_status pkv_prefix_register(pkv_pool* pool, int64_t seq_id, const uint64_t* hashes, int64_t n_hashes,
                               int64_t* n_new);
int64_t pkv_prefix_match(const pkv_pool* pool, const uint64_t* hashes, int64_t n_hashes);
pkv_status pkv_seq_attach_prefix(pkv_pool* pool, int64_t seq_id, const uint64_t* hashes, int64_t n_hashes,
                                 int64_t* n_attached);
int64_t pkv_prefix_evict(pkv_pool* pool, int64_t max_blocks);
int64_t pkv_prefix_cached_blocks(const pkv_pool* pool);        /* entries in the cache, -1 for a NULL pool */

/* Copy seq_id's block table (host int32) into out[0..capacity); *n_out = its length. */
pkv_status pkv_block_table(const pkv_pool* pool, int64_t seq_id, int32_t* out, int64_t capacity,
                           int64_t* n_out);

/* Host-side metadata for one engine iteration over the listed sequences
 * ("llm-inference-batching", the step tensors: one flat, unpadded token list
 * tagged with its request). Row i's new tokens are its last q_lens[i]
 * positions, i.e. [len - q_lens[i], len) after pkv_seq_grow. Sequences not
 * listed take no part (finished or cancelled rows leave at a step boundary).
 * Outputs (host arrays, caller-allocated):
 *   block_tables [num_seqs, max_blocks] int32, -1 past each row's blocks
 *   ctx_lens     [num_seqs]             int32, cached tokens incl. the new ones
 *   slot_mapping [sum q_lens]           int64, slot of each new token, row order
 *   q_start_loc  [num_seqs + 1]         int32, prefix sums of q_lens
 * PKV_E_SHARED if a new token falls in a block with ref_count > 1. */
pkv_status pkv_build_step(const pkv_pool* pool, const int64_t* seq_ids, const int32_t* q_lens, int32_t num_seqs,
                          int32_t max_blocks, int32_t* block_tables, int32_t* ctx_lens, int64_t* slot_mapping,
                          int32_t* q_start_loc);

/* ---------------------------------------------------------------- kernels */

/* reshape_and_cache: write token i's keys k[i] and values v[i] (device FP16,
 * [num_tokens, num_heads, 128], 16-byte aligned) of layer `layer` into slot
 * slot_mapping[i] (device int64) of the pool ("llm-inference-batching",
 * step 7: a row's new keys and values are appended; a row takes a new
 * block every 16 tokens). Slots must be distinct. A slot outside the pool is
 * skipped and flagged PKV_DEV_BAD_SLOT. */
pkv_status pkv_kv_append(pkv_pool* pool, int32_t layer, const void* k, const void* v,
                         const int64_t* slot_mapping, int32_t num_tokens, void* stream);

/* Workspace bytes pkv_decode_attn needs for num_seqs rows whose tables are
 * max_blocks wide (split-K partials: un-normalised output, max and sum per
 * row, head and partition). */
size_t pkv_decode_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t max_blocks);

/* Decode attention: for each row r and head h, the single query q[r,h,:]
 * attends positions 0..ctx_lens[r]-1 of row r's blocks, including the token
 * appended this step: out = softmax(q K^T * scale) V ("Inference
 * Infrastructure" (seeitflow), the decode steps). Long rows are split into
 * the fewest partitions of at most partition_tokens keys, of equal length in
 * whole blocks, whose softmax statistics are merged exactly ("The inference
 * engine" (wpnews), "IO-aware attention").
 *   q            device FP16 [num_seqs, num_q_heads, 128]
 *   block_tables device int32 [num_seqs, max_blocks]
 *   ctx_lens     device int32 [num_seqs], 1 <= ctx_len <= 16*max_blocks
 *   out          device FP16 [num_seqs, num_q_heads, 128], rounded once (RNE)
 *   workspace    device, >= pkv_decode_workspace_bytes(), 256-byte aligned
 * FP32 arithmetic; scale is applied in FP32 (1/sqrt(128) = 0x3DB504F3).
 * Pools with num_q_heads > num_heads: one CTA reads each K/V block once for
 * up to 16 query heads of its group and runs q K^T and P V on the tensor
 * cores (FP16 operands, P rounded to FP16, FP32 accumulation). */
pkv_status pkv_decode_attn(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                           int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs, float scale, void* out,
                           void* workspace, size_t workspace_bytes, void* stream);

/* Cascade decode for rows that share a prompt prefix ("The inference engine"
 * (wpnews), "Paging turns variable sequences into block tables": sequences
 * may point at the same immutable prefix blocks). Same inputs and result as
 * pkv_decode_attn (within the attention tolerance; the shared part runs on
 * the tensor cores with the softmax weights rounded to FP16), plus a grouping
 * of the rows: rows [group_start[i], group_start[i+1]) (device int32,
 * num_groups + 1 entries, group_start[num_groups] = num_seqs) share their first
 * group_blocks[i] table entries (device int32), which must be the same
 * physical blocks, full, and below every row's newest token. Every split-K
 * partition wholly inside a group's shared prefix is computed once for
 * several rows at a time (a CTA holds 16 query rows: 16 rows of one head over
 * a pool with one query head per K/V head, 4 rows of 4 query heads for G = 4,
 * one row's 16 heads from G = 16 up), so its K/V tiles are read from memory
 * once per group instead of once per row; the rest of each row runs as in
 * pkv_decode_attn. The two launches run side by side, and whichever
 * partial of a row arrives last merges the row's partials in partition
 * order, by the same arithmetic either way. max_group_rows = the largest
 * group. Every pool kind: FP16 with any G = num_q_heads / num_heads, and
 * 8-bit (codes dequantised as in pkv_decode_attn). No append: call
 * pkv_kv_append first. Partition plan: a row's shared prefix [0, S) is cut
 * into partitions of partition_tokens, the rest [S, ctx) as pkv_decode_attn
 * cuts a row (so a row can have one partition more than in pkv_decode_attn);
 * results are deterministic for a given grouping. The workspace must hold pkv_decode_cascade_workspace_bytes. */
pkv_status pkv_decode_attn_cascade(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                                   int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs,
                                   const int32_t* group_start, const int32_t* group_blocks, int32_t num_groups,
                                   int32_t max_group_rows, float scale, void* out, void* workspace,
                                   size_t workspace_bytes, void* stream);

size_t pkv_decode_cascade_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t max_blocks);

/* Host helper for the grouping: maximal runs of consecutive rows of host
 * block_tables [num_seqs, max_blocks] / ctx_lens that share leading blocks
 * (the first two rows' common prefix, limited to blocks wholly below each
 * row's newest token); runs shorter than min_rows become single rows with no
 * shared prefix. Writes group_start [num_groups + 1] and group_blocks
 * [num_groups] (host, capacity num_seqs + 1 and num_seqs). */
pkv_status pkv_cascade_groups(const int32_t* block_tables, const int32_t* ctx_lens, int32_t num_seqs,
                              int32_t max_blocks, int32_t min_rows, int32_t* group_start, int32_t* group_blocks,
                              int32_t* num_groups, int32_t* max_group_rows);

/* Chunked causal prefill: sequence s owns query tokens
 * [q_start_loc[s], q_start_loc[s+1]) of q ([num_tokens, num_q_heads, 128] FP16);
 * query i sits at position ctx_lens[s] - q_len + i and attends keys 0..that
 * position of s's blocks, which already hold the chunk's own K/V
 * ("llm-inference-batching", "Prefill and decode share each step"; "The
 * inference engine", "Prefill and decode ask the accelerator for different
 * work"). max_q_len bounds every q_len (it sizes the grid). Tensor cores
 * (tcgen05, accumulators in TMEM), FP32 accumulation, FP16 output. */
pkv_status pkv_prefill_attn(pkv_pool* pool, int32_t layer, const void* q, const int32_t* q_start_loc,
                            const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens,
                            int32_t num_seqs, int32_t max_q_len, float scale, void* out, void* stream);

/* Decode attention that allocates nothing. The source pages have no
 * counterpart; this is a convenience of the library.
 *
 * Same inputs, output and results as pkv_decode_attn, but the split-K
 * scratch is a 16 MiB array built into the library (one per GPU that loads
 * it, held until the process exits) instead of a caller workspace. It is for
 * callers that cannot call cudaMalloc on the decode path: a plug-in whose
 * host process owns all device memory through its own allocator, or a
 * serving loop that forbids cudaMalloc after start-up because the call can
 * synchronise the device and stall every stream.
 *
 *   - Limit: the scratch pkv_decode_workspace_bytes(pool, num_seqs,
 *     max_blocks) would report must fit in 16 MiB. That is about
 *     num_seqs x num_q_heads x P x 520 B <= 16 MiB with
 *     P = ceil(16 x max_blocks / partition_tokens), the pool's partition
 *     length (1,024 tokens by default): with 32 query heads, num_seqs x P
 *     <= ~1,000, e.g. 32 rows with tables up to 1,984 blocks at the default,
 *     or up to 992 blocks for a pool created with 512-token partitions.
 *     Larger requests are refused with PKV_E_INVALID and a message, before
 *     anything is launched.
 *   - The first call on a device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current) and keeps it for the
 *     rest of the process; make that first call before any stream capture.
 *     Do not use this entry point on a device after cudaDeviceReset (or any
 *     other reset of its primary context) in the same process: the kept
 *     address would be stale.
 *   - Every call on a device shares the one array and overwrites it. Calls
 *     whose kernels overlap on the GPU (other streams, other threads) race
 *     and give wrong results; serialise them. Each call clears the array's
 *     arrival counters on its stream (a memset, not an allocation) before its
 *     kernel. No cudaMalloc, cudaFree or allocating library routine is
 *     called. */
pkv_status pkv_decode_attn_noalloc(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                                   int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs, float scale,
                                   void* out, void* stream);

/* Whole-block copies on the device, asynchronous on `stream`.
 * pkv_copy_blocks: for i < n, block pairs[2i+1] receives a copy of block
 *   pairs[2i] (every layer, K and V: pkv_pool_bytes / num_blocks bytes);
 *   pairs is device int32 [n][2]. No block may be the destination of one pair
 *   and the source or destination of another (the pairs run concurrently).
 * pkv_swap_blocks_out: host_dst[i * block bytes ..] receives block blocks[i];
 * pkv_swap_blocks_in: block blocks[i] receives host_src[i * block bytes ..].
 *   blocks is device int32 [n]; the host buffer (n * block bytes, 16-byte
 *   aligned) must be page-locked host memory the device can address
 *   (cudaHostAlloc / cudaHostRegister; checked, PKV_E_INVALID otherwise). The
 *   kernel reads or writes it in place, so one launch gathers scattered pool
 *   blocks into one host buffer or scatters them back.
 * Block ids outside the pool are skipped and flagged (PKV_DEV_BAD_BLOCK). */
pkv_status pkv_copy_blocks(pkv_pool* pool, const int32_t* pairs, int32_t n, void* stream);
pkv_status pkv_swap_blocks_out(pkv_pool* pool, const int32_t* blocks, int32_t n, void* host_dst, void* stream);
pkv_status pkv_swap_blocks_in(pkv_pool* pool, const int32_t* blocks, int32_t n, const void* host_src, void* stream);

/* ------------------------------------------------------------------- step */

/* One mixed engine iteration: B decode rows then P prefill rows, as one flat
 * token list ("llm-inference-batching": "One step with B decode rows and a
 * prefill chunk of C prompt tokens"). Rows 0..B-1 have one token each
 * (tokens 0..B-1); rows B..B+P-1 are prefill chunks. Per-layer tensors are
 * given as a base pointer and a stride in elements between layers. */
typedef struct pkv_step_desc {
    int32_t num_decode;          /* B */
    int32_t num_prefill;         /* P */
    int32_t num_tokens;          /* T = B + sum of prefill q_lens */
    int32_t max_q_len;           /* largest prefill q_len (grid bound) */
    int32_t max_blocks;          /* width of block_tables */
    int32_t first_layer;         /* layers [first_layer, first_layer + num_layers) run in order */
    int32_t num_layers;
    float scale;
    const int32_t* block_tables; /* device [B+P, max_blocks] */
    const int32_t* ctx_lens;     /* device [B+P] */
    const int32_t* q_start_loc;  /* device [B+P+1], token offsets into the flat list */
    const int64_t* slot_mapping; /* device [T] */
    const void* q;               /* device FP16 [layers][T][num_q_heads][128] */
    const void* k;
    const void* v;
    void* out;                   /* device FP16 [layers][T][num_q_heads][128] */
    int64_t q_layer_stride, k_layer_stride, v_layer_stride, out_layer_stride; /* elements */
} pkv_step_desc;

size_t pkv_step_workspace_bytes(const pkv_pool* pool, const pkv_step_desc* step);

/* For each layer: kv_append of the prefill tokens, causal prefill over the
 * P chunks and decode attention over the B decode rows (which also appends
 * their K/V). One clear of the workspace counters per call covers all layers.
 * In a layer with both kinds of rows the prefill launch goes first and the
 * decode launch does not wait for it (decode reads and writes nothing
 * prefill touches), so decode CTAs run on the SMs prefill leaves idle. */
pkv_status pkv_step(pkv_pool* pool, const pkv_step_desc* step, void* workspace, size_t workspace_bytes,
                    void* stream);

/* ----------------------------------------------------------------- status */

/* Synchronise `stream`, read and clear the sticky device error word
 * (PKV_DEV_* bits into *device_flags if non-NULL). Returns PKV_E_TIMEOUT if
 * a wait ran out, PKV_E_DEVICE for any other flag or a CUDA error. */
pkv_status pkv_get_status(pkv_pool* pool, void* stream, uint32_t* device_flags);

/* Message for the last failure on this thread ("" if none). */
const char* pkv_last_error_string(void);
const char* pkv_status_string(pkv_status s);

/* Test hook for the bounded-wait path: one CTA waits on an mbarrier that no
 * one arrives at, gives up after timeout_ns and sets PKV_DEV_TIMEOUT. */
pkv_status pkv_debug_wait_probe(pkv_pool* pool, uint64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H */
