// pkv_host.cpp — the C ABI of libpkv: pool handle, ref-counted block manager,
// step metadata, argument validation, status word, and the per-layer step
// launcher. Host code only; kernels live in pkv_kernels.cu / pkv_prefill.cu.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <new>

#include "pkv_internal.h"

namespace {
thread_local char g_err[512] = "";

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

pkv_status check_pool(const pkv_pool* pool)
{
    if (!pool) return pkv::fail(PKV_E_INVALID, "pool is NULL");
    return PKV_OK;
}

// Kernel entry points need a pool bound to device memory.
pkv_status check_device_pool(const pkv_pool* pool)
{
    if (!pool) return pkv::fail(PKV_E_INVALID, "pool is NULL");
    if (pool->host_only) return pkv::fail(PKV_E_INVALID, "pool has no device memory (host-only block manager)");
    return PKV_OK;
}

// Make the pool's device current for the duration of a call.
struct DeviceGuard {
    int prev = -1;
    bool ok = true;
    explicit DeviceGuard(int dev)
    {
        if (cudaGetDevice(&prev) != cudaSuccess) { ok = false; return; }
        if (prev != dev && cudaSetDevice(dev) != cudaSuccess) ok = false;
    }
    ~DeviceGuard()
    {
        int cur = -1;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};
}  // namespace

namespace pkv {

pkv_status fail(pkv_status s, const char* fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    std::vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return s;
}

pkv_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(PKV_E_DEVICE, "%s: %s", what, cudaGetErrorString(e));
}

}  // namespace pkv

using pkv::fail;

extern "C" {

const char* pkv_last_error_string(void) { return g_err; }

const char* pkv_status_string(pkv_status s)
{
    switch (s) {
    case PKV_OK: return "ok";
    case PKV_E_INVALID: return "invalid argument";
    case PKV_E_NOMEM: return "free list exhausted";
    case PKV_E_SHARED: return "write into a shared block";
    case PKV_E_DEVICE: return "device error";
    case PKV_E_TIMEOUT: return "bounded wait ran out";
    }
    return "unknown status";
}

// ------------------------------------------------------------------ pool

static bool desc_ok(const pkv_pool_desc* d)
{
    if (!d) return false;
    if (d->head_dim != pkv::kHeadDim || d->block_size != pkv::kBlockSize) return false;
    if (d->dtype != PKV_DTYPE_FP16 && d->dtype != PKV_DTYPE_INT8) return false;
    if (d->num_blocks < 1 || d->num_blocks > (int64_t)1 << 31) return false;
    if (d->num_layers < 1 || d->num_layers > 1024 || d->num_heads < 1 || d->num_heads > 256) return false;
    if (d->num_q_heads != 0 &&
        (d->num_q_heads < d->num_heads || d->num_q_heads > 1024 || d->num_q_heads % d->num_heads != 0))
        return false;
    return true;
}

static int64_t tile_bytes(const pkv_pool_desc* d)
{
    return d->dtype == PKV_DTYPE_INT8 ? pkv::kTileBytesI8 : pkv::kTileBytes;
}

size_t pkv_pool_bytes(const pkv_pool_desc* d)
{
    if (!desc_ok(d)) return 0;
    return (size_t)d->num_blocks * d->num_layers * 2 * d->num_heads * (size_t)tile_bytes(d);
}

static bool bind_device(pkv_pool* p)
{
    const pkv_pool_desc* d = &p->desc;
    cudaError_t e = cudaGetDevice(&p->device);
    if (e != cudaSuccess) { pkv::cuda_fail(e, "cudaGetDevice"); return false; }
    cudaPointerAttributes attr;
    e = cudaPointerGetAttributes(&attr, d->dev_base);
    if (e != cudaSuccess || attr.type != cudaMemoryTypeDevice || attr.device != p->device) {
        cudaGetLastError();
        fail(PKV_E_INVALID, "dev_base is not device memory of the current device");
        return false;
    }
    e = pkv::status_word(p->device, &p->status_dev);
    if (e != cudaSuccess) { pkv::cuda_fail(e, "status word"); return false; }
    p->geom.base = static_cast<const char*>(d->dev_base);
    p->geom.num_blocks = d->num_blocks;
    p->geom.num_layers = d->num_layers;
    p->geom.num_heads = d->num_heads;
    p->geom.num_q_heads = d->num_q_heads;
    p->geom.group = d->num_q_heads / d->num_heads;
    p->geom.dtype = d->dtype;
    p->geom.tile_bytes = tile_bytes(d);
    p->geom.kv_bytes = (int64_t)d->num_heads * p->geom.tile_bytes;
    p->geom.layer_bytes = 2 * p->geom.kv_bytes;
    p->geom.block_bytes = (int64_t)d->num_layers * p->geom.layer_bytes;
    std::string err;
    if (d->dtype == PKV_DTYPE_FP16) {
        p->kv_tmap_ok = pkv::encode_kv_tmap(p->geom, &p->kv_tmap, &err);
        p->tile_tmap_ok = pkv::encode_tile_tmap(p->geom, &p->tile_tmap, &err);
    } else {
        p->tile_tmap_ok = pkv::encode_i8_tmap(p->geom, &p->tile_tmap, &err);
    }
    return true;
}

pkv_status pkv_pool_create(const pkv_pool_desc* d, pkv_pool** out)
{
    if (!out) return fail(PKV_E_INVALID, "out is NULL");
    *out = nullptr;
    if (!desc_ok(d))
        return fail(PKV_E_INVALID, "unsupported pool descriptor (need head_dim 128, block_size 16, FP16, "
                                   "1..1024 layers, 1..256 K/V heads, 1..2^31 blocks, num_q_heads 0 or a "
                                   "multiple of num_heads up to 1024; FP16 or INT8)");
    const bool host_only = d->dev_base == nullptr;
    if (!host_only && !aligned(d->dev_base, 256)) return fail(PKV_E_INVALID, "dev_base not 256-byte aligned");
    if (!host_only && d->bytes < pkv_pool_bytes(d))
        return fail(PKV_E_INVALID, "pool allocation smaller than pkv_pool_bytes()");
    int part = d->partition_tokens ? d->partition_tokens : pkv::kDefaultPartition;
    // the one-head decode kernel of FP16 pools with one query head per K/V head keeps a partition's block ids
    // in its lanes (2,048 tokens); the grouped-head and 8-bit kernels keep them in shared memory (4,096)
    const bool one_head = d->dtype == PKV_DTYPE_FP16 && (d->num_q_heads == 0 || d->num_q_heads == d->num_heads);
    const int max_part = one_head ? pkv::kMaxPartition : pkv::kMaxPartitionTiles;
    if (part % 64 != 0 || part < 64 || part > max_part)
        return fail(PKV_E_INVALID, "partition_tokens must be a multiple of 64 in [64, %d] for this pool", max_part);

    pkv_pool* p = new (std::nothrow) pkv_pool;
    if (!p) return fail(PKV_E_NOMEM, "host allocation failed");
    p->desc = *d;
    p->desc.free_order = nullptr;
    if (p->desc.num_q_heads == 0) p->desc.num_q_heads = d->num_heads;
    p->partition_tokens = part;
    p->host_only = host_only;
    if (!host_only && !bind_device(p)) {
        delete p;
        return PKV_E_DEVICE;  // message already set
    }


    const int64_t n = d->num_blocks;
    p->ref.assign(n, 0);
    p->cached.assign(n, 0);
    p->free_stack.resize(n);
    if (d->free_order) {
        std::vector<char> seen(n, 0);
        for (int64_t i = 0; i < n; ++i) {
            const int64_t b = d->free_order[i];
            if (b < 0 || b >= n || seen[b]) {
                delete p;
                return fail(PKV_E_INVALID, "free_order is not a permutation of 0..num_blocks-1");
            }
            seen[b] = 1;
            p->free_stack[n - 1 - i] = (int32_t)b;
        }
    } else {
        for (int64_t i = 0; i < n; ++i) p->free_stack[n - 1 - i] = (int32_t)i;
    }
    *out = p;
    return PKV_OK;
}

pkv_status pkv_pool_destroy(pkv_pool* pool)
{
    if (!pool) return fail(PKV_E_INVALID, "pool is NULL");
    delete pool;
    return PKV_OK;
}

// ---------------------------------------------------------- block manager

pkv_status pkv_seq_grow(pkv_pool* pool, int64_t seq_id, int64_t new_len)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(seq_id);
    if (it != pool->seqs.end() && it->second.swapped)
        return fail(PKV_E_INVALID, "seq %lld is swapped out", (long long)seq_id);
    const int64_t cur_len = it == pool->seqs.end() ? 0 : it->second.len;
    const int64_t cur_blocks = it == pool->seqs.end() ? 0 : (int64_t)it->second.table.size();
    if (new_len < cur_len) return fail(PKV_E_INVALID, "seq %lld: new_len %lld below current length %lld",
                                       (long long)seq_id, (long long)new_len, (long long)cur_len);
    const int64_t need = (new_len + pkv::kBlockSize - 1) / pkv::kBlockSize - cur_blocks;
    if (need > (int64_t)pool->free_stack.size())
        return fail(PKV_E_NOMEM, "seq %lld needs %lld blocks, %zu free", (long long)seq_id, (long long)need,
                    pool->free_stack.size());
    pkv::Seq& s = pool->seqs[seq_id];
    for (int64_t i = 0; i < need; ++i) {
        const int32_t b = pool->free_stack.back();
        pool->free_stack.pop_back();
        pool->ref[b] = 1;
        s.table.push_back(b);
    }
    s.len = new_len;
    return PKV_OK;
}

pkv_status pkv_seq_share_prefix(pkv_pool* pool, int64_t dst, int64_t src, int64_t n_blocks)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(src);
    if (it == pool->seqs.end()) return fail(PKV_E_INVALID, "unknown source sequence %lld", (long long)src);
    if (it->second.swapped) return fail(PKV_E_INVALID, "source %lld is swapped out", (long long)src);
    if (dst == src || pool->seqs.count(dst)) return fail(PKV_E_INVALID, "destination %lld already exists", (long long)dst);
    if (n_blocks < 0 || n_blocks * pkv::kBlockSize > it->second.len)
        return fail(PKV_E_INVALID, "only full blocks of the source can be shared");
    std::vector<int32_t> shared(it->second.table.begin(), it->second.table.begin() + n_blocks);
    for (int32_t b : shared) pool->ref[b] += 1;
    pkv::Seq& d = pool->seqs[dst];
    d.table = std::move(shared);
    d.len = n_blocks * pkv::kBlockSize;
    return PKV_OK;
}

pkv_status pkv_seq_free(pkv_pool* pool, int64_t seq_id)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return fail(PKV_E_INVALID, "unknown sequence %lld", (long long)seq_id);
    for (int32_t b : it->second.table)
        if (--pool->ref[b] == 0) pool->free_stack.push_back(b);
    pool->seqs.erase(it);
    return PKV_OK;
}

int64_t pkv_free_blocks(const pkv_pool* pool) { return pool ? (int64_t)pool->free_stack.size() : -1; }

// ------------------------------------------------------------ copy-on-write

pkv_status pkv_seq_fork(pkv_pool* pool, int64_t dst, int64_t src)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(src);
    if (it == pool->seqs.end() || it->second.swapped)
        return fail(PKV_E_INVALID, "source %lld unknown or swapped out", (long long)src);
    if (dst == src || pool->seqs.count(dst)) return fail(PKV_E_INVALID, "destination %lld already exists", (long long)dst);
    const pkv::Seq copy = it->second;
    for (int32_t b : copy.table) pool->ref[b] += 1;
    pool->seqs[dst] = copy;
    return PKV_OK;
}

pkv_status pkv_seq_cow(pkv_pool* pool, int64_t seq_id, int64_t num_new, int32_t* src_block, int32_t* dst_block)
{
    if (pkv_status s = check_pool(pool)) return s;
    if (!src_block || !dst_block) return fail(PKV_E_INVALID, "NULL output");
    *src_block = *dst_block = -1;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end() || it->second.swapped)
        return fail(PKV_E_INVALID, "seq %lld unknown or swapped out", (long long)seq_id);
    pkv::Seq& s = it->second;
    if (num_new < 0 || num_new > s.len)
        return fail(PKV_E_INVALID, "seq %lld: %lld new tokens with length %lld", (long long)seq_id,
                    (long long)num_new, (long long)s.len);
    if (num_new == 0) return PKV_OK;
    // the step writes positions [len - num_new, len): the first block among them that another table
    // also names is the one to copy
    const int64_t first = (s.len - num_new) / pkv::kBlockSize, last = (s.len - 1) / pkv::kBlockSize;
    int64_t i = first;
    while (i <= last && pool->ref[s.table[i]] == 1) ++i;
    if (i > last) return PKV_OK;
    if (pool->free_stack.empty()) return fail(PKV_E_NOMEM, "no free block for the copy");
    const int32_t b = pool->free_stack.back();
    pool->free_stack.pop_back();
    pool->ref[b] = 1;
    const int32_t old = s.table[i];
    pool->ref[old] -= 1;  // above 1 before, so it stays referenced
    s.table[i] = b;
    *src_block = old;
    *dst_block = b;
    return PKV_OK;
}

// ------------------------------------------------------------------- swap

pkv_status pkv_seq_swap_out(pkv_pool* pool, int64_t seq_id, int32_t* blocks, int64_t capacity, int64_t* n_blocks)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end() || it->second.swapped)
        return fail(PKV_E_INVALID, "seq %lld unknown or already swapped out", (long long)seq_id);
    pkv::Seq& s = it->second;
    const int64_t n = (int64_t)s.table.size();
    if (n_blocks) *n_blocks = n;
    if (capacity < n || (n > 0 && !blocks)) return fail(PKV_E_INVALID, "capacity %lld < %lld blocks", (long long)capacity,
                                                        (long long)n);
    std::copy(s.table.begin(), s.table.end(), blocks);
    for (int32_t b : s.table)
        if (--pool->ref[b] == 0) pool->free_stack.push_back(b);
    s.table.clear();
    s.swapped = true;
    return PKV_OK;
}

pkv_status pkv_seq_swap_in(pkv_pool* pool, int64_t seq_id, int32_t* blocks, int64_t capacity, int64_t* n_blocks)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end() || !it->second.swapped)
        return fail(PKV_E_INVALID, "seq %lld is not swapped out", (long long)seq_id);
    pkv::Seq& s = it->second;
    const int64_t n = (s.len + pkv::kBlockSize - 1) / pkv::kBlockSize;
    if (n_blocks) *n_blocks = n;
    if (capacity < n || (n > 0 && !blocks)) return fail(PKV_E_INVALID, "capacity %lld < %lld blocks", (long long)capacity,
                                                        (long long)n);
    if (n > (int64_t)pool->free_stack.size())
        return fail(PKV_E_NOMEM, "seq %lld needs %lld blocks, %zu free", (long long)seq_id, (long long)n,
                    pool->free_stack.size());
    for (int64_t i = 0; i < n; ++i) {
        const int32_t b = pool->free_stack.back();
        pool->free_stack.pop_back();
        pool->ref[b] = 1;
        s.table.push_back(b);
        blocks[i] = b;
    }
    s.swapped = false;
    return PKV_OK;
}

// ------------------------------------------------------------- prefix cache

// 64-bit FNV-1a, continuing from state h.
static uint64_t fnv1a64(uint64_t h, const unsigned char* p, size_t n)
{
    for (size_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 0x100000001b3ULL;
    }
    return h;
}

int64_t pkv_block_hashes(const int32_t* tokens, int64_t n_tokens, uint64_t* out, int64_t capacity)
{
    if (n_tokens < 0 || (n_tokens > 0 && !tokens)) return -1;
    const int64_t nb = n_tokens / pkv::kBlockSize;
    if (capacity < nb || (nb > 0 && !out)) return -1;
    uint64_t h = 0;
    unsigned char buf[8 + 4 * pkv::kBlockSize];
    for (int64_t i = 0; i < nb; ++i) {
        for (int k = 0; k < 8; ++k) buf[k] = (unsigned char)(h >> (8 * k));
        for (int t = 0; t < pkv::kBlockSize; ++t) {
            const uint32_t v = (uint32_t)tokens[i * pkv::kBlockSize + t];
            for (int k = 0; k < 4; ++k) buf[8 + 4 * t + k] = (unsigned char)(v >> (8 * k));
        }
        h = fnv1a64(0xcbf29ce484222325ULL, buf, sizeof(buf));
        out[i] = h;
    }
    return nb;
}

pkv_status pkv_prefix_register(pkv_pool* pool, int64_t seq_id, const uint64_t* hashes, int64_t n_hashes,
                               int64_t* n_new)
{
    if (pkv_status s = check_pool(pool)) return s;
    if (n_new) *n_new = 0;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end() || it->second.swapped)
        return fail(PKV_E_INVALID, "seq %lld unknown or swapped out", (long long)seq_id);
    if (n_hashes < 0 || (n_hashes > 0 && !hashes) || n_hashes * pkv::kBlockSize > it->second.len)
        return fail(PKV_E_INVALID, "only the sequence's full blocks can be cached");
    const uint64_t now = ++pool->clock;
    int64_t added = 0;
    for (int64_t i = 0; i < n_hashes; ++i) {
        auto e = pool->cache.find(hashes[i]);
        if (e != pool->cache.end()) {
            e->second.last_use = now;
            continue;
        }
        const int32_t b = it->second.table[i];
        if (pool->cached[b]) continue;  // already cached under another chain
        pool->cache.emplace(hashes[i], pkv::CacheEntry{b, now, i});
        pool->cached[b] = 1;
        pool->ref[b] += 1;
        ++added;
    }
    if (n_new) *n_new = added;
    return PKV_OK;
}

int64_t pkv_prefix_match(const pkv_pool* pool, const uint64_t* hashes, int64_t n_hashes)
{
    if (!pool || n_hashes < 0 || (n_hashes > 0 && !hashes)) return -1;
    int64_t n = 0;
    while (n < n_hashes && pool->cache.count(hashes[n])) ++n;
    return n;
}

pkv_status pkv_seq_attach_prefix(pkv_pool* pool, int64_t seq_id, const uint64_t* hashes, int64_t n_hashes,
                                 int64_t* n_attached)
{
    if (pkv_status s = check_pool(pool)) return s;
    if (n_attached) *n_attached = 0;
    if (pool->seqs.count(seq_id)) return fail(PKV_E_INVALID, "seq %lld already exists", (long long)seq_id);
    const int64_t n = pkv_prefix_match(pool, hashes, n_hashes);
    if (n < 0) return fail(PKV_E_INVALID, "bad hash list");
    const uint64_t now = ++pool->clock;
    pkv::Seq& s = pool->seqs[seq_id];
    for (int64_t i = 0; i < n; ++i) {
        pkv::CacheEntry& e = pool->cache.find(hashes[i])->second;
        e.last_use = now;
        pool->ref[e.block] += 1;
        s.table.push_back(e.block);
    }
    s.len = n * pkv::kBlockSize;
    if (n_attached) *n_attached = n;
    return PKV_OK;
}

int64_t pkv_prefix_evict(pkv_pool* pool, int64_t max_blocks)
{
    if (!pool || max_blocks < 0) return -1;
    struct Cand {
        uint64_t last_use;
        int64_t depth;
        int32_t block;
        uint64_t hash;
    };
    std::vector<Cand> cand;
    for (const auto& kv : pool->cache)
        if (pool->ref[kv.second.block] == 1) cand.push_back({kv.second.last_use, kv.second.depth, kv.second.block, kv.first});
    // least recently used first; deeper chain positions first among equals
    std::sort(cand.begin(), cand.end(), [](const Cand& a, const Cand& b) {
        if (a.last_use != b.last_use) return a.last_use < b.last_use;
        if (a.depth != b.depth) return a.depth > b.depth;
        if (a.block != b.block) return a.block < b.block;
        return a.hash < b.hash;
    });
    int64_t n = 0;
    for (const Cand& c : cand) {
        if (n >= max_blocks) break;
        pool->cache.erase(c.hash);
        pool->cached[c.block] = 0;
        pool->ref[c.block] = 0;
        pool->free_stack.push_back(c.block);
        ++n;
    }
    return n;
}

int64_t pkv_prefix_cached_blocks(const pkv_pool* pool) { return pool ? (int64_t)pool->cache.size() : -1; }

int32_t pkv_ref_count(const pkv_pool* pool, int64_t block)
{
    if (!pool || block < 0 || block >= pool->desc.num_blocks) return -1;
    return pool->ref[block];
}

int64_t pkv_seq_len(const pkv_pool* pool, int64_t seq_id)
{
    if (!pool) return -1;
    auto it = pool->seqs.find(seq_id);
    return it == pool->seqs.end() ? -1 : it->second.len;
}

pkv_status pkv_block_table(const pkv_pool* pool, int64_t seq_id, int32_t* out, int64_t capacity, int64_t* n_out)
{
    if (pkv_status s = check_pool(pool)) return s;
    auto it = pool->seqs.find(seq_id);
    if (it == pool->seqs.end()) return fail(PKV_E_INVALID, "unknown sequence %lld", (long long)seq_id);
    const int64_t n = (int64_t)it->second.table.size();
    if (n_out) *n_out = n;
    if (capacity < n || (n > 0 && !out)) return fail(PKV_E_INVALID, "capacity %lld < table length %lld",
                                                     (long long)capacity, (long long)n);
    std::copy(it->second.table.begin(), it->second.table.end(), out);
    return PKV_OK;
}

pkv_status pkv_build_step(const pkv_pool* pool, const int64_t* seq_ids, const int32_t* q_lens, int32_t num_seqs,
                          int32_t max_blocks, int32_t* block_tables, int32_t* ctx_lens, int64_t* slot_mapping,
                          int32_t* q_start_loc)
{
    if (pkv_status s = check_pool(pool)) return s;
    if (num_seqs < 0 || max_blocks < 1) return fail(PKV_E_INVALID, "num_seqs < 0 or max_blocks < 1");
    if (num_seqs > 0 && (!seq_ids || !q_lens || !block_tables || !ctx_lens || !slot_mapping || !q_start_loc))
        return fail(PKV_E_INVALID, "NULL array");
    if (num_seqs == 0) {
        if (q_start_loc) q_start_loc[0] = 0;
        return PKV_OK;
    }
    // validate everything first so that a refusal writes nothing
    int64_t total = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        auto it = pool->seqs.find(seq_ids[i]);
        if (it == pool->seqs.end()) return fail(PKV_E_INVALID, "row %d: unknown sequence %lld", i, (long long)seq_ids[i]);
        const pkv::Seq& s = it->second;
        if (s.swapped) return fail(PKV_E_INVALID, "row %d: sequence %lld is swapped out", i, (long long)seq_ids[i]);
        if (q_lens[i] < 1 || q_lens[i] > s.len) return fail(PKV_E_INVALID, "row %d: q_len %d outside [1, %lld]", i,
                                                            q_lens[i], (long long)s.len);
        if ((int64_t)s.table.size() > max_blocks)
            return fail(PKV_E_INVALID, "row %d: %zu blocks exceed max_blocks %d", i, s.table.size(), max_blocks);
        if (s.len > INT32_MAX) return fail(PKV_E_INVALID, "row %d: length exceeds int32", i);
        for (int64_t p = s.len - q_lens[i]; p < s.len; ++p)
            if (pool->ref[s.table[p / pkv::kBlockSize]] != 1)
                return fail(PKV_E_SHARED, "row %d: position %lld falls in a shared block", i, (long long)p);
        for (int32_t j = 0; j < i; ++j)
            if (seq_ids[j] == seq_ids[i]) return fail(PKV_E_INVALID, "sequence %lld listed twice", (long long)seq_ids[i]);
        total += q_lens[i];
        if (total > INT32_MAX) return fail(PKV_E_INVALID, "too many tokens");
    }
    int64_t tok = 0;
    q_start_loc[0] = 0;
    for (int32_t i = 0; i < num_seqs; ++i) {
        const pkv::Seq& s = pool->seqs.find(seq_ids[i])->second;
        int32_t* row = block_tables + (int64_t)i * max_blocks;
        std::fill(row, row + max_blocks, -1);
        std::copy(s.table.begin(), s.table.end(), row);
        ctx_lens[i] = (int32_t)s.len;
        for (int64_t p = s.len - q_lens[i]; p < s.len; ++p)
            slot_mapping[tok++] = (int64_t)s.table[p / pkv::kBlockSize] * pkv::kBlockSize + p % pkv::kBlockSize;
        q_start_loc[i + 1] = (int32_t)tok;
    }
    return PKV_OK;
}

// ---------------------------------------------------------------- kernels

static pkv_status check_layer(const pkv_pool* pool, int32_t layer)
{
    if (layer < 0 || layer >= pool->desc.num_layers)
        return fail(PKV_E_INVALID, "layer %d outside [0, %d)", layer, pool->desc.num_layers);
    return PKV_OK;
}

static cudaError_t launch_append_any(const pkv_pool* pool, int32_t layer, const void* k, const void* v,
                                     const int64_t* slots, int32_t num_tokens, cudaStream_t s);

pkv_status pkv_kv_append(pkv_pool* pool, int32_t layer, const void* k, const void* v, const int64_t* slot_mapping,
                         int32_t num_tokens, void* stream)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (pkv_status s = check_layer(pool, layer)) return s;
    if (num_tokens < 0) return fail(PKV_E_INVALID, "num_tokens < 0");
    if (num_tokens == 0) return PKV_OK;
    if (!k || !v || !slot_mapping) return fail(PKV_E_INVALID, "NULL k, v or slot_mapping");
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(slot_mapping, 8))
        return fail(PKV_E_INVALID, "k/v must be 16-byte aligned, slot_mapping 8-byte aligned");
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaError_t e = launch_append_any(pool, layer, k, v, slot_mapping, num_tokens, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "kv_append launch");
}

pkv_status pkv_copy_blocks(pkv_pool* pool, const int32_t* pairs, int32_t n, void* stream)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (n < 0) return fail(PKV_E_INVALID, "n < 0");
    if (n == 0) return PKV_OK;
    if (!pairs || !aligned(pairs, 4)) return fail(PKV_E_INVALID, "pairs NULL or unaligned");
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaError_t e = pkv::launch_copy_blocks(pool->geom, pairs, n, pool->status_dev, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "copy_blocks launch");
}

static pkv_status swap_blocks(pkv_pool* pool, const int32_t* blocks, int32_t n, void* host, bool to_host, void* stream)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (n < 0) return fail(PKV_E_INVALID, "n < 0");
    if (n == 0) return PKV_OK;
    if (!blocks || !host || !aligned(blocks, 4) || !aligned(host, 16))
        return fail(PKV_E_INVALID, "blocks or host buffer NULL or unaligned (host: 16 bytes)");
    cudaPointerAttributes attr;
    if (cudaPointerGetAttributes(&attr, host) != cudaSuccess || attr.type != cudaMemoryTypeHost || !attr.devicePointer) {
        cudaGetLastError();
        return fail(PKV_E_INVALID, "host buffer is not page-locked host memory the device can address");
    }
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaError_t e = pkv::launch_swap_blocks(pool->geom, blocks, n, attr.devicePointer, to_host, pool->status_dev,
                                            static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "swap launch");
}

pkv_status pkv_swap_blocks_out(pkv_pool* pool, const int32_t* blocks, int32_t n, void* host_dst, void* stream)
{
    return swap_blocks(pool, blocks, n, host_dst, true, stream);
}

pkv_status pkv_swap_blocks_in(pkv_pool* pool, const int32_t* blocks, int32_t n, const void* host_src, void* stream)
{
    return swap_blocks(pool, blocks, n, const_cast<void*>(host_src), false, stream);
}

size_t pkv_decode_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t max_blocks)
{
    if (!pool || num_seqs < 0 || max_blocks < 1) return 0;
    return pkv::decode_workspace_bytes(num_seqs, pool->desc.num_q_heads, max_blocks, pool->partition_tokens);
}

// kv_append for the pool's element type.
static cudaError_t launch_append_any(const pkv_pool* pool, int32_t layer, const void* k, const void* v,
                                     const int64_t* slots, int32_t num_tokens, cudaStream_t s)
{
    if (pool->geom.dtype == PKV_DTYPE_INT8)
        return pkv::launch_kv_append_i8(pool->geom, layer, k, v, slots, num_tokens, pool->status_dev, s);
    return pkv::launch_kv_append(pool->geom, layer, k, v, slots, num_tokens, pool->status_dev, s);
}

// The one-head decode kernel for MHA pools, the group kernel when K/V heads serve several query heads,
// the 8-bit kernel for INT8 pools.
static cudaError_t launch_decode_any(const pkv_pool* pool, int32_t layer, const void* q, const int32_t* tables,
                                     int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs, float scale,
                                     void* out, void* ws, const void* k_new, const void* v_new, const int64_t* slots,
                                     cudaStream_t s, int pdl = 0)
{
    if (pool->geom.dtype == PKV_DTYPE_INT8) {
        const pkv::DecodeWs w = pkv::decode_ws(pool->geom, ws, num_seqs, max_blocks, pool->partition_tokens);
        return pkv::launch_decode_i8(pool->geom, pool->tile_tmap, layer, q, tables, max_blocks, ctx_lens, num_seqs,
                                     scale, out, w, pool->partition_tokens, k_new, v_new, slots, pool->status_dev, s,
                                     pdl);
    }
    const pkv::DecodeWs w = pkv::decode_ws(pool->geom, ws, num_seqs, max_blocks, pool->partition_tokens);
    if (pool->geom.group == 1)
        return pkv::launch_decode(pool->geom, layer, q, tables, max_blocks, ctx_lens, num_seqs, scale, out, w,
                                  pool->partition_tokens, k_new, v_new, slots, pool->status_dev, s, nullptr, nullptr, 0,
                                  pdl);
    return pkv::launch_decode_group(pool->geom, pool->tile_tmap, layer, q, tables, max_blocks, ctx_lens, num_seqs, scale,
                                    out, w, pool->partition_tokens, k_new, v_new, slots, pool->status_dev, s, pdl);
}

static pkv_status check_decode(pkv_pool* pool, int32_t layer, const void* q, const int32_t* tables, int32_t max_blocks,
                               const int32_t* ctx_lens, int32_t num_seqs, const void* out, const void* ws,
                               size_t ws_bytes)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (pkv_status s = check_layer(pool, layer)) return s;
    if (num_seqs < 0 || max_blocks < 1 || max_blocks > (1 << 26))
        return fail(PKV_E_INVALID, "num_seqs < 0 or max_blocks outside [1, 2^26]");
    if (num_seqs > 65535) return fail(PKV_E_INVALID, "num_seqs above 65,535");
    if (num_seqs == 0) return PKV_OK;
    if (!q || !tables || !ctx_lens || !out) return fail(PKV_E_INVALID, "NULL q, tables, ctx_lens or out");
    if ((pool->geom.group > 1 || pool->geom.dtype == PKV_DTYPE_INT8) && !pool->tile_tmap_ok)
        return fail(PKV_E_DEVICE, "TMA descriptor for the pool could not be encoded");
    if (!aligned(q, 16) || !aligned(out, 16) || !aligned(tables, 4) || !aligned(ctx_lens, 4))
        return fail(PKV_E_INVALID, "q/out must be 16-byte aligned, tables/ctx_lens 4-byte aligned");
    if (pkv::decode_max_parts(max_blocks, pool->partition_tokens) > pkv::kMaxPartitionsPerRow)
        return fail(PKV_E_INVALID, "block tables of %d blocks need more than %d partitions per row", max_blocks,
                    pkv::kMaxPartitionsPerRow);
    const size_t need =
        pkv::decode_workspace_bytes(num_seqs, pool->desc.num_q_heads, max_blocks, pool->partition_tokens);
    if (pkv::decode_max_parts(max_blocks, pool->partition_tokens) > 1) {
        if (!ws || ws_bytes < need || !aligned(ws, 256))
            return fail(PKV_E_INVALID, "workspace NULL, unaligned or below %zu bytes", need);
    }
    return PKV_OK;
}

pkv_status pkv_decode_attn(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                           int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs, float scale, void* out,
                           void* workspace, size_t workspace_bytes, void* stream)
{
    if (pkv_status s = check_decode(pool, layer, q, block_tables, max_blocks, ctx_lens, num_seqs, out, workspace,
                                    workspace_bytes))
        return s;
    if (num_seqs == 0) return PKV_OK;
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::clear_decode_counters(pool->geom, num_seqs, max_blocks, pool->partition_tokens, workspace, s);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "clear decode counters");
    e = launch_decode_any(pool, layer, q, block_tables, max_blocks, ctx_lens, num_seqs, scale, out, workspace, nullptr,
                          nullptr, nullptr, s);
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "decode launch");
}

pkv_status pkv_cascade_groups(const int32_t* tables, const int32_t* ctx_lens, int32_t num_seqs, int32_t max_blocks,
                              int32_t min_rows, int32_t* group_start, int32_t* group_blocks, int32_t* num_groups,
                              int32_t* max_group_rows)
{
    if (num_seqs < 0 || max_blocks < 1 || min_rows < 1 || !num_groups || !max_group_rows)
        return fail(PKV_E_INVALID, "bad sizes or NULL output");
    if (num_seqs > 0 && (!tables || !ctx_lens || !group_start || !group_blocks)) return fail(PKV_E_INVALID, "NULL array");
    // blocks of row i that lie wholly before its newest token (a shared block never holds one)
    auto full = [&](int32_t i) { return std::max(0, std::min(max_blocks, (ctx_lens[i] - 1) / pkv::kBlockSize)); };
    auto lcp = [&](int32_t i, int32_t j, int32_t limit) {
        int32_t k = 0;
        const int32_t* a = tables + (int64_t)i * max_blocks;
        const int32_t* b = tables + (int64_t)j * max_blocks;
        while (k < limit && a[k] == b[k] && a[k] >= 0) ++k;
        return k;
    };
    int32_t G = 0, widest = 0;
    for (int32_t i = 0; i < num_seqs;) {
        int32_t j = i + 1, cp = 0;
        if (j < num_seqs) cp = lcp(i, j, std::min(full(i), full(j)));
        if (cp > 0)
            while (j < num_seqs && lcp(i, j, std::min(cp, full(j))) >= cp) ++j;
        if (cp == 0 || j - i < min_rows) {
            j = i + 1;
            cp = 0;
        }
        group_start[G] = i;
        group_blocks[G] = cp;
        widest = std::max(widest, j - i);
        ++G;
        i = j;
    }
    if (num_seqs > 0) group_start[G] = num_seqs;
    else group_start[0] = 0;
    *num_groups = G;
    *max_group_rows = widest;
    return PKV_OK;
}

pkv_status pkv_decode_attn_cascade(pkv_pool* pool, int32_t layer, const void* q, const int32_t* block_tables,
                                   int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs,
                                   const int32_t* group_start, const int32_t* group_blocks, int32_t num_groups,
                                   int32_t max_group_rows, float scale, void* out, void* workspace,
                                   size_t workspace_bytes, void* stream)
{
    if (pkv_status s = check_decode(pool, layer, q, block_tables, max_blocks, ctx_lens, num_seqs, out, workspace,
                                    workspace_bytes))
        return s;
    if (num_seqs == 0) return PKV_OK;
    const size_t need = pkv::decode_workspace_bytes(num_seqs, pool->desc.num_q_heads, max_blocks,
                                                    pool->partition_tokens, 1);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256))
        return fail(PKV_E_INVALID, "cascade workspace NULL, unaligned or below %zu bytes", need);
    if (!pool->tile_tmap_ok) return fail(PKV_E_DEVICE, "TMA descriptor for the pool could not be encoded");
    if (num_groups < 1 || num_groups > num_seqs || max_group_rows < 1 || max_group_rows > num_seqs || !group_start ||
        !group_blocks || !aligned(group_start, 4) || !aligned(group_blocks, 4))
        return fail(PKV_E_INVALID, "bad group description");
    // a shared-prefix CTA holds 16 fragment rows: the query heads of one slice of a K/V head's group for as
    // many of the group's rows as fit
    const int slices = pkv::decode_group_slices(pool->geom.group);
    const int rows_per_cta = 16 / (pool->geom.group / slices);
    const int64_t row_slices = (max_group_rows + rows_per_cta - 1) / rows_per_cta;
    if ((int64_t)num_groups * row_slices > 65535)
        return fail(PKV_E_INVALID, "too many groups x row slices (%d x %lld) for one launch", num_groups,
                    (long long)row_slices);
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // one partial slot more per row than the plain plan: the shared prefix and the rest are partitioned apart
    cudaError_t e =
        pkv::clear_decode_counters(pool->geom, num_seqs, max_blocks, pool->partition_tokens, workspace, s, 1);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "clear decode counters");
    const pkv::DecodeWs w = pkv::decode_ws(pool->geom, workspace, num_seqs, max_blocks, pool->partition_tokens, 1);
    const bool i8 = pool->geom.dtype == PKV_DTYPE_INT8;
    // (1) every group's shared prefix, once per group; (2) each row's own keys, whose last partition merges
    e = i8 ? pkv::launch_decode_i8_shared_prefix(pool->geom, pool->tile_tmap, layer, q, block_tables, max_blocks,
                                                 ctx_lens, group_start, group_blocks, num_groups, max_group_rows,
                                                 scale, out, w, pool->partition_tokens, pool->status_dev, s)
           : pkv::launch_decode_shared_prefix(pool->geom, pool->tile_tmap, layer, q, block_tables, max_blocks,
                                              ctx_lens, num_seqs, group_start, group_blocks, num_groups,
                                              max_group_rows, scale, out, w, pool->partition_tokens,
                                              pool->status_dev, s);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "cascade (shared prefix) launch");
    // the private keys' launch runs beside the shared one (programmatic launch without the dependency wait: it
    // reads only inputs that were ready before this call); the last partial of each row merges it. Fractions of
    // the HBM peak on unique bytes, beside against after: MHA 0.47 against 0.41, 8-bit 0.25 against 0.23,
    // grouped heads 0.161 against 0.153.
    if (i8)
        e = pkv::launch_decode_i8(pool->geom, pool->tile_tmap, layer, q, block_tables, max_blocks, ctx_lens, num_seqs,
                                  scale, out, w, pool->partition_tokens, nullptr, nullptr, nullptr, pool->status_dev,
                                  s, 2, group_start, group_blocks, num_groups);
    else if (pool->geom.group > 1)
        e = pkv::launch_decode_group(pool->geom, pool->tile_tmap, layer, q, block_tables, max_blocks, ctx_lens,
                                     num_seqs, scale, out, w, pool->partition_tokens, nullptr, nullptr, nullptr,
                                     pool->status_dev, s, 2, group_start, group_blocks, num_groups);
    else
        e = pkv::launch_decode(pool->geom, layer, q, block_tables, max_blocks, ctx_lens, num_seqs, scale, out, w,
                               pool->partition_tokens, nullptr, nullptr, nullptr, pool->status_dev, s, group_start,
                               group_blocks, num_groups, 2);
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "cascade decode launch");
}

size_t pkv_decode_cascade_workspace_bytes(const pkv_pool* pool, int32_t num_seqs, int32_t max_blocks)
{
    if (!pool || num_seqs < 0 || max_blocks < 1) return 0;
    return pkv::decode_workspace_bytes(num_seqs, pool->desc.num_q_heads, max_blocks, pool->partition_tokens, 1);
}

static pkv_status prefill_impl(pkv_pool* pool, int32_t layer, const void* q, const int32_t* q_start_loc,
                               const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens,
                               int32_t num_seqs, int32_t max_q_len, float scale, void* out, void* stream)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (pkv_status s = check_layer(pool, layer)) return s;
    if (num_seqs < 0 || max_blocks < 1 || max_q_len < 0) return fail(PKV_E_INVALID, "bad sizes");
    if (num_seqs == 0 || max_q_len == 0) return PKV_OK;
    if (num_seqs > 65535) return fail(PKV_E_INVALID, "num_seqs above 65,535");
    if (!q || !q_start_loc || !block_tables || !ctx_lens || !out) return fail(PKV_E_INVALID, "NULL argument");
    if (!aligned(q, 16) || !aligned(out, 16)) return fail(PKV_E_INVALID, "q/out must be 16-byte aligned");
    if (!(pool->geom.dtype == PKV_DTYPE_INT8 ? pool->tile_tmap_ok : pool->kv_tmap_ok))
        return fail(PKV_E_DEVICE, "TMA descriptor for the pool could not be encoded");
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaError_t e = pkv::launch_prefill(pool, layer, q, q_start_loc, block_tables, max_blocks, ctx_lens, num_seqs,
                                        max_q_len, scale, out, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "prefill launch");
}

pkv_status pkv_prefill_attn(pkv_pool* pool, int32_t layer, const void* q, const int32_t* q_start_loc,
                            const int32_t* block_tables, int32_t max_blocks, const int32_t* ctx_lens, int32_t num_seqs,
                            int32_t max_q_len, float scale, void* out, void* stream)
{
    return prefill_impl(pool, layer, q, q_start_loc, block_tables, max_blocks, ctx_lens, num_seqs, max_q_len, scale,
                        out, stream);
}

// ------------------------------------------------------------------- step

size_t pkv_step_workspace_bytes(const pkv_pool* pool, const pkv_step_desc* st)
{
    if (!pool || !st || st->num_decode < 0 || st->max_blocks < 1) return 0;
    return pkv::decode_workspace_bytes(st->num_decode, pool->desc.num_q_heads, st->max_blocks,
                                       pool->partition_tokens);
}

pkv_status pkv_step(pkv_pool* pool, const pkv_step_desc* st, void* workspace, size_t workspace_bytes, void* stream)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (!st) return fail(PKV_E_INVALID, "step is NULL");
    const int B = st->num_decode, P = st->num_prefill;
    if (B < 0 || P < 0 || st->num_tokens < B + P || st->max_blocks < 1 || st->num_layers < 0)
        return fail(PKV_E_INVALID, "bad step sizes");
    if (P > 0 && st->max_q_len < 1) return fail(PKV_E_INVALID, "prefill rows need max_q_len >= 1");
    if (P == 0 && st->num_tokens != B) return fail(PKV_E_INVALID, "decode-only step must have num_tokens == num_decode");
    if (st->first_layer < 0 || st->first_layer + st->num_layers > pool->desc.num_layers)
        return fail(PKV_E_INVALID, "layer range outside the pool");
    if (st->num_layers == 0 || st->num_tokens == 0) return PKV_OK;
    if (!st->block_tables || !st->ctx_lens || !st->slot_mapping || !st->q || !st->k || !st->v || !st->out)
        return fail(PKV_E_INVALID, "NULL step array");
    if (P > 0 && !st->q_start_loc) return fail(PKV_E_INVALID, "prefill rows need q_start_loc");
    if (st->q_layer_stride % 8 || st->k_layer_stride % 8 || st->v_layer_stride % 8 || st->out_layer_stride % 8)
        return fail(PKV_E_INVALID, "layer strides must be multiples of 8 elements");
    const int64_t tok = (int64_t)pool->desc.num_heads * pkv::kHeadDim * 2;  // bytes of one token's k or v row
    const char* q = static_cast<const char*>(st->q);
    const char* k = static_cast<const char*>(st->k);
    const char* v = static_cast<const char*>(st->v);
    char* out = static_cast<char*>(st->out);
    // Validate the per-layer calls once, on the first layer's pointers (the rest differ only by stride).
    if (pkv_status r = check_decode(pool, st->first_layer, q, st->block_tables, st->max_blocks, st->ctx_lens, B, out,
                                    workspace, workspace_bytes))
        return r;
    if (!aligned(k, 16) || !aligned(v, 16) || !aligned(st->slot_mapping, 8))
        return fail(PKV_E_INVALID, "k/v must be 16-byte aligned, slot_mapping 8-byte aligned");
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = pkv::clear_decode_counters(pool->geom, B, st->max_blocks, pool->partition_tokens, workspace, s);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "clear decode counters");
    for (int32_t i = 0; i < st->num_layers; ++i) {
        const int32_t layer = st->first_layer + i;
        const int64_t li = i;
        const char* ql = q + li * st->q_layer_stride * 2;
        const char* kl = k + li * st->k_layer_stride * 2;
        const char* vl = v + li * st->v_layer_stride * 2;
        char* ol = out + li * st->out_layer_stride * 2;
        if (P > 0) {  // the prefill tokens' kv_append; the decode rows append inside the decode kernel
            e = launch_append_any(pool, layer, kl + B * tok, vl + B * tok, st->slot_mapping + B, st->num_tokens - B, s);
            if (e != cudaSuccess) return pkv::cuda_fail(e, "kv_append launch");
            // Prefill first (it waits for the append that wrote the chunk's keys), then the decode rows, launched
            // with a programmatic dependency on it but without waiting: decode reads and writes nothing prefill
            // touches, so its CTAs fill the SMs prefill leaves idle and take the rest as prefill drains. The next
            // layer's append is an ordinary launch and waits for both.
            pkv_status r = prefill_impl(pool, layer, ql, st->q_start_loc + B,
                                        st->block_tables + (int64_t)B * st->max_blocks, st->max_blocks,
                                        st->ctx_lens + B, P, st->max_q_len, st->scale, ol, stream);
            if (r) return r;
            if (B > 0) {
                e = launch_decode_any(pool, layer, ql, st->block_tables, st->max_blocks, st->ctx_lens, B, st->scale,
                                      ol, workspace, kl, vl, st->slot_mapping, s, 2);
                if (e != cudaSuccess) return pkv::cuda_fail(e, "decode launch");
            }
        } else {
            // decode-only steps: every layer after the first overlaps its prologue with the previous layer
            e = launch_decode_any(pool, layer, ql, st->block_tables, st->max_blocks, st->ctx_lens, B, st->scale, ol,
                                  workspace, kl, vl, st->slot_mapping, s, i > 0 ? 1 : 0);
            if (e != cudaSuccess) return pkv::cuda_fail(e, "decode launch");
        }
    }
    return PKV_OK;
}

// ----------------------------------------------------------------- status

pkv_status pkv_get_status(pkv_pool* pool, void* stream, uint32_t* device_flags)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return pkv::cuda_fail(e, "stream synchronize");
    unsigned int flags = 0;
    e = cudaMemcpy(&flags, pool->status_dev, sizeof(flags), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return pkv::cuda_fail(e, "read status word");
    if (flags) {
        const unsigned int zero = 0;
        e = cudaMemcpy(pool->status_dev, &zero, sizeof(zero), cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return pkv::cuda_fail(e, "clear status word");
    }
    if (device_flags) *device_flags = flags;
    if (flags & PKV_DEV_TIMEOUT) return fail(PKV_E_TIMEOUT, "a kernel's bounded wait ran out (flags 0x%x)", flags);
    if (flags) return fail(PKV_E_DEVICE, "a kernel rejected a device-side input (flags 0x%x)", flags);
    return PKV_OK;
}

pkv_status pkv_debug_wait_probe(pkv_pool* pool, uint64_t timeout_ns, void* stream)
{
    if (pkv_status s = check_device_pool(pool)) return s;
    if (timeout_ns > 10ull * 1000 * 1000 * 1000) return fail(PKV_E_INVALID, "timeout above 10 s");
    DeviceGuard dg(pool->device);
    if (!dg.ok) return fail(PKV_E_DEVICE, "cannot select the pool's device");
    cudaError_t e = pkv::launch_wait_probe(timeout_ns, pool->status_dev, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PKV_OK : pkv::cuda_fail(e, "probe launch");
}

}  // extern "C"
