/*
 * pkv_oracle.c — the ORACLE for the paged KV cache path. Test infrastructure
 * only: slow, plain, single-purpose CPU code that the tests, the package's
 * smoke check and the benchmark's CPU-baseline leg compare the CUDA kernels
 * against. Nothing in the product links or calls it. It shares no header,
 * helper or constant with the CUDA library; it carries its own binary16
 * conversion and its own pool indexing.
 *
 * Arithmetic is IEEE double throughout; FP16 appears only as storage, read
 * exactly and written once with round-to-nearest-even at the end.
 *
 * What each function follows (page, section):
 *   pool geometry       "llm-inference-batching" (faangrind), "KV cache" and
 *                       the KV pool listing: a block is
 *                       [layers, 2 (K,V), heads, 16 tokens, head_dim] FP16,
 *                       2 x 32 x 32 x 128 x 2 = 524,288 B per token.
 *   slot of a position  same page, "block_table: request_id -> [block_id, ...]";
 *                       "continuous batching server" (scalablesystem),
 *                       "PagedAttention Block Table Lookup": logical block
 *                       p / 16 maps through the table, offset p % 16.
 *   kv_append           "llm-inference-batching", step 7 of the loop: a row's
 *                       new keys and values are appended to its blocks.
 *   gather              "continuous batching server", "PagedAttention Block
 *                       Table Lookup": every full block, then the leading
 *                       seq_len % 16 rows of the last block, concatenated.
 *   attention           "Inference Infrastructure" (seeitflow), the decode
 *                       steps: the new token's query attends every cached
 *                       position including its own; softmax(q K^T * scale) V.
 *   causal prefill      "llm-inference-batching", "Prefill and decode share
 *                       each step" (prompt chunks) and "The inference engine"
 *                       (wpnews), "Prefill and decode ask the accelerator for
 *                       different work" (the causal mask).
 *   split merge         "The inference engine", "IO-aware attention and
 *                       quantization attack different costs": tiles combine
 *                       exactly through their softmax statistics.
 *   grouped-query heads "Inference Infrastructure" (seeitflow), the KV cache
 *                       arithmetic: GQA shares one K/V head among a group of
 *                       query heads, MQA one K/V head among all; the cache
 *                       holds the K/V heads only. Reading: the group of K/V
 *                       head k is query heads k*G .. k*G + G-1, G = query
 *                       heads / K/V heads (query head h reads K/V head h / G).
 *   8-bit cache         "Inference Infrastructure", the KV cache arithmetic
 *                       (8 bits per element halve the cache) and "The
 *                       inference engine", "IO-aware attention and
 *                       quantization attack different costs" (scales are
 *                       metadata carried with the data). Reading (the pages
 *                       fix no scale rule): INT8, symmetric, one FP32 scale
 *                       per (token, head) vector of K or V, scale =
 *                       max|x| / 127 and code = round-half-even(x / scale),
 *                       both in IEEE single precision; the stored value is
 *                       code * scale in single precision. A tile holds the
 *                       16 x head_dim codes, then the 16 scales.
 *   block copy / swap   "The inference engine", "Paging turns variable
 *                       sequences into block tables": copy-on-write gives a
 *                       diverging branch its own copy of a shared block;
 *                       "continuous batching server", "Preemption and
 *                       Eviction: Recompute vs Swap": a victim's KV blocks
 *                       go to host memory and come back. Both are whole-
 *                       block byte copies.
 *   prefix hashes       "Serving LLMs" (sreshtalluri), "Prefix caching": each
 *                       full block is hashed together with the hash of
 *                       everything before it, starting from 0. Reading (the
 *                       page uses a language's built-in tuple hash, which is
 *                       unspecified): 64-bit FNV-1a over the previous hash
 *                       (8 bytes, little-endian) followed by the block's 16
 *                       token ids (4 bytes each, little-endian).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int64_t num_blocks;
    int32_t num_layers, num_heads, head_dim, block_size;  /* num_heads: K/V heads stored in the pool */
    int32_t num_q_heads;                                  /* query heads; 0 = num_heads (no grouping) */
    int32_t dtype;                                        /* 0: FP16 elements, 1: INT8 codes + FP32 scales */
} pkvo_geom;

enum { PKVO_FP16 = 0, PKVO_INT8 = 1 };

/* Query heads, and the K/V head that query head h reads. */
static int pkvo_q_heads(const pkvo_geom* g) { return g->num_q_heads > 0 ? g->num_q_heads : g->num_heads; }
static int pkvo_kv_head(const pkvo_geom* g, int h) { return h / (pkvo_q_heads(g) / g->num_heads); }

/* ---------------------------------------------------------------- binary16 */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double pkvo_half_to_double(uint16_t h)
{
    int sign = h >> 15, e = (h >> 10) & 0x1f, f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(0x400 | f), e - 25);    /* 1.f * 2^(e-15) */
    return sign ? -v : v;
}

/* Round a double to the nearest binary16, ties to even. */
uint16_t pkvo_double_to_half(double x)
{
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    if (isnan(x)) return 0x7e00;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7c00;
    if (a == 0.0) return sign;
    int E;
    frexp(a, &E);
    int ue = E - 1;                     /* a in [2^ue, 2^(ue+1)) */
    if (ue < -14) ue = -14;             /* subnormal spacing is 2^-24 */
    double r = rint(ldexp(a, 10 - ue)); /* significand in units of the spacing, RNE */
    if (ue == -14 && r < 1024.0) return sign | (uint16_t)r;
    if (r >= 2048.0) { r = 1024.0; ue += 1; }
    if (ue > 15) return sign | 0x7c00;
    return sign | (uint16_t)(((ue + 15) << 10) | ((int)r - 1024));
}

void pkvo_halves_to_doubles(const uint16_t* in, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = pkvo_half_to_double(in[i]);
}

void pkvo_doubles_to_halves(const double* in, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = pkvo_double_to_half(in[i]);
}

/* ------------------------------------------------------------ pool geometry */

int64_t pkvo_bytes_per_token(const pkvo_geom* g)
{
    if (g->dtype == PKVO_INT8)  /* one byte per element plus one 4-byte scale per (layer, K/V, head) row */
        return 2LL * g->num_layers * g->num_heads * (g->head_dim + 4);
    return 2LL * g->num_layers * g->num_heads * g->head_dim * 2;
}

int64_t pkvo_bytes_per_block(const pkvo_geom* g)
{
    return pkvo_bytes_per_token(g) * g->block_size;
}

int64_t pkvo_pool_bytes(const pkvo_geom* g)
{
    return pkvo_bytes_per_block(g) * g->num_blocks;
}

int64_t pkvo_blocks_for_tokens(int64_t tokens, int32_t block_size)
{
    return (tokens + block_size - 1) / block_size;
}

/* Element index of (block, layer, kv, head, token-in-block, dim). */
static int64_t elem(const pkvo_geom* g, int64_t b, int l, int kv, int h, int t, int d)
{
    int64_t i = b;
    i = i * g->num_layers + l;
    i = i * 2 + kv;
    i = i * g->num_heads + h;
    i = i * g->block_size + t;
    return i * g->head_dim + d;
}

/* Physical slot of logical position pos of a sequence: block * 16 + pos % 16. */
int64_t pkvo_slot(const int32_t* table, int64_t pos, int32_t block_size)
{
    return (int64_t)table[pos / block_size] * block_size + pos % block_size;
}

void pkvo_slots(const int32_t* tables, int32_t max_blocks, const int32_t* row_of_token,
                const int64_t* positions, int64_t T, int32_t block_size, int64_t* out)
{
    for (int64_t i = 0; i < T; ++i)
        out[i] = pkvo_slot(tables + (int64_t)row_of_token[i] * max_blocks, positions[i], block_size);
}

/* ---------------------------------------------------------------- kv_append */

/* Write token i's K row (all heads) and V row to the slot slots[i]. Returns
 * the index of the first out-of-range slot, or -1 when all were written.
 * Slots are checked before anything is written. */
static void pkvo_i8_append_row(uint8_t* pool, const pkvo_geom* g, int64_t b, int layer, int kv, int h, int t,
                               const uint16_t* x);

int64_t pkvo_kv_append(void* pool_v, const pkvo_geom* g, int layer, const uint16_t* k,
                       const uint16_t* v, const int64_t* slots, int64_t T)
{
    uint16_t* pool = (uint16_t*)pool_v;
    for (int64_t i = 0; i < T; ++i)
        if (slots[i] < 0 || slots[i] >= g->num_blocks * g->block_size) return i;
    if (g->dtype == PKVO_INT8) {
        for (int64_t i = 0; i < T; ++i)
            for (int h = 0; h < g->num_heads; ++h) {
                int64_t src = (i * g->num_heads + h) * g->head_dim;
                pkvo_i8_append_row((uint8_t*)pool_v, g, slots[i] / g->block_size, layer, 0, h,
                                   (int)(slots[i] % g->block_size), k + src);
                pkvo_i8_append_row((uint8_t*)pool_v, g, slots[i] / g->block_size, layer, 1, h,
                                   (int)(slots[i] % g->block_size), v + src);
            }
        return -1;
    }
    for (int64_t i = 0; i < T; ++i) {
        int64_t b = slots[i] / g->block_size;
        int t = (int)(slots[i] % g->block_size);
        for (int h = 0; h < g->num_heads; ++h)
            for (int d = 0; d < g->head_dim; ++d) {
                int64_t src = (i * g->num_heads + h) * g->head_dim + d;
                pool[elem(g, b, layer, 0, h, t, d)] = k[src];
                pool[elem(g, b, layer, 1, h, t, d)] = v[src];
            }
    }
    return -1;
}

/* ------------------------------------------------------------------- gather */

/* Contiguous [seq_len, head_dim] copy of one head's K (kv = 0) or V (kv = 1):
 * the full blocks in table order, then the first seq_len % 16 rows of the
 * next block. */
static void pkvo_i8_gather(const uint8_t* pool, const pkvo_geom* g, int layer, int kv, int head,
                           const int32_t* table, int64_t seq_len, double* out);

void pkvo_gather(const void* pool_v, const pkvo_geom* g, int layer, int kv, int head,
                 const int32_t* table, int64_t seq_len, double* out)
{
    const uint16_t* pool = (const uint16_t*)pool_v;
    if (g->dtype == PKVO_INT8) {
        pkvo_i8_gather((const uint8_t*)pool_v, g, layer, kv, head, table, seq_len, out);
        return;
    }
    int64_t full = seq_len / g->block_size, rem = seq_len % g->block_size, row = 0;
    for (int64_t i = 0; i < full; ++i)
        for (int t = 0; t < g->block_size; ++t, ++row)
            for (int d = 0; d < g->head_dim; ++d)
                out[row * g->head_dim + d] = pkvo_half_to_double(pool[elem(g, table[i], layer, kv, head, t, d)]);
    for (int t = 0; t < rem; ++t, ++row)
        for (int d = 0; d < g->head_dim; ++d)
            out[row * g->head_dim + d] = pkvo_half_to_double(pool[elem(g, table[full], layer, kv, head, t, d)]);
}

/* ---------------------------------------------------------------- attention */

/* o = sum_j softmax(scale * q.K_j)_j V_j over n contiguous keys. */
void pkvo_attend(const double* q, const double* K, const double* V, int64_t n, int dim,
                 double scale, double* o)
{
    double* s = (double*)malloc(sizeof(double) * (n > 0 ? n : 1));
    double m = -INFINITY, sum = 0.0;
    for (int64_t j = 0; j < n; ++j) {
        double dot = 0.0;
        for (int d = 0; d < dim; ++d) dot += q[d] * K[j * dim + d];
        s[j] = scale * dot;
        if (s[j] > m) m = s[j];
    }
    for (int64_t j = 0; j < n; ++j) { s[j] = exp(s[j] - m); sum += s[j]; }
    for (int d = 0; d < dim; ++d) o[d] = 0.0;
    for (int64_t j = 0; j < n; ++j)
        for (int d = 0; d < dim; ++d) o[d] += s[j] * V[j * dim + d];
    for (int d = 0; d < dim; ++d) o[d] /= sum;
    free(s);
}

/* Decode: row r's query (q[r, h, :]) attends positions 0 .. ctx_lens[r]-1 of
 * its own blocks, through K/V head pkvo_kv_head(h). out_f64 (optional)
 * receives the unrounded result, out_f16 (optional) the result rounded once
 * to binary16. Layout [B, query heads, dim]. */
void pkvo_decode_attn(const void* pool, const pkvo_geom* g, int layer, const uint16_t* q,
                      const int32_t* tables, int32_t max_blocks, const int32_t* ctx_lens, int32_t B,
                      double scale, double* out_f64, uint16_t* out_f16)
{
    const int H = pkvo_q_heads(g), D = g->head_dim;
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int r = 0; r < B; ++r)
        for (int h = 0; h < H; ++h) {
            int64_t n = ctx_lens[r];
            double* K = (double*)malloc(sizeof(double) * (n > 0 ? n : 1) * D);
            double* V = (double*)malloc(sizeof(double) * (n > 0 ? n : 1) * D);
            double qd[512], o[512];
            const int32_t* table = tables + (int64_t)r * max_blocks;
            pkvo_gather(pool, g, layer, 0, pkvo_kv_head(g, h), table, n, K);
            pkvo_gather(pool, g, layer, 1, pkvo_kv_head(g, h), table, n, V);
            for (int d = 0; d < D; ++d) qd[d] = pkvo_half_to_double(q[((int64_t)r * H + h) * D + d]);
            pkvo_attend(qd, K, V, n, D, scale, o);
            for (int d = 0; d < D; ++d) {
                int64_t i = ((int64_t)r * H + h) * D + d;
                if (out_f64) out_f64[i] = o[d];
                if (out_f16) out_f16[i] = pkvo_double_to_half(o[d]);
            }
            free(K);
            free(V);
        }
}

/* Chunked causal prefill: sequence s owns query tokens
 * [q_start[s], q_start[s+1]) of q ([T, query heads, dim]); they sit at logical
 * positions ctx_lens[s] - q_len + i, and query at position p attends keys
 * 0 .. p of its own blocks, through K/V head pkvo_kv_head(h). */
void pkvo_prefill_attn(const void* pool, const pkvo_geom* g, int layer, const uint16_t* q,
                       const int32_t* q_start, const int32_t* tables, int32_t max_blocks,
                       const int32_t* ctx_lens, int32_t S, double scale, double* out_f64, uint16_t* out_f16)
{
    const int H = pkvo_q_heads(g), D = g->head_dim;
    for (int s = 0; s < S; ++s) {
        int64_t n = ctx_lens[s], qlen = q_start[s + 1] - q_start[s];
        const int32_t* table = tables + (int64_t)s * max_blocks;
        #pragma omp parallel for schedule(dynamic)
        for (int h = 0; h < H; ++h) {
            double* K = (double*)malloc(sizeof(double) * (n > 0 ? n : 1) * D);
            double* V = (double*)malloc(sizeof(double) * (n > 0 ? n : 1) * D);
            double qd[512], o[512];
            pkvo_gather(pool, g, layer, 0, pkvo_kv_head(g, h), table, n, K);
            pkvo_gather(pool, g, layer, 1, pkvo_kv_head(g, h), table, n, V);
            for (int64_t i = 0; i < qlen; ++i) {
                int64_t tok = q_start[s] + i, pos = n - qlen + i;
                for (int d = 0; d < D; ++d) qd[d] = pkvo_half_to_double(q[(tok * H + h) * D + d]);
                pkvo_attend(qd, K, V, pos + 1, D, scale, o);
                for (int d = 0; d < D; ++d) {
                    int64_t idx = (tok * H + h) * D + d;
                    if (out_f64) out_f64[idx] = o[d];
                    if (out_f16) out_f16[idx] = pkvo_double_to_half(o[d]);
                }
            }
            free(K);
            free(V);
        }
    }
}

/* ----------------------------------------------------------- 8-bit cache */

/* Bytes of one (block, layer, K/V, head) tile: the codes [16][head_dim], then 16 FP32 scales. */
int64_t pkvo_i8_tile_bytes(const pkvo_geom* g)
{
    return (int64_t)g->block_size * g->head_dim + 4LL * g->block_size;
}

/* Byte offset of tile (b, l, kv, h) in the pool. */
static int64_t i8_tile(const pkvo_geom* g, int64_t b, int l, int kv, int h)
{
    int64_t tiles_before = ((b * g->num_layers + l) * 2 + kv) * g->num_heads + h;
    return tiles_before * pkvo_i8_tile_bytes(g);
}

/* Quantise one row of n FP16 values: amax = max |x|, scale = amax / 127 and
 * code = round-half-even(x / scale) clamped to [-127, 127], all in IEEE single
 * precision (each operation rounded to float); a row of zeros has scale 0 and
 * codes 0. Inputs must be finite. */
void pkvo_i8_quantize_row(const uint16_t* x, int n, int8_t* codes, float* scale_out)
{
    float amax = 0.0f;
    for (int i = 0; i < n; ++i) {
        float a = (float)fabs(pkvo_half_to_double(x[i]));  /* binary16 -> float is exact */
        if (a > amax) amax = a;
    }
    float scale = (float)(amax / 127.0f);
    for (int i = 0; i < n; ++i) {
        int c = 0;
        if (amax > 0.0f) {
            float qv = (float)((float)pkvo_half_to_double(x[i]) / scale);
            c = (int)rintf(qv);  /* default rounding mode: to nearest, ties to even */
            if (c > 127) c = 127;
            if (c < -127) c = -127;
        }
        codes[i] = (int8_t)c;
    }
    *scale_out = scale;
}

/* The stored value of a code: code * scale, rounded to float. */
double pkvo_i8_dequant(int8_t code, float scale)
{
    return (double)(float)((float)code * scale);
}

static void pkvo_i8_append_row(uint8_t* pool, const pkvo_geom* g, int64_t b, int layer, int kv, int h, int t,
                               const uint16_t* x)
{
    int8_t codes[512];
    float scale;
    pkvo_i8_quantize_row(x, g->head_dim, codes, &scale);
    uint8_t* tile = pool + i8_tile(g, b, layer, kv, h);
    memcpy(tile + (int64_t)t * g->head_dim, codes, (size_t)g->head_dim);
    memcpy(tile + (int64_t)g->block_size * g->head_dim + 4LL * t, &scale, 4);
}

static double i8_value(const uint8_t* pool, const pkvo_geom* g, int64_t b, int layer, int kv, int h, int t, int d)
{
    const uint8_t* tile = pool + i8_tile(g, b, layer, kv, h);
    float scale;
    memcpy(&scale, tile + (int64_t)g->block_size * g->head_dim + 4LL * t, 4);
    return pkvo_i8_dequant((int8_t)tile[(int64_t)t * g->head_dim + d], scale);
}

/* As pkvo_gather, reading codes and scales and returning the stored values. */
static void pkvo_i8_gather(const uint8_t* pool, const pkvo_geom* g, int layer, int kv, int head,
                           const int32_t* table, int64_t seq_len, double* out)
{
    for (int64_t j = 0; j < seq_len; ++j)
        for (int d = 0; d < g->head_dim; ++d)
            out[j * g->head_dim + d] =
                i8_value(pool, g, table[j / g->block_size], layer, kv, head, (int)(j % g->block_size), d);
}

/* ------------------------------------------------- block copy and swap */

/* Whole blocks: every layer, K and V, of a physical block, as stored. */
static int64_t block_bytes_stored(const pkvo_geom* g) { return pkvo_bytes_per_block(g); }

/* dst block pairs[2i+1] receives a copy of src block pairs[2i], in order.
 * Returns the index of the first pair naming a block outside the pool (and
 * copies nothing), or -1. */
int64_t pkvo_copy_blocks(void* pool, const pkvo_geom* g, const int32_t* pairs, int64_t n)
{
    for (int64_t i = 0; i < 2 * n; ++i)
        if (pairs[i] < 0 || pairs[i] >= g->num_blocks) return i / 2;
    const int64_t bb = block_bytes_stored(g);
    for (int64_t i = 0; i < n; ++i)
        memmove((char*)pool + pairs[2 * i + 1] * bb, (const char*)pool + pairs[2 * i] * bb, (size_t)bb);
    return -1;
}

/* host[i] = block blocks[i] (swap out); returns the first bad index or -1. */
int64_t pkvo_swap_out(const void* pool, const pkvo_geom* g, const int32_t* blocks, int64_t n, void* host)
{
    for (int64_t i = 0; i < n; ++i)
        if (blocks[i] < 0 || blocks[i] >= g->num_blocks) return i;
    const int64_t bb = block_bytes_stored(g);
    for (int64_t i = 0; i < n; ++i)
        memcpy((char*)host + i * bb, (const char*)pool + blocks[i] * bb, (size_t)bb);
    return -1;
}

/* block blocks[i] = host[i] (swap in); returns the first bad index or -1. */
int64_t pkvo_swap_in(void* pool, const pkvo_geom* g, const int32_t* blocks, int64_t n, const void* host)
{
    for (int64_t i = 0; i < n; ++i)
        if (blocks[i] < 0 || blocks[i] >= g->num_blocks) return i;
    const int64_t bb = block_bytes_stored(g);
    for (int64_t i = 0; i < n; ++i)
        memcpy((char*)pool + blocks[i] * bb, (const char*)host + i * bb, (size_t)bb);
    return -1;
}

/* ------------------------------------------------------------- prefix hashes */

/* 64-bit FNV-1a of n bytes, continuing from state h (the offset basis for a fresh hash). */
static uint64_t fnv1a64_continue(uint64_t h, const uint8_t* p, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) {
        h ^= p[i];
        h *= 1099511628211ULL;  /* the 64-bit FNV prime, 2^40 + 2^8 + 0xb3 */
    }
    return h;
}

uint64_t pkvo_fnv1a64(const uint8_t* p, int64_t n)
{
    return fnv1a64_continue(14695981039346656037ULL, p, n);  /* the 64-bit offset basis */
}

/* Chained hashes of the full blocks of a token stream: out[i] = H(out[i-1], tokens of block i), out[-1] = 0.
 * Returns the number of full blocks (n_tokens / block_size). */
int64_t pkvo_block_hashes(const int32_t* tokens, int64_t n_tokens, int32_t block_size, uint64_t* out)
{
    uint64_t h = 0;
    int64_t nb = n_tokens / block_size;
    for (int64_t i = 0; i < nb; ++i) {
        uint8_t buf[8 + 4 * 64];
        for (int k = 0; k < 8; ++k) buf[k] = (uint8_t)(h >> (8 * k));
        for (int t = 0; t < block_size; ++t) {
            uint32_t v = (uint32_t)tokens[i * block_size + t];
            for (int k = 0; k < 4; ++k) buf[8 + 4 * t + k] = (uint8_t)(v >> (8 * k));
        }
        h = pkvo_fnv1a64(buf, 8 + 4LL * block_size);
        out[i] = h;
    }
    return nb;
}

/* ------------------------------------------------------------- split merge */

/* Partial softmax statistics of one query over keys [lo, hi): running max
 * m, sum l = sum exp(s - m), un-normalised o = sum exp(s - m) v. */
void pkvo_partial(const double* q, const double* K, const double* V, int64_t lo, int64_t hi, int dim,
                  double scale, double* m_out, double* l_out, double* o)
{
    double m = -INFINITY, l = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        double dot = 0.0;
        for (int d = 0; d < dim; ++d) dot += q[d] * K[j * dim + d];
        if (scale * dot > m) m = scale * dot;
    }
    for (int d = 0; d < dim; ++d) o[d] = 0.0;
    for (int64_t j = lo; j < hi; ++j) {
        double dot = 0.0;
        for (int d = 0; d < dim; ++d) dot += q[d] * K[j * dim + d];
        double p = exp(scale * dot - m);
        l += p;
        for (int d = 0; d < dim; ++d) o[d] += p * V[j * dim + d];
    }
    *m_out = m;
    *l_out = l;
}

/* Combine P partials: M = max m_p; out = sum e^(m_p - M) o_p / sum e^(m_p - M) l_p. */
void pkvo_merge(const double* m, const double* l, const double* o, int P, int dim, double* out)
{
    double M = -INFINITY, L = 0.0;
    for (int p = 0; p < P; ++p) if (m[p] > M) M = m[p];
    for (int d = 0; d < dim; ++d) out[d] = 0.0;
    for (int p = 0; p < P; ++p) {
        double w = exp(m[p] - M);
        L += w * l[p];
        for (int d = 0; d < dim; ++d) out[d] += w * o[(int64_t)p * dim + d];
    }
    for (int d = 0; d < dim; ++d) out[d] /= L;
}

/* Decode attention computed as partitions of part_tokens keys, then merged. */
void pkvo_decode_attn_split(const void* pool, const pkvo_geom* g, int layer, const uint16_t* q,
                            const int32_t* tables, int32_t max_blocks, const int32_t* ctx_lens, int32_t B,
                            double scale, int64_t part_tokens, double* out_f64)
{
    const int H = pkvo_q_heads(g), D = g->head_dim;
    #pragma omp parallel for collapse(2) schedule(dynamic)
    for (int r = 0; r < B; ++r)
        for (int h = 0; h < H; ++h) {
            int64_t n = ctx_lens[r];
            int P = (int)((n + part_tokens - 1) / part_tokens);
            double* K = (double*)malloc(sizeof(double) * (n > 0 ? n : 1) * D);
            double* V = (double*)malloc(sizeof(double) * (n > 0 ? n : 1) * D);
            double* m = (double*)malloc(sizeof(double) * (P > 0 ? P : 1));
            double* l = (double*)malloc(sizeof(double) * (P > 0 ? P : 1));
            double* o = (double*)malloc(sizeof(double) * (P > 0 ? P : 1) * D);
            double qd[512];
            const int32_t* table = tables + (int64_t)r * max_blocks;
            pkvo_gather(pool, g, layer, 0, pkvo_kv_head(g, h), table, n, K);
            pkvo_gather(pool, g, layer, 1, pkvo_kv_head(g, h), table, n, V);
            for (int d = 0; d < D; ++d) qd[d] = pkvo_half_to_double(q[((int64_t)r * H + h) * D + d]);
            for (int p = 0; p < P; ++p) {
                int64_t lo = p * part_tokens, hi = lo + part_tokens < n ? lo + part_tokens : n;
                pkvo_partial(qd, K, V, lo, hi, D, scale, m + p, l + p, o + (int64_t)p * D);
            }
            pkvo_merge(m, l, o, P, D, out_f64 + ((int64_t)r * H + h) * D);
            free(K); free(V); free(m); free(l); free(o);
        }
}

int pkvo_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void pkvo_set_num_threads(int n)
{
#ifdef _OPENMP
    extern void omp_set_num_threads(int);
    omp_set_num_threads(n);
#else
    (void)n;
#endif
}
