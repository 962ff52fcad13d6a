// pkv_int8.cu — the 8-bit KV cache: kv_append that quantises, and decode
// attention that dequantises in its loaders.
//
// An 8-bit cache halves the bytes every decode step reads ("Inference
// Infrastructure" (seeitflow), the KV cache arithmetic); its scales are
// metadata stored with the data ("The inference engine" (wpnews),
// "IO-aware attention and quantization attack different costs"). The pages
// fix no scale rule; the library's: INT8 codes, symmetric, one FP32 scale per
// (token, head) row of K or V:
//   amax  = max |x|                      over the row's 128 FP16 values
//   scale = amax / 127                   IEEE single precision
//   code  = round-half-even(x / scale)   IEEE single division, then clamp to +-127
//   value = code * scale                 what attention reads
// A row of zeros has scale 0 and codes 0.
//
// Tile layout: each (block, layer, K/V, head) tile is 2,112 bytes, the 16 x 128
// codes (token-major) followed by the 16 scales, so one bulk copy moves a tile
// with its metadata. A block is layers x 2 x heads tiles.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kCodesBytes = kBlockSize * kHeadDim;  // 2,048
static_assert(kTileBytesI8 == kCodesBytes + 4 * kBlockSize, "8-bit tile: codes then scales");

// Quantise one row of 128 FP16 values held 4 per lane (lane l: values 4l .. 4l+3).
// Returns the lane's 4 codes packed little-endian; *scale receives the row's scale.
__device__ __forceinline__ uint32_t quantize_row_warp(const uint2 raw, float* scale)
{
    float x[4];
    half4_to_float(raw, x);
    float amax = fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3])));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    const float s = __fdiv_rn(amax, 127.f);
    uint32_t packed = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        int c = 0;
        if (amax > 0.f) c = min(max(__float2int_rn(__fdiv_rn(x[i], s)), -127), 127);
        packed |= (uint32_t)(c & 0xff) << (8 * i);
    }
    *scale = s;
    return packed;
}

// ---------------------------------------------------------------- kv_append

// One warp per (token, K/V, head) row: quantise and store its 128 codes and scale.
__global__ void __launch_bounds__(256) kv_append_i8_kernel(char* __restrict__ pool, int64_t block_bytes,
                                                           int64_t layer_off, int64_t kv_bytes, int num_heads,
                                                           const __half* __restrict__ k, const __half* __restrict__ v,
                                                           const int64_t* __restrict__ slots, int num_tokens,
                                                           int64_t num_slots, unsigned int* status)
{
    const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= 2LL * num_heads * num_tokens) return;
    const int tok = (int)(row / (2 * num_heads));
    const int rem = (int)(row - (int64_t)tok * 2 * num_heads);
    const int kv = rem / num_heads, h = rem % num_heads;
    const int64_t slot = __ldg(slots + tok);
    if (slot < 0 || slot >= num_slots) {
        if (rem == 0 && lane == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
        return;
    }
    const __half* src = (kv ? v : k) + ((int64_t)tok * num_heads + h) * kHeadDim;
    float s;
    const uint32_t codes = quantize_row_warp(__ldg(reinterpret_cast<const uint2*>(src) + lane), &s);
    const int t = (int)(slot % kBlockSize);
    char* tile = pool + slot / kBlockSize * block_bytes + layer_off + kv * kv_bytes + (int64_t)h * kTileBytesI8;
    reinterpret_cast<uint32_t*>(tile + t * kHeadDim)[lane] = codes;
    if (lane == 0) *reinterpret_cast<float*>(tile + kCodesBytes + 4 * t) = s;
}

// ---------------------------------------------------------------- decode
//
// One CTA = (partition p, K/V head k with query-head slice c, row r); it
// computes R query heads (R = 1 for a pool without grouped heads, otherwise
// up to 16 of k's group) from one copy of each 8-bit tile. Its four warps take
// the partition's blocks round-robin, each with a private two-stage ring:
// per stage the K and V codes (16 x 128 bytes each, one 4 KB stage) arrive by
// TMA with the 128-byte swizzle and the two 64-byte scale rows by bulk copies
// into a side array, all on one mbarrier. (Four stages measured slower than
// two: the rate is not set by the bytes in flight.) Per block a warp runs the attention on the tensor cores with
// mma.sync m16n8k16 (FP16 operands, FP32 accumulation); with up to 8 query heads, in the transposed form described
// at the kernel (the query heads as the MMA's 8 columns); with more, as follows:
//   S = Q C_K^T      codes become FP16 exactly (byte + 1024 - 1152), each
//                    32-bit word of 4 codes feeding one k-step pair; the
//                    contraction order of the 16 dims in a chunk is permuted
//                    (dims 4j..4j+1 to k 2j..2j+1, 4j+2..4j+3 to k 2j+8..)
//                    and q's fragments use the same order;
//   S_t *= scale_K[t], then online softmax in the log2 domain;
//   O += (P * scale_V) C_V   the V scale folds into P (rows past the context
//                    get exactly 0, never 0 x a garbage scale); a transposed
//                    ldmatrix of the codes yields token pairs for the even and
//                    for the odd dimensions of a 16-dim chunk, so each chunk
//                    is two N = 8 tiles.
// The warps merge through shared memory in warp order; split-K partials merge
// across partitions in partition order, as in the FP16 kernels. With
// `append`, the CTA with c == 0 holding a row's last partition stores the
// quantised new K/V, and the warp streaming that block quantises the same
// rows (the same arithmetic as kv_append) into its shared-memory copy.

constexpr int kQWarps = 4;
constexpr int kQStages = 2;
constexpr int kQStage = 2 * kCodesBytes;  // K codes at 0, V codes at 2,048: both 1 KB aligned for the swizzle
constexpr int kQScaleStage = 2 * 4 * kBlockSize;  // K scales, then V scales
constexpr int kQRows = 16;
constexpr int kQMaxBlocks = kMaxPartitionTiles / kBlockSize;
constexpr int kQMergeStride = kHeadDim + 4;

constexpr int kQSmRing = 0;
constexpr int kQSmScales = kQSmRing + kQWarps * kQStages * kQStage;  // [warp][stage] 128 B
constexpr int kQSmIds = kQSmScales + kQWarps * kQStages * kQScaleStage;
constexpr int kQSmBars = kQSmIds + kQMaxBlocks * 4;
constexpr int kQSmFlag = kQSmBars + kQWarps * kQStages * 8;
constexpr int kQSmBytes = kQSmFlag + 4 * kQRows;  // the last-arrival flag; cascade: one per row
constexpr int kQSmAlloc = kQSmBytes + 1024;
constexpr int kQSmMergeO = 0;
constexpr int kQSmMergeML = kQWarps * kQRows * kQMergeStride * 4;
static_assert(kQSmMergeML + kQWarps * kQRows * 8 <= kQSmBars, "merge scratch fits in the idle rings, scales and ids");

struct I8Args {
    const __half* q;
    __half* out;
    const int32_t* tables;
    int max_blocks;
    const int32_t* ctx_lens;
    char* pool;
    int64_t block_bytes;
    int64_t head_off;
    int64_t kv_bytes;
    int64_t num_blocks;
    int layer;
    int num_kv_heads;
    int num_q_heads;
    int group;
    int rows;
    int slices;
    float scale_log2;
    float* ws_o;
    float* ws_ml;
    unsigned int* counters;  // [B][num_kv_heads * slices]
    int max_parts;
    int ws_parts;
    int part_tokens;
    const __half* k_new;     // [B][num_kv_heads][128] when append
    const __half* v_new;
    const int64_t* slots;
    int append;
    int no_wait;             // launched after a kernel whose results it does not read: skip the dependency wait
    unsigned int* status;
    // cascade: rows [group_start[i], group_start[i+1]) share their first group_blocks[i] blocks. In CASCADE mode
    // the kernel computes those shared partitions for the group's rows at once; otherwise (group_start set) a
    // row's partitions cover only the keys after its group's shared prefix.
    const int32_t* group_start;
    const int32_t* group_blocks;
    int num_groups;
    int part_z;              // grid (K/V head slice, row, partition) instead of (partition, K/V head slice, row)
    int max_slices;          // CASCADE: ceil(largest group / rows per CTA)
};

// Byte offset of byte b of token t's 128 codes in a swizzled 16 x 128 B code tile.
__device__ __forceinline__ uint32_t code_off(int t, int b)
{
    return (uint32_t)(t * 128 + ((((b >> 4) ^ (t & 7))) << 4) + (b & 15));
}

// Two biased code bytes (code + 128) selected by `sel` into a half2 of code + 1,152, exactly (the byte
// under an FP16 exponent of 1,024). The MMAs run on these biased values; the bias comes off once per
// score (1,152 * sum(q)) and once per output row (1,152 * sum of the FP16 weights), so no per-value
// subtraction is needed.
constexpr float kCodeBias = 1152.f;
__device__ __forceinline__ uint32_t codes2_to_half2(uint32_t biased, uint32_t sel)
{
    return __byte_perm(biased, 0x64646464u, sel);
}

__device__ __forceinline__ float half2_sum(uint32_t h)
{
    const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h));
    return f.x + f.y;
}

__device__ __forceinline__ unsigned int q_atomic_add_acq_rel(unsigned int* p, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Up to 8 query heads per CTA: four CTAs per SM (128 registers a thread; the transposed form below fits them
// without spills, five CTAs at 96 registers spill and ran 7 % slower). An 8-bit CTA carries half the bytes of an
// FP16 one, so more of them in flight cover more of each other's start-up. 16 fragment rows (up to 16 query
// heads, or cascade's rows of a group) need more registers: three per SM.
//
// Transposed form (kT): with R <= 8 query heads the products run as S^T = C_K Q^T and O^T = C_V^T P'^T, the
// 16 MMA rows being a block's 16 tokens (for S^T) or 16 dims (for O^T) and the 8 columns the query heads, so a
// block takes 16 MMAs instead of 32 and O^T 32 accumulators a thread instead of 64. Rows of O^T: in 16-dim
// chunk c, row g is dim 16c + 2g and row g + 8 dim 16c + 2g + 1 (a transposed ldmatrix of the codes gives
// token pairs of those two dims in one word). P' moves from S^T's accumulator layout to the B operand's by
// four shuffles a block.
template <bool ROWS16, bool CASCADE>
__global__ void __launch_bounds__(kQWarps * 32, ROWS16 ? 3 : 4)
    decode_i8_kernel(const __grid_constant__ CUtensorMap tmap, const I8Args a)
{
    constexpr bool kT = !ROWS16 && !CASCADE;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    // a cascade's private keys (a partition or two a row, the grid sized for whole rows): partition-slowest grid,
    // so the CTAs with no keys come last (0.270 against 0.257 of the HBM peak on unique bytes; the FP16 cascade
    // kernels measured slower that way and keep the partition-fastest grid, whose partials of a row stay in L2)
    const int p = a.part_z ? blockIdx.z : blockIdx.x;
    const int by = a.part_z ? blockIdx.x : blockIdx.y;
    const int kvh = by / a.slices, c = by % a.slices;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;
    // The CTA's R fragment rows: query heads h0 .. h0 + hpr - 1 (hpr = a.rows) of rows r .. r + nseq - 1;
    // fragment row f is query head h0 + f % hpr of row r + f / hpr. Normal mode: one row. CASCADE: as many
    // rows of one group as 16 fragment rows hold, over the group's shared prefix.
    const int hpr = a.rows;
    const int h0 = kvh * a.group + c * hpr;
    int r, R, nseq, ctx, nparts, tok_lo, slot_p, span = a.part_tokens;
    // Cascade: the private keys' launch reads nothing this grid writes except through the split-K counters,
    // so it may start beside this one at once (whichever partial of a row arrives last merges the row)
    if (CASCADE) pdl_trigger();
    if (CASCADE) {
        const int spc = kQRows / hpr;
        const int grp = blockIdx.z / a.max_slices, sl = blockIdx.z % a.max_slices;
        const int row0 = __ldg(a.group_start + grp), row_end = __ldg(a.group_start + grp + 1);
        r = row0 + sl * spc;
        nseq = min(spc, row_end - r);
        if (nseq <= 0) return;
        R = nseq * hpr;
        ctx = __ldg(a.group_blocks + grp) * kBlockSize;  // the shared prefix: full blocks, valid for every row
        nparts = (ctx + a.part_tokens - 1) / a.part_tokens;
        if (p >= nparts) return;
        tok_lo = p * a.part_tokens;
        slot_p = p;
    } else {
        r = a.part_z ? blockIdx.y : blockIdx.z;
        nseq = 1;
        R = hpr;
        // the row's length and (cascade) its group's shared prefix: independent loads, both issued before
        // either is used (one memory round trip for a short cascade row's CTA, not two)
        ctx = __ldg(a.ctx_lens + r);
        // Cascade's other half: keys [0, S) of the row's group's shared prefix were partitioned on their own
        // (slots 0 .. nsh - 1); this CTA takes partition p of [S, ctx), slot nsh + p.
        int S = 0;
        if (a.group_start) {
            int lo = 0, hi = a.num_groups - 1;
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (__ldg(a.group_start + mid) <= r) lo = mid; else hi = mid - 1;
            }
            S = __ldg(a.group_blocks + lo) * kBlockSize;
        }
        if (ctx < 1 || ctx > a.max_blocks * kBlockSize) {
            if (p == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_CTX);
            return;
        }
        if (ctx <= S) {  // the group's shared prefix must lie below the row's newest token
            if (p == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_CTX);
            return;
        }
        // [S, ctx) goes into as few partitions as part_tokens allows, of equal length in whole blocks, so that
        // no short partition's CTA trails the launch
        const int nsh = (S + a.part_tokens - 1) / a.part_tokens;
        const int np = (ctx - S + a.part_tokens - 1) / a.part_tokens;
        span = ((ctx - S + np - 1) / np + kBlockSize - 1) / kBlockSize * kBlockSize;
        tok_lo = S + p * span;
        if (tok_lo >= ctx) return;
        nparts = nsh + (ctx - S + span - 1) / span;
        slot_p = nsh + p;
    }
    auto rh = [&](int f) { return (int64_t)(r + f / hpr) * a.num_q_heads + h0 + f % hpr; };
    const int blk_lo = tok_lo / kBlockSize;
    const int blk_hi = (min(tok_lo + span, ctx) + kBlockSize - 1) / kBlockSize;
    const int count = blk_hi - blk_lo;

    int32_t* ids = reinterpret_cast<int32_t*>(smem + kQSmIds);
    const int32_t* trow = a.tables + (int64_t)r * a.max_blocks;
    bool bad = false;
    for (int i = threadIdx.x; i < count; i += kQWarps * 32) {
        const int id = __ldg(trow + blk_lo + i);
        ids[i] = id;
        bad |= id < 0 || (int64_t)id >= a.num_blocks;
    }
    const uint32_t bar0 = sb + kQSmBars + warp * kQStages * 8;
    if (lane == 0) {
        for (int s = 0; s < kQStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        return;
    }

    const int nloc = count > warp ? (count - warp + kQWarps - 1) / kQWarps : 0;
    const uint32_t ring = sb + kQSmRing + warp * kQStages * kQStage;
    const uint32_t sring = sb + kQSmScales + warp * kQStages * kQScaleStage;
    const char* tile_k = a.pool + a.head_off + (int64_t)kvh * kTileBytesI8;
    auto issue = [&](int li) {
        const int s = li % kQStages;
        const int id = ids[warp + li * kQWarps];
        const uint32_t dst = ring + s * kQStage, bar = bar0 + 8 * s;
        const char* src = tile_k + (int64_t)id * a.block_bytes;
        mbar_arrive_expect_tx(bar, 2 * kTileBytesI8);
        tma_load_5d(dst, &tmap, 0, 0, kvh, a.layer, id, bar);
        tma_load_5d(dst + kCodesBytes, &tmap, 0, 0, a.num_kv_heads + kvh, a.layer, id, bar);
        bulk_g2s(sring + s * kQScaleStage, src + kCodesBytes, 4 * kBlockSize, bar);
        bulk_g2s(sring + s * kQScaleStage + 4 * kBlockSize, src + a.kv_bytes + kCodesBytes, 4 * kBlockSize, bar);
    };
    int issued = min(nloc, kQStages);
    if (lane == 0)
        for (int li = 0; li < issued; ++li) issue(li);

    // Only lengths, tables and this layer's codes were read so far; with a programmatic dependency on the
    // previous layer's kernel, wait for it before reading q or the new K/V and touching the workspace.
    // Without the wait (no_wait), one CTA still waits: a cascade's private launch then ends only after the shared
    // launch it runs beside, so work after the call in the stream finds both done.
    if (!a.no_wait || (a.group_start && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)) pdl_wait();

    // The new token: quantised here by the warp that streams its block, and stored by c == 0's warp 0.
    const int new_t = (ctx - 1) % kBlockSize, new_i = (ctx - 1) / kBlockSize - blk_lo;
    int patch_li = -1;
    uint32_t kcodes = 0, vcodes = 0;
    float kscale = 0.f, vscale = 0.f;
    if (!CASCADE && a.append && slot_p == nparts - 1) {
        const int64_t slot = __ldg(a.slots + r);
        const int32_t tb = __ldg(trow + (ctx - 1) / kBlockSize);
        const bool consistent =
            tb >= 0 && (int64_t)tb < a.num_blocks && slot == (int64_t)tb * kBlockSize + new_t;
        if (!consistent) {
            if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_SLOT);
        } else if (warp == new_i % kQWarps || (c == 0 && warp == 0)) {
            const int64_t src = ((int64_t)r * a.num_kv_heads + kvh) * kHeadDim;
            kcodes = quantize_row_warp(__ldg(reinterpret_cast<const uint2*>(a.k_new + src) + lane), &kscale);
            vcodes = quantize_row_warp(__ldg(reinterpret_cast<const uint2*>(a.v_new + src) + lane), &vscale);
            if (warp == new_i % kQWarps) patch_li = new_i / kQWarps;
            if (c == 0 && warp == 0) {
                char* tile = a.pool + slot / kBlockSize * a.block_bytes + a.head_off + (int64_t)kvh * kTileBytesI8;
                reinterpret_cast<uint32_t*>(tile + new_t * kHeadDim)[lane] = kcodes;
                reinterpret_cast<uint32_t*>(tile + a.kv_bytes + new_t * kHeadDim)[lane] = vcodes;
                if (lane == 0) {
                    *reinterpret_cast<float*>(tile + kCodesBytes + 4 * new_t) = kscale;
                    *reinterpret_cast<float*>(tile + a.kv_bytes + kCodesBytes + 4 * new_t) = vscale;
                }
            }
        }
    }

    // q as the A operand in the permuted contraction order: for chunk j (dims 16j..16j+15),
    // register 0 holds dims 16j+4tq, +1 and register 2 holds dims 16j+4tq+2, +3 of row g. Transposed form: q as
    // the B operand, query head g's dims 16j+4tq, +1 (register 0) and 16j+4tq+2, +3 (register 1).
    uint32_t qa[8][4];
    uint32_t qb[8][2];
    float bias_t[2] = {0.f, 0.f};  // transposed form: the scores' bias of query heads 2tq, 2tq+1
    if constexpr (kT) {
        const bool q_ok = g < R;
        const uint2* qrow = reinterpret_cast<const uint2*>(a.q + (q_ok ? rh(g) : 0) * kHeadDim);
        float sum = 0.f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint2 v = q_ok ? __ldg(qrow + 4 * j + tq) : make_uint2(0u, 0u);
            qb[j][0] = v.x;
            qb[j][1] = v.y;
            sum += half2_sum(v.x) + half2_sum(v.y);
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);  // query head g's sum, in each of its four lanes
        bias_t[0] = kCodeBias * __shfl_sync(0xffffffffu, sum, 8 * tq);
        bias_t[1] = kCodeBias * __shfl_sync(0xffffffffu, sum, 8 * tq + 4);
    } else {
        const bool lo_ok = g < R, hi_ok = ROWS16 && g + 8 < R;
        const uint32_t* qlo = reinterpret_cast<const uint32_t*>(a.q + (lo_ok ? rh(g) : 0) * kHeadDim);
        const uint32_t* qhi = reinterpret_cast<const uint32_t*>(a.q + (hi_ok ? rh(g + 8) : 0) * kHeadDim);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            qa[j][0] = lo_ok ? __ldg(qlo + 8 * j + 2 * tq) : 0u;
            qa[j][1] = hi_ok ? __ldg(qhi + 8 * j + 2 * tq) : 0u;
            qa[j][2] = lo_ok ? __ldg(qlo + 8 * j + 2 * tq + 1) : 0u;
            qa[j][3] = hi_ok ? __ldg(qhi + 8 * j + 2 * tq + 1) : 0u;
        }
    }
    // the scores' bias: 1,152 * sum(q) of rows g and g + 8 (q * 1,152 is exact in FP32)
    float bias_lo = 0.f, bias_hi = 0.f;
    if constexpr (!kT) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            bias_lo += half2_sum(qa[j][0]) + half2_sum(qa[j][2]);
            if (ROWS16) bias_hi += half2_sum(qa[j][1]) + half2_sum(qa[j][3]);
        }
        bias_lo += __shfl_xor_sync(0xffffffffu, bias_lo, 1);
        bias_lo += __shfl_xor_sync(0xffffffffu, bias_lo, 2);
        bias_hi += __shfl_xor_sync(0xffffffffu, bias_hi, 1);
        bias_hi += __shfl_xor_sync(0xffffffffu, bias_hi, 2);
        bias_lo *= kCodeBias;
        bias_hi *= kCodeBias;
    }

    float o[kT ? 8 : 16][4];
#pragma unroll
    for (int nt = 0; nt < (kT ? 8 : 16); ++nt) o[nt][0] = o[nt][1] = o[nt][2] = o[nt][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    float w_lo = 0.f, w_hi = 0.f;  // running sums of the FP16 weights the P V MMAs saw (this lane's tokens)
    const int mi = lane >> 3, rr = lane & 7;
    bool ok = true;
    for (int li = 0; li < nloc; ++li) {
        const int s = li % kQStages;
        const uint32_t kt = ring + s * kQStage, vt = kt + kCodesBytes;
        const uint32_t ks_s = sring + s * kQScaleStage, vs_s = ks_s + 4 * kBlockSize;
        const int nvalid = min(kBlockSize, ctx - (blk_lo + warp + li * kQWarps) * kBlockSize);
        if (!mbar_wait(bar0 + 8 * s, (uint32_t)(li / kQStages) & 1u)) {
            ok = false;
            break;
        }
        if (li == patch_li) {
            const uint32_t off = code_off(new_t, 4 * lane);
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(kt + off), "r"(kcodes) : "memory");
            asm volatile("st.shared.u32 [%0], %1;" ::"r"(vt + off), "r"(vcodes) : "memory");
            if (lane == 0) {
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(ks_s + 4 * new_t), "f"(kscale) : "memory");
                asm volatile("st.shared.f32 [%0], %1;" ::"r"(vs_s + 4 * new_t), "f"(vscale) : "memory");
            }
            __syncwarp();
        }
        if constexpr (kT) {
            // ---- transposed form: m_lo, l_lo, w_lo belong to query head 2tq, m_hi, l_hi, w_hi to 2tq + 1
            // S^T = C_K Q^T over chunk pairs; chunks j and j + 1 accumulate apart (shorter MMA chains)
            float sa[2][4] = {};
#pragma unroll
            for (int j = 0; j < 8; j += 2) {
                uint32_t w[4];
                ldsm_x4(kt + code_off(rr + (mi & 1) * 8, 16 * (j + (mi >> 1))), w);  // (token g | g + 8) x (j | j+1)
#pragma unroll
                for (int jj = 0; jj < 2; ++jj) {
                    const uint32_t lo = w[2 * jj] ^ 0x80808080u, hi = w[2 * jj + 1] ^ 0x80808080u;
                    const uint32_t af[4] = {codes2_to_half2(lo, 0x4140u), codes2_to_half2(hi, 0x4140u),
                                            codes2_to_half2(lo, 0x4342u), codes2_to_half2(hi, 0x4342u)};
                    mma_16816(sa[jj], af, qb[j + jj][0], qb[j + jj][1]);
                }
            }
            // element e: token g (e < 2) or g + 8, query head 2tq + (e & 1)
            float ks[2], vs[2];
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(ks[0]) : "r"(ks_s + 4 * g));
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(ks[1]) : "r"(ks_s + 4 * (g + 8)));
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(vs[0]) : "r"(vs_s + 4 * g));
            asm volatile("ld.shared.f32 %0, [%1];" : "=f"(vs[1]) : "r"(vs_s + 4 * (g + 8)));
            const bool tv[2] = {g < nvalid, g + 8 < nvalid};
            float sv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sv[e] = tv[e >> 1] ? (sa[0][e] + sa[1][e] - bias_t[e & 1]) * ks[e >> 1] * a.scale_log2 : -INFINITY;
            float mx0 = fmaxf(sv[0], sv[2]), mx1 = fmaxf(sv[1], sv[3]);
#pragma unroll
            for (int off = 4; off < 32; off <<= 1) {
                mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
                mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
            }
            const float mn0 = fmaxf(m_lo, mx0), mn1 = fmaxf(m_hi, mx1);
            const float al0 = exp2f(m_lo - mn0), al1 = exp2f(m_hi - mn1);
            m_lo = mn0;
            m_hi = mn1;
            const float p0 = exp2f(sv[0] - mn0), p1 = exp2f(sv[1] - mn1);
            const float p2 = exp2f(sv[2] - mn0), p3 = exp2f(sv[3] - mn1);
            l_lo = l_lo * al0 + (p0 + p2);
            l_hi = l_hi * al1 + (p1 + p3);
            // P' = P * scale_V, tokens past the context exactly 0; X: token g, Y: token g + 8 (query heads
            // 2tq, 2tq + 1 in the low and high halves)
            const uint32_t X = pack_half2(tv[0] ? p0 * vs[0] : 0.f, tv[0] ? p1 * vs[0] : 0.f);
            const uint32_t Y = pack_half2(tv[1] ? p2 * vs[1] : 0.f, tv[1] ? p3 * vs[1] : 0.f);
            {
                const float2 fx = __half22float2(*reinterpret_cast<const __half2*>(&X));
                const float2 fy = __half22float2(*reinterpret_cast<const __half2*>(&Y));
                w_lo = w_lo * al0 + (fx.x + fy.x);
                w_hi = w_hi * al1 + (fx.y + fy.y);
            }
            // B operand of P'^T: this lane takes query head g, tokens 2tq, 2tq+1 (b0) and 2tq+8, 2tq+9 (b1),
            // from the lanes holding tokens 2tq and 2tq + 1 for query heads 2(g/2), 2(g/2) + 1
            const int src1 = 8 * tq + (g >> 1), src2 = src1 + 4;
            const uint32_t x1 = __shfl_sync(0xffffffffu, X, src1), x2 = __shfl_sync(0xffffffffu, X, src2);
            const uint32_t y1 = __shfl_sync(0xffffffffu, Y, src1), y2 = __shfl_sync(0xffffffffu, Y, src2);
            const uint32_t sel = (g & 1) ? 0x7632u : 0x5410u;
            const uint32_t pb0 = __byte_perm(x1, x2, sel), pb1 = __byte_perm(y1, y2, sel);
            // rescale O only when some query head's running max rose in this block
            if (__any_sync(0xffffffffu, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    o[c][0] *= al0;
                    o[c][1] *= al1;
                    o[c][2] *= al0;
                    o[c][3] *= al1;
                }
            }
            // O^T += C_V^T P'^T over chunk pairs; the word of chunk cc + u holds tokens (2tq, 2tq+1) of dims
            // (2g, 2g+1) (tokens 0-7 in w[2u], 8-15 in w[2u + 1])
#pragma unroll
            for (int cc = 0; cc < 8; cc += 2) {
                uint32_t w[4];
                ldsm_x4_t(vt + code_off(rr + (mi & 1) * 8, 16 * (cc + (mi >> 1))), w);
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const uint32_t lo = w[2 * u] ^ 0x80808080u, hi = w[2 * u + 1] ^ 0x80808080u;
                    const uint32_t af[4] = {codes2_to_half2(lo, 0x4240u), codes2_to_half2(lo, 0x4341u),
                                            codes2_to_half2(hi, 0x4240u), codes2_to_half2(hi, 0x4341u)};
                    mma_16816(o[cc + u], af, pb0, pb1);
                }
            }
        } else {

        // S = Q C_K^T over chunk pairs (j, j+1); matrices (tokens 0-7 | 8-15) x (chunk j | j+1).
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int j = 0; j < 8; j += 2) {
            uint32_t w[4];
            ldsm_x4(kt + code_off(rr + (mi & 1) * 8, 16 * (j + (mi >> 1))), w);
#pragma unroll
            for (int jj = 0; jj < 2; ++jj)
#pragma unroll
                for (int nt = 0; nt < 2; ++nt) {
                    const uint32_t bw = w[jj * 2 + nt] ^ 0x80808080u;
                    mma_16816(sacc[nt], qa[j + jj], codes2_to_half2(bw, 0x4140u), codes2_to_half2(bw, 0x4342u));
                }
        }
        // element e of tile nt: row g (e < 2) or g + 8, token 8nt + 2tq + (e & 1)
        float ksc[2][2], vsc[2][2];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float2 kk, vv;
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(kk.x), "=f"(kk.y) : "r"(ks_s + 4 * (nt * 8 + 2 * tq)));
            asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(vv.x), "=f"(vv.y) : "r"(vs_s + 4 * (nt * 8 + 2 * tq)));
            ksc[nt][0] = kk.x; ksc[nt][1] = kk.y;
            vsc[nt][0] = vv.x; vsc[nt][1] = vv.y;
        }
        float sv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sv[nt][e] = (nt * 8 + 2 * tq + (e & 1) < nvalid)
                                ? (sacc[nt][e] - (e < 2 ? bias_lo : bias_hi)) * ksc[nt][e & 1] * a.scale_log2
                                : -INFINITY;
        float mx = fmaxf(fmaxf(sv[0][0], sv[0][1]), fmaxf(sv[1][0], sv[1][1]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mn_lo = fmaxf(m_lo, mx);
        const float al_lo = exp2f(m_lo - mn_lo);
        m_lo = mn_lo;
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = exp2f(sv[nt][0] - mn_lo);
            pr[nt][1] = exp2f(sv[nt][1] - mn_lo);
        }
        l_lo = l_lo * al_lo + ((pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]));
        float al_hi = 1.f;
        if (ROWS16) {
            float mh = fmaxf(fmaxf(sv[0][2], sv[0][3]), fmaxf(sv[1][2], sv[1][3]));
            mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 1));
            mh = fmaxf(mh, __shfl_xor_sync(0xffffffffu, mh, 2));
            const float mn_hi = fmaxf(m_hi, mh);
            al_hi = exp2f(m_hi - mn_hi);
            m_hi = mn_hi;
#pragma unroll
            for (int nt = 0; nt < 2; ++nt) {
                pr[nt][2] = exp2f(sv[nt][2] - mn_hi);
                pr[nt][3] = exp2f(sv[nt][3] - mn_hi);
            }
            l_hi = l_hi * al_hi + ((pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]));
        } else {
            pr[0][2] = pr[0][3] = pr[1][2] = pr[1][3] = 0.f;
        }
        // P * scale_V as the A operand (k = tokens); tokens past the context contribute exactly 0
        float pw[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                pw[nt][e] = (nt * 8 + 2 * tq + (e & 1) < nvalid) ? pr[nt][e] * vsc[nt][e & 1] : 0.f;
        const uint32_t pa[4] = {pack_half2(pw[0][0], pw[0][1]), pack_half2(pw[0][2], pw[0][3]),
                                pack_half2(pw[1][0], pw[1][1]), pack_half2(pw[1][2], pw[1][3])};
        w_lo = w_lo * al_lo + (half2_sum(pa[0]) + half2_sum(pa[2]));
        if (ROWS16) w_hi = w_hi * al_hi + (half2_sum(pa[1]) + half2_sum(pa[3]));
        // rescale O only when some row's running max rose in this block (alpha is exactly 1 otherwise)
        if (__any_sync(0xffffffffu, al_lo != 1.f || (ROWS16 && al_hi != 1.f))) {
#pragma unroll
            for (int nt = 0; nt < 16; ++nt) {
                o[nt][0] *= al_lo;
                o[nt][1] *= al_lo;
                if (ROWS16) {
                    o[nt][2] *= al_hi;
                    o[nt][3] *= al_hi;
                }
            }
        }
        // O += P' C_V over chunk pairs; matrices (tokens 0-7 | 8-15) x (chunk cc | cc+1), transposed:
        // a word holds (token 2tq: dims 2g, 2g+1; token 2tq+1: dims 2g, 2g+1) of its chunk.
#pragma unroll
        for (int cc = 0; cc < 8; cc += 2) {
            uint32_t w[4];
            ldsm_x4_t(vt + code_off(rr + (mi & 1) * 8, 16 * (cc + (mi >> 1))), w);
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const uint32_t lo = w[2 * u] ^ 0x80808080u, hi = w[2 * u + 1] ^ 0x80808080u;
                mma_16816(o[2 * (cc + u)], pa, codes2_to_half2(lo, 0x4240u), codes2_to_half2(hi, 0x4240u));
                mma_16816(o[2 * (cc + u) + 1], pa, codes2_to_half2(lo, 0x4341u), codes2_to_half2(hi, 0x4341u));
            }
        }
        }  // not the transposed form
        __syncwarp();
        if (li + kQStages < nloc) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(li + kQStages);
            }
            ++issued;
        }
    }
    pdl_trigger();
    if (!ok) {
        if (lane == 0) {
            atomicOr(a.status, PKV_DEV_TIMEOUT);
            for (int li = max(0, issued - kQStages); li < issued; ++li)
                mbar_wait(bar0 + 8 * (li % kQStages), (uint32_t)(li / kQStages) & 1u);
        }
        __syncwarp();
    }
    if constexpr (kT) {
        // sums over the block's tokens: lanes of the same tq (query heads 2tq, 2tq + 1)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) {
            l_lo += __shfl_xor_sync(0xffffffffu, l_lo, off);
            l_hi += __shfl_xor_sync(0xffffffffu, l_hi, off);
            w_lo += __shfl_xor_sync(0xffffffffu, w_lo, off);
            w_hi += __shfl_xor_sync(0xffffffffu, w_hi, off);
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            o[c][0] -= kCodeBias * w_lo;
            o[c][1] -= kCodeBias * w_hi;
            o[c][2] -= kCodeBias * w_lo;
            o[c][3] -= kCodeBias * w_hi;
        }
    } else {
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    w_lo += __shfl_xor_sync(0xffffffffu, w_lo, 1);
    w_lo += __shfl_xor_sync(0xffffffffu, w_lo, 2);
    if (ROWS16) {
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
        w_hi += __shfl_xor_sync(0xffffffffu, w_hi, 1);
        w_hi += __shfl_xor_sync(0xffffffffu, w_hi, 2);
    }
    // take the codes' bias off the outputs: sum over tokens of weight * 1,152, the same for every dimension
#pragma unroll
    for (int nt = 0; nt < 16; ++nt) {
        o[nt][0] -= kCodeBias * w_lo;
        o[nt][1] -= kCodeBias * w_lo;
        if (ROWS16) {
            o[nt][2] -= kCodeBias * w_hi;
            o[nt][3] -= kCodeBias * w_hi;
        }
    }
    }  // not the transposed form

    // ---- merge the four warps (warp order); O tile nt = 2 * chunk + parity holds dims 16 chunk + 4tq + 2e + parity
    __syncthreads();
    {
        float* mo = reinterpret_cast<float*>(smem + kQSmMergeO) + warp * kQRows * kQMergeStride;
        float* mml = reinterpret_cast<float*>(smem + kQSmMergeML) + warp * kQRows * 2;
        if constexpr (kT) {
            // O^T element (chunk c, e): dim 16c + 2g + (e >> 1), query head 2tq + (e & 1)
            const int h0r = 2 * tq, h1r = 2 * tq + 1;
#pragma unroll
            for (int c = 0; c < 8; ++c) {
                const int d0 = 16 * c + 2 * g;
                if (h0r < R) {
                    mo[h0r * kQMergeStride + d0] = o[c][0];
                    mo[h0r * kQMergeStride + d0 + 1] = o[c][2];
                }
                if (h1r < R) {
                    mo[h1r * kQMergeStride + d0] = o[c][1];
                    mo[h1r * kQMergeStride + d0 + 1] = o[c][3];
                }
            }
            if (g == 0) {
                if (h0r < R) {
                    mml[2 * h0r] = m_lo;
                    mml[2 * h0r + 1] = l_lo;
                }
                if (h1r < R) {
                    mml[2 * h1r] = m_hi;
                    mml[2 * h1r + 1] = l_hi;
                }
            }
        } else {
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int d0 = 16 * (nt >> 1) + 4 * tq + (nt & 1);
            mo[g * kQMergeStride + d0] = o[nt][0];
            mo[g * kQMergeStride + d0 + 2] = o[nt][1];
            if (ROWS16) {
                mo[(g + 8) * kQMergeStride + d0] = o[nt][2];
                mo[(g + 8) * kQMergeStride + d0 + 2] = o[nt][3];
            }
        }
        if (tq == 0) {
            mml[2 * g] = m_lo;
            mml[2 * g + 1] = l_lo;
            if (ROWS16) {
                mml[2 * (g + 8)] = m_hi;
                mml[2 * (g + 8) + 1] = l_hi;
            }
        }
        }  // not the transposed form
    }
    __syncthreads();
    const int d = threadIdx.x;
    const float* mo = reinterpret_cast<const float*>(smem + kQSmMergeO);
    const float* mml = reinterpret_cast<const float*>(smem + kQSmMergeML);
    for (int row = 0; row < R; ++row) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kQWarps; ++w) M = fmaxf(M, mml[(w * kQRows + row) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kQWarps; ++w) {
            const float wt = exp2f(mml[(w * kQRows + row) * 2] - M);
            L = fmaf(wt, mml[(w * kQRows + row) * 2 + 1], L);
            O = fmaf(wt, mo[(w * kQRows + row) * kQMergeStride + d], O);
        }
        if (!CASCADE && nparts == 1) {
            a.out[rh(row) * kHeadDim + d] = __float2half_rn(O * (1.f / L));
        } else {
            const int64_t slot = rh(row) * a.ws_parts + slot_p;
            a.ws_o[slot * kHeadDim + d] = O;
            if (d == 0) {
                a.ws_ml[slot * 2] = M;
                a.ws_ml[slot * 2 + 1] = L;
            }
        }
    }
    if (CASCADE) {
        // count the partial of each of the CTA's rows (the counter the private keys' launch counts with, which
        // may run beside this one); a row whose partials are all in is merged here, in partition order, by the
        // same arithmetic as the private kernel's merge
        unsigned int* flags = reinterpret_cast<unsigned int*>(smem + kQSmFlag);
        __syncthreads();
        if (threadIdx.x < nseq) {
            const int rr = r + threadIdx.x;
            // the row's partitions: the prefix's nparts, then its private keys cut as the private kernel cuts them
            const int n = __ldg(a.ctx_lens + rr) - ctx;
            int npriv = 0;
            if (n > 0) {
                const int np = (n + a.part_tokens - 1) / a.part_tokens;
                const int sp = ((n + np - 1) / np + kBlockSize - 1) / kBlockSize * kBlockSize;
                npriv = (n + sp - 1) / sp;
            }
            const unsigned int total = (unsigned int)(nparts + npriv);
            unsigned int* cnt = a.counters + ((int64_t)rr * a.num_kv_heads + kvh) * a.slices + c;
            flags[threadIdx.x] = q_atomic_add_acq_rel(cnt, 1u) == total - 1u ? total : 0u;
        }
        __syncthreads();
        for (int row = 0; row < R; ++row) {
            const int np_all = (int)flags[row / hpr];
            if (np_all == 0) continue;
            const int64_t base = rh(row) * a.ws_parts;
            float M = -INFINITY;
            for (int q = 0; q < np_all; ++q) M = fmaxf(M, __ldcg(a.ws_ml + (base + q) * 2));
            float L = 0.f, O = 0.f;
            for (int q = 0; q < np_all; ++q) {
                const float wt = exp2f(__ldcg(a.ws_ml + (base + q) * 2) - M);
                L = fmaf(wt, __ldcg(a.ws_ml + (base + q) * 2 + 1), L);
                O = fmaf(wt, __ldcg(a.ws_o + (base + q) * kHeadDim + d), O);
            }
            a.out[rh(row) * kHeadDim + d] = __float2half_rn(O * (1.f / L));
        }
        __syncthreads();
        if (threadIdx.x < nseq && flags[threadIdx.x])
            a.counters[((int64_t)(r + threadIdx.x) * a.num_kv_heads + kvh) * a.slices + c] = 0u;
        return;
    }
    if (nparts == 1) return;

    __syncthreads();
    unsigned int* counter = a.counters + ((int64_t)r * a.num_kv_heads + kvh) * a.slices + c;
    unsigned int* flag = reinterpret_cast<unsigned int*>(smem + kQSmFlag);
    if (threadIdx.x == 0) *flag = q_atomic_add_acq_rel(counter, 1u) == (unsigned int)(nparts - 1);
    __syncthreads();
    if (!*flag) return;
    for (int row = 0; row < R; ++row) {
        const int64_t base = rh(row) * a.ws_parts;
        float M = -INFINITY;
        for (int q = 0; q < nparts; ++q) M = fmaxf(M, __ldcg(a.ws_ml + (base + q) * 2));
        float L = 0.f, O = 0.f;
        for (int q = 0; q < nparts; ++q) {
            const float wt = exp2f(__ldcg(a.ws_ml + (base + q) * 2) - M);
            L = fmaf(wt, __ldcg(a.ws_ml + (base + q) * 2 + 1), L);
            O = fmaf(wt, __ldcg(a.ws_o + (base + q) * kHeadDim + d), O);
        }
        a.out[rh(row) * kHeadDim + d] = __float2half_rn(O * (1.f / L));
    }
    __syncthreads();
    if (threadIdx.x == 0) *counter = 0u;
}

template <bool ROWS16, bool CASCADE>
cudaError_t launch_i8(const CUtensorMap& tmap, const I8Args& a, dim3 grid, cudaStream_t stream, int pdl)
{
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_i8_kernel<ROWS16, CASCADE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kQSmAlloc);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kQWarps * 32);
    cfg.dynamicSmemBytes = kQSmAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_i8_kernel<ROWS16, CASCADE>, tmap, a);
}

}  // namespace

cudaError_t launch_kv_append_i8(const PoolGeom& g, int layer, const void* k, const void* v, const int64_t* slots,
                                int num_tokens, unsigned int* status, cudaStream_t stream)
{
    if (num_tokens == 0) return cudaSuccess;
    const int64_t threads_total = 2LL * g.num_heads * num_tokens * 32;
    const int threads = 256;
    const int64_t blocks = (threads_total + threads - 1) / threads;
    kv_append_i8_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
        const_cast<char*>(g.base), g.block_bytes, (int64_t)layer * g.layer_bytes, g.kv_bytes, g.num_heads,
        static_cast<const __half*>(k), static_cast<const __half*>(v), slots, num_tokens, g.num_blocks * kBlockSize,
        status);
    return cudaGetLastError();
}

// Map over an 8-bit pool's code tiles: [block][layer][2 x heads tiles, 2,112 B apart][16 rows][128 bytes];
// one box is a tile's 2,048 code bytes, copied with the 128-byte swizzle.
bool encode_i8_tmap(const PoolGeom& g, TensorMap128* out, std::string* err)
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
    const cuuint64_t strides[4] = {(cuuint64_t)kHeadDim, (cuuint64_t)kTileBytesI8, (cuuint64_t)g.layer_bytes,
                                   (cuuint64_t)g.block_bytes};
    const cuuint32_t box[5] = {(cuuint32_t)kHeadDim, (cuuint32_t)kBlockSize, 1, 1, 1};
    const cuuint32_t estr[5] = {1, 1, 1, 1, 1};
    CUresult r = encode(reinterpret_cast<CUtensorMap*>(out->bytes), CU_TENSOR_MAP_DATA_TYPE_UINT8, 5,
                        const_cast<char*>(g.base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        if (err) *err = "cuTensorMapEncodeTiled failed";
        return false;
    }
    return true;
}

cudaError_t launch_decode_i8(const PoolGeom& g, const TensorMap128& i8_tmap, int layer, const void* q,
                             const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                             float scale, void* out, const DecodeWs& ws, int partition_tokens, const void* k_new,
                             const void* v_new, const int64_t* slots, unsigned int* status, cudaStream_t stream,
                             int pdl, const int32_t* group_start, const int32_t* group_blocks, int num_groups)
{
    if (num_seqs == 0) return cudaSuccess;
    I8Args a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __half*>(q);
    a.out = static_cast<__half*>(out);
    a.tables = tables;
    a.max_blocks = max_blocks;
    a.ctx_lens = ctx_lens;
    a.pool = const_cast<char*>(g.base);
    a.block_bytes = g.block_bytes;
    a.head_off = (int64_t)layer * g.layer_bytes;
    a.kv_bytes = g.kv_bytes;
    a.num_blocks = g.num_blocks;
    a.layer = layer;
    a.num_kv_heads = g.num_heads;
    a.num_q_heads = g.num_q_heads;
    a.group = g.group;
    a.slices = decode_group_slices(g.group);
    a.rows = g.group / a.slices;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.ws_o = ws.o;
    a.ws_ml = ws.ml;
    a.counters = ws.counters;
    a.max_parts = decode_max_parts(max_blocks, partition_tokens);
    a.ws_parts = ws.parts;
    a.part_tokens = partition_tokens;
    a.k_new = static_cast<const __half*>(k_new);
    a.v_new = static_cast<const __half*>(v_new);
    a.slots = slots;
    a.append = k_new != nullptr;
    a.no_wait = pdl == 2;
    a.status = status;
    a.group_start = num_groups > 0 ? group_start : nullptr;
    a.group_blocks = num_groups > 0 ? group_blocks : nullptr;
    a.num_groups = num_groups;
    CUtensorMap tmap;
    static_assert(sizeof(tmap) == sizeof(i8_tmap.bytes), "tensor map size");
    memcpy(&tmap, i8_tmap.bytes, sizeof(tmap));
    a.part_z = a.group_start != nullptr;
    const dim3 grid = a.part_z ? dim3(a.num_kv_heads * a.slices, num_seqs, a.max_parts)
                               : dim3(a.max_parts, a.num_kv_heads * a.slices, num_seqs);
    return a.rows > 8 ? launch_i8<true, false>(tmap, a, grid, stream, pdl)
                      : launch_i8<false, false>(tmap, a, grid, stream, pdl);
}

cudaError_t launch_decode_i8_shared_prefix(const PoolGeom& g, const TensorMap128& i8_tmap, int layer, const void* q,
                                           const int32_t* tables, int max_blocks, const int32_t* ctx_lens,
                                           const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                                           int max_group_rows, float scale, void* out, const DecodeWs& ws,
                                           int partition_tokens, unsigned int* status, cudaStream_t stream)
{
    if (num_groups == 0) return cudaSuccess;
    I8Args a;
    memset(&a, 0, sizeof(a));
    a.q = static_cast<const __half*>(q);
    a.out = static_cast<__half*>(out);
    a.ctx_lens = ctx_lens;
    a.tables = tables;
    a.max_blocks = max_blocks;
    a.pool = const_cast<char*>(g.base);
    a.block_bytes = g.block_bytes;
    a.head_off = (int64_t)layer * g.layer_bytes;
    a.kv_bytes = g.kv_bytes;
    a.num_blocks = g.num_blocks;
    a.layer = layer;
    a.num_kv_heads = g.num_heads;
    a.num_q_heads = g.num_q_heads;
    // fragment rows: the a.rows query heads of one slice of a K/V head's group, for as many rows of the group
    // as 16 fragment rows hold
    a.group = g.group;
    a.slices = decode_group_slices(g.group);
    a.rows = g.group / a.slices;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.ws_o = ws.o;
    a.ws_ml = ws.ml;
    a.counters = ws.counters;
    a.max_parts = decode_max_parts(max_blocks, partition_tokens);
    a.ws_parts = ws.parts;
    a.part_tokens = partition_tokens;
    a.status = status;
    a.group_start = group_start;
    a.group_blocks = group_blocks;
    a.num_groups = num_groups;
    const int rows_per_cta = kQRows / a.rows;
    a.max_slices = (max_group_rows + rows_per_cta - 1) / rows_per_cta;
    CUtensorMap tmap;
    memcpy(&tmap, i8_tmap.bytes, sizeof(tmap));
    const dim3 grid(a.max_parts, g.num_heads * a.slices, num_groups * a.max_slices);
    return launch_i8<true, true>(tmap, a, grid, stream, 0);
}

}  // namespace pkv
