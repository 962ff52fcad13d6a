// pkv_decode_group.cu — decode attention when each K/V head serves a group of
// query heads (grouped-query and multi-query attention: "Inference
// Infrastructure" (seeitflow), the KV cache arithmetic, where 8 K/V heads
// serve all query heads and the cache holds only the K/V heads; "The inference
// engine" (wpnews), the section on grouped-query attention). Query head h
// reads K/V head h / G, G = query heads / K/V heads.
//
// Work unit: one CTA per (partition p, K/V head k with query-head slice c,
// row r). The CTA computes R = G / slices query heads, k*G + c*R .. + R - 1,
// all from one copy of each K/V block (slices = 1 whenever G <= 16, so every
// K/V byte is read from memory once per group). Its four warps stream the
// partition's blocks round-robin (warp w takes blocks w, w+4, ...), each with
// its own two-stage ring filled by TMA: one copy per 4 KB K or V tile, whose
// 16 token rows land as 32 rows of 128 B (token t's dimensions 0-63 in row
// 2t, 64-127 in row 2t+1) with the 128-byte swizzle.
//
// Per block a warp runs the group's attention on the tensor cores with
// mma.sync m16n8k16 (FP16 operands, FP32 accumulation): S = Q K^T with the R
// query heads as the M = 16 rows (rows past R are zero) and the block's 16
// tokens as two N = 8 tiles, then an online softmax in the log2 domain on the
// S fragments, and O += P V with P taken straight from the S fragments as the
// A operand (rounded to FP16) and V as sixteen N = 8 tiles of dimensions.
// K and V fragments come from shared memory with ldmatrix; the swizzle makes
// those reads free of bank conflicts. A warp then holds (m, l, O) of its
// blocks for every query head of the CTA; the four warps merge through shared
// memory in warp order.
//
// Split-K across partitions follows the one-head kernel: each CTA writes its
// heads' un-normalised output, max and sum to the workspace; the CTA that
// brings the (row, K/V head, slice) counter to the row's partition count
// merges all partitions in partition order and resets the counter. The
// partition plan depends only on ctx_len and partition_tokens, so a row's
// result does not depend on the rest of the batch.
//
// With `append`, the CTA with c == 0 that holds a row's last partition writes
// the row's new K/V (k_new / v_new row r, K/V head k) into slot_mapping[r], and
// the warp that streams the new token's block patches the new rows into its
// shared-memory copy, so the query sees its own new key as if the append had
// run first. Rows of a row's last block past ctx_len are zeroed in shared
// memory before P V: P is zero there, but the pool may hold anything (even
// NaN) in unwritten slots, and 0 x NaN would poison the tensor-core sum.
//
// Cascade mode (CASCADE = true, pools with one query head per K/V head): the
// MMA rows are up to 16 batch rows of a group that share their leading
// blocks (a shared prompt prefix: "The inference engine" (wpnews), "Paging
// turns variable sequences into block tables": sequences may point at the
// same immutable prefix blocks), all for one head. A CTA handles one split-K
// partition lying wholly inside the shared prefix, so each shared K/V tile is
// read from memory once per group instead of once per row; it writes each
// row's partial and counts it. The one-head kernel then computes the rows'
// remaining partitions and merges all of them.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cstring>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {
namespace {

constexpr int kGWarps = 4;                   // warps per CTA
constexpr int kGStages = 2;                  // ring stages per warp
constexpr int kGStage = 2 * kTileBytes;      // K tile + V tile of one block (8 KB)
constexpr int kGRows = 16;                   // query heads per CTA at most (the MMA's M)
constexpr int kGMaxBlocks = kMaxPartitionTiles / kBlockSize;
constexpr int kGMergeStride = kHeadDim + 4;  // floats per row of the merge scratch (bank-conflict padding)

// shared memory, offsets from a 1,024-byte aligned base
constexpr int kGSmRing = 0;                                       // [warp][stage] 8 KB
constexpr int kGSmIds = kGSmRing + kGWarps * kGStages * kGStage;  // [kGMaxBlocks] int32
constexpr int kGSmBars = kGSmIds + kGMaxBlocks * 4;               // [warp][stage] u64
constexpr int kGSmFlag = kGSmBars + kGWarps * kGStages * 8;
constexpr int kGSmBytes = kGSmFlag + 4 * kGRows;  // the last-arrival flag; cascade: one per row
constexpr int kGSmAlloc = kGSmBytes + 1024;
// the warps' merge scratch, over the ring once every copy has landed
constexpr int kGSmMergeO = 0;                                          // [warp][16][kGMergeStride] f32
constexpr int kGSmMergeML = kGWarps * kGRows * kGMergeStride * 4;     // [warp][16][2] f32
static_assert(kGSmMergeML + kGWarps * kGRows * 8 <= kGSmIds, "merge scratch fits in the ring");

struct GroupArgs {
    const __half* q;   // [B][num_q_heads][128]
    __half* out;       // [B][num_q_heads][128]
    const int32_t* tables;
    int max_blocks;
    const int32_t* ctx_lens;
    char* pool;
    int64_t block_bytes;
    int64_t head_off;  // layer * layer_bytes
    int64_t kv_bytes;
    int64_t num_blocks;
    int layer;
    int num_kv_heads;
    int num_q_heads;
    int group;         // G
    int rows;          // R: query heads per CTA
    int slices;        // G / R
    float scale_log2;
    float* ws_o;       // [B][num_q_heads][max_parts][128]
    float* ws_ml;      // [B][num_q_heads][max_parts][2]
    unsigned int* counters;  // [B][num_kv_heads * slices], zero between launches
    int max_parts;
    int ws_parts;            // partial slots per (row, query head)
    int part_tokens;
    const __half* k_new;     // [B][num_kv_heads][128] when append
    const __half* v_new;
    const int64_t* slots;    // [B] when append
    int append;
    int no_wait;             // launched after a kernel whose results it does not read: skip the dependency wait
    unsigned int* status;
    // cascade: rows [group_start[i], group_start[i+1]) share their first group_blocks[i] blocks. In CASCADE mode
    // the kernel computes those shared partitions for the group's rows at once; otherwise (group_start set) a
    // row's partitions cover only the keys after its group's shared prefix.
    const int32_t* group_start;
    const int32_t* group_blocks;
    int num_groups;
    int max_slices;          // CASCADE: ceil(largest group / sequences per CTA)
};

// Byte offset of 16-byte chunk ch (dimensions 8ch .. 8ch+7) of token t in a
// K or V tile in shared memory: row r = 2t + ch / 8 of 128 B, and the
// 128-byte swizzle puts chunk j of row r at position j ^ (r % 8).
__device__ __forceinline__ uint32_t sw_off(int t, int ch)
{
    const int r = 2 * t + (ch >> 3);
    return (uint32_t)(r * 128 + (((ch & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ unsigned int group_atomic_add_acq_rel(unsigned int* p, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// ROWS16: some row of the CTA sits in fragment rows 8..15 (R > 8).
template <bool ROWS16, bool CASCADE>
__global__ void __launch_bounds__(kGWarps * 32) decode_group_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                     const GroupArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    const int p = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int g = lane >> 2, tq = lane & 3;  // fragment row and column pair of this lane
    // The CTA's R fragment rows: query heads h0 .. h0 + hpr - 1 (hpr = a.rows, one slice of K/V head kvh's
    // group) of rows r .. r + nseq - 1; fragment row f is query head h0 + f % hpr of row r + f / hpr. Normal
    // mode: one row (nseq = 1). CASCADE: as many rows of one group as 16 fragment rows hold, over the
    // group's shared prefix, so each shared tile is read once for all of them.
    const int hpr = a.rows;
    const int kvh = blockIdx.y / a.slices, c = blockIdx.y % a.slices;
    const int h0 = kvh * a.group + c * hpr;
    int r, R, nseq, ctx, nparts, span, tok_lo, slot_p;
    // Cascade: the private keys' launch reads nothing this grid writes except through the split-K counters,
    // so it may start beside this one at once (whichever partial of a row arrives last merges the row)
    if (CASCADE) pdl_trigger();
    if (CASCADE) {
        const int spc = kGRows / hpr;  // rows per CTA
        const int grp = blockIdx.z / a.max_slices, sl = blockIdx.z % a.max_slices;
        const int row0 = __ldg(a.group_start + grp), row_end = __ldg(a.group_start + grp + 1);
        r = row0 + sl * spc;
        nseq = min(spc, row_end - r);
        if (nseq <= 0) return;
        R = nseq * hpr;
        ctx = __ldg(a.group_blocks + grp) * kBlockSize;  // the shared prefix: full blocks, valid for every row
        span = a.part_tokens;
        nparts = (ctx + span - 1) / span;  // the prefix partitioned on its own
        if (p >= nparts) return;
        tok_lo = p * span;
        slot_p = p;
    } else {
        r = blockIdx.z;
        nseq = 1;
        R = hpr;
        // the row's length and (cascade) its group's shared prefix: independent loads, both issued before
        // either is used (one memory round trip for a short cascade row's CTA, not two)
        ctx = __ldg(a.ctx_lens + r);
        // Cascade's other half: keys [0, S) of the row's group's shared prefix were partitioned on their own
        // (slots 0 .. nsh - 1, computed already); this CTA takes partition p of [S, ctx), slot nsh + p.
        int S = 0;
        if (a.group_start) {  // the row's group, by binary search over the group starts
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
        // As few partitions as part_tokens allows, of equal length in whole blocks (a row of 2,300 keys: 768,
        // 768, 764 rather than 1,024, 1,024, 252), so that no short partition's CTA trails the launch. The plan
        // depends only on ctx, S and part_tokens: a row's result is the same in any batch of the same grouping.
        if (ctx <= S) {  // the group's shared prefix must lie below the row's newest token
            if (p == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_CTX);
            return;
        }
        const int nsh = (S + a.part_tokens - 1) / a.part_tokens;
        const int np = (ctx - S + a.part_tokens - 1) / a.part_tokens;
        span = ((ctx - S + np - 1) / np + kBlockSize - 1) / kBlockSize * kBlockSize;  // <= part_tokens
        tok_lo = S + p * span;
        if (tok_lo >= ctx) return;
        nparts = nsh + (ctx - S + span - 1) / span;
        slot_p = nsh + p;
    }
    // query / output row of fragment row f, as an index of [rows][query heads]
    auto rh = [&](int f) { return (int64_t)(r + f / hpr) * a.num_q_heads + h0 + f % hpr; };
    const int blk_lo = tok_lo / kBlockSize;
    const int blk_hi = (min(tok_lo + span, ctx) + kBlockSize - 1) / kBlockSize;
    const int count = blk_hi - blk_lo;  // <= kGMaxBlocks (partition_tokens <= 4,096, a multiple of 64)

    int32_t* ids = reinterpret_cast<int32_t*>(smem + kGSmIds);
    const int32_t* trow = a.tables + (int64_t)r * a.max_blocks;
    bool bad = false;
    for (int i = threadIdx.x; i < count; i += kGWarps * 32) {
        const int id = __ldg(trow + blk_lo + i);
        ids[i] = id;
        bad |= id < 0 || (int64_t)id >= a.num_blocks;
    }
    const uint32_t bar0 = sb + kGSmBars + warp * kGStages * 8;
    if (lane == 0) {
        for (int s = 0; s < kGStages; ++s) mbar_init(bar0 + 8 * s, 1);
        fence_mbar_init();
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        return;
    }

    // This warp's blocks: i = warp + li * 4, li < nloc.
    const int nloc = count > warp ? (count - warp + kGWarps - 1) / kGWarps : 0;
    const uint32_t ring = sb + kGSmRing + warp * kGStages * kGStage;
    auto issue = [&](int li) {
        const int s = li % kGStages;
        const int id = ids[warp + li * kGWarps];
        const uint32_t dst = ring + s * kGStage, bar = bar0 + 8 * s;
        mbar_arrive_expect_tx(bar, kGStage);
        const int tile = a.layer * 2 * a.num_kv_heads + kvh;  // K tile of (layer, head); V is num_kv_heads later
        tma_load_5d(dst, &tmap, 0, 0, 0, tile, id, bar);
        tma_load_5d(dst + kTileBytes, &tmap, 0, 0, 0, tile + a.num_kv_heads, id, bar);
    };
    int issued = min(nloc, kGStages);
    if (lane == 0)
        for (int li = 0; li < issued; ++li) issue(li);

    // Only lengths, tables and this layer's K/V were read so far; with a programmatic dependency on the
    // previous layer's kernel, wait for it before reading q or the new K/V and touching the workspace.
    // Without the wait (no_wait), one CTA still waits: a cascade's private launch then ends only after the shared
    // launch it runs beside, so work after the call in the stream finds both done.
    if (!a.no_wait || (a.group_start && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)) pdl_wait();

    // The new token (position ctx - 1) is the last token of the partition's last block.
    const int new_t = (ctx - 1) % kBlockSize, new_i = (ctx - 1) / kBlockSize - blk_lo;
    int patch_li = -1;
    uint4 patch = make_uint4(0, 0, 0, 0);  // lanes 0-15: K chunk `lane`, lanes 16-31: V chunk `lane - 16`
    if (!CASCADE && a.append && slot_p == nparts - 1) {
        const int64_t slot = __ldg(a.slots + r);
        const int32_t tb = __ldg(trow + (ctx - 1) / kBlockSize);
        const bool consistent =
            tb >= 0 && (int64_t)tb < a.num_blocks && slot == (int64_t)tb * kBlockSize + new_t;
        if (!consistent) {
            if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_SLOT);
        } else {
            const uint4* src = reinterpret_cast<const uint4*>((lane < 16 ? a.k_new : a.v_new) +
                                                              ((int64_t)r * a.num_kv_heads + kvh) * kHeadDim);
            if (warp == new_i % kGWarps) {
                patch_li = new_i / kGWarps;
                patch = __ldg(src + (lane & 15));
            }
            if (c == 0 && warp == 0) {  // the global write, for later steps
                char* dst = a.pool + slot / kBlockSize * a.block_bytes + a.head_off + (int64_t)kvh * kTileBytes +
                            (slot % kBlockSize) * 256 + (lane & 15) * 16 + (lane < 16 ? 0 : a.kv_bytes);
                *reinterpret_cast<uint4*>(dst) = __ldg(src + (lane & 15));
            }
        }
    }

    // Q as the A operand: rows = the CTA's fragment rows (zero past R), k = dims.
    uint32_t qa[8][4];
    {
        const bool lo_ok = g < R, hi_ok = ROWS16 && g + 8 < R;
        const uint32_t* qlo = reinterpret_cast<const uint32_t*>(a.q + (lo_ok ? rh(g) : 0) * kHeadDim);
        const uint32_t* qhi = reinterpret_cast<const uint32_t*>(a.q + (hi_ok ? rh(g + 8) : 0) * kHeadDim);
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            qa[ks][0] = lo_ok ? __ldg(qlo + 8 * ks + tq) : 0u;
            qa[ks][1] = hi_ok ? __ldg(qhi + 8 * ks + tq) : 0u;
            qa[ks][2] = lo_ok ? __ldg(qlo + 8 * ks + 4 + tq) : 0u;
            qa[ks][3] = hi_ok ? __ldg(qhi + 8 * ks + 4 + tq) : 0u;
        }
    }

    float o[16][4];
#pragma unroll
    for (int dt = 0; dt < 16; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float m_lo = -INFINITY, m_hi = -INFINITY, l_lo = 0.f, l_hi = 0.f;
    const int mi = lane >> 3, rr = lane & 7;  // ldmatrix: this lane addresses row rr of matrix mi
    bool ok = true;
    for (int li = 0; li < nloc; ++li) {
        const int s = li % kGStages;
        const uint32_t kt = ring + s * kGStage, vt = kt + kTileBytes;
        const int nvalid = min(kBlockSize, ctx - (blk_lo + warp + li * kGWarps) * kBlockSize);
        if (!mbar_wait(bar0 + 8 * s, (uint32_t)(li / kGStages) & 1u)) {
            ok = false;
            break;
        }
        if (li == patch_li)
            st_shared_v4((lane < 16 ? kt : vt) + sw_off(new_t, lane & 15), patch);
        if (nvalid < kBlockSize)
            for (int e = lane; e < (kBlockSize - nvalid) * 16; e += 32)
                st_shared_v4(vt + sw_off(nvalid + (e >> 4), e & 15), make_uint4(0, 0, 0, 0));
        __syncwarp();

        // S = Q K^T: k-step ks covers dims 16ks..16ks+15; matrices (tokens 0-7 | 8-15) x (low | high 8 dims).
        // up to 8 query rows: even and odd k-steps accumulate apart (two chains of 4 dependent MMAs per tile
        // instead of one of 8), added at the end; 16 rows keep one chain (their registers are spoken for)
        constexpr bool kSplitS = !ROWS16;
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        float sodd[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
            uint32_t b[4];
            ldsm_x4(kt + sw_off(rr + (mi >> 1) * 8, 2 * ks + (mi & 1)), b);
            mma_16816((kSplitS && (ks & 1)) ? sodd[0] : sacc[0], qa[ks], b[0], b[1]);
            mma_16816((kSplitS && (ks & 1)) ? sodd[1] : sacc[1], qa[ks], b[2], b[3]);
        }
        if (kSplitS) {
#pragma unroll
            for (int nt = 0; nt < 2; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) sacc[nt][e] += sodd[nt][e];
        }
        // fragment element e of tile nt: row g (e < 2) or g + 8, token 8nt + 2tq + (e & 1)
        float sv[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e)
                sv[nt][e] = (nt * 8 + 2 * tq + (e & 1) < nvalid) ? sacc[nt][e] * a.scale_log2 : -INFINITY;
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
        // P as the A operand: k = tokens, tile 0 gives k 0..7, tile 1 k 8..15.
        const uint32_t pa[4] = {pack_half2(pr[0][0], pr[0][1]), pack_half2(pr[0][2], pr[0][3]),
                                pack_half2(pr[1][0], pr[1][1]), pack_half2(pr[1][2], pr[1][3])};
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            o[dt][0] *= al_lo;
            o[dt][1] *= al_lo;
            if (ROWS16) {
                o[dt][2] *= al_hi;
                o[dt][3] *= al_hi;
            }
        }
        // O += P V: dimension tiles 2dp and 2dp+1; matrices (tokens 0-7 | 8-15) x (tile 2dp | 2dp+1), transposed.
#pragma unroll
        for (int dp = 0; dp < 8; ++dp) {
            uint32_t b[4];
            ldsm_x4_t(vt + sw_off(rr + (mi & 1) * 8, 2 * dp + (mi >> 1)), b);
            mma_16816(o[2 * dp], pa, b[0], b[1]);
            mma_16816(o[2 * dp + 1], pa, b[2], b[3]);
        }
        __syncwarp();
        if (li + kGStages < nloc) {
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(li + kGStages);
            }
            ++issued;
        }
    }
    pdl_trigger();
    if (!ok) {
        if (lane == 0) {
            atomicOr(a.status, PKV_DEV_TIMEOUT);
            // copies still in flight land before the ring is reused (each stage's latest copy)
            for (int li = max(0, issued - kGStages); li < issued; ++li)
                mbar_wait(bar0 + 8 * (li % kGStages), (uint32_t)(li / kGStages) & 1u);
        }
        __syncwarp();
    }
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
    l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
    if (ROWS16) {
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    }

    // ---- merge the four warps (warp order) through shared memory
    __syncthreads();
    {
        float* mo = reinterpret_cast<float*>(smem + kGSmMergeO) + warp * kGRows * kGMergeStride;
        float* mml = reinterpret_cast<float*>(smem + kGSmMergeML) + warp * kGRows * 2;
#pragma unroll
        for (int dt = 0; dt < 16; ++dt) {
            *reinterpret_cast<float2*>(mo + g * kGMergeStride + dt * 8 + 2 * tq) = make_float2(o[dt][0], o[dt][1]);
            if (ROWS16)
                *reinterpret_cast<float2*>(mo + (g + 8) * kGMergeStride + dt * 8 + 2 * tq) =
                    make_float2(o[dt][2], o[dt][3]);
        }
        if (tq == 0) {
            mml[2 * g] = m_lo;
            mml[2 * g + 1] = l_lo;
            if (ROWS16) {
                mml[2 * (g + 8)] = m_hi;
                mml[2 * (g + 8) + 1] = l_hi;
            }
        }
    }
    __syncthreads();
    // thread t merges output dimension t % 128 of rows t / 128, t / 128 + kRowStep, ...
    constexpr int kRowStep = kGWarps * 32 / kHeadDim;
    static_assert(kGWarps * 32 % kHeadDim == 0, "whole rows per pass");
    const int d = threadIdx.x % kHeadDim, row0 = threadIdx.x / kHeadDim;
    const float* mo = reinterpret_cast<const float*>(smem + kGSmMergeO);
    const float* mml = reinterpret_cast<const float*>(smem + kGSmMergeML);
    for (int row = row0; row < R; row += kRowStep) {
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kGWarps; ++w) M = fmaxf(M, mml[(w * kGRows + row) * 2]);
        float L = 0.f, O = 0.f;
#pragma unroll
        for (int w = 0; w < kGWarps; ++w) {
            const float wt = exp2f(mml[(w * kGRows + row) * 2] - M);  // 0 for a warp without blocks
            L = fmaf(wt, mml[(w * kGRows + row) * 2 + 1], L);
            O = fmaf(wt, mo[(w * kGRows + row) * kGMergeStride + d], O);
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
        // count the partial of each of the CTA's rows (one counter per row, K/V head and slice: the one the
        // private keys' kernel counts with, which may run beside this one); a row whose partials are all in
        // is merged here, in partition order, by the same arithmetic as the private kernel's merge
        unsigned int* flags = reinterpret_cast<unsigned int*>(smem + kGSmFlag);
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
            flags[threadIdx.x] = group_atomic_add_acq_rel(cnt, 1u) == total - 1u ? total : 0u;
        }
        __syncthreads();
        for (int row = row0; row < R; row += kRowStep) {
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
            // the private kernel's final step, so that a row's result does not depend on which launch merged it
            // (pools with one query head per K/V head: decode_kernel divides; grouped heads: this kernel's merge)
            a.out[rh(row) * kHeadDim + d] = __float2half_rn(a.group == 1 ? O / L : O * (1.f / L));
        }
        __syncthreads();
        if (threadIdx.x < nseq && flags[threadIdx.x])
            a.counters[((int64_t)(r + threadIdx.x) * a.num_kv_heads + kvh) * a.slices + c] = 0u;
        return;
    }
    if (nparts == 1) return;

    // ---- split-K: the last partition of (row, K/V head, slice) to arrive merges all of them in order
    __syncthreads();
    unsigned int* counter = a.counters + ((int64_t)r * a.num_kv_heads + kvh) * a.slices + c;
    unsigned int* flag = reinterpret_cast<unsigned int*>(smem + kGSmFlag);
    if (threadIdx.x == 0) *flag = group_atomic_add_acq_rel(counter, 1u) == (unsigned int)(nparts - 1);
    __syncthreads();
    if (!*flag) return;
    for (int row = row0; row < R; row += kRowStep) {
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
cudaError_t launch_group(const CUtensorMap& tmap, const GroupArgs& a, dim3 grid, cudaStream_t stream,
                         int pdl = 0)
{
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_group_kernel<ROWS16, CASCADE>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmAlloc);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kGWarps * 32);
    cfg.dynamicSmemBytes = kGSmAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, decode_group_kernel<ROWS16, CASCADE>, tmap, a);
}

}  // namespace

// Map over the pool seen as [num_blocks][layers * 2 * heads tiles][16 tokens][2 halves][64 dims]:
// one box is a whole 4 KB tile, copied as 32 rows of 128 B with the 128-byte swizzle.
bool encode_tile_tmap(const PoolGeom& g, TensorMap128* out, std::string* err)
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
    const cuuint64_t dims[5] = {64, 2, (cuuint64_t)kBlockSize, (cuuint64_t)g.num_layers * 2 * g.num_heads,
                                (cuuint64_t)g.num_blocks};
    const cuuint64_t strides[4] = {128, (cuuint64_t)kHeadDim * 2, (cuuint64_t)kTileBytes, (cuuint64_t)g.block_bytes};
    const cuuint32_t box[5] = {64, 2, (cuuint32_t)kBlockSize, 1, 1};
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

int decode_group_slices(int group)
{
    int s = (group + kGRows - 1) / kGRows;
    while (group % s) ++s;
    return s;
}

cudaError_t launch_decode_group(const PoolGeom& g, const TensorMap128& kv_tmap, int layer, const void* q,
                                const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                                float scale, void* out, const DecodeWs& ws, int partition_tokens, const void* k_new,
                                const void* v_new, const int64_t* slots, unsigned int* status, cudaStream_t stream,
                                int pdl, const int32_t* group_start, const int32_t* group_blocks, int num_groups)
{
    if (num_seqs == 0) return cudaSuccess;
    GroupArgs a;
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
    a.max_slices = 0;
    CUtensorMap tmap;
    static_assert(sizeof(tmap) == sizeof(kv_tmap.bytes), "tensor map size");
    memcpy(&tmap, kv_tmap.bytes, sizeof(tmap));
    const dim3 grid(a.max_parts, a.num_kv_heads * a.slices, num_seqs);
    return a.rows > 8 ? launch_group<true, false>(tmap, a, grid, stream, pdl)
                      : launch_group<false, false>(tmap, a, grid, stream, pdl);
}

cudaError_t launch_decode_shared_prefix(const PoolGeom& g, const TensorMap128& kv_tmap, int layer, const void* q,
                                        const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs,
                                        const int32_t* group_start, const int32_t* group_blocks, int num_groups,
                                        int max_group_rows, float scale, void* out, const DecodeWs& ws,
                                        int partition_tokens, unsigned int* status, cudaStream_t stream)
{
    if (num_groups == 0) return cudaSuccess;
    GroupArgs a;
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
    // fragment rows: the a.rows query heads of one slice of a K/V head's group, for as many rows of the
    // group as 16 fragment rows hold (16 rows of one head each over a pool with one query head per K/V head)
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
    const int rows_per_cta = kGRows / a.rows;
    a.max_slices = (max_group_rows + rows_per_cta - 1) / rows_per_cta;
    (void)num_seqs;
    CUtensorMap tmap;
    memcpy(&tmap, kv_tmap.bytes, sizeof(tmap));
    const dim3 grid(a.max_parts, g.num_heads * a.slices, num_groups * a.max_slices);
    return launch_group<true, true>(tmap, a, grid, stream);
}

}  // namespace pkv
