// pkv_prefill.cu — chunked causal prefill attention over the paged pool on
// the 5th-generation tensor cores (tcgen05, accumulators in TMEM), with K/V
// tiles gathered from the pool's blocks by TMA.
//
// One CTA = (query tile of 128 chunk rows, head, sequence). Query row i of a
// chunk of q_len tokens sits at position ctx - q_len + i and attends keys
// 0..that position ("llm-inference-batching" (faangrind), "Prefill and
// decode share each step": a prompt is prefilled in chunks; "The inference
// engine" (wpnews), "Prefill and decode ask the accelerator for different
// work": prefill attention respects the causal mask). The chunk's own K/V
// are already in the pool (kv_append runs first), so keys come only from
// the pool, 128 at a time (8 blocks).
//
// Two independent pipelines per CTA split the key range: pipe 0 takes the
// first half of the 64-key tiles, pipe 1 the rest (the diagonal tiles), so
// the tensor core works on one pipe's MMAs while the other pipe's softmax
// runs. Each pipe has its own K/V rings, S/P and O in TMEM, MMA issuer and
// softmax warps; at the end the two partial results merge exactly through
// their softmax statistics.
//
// Warp roles (352 threads):
//   warp 0       TMA producers: lanes 0-3, one per (pipe, K|V), each with its
//                own loop: 64-key tiles = 4 blocks x two 64-dim halves (2 KB
//                boxes), into 3-stage rings.
//   warps 1, 2   MMA issuers of pipe 0 / 1 (one elected lane each; warp 1
//                also owns the TMEM allocation): S_j = Q K_j^T into S buffer
//                j%2 (A and B from shared memory), then O += P_j V_j with P
//                read from tensor memory; completion by tcgen05.commit.
//   warps 3-6,   softmax of pipe 0 / 1: thread r owns query row r (TMEM lane
//   7-10         r). Per tile it loads its 64 S values, writes
//                P = 2^(s*scale*log2e - m) in FP16 over the first half of the
//                same S buffer, and keeps the running sum. The running max m
//                is only raised when the tile's max exceeds it by more than 8
//                (a factor 256, far inside FP16/FP32 range); then the row's O
//                and sum are rescaled once the previous P V product has
//                landed. The result is exact up to rounding.
// Shared-memory operands use the 128-byte swizzle: rows of 128 B (64 halves),
// two slabs per 128-wide operand, 8-row groups 1,024 B apart.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_fp16.h>
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


namespace {

constexpr int kRows = 128;     // query rows per CTA (MMA M)
constexpr int kKeys = 64;      // keys per tile (4 blocks)
constexpr int kPipes = 2;      // independent key-range pipelines per CTA
constexpr int kStages = 3;     // K and V ring depth per pipeline
constexpr int kThreads = 352;  // producer warp, 2 MMA issuers, 2 x 4 softmax warps
constexpr int kQBytes = kRows * kHeadDim * 2;        // 32 KB
constexpr int kQSlab = kQBytes / 2;                  // 16 KB: 128 rows x 64 halves
constexpr int kTileOpBytes = kKeys * kHeadDim * 2;   // 16 KB: one 64-key K or V tile
constexpr int kTileSlab = kTileOpBytes / 2;          // 8 KB: 64 rows x 64 halves
constexpr float kRescaleThreshold = 8.f;             // log2 of the largest un-rescaled P (256)

// shared-memory map (offsets from a 1,024-byte aligned base)
constexpr int kSmQ = 0;
constexpr int kSmRing = kQBytes;                            // [pipe][K,V][stage] tiles
constexpr int kSmBars = kSmRing + kPipes * 2 * kStages * kTileOpBytes;
enum Bar { K_FULL = 0, V_FULL = 3, K_EMPTY = 6, V_EMPTY = 9, S_FULL = 12, P_FULL = 14, PV_DONE = 16, MMA_DONE = 18,
           BARS_PER_PIPE = 19 };
constexpr int kBarLx = kPipes * BARS_PER_PIPE;              // the final exchange between the pipes
constexpr int kBarQ = kBarLx + 1;                           // the Q tile is in shared memory
constexpr int kNumBars = kBarLx + 2;
constexpr int kSoftmaxThreads = 128;                        // per pipe
constexpr int kSmTmemSlot = kSmBars + kNumBars * 8;
constexpr int kSmAbort = kSmTmemSlot + 4;
constexpr int kSmBytes = kSmAbort + 12;
constexpr int kSmAlloc = kSmBytes + 1024;                   // slack to align the base

// TMEM columns per pipe (base pipe * 256): two S buffers of 64 fp32 columns
// (P, FP16, overwrites the first 32 columns of its S buffer), then O (128).
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kPipeCols = 256;
constexpr uint32_t kColS = 0;
constexpr uint32_t kColO = 128;

// Instruction descriptors, kind::f16: D = F32 (bit 4), A = B = F16,
// N >> 3 at bit 17, M >> 4 at bit 24; bit 16 makes B MN-major.
constexpr uint32_t kIdescS = (1u << 4) | ((uint32_t)(kKeys >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24);
constexpr uint32_t kIdescPV = (1u << 4) | ((uint32_t)(kHeadDim >> 3) << 17) | ((uint32_t)(kRows >> 4) << 24) |
                              (1u << 16);

struct PrefillArgs {
    const __half* q;         // [T][H][128], token index from q_start
    __half* out;             // [T][H][128]
    const int32_t* q_start;  // [S + 1]
    const int32_t* tables;   // [S][max_blocks]
    const int32_t* ctx_lens; // [S]
    int max_blocks;
    int num_heads;
    int layer;
    int max_q_len;
    int64_t num_blocks;
    float scale_log2;
    unsigned int* status;
};

// Warp-uniform bounded wait: every lane waits, the warp agrees on the
// outcome, and a timeout (or an earlier abort by any warp) stops the warp's
// role loop so that no lane reaches a .sync.aligned instruction alone.
__device__ __forceinline__ bool flag_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* status)
{
    const int lane = threadIdx.x & 31;
    if (__all_sync(0xffffffffu, mbar_try_wait(bar, parity))) return true;  // fast path
    int stop = lane == 0 ? *abort : 0;
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
    const bool ok = __all_sync(0xffffffffu, mbar_wait(bar, parity));
    if (!ok && lane == 0) {
        atomicOr(status, PKV_DEV_TIMEOUT);
        *abort = 1;
    }
    return ok;
}

// Bounded wait of a single thread (the producer lanes run independent loops).
__device__ __forceinline__ bool lane_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* status)
{
    if (mbar_try_wait(bar, parity)) return true;
    if (*abort) return false;
    if (mbar_wait(bar, parity)) return true;
    atomicOr(status, PKV_DEV_TIMEOUT);
    *abort = 1;
    return false;
}

__device__ __forceinline__ uint32_t bar_addr(uint32_t bars, int pipe, int idx)
{
    return bars + 8u * (uint32_t)(pipe * BARS_PER_PIPE + idx);
}

__global__ void __launch_bounds__(kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmap,
                                                               const PrefillArgs a)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    const int qt = blockIdx.x, h = blockIdx.y, s = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // ---- validate this sequence's metadata (all threads agree)
    const int q0 = __ldg(a.q_start + s);
    const int qlen = __ldg(a.q_start + s + 1) - q0;
    const int ctx = __ldg(a.ctx_lens + s);
    if (q0 < 0 || qlen < 1 || qlen > ctx || qlen > a.max_q_len || ctx > a.max_blocks * kBlockSize) {
        if (qt == 0 && h == 0 && threadIdx.x == 0)
            atomicOr(a.status, ctx > a.max_blocks * kBlockSize ? PKV_DEV_BAD_CTX : PKV_DEV_BAD_QLEN);
        return;
    }
    if (qt * kRows >= qlen) return;
    const int rows = min(kRows, qlen - qt * kRows);
    const int p0 = ctx - qlen + qt * kRows;  // position of row 0
    const int pos_max = p0 + rows - 1;
    const int nkt = pos_max / kKeys + 1;     // 64-key tiles
    const int nblk = pos_max / kBlockSize + 1;
    // pipe 0 takes key tiles [0, n0), pipe 1 takes [n0, nkt) (the diagonal ones)
    const int n0 = nkt / 2;
    const int32_t* trow = a.tables + (int64_t)s * a.max_blocks;
    bool bad = false;
    for (int b = threadIdx.x; b < nblk; b += kThreads) {
        const int id = __ldg(trow + b);
        bad |= id < 0 || (int64_t)id >= a.num_blocks;
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        return;
    }

    const uint32_t bars = sb + kSmBars;
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kSmAbort);
    if (threadIdx.x == 0) {
        for (int p = 0; p < kPipes; ++p) {
            for (int i = 0; i < kStages; ++i) {
                mbar_init(bar_addr(bars, p, K_FULL + i), 1);
                mbar_init(bar_addr(bars, p, V_FULL + i), 1);
                mbar_init(bar_addr(bars, p, K_EMPTY + i), 1);
                mbar_init(bar_addr(bars, p, V_EMPTY + i), 1);
            }
            for (int i = 0; i < 2; ++i) {
                mbar_init(bar_addr(bars, p, S_FULL + i), 1);
                mbar_init(bar_addr(bars, p, P_FULL + i), kSoftmaxThreads);
                mbar_init(bar_addr(bars, p, PV_DONE + i), 1);
            }
            mbar_init(bar_addr(bars, p, MMA_DONE), 1);
        }
        mbar_init(bars + 8u * kBarLx, kPipes * kSoftmaxThreads);
        mbar_init(bars + 8u * kBarQ, kThreads - 32);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tmem_alloc(sb + kSmTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kSmTmemSlot);

    if (warp >= 1) {
        // ---- Q tile -> shared memory (swizzled, K-major), rows past the chunk zero, while the
        // producers already fetch the first K/V tiles. Loads first, then stores; the MMA
        // issuers wait for the Q barrier before their first S product.
        constexpr int kLoaders = kThreads - 32;
        constexpr int kPer = (kRows * 16 + kLoaders - 1) / kLoaders;
        const int t = threadIdx.x - 32;
        uint4 v[kPer];
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int c = t + u * kLoaders, r = c >> 4, ch = c & 15;
            v[u] = make_uint4(0, 0, 0, 0);
            if (c < kRows * 16 && r < rows)
                v[u] = __ldg(reinterpret_cast<const uint4*>(
                                 a.q + ((int64_t)(q0 + qt * kRows + r) * a.num_heads + h) * kHeadDim) + ch);
        }
#pragma unroll
        for (int u = 0; u < kPer; ++u) {
            const int c = t + u * kLoaders, r = c >> 4, ch = c & 15;
            if (c < kRows * 16)
                st_shared_v4(sb + kSmQ + (ch >> 3) * kQSlab + r * 128 + (((ch & 7) ^ (r & 7)) << 4), v[u]);
        }
        fence_proxy_async_smem();
        mbar_arrive(bars + 8u * kBarQ);
    }

    if (warp == 0) {
        // ================================================= TMA producers: lanes 0-3, one per (pipe, K|V),
        // each running its own loop (no warp-wide operation in here)
        if (lane < 4) {
            const int pipe = lane >> 1, kv = lane & 1;
            const int base = pipe ? n0 : 0, n = pipe ? nkt - n0 : n0;
            const uint32_t ring = sb + kSmRing + (pipe * 2 + kv) * kStages * kTileOpBytes;
            const uint32_t full0 = bar_addr(bars, pipe, kv ? V_FULL : K_FULL);
            const uint32_t empty0 = bar_addr(bars, pipe, kv ? V_EMPTY : K_EMPTY);
            if (lane == 0) prefetch_tmap(&tmap);
            // Block ids of tile j come from a register queue filled kIdAhead tiles in advance, so that
            // the table reads' latency never sits between two tiles' copies.
            constexpr int kIdAhead = 4;
            int idq[kIdAhead][4];
#pragma unroll
            for (int u = 0; u < kIdAhead; ++u)
#pragma unroll
                for (int b = 0; b < 4; ++b) {
                    const int blk = 4 * (base + u) + b;
                    idq[u][b] = u < n && blk < nblk ? __ldg(trow + blk) : 0;
                }
            int issued = 0;
            bool stop = false;
            for (int j0 = 0; j0 < n && !stop; j0 += kIdAhead) {
#pragma unroll
                for (int u = 0; u < kIdAhead; ++u) {
                    const int j = j0 + u;
                    if (j >= n || stop) break;
                    const int st = j % kStages;
                    const uint32_t ph = (uint32_t)(j / kStages) & 1u;
                    const int g = base + j;
                    const int nb = min(4, nblk - 4 * g);
                    if (j >= kStages && !lane_wait(empty0 + 8 * st, ph ^ 1u, abort, a.status)) {
                        stop = true;
                        break;
                    }
                    mbar_arrive_expect_tx(full0 + 8 * st, nb * kTileBytes);
#pragma unroll
                    for (int b = 0; b < 4; ++b)
                        if (b < nb)
                            for (int half = 0; half < 2; ++half)
                                tma_load_5d(ring + st * kTileOpBytes + half * kTileSlab + b * 2048, &tmap, half * 64,
                                            0, kv * a.num_heads + h, a.layer, idq[u][b], full0 + 8 * st);
                    issued = j + 1;
#pragma unroll
                    for (int b = 0; b < 4; ++b) {  // refill this slot with tile j + kIdAhead
                        const int blk = 4 * (g + kIdAhead) + b;
                        idq[u][b] = j + kIdAhead < n && blk < nblk ? __ldg(trow + blk) : 0;
                    }
                }
            }
            if (*abort)
                for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j)
                    mbar_wait(full0 + 8 * (j % kStages), (uint32_t)(j / kStages) & 1u);
        }
    } else if (warp < 3) {
        // ================================================= MMA issuers, one per pipe
        const int pipe = warp - 1;
        const int base = pipe ? n0 : 0, n = pipe ? nkt - n0 : n0;
        const uint32_t tp = tmem + pipe * kPipeCols;
        const uint32_t kring = sb + kSmRing + (pipe * 2) * kStages * kTileOpBytes;
        const uint32_t vring = kring + kStages * kTileOpBytes;
        for (int j = 0; j <= n; ++j) {
            if (j < n) {
                const int ks = j % kStages, sbuf = j & 1;
                if (j == 0 && !flag_wait(bars + 8u * kBarQ, 0, abort, a.status)) break;
                if (!flag_wait(bar_addr(bars, pipe, K_FULL + ks), (uint32_t)(j / kStages) & 1u, abort, a.status))
                    break;
                // S buffer sbuf (and the P that overwrote it) is free once P V of tile j-2 is done
                if (j >= 2 &&
                    !flag_wait(bar_addr(bars, pipe, PV_DONE + sbuf), (uint32_t)((j - 2) >> 1) & 1u, abort, a.status))
                    break;
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        tc_mma_f16(tp + kColS + sbuf * 64,
                                   sw128_desc(sb + kSmQ + (kk >> 2) * kQSlab + (kk & 3) * 32, 16, 1024),
                                   sw128_desc(kring + ks * kTileOpBytes + (kk >> 2) * kTileSlab + (kk & 3) * 32, 16,
                                              1024),
                                   kIdescS, kk > 0);
                    }
                    tc_commit(bar_addr(bars, pipe, S_FULL + sbuf));
                    tc_commit(bar_addr(bars, pipe, K_EMPTY + ks));
                }
                __syncwarp();
            }
            if (j >= 1) {
                const int i = j - 1, vs = i % kStages, sbuf = i & 1;
                if (!flag_wait(bar_addr(bars, pipe, P_FULL + sbuf), (uint32_t)(i >> 1) & 1u, abort, a.status)) break;
                if (!flag_wait(bar_addr(bars, pipe, V_FULL + vs), (uint32_t)(i / kStages) & 1u, abort, a.status))
                    break;
                if (base + i == nkt - 1) {
                    // keys past the last row's position may hold anything (even NaN); zero their V rows so
                    // that P = 0 times V stays 0 in the tensor core
                    const int first = pos_max + 1 - (base + i) * kKeys;
                    for (int c = first * 8 + lane; c < kKeys * 8; c += 32) {
                        const int r = c >> 3, ch = c & 7;
                        const uint32_t at = vring + vs * kTileOpBytes + r * 128 + ch * 16;
                        st_shared_v4(at, make_uint4(0, 0, 0, 0));
                        st_shared_v4(at + kTileSlab, make_uint4(0, 0, 0, 0));
                    }
                    fence_proxy_async_smem();
                    __syncwarp();
                }
                tc_fence_after();
                if (lane == 0) {
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        tc_mma_f16_ts(tp + kColO, tp + kColS + sbuf * 64 + kk * 8,
                                      sw128_desc(vring + vs * kTileOpBytes + kk * 2048, kTileSlab, 1024), kIdescPV,
                                      (i > 0 || kk > 0) ? 1u : 0u);
                    tc_commit(bar_addr(bars, pipe, PV_DONE + sbuf));
                    tc_commit(bar_addr(bars, pipe, V_EMPTY + vs));
                }
                __syncwarp();
            }
        }
        if (lane == 0) {
            tc_commit(bar_addr(bars, pipe, MMA_DONE));
            mbar_wait(bar_addr(bars, pipe, MMA_DONE), 0);
        }
        __syncwarp();
    } else {
        // ================================================= softmax: 4 warps per pipe, thread = query row
        const int pipe = (warp - 3) >> 2;
        const int base = pipe ? n0 : 0, n = pipe ? nkt - n0 : n0;
        const int qtr = warp & 3;
        const int row = qtr * 32 + lane;
        const bool valid = row < rows;
        const int pos = p0 + row;
        const uint32_t tl = tmem + pipe * kPipeCols + ((uint32_t)(qtr * 32) << 16);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int sbuf = j & 1;
            if (!flag_wait(bar_addr(bars, pipe, S_FULL + sbuf), (uint32_t)(j >> 1) & 1u, abort, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            uint32_t sr[kKeys];
            tc_ld64(tl + kColS + sbuf * 64, sr);
            const int key0 = (base + j) * kKeys;
            if (key0 + kKeys - 1 > p0 || !valid) {
                // diagonal tile or padding row: keys past the row's position count as -inf
                const int nvis = valid ? pos - key0 + 1 : 0;
#pragma unroll
                for (int e = 0; e < kKeys; ++e)
                    if (e >= nvis) sr[e] = __float_as_uint(-INFINITY);
            }
            float mxs[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) mxs[u] = __uint_as_float(sr[u]);
#pragma unroll
            for (int e = 8; e < kKeys; ++e) mxs[e & 7] = fmaxf(mxs[e & 7], __uint_as_float(sr[e]));
            const float mx = fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                                   fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
            const float m_tile = mx * a.scale_log2;
            const bool raise = m_tile > m_used + kRescaleThreshold;  // false while the row has seen no key
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
                // the previous P V product must have landed before O is rescaled
                if (!flag_wait(bar_addr(bars, pipe, PV_DONE + ((j - 1) & 1)), (uint32_t)((j - 1) >> 1) & 1u, abort,
                               a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float f = raise ? ex2(m_used - m_tile) : 1.f;
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    float of[32];
                    uint32_t o[32];
                    tc_ld32(tl + kColO + c * 32, of);
#pragma unroll
                    for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(of[e] * f);
                    tc_st32(tl + kColO + c * 32, o);
                }
                l *= f;
            }
            if (raise) m_used = m_tile;
            // rows that have seen no visible key keep p = 0 (exp2(-inf - -inf) would be NaN)
            const float m_sub = m_used == -INFINITY ? 0.f : m_used;
            float ls[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) ls[u] = 0.f;
            uint32_t packed[32];
#pragma unroll
            for (int e = 0; e < kKeys; e += 2) {
                const float pa = ex2(fmaf(__uint_as_float(sr[e]), a.scale_log2, -m_sub));
                const float pb = ex2(fmaf(__uint_as_float(sr[e + 1]), a.scale_log2, -m_sub));
                ls[e & 7] += pa;
                ls[(e + 1) & 7] += pb;
                const __half2 hp = __floats2half2_rn(pa, pb);
                packed[e >> 1] = *reinterpret_cast<const uint32_t*>(&hp);
            }
            tc_st32(tl + kColS + sbuf * 64, packed);  // P over the first 32 columns of its S buffer
            l += ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
            tc_fence_before();
            mbar_arrive(bar_addr(bars, pipe, P_FULL + sbuf));
        }
        // ---- merge the two pipes: pipe p writes output dims [64p, 64p + 64). Each pipe's (m, l) per row
        // goes into stage 0 of its own K ring, idle once its last P V product has landed.
        const bool landed = ok && (n == 0 || flag_wait(bar_addr(bars, pipe, PV_DONE + ((n - 1) & 1)),
                                                       (uint32_t)((n - 1) >> 1) & 1u, abort, a.status));
        if (landed) {
            float2* mine = reinterpret_cast<float2*>(smem + kSmRing + pipe * 2 * kStages * kTileOpBytes);
            const float2* other = reinterpret_cast<const float2*>(smem + kSmRing + (1 - pipe) * 2 * kStages *
                                                                                     kTileOpBytes);
            mine[row] = make_float2(m_used, l);
            tc_fence_before();
            mbar_arrive(bars + 8u * kBarLx);
            if (flag_wait(bars + 8u * kBarLx, 0, abort, a.status)) {
                tc_fence_after();
                const float2 s0 = pipe == 0 ? mine[row] : other[row];
                const float2 s1 = pipe == 0 ? other[row] : mine[row];
                const float M = fmaxf(s0.x, s1.x);
                const float w0 = n0 > 0 && s0.x != -INFINITY ? ex2(s0.x - M) : 0.f;
                const float w1 = nkt - n0 > 0 && s1.x != -INFINITY ? ex2(s1.x - M) : 0.f;
                const float inv = 1.f / (w0 * s0.y + w1 * s1.y);
                const uint32_t t0 = tmem + ((uint32_t)(qtr * 32) << 16) + kColO + pipe * 64;
                uint4* dst = reinterpret_cast<uint4*>(a.out + ((int64_t)(q0 + qt * kRows + row) * a.num_heads + h) *
                                                                  kHeadDim + pipe * 64);
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    float o0[32], o1[32];
#pragma unroll
                    for (int u = 0; u < 32; ++u) o0[u] = o1[u] = 0.f;
                    // a pipe that processed no tile never wrote its O: leave it out
                    if (n0 > 0) tc_ld32(t0 + c * 32, o0);
                    if (nkt - n0 > 0) tc_ld32(t0 + kPipeCols + c * 32, o1);
                    if (valid) {
#pragma unroll
                        for (int q4 = 0; q4 < 4; ++q4) {
                            uint32_t w[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int e = q4 * 8 + 2 * u;
                                const __half2 hq = __floats2half2_rn(fmaf(w0, o0[e], w1 * o1[e]) * inv,
                                                                     fmaf(w0, o0[e + 1], w1 * o1[e + 1]) * inv);
                                w[u] = *reinterpret_cast<const uint32_t*>(&hq);
                            }
                            dst[c * 4 + q4] = make_uint4(w[0], w[1], w[2], w[3]);
                        }
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_prefill(const pkv_pool* pool, int layer, const void* q, const int32_t* q_start,
                           const int32_t* tables, int max_blocks, const int32_t* ctx_lens, int num_seqs, int max_q_len,
                           float scale, void* out, cudaStream_t stream)
{
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmAlloc);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    PrefillArgs a;
    a.q = static_cast<const __half*>(q);
    a.out = static_cast<__half*>(out);
    a.q_start = q_start;
    a.tables = tables;
    a.ctx_lens = ctx_lens;
    a.max_blocks = max_blocks;
    a.num_heads = pool->geom.num_heads;
    a.layer = layer;
    a.max_q_len = max_q_len;
    a.num_blocks = pool->geom.num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.status = pool->status_dev;
    CUtensorMap tmap;
    static_assert(sizeof(tmap) == sizeof(pool->kv_tmap.bytes), "tensor map size");
    memcpy(&tmap, pool->kv_tmap.bytes, sizeof(tmap));
    dim3 grid((max_q_len + kRows - 1) / kRows, pool->geom.num_heads, num_seqs);
    prefill_kernel<<<grid, kThreads, kSmAlloc, stream>>>(tmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
