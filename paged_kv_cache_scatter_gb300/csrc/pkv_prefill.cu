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
// are already in the pool (kv_append runs first), so keys come only from the
// pool, 128 at a time (8 blocks).
//
// Tiles are 128 keys: an M=128 N=128 QK^T product keeps the tensor core at
// its full rate (N=64 runs it at about half). Tensor memory holds three S
// buffers and O (all 512 columns). The softmax reads S_j into registers and
// writes P_j (FP16) over the first 64 columns of S_j's own buffer, where
// O += P_j V_j reads it (no shared-memory round trip). S_{j+2} goes to the
// buffer of P_{j-1}, so the only wait before it is for P_{j-1} V_{j-1}. S and
// P V are issued by two warps of their own: each waits only for its own
// operands, and while one waits the other's MMAs keep the tensor core's queue
// filled (a single issuer stalls the tensor core at every wait; its queue
// holds only a couple of MMAs).
//
// Warp roles (384 threads, three warpgroups; the producer and issuer
// warpgroups hand registers to the softmax warpgroup with setmaxnreg, so that a
// softmax thread keeps its row's 128 S values in registers):
//   warps 0-3    TMA producers of K's 64-dim halves 0, 1 and V's halves 0, 1:
//                lane b < 8 copies one 2 KB box (block b's 16 rows of the
//                warp's half) of every 128-key tile into its 3-stage ring. A
//                warp issues its TMA copies one after another, a few hundred
//                cycles each, so a tile's 32 boxes need four issuing warps
//                to arrive about as fast as the tensor core consumes them
//                (one warp: ~2,400 cycles per 64 KB tile; four: ~1,150).
//                They sleep between polls while they wait for a free slot.
//   warp 8       S issuer (the warp runs the loop, one elected lane issues;
//                the warp owns the TMEM allocation): S_j = Q K_j^T, A and B
//                from shared memory, into S buffer j%3 once K_j has landed
//                and P_{j-3} V_{j-3} has read that buffer; tcgen05.commit
//                signals S_j done and K_j's ring slot free.
//   warp 9       P V issuer: O += P_j V_j, P from tensor memory, once the
//                softmax has written P_j and V_j has landed; commits signal
//                the product done and V_j's ring slot free.
//   warps 4-7    softmax: thread r owns query row r (TMEM lane r). Per tile it
//                loads its 128 S values into registers, takes the row max,
//                and writes P =
//                2^(s*scale*log2e - m) by quarters while adding to the
//                running sum. The running max m is only raised when the
//                tile's max exceeds it by more than 8 (a factor 256, far
//                inside FP16/FP32 range); then the row's O and sum are
//                rescaled once the previous P V product has landed. The
//                result is exact up to rounding.
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

constexpr int kRows = 128;            // query rows per CTA (MMA M)
constexpr int kKeys = 128;            // keys per tile (8 blocks)
constexpr int kBlocksPerTile = kKeys / kBlockSize;
constexpr int kStagesK = 3;           // K ring depth (4 K + 2 V stages in the same space measured the same)
constexpr int kStagesV = 3;           // V ring depth
constexpr int kBufs = 3;              // S buffers in tensor memory (P_j overwrites S_j's)
constexpr int kProducerWarps = 4;     // K low, K high, V low, V high
constexpr int kFirstSoftmaxWarp = 4;
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = 8;           // S issuer; also owns the TMEM allocation
constexpr int kPvWarp = 9;            // P V issuer
constexpr int kThreads = 384;         // warps 10, 11 only fill the third warpgroup
constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;  // 168: what ptxas allows a thread at launch
constexpr int kSideRegs = 64;         // producer and issuer warpgroups
constexpr int kSoftmaxRegs = 200;     // softmax warpgroup
static_assert(2 * 128 * kSideRegs + 128 * kSoftmaxRegs <= kThreads * kLaunchRegs, "register split");
constexpr int kQBytes = kRows * kHeadDim * 2;        // 32 KB
constexpr int kQSlab = kQBytes / 2;                  // 16 KB: 128 rows x 64 halves
constexpr int kTileOpBytes = kKeys * kHeadDim * 2;   // 32 KB: one 128-key K or V tile
constexpr int kTileSlab = kTileOpBytes / 2;          // 16 KB: 128 rows x 64 halves
constexpr float kRescaleThreshold = 8.f;             // log2 of the largest un-rescaled P (256)

// shared-memory map (offsets from a 1,024-byte aligned base)
constexpr int kSmQ = 0;
constexpr int kSmKRing = kQBytes;                             // [stage] K tiles
constexpr int kSmVRing = kSmKRing + kStagesK * kTileOpBytes;  // [stage] V tiles
constexpr int kSmBars = kSmVRing + kStagesV * kTileOpBytes;
enum Bar {
    K_FULL = 0,                   // count 2: the K low and K high producers arm it
    V_FULL = K_FULL + kStagesK,
    K_EMPTY = V_FULL + kStagesV,
    V_EMPTY = K_EMPTY + kStagesK,
    S_FULL = V_EMPTY + kStagesV,  // [kBufs] per S buffer
    P_FULL = S_FULL + kBufs,      // [kBufs] count kSoftmaxThreads: P written over the buffer's S
    PV_DONE = P_FULL + kBufs,     // [kBufs]
    V_FIXED = PV_DONE + kBufs,    // the last tile's V rows past the last position are zeroed
    Q_READY = V_FIXED + 1,        // count kSoftmaxThreads
    S_ALL_DONE = Q_READY + 1,     // every S MMA finished (before the CTA frees tensor memory)
    PV_ALL_DONE = S_ALL_DONE + 1, // every P V MMA finished
    NUM_BARS = PV_ALL_DONE + 1
};
constexpr int kSmTmemSlot = kSmBars + NUM_BARS * 8;
constexpr int kSmAbort = kSmTmemSlot + 4;
constexpr int kSmBytes = kSmAbort + 12;
constexpr int kSmAlloc = kSmBytes + 1024;  // slack to align the base
static_assert(kSmAlloc <= 227 * 1024, "shared memory per CTA");

// TMEM columns: S buffers 0, 1, 2 (128 fp32 columns each; P, FP16 two per
// column, takes the first 64 of its S buffer), O (128): all 512.
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0;
constexpr uint32_t kSBufCols = 128;
constexpr uint32_t kColO = kBufs * kSBufCols;
static_assert(kColO + 128 <= kTmemCols, "tensor memory columns");

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
    int num_heads;     // K/V heads of the pool
    int num_q_heads;   // query heads: q and out rows are [num_q_heads][128]
    int group;         // query heads per K/V head; query head h reads K/V head h / group
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

// Bounded wait of a warp off the critical path (a producer waiting for a free ring slot): lane 0
// polls with a sleep between polls and broadcasts the outcome, so the waiting warp takes almost
// no issue slots from the softmax and MMA warps that share its scheduler.
__device__ __forceinline__ bool lazy_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* status)
{
    const int lane = threadIdx.x & 31;
    int r = 1;  // 1 done, 0 aborted elsewhere, 2 timed out
    if (lane == 0 && !mbar_try_wait(bar, parity)) r = *abort ? 0 : (mbar_wait_sleep(bar, parity, 256) ? 1 : 2);
    r = __shfl_sync(0xffffffffu, r, 0);
    if (r == 2 && lane == 0) {
        atomicOr(status, PKV_DEV_TIMEOUT);
        *abort = 1;
    }
    return r == 1;
}

// Shared-memory descriptor of (the operand a descriptor d describes) + off bytes: the start
// address field is address / 16 in the low 14 bits, and every operand here lies below 256 KB.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t off) { return d + (uint64_t)(off >> 4); }

// Keys e >= nvis of N S values count as -inf (diagonal tiles and padding rows only).
template <int N>
__device__ __forceinline__ void mask_tail(uint32_t* s, int nvis)
{
#pragma unroll
    for (int e = 0; e < N; ++e)
        if (e >= nvis) s[e] = __float_as_uint(-INFINITY);
}

// Max of 64 S values.
__device__ __forceinline__ float max64(const uint32_t* sr)
{
    float mxs[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mxs[u] = __uint_as_float(sr[u]);
#pragma unroll
    for (int e = 8; e < 64; ++e) mxs[e & 7] = fmaxf(mxs[e & 7], __uint_as_float(sr[e]));
    return fmaxf(fmaxf(fmaxf(mxs[0], mxs[1]), fmaxf(mxs[2], mxs[3])),
                 fmaxf(fmaxf(mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7])));
}

// Softmax of a quarter tile: 32 S values -> P = 2^(s*scale - m) as 16 FP16 pairs, written in place over
// s[0..15] (pair e/2 lands on a value already read); the sum is added to l. An s of -inf gives p = 0.
__device__ __forceinline__ void softmax_quarter(uint32_t* s, float scale_log2, float m_sub, float& l)
{
    float ls[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) ls[u] = 0.f;
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const float pa = ex2(fmaf(__uint_as_float(s[e]), scale_log2, -m_sub));
        const float pb = ex2(fmaf(__uint_as_float(s[e + 1]), scale_log2, -m_sub));
        ls[e & 3] += pa;
        ls[(e + 1) & 3] += pb;
        const __half2 hp = __floats2half2_rn(pa, pb);
        s[e >> 1] = *reinterpret_cast<const uint32_t*>(&hp);
    }
    l += (ls[0] + ls[1]) + (ls[2] + ls[3]);
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
    const int n = pos_max / kKeys + 1;       // 128-key tiles
    const int nblk = pos_max / kBlockSize + 1;
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
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile int* abort = reinterpret_cast<volatile int*>(smem + kSmAbort);
    if (threadIdx.x == 0) {
        for (int i = 0; i < kStagesK; ++i) {
            mbar_init(bar(K_FULL + i), 2);
            mbar_init(bar(K_EMPTY + i), 1);
        }
        for (int i = 0; i < kStagesV; ++i) {
            mbar_init(bar(V_FULL + i), 2);
            mbar_init(bar(V_EMPTY + i), 1);
        }
        for (int i = 0; i < kBufs; ++i) {
            mbar_init(bar(S_FULL + i), 1);
            mbar_init(bar(P_FULL + i), kSoftmaxThreads);
            mbar_init(bar(PV_DONE + i), 1);
        }
        mbar_init(bar(V_FIXED), 1);
        mbar_init(bar(Q_READY), kSoftmaxThreads);
        mbar_init(bar(S_ALL_DONE), 1);
        mbar_init(bar(PV_ALL_DONE), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sb + kSmTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kSmTmemSlot);

    // Each warpgroup sets its register budget at the top of its own branch (the same instruction in all
    // four of its warps), so that ptxas allocates each role's code with that role's budget.
    if (warp < kProducerWarps) {
        regs_dec<kSideRegs>();
        // ================================================= TMA producers: warp 0 copies K's 64-dim half 0,
        // warp 1 K's half 1, warps 2, 3 V's halves (lane < 8: block lane of each tile).
        const int kv = warp >> 1;
        const int b = lane & (kBlocksPerTile - 1), half = warp & 1;
        const bool copier = lane < kBlocksPerTile;
        const uint32_t ring = sb + (kv ? kSmVRing : kSmKRing) + half * kTileSlab;
        const uint32_t full0 = bar(kv ? V_FULL : K_FULL);
        const uint32_t empty0 = bar(kv ? V_EMPTY : K_EMPTY);
        if (lane == 0) prefetch_tmap(&tmap);
        // Block ids of tile i come from a register queue filled kIdAhead tiles in advance, so that
        // the table reads' latency never sits between two tiles' copies.
        constexpr int kIdAhead = 2;
        int idq[kIdAhead];
#pragma unroll
        for (int u = 0; u < kIdAhead; ++u) {
            const int blk = kBlocksPerTile * u + b;
            idq[u] = copier && u < n && blk < nblk ? __ldg(trow + blk) : 0;
        }
        const int stages = kv ? kStagesV : kStagesK;
        int issued = 0;
        bool stop = false;
        for (int i0 = 0; i0 < n && !stop; i0 += kIdAhead) {
#pragma unroll
            for (int u = 0; u < kIdAhead; ++u) {
                const int i = i0 + u;
                if (i >= n) break;
                const int st = i % stages;
                const uint32_t ph = (uint32_t)(i / stages) & 1u;
                const int nb = min(kBlocksPerTile, nblk - kBlocksPerTile * i);
                if (i >= stages && !lazy_wait(empty0 + 8 * st, ph ^ 1u, abort, a.status)) {
                    stop = true;
                    break;
                }
                if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, nb * (kTileBytes / 2));
                __syncwarp();
                if (copier && b < nb)
                    tma_load_5d(ring + st * kTileOpBytes + b * 2048, &tmap, half * 64, 0, kv * a.num_heads + h / a.group,
                                a.layer, idq[u], full0 + 8 * st);
                issued = i + 1;
                const int blk = kBlocksPerTile * (i + kIdAhead) + b;  // refill this slot with tile i + kIdAhead
                idq[u] = copier && i + kIdAhead < n && blk < nblk ? __ldg(trow + blk) : 0;
            }
        }
        if (warp == 2 && !stop) {
            // The last tile: keys past the last row's position may hold anything (even NaN), and rows of
            // blocks past the table's end were not copied at all. Zero those V rows (both halves, once they
            // have landed) so that P = 0 times V stays 0 in the tensor core, then release the tile.
            const int i = n - 1, st = i % kStagesV;
            if (flag_wait(full0 + 8 * st, (uint32_t)(i / kStagesV) & 1u, abort, a.status)) {
                const uint32_t vt = sb + kSmVRing + st * kTileOpBytes;
                const int first = pos_max + 1 - (n - 1) * kKeys;
                for (int c = first * 8 + lane; c < kKeys * 8; c += 32) {
                    const int r = c >> 3, ch = c & 7;
                    st_shared_v4(vt + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                    st_shared_v4(vt + kTileSlab + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(V_FIXED));
            }
        }
        // copies still in flight (after an abort) must land before the CTA exits
        for (int i = (issued > stages ? issued - stages : 0); i < issued; ++i)
            mbar_wait(full0 + 8 * (i % stages), (uint32_t)(i / stages) & 1u);
    } else if (warp >= kMmaWarp) {
        regs_dec<kSideRegs>();
        if (warp == kMmaWarp) {
        // ================================================= S issuer: the whole warp runs the loop (warp-uniform
        // waits and descriptors) and one elected lane issues each MMA and commit.
        // base descriptors; each MMA adds a constant offset (one 64-bit add instead of building a descriptor)
        const uint64_t dq = sw128_desc(sb + kSmQ, 16, 1024);
        const uint64_t dk = sw128_desc(sb + kSmKRing, 16, 1024);
        for (int j = 0; j < n; ++j) {
            const int ks = j % kStagesK, sbuf = j % kBufs;
            const bool ok = (j > 0 || flag_wait(bar(Q_READY), 0, abort, a.status)) &&
                            flag_wait(bar(K_FULL + ks), (uint32_t)(j / kStagesK) & 1u, abort, a.status) &&
                            // S buffer j%3 last held P_{j-3}, which P_{j-3} V_{j-3} must have read
                            (j < kBufs ||
                             flag_wait(bar(PV_DONE + sbuf), (uint32_t)((j - kBufs) / kBufs) & 1u, abort, a.status));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_f16_warp(tmem + kColS + sbuf * kSBufCols, desc_add(dq, (kk >> 2) * kQSlab + (kk & 3) * 32),
                                desc_add(dk, ks * kTileOpBytes + (kk >> 2) * kTileSlab + (kk & 3) * 32), kIdescS, kk > 0);
            tc_commit_warp(bar(S_FULL + sbuf));
            tc_commit_warp(bar(K_EMPTY + ks));
        }
        // every MMA this warp issued must have finished before the CTA frees its tensor memory and exits
        tc_commit_warp(bar(S_ALL_DONE));
        mbar_wait(bar(S_ALL_DONE), 0);
        __syncwarp();
        } else if (warp == kPvWarp) {
        // ================================================= P V issuer, in the same style
        const uint64_t dv = sw128_desc(sb + kSmVRing, kTileSlab, 1024);
        for (int j = 0; j < n; ++j) {
            const int vs = j % kStagesV, pbuf = j % kBufs;
            const bool ok = flag_wait(bar(P_FULL + pbuf), (uint32_t)(j / kBufs) & 1u, abort, a.status) &&
                            (j == n - 1 ? flag_wait(bar(V_FIXED), 0, abort, a.status)
                                        : flag_wait(bar(V_FULL + vs), (uint32_t)(j / kStagesV) & 1u, abort, a.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t pcol = tmem + kColS + pbuf * kSBufCols;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_f16_ts_warp(tmem + kColO, pcol + kk * 8, desc_add(dv, vs * kTileOpBytes + kk * 2048), kIdescPV,
                                   (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit_warp(bar(PV_DONE + pbuf));
            tc_commit_warp(bar(V_EMPTY + vs));
        }
        tc_commit_warp(bar(PV_ALL_DONE));
        mbar_wait(bar(PV_ALL_DONE), 0);
        __syncwarp();
        }
    } else {
        regs_inc<kSoftmaxRegs>();
        // ================================================= softmax: thread = query row
        const int qtr = warp & 3;
        const int row = qtr * 32 + lane;
        const bool valid = row < rows;
        const int pos = p0 + row;
        const uint32_t tl = tmem + ((uint32_t)(qtr * 32) << 16);
        {
            // ---- Q tile -> shared memory (swizzled, K-major), rows past the chunk zero, while the
            // producers already fetch the first K/V tiles. Loads first, then stores.
            constexpr int kPer = kRows * 16 / kSoftmaxThreads;
            const int t = threadIdx.x - kFirstSoftmaxWarp * 32;
            uint4 v[kPer];
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int c = t + u * kSoftmaxThreads, r = c >> 4, ch = c & 15;
                v[u] = make_uint4(0, 0, 0, 0);
                if (r < rows)
                    v[u] = __ldg(reinterpret_cast<const uint4*>(
                                     a.q + ((int64_t)(q0 + qt * kRows + r) * a.num_q_heads + h) * kHeadDim) +
                                 ch);
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int c = t + u * kSoftmaxThreads, r = c >> 4, ch = c & 15;
                st_shared_v4(sb + kSmQ + (ch >> 3) * kQSlab + r * 128 + (((ch & 7) ^ (r & 7)) << 4), v[u]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(Q_READY));
        }
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int sbuf = j % kBufs;
            if (!flag_wait(bar(S_FULL + sbuf), (uint32_t)(j / kBufs) & 1u, abort, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t ts = tl + kColS + sbuf * kSBufCols;
            const int key0 = j * kKeys;
            // diagonal tile: keys past the row's position count as -inf. Padding rows (past the chunk's last
            // query) are left unmasked: their Q is zero, their O is never written and rows do not mix in the
            // MMAs, so whatever they compute (even NaN from a key past the context) stays in them; masking
            // them on every tile would slow their warps, and every tile waits for the slowest softmax warp.
            const bool diag = valid && key0 + kKeys - 1 > p0;
            const int nvis = pos - key0 + 1;
            // all of S_j in registers, in two halves: the first half's max is taken while the second
            // half is still on its way from tensor memory
            uint32_t sr[kKeys];
            tc_ld64_issue(ts, sr);
            tc_wait_ld64(sr);
            tc_ld64_issue(ts + 64, sr + 64);
            if (diag) mask_tail<64>(sr, nvis);
            float mx = max64(sr);
            tc_wait_ld64(sr + 64);
            if (diag) mask_tail<64>(sr + 64, nvis - 64);
            const float m_tile = fmaxf(mx, max64(sr + 64)) * a.scale_log2;
            const bool raise = m_tile > m_used + kRescaleThreshold;  // false while the row has seen no key
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
                // the previous P V product must have landed before O is rescaled
                if (!flag_wait(bar(PV_DONE + (j - 1) % kBufs), (uint32_t)((j - 1) / kBufs) & 1u, abort,
                               a.status)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const float f = raise ? ex2(m_used - m_tile) : 1.f;
#pragma unroll 1
                for (int c = 0; c < 8; ++c) {  // 16 columns at a time: S_j occupies 128 registers meanwhile
                    uint32_t o[16];
                    tc_ld16(tl + kColO + c * 16, o);
#pragma unroll
                    for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                    tc_st16(tl + kColO + c * 16, o);
                }
                l *= f;
            }
            if (raise) m_used = m_tile;
            // rows that have seen no visible key keep p = 0 (exp2(-inf - -inf) would be NaN)
            const float m_sub = m_used == -INFINITY ? 0.f : m_used;
            // P_j goes over the S_j just read (no MMA touches this buffer until P_j V_j)
            const uint32_t tp = ts;
            // quarters of 32 keys: P of keys 32q.. goes to P columns 16q.., stored without waiting
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                softmax_quarter(sr + q * 32, a.scale_log2, m_sub, l);
                tc_st16_async(tp + q * 16, sr + q * 32);
            }
            tc_wait_st();
            tc_fence_before();
            mbar_arrive(bar(P_FULL + sbuf));
        }
        // ---- epilogue: O / l -> FP16 (each row's 256 B written by its thread)
        if (ok && flag_wait(bar(PV_DONE + (n - 1) % kBufs), (uint32_t)((n - 1) / kBufs) & 1u, abort, a.status)) {
            tc_fence_after();
            const float inv = 1.f / l;
            uint4* dst =
                reinterpret_cast<uint4*>(a.out + ((int64_t)(q0 + qt * kRows + row) * a.num_q_heads + h) * kHeadDim);
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                float o[32];
                tc_ld32(tl + kColO + c * 32, o);
                if (valid) {
#pragma unroll
                    for (int q4 = 0; q4 < 4; ++q4) {
                        uint32_t w[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            const __half2 hq = __floats2half2_rn(o[q4 * 8 + 2 * u] * inv, o[q4 * 8 + 2 * u + 1] * inv);
                            w[u] = *reinterpret_cast<const uint32_t*>(&hq);
                        }
                        dst[c * 4 + q4] = make_uint4(w[0], w[1], w[2], w[3]);
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
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
    a.num_q_heads = pool->geom.num_q_heads;
    a.group = pool->geom.group;
    a.layer = layer;
    a.max_q_len = max_q_len;
    a.num_blocks = pool->geom.num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.status = pool->status_dev;
    CUtensorMap tmap;
    static_assert(sizeof(tmap) == sizeof(pool->kv_tmap.bytes), "tensor map size");
    memcpy(&tmap, pool->kv_tmap.bytes, sizeof(tmap));
    dim3 grid((max_q_len + kRows - 1) / kRows, pool->geom.num_q_heads, num_seqs);
    prefill_kernel<<<grid, kThreads, kSmAlloc, stream>>>(tmap, a);
    return cudaGetLastError();
}

}  // namespace pkv
