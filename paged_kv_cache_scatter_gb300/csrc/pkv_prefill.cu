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
//                result is exact up to rounding. P_j is signalled to the
//                P V issuer from tile j+1, after that tile's first S load
//                (by then P_j's stores have completed without a stall).
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
constexpr int kBufs = 3;              // S buffers in tensor memory (P_j overwrites S_j's)
constexpr int kProducerWarps = 4;
constexpr int kFirstSoftmaxWarp = 4;
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = 8;           // S issuer; also owns the TMEM allocation
constexpr int kPvWarp = 9;            // P V issuer
constexpr int kFirstConvWarp = 12;    // 8-bit pools: warps 12-15 turn codes into FP16 operand tiles
constexpr int kQBytes = kRows * kHeadDim * 2;        // 32 KB
constexpr int kQSlab = kQBytes / 2;                  // 16 KB: 128 rows x 64 halves
constexpr int kTileOpBytes = kKeys * kHeadDim * 2;   // 32 KB: one 128-key K or V tile
constexpr int kTileSlab = kTileOpBytes / 2;          // 16 KB: 128 rows x 64 halves
constexpr int kScaleStage = 2 * kKeys * 4;           // 8-bit pools: a tile's 128 K then 128 V row scales (FP32)
constexpr int kScaleStages = 6;                      // 8-bit pools: scale ring depth (held until the softmax is done)
constexpr int kCodesBytes = kBlockSize * kHeadDim;   // 8-bit pools: one (block, layer, K|V, head) tile's codes
constexpr float kRescaleThreshold = 8.f;             // log2 of the largest un-rescaled P (256)

// Per pool element type: ring depths, threads, register split and the shared-memory map.
// FP16 pools: 12 warps (producers, softmax, issuers + 2 idle). 8-bit pools: a fourth warpgroup
// converts codes, the V ring has 2 stages, and the row scales have a ring of their own.
template <bool kI8>
struct Cfg {
    static constexpr int kStagesK = 3;           // K ring depth (4 K + 2 V stages in the same space measured the same)
    static constexpr int kStagesV = kI8 ? 2 : 3; // V ring depth
    static constexpr int kThreads = kI8 ? 512 : 384;
    static constexpr int kLaunchRegs = 65536 / kThreads / 8 * 8;  // what ptxas allows a thread at launch
    static constexpr int kSideRegs = 64;                          // producer and issuer warpgroups
    static constexpr int kConvRegs = 96;                          // converter warpgroup (8-bit pools)
    static constexpr int kSoftmaxRegs = 200;                      // softmax warpgroup
    static_assert(2 * 128 * kSideRegs + 128 * kSoftmaxRegs + (kI8 ? 128 * kConvRegs : 0) <= kThreads * kLaunchRegs,
                  "register split");
    // shared-memory map (offsets from a 1,024-byte aligned base)
    static constexpr int kSmQ = 0;
    static constexpr int kSmKRing = kQBytes;                             // [stage] K tiles
    static constexpr int kSmVRing = kSmKRing + kStagesK * kTileOpBytes;  // [stage] V tiles
    static constexpr int kSmScales = kSmVRing + kStagesV * kTileOpBytes; // 8-bit: [stage][K 128, V 128] f32
    static constexpr int kSmBars = kSmScales + (kI8 ? kScaleStages * kScaleStage : 0);
    // barriers
    static constexpr int K_FULL = 0;                     // count 2 (FP16: two half-tile producers) or 1 (8-bit codes)
    static constexpr int V_FULL = K_FULL + kStagesK;
    static constexpr int K_EMPTY = V_FULL + kStagesV;
    static constexpr int V_EMPTY = K_EMPTY + kStagesK;
    static constexpr int K_CONV = V_EMPTY + kStagesV;    // 8-bit: count 2, the K (or V) converter warps
    static constexpr int V_CONV = K_CONV + kStagesK;
    static constexpr int SC_FULL = V_CONV + kStagesV;    // 8-bit: [kScaleStages] count 2, the two scale producers
    static constexpr int SC_FREE = SC_FULL + kScaleStages;  // 8-bit: [kScaleStages] count 4, the softmax warps
    static constexpr int S_FULL = SC_FREE + kScaleStages;   // [kBufs] per S buffer
    static constexpr int P_FULL = S_FULL + kBufs;        // [kBufs] count kSoftmaxThreads: P written over the buffer's S
    static constexpr int PV_DONE = P_FULL + kBufs;       // [kBufs]
    static constexpr int V_FIXED = PV_DONE + kBufs;      // the last tile's V rows (FP16) or V scales (8-bit, count
                                                         // kSoftmaxThreads) past the last position zeroed
    static constexpr int Q_READY = V_FIXED + 1;          // count kSoftmaxThreads
    static constexpr int S_ALL_DONE = Q_READY + 1;       // every S MMA finished (before the CTA frees tensor memory)
    static constexpr int PV_ALL_DONE = S_ALL_DONE + 1;   // every P V MMA finished
    static constexpr int NUM_BARS = PV_ALL_DONE + 1;
    static constexpr int kSmTmemSlot = kSmBars + NUM_BARS * 8;
    static constexpr int kSmAbort = kSmTmemSlot + 4;
    static constexpr int kSmBytes = kSmAbort + 12;
    static constexpr int kSmAlloc = kSmBytes + 1024;  // slack to align the base
    static_assert(kSmAlloc <= 227 * 1024, "shared memory per CTA");
};

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
    const char* base;        // 8-bit pools: the pool, for the row scales of a tile
    int64_t block_bytes;
    int64_t layer_bytes;
    int64_t tile_bytes;
    int max_blocks;
    int num_heads;     // K/V heads of the pool
    int num_q_heads;   // query heads: q and out rows are [num_q_heads][128]
    int group;         // query heads per K/V head; query head h reads K/V head h / group
    int hpc;           // query heads per CTA: the group (group <= 128) or 1
    int tok;           // query tokens per CTA: 128 / hpc; MMA row r is token r % tok of head r / tok
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

// Max of 64 S values: three-input maxima, eight independent chains.
__device__ __forceinline__ float max64(const uint32_t* sr)
{
    auto f = [&](int e) { return __uint_as_float(sr[e]); };
    float mxs[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) mxs[u] = fmax3(f(3 * u), f(3 * u + 1), f(3 * u + 2));  // values 0..23
#pragma unroll
    for (int i = 0; i < 20; ++i) mxs[i & 7] = fmax3(mxs[i & 7], f(24 + 2 * i), f(25 + 2 * i));  // 24..63
    return fmax3(fmax3(mxs[0], mxs[1], mxs[2]), fmax3(mxs[3], mxs[4], mxs[5]), fmaxf(mxs[6], mxs[7]));
}

// Softmax of a quarter tile: 32 S values -> P = 2^(s*scale - m) as 16 FP16 pairs, written in place over
// s[0..15] (pair e/2 lands on a value already read); the sum is added to l. An s of -inf gives p = 0.
// The exponents and the sums go two at a time (f32x2 FMA and add); the 2^x stay scalar.
__device__ __forceinline__ void softmax_quarter(uint32_t* s, float scale_log2, float m_sub, float& l)
{
    const uint64_t sc2 = f32x2_pack(scale_log2, scale_log2), nm2 = f32x2_pack(-m_sub, -m_sub);
    uint64_t acc[2] = {f32x2_pack(0.f, 0.f), f32x2_pack(0.f, 0.f)};
#pragma unroll
    for (int e = 0; e < 32; e += 2) {
        const float2 x = f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])), sc2, nm2));
        const float pa = ex2(x.x), pb = ex2(x.y);
        acc[(e >> 1) & 1] = add_f32x2(acc[(e >> 1) & 1], f32x2_pack(pa, pb));
        s[e >> 1] = pack_half2(pa, pb);
    }
    const float2 a0 = f32x2_unpack(acc[0]), a1 = f32x2_unpack(acc[1]);
    l += (a0.x + a0.y) + (a1.x + a1.y);
}

// 8-bit pools: one key row r of a 128-key operand tile. Its 128 codes sit in the tile's second slab, row r,
// 16-byte chunks in 128-byte swizzle (dims 16c..16c+15 in chunk c ^ (r % 8)); the row becomes the codes as
// FP16 (exact: |code| <= 127) in both slabs (dims 0-63, 64-127), in the same swizzle, in place: this thread
// alone reads or writes row r, and it reads every chunk first. A code c becomes FP16 c via the byte
// pattern 0x64XX = 1024 + XX with XX = c + 128, less 1152. The row scales are applied by the softmax
// (K's to the scores, V's to the weights P), so no value is rounded here. Rows past the last query
// position (or of blocks not copied) become zeros: keys there may hold anything.
__device__ __forceinline__ void convert_code_row(uint32_t tile, int r, bool valid)
{
    const uint32_t s0 = tile + r * 128, s1 = tile + kTileSlab + r * 128;
    const uint32_t sw = (uint32_t)(r & 7);
    if (!valid) {
        const uint4 z = make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int c = 0; c < 8; ++c) {
            st_shared_v4(s0 + (c << 4), z);
            st_shared_v4(s1 + (c << 4), z);
        }
        return;
    }
    uint4 cw[8];
#pragma unroll
    for (int c = 0; c < 8; ++c) cw[c] = ld_shared_v4(s1 + (((uint32_t)c ^ sw) << 4));
    const __half2 bias = __float2half2_rn(1152.f);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        const uint32_t w[4] = {cw[c].x, cw[c].y, cw[c].z, cw[c].w};
        uint32_t o[8];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t u = w[k] ^ 0x80808080u;
#pragma unroll
            for (int hlf = 0; hlf < 2; ++hlf) {
                const uint32_t bits = __byte_perm(u, 0x64646464u, hlf ? 0x4342u : 0x4140u);
                const __half2 x = __hsub2(*reinterpret_cast<const __half2*>(&bits), bias);
                o[2 * k + hlf] = *reinterpret_cast<const uint32_t*>(&x);
            }
        }
        const uint32_t dst = (c >> 2) ? s1 : s0;
        const uint32_t ch = (uint32_t)(2 * (c & 3));
        st_shared_v4(dst + ((ch ^ sw) << 4), make_uint4(o[0], o[1], o[2], o[3]));
        st_shared_v4(dst + (((ch + 1) ^ sw) << 4), make_uint4(o[4], o[5], o[6], o[7]));
    }
}

// 8-bit pools: N scores times their keys' row scales (FP32, from shared memory, the same for every row).
// The scales are read through an ordinary pointer, not an asm load, so that the compiler can issue the
// reads ahead of the arithmetic (they are fenced only by the barrier waits, which clobber memory).
template <int N>
__device__ __forceinline__ void scale_columns(uint32_t* s, const float4* scales)
{
#pragma unroll
    for (int e = 0; e < N; e += 4) {
        const float4 k4 = scales[e / 4];
        const float2 a = f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(s[e]), __uint_as_float(s[e + 1])),
                                                f32x2_pack(k4.x, k4.y)));
        const float2 b = f32x2_unpack(mul_f32x2(f32x2_pack(__uint_as_float(s[e + 2]), __uint_as_float(s[e + 3])),
                                                f32x2_pack(k4.z, k4.w)));
        s[e] = __float_as_uint(a.x);
        s[e + 1] = __float_as_uint(a.y);
        s[e + 2] = __float_as_uint(b.x);
        s[e + 3] = __float_as_uint(b.y);
    }
}

// 8-bit pools: softmax_quarter with each weight times its key's V row scale before the rounding to FP16
// (O accumulates P' codes_V = P V); the running sum takes the unscaled weights. Keys past the last query
// position (the last tile) have their V scale set to 0 first, so that 0 times a garbage scale never reaches
// the P V product.
__device__ __forceinline__ void softmax_quarter_vscaled(uint32_t* s, float scale_log2, float m_sub, float& l,
                                                        const float4* vscales)
{
    const uint64_t sc2 = f32x2_pack(scale_log2, scale_log2), nm2 = f32x2_pack(-m_sub, -m_sub);
    uint64_t acc[2] = {f32x2_pack(0.f, 0.f), f32x2_pack(0.f, 0.f)};
#pragma unroll
    for (int e = 0; e < 32; e += 4) {
        const float4 v4 = vscales[e / 4];
        const float vs[4] = {v4.x, v4.y, v4.z, v4.w};
#pragma unroll
        for (int u = 0; u < 4; u += 2) {
            const float2 x =
                f32x2_unpack(fma_f32x2(f32x2_pack(__uint_as_float(s[e + u]), __uint_as_float(s[e + u + 1])), sc2, nm2));
            const uint64_t p2 = f32x2_pack(ex2(x.x), ex2(x.y));
            acc[u >> 1] = add_f32x2(acc[u >> 1], p2);
            const float2 pv = f32x2_unpack(mul_f32x2(p2, f32x2_pack(vs[u], vs[u + 1])));
            s[(e + u) >> 1] = pack_half2(pv.x, pv.y);
        }
    }
    const float2 a0 = f32x2_unpack(acc[0]), a1 = f32x2_unpack(acc[1]);
    l += (a0.x + a0.y) + (a1.x + a1.y);
}

// tmap: FP16 pools, 2 KB boxes of one block's 16 rows of one 64-dim half; 8-bit pools, a 2 KB box of one
// tile's codes (16 rows of 128).
template <bool kI8>
__global__ void __launch_bounds__(Cfg<kI8>::kThreads, 1) prefill_kernel(const __grid_constant__ CUtensorMap tmap,
                                                                         const PrefillArgs a)
{
    using C = Cfg<kI8>;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    const uint32_t sb = smem_u32(smem);
    // CTA = (tile of `tok` query tokens, group of `hpc` query heads sharing one K/V head, sequence). Its 128
    // MMA rows are (head r / tok, token r % tok): the group's K/V tiles are gathered once for all its heads.
    const int qt = blockIdx.x, s = blockIdx.z;
    const int hq0 = blockIdx.y * a.hpc, hkv = hq0 / a.group;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // Launched with a programmatic dependency on the stream's previous kernel: this grid's CTAs may be
    // placed on SMs that kernel has left (or never used) before it ends, and wait here for its results.
    // Nothing in global memory is read before this point, so any earlier kernel may produce the inputs.
    // (The trigger at the top lets a following decode launch of a mixed pkv_step layer start beside it.)
    pdl_trigger();
    // Before the dependency wait, a hint only: the first tile's K and V lines into L2, from this CTA's metadata
    // as it reads now (everything is read again after the wait; only block ids inside the pool give addresses,
    // and a stale value costs at most a wasted prefetch). The lines then come from L2 once the wait is over.
    // These reads bypass L1 (ld.global.cg), so that no line read before the wait, which the previous kernel
    // may still write, can serve a read after it.
    if (warp == kMmaWarp && lane < kBlocksPerTile * 2) {
        const int q0e = __ldcg(a.q_start + s), qle = __ldcg(a.q_start + s + 1) - q0e, ctxe = __ldcg(a.ctx_lens + s);
        if (qle >= 1 && qle <= ctxe && ctxe <= a.max_blocks * kBlockSize && qt * a.tok < qle) {
            const int pme = ctxe - qle + qt * a.tok + min(a.tok, qle - qt * a.tok) - 1;  // last position
            const int b = lane >> 1, kvl = lane & 1;  // a lane per (block, K|V) tile of 4 KB
            if (b <= pme / kBlockSize) {
                const int id = __ldcg(a.tables + (int64_t)s * a.max_blocks + b);
                if (id >= 0 && (int64_t)id < a.num_blocks)
                    bulk_prefetch_l2(a.base + (int64_t)id * a.block_bytes + (int64_t)a.layer * a.layer_bytes +
                                         (int64_t)(kvl * a.num_heads + hkv) * a.tile_bytes,
                                     (uint32_t)a.tile_bytes);
            }
        }
    }
    pdl_wait();

    // ---- validate this sequence's metadata (all threads agree)
    const int q0 = __ldg(a.q_start + s);
    const int qlen = __ldg(a.q_start + s + 1) - q0;
    const int ctx = __ldg(a.ctx_lens + s);
    if (q0 < 0 || qlen < 1 || qlen > ctx || qlen > a.max_q_len || ctx > a.max_blocks * kBlockSize) {
        if (qt == 0 && blockIdx.y == 0 && threadIdx.x == 0)
            atomicOr(a.status, ctx > a.max_blocks * kBlockSize ? PKV_DEV_BAD_CTX : PKV_DEV_BAD_QLEN);
        return;
    }
    if (qt * a.tok >= qlen) return;
    const int ntok = min(a.tok, qlen - qt * a.tok);  // this CTA's query tokens
    const int p0 = ctx - qlen + qt * a.tok;           // position of its first token
    const int pos_max = p0 + ntok - 1;
    const int n = pos_max / kKeys + 1;       // 128-key tiles
    const int nblk = pos_max / kBlockSize + 1;
    const int32_t* trow = a.tables + (int64_t)s * a.max_blocks;
    // The first S waits on two cold reads, Q and the first K tile (already on its way into L2, above): start Q
    // into L2 now (prefetch hints through the load path, not the copy engine, whose queue the first tile's boxes
    // need), a line (128 B) per thread.
    {
        const int lines_per_tok = a.hpc * 2;  // hpc rows of 256 B
        for (int i = threadIdx.x; i < ntok * lines_per_tok; i += C::kThreads)
            prefetch_l2(a.q + ((int64_t)(q0 + qt * a.tok + i / lines_per_tok) * a.num_q_heads + hq0) * kHeadDim +
                        (i % lines_per_tok) * 64);
    }
    bool bad = false;
    for (int b = threadIdx.x; b < nblk; b += C::kThreads) {
        const int id = __ldg(trow + b);
        bad |= id < 0 || (int64_t)id >= a.num_blocks;
    }
    if (__syncthreads_or(bad)) {
        if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        return;
    }

    const uint32_t bars = sb + C::kSmBars;
    auto bar = [&](int i) { return bars + 8u * (uint32_t)i; };
    volatile int* abort = reinterpret_cast<volatile int*>(smem + C::kSmAbort);
    if (threadIdx.x == 0) {
        for (int i = 0; i < C::kStagesK; ++i) {
            mbar_init(bar(C::K_FULL + i), kI8 ? 1 : 2);
            mbar_init(bar(C::K_EMPTY + i), 1);
            mbar_init(bar(C::K_CONV + i), 2);
        }
        for (int i = 0; i < C::kStagesV; ++i) {
            mbar_init(bar(C::V_FULL + i), kI8 ? 1 : 2);
            mbar_init(bar(C::V_EMPTY + i), 1);
            mbar_init(bar(C::V_CONV + i), 2);
        }
        for (int i = 0; i < kScaleStages; ++i) {
            mbar_init(bar(C::SC_FULL + i), 2);
            mbar_init(bar(C::SC_FREE + i), 4);
        }
        for (int i = 0; i < kBufs; ++i) {
            mbar_init(bar(C::S_FULL + i), 1);
            mbar_init(bar(C::P_FULL + i), kSoftmaxThreads);
            mbar_init(bar(C::PV_DONE + i), 1);
        }
        mbar_init(bar(C::V_FIXED), kI8 ? kSoftmaxThreads : 1);
        mbar_init(bar(C::Q_READY), kSoftmaxThreads);
        mbar_init(bar(C::S_ALL_DONE), 1);
        mbar_init(bar(C::PV_ALL_DONE), 1);
        *abort = 0;
        fence_mbar_init();
    }
    if (warp == kMmaWarp) {
        tmem_alloc(sb + C::kSmTmemSlot, kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + C::kSmTmemSlot);

    // Each warpgroup sets its register budget at the top of its own branch (the same instruction in all
    // four of its warps), so that ptxas allocates each role's code with that role's budget.
    if (warp < kProducerWarps) {
        regs_dec<C::kSideRegs>();
        // ================================================= TMA producers (lane < 8: block lane of each tile).
        // FP16: warp 0 copies K's 64-dim half 0, warp 1 K's half 1, warps 2, 3 V's halves.
        // 8-bit: warps 0, 2 K's and V's codes (into the tile's second slab); warps 1, 3 K's and V's row
        // scales into the scale ring, whose stages the softmax releases once it is done with the tile.
        const int kv = warp >> 1;
        const int b = lane & (kBlocksPerTile - 1), half = warp & 1;
        const bool copier = lane < kBlocksPerTile;
        const bool scales = kI8 && half;
        const int kvh = kv * a.num_heads + hkv;
        const uint32_t ring = sb + (kv ? C::kSmVRing : C::kSmKRing) + ((kI8 || half) ? kTileSlab : 0);
        const uint32_t scale_ring = sb + C::kSmScales + kv * kKeys * 4;
        const uint32_t full0 = bar(scales ? C::SC_FULL : kv ? C::V_FULL : C::K_FULL);
        const uint32_t empty0 = bar(scales ? C::SC_FREE : kv ? C::V_EMPTY : C::K_EMPTY);
        const uint32_t box_bytes = kI8 ? (half ? 4 * kBlockSize : kCodesBytes) : kTileBytes / 2;
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
        const int stages = scales ? kScaleStages : kv ? C::kStagesV : C::kStagesK;
        int issued = 0;
        bool stop = false;
        // The copy engine serves boxes in issue order and P_0 V_0 comes a whole softmax period after S_0:
        // V's producers start once S_0 is done (so K_0 has landed), so that K_0's boxes are not queued
        // behind V_0's. (S_FULL of buffer 0 cannot complete a second phase before P_0 V_0, which needs V_0,
        // so this wait cannot miss its phase; K_FULL of stage 0 could, via K_3.)
        if (kv && !scales && !flag_wait(bar(C::S_FULL), 0, abort, a.status)) stop = true;
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
                if (lane == 0) mbar_arrive_expect_tx(full0 + 8 * st, nb * box_bytes);
                __syncwarp();
                if (copier && b < nb) {
                    if (!kI8)
                        tma_load_5d(ring + st * kTileOpBytes + b * 2048, &tmap, half * 64, 0, kvh, a.layer, idq[u],
                                    full0 + 8 * st);
                    else if (!half)
                        tma_load_5d(ring + st * kTileOpBytes + b * kCodesBytes, &tmap, 0, 0, kvh, a.layer, idq[u],
                                    full0 + 8 * st);
                    else
                        bulk_g2s(scale_ring + st * kScaleStage + b * 4 * kBlockSize,
                                 a.base + (int64_t)idq[u] * a.block_bytes + (int64_t)a.layer * a.layer_bytes +
                                     (int64_t)kvh * a.tile_bytes + kCodesBytes,
                                 4 * kBlockSize, full0 + 8 * st);
                }
                issued = i + 1;
                const int blk = kBlocksPerTile * (i + kIdAhead) + b;  // refill this slot with tile i + kIdAhead
                idq[u] = copier && i + kIdAhead < n && blk < nblk ? __ldg(trow + blk) : 0;
            }
        }
        if (!kI8 && warp == 2 && !stop) {
            // The last tile: keys past the last row's position may hold anything (even NaN), and rows of
            // blocks past the table's end were not copied at all. Zero those V rows (both halves, once they
            // have landed) so that P = 0 times V stays 0 in the tensor core, then release the tile.
            const int i = n - 1, st = i % C::kStagesV;
            if (flag_wait(full0 + 8 * st, (uint32_t)(i / C::kStagesV) & 1u, abort, a.status)) {
                const uint32_t vt = sb + C::kSmVRing + st * kTileOpBytes;
                const int first = pos_max + 1 - (n - 1) * kKeys;
                for (int c = first * 8 + lane; c < kKeys * 8; c += 32) {
                    const int r = c >> 3, ch = c & 7;
                    st_shared_v4(vt + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                    st_shared_v4(vt + kTileSlab + r * 128 + ch * 16, make_uint4(0, 0, 0, 0));
                }
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::V_FIXED));
            }
        }
        // copies still in flight (after an abort) must land before the CTA exits
        for (int i = (issued > stages ? issued - stages : 0); i < issued; ++i)
            mbar_wait(full0 + 8 * (i % stages), (uint32_t)(i / stages) & 1u);
    } else if (warp >= kMmaWarp && warp < kMmaWarp + 4) {
        regs_dec<C::kSideRegs>();
        if (warp == kMmaWarp) {
        // ================================================= S issuer: the whole warp runs the loop (warp-uniform
        // waits and descriptors) and one elected lane issues each MMA and commit.
        // base descriptors; each MMA adds a constant offset (one 64-bit add instead of building a descriptor)
        const uint64_t dq = sw128_desc(sb + C::kSmQ, 16, 1024);
        const uint64_t dk = sw128_desc(sb + C::kSmKRing, 16, 1024);
        for (int j = 0; j < n; ++j) {
            const int ks = j % C::kStagesK, sbuf = j % kBufs;
            // K_j landed (FP16) or converted (8-bit)
            const bool ok = (j > 0 || flag_wait(bar(C::Q_READY), 0, abort, a.status)) &&
                            flag_wait(bar((kI8 ? C::K_CONV : C::K_FULL) + ks), (uint32_t)(j / C::kStagesK) & 1u, abort,
                                      a.status) &&
                            // S buffer j%3 last held P_{j-3}, which P_{j-3} V_{j-3} must have read
                            (j < kBufs || flag_wait(bar(C::PV_DONE + sbuf), (uint32_t)((j - kBufs) / kBufs) & 1u, abort,
                                                    a.status));
            if (!ok) break;
            tc_fence_after();
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_f16_warp(tmem + kColS + sbuf * kSBufCols, desc_add(dq, (kk >> 2) * kQSlab + (kk & 3) * 32),
                                desc_add(dk, ks * kTileOpBytes + (kk >> 2) * kTileSlab + (kk & 3) * 32), kIdescS, kk > 0);
            tc_commit_warp(bar(C::S_FULL + sbuf));
            tc_commit_warp(bar(C::K_EMPTY + ks));
        }
        // every MMA this warp issued must have finished before the CTA frees its tensor memory and exits
        tc_commit_warp(bar(C::S_ALL_DONE));
        mbar_wait(bar(C::S_ALL_DONE), 0);
        __syncwarp();
        } else if (warp == kPvWarp) {
        // ================================================= P V issuer, in the same style
        const uint64_t dv = sw128_desc(sb + C::kSmVRing, kTileSlab, 1024);
        for (int j = 0; j < n; ++j) {
            const int vs = j % C::kStagesV, pbuf = j % kBufs;
            // V_j converted (8-bit), landed (FP16), or for the last FP16 tile: landed and its tail zeroed
            const bool ok =
                flag_wait(bar(C::P_FULL + pbuf), (uint32_t)(j / kBufs) & 1u, abort, a.status) &&
                (kI8 ? flag_wait(bar(C::V_CONV + vs), (uint32_t)(j / C::kStagesV) & 1u, abort, a.status)
                     : j == n - 1 ? flag_wait(bar(C::V_FIXED), 0, abort, a.status)
                                  : flag_wait(bar(C::V_FULL + vs), (uint32_t)(j / C::kStagesV) & 1u, abort, a.status));
            if (!ok) break;
            tc_fence_after();
            const uint32_t pcol = tmem + kColS + pbuf * kSBufCols;
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
                tc_mma_f16_ts_warp(tmem + kColO, pcol + kk * 8, desc_add(dv, vs * kTileOpBytes + kk * 2048), kIdescPV,
                                   (j > 0 || kk > 0) ? 1u : 0u);
            tc_commit_warp(bar(C::PV_DONE + pbuf));
            tc_commit_warp(bar(C::V_EMPTY + vs));
        }
        tc_commit_warp(bar(C::PV_ALL_DONE));
        mbar_wait(bar(C::PV_ALL_DONE), 0);
        __syncwarp();
        }
    } else if (warp >= kFirstConvWarp) {
        regs_dec<C::kConvRegs>();
        // ================================================= 8-bit pools: code -> FP16 conversion. Warps 12, 13
        // convert K tiles and warps 14, 15 V tiles, two key rows per thread, as two independent streams (K is
        // needed two tiles before V: one stream doing both would hold K back behind V). Thread i takes rows i
        // and i + 64, so a warp's 32 rows cover all eight swizzle phases (no bank conflicts).
        const int kv = (warp - kFirstConvWarp) >> 1;
        const int r0 = threadIdx.x - (kFirstConvWarp + 2 * kv) * 32;  // rows r0, r0 + 64
        const int stages = kv ? C::kStagesV : C::kStagesK;
        const uint32_t full0 = bar(kv ? C::V_FULL : C::K_FULL), conv0 = bar(kv ? C::V_CONV : C::K_CONV);
        const uint32_t ring = sb + (kv ? C::kSmVRing : C::kSmKRing);
        for (int j = 0; j < n; ++j) {
            const int st = j % stages;
            if (!flag_wait(full0 + 8 * st, (uint32_t)(j / stages) & 1u, abort, a.status)) break;
            // the two rows one after the other: one copy of the conversion code (these warps share their
            // schedulers' instruction caches with the softmax warps)
#pragma unroll 1
            for (int u = 0; u < 2; ++u)
                convert_code_row(ring + st * kTileOpBytes, r0 + 64 * u, j * kKeys + r0 + 64 * u <= pos_max);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(conv0 + 8 * st);
        }
    } else if (warp >= kFirstSoftmaxWarp && warp < kFirstSoftmaxWarp + 4) {
        regs_inc<C::kSoftmaxRegs>();
        // ================================================= softmax: thread = query row
        const int qtr = warp & 3;
        const int row = qtr * 32 + lane;
        const int rhead = row / a.tok, rtok = row % a.tok;
        const bool valid = rhead < a.hpc && rtok < ntok;  // else a padding row (zero Q, never written)
        const int pos = p0 + rtok;
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
                const int hh = r / a.tok, tt = r % a.tok;
                v[u] = make_uint4(0, 0, 0, 0);
                if (hh < a.hpc && tt < ntok)
                    v[u] = __ldg(reinterpret_cast<const uint4*>(
                                     a.q + ((int64_t)(q0 + qt * a.tok + tt) * a.num_q_heads + hq0 + hh) * kHeadDim) +
                                 ch);
            }
#pragma unroll
            for (int u = 0; u < kPer; ++u) {
                const int c = t + u * kSoftmaxThreads, r = c >> 4, ch = c & 15;
                st_shared_v4(sb + C::kSmQ + (ch >> 3) * kQSlab + r * 128 + (((ch & 7) ^ (r & 7)) << 4), v[u]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(C::Q_READY));
        }
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n; ++j) {
            const int sbuf = j % kBufs;
            if (!flag_wait(bar(C::S_FULL + sbuf), (uint32_t)(j / kBufs) & 1u, abort, a.status)) {
                ok = false;
                break;
            }
            tc_fence_after();
            const uint32_t ts = tl + kColS + sbuf * kSBufCols;
            const int key0 = j * kKeys;
            // 8-bit pools: this tile's K and V row scales (stage j % 6 of the scale ring)
            const float4* ksc = reinterpret_cast<const float4*>(smem + C::kSmScales + (j % kScaleStages) * kScaleStage);
            const float4* vsc = ksc + kKeys / 4;
            if constexpr (kI8) {
                if (!flag_wait(bar(C::SC_FULL + j % kScaleStages), (uint32_t)(j / kScaleStages) & 1u, abort,
                               a.status)) {
                    ok = false;
                    break;
                }
                if (j == n - 1) {
                    // the last tile: keys past the last query position take V scale 0 (their scale bytes may be
                    // anything, even NaN, and their weights are 0), written by the softmax threads, one key each,
                    // before any of them reads the scales
                    const int t = threadIdx.x - kFirstSoftmaxWarp * 32;
                    if (key0 + t > pos_max) const_cast<float*>(reinterpret_cast<const float*>(vsc))[t] = 0.f;
                    mbar_arrive(bar(C::V_FIXED));
                    if (!flag_wait(bar(C::V_FIXED), 0, abort, a.status)) {
                        ok = false;
                        break;
                    }
                }
            }
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
            if constexpr (kI8) scale_columns<64>(sr, ksc);
            if (diag) mask_tail<64>(sr, nvis);
            float mx = max64(sr);
            if (j > 0) {
                // P_{j-1}, stored at the end of the previous tile: its stores have had this tile's first load and
                // max to complete, so the wait here costs the softmax nothing (P_{j-1} V_{j-1} has slack: its S
                // buffer is next needed two tiles on)
                tc_wait_st();
                tc_fence_before();
                mbar_arrive(bar(C::P_FULL + (j - 1) % kBufs));
            }
            tc_wait_ld64(sr + 64);
            if constexpr (kI8) scale_columns<64>(sr + 64, ksc + 16);
            if (diag) mask_tail<64>(sr + 64, nvis - 64);
            const float m_tile = fmaxf(mx, max64(sr + 64)) * a.scale_log2;
            const bool raise = m_tile > m_used + kRescaleThreshold;  // false while the row has seen no key
            if (j > 0 && __any_sync(0xffffffffu, raise)) {
                // the previous P V product must have landed before O is rescaled
                if (!flag_wait(bar(C::PV_DONE + (j - 1) % kBufs), (uint32_t)((j - 1) / kBufs) & 1u, abort,
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
                if constexpr (kI8)
                    softmax_quarter_vscaled(sr + q * 32, a.scale_log2, m_sub, l, vsc + q * 8);
                else
                    softmax_quarter(sr + q * 32, a.scale_log2, m_sub, l);
                tc_st16_async(tp + q * 16, sr + q * 32);
            }
            if constexpr (kI8) {
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(C::SC_FREE + j % kScaleStages));  // done with this tile's scales
            }
        }
        // the last tile's P (or, after a failed wait, no store of this thread left in flight)
        tc_wait_st();
        if (ok) {
            tc_fence_before();
            mbar_arrive(bar(C::P_FULL + (n - 1) % kBufs));
        }
        // ---- epilogue: O / l -> FP16 (each row's 256 B written by its thread)
        if (ok && flag_wait(bar(C::PV_DONE + (n - 1) % kBufs), (uint32_t)((n - 1) / kBufs) & 1u, abort, a.status)) {
            tc_fence_after();
            const float inv = 1.f / l;
            uint4* dst =
                reinterpret_cast<uint4*>(a.out + ((int64_t)(q0 + qt * a.tok + rtok) * a.num_q_heads + hq0 + rhead) *
                                         kHeadDim);
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
    const bool i8 = pool->geom.dtype == PKV_DTYPE_INT8;
    static bool attr_set[2][64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[i8][dev]) {
        cudaError_t e = i8 ? cudaFuncSetAttribute(prefill_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  Cfg<true>::kSmAlloc)
                           : cudaFuncSetAttribute(prefill_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                  Cfg<false>::kSmAlloc);
        if (e != cudaSuccess) return e;
        attr_set[i8][dev] = true;
    }
    PrefillArgs a;
    a.q = static_cast<const __half*>(q);
    a.out = static_cast<__half*>(out);
    a.q_start = q_start;
    a.tables = tables;
    a.ctx_lens = ctx_lens;
    a.base = pool->geom.base;
    a.block_bytes = pool->geom.block_bytes;
    a.layer_bytes = pool->geom.layer_bytes;
    a.tile_bytes = pool->geom.tile_bytes;
    a.max_blocks = max_blocks;
    a.num_heads = pool->geom.num_heads;
    a.num_q_heads = pool->geom.num_q_heads;
    a.group = pool->geom.group;
    a.hpc = pool->geom.group <= kRows ? pool->geom.group : 1;
    a.tok = kRows / a.hpc;
    a.layer = layer;
    a.max_q_len = max_q_len;
    a.num_blocks = pool->geom.num_blocks;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.status = pool->status_dev;
    CUtensorMap tmap;
    static_assert(sizeof(tmap) == sizeof(pool->kv_tmap.bytes), "tensor map size");
    memcpy(&tmap, (i8 ? pool->tile_tmap : pool->kv_tmap).bytes, sizeof(tmap));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((max_q_len + a.tok - 1) / a.tok, pool->geom.num_q_heads / a.hpc, num_seqs);
    cfg.blockDim = dim3(i8 ? Cfg<true>::kThreads : Cfg<false>::kThreads);
    cfg.dynamicSmemBytes = i8 ? Cfg<true>::kSmAlloc : Cfg<false>::kSmAlloc;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    // FP16 pools launch with the programmatic dependency (+1 % per chunk call); the 8-bit kernel measured
    // slower per tile with it (270 against 317 TFLOP/s on the 8-chunk schedule; 462 against 483 with the
    // current kernel: chunk 0 faster, every later chunk slower) and launches without.
    cfg.numAttrs = i8 ? 0 : 1;
    return i8 ? cudaLaunchKernelEx(&cfg, prefill_kernel<true>, tmap, a)
              : cudaLaunchKernelEx(&cfg, prefill_kernel<false>, tmap, a);
}

}  // namespace pkv
