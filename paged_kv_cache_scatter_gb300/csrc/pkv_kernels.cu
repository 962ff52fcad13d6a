// pkv_kernels.cu — kv_append (reshape_and_cache), split-K paged decode
// attention and its partition merge, for sm_103a.
//
// Pool layout (one block = every layer of 16 token positions):
//   [block][layer][K,V][head][16 tokens][128 dims] FP16
// so one head's K (or V) for one block is a contiguous 4,096-byte tile, and
// consecutive heads of the same block/layer are 4,096 B apart
// ("llm-inference-batching" (faangrind), the KV pool listing).
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "pkv_internal.h"
#include "ptx.cuh"

namespace pkv {

// Sticky per-device error word (PKV_DEV_* bits). Host code takes its device
// address once per device with cudaGetSymbolAddress and passes it to kernels.
__device__ unsigned int g_status_word;

cudaError_t status_word(int device, unsigned int** out)
{
    int cur = 0;
    cudaError_t e = cudaGetDevice(&cur);
    if (e != cudaSuccess) return e;
    if (cur != device && (e = cudaSetDevice(device)) != cudaSuccess) return e;
    e = cudaGetSymbolAddress(reinterpret_cast<void**>(out), g_status_word);
    if (cur != device) cudaSetDevice(cur);
    return e;
}

// ======================================================================
// kv_append: one thread moves one 16-byte chunk. A token's K row for one
// head is 256 B (16 chunks) and lands at tile offset (slot % 16) * 256 of
// its block's (layer, K, head) tile; V likewise in the V half.
// "llm-inference-batching", step 7: new keys and values are appended.
// Grid (chunk blocks, tokens): a block's threads are chunks c = K|V x heads x
// 16 + head x 16 + chunk of one token (blockIdx.y, plus multiples of
// gridDim.y past 65,535 tokens), so no thread divides by a runtime value; the
// new row's load does not depend on the slot and is issued beside it.

__global__ void __launch_bounds__(256) kv_append_kernel(char* __restrict__ pool, int64_t block_bytes,
                                                        int64_t layer_off, int64_t kv_bytes, int num_heads,
                                                        const uint4* __restrict__ k, const uint4* __restrict__ v,
                                                        const int64_t* __restrict__ slots, int num_tokens,
                                                        int64_t num_slots, unsigned int* status)
{
    const int hc = num_heads * 16;  // chunks of one token's K (or V) rows
    const int c = blockIdx.x * blockDim.x + threadIdx.x;
    if (c >= 2 * hc) return;
    const int kv = c >= hc;
    const int h = (c - kv * hc) >> 4, chunk = c & 15;
    for (int tok = blockIdx.y; tok < num_tokens; tok += gridDim.y) {
        const int64_t slot = __ldg(slots + tok);
        const uint4 val = __ldg((kv ? v : k) + ((int64_t)tok * num_heads + h) * 16 + chunk);
        if (slot < 0 || slot >= num_slots) {
            if (c == 0) atomicOr(status, PKV_DEV_BAD_SLOT);
            continue;
        }
        const int64_t blk = slot >> 4;
        const int t = (int)(slot & 15);
        *reinterpret_cast<uint4*>(pool + blk * block_bytes + layer_off + kv * kv_bytes + (int64_t)h * kTileBytes +
                                  t * 256 + chunk * 16) = val;
    }
}

cudaError_t launch_kv_append(const PoolGeom& g, int layer, const void* k, const void* v, const int64_t* slots,
                             int num_tokens, unsigned int* status, cudaStream_t stream)
{
    if (num_tokens == 0) return cudaSuccess;
    const int chunks = 2 * g.num_heads * 16;
    const int threads = chunks < 256 ? chunks : 256;  // a multiple of 32
    const dim3 grid((unsigned)((chunks + threads - 1) / threads), (unsigned)(num_tokens < 65535 ? num_tokens : 65535));
    kv_append_kernel<<<grid, threads, 0, stream>>>(
        const_cast<char*>(g.base), g.block_bytes, (int64_t)layer * g.layer_bytes, g.kv_bytes, g.num_heads,
        static_cast<const uint4*>(k), static_cast<const uint4*>(v), slots, num_tokens, g.num_blocks * kBlockSize,
        status);
    return cudaGetLastError();
}

// ======================================================================
// Decode attention.
//
// One CTA = (partition p, head h, row r); a partition is partition_tokens
// consecutive keys (a whole number of blocks). Its WARPS warps take the
// partition's blocks round-robin; each warp is an independent streaming
// consumer with a private ring of STAGES stages, one block (K tile + V tile,
// 8 KB) per stage, filled by 1-D bulk async copies that complete on an
// mbarrier. Lane 0 of the warp issues the copies; the whole warp consumes.
//
// Per block: lane = (token t = lane/2, half hf = lane%2) forms q.k_t over 64
// dims (the two halves meet with one shuffle), the warp takes the block max
// (online softmax in the log2 domain, the scale pre-multiplied by log2 e),
// and each lane then owns 4 output dims for the P.V update.
//
// The warps' states merge in shared memory in fixed order. A single-partition
// row writes its FP16 output directly. Otherwise each partition writes its
// un-normalised output, max and sum to the workspace and bumps a per-(row,
// head) counter; the CTA that brings the counter to the row's partition
// count merges all partitions in partition order and resets the counter to
// zero ("The inference engine" (wpnews), "IO-aware attention": tiles combine
// exactly through their softmax statistics). The partition plan depends only
// on ctx_len and partition_tokens, so a row's result is the same in any batch.
//
// With `append` set, the kernel also performs kv_append for the decode rows:
// the CTA holding a row's last partition writes the row's new K/V (token r of
// k_new / v_new) for its head into the slot slot_mapping[r], and the warp that
// streams that block patches the new row into its shared-memory copy, so the
// query sees its own new key exactly as if the append had run first.

constexpr int kDecodeWarps = 4;
constexpr int kDecodeStages = 2;
constexpr int kCascadeWarps = 2;  // cascade decode's private-key launch
constexpr int kStageBytes = 2 * kTileBytes;
constexpr int kMaxMergeParts = kMaxPartitionsPerRow;  // s_w and s_l of the merge fit in the idle rings

struct DecodeArgs {
    char* pool;
    int64_t block_bytes;
    int64_t head_off;   // layer * layer_bytes (the head offset is added per CTA)
    int64_t kv_bytes;
    int64_t num_blocks;
    int num_heads;
    const __half* q;
    const int32_t* tables;
    int max_blocks;
    const int32_t* ctx_lens;
    float scale_log2;
    __half* out;
    float* ws_o;            // [B][H][max_parts][128]
    float* ws_ml;           // [B][H][max_parts][2]
    unsigned int* counters; // [B][H], zero between launches
    int max_parts;
    int ws_parts;           // partial slots per (row, head)
    int part_tokens;
    const __half* k_new;    // [B][H][128] when append
    const __half* v_new;
    const int64_t* slots;   // [B] when append
    int append;
    int no_wait;             // launched after a kernel whose results it does not read: skip the dependency wait
    unsigned int* status;
    // cascade: a row's partitions wholly inside its group's shared prefix were computed already
    const int32_t* group_start;   // [num_groups + 1] or NULL
    const int32_t* group_blocks;  // [num_groups]
    int num_groups;
};

template <int WARPS, int STAGES>
struct DecodeLayout {
    static constexpr int kRing = WARPS * STAGES * kStageBytes;
    static constexpr int kPbuf = kRing;                        // [WARPS][16] float
    static constexpr int kStats = kPbuf + WARPS * 16 * 4;      // [WARPS][2] float
    static constexpr int kBars = kStats + WARPS * 2 * 4;       // [WARPS][STAGES][2] u64
    static constexpr int kFlag = kBars + WARPS * STAGES * 2 * 8;
    static constexpr int kBytes = kFlag + 16;
};

// Counter bump with release (prior writes of this CTA, ordered by a CTA
// barrier, become visible first) and acquire (the other partitions' writes
// are visible to this CTA afterwards) at GPU scope.
__device__ __forceinline__ unsigned int atomic_add_acq_rel_gpu(unsigned int* p, unsigned int v)
{
    unsigned int old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

template <int WARPS, int STAGES>
__global__ void __launch_bounds__(WARPS * 32) decode_kernel(const DecodeArgs a)
{
    using Lay = DecodeLayout<WARPS, STAGES>;
    extern __shared__ __align__(1024) unsigned char smem[];
    // Grid (partition, head, row): the partitions of one (row, head) are
    // dispatched next to each other, so their partials are still in L2 when
    // the last of them merges.
    const int p = blockIdx.x, h = blockIdx.y, r = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    // The row's length and (cascade) its group's shared prefix are independent loads: both are issued before
    // either is used, so a short cascade row's CTA waits for one memory round trip here, not two.
    const int ctx = __ldg(a.ctx_lens + r);
    // Partition plan: keys [0, ctx) in partitions of at most part_tokens. Cascade: keys [0, S) of the row's group's
    // shared prefix are partitioned on their own (computed already, slots 0 .. nsh-1); this CTA takes
    // partition p of [S, ctx), slot nsh + p.
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
        if (p == 0 && h == 0 && threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_CTX);
        return;
    }
    // [S, ctx) goes into as few partitions as part_tokens allows, of equal length in whole blocks (1,043 keys:
    // 528 + 515, not 1,024 + 19), so that no short partition's CTA trails the launch.
    if (ctx <= S) {  // the group's shared prefix must lie below the row's newest token
        if (p == 0 && h == 0 && threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_CTX);
        return;
    }
    const int nsh = (S + a.part_tokens - 1) / a.part_tokens;
    const int np = (ctx - S + a.part_tokens - 1) / a.part_tokens;
    const int span = ((ctx - S + np - 1) / np + kBlockSize - 1) / kBlockSize * kBlockSize;
    const int tok_lo = S + p * span;
    if (tok_lo >= ctx) return;
    const int nparts = nsh + (ctx - S + span - 1) / span;
    const int slot_p = nsh + p;
    const int blk_lo = tok_lo >> 4;
    const int blk_hi = (min(tok_lo + span, ctx) + 15) >> 4;
    const int nblk = blk_hi - blk_lo;
    int count = nblk > warp ? (nblk - warp + WARPS - 1) / WARPS : 0;  // <= 32 by construction

    unsigned char* ring = smem + warp * STAGES * kStageBytes;
    float* pbuf = reinterpret_cast<float*>(smem + Lay::kPbuf) + warp * 16;
    float* stats = reinterpret_cast<float*>(smem + Lay::kStats);
    const uint32_t bar0 = smem_u32(smem + Lay::kBars) + warp * STAGES * 16;

    // Physical block ids of this warp's blocks: lane i holds the i-th.
    const int32_t* trow = a.tables + (int64_t)r * a.max_blocks;
    int my_id = 0;
    bool bad = false;
    if (lane < count) {
        my_id = __ldg(trow + blk_lo + warp + lane * WARPS);
        bad = my_id < 0 || (int64_t)my_id >= a.num_blocks;
    }
    if (__any_sync(0xffffffffu, bad)) {
        if (lane == 0) atomicOr(a.status, PKV_DEV_BAD_BLOCK);
        count = 0;
    }

    const char* kbase = a.pool + a.head_off + (int64_t)h * kTileBytes;
    if (lane == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar0 + 16 * s, 1);
            mbar_init(bar0 + 16 * s + 8, 1);
        }
        fence_mbar_init();
    }
    __syncwarp();

    // Prologue: fill the ring.
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
        const int id = __shfl_sync(0xffffffffu, my_id, s);
        if (s < count && lane == 0) {
            const char* src = kbase + (int64_t)id * a.block_bytes;
            const uint32_t dst = smem_u32(ring + s * kStageBytes);
            mbar_arrive_expect_tx(bar0 + 16 * s, kTileBytes);
            bulk_g2s(dst, src, kTileBytes, bar0 + 16 * s);
            mbar_arrive_expect_tx(bar0 + 16 * s + 8, kTileBytes);
            bulk_g2s(dst + kTileBytes, src + a.kv_bytes, kTileBytes, bar0 + 16 * s + 8);
        }
    }

    // Everything above reads only what the step's earlier layers never write (lengths, tables, this
    // layer's K/V). With a programmatic dependency on the previous layer's kernel, wait for it here, before
    // reading q or the new K/V and before touching the workspace or the output.
    // Without the wait (no_wait), one CTA still waits: a cascade's private launch then ends only after the shared
    // launch it runs beside, so work after the call in the stream finds both done.
    if (!a.no_wait || (a.group_start && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0)) pdl_wait();

    // The new token (position ctx - 1) lives in this partition's last block.
    const int last_local = ((ctx - 1) >> 4) - blk_lo;
    int patch_iter = -1;  // iteration of this warp that streams the new token's block
    uint4 knew = make_uint4(0, 0, 0, 0), vnew = make_uint4(0, 0, 0, 0);
    if (a.append && slot_p == nparts - 1) {
        const int64_t slot = __ldg(a.slots + r);
        const int32_t tb = __ldg(trow + ((ctx - 1) >> 4));
        const bool consistent = slot == (int64_t)tb * kBlockSize + ((ctx - 1) & 15) && tb >= 0 &&
                                (int64_t)tb < a.num_blocks;
        if (!consistent) {
            if (threadIdx.x == 0) atomicOr(a.status, PKV_DEV_BAD_SLOT);
        } else {
            const uint4* ks = reinterpret_cast<const uint4*>(a.k_new + ((int64_t)r * a.num_heads + h) * kHeadDim);
            const uint4* vs = reinterpret_cast<const uint4*>(a.v_new + ((int64_t)r * a.num_heads + h) * kHeadDim);
            if (warp == last_local % WARPS) {
                patch_iter = last_local / WARPS;
                knew = __ldg(ks + (lane & 15));
                vnew = __ldg(vs + (lane & 15));
            }
            if (warp == 0) {  // the global write, for later steps: lanes 0-15 K, 16-31 V
                char* dst = a.pool + slot / kBlockSize * a.block_bytes + a.head_off + (int64_t)h * kTileBytes +
                            (slot % kBlockSize) * 256 + (lane & 15) * 16 + (lane < 16 ? 0 : a.kv_bytes);
                *reinterpret_cast<uint4*>(dst) = __ldg((lane < 16 ? ks : vs) + (lane & 15));
            }
        }
    }

    // q, rotated per lane so that the K-tile reads below are free of bank
    // conflicts: register chunk j holds dims hf*64 + ((j + lane) & 7)*8 .. +8.
    const int t = lane >> 1, hf = lane & 1;
    float qf[8][8];
    {
        const __half* qrow = a.q + ((int64_t)r * a.num_heads + h) * kHeadDim + hf * 64;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qrow + ((j + lane) & 7) * 8));
            half8_to_float(raw, qf[j]);
        }
    }

    float m_run = -INFINITY, l_lane = 0.f;
    float o[4] = {0.f, 0.f, 0.f, 0.f};
    bool timed_out = false;
    int i = 0;
    for (; i < count; ++i) {
        const int s = i % STAGES;
        const uint32_t par = (uint32_t)(i / STAGES) & 1u;
        const uint32_t bk = bar0 + 16 * s, bv = bk + 8;
        unsigned char* kt = ring + s * kStageBytes;
        unsigned char* vt = kt + kTileBytes;
        const int key0 = (blk_lo + warp + i * WARPS) * kBlockSize;
        const int nvalid = min(kBlockSize, ctx - key0);

        if (!mbar_wait(bk, par)) { timed_out = true; break; }
        if (i == patch_iter) {
            if (lane < 16) *reinterpret_cast<uint4*>(kt + ((ctx - 1) & 15) * 256 + lane * 16) = knew;
            __syncwarp();
        }
        float acc = 0.f;
        {
            const uint4* krow = reinterpret_cast<const uint4*>(kt + t * 256 + hf * 128);
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                float kf[8];
                half8_to_float(krow[(j + lane) & 7], kf);
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(qf[j][e], kf[e], acc);
            }
        }
        acc += __shfl_xor_sync(0xffffffffu, acc, 1);
        const float sc = (t < nvalid) ? acc * a.scale_log2 : -INFINITY;
        float mb = sc;
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 4));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 8));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 16));
        const float m_new = fmaxf(m_run, mb);
        const float alpha = exp2f(m_run - m_new);
        const float pt = exp2f(sc - m_new);
        l_lane = l_lane * alpha + (hf == 0 ? pt : 0.f);
        m_run = m_new;
        if (hf == 0) pbuf[t] = pt;
        __syncwarp();

        if (!mbar_wait(bv, par)) { timed_out = true; break; }
        if (i == patch_iter) {
            if (lane < 16) *reinterpret_cast<uint4*>(vt + ((ctx - 1) & 15) * 256 + lane * 16) = vnew;
            __syncwarp();
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) o[e] *= alpha;
        {
            const float4* pp = reinterpret_cast<const float4*>(pbuf);
            const unsigned char* vcol = vt + lane * 8;
#pragma unroll
            for (int tq = 0; tq < 4; ++tq) {
                const float4 p4 = pp[tq];
                const float pv[4] = {p4.x, p4.y, p4.z, p4.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int tt = tq * 4 + e;
                    if (tt < nvalid) {  // rows past ctx may hold anything, even NaN
                        float vf[4];
                        half4_to_float(*reinterpret_cast<const uint2*>(vcol + tt * 256), vf);
#pragma unroll
                        for (int c = 0; c < 4; ++c) o[c] = fmaf(pv[e], vf[c], o[c]);
                    }
                }
            }
        }
        __syncwarp();
        if (i + STAGES < count) {
            const int id = __shfl_sync(0xffffffffu, my_id, i + STAGES);
            if (lane == 0) {
                fence_proxy_async_smem();
                const char* src = kbase + (int64_t)id * a.block_bytes;
                const uint32_t dst = smem_u32(ring + s * kStageBytes);
                mbar_arrive_expect_tx(bk, kTileBytes);
                bulk_g2s(dst, src, kTileBytes, bk);
                mbar_arrive_expect_tx(bv, kTileBytes);
                bulk_g2s(dst + kTileBytes, src + a.kv_bytes, kTileBytes, bv);
            }
        }
    }
    pdl_trigger();  // the next layer's CTAs may start their prologue as this grid drains
    if (timed_out) {
        // Give the copies still in flight into this warp's ring a bounded
        // chance to land before the shared memory is reused or released.
        if (lane == 0) atomicOr(a.status, PKV_DEV_TIMEOUT);
        for (int k = i; k < count && k < i + STAGES; ++k) {
            const uint32_t bk = bar0 + 16 * (k % STAGES);
            const uint32_t par = (uint32_t)(k / STAGES) & 1u;
            mbar_wait(bk, par);
            mbar_wait(bk + 8, par);
        }
    }

    // Merge the warps. Warp w's partial output goes into its own (now idle) ring.
    float l_w = l_lane;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) l_w += __shfl_xor_sync(0xffffffffu, l_w, off);
    float* mo = reinterpret_cast<float*>(ring);
    *reinterpret_cast<float4*>(mo + lane * 4) = make_float4(o[0], o[1], o[2], o[3]);
    if (lane == 0) {
        stats[warp * 2] = m_run;
        stats[warp * 2 + 1] = l_w;
    }
    __syncthreads();

    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < WARPS; ++w) M = fmaxf(M, stats[w * 2]);
    float L = 0.f, wt[WARPS];
#pragma unroll
    for (int w = 0; w < WARPS; ++w) {
        wt[w] = (stats[w * 2] == -INFINITY) ? 0.f : exp2f(stats[w * 2] - M);
        L = fmaf(wt[w], stats[w * 2 + 1], L);
    }
    const int64_t rh = (int64_t)r * a.num_heads + h;
    if (nparts == 1) {
        for (int d = threadIdx.x; d < kHeadDim; d += WARPS * 32) {
            float O = 0.f;
#pragma unroll
            for (int w = 0; w < WARPS; ++w)
                O = fmaf(wt[w], reinterpret_cast<const float*>(smem + w * STAGES * kStageBytes)[d], O);
            a.out[rh * kHeadDim + d] = __float2half_rn(O / L);
        }
        return;
    }
    const int64_t slot = rh * a.ws_parts + slot_p;
    for (int d = threadIdx.x; d < kHeadDim; d += WARPS * 32) {
        float O = 0.f;
#pragma unroll
        for (int w = 0; w < WARPS; ++w)
            O = fmaf(wt[w], reinterpret_cast<const float*>(smem + w * STAGES * kStageBytes)[d], O);
        a.ws_o[slot * kHeadDim + d] = O;
    }
    if (threadIdx.x == 0) {
        a.ws_ml[slot * 2] = M;
        a.ws_ml[slot * 2 + 1] = L;
    }
    // Publish the partial, then count it (one release by thread 0 after the
    // CTA barrier covers every thread's writes); the last partition to
    // arrive merges all of them in partition order.
    __syncthreads();
    unsigned int* flag = reinterpret_cast<unsigned int*>(smem + Lay::kFlag);
    if (threadIdx.x == 0) *flag = atomic_add_acq_rel_gpu(a.counters + rh, 1u) == (unsigned int)(nparts - 1);
    __syncthreads();
    if (!*flag) return;
    const int64_t base = rh * a.ws_parts;
    float* s_w = reinterpret_cast<float*>(smem);  // the rings are idle now
    float* s_l = s_w + kMaxMergeParts;
    for (int q = threadIdx.x; q < nparts; q += WARPS * 32) {
        s_w[q] = __ldcg(a.ws_ml + (base + q) * 2);
        s_l[q] = __ldcg(a.ws_ml + (base + q) * 2 + 1);
    }
    __syncthreads();
    float Mx = -INFINITY;
    for (int q = 0; q < nparts; ++q) Mx = fmaxf(Mx, s_w[q]);
    __syncthreads();
    for (int q = threadIdx.x; q < nparts; q += WARPS * 32) s_w[q] = exp2f(s_w[q] - Mx);
    __syncthreads();
    float Lt = 0.f;
    for (int q = 0; q < nparts; ++q) Lt = fmaf(s_w[q], s_l[q], Lt);
    for (int d = threadIdx.x; d < kHeadDim; d += WARPS * 32) {
        float O = 0.f;
#pragma unroll 8
        for (int q = 0; q < nparts; ++q) O = fmaf(s_w[q], __ldcg(a.ws_o + (base + q) * kHeadDim + d), O);
        a.out[rh * kHeadDim + d] = __float2half_rn(O / Lt);
    }
    if (threadIdx.x == 0) a.counters[rh] = 0u;
}

int decode_max_parts(int max_blocks, int partition_tokens)
{
    const int64_t max_tokens = (int64_t)max_blocks * kBlockSize;
    return (int)((max_tokens + partition_tokens - 1) / partition_tokens);
}

namespace {
struct WsLayout {
    size_t o_bytes, ml_off, ctr_off, total;
};

WsLayout ws_layout(int num_seqs, int num_q_heads, int64_t parts)
{
    const int64_t slots = (int64_t)num_seqs * num_q_heads * parts;
    WsLayout w;
    w.o_bytes = ((size_t)slots * kHeadDim * sizeof(float) + 255) & ~(size_t)255;
    w.ml_off = w.o_bytes;
    w.ctr_off = (w.ml_off + (size_t)slots * 2 * sizeof(float) + 255) & ~(size_t)255;
    w.total = w.ctr_off + (((size_t)num_seqs * num_q_heads * sizeof(unsigned int) + 255) & ~(size_t)255);
    return w;
}
}  // namespace

size_t decode_workspace_bytes(int num_seqs, int num_q_heads, int max_blocks, int partition_tokens, int extra_parts)
{
    const int parts = decode_max_parts(max_blocks, partition_tokens) + extra_parts;
    if (parts <= 1) return 256;
    return ws_layout(num_seqs, num_q_heads, parts).total;
}

DecodeWs decode_ws(const PoolGeom& g, void* ws, int num_seqs, int max_blocks, int partition_tokens, int extra_parts)
{
    const int parts = decode_max_parts(max_blocks, partition_tokens) + extra_parts;
    DecodeWs d{nullptr, nullptr, nullptr, parts};
    if (parts <= 1) return d;
    const WsLayout w = ws_layout(num_seqs, g.num_q_heads, parts);
    d.o = static_cast<float*>(ws);
    d.ml = reinterpret_cast<float*>(static_cast<char*>(ws) + w.ml_off);
    d.counters = reinterpret_cast<unsigned int*>(static_cast<char*>(ws) + w.ctr_off);
    return d;
}

cudaError_t clear_decode_counters(const PoolGeom& g, int num_seqs, int max_blocks, int partition_tokens, void* ws,
                                  cudaStream_t stream, int extra_parts)
{
    const int parts = decode_max_parts(max_blocks, partition_tokens) + extra_parts;
    if (num_seqs == 0 || parts <= 1) return cudaSuccess;
    const WsLayout w = ws_layout(num_seqs, g.num_q_heads, parts);
    return cudaMemsetAsync(static_cast<char*>(ws) + w.ctr_off, 0,
                           (size_t)num_seqs * g.num_q_heads * sizeof(unsigned int), stream);
}

cudaError_t launch_decode(const PoolGeom& g, int layer, const void* q, const int32_t* tables, int max_blocks,
                          const int32_t* ctx_lens, int num_seqs, float scale, void* out, const DecodeWs& w,
                          int partition_tokens, const void* k_new, const void* v_new, const int64_t* slots,
                          unsigned int* status, cudaStream_t stream, const int32_t* group_start,
                          const int32_t* group_blocks, int num_groups, int pdl)
{
    if (num_seqs == 0) return cudaSuccess;
    // Cascade decode's private keys are a few hundred per row: CTAs of two warps (half the shared memory, so
    // twice as many resident per SM) overlap more of their start-up with each other's streaming.
    // (A warp's lanes hold its block ids, at most 32: two warps cover partitions of up to 1,024 keys.)
    const bool cascade = num_groups > 0 && partition_tokens <= 32 * kCascadeWarps * kBlockSize;
    using Lay = DecodeLayout<kDecodeWarps, kDecodeStages>;
    using LayC = DecodeLayout<kCascadeWarps, kDecodeStages>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 64 && !attr_set[dev]) {
        cudaError_t e = cudaFuncSetAttribute(decode_kernel<kDecodeWarps, kDecodeStages>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kBytes);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(decode_kernel<kCascadeWarps, kDecodeStages>,
                                     cudaFuncAttributeMaxDynamicSharedMemorySize, LayC::kBytes);
        if (e != cudaSuccess) return e;
        attr_set[dev] = true;
    }
    DecodeArgs a;
    a.pool = const_cast<char*>(g.base);
    a.block_bytes = g.block_bytes;
    a.head_off = (int64_t)layer * g.layer_bytes;
    a.kv_bytes = g.kv_bytes;
    a.num_blocks = g.num_blocks;
    a.num_heads = g.num_heads;
    a.q = static_cast<const __half*>(q);
    a.tables = tables;
    a.max_blocks = max_blocks;
    a.ctx_lens = ctx_lens;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.out = static_cast<__half*>(out);
    a.max_parts = decode_max_parts(max_blocks, partition_tokens);
    a.part_tokens = partition_tokens;
    a.k_new = static_cast<const __half*>(k_new);
    a.v_new = static_cast<const __half*>(v_new);
    a.slots = slots;
    a.append = k_new != nullptr;
    a.no_wait = pdl == 2;
    a.status = status;
    a.group_start = num_groups > 0 ? group_start : nullptr;
    a.group_blocks = group_blocks;
    a.num_groups = num_groups;
    a.ws_parts = w.parts;
    a.ws_o = w.o;
    a.ws_ml = w.ml;
    a.counters = w.counters;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(a.max_parts, g.num_heads, num_seqs);
    cfg.blockDim = dim3((cascade ? kCascadeWarps : kDecodeWarps) * 32);
    cfg.dynamicSmemBytes = cascade ? LayC::kBytes : Lay::kBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cascade ? cudaLaunchKernelEx(&cfg, decode_kernel<kCascadeWarps, kDecodeStages>, a)
                   : cudaLaunchKernelEx(&cfg, decode_kernel<kDecodeWarps, kDecodeStages>, a);
}

// ======================================================================
// Bounded-wait probe: one thread waits on an mbarrier that nothing arrives
// at, gives up after timeout_ns and records PKV_DEV_TIMEOUT.

__global__ void wait_probe_kernel(uint64_t timeout_ns, unsigned int* status)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x == 0) {
        const uint32_t b = smem_u32(&bar);
        mbar_init(b, 1);
        fence_mbar_init();
        if (!mbar_wait(b, 0, timeout_ns)) atomicOr(status, PKV_DEV_TIMEOUT);
    }
}

cudaError_t launch_wait_probe(uint64_t timeout_ns, unsigned int* status, cudaStream_t stream)
{
    wait_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns, status);
    return cudaGetLastError();
}

}  // namespace pkv
