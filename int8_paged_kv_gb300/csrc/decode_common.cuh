// Shared machinery of the decode kernels (one copy per translation unit):
// the launch parameters, the work split and block-table walk, the bulk-copy
// chunk ring, the CTA merge of warp states and the split-context combine.
// The kernel families live in decode.cu (tensor-core and CUDA-core tiles,
// the prep kernel and the plan), decode_umma.cu (tcgen05), decode_f32.cu
// (the f32 cache) and decode_cq.cu (the contiguous q8 cache).
#pragma once

#include <algorithm>
#include <cfloat>
#include <climits>
#include <cstdint>
#include <cstring>
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "device_util.cuh"
#include "kernels.h"

namespace pa_q8 {

struct Params {
    float *out;
    const float *q;
    const uint32_t *kc;
    const uint32_t *vc;
    const uint32_t *bt;
    const uint32_t *cl;
    int S, H, Hk, B, Nb;
    int log2B;              // block_size is a power of two
    int log2ptok;           // piece = min(block_size, 32) tokens
    int64_t num_blocks;
    float scale_log2;       // scale * log2(e)
    int PT;                 // most tokens a partition holds
    int NP;                 // most partitions a sequence is split into (grid x)
    int r;                  // num_heads / num_kv_heads
    int R;                  // query rows per sequence (1 = single-query decode)
    int rv;                 // R * r: (row, head) "virtual heads" per kv head
    int heads_per_cta;
    int head_groups;
    const unsigned long long *order;  // [S]: (clamped length << 32 | sequence) of grid z,
                                      // longest context first
    uint32_t *counters;     // [S][gridDim.y]: partitions of the group finished so far;
                            // nullptr: a combine grid of its own merges the partials
    int rec_slots;          // partial records per (row, partition): 1 (the CTA's merged
                            // state), or the token-slot warps' own (combine grid only)
    float *part;            // [S][R][H][NP][rec_slots][D + 4]: A, then m, l (and two spare words)
    uint32_t *status;
    // fused append of the newest R tokens (nk == nullptr: none)
    const float *nk;
    const float *nv;
    int64_t nk_stride, nv_stride;
    uint32_t *kc_w;         // the caches, written by the append
    uint32_t *vc_w;
    int contiguous;         // contiguous q8 cache (decode_cq_kernel)
    int per_sm;             // CTAs per SM the plan sized its waves for (the contiguous
                            // head-size-128 kernel is built for 2 and for 3)
};

// Launchers of the families in their own translation units (head sizes
// 64 / 128 / 256 as they support; anything else is cudaErrorInvalidValue).
cudaError_t launch_umma_family(const Params &P, int head_size, cudaStream_t st);
cudaError_t launch_f32_family(const Params &P, int head_size, cudaStream_t st);
cudaError_t launch_cq_family(const Params &P, int head_size, cudaStream_t st);

namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kChunk = 32;                 // tokens per warp chunk
constexpr int kLazy = 8;                   // rescale only when a logit passes the reference max by 2^8
constexpr int kVScaleBias = 131;           // weights carry 2^(131 - E): p * vs * 2^(131-E) < 2^13

// (row, head) pairs one tcgen05 CTA serves
constexpr int kUmmaHeads = 64;
// The automatic plan takes tcgen05 from this many (row, head) pairs per kv
// head on (measured: 24 pairs at head size 128 tcgen05 0.54 against mma.sync
// 0.69 ms on the 256-sequence batch, level on 8 long contexts; 16 pairs
// mma.sync 0.39 against 0.53 ms); at head size 256 above 32 (32 MQA rows:
// 44.7 against 46.4 us).
__host__ __device__ constexpr int umma_auto_pairs(int head_size) { return head_size == 256 ? 33 : 24; }

#ifndef PA_Q8_TC_SLOTS
#define PA_Q8_TC_SLOTS 4                   // token-slot warps per head tile
#endif
#ifndef PA_Q8_TC_RING_64
#define PA_Q8_TC_RING_64 3                 // chunk buffers per slot, head size 64
#endif
#ifndef PA_Q8_TC_RING_128
#define PA_Q8_TC_RING_128 2
#endif
#ifndef PA_Q8_TC_RING_256
#define PA_Q8_TC_RING_256 2
#endif
// Head size 256, one-tile (8-head) tensor-core CTAs: CTAs per SM the
// register budget targets (shared memory holds one at ring depth 2)
#ifndef PA_Q8_TC_MINB_256
#define PA_Q8_TC_MINB_256 1
#endif
// Virtual heads per one-tile tensor-core CTA (decode_tc_kernel) at head
// sizes 64 / 128.  Several such CTAs per kv head each read the K/V (the
// second read mostly from L2) and convert its codes again.
#ifndef PA_Q8_TC_MAX_HEADS
#define PA_Q8_TC_MAX_HEADS 8
#endif
// More than 8 pairs per kv head at head sizes 64 / 128 may instead take the
// two-tile kernel (decode_tc2_kernel: 16 heads per CTA, one conversion for
// both tiles); 0 keeps every group on one-tile CTAs
#ifndef PA_Q8_TC_WIDE
#define PA_Q8_TC_WIDE 1
#endif
#ifndef PA_Q8_TC_MINB_128
#define PA_Q8_TC_MINB_128 3                // CTAs per SM the register budget targets
#endif


// Which CTA this is and the token range it owns.  The CTA serves virtual
// heads h0 .. h0 + nh - 1 of kv head g: virtual head vh is query row
// b = vh / r, head g * r + vh % r of that row.
struct Work {
    int s, g, h0, nh, p;
    int c;          // clamped context length
    int t_begin;    // first logical token of the partition
    int len;        // tokens in the partition
    int np;         // partitions of this sequence
    bool single;    // the partition is the whole context
};

// Which (sequence, partition, kv head group) this CTA serves.  A context of
// c tokens is cut into np = ceil(c / PT) partitions of PT tokens, the last
// one taking the rest: each sequence gets its own partition count from its
// own length (as the split-T decode of "attention.rs", attention_b, sizes each
// row's workgroups from its visible length), so only contexts longer than PT
// are split.  CTAs with p >= np have nothing to stream and return false; so
// does partition 0 of an empty context, whose rows write_zero_rows writes.
__device__ __forceinline__ bool setup_work(const Params &P, Work &w) {
    // a split grid merged by a separate combine grid lets that grid launch
    // now; its CTAs then wait (griddepcontrol.wait) for this one to finish
    grid_dependents_launch();
    w.p = blockIdx.x;
    w.g = blockIdx.y / P.head_groups;
    const int hg = blockIdx.y % P.head_groups;
    w.h0 = hg * P.heads_per_cta;
    w.nh = min(P.heads_per_cta, P.rv - w.h0);
    const int64_t cap = (int64_t)P.Nb * P.B;
    if (P.order) {
        // written by the prep kernel that precedes this grid on the stream
        grid_dependency_wait();
        const unsigned long long e = __ldcg(P.order + blockIdx.z);
        w.s = (int)(e & 0xFFFFFFFFull);
        w.c = (int)(e >> 32);
    } else {
        w.s = (int)blockIdx.z;
        const int64_t craw = __ldg(P.cl + w.s);
        w.c = (int)(craw < cap ? craw : cap);
    }
    w.np = max(1, (w.c + P.PT - 1) / P.PT);
    w.t_begin = w.p * P.PT;
    w.len = min(w.c - w.t_begin, P.PT);
    w.single = w.np == 1;
    return w.len > 0;
}

// Row of q / out (in units of head_size) of virtual head vh of the CTA's
// group: sequence s, query row vh / r, head g * r + vh % r.
__device__ __forceinline__ int64_t qrow(const Params &P, const Work &w, int vh) {
    if (P.R == 1) return (int64_t)w.s * P.H + (int64_t)w.g * P.r + vh;      // single query: no division
    const int b = vh / P.r;
    return ((int64_t)w.s * P.R + b) * P.H + (int64_t)w.g * P.r + (vh - b * P.r);
}

// Tokens of this partition virtual head vh attends to: query row b sees the
// first c - (R - 1 - b) tokens of the context ("attention.rs", attention_b:
// t_len = base_pos + b + 1).
__device__ __forceinline__ int row_len(const Params &P, const Work &w, int vh) {
    const int cb = P.R == 1 ? w.c : w.c - (P.R - 1 - vh / P.r);
    return max(0, min(cb - w.t_begin, w.len));
}

// Fused append: quantise the sequence's newest R tokens (positions c-R ..
// c-1 of the clamped context; row b of the new K/V rows is position c-R+b)
// that fall in this CTA's partition, for its kv head, and store their K and V
// token vectors in the cache -- the writer's arithmetic, one warp per vector.
// Every CTA whose tiles hold such a token stores it, all with the same bits,
// so a tile copy observes the token's words whichever store it sees; the
// caller's CTA barrier (after the proxy fence here) orders the stores before
// this CTA's bulk copies.
template <int D>
__device__ void append_tokens(const Params &P, const Work &w) {
    constexpr int WORDS = D / 4;
    constexpr int NW = (WORDS + 31) / 32;          // words per lane (head size 64: lanes 0..15)
    const int first = w.c - P.R;                    // position of new row 0 (may be < 0)
    const int t_lo = max(first, w.t_begin), t_hi = min(w.c, w.t_begin + w.len);
    const int nvec = 2 * max(0, t_hi - t_lo);       // (token, K or V) vectors
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int v = warp; v < nvec; v += (int)(blockDim.x >> 5)) {
        const int t = t_lo + (v >> 1);
        const bool is_v = v & 1;
        const int64_t row = (int64_t)w.s * P.R + (t - first);
        const float4 *src = reinterpret_cast<const float4 *>(
            (is_v ? P.nv + row * P.nv_stride : P.nk + row * P.nk_stride) + (int64_t)w.g * D);
        float4 x[NW];
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const int wd = lane + 32 * i;
            x[i] = wd < WORDS ? __ldg(src + wd) : make_float4(0.f, 0.f, 0.f, 0.f);
            m = fmaxf(m, fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)), fmaxf(fabsf(x[i].z), fabsf(x[i].w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float inv = m > 0.0f ? __fdiv_rn(127.0f, m) : 0.0f;
        const float scale = m > 0.0f ? __fdiv_rn(m, 127.0f) : 1.0f;
        const uint32_t pb = __ldg(P.bt + (int64_t)w.s * P.Nb + (t >> P.log2B));
        if ((int64_t)pb >= P.num_blocks) {         // warp-uniform; the table walk flags it
            continue;
        }
        uint32_t *dst = (is_v ? P.vc_w : P.kc_w) +
                        (((int64_t)pb * P.Hk + w.g) * P.B + (t & (P.B - 1))) * (WORDS + 1);
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            const int wd = lane + 32 * i;
            if (wd < WORDS) dst[wd] = pack_word(x[i], inv);
        }
        if (lane == 0) dst[WORDS] = __float_as_uint(scale);
    }
    fence_proxy_async_global();
}

// Zero output rows of a sequence whose context is empty (partition 0 only).
template <int D>
__device__ void write_zero_rows(const Params &P, const Work &w) {
    if (w.p != 0 || w.c != 0) return;
    for (int i = threadIdx.x; i < w.nh * D; i += blockDim.x) {
        const int hh = i / D, d = i % D;
        P.out[qrow(P, w, w.h0 + hh) * D + d] = 0.0f;
    }
}

__host__ __device__ constexpr uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

// Bytes of the CTA merge's scratch (merge_and_store): per-slot (m, l, E)
// and accumulators of every head, then the per-head factors.  The kernels
// carve it out of their chunk ring once the streams are drained, so it must
// fit there (checked at compile time per kernel).
__host__ __device__ constexpr uint32_t merge_scratch_bytes(int D, int slots, int heads) {
    return (uint32_t)(slots * heads * (3 + D) + heads * (slots + 2)) * 4u;
}
__host__ __device__ constexpr uint32_t ring_bytes(int D, int streams, int ring) {
    return (uint32_t)streams * ring * ((2u * kChunk * (D / 4 + 1) * 4 + 127) / 128 * 128);
}

// Shared-memory layout (bytes from the dynamic base).
struct Layout {
    uint32_t bars;        // [streams][ring] full barriers
    uint32_t table;       // physical block of each piece of the partition
    uint32_t extra;       // kernel-specific (q fragments, or q and weights)
    uint32_t ring;        // [streams][ring] chunk buffers
    uint32_t slot_bytes;  // one chunk: K rows [32][W] then V rows [32][W]
    uint32_t total;
};

__host__ __device__ inline Layout make_layout(int D, int streams, int ring, int PT, int B,
                                              uint32_t extra_bytes) {
    Layout L{};
    const int W = D / 4 + 1;
    const int ptok = B < kChunk ? B : kChunk;
    const int pieces = (PT + ptok - 1) / ptok + 1;
    L.bars = 0;
    L.table = align_up(streams * ring * 8, 16);
    L.extra = align_up(L.table + pieces * 4, 128);
    L.ring = align_up(L.extra + extra_bytes, 128);
    L.slot_bytes = align_up(2u * kChunk * W * 4, 128);
    L.total = L.ring + streams * ring * L.slot_bytes;
    return L;
}

// Load the partition's block-table slice (one entry per piece of
// min(B, 32) tokens); entries out of range become kPadSlot and are flagged.
// Four entries per thread are loaded before any is stored, so a long
// partition's table costs one memory round trip, not one per pass.
__device__ void load_table(const Params &P, const Work &w, uint32_t *table) {
    constexpr int U = 4;
    const int n = (w.len + (1 << P.log2ptok) - 1) >> P.log2ptok;
    const uint32_t *row = P.bt + (int64_t)w.s * P.Nb;
    for (int i0 = threadIdx.x; i0 < n; i0 += U * blockDim.x) {
        uint32_t pb[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * (int)blockDim.x;
            pb[u] = i < n ? __ldg(row + ((w.t_begin + (i << P.log2ptok)) >> P.log2B)) : 0u;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * (int)blockDim.x;
            if (i < n) {
                if ((int64_t)pb[u] >= P.num_blocks) {
                    flag_error(P.status, kDevBadBlock);
                    pb[u] = kPadSlot;
                }
                table[i] = pb[u];
            }
        }
    }
}

// Copy chunk c of the partition (32 tokens; pieces of min(B, 32) tokens,
// each a contiguous run of one (block, kv head) tile) into the chunk buffer
// at `slot`, completing on `bar`.  Whole warp; lane i copies piece i.
template <int D>
__device__ __forceinline__ void issue_chunk(const Params &P, const Work &w, const uint32_t *table,
                                            int c, uint32_t slot, uint32_t bar, uint64_t policy) {
    constexpr int W = D / 4 + 1;
    const int lane = threadIdx.x & 31;
    const int t = c * kChunk + (lane << P.log2ptok);   // partition-relative token
    uint32_t bytes = 0;
    int64_t base = 0;
    if (lane < (kChunk >> P.log2ptok) && t < w.len) {
        const uint32_t pb = table[t >> P.log2ptok];
        if (pb != kPadSlot) {
            const int off = (w.t_begin + t) & (P.B - 1);
            base = (((int64_t)pb * P.Hk + w.g) << P.log2B) * W + (int64_t)off * W;
            bytes = (uint32_t)W * 4 << P.log2ptok;
        }
    }
    const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes) * 2u;
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (bytes) {
        fence_proxy_async_smem();
        const uint32_t dst = slot + (((uint32_t)lane * W * 4) << P.log2ptok);
        bulk_copy_g2s(dst, P.kc + base, bytes, bar, policy);
        bulk_copy_g2s(dst + kChunk * W * 4, P.vc + base, bytes, bar, policy);
    }
}

// Wait (bounded) for chunk buffers still being filled before a warp leaves.
__device__ void drain(const Params &P, uint32_t bars, int ring, int consumed, int issued) {
    if ((threadIdx.x & 31) != 0) return;
    for (int i = consumed; i < issued; ++i) {
        if (!mbar_wait(bars + 8 * (i % ring), (i / ring) & 1)) {
            flag_error(P.status, kDevWaitTimeout);
            return;
        }
    }
}

// ----------------------------------------------------------------- epilogue
//
// Merge the per-warp online-softmax states of the CTA (m in log2 units, l,
// acc scaled by 2^(E - 139)) and write the output rows, or this
// partition's partial (M, L, A) for the combine.
//
// Log-sum-exp merge of all np partitions of this CTA's heads (run by the
// last CTA of a (sequence, head group) to finish):
// out = sum_p A_p 2^(M_p - M*) / sum_p L_p 2^(M_p - M*), M* = max M_p.
// A head's np partial records (A_p, M_p, L_p; D + 4 floats each) are
// contiguous in the workspace and were written by other CTAs (or this one).
// `scratch` is the start of shared memory this CTA no longer needs, up to the
// end of its dynamic allocation.  As many heads' records as fit come in with
// one bulk copy per head, so a batch of heads costs one memory round trip;
// the weights 2^(M_p - M*) then go into each record's spare word.  A head
// whose records alone do not fit is read with vector loads instead.
template <int D>
__device__ __forceinline__ void combine_rows(const Params &P, const Work &w, int np, uint8_t *scratch) {
    constexpr int DP = D + 4;            // floats per partial record
    constexpr int D4 = D / 4;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    const int nh = w.nh;
    extern __shared__ __align__(16) uint8_t combine_dsm[];
    uint32_t dyn;
    asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    const uintptr_t end = reinterpret_cast<uintptr_t>(combine_dsm) + dyn;
    const uintptr_t base = (reinterpret_cast<uintptr_t>(scratch) + 15) & ~(uintptr_t)15;
    float *iL = reinterpret_cast<float *>(base + 16);                  // after the barrier: [nh] 1/L
    const uintptr_t buf = (reinterpret_cast<uintptr_t>(iL + nh) + 127) & ~(uintptr_t)127;
    const size_t head_bytes = (size_t)np * DP * 4;
    const size_t fit = buf + head_bytes <= end ? (end - buf) / head_bytes : 0;
    const int hb = fit < (size_t)nh ? (int)fit : nh;                   // heads per batch
    auto record = [&](int h) { return P.part + qrow(P, w, w.h0 + h) * P.NP * DP; };

    if (hb > 0) {
        const uint32_t bar = smem_addr(reinterpret_cast<void *>(base));
        const uint64_t policy = l2_policy_evict_first();
        if (threadIdx.x == 0) {
            mbar_init(bar, 1);
            fence_mbar_init();
        }
        __syncthreads();
        float *rows = reinterpret_cast<float *>(buf);                  // [hb][np][DP]
        for (int h0 = 0, ph = 0; h0 < nh; h0 += hb, ph ^= 1) {
            const int n = min(hb, nh - h0);
            if (h0 > 0) __syncthreads();                               // the previous batch is consumed
            if (warp == 0) {
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)(n * head_bytes));
                __syncwarp();
                // other CTAs' generic stores, seen through the arrival counter,
                // before this thread's bulk (async proxy) reads of them; and
                // this CTA's earlier generic use of the buffer before the
                // copies overwrite it
                fence_proxy_async_global();
                fence_proxy_async_smem();
                for (int h = lane; h < n; h += 32)
                    bulk_copy_g2s(smem_addr(rows + (size_t)h * np * DP), record(h0 + h), (uint32_t)head_bytes, bar,
                                  policy);
            }
            if (!mbar_wait(bar, (uint32_t)ph)) {
                flag_error(P.status, kDevWaitTimeout);
                return;
            }
            // M* and 1/L per head (a warp per head, lanes over partitions); each
            // partition's weight goes into its record's spare word
            for (int h = warp; h < n; h += nwarps) {
                float *rh = rows + (size_t)h * np * DP;
                float M = -INFINITY;
                for (int p = lane; p < np; p += 32) M = fmaxf(M, rh[p * DP + D]);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
                if (M == -INFINITY) M = 0.0f;       // a query row that sees no token: weights 0, row 0
                float L = 0.0f;
                for (int p = lane; p < np; p += 32) {
                    const float e = fast_exp2(rh[p * DP + D] - M);
                    L += rh[p * DP + D + 1] * e;
                    rh[p * DP + D + 2] = e;
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
                if (lane == 0) iL[h0 + h] = L > 0.0f ? 1.0f / L : 0.0f;
            }
            __syncthreads();
            // out[h][d] = (1/L) sum_p A_p[h][d] 2^(M_p - M*), summed over p in order
            for (int i = threadIdx.x; i < n * D4; i += blockDim.x) {
                const int hl = i / D4, d4 = i - hl * D4;
                const float *rh = rows + (size_t)hl * np * DP;
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
                for (int p = 0; p < np; ++p) {
                    const float4 v = reinterpret_cast<const float4 *>(rh + p * DP)[d4];
                    const float x = rh[p * DP + D + 2];
                    a.x = fmaf(v.x, x, a.x);
                    a.y = fmaf(v.y, x, a.y);
                    a.z = fmaf(v.z, x, a.z);
                    a.w = fmaf(v.w, x, a.w);
                }
                const float il = iL[h0 + hl];
                reinterpret_cast<float4 *>(P.out + qrow(P, w, w.h0 + h0 + hl) * D)[d4] =
                    make_float4(a.x * il, a.y * il, a.z * il, a.w * il);
            }
        }
        return;
    }
    // Records too large for shared memory: M* and 1/L per head from the (m, l)
    // words, then the weighted sums with eight partitions' vector loads in
    // flight per thread, each weight recomputed from its m.
    float *Ms = iL + nh;
    for (int h = warp; h < nh; h += nwarps) {
        const float *rh = record(h);
        float M = -INFINITY;
        for (int p = lane; p < np; p += 32) M = fmaxf(M, __ldcg(rh + (size_t)p * DP + D));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        if (M == -INFINITY) M = 0.0f;
        float L = 0.0f;
        for (int p = lane; p < np; p += 32) {
            const float2 ml = __ldcg(reinterpret_cast<const float2 *>(rh + (size_t)p * DP + D));
            L += ml.y * fast_exp2(ml.x - M);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
        if (lane == 0) {
            Ms[h] = M;
            iL[h] = L > 0.0f ? 1.0f / L : 0.0f;
        }
    }
    __syncthreads();
    constexpr int PU = 8;
    for (int i = threadIdx.x; i < nh * D4; i += blockDim.x) {
        const int h = i / D4, d4 = i - h * D4;
        const float *rh = record(h);
        const float M = Ms[h];
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int p0 = 0; p0 < np; p0 += PU) {
            float4 v[PU];
            float m[PU];
#pragma unroll
            for (int j = 0; j < PU; ++j) {
                const int p = min(p0 + j, np - 1);
                v[j] = __ldcg(reinterpret_cast<const float4 *>(rh + (size_t)p * DP) + d4);
                m[j] = __ldcg(rh + (size_t)p * DP + D);
            }
#pragma unroll
            for (int j = 0; j < PU; ++j) {
                if (p0 + j < np) {
                    const float x = fast_exp2(m[j] - M);
                    a.x = fmaf(v[j].x, x, a.x);
                    a.y = fmaf(v[j].y, x, a.y);
                    a.z = fmaf(v[j].z, x, a.z);
                    a.w = fmaf(v[j].w, x, a.w);
                }
            }
        }
        const float il = iL[h];
        reinterpret_cast<float4 *>(P.out + qrow(P, w, w.h0 + h) * D)[d4] =
            make_float4(a.x * il, a.y * il, a.z * il, a.w * il);
    }
}

// combine_rows as a call of its own, for kernels whose register budget is
// tight (the tcgen05 family: 96 per thread): it runs once per split sequence,
// and keeping it out of line keeps its registers out of the streaming loop's
// allocation.  The other families inline it (measured slightly faster).
template <int D>
__device__ __noinline__ void combine_rows_outlined(const Params &P, const Work &w, int np, uint8_t *scratch) {
    combine_rows<D>(P, w, np, scratch);
}

// Split context, after this CTA stored its partial records: the last CTA of
// the (sequence, head group) to arrive merges every partition (threadfence /
// counter handshake).  Called by every thread of the CTA; scratch is shared
// memory free up to the end of the dynamic allocation.
template <int D, bool kOutlineCombine = false>
__device__ void arrive_and_combine(const Params &P, const Work &w, uint8_t *scratch) {
    if (P.counters == nullptr) return;       // merged by the combine grid that follows
    __threadfence();
    __syncthreads();
    const int np = w.np;
    int *last = reinterpret_cast<int *>(scratch);
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(P.counters + (int64_t)w.s * gridDim.y + blockIdx.y, 1u);
        *last = (prev == (uint32_t)(np - 1));
    }
    __syncthreads();
    const bool is_last = *last != 0;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    if constexpr (kOutlineCombine) combine_rows_outlined<D>(P, w, np, scratch);
    else combine_rows<D>(P, w, np, scratch);
}

template <int D, bool kOutlineCombine = false>
__device__ void merge_and_store(const Params &P, const Work &w, const float *ml, const float *accs,
                                int n_slots, int heads_stride, float *fac) {
    // ml: [slot][head][3] = (m, l, E); accs: [slot][head][D]; fac: scratch
    // [head][n_slots + 2] = per-slot factors, M, L, then room for the
    // combine's weights.  Called by every thread of the CTA.
    for (int hh = threadIdx.x; hh < w.nh; hh += blockDim.x) {
        float M = -INFINITY;
        for (int sl = 0; sl < n_slots; ++sl) M = fmaxf(M, ml[(sl * heads_stride + hh) * 3]);
        float Lsum = 0.0f;
        float *f = fac + hh * (n_slots + 2);
        for (int sl = 0; sl < n_slots; ++sl) {
            const float *e = ml + (sl * heads_stride + hh) * 3;
            float x = 0.0f;
            if (e[0] != -INFINITY) {
                const float wgt = fast_exp2(e[0] - M);
                Lsum += e[1] * wgt;
                x = wgt * ldexpf(1.0f, __float2int_rn(e[2]) - kVScaleBias);
            }
            f[sl] = x;
        }
        f[n_slots] = M;
        f[n_slots + 1] = Lsum;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < w.nh * D; i += blockDim.x) {
        const int hh = i / D, d = i % D;
        const float *f = fac + hh * (n_slots + 2);
        float A = 0.0f;
        for (int sl = 0; sl < n_slots; ++sl) A = fmaf(accs[(sl * heads_stride + hh) * D + d], f[sl], A);
        const int64_t qr = qrow(P, w, w.h0 + hh);
        if (w.single) {
            // a query row that sees no token (L = 0) gets a zero row
            P.out[qr * D + d] = f[n_slots + 1] > 0.0f ? A / f[n_slots + 1] : 0.0f;
        } else {
            float *rec = P.part + (qr * P.NP + w.p) * (D + 4);
            rec[d] = A;
            if (d == 0) {
                rec[D] = f[n_slots];
                rec[D + 1] = f[n_slots + 1];
            }
        }
    }
    if (w.single) return;
    // the merge's own scratch (ml, accs) is no longer needed
    arrive_and_combine<D, kOutlineCombine>(P, w, reinterpret_cast<uint8_t *>(const_cast<float *>(ml)));
}

// The attention grid is launched as a programmatic dependent of the prep
// kernel before it on the stream: its launch overlaps the prep kernel, and
// each CTA waits (griddepcontrol.wait) before it reads the prep's output.
template <typename K, typename A>
cudaError_t launch_attn_arg(K kernel, const Params &P, const A &arg, uint32_t smem_bytes, int threads,
                            cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(P.NP, P.Hk * P.head_groups, P.S);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem_bytes;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = P.order ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kernel, arg);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename K>
cudaError_t launch_attn(K kernel, const Params &P, uint32_t smem_bytes, int threads, cudaStream_t st) {
    return launch_attn_arg(kernel, P, P, smem_bytes, threads, st);
}

}  // namespace
}  // namespace pa_q8
