// Paged-attention decode over the int8 KV cache, and the log-sum-exp merge
// of split-context partials.
//
// What is computed ("paged_attn_q8.comp", hanzo-ml 0.11.92, header comment
// and main()): for each sequence s and query head h, with kv head
// g = h / (num_heads / num_kv_heads) and c = min(context_len, max_blocks *
// block_size), out[s,h] = sum_t softmax_t(scale * q . k_t) v_t, where k_t and
// v_t are the codes of logical token t (block block_tables[s][t / B], offset
// t % B) times that token's scale.  The context may be split into
// partitions whose (max, sum, weighted sum) partials are merged by their
// log-sum-exp, as the split-T decode and attn_combine dispatches of
// "attention.rs" (attention_b) do.
//
// GB300 design (not the pages'): one CTA per (sequence, kv head,
// partition) serves every query head of the GQA group from one read of the
// group's K/V.  The partition is cut into 32-token chunks dealt round-robin
// to the CTA's token-slot warps.  Every slot owns a small ring of shared-
// memory chunk buffers: it copies its next chunks' K and V rows -- runs of
// (block, kv head) tiles, block_size * (head_size + 4) contiguous bytes --
// with 1-D bulk copies (cp.async.bulk) completing on per-buffer mbarriers,
// then dequantises in registers and runs a single-pass online softmax.  No
// cross-warp handshake sits on the streaming path.  Two consumer families:
//   * tensor core: per chunk, S = Q K^T and O += P V as mma.sync m16n8k16
//     f16 tiles; q and P enter as hi + lo f16 pairs (rows 0-7 = hi, rows
//     8-15 = lo of the same 8 heads), int8 codes are exact in f16;
//   * CUDA core: f32 FMA dot products (lane = token) and weighted sums
//     (lane = 4 head dims).
// Every wait is bounded; a wait that gives up flags the status word, and a
// warp leaves only after the copies it issued have landed.
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
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kChunk = 32;                 // tokens per warp chunk
constexpr int kLazy = 8;                   // rescale only when a logit passes the reference max by 2^8
constexpr int kVScaleBias = 131;           // weights carry 2^(131 - E): p * vs * 2^(131-E) < 2^13

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
// Virtual heads per tensor-core CTA for head sizes 64 / 128.  Each head tile
// converts the chunk's codes itself, so a 16-head CTA does twice the work of
// an 8-head one on one CTA per SM; two 8-head CTAs (three per SM) finish
// sooner, their second K/V read mostly served by L2.
#ifndef PA_Q8_TC_MAX_HEADS
#define PA_Q8_TC_MAX_HEADS 8
#endif
#ifndef PA_Q8_TC_MINB_128
#define PA_Q8_TC_MINB_128 3                // CTAs per SM the register budget targets
#endif

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
    int PT;                 // tokens per partition
    int NP;                 // partitions per sequence (grid x)
    int r;                  // num_heads / num_kv_heads
    int R;                  // query rows per sequence (1 = single-query decode)
    int rv;                 // R * r: (row, head) "virtual heads" per kv head
    int heads_per_cta;
    int head_groups;
    const unsigned long long *order;  // [S]: (clamped length << 32 | sequence) of grid z,
                                      // longest context first
    uint32_t *counters;     // [S][gridDim.y]: partitions of the group finished so far
    float *pml;             // [S][R][H][NP][2]
    float *pacc;            // [S][R][H][NP][D]
    uint32_t *status;
    // fused append of the newest R tokens (nk == nullptr: none)
    const float *nk;
    const float *nv;
    int64_t nk_stride, nv_stride;
    uint32_t *kc_w;         // the caches, written by the append
    uint32_t *vc_w;
    int contiguous;         // contiguous q8 cache (decode_cq_kernel)
};

// Which CTA this is and the token range it owns.  The CTA serves virtual
// heads h0 .. h0 + nh - 1 of kv head g: virtual head vh is query row
// b = vh / r, head g * r + vh % r of that row.
struct Work {
    int s, g, h0, nh, p;
    int c;          // clamped context length
    int t_begin;    // first logical token of the partition
    int len;        // tokens in the partition
    bool single;    // the partition is the whole context
};

__device__ __forceinline__ bool setup_work(const Params &P, Work &w) {
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
    w.t_begin = w.p * P.PT;
    w.len = min(w.c - w.t_begin, P.PT);
    w.single = w.c <= P.PT;
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
    return max(0, min(cb - w.t_begin, P.PT));
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
    const int t_lo = max(first, w.t_begin), t_hi = min(w.c, w.t_begin + P.PT);
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
// partition's partial (M, L, A) for the combine kernel.
// Log-sum-exp merge of all np partitions of this CTA's heads (run by the
// last CTA of a (sequence, head group) to finish):
// out = sum_p A_p 2^(M_p - M*) / sum_p L_p 2^(M_p - M*), M* = max M_p.
// The partials of other CTAs are read through L2 (__ldcg).  scratch holds
// (M*, 1/L) per head.
template <int D>
__device__ void combine_rows(const Params &P, const Work &w, int np, float *scratch) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = blockDim.x >> 5;
    for (int hh = warp; hh < w.nh; hh += nwarps) {
        const int64_t row0 = qrow(P, w, w.h0 + hh) * P.NP;
        // up to 32 partitions: each lane's (m, l) is read once
        const float2 ml0 = lane < np ? __ldcg(reinterpret_cast<const float2 *>(P.pml + (row0 + lane) * 2))
                                     : make_float2(-INFINITY, 0.0f);
        float M = ml0.x;
        for (int p = lane + 32; p < np; p += 32) M = fmaxf(M, __ldcg(P.pml + (row0 + p) * 2));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        if (M == -INFINITY) M = 0.0f;       // a query row that sees no token: weights 0, row 0
        float L = lane < np ? ml0.y * fast_exp2(ml0.x - M) : 0.0f;
        for (int p = lane + 32; p < np; p += 32)
            L += __ldcg(P.pml + (row0 + p) * 2 + 1) * fast_exp2(__ldcg(P.pml + (row0 + p) * 2) - M);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);
        if (lane == 0) {
            scratch[2 * hh] = M;
            scratch[2 * hh + 1] = L > 0.0f ? 1.0f / L : 0.0f;
        }
    }
    __syncthreads();
    // four output elements per thread at a time, eight partitions deep, so
    // their loads overlap; the sum still runs over p in order
    constexpr int U = 4, PU = 8;
    const int n_out = w.nh * D;
    for (int i0 = threadIdx.x; i0 < n_out; i0 += U * blockDim.x) {
        float a[U], M[U];
        int64_t prow[U];
        int dd[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = min(i0 + u * (int)blockDim.x, n_out - 1);
            const int hh = i / D;
            dd[u] = i % D;
            prow[u] = qrow(P, w, w.h0 + hh) * P.NP;
            M[u] = scratch[2 * hh];
            a[u] = 0.0f;
        }
        for (int p0 = 0; p0 < np; p0 += PU) {
            float v[U][PU], m[U][PU];
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int j = 0; j < PU; ++j) {
                    const int p = min(p0 + j, np - 1);
                    v[u][j] = __ldcg(P.pacc + (prow[u] + p) * D + dd[u]);
                    m[u][j] = __ldcg(P.pml + (prow[u] + p) * 2);
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
#pragma unroll
                for (int j = 0; j < PU; ++j)
                    if (p0 + j < np) a[u] = fmaf(v[u][j], fast_exp2(m[u][j] - M[u]), a[u]);
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int i = i0 + u * (int)blockDim.x;
            if (i < n_out) {
                const int hh = i / D;
                P.out[qrow(P, w, w.h0 + hh) * D + dd[u]] = a[u] * scratch[2 * hh + 1];
            }
        }
    }
}

template <int D>
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
            const int64_t row = qr * P.NP + w.p;
            P.pacc[row * D + d] = A;
            if (d == 0) {
                P.pml[row * 2] = f[n_slots];
                P.pml[row * 2 + 1] = f[n_slots + 1];
            }
        }
    }
    if (w.single) return;
    // Split context: the last CTA of this (sequence, head group) to arrive
    // merges every partition (threadfence / counter handshake).
    __threadfence();
    __syncthreads();
    const int np = (w.c + P.PT - 1) / P.PT;
    int *last = reinterpret_cast<int *>(fac);
    if (threadIdx.x == 0) {
        const uint32_t prev = atomicAdd(P.counters + (int64_t)w.s * gridDim.y + blockIdx.y, 1u);
        *last = (prev == (uint32_t)(np - 1));
    }
    __syncthreads();
    const bool is_last = *last != 0;
    __syncthreads();
    if (!is_last) return;
    __threadfence();
    combine_rows<D>(P, w, np, fac);
}

// ============================================================ tensor cores
//
// Warp (head tile ht, token slot ts) owns query heads h0 + 8 ht + (0..7) and
// chunks ts, ts + SLOTS, ...; the HT warps of one token slot share its
// chunk stream.  Fragment coordinates: gq = lane / 4, cq = lane % 4.
//
// K dimension of S = Q K^T: k-step ks uses, for lane column cq, code word
// kword(cq, ks) of a token row -- 4 consecutive head dims in one u32.  The
// A fragment (q) follows the same dimension order, so the sum is the plain
// dot product.  Rows gq and gq + 8 of A are the hi and lo f16 parts of head
// gq.
//
// N dimension of O = P V: the V words of four tokens at word vword(gq, jj)
// give, byte lane e, the B fragments of n-tile 4 jj + e; output column n of
// n-tile i is head dim 4 * vword(n, i / 4) + i % 4.  Both word maps visit
// every word once and make a warp's shared-memory reads hit 32 distinct
// banks when the token row stride (head_size/4 + 1 words) is 1 mod 32
// (head sizes 128 and 256).
template <int D>
__device__ __forceinline__ int kword(int cq, int ks) {
    if constexpr (D == 64) return 4 * cq + ks;
    else return 8 * cq + (ks & 7) + 32 * (ks >> 3);
}

template <int D>
__device__ __forceinline__ int vword(int n, int jj) {
    if constexpr (D == 64) return 4 * (n & 3) + (n >> 2) + 2 * jj;
    else return 8 * (n & 3) + (n >> 2) + 2 * (jj & 3) + 32 * (jj >> 2);
}

template <int D, int HT>
__host__ __device__ constexpr uint32_t tc_extra_bytes() {
    return D == 256 ? (uint32_t)HT * (D / 16) * 32 * 16 : 0u;
}

template <int D>
__host__ __device__ constexpr int tc_ring() { return D == 64 ? PA_Q8_TC_RING_64 : (D == 128 ? PA_Q8_TC_RING_128 : PA_Q8_TC_RING_256); }

template <int D, int HT>
__host__ __device__ constexpr int tc_min_blocks() { return (D == 256 || HT == 2) ? 1 : (D == 128 ? PA_Q8_TC_MINB_128 : 3); }

template <int D, int HT>
__global__ void __launch_bounds__(HT * PA_Q8_TC_SLOTS * 32, tc_min_blocks<D, HT>())
decode_tc_kernel(Params P) {
    constexpr int SLOTS = PA_Q8_TC_SLOTS;
    constexpr int RING = tc_ring<D>();
    constexpr int W = D / 4 + 1;
    constexpr int NKS = D / 16;          // k-steps of Q K^T
    constexpr int NT = D / 8;            // n-tiles of P V
    constexpr int NJ = D / 32;           // V words per row group
    constexpr bool kQInSmem = (D == 256);

    extern __shared__ __align__(128) uint8_t smem[];
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const Layout L = make_layout(D, SLOTS, RING, P.PT, P.B, tc_extra_bytes<D, HT>());
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ht = warp / SLOTS, ts = warp % SLOTS;
    const int gq = lane >> 2, cq = lane & 3;
    const uint32_t bars = smem_addr(smem + L.bars) + 8 * RING * ts;      // this slot's barriers
    const uint32_t ring = smem_addr(smem + L.ring) + RING * L.slot_bytes * ts;
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    const int nchunks = (w.len + kChunk - 1) / kChunk;
    const int my_n = ts < nchunks ? (nchunks - ts + SLOTS - 1) / SLOTS : 0;
    const uint64_t policy = l2_policy_evict_first();

    if (ht == 0 && lane == 0) {
        for (int k = 0; k < RING; ++k) mbar_init(bars + 8 * k, 1);
        fence_mbar_init();
    }
    const int nh_tile = max(0, min(8, w.nh - 8 * ht));
    const bool row_ok = gq < nh_tile;
    const int vh = w.h0 + 8 * ht + gq;                      // this thread's virtual head
    // q is loaded before the block table so the two round trips overlap
    // (head size 256 reads q below, into shared memory)
    float4 qraw[kQInSmem ? 1 : NKS];
    if constexpr (!kQInSmem) {
        const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok ? vh : w.h0) * D);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks)
            qraw[ks] = row_ok ? __ldg(qv + kword<D>(cq, ks)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }

    if (P.nk) append_tokens<D>(P, w);
    load_table(P, w, const_cast<uint32_t *>(table));
    __syncthreads();

    int issued = 0;
    if (ht == 0) {
        for (; issued < RING && issued < my_n; ++issued)
            issue_chunk<D>(P, w, table, ts + SLOTS * issued, ring + issued * L.slot_bytes,
                           bars + 8 * issued, policy);
    }
    // tokens this row sees in the partition (query row b sees c - (R-1-b));
    // chunks below the warp's smallest length need no masking
    const int len_row = row_ok ? row_len(P, w, vh) : w.len;
    const int len_min = __reduce_min_sync(0xFFFFFFFFu, (unsigned)len_row);

    // q of head gq scaled by 2^-eq into [1, 2) in magnitude, as hi/lo f16
    // pairs.  Head size 256 keeps these fragments in shared memory.
    uint32_t aq[kQInSmem ? 1 : NKS][4];
    uint4 *qf = reinterpret_cast<uint4 *>(smem + L.extra);           // [HT][NKS][32]
    float qk2;
    {
        const float4 *qv = reinterpret_cast<const float4 *>(
            P.q + qrow(P, w, row_ok ? vh : w.h0) * D);
        auto qload = [&](int ks) -> float4 {
            if constexpr (kQInSmem) return row_ok ? __ldg(qv + kword<D>(cq, ks)) : make_float4(0.f, 0.f, 0.f, 0.f);
            else return qraw[ks];
        };
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = qload(ks);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);      // 2^-eq
        qk2 = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = qload(ks);
            uint32_t f0, f1, f2, f3;
            split_f16x2(v.x * down, v.y * down, f0, f1);
            split_f16x2(v.z * down, v.w * down, f2, f3);
            if constexpr (kQInSmem) {
                if (ts == 0) qf[(ht * NKS + ks) * 32 + lane] = make_uint4(f0, f1, f2, f3);
            } else {
                aq[ks][0] = f0; aq[ks][1] = f1; aq[ks][2] = f2; aq[ks][3] = f3;
            }
        }
        if constexpr (kQInSmem) __syncthreads();
    }

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    float m = -INFINITY, lsum = 0.0f;
    int E = 12;                       // running max biased exponent of V scales (>= 12)
    float wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);

    const F16Consts fk;
    bool ok = true;
    int i = 0;
    for (; i < my_n; ++i) {
        const int k = i % RING;
        bool got = mbar_wait(bars + 8 * k, (i / RING) & 1);
        if constexpr (HT > 1) got = !named_barrier_or(1 + ts, HT * 32, !got);
        if (!got) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(smem + L.ring) +
                             (RING * ts + k) * (L.slot_bytes / 4);
        const uint32_t *sV = sK + kChunk * W;
        const int t0 = (ts + SLOTS * i) * kChunk;              // partition-relative
        const bool full = t0 + kChunk <= len_min;

        // ---- S = Q K^T for the 32 tokens (n-tile j holds tokens 8j .. 8j+7)
        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const int wd = kword<D>(cq, ks);
            uint32_t a[4];
            if constexpr (kQInSmem) {
                const uint4 f = qf[(ht * NKS + ks) * 32 + lane];
                a[0] = f.x; a[1] = f.y; a[2] = f.z; a[3] = f.w;
            } else {
                a[0] = aq[ks][0]; a[1] = aq[ks][1]; a[2] = aq[ks][2]; a[3] = aq[ks][3];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t b0, b1;
                codes4_to_f16x2(sK[(8 * j + gq) * W + wd], b0, b1, fk);
                mma_16816(s[j], a, b0, b1);
            }
        }
        // ---- online softmax over this thread's 8 tokens: 8j + 2cq + e
        float z[8], vs[8];
        float cmax = -INFINITY, vmax = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 8 * j + 2 * cq + e;
                const float kscale = __uint_as_float(sK[t * W + D / 4]);
                float zz = (s[j][e] + s[j][e + 2]) * kscale * qk2;
                float vv = __uint_as_float(sV[t * W + D / 4]);
                if (!full) {
                    const bool valid = t0 + t < len_row;
                    zz = valid ? zz : -INFINITY;
                    vv = valid ? vv : 0.0f;
                }
                z[2 * j + e] = zz;
                vs[2 * j + e] = vv;
                cmax = fmaxf(cmax, zz);
                vmax = fmaxf(vmax, vv);
            }
        }
        cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 1));
        cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 2));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 2));
        // Lazy reference max: weights 2^(z - m) may reach 2^kLazy before the
        // accumulators are rescaled; kVScaleBias leaves room for that in f16.
        const int Ec = (int)(__float_as_uint(vmax) >> 23);
        if (__any_sync(0xFFFFFFFFu, cmax > m + (float)kLazy || Ec > E)) {
            const float m_new = fmaxf(m, cmax);
            const int E_new = max(E, Ec);
            const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
            const float ea = (E - E_new < -126) ? 0.0f : __uint_as_float((uint32_t)(127 + E - E_new) << 23);
            const float fa = alpha * ea;
            // rows whose max did not move keep alpha = 1, ea may still shrink them
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                acc[n][0] *= fa; acc[n][1] *= fa; acc[n][2] *= fa; acc[n][3] *= fa;
            }
            lsum *= alpha;
            m = m_new;
            E = E_new;
            wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
        }
        // a row that has seen no token yet keeps m = -inf; its z are all -inf
        const float m_ref = m == -INFINITY ? 0.0f : m;
        float pw[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const float p = fast_exp2(z[u] - m_ref);    // <= 2^kLazy; masked tokens: 2^-inf = 0
            lsum += p;
            pw[u] = p * vs[u] * wscale;
        }
        // ---- O += P V, two k-steps of 16 tokens
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            uint32_t ap[4];
            split_f16x2(pw[4 * kk + 0], pw[4 * kk + 1], ap[0], ap[1]);
            split_f16x2(pw[4 * kk + 2], pw[4 * kk + 3], ap[2], ap[3]);
            const uint32_t *r0 = sV + (16 * kk + 2 * cq) * W;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                const int wd = vword<D>(gq, jj);
                const uint32_t x0 = r0[wd], x1 = r0[W + wd], x8 = r0[8 * W + wd], x9 = r0[9 * W + wd];
                mma_16816(acc[4 * jj + 0], ap, codes_pair_to_f16x2<0>(x0, x1, fk), codes_pair_to_f16x2<0>(x8, x9, fk));
                mma_16816(acc[4 * jj + 1], ap, codes_pair_to_f16x2<1>(x0, x1, fk), codes_pair_to_f16x2<1>(x8, x9, fk));
                mma_16816(acc[4 * jj + 2], ap, codes_pair_to_f16x2<2>(x0, x1, fk), codes_pair_to_f16x2<2>(x8, x9, fk));
                mma_16816(acc[4 * jj + 3], ap, codes_pair_to_f16x2<3>(x0, x1, fk), codes_pair_to_f16x2<3>(x8, x9, fk));
            }
        }
        // ---- release the buffer, refill it with this slot's chunk i + RING
        if constexpr (HT > 1) named_barrier(1 + ts, HT * 32);
        else __syncwarp();
        if (ht == 0 && issued < my_n) {
            issue_chunk<D>(P, w, table, ts + SLOTS * issued, ring + k * L.slot_bytes, bars + 8 * k, policy);
            ++issued;
        }
    }
    if (ht == 0) drain(P, bars, RING, i, issued);

    // All warps are past their rings; reuse them as merge scratch.
    if (__syncthreads_or(!ok)) return;
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 2);
    float *ml = reinterpret_cast<float *>(smem + L.ring);            // [slot][HT*8][3]
    float *accs = ml + SLOTS * HT * 8 * 3;                            // [slot][HT*8][D]
    const int hl = 8 * ht + gq;                                        // CTA-local head
    if (cq == 0) {
        float *e = ml + (ts * HT * 8 + hl) * 3;
        e[0] = m; e[1] = lsum; e[2] = (float)E;
    }
    float *arow = accs + (ts * HT * 8 + hl) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        arow[4 * vword<D>(2 * cq, n / 4) + (n & 3)] = acc[n][0] + acc[n][2];
        arow[4 * vword<D>(2 * cq + 1, n / 4) + (n & 3)] = acc[n][1] + acc[n][3];
    }
    __syncthreads();
    merge_and_store<D>(P, w, ml, accs, SLOTS, HT * 8, accs + SLOTS * HT * 8 * D);
}

// ============================================================== CUDA cores
//
// Warp ts owns chunks ts, ts + 4, ... of the partition.  QK: lane = token;
// the CTA's q rows are read from shared memory (broadcast) as f32.
// Softmax: per head, warp-wide max; weights p * v_scale go to shared memory.
// PV: lane = code word (4 head dims); for head size 64 the two half warps
// take alternate tokens, for 256 each lane takes two words.
constexpr int kCcSlots = 4;

template <int D>
__host__ __device__ constexpr int cc_ring() { return D == 256 ? 2 : 3; }

__device__ __forceinline__ void codes4_to_f32(uint32_t x, float &a, float &b, float &c, float &d) {
    // offset-binary byte under 0x4B000000 is 2^23 + code + 128 exactly
    const uint32_t u = x ^ 0x80808080u;
    const uint32_t hi = 0x4B000000u;
    a = __uint_as_float(prmt_i<0x7650u>(u, hi)) - 8388736.0f;
    b = __uint_as_float(prmt_i<0x7651u>(u, hi)) - 8388736.0f;
    c = __uint_as_float(prmt_i<0x7652u>(u, hi)) - 8388736.0f;
    d = __uint_as_float(prmt_i<0x7653u>(u, hi)) - 8388736.0f;
}

// shared memory beside the ring: q rows [NH][D], weights [slot][NH][32], row lags [NH]
template <int D, int NH>
__host__ __device__ constexpr uint32_t cc_extra() { return NH * D * 4 + kCcSlots * 32 * NH * 4 + NH * 4; }

template <int D, int NH>
__global__ void __launch_bounds__(kCcSlots * 32, (D == 256 ? 1 : 2))
decode_cc_kernel(Params P) {
    constexpr int RING = cc_ring<D>();
    constexpr int W = D / 4 + 1;
    constexpr int WORDS = D / 4;
    constexpr int LW = WORDS < 32 ? WORDS : 32;      // lanes per token row in PV
    constexpr int TG = 32 / LW;                      // token groups in PV (2 for D = 64)
    constexpr int NWL = WORDS / LW;                  // words per lane in PV

    extern __shared__ __align__(128) uint8_t smem[];
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const Layout L = make_layout(D, kCcSlots, RING, P.PT, P.B, cc_extra<D, NH>());
    const int ts = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t bars = smem_addr(smem + L.bars) + 8 * RING * ts;
    const uint32_t ring = smem_addr(smem + L.ring) + RING * L.slot_bytes * ts;
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    float *sq = reinterpret_cast<float *>(smem + L.extra);             // [NH][D]
    float *myw = sq + NH * D + ts * 32 * NH;                           // [NH][32]
    int *slag = reinterpret_cast<int *>(sq + NH * D + kCcSlots * 32 * NH);   // [NH]
    const int nchunks = (w.len + kChunk - 1) / kChunk;
    const int my_n = ts < nchunks ? (nchunks - ts + kCcSlots - 1) / kCcSlots : 0;
    const uint64_t policy = l2_policy_evict_first();

    if (lane == 0) {
        for (int k = 0; k < RING; ++k) mbar_init(bars + 8 * k, 1);
        fence_mbar_init();
    }
    if (P.nk) append_tokens<D>(P, w);
    load_table(P, w, const_cast<uint32_t *>(table));
    for (int i = threadIdx.x; i < NH * D; i += blockDim.x) {
        const int hh = i / D;
        sq[i] = hh < w.nh ? __ldg(P.q + qrow(P, w, w.h0 + hh) * D + (i % D)) : 0.0f;
    }
    // query row b of R sees the first c - (R-1-b) tokens: its lag behind the context
    if (threadIdx.x < NH)
        slag[threadIdx.x] = (int)threadIdx.x < w.nh ? P.R - 1 - (w.h0 + (int)threadIdx.x) / P.r : INT_MAX;
    __syncthreads();
    int issued = 0;
    for (; issued < RING && issued < my_n; ++issued)
        issue_chunk<D>(P, w, table, ts + kCcSlots * issued, ring + issued * L.slot_bytes,
                       bars + 8 * issued, policy);

    const float4 *sq4 = reinterpret_cast<const float4 *>(sq);
    float m[NH], lsum[NH], acc[NH][NWL][4];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        m[hh] = -INFINITY;
        lsum[hh] = 0.0f;
#pragma unroll
        for (int u = 0; u < NWL; ++u) acc[hh][u][0] = acc[hh][u][1] = acc[hh][u][2] = acc[hh][u][3] = 0.0f;
    }

    bool ok = true;
    int i = 0;
    for (; i < my_n; ++i) {
        const int k = i % RING;
        if (!mbar_wait(bars + 8 * k, (i / RING) & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(smem + L.ring) +
                             (RING * ts + k) * (L.slot_bytes / 4);
        const uint32_t *sV = sK + kChunk * W;
        const int t0 = (ts + kCcSlots * i) * kChunk;
        // ---- logits, lane = token
        const bool valid = t0 + lane < w.len;
        const int ahead = w.c - w.t_begin - t0 - lane;        // tokens from this one to the context end
        float dot[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) dot[hh] = 0.0f;
        const uint32_t *krow = sK + lane * W;
#pragma unroll 4
        for (int wd = 0; wd < WORDS; ++wd) {
            float c0, c1, c2, c3;
            codes4_to_f32(krow[wd], c0, c1, c2, c3);
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float4 qv = sq4[hh * WORDS + wd];
                dot[hh] = fmaf(qv.x, c0, fmaf(qv.y, c1, fmaf(qv.z, c2, fmaf(qv.w, c3, dot[hh]))));
            }
        }
        const float kscale = __uint_as_float(krow[WORDS]) * P.scale_log2;
        const float vscale = valid ? __uint_as_float(sV[lane * W + WORDS]) : 0.0f;
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            const bool seen = valid && slag[hh] < ahead;      // causal limit of this query row
            const float z = seen ? dot[hh] * kscale : -INFINITY;
            float cm = z;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
            const float m_new = fmaxf(m[hh], cm);
            if (m_new != m[hh]) {        // warp-uniform
                const float alpha = (m[hh] == -INFINITY) ? 0.0f : fast_exp2(m[hh] - m_new);
                lsum[hh] *= alpha;
#pragma unroll
                for (int u = 0; u < NWL; ++u) {
                    acc[hh][u][0] *= alpha; acc[hh][u][1] *= alpha;
                    acc[hh][u][2] *= alpha; acc[hh][u][3] *= alpha;
                }
                m[hh] = m_new;
            }
            const float p = seen ? fast_exp2(z - m[hh]) : 0.0f;
            lsum[hh] += p;
            myw[hh * 32 + lane] = p * vscale;
        }
        __syncwarp();
        // ---- weighted sum, lane = code word(s)
        const int ntok = min(kChunk, w.len - t0);
        const int tg = lane / LW, lw = lane % LW;
#pragma unroll 2
        for (int tt = tg; tt < ntok; tt += TG) {
            const uint32_t *vrow = sV + tt * W;
            float v[NWL][4];
#pragma unroll
            for (int u = 0; u < NWL; ++u) codes4_to_f32(vrow[lw + 32 * u], v[u][0], v[u][1], v[u][2], v[u][3]);
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float wt = myw[hh * 32 + tt];
#pragma unroll
                for (int u = 0; u < NWL; ++u) {
                    acc[hh][u][0] = fmaf(wt, v[u][0], acc[hh][u][0]);
                    acc[hh][u][1] = fmaf(wt, v[u][1], acc[hh][u][1]);
                    acc[hh][u][2] = fmaf(wt, v[u][2], acc[hh][u][2]);
                    acc[hh][u][3] = fmaf(wt, v[u][3], acc[hh][u][3]);
                }
            }
        }
        __syncwarp();
        if (issued < my_n) {
            issue_chunk<D>(P, w, table, ts + kCcSlots * issued, ring + k * L.slot_bytes, bars + 8 * k, policy);
            ++issued;
        }
    }
    drain(P, bars, RING, i, issued);

    if (__syncthreads_or(!ok)) return;
    float *ml = reinterpret_cast<float *>(smem + L.ring);      // [slot][NH][3]
    float *accs = ml + kCcSlots * NH * 3;                       // [slot][NH][D]
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        float l = lsum[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
#pragma unroll
        for (int u = 0; u < NWL; ++u) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float a = acc[hh][u][e];
                if constexpr (TG == 2) a += __shfl_xor_sync(0xFFFFFFFFu, a, 16);
                acc[hh][u][e] = a;
            }
        }
        if (lane == 0) {
            float *e = ml + (ts * NH + hh) * 3;
            e[0] = m[hh]; e[1] = l; e[2] = (float)kVScaleBias;
        }
        if (lane < LW) {
#pragma unroll
            for (int u = 0; u < NWL; ++u) {
                float *dst = accs + (ts * NH + hh) * D + 4 * (lane + 32 * u);
                dst[0] = acc[hh][u][0]; dst[1] = acc[hh][u][1];
                dst[2] = acc[hh][u][2]; dst[3] = acc[hh][u][3];
            }
        }
    }
    __syncthreads();
    merge_and_store<D>(P, w, ml, accs, kCcSlots, NH, accs + kCcSlots * NH * D);
}

// ================================================= contiguous q8 cache
//
// The contiguous cache with a side scale region ("attention.rs": the
// kv_append_q8 dispatch and kv_q8_side): per sequence, [max_t][kv_row] int8
// codes (u32 words, kv_row = Hk * D) then [max_t][kv_row / 32] f32 scales,
// one per 32-element group; sequences back to back.  P.Nb holds max_t (and
// P.B = 1): position t of sequence s is token t, no block table.
//
// The tensor-core tile of decode_tc_kernel with three changes:
//  - lane = token: each lane bulk-copies its token's K and V code rows (D
//    bytes) and scale rows (D / 8 bytes) of kv head g into the chunk buffer;
//    code rows sit WC = D/4 + 4 words apart (16-byte rows, WC = 4 mod 32);
//  - the word maps kword = 4 ks + cq and vword = n + 8 jj are bank-conflict
//    free at that stride, and keep each k-step of QK and each 4 n-tiles of PV
//    inside one 32-element group;
//  - QK accumulates each group separately and adds it times the token's
//    group scale; PV weights are p * v_scale[token][group] per group.

template <int D>
__host__ __device__ constexpr int cq_wc() { return D / 4 + 4; }

template <int D>
__host__ __device__ constexpr uint32_t cq_slot_bytes() {
    return 2u * (kChunk * cq_wc<D>() * 4u + kChunk * (D / 32) * 4u);
}

constexpr int kCqRing = 2;

// [barriers] [q fragments (head size 256)] [chunk buffers: slot x ring]
struct CqLayout {
    uint32_t extra, ring, total;
};

template <int D>
__host__ __device__ inline CqLayout make_cq_layout() {
    CqLayout L{};
    L.extra = align_up(PA_Q8_TC_SLOTS * kCqRing * 8, 128);
    L.ring = align_up(L.extra + (D == 256 ? (uint32_t)(D / 16) * 32 * 16 : 0u), 128);
    L.total = L.ring + PA_Q8_TC_SLOTS * kCqRing * cq_slot_bytes<D>();
    return L;
}

template <int D>
__device__ __forceinline__ void issue_cq_chunk(const Params &P, const Work &w, int c, uint32_t slot, uint32_t bar,
                                               uint64_t policy) {
    constexpr int WC = cq_wc<D>();
    constexpr uint32_t CODES = kChunk * WC * 4u, SCALES = kChunk * (D / 32) * 4u;
    const int lane = threadIdx.x & 31;
    const int t = c * kChunk + lane;                      // partition-relative token
    const int n = min(kChunk, w.len - c * kChunk);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)n * 2u * (D + D / 8));
    __syncwarp();
    if (t < w.len) {
        fence_proxy_async_smem();
        const int64_t kv_row = (int64_t)P.Hk * D, max_t = P.Nb;
        const int64_t seq_words = max_t * (kv_row / 4) + max_t * (kv_row / 32);
        const int64_t pos = (int64_t)w.t_begin + t;
        const int64_t code = (int64_t)w.s * seq_words + pos * (kv_row / 4) + (int64_t)w.g * (D / 4);
        const int64_t scale = (int64_t)w.s * seq_words + max_t * (kv_row / 4) + pos * (kv_row / 32) +
                              (int64_t)w.g * (D / 32);
        bulk_copy_g2s(slot + lane * WC * 4, P.kc + code, D, bar, policy);
        bulk_copy_g2s(slot + CODES + lane * (D / 8), P.kc + scale, D / 8, bar, policy);
        bulk_copy_g2s(slot + CODES + SCALES + lane * WC * 4, P.vc + code, D, bar, policy);
        bulk_copy_g2s(slot + 2 * CODES + SCALES + lane * (D / 8), P.vc + scale, D / 8, bar, policy);
    }
}

// Head size 128: the chunk moves as four 3-D tensor copies (TMA) over the
// caches seen as [sequence][position][kv_row bytes] codes and [sequence]
// [position][kv_row / 32] scales (the sequence stride covers both regions):
// code boxes of 128 bytes x 32 positions with the 128-byte swizzle (16-byte
// chunk c of row r at c ^ (r % 8)), scale boxes of 4 floats x 32 positions.
// The word maps stay conflict-free under the swizzle: QK reads chunk ks ^ gq
// of rows 8j + gq, PV reads chunk ((gq >> 2) + 2jj) ^ (row % 8).
struct CqTmaParams {
    Params p;
    CUtensorMap kcodes, kscales, vcodes, vscales;
};

constexpr uint32_t kCqTmaCodes = kChunk * 128u, kCqTmaScales = kChunk * 16u;
constexpr uint32_t kCqTmaSlot = 2u * kCqTmaCodes + 2u * kCqTmaScales;      // 9216 = 9 x 1024

// [barriers] [ring, 1024-aligned at run time: slot x ring] (+1024 slack)
__host__ __device__ inline uint32_t cq_tma_smem_bytes() {
    return 1024u + PA_Q8_TC_SLOTS * kCqRing * 8u + PA_Q8_TC_SLOTS * kCqRing * kCqTmaSlot + 1024u;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, int x, int y, int z, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar), "l"(policy)
        : "memory");
}

// Byte offset of code word w of row r in a swizzled 128-byte-row box.
__device__ __forceinline__ uint32_t sw128(int r, int w) {
    return (uint32_t)(r * 128 + ((((w >> 2) ^ r) & 7) << 4) + (w & 3) * 4);
}

template <int D>
__global__ void __launch_bounds__(PA_Q8_TC_SLOTS * 32, 2)
decode_cq_tma_kernel(const __grid_constant__ CqTmaParams CP) {
    static_assert(D == 128, "tensor-copy contiguous decode: head size 128");
    const Params &P = CP.p;
    constexpr int SLOTS = PA_Q8_TC_SLOTS;
    constexpr int RING = kCqRing;
    constexpr int G = D / 32;
    constexpr int NKS = D / 16;
    constexpr int NT = D / 8;
    constexpr int NJ = D / 32;

    extern __shared__ __align__(128) uint8_t smem[];
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ts = warp;
    const int gq = lane >> 2, cq = lane & 3;
    const uint32_t s0 = smem_addr(smem);
    const uint32_t bars = s0 + 8 * RING * ts;
    const uint32_t ring0 = (s0 + SLOTS * RING * 8u + 1023u) & ~1023u;
    const uint32_t ring = ring0 + RING * kCqTmaSlot * ts;
    const int nchunks = (w.len + kChunk - 1) / kChunk;
    const int my_n = ts < nchunks ? (nchunks - ts + SLOTS - 1) / SLOTS : 0;
    const uint64_t policy = l2_policy_evict_first();

    if (lane == 0) {
        for (int k = 0; k < RING; ++k) mbar_init(bars + 8 * k, 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](int c, int k) {           // chunk c into buffer k: four boxes (lanes 0-3)
        const uint32_t dst = ring + k * kCqTmaSlot, bar = bars + 8 * k;
        if (lane == 0) mbar_arrive_expect_tx(bar, kCqTmaSlot);
        __syncwarp();
        if (lane < 4) {
            fence_proxy_async_smem();
            const int y = w.t_begin + c * kChunk;
            if (lane == 0) tma_load_3d(dst, &CP.kcodes, w.g * D, y, w.s, bar, policy);
            else if (lane == 1) tma_load_3d(dst + kCqTmaCodes, &CP.vcodes, w.g * D, y, w.s, bar, policy);
            else if (lane == 2) tma_load_3d(dst + 2 * kCqTmaCodes, &CP.kscales, w.g * G, y, w.s, bar, policy);
            else tma_load_3d(dst + 2 * kCqTmaCodes + kCqTmaScales, &CP.vscales, w.g * G, y, w.s, bar, policy);
        }
    };
    int issued = 0;
    for (; issued < RING && issued < my_n; ++issued) issue(ts + SLOTS * issued, issued);

    const bool row_ok = gq < w.nh;
    const int vh = w.h0 + gq;
    const int len_row = row_ok ? row_len(P, w, vh) : w.len;
    const int len_min = __reduce_min_sync(0xFFFFFFFFu, (unsigned)len_row);

    uint32_t aq[NKS][4];
    float qk2;
    {
        const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok ? vh : w.h0) * D);
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok ? __ldg(qv + 4 * ks + cq) : make_float4(0.f, 0.f, 0.f, 0.f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);      // 2^-eq
        qk2 = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok ? __ldg(qv + 4 * ks + cq) : make_float4(0.f, 0.f, 0.f, 0.f);
            split_f16x2(v.x * down, v.y * down, aq[ks][0], aq[ks][1]);
            split_f16x2(v.z * down, v.w * down, aq[ks][2], aq[ks][3]);
        }
    }

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    float m = -INFINITY, lsum = 0.0f;
    int E = 12;
    float wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
    const F16Consts fk;

    bool ok = true;
    int i = 0;
    for (; i < my_n; ++i) {
        const int k = i % RING;
        if (!mbar_wait(bars + 8 * k, (i / RING) & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        const uint8_t *base = smem + (ring0 - s0) + (RING * ts + k) * kCqTmaSlot;
        const uint8_t *sK = base, *sV = base + kCqTmaCodes;
        const float *sKs = reinterpret_cast<const float *>(base + 2 * kCqTmaCodes);
        const float *sVs = sKs + kChunk * G;
        const int t0 = (ts + SLOTS * i) * kChunk;
        const bool full = t0 + kChunk <= len_min;

        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float sg[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) sg[j][0] = sg[j][1] = sg[j][2] = sg[j][3] = 0.0f;
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
                const int ks = 2 * g + kh;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t b0, b1;
                    codes4_to_f16x2(*reinterpret_cast<const uint32_t *>(sK + sw128(8 * j + gq, 4 * ks + cq)), b0, b1,
                                    fk);
                    mma_16816(sg[j], aq[ks], b0, b1);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float k0 = sKs[(8 * j + 2 * cq) * G + g], k1 = sKs[(8 * j + 2 * cq + 1) * G + g];
                s[j][0] = fmaf(sg[j][0], k0, s[j][0]);
                s[j][1] = fmaf(sg[j][1], k1, s[j][1]);
                s[j][2] = fmaf(sg[j][2], k0, s[j][2]);
                s[j][3] = fmaf(sg[j][3], k1, s[j][3]);
            }
        }
        float z[8];
        float cmax = -INFINITY, vmax = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 8 * j + 2 * cq + e;
                float zz = (s[j][e] + s[j][e + 2]) * qk2;
                float vv = 0.0f;
#pragma unroll
                for (int g = 0; g < G; ++g) vv = fmaxf(vv, sVs[t * G + g]);
                if (!full) {
                    const bool valid = t0 + t < len_row;
                    zz = valid ? zz : -INFINITY;
                    vv = valid ? vv : 0.0f;
                }
                z[2 * j + e] = zz;
                cmax = fmaxf(cmax, zz);
                vmax = fmaxf(vmax, vv);
            }
        }
        cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 1));
        cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 2));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 2));
        const int Ec = (int)(__float_as_uint(vmax) >> 23);
        if (__any_sync(0xFFFFFFFFu, cmax > m + (float)kLazy || Ec > E)) {
            const float m_new = fmaxf(m, cmax);
            const int E_new = max(E, Ec);
            const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
            const float ea = (E - E_new < -126) ? 0.0f : __uint_as_float((uint32_t)(127 + E - E_new) << 23);
            const float fa = alpha * ea;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                acc[n][0] *= fa; acc[n][1] *= fa; acc[n][2] *= fa; acc[n][3] *= fa;
            }
            lsum *= alpha;
            m = m_new;
            E = E_new;
            wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
        }
        const float m_ref = m == -INFINITY ? 0.0f : m;
        float p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            p[u] = fast_exp2(z[u] - m_ref);
            lsum += p[u];
            p[u] *= wscale;
        }
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
            const int wd = gq + 8 * jj;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                float pw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = 16 * kk + 2 * cq + (u & 1) + 8 * (u >> 1);
                    const bool valid = full || t0 + t < len_row;
                    pw[u] = valid ? p[4 * kk + u] * sVs[t * G + jj] : 0.0f;
                }
                uint32_t ap[4];
                split_f16x2(pw[0], pw[1], ap[0], ap[1]);
                split_f16x2(pw[2], pw[3], ap[2], ap[3]);
                const int r = 16 * kk + 2 * cq;
                const uint32_t x0 = *reinterpret_cast<const uint32_t *>(sV + sw128(r, wd));
                const uint32_t x1 = *reinterpret_cast<const uint32_t *>(sV + sw128(r + 1, wd));
                const uint32_t x8 = *reinterpret_cast<const uint32_t *>(sV + sw128(r + 8, wd));
                const uint32_t x9 = *reinterpret_cast<const uint32_t *>(sV + sw128(r + 9, wd));
                mma_16816(acc[4 * jj + 0], ap, codes_pair_to_f16x2<0>(x0, x1, fk), codes_pair_to_f16x2<0>(x8, x9, fk));
                mma_16816(acc[4 * jj + 1], ap, codes_pair_to_f16x2<1>(x0, x1, fk), codes_pair_to_f16x2<1>(x8, x9, fk));
                mma_16816(acc[4 * jj + 2], ap, codes_pair_to_f16x2<2>(x0, x1, fk), codes_pair_to_f16x2<2>(x8, x9, fk));
                mma_16816(acc[4 * jj + 3], ap, codes_pair_to_f16x2<3>(x0, x1, fk), codes_pair_to_f16x2<3>(x8, x9, fk));
            }
        }
        __syncwarp();
        if (issued < my_n) {
            issue(ts + SLOTS * issued, k);
            ++issued;
        }
    }
    drain(P, bars, RING, i, issued);

    if (__syncthreads_or(!ok)) return;
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 2);
    float *ml = reinterpret_cast<float *>(smem + (ring0 - s0));       // [slot][8][3]
    float *accs = ml + SLOTS * 8 * 3;                                 // [slot][8][D]
    if (cq == 0) {
        float *e = ml + (ts * 8 + gq) * 3;
        e[0] = m; e[1] = lsum; e[2] = (float)E;
    }
    float *arow = accs + (ts * 8 + gq) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        arow[4 * (2 * cq + 8 * (n >> 2)) + (n & 3)] = acc[n][0] + acc[n][2];
        arow[4 * (2 * cq + 1 + 8 * (n >> 2)) + (n & 3)] = acc[n][1] + acc[n][3];
    }
    __syncthreads();
    merge_and_store<D>(P, w, ml, accs, SLOTS, 8, accs + SLOTS * 8 * D);
}

template <int D>
__global__ void __launch_bounds__(PA_Q8_TC_SLOTS * 32, 2)
decode_cq_kernel(Params P) {
    constexpr int SLOTS = PA_Q8_TC_SLOTS;
    constexpr int RING = kCqRing;
    constexpr int WC = cq_wc<D>();
    constexpr int G = D / 32;            // scale groups per row
    constexpr int NKS = D / 16;
    constexpr int NT = D / 8;
    constexpr int NJ = D / 32;
    constexpr bool kQInSmem = (D == 256);
    constexpr uint32_t CODES = kChunk * WC * 4u, SCALES = kChunk * G * 4u;

    extern __shared__ __align__(128) uint8_t smem[];
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const CqLayout L = make_cq_layout<D>();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ts = warp;
    const int gq = lane >> 2, cq = lane & 3;
    const uint32_t bars = smem_addr(smem) + 8 * RING * ts;
    const uint32_t ring = smem_addr(smem + L.ring) + RING * cq_slot_bytes<D>() * ts;
    const int nchunks = (w.len + kChunk - 1) / kChunk;
    const int my_n = ts < nchunks ? (nchunks - ts + SLOTS - 1) / SLOTS : 0;
    const uint64_t policy = l2_policy_evict_first();

    if (lane == 0) {
        for (int k = 0; k < RING; ++k) mbar_init(bars + 8 * k, 1);
        fence_mbar_init();
    }
    __syncthreads();
    int issued = 0;
    for (; issued < RING && issued < my_n; ++issued)
        issue_cq_chunk<D>(P, w, ts + SLOTS * issued, ring + issued * cq_slot_bytes<D>(), bars + 8 * issued, policy);

    const bool row_ok = gq < w.nh;
    const int vh = w.h0 + gq;
    const int len_row = row_ok ? row_len(P, w, vh) : w.len;
    const int len_min = __reduce_min_sync(0xFFFFFFFFu, (unsigned)len_row);

    uint32_t aq[kQInSmem ? 1 : NKS][4];
    uint4 *qf = reinterpret_cast<uint4 *>(smem + L.extra);           // [NKS][32]
    float qk2;
    {
        const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok ? vh : w.h0) * D);
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok ? __ldg(qv + 4 * ks + cq) : make_float4(0.f, 0.f, 0.f, 0.f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);      // 2^-eq
        qk2 = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok ? __ldg(qv + 4 * ks + cq) : make_float4(0.f, 0.f, 0.f, 0.f);
            uint32_t f0, f1, f2, f3;
            split_f16x2(v.x * down, v.y * down, f0, f1);
            split_f16x2(v.z * down, v.w * down, f2, f3);
            if constexpr (kQInSmem) {
                if (ts == 0) qf[ks * 32 + lane] = make_uint4(f0, f1, f2, f3);
            } else {
                aq[ks][0] = f0; aq[ks][1] = f1; aq[ks][2] = f2; aq[ks][3] = f3;
            }
        }
        if constexpr (kQInSmem) __syncthreads();
    }

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    float m = -INFINITY, lsum = 0.0f;
    int E = 12;
    float wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
    const F16Consts fk;

    bool ok = true;
    int i = 0;
    for (; i < my_n; ++i) {
        const int k = i % RING;
        if (!mbar_wait(bars + 8 * k, (i / RING) & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        const uint8_t *base = smem + L.ring + (RING * ts + k) * cq_slot_bytes<D>();
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(base);
        const float *sKs = reinterpret_cast<const float *>(base + CODES);
        const uint32_t *sV = reinterpret_cast<const uint32_t *>(base + CODES + SCALES);
        const float *sVs = reinterpret_cast<const float *>(base + 2 * CODES + SCALES);
        const int t0 = (ts + SLOTS * i) * kChunk;
        const bool full = t0 + kChunk <= len_min;

        // ---- S = sum over groups of (Q_g K_g^T) x the tokens' group scales
        float s[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) s[j][0] = s[j][1] = s[j][2] = s[j][3] = 0.0f;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float sg[4][4];
#pragma unroll
            for (int j = 0; j < 4; ++j) sg[j][0] = sg[j][1] = sg[j][2] = sg[j][3] = 0.0f;
#pragma unroll
            for (int kh = 0; kh < 2; ++kh) {
                const int ks = 2 * g + kh;
                uint32_t a[4];
                if constexpr (kQInSmem) {
                    const uint4 f = qf[ks * 32 + lane];
                    a[0] = f.x; a[1] = f.y; a[2] = f.z; a[3] = f.w;
                } else {
                    a[0] = aq[ks][0]; a[1] = aq[ks][1]; a[2] = aq[ks][2]; a[3] = aq[ks][3];
                }
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t b0, b1;
                    codes4_to_f16x2(sK[(8 * j + gq) * WC + 4 * ks + cq], b0, b1, fk);
                    mma_16816(sg[j], a, b0, b1);
                }
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const float k0 = sKs[(8 * j + 2 * cq) * G + g], k1 = sKs[(8 * j + 2 * cq + 1) * G + g];
                s[j][0] = fmaf(sg[j][0], k0, s[j][0]);
                s[j][1] = fmaf(sg[j][1], k1, s[j][1]);
                s[j][2] = fmaf(sg[j][2], k0, s[j][2]);
                s[j][3] = fmaf(sg[j][3], k1, s[j][3]);
            }
        }
        // ---- online softmax over this thread's 8 tokens: 8j + 2cq + e
        float z[8];
        float cmax = -INFINITY, vmax = 0.0f;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 8 * j + 2 * cq + e;
                float zz = (s[j][e] + s[j][e + 2]) * qk2;
                float vv = 0.0f;
#pragma unroll
                for (int g = 0; g < G; ++g) vv = fmaxf(vv, sVs[t * G + g]);
                if (!full) {
                    const bool valid = t0 + t < len_row;
                    zz = valid ? zz : -INFINITY;
                    vv = valid ? vv : 0.0f;
                }
                z[2 * j + e] = zz;
                cmax = fmaxf(cmax, zz);
                vmax = fmaxf(vmax, vv);
            }
        }
        cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 1));
        cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 2));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 1));
        vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 2));
        const int Ec = (int)(__float_as_uint(vmax) >> 23);
        if (__any_sync(0xFFFFFFFFu, cmax > m + (float)kLazy || Ec > E)) {
            const float m_new = fmaxf(m, cmax);
            const int E_new = max(E, Ec);
            const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
            const float ea = (E - E_new < -126) ? 0.0f : __uint_as_float((uint32_t)(127 + E - E_new) << 23);
            const float fa = alpha * ea;
#pragma unroll
            for (int n = 0; n < NT; ++n) {
                acc[n][0] *= fa; acc[n][1] *= fa; acc[n][2] *= fa; acc[n][3] *= fa;
            }
            lsum *= alpha;
            m = m_new;
            E = E_new;
            wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
        }
        const float m_ref = m == -INFINITY ? 0.0f : m;
        float p[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            p[u] = fast_exp2(z[u] - m_ref);                  // masked tokens: 2^-inf = 0
            lsum += p[u];
            p[u] *= wscale;
        }
        // ---- O += P V, per scale group (its 4 n-tiles), two k-steps of 16 tokens
#pragma unroll
        for (int jj = 0; jj < NJ; ++jj) {
            const int wd = gq + 8 * jj;
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                float pw[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int t = 16 * kk + 2 * cq + (u & 1) + 8 * (u >> 1);   // tokens of p[4kk + u]
                    const bool valid = full || t0 + t < len_row;
                    pw[u] = valid ? p[4 * kk + u] * sVs[t * G + jj] : 0.0f;
                }
                uint32_t ap[4];
                split_f16x2(pw[0], pw[1], ap[0], ap[1]);
                split_f16x2(pw[2], pw[3], ap[2], ap[3]);
                const uint32_t *r0 = sV + (16 * kk + 2 * cq) * WC;
                const uint32_t x0 = r0[wd], x1 = r0[WC + wd], x8 = r0[8 * WC + wd], x9 = r0[9 * WC + wd];
                mma_16816(acc[4 * jj + 0], ap, codes_pair_to_f16x2<0>(x0, x1, fk), codes_pair_to_f16x2<0>(x8, x9, fk));
                mma_16816(acc[4 * jj + 1], ap, codes_pair_to_f16x2<1>(x0, x1, fk), codes_pair_to_f16x2<1>(x8, x9, fk));
                mma_16816(acc[4 * jj + 2], ap, codes_pair_to_f16x2<2>(x0, x1, fk), codes_pair_to_f16x2<2>(x8, x9, fk));
                mma_16816(acc[4 * jj + 3], ap, codes_pair_to_f16x2<3>(x0, x1, fk), codes_pair_to_f16x2<3>(x8, x9, fk));
            }
        }
        __syncwarp();
        if (issued < my_n) {
            issue_cq_chunk<D>(P, w, ts + SLOTS * issued, ring + k * cq_slot_bytes<D>(), bars + 8 * k, policy);
            ++issued;
        }
    }
    drain(P, bars, RING, i, issued);

    if (__syncthreads_or(!ok)) return;
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 2);
    float *ml = reinterpret_cast<float *>(smem + L.ring);            // [slot][8][3]
    float *accs = ml + SLOTS * 8 * 3;                                 // [slot][8][D]
    if (cq == 0) {
        float *e = ml + (ts * 8 + gq) * 3;
        e[0] = m; e[1] = lsum; e[2] = (float)E;
    }
    float *arow = accs + (ts * 8 + gq) * D;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
        // acc[n]: columns 2cq, 2cq+1 of n-tile n = dims 4 (vword(2cq / 2cq+1)) + (n & 3)
        arow[4 * (2 * cq + 8 * (n >> 2)) + (n & 3)] = acc[n][0] + acc[n][2];
        arow[4 * (2 * cq + 1 + 8 * (n >> 2)) + (n & 3)] = acc[n][1] + acc[n][3];
    }
    __syncthreads();
    merge_and_store<D>(P, w, ml, accs, SLOTS, 8, accs + SLOTS * 8 * D);
}

// ======================================================== tcgen05 (multi-row)
//
// Many virtual heads per kv head (multi-row decode: R query rows x r heads)
// make the contraction GEMM-shaped, so it runs on the 5th-generation tensor
// cores: one CTA serves up to 64 virtual heads of one kv head for one
// partition.  TMEM lane quadrant q holds M rows 32q .. 32q+31: rows 32q + j
// (j < 16) the hi f16 part of virtual head 16q + j's q (scaled by 2^-eq like
// the mma.sync kernel), rows 32q + 16 + j its lo part, so a logit's two
// halves are one shuffle apart.  TMEM holds S twice (columns 0-31, 32-63) and
// O (D columns).
//
// Warp roles, linked only by mbarriers (every wait bounded and abortable):
//  - warps 0-3, softmax: warp q owns quadrant q (idle when it holds no head).
//    Per chunk: S row -> online softmax (hi/lo partner threads take 16 tokens
//    each; lazy rescale of O rows in TMEM) -> P tile rows (w = p * v_scale *
//    2^(131 - E), split hi/lo like the mma.sync kernel).
//  - warps 4-6, conversion: per chunk the raw codes (bulk-copied ring, as in
//    the other families) become f16 K [32][D] and V^T [D][32] tiles (K-major
//    core matrices) and the token scales a small table.
//  - warp 7: refills the ring; its lane 0 issues S = Q.K^T (M 128, N 32, K D)
//    and, one chunk behind, O += P.V (M 128, N D, K 32).
// K, V^T, P and S are double buffered by chunk parity.  Signals per buffer
// b = chunk & 1: conv[b] (96 conversion threads), s_free[b] / p_ready[b]
// (the active softmax threads), qk[b] / pv[b] (tcgen05.commit).  A waiter
// never falls two phases behind: the next phase of each barrier needs a step
// that follows the wait.

constexpr int kUmmaHeads = 64;
constexpr int kUmmaThreads = 256;
constexpr int kUmmaConvThreads = 96;

template <int D>
__host__ __device__ constexpr int umma_ring() { return 3; }
template <int D>
__host__ __device__ constexpr uint32_t umma_tmem_cols() { return D == 64 ? 128u : (D == 128 ? 256u : 512u); }
// resident CTAs per SM: TMEM (512 columns) and registers (2 x 256 threads x 128)
template <int D>
__host__ __device__ constexpr int umma_ctas_per_sm() { return D == 256 ? 1 : 2; }

// Byte offset of element (r, k) of an f16 operand tile with kdim columns in
// the K-major core-matrix layout (LBO = 128, SBO = kdim / 8 * 128).
__device__ __forceinline__ uint32_t kmaj_off(int r, int k, int kdim) {
    return (uint32_t)(((r >> 3) * (kdim >> 3) + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// barrier slots (8 bytes each) after the ring's
enum UmmaBar { kBarQk = 0, kBarPv = 2, kBarConv = 4, kBarSFree = 6, kBarPReady = 8, kUmmaBars = 10 };

struct UmmaLayout {
    uint32_t misc, scales, table, ops, ring, slot_bytes, total;
};

// [barriers: ring, kUmmaBars] [TMEM address, abort flag] [token scales 2 x
// (K, V) x 32] [table] [operand tiles Q, K x2, V^T x2, P x2] [raw chunk ring].
// Total at least a 1/(n+1) share of the shared memory, so no more CTAs share
// an SM than its TMEM serves.
template <int D>
__host__ __device__ inline UmmaLayout make_umma_layout(int PT, int B) {
    constexpr int RING = umma_ring<D>();
    UmmaLayout L{};
    const int ptok = B < kChunk ? B : kChunk;
    const int pieces = (PT + ptok - 1) / ptok + 1;
    L.misc = (RING + kUmmaBars) * 8;
    L.scales = align_up(L.misc + 8, 16);
    L.table = L.scales + 2 * 2 * kChunk * 4;
    L.ops = align_up(L.table + pieces * 4, 128);
    const uint32_t ops_bytes = 128u * D * 2 + 2u * (32u * D * 2 + (uint32_t)D * 32 * 2 + 128u * 32 * 2);
    L.ring = align_up(L.ops + ops_bytes, 128);
    L.slot_bytes = align_up(2u * kChunk * (D / 4 + 1) * 4, 128);
    L.total = L.ring + RING * L.slot_bytes;
    const uint32_t floor_bytes = 232448u / (umma_ctas_per_sm<D>() + 1) + 128u;
    if (L.total < floor_bytes) L.total = floor_bytes;
    return L;
}

template <int D>
__global__ void __launch_bounds__(kUmmaThreads, umma_ctas_per_sm<D>())
decode_umma_kernel(Params P) {
    constexpr int RING = umma_ring<D>();
    constexpr int W = D / 4 + 1;
    constexpr uint32_t TCOLS = umma_tmem_cols<D>();
    constexpr uint32_t Q_BYTES = 128u * D * 2, K_BYTES = 32u * D * 2, V_BYTES = (uint32_t)D * 32 * 2;
    constexpr uint32_t P_BYTES = 128u * kChunk * 2;
    constexpr uint32_t IDESC_QK = umma_idesc_f16(128, 32), IDESC_PV = umma_idesc_f16(128, D);

    extern __shared__ __align__(128) uint8_t smem[];
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const UmmaLayout L = make_umma_layout<D>(P.PT, P.B);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const uint32_t s0 = smem_addr(smem);
    const uint32_t ring_bars = s0, bars = s0 + 8 * RING;
    auto bar = [&](int kind, int b) { return bars + 8 * (kind + b); };
    const uint32_t tmem_slot = s0 + L.misc;
    volatile uint32_t *abort = reinterpret_cast<volatile uint32_t *>(smem + L.misc + 4);
    float *ksc = reinterpret_cast<float *>(smem + L.scales);           // [2][32]
    float *vsc = ksc + 2 * kChunk;                                       // [2][32]
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    uint8_t *sQ = smem + L.ops, *sK0 = sQ + Q_BYTES, *sV0 = sK0 + 2 * K_BYTES, *sP0 = sV0 + 2 * V_BYTES;
    const uint32_t aQ = s0 + L.ops, aK0 = aQ + Q_BYTES, aV0 = aK0 + 2 * K_BYTES, aP0 = aV0 + 2 * V_BYTES;
    const uint32_t ring = s0 + L.ring;
    const uint64_t policy = l2_policy_evict_first();
    const int nquad = min(4, (w.nh + 15) / 16);         // quadrants that hold a real head
    const int nch = (w.len + kChunk - 1) / kChunk;

    if (warp == 0) tmem_alloc(tmem_slot, TCOLS);
    if (tid == 0) {
        for (int k = 0; k < RING; ++k) mbar_init(ring_bars + 8 * k, 1);
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kBarQk, b), 1);
            mbar_init(bar(kBarPv, b), 1);
            mbar_init(bar(kBarConv, b), kUmmaConvThreads);
            mbar_init(bar(kBarSFree, b), 32 * nquad);
            mbar_init(bar(kBarPReady, b), 32 * nquad);
        }
        *abort = 0u;
        fence_mbar_init();
    }
    load_table(P, w, const_cast<uint32_t *>(table));
    for (int i = tid; i < 2 * 128 * kChunk / 8; i += kUmmaThreads)    // P rows of heads that do not exist stay 0
        reinterpret_cast<uint4 *>(sP0)[i] = make_uint4(0u, 0u, 0u, 0u);

    // softmax threads: this thread's M row (virtual head hl, hi or lo part)
    const int hl = 16 * (warp & 3) + (lane & 15);
    const bool row_ok = warp < 4 && hl < w.nh;
    const int vh = w.h0 + hl;
    const bool lo_part = lane >= 16;
    const int half = lo_part ? 16 : 0;
    const int len_row = row_ok ? row_len(P, w, vh) : 0;
    const int row = 32 * (warp & 3) + lane, row_hi = 32 * (warp & 3) + (lane & 15), row_lo = row_hi + 16;
    float qk2 = 0.0f;
    if (warp < 4) {      // Q row: q * 2^-eq as hi (or lo) f16, K-major
        const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok ? vh : w.h0) * D);
        float mx = 0.0f;
        for (int c = 0; c < D / 4; ++c) {
            const float4 v = row_ok ? __ldg(qv + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);      // 2^-eq
        qk2 = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
        for (int c = 0; c < D / 8; ++c) {
            const float4 a = row_ok ? __ldg(qv + 2 * c) : make_float4(0.f, 0.f, 0.f, 0.f);
            const float4 b = row_ok ? __ldg(qv + 2 * c + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
            uint32_t h[4], l[4];
            split_f16x2(a.x * down, a.y * down, h[0], l[0]);
            split_f16x2(a.z * down, a.w * down, h[1], l[1]);
            split_f16x2(b.x * down, b.y * down, h[2], l[2]);
            split_f16x2(b.z * down, b.w * down, h[3], l[3]);
            *reinterpret_cast<uint4 *>(sQ + kmaj_off(row, 8 * c, D)) =
                lo_part ? make_uint4(l[0], l[1], l[2], l[3]) : make_uint4(h[0], h[1], h[2], h[3]);
        }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<const volatile uint32_t *>(smem + L.misc);
    const uint32_t tO = tmem + 64;

    // softmax state (warps 0-3) and the issuer's commit record (warp 7, lane 0)
    float m = -INFINITY, lsum = 0.0f;
    int E = 12;
    int last_commit = -1;            // barrier slot address offset of the newest commit, -1 none
    uint32_t last_parity = 0;
    int issued = 0;                  // chunks whose ring copy warp 7 started

    if (warp == 7) {
        // ---- ring refills and MMA issue
        for (; issued < RING && issued < nch; ++issued)
            issue_chunk<D>(P, w, table, issued, ring + issued * L.slot_bytes, ring_bars + 8 * issued, policy);
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1;
            if (!mbar_wait_abortable(bar(kBarConv, b), (i >> 1) & 1, abort)) break;    // K(i), V(i) ready
            if (issued < nch) {                                // chunk i's raw slot is free
                issue_chunk<D>(P, w, table, issued, ring + (issued % RING) * L.slot_bytes,
                               ring_bars + 8 * (issued % RING), policy);
                ++issued;
            }
            bool go = true;
            if (lane == 0) {
                if (i >= 2) go = mbar_wait_abortable(bar(kBarSFree, b), ((i - 2) >> 1) & 1, abort);
                if (go) {
                    tc_fence_after();
                    const uint32_t aK = aK0 + b * K_BYTES, tS = tmem + 32 * b;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma_f16(tS, umma_smem_desc(aQ + ks * 256, 128, D * 16),
                                 umma_smem_desc(aK + ks * 256, 128, D * 16), IDESC_QK, ks > 0);
                    umma_commit(bar(kBarQk, b));
                    last_commit = kBarQk + b;
                    last_parity = (i >> 1) & 1;
                }
                if (go && i >= 1) {                            // O += P(i-1) . V(i-1)
                    const int j = i - 1, bj = j & 1;
                    go = mbar_wait_abortable(bar(kBarPReady, bj), (j >> 1) & 1, abort);
                    if (go) {
                        tc_fence_after();
                        const uint32_t aP = aP0 + bj * P_BYTES, aV = aV0 + bj * V_BYTES;
                        umma_f16(tO, umma_smem_desc(aP, 128, 512), umma_smem_desc(aV, 128, 512), IDESC_PV, j > 0);
                        umma_f16(tO, umma_smem_desc(aP + 256, 128, 512), umma_smem_desc(aV + 256, 128, 512),
                                 IDESC_PV, true);
                        umma_commit(bar(kBarPv, bj));
                        last_commit = kBarPv + bj;
                        last_parity = (j >> 1) & 1;
                    }
                }
            }
            if (!__shfl_sync(0xFFFFFFFFu, (int)go, 0)) break;
        }
        if (lane == 0 && !*abort && nch > 0) {                // the last chunk's PV
            const int j = nch - 1, bj = j & 1;
            if (mbar_wait_abortable(bar(kBarPReady, bj), (j >> 1) & 1, abort)) {
                tc_fence_after();
                const uint32_t aP = aP0 + bj * P_BYTES, aV = aV0 + bj * V_BYTES;
                umma_f16(tO, umma_smem_desc(aP, 128, 512), umma_smem_desc(aV, 128, 512), IDESC_PV, j > 0);
                umma_f16(tO, umma_smem_desc(aP + 256, 128, 512), umma_smem_desc(aV + 256, 128, 512), IDESC_PV,
                         true);
                umma_commit(bar(kBarPv, bj));
                last_commit = kBarPv + bj;
                last_parity = (j >> 1) & 1;
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---- conversion (96 threads)
        const int ct = tid - 128;
        const F16Consts fk;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1, k = i % RING;
            const uint32_t *rawK = reinterpret_cast<const uint32_t *>(smem + L.ring + k * L.slot_bytes);
            const uint32_t *rawV = rawK + kChunk * W;
            if (!mbar_wait_abortable(ring_bars + 8 * k, (i / RING) & 1, abort)) break;
            if (i >= 2 && !mbar_wait_abortable(bar(kBarQk, b), ((i - 2) >> 1) & 1, abort)) break;   // K tile free
            uint8_t *dK = sK0 + b * K_BYTES;
            for (int u = ct; u < kChunk * D / 8; u += kUmmaConvThreads) {   // lane = token: 8 bank groups
                const int t = u % kChunk, c8 = u / kChunk;
                uint32_t a0, a1, a2, a3;
                codes4_to_f16x2(rawK[t * W + 2 * c8], a0, a1, fk);
                codes4_to_f16x2(rawK[t * W + 2 * c8 + 1], a2, a3, fk);
                *reinterpret_cast<uint4 *>(dK + kmaj_off(t, 8 * c8, D)) = make_uint4(a0, a1, a2, a3);
            }
            // V tile and scale table b free: PV(i-2) done, so softmax(i-2) is too
            if (i >= 2 && !mbar_wait_abortable(bar(kBarPv, b), ((i - 2) >> 1) & 1, abort)) break;
            if (ct < kChunk) ksc[b * kChunk + ct] = __uint_as_float(rawK[ct * W + D / 4]);
            else if (ct < 2 * kChunk) vsc[b * kChunk + ct - kChunk] = __uint_as_float(rawV[(ct - kChunk) * W + D / 4]);
            uint8_t *dV = sV0 + b * V_BYTES;
            for (int u = ct; u < D * (kChunk / 8); u += kUmmaConvThreads) {  // lane = head dim: 8 bank groups
                const int d = u % D, tg = u / D;
                const uint32_t *src = rawV + (8 * tg) * W + (d >> 2);
                const uint32_t e = (uint32_t)(d & 3);
                const uint32_t sel = e | (e << 4) | ((e + 4) << 8) | ((e + 4) << 12);
                uint32_t h[4];
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    h[j] = sub_1152_x2(and_xor_i<0x00FF00FFu>(prmt_r(src[2 * j * W], src[(2 * j + 1) * W], sel),
                                                            fk.bias),
                                       fk.bias);
                *reinterpret_cast<uint4 *>(dV + kmaj_off(d, 8 * tg, kChunk)) = make_uint4(h[0], h[1], h[2], h[3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarConv, b));
        }
    } else if (warp < nquad) {
        // ---- softmax (quadrant warp)
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        float wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
        bool ok = true;
        for (int i = 0; ok && i < nch; ++i) {
            const int b = i & 1;
            ok = mbar_wait_abortable(bar(kBarQk, b), (i >> 1) & 1, abort);
            ok = ok && mbar_wait_abortable(bar(kBarConv, b), (i >> 1) & 1, abort);     // the scale table
            if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            tc_fence_after();
            float sv[32], z[16];
            tmem_ld32(tmem + 32 * b + lane_off, sv);      // TMEM addresses are warp-uniform
            tc_fence_before();
            mbar_arrive(bar(kBarSFree, b));
#pragma unroll
            for (int j = 0; j < 16; ++j) {                // own half + the partner's row at those tokens
                const float mine = lo_part ? sv[16 + j] : sv[j], send = lo_part ? sv[j] : sv[16 + j];
                z[j] = mine + __shfl_xor_sync(0xFFFFFFFFu, send, 16);
            }
            const float *ks = ksc + b * kChunk + half, *vs = vsc + b * kChunk + half;
            const int t0 = i * kChunk + half;
            float cmax = -INFINITY, vmax = 0.0f;
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const bool valid = t0 + j < len_row;
                z[j] = valid ? z[j] * ks[j] * qk2 : -INFINITY;
                cmax = fmaxf(cmax, z[j]);
                vmax = fmaxf(vmax, valid ? vs[j] : 0.0f);
            }
            cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 16));
            vmax = fmaxf(vmax, __shfl_xor_sync(0xFFFFFFFFu, vmax, 16));
            const int Ec = (int)(__float_as_uint(vmax) >> 23);
            const bool need = cmax > m + (float)kLazy || Ec > E;
            float fa = 1.0f;
            if (need) {
                const float m_new = fmaxf(m, cmax);
                const int E_new = max(E, Ec);
                const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
                const float ea = (E - E_new < -126) ? 0.0f : __uint_as_float((uint32_t)(127 + E - E_new) << 23);
                fa = alpha * ea;
                lsum *= alpha;
                m = m_new;
                E = E_new;
                wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
            }
            if (i >= 1 && __any_sync(0xFFFFFFFFu, need)) {      // O rows once PV(i-1) is done
                ok = mbar_wait_abortable(bar(kBarPv, (i - 1) & 1), ((i - 1) >> 1) & 1, abort);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < D / 32; ++c) {
                    float o[32];
                    tmem_ld32(tO + lane_off + 32 * c, o);
#pragma unroll
                    for (int j = 0; j < 32; ++j) o[j] *= fa;
                    tmem_st32(tO + lane_off + 32 * c, o);
                }
            }
            if (i >= 2) {                                       // P tile b free: PV(i-2) done
                ok = mbar_wait_abortable(bar(kBarPv, b), ((i - 2) >> 1) & 1, abort);
                if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
            }
            const float m_ref = m == -INFINITY ? 0.0f : m;
            uint8_t *dP = sP0 + b * P_BYTES;
#pragma unroll
            for (int c = 0; c < 2; ++c) {                 // tokens half + 8c .. +7, both rows of the head
                uint32_t ph[4], pl[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int j = 8 * c + 2 * e;
                    const float p0 = fast_exp2(z[j] - m_ref), p1 = fast_exp2(z[j + 1] - m_ref);
                    lsum += p0 + p1;
                    const float w0 = t0 + j < len_row ? vs[j] : 0.0f, w1 = t0 + j + 1 < len_row ? vs[j + 1] : 0.0f;
                    split_f16x2(p0 * w0 * wscale, p1 * w1 * wscale, ph[e], pl[e]);
                }
                *reinterpret_cast<uint4 *>(dP + kmaj_off(row_hi, half + 8 * c, kChunk)) =
                    make_uint4(ph[0], ph[1], ph[2], ph[3]);
                *reinterpret_cast<uint4 *>(dP + kmaj_off(row_lo, half + 8 * c, kChunk)) =
                    make_uint4(pl[0], pl[1], pl[2], pl[3]);
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(kBarPReady, b));
        }
        // the last PV, then this warp's O rows (hi + lo) into the merge scratch
        if (ok && nch > 0) ok = mbar_wait_abortable(bar(kBarPv, (nch - 1) & 1), ((nch - 1) >> 1) & 1, abort);
        if (__all_sync(0xFFFFFFFFu, ok)) {
            tc_fence_after();
            float *ml = reinterpret_cast<float *>(sQ);                  // [64][3]   (operand tiles are free)
            float *accs = ml + kUmmaHeads * 3;                          // [64][D]
            // every PV has completed: no MMA reads the Q tile any more
            for (int c = 0; c < D / 32; ++c) {
                float o[32];
                tmem_ld32(tO + lane_off + 32 * c, o);
#pragma unroll
                for (int j = 0; j < 32; ++j) o[j] += __shfl_xor_sync(0xFFFFFFFFu, o[j], 16);
                if (!lo_part) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) accs[hl * D + 32 * c + j] = o[j];
                }
            }
            const float l_row = lsum + __shfl_xor_sync(0xFFFFFFFFu, lsum, 16);
            if (!lo_part) {
                ml[hl * 3] = m;
                ml[hl * 3 + 1] = l_row;
                ml[hl * 3 + 2] = (float)E;
            }
        } else {
            *abort = 1u;
        }
    }
    __syncthreads();
    const bool failed = *abort != 0u;
    if (failed && warp == 7 && lane == 0) {
        // stop only after the newest MMA (and so every earlier one) completed
        if (last_commit >= 0) mbar_wait(bars + 8 * last_commit, last_parity);
        for (int c = max(0, issued - RING); c < issued; ++c)     // and the ring copies in flight
            mbar_wait(ring_bars + 8 * (c % RING), (c / RING) & 1);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TCOLS);
    }
    if (failed) {
        if (tid == 0) flag_error(P.status, kDevWaitTimeout);
        return;
    }
    float *ml = reinterpret_cast<float *>(sQ);
    float *accs = ml + kUmmaHeads * 3;
    merge_and_store<D>(P, w, ml, accs, 1, kUmmaHeads, accs + kUmmaHeads * D);
}

// ============================================================== f32 cache
//
// The f32 variant of the cache, token vectors of head_size f32 values and no
// scale word: [num_blocks][Hk][B][D] f32 (the q8 layout with f32 elements;
// "paged_attn_q8.comp" names "paged_attn.comp" as the same math over an f32
// cache).  CUDA cores, with the CUDA-core family's streams, softmax and merge.
//
// Tiles move with 2-D tensor copies over the cache seen as rows of D floats:
// one box is 32 floats (128 B) of min(B, 32) rows, copied with the 128-byte
// swizzle, so 16-byte chunk c of token row t lands at chunk c ^ (t % 8) of
// that row's 128 bytes.  A chunk buffer holds [D/32 segments][32 tokens][32
// floats]; lane = token reads of one chunk index by eight lanes then touch
// eight different bank groups (the rows are 512 B apart at D = 128, which
// without the swizzle would put all of them in one bank group).
// Each warp owns chunks ts, ts + SLOTS, ...; the K and V halves of its buffer
// have their own mbarrier, so the next chunk's keys are in flight during this
// chunk's PV and its values during the next QK.

template <int D>
__host__ __device__ constexpr int f32_slots() { return D == 64 ? 8 : (D == 128 ? 6 : 3); }

constexpr uint32_t kF32SegBytes = kChunk * 128;        // one 32-float column of a chunk

struct F32Params {
    Params p;
    CUtensorMap tk;        // the key cache as [rows = num_blocks * Hk * B][D] f32
    CUtensorMap tv;
};

// shared memory beside the buffers: q rows [NH][D], weights [slot][NH][32], row lags [NH]
template <int D, int NH>
__host__ __device__ constexpr uint32_t f32_extra() { return NH * D * 4 + f32_slots<D>() * 32 * NH * 4 + NH * 4; }

struct F32Layout {
    uint32_t table, extra, ring, half_bytes, total;
};

// [barriers: slot x (K, V)] [table] [extra] [buffers, 1024-aligned: slot x (K, V)]
// (+1024 so the buffers' shared address can be rounded up to 1024)
__host__ __device__ inline F32Layout make_f32_layout(int D, int slots, int PT, int B, uint32_t extra_bytes) {
    F32Layout L{};
    const int ptok = B < kChunk ? B : kChunk;
    const int pieces = (PT + ptok - 1) / ptok + 1;
    L.table = align_up(slots * 16, 16);
    L.extra = align_up(L.table + pieces * 4, 128);
    L.ring = align_up(L.extra + extra_bytes, 1024);
    L.half_bytes = (uint32_t)kChunk * D * 4;
    L.total = L.ring + 2u * slots * L.half_bytes + 1024u;
    return L;
}

// Copy the K or V half of chunk c: lane = (piece of min(B, 32) tokens,
// 32-float column), one tensor copy each.  Pieces past the partition's end
// or in an out-of-range block are not copied (their rows are never used as
// values, or the block was flagged by the table walk).
template <int D>
__device__ __forceinline__ void issue_f32_half(const Params &P, const Work &w, const uint32_t *table,
                                               const CUtensorMap *tmap, int c, uint32_t dst, uint32_t bar,
                                               uint64_t policy) {
    constexpr int NSEG = D / 32;
    const int lane = threadIdx.x & 31;
    const int piece = lane / NSEG, seg = lane % NSEG;
    const int t = c * kChunk + (piece << P.log2ptok);      // partition-relative token
    bool go = false;
    int y = 0;
    if (piece < (kChunk >> P.log2ptok) && t < w.len) {
        const uint32_t pb = table[t >> P.log2ptok];
        if (pb != kPadSlot) {
            const int off = (w.t_begin + t) & (P.B - 1);
            y = (int)((((int64_t)pb * P.Hk + w.g) << P.log2B) + off);
            go = true;
        }
    }
    const uint32_t bytes = go ? 128u << P.log2ptok : 0u;
    const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes);
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (go) {
        fence_proxy_async_smem();
        tma_load_2d(dst + seg * kF32SegBytes + ((uint32_t)piece << P.log2ptok) * 128u, tmap, seg * 32, y,
                    bar, policy);
    }
}

template <int D, int NH>
__global__ void __launch_bounds__(f32_slots<D>() * 32, 1)
decode_f32_kernel(const __grid_constant__ F32Params FP) {
    const Params &P = FP.p;
    constexpr int SLOTS = f32_slots<D>();
    constexpr int NSEG = D / 32;
    constexpr int WORDS = D / 4;                     // 16-byte groups per row
    constexpr int LW = WORDS < 32 ? WORDS : 32;      // lanes per token row in PV
    constexpr int TG = 32 / LW;                      // token groups in PV (2 for D = 64)
    constexpr int NWL = WORDS / LW;                  // groups per lane in PV

    extern __shared__ __align__(128) uint8_t smem[];     // the buffers are aligned to 1024 at run time
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const F32Layout L = make_f32_layout(D, SLOTS, P.PT, P.B, f32_extra<D, NH>());
    const int ts = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t s0 = smem_addr(smem);
    const uint32_t kbar = s0 + 16 * ts, vbar = kbar + 8;
    const uint32_t ring = (s0 + L.ring + 1023u) & ~1023u;
    const uint32_t kbuf = ring + 2u * ts * L.half_bytes, vbuf = kbuf + L.half_bytes;
    const float *sK = reinterpret_cast<const float *>(smem + (kbuf - s0));
    const float *sV = reinterpret_cast<const float *>(smem + (vbuf - s0));
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    float *sq = reinterpret_cast<float *>(smem + L.extra);                  // [NH][D]
    float *myw = sq + NH * D + ts * 32 * NH;                                // [NH][32]
    int *slag = reinterpret_cast<int *>(sq + NH * D + SLOTS * 32 * NH);     // [NH]
    const int nchunks = (w.len + kChunk - 1) / kChunk;
    const int my_n = ts < nchunks ? (nchunks - ts + SLOTS - 1) / SLOTS : 0;
    const uint64_t policy = l2_policy_evict_first();

    if (lane == 0) {
        mbar_init(kbar, 1);
        mbar_init(vbar, 1);
        fence_mbar_init();
    }
    load_table(P, w, const_cast<uint32_t *>(table));
    for (int i = threadIdx.x; i < NH * D; i += blockDim.x) {
        const int hh = i / D;
        sq[i] = hh < w.nh ? __ldg(P.q + qrow(P, w, w.h0 + hh) * D + (i % D)) : 0.0f;
    }
    if (threadIdx.x < NH)
        slag[threadIdx.x] = (int)threadIdx.x < w.nh ? P.R - 1 - (w.h0 + (int)threadIdx.x) / P.r : INT_MAX;
    __syncthreads();
    int k_issued = 0, v_issued = 0, k_done = 0, v_done = 0;
    if (my_n > 0) {
        issue_f32_half<D>(P, w, table, &FP.tk, ts, kbuf, kbar, policy);
        issue_f32_half<D>(P, w, table, &FP.tv, ts, vbuf, vbar, policy);
        k_issued = v_issued = 1;
    }

    const float4 *sq4 = reinterpret_cast<const float4 *>(sq);
    float m[NH], lsum[NH], acc[NH][NWL][4];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        m[hh] = -INFINITY;
        lsum[hh] = 0.0f;
#pragma unroll
        for (int u = 0; u < NWL; ++u) acc[hh][u][0] = acc[hh][u][1] = acc[hh][u][2] = acc[hh][u][3] = 0.0f;
    }

    bool ok = true;
    const int rsw = lane & 7;                        // swizzle phase of this lane's row in QK
    for (int i = 0; i < my_n; ++i) {
        const int c = ts + SLOTS * i;
        const int t0 = c * kChunk;
        if (!mbar_wait(kbar, i & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        ++k_done;
        // ---- logits, lane = token
        const bool valid = t0 + lane < w.len;
        const int ahead = w.c - w.t_begin - t0 - lane;         // tokens from this one to the context end
        float dot[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) dot[hh] = 0.0f;
        const float *krow = sK + lane * 32;
#pragma unroll
        for (int sg = 0; sg < NSEG; ++sg) {
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 kv = *reinterpret_cast<const float4 *>(krow + sg * (kChunk * 32) + ((q4 ^ rsw) << 2));
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const float4 qv = sq4[hh * WORDS + sg * 8 + q4];
                    dot[hh] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, fmaf(qv.w, kv.w, dot[hh]))));
                }
            }
        }
        __syncwarp();
        if (i + 1 < my_n) {            // keys consumed: the next chunk's keys into the same half
            issue_f32_half<D>(P, w, table, &FP.tk, c + SLOTS, kbuf, kbar, policy);
            ++k_issued;
        }
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) {
            const bool seen = valid && slag[hh] < ahead;      // causal limit of this query row
            const float z = seen ? dot[hh] * P.scale_log2 : -INFINITY;
            float cm = z;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
            const float m_new = fmaxf(m[hh], cm);
            if (m_new != m[hh]) {        // warp-uniform
                const float alpha = (m[hh] == -INFINITY) ? 0.0f : fast_exp2(m[hh] - m_new);
                lsum[hh] *= alpha;
#pragma unroll
                for (int u = 0; u < NWL; ++u) {
                    acc[hh][u][0] *= alpha; acc[hh][u][1] *= alpha;
                    acc[hh][u][2] *= alpha; acc[hh][u][3] *= alpha;
                }
                m[hh] = m_new;
            }
            const float p = seen ? fast_exp2(z - m[hh]) : 0.0f;
            lsum[hh] += p;
            myw[hh * 32 + lane] = p;
        }
        __syncwarp();
        if (!mbar_wait(vbar, i & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        ++v_done;
        // ---- weighted sum, lane = 4 head dims; only tokens inside the context
        const int ntok = min(kChunk, w.len - t0);
        const int tg = lane / LW, lw = lane % LW;
#pragma unroll 2
        for (int tt = tg; tt < ntok; tt += TG) {
            const float *vrow = sV + tt * 32;
            float4 v[NWL];
#pragma unroll
            for (int u = 0; u < NWL; ++u) {
                const int g4 = lw + 32 * u;                     // 16-byte group: column g4 / 8, chunk g4 % 8
                v[u] = *reinterpret_cast<const float4 *>(vrow + (g4 >> 3) * (kChunk * 32) +
                                                         (((g4 & 7) ^ (tt & 7)) << 2));
            }
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float wt = myw[hh * 32 + tt];
#pragma unroll
                for (int u = 0; u < NWL; ++u) {
                    acc[hh][u][0] = fmaf(wt, v[u].x, acc[hh][u][0]);
                    acc[hh][u][1] = fmaf(wt, v[u].y, acc[hh][u][1]);
                    acc[hh][u][2] = fmaf(wt, v[u].z, acc[hh][u][2]);
                    acc[hh][u][3] = fmaf(wt, v[u].w, acc[hh][u][3]);
                }
            }
        }
        __syncwarp();
        if (i + 1 < my_n) {
            issue_f32_half<D>(P, w, table, &FP.tv, c + SLOTS, vbuf, vbar, policy);
            ++v_issued;
        }
    }
    // a warp leaves only after every copy it issued has landed (bounded)
    if (lane == 0) {
        for (; k_done < k_issued; ++k_done)
            if (!mbar_wait(kbar, k_done & 1)) { flag_error(P.status, kDevWaitTimeout); break; }
        for (; v_done < v_issued; ++v_done)
            if (!mbar_wait(vbar, v_done & 1)) { flag_error(P.status, kDevWaitTimeout); break; }
    }

    if (__syncthreads_or(!ok)) return;
    float *ml = reinterpret_cast<float *>(smem + L.ring);      // [slot][NH][3]
    float *accs = ml + SLOTS * NH * 3;                          // [slot][NH][D]
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        float l = lsum[hh];
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
#pragma unroll
        for (int u = 0; u < NWL; ++u) {
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                float a = acc[hh][u][e];
                if constexpr (TG == 2) a += __shfl_xor_sync(0xFFFFFFFFu, a, 16);
                acc[hh][u][e] = a;
            }
        }
        if (lane == 0) {
            float *e = ml + (ts * NH + hh) * 3;
            e[0] = m[hh]; e[1] = l; e[2] = (float)kVScaleBias;
        }
        if (lane < LW) {
#pragma unroll
            for (int u = 0; u < NWL; ++u) {
                float *dst = accs + (ts * NH + hh) * D + 4 * (lane + 32 * u);
                dst[0] = acc[hh][u][0]; dst[1] = acc[hh][u][1];
                dst[2] = acc[hh][u][2]; dst[3] = acc[hh][u][3];
            }
        }
    }
    __syncthreads();
    merge_and_store<D>(P, w, ml, accs, SLOTS, NH, accs + SLOTS * NH * D);
}

// ==================================================================== prep
//
// One CTA before the attention grid: zero the split-context arrival
// counters and order the sequences longest (clamped) context first, so the
// block scheduler starts the longest-running CTAs first and the grid's tail
// holds only short ones.  (length, index) keys in shared memory: ranked by
// counting for up to blockDim sequences, bitonic-sorted up to kPrepMaxSort;
// beyond that the order is the identity.
constexpr int kPrepThreads = 1024;
constexpr int kPrepMaxSort = 8192;

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const uint32_t *context_lens, int S, int64_t cap,
                                                            unsigned long long *order, uint32_t *counters,
                                                            int64_t n_counters) {
    extern __shared__ unsigned long long keys[];
    // the attention grid may launch now; it waits for this grid's writes
    grid_dependents_launch();
    for (int64_t i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
    if (S > kPrepMaxSort) {
        for (int i = threadIdx.x; i < S; i += blockDim.x) {
            const int64_t c = min((int64_t)__ldg(context_lens + i), cap);
            order[i] = ((unsigned long long)c << 32) | (unsigned)i;
        }
        return;
    }
    int n = 1;
    while (n < S) n <<= 1;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        if (i < S) {
            const int64_t c = min((int64_t)__ldg(context_lens + i), cap);
            keys[i] = ((unsigned long long)(cap - c) << 32) | (unsigned)i;   // ascending = longest first
        } else {
            keys[i] = ~0ull;
        }
    }
    __syncthreads();
    if (S <= (int)blockDim.x) {
        // G threads per sequence (a power of two, at most a warp): each counts
        // the smaller keys (all distinct) in its stride of the S keys, the
        // group sums them into the sequence's rank
        int G = 1;
        while (G < 32 && 2 * G * S <= (int)blockDim.x) G <<= 1;
        const int i = threadIdx.x / G, part = threadIdx.x % G;
        int rank = 0;
        const unsigned long long mine = i < S ? keys[i] : 0ull;
        if (i < S) {
#pragma unroll 8
            for (int j = part; j < S; j += G) rank += keys[j] < mine;
        }
        for (int o = G >> 1; o > 0; o >>= 1) rank += __shfl_xor_sync(0xFFFFFFFFu, rank, o);
        if (i < S && part == 0)
            order[rank] = ((unsigned long long)(cap - (int64_t)(mine >> 32)) << 32) | (unsigned)i;
        return;
    }
    // bitonic sort of the n (power of two) keys, ascending
    for (int k = 2; k <= n; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < n; i += blockDim.x) {
                const int l = i ^ j;
                if (l > i) {
                    const unsigned long long a = keys[i], b = keys[l];
                    if ((a > b) == ((i & k) == 0)) {
                        keys[i] = b;
                        keys[l] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    for (int i = threadIdx.x; i < S; i += blockDim.x)
        order[i] = ((unsigned long long)(cap - (int64_t)(keys[i] >> 32)) << 32) | (keys[i] & 0xFFFFFFFFull);
}

// ============================================================== selftest
__global__ void wait_selftest_kernel(uint64_t limit_ns, uint32_t *status) {
    __shared__ __align__(8) uint64_t bar;
    const uint32_t b = smem_addr(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // nothing arrives on this barrier: the wait must give up
        if (!mbar_wait(b, 0, limit_ns)) flag_error(status, kDevWaitTimeout);
    }
}

// ================================================================== launch

Params make_params(const DecodeArgs &a) {
    Params P{};
    P.out = a.out; P.q = a.q; P.kc = a.key_cache; P.vc = a.value_cache;
    P.bt = a.block_tables; P.cl = a.context_lens;
    P.S = a.num_seqs; P.H = a.num_heads; P.Hk = a.num_kv_heads; P.B = a.block_size;
    P.log2B = 0;
    while ((1 << P.log2B) < a.block_size) ++P.log2B;
    P.log2ptok = P.log2B < 5 ? P.log2B : 5;
    P.Nb = a.max_blocks_per_seq; P.num_blocks = a.num_blocks;
    P.scale_log2 = a.scale * kLog2e;
    P.PT = a.partition_tokens; P.NP = a.num_partitions;
    P.r = a.num_heads / a.num_kv_heads;
    P.R = a.num_rows;
    P.rv = P.R * P.r;
    P.heads_per_cta = a.heads_per_cta; P.head_groups = a.head_groups;
    P.order = a.order; P.counters = a.counters; P.pml = a.partial_ml; P.pacc = a.partial_acc; P.status = a.status;
    P.nk = a.new_key; P.nv = a.new_value;
    P.nk_stride = a.new_key_stride; P.nv_stride = a.new_value_stride;
    P.contiguous = a.contiguous;
    P.kc_w = const_cast<uint32_t *>(a.key_cache);      // written only by the fused append
    P.vc_w = const_cast<uint32_t *>(a.value_cache);
    return P;
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

// cuTensorMapEncodeTiled, looked up once through the runtime (no link
// against the driver library).
using EncodeTiledFn = PFN_cuTensorMapEncodeTiled_v12000;

EncodeTiledFn tensor_map_encoder() {
    static const EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}

// An f32 cache [num_blocks * Hk * B rows][D] as a 2-D tensor with boxes of
// 32 floats x min(B, 32) rows and the 128-byte swizzle.
bool encode_f32_cache_map(CUtensorMap *map, const void *cache, int64_t rows, int D, int ptok) {
    const EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)D, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)D * 4u};
    const cuuint32_t box[2] = {32u, (cuuint32_t)ptok};
    const cuuint32_t elem[2] = {1u, 1u};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(cache), dims, strides, box, elem,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Tensor maps of one contiguous cache (head size 128): codes as u8
// [S][max_t][kv_row], scales as f32 [S][max_t][kv_row / 32].
bool encode_cq_maps(CUtensorMap *codes, CUtensorMap *scales, const void *cache, int S, int64_t max_t, int Hk) {
    const EncodeTiledFn enc = tensor_map_encoder();
    if (!enc) return false;
    const int64_t kv_row = (int64_t)Hk * 128;
    const uint64_t seq_bytes = (uint64_t)(max_t * kv_row + max_t * (kv_row / 32) * 4);
    const cuuint32_t elem[3] = {1u, 1u, 1u};
    {
        const cuuint64_t dims[3] = {(cuuint64_t)kv_row, (cuuint64_t)max_t, (cuuint64_t)S};
        const cuuint64_t strides[2] = {(cuuint64_t)kv_row, seq_bytes};
        const cuuint32_t box[3] = {128u, (cuuint32_t)kChunk, 1u};
        if (enc(codes, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(cache), dims, strides, box, elem,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    {
        const void *sbase = static_cast<const uint8_t *>(cache) + max_t * kv_row;
        const cuuint64_t dims[3] = {(cuuint64_t)(kv_row / 32), (cuuint64_t)max_t, (cuuint64_t)S};
        const cuuint64_t strides[2] = {(cuuint64_t)(kv_row / 32) * 4u, seq_bytes};
        const cuuint32_t box[3] = {4u, (cuuint32_t)kChunk, 1u};
        if (enc(scales, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void *>(sbase), dims, strides, box, elem,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

cudaError_t launch_cq_tma(const Params &P, cudaStream_t st) {
    CqTmaParams CP;
    std::memset(&CP, 0, sizeof CP);
    CP.p = P;
    if (!encode_cq_maps(&CP.kcodes, &CP.kscales, P.kc, P.S, P.Nb, P.Hk) ||
        !encode_cq_maps(&CP.vcodes, &CP.vscales, P.vc, P.S, P.Nb, P.Hk))
        return cudaErrorNotSupported;
    return launch_attn_arg(decode_cq_tma_kernel<128>, P, CP, cq_tma_smem_bytes(), PA_Q8_TC_SLOTS * 32, st);
}

template <int D, int NH>
cudaError_t launch_f32_nh(const F32Params &FP, cudaStream_t st) {
    const F32Layout L = make_f32_layout(D, f32_slots<D>(), FP.p.PT, FP.p.B, f32_extra<D, NH>());
    return launch_attn_arg(decode_f32_kernel<D, NH>, FP.p, FP, L.total, f32_slots<D>() * 32, st);
}

template <int D>
cudaError_t launch_f32(const Params &P, cudaStream_t st) {
    F32Params FP;
    std::memset(&FP, 0, sizeof FP);
    FP.p = P;
    const int64_t rows = P.num_blocks * P.Hk * P.B;
    const int ptok = 1 << P.log2ptok;
    if (!encode_f32_cache_map(&FP.tk, P.kc, rows, D, ptok) || !encode_f32_cache_map(&FP.tv, P.vc, rows, D, ptok))
        return cudaErrorNotSupported;
    switch (P.heads_per_cta) {
        case 1: return launch_f32_nh<D, 1>(FP, st);
        case 2: return launch_f32_nh<D, 2>(FP, st);
        case 4: return launch_f32_nh<D, 4>(FP, st);
        case 8: return launch_f32_nh<D, 8>(FP, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_tc(const Params &P, cudaStream_t st) {
    constexpr int SLOTS = PA_Q8_TC_SLOTS;
    constexpr int RING = tc_ring<D>();
    if constexpr (D == 256) {       // 16-head CTAs: head size 256 only (make_plan)
        if (P.heads_per_cta > 8) {
            const Layout L = make_layout(D, SLOTS, RING, P.PT, P.B, tc_extra_bytes<D, 2>());
            return launch_attn(decode_tc_kernel<D, 2>, P, L.total, 2 * SLOTS * 32, st);
        }
    }
    const Layout L = make_layout(D, SLOTS, RING, P.PT, P.B, tc_extra_bytes<D, 1>());
    return launch_attn(decode_tc_kernel<D, 1>, P, L.total, SLOTS * 32, st);
}

template <int D, int NH>
cudaError_t launch_cc_nh(const Params &P, cudaStream_t st) {
    const Layout L = make_layout(D, kCcSlots, cc_ring<D>(), P.PT, P.B, cc_extra<D, NH>());
    return launch_attn(decode_cc_kernel<D, NH>, P, L.total, kCcSlots * 32, st);
}

template <int D>
cudaError_t launch_cc(const Params &P, cudaStream_t st) {
    switch (P.heads_per_cta) {
        case 1: return launch_cc_nh<D, 1>(P, st);
        case 2: return launch_cc_nh<D, 2>(P, st);
        case 4: return launch_cc_nh<D, 4>(P, st);
        case 8: return launch_cc_nh<D, 8>(P, st);
        case 16: return launch_cc_nh<D, 16>(P, st);
        default: return cudaErrorInvalidValue;
    }
}

template <int D>
cudaError_t launch_d(const Params &P, int kernel, cudaStream_t st) {
    if (P.order) {
        const int64_t n_counters = P.NP > 1 ? (int64_t)P.S * P.Hk * P.head_groups : 0;
        int n = 1;
        while (n < P.S && n < kPrepMaxSort) n <<= 1;
        const size_t smem = (size_t)n * sizeof(unsigned long long);
        cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        prep_kernel<<<1, kPrepThreads, smem, st>>>(P.cl, P.S, (int64_t)P.Nb * P.B,
                                                   const_cast<unsigned long long *>(P.order),
                                                   P.counters, n_counters);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (kernel == kF32) return launch_f32<D>(P, st);
    if (P.contiguous) {
        if constexpr (D == 64) {
            return cudaErrorInvalidValue;                 // head sizes 128 and 256 only
        } else if constexpr (D == 128) {
            return launch_cq_tma(P, st);
        } else {
            const CqLayout L = make_cq_layout<D>();
            return launch_attn(decode_cq_kernel<D>, P, L.total, PA_Q8_TC_SLOTS * 32, st);
        }
    }
    if (kernel == kTcgen05) {
        const UmmaLayout L = make_umma_layout<D>(P.PT, P.B);
        return launch_attn(decode_umma_kernel<D>, P, L.total, kUmmaThreads, st);
    }
    return (kernel == kCudaCore) ? launch_cc<D>(P, st) : launch_tc<D>(P, st);
}

}  // namespace

bool make_plan(DecodeArgs &a, int requested_kernel, int requested_partition, int num_sms) {
    if (a.num_rows < 1) a.num_rows = 1;
    // (query row, head) pairs served per kv head: the rows of one sequence
    // share their kv group's K/V read like the heads of a GQA group
    const int r = a.num_rows * (a.num_heads / a.num_kv_heads);
    // automatic: tcgen05 when a kv head has enough (row, head) pairs to fill
    // its CTAs (64 each); the mma.sync tensor-core family otherwise
    a.kernel = requested_kernel != kAuto ? requested_kernel : (r >= kUmmaHeads ? kTcgen05 : kTensorCore);
    if (a.kernel == kTcgen05) {
        a.heads_per_cta = r < kUmmaHeads ? r : kUmmaHeads;
    } else if (a.kernel == kTensorCore && a.contiguous) {
        a.heads_per_cta = r < 8 ? r : 8;                  // the contiguous-cache kernel: one head tile
    } else if (a.kernel == kTensorCore) {
        const int cap = a.head_size == 256 ? 16 : PA_Q8_TC_MAX_HEADS;
        a.heads_per_cta = r < cap ? r : cap;
    } else {
        int hp = a.kernel == kF32 ? 8 : 16;
        while (hp > 1 && (r % hp) != 0) hp >>= 1;
        a.heads_per_cta = hp;
    }
    a.head_groups = (r + a.heads_per_cta - 1) / a.heads_per_cta;
    const int64_t max_ctx = (int64_t)a.max_blocks_per_seq * a.block_size;
    int pt = requested_partition;
    if (pt <= 0) {
        // CTAs resident per SM for this kernel configuration
        const int hd = a.head_size;
        const bool big_tile = hd == 256 || a.heads_per_cta > 8;
        const int per_sm = a.contiguous          ? (hd == 256 ? 1 : 2)
                           : a.kernel == kF32       ? 1
                           : a.kernel == kTcgen05 ? (hd == 256 ? 1 : 2)
                           : a.kernel == kCudaCore ? (hd == 256 ? 1 : 2)
                                                   : (big_tile ? 1 : 3);
        const int64_t slots = (int64_t)per_sm * num_sms;
        const int64_t units = (int64_t)a.num_seqs * a.num_kv_heads * a.head_groups;
        if (units >= slots) {
            // Enough (sequence, kv head) work items: one partition per context
            // (up to 8192 tokens).  The grid runs the longest contexts first,
            // so the tail holds short ones.
            pt = (int)std::min<int64_t>((max_ctx + 127) / 128 * 128, 8192);
        } else {
            // Few, long contexts: split so that the expected work (contexts
            // taken at half their maximum) fills about two waves of resident
            // CTAs (one wave for one-CTA-per-SM kernels), rounded to the
            // nearest power of two in 256 .. 8192 tokens.
            const int64_t waves = per_sm > 1 ? 2 : 1;
            const double want = (double)units * (double)max_ctx / 2.0 / (double)(waves * slots);
            pt = 256;
            while (pt < 8192 && (double)pt * 1.4142135 < want) pt <<= 1;
        }
    }
    if (pt % 128 != 0 || pt > 16384) return false;
    a.partition_tokens = pt;
    const int64_t np = (max_ctx + pt - 1) / pt;
    if (np > 0x7FFFFFFF || np < 1) return false;
    a.num_partitions = (int)np;
    {
        const int hd = a.head_size;
        const bool big_tile = hd == 256 || a.heads_per_cta > 8;
        const int per_sm = a.contiguous          ? (hd == 256 ? 1 : 2)
                           : a.kernel == kF32       ? 1
                           : a.kernel == kTcgen05 ? (hd == 256 ? 1 : 2)
                           : a.kernel == kCudaCore ? (hd == 256 ? 1 : 2)
                                                   : (big_tile ? 1 : 3);
        a.one_wave = np == 1 && (int64_t)a.num_seqs * a.num_kv_heads * a.head_groups <= (int64_t)per_sm * num_sms;
    }
    return true;
}

namespace {
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
}

size_t plan_workspace_bytes(const DecodeArgs &a) {
    const size_t order = round256((size_t)a.num_seqs * sizeof(unsigned long long));
    if (a.num_partitions <= 1) return order;
    const size_t groups = (size_t)a.num_seqs * a.num_kv_heads * a.head_groups;
    const size_t rows = (size_t)a.num_seqs * a.num_rows * a.num_heads * a.num_partitions;
    return order + round256(groups * sizeof(uint32_t)) + round256(rows * 2 * sizeof(float)) +
           rows * a.head_size * sizeof(float);
}

void plan_workspace_layout(DecodeArgs &a, void *workspace) {
    char *p = static_cast<char *>(workspace);
    a.order = reinterpret_cast<unsigned long long *>(p);
    p += round256((size_t)a.num_seqs * sizeof(unsigned long long));
    if (a.num_partitions <= 1) return;
    const size_t groups = (size_t)a.num_seqs * a.num_kv_heads * a.head_groups;
    const size_t rows = (size_t)a.num_seqs * a.num_rows * a.num_heads * a.num_partitions;
    a.counters = reinterpret_cast<uint32_t *>(p);
    p += round256(groups * sizeof(uint32_t));
    a.partial_ml = reinterpret_cast<float *>(p);
    p += round256(rows * 2 * sizeof(float));
    a.partial_acc = reinterpret_cast<float *>(p);
}

int64_t plan_num_ctas(const DecodeArgs &a) {
    return (int64_t)a.num_partitions * a.num_kv_heads * a.head_groups * a.num_seqs;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    Params P = make_params(a);
    if (a.one_wave) P.order = nullptr;       // every CTA starts at once: no order, no prep kernel
    switch (a.head_size) {
        case 64: return launch_d<64>(P, a.kernel, stream);
        case 128: return launch_d<128>(P, a.kernel, stream);
        case 256: return launch_d<256>(P, a.kernel, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_wait_selftest(uint32_t timeout_us, uint32_t *status, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>((uint64_t)timeout_us * 1000ull, status);
    return cudaGetLastError();
}

}  // namespace pa_q8
