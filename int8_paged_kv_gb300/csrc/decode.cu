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
// group's K/V.  A producer warp walks the block table and copies whole
// (block, kv head) tiles -- block_size * (head_size + 4) contiguous bytes --
// with 1-D bulk copies (cp.async.bulk) into a ring of shared-memory stages
// guarded by mbarriers; consumer warps dequantise in registers and run a
// single-pass online softmax.  Two consumer families:
//   * tensor core: per 16-token chunk, S = Q K^T and O += P V as
//     mma.sync m16n8k16 f16 tiles; q and P enter as hi + lo f16 pairs
//     (rows 0-7 = hi, rows 8-15 = lo), int8 codes are exact in f16;
//   * CUDA core: f32 FMA dot products (lane = token) and weighted sums
//     (lane = 4 head dims).
// Every wait is bounded; a wait that gives up flags the status word and the
// CTA leaves after the copies it issued have landed.
#include <cfloat>
#include <cstdint>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"

namespace pa_q8 {
namespace {

constexpr float kLog2e = 1.4426950408889634f;
constexpr int kConsumerWarpsPerTile = 4;   // token slots per head tile
constexpr int kTcTokensPerStage = 64;      // 4 warps x 16-token chunks
constexpr int kCcTokensPerStage = 128;     // 4 warps x 32-token chunks
constexpr int kVScaleBias = 139;           // weights carry 2^(139 - E): below 2^13

struct Params {
    float *out;
    const float *q;
    const uint32_t *kc;
    const uint32_t *vc;
    const uint32_t *bt;
    const uint32_t *cl;
    int S, H, Hk, B, Nb;
    int64_t num_blocks;
    float scale_log2;       // scale * log2(e)
    int PT;                 // tokens per partition
    int NP;                 // partitions per sequence (grid x)
    int r;                  // num_heads / num_kv_heads
    int heads_per_cta;
    int head_groups;
    float *pml;             // [S][H][NP][2]
    float *pacc;            // [S][H][NP][D]
    uint32_t *status;
};

// Which CTA this is and the token range it owns.
struct Work {
    int s, g, h0, nh, p;
    int c;          // clamped context length
    int t_begin;    // first logical token of the partition
    int len;        // tokens in the partition
    bool single;    // the partition is the whole context
};

__device__ __forceinline__ bool setup_work(const Params &P, Work &w) {
    w.p = blockIdx.x;
    w.s = blockIdx.z;
    w.g = blockIdx.y / P.head_groups;
    const int hg = blockIdx.y % P.head_groups;
    w.h0 = w.g * P.r + hg * P.heads_per_cta;
    w.nh = min(P.heads_per_cta, P.r - hg * P.heads_per_cta);
    const int64_t cap = (int64_t)P.Nb * P.B;
    const int64_t craw = __ldg(P.cl + w.s);
    w.c = (int)(craw < cap ? craw : cap);
    w.t_begin = w.p * P.PT;
    w.len = min(w.c - w.t_begin, P.PT);
    w.single = w.c <= P.PT;
    return w.len > 0;
}

// Zero output rows of a sequence whose context is empty (partition 0 only).
template <int D>
__device__ void write_zero_rows(const Params &P, const Work &w) {
    if (w.p != 0 || w.c != 0) return;
    for (int i = threadIdx.x; i < w.nh * D; i += blockDim.x) {
        const int hh = i / D, d = i % D;
        P.out[((int64_t)w.s * P.H + w.h0 + hh) * D + d] = 0.0f;
    }
}

// Shared-memory layout, in bytes from the (128-aligned) dynamic base.
struct Layout {
    uint32_t bars;       // full[NST], empty[NST]
    uint32_t table;      // physical block of each piece of the partition
    uint32_t extra;      // kernel-specific (CUDA core: q and weights)
    uint32_t stages;     // ring
    uint32_t stage_bytes;
    uint32_t total;
};

__host__ __device__ constexpr uint32_t align_up(uint32_t x, uint32_t a) { return (x + a - 1) / a * a; }

__host__ __device__ inline Layout make_layout(int D, int TPS, int NST, int PT, int B, uint32_t extra_bytes) {
    Layout L{};
    const int W = D / 4 + 1;
    const int ptok = B < TPS ? B : TPS;
    const int pieces = (PT + ptok - 1) / ptok + 1;
    L.bars = 0;
    L.table = align_up(2 * NST * 8, 16);
    L.extra = align_up(L.table + pieces * 4, 128);
    L.stages = align_up(L.extra + extra_bytes, 128);
    L.stage_bytes = align_up(2u * TPS * W * 4, 128);
    L.total = L.stages + NST * L.stage_bytes;
    return L;
}

// ------------------------------------------------------------------ producer
//
// The partition is cut into stages of TPS tokens; each stage is
// max(1, TPS / B) pieces of min(B, TPS) tokens, each piece one contiguous
// run of a (block, kv head) tile.  Lane i of the producer warp copies piece
// i of a stage (K and V), after lane 0 has announced the stage's bytes.
template <int D, int TPS, int NST>
__device__ void producer(const Params &P, const Work &w, uint8_t *smem, const Layout &L,
                         int n_stages, volatile int *abort_flag) {
    constexpr int W = D / 4 + 1;
    const int lane = threadIdx.x & 31;
    const int ptok = P.B < TPS ? P.B : TPS;
    const int pieces_per_stage = TPS / ptok;
    const uint32_t piece_bytes = (uint32_t)ptok * W * 4;
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    const uint32_t bars = smem_addr(smem + L.bars);
    const uint32_t ring = smem_addr(smem + L.stages);
    const uint64_t policy = l2_policy_evict_first();
    const int64_t head_tile_words = (int64_t)P.B * W;      // one (block, kv head) tile
    int issued = 0;

    for (int j = 0; j < n_stages; ++j) {
        const int k = j % NST;
        const uint32_t full = bars + 8 * k, empty = bars + 8 * (NST + k);
        if (j >= NST) {
            bool ok = true;
            if (lane == 0) ok = mbar_wait(empty, ((j / NST) - 1) & 1);
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok || *abort_flag) {
                if (lane == 0) { *abort_flag = 1; flag_error(P.status, kDevWaitTimeout); }
                break;
            }
        }
        uint32_t bytes = 0;
        const uint32_t *src_k = nullptr, *src_v = nullptr;
        const int t = j * TPS + lane * ptok;             // first token of my piece (partition-relative)
        if (lane < pieces_per_stage && t < w.len) {
            const int tabs = w.t_begin + t;              // logical token in the sequence
            const uint32_t pb = table[t / ptok];
            if (pb != kPadSlot) {
                const int64_t base = ((int64_t)pb * P.Hk + w.g) * head_tile_words + (int64_t)(tabs % P.B) * W;
                src_k = P.kc + base;
                src_v = P.vc + base;
                bytes = piece_bytes;
            }
        }
        const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes) * 2u;
        if (lane == 0) mbar_arrive_expect_tx(full, total);
        __syncwarp();
        if (bytes) {
            const uint32_t dst = ring + k * L.stage_bytes + lane * piece_bytes;
            bulk_copy_g2s(dst, src_k, bytes, full, policy);
            bulk_copy_g2s(dst + TPS * W * 4, src_v, bytes, full, policy);
        }
        issued = j + 1;
    }
    // Leave only once every copy this warp issued has landed in shared memory.
    if (lane == 0) {
        const int first = issued > NST ? issued - NST : 0;
        for (int j = first; j < issued; ++j) {
            if (!mbar_wait(bars + 8 * (j % NST), (j / NST) & 1)) {
                flag_error(P.status, kDevWaitTimeout);
                break;
            }
        }
    }
}

// Load the partition's block-table slice into shared memory (one entry per
// piece); entries out of range become kPadSlot and are flagged.
template <int TPS>
__device__ void load_table(const Params &P, const Work &w, uint32_t *table) {
    const int ptok = P.B < TPS ? P.B : TPS;
    const int n = (w.len + ptok - 1) / ptok;
    const uint32_t *row = P.bt + (int64_t)w.s * P.Nb;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
        const int tabs = w.t_begin + i * ptok;
        uint32_t pb = __ldg(row + tabs / P.B);
        if ((int64_t)pb >= P.num_blocks) {
            flag_error(P.status, kDevBadBlock);
            pb = kPadSlot;
        }
        table[i] = pb;
    }
}

__device__ __forceinline__ void init_barriers(uint32_t bars, int nst, int consumer_warps) {
    if (threadIdx.x == 0) {
        for (int k = 0; k < nst; ++k) {
            mbar_init(bars + 8 * k, 1);
            mbar_init(bars + 8 * (nst + k), consumer_warps);
        }
        fence_mbar_init();
    }
}

// ----------------------------------------------------------------- epilogue
//
// Merge the per-warp online-softmax states of the CTA (m in log2 units, l,
// acc scaled by 2^(E - 139)) and write the output rows, or this
// partition's partial (M, L, A) for the combine kernel.
template <int D>
__device__ void merge_and_store(const Params &P, const Work &w, const float *ml, const float *accs,
                                int n_slots, int heads_per_slotgroup, int nthreads) {
    // ml: [slot][head][3] = (m, l, E); accs: [slot][head][D]; slot = warp's token slot
    // within its head tile; head = CTA-local head index.
    const int tid = threadIdx.x;
    for (int i = tid; i < w.nh * D; i += nthreads) {
        const int hh = i / D, d = i % D;
        float M = -INFINITY;
        for (int sl = 0; sl < n_slots; ++sl) M = fmaxf(M, ml[(sl * heads_per_slotgroup + hh) * 3]);
        float Lsum = 0.0f, A = 0.0f;
        if (M != -INFINITY) {
            for (int sl = 0; sl < n_slots; ++sl) {
                const float *e = ml + (sl * heads_per_slotgroup + hh) * 3;
                if (e[0] == -INFINITY) continue;
                const float wgt = fast_exp2(e[0] - M);
                const int E = __float2int_rn(e[2]);
                const float unscale = ldexpf(1.0f, E - kVScaleBias);
                Lsum += e[1] * wgt;
                A += accs[(sl * heads_per_slotgroup + hh) * D + d] * (wgt * unscale);
            }
        }
        const int h = w.h0 + hh;
        if (w.single) {
            P.out[((int64_t)w.s * P.H + h) * D + d] = A / Lsum;
        } else {
            const int64_t row = ((int64_t)w.s * P.H + h) * P.NP + w.p;
            P.pacc[row * D + d] = A;
            if (d == 0) {
                P.pml[row * 2] = M;
                P.pml[row * 2 + 1] = Lsum;
            }
        }
    }
}

// ============================================================ tensor cores
//
// Consumer warp (head tile ht, token slot ts) owns query heads
// h0 + 8 ht + (0..7) and, in every stage, the 16-token chunks ts, ts+4, ...
// Fragment coordinates: gq = lane / 4 (row group), cq = lane % 4.
//
// K dimension of S = Q K^T: k-step ks uses, for lane column cq, code word
// kword(cq, ks) of the token row -- 4 consecutive head dims in one u32.  The
// A fragment (q) follows the same dimension order, so the sum is the plain
// dot product.  Rows gq and gq + 8 of A are hi and lo f16 parts of head gq.
//
// N dimension of O = P V: the V words of four tokens at word vword(gq, jj)
// give, byte lane e, the B fragments of n-tile 4 jj + e; output column n of
// n-tile i is head dim 4 * vword(n, i / 4) + i % 4.  Both word maps visit
// every word once and make the shared-memory reads of a warp hit 32
// distinct banks when the token row stride (head_size/4 + 1 words) is
// 1 mod 32 (head sizes 128 and 256).
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

template <int D, int HT, int NST>
__global__ void __launch_bounds__((HT * kConsumerWarpsPerTile + 1) * 32, (D == 256 || HT == 2) ? 1 : 2)
decode_tc_kernel(Params P) {
    constexpr int TPS = kTcTokensPerStage;
    constexpr int W = D / 4 + 1;
    constexpr int NKS = D / 16;          // k-steps of QK^T
    constexpr int NT = D / 8;            // n-tiles of PV
    constexpr int NJ = D / 32;           // V words per row group
    constexpr int NCW = HT * kConsumerWarpsPerTile;
    constexpr int CHUNKS = TPS / 16;

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const Layout L = make_layout(D, TPS, NST, P.PT, P.B, tc_extra_bytes<D, HT>());
    const uint32_t bars = smem_addr(smem + L.bars);
    const int n_stages = (w.len + TPS - 1) / TPS;
    if (threadIdx.x == 0) abort_flag = 0;
    init_barriers(bars, NST, NCW);
    load_table<TPS>(P, w, reinterpret_cast<uint32_t *>(smem + L.table));
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == NCW) {
        producer<D, TPS, NST>(P, w, smem, L, n_stages, &abort_flag);
        return;
    }

    const int ht = warp / kConsumerWarpsPerTile, ts = warp % kConsumerWarpsPerTile;
    const int gq = lane >> 2, cq = lane & 3;
    const int nh_tile = max(0, min(8, w.nh - 8 * ht));
    const bool row_ok = gq < nh_tile;
    const int h = w.h0 + 8 * ht + gq;

    // q of head gq, scaled by 2^-Eq into [1, 2) in magnitude, as hi/lo f16
    // pairs.  Head size 256 keeps these fragments in shared memory (one
    // 16-byte load per k-step) to leave registers for the accumulators.
    constexpr bool kQInSmem = (D == 256);
    uint32_t aq[kQInSmem ? 1 : NKS][4];
    uint4 *qf = reinterpret_cast<uint4 *>(smem + L.extra);          // [HT][NKS][32]
    float qk2 = 0.0f;
    {
        const float *qrow = P.q + ((int64_t)w.s * P.H + (row_ok ? h : w.h0)) * D;
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok ? __ldg(reinterpret_cast<const float4 *>(qrow) + kword<D>(cq, ks))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);      // 2^-eq
        qk2 = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok ? __ldg(reinterpret_cast<const float4 *>(qrow) + kword<D>(cq, ks))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            __half h0, l0, h1, l1, h2, l2, h3, l3;
            split_f16(v.x * down, h0, l0);
            split_f16(v.y * down, h1, l1);
            split_f16(v.z * down, h2, l2);
            split_f16(v.w * down, h3, l3);
            const uint32_t f0 = pack_half2(h0, h1), f1 = pack_half2(l0, l1);
            const uint32_t f2 = pack_half2(h2, h3), f3 = pack_half2(l2, l3);
            if constexpr (kQInSmem) {
                if (ts == 0) qf[(ht * NKS + ks) * 32 + lane] = make_uint4(f0, f1, f2, f3);
            } else {
                aq[ks][0] = f0; aq[ks][1] = f1; aq[ks][2] = f2; aq[ks][3] = f3;
            }
        }
        if constexpr (kQInSmem) named_barrier(2, NCW * 32);
    }

    float acc[NT][4];
#pragma unroll
    for (int i = 0; i < NT; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.0f;
    float m = -INFINITY, lsum = 0.0f;
    int E = 12;                       // running max biased exponent of V scales (>= 12)
    float wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);

    bool ok = true;
    for (int j = 0; j < n_stages; ++j) {
        const int k = j % NST;
        const uint32_t full = bars + 8 * k;
        if (!mbar_wait(full, (j / NST) & 1) || abort_flag) {
            if (lane == 0) { abort_flag = 1; flag_error(P.status, kDevWaitTimeout); }
            ok = false;
            break;
        }
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(smem + L.stages + k * L.stage_bytes);
        const uint32_t *sV = sK + TPS * W;
        const int stage_t0 = j * TPS;

#pragma unroll 1
        for (int ch = ts; ch < CHUNKS; ch += kConsumerWarpsPerTile) {
            const int rb = ch * 16;
            if (stage_t0 + rb >= w.len) break;
            float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
                const int wd = kword<D>(cq, ks);
                uint32_t b0, b1, b2, b3;
                codes4_to_f16x2(sK[(rb + gq) * W + wd], b0, b1);
                codes4_to_f16x2(sK[(rb + 8 + gq) * W + wd], b2, b3);
                if constexpr (kQInSmem) {
                    const uint4 f = qf[(ht * NKS + ks) * 32 + lane];
                    const uint32_t a[4] = {f.x, f.y, f.z, f.w};
                    mma_16816(s0, a, b0, b1);
                    mma_16816(s1, a, b2, b3);
                } else {
                    mma_16816(s0, aq[ks], b0, b1);
                    mma_16816(s1, aq[ks], b2, b3);
                }
            }
            // this thread's four tokens: rb + 2cq + {0, 1, 8, 9}
            const int tA = rb + 2 * cq;
            const int tt[4] = {tA, tA + 1, tA + 8, tA + 9};
            const float sc[4] = {s0[0] + s0[2], s0[1] + s0[3], s1[0] + s1[2], s1[1] + s1[3]};
            float z[4], vs[4];
            uint32_t vbits = 0;
            float cmax = -INFINITY;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool valid = stage_t0 + tt[u] < w.len;
                const float ks_ = __uint_as_float(sK[tt[u] * W + D / 4]);
                vs[u] = __uint_as_float(sV[tt[u] * W + D / 4]);
                z[u] = valid ? sc[u] * ks_ * qk2 : -INFINITY;
                vs[u] = valid ? vs[u] : 0.0f;
                vbits = max(vbits, __float_as_uint(vs[u]) & 0x7FFFFFFFu);
                cmax = fmaxf(cmax, z[u]);
            }
            cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 1));
            cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 2));
            vbits = max(vbits, __shfl_xor_sync(0xFFFFFFFFu, vbits, 1));
            vbits = max(vbits, __shfl_xor_sync(0xFFFFFFFFu, vbits, 2));
            const int Ec = (int)(vbits >> 23);
            const float m_new = fmaxf(m, cmax);
            const int E_new = max(E, Ec);
            const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
            if (__any_sync(0xFFFFFFFFu, m_new != m || E_new != E)) {
                const float ea = (E_new == E) ? 1.0f
                                 : (E - E_new < -126 ? 0.0f
                                                     : __uint_as_float((uint32_t)(127 + E - E_new) << 23));
                const float fa = (m == -INFINITY) ? 0.0f : alpha * ea;
#pragma unroll
                for (int i = 0; i < NT; ++i) {
                    acc[i][0] *= fa; acc[i][1] *= fa; acc[i][2] *= fa; acc[i][3] *= fa;
                }
                lsum *= alpha;
                m = m_new;
                E = E_new;
                wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
            }
            float pw[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float p = (z[u] == -INFINITY) ? 0.0f : fast_exp2(z[u] - m);
                lsum += p;
                pw[u] = p * vs[u] * wscale;
            }
            uint32_t ap[4];
            {
                __half hA, lA, hB, lB, hC, lC, hD, lD;
                split_f16(pw[0], hA, lA);
                split_f16(pw[1], hB, lB);
                split_f16(pw[2], hC, lC);
                split_f16(pw[3], hD, lD);
                ap[0] = pack_half2(hA, hB);
                ap[1] = pack_half2(lA, lB);
                ap[2] = pack_half2(hC, hD);
                ap[3] = pack_half2(lC, lD);
            }
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                const int wd = vword<D>(gq, jj);
                const uint32_t x0 = sV[tt[0] * W + wd], x1 = sV[tt[1] * W + wd];
                const uint32_t x8 = sV[tt[2] * W + wd], x9 = sV[tt[3] * W + wd];
                mma_16816(acc[4 * jj + 0], ap, codes_pair_to_f16x2<0>(x0, x1), codes_pair_to_f16x2<0>(x8, x9));
                mma_16816(acc[4 * jj + 1], ap, codes_pair_to_f16x2<1>(x0, x1), codes_pair_to_f16x2<1>(x8, x9));
                mma_16816(acc[4 * jj + 2], ap, codes_pair_to_f16x2<2>(x0, x1), codes_pair_to_f16x2<2>(x8, x9));
                mma_16816(acc[4 * jj + 3], ap, codes_pair_to_f16x2<3>(x0, x1), codes_pair_to_f16x2<3>(x8, x9));
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (NST + k));
    }

    // All consumer warps are past the ring; reuse it as merge scratch.
    if (named_barrier_or(1, NCW * 32, !ok)) return;
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 1);
    lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, 2);
    float *ml = reinterpret_cast<float *>(smem + L.stages);          // [slot][HT*8][3]
    float *accs = ml + kConsumerWarpsPerTile * HT * 8 * 3;             // [slot][HT*8][D]
    const int hl = 8 * ht + gq;                                         // CTA-local head
    if (cq == 0) {
        float *e = ml + (ts * HT * 8 + hl) * 3;
        e[0] = m; e[1] = lsum; e[2] = (float)E;
    }
    float *arow = accs + (ts * HT * 8 + hl) * D;
#pragma unroll
    for (int i = 0; i < NT; ++i) {
        const int n0 = 2 * cq, n1 = 2 * cq + 1;
        arow[4 * vword<D>(n0, i / 4) + (i & 3)] = acc[i][0] + acc[i][2];
        arow[4 * vword<D>(n1, i / 4) + (i & 3)] = acc[i][1] + acc[i][3];
    }
    named_barrier(1, NCW * 32);
    merge_and_store<D>(P, w, ml, accs, kConsumerWarpsPerTile, HT * 8, NCW * 32);
}

// ============================================================== CUDA cores
//
// Consumer warp ts owns 32-token chunk ts of every stage.  QK: lane = token,
// the warp's heads' q rows are read from shared memory (broadcast) as f32.
// Softmax: per head, warp-wide max; weights p * v_scale go to shared
// memory.  PV: lane = code word (4 head dims; for head size 64 the two half
// warps take alternate tokens, for 256 each lane takes two words).
__device__ __forceinline__ void codes4_to_f32(uint32_t x, float &a, float &b, float &c, float &d) {
    // offset-binary byte under 0x4B000000 is 2^23 + code + 128 exactly
    const uint32_t u = x ^ 0x80808080u;
    a = __uint_as_float(prmt(u, 0x4B000000u, 0x7650u)) - 8388736.0f;
    b = __uint_as_float(prmt(u, 0x4B000000u, 0x7651u)) - 8388736.0f;
    c = __uint_as_float(prmt(u, 0x4B000000u, 0x7652u)) - 8388736.0f;
    d = __uint_as_float(prmt(u, 0x4B000000u, 0x7653u)) - 8388736.0f;
}

template <int D, int NH, int NST>
__global__ void __launch_bounds__((kConsumerWarpsPerTile + 1) * 32, (D == 256 ? 1 : 2))
decode_cc_kernel(Params P) {
    constexpr int TPS = kCcTokensPerStage;
    constexpr int W = D / 4 + 1;
    constexpr int WORDS = D / 4;
    constexpr int NCW = kConsumerWarpsPerTile;
    constexpr int LW = WORDS < 32 ? WORDS : 32;      // lanes per token row in PV
    constexpr int TG = 32 / LW;                      // token groups in PV (2 for D = 64)
    constexpr int NWL = WORDS / LW;                  // words per lane in PV

    extern __shared__ __align__(128) uint8_t smem[];
    __shared__ int abort_flag;
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const uint32_t extra = NH * D * 4 + NCW * 32 * NH * 4;
    const Layout L = make_layout(D, TPS, NST, P.PT, P.B, extra);
    const uint32_t bars = smem_addr(smem + L.bars);
    const int n_stages = (w.len + TPS - 1) / TPS;
    float *sq = reinterpret_cast<float *>(smem + L.extra);             // [NH][D]
    float *sw = sq + NH * D;                                           // [warp][NH][32]
    if (threadIdx.x == 0) abort_flag = 0;
    init_barriers(bars, NST, NCW);
    load_table<TPS>(P, w, reinterpret_cast<uint32_t *>(smem + L.table));
    for (int i = threadIdx.x; i < NH * D; i += blockDim.x) {
        const int hh = i / D;
        sq[i] = hh < w.nh ? __ldg(P.q + ((int64_t)w.s * P.H + w.h0 + hh) * D + (i % D)) : 0.0f;
    }
    __syncthreads();

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (warp == NCW) {
        producer<D, TPS, NST>(P, w, smem, L, n_stages, &abort_flag);
        return;
    }
    const int ts = warp;
    const float4 *sq4 = reinterpret_cast<const float4 *>(sq);
    float *myw = sw + ts * 32 * NH;

    float m[NH], lsum[NH], acc[NH][NWL][4];
#pragma unroll
    for (int hh = 0; hh < NH; ++hh) {
        m[hh] = -INFINITY;
        lsum[hh] = 0.0f;
#pragma unroll
        for (int u = 0; u < NWL; ++u) acc[hh][u][0] = acc[hh][u][1] = acc[hh][u][2] = acc[hh][u][3] = 0.0f;
    }

    bool ok = true;
    for (int j = 0; j < n_stages; ++j) {
        const int k = j % NST;
        if (!mbar_wait(bars + 8 * k, (j / NST) & 1) || abort_flag) {
            if (lane == 0) { abort_flag = 1; flag_error(P.status, kDevWaitTimeout); }
            ok = false;
            break;
        }
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(smem + L.stages + k * L.stage_bytes);
        const uint32_t *sV = sK + TPS * W;
        const int rb = ts * 32;
        const int stage_t0 = j * TPS;
        if (stage_t0 + rb < w.len) {
            // ---- logits, lane = token
            const int t = rb + lane;
            const bool valid = stage_t0 + t < w.len;
            float dot[NH];
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) dot[hh] = 0.0f;
            const uint32_t *krow = sK + t * W;
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
            const float vscale = valid ? __uint_as_float(sV[t * W + WORDS]) : 0.0f;
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float z = valid ? dot[hh] * kscale : -INFINITY;
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
                const float p = valid ? fast_exp2(z - m[hh]) : 0.0f;
                lsum[hh] += p;
                myw[hh * 32 + lane] = p * vscale;
            }
            __syncwarp();
            // ---- weighted sum, lane = code word(s)
            const int ntok = min(32, w.len - stage_t0 - rb);
            const int tg = lane / LW, lw = lane % LW;
#pragma unroll 2
            for (int tt = tg; tt < ntok; tt += TG) {
                const uint32_t *vrow = sV + (rb + tt) * W;
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
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bars + 8 * (NST + k));
    }

    if (named_barrier_or(1, NCW * 32, !ok)) return;
    float *ml = reinterpret_cast<float *>(smem + L.stages);    // [slot][NH][3]
    float *accs = ml + NCW * NH * 3;                            // [slot][NH][D]
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
    named_barrier(1, NCW * 32);
    merge_and_store<D>(P, w, ml, accs, NCW, NH, NCW * 32);
}

// ================================================================= combine
//
// out[s,h] = sum_p A_p 2^(M_p - M*) / sum_p L_p 2^(M_p - M*), M* = max M_p,
// over the partitions of sequences that have more than one.
template <int D>
__global__ void __launch_bounds__(128) combine_kernel(Params P) {
    const int h = blockIdx.x, s = blockIdx.y;
    const int64_t cap = (int64_t)P.Nb * P.B;
    const int64_t craw = __ldg(P.cl + s);
    const int c = (int)(craw < cap ? craw : cap);
    const int np = (c + P.PT - 1) / P.PT;
    if (np <= 1) return;
    const int64_t row0 = ((int64_t)s * P.H + h) * P.NP;
    __shared__ float s_w[1024];
    __shared__ float s_inv;
    float M = -INFINITY;
    for (int p = threadIdx.x; p < np; p += blockDim.x) M = fmaxf(M, P.pml[(row0 + p) * 2]);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    __shared__ float s_red[4];
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = M;
    __syncthreads();
    M = fmaxf(fmaxf(s_red[0], s_red[1]), fmaxf(s_red[2], s_red[3]));
    float Lp = 0.0f;
    for (int p = threadIdx.x; p < np; p += blockDim.x) {
        const float wgt = fast_exp2(P.pml[(row0 + p) * 2] - M);
        if (p < 1024) s_w[p] = wgt;
        Lp += P.pml[(row0 + p) * 2 + 1] * wgt;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) Lp += __shfl_xor_sync(0xFFFFFFFFu, Lp, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = Lp;
    __syncthreads();
    if (threadIdx.x == 0) s_inv = 1.0f / (s_red[0] + s_red[1] + s_red[2] + s_red[3]);
    __syncthreads();
    const float inv = s_inv;
    for (int d = threadIdx.x; d < D; d += blockDim.x) {
        float a = 0.0f;
        for (int p = 0; p < np; ++p) {
            const float wgt = p < 1024 ? s_w[p] : fast_exp2(P.pml[(row0 + p) * 2] - M);
            a = fmaf(P.pacc[(row0 + p) * D + d], wgt, a);
        }
        P.out[((int64_t)s * P.H + h) * D + d] = a * inv;
    }
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

template <int D>
constexpr int tc_stages() { return D == 64 ? 8 : (D == 128 ? 6 : 5); }
template <int D>
constexpr int cc_stages() { return D == 256 ? 2 : 3; }

Params make_params(const DecodeArgs &a) {
    Params P{};
    P.out = a.out; P.q = a.q; P.kc = a.key_cache; P.vc = a.value_cache;
    P.bt = a.block_tables; P.cl = a.context_lens;
    P.S = a.num_seqs; P.H = a.num_heads; P.Hk = a.num_kv_heads; P.B = a.block_size;
    P.Nb = a.max_blocks_per_seq; P.num_blocks = a.num_blocks;
    P.scale_log2 = a.scale * kLog2e;
    P.PT = a.partition_tokens; P.NP = a.num_partitions;
    P.r = a.num_heads / a.num_kv_heads;
    P.heads_per_cta = a.heads_per_cta; P.head_groups = a.head_groups;
    P.pml = a.partial_ml; P.pacc = a.partial_acc; P.status = a.status;
    return P;
}

template <typename K>
cudaError_t launch_attn(K kernel, const Params &P, uint32_t smem_bytes, int threads, cudaStream_t st) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes);
    if (e != cudaSuccess) return e;
    dim3 grid(P.NP, P.Hk * P.head_groups, P.S);
    kernel<<<grid, threads, smem_bytes, st>>>(P);
    return cudaGetLastError();
}

template <int D>
cudaError_t launch_tc(const Params &P, cudaStream_t st) {
    constexpr int NST = tc_stages<D>();
    if (P.heads_per_cta > 8) {
        const Layout L = make_layout(D, kTcTokensPerStage, NST, P.PT, P.B, tc_extra_bytes<D, 2>());
        return launch_attn(decode_tc_kernel<D, 2, NST>, P, L.total, (2 * kConsumerWarpsPerTile + 1) * 32, st);
    }
    const Layout L = make_layout(D, kTcTokensPerStage, NST, P.PT, P.B, tc_extra_bytes<D, 1>());
    return launch_attn(decode_tc_kernel<D, 1, NST>, P, L.total, (kConsumerWarpsPerTile + 1) * 32, st);
}

template <int D, int NH>
cudaError_t launch_cc_nh(const Params &P, cudaStream_t st) {
    constexpr int NST = cc_stages<D>();
    const uint32_t extra = NH * D * 4 + kConsumerWarpsPerTile * 32 * NH * 4;
    const Layout L = make_layout(D, kCcTokensPerStage, NST, P.PT, P.B, extra);
    return launch_attn(decode_cc_kernel<D, NH, NST>, P, L.total, (kConsumerWarpsPerTile + 1) * 32, st);
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
    cudaError_t e = (kernel == kCudaCore) ? launch_cc<D>(P, st) : launch_tc<D>(P, st);
    if (e != cudaSuccess || P.NP <= 1) return e;
    combine_kernel<D><<<dim3(P.H, P.S), 128, 0, st>>>(P);
    return cudaGetLastError();
}

}  // namespace

bool make_plan(DecodeArgs &a, int requested_kernel, int requested_partition, int num_sms) {
    const int r = a.num_heads / a.num_kv_heads;
    a.kernel = requested_kernel == kAuto ? kTensorCore : requested_kernel;
    if (a.kernel == kTensorCore) {
        a.heads_per_cta = r < 16 ? r : 16;
    } else {
        int hp = 16;
        while (hp > 1 && (r % hp) != 0) hp >>= 1;
        a.heads_per_cta = hp;
    }
    a.head_groups = (r + a.heads_per_cta - 1) / a.heads_per_cta;
    const int64_t max_ctx = (int64_t)a.max_blocks_per_seq * a.block_size;
    int pt = requested_partition;
    if (pt <= 0) {
        const int64_t units = (int64_t)a.num_seqs * a.num_kv_heads * a.head_groups;
        const int64_t target = 4LL * num_sms;
        pt = 2048;
        while (pt > 256 && units * ((max_ctx / 2 + pt - 1) / pt) < target) pt >>= 1;
        if (pt > 2048) pt = 2048;
    }
    if (pt % kCcTokensPerStage != 0 || pt > 16384) return false;
    a.partition_tokens = pt;
    const int64_t np = (max_ctx + pt - 1) / pt;
    if (np > 0x7FFFFFFF || np < 1) return false;
    a.num_partitions = (int)(np < 1 ? 1 : np);
    return true;
}

size_t plan_workspace_bytes(const DecodeArgs &a) {
    if (a.num_partitions <= 1) return 0;
    const size_t rows = (size_t)a.num_seqs * a.num_heads * a.num_partitions;
    const size_t ml = rows * 2 * sizeof(float);
    return ((ml + 255) / 256) * 256 + rows * a.head_size * sizeof(float);
}

int64_t plan_num_ctas(const DecodeArgs &a) {
    return (int64_t)a.num_partitions * a.num_kv_heads * a.head_groups * a.num_seqs;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    const Params P = make_params(a);
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
