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
// Split contexts are merged by the last CTA of each group to finish, or, when
// the whole split grid fits in one wave, by combine_kernel, a grid of its own
// launched as a programmatic dependent of the attention grid.
// Every wait is bounded; a wait that gives up flags the status word, and a
// warp leaves only after the copies it issued have landed.
#include "decode_common.cuh"

// Partition length, in quarters of the table's capacity, when the sequences
// fill less than two waves of resident CTAs (4: no cut)
#ifndef PA_Q8_TAIL_CUT_X4
#define PA_Q8_TAIL_CUT_X4 3
#endif
// Split grids that fit in one wave merge their partials in a combine grid of
// their own (0: always by the last CTA of each group)
#ifndef PA_Q8_SEP_COMBINE
#define PA_Q8_SEP_COMBINE 1
#endif
// With such a combine grid, one-tile tensor-core CTAs store one record per
// token-slot warp instead of merging their warps (0: CTA merge)
#ifndef PA_Q8_SLOT_RECORDS
#define PA_Q8_SLOT_RECORDS 1
#endif

namespace pa_q8 {
namespace {

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

// Head size 256: the q fragments of every head tile ([HT][D/16][32] uint4),
// then each head's logit factor ([HT * 8] f32).
// Head dims (in float4 units) held at float4 slot t of a per-warp record:
// the slot order of the record store above.
template <int D>
__device__ __forceinline__ int tc_record_dim4(int t) {
    return vword<D>(2 * (t & 3) + ((t >> 2) & 1), t >> 3);
}

template <int D, int HT>
__host__ __device__ constexpr uint32_t tc_extra_bytes() {
    return D == 256 ? (uint32_t)HT * (D / 16) * 32 * 16 + (uint32_t)HT * 8 * 4 : 0u;
}

template <int D>
__host__ __device__ constexpr int tc_ring() { return D == 64 ? PA_Q8_TC_RING_64 : (D == 128 ? PA_Q8_TC_RING_128 : PA_Q8_TC_RING_256); }

template <int D, int HT>
__host__ __device__ constexpr int tc_min_blocks() {
    return HT == 2 ? 1 : (D == 256 ? PA_Q8_TC_MINB_256 : (D == 128 ? PA_Q8_TC_MINB_128 : 3));
}

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
    // q is loaded before the block table so the two round trips overlap.
    // Head size 256 keeps its fragments in shared memory, built by the
    // token slot 0 warp of each head tile alone, so only that warp loads q.
    const bool q_builder = !kQInSmem || ts == 0;
    float4 qraw[NKS];
    if (q_builder) {
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
    float *qk2s = reinterpret_cast<float *>(qf + HT * NKS * 32);      // [HT * 8]
    float qk2 = 0.0f;
    if (q_builder) {
        auto qload = [&](int ks) -> float4 { return qraw[ks]; };
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
                qf[(ht * NKS + ks) * 32 + lane] = make_uint4(f0, f1, f2, f3);
            } else {
                aq[ks][0] = f0; aq[ks][1] = f1; aq[ks][2] = f2; aq[ks][3] = f3;
            }
        }
        if (kQInSmem && cq == 0) qk2s[ht * 8 + gq] = qk2;
    }
    if constexpr (kQInSmem) {
        __syncthreads();
        qk2 = qk2s[ht * 8 + gq];
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
    if (P.rec_slots > 1) {
        // The combine grid merges every row: each warp stores its own
        // record (A in true units, m, l) for the rows of its head tile, and
        // no CTA merge runs.  For a fixed word group jj and column pair half
        // e, a thread's four accumulators are four consecutive head dims
        // (4 vword(2 cq + e, jj) ..): one float4, stored at float4 slot
        // (2 jj + e) * 4 + cq of the record, so the four threads of a row
        // write 64 contiguous bytes; the combine grid maps the slots back to
        // head dims (tc_record_dim4).
        if (row_ok) {
            const float f = ldexpf(1.0f, E - kVScaleBias);
            float *rec = P.part + ((qrow(P, w, vh) * P.NP + w.p) * SLOTS + ts) * (D + 4);
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    float4 v;
                    v.x = (acc[4 * jj + 0][e] + acc[4 * jj + 0][e + 2]) * f;
                    v.y = (acc[4 * jj + 1][e] + acc[4 * jj + 1][e + 2]) * f;
                    v.z = (acc[4 * jj + 2][e] + acc[4 * jj + 2][e + 2]) * f;
                    v.w = (acc[4 * jj + 3][e] + acc[4 * jj + 3][e + 2]) * f;
                    reinterpret_cast<float4 *>(rec)[(2 * jj + e) * 4 + cq] = v;
                }
            }
            if (cq == 0) {
                rec[D] = m;
                rec[D + 1] = lsum;
            }
        }
        return;
    }
    float *ml = reinterpret_cast<float *>(smem + L.ring);            // [slot][HT*8][3]
    float *accs = ml + SLOTS * HT * 8 * 3;                            // [slot][HT*8][D]
    static_assert(merge_scratch_bytes(D, SLOTS, HT * 8) <= ring_bytes(D, SLOTS, RING),
                  "the merge scratch must fit in the chunk ring");
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

// ============================================== tensor cores, 16 heads per warp
//
// For 9 .. 16 (query row, head) pairs per kv head at head sizes 64 / 128
// (multi-row decodes): the tensor-core tile with two 8-head A tiles per warp
// (u = 0, 1: virtual heads h0 + 8u + gq).  Every chunk's codes become B
// fragments once and feed both tiles' MMAs, so the conversion -- most of a
// warp's instructions -- serves 16 heads without leaving registers.  The q
// fragments of both tiles live in shared memory; the token scales are read
// once for both.

template <int D>
__host__ __device__ constexpr uint32_t tc2_extra_bytes() { return 2u * (D / 16) * 32 * 16; }

template <int D>
__global__ void __launch_bounds__(PA_Q8_TC_SLOTS * 32, 2)
decode_tc2_kernel(Params P) {
    constexpr int SLOTS = PA_Q8_TC_SLOTS;
    constexpr int RING = tc_ring<D>();
    constexpr int W = D / 4 + 1;
    constexpr int NKS = D / 16;
    constexpr int NT = D / 8;
    constexpr int NJ = D / 32;

    extern __shared__ __align__(128) uint8_t smem[];
    Work w;
    if (!setup_work(P, w)) {
        write_zero_rows<D>(P, w);
        return;
    }
    const Layout L = make_layout(D, SLOTS, RING, P.PT, P.B, tc2_extra_bytes<D>());
    const int ts = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, cq = lane & 3;
    const uint32_t bars = smem_addr(smem + L.bars) + 8 * RING * ts;
    const uint32_t ring = smem_addr(smem + L.ring) + RING * L.slot_bytes * ts;
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    uint4 *qf = reinterpret_cast<uint4 *>(smem + L.extra);           // [2][NKS][32]
    const int nchunks = (w.len + kChunk - 1) / kChunk;
    const int my_n = ts < nchunks ? (nchunks - ts + SLOTS - 1) / SLOTS : 0;
    const uint64_t policy = l2_policy_evict_first();

    if (lane == 0) {
        for (int k = 0; k < RING; ++k) mbar_init(bars + 8 * k, 1);
        fence_mbar_init();
    }
    if (P.nk) append_tokens<D>(P, w);
    load_table(P, w, const_cast<uint32_t *>(table));

    bool row_ok[2];
    int len_row[2];
    float qk2[2];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        row_ok[u] = 8 * u + gq < w.nh;
        const int vh = w.h0 + 8 * u + gq;
        len_row[u] = row_ok[u] ? row_len(P, w, vh) : w.len;
        // q of this row scaled by 2^-eq into [1, 2) in magnitude, as hi/lo f16
        // pairs; warp u writes tile u's fragments
        const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok[u] ? vh : w.h0) * D);
        float mx = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const float4 v = row_ok[u] ? __ldg(qv + kword<D>(cq, ks)) : make_float4(0.f, 0.f, 0.f, 0.f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 2));
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);
        qk2[u] = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
        if (ts == u) {
#pragma unroll
            for (int ks = 0; ks < NKS; ++ks) {
                const float4 v = row_ok[u] ? __ldg(qv + kword<D>(cq, ks)) : make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t f0, f1, f2, f3;
                split_f16x2(v.x * down, v.y * down, f0, f1);
                split_f16x2(v.z * down, v.w * down, f2, f3);
                qf[(u * NKS + ks) * 32 + lane] = make_uint4(f0, f1, f2, f3);
            }
        }
    }
    __syncthreads();

    int issued = 0;
    for (; issued < RING && issued < my_n; ++issued)
        issue_chunk<D>(P, w, table, ts + SLOTS * issued, ring + issued * L.slot_bytes, bars + 8 * issued, policy);
    const int len_min = __reduce_min_sync(0xFFFFFFFFu, (unsigned)min(len_row[0], len_row[1]));

    float acc[2][NT][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
        for (int n = 0; n < NT; ++n) acc[u][n][0] = acc[u][n][1] = acc[u][n][2] = acc[u][n][3] = 0.0f;
    float m[2] = {-INFINITY, -INFINITY}, lsum[2] = {0.0f, 0.0f};
    int E[2] = {12, 12};
    float wscale[2];
    wscale[0] = wscale[1] = __uint_as_float((uint32_t)(kVScaleBias + 127 - 12) << 23);

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
        const uint32_t *sK = reinterpret_cast<const uint32_t *>(smem + L.ring) + (RING * ts + k) * (L.slot_bytes / 4);
        const uint32_t *sV = sK + kChunk * W;
        const int t0 = (ts + SLOTS * i) * kChunk;
        const bool full = t0 + kChunk <= len_min;

        // ---- S = Q K^T for both tiles from one conversion of the codes
        float s[2][4][4];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int j = 0; j < 4; ++j) s[u][j][0] = s[u][j][1] = s[u][j][2] = s[u][j][3] = 0.0f;
#pragma unroll
        for (int ks = 0; ks < NKS; ++ks) {
            const int wd = kword<D>(cq, ks);
            const uint4 f0 = qf[ks * 32 + lane], f1 = qf[(NKS + ks) * 32 + lane];
            const uint32_t a0[4] = {f0.x, f0.y, f0.z, f0.w}, a1[4] = {f1.x, f1.y, f1.z, f1.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                uint32_t b0, b1;
                codes4_to_f16x2(sK[(8 * j + gq) * W + wd], b0, b1, fk);
                mma_16816(s[0][j], a0, b0, b1);
                mma_16816(s[1][j], a1, b0, b1);
            }
        }
        // ---- online softmax per tile over this thread's 8 tokens 8j + 2cq + e
        float ksv[8], vsv[8];
#pragma unroll
        for (int j = 0; j < 4; ++j)
#pragma unroll
            for (int e = 0; e < 2; ++e) {
                const int t = 8 * j + 2 * cq + e;
                ksv[2 * j + e] = __uint_as_float(sK[t * W + D / 4]);
                vsv[2 * j + e] = __uint_as_float(sV[t * W + D / 4]);
            }
        uint32_t ap[2][2][4];                 // [tile][k-step][4]: P as hi/lo f16 pairs
#pragma unroll
        for (int u = 0; u < 2; ++u) {
            float z[8], vs[8];
            float cmax = -INFINITY, vmax = 0.0f;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int t = 8 * j + 2 * cq + e;
                    float zz = (s[u][j][e] + s[u][j][e + 2]) * ksv[2 * j + e] * qk2[u];
                    float vv = vsv[2 * j + e];
                    if (!full) {
                        const bool valid = t0 + t < len_row[u];
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
            const int Ec = (int)(__float_as_uint(vmax) >> 23);
            if (__any_sync(0xFFFFFFFFu, cmax > m[u] + (float)kLazy || Ec > E[u])) {
                const float m_new = fmaxf(m[u], cmax);
                const int E_new = max(E[u], Ec);
                const float alpha = (m[u] == -INFINITY) ? 0.0f : fast_exp2(m[u] - m_new);
                const float ea = (E[u] - E_new < -126) ? 0.0f : __uint_as_float((uint32_t)(127 + E[u] - E_new) << 23);
                const float fa = alpha * ea;
#pragma unroll
                for (int n = 0; n < NT; ++n) {
                    acc[u][n][0] *= fa; acc[u][n][1] *= fa; acc[u][n][2] *= fa; acc[u][n][3] *= fa;
                }
                lsum[u] *= alpha;
                m[u] = m_new;
                E[u] = E_new;
                wscale[u] = __uint_as_float((uint32_t)(kVScaleBias + 127 - E[u]) << 23);
            }
            const float m_ref = m[u] == -INFINITY ? 0.0f : m[u];
            float pw[8];
#pragma unroll
            for (int x = 0; x < 8; ++x) {
                const float p = fast_exp2(z[x] - m_ref);
                lsum[u] += p;
                pw[x] = p * vs[x] * wscale[u];
            }
#pragma unroll
            for (int kk = 0; kk < 2; ++kk) {
                split_f16x2(pw[4 * kk + 0], pw[4 * kk + 1], ap[u][kk][0], ap[u][kk][1]);
                split_f16x2(pw[4 * kk + 2], pw[4 * kk + 3], ap[u][kk][2], ap[u][kk][3]);
            }
        }
        // ---- O += P V for both tiles from one conversion of the codes
#pragma unroll
        for (int kk = 0; kk < 2; ++kk) {
            const uint32_t *r0 = sV + (16 * kk + 2 * cq) * W;
#pragma unroll
            for (int jj = 0; jj < NJ; ++jj) {
                const int wd = vword<D>(gq, jj);
                const uint32_t x0 = r0[wd], x1 = r0[W + wd], x8 = r0[8 * W + wd], x9 = r0[9 * W + wd];
                uint32_t b[4][2];
                b[0][0] = codes_pair_to_f16x2<0>(x0, x1, fk); b[0][1] = codes_pair_to_f16x2<0>(x8, x9, fk);
                b[1][0] = codes_pair_to_f16x2<1>(x0, x1, fk); b[1][1] = codes_pair_to_f16x2<1>(x8, x9, fk);
                b[2][0] = codes_pair_to_f16x2<2>(x0, x1, fk); b[2][1] = codes_pair_to_f16x2<2>(x8, x9, fk);
                b[3][0] = codes_pair_to_f16x2<3>(x0, x1, fk); b[3][1] = codes_pair_to_f16x2<3>(x8, x9, fk);
#pragma unroll
                for (int e4 = 0; e4 < 4; ++e4) {
                    mma_16816(acc[0][4 * jj + e4], ap[0][kk], b[e4][0], b[e4][1]);
                    mma_16816(acc[1][4 * jj + e4], ap[1][kk], b[e4][0], b[e4][1]);
                }
            }
        }
        __syncwarp();
        if (issued < my_n) {
            issue_chunk<D>(P, w, table, ts + SLOTS * issued, ring + k * L.slot_bytes, bars + 8 * k, policy);
            ++issued;
        }
    }
    drain(P, bars, RING, i, issued);

    if (__syncthreads_or(!ok)) return;
    float *ml = reinterpret_cast<float *>(smem + L.ring);            // [slot][16][3]
    float *accs = ml + SLOTS * 16 * 3;                                // [slot][16][D]
    static_assert(merge_scratch_bytes(D, SLOTS, 16) <= ring_bytes(D, SLOTS, RING),
                  "the merge scratch must fit in the chunk ring");
#pragma unroll
    for (int u = 0; u < 2; ++u) {
        float l = lsum[u];
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 1);
        l += __shfl_xor_sync(0xFFFFFFFFu, l, 2);
        const int hl = 8 * u + gq;
        if (cq == 0) {
            float *e = ml + (ts * 16 + hl) * 3;
            e[0] = m[u]; e[1] = l; e[2] = (float)E[u];
        }
        float *arow = accs + (ts * 16 + hl) * D;
#pragma unroll
        for (int n = 0; n < NT; ++n) {
            arow[4 * vword<D>(2 * cq, n / 4) + (n & 3)] = acc[u][n][0] + acc[u][n][2];
            arow[4 * vword<D>(2 * cq + 1, n / 4) + (n & 3)] = acc[u][n][1] + acc[u][n][3];
        }
    }
    __syncthreads();
    merge_and_store<D>(P, w, ml, accs, SLOTS, 16, accs + SLOTS * 16 * D);
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
    static_assert(merge_scratch_bytes(D, kCcSlots, NH) <= ring_bytes(D, kCcSlots, RING),
                  "the merge scratch must fit in the chunk ring");
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

// ==================================================================== prep
//
// One CTA before the attention grid: zero the split-context arrival
// counters and order the sequences longest (clamped) context first, so the
// block scheduler starts the longest-running CTAs first and the grid's tail
// holds only short ones.  (length, index) keys in shared memory: ranked by
// counting for up to blockDim sequences, bitonic-sorted up to kPrepMaxSort;
// beyond that the order is the identity.
//
// Launched as a programmatic dependent of the kernel before it (the library's
// writers let it start once all their CTAs are running): it reads only the
// context lengths, which that kernel does not write, and waits for it to
// finish before writing the workspace.  The attention grid waits for this one,
// so it sees the writer's cache words too.
constexpr int kPrepThreads = 1024;
constexpr int kPrepMaxSort = 8192;

__global__ void __launch_bounds__(kPrepThreads) prep_kernel(const uint32_t *context_lens, int S, int64_t cap,
                                                            unsigned long long *order, uint32_t *counters,
                                                            int64_t n_counters) {
    extern __shared__ unsigned long long keys[];
    // the attention grid may launch now; it waits for this grid's writes
    grid_dependents_launch();
    if (S > kPrepMaxSort) {
        grid_dependency_wait();
        for (int64_t i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
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
        grid_dependency_wait();
        for (int64_t c = threadIdx.x; c < n_counters; c += blockDim.x) counters[c] = 0u;
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
    grid_dependency_wait();
    for (int64_t i = threadIdx.x; i < n_counters; i += blockDim.x) counters[i] = 0u;
    for (int i = threadIdx.x; i < S; i += blockDim.x)
        order[i] = ((unsigned long long)(cap - (int64_t)(keys[i] >> 32)) << 32) | (keys[i] & 0xFFFFFFFFull);
}

// ============================================================== combine
//
// The log-sum-exp merge of split-context partials as a grid of its own
// ("attention.rs", the attn_combine dispatch after the split-T decode), for
// plans whose split grid fits in one wave: there the merge by the group's
// last CTA sits at the end of the critical path, one CTA working through
// every head of its group.  Here one warp (two at head size 256, each with
// half the dims) merges one output row (sequence, query row, head) from its
// records -- one per partition, or one per token-slot warp of each partition
// (rec_slots) --: M = max_r m_r, L = sum_r l_r 2^(m_r - M), out = (1/L)
// sum_r A_r 2^(m_r - M), summed over r in order, with the first 32 records'
// A loads in flight while M and L are reduced.  Launched as a programmatic
// dependent of the attention grid: it waits for that grid's completion and
// memory before the first load.  With one record per partition, rows of a
// context that fits one partition were written by the attention CTA and are
// left alone.
constexpr int kCombineThreads = 256;

template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(Params P) {
    constexpr int DP = D + 4;                 // floats per partial record
    constexpr int WPR = D > 128 ? D / 128 : 1;    // warps per row
    constexpr int V4W = D / 4 / WPR;          // float4 of the row per warp (32, or 16 at head size 64)
    constexpr int RU = 32;                    // records' loads in flight per thread
    grid_dependency_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t gw = (int64_t)blockIdx.x * (kCombineThreads / 32) + warp;
    const int64_t row = gw / WPR;             // (s * R + b) * H + h
    if (row >= (int64_t)P.S * P.R * P.H) return;
    const int s = (int)(row / ((int64_t)P.R * P.H));
    const int64_t cap = (int64_t)P.Nb * P.B;
    const int64_t craw = __ldg(P.cl + s);
    const int c = (int)(craw < cap ? craw : cap);
    const int nrec = (c + P.PT - 1) / P.PT * P.rec_slots;     // records of this row
    if (nrec <= 1) return;
    const float *rec = P.part + row * P.NP * P.rec_slots * DP;
    const int d4 = (int)(gw % WPR) * V4W + lane;              // this thread's float4 of the row
    const bool act = lane < V4W;

    float4 v[RU];
    float mp[RU];
    auto load = [&](int r0) {
#pragma unroll
        for (int j = 0; j < RU; ++j) {
            const float *r = rec + (size_t)min(r0 + j, nrec - 1) * DP;
            mp[j] = __ldcg(r + D);
            if (act) v[j] = __ldcg(reinterpret_cast<const float4 *>(r) + d4);
        }
    };
    load(0);
    // (m, l) of record lane (and lane + 32, ...), in flight with the A loads
    const float2 ml0 = lane < nrec ? __ldcg(reinterpret_cast<const float2 *>(rec + (size_t)lane * DP + D))
                                   : make_float2(-INFINITY, 0.0f);
    float M = ml0.x;
    for (int r = lane + 32; r < nrec; r += 32) M = fmaxf(M, __ldcg(rec + (size_t)r * DP + D));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
    if (M == -INFINITY) M = 0.0f;             // a query row that sees no token: weights 0, row 0
    float L = ml0.y * fast_exp2(ml0.x - M);
    for (int r = lane + 32; r < nrec; r += 32) {
        const float2 ml = __ldcg(reinterpret_cast<const float2 *>(rec + (size_t)r * DP + D));
        L += ml.y * fast_exp2(ml.x - M);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) L += __shfl_xor_sync(0xFFFFFFFFu, L, o);

    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int r0 = 0;;) {
#pragma unroll
        for (int j = 0; j < RU; ++j) {
            if (r0 + j < nrec) {
                const float x = fast_exp2(mp[j] - M);
                a.x = fmaf(v[j].x, x, a.x);
                a.y = fmaf(v[j].y, x, a.y);
                a.z = fmaf(v[j].z, x, a.z);
                a.w = fmaf(v[j].w, x, a.w);
            }
        }
        r0 += RU;
        if (r0 >= nrec) break;
        load(r0);
    }
    const float il = L > 0.0f ? 1.0f / L : 0.0f;
    // per-warp records keep the tensor-core fragment order
    const int o4 = P.rec_slots > 1 ? tc_record_dim4<D>(d4) : d4;
    if (act) reinterpret_cast<float4 *>(P.out + row * D)[o4] = make_float4(a.x * il, a.y * il, a.z * il, a.w * il);
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
    P.order = a.order; P.counters = a.counters; P.part = a.partials; P.status = a.status;
    P.nk = a.new_key; P.nv = a.new_value;
    P.nk_stride = a.new_key_stride; P.nv_stride = a.new_value_stride;
    P.contiguous = a.contiguous;
    P.per_sm = a.per_sm;
    P.rec_slots = a.rec_slots > 1 ? a.rec_slots : 1;
    P.kc_w = const_cast<uint32_t *>(a.key_cache);      // written only by the fused append
    P.vc_w = const_cast<uint32_t *>(a.value_cache);
    return P;
}

template <int D>
cudaError_t launch_tc(const Params &P, cudaStream_t st) {
    constexpr int SLOTS = PA_Q8_TC_SLOTS;
    constexpr int RING = tc_ring<D>();
    if constexpr (D <= 128) {       // 9 .. 16 pairs: two 8-head tiles per warp
        if (P.heads_per_cta > 8) {
            const Layout L = make_layout(D, SLOTS, RING, P.PT, P.B, tc2_extra_bytes<D>());
            return launch_attn(decode_tc2_kernel<D>, P, L.total, SLOTS * 32, st);
        }
    }
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
        const int64_t n_counters = P.NP > 1 && P.counters ? (int64_t)P.S * P.Hk * P.head_groups : 0;
        int n = 1;
        while (n < P.S && n < kPrepMaxSort) n <<= 1;
        const size_t smem = (size_t)n * sizeof(unsigned long long);
        cudaError_t e = cudaFuncSetAttribute(prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(1);
        cfg.blockDim = dim3(kPrepThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, prep_kernel, P.cl, P.S, (int64_t)P.Nb * P.B,
                               const_cast<unsigned long long *>(P.order), P.counters, n_counters);
        if (e != cudaSuccess) return e;
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    cudaError_t e;
    if (kernel == kF32) e = launch_f32_family(P, D, st);
    else if (P.contiguous) e = launch_cq_family(P, D, st);
    else if (kernel == kTcgen05) e = launch_umma_family(P, D, st);
    else e = (kernel == kCudaCore) ? launch_cc<D>(P, st) : launch_tc<D>(P, st);
    if (e != cudaSuccess || P.NP <= 1 || P.counters != nullptr) return e;
    // split contexts without arrival counters: the combine grid, launched as a
    // programmatic dependent of the attention grid
    const int64_t warps = (int64_t)P.S * P.R * P.H * (D > 128 ? D / 128 : 1);     // warps per row: combine_kernel
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + kCombineThreads / 32 - 1) / (kCombineThreads / 32)));
    cfg.blockDim = dim3(kCombineThreads);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, combine_kernel<D>, P);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// CTAs of the chosen kernel resident per SM (registers and shared memory as
// built): the partition planner sizes its waves and the one-wave test by it.
int resident_per_sm(const DecodeArgs &a) {
    const int hd = a.head_size;
    if (hd == 256) return a.heads_per_cta > 8 || a.kernel != kTensorCore ? 1 : PA_Q8_TC_MINB_256;
    if (a.contiguous) return 3;
    if (a.kernel == kF32) return 1;
    if (a.kernel == kTcgen05 || a.kernel == kCudaCore) return 2;
    return a.heads_per_cta > 8 ? 2 : 3;
}

}  // namespace

bool make_plan(DecodeArgs &a, int requested_kernel, int requested_partition, int num_sms) {
    if (a.num_rows < 1) a.num_rows = 1;
    // (query row, head) pairs served per kv head: the rows of one sequence
    // share their kv group's K/V read like the heads of a GQA group
    const int r = a.num_rows * (a.num_heads / a.num_kv_heads);
    // automatic: tcgen05 from umma_auto_pairs (row, head) pairs per kv head
    // on (one CTA serves up to 64), the mma.sync tensor-core family below
    a.kernel = requested_kernel != kAuto ? requested_kernel
                                         : (r >= umma_auto_pairs(a.head_size) ? kTcgen05 : kTensorCore);
    if (a.kernel == kTcgen05) {
        a.heads_per_cta = r < kUmmaHeads ? r : kUmmaHeads;
    } else if (a.kernel == kTensorCore && a.contiguous) {
        a.heads_per_cta = r < 8 ? r : 8;                  // the contiguous-cache kernel: one head tile
    } else if (a.kernel == kTensorCore) {
        // head size 256: 16-head CTAs.  At 64 / 128, more than 8 pairs take the
        // two-tile kernel (16 per CTA) when it needs fewer CTA-equivalents: a
        // 16-head CTA costs about 1.75 eight-head ones (measured on the
        // 256-sequence batch at 16 pairs), so 24 or 40 pairs stay on 8-head CTAs
        const int n8 = (r + 7) / 8, n16 = (r + 15) / 16;
        const bool wide = PA_Q8_TC_WIDE && a.head_size <= 128 && r > 8 && 7 * n16 < 4 * n8;
        int cap = wide ? 16 : PA_Q8_TC_MAX_HEADS;
        // head size 256: 16 heads per CTA (two head tiles, one CTA per SM),
        // one read of each K/V tile per 16 heads.  Few sequences then take
        // short partitions (the rule below) rather than two 8-head CTAs per
        // group: 32 MQA sequences of up to 4095 tokens, 512-token partitions,
        // 26.3 us against 27.3 us.
        if (a.head_size == 256) cap = 16;
        a.heads_per_cta = r < cap ? r : cap;
    } else {
        int hp = a.kernel == kF32 ? 8 : 16;
        while (hp > 1 && (r % hp) != 0) hp >>= 1;
        a.heads_per_cta = hp;
    }
    a.head_groups = (r + a.heads_per_cta - 1) / a.heads_per_cta;
    const int64_t max_ctx = (int64_t)a.max_blocks_per_seq * a.block_size;
    const int64_t units = (int64_t)a.num_seqs * a.num_kv_heads * a.head_groups;
    int per_sm = resident_per_sm(a);
    int pt = requested_partition;
    if (pt <= 0) {
        const int64_t slots = (int64_t)per_sm * num_sms;
        if (units >= slots) {
            // Enough (sequence, kv head) work items: one partition per context
            // (up to 8192 tokens).  The grid runs the longest contexts first,
            // so the tail holds short ones.  Within two waves, the longest
            // contexts alone would set that tail: those in the top quarter of
            // the table's capacity are cut in two (measured on 64 x U[512,
            // 4096] contexts: 3072-token partitions 65-66 us against 68 us)
            const int64_t cut = units < 2 * slots ? (max_ctx * PA_Q8_TAIL_CUT_X4 + 3) / 4 : max_ctx;
            pt = (int)std::min<int64_t>((cut + 127) / 128 * 128, 8192);
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
    if (a.contiguous && a.head_size == 128) {
        // Two builds of the kernel: 3 CTAs per SM (168 registers) keep more
        // loads in flight per SM; 2 per SM (no register limit below 255) run
        // each CTA faster.  With four or more waves of 3 per SM expected
        // (contexts taken at half their maximum) occupancy wins; with fewer,
        // the longest CTAs set the time and the faster CTA wins (measured:
        // 256-sequence lognormal batch 3; 64 x U[512, 4096] and 8 x
        // U[32K, 128K] contexts 2).
        const int64_t live = units * std::max<int64_t>(1, (max_ctx / 2 + pt - 1) / pt);
        per_sm = live >= 4 * 3 * (int64_t)num_sms ? 3 : 2;
    }
    a.per_sm = per_sm;
    a.one_wave = np == 1 && units <= (int64_t)per_sm * num_sms;
    // A split grid whose expected CTAs (contexts taken at half their maximum)
    // all fit at once: the partials are merged by a combine grid of its own,
    // a warp per output row, instead of by the last CTA of each group, whose
    // merge of every head would end the critical path.  Such a grid needs no
    // longest-first order and no arrival counters, so no prep kernel.
    const int64_t expect = units * std::max<int64_t>(1, (max_ctx / 2 + pt - 1) / pt);
    a.sep_combine = PA_Q8_SEP_COMBINE && np > 1 && expect <= (int64_t)per_sm * num_sms;
    // The one-tile tensor-core kernel then skips its CTA merge too: each
    // token-slot warp stores its own record, and the combine grid merges every
    // row (one partition or several).
    a.rec_slots = a.sep_combine && PA_Q8_SLOT_RECORDS && a.kernel == kTensorCore && !a.contiguous &&
                          (a.heads_per_cta <= 8 || a.head_size == 256) ? PA_Q8_TC_SLOTS : 1;
    return true;
}

namespace {
size_t round256(size_t x) { return (x + 255) / 256 * 256; }
}

size_t plan_workspace_bytes(const DecodeArgs &a) {
    const size_t order = round256((size_t)a.num_seqs * sizeof(unsigned long long));
    if (a.num_partitions <= 1) return order;
    const size_t groups = (size_t)a.num_seqs * a.num_kv_heads * a.head_groups;
    const size_t rows = (size_t)a.num_seqs * a.num_rows * a.num_heads * a.num_partitions * (a.rec_slots > 1 ? a.rec_slots : 1);
    return order + round256(groups * sizeof(uint32_t)) + rows * (a.head_size + 4) * sizeof(float);
}

void plan_workspace_layout(DecodeArgs &a, void *workspace) {
    char *p = static_cast<char *>(workspace);
    a.order = reinterpret_cast<unsigned long long *>(p);
    p += round256((size_t)a.num_seqs * sizeof(unsigned long long));
    if (a.num_partitions <= 1) return;
    const size_t groups = (size_t)a.num_seqs * a.num_kv_heads * a.head_groups;
    a.counters = reinterpret_cast<uint32_t *>(p);
    p += round256(groups * sizeof(uint32_t));
    a.partials = reinterpret_cast<float *>(p);
}

int64_t plan_num_ctas(const DecodeArgs &a) {
    return (int64_t)a.num_partitions * a.num_kv_heads * a.head_groups * a.num_seqs;
}

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream) {
    Params P = make_params(a);
    // every CTA starts at once: no order, and without counters no prep kernel
    if (a.one_wave || a.sep_combine) P.order = nullptr;
    if (a.sep_combine) P.counters = nullptr;
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
