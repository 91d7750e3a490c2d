// Multi-row decode on 5th-generation tensor cores: decode_umma_kernel
// (tcgen05.mma, f32 accumulators in TMEM, warp-specialised conversion,
// softmax and issue roles).
#include "decode_common.cuh"

namespace pa_q8 {
namespace {

// ======================================================== tcgen05 (multi-row)
//
// Many virtual heads per kv head (multi-row decode: R query rows x r heads)
// make the contraction GEMM-shaped, so it runs on the 5th-generation tensor
// cores: one CTA serves up to 64 virtual heads of one kv head for one
// partition.  TMEM lane quadrant q holds M rows 32q .. 32q+31: rows 32q + j
// (j < 16) the hi f16 part of virtual head 16q + j's q (scaled by 2^-eq like
// the mma.sync kernel), rows 32q + 16 + j its lo part, so a logit's two
// halves are one shuffle apart.  TMEM holds S twice (columns 0-31, 32-63), O
// (D columns) and the Q tile itself (D / 2 columns, two f16 per column of a
// row's lane), which QK takes as its A operand from tensor memory.
//
// Warp roles, linked only by mbarriers (every wait bounded and abortable):
//  - warps 0-3, softmax: warp q owns quadrant q (idle when it holds no head).
//    Per chunk: S row -> online softmax (hi/lo partner threads take 16 tokens
//    each; lazy rescale of O rows in TMEM) -> P tile rows (w = p * v_scale *
//    2^(131 - E), split hi/lo like the mma.sync kernel).
//  - warps 4-6, conversion: per chunk the raw codes (bulk-copied ring, as in
//    the other families) become f16 K and V tiles [32 tokens][D] in the
//    same core-matrix layout (K-major for QK's B, MN-major for PV's B) and
//    the token scales a small table.
//  - warp 7: its lane 0 issues S = Q.K^T (M 128, N 32, K D) and O += P.V
//    (M 128, N D, K 32), each as soon as its inputs are ready.
//  - warp 8: refills the raw ring, chunk c into the slot of chunk c - ring
//    once the conversion has read that slot (slot_free[slot]).  A refill
//    costs about as much as issuing both MMAs of a chunk, so it has a warp of
//    its own.
// K, V, P and S are double buffered by chunk parity.  Signals per buffer
// b = chunk & 1: k_ready[b] (96 conversion threads: K tile and the token
// scale table written), v_ready[b] (the same threads: V tile written),
// s_free[b] / p_ready[b] (the active softmax threads), qk[b] / pv[b]
// (tcgen05.commit).  QK and the softmax wait only for k_ready, so a chunk's
// logits do not wait for its V tile, whose conversion waits for PV two chunks
// back.  A waiter never falls two phases behind: the next phase of each
// barrier needs a step that follows the wait (v_ready(j + 2) needs PV(j),
// issued after the issue warp saw v_ready(j); slot_free for chunk c + ring
// needs the refill issued after the wait for chunk c).

// conversion warps (4 measured slower than 3: large R = 8 0.96 against 0.93 ms)
#ifndef PA_Q8_UMMA_CONV_WARPS
#define PA_Q8_UMMA_CONV_WARPS 3
#endif
// warps 0-3 softmax, then the conversion warps, the issue warp, the refill warp
constexpr int kUmmaConvWarps = PA_Q8_UMMA_CONV_WARPS;
constexpr int kUmmaIssueWarp = 4 + kUmmaConvWarps;
constexpr int kUmmaRefillWarp = kUmmaIssueWarp + 1;
constexpr int kUmmaThreads = 32 * (kUmmaRefillWarp + 1);
// instruction-descriptor bit: the B operand is MN-major (N contiguous)
constexpr uint32_t kUmmaBMnMajor = 1u << 16;
constexpr int kUmmaConvThreads = 32 * kUmmaConvWarps;
// longest suspension of the issue warp on one pending input before it polls
// the other again (64 and 32 ns measured the same)
constexpr uint32_t kIssuePollNs = 256;

template <int D>
__host__ __device__ constexpr int umma_ring() { return 3; }
// TMEM columns: S twice (64), O (D), the Q tile (D / 2: two f16 per column)
template <int D>
__host__ __device__ constexpr uint32_t umma_tmem_cols() { return D == 256 ? 512u : 256u; }
// resident CTAs per SM: TMEM (512 columns) and registers (2 x 288 threads)
template <int D>
__host__ __device__ constexpr int umma_ctas_per_sm() { return D == 256 ? 1 : 2; }

// Byte offset of element (r, k) of an f16 operand tile with kdim columns in
// the K-major core-matrix layout (LBO = 128, SBO = kdim / 8 * 128).
__device__ __forceinline__ uint32_t kmaj_off(int r, int k, int kdim) {
    return (uint32_t)(((r >> 3) * (kdim >> 3) + (k >> 3)) * 128 + (r & 7) * 16 + (k & 7) * 2);
}

// barrier slots (8 bytes each) after the ring's
enum UmmaBar { kBarQk = 0, kBarPv = 2, kBarVReady = 4, kBarSFree = 6, kBarPReady = 8, kBarKReady = 10,
               kBarSlotFree = 12, kUmmaBars = 16 };     // slot_free: one per raw ring slot (ring <= 4)

struct UmmaLayout {
    uint32_t misc, scales, table, ops, ring, slot_bytes, total;
};

// [barriers: ring, kUmmaBars] [TMEM address, abort flag] [token scales 2 x
// (K, V) x 32] [table] [operand tiles Q, K x2, V x2, P x2] [raw chunk ring].
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
    static_assert(RING <= kUmmaBars - kBarSlotFree, "one slot_free barrier per raw ring slot");
    constexpr int W = D / 4 + 1;
    constexpr uint32_t TCOLS = umma_tmem_cols<D>();
    constexpr uint32_t Q_BYTES = 128u * D * 2, K_BYTES = 32u * D * 2, V_BYTES = (uint32_t)D * 32 * 2;
    constexpr uint32_t P_BYTES = 128u * kChunk * 2;
    constexpr uint32_t IDESC_QK = umma_idesc_f16(128, 32), IDESC_PV = umma_idesc_f16(128, D) | kUmmaBMnMajor;

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
        for (int k = 0; k < RING; ++k) {
            mbar_init(ring_bars + 8 * k, 1);
            mbar_init(bar(kBarSlotFree, k), kUmmaConvThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(kBarQk, b), 1);
            mbar_init(bar(kBarPv, b), 1);
            mbar_init(bar(kBarKReady, b), kUmmaConvThreads);
            mbar_init(bar(kBarVReady, b), kUmmaConvThreads);
            mbar_init(bar(kBarSFree, b), 32 * nquad);
            mbar_init(bar(kBarPReady, b), 32 * nquad);
        }
        *abort = 0u;
        fence_mbar_init();
    }
    // fused append: the newest tokens' vectors are stored (and fenced for the
    // async proxy) before the barrier that precedes the first bulk copy
    if (P.nk) append_tokens<D>(P, w);
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
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();                                  // barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<const volatile uint32_t *>(smem + L.misc);
    const uint32_t tO = tmem + 64;
    const uint32_t tQ = tO + D;                       // the Q tile: D / 2 columns
    float qk2 = 0.0f;
    if (warp < 4) {
        // Q row: q * 2^-eq as hi (or lo) f16, two per column of this thread's TMEM lane
        const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok ? vh : w.h0) * D);
        float mx = 0.0f;
        for (int c = 0; c < D / 4; ++c) {
            const float4 v = row_ok ? __ldg(qv + c) : make_float4(0.f, 0.f, 0.f, 0.f);
            mx = fmaxf(mx, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
        }
        const int eq = mx > 0.0f ? (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127 : 0;
        const float down = __uint_as_float((uint32_t)(127 - eq) << 23);      // 2^-eq
        qk2 = P.scale_log2 * __uint_as_float((uint32_t)(127 + min(eq, 127)) << 23);
        const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
        for (int c0 = 0; c0 < D / 2; c0 += 32) {
            float words[32];
#pragma unroll
            for (int j = 0; j < 32; j += 4) {                 // words c0 + j .. + 3: elements 2(c0 + j) .. + 7
                const int e4 = (2 * (c0 + j)) / 4;
                const float4 a = row_ok ? __ldg(qv + e4) : make_float4(0.f, 0.f, 0.f, 0.f);
                const float4 b = row_ok ? __ldg(qv + e4 + 1) : make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t h[4], l[4];
                split_f16x2(a.x * down, a.y * down, h[0], l[0]);
                split_f16x2(a.z * down, a.w * down, h[1], l[1]);
                split_f16x2(b.x * down, b.y * down, h[2], l[2]);
                split_f16x2(b.z * down, b.w * down, h[3], l[3]);
#pragma unroll
                for (int u = 0; u < 4; ++u) words[j + u] = __uint_as_float(lo_part ? l[u] : h[u]);
            }
            tmem_st32(tQ + lane_base + c0, words);
        }
    }
    tc_fence_before();
    __syncthreads();                                  // the Q tile is in TMEM
    tc_fence_after();

    // softmax state (warps 0-3) and the issuer's commit record (warp 7, lane 0)
    float m = -INFINITY, lsum = 0.0f;
    int E = 12;
    int last_commit = -1;            // barrier slot address offset of the newest commit, -1 none
    uint32_t last_parity = 0;
    int issued = 0;                  // chunks whose ring copy warp 8 started

    if (warp == kUmmaRefillWarp) {
        // ---- ring refills: the first RING chunks at once, then chunk c into
        // the slot of chunk c - RING once the conversion has read it
        for (; issued < nch; ++issued) {
            const int k = issued % RING;
            const bool ok = issued < RING ||
                            mbar_wait_abortable(bar(kBarSlotFree, k), ((issued - RING) / RING) & 1, abort);
            if (!__all_sync(0xFFFFFFFFu, ok)) break;          // issue_chunk is warp-collective
            issue_chunk<D>(P, w, table, issued, ring + k * L.slot_bytes, ring_bars + 8 * k, policy);
        }
    } else if (warp == kUmmaIssueWarp) {
        // ---- MMA issue.  Lane 0 polls the inputs and issues whichever MMA is
        // ready: QK(nq) once chunk nq's K tile is converted (and S buffer
        // nq & 1 was read), PV(np) once P(np) is written and V(np) is
        // converted.  No barrier runs two phases ahead of the poll: each one's
        // next phase needs an MMA this warp has not issued yet.
        int nq = 0, np = 0;                                   // next QK / PV to issue
        uint64_t idle_since = 0;
        uint32_t polls = 0;
        while (np < nch) {
            int act = 0;
            if (lane == 0) {
                if (nq < nch && mbar_try_wait(bar(kBarKReady, nq & 1), (nq >> 1) & 1) &&
                    (nq < 2 || mbar_try_wait(bar(kBarSFree, nq & 1), ((nq - 2) >> 1) & 1)))
                    act |= 1;
                bool p_ok = false;
                if (np < nq) {
                    p_ok = mbar_try_wait(bar(kBarPReady, np & 1), (np >> 1) & 1);
                    if (p_ok && mbar_try_wait(bar(kBarVReady, np & 1), (np >> 1) & 1)) act |= 2;
                }
                if (act == 0) {
                    // nothing ready: suspend briefly on the oldest pending input, then
                    // poll again; give up after the wait limit or on the CTA's abort
                    if (np < nq) {
                        if (p_ok) mbar_try_wait_suspend(bar(kBarVReady, np & 1), (np >> 1) & 1, kIssuePollNs);
                        else mbar_try_wait_suspend(bar(kBarPReady, np & 1), (np >> 1) & 1, kIssuePollNs);
                    } else {
                        mbar_try_wait_suspend(bar(kBarKReady, nq & 1), (nq >> 1) & 1, kIssuePollNs);
                    }
                    if (polls++ == 0) idle_since = global_timer_ns();
                    if ((polls & 15u) == 0) {
                        if (*abort) act = 4;
                        else if (global_timer_ns() - idle_since > kWaitLimitNs) {
                            *abort = 1u;
                            act = 4;
                        }
                    }
                } else {
                    polls = 0;
                }
            }
            act = __shfl_sync(0xFFFFFFFFu, act, 0);
            if (act & 4) break;
            if (lane == 0 && (act & 1)) {                        // S = Q . K(nq)^T
                tc_fence_after();
                const int b = nq & 1;
                const uint32_t aK = aK0 + b * K_BYTES, tS = tmem + 32 * b;
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks)
                    umma_f16_ta(tS, tQ + 8 * ks, umma_smem_desc(aK + ks * 256, 128, D * 16), IDESC_QK, ks > 0);
                umma_commit(bar(kBarQk, b));
                last_commit = kBarQk + b;
                last_parity = (nq >> 1) & 1;
            }
            if (lane == 0 && (act & 2)) {                        // O += P(np) . V(np)
                tc_fence_after();
                const int bj = np & 1;
                const uint32_t aP = aP0 + bj * P_BYTES, aV = aV0 + bj * V_BYTES;
                // V tile: token rows of D dims = the MN-major B layout, 8-token
                // blocks LBO = D * 16 bytes apart, 8-dim blocks SBO = 128 apart
                umma_f16(tO, umma_smem_desc(aP, 128, 512), umma_smem_desc(aV, D * 16, 128), IDESC_PV, np > 0);
                umma_f16(tO, umma_smem_desc(aP + 256, 128, 512), umma_smem_desc(aV + 2 * D * 16, D * 16, 128),
                         IDESC_PV, true);
                umma_commit(bar(kBarPv, bj));
                last_commit = kBarPv + bj;
                last_parity = (np >> 1) & 1;
            }
            if (act & 2) ++np;
            if (act & 1) ++nq;
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---- conversion (kUmmaConvThreads threads)
        const int ct = tid - 128;
        static_assert(kUmmaConvThreads % kChunk == 0, "conversion threads: whole warps per token lane");
        constexpr int kConvColStep = kUmmaConvThreads / kChunk;
        const int tok = ct % kChunk, col0 = ct / kChunk;
        const F16Consts fk;
        for (int i = 0; i < nch; ++i) {
            const int b = i & 1, k = i % RING;
            const uint32_t *rawK = reinterpret_cast<const uint32_t *>(smem + L.ring + k * L.slot_bytes);
            const uint32_t *rawV = rawK + kChunk * W;
            if (!mbar_wait_abortable(ring_bars + 8 * k, (i / RING) & 1, abort)) break;
            if (i >= 2 && !mbar_wait_abortable(bar(kBarQk, b), ((i - 2) >> 1) & 1, abort)) break;   // K tile free
            uint8_t *dK = sK0 + b * K_BYTES;
            // element u = ct + kUmmaConvThreads * k of the [8-code column][token]
            // walk: lane = token (8 bank groups); the thread count is a multiple
            // of 32, so this thread's token is fixed and its column steps by
            // kConvColStep (128 bytes each in the tile)
            {
                const uint32_t *src = rawK + tok * W;
                uint8_t *dst = dK + kmaj_off(tok, 0, D);
                for (int c8 = col0; c8 < D / 8; c8 += kConvColStep) {
                    uint32_t a0, a1, a2, a3;
                    codes4_to_f16x2(src[2 * c8], a0, a1, fk);
                    codes4_to_f16x2(src[2 * c8 + 1], a2, a3, fk);
                    *reinterpret_cast<uint4 *>(dst + 128 * c8) = make_uint4(a0, a1, a2, a3);
                }
            }
            // scale table b free: softmax(i-2) wrote P(i-2), after its last read of the table
            if (i >= 2 && !mbar_wait_abortable(bar(kBarPReady, b), ((i - 2) >> 1) & 1, abort)) break;
            if (ct < kChunk) ksc[b * kChunk + ct] = __uint_as_float(rawK[ct * W + D / 4]);
            else if (ct < 2 * kChunk) vsc[b * kChunk + ct - kChunk] = __uint_as_float(rawV[(ct - kChunk) * W + D / 4]);
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarKReady, b));
            // V tile b free: PV(i-2) done
            if (i >= 2 && !mbar_wait_abortable(bar(kBarPv, b), ((i - 2) >> 1) & 1, abort)) break;
            uint8_t *dV = sV0 + b * V_BYTES;
            {                                                 // as K: the PV B operand is MN-major
                const uint32_t *src = rawV + tok * W;
                uint8_t *dst = dV + kmaj_off(tok, 0, D);
                for (int c8 = col0; c8 < D / 8; c8 += kConvColStep) {
                    uint32_t a0, a1, a2, a3;
                    codes4_to_f16x2(src[2 * c8], a0, a1, fk);
                    codes4_to_f16x2(src[2 * c8 + 1], a2, a3, fk);
                    *reinterpret_cast<uint4 *>(dst + 128 * c8) = make_uint4(a0, a1, a2, a3);
                }
            }
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarVReady, b));
            mbar_arrive(bar(kBarSlotFree, k));                // raw slot k read for the last time
        }
    } else if (warp < nquad) {
        // ---- softmax (quadrant warp)
        const uint32_t lane_off = (uint32_t)(32 * warp) << 16;
        float wscale = __uint_as_float((uint32_t)(kVScaleBias + 127 - E) << 23);
        // chunks below every row's length in this warp need no masking (0 when a
        // lane holds no head: that warp always masks)
        const int len_full = (int)__reduce_min_sync(0xFFFFFFFFu, (unsigned)(row_ok ? len_row : 0));
        bool ok = true;
        for (int i = 0; ok && i < nch; ++i) {
            const int b = i & 1;
            ok = mbar_wait_abortable(bar(kBarQk, b), (i >> 1) & 1, abort);
            ok = ok && mbar_wait_abortable(bar(kBarKReady, b), (i >> 1) & 1, abort);   // the scale table
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
            // this thread's 16 token scales, as 16-byte vectors
            float ks[16], vs[16];
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
                const float4 a = reinterpret_cast<const float4 *>(ksc + b * kChunk + half)[q4];
                const float4 c = reinterpret_cast<const float4 *>(vsc + b * kChunk + half)[q4];
                ks[4 * q4] = a.x; ks[4 * q4 + 1] = a.y; ks[4 * q4 + 2] = a.z; ks[4 * q4 + 3] = a.w;
                vs[4 * q4] = c.x; vs[4 * q4 + 1] = c.y; vs[4 * q4 + 2] = c.z; vs[4 * q4 + 3] = c.w;
            }
            const int t0 = i * kChunk + half;
            float cmax = -INFINITY, vmax = 0.0f;
            if ((i + 1) * kChunk <= len_full) {                 // warp-uniform: every row sees the whole chunk
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    z[j] = z[j] * ks[j] * qk2;
                    cmax = fmaxf(cmax, z[j]);
                    vmax = fmaxf(vmax, vs[j]);
                }
            } else {
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const bool valid = t0 + j < len_row;
                    z[j] = valid ? z[j] * ks[j] * qk2 : -INFINITY;
                    vs[j] = valid ? vs[j] : 0.0f;
                    cmax = fmaxf(cmax, z[j]);
                    vmax = fmaxf(vmax, vs[j]);
                }
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
                    split_f16x2(p0 * vs[j] * wscale, p1 * vs[j + 1] * wscale, ph[e], pl[e]);
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
    if (failed && warp == kUmmaIssueWarp && lane == 0) {
        // stop only after the newest MMA (and so every earlier one) completed
        if (last_commit >= 0) mbar_wait(bars + 8 * last_commit, last_parity);
    }
    if (failed && warp == kUmmaRefillWarp && lane == 0) {
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
    merge_and_store<D, true>(P, w, ml, accs, 1, kUmmaHeads, accs + kUmmaHeads * D);
}

template <int D>
cudaError_t launch_umma(const Params &P, cudaStream_t st) {
    const UmmaLayout L = make_umma_layout<D>(P.PT, P.B);
    return launch_attn(decode_umma_kernel<D>, P, L.total, kUmmaThreads, st);
}

}  // namespace

cudaError_t launch_umma_family(const Params &P, int head_size, cudaStream_t st) {
    switch (head_size) {
        case 64: return launch_umma<64>(P, st);
        case 128: return launch_umma<128>(P, st);
        case 256: return launch_umma<256>(P, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa_q8
