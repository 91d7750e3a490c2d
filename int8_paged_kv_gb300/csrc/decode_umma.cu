// Multi-row decode on 5th-generation tensor cores: decode_umma_kernel
// (tcgen05.mma, f32 accumulators in TMEM, warp-specialised conversion,
// softmax and issue roles).
#include <type_traits>

#include "decode_common.cuh"

namespace pa_q8 {
namespace {

// ======================================================== tcgen05 (multi-row)
//
// Many virtual heads per kv head (multi-row decode: R query rows x r heads)
// make the contraction GEMM-shaped, so it runs on the 5th-generation tensor
// cores: one CTA serves up to 64 virtual heads of one kv head for one
// partition.
//
// Precision: K and V codes are exact in f16; q and the weights P are not, so
// each is split into an f16 hi part and the f16 residual (lo), about 22
// significant bits together (q scaled by 2^-eq per row first, like the
// mma.sync kernel).  The two parts are separate rows of the M = 128 MMAs:
// TMEM lane quadrant q holds rows 32q + j (j < 16: the hi part of virtual
// head 16q + j) and 32q + 16 + j (its lo part), for the Q tile (the A
// operand of S = Q.K^T, read from tensor memory: D / 2 columns, two f16 per
// column), for S (two chunk buffers of 32 columns) and for O (D columns),
// and the P tile in shared memory has the same rows.  A logit is the sum of
// its two rows, an output row the sum of its two O rows.
//
// Each softmax thread owns one virtual head and 16 of a chunk's 32 tokens:
// two 16x32bx2 loads (lane bases 32q and 32q + 16) give thread t the hi and
// the lo row of head 16q + t % 16 at tokens 16 (t / 16) .. + 15, so a logit
// is one paired add; the two threads of a head exchange only the chunk
// maximum and, at the end, their weight sums.  With 32 heads or fewer the
// softmax warps of quadrants without heads stay idle (giving them tokens
// 16-31 of each chunk on copies of the Q rows measured 2-4% slower).
//
// Warp roles, linked only by mbarriers (every wait bounded and abortable):
//  - warps 0-3, softmax: first the Q tile (row max -> 2^-eq -> hi/lo into
//    tensor memory, while the ring fills), then per chunk: S half-rows ->
//    online softmax with a lazy reference max (O rows rescaled in TMEM only
//    when it moves past 2^kLazy, or the weight scale changes) -> P half-rows
//    as hi and lo f16.  The per-logit arithmetic runs on f32 pairs.
//  - warps 4-6, conversion: per chunk the raw codes (bulk-copied ring, as in
//    the other families) become f16 K and V tiles [32 tokens][D] in the
//    core-matrix layout (K-major for QK's B, MN-major for PV's B).  Warps 4-5
//    convert K and write the chunk's scale table: the K scales, the V scales
//    times the weight scale 2^(131 - E) (E the largest V-scale exponent of
//    the partition so far), and E; tokens past the partition get scale 0.
//    Warp 6 converts V.  So a K tile never waits behind the V tile of the
//    chunk before, whose buffer frees only when PV two chunks back is done.
//  - warps 7 and 8: lane 0 of warp 8 issues S = Q.K^T, lane 0 of warp 7
//    O += P.V, each as soon as its inputs are ready.  A thread's MMAs run
//    one after another (about 25 ns each at these shapes), so the two
//    streams from two threads overlap.
//  - warp 9: refills the raw ring (four chunks), chunk c into the slot of
//    chunk c - 4 once both conversion groups have read it (slot_free[slot]).
// S, P and V tiles are double buffered by chunk parity b = chunk & 1; K tiles
// and scale tables are four deep, b4 = chunk & 3.  Signals: k_ready[b4]
// (warps 4-5: K tile and scale table written), qk[b4] (tcgen05.commit of
// QK), p_ready[b4] (the active softmax threads: P written, so the table is
// free), s_free[b] (S read), v_ready[b] (warp 6: V tile written), pv[b]
// (commit of PV), and q_ready once (the 128 softmax threads: Q tile stored).
// QK and the softmax wait only for k_ready, so a chunk's logits do not wait
// for its V tile, whose conversion waits for PV two chunks back.  A waiter
// never falls two phases behind: the next phase of each barrier needs a step
// that follows the wait (v_ready(j + 2) needs PV(j), issued after the issue
// warp saw v_ready(j); k_ready(j + 4) needs p_ready(j), which the softmax
// gives after its wait for k_ready(j); slot_free for chunk c + 4 needs the
// refill issued after the wait for chunk c).

// Warp roles: 0-3 softmax, 4-5 K conversion (and the scale tables), 6 V
// conversion, 7 PV issue, 8 QK issue, 9 ring refill.  Ten warps: two CTAs
// per SM then put at most five warps on an SM sub-partition, which leaves
// 96 registers a thread.
constexpr int kUmmaKConvWarps = 2;                        // one for the K scales, one for the V scales
constexpr int kUmmaVConvWarps = 1;
constexpr int kUmmaKConvThreads = 32 * kUmmaKConvWarps;
constexpr int kUmmaVConvThreads = 32 * kUmmaVConvWarps;
constexpr int kUmmaConvThreads = kUmmaKConvThreads + kUmmaVConvThreads;
// (Warp w runs on SM sub-partition w % 4; other placements of the K, V and
// PV warps measured within 1%.)
constexpr int kUmmaKWarp0 = 4, kUmmaVWarp = 6, kUmmaPvWarp = 7;
constexpr int kUmmaQkWarp = 8;
constexpr int kUmmaRefillWarp = 9;
constexpr int kUmmaThreads = 32 * (kUmmaRefillWarp + 1);
static_assert(kUmmaKConvWarps == 2 && kUmmaVConvWarps == 1, "the role table above");
// instruction-descriptor bit: the B operand is MN-major (N contiguous)
constexpr uint32_t kUmmaBMnMajor = 1u << 16;
static_assert(kUmmaHeads == 64, "64 virtual heads: hi and lo rows of one M = 128 tile");

template <int D>
// raw chunks in flight per CTA (4: 2-3% faster than 3 on the large batch at 32
// and 64 pairs; 5 no faster)
__host__ __device__ constexpr int umma_ring() { return 4; }
// TMEM columns: S twice (64), O (D), the Q tile (D / 2)
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
// K tiles and scale tables are kept for kKDepth chunks (their signals qk,
// k_ready and p_ready too), so the K conversion runs up to four chunks ahead
// of the softmax; S, P and V tiles are double buffered.
constexpr int kKDepth = 4;      // measured 1-2% faster than 2 deep (large R = 8, 4, long R = 8)
// V tiles (and their signals pv, v_ready) are kept for kVDepth chunks (3 or 4
// deep measured no faster than 2 with the four-chunk ring)
constexpr int kVDepth = 2;
enum UmmaBar { kBarQk = 0, kBarPv = 4, kBarVReady = 8, kBarSFree = 12, kBarPReady = 14, kBarKReady = 18,
               kBarQReady = 22, kBarSlotFree = 23, kUmmaBars = 31 };   // slot_free: one per raw ring slot (ring <= 8)

struct UmmaLayout {
    uint32_t misc, scales, table, ops, ring, slot_bytes, total;
};

// [barriers: ring, kUmmaBars] [TMEM address, abort flag] [scale tables: K
// 4 x 32, weighted V 4 x 32, E 4] [block table] [operand tiles K x4, V x2,
// P x2] [raw chunk ring].  Total at least a 1/(n+1) share of the
// shared memory, so no more CTAs share an SM than its TMEM serves.
template <int D>
__host__ __device__ inline UmmaLayout make_umma_layout(int PT, int B) {
    constexpr int RING = umma_ring<D>();
    UmmaLayout L{};
    const int ptok = B < kChunk ? B : kChunk;
    const int pieces = (PT + ptok - 1) / ptok + 1;
    L.misc = (RING + kUmmaBars) * 8;
    L.scales = align_up(L.misc + 8, 16);
    L.table = L.scales + align_up(kKDepth * (2 * kChunk * 4 + 4), 16);
    L.ops = align_up(L.table + pieces * 4, 128);
    const uint32_t ops_bytes = kKDepth * 32u * D * 2 + kVDepth * (uint32_t)D * 32 * 2 + 2u * 128u * kChunk * 2;
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
    static_assert(64 + D + D / 2 <= (int)TCOLS, "S twice, O and the Q tile in the allocation");
    constexpr uint32_t K_BYTES = 32u * D * 2, V_BYTES = (uint32_t)D * 32 * 2;
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
    float *ksc = reinterpret_cast<float *>(smem + L.scales);           // [4][32] K scales x scale x log2(e)
    float *vwc = ksc + kKDepth * kChunk;                                 // [4][32] V scales x 2^(131 - E)
    int *ecc = reinterpret_cast<int *>(vwc + kKDepth * kChunk);          // [4] E
    const uint32_t *table = reinterpret_cast<const uint32_t *>(smem + L.table);
    uint8_t *sK0 = smem + L.ops, *sV0 = sK0 + kKDepth * K_BYTES, *sP0 = sV0 + kVDepth * V_BYTES;
    const uint32_t aK0 = s0 + L.ops, aV0 = aK0 + kKDepth * K_BYTES, aP0 = aV0 + kVDepth * V_BYTES;
    const uint32_t ring = s0 + L.ring;
    const uint64_t policy = l2_policy_evict_first();
    const int nsoft = min(4, (w.nh + 15) / 16);          // softmax warps with work
    const int nch = (w.len + kChunk - 1) / kChunk;

    // softmax threads: virtual head hl (M row) and token half of each chunk
    const int qd = warp & 3;                             // TMEM lane quadrant
    const int hl = 16 * qd + (lane & 15);
    const int half = lane >> 4;
    const bool row_ok = warp < 4 && hl < w.nh;
    const bool soft_active = warp < nsoft;
    const int vh = w.h0 + hl;
    const int len_row = row_ok ? row_len(P, w, vh) : 0;
    if (warp == 0) tmem_alloc(tmem_slot, TCOLS);
    // Q rows: the softmax warps load their q elements first, so the loads
    // overlap the setup below.  Thread t covers, in each 64-element block k
    // of its head's q, elements 64k + 32 (t / 16) .. + 31, which become TMEM
    // words 32k + 16 (t / 16) .. + 15 of the head's hi row and of its lo row.
    // The loads here only give each row's largest magnitude.
    // q is scaled by 2^-eq, eq the row's largest exponent kept within the
    // normal range, so the f16 parts keep their bits; logits are
    // (q 2^-eq . k) (k scale x scale x log2 e) x 2^eq.  The blocks are read
    // again (from L1) for the split once the TMEM is allocated (keeping the
    // split words in registers instead measured 1-2% slower: 96 registers).
    constexpr int NBLK = D / 64;                      // 64-element blocks (head size 64: one)
    const float4 *qv = reinterpret_cast<const float4 *>(P.q + qrow(P, w, row_ok ? vh : w.h0) * D) + 8 * half;
    float qk2 = 1.0f, qdown = 1.0f;                   // the row's 2^eq and 2^-eq
    if (warp < 4) {
        float4 v[8 * NBLK];
#pragma unroll
        for (int k = 0; k < NBLK; ++k)
#pragma unroll
            for (int u = 0; u < 8; ++u)
                v[8 * k + u] = row_ok ? __ldg(qv + 16 * k + u) : make_float4(0.f, 0.f, 0.f, 0.f);
        float mx = 0.0f;
#pragma unroll
        for (int c = 0; c < 8 * NBLK; ++c)
            mx = max3f(mx, fmaxf(fabsf(v[c].x), fabsf(v[c].y)), fmaxf(fabsf(v[c].z), fabsf(v[c].w)));
        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
        const int eq = mx > 0.0f ? max(-126, min(126, (int)((__float_as_uint(mx) >> 23) & 0xFF) - 127)) : 0;
        qdown = __uint_as_float((uint32_t)(127 - eq) << 23);
        qk2 = __uint_as_float((uint32_t)(127 + eq) << 23);
    }
    if (tid == 0) {
        for (int k = 0; k < RING; ++k) {
            mbar_init(ring_bars + 8 * k, 1);
            mbar_init(bar(kBarSlotFree, k), kUmmaConvThreads);
        }
        for (int b = 0; b < kKDepth; ++b) {
            mbar_init(bar(kBarQk, b), 1);
            mbar_init(bar(kBarKReady, b), kUmmaKConvThreads);
            mbar_init(bar(kBarPReady, b), 32 * nsoft);
        }
        for (int b = 0; b < kVDepth; ++b) {
            mbar_init(bar(kBarPv, b), 1);
            mbar_init(bar(kBarVReady, b), kUmmaVConvThreads);
        }
        for (int b = 0; b < 2; ++b) mbar_init(bar(kBarSFree, b), 32 * nsoft);
        mbar_init(bar(kBarQReady, 0), 128);
        *abort = 0u;
        fence_mbar_init();
    }
    // fused append: the newest tokens' vectors are stored (and fenced for the
    // async proxy) before the barrier that precedes the first bulk copy
    if (P.nk) append_tokens<D>(P, w);
    load_table(P, w, const_cast<uint32_t *>(table));
    for (int i = tid; i < 2 * (int)P_BYTES / 16; i += kUmmaThreads)    // P rows of heads that do not exist stay 0
        reinterpret_cast<uint4 *>(sP0)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();                                  // barriers initialised, TMEM allocated
    tc_fence_after();
    const uint32_t tmem = *reinterpret_cast<const volatile uint32_t *>(smem + L.misc);
    const uint32_t tO = tmem + 64;
    const uint32_t tQ = tO + D;                       // the Q tile: D / 2 columns

    const uint32_t lane_hi = (uint32_t)(32 * (warp & 3)) << 16;        // the quadrant's hi rows
    const uint32_t lane_lo = (uint32_t)(32 * (warp & 3) + 16) << 16;   // and its lo rows

    // softmax state (warps 0-3) and the issuers' commit records (lane 0)
    float m = -INFINITY;
    float2 lsum = make_float2(0.0f, 0.0f);
    int E = 12;
    int last_commit = -1;            // barrier slot address offset of the newest commit, -1 none
    uint32_t last_parity = 0;
    int issued = 0;                  // chunks whose ring copy the refill warp started

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
    } else if (warp == kUmmaQkWarp || warp == kUmmaPvWarp) {
        // ---- MMA issue, one warp per stream (a thread's MMAs run one after
        // the other, so QK and PV from two threads overlap).  Lane 0 waits for
        // the inputs and issues:
        //  QK(c) once chunk c's K tile is converted and S buffer c & 1 was read
        //  PV(c) once P(c) is written and V(c) is converted.
        // (b: the double buffers of S, P, V; b4: those of K tiles and tables)
        // No barrier runs two phases ahead of a wait: each one's next phase
        // needs an MMA of this stream that is not issued yet.
        const bool qk = warp == kUmmaQkWarp;
        bool ok = __all_sync(0xFFFFFFFFu, !qk || mbar_wait_abortable(bar(kBarQReady, 0), 0, abort));
        for (int c = 0; ok && c < nch; ++c) {
            const int b = c & 1, b4 = c & (kKDepth - 1);
            const uint32_t par = (c >> 1) & 1, par4 = (c / kKDepth) & 1;
            if (lane == 0) {
                if (qk) {
                    ok = mbar_wait_abortable(bar(kBarKReady, b4), par4, abort) &&
                         (c < 2 || mbar_wait_abortable(bar(kBarSFree, b), par ^ 1, abort));
                } else {
                    ok = mbar_wait_abortable(bar(kBarPReady, b4), par4, abort) &&
                         mbar_wait_abortable(bar(kBarVReady, c % kVDepth), (c / kVDepth) & 1, abort);
                }
            }
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
            if (!ok) break;
            if (lane == 0) {
                tc_fence_after();
                if (qk) {                                          // S = Q . K(c)^T, Q from TMEM
                    const uint32_t aK = aK0 + b4 * K_BYTES, tS = tmem + 32 * b;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks)
                        umma_f16_ta(tS, tQ + 8 * ks, umma_smem_desc(aK + ks * 256, 128, 16 * D), IDESC_QK, ks > 0);
                    umma_commit(bar(kBarQk, b4));
                    last_commit = kBarQk + b4;
                    last_parity = par4;
                } else {                                           // O += P(c) . V(c)
                    const uint32_t aP = aP0 + b * P_BYTES, aV = aV0 + (c % kVDepth) * V_BYTES;
                    // V tile: token rows of D dims = the MN-major B layout, 8-token
                    // blocks LBO = D * 16 bytes apart, 8-dim blocks SBO = 128 apart;
                    // k-steps 0, 1: tokens 0-15, 16-31
                    umma_f16(tO, umma_smem_desc(aP, 128, 512), umma_smem_desc(aV, D * 16, 128), IDESC_PV, c > 0);
                    umma_f16(tO, umma_smem_desc(aP + 256, 128, 512), umma_smem_desc(aV + 2 * D * 16, D * 16, 128),
                             IDESC_PV, true);
                    umma_commit(bar(kBarPv, c % kVDepth));
                    last_commit = kBarPv + c % kVDepth;
                    last_parity = (c / kVDepth) & 1;
                }
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ---- conversion: K group (warps 4-5) and V group (warp 6).  A tile
        // is 32 tokens x D / 8 columns of 8 codes; thread g of a group takes
        // token g % 32 (lane = token: conflict-free reads of the 33-word rows
        // and 128-byte runs of core-matrix rows) and columns g / 32 + gw k, gw
        // the group's warps, eight columns' loads in flight at a time.
        const bool kgroup = warp >= kUmmaKWarp0 && warp < kUmmaKWarp0 + kUmmaKConvWarps;
        const int g = kgroup ? tid - 32 * kUmmaKWarp0 : tid - 32 * kUmmaVWarp;
        const int gw = kgroup ? kUmmaKConvWarps : kUmmaVConvWarps;
        static_assert(kUmmaKConvThreads >= 2 * kChunk, "one K-group thread per K scale and per V scale");
        static_assert((D / 8) % kUmmaKConvWarps == 0 && (D / 8) % kUmmaVConvWarps == 0, "whole columns per warp");
        const int tok = g % kChunk, col0 = g / kChunk;
        const F16Consts fk;
        auto convert_tile = [&](auto ncols_c, const uint32_t *raw, uint8_t *tile) {
            constexpr int ncols = decltype(ncols_c)::value;      // columns per thread and tile
            const uint32_t *src = raw + tok * W;
            uint8_t *dst = tile + kmaj_off(tok, 0, D);
#pragma unroll
            for (int k0 = 0; k0 < ncols; k0 += 8) {
                uint32_t wd[16];
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int c8 = col0 + gw * (k0 + k);
                    if (k0 + k < ncols) {
                        wd[2 * k] = src[2 * c8];
                        wd[2 * k + 1] = src[2 * c8 + 1];
                    }
                }
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (k0 + k < ncols) {
                        uint32_t a0, a1, a2, a3;
                        codes4_to_f16x2(wd[2 * k], a0, a1, fk);
                        codes4_to_f16x2(wd[2 * k + 1], a2, a3, fk);
                        *reinterpret_cast<uint4 *>(dst + 128 * (col0 + gw * (k0 + k))) = make_uint4(a0, a1, a2, a3);
                    }
                }
            }
        };
        int Ew = 12;                                           // weight-scale exponent (second K warp)
        for (int i = 0; i < nch; ++i) {
            const int k = i % RING;
            const uint32_t *rawK = reinterpret_cast<const uint32_t *>(smem + L.ring + k * L.slot_bytes);
            const uint32_t *rawV = rawK + kChunk * W;
            // every wait's outcome is made warp-uniform: a K-group warp reduces over its lanes
            if (!__all_sync(0xFFFFFFFFu, mbar_wait_abortable(ring_bars + 8 * k, (i / RING) & 1, abort))) break;
            if (kgroup) {
                const int b4 = i & (kKDepth - 1);
                const uint32_t prev4 = ((i / kKDepth) & 1) ^ 1;   // the phase of chunk i - kKDepth
                if (i >= kKDepth && !__all_sync(0xFFFFFFFFu, mbar_wait_abortable(bar(kBarQk, b4), prev4, abort)))
                    break;                                    // K tile free: QK(i - 4) done
                convert_tile(std::integral_constant<int, D / 8 / kUmmaKConvWarps>(), rawK, sK0 + b4 * K_BYTES);
                // scale table b4 free: softmax(i-4) wrote P(i-4), after its last read of the table
                if (i >= kKDepth &&
                    !__all_sync(0xFFFFFFFFu, mbar_wait_abortable(bar(kBarPReady, b4), prev4, abort)))
                    break;
                const int tk = i * kChunk;                      // partition-relative first token
                if (g < kChunk) {                               // K scale x scale x log2(e)
                    ksc[b4 * kChunk + g] = tk + g < w.len ? __uint_as_float(rawK[g * W + D / 4]) * P.scale_log2 : 0.0f;
                } else if (g < 2 * kChunk) {                    // one whole warp: the V scales
                    const int t = g - kChunk;
                    const float vs = tk + t < w.len ? __uint_as_float(rawV[t * W + D / 4]) : 0.0f;
                    const int ev = (int)(__float_as_uint(fmaxf(vs, 0.0f)) >> 23);
                    Ew = max(Ew, (int)__reduce_max_sync(0xFFFFFFFFu, (unsigned)ev));
                    vwc[b4 * kChunk + t] = vs * __uint_as_float((uint32_t)(kVScaleBias + 127 - Ew) << 23);
                    if (t == 0) ecc[b4] = Ew;
                }
                fence_proxy_async_smem();
                mbar_arrive(bar(kBarKReady, b4));
            } else {
                // V tile b free: PV(i-2) done
                const int bv = i % kVDepth;                     // V tile bv free: PV(i - kVDepth) done
                if (i >= kVDepth &&
                    !__all_sync(0xFFFFFFFFu, mbar_wait_abortable(bar(kBarPv, bv), ((i / kVDepth) & 1) ^ 1, abort)))
                    break;
                // as K: the PV B operand is MN-major
                convert_tile(std::integral_constant<int, D / 8 / kUmmaVConvWarps>(), rawV, sV0 + bv * V_BYTES);
                fence_proxy_async_smem();
                mbar_arrive(bar(kBarVReady, bv));
            }
            mbar_arrive(bar(kBarSlotFree, k));                // raw slot k read for the last time (by this group)
        }
    } else {
        // ---- softmax warps: the Q tile first (all four warps; rows of heads
        // that do not exist are written as zeros), as 16x32bx2 stores at lane
        // bases 32q (hi rows) and 32q + 16 (lo rows)
        {
#pragma unroll 1
            for (int k = 0; k < NBLK; ++k) {
                float4 v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) v[u] = row_ok ? __ldg(qv + 16 * k + u) : make_float4(0.f, 0.f, 0.f, 0.f);
                uint32_t hw[16], lw[16];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const float4 a = v[u];
                    split_f16x2_fma(a.x * qdown, a.y * qdown, hw[2 * u], lw[2 * u]);
                    split_f16x2_fma(a.z * qdown, a.w * qdown, hw[2 * u + 1], lw[2 * u + 1]);
                }
                tmem_st16x2_nowait(tQ + lane_hi + 32 * k, hw);
                tmem_st16x2_nowait(tQ + lane_lo + 32 * k, lw);
            }
            tmem_wait_st();
            tc_fence_before();
            mbar_arrive(bar(kBarQReady, 0));
        }
        if (soft_active) {
            // ---- softmax (this warp's 16 pairs)
            // chunks below every row's length in this warp need no masking (0 when a
            // lane holds no pair: that warp always masks)
            const int len_full = (int)__reduce_min_sync(0xFFFFFFFFu, (unsigned)(row_ok ? len_row : 0));
            const int row_h = 32 * qd + (lane & 15), row_l = row_h + 16;   // this pair's hi and lo rows
            bool ok = true;
            // NT = 16 tokens of each chunk per thread (tokens 16 half ..)
            auto run = [&]() {
                constexpr int NT = 16;
                constexpr int NP = NT / 2;
                const int tok0 = 16 * half;
                // this thread's P tile words: hi row then lo row, 8 tokens per 16 bytes
                uint32_t p_off[NT / 4];
#pragma unroll
                for (int k = 0; k < NT / 8; ++k) {
                    p_off[k] = kmaj_off(row_h, tok0 + 8 * k, kChunk);
                    p_off[NT / 8 + k] = kmaj_off(row_l, tok0 + 8 * k, kChunk);
                }
                for (int i = 0; ok && i < nch; ++i) {
                    const int b = i & 1, b4 = i & (kKDepth - 1);
                    const uint32_t par4 = (i / kKDepth) & 1;
                    ok = mbar_wait_abortable(bar(kBarQk, b4), par4, abort);
                    ok = ok && mbar_wait_abortable(bar(kBarKReady, b4), par4, abort);   // the scale table
                    if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    tc_fence_after();
                    float zh[NT], zl[NT];                        // this pair's hi and lo rows at its tokens
                    tmem_ld16x2(tmem + 32 * b + lane_hi, zh);
                    tmem_ld16x2(tmem + 32 * b + lane_lo, zl);
                    tc_fence_before();
                    mbar_arrive(bar(kBarSFree, b));
                    float ks[NT], vw[NT];
#pragma unroll
                    for (int q4 = 0; q4 < NT / 4; ++q4) {
                        const float4 a = reinterpret_cast<const float4 *>(ksc + b4 * kChunk + tok0)[q4];
                        const float4 c = reinterpret_cast<const float4 *>(vwc + b4 * kChunk + tok0)[q4];
                        ks[4 * q4] = a.x; ks[4 * q4 + 1] = a.y; ks[4 * q4 + 2] = a.z; ks[4 * q4 + 3] = a.w;
                        vw[4 * q4] = c.x; vw[4 * q4 + 1] = c.y; vw[4 * q4 + 2] = c.z; vw[4 * q4 + 3] = c.w;
                    }
                    const int Ei = ecc[b4];
                    float2 t2[NP];                               // z x k scale x scale x log2 e; -inf where masked
#pragma unroll
                    for (int u = 0; u < NP; ++u)
                        t2[u] = mul_f2(add_f2(make_float2(zh[2 * u], zh[2 * u + 1]), make_float2(zl[2 * u], zl[2 * u + 1])),
                                       make_float2(ks[2 * u], ks[2 * u + 1]));
                    if ((i + 1) * kChunk > len_full) {           // warp-uniform: some row ends in this chunk
                        const int t0 = i * kChunk + tok0;
#pragma unroll
                        for (int u = 0; u < NP; ++u) {
                            if (t0 + 2 * u >= len_row) t2[u].x = -INFINITY;
                            if (t0 + 2 * u + 1 >= len_row) t2[u].y = -INFINITY;
                        }
                    }
                    // a tree of three-input maxima
                    const float c0 = max3f(t2[0].x, t2[0].y, t2[1].x), c1 = max3f(t2[1].y, t2[2].x, t2[2].y);
                    const float c2 = max3f(t2[3].x, t2[3].y, t2[4].x), c3 = max3f(t2[4].y, t2[5].x, t2[5].y);
                    const float c4 = max3f(t2[6].x, t2[6].y, t2[7].x);
                    float cmax = fmaxf(max3f(c0, c1, c2), max3f(c3, c4, t2[7].y));
                    cmax = fmaxf(cmax, __shfl_xor_sync(0xFFFFFFFFu, cmax, 16));   // the pair's other tokens
                    const float cm = cmax * qk2;                 // qk2 = 2^eq > 0: the max of the logits
                    // the same decision in both threads of a pair (same cm, m, E)
                    const bool need = cm > m + (float)kLazy || Ei > E;
                    float fa = 1.0f;
                    if (need) {
                        const float m_new = fmaxf(m, cm);
                        const float alpha = (m == -INFINITY) ? 0.0f : fast_exp2(m - m_new);
                        const float ea = (E - Ei < -126) ? 0.0f : __uint_as_float((uint32_t)(127 + E - Ei) << 23);
                        fa = alpha * ea;
                        lsum.x *= alpha;
                        lsum.y *= alpha;
                        m = m_new;
                        E = Ei;
                    }
                    if (i >= 1 && __any_sync(0xFFFFFFFFu, need)) {  // O rows once PV(i-1) is done
                        ok = mbar_wait_abortable(bar(kBarPv, (i - 1) % kVDepth), ((i - 1) / kVDepth) & 1, abort);
                        if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                        tc_fence_after();
#pragma unroll 1
                        for (int c = 0; c < D / 16; ++c) {            // hi rows, then lo rows
                            const uint32_t a = tO + (c & 1 ? lane_lo : lane_hi) + 32 * (c >> 1);
                            float o[16];
                            tmem_ld16x2(a, o);
#pragma unroll
                            for (int j = 0; j < 16; ++j) o[j] *= fa;
                            tmem_st16x2(a, o);
                        }
                    }
                    if (i >= 2) {                                   // P tile b free: PV(i-2) done
                        ok = mbar_wait_abortable(bar(kBarPv, (i - 2) % kVDepth), ((i - 2) / kVDepth) & 1, abort);
                        if (!__all_sync(0xFFFFFFFFu, ok)) { ok = false; break; }
                    }
                    const float m_ref = m == -INFINITY ? 0.0f : m;
                    const float2 q2 = make_float2(qk2, qk2), nm2 = make_float2(-m_ref, -m_ref);
                    uint32_t ph[NP], pl[NP];
                    float2 pp[NP];
#pragma unroll
                    for (int u = 0; u < NP; ++u) {
                        const float2 a = fma_f2(t2[u], q2, nm2);    // masked tokens: 2^-inf = 0
                        pp[u] = make_float2(fast_exp2(a.x), fast_exp2(a.y));
                        const float2 pw = mul_f2(pp[u], make_float2(vw[2 * u], vw[2 * u + 1]));
                        split_f16x2_fma(pw.x, pw.y, ph[u], pl[u]);
                    }
                    // the chunk's weights summed as a tree, then added to the row's sum
                    lsum = add_f2(lsum, add_f2(add_f2(add_f2(pp[0], pp[1]), add_f2(pp[2], pp[3])),
                                               add_f2(add_f2(pp[4], pp[5]), add_f2(pp[6], pp[7]))));
                    uint8_t *dP = sP0 + b * P_BYTES;
#pragma unroll
                    for (int k = 0; k < NT / 8; ++k) {
                        *reinterpret_cast<uint4 *>(dP + p_off[k]) =
                            make_uint4(ph[4 * k], ph[4 * k + 1], ph[4 * k + 2], ph[4 * k + 3]);
                        *reinterpret_cast<uint4 *>(dP + p_off[NT / 8 + k]) =
                            make_uint4(pl[4 * k], pl[4 * k + 1], pl[4 * k + 2], pl[4 * k + 3]);
                    }
                    fence_proxy_async_smem();
                    tc_fence_before();
                    mbar_arrive(bar(kBarPReady, b4));
                }
            };
            run();
            // the last PV, then this thread's half of its pair's output row (hi +
            // lo rows of O), normalised (one partition) or as the partition's
            // record (m, l and the unnormalised row in the V scales' units)
            if (ok) ok = mbar_wait_abortable(bar(kBarPv, (nch - 1) % kVDepth), ((nch - 1) / kVDepth) & 1, abort);
            if (__all_sync(0xFFFFFFFFu, ok)) {
                tc_fence_after();
                const float l_half = lsum.x + lsum.y;
                const float l_row = l_half + __shfl_xor_sync(0xFFFFFFFFu, l_half, 16);
                const float fE = m == -INFINITY ? 0.0f : ldexpf(1.0f, E - kVScaleBias);   // O = 2^(131-E) sum p v
                float f = fE;
                float *dst = nullptr;
                if (row_ok) {
                    const int64_t qr = qrow(P, w, vh);
                    if (w.single) {
                        // a query row that sees no token (l = 0) gets a zero row
                        f = l_row > 0.0f ? fE / l_row : 0.0f;
                        dst = P.out + qr * D;
                    } else {
                        dst = P.part + (qr * P.NP + w.p) * (D + 4);
                        if (half == 0) {
                            dst[D] = m;
                            dst[D + 1] = l_row;
                        }
                    }
                }
                for (int c = 0; c < D / 32; ++c) {
                    float oh[16], ol[16];
                    tmem_ld16x2(tO + lane_hi + 32 * c, oh);
                    tmem_ld16x2(tO + lane_lo + 32 * c, ol);
                    if (dst) {
                        float4 *d4 = reinterpret_cast<float4 *>(dst + 32 * c + 16 * half);
#pragma unroll
                        for (int j = 0; j < 4; ++j)
                            d4[j] = make_float4((oh[4 * j] + ol[4 * j]) * f, (oh[4 * j + 1] + ol[4 * j + 1]) * f,
                                                (oh[4 * j + 2] + ol[4 * j + 2]) * f, (oh[4 * j + 3] + ol[4 * j + 3]) * f);
                    }
                }
            } else {
                *abort = 1u;
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    const bool failed = *abort != 0u;
    if (failed && (warp == kUmmaQkWarp || warp == kUmmaPvWarp) && lane == 0) {
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
    // split context: the records are out; the last CTA of the group merges
    // them, with the operand tiles and the (drained) ring as scratch
    if (!w.single) arrive_and_combine<D, true>(P, w, sK0);
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
