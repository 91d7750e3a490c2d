// Decode over the contiguous q8 cache (per-sequence code rows and a side
// region of 32-element group scales): decode_cq_tma_kernel (head size 128,
// 3-D tensor copies) and decode_cq_kernel (head size 256).
#include "decode_common.cuh"

namespace pa_q8 {
namespace {

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

// [barriers] [ring, 1024-aligned at run time: slot x ring]: the ring starts
// at most 1023 bytes past the barriers.  About 73 KB, so three CTAs can share
// an SM (the build for three per SM is held to 168 registers for that).
__host__ __device__ inline uint32_t cq_tma_smem_bytes() {
    return align_up(PA_Q8_TC_SLOTS * kCqRing * 8u + 1023u + PA_Q8_TC_SLOTS * kCqRing * kCqTmaSlot, 128u);
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

// MINB: CTAs per SM the build is for (2 or 3; the plan picks one)
template <int D, int MINB>
__global__ void __launch_bounds__(PA_Q8_TC_SLOTS * 32, MINB)
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
    if (P.per_sm >= 3)
        return launch_attn_arg(decode_cq_tma_kernel<128, 3>, P, CP, cq_tma_smem_bytes(), PA_Q8_TC_SLOTS * 32, st);
    return launch_attn_arg(decode_cq_tma_kernel<128, 2>, P, CP, cq_tma_smem_bytes(), PA_Q8_TC_SLOTS * 32, st);
}

}  // namespace

cudaError_t launch_cq_family(const Params &P, int head_size, cudaStream_t st) {
    switch (head_size) {
        case 128: return launch_cq_tma(P, st);
        case 256: {
            const CqLayout L = make_cq_layout<256>();
            return launch_attn(decode_cq_kernel<256>, P, L.total, PA_Q8_TC_SLOTS * 32, st);
        }
        default: return cudaErrorInvalidValue;              // head sizes 128 and 256 only
    }
}

}  // namespace pa_q8
