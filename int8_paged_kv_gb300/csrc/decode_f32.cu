// Decode over the f32 cache [blocks][Hk][B][D]: decode_f32_kernel, K/V
// tiles by 2-D tensor copies with the 128-byte swizzle, CUDA-core dot
// products.
#include "decode_common.cuh"

namespace pa_q8 {
namespace {

// ============================================================== f32 cache
//
// The f32 variant of the cache, token vectors of head_size f32 values and no
// scale word: [num_blocks][Hk][B][D] f32 (the q8 layout with f32 elements;
// "paged_attn_q8.comp" names "paged_attn.comp" as the same math over an f32
// cache).  CUDA cores, with the CUDA-core family's streams, softmax and merge.
//
// Tiles move with 2-D tensor copies over the cache seen as rows of D floats:
// one box is 32 floats (128 B) of min(B, 16) rows, copied with the 128-byte
// swizzle, so 16-byte chunk c of token row t lands at chunk c ^ (t % 8) of
// that row's 128 bytes.  A chunk of 16 tokens keeps a warp's K and V buffers
// at 2 * 16 * D * 4 bytes, so 12 token-stream warps share an SM at head size
// 128 (latency hiding for the FMA-bound GQA-8 case).  A buffer holds [D/32
// segments][16 tokens][32 floats].  QK: lane = (token, half of the head
// dims); eight lanes reading one chunk index touch eight bank groups thanks
// to the swizzle, and one shuffle adds the two halves' partial dots.  PV:
// lane = 4 head dims.  Each warp owns chunks ts, ts + SLOTS, ...; the K and V
// halves of its buffer have their own mbarrier, so the next chunk's keys are
// in flight during this chunk's PV and its values during the next QK.

// Token-stream warps per CTA: a warp's K and V chunk buffers take 2 * 16 * D
// * 4 bytes (16 KB at head size 128), so 12 of them fill about 200 KB.
template <int D>
__host__ __device__ constexpr int f32_slots() { return D == 256 ? 6 : 12; }

constexpr int kF32Chunk = 16;                           // tokens per chunk
constexpr uint32_t kF32SegBytes = kF32Chunk * 128;      // one 32-float column of a chunk

struct F32Params {
    Params p;
    CUtensorMap tk;        // the key cache as [rows = num_blocks * Hk * B][D] f32
    CUtensorMap tv;
};

// shared memory beside the buffers: q rows [NH][D], weights [slot][NH][32], row lags [NH]
template <int D, int NH>
__host__ __device__ constexpr uint32_t f32_extra() { return NH * D * 4 + f32_slots<D>() * kF32Chunk * NH * 4 + NH * 4; }

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
    L.half_bytes = (uint32_t)kF32Chunk * D * 4;
    L.total = L.ring + 2u * slots * L.half_bytes + 1024u;
    return L;
}

// Copy the K or V half of chunk c (16 tokens): lane = (piece of min(B, 16)
// tokens, 32-float column), one tensor copy each.  Pieces past the
// partition's end or in an out-of-range block are not copied (their rows are
// never used as values, or the block was flagged by the table walk).  The
// table holds one block per min(B, 32) tokens, so a piece lies in one entry.
template <int D>
__device__ __forceinline__ void issue_f32_half(const Params &P, const Work &w, const uint32_t *table,
                                               const CUtensorMap *tmap, int c, uint32_t dst, uint32_t bar,
                                               uint64_t policy) {
    constexpr int NSEG = D / 32;
    const int lane = threadIdx.x & 31;
    const int log2f = min(P.log2B, 4);                      // box rows: min(B, 16)
    const int piece = lane / NSEG, seg = lane % NSEG;
    const int t = c * kF32Chunk + (piece << log2f);         // partition-relative token
    bool go = false;
    int y = 0;
    if (piece < (kF32Chunk >> log2f) && t < w.len) {
        const uint32_t pb = table[t >> P.log2ptok];
        if (pb != kPadSlot) {
            const int off = (w.t_begin + t) & (P.B - 1);
            y = (int)((((int64_t)pb * P.Hk + w.g) << P.log2B) + off);
            go = true;
        }
    }
    const uint32_t bytes = go ? 128u << log2f : 0u;
    const uint32_t total = __reduce_add_sync(0xFFFFFFFFu, bytes);
    if (lane == 0) mbar_arrive_expect_tx(bar, total);
    __syncwarp();
    if (go) {
        fence_proxy_async_smem();
        tma_load_2d(dst + seg * kF32SegBytes + ((uint32_t)piece << log2f) * 128u, tmap, seg * 32, y, bar,
                    policy);
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
    constexpr int C = kF32Chunk;

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
    float *myw = sq + NH * D + ts * C * NH;                                 // [NH][C]
    int *slag = reinterpret_cast<int *>(sq + NH * D + SLOTS * C * NH);      // [NH]
    const int nchunks = (w.len + C - 1) / C;
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
    // QK: lane = (token tl of the chunk, half dh of the head dims); the two
    // halves' partial dots are summed with one shuffle, so both hold the
    // logits and the softmax below stays warp-uniform
    const int tl = lane & (C - 1), dh = lane >> 4;
    const int rsw = tl & 7;                          // swizzle phase of this lane's row
    for (int i = 0; i < my_n; ++i) {
        const int c = ts + SLOTS * i;
        const int t0 = c * C;
        if (!mbar_wait(kbar, i & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        ++k_done;
        // ---- logits
        const bool valid = t0 + tl < w.len;
        const int ahead = w.c - w.t_begin - t0 - tl;           // tokens from this one to the context end
        float dot[NH];
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) dot[hh] = 0.0f;
        const float *krow = sK + tl * 32;
#pragma unroll
        for (int sh = 0; sh < NSEG / 2; ++sh) {
            const int sg = dh * (NSEG / 2) + sh;
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4) {
                const float4 kv = *reinterpret_cast<const float4 *>(krow + sg * (C * 32) + ((q4 ^ rsw) << 2));
#pragma unroll
                for (int hh = 0; hh < NH; ++hh) {
                    const float4 qv = sq4[hh * WORDS + sg * 8 + q4];
                    dot[hh] = fmaf(qv.x, kv.x, fmaf(qv.y, kv.y, fmaf(qv.z, kv.z, fmaf(qv.w, kv.w, dot[hh]))));
                }
            }
        }
#pragma unroll
        for (int hh = 0; hh < NH; ++hh) dot[hh] += __shfl_xor_sync(0xFFFFFFFFu, dot[hh], 16);
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
            for (int o = C / 2; o > 0; o >>= 1) cm = fmaxf(cm, __shfl_xor_sync(0xFFFFFFFFu, cm, o));
            const float m_new = fmaxf(m[hh], cm);
            if (m_new != m[hh]) {        // warp-uniform: both halves hold the same logits
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
            lsum[hh] += p;                                    // each half counts its 16 tokens once
            if (dh == 0) myw[hh * C + tl] = p;
        }
        __syncwarp();
        if (!mbar_wait(vbar, i & 1)) {
            if (lane == 0) flag_error(P.status, kDevWaitTimeout);
            ok = false;
            break;
        }
        ++v_done;
        // ---- weighted sum, lane = 4 head dims; only tokens inside the context
        const int ntok = min(C, w.len - t0);
        const int tg = lane / LW, lw = lane % LW;
#pragma unroll 2
        for (int tt = tg; tt < ntok; tt += TG) {
            const float *vrow = sV + tt * 32;
            float4 v[NWL];
#pragma unroll
            for (int u = 0; u < NWL; ++u) {
                const int g4 = lw + 32 * u;                     // 16-byte group: column g4 / 8, chunk g4 % 8
                v[u] = *reinterpret_cast<const float4 *>(vrow + (g4 >> 3) * (C * 32) +
                                                         (((g4 & 7) ^ (tt & 7)) << 2));
            }
#pragma unroll
            for (int hh = 0; hh < NH; ++hh) {
                const float wt = myw[hh * C + tt];
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
        float l = lsum[hh];                 // each half holds the sums of all 16 token lanes
#pragma unroll
        for (int o = C / 2; o > 0; o >>= 1) l += __shfl_xor_sync(0xFFFFFFFFu, l, o);
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
// 32 floats x min(B, 16) rows and the 128-byte swizzle.
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
    const int ptok = 1 << (P.log2B < 4 ? P.log2B : 4);     // box rows: min(B, 16)
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

}  // namespace

cudaError_t launch_f32_family(const Params &P, int head_size, cudaStream_t st) {
    switch (head_size) {
        case 64: return launch_f32<64>(P, st);
        case 128: return launch_f32<128>(P, st);
        case 256: return launch_f32<256>(P, st);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa_q8
