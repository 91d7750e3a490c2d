// Quantise-and-scatter writer for the int8 paged KV cache.
//
// Computes what main() of "reshape_and_cache_q8.comp" (hanzo-ml 0.11.93)
// computes, per (token, kv_head) and separately for K and V: amax = max |x|;
// inv = 127/amax (0 for amax = 0); code = clamp(round(x * inv), -127, 127),
// halves away from zero; 4 codes per u32 (code l in byte l); then the f32
// bits of amax/127 (1.0 for amax = 0); slot 0xFFFFFFFF skips the row.
//
// GB300 mapping: a warp per (token, pair of kv heads), eight lanes per K or
// V vector, so the per-vector reductions and divisions of four vectors share
// instructions.  Large appends of 16-byte aligned rows run as one wave of
// CTAs whose warps walk a series of tokens, reading each token's slot ahead of
// its rows (PAD rows are never read); other appends take one token per warp,
// its 16-byte row loads issued before the slot read.
// Every f32 operation is an explicit round-to-nearest intrinsic, so nothing
// is contracted or approximated and the words match an IEEE reference bit
// for bit.
#include <cstdint>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"

namespace pa_q8 {
namespace {

constexpr int kWriterWarps = 8;
// The walking writer (one wave of CTAs, each warp a series of tokens) takes
// appends of at least kWalkTokensPerWarp tokens per warp of that wave
#ifndef PA_Q8_WRITER_WALK
#define PA_Q8_WRITER_WALK 1
#endif
constexpr int kWalkTokensPerWarp = 2;
// tokens whose rows a walking warp has in flight
#ifndef PA_Q8_WRITER_WALK_DEPTH
#define PA_Q8_WRITER_WALK_DEPTH 1
#endif
constexpr int kWalkDepth = PA_Q8_WRITER_WALK_DEPTH;

template <bool kVec>
__device__ __forceinline__ float4 load4(const float *p) {
    if constexpr (kVec) {
        return __ldcs(reinterpret_cast<const float4 *>(p));   // read once: streaming
    } else {
        return make_float4(__ldcs(p), __ldcs(p + 1), __ldcs(p + 2), __ldcs(p + 3));
    }
}

// D: head_size.  A warp owns one token and two kv heads (h0, h0 + 1): four
// vectors K(h0), V(h0), K(h0+1), V(h0+1), eight lanes each (lane group
// v = lane / 8).  Lane j of a group holds words j, j + 8, ... (NW = D/32 of
// them), so every load and store instruction covers contiguous 128-byte /
// 32-byte runs per vector.  Because the four groups run side by side, one
// instruction sequence computes all four amax reductions (3 shuffle levels)
// and all four divisions.  The K/V loads are issued before the slot is looked
// at, so the memory round trips overlap (a PAD row's data is read and
// dropped).  log2_block < 0 means block_size is not a power of two.
constexpr int kLanesPerVector = 8;

template <int D, bool kVec>
__global__ void __launch_bounds__(kWriterWarps * 32)
quant_scatter_kernel(const float *__restrict__ key, const float *__restrict__ value,
                     uint32_t *__restrict__ key_cache, uint32_t *__restrict__ value_cache,
                     const uint32_t *__restrict__ slot_mapping, int num_tokens,
                     int64_t key_stride, int64_t value_stride, int num_kv_heads,
                     int block_size, int log2_block, int64_t num_slots, uint32_t *status) {
    // a decode launched next may start its prep (which reads only the
    // context lengths until this grid has finished)
    grid_dependents_launch();
    constexpr int WORDS = D / 4;
    constexpr int G = kLanesPerVector;
    constexpr int NW = WORDS / G;
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * kWriterWarps + (threadIdx.x >> 5);
    if (tok >= num_tokens) return;
    const int v = lane / G, j = lane % G;
    const bool is_v = v & 1;
    const int h = 2 * blockIdx.y + (v >> 1);
    const bool live = h < num_kv_heads;                 // an odd head count leaves a pair half empty
    const float *src = is_v ? value + (int64_t)tok * value_stride + (int64_t)h * D
                            : key + (int64_t)tok * key_stride + (int64_t)h * D;
    float4 x[NW];
#pragma unroll
    for (int i = 0; i < NW; ++i)
        x[i] = live ? load4<kVec>(src + 4 * (j + G * i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t slot = __ldg(slot_mapping + tok);

    float m = 0.0f;
#pragma unroll
    for (int i = 0; i < NW; ++i)
        m = fmaxf(m, fmaxf(fmaxf(fabsf(x[i].x), fabsf(x[i].y)), fmaxf(fabsf(x[i].z), fabsf(x[i].w))));
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float inv = m > 0.0f ? __fdiv_rn(127.0f, m) : 0.0f;
    const float scale = m > 0.0f ? __fdiv_rn(m, 127.0f) : 1.0f;
    if (slot == kPadSlot || !live) return;
    if ((int64_t)slot >= num_slots) {
        if (lane == 0) flag_error(status, kDevBadSlot);
        return;
    }
    uint32_t blk, off;
    if (log2_block >= 0) {
        blk = slot >> log2_block;
        off = slot & ((1u << log2_block) - 1u);
    } else {
        blk = slot / (uint32_t)block_size;
        off = slot - blk * (uint32_t)block_size;
    }
    const int64_t dst = (((int64_t)blk * num_kv_heads + h) * block_size + off) * (WORDS + 1);
    uint32_t *cache = is_v ? value_cache : key_cache;
#pragma unroll
    for (int i = 0; i < NW; ++i) cache[dst + j + G * i] = pack_word(x[i], inv);
    if (j == 0) cache[dst + WORDS] = __float_as_uint(scale);
}

// The same arithmetic with every warp walking a strided series of tokens for
// one pair of kv heads (16-byte aligned rows only), as one wave of CTAs.  A
// token's slot is read DEPTH + 1 tokens ahead and its rows DEPTH tokens
// ahead, so a PAD row is never read and no slot round trip sits in front of
// the row loads: while a warp quantises token i, the rows of the next DEPTH
// tokens and the slot of the one after are in flight.  One token ahead
// measured as fast as the one-token warps (30.6 against 30.7 us for the
// 16384-row append) with 5% fewer bytes read; two and three ahead were slower
// (31.6, 31.0 us: more registers, fewer CTAs per SM).
template <int D, int DEPTH>
__global__ void __launch_bounds__(kWriterWarps * 32)
quant_scatter_walk_kernel(const float *__restrict__ key, const float *__restrict__ value,
                          uint32_t *__restrict__ key_cache, uint32_t *__restrict__ value_cache,
                          const uint32_t *__restrict__ slot_mapping, int num_tokens,
                          int64_t key_stride, int64_t value_stride, int num_kv_heads,
                          int block_size, int log2_block, int64_t num_slots, uint32_t *status) {
    grid_dependents_launch();
    constexpr int WORDS = D / 4;
    constexpr int G = kLanesPerVector;
    constexpr int NW = WORDS / G;
    const int lane = threadIdx.x & 31;
    const int stride = (int)gridDim.x * kWriterWarps;
    int tok = blockIdx.x * kWriterWarps + (threadIdx.x >> 5);
    const int v = lane / G, j = lane % G;
    const bool is_v = v & 1;
    const int h = 2 * blockIdx.y + (v >> 1);
    const bool live = h < num_kv_heads;
    const float *base = is_v ? value + (int64_t)h * D : key + (int64_t)h * D;
    const int64_t row_stride = is_v ? value_stride : key_stride;
    uint32_t *cache = is_v ? value_cache : key_cache;
    auto slot_at = [&](int t) { return t < num_tokens ? __ldg(slot_mapping + t) : kPadSlot; };
    auto load_rows = [&](int t, uint32_t slot, float4 (&x)[NW]) {
        const bool want = live && t < num_tokens && slot != kPadSlot;
        const float *src = base + (int64_t)t * row_stride;
#pragma unroll
        for (int i = 0; i < NW; ++i)
            x[i] = want ? load4<true>(src + 4 * (j + G * i)) : make_float4(0.f, 0.f, 0.f, 0.f);
    };
    // rows of the next DEPTH tokens in flight (x[0] the current one), slots of
    // one more token ahead
    uint32_t sl[DEPTH + 1];
    float4 x[DEPTH][NW];
#pragma unroll
    for (int d = 0; d <= DEPTH; ++d) sl[d] = slot_at(tok + d * stride);
#pragma unroll
    for (int d = 0; d < DEPTH; ++d) load_rows(tok + d * stride, sl[d], x[d]);
    for (; tok < num_tokens; tok += stride) {
        const uint32_t slot = sl[0];
        float4 cur[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) cur[i] = x[0][i];
        // shift the window: rows of token tok + DEPTH * stride, slot one further
#pragma unroll
        for (int d = 0; d + 1 < DEPTH; ++d) {
#pragma unroll
            for (int i = 0; i < NW; ++i) x[d][i] = x[d + 1][i];
        }
#pragma unroll
        for (int d = 0; d < DEPTH; ++d) sl[d] = sl[d + 1];
        load_rows(tok + DEPTH * stride, sl[DEPTH - 1], x[DEPTH - 1]);
        sl[DEPTH] = slot_at(tok + (DEPTH + 1) * stride);
        float m = 0.0f;
#pragma unroll
        for (int i = 0; i < NW; ++i)
            m = fmaxf(m, fmaxf(fmaxf(fabsf(cur[i].x), fabsf(cur[i].y)), fmaxf(fabsf(cur[i].z), fabsf(cur[i].w))));
#pragma unroll
        for (int o = G / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
        const float inv = m > 0.0f ? __fdiv_rn(127.0f, m) : 0.0f;
        const float scale = m > 0.0f ? __fdiv_rn(m, 127.0f) : 1.0f;
        if (slot != kPadSlot && live) {
            if ((int64_t)slot >= num_slots) {
                if (j == 0) flag_error(status, kDevBadSlot);
            } else {
                uint32_t blk, off;
                if (log2_block >= 0) {
                    blk = slot >> log2_block;
                    off = slot & ((1u << log2_block) - 1u);
                } else {
                    blk = slot / (uint32_t)block_size;
                    off = slot - blk * (uint32_t)block_size;
                }
                const int64_t dst = (((int64_t)blk * num_kv_heads + h) * block_size + off) * (WORDS + 1);
#pragma unroll
                for (int i = 0; i < NW; ++i) cache[dst + j + G * i] = pack_word(cur[i], inv);
                if (j == 0) cache[dst + WORDS] = __float_as_uint(scale);
            }
        }
    }
}

template <int D>
cudaError_t launch_d(const WriterArgs &a, cudaStream_t stream) {
    const int64_t head_pairs = (a.num_kv_heads + 1) / 2;
    if (a.num_tokens > 0x7FFFFFFF - kWriterWarps || head_pairs > 65535) return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((a.num_tokens + kWriterWarps - 1) / kWriterWarps), (unsigned)head_pairs);
    const bool vec = ((reinterpret_cast<uintptr_t>(a.key) | reinterpret_cast<uintptr_t>(a.value)) & 15u) == 0 &&
                     (a.key_stride % 4) == 0 && (a.value_stride % 4) == 0;
    const int64_t num_slots = a.num_blocks * a.block_size;
    int log2_block = -1;
    if ((a.block_size & (a.block_size - 1)) == 0) {
        log2_block = 0;
        while ((1 << log2_block) < a.block_size) ++log2_block;
    }
    int sms = 0, dev = 0, per_sm = 0;
    if (PA_Q8_WRITER_WALK && vec && cudaGetDevice(&dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_scatter_walk_kernel<D, kWalkDepth>,
                                                      kWriterWarps * 32, 0) ==
            cudaSuccess &&
        per_sm > 0 && grid.x > (unsigned)(kWalkTokensPerWarp * per_sm * sms / head_pairs)) {
        // enough tokens for every warp to walk several: one wave of CTAs
        const dim3 wgrid((unsigned)((per_sm * sms + head_pairs - 1) / head_pairs), (unsigned)head_pairs);
        quant_scatter_walk_kernel<D, kWalkDepth><<<wgrid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, (int)a.num_tokens,
            a.key_stride, a.value_stride, a.num_kv_heads, a.block_size, log2_block, num_slots, a.status);
    } else if (vec) {
        cudaGetLastError();
        quant_scatter_kernel<D, true><<<grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, (int)a.num_tokens,
            a.key_stride, a.value_stride, a.num_kv_heads, a.block_size, log2_block, num_slots, a.status);
    } else {
        quant_scatter_kernel<D, false><<<grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, (int)a.num_tokens,
            a.key_stride, a.value_stride, a.num_kv_heads, a.block_size, log2_block, num_slots, a.status);
    }
    return cudaGetLastError();
}

// ----------------------------------------------------- contiguous q8 cache
//
// The contiguous cache with a side scale region ("attention.rs", the
// kv_append_q8 dispatch): per sequence, [max_t][kv_row] int8 codes (4 per
// u32 word, kv_row = num_kv_heads * head_size) then [max_t][kv_row / 32] f32
// scales, one per 32-element group; sequences back to back.  A row's slot is
// sequence * max_t + position (0xFFFFFFFF skips it).  One warp per (token,
// pair of groups): vectors K(g0), V(g0), K(g1), V(g1), eight lanes each, one
// word per lane -- the paged writer's arithmetic on 32-value groups.
template <bool kVec>
__global__ void __launch_bounds__(kWriterWarps * 32)
cq_append_kernel(const float *__restrict__ key, const float *__restrict__ value,
                 uint32_t *__restrict__ key_cache, uint32_t *__restrict__ value_cache,
                 const uint32_t *__restrict__ slot_mapping, int num_tokens, int64_t key_stride,
                 int64_t value_stride, int kv_row, int64_t max_t, int64_t num_slots, uint32_t *status) {
    grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * kWriterWarps + (threadIdx.x >> 5);
    if (tok >= num_tokens) return;
    const int v = lane / kLanesPerVector, j = lane % kLanesPerVector;
    const bool is_v = v & 1;
    const int groups = kv_row / 32;
    const int grp = 2 * blockIdx.y + (v >> 1);
    const bool live = grp < groups;
    const float *src = (is_v ? value + (int64_t)tok * value_stride : key + (int64_t)tok * key_stride) + 32 * grp + 4 * j;
    const float4 x = live ? load4<kVec>(src) : make_float4(0.f, 0.f, 0.f, 0.f);
    const uint32_t slot = __ldg(slot_mapping + tok);
    float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
#pragma unroll
    for (int o = kLanesPerVector / 2; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, o));
    const float inv = m > 0.0f ? __fdiv_rn(127.0f, m) : 0.0f;
    const float scale = m > 0.0f ? __fdiv_rn(m, 127.0f) : 1.0f;
    if (slot == kPadSlot || !live) return;
    if ((int64_t)slot >= num_slots) {
        if (lane == 0) flag_error(status, kDevBadSlot);
        return;
    }
    const int64_t s = slot / max_t, t = slot - s * max_t;
    const int64_t base = s * (max_t * (kv_row / 4) + max_t * groups);
    uint32_t *cache = is_v ? value_cache : key_cache;
    cache[base + t * (kv_row / 4) + 8 * grp + j] = pack_word(x, inv);
    if (j == 0) cache[base + max_t * (kv_row / 4) + t * groups + grp] = __float_as_uint(scale);
}

// ------------------------------------------------------------ f32 cache
//
// The f32 cache's writer: each (token, kv head) K and V vector is copied to
// its slot of the f32 cache [num_blocks][Hk][B][D] (slot 0xFFFFFFFF skips the
// row, as in the q8 writer).  One warp per (token, kv head); lanes move 16-byte
// groups when the rows allow it, single floats otherwise.
template <int D, bool kVec>
__global__ void __launch_bounds__(kWriterWarps * 32)
f32_scatter_kernel(const float *__restrict__ key, const float *__restrict__ value,
                   float *__restrict__ key_cache, float *__restrict__ value_cache,
                   const uint32_t *__restrict__ slot_mapping, int num_tokens, int64_t key_stride,
                   int64_t value_stride, int num_kv_heads, int log2_block, int64_t num_slots,
                   uint32_t *status) {
    grid_dependents_launch();
    const int lane = threadIdx.x & 31;
    const int tok = blockIdx.x * kWriterWarps + (threadIdx.x >> 5);
    const int h = blockIdx.y;
    if (tok >= num_tokens) return;
    const uint32_t slot = __ldg(slot_mapping + tok);
    if (slot == kPadSlot) return;
    if ((int64_t)slot >= num_slots) {
        if (lane == 0) flag_error(status, kDevBadSlot);
        return;
    }
    const uint32_t blk = slot >> log2_block, off = slot & ((1u << log2_block) - 1u);
    const int64_t dst = (((int64_t)blk * num_kv_heads + h) << log2_block | off) * D;
    const float *ks = key + (int64_t)tok * key_stride + (int64_t)h * D;
    const float *vs = value + (int64_t)tok * value_stride + (int64_t)h * D;
    if constexpr (kVec) {
#pragma unroll
        for (int i = lane; i < D / 4; i += 32) {
            const float4 a = __ldcs(reinterpret_cast<const float4 *>(ks) + i);
            const float4 b = __ldcs(reinterpret_cast<const float4 *>(vs) + i);
            reinterpret_cast<float4 *>(key_cache + dst)[i] = a;
            reinterpret_cast<float4 *>(value_cache + dst)[i] = b;
        }
    } else {
#pragma unroll 4
        for (int i = lane; i < D; i += 32) {
            key_cache[dst + i] = __ldcs(ks + i);
            value_cache[dst + i] = __ldcs(vs + i);
        }
    }
}

template <int D>
cudaError_t launch_f32_d(const WriterArgs &a, cudaStream_t stream) {
    if (a.num_tokens > 0x7FFFFFFF - kWriterWarps || a.num_kv_heads > 65535) return cudaErrorInvalidValue;
    if ((a.block_size & (a.block_size - 1)) != 0) return cudaErrorInvalidValue;
    int log2_block = 0;
    while ((1 << log2_block) < a.block_size) ++log2_block;
    const dim3 grid((unsigned)((a.num_tokens + kWriterWarps - 1) / kWriterWarps), (unsigned)a.num_kv_heads);
    const bool vec = ((reinterpret_cast<uintptr_t>(a.key) | reinterpret_cast<uintptr_t>(a.value) |
                       reinterpret_cast<uintptr_t>(a.key_cache) | reinterpret_cast<uintptr_t>(a.value_cache)) &
                      15u) == 0 &&
                     (a.key_stride % 4) == 0 && (a.value_stride % 4) == 0;
    float *kc = reinterpret_cast<float *>(a.key_cache);
    float *vc = reinterpret_cast<float *>(a.value_cache);
    const int64_t num_slots = a.num_blocks * a.block_size;
    if (vec) {
        f32_scatter_kernel<D, true><<<grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, kc, vc, a.slot_mapping, (int)a.num_tokens, a.key_stride, a.value_stride,
            a.num_kv_heads, log2_block, num_slots, a.status);
    } else {
        f32_scatter_kernel<D, false><<<grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, kc, vc, a.slot_mapping, (int)a.num_tokens, a.key_stride, a.value_stride,
            a.num_kv_heads, log2_block, num_slots, a.status);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_writer(const WriterArgs &a, cudaStream_t stream) {
    switch (a.head_size) {
        case 64: return launch_d<64>(a, stream);
        case 128: return launch_d<128>(a, stream);
        case 256: return launch_d<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_cq_append(const WriterArgs &a, int64_t max_t, cudaStream_t stream) {
    const int kv_row = a.num_kv_heads * a.head_size;
    const int64_t group_pairs = (kv_row / 32 + 1) / 2;
    if (a.num_tokens > 0x7FFFFFFF - kWriterWarps || group_pairs > 65535 || kv_row % 32 != 0)
        return cudaErrorInvalidValue;
    const dim3 grid((unsigned)((a.num_tokens + kWriterWarps - 1) / kWriterWarps), (unsigned)group_pairs);
    const bool vec = ((reinterpret_cast<uintptr_t>(a.key) | reinterpret_cast<uintptr_t>(a.value)) & 15u) == 0 &&
                     (a.key_stride % 4) == 0 && (a.value_stride % 4) == 0;
    const int64_t num_slots = a.num_blocks * max_t;        // num_blocks carries the sequence count
    if (vec) {
        cq_append_kernel<true><<<grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, (int)a.num_tokens, a.key_stride,
            a.value_stride, kv_row, max_t, num_slots, a.status);
    } else {
        cq_append_kernel<false><<<grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, (int)a.num_tokens, a.key_stride,
            a.value_stride, kv_row, max_t, num_slots, a.status);
    }
    return cudaGetLastError();
}

cudaError_t launch_writer_f32(const WriterArgs &a, cudaStream_t stream) {
    switch (a.head_size) {
        case 64: return launch_f32_d<64>(a, stream);
        case 128: return launch_f32_d<128>(a, stream);
        case 256: return launch_f32_d<256>(a, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace pa_q8
