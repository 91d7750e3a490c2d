// Quantise-and-scatter writer for the int8 paged KV cache.
//
// Computes what main() of "reshape_and_cache_q8.comp" (hanzo-ml 0.11.93)
// computes, per (token, kv_head) and separately for K and V: amax = max |x|;
// inv = 127/amax (0 for amax = 0); code = clamp(round(x * inv), -127, 127),
// halves away from zero; 4 codes per u32 (code l in byte l); then the f32
// bits of amax/127 (1.0 for amax = 0); slot 0xFFFFFFFF skips the row.
//
// GB300 mapping: one warp per (token, kv_head).  Each lane loads 16-byte
// vectors of K and of V (both in flight at once), the amax is a warp
// shuffle reduction, and lane j stores code word j (consecutive lanes,
// consecutive words).  Every f32 operation is an explicit round-to-nearest
// intrinsic, so nothing is contracted or approximated and the words match
// an IEEE reference bit for bit.
#include <cstdint>
#include <cuda_runtime.h>

#include "device_util.cuh"
#include "kernels.h"

namespace pa_q8 {
namespace {

constexpr int kWriterWarps = 8;

__device__ __forceinline__ uint32_t quantise_code(float x, float inv) {
    float t = __fmul_rn(x, inv);
    if (t != t) return 0u;                    // 0 * inf (127/amax overflowed): code 0
    t = fminf(fmaxf(roundf(t), -127.0f), 127.0f);
    return static_cast<uint32_t>(__float2int_rn(t)) & 0xFFu;
}

__device__ __forceinline__ uint32_t pack_word(float4 x, float inv) {
    return quantise_code(x.x, inv) | (quantise_code(x.y, inv) << 8) |
           (quantise_code(x.z, inv) << 16) | (quantise_code(x.w, inv) << 24);
}

template <int G>
__device__ __forceinline__ float group_max(float v) {
#pragma unroll
    for (int o = G / 2; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}

template <bool kVec>
__device__ __forceinline__ float4 load4(const float *p) {
    if constexpr (kVec) {
        return __ldcs(reinterpret_cast<const float4 *>(p));   // read once: streaming
    } else {
        return make_float4(__ldcs(p), __ldcs(p + 1), __ldcs(p + 2), __ldcs(p + 3));
    }
}

// D: head_size.  WORDS = D/4 code words per vector; G = lanes per vector
// (16 for D = 64, else 32); NW = words per lane.  For D = 64 lanes 0-15
// quantise K and lanes 16-31 quantise V; otherwise every lane does both.
template <int D, bool kVec>
__global__ void __launch_bounds__(kWriterWarps * 32)
quant_scatter_kernel(const float *__restrict__ key, const float *__restrict__ value,
                     uint32_t *__restrict__ key_cache, uint32_t *__restrict__ value_cache,
                     const uint32_t *__restrict__ slot_mapping, int64_t num_tokens,
                     int64_t key_stride, int64_t value_stride, int num_kv_heads,
                     int block_size, int64_t num_slots, uint32_t *status) {
    constexpr int WORDS = D / 4;
    constexpr int G = WORDS < 32 ? WORDS : 32;
    constexpr int NW = WORDS / G;
    constexpr bool kSplit = (G == 16);        // half-warp per vector
    const int lane = threadIdx.x & 31;
    const int64_t item = (int64_t)blockIdx.x * kWriterWarps + (threadIdx.x >> 5);
    if (item >= num_tokens * num_kv_heads) return;
    const int64_t tok = item / num_kv_heads;
    const int h = (int)(item - tok * num_kv_heads);

    const uint32_t slot = __ldg(slot_mapping + tok);
    if (slot == kPadSlot) return;
    if ((int64_t)slot >= num_slots) {
        if (lane == 0) flag_error(status, kDevBadSlot);
        return;
    }
    const int64_t blk = slot / (uint32_t)block_size;
    const int64_t off = slot - blk * block_size;
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * (WORDS + 1);

    if constexpr (kSplit) {
        const bool is_v = lane >= 16;
        const int j = lane & 15;
        const float *src = is_v ? value + tok * value_stride + (int64_t)h * D
                                : key + tok * key_stride + (int64_t)h * D;
        const float4 x = load4<kVec>(src + 4 * j);
        float m = fmaxf(fmaxf(fabsf(x.x), fabsf(x.y)), fmaxf(fabsf(x.z), fabsf(x.w)));
        m = group_max<16>(m);
        const float inv = m > 0.0f ? __fdiv_rn(127.0f, m) : 0.0f;
        uint32_t *cache = is_v ? value_cache : key_cache;
        cache[dst + j] = pack_word(x, inv);
        if (j == 0) cache[dst + WORDS] = __float_as_uint(m > 0.0f ? __fdiv_rn(m, 127.0f) : 1.0f);
    } else {
        const float *ksrc = key + tok * key_stride + (int64_t)h * D;
        const float *vsrc = value + tok * value_stride + (int64_t)h * D;
        float4 xk[NW], xv[NW];
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            xk[i] = load4<kVec>(ksrc + 4 * (lane + 32 * i));
            xv[i] = load4<kVec>(vsrc + 4 * (lane + 32 * i));
        }
        float mk = 0.0f, mv = 0.0f;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            mk = fmaxf(mk, fmaxf(fmaxf(fabsf(xk[i].x), fabsf(xk[i].y)),
                                 fmaxf(fabsf(xk[i].z), fabsf(xk[i].w))));
            mv = fmaxf(mv, fmaxf(fmaxf(fabsf(xv[i].x), fabsf(xv[i].y)),
                                 fmaxf(fabsf(xv[i].z), fabsf(xv[i].w))));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            mk = fmaxf(mk, __shfl_xor_sync(0xFFFFFFFFu, mk, o));
            mv = fmaxf(mv, __shfl_xor_sync(0xFFFFFFFFu, mv, o));
        }
        const float ik = mk > 0.0f ? __fdiv_rn(127.0f, mk) : 0.0f;
        const float iv = mv > 0.0f ? __fdiv_rn(127.0f, mv) : 0.0f;
#pragma unroll
        for (int i = 0; i < NW; ++i) {
            key_cache[dst + lane + 32 * i] = pack_word(xk[i], ik);
            value_cache[dst + lane + 32 * i] = pack_word(xv[i], iv);
        }
        if (lane == 0) {
            key_cache[dst + WORDS] = __float_as_uint(mk > 0.0f ? __fdiv_rn(mk, 127.0f) : 1.0f);
            value_cache[dst + WORDS] = __float_as_uint(mv > 0.0f ? __fdiv_rn(mv, 127.0f) : 1.0f);
        }
    }
}

template <int D>
cudaError_t launch_d(const WriterArgs &a, cudaStream_t stream) {
    const int64_t items = a.num_tokens * a.num_kv_heads;
    const int64_t grid = (items + kWriterWarps - 1) / kWriterWarps;
    if (grid > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const bool vec = ((reinterpret_cast<uintptr_t>(a.key) | reinterpret_cast<uintptr_t>(a.value)) & 15u) == 0 &&
                     (a.key_stride % 4) == 0 && (a.value_stride % 4) == 0;
    const int64_t num_slots = a.num_blocks * a.block_size;
    if (vec) {
        quant_scatter_kernel<D, true><<<(unsigned)grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, a.num_tokens,
            a.key_stride, a.value_stride, a.num_kv_heads, a.block_size, num_slots, a.status);
    } else {
        quant_scatter_kernel<D, false><<<(unsigned)grid, kWriterWarps * 32, 0, stream>>>(
            a.key, a.value, a.key_cache, a.value_cache, a.slot_mapping, a.num_tokens,
            a.key_stride, a.value_stride, a.num_kv_heads, a.block_size, num_slots, a.status);
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

}  // namespace pa_q8
