// Device helpers for the pa_q8 kernels (sm_103a): mbarriers, 1-D bulk
// copies global -> shared, bounded waits, warp reductions and the f16 tensor
// core tile.  Inline PTX only; no library code.
#pragma once

#include <cstdint>
#include <cuda_fp16.h>

namespace pa_q8 {

constexpr uint32_t kPadSlot = 0xFFFFFFFFu;
constexpr uint32_t kDevBadBlock = 0x1u;
constexpr uint32_t kDevBadSlot = 0x2u;
constexpr uint32_t kDevWaitTimeout = 0x4u;
constexpr uint64_t kWaitLimitNs = 1000000000ull;  // a stage wait normally takes microseconds

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void flag_error(uint32_t *status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}

// ---------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.release.cta.shared::cta.b64 st, [%0];\n\t}"
                 ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\t"
                 "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 st, [%0], %1;\n\t}"
                 ::"r"(bar), "r"(bytes) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase with the given parity to complete, for at most
// limit_ns of global time.  Returns false when it gave up.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint64_t limit_ns = kWaitLimitNs) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 31u) == 0 && global_timer_ns() - t0 > limit_ns) return false;
    }
}

// mbar_wait that also gives up once *abort is set (by any thread of the CTA);
// a thread whose own wait runs out of time sets it, so one stuck stage ends
// every waiter of the CTA within one time limit.
// Like mbar_try_wait, but the hardware may suspend the thread for up to
// hint_ns while the phase is incomplete (fewer issue slots spent waiting).
__device__ __forceinline__ bool mbar_try_wait_suspend(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_abortable(uint32_t bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait_suspend(bar, parity, 2000u)) return true;
        if ((i & 31u) == 0) {
            if (*abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                *abort = 1u;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------ bulk copies

// One contiguous run of `bytes` (multiple of 16; both addresses 16-byte
// aligned) from global memory into this CTA's shared memory; completion is
// counted on `bar` as transaction bytes.  Streaming data: evict-first in L2.
__device__ __forceinline__ void bulk_copy_g2s(uint32_t dst, const void *src, uint32_t bytes,
                                              uint32_t bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// Order this thread's earlier shared-memory accesses (made visible to it by
// a preceding __syncwarp / bar.sync) before its later async-proxy copies.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// 2-D tensor copy (TMA) of one box of the tensor map `tmap` (a
// __grid_constant__ kernel parameter) at element coordinates (x, y) into
// shared memory at `dst`, completing `bar`'s transaction count.  x times the
// element size must be a multiple of 16 bytes.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int x, int y, uint32_t bar,
                                            uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;"
        :: "r"(dst), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
        : "memory");
}

// Order this thread's generic stores to global memory before bulk copies
// (async proxy) that a CTA barrier later lets another thread issue.
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// ----------------------------------------------- 5th-generation tensor cores
//
// tcgen05 with one CTA (cta_group::1): f16 operands in shared memory, f32
// accumulators in tensor memory (TMEM: 128 lanes x 512 32-bit columns per
// SM).  Operand tiles use the canonical layouts without swizzle: 8 x 16-byte
// core matrices, LBO bytes apart along K and SBO bytes apart along M/N.  In
// the K-major layout a core matrix holds 8 M/N rows of 8 K elements; an
// MN-major B operand (instruction-descriptor bit 16) holds 8 K rows of 8 N
// elements.

__device__ __forceinline__ uint64_t umma_smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46);
}

// kind::f16 instruction descriptor: f16 A and B (K-major), f32 accumulator, M x N.
__host__ __device__ constexpr uint32_t umma_idesc_f16(int m, int n) {
    return (1u << 4) | ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

// One warp allocates `ncols` TMEM columns (a power of two >= 32); the base
// address lands in shared memory at `dst`.
__device__ __forceinline__ void tmem_alloc(uint32_t dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" :: "r"(dst), "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// D (TMEM) = A . B^T (+ D when accumulate), issued by one thread.
__device__ __forceinline__ void umma_f16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                         bool accumulate) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}"
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
                 : "memory");
}

// D (TMEM) = A . B^T (+ D when accumulate) with A in tensor memory: lane m
// holds row m of A, two consecutive f16 K elements per 32-bit column (16 K
// elements = 8 columns per instruction); B in shared memory as above.
__device__ __forceinline__ void umma_f16_ta(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                            bool accumulate) {
    asm volatile("{\n.reg .pred p;\nsetp.ne.b32 p, %4, 0;\n"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"((uint32_t)accumulate)
                 : "memory");
}

// Arrive once on `bar` when every tcgen05.mma this thread issued so far is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" :: "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane (warp w owns lanes
// 32(w%4)..); the address must be the same in every thread of the warp.
__device__ __forceinline__ void tmem_ld32(uint32_t addr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
}

__device__ __forceinline__ void tmem_st32(uint32_t addr, const float (&v)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(addr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                    "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                    "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                    "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                    "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
                    "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
                    "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
                    "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
                    "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
                    "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// 16 consecutive 32-bit columns of 16 TMEM lanes, split across the warp
// (shape 16x32bx2, half-split offset 16): threads t < 16 read lane
// base + t at columns addr .. addr + 15, threads t >= 16 read lane
// base + t - 16 at columns addr + 16 .. addr + 31.  An M = 64 accumulator
// keeps its rows in lanes 0-15 of each warp's 32, so this gives the two
// halves of a row's 32 columns to threads t and t + 16.
__device__ __forceinline__ void tmem_ld16x2(uint32_t addr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile("tcgen05.ld.sync.aligned.16x32bx2.x16.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16], 16;"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15])
                 : "r"(addr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] = __uint_as_float(r[j]);
}

// The store of the same shape, without waiting (tcgen05.wait::st before the
// columns are used).
__device__ __forceinline__ void tmem_st16x2_nowait(uint32_t addr, const uint32_t (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], 16, "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(addr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
                    "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
                 : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// The store of the same shape; waits until the columns are written.
__device__ __forceinline__ void tmem_st16x2(uint32_t addr, const float (&v)[16]) {
    asm volatile("tcgen05.st.sync.aligned.16x32bx2.x16.b32 [%0], 16, "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(addr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
                    "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
                    "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
                    "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
                    "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
                    "r"(__float_as_uint(v[15]))
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// ------------------------------------------------- paired f32 arithmetic
// One instruction for two f32 lanes (round to nearest even, no flush), the
// same results as two scalar operations.

__device__ __forceinline__ unsigned long long f2_bits(float2 a) {
    return (unsigned long long)__float_as_uint(a.x) | ((unsigned long long)__float_as_uint(a.y) << 32);
}
__device__ __forceinline__ float2 bits_f2(unsigned long long b) {
    return make_float2(__uint_as_float((uint32_t)b), __uint_as_float((uint32_t)(b >> 32)));
}
__device__ __forceinline__ float2 mul_f2(float2 a, float2 b) {
    unsigned long long d;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 fma_f2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)), "l"(f2_bits(c)));
    return bits_f2(d);
}
__device__ __forceinline__ float2 add_f2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(f2_bits(a)), "l"(f2_bits(b)));
    return bits_f2(d);
}

// max(a, b, c) in one instruction
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float d;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
    return d;
}

// (a, b) as f16x2 hi = rn(a, b) and lo = rn(a - hi.x, b - hi.y): the
// residual of each lane is one f32 fma with an f16 operand (hi * -1 + x,
// exact: hi is x rounded to f16), so the pair costs four instructions.
__device__ __forceinline__ void split_f16x2_fma(float a, float b, uint32_t &hi, uint32_t &lo) {
    asm("{\n\t.reg .b16 h0, h1, m1;\n\t.reg .f32 r0, r1;\n\t"
        "cvt.rn.f16x2.f32 %0, %3, %2;\n\t"
        "mov.b32 {h0, h1}, %0;\n\t"
        "mov.b16 m1, 0xBC00;\n\t"
        "fma.rn.f32.f16 r0, h0, m1, %2;\n\t"
        "fma.rn.f32.f16 r1, h1, m1, %3;\n\t"
        "cvt.rn.f16x2.f32 %1, r1, r0;\n\t}"
        : "=r"(hi), "=r"(lo)
        : "f"(a), "f"(b));
}

// ----------------------------------------------- programmatic dependent launch

// Block until the grid this one depends on (launched before it on the
// stream) has finished and its memory is visible.  No-op without a
// programmatic dependency.
__device__ __forceinline__ void grid_dependency_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// Allow the dependent grid to be launched before this one finishes.
__device__ __forceinline__ void grid_dependents_launch() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------------- misc

__device__ __forceinline__ void named_barrier(uint32_t id, uint32_t threads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// bar.sync over `threads` threads that also ORs a predicate across them.
__device__ __forceinline__ bool named_barrier_or(uint32_t id, uint32_t threads, bool pred) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 p, %1, 0;\n\t"
        "barrier.cta.red.or.pred q, %2, %3, p;\n\t"
        "selp.u32 %0, 1, 0, q;\n\t}"
        : "=r"(r)
        : "r"((uint32_t)pred), "r"(id), "r"(threads)
        : "memory");
    return r != 0;
}

__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(sel));
    return d;
}

// prmt with a compile-time selector (an immediate operand)
template <uint32_t SEL>
__device__ __forceinline__ uint32_t prmt_i(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "n"(SEL));
    return d;
}

// ----------------------------------------------- int8 token-vector encoding

// Code of x: round(x * inv) with halves away from zero, clamped to
// [-127, 127].  For |t| < 2^23, adding 0.5 to |t| rounded toward zero and
// truncating gives floor(|t| + 0.5) exactly (every integer below 2^24 is an
// f32, so rounding down never skips one).  The f32 -> s32 conversion
// saturates: NaN (0 * inf, when 127/amax overflowed) becomes 0 and +inf
// becomes INT_MAX, clamped to 127 next.
__device__ __forceinline__ int quantise_code(float x, float inv) {
    const float t = __fmul_rn(x, inv);
    const int a = min(__float2int_rz(__fadd_rz(fabsf(t), 0.5f)), 127);
    return t < 0.0f ? -a : a;
}

// Four codes into one word, code l in byte l.
__device__ __forceinline__ uint32_t pack_word(float4 x, float inv) {
    const uint32_t c0 = (uint32_t)quantise_code(x.x, inv), c1 = (uint32_t)quantise_code(x.y, inv);
    const uint32_t c2 = (uint32_t)quantise_code(x.z, inv), c3 = (uint32_t)quantise_code(x.w, inv);
    return prmt_i<0x5410u>(prmt_i<0x0040u>(c0, c1), prmt_i<0x0040u>(c2, c3));
}


// (a & MASK) ^ c in one LOP3, MASK an immediate
template <uint32_t MASK>
__device__ __forceinline__ uint32_t and_xor_i(uint32_t a, uint32_t c) {
    uint32_t d;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;" : "=r"(d) : "r"(a), "n"(MASK), "r"(c));
    return d;
}

// Two f16 lanes 0x64XX (= 1024 + XX) minus 1152 -> the signed codes XX - 128.
__device__ __forceinline__ uint32_t sub_1152_x2(uint32_t v, uint32_t bias) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(v), "r"(bias));
    return d;
}

// Constants of the int8 -> f16 conversions, kept in registers by the caller.
struct F16Consts {
    uint32_t exp64 = 0x64646464u;     // 0x64 in every byte: f16 exponent of 1024
    uint32_t bias = 0x64806480u;      // f16x2 (1152, 1152); also 0x64 | 0x80 per half
};

// Codes in byte lanes 0,1 (lo) and 2,3 (hi) of a word -> two f16x2 values.
// Exact: every int8 is an f16.
__device__ __forceinline__ void codes4_to_f16x2(uint32_t w, uint32_t &lo, uint32_t &hi,
                                                const F16Consts &k) {
    const uint32_t u = w ^ 0x80808080u;         // two's complement -> offset binary
    lo = sub_1152_x2(prmt_i<0x4140u>(u, k.exp64), k.bias);
    hi = sub_1152_x2(prmt_i<0x4342u>(u, k.exp64), k.bias);
}

// Byte lane e of a and of b -> f16x2 (code_a[e], code_b[e]).
template <int E>
__device__ __forceinline__ uint32_t codes_pair_to_f16x2(uint32_t a, uint32_t b, const F16Consts &k) {
    // d = [a.e, a.e, b.e, b.e]; bytes 1 and 3 then become 0x64, bytes 0 and 2 flip sign
    constexpr uint32_t sel = (uint32_t)E | ((uint32_t)E << 4) | ((uint32_t)(E + 4) << 8) |
                             ((uint32_t)(E + 4) << 12);
    return sub_1152_x2(and_xor_i<0x00FF00FFu>(prmt_i<sel>(a, b), k.bias), k.bias);
}

// D = A(16x16, f16, row) * B(16x8, f16, col) + D, f32 accumulate.
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                          uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t pack_half2(__half lo, __half hi) {
    return (uint32_t)__half_as_ushort(lo) | ((uint32_t)__half_as_ushort(hi) << 16);
}

// x = hi + lo with hi = f16(x), lo = f16(x - hi): 22 significant bits.
__device__ __forceinline__ void split_f16(float x, __half &hi, __half &lo) {
    hi = __float2half_rn(x);
    lo = __float2half_rn(x - __half2float(hi));
}

// The same split for a pair (a, b) -> packed f16x2 hi = (hi(a), hi(b)) and
// lo = (lo(a), lo(b)); a sits in the low half.
__device__ __forceinline__ void split_f16x2(float a, float b, uint32_t &hi, uint32_t &lo) {
    const __half2 h = __floats2half2_rn(a, b);
    const __half2 l = __floats2half2_rn(a - __low2float(h), b - __high2float(h));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

}  // namespace pa_q8
