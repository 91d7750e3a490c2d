/*
 * pa_q8 -- int8 paged-KV attention decode for NVIDIA GB300 (sm_103a).
 *
 * C ABI of libpa_q8.so.  Plain pointers and sizes only; every pointer named
 * "device" is a CUDA device address the caller allocated and owns.  The
 * library keeps no per-call state and makes no allocation call: scratch (the
 * split-context partials) lives in a workspace the caller passes in, or, for
 * pa_q8_decode_noalloc, in a fixed buffer compiled into the library.  That
 * buffer (PA_Q8_NOALLOC_SCRATCH_BYTES, 64 MiB) sits in the same device module
 * as the library's status word, so every device on which any entry point has
 * run holds it until the process exits, whether or not pa_q8_decode_noalloc
 * is called there.  The library looks up the device addresses of those two
 * symbols once per device and caches them: after cudaDeviceReset (or any
 * other teardown of a device's primary context) the cached addresses are
 * stale, so the library must not be called again on that device in the same
 * process.
 * All work is queued on the caller's CUDA stream (a cudaStream_t passed as
 * void*; NULL = the legacy default stream) and no function synchronises,
 * except pa_q8_device_status which reads a flag back.
 *
 * Programmatic dependent launch: the writers let the next kernel on the
 * stream start once all their CTAs run, and a decode's first kernel (its
 * ordering pass) is launched to take that chance.  That kernel reads only
 * context_lens before the previous kernel has finished, and waits for it
 * before anything else; every later step of the decode waits for it in turn.
 * A decode whose split-context grid fits in one wave has no ordering pass;
 * its partials are merged by a second kernel, launched as a programmatic
 * dependent of the attention kernel, which waits for that kernel to finish
 * before it reads anything.
 * So context_lens must be final when the kernel before the decode starts,
 * which stream order gives unless that kernel is itself one (of the caller's)
 * that writes context_lens and allows early dependents.
 *
 * Data layout (header comments of the "paged_attn_q8.comp" and
 * "reshape_and_cache_q8.comp" pages, hanzo-ml 0.11.92 / 0.11.93):
 *
 *   key_cache, value_cache : u32 [num_blocks][num_kv_heads][block_size][W],
 *                            W = head_size/4 + 1.  A token vector holds
 *                            head_size/4 code words (4 int8 codes per word,
 *                            code l in bits 8l..8l+7, two's complement)
 *                            followed by one word with the f32 bit pattern of
 *                            the token's scale.  value = code * scale.
 *   block_tables           : u32 [num_seqs][max_blocks_per_seq]; logical
 *                            token t of a sequence is in physical block
 *                            block_tables[s][t / block_size], offset
 *                            t % block_size.  Entries past a sequence's last
 *                            block are never read.
 *   context_lens           : u32 [num_seqs]; clamped to
 *                            max_blocks_per_seq * block_size.
 *   q, out                 : f32 [num_seqs][num_heads][head_size], contiguous.
 *   query head h reads kv head h / (num_heads / num_kv_heads).
 *
 * Return values: PA_Q8_OK or a negative pa_q8_status; nothing throws.
 * Argument errors are found on the host before anything is queued.  Errors
 * a kernel finds while running (a block id or slot out of range, a wait
 * that gave up) set sticky bits in a per-device status word that
 * pa_q8_device_status reads; the offending access is skipped, never made.
 */
#ifndef PA_Q8_H
#define PA_Q8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_q8_status {
    PA_Q8_OK = 0,
    PA_Q8_EINVAL = -1,        /* a size <= 0, a NULL pointer, H % Hk != 0, D or B not a multiple of 4 */
    PA_Q8_EUNSUPPORTED = -2,  /* valid but without a kernel: head_size not in {64,128,256},
                                 block_size not a power of two in [4,1024], ... */
    PA_Q8_EALIGN = -3,        /* a pointer or stride without the alignment stated below */
    PA_Q8_ECUDA = -4,         /* the CUDA runtime refused a launch or query */
    PA_Q8_EWORKSPACE = -5     /* workspace_bytes below pa_q8_decode_workspace_size() */
} pa_q8_status;

/* Sticky device-side error bits (pa_q8_device_status). */
#define PA_Q8_DEV_BAD_BLOCK    0x1u  /* a block_tables entry >= num_blocks was skipped      */
#define PA_Q8_DEV_BAD_SLOT     0x2u  /* a slot_mapping entry >= num_blocks*block_size (not PAD) */
#define PA_Q8_DEV_WAIT_TIMEOUT 0x4u  /* a bounded in-kernel wait gave up; the output is void */

/* Kernel families for pa_q8_decode_ex. */
#define PA_Q8_KERNEL_AUTO 0
#define PA_Q8_KERNEL_CUDA_CORE 1     /* f32 FMA dot products and weighted sums      */
#define PA_Q8_KERNEL_TENSOR_CORE 2   /* mma.sync f16 tiles with hi/lo split operands */
#define PA_Q8_KERNEL_TCGEN05 3       /* tcgen05.mma, TMEM accumulators: up to 64 (row, head)
                                        pairs per kv head and CTA; automatic when a kv head
                                        has >= 24 pairs (num_rows * num_heads/num_kv_heads),
                                        > 32 at head size 256                              */

typedef struct pa_q8_decode_options {
    int kernel;            /* PA_Q8_KERNEL_*                                           */
    int partition_tokens;  /* context tokens per split-context partition; 0 = automatic;
                              otherwise a multiple of 128 (at most 16384); partitions
                              need not align with blocks                                */
} pa_q8_decode_options;

/*
 * pa_q8_reshape_and_cache -- quantise new K/V rows and scatter them into the
 * paged int8 caches ("reshape_and_cache_q8.comp", main()).
 *
 * For every row i with slot_mapping[i] != 0xFFFFFFFF and every kv head h,
 * separately for K and V: amax = max_d |x_d|; inv = 127/amax (0 if amax is
 * 0); code_d = clamp(round(x_d * inv), -127, 127) with halves rounded away
 * from zero; the codes and the scale word (f32 bits of amax/127, or of 1.0
 * when amax is 0) are written to the token vector at [slot / block_size,
 * h, slot % block_size].  Each f32 operation is IEEE round-to-nearest, so
 * the words are reproducible bit for bit.
 *
 *   key, value      device f32; row i, head h starts at key + i*key_stride + h*head_size
 *   key_stride,
 *   value_stride    f32 elements between consecutive rows (>= num_kv_heads*head_size)
 *   key_cache,
 *   value_cache     device u32 caches (layout above), 4-byte aligned; written in place
 *   slot_mapping    device u32 [num_tokens]; 0xFFFFFFFF = skip the row; duplicate
 *                   non-PAD slots are a caller error (unspecified result)
 *   num_tokens      rows; 0 is a no-op
 *   num_blocks      physical blocks in each cache; slots >= num_blocks*block_size are
 *                   skipped and flagged PA_Q8_DEV_BAD_SLOT
 *   stream          cudaStream_t or NULL
 * Alignment: none required; 16-byte aligned rows (key/value pointers and strides
 * multiples of 4 floats) take the vector-load kernel.
 */
int pa_q8_reshape_and_cache(const float *key, const float *value,
                            uint32_t *key_cache, uint32_t *value_cache,
                            const uint32_t *slot_mapping, int64_t num_tokens,
                            int64_t key_stride, int64_t value_stride,
                            int num_kv_heads, int head_size, int block_size,
                            int64_t num_blocks, void *stream);

/*
 * pa_q8_decode -- single-query paged attention over the int8 caches
 * ("paged_attn_q8.comp": output = softmax(scale * q . K^T) . V per (seq,
 * head), K and V dequantised as code * token scale; the split-context
 * partials and their log-sum-exp merge follow the split-T decode and
 * attn_combine steps of "attention.rs", attention_b).
 *
 *   out             device f32 [num_seqs][num_heads][head_size] (written; 16-byte aligned)
 *   q               device f32 [num_seqs][num_heads][head_size] (16-byte aligned)
 *   key_cache,
 *   value_cache     device u32 caches, 16-byte aligned; block_size % 4 == 0 makes every
 *                   (block, kv head) tile a 16-byte aligned run of block_size*(head_size+4)
 *                   bytes, which the kernels copy whole
 *   block_tables    device u32 [num_seqs][max_blocks_per_seq]
 *   context_lens    device u32 [num_seqs]; 0 gives a zero output row
 *   num_blocks      physical blocks; table entries >= num_blocks are skipped and flagged
 *   scale           softmax scale (e.g. 1/sqrt(head_size))
 *   workspace       device scratch of >= pa_q8_decode_workspace_size() bytes (never 0),
 *                   16-byte aligned; its contents need no initialisation and are
 *                   overwritten (sequence order, split-context partials)
 *   stream          cudaStream_t or NULL
 * Concurrent calls on different streams need different workspaces.
 */
int pa_q8_decode(float *out, const float *q,
                 const uint32_t *key_cache, const uint32_t *value_cache,
                 const uint32_t *block_tables, const uint32_t *context_lens,
                 int num_seqs, int num_heads, int num_kv_heads, int head_size,
                 int block_size, int max_blocks_per_seq, int64_t num_blocks,
                 float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_q8_decode_noalloc -- pa_q8_decode for callers that cannot allocate.
 * The pages have no counterpart to this entry point.
 *
 * Some callers cannot give the library device memory for scratch: a plugin
 * hosted by another runtime that owns every device allocation and hands its
 * plugins no allocator, or a serving loop whose latency budget rules out
 * allocation calls.  This entry point takes no workspace and allocates
 * nothing: the split-context partials go to a fixed buffer of
 * PA_Q8_NOALLOC_SCRATCH_BYTES compiled into the library (every GPU that
 * loads the library holds it until the process exits).  Arguments, layouts,
 * kernels and results are those of pa_q8_decode.
 *   - Sizes whose partials exceed the buffer return PA_Q8_EWORKSPACE
 *     (pa_q8_decode_workspace_size() gives the bytes a shape needs).
 *   - The first call on a device looks up the buffer's device address
 *     (cudaGetSymbolAddress) with that device current and caches it.
 *   - All calls on a device share the buffer: calls whose work overlaps on
 *     the GPU (different streams, concurrent launches) race on it.  The
 *     buffer keeps the previous call's contents, none of which is read as
 *     an initial value.
 */
#define PA_Q8_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)
int pa_q8_decode_noalloc(float *out, const float *q,
                         const uint32_t *key_cache, const uint32_t *value_cache,
                         const uint32_t *block_tables, const uint32_t *context_lens,
                         int num_seqs, int num_heads, int num_kv_heads, int head_size,
                         int block_size, int max_blocks_per_seq, int64_t num_blocks,
                         float scale, void *stream);

/* Workspace bytes pa_q8_decode needs for these sizes: the sequence order
 * (longest context first) and, when a sequence can span more than one
 * partition, the split-context partials.  Returns 0 for invalid sizes; the
 * decode call reports those. */
size_t pa_q8_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                   int head_size, int block_size, int max_blocks_per_seq);

/* pa_q8_decode with an explicit kernel family and partition size (opts may
 * be NULL = automatic).  Every choice computes the same result within f32
 * rounding. */
int pa_q8_decode_ex(float *out, const float *q,
                    const uint32_t *key_cache, const uint32_t *value_cache,
                    const uint32_t *block_tables, const uint32_t *context_lens,
                    int num_seqs, int num_heads, int num_kv_heads, int head_size,
                    int block_size, int max_blocks_per_seq, int64_t num_blocks,
                    float scale, void *workspace, size_t workspace_bytes, void *stream,
                    const pa_q8_decode_options *opts);

size_t pa_q8_decode_workspace_size_ex(int num_seqs, int num_heads, int num_kv_heads,
                                      int head_size, int block_size, int max_blocks_per_seq,
                                      const pa_q8_decode_options *opts);

/*
 * pa_q8_decode_rows -- causal decode of several query rows per sequence
 * ("attention.rs", attention_b: the loop over rows b whose visible length is
 * the base position + b + 1).  Sequence s holds c = min(context_lens[s],
 * max_blocks_per_seq * block_size) tokens in the caches, the last num_rows of
 * which belong to the rows being decoded: query row b (0 <= b < num_rows)
 * attends to the first c - (num_rows - 1 - b) tokens; a row that sees none is
 * written as zeros.  num_rows = 1 is pa_q8_decode_ex.
 *
 *   out, q          device f32 [num_seqs][num_rows][num_heads][head_size], 16-byte aligned
 *   num_rows        query rows per sequence, >= 1; num_kv_heads * num_rows *
 *                   (num_heads / num_kv_heads) <= 65535
 *   workspace       >= pa_q8_decode_rows_workspace_size() bytes (never 0)
 * Every other argument, the status codes and the kernel families are those
 * of pa_q8_decode_ex.  The rows of a kv head share each K/V tile the kernel
 * copies, so the cache is read once per call whatever num_rows is.
 */
int pa_q8_decode_rows(float *out, const float *q,
                      const uint32_t *key_cache, const uint32_t *value_cache,
                      const uint32_t *block_tables, const uint32_t *context_lens,
                      int num_seqs, int num_rows, int num_heads, int num_kv_heads,
                      int head_size, int block_size, int max_blocks_per_seq,
                      int64_t num_blocks, float scale, void *workspace,
                      size_t workspace_bytes, void *stream, const pa_q8_decode_options *opts);

/*
 * pa_q8_decode_append -- one decode step with the newest tokens' K/V
 * appended inside the attention launch: reshape_and_cache_q8 of those rows
 * followed by pa_q8_decode_rows, in that order (append, then attend), as one
 * attention launch (after the ordering prep, when the plan has one).
 *
 * context_lens[s] counts the new tokens: row b (0 <= b < num_rows) of the
 * new K/V rows is position c - num_rows + b of sequence s, c = min(
 * context_lens[s], max_blocks_per_seq * block_size); it is quantised exactly
 * as pa_q8_reshape_and_cache does (same words, bit for bit) and stored at
 * slot block_tables[s][p / block_size] * block_size + p % block_size.  Rows
 * whose position is negative (c < num_rows) are not stored.  Query row b then
 * attends to the first c - (num_rows - 1 - b) tokens, its own among them.
 *
 *   key, value      device f32 rows, row (s, b) at key + (s * num_rows + b) *
 *                   key_stride holding num_kv_heads * head_size floats (kv head
 *                   major); 16-byte aligned, strides multiples of 4 floats
 *   key_cache,
 *   value_cache     written (the new tokens' slots) and read
 * Every other argument, the workspace (pa_q8_decode_rows_workspace_size),
 * the kernel families (each stores the new tokens itself) and the status
 * codes are those of pa_q8_decode_rows.  A slot whose block id is
 * >= num_blocks is neither written nor read, and flagged
 * PA_Q8_DEV_BAD_BLOCK.
 */
int pa_q8_decode_append(float *out, const float *q, const float *key, const float *value,
                        int64_t key_stride, int64_t value_stride,
                        uint32_t *key_cache, uint32_t *value_cache,
                        const uint32_t *block_tables, const uint32_t *context_lens,
                        int num_seqs, int num_rows, int num_heads, int num_kv_heads,
                        int head_size, int block_size, int max_blocks_per_seq,
                        int64_t num_blocks, float scale, void *workspace,
                        size_t workspace_bytes, void *stream, const pa_q8_decode_options *opts);

size_t pa_q8_decode_rows_workspace_size(int num_seqs, int num_rows, int num_heads,
                                        int num_kv_heads, int head_size, int block_size,
                                        int max_blocks_per_seq, const pa_q8_decode_options *opts);

/*
 * ---- The f32 cache variant ------------------------------------------------
 * "paged_attn_q8.comp" (header comment) describes itself as the math of
 * "paged_attn.comp" over an int8 cache instead of an f32 one ("1 byte/elem
 * vs the f32 cache's 4"), and "reshape_and_cache_q8.comp" says its slot rule
 * mirrors the f32 writer.  Neither f32 shader is on the pages; the layout
 * read here is the q8 one with f32 elements and no scale word:
 *   f32 [num_blocks][num_kv_heads][block_size][head_size].
 * Same arguments, statuses, device flags and result semantics as the q8
 * calls; block_size a power of two (>= 8 for the decode, whose tiles move as
 * 2-D tensor copies), num_blocks * num_kv_heads * block_size < 2^31.
 */

/* Copy each (token, kv head) K and V vector to its slot of the f32 caches;
 * slot 0xFFFFFFFF skips the row, slots >= num_blocks * block_size are skipped
 * and flagged PA_Q8_DEV_BAD_SLOT.  Rows as in pa_q8_reshape_and_cache (any
 * 4-byte alignment; 16-byte aligned rows and caches take 16-byte moves). */
int pa_f32_reshape_and_cache(const float *key, const float *value,
                             float *key_cache, float *value_cache,
                             const uint32_t *slot_mapping, int64_t num_tokens,
                             int64_t key_stride, int64_t value_stride,
                             int num_kv_heads, int head_size, int block_size,
                             int64_t num_blocks, void *stream);

/* pa_q8_decode over the f32 caches (16-byte aligned), output = softmax(scale
 * * q . K^T) . V per (seq, head) with the same GQA map, clamp, empty-context
 * rule and split-context combine.  opts may set partition_tokens; its kernel
 * must be PA_Q8_KERNEL_AUTO (the f32 cache has one kernel family). */
int pa_f32_decode(float *out, const float *q,
                  const float *key_cache, const float *value_cache,
                  const uint32_t *block_tables, const uint32_t *context_lens,
                  int num_seqs, int num_heads, int num_kv_heads, int head_size,
                  int block_size, int max_blocks_per_seq, int64_t num_blocks,
                  float scale, void *workspace, size_t workspace_bytes, void *stream,
                  const pa_q8_decode_options *opts);

size_t pa_f32_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads,
                                    int head_size, int block_size, int max_blocks_per_seq,
                                    const pa_q8_decode_options *opts);

/*
 * ---- The contiguous q8 cache with a side scale region ----------------------
 * "attention.rs" (cherenkov qwen4_exp gpu) appends a step's K/V rows to a
 * per-sequence contiguous q8 cache with its kv_append_q8 dispatch (row =
 * kv_row, t0, nb, scale_off = kv_q8_side(max_t, kv_row); nb * (kv_row/32) * 2
 * subgroups) and attends over it.  The shader is not on the page; the layout
 * read here, one u32 buffer per cache (K, V), sequences back to back:
 *   sequence s at word s * pa_q8c_cache_words(max_t, num_kv_heads, head_size):
 *     codes  [max_t][kv_row / 4] words, kv_row = num_kv_heads * head_size,
 *            int8 code e of a row in byte e % 4 of word e / 4 (kv head major);
 *     scales [max_t][kv_row / 32] f32 bit patterns, scale j of a row covering
 *            codes 32j .. 32j + 31 (amax / 127 of that group, 1.0 when 0),
 *            starting at word max_t * kv_row / 4 of the sequence (scale_off).
 * A 32-element group is quantised like a paged token vector (same rounding,
 * same words for the same values).
 */
size_t pa_q8c_cache_words(int64_t max_t, int num_kv_heads, int head_size);

/* Quantise rows into the contiguous caches: row i (f32, kv_row floats, row
 * stride key_stride / value_stride) goes to position slot % max_t of sequence
 * slot / max_t, slot = slot_mapping[i]; 0xFFFFFFFF skips the row, slots >=
 * num_seqs * max_t are skipped and flagged PA_Q8_DEV_BAD_SLOT.  head_size 64,
 * 128 or 256. */
int pa_q8c_append(const float *key, const float *value, int64_t key_stride, int64_t value_stride,
                  uint32_t *key_cache, uint32_t *value_cache, const uint32_t *slot_mapping,
                  int64_t num_tokens, int num_kv_heads, int head_size, int64_t max_t, int num_seqs,
                  void *stream);

/* Single-query decode over the contiguous caches: out[s, h] = softmax(scale *
 * q[s, h] . K^T) . V over positions [0, min(context_lens[s], max_t)) of
 * sequence s, K and V dequantised as code * group scale, kv head h / (num_heads
 * / num_kv_heads); empty context -> zeros.  q, out [num_seqs][num_heads][head_size]
 * f32, 16-byte aligned; caches 16-byte aligned; head_size 128 or 256 (64 is
 * EUNSUPPORTED: its 8-byte scale rows cannot be bulk-copied).  opts: kernel
 * AUTO or TENSOR_CORE, partition_tokens as for pa_q8_decode_ex. */
int pa_q8c_decode(float *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                  const uint32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads,
                  int head_size, int64_t max_t, float scale, void *workspace, size_t workspace_bytes,
                  void *stream, const pa_q8_decode_options *opts);

size_t pa_q8c_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                    int64_t max_t, const pa_q8_decode_options *opts);

/* The launch plan pa_q8_decode_ex would use (no launch): kernel family,
 * tokens per partition, partitions per sequence (grid x), CTAs launched for
 * the attention kernel.  Any output pointer may be NULL.  Needs a current
 * CUDA device (it reads the SM count). */
int pa_q8_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                      int block_size, int max_blocks_per_seq,
                      const pa_q8_decode_options *opts, int *kernel, int *partition_tokens,
                      int *num_partitions, int64_t *num_ctas);

/* Read (and with clear != 0, reset) the sticky device status bits of the
 * current device.  Synchronises `stream` first. */
int pa_q8_device_status(uint32_t *bits, int clear, void *stream);

/* Launch a one-CTA kernel that waits on a barrier nothing will release,
 * with the given limit in microseconds (1..10^6).  The kernel gives up,
 * sets PA_Q8_DEV_WAIT_TIMEOUT and exits; the context stays usable.  This
 * is how the bounded-wait path of the decode kernels is exercised without
 * faulting or hanging a GPU. */
int pa_q8_selftest_wait_timeout(uint32_t timeout_us, void *stream);

/* Human-readable text for a pa_q8_status value (static storage). */
const char *pa_q8_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int pa_q8_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_Q8_H */
