// Internal launch interface between the C-ABI layer (abi.cu) and the
// kernels.  Host-side structs only; argument checking happens in abi.cu.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace pa_q8 {

struct WriterArgs {
    const float *key;
    const float *value;
    uint32_t *key_cache;
    uint32_t *value_cache;
    const uint32_t *slot_mapping;
    int64_t num_tokens;
    int64_t key_stride;
    int64_t value_stride;
    int num_kv_heads;
    int head_size;
    int block_size;
    int64_t num_blocks;
    uint32_t *status;
};

cudaError_t launch_writer(const WriterArgs &a, cudaStream_t stream);
// The contiguous q8 cache's append (per-sequence code rows + side scale
// region, 32-element groups); a.num_blocks holds the number of sequences.
cudaError_t launch_cq_append(const WriterArgs &a, int64_t max_t, cudaStream_t stream);
// The f32 cache's writer: key_cache / value_cache hold f32 [blocks][Hk][B][D].
cudaError_t launch_writer_f32(const WriterArgs &a, cudaStream_t stream);

// kTcgen05: 5th-generation tensor cores (many virtual heads per kv head);
// kF32: the f32-cache decode (pa_f32_decode only)
enum KernelFamily { kAuto = 0, kCudaCore = 1, kTensorCore = 2, kTcgen05 = 3, kF32 = 8 };

struct DecodeArgs {
    float *out;
    const float *q;
    const uint32_t *key_cache;
    const uint32_t *value_cache;
    const uint32_t *block_tables;
    const uint32_t *context_lens;
    int num_seqs;
    int num_rows;          // query rows per sequence (causal: row b sees c - (rows - 1 - b) tokens)
    int num_heads;
    int num_kv_heads;
    int head_size;
    int block_size;
    int max_blocks_per_seq;
    int64_t num_blocks;
    float scale;
    // plan (filled by make_plan)
    int kernel;            // kCudaCore, kTensorCore, kTcgen05 or kF32
    int partition_tokens;  // tokens per partition
    int num_partitions;    // partitions per sequence (grid x)
    int heads_per_cta;     // query heads one CTA serves (one kv head's group, or part of it)
    int head_groups;       // CTAs per (seq, kv head, partition) along the group
    int one_wave;          // one partition per context and every CTA resident at once: no
                           // ordering and no combine counters, so no prep kernel
    int sep_combine;       // split contexts merged by a combine grid of its own (launched as a
                           // programmatic dependent), not by the last CTA of each group: no
                           // arrival counters, no ordering, so no prep kernel
    int rec_slots;         // partial records per (row, partition): 1, or the token-slot warps
                           // of a one-tile tensor-core CTA, each storing its own (combine grid)
    int per_sm;            // CTAs per SM the waves are sized for (selects the contiguous
                           // kernel's register budget)
    // workspace: sequence order [S] (u64: clamped length << 32 | sequence,
    // longest context first); when partitions > 1 also arrival counters
    // [S][Hk * head_groups] (u32) and one partial record per (sequence, query
    // row, head, partition) -- or rec_slots of them --: [S][R][H][P][rec_slots]
    // [head_size + 4] f32, the weighted sum A followed by m, l and two spare words
    unsigned long long *order;
    uint32_t *counters;
    float *partials;
    uint32_t *status;
    // fused append (new_key == nullptr: none): rows [num_seqs][num_rows] of
    // num_kv_heads * head_size floats, row (s, b) at new_key + (s * num_rows +
    // b) * new_key_stride; the token of row b is position c - num_rows + b
    const float *new_key;
    const float *new_value;
    int64_t new_key_stride;
    int64_t new_value_stride;
    // contiguous q8 cache (per sequence: code rows, then group scales); then
    // block_size = 1, max_blocks_per_seq = max_t and block_tables is unused
    int contiguous;
};

struct DecodePlanLimits {
    int num_sms;
};

// Fill the plan fields of `a` (kernel family, partition size, grid).
// Returns false if no kernel serves these sizes.
bool make_plan(DecodeArgs &a, int requested_kernel, int requested_partition, int num_sms);

// Workspace bytes for a plan.
size_t plan_workspace_bytes(const DecodeArgs &a);

// Point the scratch fields of `a` into a workspace of plan_workspace_bytes(a).
void plan_workspace_layout(DecodeArgs &a, void *workspace);

// Grid size of the attention kernel for a plan.
int64_t plan_num_ctas(const DecodeArgs &a);

cudaError_t launch_decode(const DecodeArgs &a, cudaStream_t stream);

cudaError_t launch_wait_selftest(uint32_t timeout_us, uint32_t *status, cudaStream_t stream);

}  // namespace pa_q8
