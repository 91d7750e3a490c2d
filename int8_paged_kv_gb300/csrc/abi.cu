// C ABI of libpa_q8.so: argument checks, launch planning, status strings.
// Every check happens on the host before anything is queued; the kernels
// are in writer.cu and the decode*.cu files.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "pa_q8.h"
#include "kernels.h"

namespace {

// Per-device sticky status bits written by the kernels.
__device__ uint32_t g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
uint32_t *g_status_ptr[kMaxDevices];
int g_num_sms[kMaxDevices];

// Device address of the status word and the SM count of the current device,
// looked up once per device.
int device_info(uint32_t **status, int *num_sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_status_ptr[dev]) {
        void *p = nullptr;
        int sms = 0;
        if (cudaGetSymbolAddress(&p, g_device_status) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return PA_Q8_ECUDA;
        }
        g_status_ptr[dev] = static_cast<uint32_t *>(p);
        g_num_sms[dev] = sms;
    }
    if (status) *status = g_status_ptr[dev];
    if (num_sms) *num_sms = g_num_sms[dev];
    return PA_Q8_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
bool head_size_ok(int d) { return d == 64 || d == 128 || d == 256; }

int check_decode_shape(int num_seqs, int num_heads, int num_kv_heads, int head_size, int block_size,
                       int max_blocks_per_seq, int num_rows = 1) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 ||
        max_blocks_per_seq <= 0 || num_rows <= 0)
        return PA_Q8_EINVAL;
    if (num_heads % num_kv_heads != 0 || head_size % 4 != 0 || block_size % 4 != 0) return PA_Q8_EINVAL;
    if (!head_size_ok(head_size) || !pow2(block_size) || block_size > 1024) return PA_Q8_EUNSUPPORTED;
    if (num_seqs > 65535) return PA_Q8_EUNSUPPORTED;            // grid z
    // grid y = kv heads x groups of (row, head) pairs; at worst one pair per group
    if ((int64_t)num_kv_heads * num_rows * (num_heads / num_kv_heads) > 65535) return PA_Q8_EUNSUPPORTED;
    if ((int64_t)max_blocks_per_seq * block_size > (int64_t)1 << 30) return PA_Q8_EUNSUPPORTED;
    return PA_Q8_OK;
}

// f32: the f32-cache decode, whose only kernel family is its own (opts->kernel
// must be automatic).
int plan_for(pa_q8::DecodeArgs &a, const pa_q8_decode_options *opts, int num_sms, bool f32 = false) {
    int kernel = opts ? opts->kernel : PA_Q8_KERNEL_AUTO;
    const int pt = opts ? opts->partition_tokens : 0;
    if (kernel < PA_Q8_KERNEL_AUTO || kernel > PA_Q8_KERNEL_TCGEN05) return PA_Q8_EINVAL;
    if (f32) {
        if (kernel != PA_Q8_KERNEL_AUTO) return PA_Q8_EINVAL;
        kernel = pa_q8::kF32;
    }
    if (pt < 0 || (pt > 0 && pt % 128 != 0)) return PA_Q8_EINVAL;
    if (!pa_q8::make_plan(a, kernel, pt, num_sms)) return PA_Q8_EUNSUPPORTED;
    return PA_Q8_OK;
}

// Extra limits of the f32-cache decode: tensor copies of min(B, 32)-row
// boxes 1024-byte aligned in shared memory (B >= 8), row coordinates in s32.
int check_f32_shape(int num_kv_heads, int block_size, int64_t num_blocks) {
    if (block_size < 8) return PA_Q8_EUNSUPPORTED;
    if (num_blocks > 0 && num_blocks * num_kv_heads * block_size > (int64_t)0x7FFFFFFF) return PA_Q8_EUNSUPPORTED;
    return PA_Q8_OK;
}

void fill_shape(pa_q8::DecodeArgs &a, int num_seqs, int num_heads, int num_kv_heads, int head_size,
                int block_size, int max_blocks_per_seq, int num_rows = 1) {
    std::memset(&a, 0, sizeof a);
    a.num_seqs = num_seqs;
    a.num_rows = num_rows;
    a.num_heads = num_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_size = head_size;
    a.block_size = block_size;
    a.max_blocks_per_seq = max_blocks_per_seq;
}

size_t workspace_impl(int num_seqs, int num_rows, int num_heads, int num_kv_heads, int head_size,
                      int block_size, int max_blocks_per_seq, const pa_q8_decode_options *opts,
                      bool f32 = false) {
    if (check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq,
                           num_rows) != PA_Q8_OK)
        return 0;
    if (f32 && check_f32_shape(num_kv_heads, block_size, 0) != PA_Q8_OK) return 0;
    pa_q8::DecodeArgs a;
    fill_shape(a, num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, num_rows);
    int sms = 0;
    if (device_info(nullptr, &sms) != PA_Q8_OK) sms = 152;     // size query without a device
    if (plan_for(a, opts, sms, f32) != PA_Q8_OK) return 0;
    return pa_q8::plan_workspace_bytes(a);
}

// New K/V rows of the fused append (key == nullptr: plain decode).
struct AppendRows {
    const float *key = nullptr;
    const float *value = nullptr;
    int64_t key_stride = 0;
    int64_t value_stride = 0;
};

int decode_impl(float *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                const uint32_t *block_tables, const uint32_t *context_lens, int num_seqs, int num_rows,
                int num_heads, int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq,
                int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes, void *stream,
                const pa_q8_decode_options *opts, const AppendRows &app = AppendRows{},
                bool f32 = false) {
    int rc = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq,
                                num_rows);
    if (rc != PA_Q8_OK) return rc;
    if (num_blocks <= 0) return PA_Q8_EINVAL;
    if (f32 && (rc = check_f32_shape(num_kv_heads, block_size, num_blocks)) != PA_Q8_OK) return rc;
    if (!out || !q || !key_cache || !value_cache || !block_tables || !context_lens) return PA_Q8_EINVAL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache) ||
        !aligned4(block_tables) || !aligned4(context_lens))
        return PA_Q8_EALIGN;
    if (app.key) {
        const int64_t row = (int64_t)num_kv_heads * head_size;
        if (!app.value || app.key_stride < row || app.value_stride < row) return PA_Q8_EINVAL;
        if (!aligned16(app.key) || !aligned16(app.value) || app.key_stride % 4 || app.value_stride % 4)
            return PA_Q8_EALIGN;
    }
    uint32_t *status = nullptr;
    int sms = 0;
    rc = device_info(&status, &sms);
    if (rc != PA_Q8_OK) return rc;
    pa_q8::DecodeArgs a;
    fill_shape(a, num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, num_rows);
    rc = plan_for(a, opts, sms, f32);
    if (rc != PA_Q8_OK) return rc;
    const size_t need = pa_q8::plan_workspace_bytes(a);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return PA_Q8_EWORKSPACE;
        if (!aligned16(workspace)) return PA_Q8_EALIGN;
        pa_q8::plan_workspace_layout(a, workspace);
    }
    a.out = out;
    a.q = q;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.block_tables = block_tables;
    a.context_lens = context_lens;
    a.num_blocks = num_blocks;
    a.scale = scale;
    a.status = status;
    a.new_key = app.key;
    a.new_value = app.value;
    a.new_key_stride = app.key_stride;
    a.new_value_stride = app.value_stride;
    if (pa_q8::launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    return PA_Q8_OK;
}

int cq_shape(int num_seqs, int num_heads, int num_kv_heads, int head_size, int64_t max_t) {
    if (num_seqs <= 0 || num_heads <= 0 || num_kv_heads <= 0 || head_size <= 0 || max_t <= 0) return PA_Q8_EINVAL;
    if (num_heads % num_kv_heads != 0 || head_size % 32 != 0) return PA_Q8_EINVAL;
    if (head_size != 128 && head_size != 256) return PA_Q8_EUNSUPPORTED;
    if (num_seqs > 65535 || (int64_t)num_kv_heads * (num_heads / num_kv_heads) > 65535) return PA_Q8_EUNSUPPORTED;
    if (max_t > (int64_t)1 << 30) return PA_Q8_EUNSUPPORTED;
    return PA_Q8_OK;
}

void cq_fill(pa_q8::DecodeArgs &a, int num_seqs, int num_heads, int num_kv_heads, int head_size, int64_t max_t) {
    fill_shape(a, num_seqs, num_heads, num_kv_heads, head_size, 1, (int)max_t);
    a.contiguous = 1;
}

int cq_plan(pa_q8::DecodeArgs &a, const pa_q8_decode_options *opts, int sms) {
    pa_q8_decode_options o = opts ? *opts : pa_q8_decode_options{};
    if (o.kernel != PA_Q8_KERNEL_AUTO && o.kernel != PA_Q8_KERNEL_TENSOR_CORE) return PA_Q8_EINVAL;
    o.kernel = PA_Q8_KERNEL_TENSOR_CORE;
    return plan_for(a, &o, sms);
}

}  // namespace

extern "C" {

int pa_q8_version(void) { return 10000; }

const char *pa_q8_status_string(int status) {
    switch (status) {
        case PA_Q8_OK: return "ok";
        case PA_Q8_EINVAL: return "invalid argument";
        case PA_Q8_EUNSUPPORTED: return "unsupported shape (head_size 64/128/256, block_size a power of two 4..1024)";
        case PA_Q8_EALIGN: return "misaligned pointer or stride";
        case PA_Q8_ECUDA: return "CUDA runtime error";
        case PA_Q8_EWORKSPACE: return "workspace too small";
        default: return "unknown status";
    }
}

int pa_q8_reshape_and_cache(const float *key, const float *value, uint32_t *key_cache,
                            uint32_t *value_cache, const uint32_t *slot_mapping, int64_t num_tokens,
                            int64_t key_stride, int64_t value_stride, int num_kv_heads, int head_size,
                            int block_size, int64_t num_blocks, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_Q8_EINVAL;
    if (head_size % 4 != 0 || block_size % 4 != 0) return PA_Q8_EINVAL;
    if (!head_size_ok(head_size)) return PA_Q8_EUNSUPPORTED;
    if (key_stride < (int64_t)num_kv_heads * head_size || value_stride < (int64_t)num_kv_heads * head_size)
        return PA_Q8_EINVAL;
    if (num_blocks * block_size > (int64_t)0xFFFFFFFFu) return PA_Q8_EUNSUPPORTED;
    if (num_tokens == 0) return PA_Q8_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_Q8_EINVAL;
    if (!aligned4(key) || !aligned4(value) || !aligned4(key_cache) || !aligned4(value_cache) ||
        !aligned4(slot_mapping))
        return PA_Q8_EALIGN;
    uint32_t *status = nullptr;
    int rc = device_info(&status, nullptr);
    if (rc != PA_Q8_OK) return rc;
    pa_q8::WriterArgs a{key, value, key_cache, value_cache, slot_mapping, num_tokens, key_stride,
                        value_stride, num_kv_heads, head_size, block_size, num_blocks, status};
    if (pa_q8::launch_writer(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    return PA_Q8_OK;
}

size_t pa_q8_decode_workspace_size_ex(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                      int block_size, int max_blocks_per_seq,
                                      const pa_q8_decode_options *opts) {
    return workspace_impl(num_seqs, 1, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, opts);
}

int pa_q8_decode_append(float *out, const float *q, const float *key, const float *value,
                        int64_t key_stride, int64_t value_stride, uint32_t *key_cache,
                        uint32_t *value_cache, const uint32_t *block_tables, const uint32_t *context_lens,
                        int num_seqs, int num_rows, int num_heads, int num_kv_heads, int head_size,
                        int block_size, int max_blocks_per_seq, int64_t num_blocks, float scale,
                        void *workspace, size_t workspace_bytes, void *stream,
                        const pa_q8_decode_options *opts) {
    AppendRows app;
    app.key = key;
    app.value = value;
    app.key_stride = key_stride;
    app.value_stride = value_stride;
    if (!key) return PA_Q8_EINVAL;
    return decode_impl(out, q, key_cache, value_cache, block_tables, context_lens, num_seqs, num_rows,
                       num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, num_blocks, scale,
                       workspace, workspace_bytes, stream, opts, app);
}

int pa_f32_reshape_and_cache(const float *key, const float *value, float *key_cache, float *value_cache,
                             const uint32_t *slot_mapping, int64_t num_tokens, int64_t key_stride,
                             int64_t value_stride, int num_kv_heads, int head_size, int block_size,
                             int64_t num_blocks, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_Q8_EINVAL;
    if (head_size % 4 != 0) return PA_Q8_EINVAL;
    if (!head_size_ok(head_size) || !pow2(block_size) || block_size > 1024) return PA_Q8_EUNSUPPORTED;
    if (key_stride < (int64_t)num_kv_heads * head_size || value_stride < (int64_t)num_kv_heads * head_size)
        return PA_Q8_EINVAL;
    if (num_blocks * block_size > (int64_t)0xFFFFFFFFu || num_kv_heads > 65535) return PA_Q8_EUNSUPPORTED;
    if (num_tokens == 0) return PA_Q8_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_Q8_EINVAL;
    if (!aligned4(key) || !aligned4(value) || !aligned4(key_cache) || !aligned4(value_cache) ||
        !aligned4(slot_mapping))
        return PA_Q8_EALIGN;
    uint32_t *status = nullptr;
    int rc = device_info(&status, nullptr);
    if (rc != PA_Q8_OK) return rc;
    pa_q8::WriterArgs a{key, value, reinterpret_cast<uint32_t *>(key_cache),
                        reinterpret_cast<uint32_t *>(value_cache), slot_mapping, num_tokens, key_stride,
                        value_stride, num_kv_heads, head_size, block_size, num_blocks, status};
    if (pa_q8::launch_writer_f32(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    return PA_Q8_OK;
}

int pa_f32_decode(float *out, const float *q, const float *key_cache, const float *value_cache,
                  const uint32_t *block_tables, const uint32_t *context_lens, int num_seqs, int num_heads,
                  int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq, int64_t num_blocks,
                  float scale, void *workspace, size_t workspace_bytes, void *stream,
                  const pa_q8_decode_options *opts) {
    return decode_impl(out, q, reinterpret_cast<const uint32_t *>(key_cache),
                       reinterpret_cast<const uint32_t *>(value_cache), block_tables, context_lens, num_seqs, 1,
                       num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, num_blocks, scale,
                       workspace, workspace_bytes, stream, opts, AppendRows{}, true);
}

size_t pa_f32_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                    int block_size, int max_blocks_per_seq, const pa_q8_decode_options *opts) {
    return workspace_impl(num_seqs, 1, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, opts,
                          true);
}

size_t pa_q8c_cache_words(int64_t max_t, int num_kv_heads, int head_size) {
    if (max_t <= 0 || num_kv_heads <= 0 || head_size <= 0 || head_size % 32 != 0) return 0;
    const int64_t kv_row = (int64_t)num_kv_heads * head_size;
    return (size_t)(max_t * (kv_row / 4) + max_t * (kv_row / 32));
}

int pa_q8c_append(const float *key, const float *value, int64_t key_stride, int64_t value_stride,
                  uint32_t *key_cache, uint32_t *value_cache, const uint32_t *slot_mapping, int64_t num_tokens,
                  int num_kv_heads, int head_size, int64_t max_t, int num_seqs, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_size <= 0 || max_t <= 0 || num_seqs <= 0) return PA_Q8_EINVAL;
    if (head_size % 32 != 0) return PA_Q8_EINVAL;
    if (!head_size_ok(head_size)) return PA_Q8_EUNSUPPORTED;
    const int64_t kv_row = (int64_t)num_kv_heads * head_size;
    if (key_stride < kv_row || value_stride < kv_row) return PA_Q8_EINVAL;
    if ((int64_t)num_seqs * max_t > (int64_t)0xFFFFFFFFu || kv_row / 64 > 65535) return PA_Q8_EUNSUPPORTED;
    if (num_tokens == 0) return PA_Q8_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_Q8_EINVAL;
    if (!aligned4(key) || !aligned4(value) || !aligned4(key_cache) || !aligned4(value_cache) ||
        !aligned4(slot_mapping))
        return PA_Q8_EALIGN;
    uint32_t *status = nullptr;
    int rc = device_info(&status, nullptr);
    if (rc != PA_Q8_OK) return rc;
    pa_q8::WriterArgs a{key, value, key_cache, value_cache, slot_mapping, num_tokens, key_stride,
                        value_stride, num_kv_heads, head_size, 1, num_seqs, status};
    if (pa_q8::launch_cq_append(a, max_t, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    return PA_Q8_OK;
}


size_t pa_q8c_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size, int64_t max_t,
                                    const pa_q8_decode_options *opts) {
    if (cq_shape(num_seqs, num_heads, num_kv_heads, head_size, max_t) != PA_Q8_OK) return 0;
    pa_q8::DecodeArgs a;
    cq_fill(a, num_seqs, num_heads, num_kv_heads, head_size, max_t);
    int sms = 0;
    if (device_info(nullptr, &sms) != PA_Q8_OK) sms = 152;
    if (cq_plan(a, opts, sms) != PA_Q8_OK) return 0;
    return pa_q8::plan_workspace_bytes(a);
}

int pa_q8c_decode(float *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                  const uint32_t *context_lens, int num_seqs, int num_heads, int num_kv_heads, int head_size,
                  int64_t max_t, float scale, void *workspace, size_t workspace_bytes, void *stream,
                  const pa_q8_decode_options *opts) {
    int rc = cq_shape(num_seqs, num_heads, num_kv_heads, head_size, max_t);
    if (rc != PA_Q8_OK) return rc;
    if (!out || !q || !key_cache || !value_cache || !context_lens) return PA_Q8_EINVAL;
    if (!aligned16(out) || !aligned16(q) || !aligned16(key_cache) || !aligned16(value_cache) || !aligned4(context_lens))
        return PA_Q8_EALIGN;
    uint32_t *status = nullptr;
    int sms = 0;
    rc = device_info(&status, &sms);
    if (rc != PA_Q8_OK) return rc;
    pa_q8::DecodeArgs a;
    cq_fill(a, num_seqs, num_heads, num_kv_heads, head_size, max_t);
    rc = cq_plan(a, opts, sms);
    if (rc != PA_Q8_OK) return rc;
    const size_t need = pa_q8::plan_workspace_bytes(a);
    if (!workspace || workspace_bytes < need) return PA_Q8_EWORKSPACE;
    if (!aligned16(workspace)) return PA_Q8_EALIGN;
    pa_q8::plan_workspace_layout(a, workspace);
    a.out = out;
    a.q = q;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.context_lens = context_lens;
    a.num_blocks = num_seqs;
    a.scale = scale;
    a.status = status;
    if (pa_q8::launch_decode(a, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    return PA_Q8_OK;
}

size_t pa_q8_decode_rows_workspace_size(int num_seqs, int num_rows, int num_heads, int num_kv_heads,
                                        int head_size, int block_size, int max_blocks_per_seq,
                                        const pa_q8_decode_options *opts) {
    return workspace_impl(num_seqs, num_rows, num_heads, num_kv_heads, head_size, block_size,
                          max_blocks_per_seq, opts);
}

size_t pa_q8_decode_workspace_size(int num_seqs, int num_heads, int num_kv_heads, int head_size,
                                   int block_size, int max_blocks_per_seq) {
    return pa_q8_decode_workspace_size_ex(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                          max_blocks_per_seq, nullptr);
}

int pa_q8_decode_plan(int num_seqs, int num_heads, int num_kv_heads, int head_size, int block_size,
                      int max_blocks_per_seq, const pa_q8_decode_options *opts, int *kernel,
                      int *partition_tokens, int *num_partitions, int64_t *num_ctas) {
    int rc = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq);
    if (rc != PA_Q8_OK) return rc;
    int sms = 0;
    rc = device_info(nullptr, &sms);
    if (rc != PA_Q8_OK) return rc;
    pa_q8::DecodeArgs a;
    fill_shape(a, num_seqs, num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq);
    rc = plan_for(a, opts, sms);
    if (rc != PA_Q8_OK) return rc;
    if (kernel) *kernel = a.kernel;
    if (partition_tokens) *partition_tokens = a.partition_tokens;
    if (num_partitions) *num_partitions = a.num_partitions;
    if (num_ctas) *num_ctas = pa_q8::plan_num_ctas(a);
    return PA_Q8_OK;
}

int pa_q8_decode_ex(float *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                    const uint32_t *block_tables, const uint32_t *context_lens, int num_seqs, int num_heads,
                    int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq,
                    int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes, void *stream,
                    const pa_q8_decode_options *opts) {
    return decode_impl(out, q, key_cache, value_cache, block_tables, context_lens, num_seqs, 1, num_heads,
                       num_kv_heads, head_size, block_size, max_blocks_per_seq, num_blocks, scale, workspace,
                       workspace_bytes, stream, opts);
}

int pa_q8_decode_rows(float *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                      const uint32_t *block_tables, const uint32_t *context_lens, int num_seqs, int num_rows,
                      int num_heads, int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq,
                      int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes, void *stream,
                      const pa_q8_decode_options *opts) {
    return decode_impl(out, q, key_cache, value_cache, block_tables, context_lens, num_seqs, num_rows,
                       num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq, num_blocks, scale,
                       workspace, workspace_bytes, stream, opts);
}

int pa_q8_decode(float *out, const float *q, const uint32_t *key_cache, const uint32_t *value_cache,
                 const uint32_t *block_tables, const uint32_t *context_lens, int num_seqs, int num_heads,
                 int num_kv_heads, int head_size, int block_size, int max_blocks_per_seq, int64_t num_blocks,
                 float scale, void *workspace, size_t workspace_bytes, void *stream) {
    return pa_q8_decode_ex(out, q, key_cache, value_cache, block_tables, context_lens, num_seqs, num_heads,
                           num_kv_heads, head_size, block_size, max_blocks_per_seq, num_blocks, scale, workspace,
                           workspace_bytes, stream, nullptr);
}

int pa_q8_device_status(uint32_t *bits, int clear, void *stream) {
    if (!bits) return PA_Q8_EINVAL;
    uint32_t *status = nullptr;
    int rc = device_info(&status, nullptr);
    if (rc != PA_Q8_OK) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaMemcpyAsync(bits, status, sizeof(uint32_t), cudaMemcpyDeviceToHost, st) != cudaSuccess ||
        cudaStreamSynchronize(st) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    if (clear && *bits) {
        if (cudaMemsetAsync(status, 0, sizeof(uint32_t), st) != cudaSuccess ||
            cudaStreamSynchronize(st) != cudaSuccess) {
            cudaGetLastError();
            return PA_Q8_ECUDA;
        }
    }
    return PA_Q8_OK;
}

int pa_q8_selftest_wait_timeout(uint32_t timeout_us, void *stream) {
    if (timeout_us < 1 || timeout_us > 1000000) return PA_Q8_EINVAL;
    uint32_t *status = nullptr;
    int rc = device_info(&status, nullptr);
    if (rc != PA_Q8_OK) return rc;
    if (pa_q8::launch_wait_selftest(timeout_us, status, static_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    return PA_Q8_OK;
}

}  // extern "C"

// ------------------------------------------------- decode without allocation
//
// Some callers cannot give this library device memory for scratch: a plugin
// hosted by another runtime that owns every device allocation and hands its
// plugins no allocator, or a serving loop whose latency budget rules out
// allocation calls (they can synchronise the device and take unbounded
// time).  pa_q8_decode_noalloc serves them: it keeps the split-context
// partials in a buffer compiled into this library, a fixed 64 MiB that every
// GPU loading the library holds until the process exits.  Host code cannot
// use the array's name as a device address (it is a host-side stand-in), so
// the first call on each device looks the address up with
// cudaGetSymbolAddress while that device is current and caches it.  All
// calls on a device share the buffer, and calls whose kernels overlap on the
// GPU race on it.  The buffer keeps the previous call's partials; nothing in
// it needs to start at zero, since every partial the combine step reads is
// written earlier in the same call.
namespace {

constexpr size_t kNoAllocScratchBytes = PA_Q8_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];
void *g_noalloc_ptr[kMaxDevices];

int noalloc_scratch(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return PA_Q8_ECUDA;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_noalloc_ptr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            cudaGetLastError();
            return PA_Q8_ECUDA;
        }
        g_noalloc_ptr[dev] = p;
    }
    *ptr = g_noalloc_ptr[dev];
    return PA_Q8_OK;
}

}  // namespace

extern "C" int pa_q8_decode_noalloc(float *out, const float *q, const uint32_t *key_cache,
                                    const uint32_t *value_cache, const uint32_t *block_tables,
                                    const uint32_t *context_lens, int num_seqs, int num_heads,
                                    int num_kv_heads, int head_size, int block_size,
                                    int max_blocks_per_seq, int64_t num_blocks, float scale,
                                    void *stream) {
    const int rc = check_decode_shape(num_seqs, num_heads, num_kv_heads, head_size, block_size,
                                      max_blocks_per_seq);
    if (rc != PA_Q8_OK) return rc;
    void *scratch = nullptr;
    const int src = noalloc_scratch(&scratch);
    if (src != PA_Q8_OK) return src;
    // Same launch plan and kernels as pa_q8_decode; partials that would not
    // fit in the fixed buffer make it return PA_Q8_EWORKSPACE.
    return pa_q8_decode_ex(out, q, key_cache, value_cache, block_tables, context_lens, num_seqs,
                           num_heads, num_kv_heads, head_size, block_size, max_blocks_per_seq,
                           num_blocks, scale, scratch, kNoAllocScratchBytes, stream, nullptr);
}
