// The kvfp8 C ABI: host-side validation, then one enqueue on the caller's stream.
// Declarations, argument meanings and error behaviour: include/kvfp8.h.
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>

#include "../../include/kvfp8.h"
#include "kvfp8_internal.h"

namespace {

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned(const void *p, uintptr_t n) { return (reinterpret_cast<uintptr_t>(p) & (n - 1)) == 0; }

bool dtype_ok(kvfp8_dtype t) { return t == KVFP8_BF16 || t == KVFP8_F32; }

kvfp8_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return KVFP8_OK;
    if (e == cudaErrorNotSupported) return KVFP8_ERR_UNSUPPORTED;
    return KVFP8_ERR_CUDA;
}

bool cache_dtype_ok(kvfp8_cache_dtype t) { return t == KVFP8_CACHE_E4M3 || t == KVFP8_CACHE_BF16; }

bool block_size_ok_for_decode(int32_t bs) {
    return bs == 8 || bs == 16 || bs == 32 || bs == 64 || bs == 128 || bs == 256;
}

}  // namespace

namespace kvfp8 {

kvfp8_status validate_decode(const void *out, const void *query, const uint8_t *key_cache,
                             const uint8_t *value_cache, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *seq_lens,
                             int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, float sm_scale,
                             int scale_dtype, bool *nothing_to_do) {
    *nothing_to_do = false;
    if (!dtype_ok(static_cast<kvfp8_dtype>(scale_dtype))) return KVFP8_ERR_DTYPE;
    if (num_seqs < 0 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || num_blocks < 1 ||
        max_blocks_per_seq < 1)
        return KVFP8_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVFP8_ERR_SHAPE;
    if (!block_size_ok_for_decode(block_size)) return KVFP8_ERR_SHAPE;
    if (n_q / n_kv > 128) return KVFP8_ERR_UNSUPPORTED;  // past the tensor-core kernel's rows
    if (static_cast<int64_t>(num_blocks) * block_size > 0x7FFFFFFFLL ||
        static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
        return KVFP8_ERR_SHAPE;
    if (std::isnan(sm_scale) || std::isinf(sm_scale)) return KVFP8_ERR_SCALE;
    if (num_seqs == 0) {
        *nothing_to_do = true;
        return KVFP8_OK;
    }
    if (!out || !query || !key_cache || !value_cache || !block_tables || !seq_lens)
        return KVFP8_ERR_NULL;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache) || !aligned(block_tables, 4) || !aligned(seq_lens, 4))
        return KVFP8_ERR_ALIGN;
    return KVFP8_OK;
}

kvfp8_status launch_decode_validated(void *out, const void *query, const uint8_t *key_cache,
                                     const uint8_t *value_cache, const int32_t *block_tables,
                                     int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                     int32_t num_seqs, int32_t n_q, int32_t n_kv,
                                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float sm_scale, const void *k_scale, const void *v_scale,
                                     int scale_dtype, void *workspace, uint32_t *status,
                                     kvfp8_stream_t stream) {
    DecodeArgs d;
    d.out = out;
    d.query = query;
    d.key_cache = key_cache;
    d.value_cache = value_cache;
    d.block_tables = block_tables;
    d.max_blocks_per_seq = max_blocks_per_seq;
    d.seq_lens = seq_lens;
    d.num_seqs = num_seqs;
    d.n_q = n_q;
    d.n_kv = n_kv;
    d.head_dim = head_dim;
    d.block_size = block_size;
    d.num_blocks = num_blocks;
    d.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    d.k_scale = k_scale;
    d.v_scale = v_scale;
    d.scale_dtype = scale_dtype;
    d.workspace = workspace;
    d.status = status;
    d.qsl = nullptr;
    d.qmax = 1;
    d.qrows = num_seqs;
    d.k_bf16 = 0;
    d.v_bf16 = 0;
    return from_cuda(launch_paged_decode(d, reinterpret_cast<cudaStream_t>(stream)));
}

}  // namespace kvfp8

extern "C" {

kvfp8_status kvfp8_reshape_and_cache(const void *key, const void *value, kvfp8_dtype src_dtype,
                                     int64_t key_stride, int64_t value_stride, int64_t num_tokens,
                                     uint8_t *key_cache, uint8_t *value_cache, int32_t num_blocks,
                                     int32_t block_size, int32_t n_kv, int32_t head_dim,
                                     const int64_t *slot_mapping, const void *k_scale,
                                     const void *v_scale, kvfp8_dtype scale_dtype,
                                     uint32_t *status, kvfp8_stream_t stream) {
    if (!dtype_ok(src_dtype) || !dtype_ok(scale_dtype)) return KVFP8_ERR_DTYPE;
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || block_size > 1024 || n_kv < 1 ||
        head_dim < 1)
        return KVFP8_ERR_SHAPE;
    const int64_t row = static_cast<int64_t>(n_kv) * head_dim;
    if (row % 8 != 0 || row > (1 << 20) || key_stride < row || value_stride < row)
        return KVFP8_ERR_SHAPE;
    if (num_tokens == 0) return KVFP8_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return KVFP8_ERR_NULL;
    const int64_t esz = src_dtype == KVFP8_F32 ? 4 : 2;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (key_stride * esz) % 16 != 0 || (value_stride * esz) % 16 != 0 || !aligned(slot_mapping, 8))
        return KVFP8_ERR_ALIGN;
    kvfp8::ReshapeArgs a;
    a.key = key;
    a.value = value;
    a.src_dtype = src_dtype;
    a.key_stride = key_stride;
    a.value_stride = value_stride;
    a.num_tokens = num_tokens;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
    a.row_elems = static_cast<int32_t>(row);
    a.slot_mapping = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.scale_dtype = scale_dtype;
    a.status = status;
    a.positions = nullptr;
    a.cos_sin = nullptr;
    a.max_pos = 0;
    a.rot = 0;
    a.neox = 0;
    a.head_dim = head_dim;
    a.k_bf16 = 0;
    a.v_bf16 = 0;
    return from_cuda(kvfp8::launch_reshape_and_cache(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvfp8_status kvfp8_rope_reshape_and_cache(
    const void *key, const void *value, kvfp8_dtype src_dtype, int64_t key_stride,
    int64_t value_stride, int64_t num_tokens, uint8_t *key_cache, uint8_t *value_cache,
    int32_t num_blocks, int32_t block_size, int32_t n_kv, int32_t head_dim,
    const int64_t *slot_mapping, const int64_t *positions, const float *cos_sin_cache,
    int64_t max_position, int32_t rot_dim, int32_t is_neox, const void *k_scale,
    const void *v_scale, kvfp8_dtype scale_dtype, uint32_t *status, kvfp8_stream_t stream) {
    if (!dtype_ok(src_dtype) || !dtype_ok(scale_dtype)) return KVFP8_ERR_DTYPE;
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || block_size > 1024 || n_kv < 1 ||
        max_position < 1)
        return KVFP8_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVFP8_ERR_SHAPE;
    if (rot_dim < 16 || rot_dim > head_dim || (rot_dim & (rot_dim - 1)) != 0) return KVFP8_ERR_SHAPE;
    const int64_t row = static_cast<int64_t>(n_kv) * head_dim;
    if (key_stride < row || value_stride < row) return KVFP8_ERR_SHAPE;
    if (row > 2048) return KVFP8_ERR_UNSUPPORTED;
    if (num_tokens == 0) return KVFP8_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping || !positions ||
        !cos_sin_cache)
        return KVFP8_ERR_NULL;
    const int64_t esz = src_dtype == KVFP8_F32 ? 4 : 2;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (key_stride * esz) % 16 != 0 || (value_stride * esz) % 16 != 0 ||
        !aligned(slot_mapping, 8) || !aligned(positions, 8) || !aligned16(cos_sin_cache))
        return KVFP8_ERR_ALIGN;
    kvfp8::ReshapeArgs a;
    a.key = key;
    a.value = value;
    a.src_dtype = src_dtype;
    a.key_stride = key_stride;
    a.value_stride = value_stride;
    a.num_tokens = num_tokens;
    a.key_cache = key_cache;
    a.value_cache = value_cache;
    a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
    a.row_elems = static_cast<int32_t>(row);
    a.slot_mapping = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.scale_dtype = scale_dtype;
    a.status = status;
    a.positions = positions;
    a.cos_sin = cos_sin_cache;
    a.max_pos = max_position;
    a.rot = rot_dim;
    a.neox = is_neox ? 1 : 0;
    a.head_dim = head_dim;
    a.k_bf16 = 0;
    a.v_bf16 = 0;
    return from_cuda(kvfp8::launch_reshape_and_cache(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t kvfp8_paged_decode_workspace_size(int32_t num_seqs, int32_t n_q, int32_t head_dim) {
    if (num_seqs < 0 || n_q < 1 || head_dim < 1) return 0;
    return kvfp8::decode_workspace_layout(num_seqs, n_q, head_dim).total;
}

kvfp8_status kvfp8_paged_decode_attention(void *out, const void *query, const uint8_t *key_cache,
                                          const uint8_t *value_cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                          int32_t num_seqs, int32_t n_q, int32_t n_kv,
                                          int32_t head_dim, int32_t block_size,
                                          int32_t num_blocks, float sm_scale,
                                          const void *k_scale, const void *v_scale,
                                          kvfp8_dtype scale_dtype, void *workspace,
                                          size_t workspace_bytes, uint32_t *status,
                                          kvfp8_stream_t stream) {
    bool nothing_to_do = false;
    const kvfp8_status v = kvfp8::validate_decode(
        out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
        n_q, n_kv, head_dim, block_size, num_blocks, sm_scale, scale_dtype, &nothing_to_do);
    if (v != KVFP8_OK || nothing_to_do) return v;
    if (!workspace) return KVFP8_ERR_NULL;
    if (!aligned16(workspace)) return KVFP8_ERR_ALIGN;
    if (workspace_bytes < kvfp8_paged_decode_workspace_size(num_seqs, n_q, head_dim))
        return KVFP8_ERR_WORKSPACE;
    return kvfp8::launch_decode_validated(out, query, key_cache, value_cache, block_tables,
                                          max_blocks_per_seq, seq_lens, num_seqs, n_q, n_kv,
                                          head_dim, block_size, num_blocks, sm_scale, k_scale,
                                          v_scale, scale_dtype, workspace, status, stream);
}

size_t kvfp8_paged_attention_multi_workspace_size(int32_t num_seqs, int32_t n_q, int32_t n_kv,
                                                  int32_t head_dim, int32_t max_query_len) {
    if (num_seqs < 0 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || head_dim < 1 || max_query_len < 1)
        return 0;
    if (!kvfp8::multi_uses_decode_kernel(n_q, n_kv, head_dim, max_query_len)) return 0;
    return kvfp8::decode_workspace_layout(num_seqs, n_q * max_query_len, head_dim).total;
}

kvfp8_status kvfp8_paged_attention_multi(
    void *out, const void *query, const int32_t *query_start_loc, int32_t num_query_rows,
    int32_t max_query_len, const uint8_t *key_cache, const uint8_t *value_cache, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
    int32_t n_kv, int32_t head_dim, int32_t block_size, int32_t num_blocks, float sm_scale,
    const void *k_scale, const void *v_scale, kvfp8_dtype scale_dtype, void *workspace,
    size_t workspace_bytes, uint32_t *status, kvfp8_stream_t stream) {
    if (!dtype_ok(scale_dtype)) return KVFP8_ERR_DTYPE;
    if (num_seqs < 0 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || max_query_len < 1 ||
        num_query_rows < 0 || num_blocks < 1 || max_blocks_per_seq < 1)
        return KVFP8_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVFP8_ERR_SHAPE;
    if (!block_size_ok_for_decode(block_size)) return KVFP8_ERR_SHAPE;
    const bool split_kv = kvfp8::multi_uses_decode_kernel(n_q, n_kv, head_dim, max_query_len);
    if (!split_kv && (n_q / n_kv > 128 ||
                      (static_cast<int64_t>(max_query_len) * (n_q / n_kv) + 127) / 128 * n_kv *
                              num_seqs > 0x7FFFFFFFLL))
        return KVFP8_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(num_blocks) * block_size > 0x7FFFFFFFLL ||
        static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
        return KVFP8_ERR_SHAPE;
    if (std::isnan(sm_scale) || std::isinf(sm_scale)) return KVFP8_ERR_SCALE;
    if (num_seqs == 0) return KVFP8_OK;
    if (!out || !query || !query_start_loc || !key_cache || !value_cache || !block_tables ||
        !seq_lens || (split_kv && !workspace))
        return KVFP8_ERR_NULL;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
        !aligned(query_start_loc, 4) || (split_kv && !aligned16(workspace)))
        return KVFP8_ERR_ALIGN;
    if (workspace_bytes <
        kvfp8_paged_attention_multi_workspace_size(num_seqs, n_q, n_kv, head_dim, max_query_len))
        return KVFP8_ERR_WORKSPACE;
    kvfp8::DecodeArgs d;
    d.out = out;
    d.query = query;
    d.key_cache = key_cache;
    d.value_cache = value_cache;
    d.block_tables = block_tables;
    d.max_blocks_per_seq = max_blocks_per_seq;
    d.seq_lens = seq_lens;
    d.num_seqs = num_seqs;
    d.n_q = n_q;
    d.n_kv = n_kv;
    d.head_dim = head_dim;
    d.block_size = block_size;
    d.num_blocks = num_blocks;
    d.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    d.k_scale = k_scale;
    d.v_scale = v_scale;
    d.scale_dtype = scale_dtype;
    d.workspace = workspace;
    d.status = status;
    d.qsl = query_start_loc;
    d.qmax = max_query_len;
    d.qrows = num_query_rows;
    d.k_bf16 = 0;
    d.v_bf16 = 0;
    return from_cuda(kvfp8::launch_paged_decode(d, reinterpret_cast<cudaStream_t>(stream)));
}

kvfp8_status kvfp8_reshape_and_cache_mixed(
    const void *key, const void *value, kvfp8_dtype src_dtype, int64_t key_stride,
    int64_t value_stride, int64_t num_tokens, void *key_cache, kvfp8_cache_dtype k_cache_dtype,
    void *value_cache, kvfp8_cache_dtype v_cache_dtype, int32_t num_blocks, int32_t block_size,
    int32_t n_kv, int32_t head_dim, const int64_t *slot_mapping, const void *k_scale,
    const void *v_scale, kvfp8_dtype scale_dtype, uint32_t *status, kvfp8_stream_t stream) {
    if (!dtype_ok(src_dtype) || !dtype_ok(scale_dtype) || !cache_dtype_ok(k_cache_dtype) ||
        !cache_dtype_ok(v_cache_dtype))
        return KVFP8_ERR_DTYPE;
    if (num_tokens < 0 || num_blocks < 1 || block_size < 1 || block_size > 1024 || n_kv < 1 ||
        head_dim < 1)
        return KVFP8_ERR_SHAPE;
    const int64_t row = static_cast<int64_t>(n_kv) * head_dim;
    if (row % 8 != 0 || key_stride < row || value_stride < row) return KVFP8_ERR_SHAPE;
    if (row > 2048) return KVFP8_ERR_UNSUPPORTED;
    if (num_tokens == 0) return KVFP8_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return KVFP8_ERR_NULL;
    const int64_t esz = src_dtype == KVFP8_F32 ? 4 : 2;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        (key_stride * esz) % 16 != 0 || (value_stride * esz) % 16 != 0 || !aligned(slot_mapping, 8))
        return KVFP8_ERR_ALIGN;
    kvfp8::ReshapeArgs a;
    a.key = key;
    a.value = value;
    a.src_dtype = src_dtype;
    a.key_stride = key_stride;
    a.value_stride = value_stride;
    a.num_tokens = num_tokens;
    a.key_cache = static_cast<uint8_t *>(key_cache);
    a.value_cache = static_cast<uint8_t *>(value_cache);
    a.num_slots = static_cast<int64_t>(num_blocks) * block_size;
    a.row_elems = static_cast<int32_t>(row);
    a.slot_mapping = slot_mapping;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.scale_dtype = scale_dtype;
    a.status = status;
    a.positions = nullptr;
    a.cos_sin = nullptr;
    a.max_pos = 0;
    a.rot = 0;
    a.neox = 0;
    a.head_dim = head_dim;
    a.k_bf16 = k_cache_dtype == KVFP8_CACHE_BF16 ? 1 : 0;
    a.v_bf16 = v_cache_dtype == KVFP8_CACHE_BF16 ? 1 : 0;
    return from_cuda(kvfp8::launch_reshape_and_cache(a, reinterpret_cast<cudaStream_t>(stream)));
}

kvfp8_status kvfp8_paged_decode_attention_mixed(
    void *out, const void *query, const void *key_cache, kvfp8_cache_dtype k_cache_dtype,
    const void *value_cache, kvfp8_cache_dtype v_cache_dtype, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
    int32_t n_kv, int32_t head_dim, int32_t block_size, int32_t num_blocks, float sm_scale,
    const void *k_scale, const void *v_scale, kvfp8_dtype scale_dtype, void *workspace,
    size_t workspace_bytes, uint32_t *status, kvfp8_stream_t stream) {
    if (!cache_dtype_ok(k_cache_dtype) || !cache_dtype_ok(v_cache_dtype)) return KVFP8_ERR_DTYPE;
    if (k_cache_dtype == KVFP8_CACHE_E4M3 && v_cache_dtype == KVFP8_CACHE_E4M3)
        return kvfp8_paged_decode_attention(
            out, query, static_cast<const uint8_t *>(key_cache),
            static_cast<const uint8_t *>(value_cache), block_tables, max_blocks_per_seq, seq_lens,
            num_seqs, n_q, n_kv, head_dim, block_size, num_blocks, sm_scale, k_scale, v_scale,
            scale_dtype, workspace, workspace_bytes, status, stream);
    if (!dtype_ok(scale_dtype)) return KVFP8_ERR_DTYPE;
    if (num_seqs < 0 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || num_blocks < 1 ||
        max_blocks_per_seq < 1)
        return KVFP8_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVFP8_ERR_SHAPE;
    if (!block_size_ok_for_decode(block_size)) return KVFP8_ERR_SHAPE;
    if (static_cast<int64_t>(num_blocks) * block_size > 0x7FFFFFFFLL ||
        static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
        return KVFP8_ERR_SHAPE;
    if (k_cache_dtype == v_cache_dtype ||
        !kvfp8::mixed_uses_decode_kernel(n_q, n_kv, head_dim, 1))
        return KVFP8_ERR_UNSUPPORTED;
    if (std::isnan(sm_scale) || std::isinf(sm_scale)) return KVFP8_ERR_SCALE;
    if (num_seqs == 0) return KVFP8_OK;
    if (!out || !query || !key_cache || !value_cache || !block_tables || !seq_lens || !workspace)
        return KVFP8_ERR_NULL;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
        !aligned16(workspace))
        return KVFP8_ERR_ALIGN;
    if (workspace_bytes < kvfp8_paged_decode_workspace_size(num_seqs, n_q, head_dim))
        return KVFP8_ERR_WORKSPACE;
    kvfp8::DecodeArgs d;
    d.out = out;
    d.query = query;
    d.key_cache = static_cast<const uint8_t *>(key_cache);
    d.value_cache = static_cast<const uint8_t *>(value_cache);
    d.block_tables = block_tables;
    d.max_blocks_per_seq = max_blocks_per_seq;
    d.seq_lens = seq_lens;
    d.num_seqs = num_seqs;
    d.n_q = n_q;
    d.n_kv = n_kv;
    d.head_dim = head_dim;
    d.block_size = block_size;
    d.num_blocks = num_blocks;
    d.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    d.k_scale = k_scale;
    d.v_scale = v_scale;
    d.scale_dtype = scale_dtype;
    d.workspace = workspace;
    d.status = status;
    d.qsl = nullptr;
    d.qmax = 1;
    d.qrows = num_seqs;
    d.k_bf16 = k_cache_dtype == KVFP8_CACHE_BF16 ? 1 : 0;
    d.v_bf16 = v_cache_dtype == KVFP8_CACHE_BF16 ? 1 : 0;
    return from_cuda(kvfp8::launch_paged_decode(d, reinterpret_cast<cudaStream_t>(stream)));
}

kvfp8_status kvfp8_paged_attention_multi_mixed(
    void *out, const void *query, const int32_t *query_start_loc, int32_t num_query_rows,
    int32_t max_query_len, const void *key_cache, kvfp8_cache_dtype k_cache_dtype,
    const void *value_cache, kvfp8_cache_dtype v_cache_dtype, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
    int32_t n_kv, int32_t head_dim, int32_t block_size, int32_t num_blocks, float sm_scale,
    const void *k_scale, const void *v_scale, kvfp8_dtype scale_dtype, void *workspace,
    size_t workspace_bytes, uint32_t *status, kvfp8_stream_t stream) {
    if (!cache_dtype_ok(k_cache_dtype) || !cache_dtype_ok(v_cache_dtype)) return KVFP8_ERR_DTYPE;
    if (k_cache_dtype == KVFP8_CACHE_E4M3 && v_cache_dtype == KVFP8_CACHE_E4M3)
        return kvfp8_paged_attention_multi(
            out, query, query_start_loc, num_query_rows, max_query_len,
            static_cast<const uint8_t *>(key_cache), static_cast<const uint8_t *>(value_cache),
            block_tables, max_blocks_per_seq, seq_lens, num_seqs, n_q, n_kv, head_dim, block_size,
            num_blocks, sm_scale, k_scale, v_scale, scale_dtype, workspace, workspace_bytes, status,
            stream);
    if (!dtype_ok(scale_dtype)) return KVFP8_ERR_DTYPE;
    if (num_seqs < 0 || n_q < 1 || n_kv < 1 || n_q % n_kv != 0 || max_query_len < 1 ||
        num_query_rows < 0 || num_blocks < 1 || max_blocks_per_seq < 1)
        return KVFP8_ERR_SHAPE;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return KVFP8_ERR_SHAPE;
    if (!block_size_ok_for_decode(block_size)) return KVFP8_ERR_SHAPE;
    if (static_cast<int64_t>(num_blocks) * block_size > 0x7FFFFFFFLL ||
        static_cast<int64_t>(max_blocks_per_seq) * block_size > 0x7FFFFFFFLL)
        return KVFP8_ERR_SHAPE;
    if (k_cache_dtype == v_cache_dtype ||
        !kvfp8::mixed_uses_decode_kernel(n_q, n_kv, head_dim, max_query_len))
        return KVFP8_ERR_UNSUPPORTED;
    if (std::isnan(sm_scale) || std::isinf(sm_scale)) return KVFP8_ERR_SCALE;
    if (num_seqs == 0) return KVFP8_OK;
    if (!out || !query || !query_start_loc || !key_cache || !value_cache || !block_tables ||
        !seq_lens || !workspace)
        return KVFP8_ERR_NULL;
    if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) ||
        !aligned16(value_cache) || !aligned(block_tables, 4) || !aligned(seq_lens, 4) ||
        !aligned(query_start_loc, 4) || !aligned16(workspace))
        return KVFP8_ERR_ALIGN;
    if (workspace_bytes <
        kvfp8_paged_attention_multi_workspace_size(num_seqs, n_q, n_kv, head_dim, max_query_len))
        return KVFP8_ERR_WORKSPACE;
    kvfp8::DecodeArgs d;
    d.out = out;
    d.query = query;
    d.key_cache = static_cast<const uint8_t *>(key_cache);
    d.value_cache = static_cast<const uint8_t *>(value_cache);
    d.block_tables = block_tables;
    d.max_blocks_per_seq = max_blocks_per_seq;
    d.seq_lens = seq_lens;
    d.num_seqs = num_seqs;
    d.n_q = n_q;
    d.n_kv = n_kv;
    d.head_dim = head_dim;
    d.block_size = block_size;
    d.num_blocks = num_blocks;
    d.sm_scale = sm_scale > 0.f ? sm_scale : 1.0f / std::sqrt(static_cast<float>(head_dim));
    d.k_scale = k_scale;
    d.v_scale = v_scale;
    d.scale_dtype = scale_dtype;
    d.workspace = workspace;
    d.status = status;
    d.qsl = query_start_loc;
    d.qmax = max_query_len;
    d.qrows = num_query_rows;
    d.k_bf16 = k_cache_dtype == KVFP8_CACHE_BF16 ? 1 : 0;
    d.v_bf16 = v_cache_dtype == KVFP8_CACHE_BF16 ? 1 : 0;
    return from_cuda(kvfp8::launch_paged_decode(d, reinterpret_cast<cudaStream_t>(stream)));
}

kvfp8_status kvfp8_dequant(void *dst, kvfp8_dtype dst_dtype, const uint8_t *src, int64_t n,
                           const void *scale, kvfp8_dtype scale_dtype, kvfp8_stream_t stream) {
    if (!dtype_ok(dst_dtype) || !dtype_ok(scale_dtype)) return KVFP8_ERR_DTYPE;
    if (n < 0) return KVFP8_ERR_SHAPE;
    if (n == 0) return KVFP8_OK;
    if (!dst || !src) return KVFP8_ERR_NULL;
    if (!aligned16(dst) || !aligned16(src)) return KVFP8_ERR_ALIGN;
    return from_cuda(kvfp8::launch_dequant(dst, dst_dtype, src, n, scale, scale_dtype,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

kvfp8_status kvfp8_check_scale_host(float s) {
    return (std::isfinite(s) && s != 0.0f) ? KVFP8_OK : KVFP8_ERR_SCALE;
}

const char *kvfp8_status_string(kvfp8_status s) {
    switch (s) {
        case KVFP8_OK: return "ok";
        case KVFP8_ERR_NULL: return "null pointer";
        case KVFP8_ERR_SHAPE: return "shape out of range";
        case KVFP8_ERR_DTYPE: return "unsupported dtype";
        case KVFP8_ERR_SCALE: return "scale must be finite and nonzero";
        case KVFP8_ERR_ALIGN: return "pointer or stride not 16-byte aligned";
        case KVFP8_ERR_WORKSPACE: return "workspace too small";
        case KVFP8_ERR_CUDA: return "CUDA error";
        case KVFP8_ERR_UNSUPPORTED: return "unsupported configuration";
    }
    return "unknown status";
}

}  // extern "C"
