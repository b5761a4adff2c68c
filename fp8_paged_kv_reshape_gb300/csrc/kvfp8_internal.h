// Internal launch interface between the C ABI (kvfp8_api.cu) and the kernels.
// Arguments arrive here already validated on the host.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cstdlib>
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <tuple>

#include "../../include/kvfp8.h"

namespace kvfp8 {

// A tuning knob read from the environment (launch shapes and kernel choices only).
inline int env_int(const char *name, int dflt) {
    const char *v = std::getenv(name);
    return v ? std::atoi(v) : dflt;
}

// ---------------------------------------------------------------- launch facts
// Device attributes and per-kernel occupancy do not change during a process, but querying
// them costs microseconds of host time per call; they are looked up once per device (and
// kernel, block size, shared memory) and kept.  A per-kernel dynamic shared memory limit is
// raised once per device, when a larger size is first needed.

struct DeviceFacts {
    int sms;         // multiprocessors
    int smem_optin;  // largest opt-in dynamic shared memory per block
};

inline cudaError_t device_facts(DeviceFacts *f) {
    static std::mutex mu;
    static std::map<int, DeviceFacts> cache;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(dev);
    if (it == cache.end()) {
        DeviceFacts d;
        if ((err = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) !=
            cudaSuccess)
            return err;
        if ((err = cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin,
                                          dev)) != cudaSuccess)
            return err;
        it = cache.emplace(dev, d).first;
    }
    *f = it->second;
    return cudaSuccess;
}

// Resident blocks per SM of `kernel` at `threads` per block and `smem` dynamic bytes, after
// making sure the kernel may use `smem` bytes of dynamic shared memory on this device.
template <typename K>
cudaError_t kernel_occupancy(K kernel, int threads, size_t smem, int *occ) {
    static std::mutex mu;
    static std::map<std::tuple<const void *, int, int, size_t>, int> occ_cache;
    static std::map<std::pair<const void *, int>, size_t> smem_set;
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const void *fn = reinterpret_cast<const void *>(kernel);
    std::lock_guard<std::mutex> lock(mu);
    auto key = std::make_tuple(fn, dev, threads, smem);
    auto it = occ_cache.find(key);
    if (it != occ_cache.end()) {
        *occ = it->second;
        return cudaSuccess;
    }
    if (smem > 48 * 1024) {
        size_t &cur = smem_set[std::make_pair(fn, dev)];
        if (smem > cur) {
            if ((err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                            static_cast<int>(smem))) != cudaSuccess)
                return err;
            cur = smem;
        }
    }
    int o = 0;
    if ((err = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, kernel, threads, smem)) !=
        cudaSuccess)
        return err;
    occ_cache.emplace(key, o);
    *occ = o;
    return cudaSuccess;
}

struct ReshapeArgs {
    const void *key;
    const void *value;
    int src_dtype;
    int64_t key_stride;    // elements
    int64_t value_stride;  // elements
    int64_t num_tokens;
    uint8_t *key_cache;
    uint8_t *value_cache;
    int64_t num_slots;     // num_blocks * block_size
    int32_t row_elems;     // n_kv * head_dim, multiple of 8
    const int64_t *slot_mapping;
    const void *k_scale;
    const void *v_scale;
    int scale_dtype;
    uint32_t *status;
    // rope on K before the store (kvfp8_rope_reshape_and_cache); cos_sin == nullptr: none
    const int64_t *positions;
    const float *cos_sin;  // [max_pos][rot]: cos half, then sin half
    int64_t max_pos;
    int32_t rot;
    int32_t neox;
    int32_t head_dim;
    // mixed cache dtypes: 1 = that side's cache is bf16 (unscaled), 0 = E4M3
    int32_t k_bf16;
    int32_t v_bf16;
};

cudaError_t launch_reshape_and_cache(const ReshapeArgs &a, cudaStream_t stream);

// Split-KV decode attention: work is cut into 16-token chunks, the chunks of all
// sequences are concatenated and every CTA of a fixed-size grid takes an equal
// contiguous range of them.
constexpr int kChunkTokens = 16;
constexpr int kMaxDecodeCtas = 1024;

struct DecodeArgs {
    void *out;
    const void *query;
    const uint8_t *key_cache;
    const uint8_t *value_cache;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t n_q;
    int32_t n_kv;
    int32_t head_dim;
    int32_t block_size;
    int32_t num_blocks;
    float sm_scale;  // > 0
    const void *k_scale;
    const void *v_scale;
    int scale_dtype;
    void *workspace;
    uint32_t *status;
    // multi-query (causal) form: sequence b's query rows start at qsl[b]; qmax is the
    // largest per-sequence query count.  Decode: qsl == nullptr, qmax == 1.
    const int32_t *qsl;
    int32_t qmax;
    int32_t qrows;  // rows of query and out
    // mixed cache dtypes: 1 = that side's cache is bf16 (2 bytes per element, no scale)
    int32_t k_bf16;
    int32_t v_bf16;
};

// Workspace layout, shared by the size query and the launcher; rows = query rows per
// sequence (n_q for decode, max query count * n_q for the multi-query form).
struct DecodeWorkspace {
    size_t cstart_off, cta_off, lse_off, o_off, total;
};
DecodeWorkspace decode_workspace_layout(int32_t num_seqs, int32_t rows, int32_t head_dim);

// Returns cudaErrorNotSupported for a shape without a kernel instance, or the first
// CUDA error met while encoding tensor maps / launching.
cudaError_t launch_paged_decode(const DecodeArgs &a, cudaStream_t stream);
// The mixed-dtype instances (exactly one of k_bf16 / v_bf16 set); called by the above.
cudaError_t launch_paged_decode_mixed(const DecodeArgs &a, cudaStream_t stream);
// True when the split-KV kernel has a mixed-dtype instance for this shape (up to 16 score
// columns per kv head, 8 at head_dim 256); the tensor-core kernel has none.
bool mixed_uses_decode_kernel(int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t max_query_len);

// Multi-query (causal) attention on the tensor cores (tcgen05): long query chunks, or kv-head
// counts the split-KV decode kernel does not cover.  Needs no workspace.
cudaError_t launch_prefill_attention(const DecodeArgs &a, cudaStream_t stream);
// True when kvfp8_paged_attention_multi takes the split-KV decode kernel for this shape
// (and so needs a workspace); false when it takes the prefill kernel.
bool multi_uses_decode_kernel(int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t max_query_len);

// Host validation of kvfp8_paged_decode_attention's arguments other than the workspace,
// in the order that call checks them; *nothing_to_do is set (with KVFP8_OK) for an empty
// batch.  Shared with the no-allocation entry point so both report the same errors.
kvfp8_status validate_decode(const void *out, const void *query, const uint8_t *key_cache,
                             const uint8_t *value_cache, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *seq_lens,
                             int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim,
                             int32_t block_size, int32_t num_blocks, float sm_scale,
                             int scale_dtype, bool *nothing_to_do);
// The decode launch for arguments validate_decode accepted, with a workspace of at least
// kvfp8_paged_decode_workspace_size bytes (16-byte aligned).
kvfp8_status launch_decode_validated(void *out, const void *query, const uint8_t *key_cache,
                                     const uint8_t *value_cache, const int32_t *block_tables,
                                     int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                     int32_t num_seqs, int32_t n_q, int32_t n_kv,
                                     int32_t head_dim, int32_t block_size, int32_t num_blocks,
                                     float sm_scale, const void *k_scale, const void *v_scale,
                                     int scale_dtype, void *workspace, uint32_t *status,
                                     kvfp8_stream_t stream);

cudaError_t launch_dequant(void *dst, int dst_dtype, const uint8_t *src, int64_t n,
                           const void *scale, int scale_dtype, cudaStream_t stream);

}  // namespace kvfp8
