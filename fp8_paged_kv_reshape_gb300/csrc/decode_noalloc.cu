// kvfp8_paged_decode_attention_noalloc: paged decode attention for callers that cannot
// allocate device memory (a plug-in whose host runtime owns every device allocation, a
// serving loop that must not allocate once it is running, a caller with no allocator of
// its own).  It is kvfp8_paged_decode_attention with the split-KV scratch placed in a
// file-scope device array of KVFP8_NOALLOC_SCRATCH_BYTES instead of a caller workspace.
//
// The array is part of this library's device image: every GPU that loads the library
// holds it until the process exits.  Host code must not hand the array's name to a
// kernel (on the host it is only a stand-in for the symbol); its device address is looked
// up once per device with cudaGetSymbolAddress, with that device current, on the first
// call made on that device, so make that first call before any stream capture.  All
// calls share the array and it keeps the last call's contents; nothing in it needs to
// start at zero (each call writes every scratch byte it later reads), but calls that
// overlap on the GPU race on it.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/kvfp8.h"
#include "kvfp8_internal.h"

namespace {

constexpr size_t kScratchBytes = KVFP8_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) uint8_t g_decode_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_decode_scratch, per device

// The scratch array's device address on the current device (looked up once per device).
cudaError_t scratch_address(void **addr) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_decode_scratch);
        if (err != cudaSuccess) return err;
        g_scratch_addr[dev] = p;
    }
    *addr = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" kvfp8_status kvfp8_paged_decode_attention_noalloc(
    void *out, const void *query, const uint8_t *key_cache, const uint8_t *value_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
    int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float sm_scale, const void *k_scale, const void *v_scale,
    kvfp8_dtype scale_dtype, uint32_t *status, kvfp8_stream_t stream) {
    // The same argument checks, in the same order, as the workspace entry point: a call it
    // would reject is rejected here with the same code, before the scratch is looked at.
    bool nothing_to_do = false;
    const kvfp8_status v = kvfp8::validate_decode(
        out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
        n_q, n_kv, head_dim, block_size, num_blocks, sm_scale, scale_dtype, &nothing_to_do);
    if (v != KVFP8_OK || nothing_to_do) return v;
    // A batch whose scratch would not fit the fixed array is refused before anything runs.
    if (kvfp8_paged_decode_workspace_size(num_seqs, n_q, head_dim) > kScratchBytes)
        return KVFP8_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (scratch_address(&scratch) != cudaSuccess) return KVFP8_ERR_CUDA;
    return kvfp8::launch_decode_validated(out, query, key_cache, value_cache, block_tables,
                                          max_blocks_per_seq, seq_lens, num_seqs, n_q, n_kv,
                                          head_dim, block_size, num_blocks, sm_scale, k_scale,
                                          v_scale, scale_dtype, scratch, status, stream);
}
