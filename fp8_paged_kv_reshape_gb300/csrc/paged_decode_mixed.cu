// Paged decode attention with mixed cache dtypes: E4M3 on one side (K or V, scaled), bf16
// on the other (unscaled) -- llama.cpp "llama : Add FP8 KV-cache support (#28392)",
// tests/test-fp8.cpp check_fp8_attention, which quantizes K only, V only or both, and
// tests/test-backend-ops.cpp, which adds the F8/F16 mixes.  All-E4M3 calls go to
// paged_decode.cu.  Single-query decode, head_dim 64 or 128, up to 16 heads per group.
#include "paged_decode_kernel.cuh"

namespace kvfp8 {

cudaError_t launch_paged_decode_mixed(const DecodeArgs &d, cudaStream_t stream) {
    if (d.num_seqs == 0) return cudaSuccess;
    if (d.qsl != nullptr || d.k_bf16 == d.v_bf16)
        return cudaErrorNotSupported;
    const int group = d.n_q / d.n_kv;
    if (group > 16) return cudaErrorNotSupported;
    const DecodeWorkspace ws = decode_workspace_layout(d.num_seqs, d.n_q, d.head_dim);
    const bool two = group > 8;
    if (d.k_bf16) {
        switch (d.head_dim) {
            case 64: return two ? run<64, 2, false, true, false>(d, ws, stream)
                                : run<64, 1, false, true, false>(d, ws, stream);
            case 128: return two ? run<128, 2, false, true, false>(d, ws, stream)
                                 : run<128, 1, false, true, false>(d, ws, stream);
            default: return cudaErrorNotSupported;
        }
    }
    switch (d.head_dim) {
        case 64: return two ? run<64, 2, false, false, true>(d, ws, stream)
                            : run<64, 1, false, false, true>(d, ws, stream);
        case 128: return two ? run<128, 2, false, false, true>(d, ws, stream)
                             : run<128, 1, false, false, true>(d, ws, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace kvfp8
