// Paged decode attention with mixed cache dtypes: E4M3 on one side (K or V, scaled), bf16
// on the other (unscaled) -- llama.cpp "llama : Add FP8 KV-cache support (#28392)",
// tests/test-fp8.cpp check_fp8_attention, which quantizes K only, V only or both, and
// tests/test-backend-ops.cpp, which adds the F8/F16 mixes.  All-E4M3 calls go to
// paged_decode.cu.  Single-query decode and the multi-query (causal) form, both on the
// split-KV kernel: up to 16 score columns per kv head at head_dim 64 and 128, up to 8 at 256.
#include "paged_decode_kernel.cuh"

namespace kvfp8 {

namespace {

template <bool kMulti, bool KT16, bool VT16>
cudaError_t run_mixed(const DecodeArgs &d, const DecodeWorkspace &ws, int nt, cudaStream_t stream) {
    switch (d.head_dim) {
        case 64: return nt == 1 ? run<64, 1, kMulti, KT16, VT16>(d, ws, stream)
                                : run<64, 2, kMulti, KT16, VT16>(d, ws, stream);
        case 128: return nt == 1 ? run<128, 1, kMulti, KT16, VT16>(d, ws, stream)
                                 : run<128, 2, kMulti, KT16, VT16>(d, ws, stream);
        case 256: return nt == 1 ? run<256, 1, kMulti, KT16, VT16>(d, ws, stream)
                                 : cudaErrorNotSupported;
        default: return cudaErrorNotSupported;
    }
}

}  // namespace

bool mixed_uses_decode_kernel(int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t max_query_len) {
    const int64_t cols = static_cast<int64_t>(max_query_len) * (n_q / n_kv);
    return cols <= 16 && !(head_dim == 256 && cols > 8);
}

cudaError_t launch_paged_decode_mixed(const DecodeArgs &d, cudaStream_t stream) {
    if (d.num_seqs == 0) return cudaSuccess;
    if (d.k_bf16 == d.v_bf16) return cudaErrorNotSupported;
    if (!mixed_uses_decode_kernel(d.n_q, d.n_kv, d.head_dim, d.qmax)) return cudaErrorNotSupported;
    const DecodeWorkspace ws = decode_workspace_layout(d.num_seqs, d.qmax * d.n_q, d.head_dim);
    const int nt = d.qmax * (d.n_q / d.n_kv) <= 8 ? 1 : 2;
    const bool multi = d.qsl != nullptr;
    if (d.k_bf16)
        return multi ? run_mixed<true, true, false>(d, ws, nt, stream)
                     : run_mixed<false, true, false>(d, ws, nt, stream);
    return multi ? run_mixed<true, false, true>(d, ws, nt, stream)
                 : run_mixed<false, false, true>(d, ws, nt, stream);
}

}  // namespace kvfp8
