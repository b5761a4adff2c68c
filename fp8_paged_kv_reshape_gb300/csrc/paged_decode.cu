// Paged decode attention over the FP8 (E4M3) cache: the all-E4M3 kernel instances, the
// workspace layout and the dispatch on head_dim / query columns.  The kernels themselves
// are in paged_decode_kernel.cuh.
#include "paged_decode_kernel.cuh"

namespace kvfp8 {

DecodeWorkspace decode_workspace_layout(int32_t num_seqs, int32_t n_q, int32_t head_dim) {
    auto up = [](size_t x) { return (x + 255) & ~static_cast<size_t>(255); };
    const size_t parts = static_cast<size_t>(num_seqs) + kMaxDecodeCtas;
    DecodeWorkspace w;
    w.cstart_off = 0;
    w.cta_off = up(sizeof(int32_t) * (static_cast<size_t>(num_seqs) + 1));
    w.lse_off = w.cta_off + up(sizeof(CtaPlan) * kMaxDecodeCtas);
    w.o_off = w.lse_off + up(sizeof(float) * parts * n_q);
    w.total = w.o_off + up(sizeof(float) * parts * n_q * head_dim);
    return w;
}

bool multi_uses_decode_kernel(int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t max_query_len) {
    const int64_t cols = static_cast<int64_t>(max_query_len) * (n_q / n_kv);
    (void)n_kv;
    return cols <= 16 && !(head_dim == 256 && cols > 8);
}

cudaError_t launch_paged_decode(const DecodeArgs &d, cudaStream_t stream) {
    if (d.num_seqs == 0) return cudaSuccess;
    if (d.k_bf16 || d.v_bf16) return launch_paged_decode_mixed(d, stream);
    // score columns past the split-KV kernel's 16 per kv head (8 at head_dim 256): long query
    // chunks, or single-query groups of more heads, run on the tensor-core kernel
    if (!multi_uses_decode_kernel(d.n_q, d.n_kv, d.head_dim, d.qmax))
        return launch_prefill_attention(d, stream);
    const DecodeWorkspace ws = decode_workspace_layout(d.num_seqs, d.qmax * d.n_q, d.head_dim);
    const int group = d.n_q / d.n_kv;
    const int cols = d.qmax * group;  // score columns per kv head
    if (cols > 16) return cudaErrorNotSupported;
    const int nt = cols <= 8 ? 1 : 2;
    if (d.qsl == nullptr) {
        switch (d.head_dim) {
            case 64: return nt == 1 ? run<64, 1, false, false, false>(d, ws, stream) : run<64, 2, false, false, false>(d, ws, stream);
            case 128: return nt == 1 ? run<128, 1, false, false, false>(d, ws, stream) : run<128, 2, false, false, false>(d, ws, stream);
            case 256: return nt == 1 ? run<256, 1, false, false, false>(d, ws, stream) : cudaErrorNotSupported;
            default: return cudaErrorNotSupported;
        }
    }
    switch (d.head_dim) {
        case 64: return nt == 1 ? run<64, 1, true, false, false>(d, ws, stream) : run<64, 2, true, false, false>(d, ws, stream);
        case 128: return nt == 1 ? run<128, 1, true, false, false>(d, ws, stream) : run<128, 2, true, false, false>(d, ws, stream);
        case 256: return nt == 1 ? run<256, 1, true, false, false>(d, ws, stream) : cudaErrorNotSupported;
        default: return cudaErrorNotSupported;
    }
}

}  // namespace kvfp8
