// reshape_and_cache for an FP8 (E4M3) paged KV cache, sm_103a.
//
// What it computes (llama.cpp "llama : Add FP8 KV-cache support (#28392)",
// llama-graph.cpp build_attn_scale_kv_inputs + llama-kv-cache.cpp cpy_k/cpy_v):
// every element of every non-padding token row is divided by the layer's scalar scale
// (IEEE float quotient), rounded to E4M3 (nearest even, saturating at +-448), and the
// row's n_kv*head_dim bytes land at slot * n_kv*head_dim in the cache.
//
// Design: HBM-streaming.  One warp owns one (token, K|V) row; a lane moves 8 elements
// per 16-byte load (bf16) and issues all of its loads for the row before converting,
// so a 1 KiB-row warp keeps 2 KiB of reads in flight.  Loads are streaming (evict
// first: every input byte is read once); each lane writes 8 contiguous output bytes so
// a warp's stores cover whole 256-byte spans of the destination row.  Per element the
// work is one unpack, one correctly rounded divide (__fdiv_rn) and half a packed
// convert; a NaN check on the packed bytes sends the rare NaN/inf words to a slow path
// that sets the sign the way the CPU reference does.
#include <cuda_runtime.h>

#include "kvfp8_device.cuh"
#include "kvfp8_internal.h"

namespace kvfp8 {
namespace {

constexpr int kWarps = 8;    // rows per CTA
constexpr int kUnroll = 4;   // 8-element groups per lane kept in flight

// Re-derive one byte of a word whose packed code came out as a NaN code: a NaN element
// keeps its own sign (sign(x)|0x7F); an infinite quotient saturates (sign(q)|0x7E).
__device__ __forceinline__ uint32_t fix_byte(uint32_t w, uint32_t nanmask, int i, float x, float q) {
    if (((nanmask >> (8 * i)) & 0xFFu) == 0u) return w;
    const uint32_t code = isnan(x) ? ((signbit(x) ? 0x80u : 0u) | 0x7Fu)
                                   : ((signbit(q) ? 0x80u : 0u) | 0x7Eu);
    return (w & ~(0xFFu << (8 * i))) | (code << (8 * i));
}

__device__ __noinline__ uint32_t patch_word(uint32_t w, uint32_t nanmask, float x0, float x1,
                                            float x2, float x3, float q0, float q1, float q2,
                                            float q3) {
    w = fix_byte(w, nanmask, 0, x0, q0);
    w = fix_byte(w, nanmask, 1, x1, q1);
    w = fix_byte(w, nanmask, 2, x2, q2);
    return fix_byte(w, nanmask, 3, x3, q3);
}

// Eight floats -> eight E4M3 bytes (x[0] in the lowest byte), divided by s.
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], float s) {
    float q[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(x[i], s);
    uint32_t w0 = e4m3x2_from_f32(q[0], q[1]) | (e4m3x2_from_f32(q[2], q[3]) << 16);
    uint32_t w1 = e4m3x2_from_f32(q[4], q[5]) | (e4m3x2_from_f32(q[6], q[7]) << 16);
    const uint32_t m0 = nan_byte_mask(w0);
    const uint32_t m1 = nan_byte_mask(w1);
    if (__builtin_expect((m0 | m1) != 0u, 0)) {
        if (m0) w0 = patch_word(w0, m0, x[0], x[1], x[2], x[3], q[0], q[1], q[2], q[3]);
        if (m1) w1 = patch_word(w1, m1, x[4], x[5], x[6], x[7], q[4], q[5], q[6], q[7]);
    }
    return make_uint2(w0, w1);
}

template <bool kF32>
struct Group;  // one 8-element group of a source row

template <>
struct Group<false> {  // bf16: 16 bytes
    uint4 v;
    __device__ __forceinline__ void load(const uint8_t *p) {
        v = __ldcs(reinterpret_cast<const uint4 *>(p));
    }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
        x[4] = bf16lo(v.z); x[5] = bf16hi(v.z); x[6] = bf16lo(v.w); x[7] = bf16hi(v.w);
    }
    static constexpr int kBytes = 16;
};

template <>
struct Group<true> {  // fp32: 32 bytes
    float4 a, b;
    __device__ __forceinline__ void load(const uint8_t *p) {
        a = __ldcs(reinterpret_cast<const float4 *>(p));
        b = __ldcs(reinterpret_cast<const float4 *>(p) + 1);
    }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    static constexpr int kBytes = 32;
};

template <bool kF32>
__global__ void __launch_bounds__(kWarps * 32)
reshape_and_cache_kernel(const ReshapeArgs a) {
    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t row = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    if (row >= 2 * a.num_tokens) return;
    const int64_t tok = row >> 1;
    const bool is_v = (row & 1) != 0;

    const int64_t slot = __ldg(a.slot_mapping + tok);
    if (slot == -1) return;  // padding token
    if (slot < 0 || slot >= a.num_slots) {
        if (lane == 0 && !is_v) flag(a.status, KVFP8_DEV_BAD_SLOT);
        return;
    }
    const float s = is_v ? sv : sk;
    const int64_t stride = is_v ? a.value_stride : a.key_stride;
    const uint8_t *src = static_cast<const uint8_t *>(is_v ? a.value : a.key) +
                         tok * stride * (kF32 ? 4 : 2);
    uint8_t *dst = (is_v ? a.value_cache : a.key_cache) + slot * a.row_elems;
    const int groups = a.row_elems >> 3;

    for (int g0 = lane; g0 < groups; g0 += 32 * kUnroll) {
        Group<kF32> in[kUnroll];
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int g = g0 + 32 * u;
            if (g < groups) in[u].load(src + static_cast<int64_t>(g) * Group<kF32>::kBytes);
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int g = g0 + 32 * u;
            if (g < groups) {
                float x[8];
                in[u].unpack(x);
                *reinterpret_cast<uint2 *>(dst + static_cast<int64_t>(g) * 8) = quantize8(x, s);
            }
        }
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ReshapeArgs &a, cudaStream_t stream) {
    if (a.num_tokens == 0) return cudaSuccess;
    const int64_t rows = 2 * a.num_tokens;
    const int64_t blocks = (rows + kWarps - 1) / kWarps;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(blocks)), block(kWarps * 32);
    if (a.src_dtype == KVFP8_F32)
        reshape_and_cache_kernel<true><<<grid, block, 0, stream>>>(a);
    else
        reshape_and_cache_kernel<false><<<grid, block, 0, stream>>>(a);
    return cudaGetLastError();
}

}  // namespace kvfp8
