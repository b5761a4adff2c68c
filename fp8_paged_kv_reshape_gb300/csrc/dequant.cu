// E4M3 bytes -> scale * value (fp32 or bf16), sm_103a.
//
// The rope-shift path of llama.cpp "llama : Add FP8 KV-cache support (#28392)"
// (llama-kv-cache.cpp build_rope_shift) dequantizes the F8 cache, rotates it and
// requantizes; tests/test-fp8.cpp check_fp8_context_shift holds the result to
// quantize(rope(decode(bytes))) byte for byte.  This kernel is the decode half.
//
// Streaming: each thread converts 16 bytes per step (one 16-byte load, eight packed
// e4m3x2 -> f16x2 converts, exact widening to fp32, one fp32 multiply per element).
#include <cuda_runtime.h>

#include "kvfp8_device.cuh"
#include "kvfp8_internal.h"

namespace kvfp8 {
namespace {

__device__ __forceinline__ float2 f32x2_from_f16x2(uint32_t h) {
    const __half2 v = *reinterpret_cast<const __half2 *>(&h);
    return __half22float2(v);
}

template <bool kBF16Out>
__global__ void __launch_bounds__(256)
dequant_kernel(void *dst, const uint8_t *src, int64_t n, const void *scale, int scale_dtype) {
    const float s = load_scale(scale, scale_dtype);
    const bool has_scale = scale != nullptr;
    const int64_t nvec = n >> 4;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * blockDim.x;
    for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < nvec;
         i += stride) {
        const uint4 v = __ldcs(reinterpret_cast<const uint4 *>(src) + i);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        float f[16];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float2 lo = f32x2_from_f16x2(f16x2_from_e4m3x2(w[k]));
            const float2 hi = f32x2_from_f16x2(f16x2_from_e4m3x2_hi(w[k]));
            f[4 * k + 0] = lo.x;
            f[4 * k + 1] = lo.y;
            f[4 * k + 2] = hi.x;
            f[4 * k + 3] = hi.y;
        }
        if (has_scale) {
#pragma unroll
            for (int k = 0; k < 16; ++k) f[k] = __fmul_rn(s, f[k]);
        }
        if (kBF16Out) {
            uint4 o0, o1;
            o0.x = bf16x2_from_f32(f[0], f[1]);
            o0.y = bf16x2_from_f32(f[2], f[3]);
            o0.z = bf16x2_from_f32(f[4], f[5]);
            o0.w = bf16x2_from_f32(f[6], f[7]);
            o1.x = bf16x2_from_f32(f[8], f[9]);
            o1.y = bf16x2_from_f32(f[10], f[11]);
            o1.z = bf16x2_from_f32(f[12], f[13]);
            o1.w = bf16x2_from_f32(f[14], f[15]);
            uint4 *d = reinterpret_cast<uint4 *>(dst) + 2 * i;
            d[0] = o0;
            d[1] = o1;
        } else {
            float4 *d = reinterpret_cast<float4 *>(dst) + 4 * i;
#pragma unroll
            for (int k = 0; k < 4; ++k)
                d[k] = make_float4(f[4 * k], f[4 * k + 1], f[4 * k + 2], f[4 * k + 3]);
        }
    }
    // ragged tail (< 16 bytes), one element per thread of the first block
    if (blockIdx.x == 0 && threadIdx.x < (n & 15)) {
        const int64_t j = (nvec << 4) + threadIdx.x;
        float x = __half2float(__ushort_as_half(
            static_cast<uint16_t>(f16x2_from_e4m3x2(static_cast<uint32_t>(src[j])) & 0xFFFFu)));
        if (has_scale) x = __fmul_rn(s, x);
        if (kBF16Out)
            reinterpret_cast<uint16_t *>(dst)[j] = static_cast<uint16_t>(bf16x2_from_f32(x, 0.f) & 0xFFFFu);
        else
            reinterpret_cast<float *>(dst)[j] = x;
    }
}

}  // namespace

cudaError_t launch_dequant(void *dst, int dst_dtype, const uint8_t *src, int64_t n,
                           const void *scale, int scale_dtype, cudaStream_t stream) {
    if (n == 0) return cudaSuccess;
    DeviceFacts f;
    cudaError_t err = device_facts(&f);
    if (err != cudaSuccess) return err;
    const int sms = f.sms;
    const int64_t nvec = (n >> 4) > 0 ? (n >> 4) : 1;
    const int64_t want = (nvec + 255) / 256;
    const int blocks = static_cast<int>(want < 8LL * sms ? want : 8LL * sms);
    if (dst_dtype == KVFP8_BF16)
        dequant_kernel<true><<<blocks, 256, 0, stream>>>(dst, src, n, scale, scale_dtype);
    else
        dequant_kernel<false><<<blocks, 256, 0, stream>>>(dst, src, n, scale, scale_dtype);
    return cudaGetLastError();
}

}  // namespace kvfp8
