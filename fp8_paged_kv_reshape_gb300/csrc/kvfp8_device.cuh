// Device helpers shared by the kvfp8 kernels (sm_103a).
//
// E4M3 conversions use the hardware's packed converters:
//   cvt.rn.satfinite.e4m3x2.f32  two floats -> two E4M3 bytes, round to nearest even,
//                                finite values past 448 (and +-inf) clamp to +-448
//   cvt.rn.f16x2.e4m3x2          two E4M3 bytes -> two fp16 (exact: every E4M3 value
//                                is an fp16 value)
// which implement the codec of the osimons/ocp_fp8_kv branch of llama.cpp
// (ggml-impl.h ggml_fp32_to_f8_e4m3 / ggml_f8_e4m3_to_fp32) except for the sign of a
// NaN, which callers patch from the input bits.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "../../include/kvfp8.h"

namespace kvfp8 {

// Shared-memory address of a generic pointer into this CTA's shared memory.
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- status word

__device__ __forceinline__ void flag(uint32_t *status, uint32_t bit) {
    if (status != nullptr) atomicOr(status, bit);
}

// ---------------------------------------------------------------- scales

// A per-layer scalar scale: fp32, or bf16 widened exactly; a null pointer means 1.
__device__ __forceinline__ float load_scale(const void *p, int dtype) {
    if (p == nullptr) return 1.0f;
    if (dtype == KVFP8_BF16) {
        const uint16_t h = *reinterpret_cast<const uint16_t *>(p);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    return *reinterpret_cast<const float *>(p);
}

// finite and nonzero (negative allowed)
__device__ __forceinline__ bool scale_ok(float s) {
    return isfinite(s) && s != 0.0f;
}

// ---------------------------------------------------------------- E4M3

// Two floats -> two E4M3 bytes in a 16-bit value; lo lands in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 bytes (low 16 bits of v) -> fp16x2, low byte in the low half.
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t v) {
    uint32_t r;
    const uint16_t h = static_cast<uint16_t>(v & 0xFFFFu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

__device__ __forceinline__ uint32_t f16x2_from_e4m3x2_hi(uint32_t v) {
    uint32_t r;
    const uint16_t h = static_cast<uint16_t>(v >> 16);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

// Per-byte 0xFF mask of the bytes of w that are E4M3 NaN codes (0x7F or 0xFF).
__device__ __forceinline__ uint32_t nan_byte_mask(uint32_t w) {
    return __vcmpeq4(w & 0x7F7F7F7Fu, 0x7F7F7F7Fu);
}

// ---------------------------------------------------------------- bf16 / fp16

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t f16x2_from_f32(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

__device__ __forceinline__ uint32_t bf16x2_from_f32(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

}  // namespace kvfp8
