// reshape_and_cache for an FP8 (E4M3) paged KV cache, sm_103a.
//
// What it computes (llama.cpp "llama : Add FP8 KV-cache support (#28392)",
// llama-graph.cpp build_attn_scale_kv_inputs + llama-kv-cache.cpp cpy_k/cpy_v):
// every element of every non-padding token row is divided by the layer's scalar scale
// (IEEE float quotient), rounded to E4M3 (nearest even, saturating at +-448), and the
// row's n_kv*head_dim bytes land at slot * n_kv*head_dim in the cache.
//
// Design: HBM-streaming with few instructions per element.
//  * Persistent warps.  A warp owns every (gridDim*8)-th row of the (token, K|V) row
//    sequence, so it always handles K rows or always V rows (one scale per warp), and
//    keeps two rows in registers: while it converts and stores one, the 16-byte
//    streaming loads of the next are in flight; slot indices are fetched two rows ahead.
//  * Division.  The quotient must be the IEEE float quotient x/s (correctly rounded).
//    With y = RN(1/|s|) computed once per thread, q0 = RN(x*y) is within two ulps;
//    one residual step q1 = q0 + (x - q0*|s|)*y (fused multiply-adds) makes it faithful
//    and a second step gives RN(x/|s|) by Markstein's theorem (y within half an ulp of
//    1/|s|, q1 faithful, exact FMA residual; see Markstein, "Computation of elementary
//    functions on the IBM RISC System/6000 processor", IBM J. R&D 34(1), 1990).  The
//    theorem's range conditions hold whenever 2^-60 <= |s| <= 2^60 and the quotient
//    decides the byte; other scales take __fdiv_rn.  Signs are set from the operands
//    (zeros included), and the few words whose packed codes come out as NaN (a NaN
//    element, an infinite element, or a quotient so large that the steps overflow) get
//    their bytes re-derived from the operands.
//  * Rows of more than 2048 elements take a plain per-row loop.
//  * Wide rows.  Rows of 512-2048 elements with 32-byte aligned sources are read 16
//    elements per lane (one 32-byte load for bf16) and stored as one 16-byte code store.
//  * L2 placement.  Source loads skip L1; cache stores carry an evict-first L2 policy so
//    that the written lines reach HBM while this kernel runs rather than after it.
#include <cuda_runtime.h>

#include <algorithm>

#include "kvfp8_device.cuh"
#include "kvfp8_internal.h"

namespace kvfp8 {
namespace {

constexpr int kWarps = 8;  // per CTA

// Packed fp32 pairs: the f32x2 arithmetic of sm_100+ does two IEEE round-to-nearest
// operations (no flush to zero) per instruction, halving the issue cost of the divide and
// of the rope rotation.  Lane 0 of a pair is the low half.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void unpack2(uint64_t v, float &lo, float &hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ uint64_t mul2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t sub2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// The reciprocal-and-corrections divide of the header note, for |s| in [2^-60, 2^60].
struct FastDiv {
    float sa;    // |s|
    float y;     // RN(1 / |s|)
    uint32_t neg;  // 0x80808080 when s < 0 (the byte signs are flipped after packing)
    uint64_t y2, nsa2;  // (y, y) and (-|s|, -|s|) for the packed form
    __device__ __forceinline__ explicit FastDiv(float s) {
        sa = fabsf(s);
        y = __fdiv_rn(1.0f, sa);  // correctly rounded reciprocal
        neg = signbit(s) ? 0x80808080u : 0u;
        y2 = pack2(y, y);
        nsa2 = pack2(-sa, -sa);
    }
    // RN(x / |s|) for a pair: q0 = x*y, then two residual steps q += fma(q, -|s|, x) * y,
    // each operation on both lanes (fma(q, -|s|, x) equals fma(-q, |s|, x): negation is
    // exact).  The sign is that of x except for x = -0, where the residual sums give +0;
    // the caller ORs the sign bits of x into the codes.
    __device__ __forceinline__ void quot2(float x0, float x1, float &r0, float &r1) const {
        const uint64_t x = pack2(x0, x1);
        const uint64_t q0 = mul2(x, y2);
        const uint64_t e0 = fma2(q0, nsa2, x);
        const uint64_t q1 = fma2(e0, y2, q0);
        const uint64_t e1 = fma2(q1, nsa2, x);
        unpack2(fma2(e1, y2, q1), r0, r1);
    }
};

__device__ __forceinline__ uint32_t fix_byte(uint32_t w, uint32_t nanmask, int i, float x,
                                             bool s_neg) {
    if (((nanmask >> (8 * i)) & 0xFFu) == 0u) return w;
    // a NaN element keeps its own sign; anything else that produced a NaN code is a
    // quotient out of range, which saturates with the quotient's sign
    const uint32_t code = isnan(x) ? ((signbit(x) ? 0x80u : 0u) | 0x7Fu)
                                   : (((signbit(x) != s_neg) ? 0x80u : 0u) | 0x7Eu);
    return (w & ~(0xFFu << (8 * i))) | (code << (8 * i));
}

__device__ __noinline__ uint32_t patch_word(uint32_t w, uint32_t nanmask, float x0, float x1,
                                            float x2, float x3, bool s_neg) {
    w = fix_byte(w, nanmask, 0, x0, s_neg);
    w = fix_byte(w, nanmask, 1, x1, s_neg);
    w = fix_byte(w, nanmask, 2, x2, s_neg);
    return fix_byte(w, nanmask, 3, x3, s_neg);
}

// The sign bits of eight floats at bit 7 of the bytes of two words (element i in byte i % 4
// of word i / 4); the other bits are left over and masked by the caller.
__device__ __forceinline__ uint2 sign_bytes(const float (&x)[8]) {
    auto w = [&](int i) { return __float_as_uint(x[i]); };
    const uint32_t a = __byte_perm(w(0), w(1), 0x0073), b = __byte_perm(w(2), w(3), 0x0073);
    const uint32_t c = __byte_perm(w(4), w(5), 0x0073), d = __byte_perm(w(6), w(7), 0x0073);
    return make_uint2(__byte_perm(a, b, 0x5410), __byte_perm(c, d, 0x5410));
}
// the same for eight bf16 values in four words (the high byte of each)
__device__ __forceinline__ uint2 sign_bytes_bf16(uint32_t w0, uint32_t w1, uint32_t w2, uint32_t w3) {
    return make_uint2(__byte_perm(w0, w1, 0x7531), __byte_perm(w2, w3, 0x7531));
}

// Eight floats -> eight E4M3 bytes (x[0] in the lowest byte): E4M3(x / s).  sgn: the sign
// bits of x as sign_bytes gives them (used by the fast divide only).
template <bool kFast>
__device__ __forceinline__ uint2 quantize8(const float (&x)[8], float s, const FastDiv &fd, uint2 sgn) {
    float q[8];
    if (kFast) {
#pragma unroll
        for (int i = 0; i < 8; i += 2) fd.quot2(x[i], x[i + 1], q[i], q[i + 1]);
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) q[i] = __fdiv_rn(x[i], s);
    }
    uint32_t w0 = e4m3x2_from_f32(q[0], q[1]) | (e4m3x2_from_f32(q[2], q[3]) << 16);
    uint32_t w1 = e4m3x2_from_f32(q[4], q[5]) | (e4m3x2_from_f32(q[6], q[7]) << 16);
    if (kFast) {  // sign(x) (which a zero quotient may have lost), then sign(s)
        w0 = (w0 | (sgn.x & 0x80808080u)) ^ fd.neg;
        w1 = (w1 | (sgn.y & 0x80808080u)) ^ fd.neg;
    }
    // any NaN code (a byte whose low seven bits are all set)?  Adding 1 to each byte of the
    // low-seven-bit part carries into bit 7 exactly there, and never into the next byte.
    const uint32_t t0 = (w0 & 0x7F7F7F7Fu) + 0x01010101u, t1 = (w1 & 0x7F7F7F7Fu) + 0x01010101u;
    if (__builtin_expect(((t0 | t1) & 0x80808080u) != 0u, 0)) {
        const uint32_t m0 = nan_byte_mask(w0);
        const uint32_t m1 = nan_byte_mask(w1);
        const bool s_neg = signbit(s);
        if (m0) w0 = patch_word(w0, m0, x[0], x[1], x[2], x[3], s_neg);
        if (m1) w1 = patch_word(w1, m1, x[4], x[5], x[6], x[7], s_neg);
    }
    return make_uint2(w0, w1);
}

// Cache placement of the streams.  Source rows are read once: loads skip L1 and keep the
// normal L2 priority.  Cache rows are written once: stores carry an L2 evict-first policy, so
// the written lines are the first the L2 writes back, while this kernel runs, instead of
// staying dirty in L2 after it ends (where the next kernel would pay for their write-back).
__device__ __forceinline__ uint4 ld_na_v4(const uint8_t *p) {
    uint4 v;
    asm volatile("ld.global.L1::no_allocate.v4.b32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}
__device__ __forceinline__ uint64_t evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ void st_ef(uint8_t *p, uint2 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v2.b32 [%0], {%1,%2}, %3;" ::"l"(p), "r"(v.x), "r"(v.y),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void st_ef(uint8_t *p, uint4 v, uint64_t pol) {
    asm volatile("st.global.L2::cache_hint.v4.b32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(pol)
                 : "memory");
}

template <bool kF32>
struct Group;  // one 8-element group of a source row

template <>
struct Group<false> {  // bf16: 16 bytes
    uint4 v;
    __device__ __forceinline__ void load(const uint8_t *p) { v = ld_na_v4(p); }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = bf16lo(v.x); x[1] = bf16hi(v.x); x[2] = bf16lo(v.y); x[3] = bf16hi(v.y);
        x[4] = bf16lo(v.z); x[5] = bf16hi(v.z); x[6] = bf16lo(v.w); x[7] = bf16hi(v.w);
    }
    // the same group of lane ^ m (packed: four shuffles for eight values)
    __device__ __forceinline__ Group xor_lane(int m) const {
        Group g;
        g.v.x = __shfl_xor_sync(0xFFFFFFFFu, v.x, m);
        g.v.y = __shfl_xor_sync(0xFFFFFFFFu, v.y, m);
        g.v.z = __shfl_xor_sync(0xFFFFFFFFu, v.z, m);
        g.v.w = __shfl_xor_sync(0xFFFFFFFFu, v.w, m);
        return g;
    }
    // the elements as bf16 pairs (a bf16 source is copied unchanged)
    __device__ __forceinline__ void bf16_words(uint32_t (&o)[4]) const {
        o[0] = v.x; o[1] = v.y; o[2] = v.z; o[3] = v.w;
    }
    __device__ __forceinline__ uint2 signs8(int) const { return sign_bytes_bf16(v.x, v.y, v.z, v.w); }
    static constexpr int kElems = 8;
    static constexpr int kBytes = 16;
};

template <>
struct Group<true> {  // fp32: 32 bytes
    float4 a, b;
    __device__ __forceinline__ void load(const uint8_t *p) {
        const uint4 x = ld_na_v4(p), y = ld_na_v4(p + 16);
        a = make_float4(__uint_as_float(x.x), __uint_as_float(x.y), __uint_as_float(x.z),
                        __uint_as_float(x.w));
        b = make_float4(__uint_as_float(y.x), __uint_as_float(y.y), __uint_as_float(y.z),
                        __uint_as_float(y.w));
    }
    __device__ __forceinline__ void unpack(float (&x)[8]) const {
        x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
        x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
    }
    __device__ __forceinline__ Group xor_lane(int m) const {
        Group g;
        g.a = make_float4(__shfl_xor_sync(0xFFFFFFFFu, a.x, m), __shfl_xor_sync(0xFFFFFFFFu, a.y, m),
                          __shfl_xor_sync(0xFFFFFFFFu, a.z, m), __shfl_xor_sync(0xFFFFFFFFu, a.w, m));
        g.b = make_float4(__shfl_xor_sync(0xFFFFFFFFu, b.x, m), __shfl_xor_sync(0xFFFFFFFFu, b.y, m),
                          __shfl_xor_sync(0xFFFFFFFFu, b.z, m), __shfl_xor_sync(0xFFFFFFFFu, b.w, m));
        return g;
    }
    // the elements rounded to bf16 pairs (nearest even)
    __device__ __forceinline__ void bf16_words(uint32_t (&o)[4]) const {
        o[0] = bf16x2_from_f32(a.x, a.y); o[1] = bf16x2_from_f32(a.z, a.w);
        o[2] = bf16x2_from_f32(b.x, b.y); o[3] = bf16x2_from_f32(b.z, b.w);
    }
    __device__ __forceinline__ uint2 signs8(int) const {
        const float x[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
        return sign_bytes(x);
    }
    static constexpr int kElems = 8;
    static constexpr int kBytes = 32;
};

// 32-byte load (sm_100+): eight words in one instruction; p 32-byte aligned.
__device__ __forceinline__ void ld_na_v8(const uint8_t *p, uint32_t *w) {
    asm volatile("ld.global.L1::no_allocate.v8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]), "=r"(w[4]), "=r"(w[5]),
                   "=r"(w[6]), "=r"(w[7])
                 : "l"(p));
}

// Sixteen consecutive elements of a source row for the wide path: one 32-byte load (bf16)
// or two (fp32) per lane, and 16 output bytes per lane, stored with one 16-byte store.
// Rows and their start must be 32-byte aligned.
template <bool kF32>
struct Wide;

template <>
struct Wide<false> {  // bf16: 32 bytes
    uint32_t w[8];
    __device__ __forceinline__ void load(const uint8_t *p) { ld_na_v8(p, w); }
    __device__ __forceinline__ void unpack(float (&x)[16]) const {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            x[2 * i] = bf16lo(w[i]);
            x[2 * i + 1] = bf16hi(w[i]);
        }
    }
    __device__ __forceinline__ void bf16_words(uint32_t (&o)[8]) const {
#pragma unroll
        for (int i = 0; i < 8; ++i) o[i] = w[i];
    }
    // sign bytes of elements 8h .. 8h+7
    __device__ __forceinline__ uint2 signs8(int h) const {
        return sign_bytes_bf16(w[4 * h], w[4 * h + 1], w[4 * h + 2], w[4 * h + 3]);
    }
    static constexpr int kElems = 16;
    static constexpr int kBytes = 32;
};

template <>
struct Wide<true> {  // fp32: 64 bytes
    uint32_t w[16];
    __device__ __forceinline__ void load(const uint8_t *p) {
        ld_na_v8(p, w);
        ld_na_v8(p + 32, w + 8);
    }
    __device__ __forceinline__ void unpack(float (&x)[16]) const {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = __uint_as_float(w[i]);
    }
    __device__ __forceinline__ void bf16_words(uint32_t (&o)[8]) const {
#pragma unroll
        for (int i = 0; i < 8; ++i)
            o[i] = bf16x2_from_f32(__uint_as_float(w[2 * i]), __uint_as_float(w[2 * i + 1]));
    }
    __device__ __forceinline__ uint2 signs8(int h) const {
        float x[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) x[i] = __uint_as_float(w[8 * h + i]);
        return sign_bytes(x);
    }
    static constexpr int kElems = 16;
    static constexpr int kBytes = 64;
};

struct RowCtx {
    const uint8_t *src;  // K or V base
    uint8_t *cache;
    int64_t stride_bytes;
    float s;
    uint64_t pol;  // L2 policy of the cache stores
};

__device__ __forceinline__ int64_t slot_of(const ReshapeArgs &a, int64_t row, int64_t rows) {
    return row < rows ? __ldg(a.slot_mapping + (row >> 1)) : -1;
}

// A row is written iff its slot is in range; -1 is padding; anything else is flagged
// (once per token, by its K row) and skipped.
__device__ __forceinline__ bool row_ok(const ReshapeArgs &a, int64_t row, int64_t slot, int lane) {
    if (slot >= 0 && slot < a.num_slots) return true;
    if (slot != -1 && lane == 0 && (row & 1) == 0) flag(a.status, KVFP8_DEV_BAD_SLOT);
    return false;
}

template <typename G, int U>
__device__ __forceinline__ void load_row(G (&buf)[U], const RowCtx &c, int64_t row, int units,
                                         int lane) {
    const uint8_t *p = c.src + (row >> 1) * c.stride_bytes;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int g = lane + 32 * u;
        if (g < units) buf[u].load(p + static_cast<int64_t>(g) * G::kBytes);
    }
}

// A side whose cache is bf16 (mixed cache dtypes): the row is stored at 16 bits, rounded to
// bf16 (a bf16 source is copied unchanged), with no scale.
template <typename G, int U>
__device__ __forceinline__ void store_row_bf16(const G (&buf)[U], const RowCtx &c, int64_t slot,
                                               int row_elems, int units, int lane) {
    uint8_t *dst = c.cache + slot * row_elems * 2;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int g = lane + 32 * u;
        if (g < units) {
            uint32_t o[G::kElems / 2];
            buf[u].bf16_words(o);
            uint4 *q = reinterpret_cast<uint4 *>(dst + static_cast<int64_t>(g) * G::kElems * 2);
#pragma unroll
            for (int i = 0; i < G::kElems / 8; ++i)
                st_ef(reinterpret_cast<uint8_t *>(q + i),
                      make_uint4(o[4 * i], o[4 * i + 1], o[4 * i + 2], o[4 * i + 3]), c.pol);
        }
    }
}

// E4M3 codes of a row: 8 bytes per lane and unit (8-element groups) or 16 (wide units).
template <typename G, int U, bool kFast>
__device__ __forceinline__ void store_row(const G (&buf)[U], const RowCtx &c, const FastDiv &fd,
                                          int64_t slot, int row_elems, int units, int lane) {
    uint8_t *dst = c.cache + slot * row_elems;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int g = lane + 32 * u;
        if (g < units) {
            float x[G::kElems];
            buf[u].unpack(x);
            if constexpr (G::kElems == 8) {
                st_ef(dst + static_cast<int64_t>(g) * 8, quantize8<kFast>(x, c.s, fd, buf[u].signs8(0)),
                      c.pol);
            } else {
                const uint2 lo = quantize8<kFast>(*reinterpret_cast<const float(*)[8]>(x), c.s, fd,
                                                  buf[u].signs8(0));
                const uint2 hi = quantize8<kFast>(*reinterpret_cast<const float(*)[8]>(x + 8), c.s,
                                                  fd, buf[u].signs8(1));
                st_ef(dst + static_cast<int64_t>(g) * 16, make_uint4(lo.x, lo.y, hi.x, hi.y), c.pol);
            }
        }
    }
}

__device__ __forceinline__ bool fast_range(float s) {
    const float sa = fabsf(s);
    return sa >= 0x1p-60f && sa <= 0x1p60f;
}

// The rows of one warp (every stride-th row from r), two in flight.  kMode: 0 = E4M3 with
// the fast divide, 1 = E4M3 with __fdiv_rn, 2 = bf16 cache (mixed cache dtypes).
template <typename G, int U, int kMode>
__device__ __forceinline__ void pipelined_rows(const ReshapeArgs &a, const RowCtx &c, int64_t r,
                                               int64_t stride, int64_t rows, int lane) {
    constexpr bool kFast = kMode == 0;
    const FastDiv fd(c.s);
    const int units = a.row_elems / G::kElems;
    G A[U], B[U];
    // the first row's source is read before its slot is known (the source row exists for
    // every token; a padding row's bytes are simply not stored), so the warp's first loads do
    // not wait behind the slot load
    if (r < rows) load_row(A, c, r, units, lane);
    int64_t s1 = slot_of(a, r, rows);
    int64_t s2 = slot_of(a, r + stride, rows);
    bool ok1 = r < rows && row_ok(a, r, s1, lane);
    while (r < rows) {
        int64_t rn = r + stride;
        bool ok2 = rn < rows && row_ok(a, rn, s2, lane);
        if (ok2) load_row(B, c, rn, units, lane);
        int64_t s3 = slot_of(a, rn + stride, rows);
        if (ok1) {
            if (kMode == 2) store_row_bf16(A, c, s1, a.row_elems, units, lane);
            else store_row<G, U, kFast>(A, c, fd, s1, a.row_elems, units, lane);
        }
        r = rn; s1 = s2; s2 = s3; ok1 = ok2;
        if (r >= rows) break;
        rn = r + stride;
        ok2 = rn < rows && row_ok(a, rn, s2, lane);
        if (ok2) load_row(A, c, rn, units, lane);
        s3 = slot_of(a, rn + stride, rows);
        if (ok1) {
            if (kMode == 2) store_row_bf16(B, c, s1, a.row_elems, units, lane);
            else store_row<G, U, kFast>(B, c, fd, s1, a.row_elems, units, lane);
        }
        r = rn; s1 = s2; s2 = s3; ok1 = ok2;
    }
}

// Rows of up to 32*U units of G::kElems elements.
template <typename G, int U>
__global__ void __launch_bounds__(kWarps * 32) reshape_pipelined_kernel(const ReshapeArgs a) {
    constexpr bool kF32 = G::kBytes == 4 * G::kElems;
    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    if ((!a.k_bf16 && !scale_ok(sk)) || (!a.v_bf16 && !scale_ok(sv))) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t rows = 2 * a.num_tokens;
    const int64_t stride = static_cast<int64_t>(gridDim.x) * kWarps;  // even
    const int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    const bool is_v = (r & 1) != 0;  // fixed for the warp: the stride is even
    RowCtx c;
    c.src = static_cast<const uint8_t *>(is_v ? a.value : a.key);
    c.cache = is_v ? a.value_cache : a.key_cache;
    c.stride_bytes = (is_v ? a.value_stride : a.key_stride) * (kF32 ? 4 : 2);
    c.s = is_v ? sv : sk;
    c.pol = evict_first_policy();
    if (is_v ? a.v_bf16 : a.k_bf16)  // uniform per warp
        pipelined_rows<G, U, 2>(a, c, r, stride, rows, lane);
    else if (fast_range(c.s))
        pipelined_rows<G, U, 0>(a, c, r, stride, rows, lane);
    else
        pipelined_rows<G, U, 1>(a, c, r, stride, rows, lane);
}

// ---------------------------------------------------------------- rope + cache write
//
// K rows are rotated (rope) before the divide/encode; V rows are stored as above.  The
// rotation of a pair (a, b) by the table entry (c, s) is a' = a*c - b*s, b' = a*s + b*c,
// each product and sum rounded to float in that order (no fused multiply-add), so the
// bytes match a plain CPU evaluation.  In the NeoX layout dim i pairs with i + rot/2: a
// lane's 8-dim group and its partner group sit rot/16 lanes apart inside the head's
// lane block, and are exchanged with one shuffle per value.  In the GPT-J layout pairs
// are adjacent dims inside the group.  The table values a lane needs are the same for
// every head of a row, so they are read once per row, issued with the row's data loads.

__device__ __forceinline__ bool pos_ok(const ReshapeArgs &a, int64_t pos) {
    return pos >= 0 && pos < a.max_pos;
}

// The cos/sin a lane needs for one row.  A lane's 8-dim groups g = lane + 32u all start at
// the same dim of their head, d0 = 8*lane mod head_dim (head_dim divides 256), so one set
// of table values serves the whole row; it is fetched together with the row's data, two
// rows ahead of its use.  NeoX: 8 cos and 8 sin of pairs ci..ci+7; GPT-J: 4 of each.
struct RopeCS {
    float c[8], s[8];
};

__device__ __forceinline__ void load_cs(RopeCS &t, const ReshapeArgs &a, int64_t pos, int lane) {
    const int d0 = (lane * 8) % a.head_dim;
    if (d0 >= a.rot) return;  // pass-through dims
    const float *cs = a.cos_sin + pos * a.rot;
    const int half = a.rot >> 1;
    if (a.neox) {
        const int ci = d0 < half ? d0 : d0 - half;
        const float4 c0 = __ldg(reinterpret_cast<const float4 *>(cs + ci));
        const float4 c1 = __ldg(reinterpret_cast<const float4 *>(cs + ci + 4));
        const float4 s0 = __ldg(reinterpret_cast<const float4 *>(cs + half + ci));
        const float4 s1 = __ldg(reinterpret_cast<const float4 *>(cs + half + ci + 4));
        t.c[0] = c0.x; t.c[1] = c0.y; t.c[2] = c0.z; t.c[3] = c0.w;
        t.c[4] = c1.x; t.c[5] = c1.y; t.c[6] = c1.z; t.c[7] = c1.w;
        t.s[0] = s0.x; t.s[1] = s0.y; t.s[2] = s0.z; t.s[3] = s0.w;
        t.s[4] = s1.x; t.s[5] = s1.y; t.s[6] = s1.z; t.s[7] = s1.w;
    } else {
        const float4 cv = __ldg(reinterpret_cast<const float4 *>(cs + d0 / 2));
        const float4 sv = __ldg(reinterpret_cast<const float4 *>(cs + half + d0 / 2));
        t.c[0] = cv.x; t.c[1] = cv.y; t.c[2] = cv.z; t.c[3] = cv.w;
        t.s[0] = sv.x; t.s[1] = sv.y; t.s[2] = sv.z; t.s[3] = sv.w;
    }
}

template <bool kF32, int U, bool kFast>
__device__ __forceinline__ void store_row_rope(const Group<kF32> (&buf)[U], const RopeCS &t,
                                               const RowCtx &c, const FastDiv &fd,
                                               const ReshapeArgs &a, int64_t slot, int groups,
                                               int lane) {
    uint8_t *dst = c.cache + slot * a.row_elems;
    const int half = a.rot >> 1;
    const int partner = half >> 3;  // lanes between a group and its NeoX partner
    const int d0 = (lane * 8) % a.head_dim;
    const bool rotated = d0 < a.rot;
    const bool first = d0 < half;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int g = lane + 32 * u;
        float x[8];
        buf[u].unpack(x);  // lanes past the row hold stale values; they only feed shuffles
        if (a.neox) {
            float y[8];  // the partner group's values, shuffled packed (half the shuffles for bf16)
            buf[u].xor_lane(partner).unpack(y);
            if (g < groups && rotated) {
                // first half: x*c - y*s; second half: y*s + x*c (= x*c + y*s exactly)
#pragma unroll
                for (int i = 0; i < 8; i += 2) {
                    const uint64_t xc = mul2(pack2(x[i], x[i + 1]), pack2(t.c[i], t.c[i + 1]));
                    const uint64_t ys = mul2(pack2(y[i], y[i + 1]), pack2(t.s[i], t.s[i + 1]));
                    unpack2(first ? sub2(xc, ys) : add2(xc, ys), x[i], x[i + 1]);
                }
            }
        } else if (g < groups && rotated) {
            // pairs (p, q) = (x[2j], x[2j+1]), two pairs per packed operation:
            // p' = p*c - q*s, q' = p*s + q*c
#pragma unroll
            for (int j = 0; j < 4; j += 2) {
                const uint64_t p = pack2(x[2 * j], x[2 * j + 2]);
                const uint64_t q = pack2(x[2 * j + 1], x[2 * j + 3]);
                const uint64_t c = pack2(t.c[j], t.c[j + 1]);
                const uint64_t sn = pack2(t.s[j], t.s[j + 1]);
                unpack2(sub2(mul2(p, c), mul2(q, sn)), x[2 * j], x[2 * j + 2]);
                unpack2(add2(mul2(p, sn), mul2(q, c)), x[2 * j + 1], x[2 * j + 3]);
            }
        }
        if (g < groups)
            st_ef(dst + static_cast<int64_t>(g) * 8, quantize8<kFast>(x, c.s, fd, sign_bytes(x)), c.pol);
    }
}

// The tokens of one warp (every W-th token from t, W = warps in the grid): the K row of
// each, rotated, then its V row.  One row's loads are in flight while the other row is
// stored, so K and V work is spread evenly over the warps; the table values of the next
// token travel with its K row's loads.
template <bool kF32, int U, bool kFast>
__device__ __forceinline__ void rope_token_rows(const ReshapeArgs &a, const RowCtx &ck,
                                                const RowCtx &cv, int64_t t, int64_t W,
                                                int lane) {
    const FastDiv fk(ck.s), fv(cv.s);
    const int groups = a.row_elems >> 3;
    const int64_t T = a.num_tokens;
    auto slot_at = [&](int64_t tok) -> int64_t {
        return tok < T ? __ldg(a.slot_mapping + tok) : -1;
    };
    auto pos_at = [&](int64_t tok) -> int64_t { return tok < T ? __ldg(a.positions + tok) : 0; };
    auto ok_of = [&](int64_t tok, int64_t slot, int64_t pos) -> bool {
        if (tok >= T) return false;
        if (slot >= 0 && slot < a.num_slots && pos_ok(a, pos)) return true;
        if (slot != -1 && lane == 0) flag(a.status, KVFP8_DEV_BAD_SLOT);
        return false;
    };
    Group<kF32> A[U], B[U];  // the K row and the V row
    RopeCS tc;
    int64_t s1 = slot_at(t), p1 = pos_at(t);
    int64_t s2 = slot_at(t + W), p2 = pos_at(t + W);
    // the first token's rows are read before its slot and position are known (the source
    // rows exist for every token), so the warp's first loads do not wait behind those loads
    if (t < T) {
        load_row(A, ck, 2 * t, groups, lane);
        load_row(B, cv, 2 * t + 1, groups, lane);
    }
    bool ok1 = ok_of(t, s1, p1);
    if (ok1) load_cs(tc, a, p1, lane);
    while (t < T) {
        const int64_t tn = t + W;
        const bool ok2 = ok_of(tn, s2, p2);
        const int64_t s3 = slot_at(tn + W), p3 = pos_at(tn + W);
        if (ok1) store_row_rope<kF32, U, kFast>(A, tc, ck, fk, a, s1, groups, lane);
        if (ok2) {
            load_row(A, ck, 2 * tn, groups, lane);
            load_cs(tc, a, p2, lane);
        }
        if (ok1) store_row<Group<kF32>, U, kFast>(B, cv, fv, s1, a.row_elems, groups, lane);
        if (ok2) load_row(B, cv, 2 * tn + 1, groups, lane);
        t = tn; s1 = s2; s2 = s3; p1 = p2; p2 = p3; ok1 = ok2;
    }
}

template <bool kF32, int U>
__global__ void __launch_bounds__(kWarps * 32) rope_reshape_kernel(const ReshapeArgs a) {
    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t W = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5);
    RowCtx ck, cv;
    ck.src = static_cast<const uint8_t *>(a.key);
    ck.cache = a.key_cache;
    ck.stride_bytes = a.key_stride * (kF32 ? 4 : 2);
    ck.s = sk;
    ck.pol = evict_first_policy();
    cv.src = static_cast<const uint8_t *>(a.value);
    cv.cache = a.value_cache;
    cv.stride_bytes = a.value_stride * (kF32 ? 4 : 2);
    cv.s = sv;
    cv.pol = ck.pol;
    if (fast_range(sk) && fast_range(sv))
        rope_token_rows<kF32, U, true>(a, ck, cv, t, W, lane);
    else
        rope_token_rows<kF32, U, false>(a, ck, cv, t, W, lane);
}

// ---------------------------------------------------------------- rope + cache write, staged
//
// The rope write with its source rows staged in shared memory (bf16 sources, 16-element
// units).  The kernel above keeps each warp's next rows in registers, and the rotation's
// table values and temporaries take so many registers (117) that 16 warps fit an SM, with
// about one row per warp in flight: too few bytes in flight to cover HBM latency, and too
// few warps to cover the conversion's own latencies.  Here each warp owns two slots, one
// for a token's K row (with its table row) and one for its V row, each filled by bulk copies
// (cp.async.bulk, issued by one lane) that complete on the slot's own mbarrier: the next
// token's K row is fetched while this token's V row is converted, and its V row while its K
// row is.  A lane converts 16 consecutive elements, in two halves of 8 (64 registers), and
// stores their codes with one 16-byte store; the NeoX partner unit and the table values are
// read from shared memory, not shuffled or kept in registers.  A warp needs ~4.6 KB at
// 1024-element rows, so four CTAs of 8 warps share an SM.  Measured on llama3_8b's rope
// step (fraction of the copy peak): whole units, a ring of two or three tokens, 16 warps
// per SM 0.790; half units, two tokens, 24 warps 0.818-0.833; these two row slots, 32 warps
// 0.827 (0.818 for the 24-warp form on the same box), and on the shorter prefill write
// 0.659 (0.635).  The arithmetic, and so every byte, is that of store_row_rope and store_row.

__device__ __forceinline__ void ring_bar_init(uint32_t bar) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void ring_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void ring_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ bool ring_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// bounded wait (~2 s at 2 GHz); false when it runs out
__device__ __forceinline__ bool ring_wait(uint32_t bar, uint32_t parity) {
    if (ring_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (ring_try(bar, parity)) return true;
        if ((it & 15u) == 15u && clock64() - t0 > 4000000000LL) return false;
    }
    return false;
}
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
        "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}
__device__ __forceinline__ uint4 lds16(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ float4 lds16f(uint32_t addr) {
    const uint4 v = lds16(addr);
    return make_float4(__uint_as_float(v.x), __uint_as_float(v.y), __uint_as_float(v.z), __uint_as_float(v.w));
}
// The staged path takes bf16 sources with rows of 16-element units, and NeoX rotations of
// at least 32 dims (a unit and its partner then lie in different halves).
bool rope_ring_ok(const ReshapeArgs &a) {
    return a.src_dtype != KVFP8_F32 && a.row_elems % 16 == 0 && a.row_elems <= 2048 &&
           (!a.neox || a.rot >= 32);
}

// One K row of a staged token: rotate and encode the lane's units (the row's source at
// shared-memory address ks, its table row at cs).
template <int U, bool kFast>
__device__ __forceinline__ void ring_k_row(const ReshapeArgs &a, uint32_t ks, uint32_t cs, uint8_t *kdst,
                                           int lane, float sk, const FastDiv &fk, uint64_t pol) {
    const int units = a.row_elems >> 4;
    const int half = a.rot >> 1;
    // the lane's units all start at the same dim of their head (head_dim divides 512)
    const int d0 = (lane * 16) % a.head_dim;
    const bool rotated = d0 < a.rot;
    const bool first = d0 < half;
    // NeoX: cos/sin of pairs ci.. (dims d0.. and their partners); GPT-J: of pairs d0/2..
    const int ci = a.neox ? (first ? d0 : d0 - half) : d0 / 2;
    const int step = half >> 4;  // units between a NeoX unit and its partner
    // K: each unit in two halves of 8 elements (fewer values live at once), one
    // 16-byte store of codes
#pragma unroll 1
    for (int q = 0; q < U; ++q) {
        const int u = lane + 32 * q;
        if (u >= units) break;
        uint32_t code[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 wx = lds16(ks + 32 * u + 16 * h);
            float x[8];
            x[0] = bf16lo(wx.x); x[1] = bf16hi(wx.x); x[2] = bf16lo(wx.y); x[3] = bf16hi(wx.y);
            x[4] = bf16lo(wx.z); x[5] = bf16hi(wx.z); x[6] = bf16lo(wx.w); x[7] = bf16hi(wx.w);
            uint2 sg;
            if (rotated) {
                if (a.neox) {
                    // first half: x*c - y*s; second half: y*s + x*c (= x*c + y*s exactly)
                    const uint4 wy = lds16(ks + 32 * (first ? u + step : u - step) + 16 * h);
                    const float y[8] = {bf16lo(wy.x), bf16hi(wy.x), bf16lo(wy.y), bf16hi(wy.y),
                                        bf16lo(wy.z), bf16hi(wy.z), bf16lo(wy.w), bf16hi(wy.w)};
                    const float4 c0 = lds16f(cs + 4 * (ci + 8 * h)), c1 = lds16f(cs + 4 * (ci + 8 * h + 4));
                    const float4 s0 = lds16f(cs + 4 * (half + ci + 8 * h)), s1 = lds16f(cs + 4 * (half + ci + 8 * h + 4));
                    const float c[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
                    const float sn[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
#pragma unroll
                    for (int i = 0; i < 8; i += 2) {
                        const uint64_t xc = mul2(pack2(x[i], x[i + 1]), pack2(c[i], c[i + 1]));
                        const uint64_t ys = mul2(pack2(y[i], y[i + 1]), pack2(sn[i], sn[i + 1]));
                        unpack2(first ? sub2(xc, ys) : add2(xc, ys), x[i], x[i + 1]);
                    }
                } else {
                    // pairs (p, q) = (x[2j], x[2j+1]): p' = p*c - q*s, q' = p*s + q*c
                    const float4 cv = lds16f(cs + 4 * (ci + 4 * h));
                    const float4 sv4 = lds16f(cs + 4 * (half + ci + 4 * h));
                    const float c[4] = {cv.x, cv.y, cv.z, cv.w};
                    const float sn[4] = {sv4.x, sv4.y, sv4.z, sv4.w};
#pragma unroll
                    for (int j = 0; j < 4; j += 2) {
                        const uint64_t p = pack2(x[2 * j], x[2 * j + 2]);
                        const uint64_t qq = pack2(x[2 * j + 1], x[2 * j + 3]);
                        const uint64_t cc = pack2(c[j], c[j + 1]);
                        const uint64_t ss = pack2(sn[j], sn[j + 1]);
                        unpack2(sub2(mul2(p, cc), mul2(qq, ss)), x[2 * j], x[2 * j + 2]);
                        unpack2(add2(mul2(p, ss), mul2(qq, cc)), x[2 * j + 1], x[2 * j + 3]);
                    }
                }
                sg = sign_bytes(x);
            } else {
                sg = sign_bytes_bf16(wx.x, wx.y, wx.z, wx.w);
            }
            const uint2 cd = quantize8<kFast>(x, sk, fk, sg);
            code[2 * h] = cd.x;
            code[2 * h + 1] = cd.y;
        }
        st_ef(kdst + 16 * u, make_uint4(code[0], code[1], code[2], code[3]), pol);
    }
}

// One V row of a staged token: encode the lane's units (source at shared-memory address vs).
template <int U, bool kFast>
__device__ __forceinline__ void ring_v_row(const ReshapeArgs &a, uint32_t vs, uint8_t *vdst, int lane,
                                           float sv, const FastDiv &fv, uint64_t pol) {
    const int units = a.row_elems >> 4;
#pragma unroll 1
    for (int q = 0; q < U; ++q) {
        const int u = lane + 32 * q;
        if (u >= units) break;
        uint32_t code[4];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const uint4 wx = lds16(vs + 32 * u + 16 * h);
            const float x[8] = {bf16lo(wx.x), bf16hi(wx.x), bf16lo(wx.y), bf16hi(wx.y),
                                bf16lo(wx.z), bf16hi(wx.z), bf16lo(wx.w), bf16hi(wx.w)};
            const uint2 cd = quantize8<kFast>(x, sv, fv, sign_bytes_bf16(wx.x, wx.y, wx.z, wx.w));
            code[2 * h] = cd.x;
            code[2 * h + 1] = cd.y;
        }
        st_ef(vdst + 16 * u, make_uint4(code[0], code[1], code[2], code[3]), pol);
    }
}

constexpr int kRowHeader = 32;  // two mbarriers, then the K and V slots' cache slot indices
__host__ __device__ constexpr int rowring_region_bytes(int row_elems, int rot) {
    return kRowHeader + 2 * row_elems * 2 + rot * 4;
}

template <int U, bool kFast>
__device__ __forceinline__ void ring_rows(const ReshapeArgs &a, uint32_t region, uint8_t *region_p,
                                          int64_t t, int64_t W, int lane, float sk, float sv) {
    const FastDiv fk(sk), fv(sv);
    const uint64_t pol = evict_first_policy();
    const int64_t T = a.num_tokens;
    const int rb = a.row_elems * 2;                       // source row bytes
    const uint32_t bk = region, bv = region + 8;
    volatile int64_t *meta = reinterpret_cast<volatile int64_t *>(region_p + 16);  // K slot, V slot
    const uint32_t ks = region + kRowHeader, cs = ks + rb, vs = cs + a.rot * 4;
    const int64_t kstride = a.key_stride * 2, vstride = a.value_stride * 2;
    const uint8_t *kbase = static_cast<const uint8_t *>(a.key);
    const uint8_t *vbase = static_cast<const uint8_t *>(a.value);
    auto slot_at = [&](int64_t tok) -> int64_t { return tok < T ? __ldg(a.slot_mapping + tok) : -1; };
    auto pos_at = [&](int64_t tok) -> int64_t { return tok < T ? __ldg(a.positions + tok) : 0; };
    // first lane: fetch token tok's K row and table row (its slot and position, read one
    // token ahead, are checked here); returns the cache slot its rows go to, -1 for none, in
    // which case the K slot's phase completes without copies
    auto issue_k = [&](int64_t tok, int64_t slot, int64_t pos) -> int64_t {
        const bool ok = slot >= 0 && slot < a.num_slots && pos_ok(a, pos);
        if (!ok && slot != -1) flag(a.status, KVFP8_DEV_BAD_SLOT);
        const int64_t st = ok ? slot : -1;
        meta[0] = st;
        if (ok) {
            ring_arrive_tx(bk, static_cast<uint32_t>(rb + a.rot * 4));
            bulk_g2s(ks, kbase + tok * kstride, rb, bk);
            bulk_g2s(cs, a.cos_sin + pos * a.rot, static_cast<uint32_t>(a.rot * 4), bk);
        } else {
            ring_arrive(bk);
        }
        return st;
    };
    // first lane: fetch token tok's V row (st: its cache slot, -1 for none)
    auto issue_v = [&](int64_t tok, int64_t st) {
        meta[1] = st;
        if (st >= 0) {
            ring_arrive_tx(bv, static_cast<uint32_t>(rb));
            bulk_g2s(vs, vbase + tok * vstride, rb, bv);
        } else {
            ring_arrive(bv);
        }
    };
    int issued_k = 0, issued_v = 0, done_k = 0, done_v = 0;  // rows fetched / converted
    int64_t nslot = -1, npos = 0;  // the next token's slot and position (first lane)
    if (lane == 0) {
        ring_bar_init(bk);
        ring_bar_init(bv);
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
        if (t < T) {
            const int64_t st = issue_k(t, slot_at(t), pos_at(t));
            issue_v(t, st);
            issued_k = issued_v = 1;
        }
        nslot = slot_at(t + W);
        npos = pos_at(t + W);
    }
    __syncwarp();
    bool ok = true;
    for (int j = 0; t + j * W < T; ++j) {
        const int64_t tok = t + j * W;
        const bool more = tok + W < T;
        ok = __all_sync(0xFFFFFFFFu, ring_wait(bk, static_cast<uint32_t>(j & 1)));
        if (!ok) break;
        ++done_k;
        int64_t slot = meta[0];
        if (slot >= 0) ring_k_row<U, kFast>(a, ks, cs, a.key_cache + slot * a.row_elems, lane, sk, fk, pol);
        __syncwarp();  // every lane is done reading the K slot
        int64_t next_v = -1;
        if (lane == 0 && more) {
            // the slot's shared-memory reads (generic proxy) before the copies that overwrite
            // it (async proxy)
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            next_v = issue_k(tok + W, nslot, npos);
            ++issued_k;
            nslot = slot_at(tok + 2 * W);
            npos = pos_at(tok + 2 * W);
        }
        ok = __all_sync(0xFFFFFFFFu, ring_wait(bv, static_cast<uint32_t>(j & 1)));
        if (!ok) break;
        ++done_v;
        slot = meta[1];
        if (slot >= 0) ring_v_row<U, kFast>(a, vs, a.value_cache + slot * a.row_elems, lane, sv, fv, pol);
        __syncwarp();  // every lane is done reading the V slot
        if (lane == 0 && more) {
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            issue_v(tok + W, next_v);
            ++issued_v;
        }
    }
    if (!ok && lane == 0) {
        flag(a.status, KVFP8_DEV_TIMEOUT);
        // let the copies still in flight land before the CTA's shared memory goes away
        for (int k = done_k; k < issued_k; ++k) ring_wait(bk, static_cast<uint32_t>(k & 1));
        for (int k = done_v; k < issued_v; ++k) ring_wait(bv, static_cast<uint32_t>(k & 1));
    }
}

template <int U>
__global__ void __launch_bounds__(kWarps * 32) rope_ring_kernel(const ReshapeArgs a) {
    extern __shared__ __align__(128) uint8_t ring_smem[];
    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t W = static_cast<int64_t>(gridDim.x) * kWarps;
    const int64_t t = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
    uint8_t *region_p = ring_smem + warp * rowring_region_bytes(a.row_elems, a.rot);
    const uint32_t region = smem_u32(region_p);
    if (fast_range(sk) && fast_range(sv))
        ring_rows<U, true>(a, region, region_p, t, W, lane, sk, sv);
    else
        ring_rows<U, false>(a, region, region_p, t, W, lane, sk, sv);
}

// Any row length: one warp per row, groups streamed in rounds of 4 per lane.
template <bool kF32>
__global__ void __launch_bounds__(kWarps * 32) reshape_rowloop_kernel(const ReshapeArgs a) {
    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    const int lane = threadIdx.x & 31;
    const int64_t rows = 2 * a.num_tokens;
    const uint64_t pol = evict_first_policy();
    for (int64_t r = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); r < rows;
         r += static_cast<int64_t>(gridDim.x) * kWarps) {
        const int64_t slot = __ldg(a.slot_mapping + (r >> 1));
        if (!row_ok(a, r, slot, lane)) continue;
        const bool is_v = (r & 1) != 0;
        const float s = is_v ? sv : sk;
        const FastDiv fd(s);
        const bool fast = fast_range(s);
        const uint8_t *src = static_cast<const uint8_t *>(is_v ? a.value : a.key) +
                             (r >> 1) * (is_v ? a.value_stride : a.key_stride) * (kF32 ? 4 : 2);
        uint8_t *dst = (is_v ? a.value_cache : a.key_cache) + slot * a.row_elems;
        const int groups = a.row_elems >> 3;
        for (int g0 = lane; g0 < groups; g0 += 32 * 4) {
            Group<kF32> in[4];
#pragma unroll
            for (int u = 0; u < 4; ++u)
                if (g0 + 32 * u < groups)
                    in[u].load(src + static_cast<int64_t>(g0 + 32 * u) * Group<kF32>::kBytes);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int g = g0 + 32 * u;
                if (g < groups) {
                    float x[8];
                    in[u].unpack(x);
                    st_ef(dst + static_cast<int64_t>(g) * 8,
                          fast ? quantize8<true>(x, s, fd, in[u].signs8(0))
                               : quantize8<false>(x, s, fd, in[u].signs8(0)),
                          pol);
                }
            }
        }
    }
}

// A grid of at most one resident wave, no more warps than units of work (rows, or tokens
// for the rope kernel).
template <typename K>
cudaError_t launch_persistent(K kernel, const ReshapeArgs &a, cudaStream_t stream,
                              int64_t units, size_t smem = 0) {
    DeviceFacts f;
    int occ = 0;
    cudaError_t err = device_facts(&f);
    if (err != cudaSuccess) return err;
    if (smem > static_cast<size_t>(f.smem_optin)) return cudaErrorNotSupported;
    if ((err = kernel_occupancy(kernel, kWarps * 32, smem, &occ)) != cudaSuccess) return err;
    const int64_t want = (units + kWarps - 1) / kWarps;
    const int64_t full = static_cast<int64_t>(f.sms) * std::max(occ, 1);
    const unsigned blocks = static_cast<unsigned>(std::min(want, full));
    kernel<<<blocks, kWarps * 32, smem, stream>>>(a);
    return cudaGetLastError();
}

// The wide path (16 elements and one 16-byte store of codes per lane and unit) needs rows of
// at least 512 elements, a multiple of 16, and 32-byte aligned source rows.
bool wide_ok(const ReshapeArgs &a) {
    const int64_t esz = a.src_dtype == KVFP8_F32 ? 4 : 2;
    const uintptr_t bases = reinterpret_cast<uintptr_t>(a.key) | reinterpret_cast<uintptr_t>(a.value);
    return a.row_elems % 16 == 0 && a.row_elems >= 512 && a.row_elems <= 2048 &&
           (bases & 31u) == 0 && (a.key_stride * esz) % 32 == 0 && (a.value_stride * esz) % 32 == 0;
}

template <bool kF32>
cudaError_t dispatch(const ReshapeArgs &a, cudaStream_t stream) {
    const int64_t rows = 2 * a.num_tokens;
    if (wide_ok(a)) {
        const int per_lane = (a.row_elems / 16 + 31) / 32;  // 16-element units per lane
        if (per_lane <= 1) return launch_persistent(reshape_pipelined_kernel<Wide<kF32>, 1>, a, stream, rows);
        if (per_lane <= 2) return launch_persistent(reshape_pipelined_kernel<Wide<kF32>, 2>, a, stream, rows);
        return launch_persistent(reshape_pipelined_kernel<Wide<kF32>, 4>, a, stream, rows);
    }
    const int per_lane = (a.row_elems / 8 + 31) / 32;  // 8-element groups per lane
    if (per_lane <= 1) return launch_persistent(reshape_pipelined_kernel<Group<kF32>, 1>, a, stream, rows);
    if (per_lane <= 2) return launch_persistent(reshape_pipelined_kernel<Group<kF32>, 2>, a, stream, rows);
    if (per_lane <= 4) return launch_persistent(reshape_pipelined_kernel<Group<kF32>, 4>, a, stream, rows);
    if (per_lane <= 8) return launch_persistent(reshape_pipelined_kernel<Group<kF32>, 8>, a, stream, rows);
    return launch_persistent(reshape_rowloop_kernel<kF32>, a, stream, rows);
}

template <bool kF32>
cudaError_t dispatch_rope(const ReshapeArgs &a, cudaStream_t stream) {
    if (!kF32 && rope_ring_ok(a)) {
        const size_t smem = static_cast<size_t>(kWarps) * rowring_region_bytes(a.row_elems, a.rot);
        const int units = (a.row_elems / 16 + 31) / 32;  // 16-element units per lane
        if (units <= 1) return launch_persistent(rope_ring_kernel<1>, a, stream, a.num_tokens, smem);
        if (units <= 2) return launch_persistent(rope_ring_kernel<2>, a, stream, a.num_tokens, smem);
        return launch_persistent(rope_ring_kernel<4>, a, stream, a.num_tokens, smem);
    }
    const int per_lane = (a.row_elems / 8 + 31) / 32;
    if (per_lane <= 1) return launch_persistent(rope_reshape_kernel<kF32, 1>, a, stream, a.num_tokens);
    if (per_lane <= 2) return launch_persistent(rope_reshape_kernel<kF32, 2>, a, stream, a.num_tokens);
    if (per_lane <= 4) return launch_persistent(rope_reshape_kernel<kF32, 4>, a, stream, a.num_tokens);
    if (per_lane <= 8) return launch_persistent(rope_reshape_kernel<kF32, 8>, a, stream, a.num_tokens);
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_reshape_and_cache(const ReshapeArgs &a, cudaStream_t stream) {
    if (a.num_tokens == 0) return cudaSuccess;
    if ((a.k_bf16 || a.v_bf16) && (a.cos_sin != nullptr || a.row_elems > 2048))
        return cudaErrorNotSupported;  // mixed dtypes: the pipelined plain store only
    if (a.cos_sin != nullptr)
        return a.src_dtype == KVFP8_F32 ? dispatch_rope<true>(a, stream)
                                        : dispatch_rope<false>(a, stream);
    return a.src_dtype == KVFP8_F32 ? dispatch<true>(a, stream) : dispatch<false>(a, stream);
}

}  // namespace kvfp8
