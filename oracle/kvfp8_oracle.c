/*
 * kvfp8 oracle -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, single-threaded CPU statement of what the FP8 (OCP E4M3)
 * paged KV-cache path computes.  Only the test suite, the package smoke check
 * and the benchmark's CPU-baseline leg may load this library; the product path
 * never does.  It shares no code, header, table or helper with the CUDA
 * library: every step below is written out again from the source pages.
 *
 * Sources (cited by page title and section):
 *   [P1] "llama : Add FP8 KV-cache support (#28392)", llama.cpp commit 202c1a229
 *   [P2] llama.cpp compare osimons/ocp_fp8_kv (the branch that prints the E4M3
 *        codec: ggml-impl.h, ggml-quants.c, tests/test-quantize-fns.cpp)
 *   [P3] vllm.cpp PR #1641 "feat(KV-FP8): W3 -- half-sized KV blocks the runner
 *        actually serves, and a default scale that knows it was declared"
 *
 * Readings taken where the pages are silent are marked READING.
 * Parity status of every function: pinned by tests/test_oracle_*.py.
 *
 * Build: plain C11, no fast-math, -ffp-contract=off so that no multiply-add is
 * fused behind the reader's back (the encode path never needs it; the
 * attention sums are in double and the choice only fixes the rounding order).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Status bits, same meaning as the library's device status word (the values
 * are restated here, not shared). */
enum {
    KVO_OK = 0,
    KVO_BAD_SCALE = 1u << 0,
    KVO_BAD_SLOT = 1u << 1,
    KVO_BAD_BLOCK = 1u << 2,
};

enum { KVO_BF16 = 0, KVO_F32 = 1 };

/* ---------------------------------------------------------------------- */
/* E4M3 decode.  [P2] ggml-impl.h, ggml_f8_e4m3_to_fp32; the same map is
 * restated in [P2] tests/test-quantize-fns.cpp (f8_e4m3_to_fp32_ref) and in
 * [P2] gguf-py quants.py (class F8_E4M3).
 *   magnitude 0x7F            -> NaN (both 0x7F and 0xFF)
 *   exponent field 0          -> mantissa * 2^-9          (subnormal grid)
 *   exponent field e in 1..15 -> (1 + mantissa/8) * 2^(e-7)
 *   the sign bit is applied last, so 0x80 decodes to -0.0
 * Every finite value is exact in double (and in float). */
double kvo_e4m3_decode(uint8_t code)
{
    const int mag = code & 0x7F;
    if (mag == 0x7F)
        return NAN;
    const int e = mag >> 3;
    const int m = mag & 7;
    double v;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(8.0 + (double)m, e - 10); /* (1 + m/8) * 2^(e-7) */
    return (code & 0x80) ? -v : v;
}

/* Round to the nearest integer, ties to the even neighbour.
 * [P2] ggml-impl.h, ggml_round_to_nearest_even: floor, then step up when the
 * remainder is above one half, or exactly one half with an odd floor.
 * Callers pass values whose remainders are exact in float. */
static int kvo_round_half_even(float v)
{
    const float lo = floorf(v);
    const float rem = v - lo; /* exact: v and lo share a binade or lo is 0 */
    int n = (int)lo;
    if (rem > 0.5f || (rem == 0.5f && (n & 1)))
        n += 1;
    return n;
}

/* E4M3 encode of one float, round-to-nearest-even, saturating.
 * [P2] ggml-impl.h, ggml_fp32_to_f8_e4m3.  Steps, in the page's order:
 *   1. take the sign bit (so -0.0 and negative NaN keep it);
 *   2. NaN -> sign|0x7F;  zero -> sign;  inf or |y| >= 448 -> sign|0x7E;
 *   3. |y| < 2^-6 (below the smallest normal): the code is the RNE integer
 *      of |y| * 2^9 on the uniform subnormal grid (8 lands on the smallest
 *      normal, code 0x08, which is the right answer);
 *   4. otherwise split |y| = f * 2^E with f in [1,2), round (f - 1) * 8 to
 *      three mantissa bits with RNE, carry a rounded-up mantissa of 8 into
 *      the exponent, and saturate anything past 448 to 0x7E.
 * Written here with the mantissa kept as an integer n = 8 + mantissa in
 * [8, 16]; the products |y|*2^9 and f*8 are exact in float. */
uint8_t kvo_e4m3_encode(float y)
{
    const uint8_t sign = signbit(y) ? 0x80 : 0x00;
    const float a = fabsf(y);
    if (isnan(a))
        return sign | 0x7F;
    if (a == 0.0f)
        return sign;
    if (isinf(a) || a >= 448.0f)
        return sign | 0x7E;
    if (a < 0.015625f) /* 2^-6 */
        return sign | (uint8_t)kvo_round_half_even(a * 512.0f);

    int e2;
    const float half_frac = frexpf(a, &e2); /* a = half_frac * 2^e2, half_frac in [0.5,1) */
    int unbiased = e2 - 1;                   /* a = f * 2^unbiased, f in [1,2) */
    int n = kvo_round_half_even(half_frac * 16.0f); /* = RNE(f * 8), in [8,16] */
    if (n == 16) {
        n = 8;
        unbiased += 1;
    }
    const int biased = unbiased + 7;
    const int man = n - 8;
    if (biased > 15 || (biased == 15 && man > 6))
        return sign | 0x7E;
    return sign | (uint8_t)(biased << 3) | (uint8_t)man;
}

/* Encode n floats (the same map, element by element). */
void kvo_e4m3_encode_n(const float *y, uint8_t *out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = kvo_e4m3_encode(y[i]);
}

/* bf16 -> float is exact: the 16 bits are the top half of the float. */
float kvo_bf16_to_f32(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float -> bf16 with round-to-nearest-even on the 16 dropped bits; NaN stays
 * NaN (quiet, sign kept).  Used only to state the dequant output dtype. */
uint16_t kvo_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if (isnan(f))
        return (uint16_t)((u >> 16) | 0x0040);
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* Per-layer scalar scale.  [P1] conversion/base.py _prepare_kv_cache_scales
 * accepts a BF16 or FP32 scalar and widens it to float; [P1]
 * llama-model.cpp load_tensors then holds it as F32.  bf16 widening is exact. */
float kvo_scale_value(const void *p, int dtype)
{
    if (dtype == KVO_BF16)
        return kvo_bf16_to_f32(*(const uint16_t *)p);
    return *(const float *)p;
}

/* [P1] llama-context.cpp llama_init_from_model and conversion/base.py: a
 * cache scale must be finite and nonzero.  A negative scale is allowed. */
int kvo_scale_ok(float s)
{
    return isfinite(s) && s != 0.0f;
}

/* One cached byte for one element.  [P1] llama-graph.cpp
 * build_attn_scale_kv_inputs stores K/s_k and V/s_v (ggml_div), then the cache
 * copy converts to F8_E4M3; [P3] ("the store divides by the scale").
 * The quotient is the IEEE float quotient (one rounding), then it is encoded
 * (a second rounding).
 * READING: for a NaN element the quotient's sign is not fixed by IEEE 754; the
 * CPU backends the pages run on hand the NaN operand through a division
 * unchanged, so the code keeps the element's own sign bit: sign(x)|0x7F. */
uint8_t kvo_store_code(float x, float s)
{
    if (isnan(x))
        return (signbit(x) ? 0x80 : 0x00) | 0x7F;
    const float y = x / s;
    return kvo_e4m3_encode(y);
}

static float kvo_load_src(const void *base, int dtype, int64_t idx)
{
    if (dtype == KVO_BF16)
        return kvo_bf16_to_f32(((const uint16_t *)base)[idx]);
    return ((const float *)base)[idx];
}

/* reshape_and_cache into paged blocks.
 * [P1] llama-kv-cache.cpp cpy_k / cpy_v scatter the rows of k_cur
 * [head_dim, n_kv, n_tokens] to destination rows given by an I64 index per
 * token; [P3] sizes the pages at one byte per element.
 * READING (cache layout): key_cache and value_cache are separate arrays laid
 * out [num_blocks][block_size][n_kv][head_dim] bytes; slot = block*block_size
 * + offset; slot -1 marks a padding token that is skipped; any other slot
 * outside [0, num_blocks*block_size) is skipped and flagged.
 * Bytes that are not written keep their prior contents.
 * Returns a bit set of KVO_* status flags. */
uint32_t kvo_reshape_and_cache(const void *key, const void *value, int src_dtype,
                               int64_t key_stride, int64_t value_stride, int64_t num_tokens,
                               uint8_t *key_cache, uint8_t *value_cache,
                               int32_t num_blocks, int32_t block_size, int32_t n_kv,
                               int32_t head_dim, const int64_t *slot_mapping,
                               float k_scale, float v_scale)
{
    uint32_t status = 0;
    if (!kvo_scale_ok(k_scale) || !kvo_scale_ok(v_scale))
        return KVO_BAD_SCALE;
    const int64_t row = (int64_t)n_kv * head_dim;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= num_slots) {
            status |= KVO_BAD_SLOT;
            continue;
        }
        const int64_t blk = slot / block_size;
        const int64_t off = slot % block_size;
        uint8_t *kdst = key_cache + (blk * block_size + off) * row;
        uint8_t *vdst = value_cache + (blk * block_size + off) * row;
        for (int32_t h = 0; h < n_kv; ++h) {
            for (int32_t d = 0; d < head_dim; ++d) {
                const int64_t e = (int64_t)h * head_dim + d;
                kdst[e] = kvo_store_code(kvo_load_src(key, src_dtype, i * key_stride + e), k_scale);
                vdst[e] = kvo_store_code(kvo_load_src(value, src_dtype, i * value_stride + e), v_scale);
            }
        }
    }
    return status;
}

/* Rotary position embedding of one head's vector, in float.
 * [P1] llama-graph.cpp build_attn: "expand k later to enable rope fusion which directly
 * writes into k-v cache" -- the fused form rotates K and stores it in one pass.
 * READING (the pages leave rope to the model): the caller supplies the table
 * cos_sin[pos][0..rot/2) = cos, cos_sin[pos][rot/2..rot) = sin (fp32), and each pair
 * (a, b) of the first rot dims becomes
 *     a' = a*cos - b*sin,   b' = a*sin + b*cos
 * with every product and sum rounded to float in that order (no fused multiply-add).
 * neox != 0 pairs dim i with dim i + rot/2 (GPT-NeoX layout); neox == 0 pairs 2i with
 * 2i+1 (GPT-J layout).  Pair i uses cos/sin entry i.  Dims >= rot pass through. */
void kvo_rope(float *x, int32_t head_dim, int32_t rot, int neox, const float *cs_row)
{
    const int32_t half = rot / 2;
    for (int32_t i = 0; i < half; ++i) {
        const int32_t ia = neox ? i : 2 * i;
        const int32_t ib = neox ? i + half : 2 * i + 1;
        const float c = cs_row[i], sn = cs_row[half + i];
        const float a = x[ia], b = x[ib];
        const float ac = a * c, bs = b * sn, as = a * sn, bc = b * c;
        x[ia] = ac - bs;
        x[ib] = as + bc;
    }
    (void)head_dim;
}

/* reshape_and_cache with rope applied to K first (positions[i] selects the table row);
 * V is stored as in kvo_reshape_and_cache.  Status bits as there; a position outside
 * [0, max_pos) flags KVO_BAD_SLOT and skips the row. */
uint32_t kvo_rope_reshape_and_cache(const void *key, const void *value, int src_dtype,
                                    int64_t key_stride, int64_t value_stride,
                                    int64_t num_tokens, uint8_t *key_cache,
                                    uint8_t *value_cache, int32_t num_blocks,
                                    int32_t block_size, int32_t n_kv, int32_t head_dim,
                                    const int64_t *slot_mapping, const int64_t *positions,
                                    const float *cos_sin, int64_t max_pos, int32_t rot,
                                    int neox, float k_scale, float v_scale)
{
    uint32_t status = 0;
    if (!kvo_scale_ok(k_scale) || !kvo_scale_ok(v_scale))
        return KVO_BAD_SCALE;
    const int64_t row = (int64_t)n_kv * head_dim;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    float *buf = (float *)malloc(sizeof(float) * (size_t)head_dim);
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= num_slots || positions[i] < 0 || positions[i] >= max_pos) {
            status |= KVO_BAD_SLOT;
            continue;
        }
        const float *cs_row = cos_sin + positions[i] * rot;
        uint8_t *kdst = key_cache + slot * row;
        uint8_t *vdst = value_cache + slot * row;
        for (int32_t h = 0; h < n_kv; ++h) {
            for (int32_t d = 0; d < head_dim; ++d)
                buf[d] = kvo_load_src(key, src_dtype, i * key_stride + (int64_t)h * head_dim + d);
            kvo_rope(buf, head_dim, rot, neox, cs_row);
            for (int32_t d = 0; d < head_dim; ++d) {
                const int64_t e = (int64_t)h * head_dim + d;
                kdst[e] = kvo_store_code(buf[d], k_scale);
                vdst[e] = kvo_store_code(kvo_load_src(value, src_dtype, i * value_stride + e), v_scale);
            }
        }
    }
    free(buf);
    return status;
}

/* Dequantize n bytes: dst = s * decode(code), the product taken in float.
 * [P1] llama-kv-cache.cpp build_rope_shift routes F8_E4M3 through the
 * dequantize -> rope -> requantize path; [P1] tests/test-fp8.cpp
 * check_fp8_context_shift decodes the stored bytes with to_float.
 * dst_dtype KVO_F32 writes floats, KVO_BF16 rounds the float to bf16 (RNE).
 * has_scale == 0 means no scale (the decoded value itself). */
void kvo_dequant(void *dst, int dst_dtype, const uint8_t *src, int64_t n, int has_scale, float scale)
{
    for (int64_t i = 0; i < n; ++i) {
        float v = (float)kvo_e4m3_decode(src[i]);
        if (has_scale)
            v = scale * v;
        if (dst_dtype == KVO_F32)
            ((float *)dst)[i] = v;
        else
            ((uint16_t *)dst)[i] = kvo_f32_to_bf16(v);
    }
}

/* Single-query (decode) paged attention for one (sequence, query head).
 * Definition: [P1] tests/test-fp8.cpp check_fp8_attention computes, in
 * double, scores = q.k / sqrt(head_size) over every past token, a max-shifted
 * softmax, and the probability-weighted sum of V, on K and V that went through
 * divide-by-scale, E4M3 round trip and multiply-by-scale.  [P1]
 * llama-graph.cpp moves s_k onto q and s_v onto the output; both are the same
 * numbers as dequantizing by the scales, which is what is written here.
 * READINGS: the query of sequence b attends to all seq_lens[b] cached tokens;
 * q head h reads kv head h / (n_q / n_kv); token t of a sequence lives in
 * physical block block_tables[b][t / block_size] at row t % block_size;
 * a sequence of length 0 gives a zero output.
 * out: head_dim doubles.  Returns KVO_BAD_BLOCK if a block id is out of range
 * (that token is then left out). */
uint32_t kvo_decode_one(double *out, const uint16_t *q_row, const uint8_t *key_cache,
                        const uint8_t *value_cache, const int32_t *block_table_row,
                        int32_t seq_len, int32_t n_kv, int32_t kv_head, int32_t head_dim,
                        int32_t block_size, int32_t num_blocks, double sm_scale,
                        float k_scale, float v_scale)
{
    uint32_t status = 0;
    for (int32_t d = 0; d < head_dim; ++d)
        out[d] = 0.0;
    if (seq_len <= 0)
        return 0;
    const int64_t row = (int64_t)n_kv * head_dim;
    double *score = (double *)malloc(sizeof(double) * (size_t)seq_len);
    uint8_t *ok = (uint8_t *)malloc((size_t)seq_len);
    double best = -INFINITY;
    for (int32_t t = 0; t < seq_len; ++t) {
        const int32_t phys = block_table_row[t / block_size];
        ok[t] = phys >= 0 && phys < num_blocks;
        if (!ok[t]) {
            status |= KVO_BAD_BLOCK;
            continue;
        }
        const uint8_t *k = key_cache + ((int64_t)phys * block_size + t % block_size) * row +
                           (int64_t)kv_head * head_dim;
        double dot = 0.0;
        for (int32_t d = 0; d < head_dim; ++d) {
            const double kd = (double)k_scale * kvo_e4m3_decode(k[d]);
            dot += (double)kvo_bf16_to_f32(q_row[d]) * kd;
        }
        score[t] = sm_scale * dot;
        if (score[t] > best)
            best = score[t];
    }
    double denom = 0.0;
    for (int32_t t = 0; t < seq_len; ++t) {
        if (!ok[t])
            continue;
        score[t] = exp(score[t] - best);
        denom += score[t];
    }
    for (int32_t t = 0; t < seq_len; ++t) {
        if (!ok[t])
            continue;
        const int32_t phys = block_table_row[t / block_size];
        const uint8_t *v = value_cache + ((int64_t)phys * block_size + t % block_size) * row +
                           (int64_t)kv_head * head_dim;
        const double p = score[t] / denom;
        for (int32_t d = 0; d < head_dim; ++d)
            out[d] += p * ((double)v_scale * kvo_e4m3_decode(v[d]));
    }
    free(score);
    free(ok);
    return status;
}

/* Mixed cache dtypes.  [P1] tests/test-fp8.cpp check_fp8_attention runs the FP8 cache on
 * K only, on V only, or on both (type_k / type_v F8_E4M3 or F16), each FP8 side with its
 * own scale and the other side unscaled; test-backend-ops adds the F8/F16 mixes.  Here the
 * 16-bit side is bf16: the cache holds the source value rounded to bf16 (RNE; exact for a
 * bf16 source) and reads back as that value, with no scale.
 * kind: 0 = E4M3 bytes (scaled), 1 = bf16 (unscaled). */
static double kvo_cache_value(const void *cache, int kind, int64_t idx, float scale)
{
    if (kind == 0)
        return (double)scale * kvo_e4m3_decode(((const uint8_t *)cache)[idx]);
    return (double)kvo_bf16_to_f32(((const uint16_t *)cache)[idx]);
}

/* reshape_and_cache with a per-side cache kind (see kvo_cache_value). */
uint32_t kvo_reshape_and_cache_mixed(const void *key, const void *value, int src_dtype,
                                     int64_t num_tokens, void *key_cache, int k_kind,
                                     void *value_cache, int v_kind, int32_t num_blocks,
                                     int32_t block_size, int32_t n_kv, int32_t head_dim,
                                     const int64_t *slot_mapping, float k_scale, float v_scale)
{
    if ((k_kind == 0 && !kvo_scale_ok(k_scale)) || (v_kind == 0 && !kvo_scale_ok(v_scale)))
        return KVO_BAD_SCALE;
    uint32_t status = 0;
    const int64_t row = (int64_t)n_kv * head_dim;
    const int64_t num_slots = (int64_t)num_blocks * block_size;
    for (int64_t i = 0; i < num_tokens; ++i) {
        const int64_t slot = slot_mapping[i];
        if (slot == -1)
            continue;
        if (slot < 0 || slot >= num_slots) {
            status |= KVO_BAD_SLOT;
            continue;
        }
        for (int64_t e = 0; e < row; ++e) {
            const float kx = kvo_load_src(key, src_dtype, i * row + e);
            const float vx = kvo_load_src(value, src_dtype, i * row + e);
            if (k_kind == 0)
                ((uint8_t *)key_cache)[slot * row + e] = kvo_store_code(kx, k_scale);
            else
                ((uint16_t *)key_cache)[slot * row + e] = kvo_f32_to_bf16(kx);
            if (v_kind == 0)
                ((uint8_t *)value_cache)[slot * row + e] = kvo_store_code(vx, v_scale);
            else
                ((uint16_t *)value_cache)[slot * row + e] = kvo_f32_to_bf16(vx);
        }
    }
    return status;
}

/* Decode attention with a per-side cache kind; otherwise as kvo_paged_decode_attention. */
uint32_t kvo_paged_decode_attention_mixed(double *out, const uint16_t *query,
                                          const void *key_cache, int k_kind,
                                          const void *value_cache, int v_kind,
                                          const int32_t *block_tables, int32_t max_blocks_per_seq,
                                          const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
                                          int32_t n_kv, int32_t head_dim, int32_t block_size,
                                          int32_t num_blocks, double sm_scale, float k_scale,
                                          float v_scale)
{
    if ((k_kind == 0 && !kvo_scale_ok(k_scale)) || (v_kind == 0 && !kvo_scale_ok(v_scale)))
        return KVO_BAD_SCALE;
    if (sm_scale <= 0.0)
        sm_scale = 1.0 / sqrt((double)head_dim);
    uint32_t status = 0;
    const int32_t group = n_q / n_kv;
    const int64_t row = (int64_t)n_kv * head_dim;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t len = seq_lens[b];
        if (len > max_blocks_per_seq * block_size) {
            status |= KVO_BAD_BLOCK;
            len = max_blocks_per_seq * block_size;
        }
        if (len < 0)
            len = 0;
        const int32_t *bt = block_tables + (int64_t)b * max_blocks_per_seq;
        double *score = (double *)malloc(sizeof(double) * (size_t)(len > 0 ? len : 1));
        for (int32_t h = 0; h < n_q; ++h) {
            const int32_t kvh = h / group;
            const uint16_t *q = query + ((int64_t)b * n_q + h) * head_dim;
            double *o = out + ((int64_t)b * n_q + h) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d)
                o[d] = 0.0;
            if (len == 0)
                continue;
            double best = -INFINITY;
            for (int32_t t = 0; t < len; ++t) {
                const int32_t phys = bt[t / block_size];
                if (phys < 0 || phys >= num_blocks) {  /* token left out, flagged */
                    status |= KVO_BAD_BLOCK;
                    score[t] = -INFINITY;
                    continue;
                }
                const int64_t base = ((int64_t)phys * block_size + t % block_size) * row +
                                     (int64_t)kvh * head_dim;
                double dot = 0.0;
                for (int32_t d = 0; d < head_dim; ++d)
                    dot += (double)kvo_bf16_to_f32(q[d]) * kvo_cache_value(key_cache, k_kind, base + d, k_scale);
                score[t] = sm_scale * dot;
                if (score[t] > best)
                    best = score[t];
            }
            double denom = 0.0;
            for (int32_t t = 0; t < len; ++t) {
                score[t] = exp(score[t] - best);
                denom += score[t];
            }
            for (int32_t t = 0; t < len; ++t) {
                if (score[t] == 0.0)
                    continue;
                const int64_t base = ((int64_t)bt[t / block_size] * block_size + t % block_size) * row +
                                     (int64_t)kvh * head_dim;
                const double p = score[t] / denom;
                for (int32_t d = 0; d < head_dim; ++d)
                    o[d] += p * kvo_cache_value(value_cache, v_kind, base + d, v_scale);
            }
        }
        free(score);
    }
    return status;
}

/* Whole-batch decode attention: out is [num_seqs][n_q][head_dim] doubles,
 * query is [num_seqs][n_q][head_dim] bf16, block_tables is
 * [num_seqs][max_blocks_per_seq] int32.  sm_scale <= 0 selects
 * 1/sqrt(head_dim) ([P1] tests/test-fp8.cpp, 1.0f/sqrtf(head_size)). */
uint32_t kvo_paged_decode_attention(double *out, const uint16_t *query, const uint8_t *key_cache,
                                    const uint8_t *value_cache, const int32_t *block_tables,
                                    int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                    int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim,
                                    int32_t block_size, int32_t num_blocks, double sm_scale,
                                    float k_scale, float v_scale)
{
    uint32_t status = 0;
    if (!kvo_scale_ok(k_scale) || !kvo_scale_ok(v_scale))
        return KVO_BAD_SCALE;
    if (sm_scale <= 0.0)
        sm_scale = 1.0 / sqrt((double)head_dim);
    const int32_t group = n_q / n_kv;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t len = seq_lens[b];
        if (len > max_blocks_per_seq * block_size) {
            status |= KVO_BAD_BLOCK;
            len = max_blocks_per_seq * block_size;
        }
        for (int32_t h = 0; h < n_q; ++h) {
            status |= kvo_decode_one(out + ((int64_t)b * n_q + h) * head_dim,
                                     query + ((int64_t)b * n_q + h) * head_dim, key_cache,
                                     value_cache, block_tables + (int64_t)b * max_blocks_per_seq,
                                     len, n_kv, h / group, head_dim, block_size, num_blocks,
                                     sm_scale, k_scale, v_scale);
        }
    }
    return status;
}

/* Multi-query (causal) paged attention: sequence b holds seq_lens[b] cached tokens, the
 * last n_b = query_start_loc[b+1] - query_start_loc[b] of which are new; its query token
 * j (0 <= j < n_b) sits at position p = seq_lens[b] - n_b + j and attends to the cached
 * tokens t <= p.  [P1] tests/test-fp8.cpp check_fp8_attention: a batch of 4 tokens,
 * each attending to every past token up to and including itself (past <= token).
 * query and out are [total_q][n_q][head_dim] with sequence b's rows starting at
 * query_start_loc[b].  n_b > seq_lens[b] flags KVO_BAD_BLOCK (positions below 0 attend to
 * nothing and give zeros). */
uint32_t kvo_paged_attention_multi(double *out, const uint16_t *query,
                                   const int32_t *query_start_loc, const uint8_t *key_cache,
                                   const uint8_t *value_cache, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                   int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim,
                                   int32_t block_size, int32_t num_blocks, double sm_scale,
                                   float k_scale, float v_scale)
{
    uint32_t status = 0;
    if (!kvo_scale_ok(k_scale) || !kvo_scale_ok(v_scale))
        return KVO_BAD_SCALE;
    if (sm_scale <= 0.0)
        sm_scale = 1.0 / sqrt((double)head_dim);
    const int32_t group = n_q / n_kv;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t len = seq_lens[b];
        if (len > max_blocks_per_seq * block_size) {
            status |= KVO_BAD_BLOCK;
            len = max_blocks_per_seq * block_size;
        }
        const int32_t q0 = query_start_loc[b];
        const int32_t nb = query_start_loc[b + 1] - q0;
        if (nb > len)
            status |= KVO_BAD_BLOCK;
        for (int32_t j = 0; j < nb; ++j) {
            const int32_t p = len - nb + j;  /* attends to tokens 0..p */
            for (int32_t h = 0; h < n_q; ++h) {
                const int64_t row = ((int64_t)(q0 + j) * n_q + h) * head_dim;
                status |= kvo_decode_one(out + row, query + row, key_cache, value_cache,
                                         block_tables + (int64_t)b * max_blocks_per_seq,
                                         p + 1 > 0 ? p + 1 : 0, n_kv, h / group, head_dim,
                                         block_size, num_blocks, sm_scale, k_scale, v_scale);
            }
        }
    }
    return status;
}

/* Multi-query (causal) attention with a per-side cache kind: the two forms above put
 * together.  [P1] tests/test-fp8.cpp check_fp8_attention runs its batch of new tokens
 * (each attending to every past token up to itself) over a cache with K only, V only or
 * both in FP8, the other side at 16 bits and unscaled.  Sequence b's query token j sits at
 * position p = len - n_b + j and its output is the single-query decode over the cache
 * prefix 0..p, so each row is kvo_paged_decode_attention_mixed of that one query with
 * sequence length p + 1 (no token past p is visible). */
uint32_t kvo_paged_attention_multi_mixed(double *out, const uint16_t *query,
                                         const int32_t *query_start_loc, const void *key_cache,
                                         int k_kind, const void *value_cache, int v_kind,
                                         const int32_t *block_tables, int32_t max_blocks_per_seq,
                                         const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
                                         int32_t n_kv, int32_t head_dim, int32_t block_size,
                                         int32_t num_blocks, double sm_scale, float k_scale,
                                         float v_scale)
{
    if ((k_kind == 0 && !kvo_scale_ok(k_scale)) || (v_kind == 0 && !kvo_scale_ok(v_scale)))
        return KVO_BAD_SCALE;
    uint32_t status = 0;
    for (int32_t b = 0; b < num_seqs; ++b) {
        int32_t len = seq_lens[b];
        if (len > max_blocks_per_seq * block_size) {
            status |= KVO_BAD_BLOCK;
            len = max_blocks_per_seq * block_size;
        }
        const int32_t q0 = query_start_loc[b];
        const int32_t nb = query_start_loc[b + 1] - q0;
        if (nb > len)
            status |= KVO_BAD_BLOCK;
        for (int32_t j = 0; j < nb; ++j) {
            const int32_t p = len - nb + j;  /* attends to tokens 0..p */
            const int32_t visible = p + 1 > 0 ? p + 1 : 0;
            const int64_t row = (int64_t)(q0 + j) * n_q * head_dim;
            status |= kvo_paged_decode_attention_mixed(
                out + row, query + row, key_cache, k_kind, value_cache, v_kind,
                block_tables + (int64_t)b * max_blocks_per_seq, max_blocks_per_seq, &visible, 1,
                n_q, n_kv, head_dim, block_size, num_blocks, sm_scale, k_scale, v_scale);
        }
    }
    return status;
}

/* Attention for a chosen list of (sequence, q head) pairs only, for sampled
 * checks at full size: pairs holds n_pairs (seq, head) int32 pairs and out is
 * [n_pairs][head_dim]. */
uint32_t kvo_paged_decode_attention_pairs(double *out, const int32_t *pairs, int32_t n_pairs,
                                          const uint16_t *query, const uint8_t *key_cache,
                                          const uint8_t *value_cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                          int32_t n_q, int32_t n_kv, int32_t head_dim,
                                          int32_t block_size, int32_t num_blocks, double sm_scale,
                                          float k_scale, float v_scale)
{
    uint32_t status = 0;
    if (!kvo_scale_ok(k_scale) || !kvo_scale_ok(v_scale))
        return KVO_BAD_SCALE;
    if (sm_scale <= 0.0)
        sm_scale = 1.0 / sqrt((double)head_dim);
    const int32_t group = n_q / n_kv;
    for (int32_t i = 0; i < n_pairs; ++i) {
        const int32_t b = pairs[2 * i];
        const int32_t h = pairs[2 * i + 1];
        int32_t len = seq_lens[b];
        if (len > max_blocks_per_seq * block_size) {
            status |= KVO_BAD_BLOCK;
            len = max_blocks_per_seq * block_size;
        }
        status |= kvo_decode_one(out + (int64_t)i * head_dim,
                                 query + ((int64_t)b * n_q + h) * head_dim, key_cache, value_cache,
                                 block_tables + (int64_t)b * max_blocks_per_seq, len, n_kv,
                                 h / group, head_dim, block_size, num_blocks, sm_scale, k_scale,
                                 v_scale);
    }
    return status;
}
