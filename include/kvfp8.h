/*
 * kvfp8 -- FP8 (OCP E4M3) paged KV cache for GB300 (sm_103a): C ABI.
 *
 * Three operations, all enqueued on a caller-supplied CUDA stream:
 *   kvfp8_reshape_and_cache       bf16/f32 K,V rows -> divide by a per-layer scalar
 *                                 scale -> E4M3 (RNE, saturating at +-448) -> scatter
 *                                 into paged blocks at one byte per element
 *   kvfp8_paged_decode_attention  one query per sequence reads the FP8 cache through
 *                                 block tables, dequantizes in registers by the same
 *                                 scales, and computes softmax(q.K^T * s) V with GQA
 *   kvfp8_dequant                 bytes -> scale * value, for the rope-shift path
 *                                 (dequantize, rotate, requantize)
 *
 * Sources, by page title and section:
 *   [P1] llama.cpp commit 202c1a229 "llama : Add FP8 KV-cache support (#28392)"
 *   [P2] llama.cpp compare osimons/ocp_fp8_kv (ggml-impl.h: the E4M3 codec)
 *   [P3] vllm.cpp PR #1641 "feat(KV-FP8): W3 -- half-sized KV blocks the runner
 *        actually serves, and a default scale that knows it was declared"
 *
 * Conventions common to every call
 *   - Every pointer argument named "device" must be device memory of the current
 *     device, 16-byte aligned (int64 slot mappings: 8-byte; int32 block tables and
 *     sequence lengths: 4-byte).  The caller owns all memory, including workspaces;
 *     the library allocates nothing and never synchronizes.
 *   - Host-checkable errors (null pointers, shapes, dtypes, alignment, workspace
 *     size) are returned before anything is enqueued; nothing is written then.
 *   - Errors only the device can see (a scale that is zero or not finite, a slot or
 *     block id out of range) skip the offending element/row/token and OR a bit into
 *     the optional device word *status (KVFP8_DEV_*).  Nothing traps or spins
 *     forever; the caller reads *status when it wants to.
 *   - Launch failures are returned as KVFP8_ERR_CUDA.
 *   - Cache layout (shared by K and V, which are separate arrays):
 *       uint8 [num_blocks][block_size][n_kv][head_dim]
 *     so token slot s = block * block_size + offset owns the n_kv*head_dim bytes at
 *     s * n_kv * head_dim.  One byte per element: a block is exactly half the bytes
 *     of the same block in bf16 ([P3] section "Three surfaces that no gate
 *     reached", KVBytesPerBlock halved).
 */
#ifndef KVFP8_H
#define KVFP8_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define KVFP8_API __attribute__((visibility("default")))
#else
#define KVFP8_API
#endif

/* Same type as cudaStream_t; 0 is the legacy default stream. */
typedef struct CUstream_st *kvfp8_stream_t;

typedef enum {
    KVFP8_OK = 0,
    KVFP8_ERR_NULL = 1,        /* a required pointer is null */
    KVFP8_ERR_SHAPE = 2,       /* a size or shape is out of the supported range */
    KVFP8_ERR_DTYPE = 3,       /* unsupported dtype code */
    KVFP8_ERR_SCALE = 4,       /* a host-known scale is zero or not finite */
    KVFP8_ERR_ALIGN = 5,       /* a pointer or stride breaks the 16-byte rule */
    KVFP8_ERR_WORKSPACE = 6,   /* workspace_bytes below kvfp8_paged_decode_workspace_size */
    KVFP8_ERR_CUDA = 7,        /* a CUDA launch or driver call failed */
    KVFP8_ERR_UNSUPPORTED = 8  /* a valid shape this build has no kernel for */
} kvfp8_status;

typedef enum {
    KVFP8_BF16 = 0,
    KVFP8_F32 = 1
} kvfp8_dtype;

/* Element type of one side's cache in the mixed-dtype calls. */
typedef enum {
    KVFP8_CACHE_E4M3 = 0, /* uint8 E4M3 codes, dequantized by that side's scale */
    KVFP8_CACHE_BF16 = 1  /* bf16 values, no scale */
} kvfp8_cache_dtype;

/* Bits ORed into the optional device status word. */
#define KVFP8_DEV_BAD_SCALE (1u << 0) /* a device scale was zero or not finite: nothing written */
#define KVFP8_DEV_BAD_SLOT  (1u << 1) /* a slot outside [-1, num_blocks*block_size): row skipped */
#define KVFP8_DEV_BAD_BLOCK (1u << 2) /* a block id outside [0, num_blocks), or a seq_len above
                                         max_blocks_per_seq*block_size (clamped) or negative */
#define KVFP8_DEV_TIMEOUT   (1u << 3) /* a bounded wait inside a kernel gave up; output invalid */

/*
 * Quantize K and V rows and scatter them into the paged caches.
 *
 * Defined by: [P1] llama-graph.cpp build_attn_scale_kv_inputs (K/s_k and V/s_v via
 * ggml_div before the cache copy) and llama-kv-cache.cpp cpy_k/cpy_v (rows stored at a
 * per-token I64 destination index); [P2] ggml-impl.h ggml_fp32_to_f8_e4m3 (the encode);
 * [P3] vt::ReshapeAndCacheFp8 (one shared source dtype for K and V).
 *
 * For every token i with slot = slot_mapping[i] != -1 and every (h, d):
 *   key_cache  [slot][h][d] = E4M3( fp32(key  [i*key_stride   + h*head_dim + d]) / k_scale )
 *   value_cache[slot][h][d] = E4M3( fp32(value[i*value_stride + h*head_dim + d]) / v_scale )
 * where "/" is the IEEE float quotient (correctly rounded) and E4M3 rounds to nearest
 * even, maps |y| >= 448 and +-inf to +-448 (0x7E/0xFE), keeps -0 as 0x80, and maps a NaN
 * element to sign(element)|0x7F.  Bytes of slots not written keep their contents.
 *
 * key, value        device, src_dtype elements; token i's row starts at i*stride elements
 * src_dtype         KVFP8_BF16 or KVFP8_F32, shared by key and value
 * key_stride,
 * value_stride      row strides in elements (>= n_kv*head_dim; stride*elem_size % 16 == 0)
 * num_tokens        >= 0 (0 enqueues nothing)
 * key_cache,
 * value_cache       device uint8 caches, layout above
 * num_blocks        >= 1;  block_size in [1, 1024];  n_kv >= 1;  head_dim >= 1 with
 *                   n_kv*head_dim a multiple of 8
 * slot_mapping      device int64 [num_tokens]; -1 = padding token (skipped)
 * k_scale, v_scale  device scalars of scale_dtype (bf16 is widened exactly), or NULL for
 *                   a scale of 1.  Must be finite and nonzero; negative is allowed.
 * status            device uint32 or NULL
 */
KVFP8_API kvfp8_status kvfp8_reshape_and_cache(const void *key, const void *value, kvfp8_dtype src_dtype,
                                     int64_t key_stride, int64_t value_stride, int64_t num_tokens,
                                     uint8_t *key_cache, uint8_t *value_cache, int32_t num_blocks,
                                     int32_t block_size, int32_t n_kv, int32_t head_dim,
                                     const int64_t *slot_mapping, const void *k_scale,
                                     const void *v_scale, kvfp8_dtype scale_dtype,
                                     uint32_t *status, kvfp8_stream_t stream);

/*
 * kvfp8_reshape_and_cache with rotary position embedding applied to K first, in the same
 * pass (V is stored unrotated).
 *
 * Defined by: [P1] llama-graph.cpp build_attn ("rope fusion which directly writes into
 * k-v cache"); the rotation itself is the model's, so its form is fixed here: for token i
 * with p = positions[i], table row T = cos_sin_cache[p] (cos in T[0..rot/2), sin in
 * T[rot/2..rot)), every pair (a, b) of the first rot_dim dims of each K head becomes
 *   a' = a*cos - b*sin,   b' = a*sin + b*cos      (pair j uses cos/sin entry j)
 * with each product and sum rounded to float in that order (no fused multiply-add).
 * is_neox != 0: dim j pairs with j + rot_dim/2 (GPT-NeoX); 0: dim 2j with 2j+1 (GPT-J).
 * Dims >= rot_dim pass through.  Then K and V are stored exactly as by
 * kvfp8_reshape_and_cache.
 *
 * Arguments as kvfp8_reshape_and_cache, plus:
 * positions       device int64 [num_tokens]; a position outside [0, max_position) skips the
 *                 token and sets KVFP8_DEV_BAD_SLOT
 * cos_sin_cache   device float32 [max_position][rot_dim], 16-byte aligned
 * rot_dim         a power of two in [16, head_dim]
 * head_dim must be 64, 128 or 256; rows of more than 2048 elements (n_kv*head_dim) return
 * KVFP8_ERR_UNSUPPORTED.
 */
KVFP8_API kvfp8_status kvfp8_rope_reshape_and_cache(
    const void *key, const void *value, kvfp8_dtype src_dtype, int64_t key_stride,
    int64_t value_stride, int64_t num_tokens, uint8_t *key_cache, uint8_t *value_cache,
    int32_t num_blocks, int32_t block_size, int32_t n_kv, int32_t head_dim,
    const int64_t *slot_mapping, const int64_t *positions, const float *cos_sin_cache,
    int64_t max_position, int32_t rot_dim, int32_t is_neox, const void *k_scale,
    const void *v_scale, kvfp8_dtype scale_dtype, uint32_t *status, kvfp8_stream_t stream);

/*
 * Workspace bytes kvfp8_paged_decode_attention needs for this batch shape (split-KV
 * partial results and the per-call chunk plan).  Pure host arithmetic.
 */
KVFP8_API size_t kvfp8_paged_decode_workspace_size(int32_t num_seqs, int32_t n_q, int32_t head_dim);

/*
 * Single-query (decode) paged attention over the FP8 cache.
 *
 * Defined by: [P1] tests/test-fp8.cpp check_fp8_attention (softmax(q.k/sqrt(d)) V over
 * all past tokens, on K and V rounded through the cache format) and llama-graph.cpp
 * build_attn_scale_kv_inputs / build_attn_scale_kv_output ((Q*s_k).(K/s_k) = Q.K and
 * P*(V/s_v)*s_v = P*V: dequantizing by the same scales); [P2] ggml-impl.h
 * ggml_f8_e4m3_to_fp32 (the decode).
 *
 * For every sequence b and query head h, with G = n_q / n_kv, kv = h / G,
 * L = seq_lens[b] and token t < L stored in physical block block_tables[b][t / block_size]
 * at row t % block_size:
 *   s_t = sm_scale * k_scale * sum_d q[b][h][d] * E4M3dec(K[t][kv][d])
 *   out[b][h][d] = v_scale * sum_t softmax(s)_t * E4M3dec(V[t][kv][d])   (bf16)
 * L == 0 gives a zero row.  Accumulation is fp32; q and the decoded cache enter the
 * tensor cores as fp16 (exact for the cache; q must lie within fp16 range).
 *
 * out               device bf16 [num_seqs][n_q][head_dim]
 * query             device bf16 [num_seqs][n_q][head_dim]
 * key_cache,
 * value_cache       device uint8 caches, layout above
 * block_tables      device int32 [num_seqs][max_blocks_per_seq]
 * seq_lens          device int32 [num_seqs]
 * num_seqs >= 0; n_q % n_kv == 0; head_dim in {64, 128, 256}; block_size in
 * {8, 16, 32, 64, 128, 256}; num_blocks*block_size < 2^31.  Any n_kv: a CTA serves a
 * group of at most 8 kv heads (4 when a kv head has 9-16 score columns at head_dim 128 on
 * an FP8 cache; the largest divisor of n_kv up to that), the groups side by side.  Groups of up to 16 query heads per kv head (8 at head_dim 256) run on the
 * split-KV kernel; larger ones, up to 128, on the tensor-core kernel of
 * kvfp8_paged_attention_multi; more return KVFP8_ERR_UNSUPPORTED.
 * sm_scale          <= 0 selects 1/sqrt(head_dim)
 * k_scale, v_scale  device scalars of scale_dtype, or NULL for 1
 * workspace         device, >= kvfp8_paged_decode_workspace_size(...) bytes, contents
 *                   need no initialization; calls that overlap on the GPU must not share it
 * status            device uint32 or NULL
 */
KVFP8_API kvfp8_status kvfp8_paged_decode_attention(void *out, const void *query, const uint8_t *key_cache,
                                          const uint8_t *value_cache, const int32_t *block_tables,
                                          int32_t max_blocks_per_seq, const int32_t *seq_lens,
                                          int32_t num_seqs, int32_t n_q, int32_t n_kv,
                                          int32_t head_dim, int32_t block_size,
                                          int32_t num_blocks, float sm_scale,
                                          const void *k_scale, const void *v_scale,
                                          kvfp8_dtype scale_dtype, void *workspace,
                                          size_t workspace_bytes, uint32_t *status,
                                          kvfp8_stream_t stream);

/*
 * Size in bytes of the fixed device scratch array that
 * kvfp8_paged_decode_attention_noalloc uses in place of a caller workspace (32 MiB).
 */
#define KVFP8_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

/*
 * kvfp8_paged_decode_attention for callers that cannot allocate device memory: same
 * arguments, outputs and errors, minus the workspace.  The source pages have no
 * counterpart of this call; it exists for callers that cannot call cudaMalloc (a
 * plug-in whose host runtime owns every device allocation, a serving loop that must not
 * allocate once it runs, a caller with no allocator of its own).
 *
 * The split-KV scratch is a fixed device array of KVFP8_NOALLOC_SCRATCH_BYTES inside this
 * library, held by every GPU that loads the library until the process exits.  A batch
 * whose kvfp8_paged_decode_workspace_size exceeds it returns KVFP8_ERR_WORKSPACE before
 * anything is enqueued.  The call allocates nothing.  The first call on each device looks
 * up the array's device address (with that device current); make that first call
 * before any stream capture.  All calls share the array, which keeps the last call's
 * contents (nothing in it needs to start at zero); calls that overlap on the GPU race on
 * it, so order them on one stream or serialize them.
 */
KVFP8_API kvfp8_status kvfp8_paged_decode_attention_noalloc(
    void *out, const void *query, const uint8_t *key_cache, const uint8_t *value_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
    int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float sm_scale, const void *k_scale, const void *v_scale,
    kvfp8_dtype scale_dtype, uint32_t *status, kvfp8_stream_t stream);

/*
 * Multi-query (causal) paged attention over the FP8 cache: several new tokens per
 * sequence, each attending to the cached tokens up to and including itself.
 *
 * Defined by: [P1] tests/test-fp8.cpp check_fp8_attention (a batch of new tokens, each
 * attending to every past token up to itself, on K/V rounded through the cache format);
 * the arithmetic is that of kvfp8_paged_decode_attention.
 *
 * Sequence b holds L = seq_lens[b] cached tokens (the new tokens already written), the last
 * n_b = query_start_loc[b+1] - query_start_loc[b] of them new.  Its query token j
 * (0 <= j < n_b) is row query_start_loc[b] + j of query and out, sits at position
 * p = L - n_b + j, and attends to tokens t <= p:
 *   out[row][h] = v_scale * sum_{t<=p} softmax_t(sm_scale*k_scale*q[row][h].dec(K_t)) dec(V_t)
 * n_b = 1 for every sequence is kvfp8_paged_decode_attention.
 *
 * Two kernels serve the call.  With max_query_len * (n_q / n_kv) <= 16 score columns per
 * kv head (<= 8 at head_dim 256) the split-KV decode kernel runs and needs the workspace
 * below.  Every other shape (long query chunks,
 * prefill) runs on the tensor cores (tcgen05, accumulators in tensor memory), one CTA per
 * 128 (query token, head) rows of a kv head (256 rows, as two tiles sharing each K/V tile,
 * when there are more than 128 rows at head_dim 64 or 128), with no workspace; it needs
 * n_q / n_kv <= 128 and num_seqs * n_kv * ceil(max_query_len * (n_q / n_kv) / 128) < 2^31
 * CTAs, else KVFP8_ERR_UNSUPPORTED.
 *
 * out, query        device bf16 [num_query_rows][n_q][head_dim]
 * query_start_loc   device int32 [num_seqs + 1], non-decreasing; a sequence whose rows
 *                   fall outside [0, num_query_rows) or number more than max_query_len is
 *                   skipped and sets KVFP8_DEV_BAD_BLOCK; n_b > L also sets it (positions
 *                   below zero attend to nothing and give zero rows)
 * max_query_len     >= 1
 * workspace         >= kvfp8_paged_attention_multi_workspace_size(...) bytes (may be NULL
 *                   when that is 0)
 * Everything else as kvfp8_paged_decode_attention.
 */
/*
 * Workspace bytes kvfp8_paged_attention_multi needs for this shape: the split-KV partials
 * (kvfp8_paged_decode_workspace_size(num_seqs, n_q * max_query_len, head_dim)) when the
 * decode kernel serves it, 0 when the tensor-core kernel does.  Pure host arithmetic.
 */
KVFP8_API size_t kvfp8_paged_attention_multi_workspace_size(int32_t num_seqs, int32_t n_q,
                                                            int32_t n_kv, int32_t head_dim,
                                                            int32_t max_query_len);

KVFP8_API kvfp8_status kvfp8_paged_attention_multi(
    void *out, const void *query, const int32_t *query_start_loc, int32_t num_query_rows,
    int32_t max_query_len, const uint8_t *key_cache, const uint8_t *value_cache,
    const int32_t *block_tables, int32_t max_blocks_per_seq, const int32_t *seq_lens,
    int32_t num_seqs, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t block_size,
    int32_t num_blocks, float sm_scale, const void *k_scale, const void *v_scale,
    kvfp8_dtype scale_dtype, void *workspace, size_t workspace_bytes, uint32_t *status,
    kvfp8_stream_t stream);

/*
 * Mixed cache dtypes: FP8 on one side only.
 *
 * Defined by: [P1] tests/test-fp8.cpp check_fp8_attention, which quantizes K only, V only
 * or both (type_k / type_v F8_E4M3 or F16, the FP8 side with its own scale, the other
 * unscaled), and tests/test-backend-ops.cpp, which adds the F8/F16 cache mixes.  Here the
 * 16-bit side is bf16.
 *
 * A KVFP8_CACHE_BF16 side's cache is bf16 [num_blocks][block_size][n_kv][head_dim] (two
 * bytes per element, so slot s owns the 2*n_kv*head_dim bytes at 2*s*n_kv*head_dim); its
 * scale pointer is ignored (may be NULL) and never checked.  The KVFP8_CACHE_E4M3 side is
 * exactly as in the all-FP8 calls.
 *
 * kvfp8_reshape_and_cache_mixed: as kvfp8_reshape_and_cache; a bf16 side stores the
 * source value rounded to bf16 (round to nearest even; a bf16 source is copied as it is;
 * a NaN stays a NaN, its payload unspecified).  n_kv*head_dim <= 2048, else
 * KVFP8_ERR_UNSUPPORTED.
 */
KVFP8_API kvfp8_status kvfp8_reshape_and_cache_mixed(
    const void *key, const void *value, kvfp8_dtype src_dtype, int64_t key_stride,
    int64_t value_stride, int64_t num_tokens, void *key_cache, kvfp8_cache_dtype k_cache_dtype,
    void *value_cache, kvfp8_cache_dtype v_cache_dtype, int32_t num_blocks, int32_t block_size,
    int32_t n_kv, int32_t head_dim, const int64_t *slot_mapping, const void *k_scale,
    const void *v_scale, kvfp8_dtype scale_dtype, uint32_t *status, kvfp8_stream_t stream);

/*
 * kvfp8_paged_decode_attention with a per-side cache dtype:
 *   s_t = sm_scale * sum_d q[b][h][d] * Kval(t, kv, d),  out = sum_t softmax(s)_t Vval(t, kv, d)
 * where an E4M3 side's value is scale * E4M3dec(byte) and a bf16 side's is the stored bf16.
 * A bf16 K enters the tensor cores against bf16 q (exact products); a bf16 V against the
 * probabilities split into two bf16 parts (16 significant bits).
 * This build: exactly one side bf16 (both E4M3 is kvfp8_paged_decode_attention; both
 * bf16 returns KVFP8_ERR_UNSUPPORTED); n_q/n_kv <= 16 at head_dim 64 and 128, <= 8 at 256
 * (larger groups return KVFP8_ERR_UNSUPPORTED).
 * Workspace: kvfp8_paged_decode_workspace_size(num_seqs, n_q, head_dim).  Everything else
 * as kvfp8_paged_decode_attention.
 */
KVFP8_API kvfp8_status kvfp8_paged_decode_attention_mixed(
    void *out, const void *query, const void *key_cache, kvfp8_cache_dtype k_cache_dtype,
    const void *value_cache, kvfp8_cache_dtype v_cache_dtype, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
    int32_t n_kv, int32_t head_dim, int32_t block_size, int32_t num_blocks, float sm_scale,
    const void *k_scale, const void *v_scale, kvfp8_dtype scale_dtype, void *workspace,
    size_t workspace_bytes, uint32_t *status, kvfp8_stream_t stream);

/*
 * kvfp8_paged_attention_multi with a per-side cache dtype: causal multi-query attention
 * (each new token attends to the cached tokens up to and including its own position) where
 * an E4M3 side reads as scale * E4M3dec(byte) and a bf16 side as the stored bf16, unscaled.
 *
 * Defined by: [P1] tests/test-fp8.cpp check_fp8_attention, whose batch of new tokens runs
 * over a cache with K only, V only or both in FP8 (the other side at 16 bits, unscaled),
 * and tests/test-backend-ops.cpp (the F8/F16 cache mixes with several query rows).
 *
 * Both sides E4M3 is kvfp8_paged_attention_multi (and is passed to it).  With one bf16 side
 * this build runs the split-KV kernel only: max_query_len * (n_q / n_kv) <= 16 score
 * columns per kv head (<= 8 at head_dim 256); longer query chunks return
 * KVFP8_ERR_UNSUPPORTED, as do both sides bf16.  Workspace:
 * kvfp8_paged_attention_multi_workspace_size(num_seqs, n_q, n_kv, head_dim, max_query_len).
 * Cache layouts as kvfp8_paged_decode_attention_mixed; everything else as
 * kvfp8_paged_attention_multi.
 */
KVFP8_API kvfp8_status kvfp8_paged_attention_multi_mixed(
    void *out, const void *query, const int32_t *query_start_loc, int32_t num_query_rows,
    int32_t max_query_len, const void *key_cache, kvfp8_cache_dtype k_cache_dtype,
    const void *value_cache, kvfp8_cache_dtype v_cache_dtype, const int32_t *block_tables,
    int32_t max_blocks_per_seq, const int32_t *seq_lens, int32_t num_seqs, int32_t n_q,
    int32_t n_kv, int32_t head_dim, int32_t block_size, int32_t num_blocks, float sm_scale,
    const void *k_scale, const void *v_scale, kvfp8_dtype scale_dtype, void *workspace,
    size_t workspace_bytes, uint32_t *status, kvfp8_stream_t stream);

/*
 * Dequantize n E4M3 bytes: dst[i] = scale * E4M3dec(src[i]), product in fp32, then
 * rounded to dst_dtype (bf16: round to nearest even).  NaN codes give NaN.
 *
 * Defined by: [P1] llama-kv-cache.cpp build_rope_shift (F8 joins the dequantize ->
 * rope -> requantize path) and tests/test-fp8.cpp check_fp8_context_shift (stored bytes
 * after a shift equal quantize(rope(decode(bytes)))).  Requantize with
 * kvfp8_reshape_and_cache.  Rope is linear, so the shift path may run scale-free
 * (scale = NULL) as long as dequant and requant agree.
 *
 * dst    device, dst_dtype [n];  src device uint8 [n];  n >= 0
 * scale  device scalar of scale_dtype, or NULL for 1
 */
KVFP8_API kvfp8_status kvfp8_dequant(void *dst, kvfp8_dtype dst_dtype, const uint8_t *src, int64_t n,
                           const void *scale, kvfp8_dtype scale_dtype, kvfp8_stream_t stream);

/*
 * Host-side scale check: KVFP8_OK if s is finite and nonzero, else KVFP8_ERR_SCALE.
 * [P1] llama-context.cpp llama_init_from_model ("must be finite and nonzero").
 */
KVFP8_API kvfp8_status kvfp8_check_scale_host(float s);

/* Static, human-readable name of a status code. */
KVFP8_API const char *kvfp8_status_string(kvfp8_status s);

#ifdef __cplusplus
}
#endif

#endif /* KVFP8_H */
