// Causal multi-query attention over the FP8 (E4M3) cache for long query chunks (prefill),
// sm_103a tensor cores (tcgen05) with accumulators in tensor memory.
//
// What it computes is kvfp8_paged_attention_multi (llama.cpp "llama : Add FP8 KV-cache
// support (#28392)", tests/test-fp8.cpp check_fp8_attention: a batch of new tokens, each
// attending to every cached token up to its own position, on K/V rounded through the cache
// format).  The decode kernel covers up to 16 (query token, head) score columns per kv
// head; past that the rows form a real M dimension and the contraction is dense, so:
//
// Two kernels: prefill_kernel below (one row tile of 128 per CTA), and prefill2_kernel
// further down (two row tiles per CTA sharing each converted K/V tile), which takes the
// long chunks at head_dim 64 and 128.
//
//  * Work unit: one CTA per (sequence, kv head, tile of 128 score rows).  A row is a
//    (query token j, head g of the kv head's group) pair, row = j*G + g, so all rows of a
//    tile share one K/V stream.  Keys are visited in tiles of 64 up to the tile's last
//    causal position, each row tile starting at its own key tile (the online softmax takes
//    the keys in any order).  The grid runs kv head fastest, then row tile, then sequence.
//  * Warp-specialized, every stage overlapped with the others (14 warps):
//      - warp 13 issues the TMA loads of the FP8 K/V tiles (per-head-segment boxes of the
//        cache map, one lane per box) into a four-stage ring;
//      - warps 4-11 convert the tile's q rows bf16 -> f16 once, and each K tile
//        e4m3 -> f16, into the K-major 128-byte-swizzled operand layout, and each V tile
//        e4m3 -> f16 transposed (V^T: head dims as rows, keys along K), so both products
//        take K-major operands; K, V^T and the score buffers are triple-buffered;
//      - one thread of warp 12 issues S(i) = Q.K(i)^T (tcgen05.mma kind::f16, M = 128,
//        N = 64, fp32 in tensor memory) and then O += P(i-1).V(i-1) (A = P from tensor
//        memory, B = V^T from shared memory), so the next scores are computed while the
//        softmax works on the current ones.  Up to head_dim 128 V^T carries a row of ones,
//        so the same product also sums each row of P;
//      - warps 0-3 (one TMEM lane quarter each, one score row per thread) read S, apply
//        the causal mask and the online softmax (log2 domain), and write P (f16) back over
//        S.  O is rescaled in TMEM only when a row's running maximum grows by more than
//        2^8 (P <= 2^8 stays well inside fp16); at the end they divide by the row sum,
//        apply v_scale and store bf16.
//  * All waits are bounded (mbarriers with a clock64 limit); a wait that runs out sets
//    KVFP8_DEV_TIMEOUT.  Tensor memory is always released before the CTA exits.
#include "paged_decode_kernel.cuh"

namespace kvfp8 {
namespace {

constexpr int kPfRows = 128;   // score rows per CTA (TMEM lanes)
constexpr int kPfKeys = 64;    // keys per tile

// ---------------------------------------------------------------- tcgen05 wrappers

__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
// D (TMEM) (+)= A (shared memory descriptor) x B (shared memory descriptor)
__device__ __forceinline__ void umma_ss(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d),
        "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// D (TMEM) (+)= A (TMEM) x B (shared memory descriptor)
__device__ __forceinline__ void umma_ts(uint32_t d, uint32_t a, uint64_t b, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d),
        "r"(a), "l"(b), "r"(idesc), "r"(accumulate)
        : "memory");
}
// arrive on the mbarrier once every tcgen05.mma this thread issued before has completed
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// four 8x8 b16 matrices stored transposed: lane t gives (rows 2(t%4), 2(t%4)+1; column t/4)
// of matrix j in r[j], and the address of row t%8 of matrix t/8
__device__ __forceinline__ void stsm_x4_t(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                          uint32_t r3) {
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1,%2,%3,%4};" ::"r"(addr),
                 "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// generic-proxy shared-memory writes become visible to the tensor core (async proxy)
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// Shared-memory matrix descriptor: K-major operand in the 128-byte swizzle layout (rows of
// 128 bytes, 16-byte chunks XOR-ed with row % 8, 8-row groups 1024 bytes apart).
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu)  // start address
           | (1ull << 16)                                 // leading byte offset (unused here)
           | (static_cast<uint64_t>(1024 >> 4) << 32)     // stride byte offset: 8 rows
           | (1ull << 46)                                 // descriptor version
           | (2ull << 61);                                // 128-byte swizzle
}
// The descriptor of an address off bytes (a multiple of 16) past one whose descriptor is d:
// the start-address field is (address >> 4) in 14 bits, and every shared-memory address of
// a CTA is below 2^18, so the field never carries into the next one.
__device__ __forceinline__ uint64_t desc_at(uint64_t d, uint32_t off) { return d + (off >> 4); }

// Instruction descriptor, kind::f16: f16 A and B, fp32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major block
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

// packed fp32 pairs (sm_100+ f32x2 arithmetic: two IEEE round-to-nearest operations)
__device__ __forceinline__ uint64_t pk2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t pk2u(uint32_t lo, uint32_t hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "r"(lo), "r"(hi));
    return r;
}
__device__ __forceinline__ float2 upk2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint64_t add_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t mul_f32x2(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
__device__ __forceinline__ float min3f(float a, float b, float c) {
    float r;
    asm("min.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}
// 2^x on an f16 pair (the tensor core takes P as f16)
__device__ __forceinline__ uint32_t ex2_f16x2(uint32_t x) {
    uint32_t r;
    asm("ex2.approx.f16x2 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}
__device__ __forceinline__ float f16lo_f32(uint32_t h) {
    float r;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(r) : "r"(h));
    return r;
}
__device__ __forceinline__ float f16hi_f32(uint32_t h) {
    float r;
    asm("{\n\t.reg .b16 l, u;\n\tmov.b32 {l, u}, %1;\n\tcvt.f32.f16 %0, u;\n\t}" : "=f"(r) : "r"(h));
    return r;
}
// the largest (kMax) or smallest of 64 scores, four independent chains of 3-input ops
template <bool kMax>
__device__ __forceinline__ float extreme64(const uint32_t (&s)[2][32]) {
    auto v = [&](int c) { return __uint_as_float(s[c >> 5][c & 31]); };
    auto op = [](float a, float b, float c) { return kMax ? max3f(a, b, c) : min3f(a, b, c); };
    float a0 = v(0), a1 = v(1), a2 = v(2), a3 = v(3);
#pragma unroll
    for (int c = 4; c < 60; c += 8) {
        a0 = op(a0, v(c), v(c + 1));
        a1 = op(a1, v(c + 2), v(c + 3));
        a2 = op(a2, v(c + 4), v(c + 5));
        a3 = op(a3, v(c + 6), v(c + 7));
    }
    a0 = op(a0, v(60), v(61));
    a1 = op(a1, v(62), v(63));
    return op(a0, a1, kMax ? fmaxf(a2, a3) : fminf(a2, a3));
}

struct PrefillArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *query;
    const int32_t *qsl;
    int32_t qmax, qrows;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t n_q, n_kv, group, block_size, num_blocks, max_len;
    float sm_scale;
    const void *k_scale;
    const void *v_scale;
    int32_t scale_dtype;
    uint32_t *status;
    int32_t box_rows;
    int32_t row_tiles;  // tiles of 128 score rows per (sequence, kv head)
};

// ---------------------------------------------------------------- work order
//
// The CTAs of the sequences with the most keys go first.  The hardware starts CTAs in index
// order as SMs free up, so giving the low indices to the longest sequences keeps one of them
// from starting last and running alone at the end (longest-processing-time-first list
// scheduling; with lengths log-uniform over 16..32768 tokens, as in a serving mix, index
// order leaves the last SMs busy ~20 % past the mean).  Sequences are ranked by a bucket of
// their length, four buckets per octave (lengths in one bucket differ by less than 19 %),
// longest bucket first, and by index within a bucket.

__device__ __forceinline__ int length_bucket(int len, int max_len) {
    const int l = min(max(len, 0), max_len);
    if (l == 0) return 0;
    const int b = 31 - __clz(l);                                     // floor(log2 l), 0..30
    const int frac = b >= 2 ? (l >> (b - 2)) & 3 : (l << (2 - b)) & 3;  // next two bits
    return 1 + 4 * b + frac;                                         // 1..124
}

// The sequence of rank u (0 = longest).  Every thread of the CTA calls it (it synchronizes
// the CTA); scratch is 168 words of this CTA's shared memory, free until it returns.
__device__ __forceinline__ int seq_of_rank(const int32_t *seq_lens, int num_seqs, int max_len, int u,
                           uint32_t *scratch) {
    if (num_seqs <= 1) return u;
    uint32_t *cnt = scratch;                      // [128] sequences per bucket
    // bucket of rank u, rank within it, the result, and whether the result is final
    volatile uint32_t *pick = scratch + 128;
    volatile uint32_t *wsum = scratch + 136;      // [32] per-warp counts of one round
    const int tid = threadIdx.x, nthr = blockDim.x, warp = tid >> 5, lane = tid & 31;
    const int nwarps = nthr >> 5;
    // bucket of sequence tid, kept for the histogram and the first round of the scan
    const int my_bucket = tid < num_seqs ? length_bucket(seq_lens[tid], max_len) : -1;
    if (num_seqs <= nthr) {  // lengths all in one bucket (a batch of equal lengths): index order
        const int b0 = length_bucket(seq_lens[0], max_len);
        if (__syncthreads_and(tid >= num_seqs || my_bucket == b0)) return u;
    }
    for (int b = tid; b < 128; b += nthr) cnt[b] = 0u;
    if (tid == 0) {  // (u < num_seqs always finds its bucket; index order otherwise)
        pick[0] = 0u;
        pick[1] = 0u;
        pick[2] = static_cast<uint32_t>(u);
        pick[3] = 0u;
    }
    __syncthreads();
    for (int s = tid; s < num_seqs; s += nthr)
        atomicAdd(&cnt[s == tid ? my_bucket : length_bucket(seq_lens[s], max_len)], 1u);
    __syncthreads();
    if (warp == 0) {
        // lane l holds buckets 127-4l .. 124-4l, so lanes run longest first
        uint32_t c[4], tot = 0;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            c[q] = cnt[127 - 4 * lane - q];
            tot += c[q];
        }
        uint32_t incl = tot;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += v;
        }
        uint32_t before = incl - tot;
        const uint32_t uu = static_cast<uint32_t>(u);
        if (uu >= before && uu < incl) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (uu < before + c[q]) {
                    pick[0] = static_cast<uint32_t>(127 - 4 * lane - q);
                    pick[1] = uu - before;
                    // every sequence in one bucket (a batch of equal lengths): index order
                    if (c[q] == static_cast<uint32_t>(num_seqs)) pick[3] = 1u;
                    break;
                }
                before += c[q];
            }
        }
    }
    __syncthreads();
    if (pick[3] != 0u) return u;
    const int B = static_cast<int>(pick[0]);
    const uint32_t k = pick[1];
    // the k-th sequence of bucket B in index order, nthr sequences a round
    uint32_t seen = 0;
    for (int s0 = 0; s0 < num_seqs; s0 += nthr) {
        const int s = s0 + tid;
        const int b = s0 == 0 ? my_bucket : (s < num_seqs ? length_bucket(seq_lens[s], max_len) : -1);
        const bool in = s < num_seqs && b == B;
        const uint32_t bal = __ballot_sync(0xFFFFFFFFu, in);
        if (lane == 0) wsum[warp] = static_cast<uint32_t>(__popc(bal));
        __syncthreads();
        uint32_t pre = seen, tot = 0;
        for (int w = 0; w < nwarps; ++w) {
            const uint32_t v = wsum[w];
            if (w < warp) pre += v;
            tot += v;
        }
        pre += static_cast<uint32_t>(__popc(bal & ((1u << lane) - 1u)));
        if (in && pre == k) pick[2] = static_cast<uint32_t>(s);
        seen += tot;
        __syncthreads();  // pick[2] is written; wsum may be reused
        if (seen > k) break;
    }
    return static_cast<int>(pick[2]);
}

// Shared-memory plan (byte offsets from a 1024-aligned base).  Q is converted once; K and
// V^T (f16) have NB buffers, and so do the scores in tensor memory; the FP8 staging ring has
// NS stages.  At head_dim 256 the f16 buffers fill the shared memory: NB = 2, NS = 1.
template <int HD>
struct PfSmem {
    static constexpr int kSeg = HD >= 128 ? 128 : 64;             // fp8 TMA box row (swizzle span)
    static constexpr int kSegs = HD / kSeg;
    static constexpr int kNB = HD >= 256 ? 2 : 3;                  // f16 K/V^T and S buffers
    static constexpr int kNS = HD >= 256 ? 1 : 4;                  // FP8 staging stages
    static constexpr int kQ = 0;                                   // Q f16: HD/64 blocks x 128 rows x 128 B
    static constexpr int kKBuf = HD * 128;                         // one K f16 buffer: HD/64 x 64 rows x 128 B
    // Up to head_dim 128, V^T carries 16 more rows: a row of ones then zeros, so the O
    // product also accumulates each score row's sum of P (column HD of O) in fp32.  At 256
    // there is no room (the product's N would pass 256 and shared memory would overflow):
    // the softmax warps sum P themselves.
    static constexpr bool kSumCol = HD <= 128;
    static constexpr int kVRows = HD + (kSumCol ? 16 : 0);
    static constexpr int kVBuf = kVRows * 128;                     // one V^T f16 buffer: rows x 128 B
    static constexpr int kK = kQ + HD * 256;
    static constexpr int kV = kK + kNB * kKBuf;
    static constexpr int kStage = kV + kNB * kVBuf;                // fp8 K then V, per stage
    static constexpr int kStageBytes = 2 * kPfKeys * HD;
    static constexpr int kBars = kStage + kNS * kStageBytes;
    // mbarriers: full[NS], empty[NS], then per buffer kv_ready, kv_free, s_ready, p_ready,
    // and one to drain the tensor core on a timeout.  kv_free[b] completes when the products
    // of the buffer's tile are done (one commit after its O product covers its S product
    // too); it also tells that O is up to date.
    static constexpr int kFull = kBars, kEmpty = kFull + 8 * kNS, kKvReady = kEmpty + 8 * kNS;
    static constexpr int kKvFree = kKvReady + 8 * kNB, kSReady = kKvFree + 8 * kNB;
    static constexpr int kPReady = kSReady + 8 * kNB;
    static constexpr int kDrain = kPReady + 8 * kNB;
    static constexpr int kMeta = kDrain + 8;                       // valid-key mask per stage
    static constexpr int kBufMask = kMeta + 8 * kNS;               // valid-key mask per K/V buffer
    static constexpr int kMisc = kBufMask + 8 * kNB;               // tmem base, abort flag
    static constexpr int kTotal = kMisc + 16;
    // tensor memory: S[NB] (64 fp32 columns each; P as f16 over the first 32), then O
    static constexpr uint32_t kColO = 64 * kNB;
    static constexpr uint32_t kTmemCols = kColO + HD + 32 <= 256 ? 256 : 512;
};

// Warp roles (448 threads): warps 0-3 softmax + epilogue (TMEM lane quarters 0-3, one score
// row per thread), warps 4-11 conversion, warp 12 tensor-core issue (and TMEM allocation),
// warp 13 TMA.
constexpr int kPfConvWarps = 8;
constexpr int kPfMmaWarp = 4 + kPfConvWarps, kPfTmaWarp = kPfMmaWarp + 1;
constexpr int kPfWarps = kPfTmaWarp + 1;

template <int HD>
__global__ void __launch_bounds__(kPfWarps * 32, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
               const PrefillArgs a) {
    using L = PfSmem<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *bp = smem_raw + (base - raw);
    volatile uint64_t *meta = reinterpret_cast<volatile uint64_t *>(bp + L::kMeta);
    volatile uint64_t *buf_mask = reinterpret_cast<volatile uint64_t *>(bp + L::kBufMask);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bp + L::kMisc);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(bp + L::kMisc + 4);
    auto bar = [&](int off, int i) { return base + static_cast<uint32_t>(off + 8 * i); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // kv head fastest, then row tile, then sequence (longest first): the CTAs resident at one
    // time read every kv head's slice of the same cache rows, and a (sequence, kv head)'s row
    // tiles run together, so its K/V tiles are fetched from HBM once and re-read from L2
    const int kvh = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.n_kv));
    const int tile = static_cast<int>((blockIdx.x / static_cast<unsigned>(a.n_kv)) % static_cast<unsigned>(a.row_tiles));
    const int rank = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.n_kv * a.row_tiles));

    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    // the K buffers are free scratch until the pipeline starts
    const int seq = seq_of_rank(a.seq_lens, a.num_seqs, a.max_len, rank,
                                reinterpret_cast<uint32_t *>(bp + L::kK));
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && tid == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    // this sequence's query rows (qsl == nullptr: one query per sequence, row seq) and cached
    // length (flagged once, by its first CTA)
    const int raw_nq = a.qsl ? a.qsl[seq + 1] - a.qsl[seq] : 1;
    const QueryRange qr = a.qsl ? query_range(a.qsl, seq, a.qmax, a.qrows) : QueryRange{seq, 1};
    const int Lraw = a.seq_lens[seq];
    const int Ls = min(max(Lraw, 0), a.max_len);
    // (more new tokens than cached ones is an error of the multi-query form only: a decode
    // query on an empty sequence gives a zero row)
    if (tile == 0 && kvh == 0 && tid == 0 &&
        (qr.count != raw_nq || Lraw < 0 || Lraw > a.max_len || (a.qsl && qr.count > Ls)))
        flag(a.status, KVFP8_DEV_BAD_BLOCK);
    const int nb = qr.count, G = a.group;
    const int row0 = tile * kPfRows;                 // first score row of this tile
    if (row0 >= nb * G) return;                      // no rows here
    const int j_last = min(nb, (row0 + kPfRows + G - 1) / G) - 1;
    const int kend = Ls - nb + j_last + 1;           // keys the tile's last row may see
    const int ntiles = kend > 0 ? (kend + kPfKeys - 1) / kPfKeys : 0;
    // The row tiles of one (sequence, kv head) run side by side on one K/V stream; each
    // starts its pass at its own key tile (the online softmax takes the keys in any order),
    // so they read different lines of the stream at any one time.
    const int rot = ntiles > 0 ? static_cast<int>((static_cast<int64_t>(tile) * ntiles) / a.row_tiles) % ntiles : 0;
    auto key_tile = [&](int i) { const int k = i + rot; return k >= ntiles ? k - ntiles : k; };

    if (ntiles == 0) {  // every row of the tile sees no key: zero rows
        if (tid < kPfRows) {
            const int r = row0 + tid;
            if (r < nb * G) {
                const int j = r / G, g = r % G;
                uint4 *o = reinterpret_cast<uint4 *>(
                    a.out + ((static_cast<int64_t>(qr.q0) + j) * a.n_q + kvh * G + g) * HD);
                for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < L::kNS; ++s) {
            mbar_init(bar(L::kFull, s), 1);
            mbar_init(bar(L::kEmpty, s), kPfConvWarps);
        }
        for (int b = 0; b < L::kNB; ++b) {
            mbar_init(bar(L::kKvReady, b), kPfConvWarps);
            mbar_init(bar(L::kKvFree, b), 1);
            mbar_init(bar(L::kSReady, b), 1);
            mbar_init(bar(L::kPReady, b), 4);
        }
        mbar_init(bar(L::kDrain, 0), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kPfMmaWarp) {
        tmem_alloc(base + L::kMisc, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kPfTmaWarp && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const volatile int32_t never = 0;

    if (warp == kPfTmaWarp) {
        // ------------------------------------------------------------ TMA producer
        // The warp holds 32 block-table entries, one per lane (refreshed as the tiles move
        // past them).  A tile is nbox boxes of K and nbox of V: lane p < nbox works out K box
        // p and lane nbox + p V box p, side by side; lane 0 waits for a free stage and posts
        // the expected bytes, then every lane with a box issues its own copy.  (This warp
        // shares its scheduler with compute-heavy warps: its per-tile work is kept to a few
        // dozen instructions, with no division.)
        const int32_t *bt = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
        const int bs = a.block_size, br = a.box_rows;
        const int lbs = __ffs(bs) - 1;  // block_size is a power of two
        const int nbox = kPfKeys / br;
        const bool k_lane = lane < nbox;
        const int p = k_lane ? lane : lane - nbox;  // this lane's box within the tile
        const bool box_lane = lane < 2 * nbox;
        const CUtensorMap *map = k_lane ? &tmk : &tmv;
        const uint32_t side = k_lane ? 0u : static_cast<uint32_t>(kPfKeys * HD);
        int wbase = -(1 << 30);
        int32_t win = -1;
        int issued = 0;
        bool aborted = false;
        for (int i = 0; i < ntiles; ++i) {
            const int st = i % L::kNS;
            const int t0 = key_tile(i) * kPfKeys;
            const int e0 = t0 >> lbs, e1 = (min(kend, t0 + kPfKeys) - 1) >> lbs;
            if (e0 < wbase || e1 >= wbase + 32) {  // next window of block-table entries
                wbase = e0;
                win = wbase + lane < a.max_blocks_per_seq ? bt[wbase + lane] : -1;
            }
            // this lane's box: its first key t, the block holding it, and whether it is
            // copied (keys past kend are left out; a bad block is flagged and left out)
            const int t = t0 + p * br;
            const int blk = __shfl_sync(0xFFFFFFFFu, win, ((t >> lbs) - wbase) & 31);
            const bool live = box_lane && t < kend;
            const bool good = live && blk >= 0 && blk < a.num_blocks;
            if (live && !good && k_lane) flag(a.status, KVFP8_DEV_BAD_BLOCK);
            const int row = blk * bs + (t & (bs - 1));
            uint64_t part = 0;
            if (good && k_lane) {
                const int nk = min(br, kend - t);
                part = (nk >= 64 ? ~0ull : ((1ull << nk) - 1)) << (p * br);
            }
            const uint64_t mask =
                static_cast<uint64_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(part))) |
                static_cast<uint64_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(part >> 32))) << 32;
            const int boxes = __popc(__ballot_sync(0xFFFFFFFFu, good && k_lane));
            if (lane == 0) {
                if (!mbar_wait(bar(L::kEmpty, st), ((i / L::kNS) & 1) ^ 1u, abort_flag)) {
                    aborted = true;
                } else {
                    meta[st] = mask;
                    const uint32_t full = bar(L::kFull, st);
                    if (boxes > 0)
                        mbar_arrive_tx(full, static_cast<uint32_t>(boxes * L::kSegs * 2 * br * L::kSeg));
                    else
                        mbar_arrive(full);
                    ++issued;
                }
            }
            aborted = __shfl_sync(0xFFFFFFFFu, aborted, 0);
            if (aborted) break;
            // the expected bytes are posted: each lane with a box copies it
            if (good) {
                const uint32_t full = bar(L::kFull, st);
                const uint32_t dst = base + L::kStage + st * L::kStageBytes + side +
                                     static_cast<uint32_t>(p * br * L::kSeg);
#pragma unroll
                for (int sgi = 0; sgi < L::kSegs; ++sgi)
                    tma_load_3d(dst + static_cast<uint32_t>(sgi * kPfKeys * L::kSeg), map, 0,
                                kvh * L::kSegs + sgi, row, full);
            }
        }
        if (aborted && lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
            // let copies already issued land before the CTA's shared memory goes away
            for (int k = max(0, issued - L::kNS); k < issued; ++k)
                mbar_wait(bar(L::kFull, k % L::kNS), (k / L::kNS) & 1, &never);
        }
    } else if (warp == kPfMmaWarp) {
        // ------------------------------------------------------------ tensor-core issue
        // S(i) is issued before O(i-1), so the tensor core computes the next scores while the
        // softmax warps work on the current ones.
        if (lane == 0) {
            const uint32_t idesc_s = f16_idesc(kPfRows, kPfKeys), idesc_o = f16_idesc(kPfRows, L::kVRows);
            // operand descriptors computed once; each product adds its constant offset
            const uint64_t qdesc = sw128_desc(base + L::kQ), kdesc = sw128_desc(base + L::kK),
                           vdesc = sw128_desc(base + L::kV);
            bool ok = true;
            auto issue_o = [&](int t) {  // O += P(t) . V(t), then release tile t's buffers
                const int b = t % L::kNB;
                if (!mbar_wait(bar(L::kPReady, b), (t / L::kNB) & 1, abort_flag)) return false;
                tc_fence_after();
                const uint64_t vb = desc_at(vdesc, b * L::kVBuf);
#pragma unroll
                for (int k = 0; k < kPfKeys / 16; ++k)
                    umma_ts(tmem + L::kColO, tmem + 64 * b + 8 * k, desc_at(vb, k * 32), idesc_o,
                            (t > 0 || k > 0) ? 1u : 0u);
                umma_commit(bar(L::kKvFree, b));
                return true;
            };
            for (int i = 0; i < ntiles && ok; ++i) {
                const int b = i % L::kNB;
                ok = mbar_wait(bar(L::kKvReady, b), (i / L::kNB) & 1, abort_flag);
                // S(i) overwrites the buffer that held P(i-NB): O(i-NB) must have read it
                if (ok && i >= L::kNB)
                    ok = mbar_wait(bar(L::kKvFree, b), ((i / L::kNB) & 1) ^ 1u, abort_flag);
                if (!ok) break;
                tc_fence_after();
                const uint64_t kb = desc_at(kdesc, b * L::kKBuf);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint64_t ad = desc_at(qdesc, (k >> 2) * (kPfRows * 128) + (k & 3) * 32);
                    const uint64_t bd = desc_at(kb, (k >> 2) * (kPfKeys * 128) + (k & 3) * 32);
                    umma_ss(tmem + 64 * b, ad, bd, idesc_s, k > 0 ? 1u : 0u);
                }
                umma_commit(bar(L::kSReady, b));
                if (i >= 1) ok = issue_o(i - 1);
            }
            if (ok) ok = issue_o(ntiles - 1);
            if (!ok) {
                flag(a.status, KVFP8_DEV_TIMEOUT);
                *abort_flag = 1;
                // let the products already issued finish before tensor memory is released
                umma_commit(bar(L::kDrain, 0));
                mbar_wait(bar(L::kDrain, 0), 0, &never);
            }
        }
    } else if (warp >= 4) {
        // ------------------------------------------------------------ conversion warps
        const int ct = tid - 128;  // 0 .. 32*kPfConvWarps-1
        constexpr int kCT = 32 * kPfConvWarps;
        if (ct < kPfRows) {  // q rows -> f16, 128-byte-swizzled K-major blocks of 64 head dims; row ct
            const int r = row0 + ct;
            const bool row_ok = r < nb * G;
            const int jq = row_ok ? r / G : 0, gq = row_ok ? r % G : 0;
            const __nv_bfloat16 *qrow =
                a.query + ((static_cast<int64_t>(qr.q0) + jq) * a.n_q + kvh * G + gq) * HD;
#pragma unroll 4
            for (int c = 0; c < HD / 8; ++c) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (row_ok) w = *reinterpret_cast<const uint4 *>(qrow + 8 * c);
                uint4 h;
                h.x = f16x2_from_f32(bf16lo(w.x), bf16hi(w.x));
                h.y = f16x2_from_f32(bf16lo(w.y), bf16hi(w.y));
                h.z = f16x2_from_f32(bf16lo(w.z), bf16hi(w.z));
                h.w = f16x2_from_f32(bf16lo(w.w), bf16hi(w.w));
                *reinterpret_cast<uint4 *>(bp + L::kQ + (c >> 3) * (kPfRows * 128) + sw128(ct, c & 7)) = h;
            }
        }
        if (L::kSumCol) {  // V^T rows HD..HD+15 of every buffer: ones, then zeros
            for (int e = ct; e < L::kNB * 128; e += kCT) {
                const int bb = e >> 7, w = e & 127;  // 128 16-byte words per buffer
                const uint32_t one = w < 8 ? 0x3C003C00u : 0u;
                *reinterpret_cast<uint4 *>(bp + L::kV + bb * L::kVBuf + HD * 128 + 16 * w) =
                    make_uint4(one, one, one, one);
            }
        }
        bool ok = true;
        for (int i = 0; i < ntiles && ok; ++i) {
            const int st = i % L::kNS, b = i % L::kNB;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kFull, st), (i / L::kNS) & 1, abort_flag));
            // the buffer's previous tile (i-NB) has been through both products
            if (ok)
                ok = __all_sync(0xFFFFFFFFu,
                                mbar_wait(bar(L::kKvFree, b), ((i / L::kNB) & 1) ^ 1u, abort_flag));
            if (!ok) break;
            const uint64_t mask = meta[st];
            const uint8_t *kst = bp + L::kStage + st * L::kStageBytes;
            const uint8_t *vst = kst + kPfKeys * HD;
            uint8_t *kdst0 = bp + L::kK + b * L::kKBuf;
            uint8_t *vdst = bp + L::kV + b * L::kVBuf;
            // K: 64 keys x HD/8 chunks of 8 fp8 -> one 16-byte f16 chunk (invalid keys: zeros);
            // eight consecutive threads take the eight chunks of one 64-dim block row, so each
            // quarter-warp's stores cover all 32 banks.
            // V^T by 8-key x 32-dim blocks: lane t converts dims (8j + 2(t%4), +1) of key t/4
            // (one e4m3 pair -> f16x2 per matrix j) and stmatrix.trans writes each dim's 8 keys
            // as one 16-byte row of V^T (head dims as rows, keys along K).
            // Every load of a round is issued before the first conversion, so their latencies
            // overlap (a store to shared memory would otherwise hold back the next load).
            constexpr int kKT = kPfKeys * (HD / 8) / kCT;                    // K tasks per thread
            constexpr int kVB = (kPfKeys / 8) * (HD / 32) / kPfConvWarps;    // V^T blocks per warp
            constexpr int kVG = kVB < 4 ? kVB : 4;                           // V^T blocks per round
            const int w4 = warp - 4;
            const uint32_t vbase = base + L::kV + b * L::kVBuf;
            const uint32_t vsel = static_cast<uint32_t>(2 * (lane & 3)) | static_cast<uint32_t>(2 * (lane & 3) + 1) << 4;
            uint2 kw[kKT];
            uint4 vw[kVG][2];
            auto v_load = [&](int g0) {
#pragma unroll
                for (int j = 0; j < kVG; ++j) {
                    const int blk = w4 + (g0 + j) * kPfConvWarps;
                    const int ko = blk % (kPfKeys / 8), dg = blk / (kPfKeys / 8);
                    const int key = ko * 8 + (lane >> 2);
                    const int sgi = (32 * dg) / L::kSeg, cc = ((32 * dg) % L::kSeg) >> 4;
                    const uint8_t *vrow = vst + sgi * kPfKeys * L::kSeg;
                    vw[j][0] = *reinterpret_cast<const uint4 *>(vrow + swz<L::kSeg>(key, cc));
                    vw[j][1] = *reinterpret_cast<const uint4 *>(vrow + swz<L::kSeg>(key, cc + 1));
                    if (!((mask >> key) & 1ull)) vw[j][0] = vw[j][1] = make_uint4(0u, 0u, 0u, 0u);
                }
            };
            auto v_store = [&](int g0) {
#pragma unroll
                for (int j = 0; j < kVG; ++j) {
                    const int blk = w4 + (g0 + j) * kPfConvWarps;
                    const int ko = blk % (kPfKeys / 8), dg = blk / (kPfKeys / 8);
                    const uint4 lo = vw[j][0], hi = vw[j][1];
                    const uint32_t wd[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    uint32_t r[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q)  // bytes 8q + 2(t%4), +1 of the key's 32
                        r[q] = f16x2_from_e4m3x2(__byte_perm(wd[2 * q], wd[2 * q + 1], vsel));
                    const int n = 32 * dg + 8 * (lane >> 3) + (lane & 7);  // V^T row this lane addresses
                    stsm_x4_t(vbase + sw128(n, ko), r[0], r[1], r[2], r[3]);
                }
            };
#pragma unroll
            for (int j = 0; j < kKT; ++j) {
                const int task = ct + j * kCT;
                const int key = task / (HD / 8), c = task % (HD / 8);  // dims 8c .. 8c+7
                const int sgi = (8 * c) / L::kSeg, within = (8 * c) % L::kSeg;
                kw[j] = *reinterpret_cast<const uint2 *>(kst + sgi * kPfKeys * L::kSeg +
                                                         swz<L::kSeg>(key, within >> 4) + (within & 8));
                if (!((mask >> key) & 1ull)) kw[j] = make_uint2(0u, 0u);
            }
            v_load(0);
#pragma unroll
            for (int j = 0; j < kKT; ++j) {
                const int task = ct + j * kCT;
                const int key = task / (HD / 8), c = task % (HD / 8);
                const uint2 w = kw[j];
                uint4 h;
                h.x = f16x2_from_e4m3x2(w.x);
                h.y = f16x2_from_e4m3x2_hi(w.x);
                h.z = f16x2_from_e4m3x2(w.y);
                h.w = f16x2_from_e4m3x2_hi(w.y);
                *reinterpret_cast<uint4 *>(kdst0 + (c >> 3) * (kPfKeys * 128) + sw128(key, c & 7)) = h;
            }
            v_store(0);
#pragma unroll
            for (int g0 = kVG; g0 < kVB; g0 += kVG) {
                v_load(g0);
                v_store(g0);
            }
            if (ct == 0) buf_mask[b] = mask;  // for the softmax warps, released with kv_ready
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(L::kEmpty, st));     // the FP8 stage may be refilled
                mbar_arrive(bar(L::kKvReady, b));    // K(i), V^T(i) (and Q) are ready
            }
        }
        if (!ok && lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    } else {
        // ------------------------------------------------------------ softmax warps
        const int r = row0 + tid;                   // this thread's score row (TMEM lane tid)
        const bool row_ok = r < nb * G;
        const int jq = row_ok ? r / G : 0, gq = row_ok ? r % G : 0;
        const int pos = Ls - nb + jq;               // last key position the row may see
        const float score_scale = a.sm_scale * sk * 1.4426950408889634f;  // log2(e)
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        float m_used = -INFINITY, lsum = 0.f;
        bool ok = true;
        for (int i = 0; i < ntiles && ok; ++i) {
            const int b = i % L::kNB, ph = (i / L::kNB) & 1;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kSReady, b), ph, abort_flag));
            // the tile's valid-key mask (already complete: S(i) needed the same phase)
            if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kKvReady, b), ph, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const uint64_t mask = buf_mask[b];
            uint32_t s[2][32];
            tmem_ld32(lane_addr + 64 * b, s[0]);
            tmem_ld32(lane_addr + 64 * b + 32, s[1]);
            tmem_wait_ld();
            // causal mask, scale, running maximum (a key past the row's position, past the
            // sequence or in a bad block scores -inf; keys past kend are past every position).
            // A tile every row of the warp sees whole takes no mask: the maximum is taken on
            // the raw scores (the smallest when the scale is negative) and scaled once, and
            // the scale is applied inside the exponent's fma.
            const int k0 = key_tile(i) * kPfKeys;
            const int vis_n = row_ok ? min(kPfKeys, max(0, pos - k0 + 1)) : 0;  // keys 0..vis_n-1
            const uint64_t vis = mask & (vis_n >= 64 ? ~0ull : ((1ull << vis_n) - 1));
            float mx, mult;
            if (__all_sync(0xFFFFFFFFu, vis == ~0ull)) {
                mx = (score_scale >= 0.f ? extreme64<true>(s) : extreme64<false>(s)) * score_scale;
                mult = score_scale;
            } else {
                mx = -INFINITY;
                mult = 1.f;
#pragma unroll
                for (int h = 0; h < 2; ++h)
#pragma unroll
                    for (int c = 0; c < 32; ++c) {
                        const float v = ((vis >> (32 * h + c)) & 1ull)
                                            ? __uint_as_float(s[h][c]) * score_scale
                                            : -INFINITY;
                        s[h][c] = __float_as_uint(v);
                        mx = fmaxf(mx, v);
                    }
            }
            // rescale O only when the maximum grew by more than 2^8 (first visible keys: O is
            // still zero for this row, nothing to rescale)
            float factor = 1.f;
            if (mx > -INFINITY) {
                if (m_used == -INFINITY) {
                    m_used = mx;
                } else if (mx > m_used + 8.f) {
                    factor = ex2(m_used - mx);
                    m_used = mx;
                }
            }
            if (__any_sync(0xFFFFFFFFu, factor != 1.f)) {
                // O(i-1) must be complete before O is rescaled (with its row-sum column)
                ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kKvFree, (i - 1) % L::kNB),
                                                       ((i - 1) / L::kNB) & 1, abort_flag));
                if (!ok) break;
                tc_fence_after();
                lsum *= factor;
#pragma unroll 1
                for (int c0 = 0; c0 < (L::kSumCol ? HD + 32 : HD); c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + L::kColO + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * factor);
                    tmem_st32(lane_addr + L::kColO + c0, o);
                }
            }
            // P = 2^(s*mult - m) as f16 pairs over the first 32 columns of this S buffer: one
            // packed fma, one f16 pack and one f16x2 exp2 per pair (x <= 2^3 by the rescale
            // rule, so P <= 2^8)
            uint32_t p[32];
            const float msub = m_used == -INFINITY ? 0.f : m_used;
            const uint64_t mul2 = pk2(mult, mult), sub2 = pk2(-msub, -msub);
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int h = c >> 4, e = (2 * c) & 31;
                const float2 x = upk2(fma_f32x2(pk2u(s[h][e], s[h][e + 1]), mul2, sub2));
                p[c] = ex2_f16x2(f16x2_from_f32(x.x, x.y));
                if (!L::kSumCol) lsum += f16lo_f32(p[c]) + f16hi_f32(p[c]);
            }
            tmem_st32(lane_addr + 64 * b, p);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kPReady, b));
        }
        if (ok)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kKvFree, (ntiles - 1) % L::kNB),
                                                   ((ntiles - 1) / L::kNB) & 1, abort_flag));
        if (ok) {
            tc_fence_after();
            if (L::kSumCol) {  // the row's sum of P, accumulated by the O product
                uint32_t o[32];
                tmem_ld32(lane_addr + L::kColO + HD, o);
                tmem_wait_ld();
                lsum = __uint_as_float(o[0]);
            }
            const float inv = lsum > 0.f ? sv / lsum : 0.f;
            uint4 *orow = reinterpret_cast<uint4 *>(
                a.out + ((static_cast<int64_t>(qr.q0) + jq) * a.n_q + kvh * G + gq) * HD);
#pragma unroll 1
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(lane_addr + L::kColO + c0, o);
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w;
                        w.x = bf16x2_from_f32(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv);
                        w.y = bf16x2_from_f32(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                        w.z = bf16x2_from_f32(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
                        w.w = bf16x2_from_f32(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
                        orow[(c0 + c) / 8] = w;
                    }
                }
            }
        } else if (lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kPfMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

// ---------------------------------------------------------------- two row tiles per CTA
//
// For head_dim 64 and 128 when a (sequence, kv head) has more than 128 score rows: one CTA
// takes 256 rows as two row tiles that share every converted K/V tile, so the copies and
// the conversion are paid once per two tiles of tensor work.  Keys go in tiles of 128: the
// score product S = Q.K^T then has N = 128, where a kind::f16 product runs at the tensor
// core's full rate (at N = 64 the shared-memory reads of its two operands bound it to about
// two thirds of that), and each tile costs half as many products, commits and waits.
//
// Tensor memory (512 columns at head_dim 128): S[r] at 128*r (P written over its first 64
// columns as f16), O[r] at 256 + head_dim*r.  Each row tile has one score buffer: the tensor
// core runs the products one thread issues in order, and S(r, i+1) is issued after O(r, i),
// so the next scores land only after the product that reads P.  The two row tiles take
// turns: while one row tile's softmax works, the tensor core runs the other's O and next S.
// The commit that signals S(r, i) also covers O(r, i-1), so the softmax may rescale O as
// soon as its scores are ready.  The rows sum P themselves (fp32, in pairs).
//
// FP8 K/V arrive by TMA in halves of 64 keys (a staging ring of NS halves) and are converted
// into two f16 K buffers and two V^T buffers of 128 keys.  A K buffer is free once both row
// tiles' S products are done with it; a V^T buffer (and the valid-key masks stored with it)
// once both O products are.
//
// Warps (14): 0-3 softmax of row tile 0, 4-7 softmax of row tile 1 (warp w reads TMEM
// lanes 32*(w%4)..+31), 8-11 conversion, 12 tensor-core issue (and TMEM allocation), 13 TMA.
constexpr int kP2Rows = 2 * kPfRows;
constexpr int kP2Keys = 2 * kPfKeys;   // keys per tile; FP8 staging and conversion go by halves
constexpr int kP2ConvWarps = 4;
constexpr int kP2MmaWarp = 8 + kP2ConvWarps, kP2TmaWarp = kP2MmaWarp + 1;
constexpr int kP2Warps = kP2TmaWarp + 1;

template <int HD>
struct Pf2Smem {
    static constexpr int kSeg = HD >= 128 ? 128 : 64;
    static constexpr int kSegs = HD / kSeg;
    static constexpr int kNS = HD >= 128 ? 2 : 4;                  // FP8 staging halves
    static constexpr int kQTile = HD * 256;                        // one row tile of Q (f16)
    static constexpr int kQ = 0;
    // K f16: HD/64 blocks x 128 keys x 128 B; V^T f16: 2 key blocks x HD rows x 128 B
    static constexpr int kKBuf = HD * 256, kVBuf = HD * 256;
    static constexpr int kK = kQ + 2 * kQTile;
    static constexpr int kV = kK + 2 * kKBuf;
    static constexpr int kStage = kV + 2 * kVBuf;
    static constexpr int kStageBytes = 2 * kPfKeys * HD;           // FP8 K then V of 64 keys
    static constexpr int kBars = kStage + kNS * kStageBytes;
    // mbarriers: full[NS], empty[NS], then per buffer k_ready, v_ready, k_free, v_free, then
    // per row tile s_ready, p_ready, o_done, and one to drain the tensor core on a timeout
    static constexpr int kFull = kBars, kEmpty = kFull + 8 * kNS, kKReady = kEmpty + 8 * kNS;
    static constexpr int kVReady = kKReady + 16, kKFree = kVReady + 16, kVFree = kKFree + 16;
    static constexpr int kSReady = kVFree + 16, kPReady = kSReady + 16, kODone = kPReady + 16;
    static constexpr int kDrain = kODone + 16;
    static constexpr int kMeta = kDrain + 8;                       // valid-key mask per stage
    static constexpr int kBufMask = kMeta + 8 * kNS;               // per V^T buffer, two halves
    static constexpr int kMisc = kBufMask + 32;                    // tmem base, abort flag
    static constexpr int kTotal = kMisc + 16;
    static constexpr uint32_t kTmemCols = 512;
    __host__ __device__ static constexpr uint32_t col_s(int r) { return static_cast<uint32_t>(128 * r); }
    __host__ __device__ static constexpr uint32_t col_o(int r) { return static_cast<uint32_t>(256 + HD * r); }
    // P of keys 16k..16k+15 (f16 pairs, 8 columns): the first half of the 32 columns that
    // held the scores of keys 32(k/2)..+31, so each 32-key chunk's P overwrites only its own
    // scores
    __host__ __device__ static constexpr uint32_t col_p(int k) { return static_cast<uint32_t>(32 * (k >> 1) + 8 * (k & 1)); }
};

// the largest (kMax) or smallest of 32 scores, four chains of 3-input ops
template <bool kMax>
__device__ __forceinline__ float extreme32(const uint32_t (&s)[32]) {
    auto v = [&](int c) { return __uint_as_float(s[c]); };
    auto op = [](float a, float b, float c) { return kMax ? max3f(a, b, c) : min3f(a, b, c); };
    float a0 = v(0), a1 = v(1), a2 = v(2), a3 = v(3);
#pragma unroll
    for (int c = 4; c < 28; c += 8) {
        a0 = op(a0, v(c), v(c + 1));
        a1 = op(a1, v(c + 2), v(c + 3));
        a2 = op(a2, v(c + 4), v(c + 5));
        a3 = op(a3, v(c + 6), v(c + 7));
    }
    a0 = op(a0, v(28), v(29));
    a1 = op(a1, v(30), v(31));
    return op(a0, a1, kMax ? fmaxf(a2, a3) : fminf(a2, a3));
}

__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
                 : "memory");
}

template <int HD>
__global__ void __launch_bounds__(kP2Warps * 32, 1)
prefill2_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                const PrefillArgs a) {
    using L = Pf2Smem<HD>;
    static_assert(L::kTotal + 1024 <= 232448, "shared memory");
    static_assert(L::col_o(1) + HD <= L::kTmemCols, "tensor memory");
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *bp = smem_raw + (base - raw);
    volatile uint64_t *meta = reinterpret_cast<volatile uint64_t *>(bp + L::kMeta);
    volatile uint64_t *buf_mask = reinterpret_cast<volatile uint64_t *>(bp + L::kBufMask);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bp + L::kMisc);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(bp + L::kMisc + 4);
    auto bar = [&](int off, int i) { return base + static_cast<uint32_t>(off + 8 * i); };

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int kvh = static_cast<int>(blockIdx.x % static_cast<unsigned>(a.n_kv));
    const int ctile = static_cast<int>((blockIdx.x / static_cast<unsigned>(a.n_kv)) % static_cast<unsigned>(a.row_tiles));
    const int rank = static_cast<int>(blockIdx.x / static_cast<unsigned>(a.n_kv * a.row_tiles));

    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    // longest sequences first; the K buffers are free scratch until the pipeline starts
    const int seq = seq_of_rank(a.seq_lens, a.num_seqs, a.max_len, rank,
                                reinterpret_cast<uint32_t *>(bp + L::kK));
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && tid == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    const int raw_nq = a.qsl[seq + 1] - a.qsl[seq];
    const QueryRange qr = query_range(a.qsl, seq, a.qmax, a.qrows);
    const int Lraw = a.seq_lens[seq];
    const int Ls = min(max(Lraw, 0), a.max_len);
    if (ctile == 0 && kvh == 0 && tid == 0 &&
        (qr.count != raw_nq || Lraw < 0 || Lraw > a.max_len || qr.count > Ls))
        flag(a.status, KVFP8_DEV_BAD_BLOCK);
    const int nb = qr.count, G = a.group;
    const int row0 = ctile * kP2Rows;                 // first score row of this CTA
    if (row0 >= nb * G) return;
    const int j_last = min(nb, (row0 + kP2Rows + G - 1) / G) - 1;
    const int kend = Ls - nb + j_last + 1;            // keys the CTA's last row may see
    const int ntiles = kend > 0 ? (kend + kP2Keys - 1) / kP2Keys : 0;
    const int rot = ntiles > 0 ? static_cast<int>((static_cast<int64_t>(ctile) * ntiles) / a.row_tiles) % ntiles : 0;
    auto key_tile = [&](int i) { const int k = i + rot; return k >= ntiles ? k - ntiles : k; };

    if (ntiles == 0) {  // every row of the CTA sees no key: zero rows
        if (tid < kP2Rows) {
            const int r = row0 + tid;
            if (r < nb * G) {
                const int j = r / G, g = r % G;
                uint4 *o = reinterpret_cast<uint4 *>(
                    a.out + ((static_cast<int64_t>(qr.q0) + j) * a.n_q + kvh * G + g) * HD);
                for (int c = 0; c < HD / 8; ++c) o[c] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        return;
    }

    if (tid == 0) {
        for (int s = 0; s < L::kNS; ++s) {
            mbar_init(bar(L::kFull, s), 1);
            mbar_init(bar(L::kEmpty, s), kP2ConvWarps);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bar(L::kKReady, b), kP2ConvWarps);
            mbar_init(bar(L::kVReady, b), kP2ConvWarps);
            mbar_init(bar(L::kKFree, b), 1);
            mbar_init(bar(L::kVFree, b), 1);
            mbar_init(bar(L::kSReady, b), 1);
            mbar_init(bar(L::kPReady, b), 4);
            mbar_init(bar(L::kODone, b), 1);
        }
        mbar_init(bar(L::kDrain, 0), 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == kP2MmaWarp) {
        tmem_alloc(base + L::kMisc, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == kP2TmaWarp && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const volatile int32_t never = 0;

    if (warp == kP2TmaWarp) {
        // ------------------------------------------------------------ TMA producer
        // half h of the key pass (64 keys of tile h/2): lane p < nbox fetches K box p, lane
        // nbox + p V box p
        const int32_t *bt = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
        const int bs = a.block_size, br = a.box_rows;
        const int lbs = __ffs(bs) - 1;
        const int nbox = kPfKeys / br;
        const bool k_lane = lane < nbox;
        const int p = k_lane ? lane : lane - nbox;
        const bool box_lane = lane < 2 * nbox;
        const CUtensorMap *map = k_lane ? &tmk : &tmv;
        const uint32_t side = k_lane ? 0u : static_cast<uint32_t>(kPfKeys * HD);
        int wbase = -(1 << 30);
        int32_t win = -1;
        int issued = 0;
        bool aborted = false;
        for (int h = 0; h < 2 * ntiles; ++h) {
            const int st = h % L::kNS;
            const int t0 = key_tile(h >> 1) * kP2Keys + (h & 1) * kPfKeys;
            const int t = t0 + p * br;
            const bool any = t0 < kend;
            if (any) {
                const int e0 = t0 >> lbs, e1 = (min(kend, t0 + kPfKeys) - 1) >> lbs;
                if (e0 < wbase || e1 >= wbase + 32) {
                    wbase = e0;
                    win = wbase + lane < a.max_blocks_per_seq ? bt[wbase + lane] : -1;
                }
            }
            const int blk = __shfl_sync(0xFFFFFFFFu, win, ((t >> lbs) - wbase) & 31);
            const bool live = any && box_lane && t < kend;
            const bool good = live && blk >= 0 && blk < a.num_blocks;
            if (live && !good && k_lane) flag(a.status, KVFP8_DEV_BAD_BLOCK);
            const int row = blk * bs + (t & (bs - 1));
            uint64_t part = 0;
            if (good && k_lane) {
                const int nk = min(br, kend - t);
                part = (nk >= 64 ? ~0ull : ((1ull << nk) - 1)) << (p * br);
            }
            const uint64_t mask =
                static_cast<uint64_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(part))) |
                static_cast<uint64_t>(__reduce_or_sync(0xFFFFFFFFu, static_cast<uint32_t>(part >> 32))) << 32;
            const int boxes = __popc(__ballot_sync(0xFFFFFFFFu, good && k_lane));
            if (lane == 0) {
                if (!mbar_wait(bar(L::kEmpty, st), ((h / L::kNS) & 1) ^ 1u, abort_flag)) {
                    aborted = true;
                } else {
                    meta[st] = mask;
                    const uint32_t full = bar(L::kFull, st);
                    if (boxes > 0)
                        mbar_arrive_tx(full, static_cast<uint32_t>(boxes * L::kSegs * 2 * br * L::kSeg));
                    else
                        mbar_arrive(full);
                    ++issued;
                }
            }
            aborted = __shfl_sync(0xFFFFFFFFu, aborted, 0);
            if (aborted) break;
            if (good) {
                const uint32_t full = bar(L::kFull, st);
                const uint32_t dst = base + L::kStage + st * L::kStageBytes + side +
                                     static_cast<uint32_t>(p * br * L::kSeg);
#pragma unroll
                for (int sgi = 0; sgi < L::kSegs; ++sgi)
                    tma_load_3d(dst + static_cast<uint32_t>(sgi * kPfKeys * L::kSeg), map, 0,
                                kvh * L::kSegs + sgi, row, full);
            }
        }
        if (aborted && lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
            for (int k = max(0, issued - L::kNS); k < issued; ++k)
                mbar_wait(bar(L::kFull, k % L::kNS), (k / L::kNS) & 1, &never);
        }
    }
    else if (warp == kP2MmaWarp) {
        // ------------------------------------------------------------ tensor-core issue
        // S(r, 0) for both row tiles, then per tile i and row tile r: O(r, i) once P(r, i) is
        // ready, then S(r, i+1) into the same columns.
        if (lane == 0) {
            const uint32_t idesc_s = f16_idesc(kPfRows, kP2Keys), idesc_o = f16_idesc(kPfRows, HD);
            // operand descriptors computed once; each product adds its constant offset
            const uint64_t qdesc = sw128_desc(base + L::kQ), kdesc = sw128_desc(base + L::kK),
                           vdesc = sw128_desc(base + L::kV);
            auto issue_s = [&](int i, int r) {
                const uint64_t qd = desc_at(qdesc, r * L::kQTile);
                const uint64_t kb = desc_at(kdesc, (i & 1) * L::kKBuf);
#pragma unroll
                for (int k = 0; k < HD / 16; ++k)
                    umma_ss(tmem + L::col_s(r), desc_at(qd, (k >> 2) * (kPfRows * 128) + (k & 3) * 32),
                            desc_at(kb, (k >> 2) * (kP2Keys * 128) + (k & 3) * 32), idesc_s,
                            k > 0 ? 1u : 0u);
                umma_commit(bar(L::kSReady, r));
            };
            auto issue_o = [&](int i, int r) {
                const uint64_t vb = desc_at(vdesc, (i & 1) * L::kVBuf);
#pragma unroll
                for (int k = 0; k < kP2Keys / 16; ++k)
                    umma_ts(tmem + L::col_o(r), tmem + L::col_s(r) + L::col_p(k),
                            desc_at(vb, (k >> 2) * (HD * 128) + (k & 3) * 32), idesc_o,
                            (i > 0 || k > 0) ? 1u : 0u);
            };
            bool ok = mbar_wait(bar(L::kKReady, 0), 0, abort_flag);
            if (ok) {
                tc_fence_after();
                issue_s(0, 0);
                issue_s(0, 1);
                umma_commit(bar(L::kKFree, 0));
            }
            for (int i = 0; i < ntiles && ok; ++i) {
                const int b = i & 1;
                ok = mbar_wait(bar(L::kVReady, b), (i >> 1) & 1, abort_flag);
#pragma unroll
                for (int r = 0; r < 2; ++r) {
                    if (ok) ok = mbar_wait(bar(L::kPReady, r), i & 1, abort_flag);
                    if (ok && r == 0 && i + 1 < ntiles)
                        ok = mbar_wait(bar(L::kKReady, (i + 1) & 1), ((i + 1) >> 1) & 1, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    issue_o(i, r);
                    if (i + 1 == ntiles) umma_commit(bar(L::kODone, r));
                    if (r == 1) umma_commit(bar(L::kVFree, b));
                    if (i + 1 < ntiles) {
                        issue_s(i + 1, r);
                        if (r == 1) umma_commit(bar(L::kKFree, (i + 1) & 1));
                    }
                }
            }
            if (!ok) {
                flag(a.status, KVFP8_DEV_TIMEOUT);
                *abort_flag = 1;
                // let the products already issued finish before tensor memory is released
                umma_commit(bar(L::kDrain, 0));
                mbar_wait(bar(L::kDrain, 0), 0, &never);
            }
        }
    }
    else if (warp >= 8) {
        // ------------------------------------------------------------ conversion warps
        const int ct = tid - 256;  // 0 .. 32*kP2ConvWarps-1
        constexpr int kCT = 32 * kP2ConvWarps;
        // q rows -> f16, 128-byte-swizzled K-major blocks of 64 head dims: rows ct and ct+128
#pragma unroll 1
        for (int rr = ct; rr < kP2Rows; rr += kCT) {
            const int r = row0 + rr;
            const bool row_ok = r < nb * G;
            const int jq = row_ok ? r / G : 0, gq = row_ok ? r % G : 0;
            const __nv_bfloat16 *qrow =
                a.query + ((static_cast<int64_t>(qr.q0) + jq) * a.n_q + kvh * G + gq) * HD;
            uint8_t *qt = bp + L::kQ + (rr / kPfRows) * L::kQTile;
            const int lr = rr % kPfRows;
#pragma unroll 4
            for (int c = 0; c < HD / 8; ++c) {
                uint4 w = make_uint4(0u, 0u, 0u, 0u);
                if (row_ok) w = *reinterpret_cast<const uint4 *>(qrow + 8 * c);
                uint4 h;
                h.x = f16x2_from_f32(bf16lo(w.x), bf16hi(w.x));
                h.y = f16x2_from_f32(bf16lo(w.y), bf16hi(w.y));
                h.z = f16x2_from_f32(bf16lo(w.z), bf16hi(w.z));
                h.w = f16x2_from_f32(bf16lo(w.w), bf16hi(w.w));
                *reinterpret_cast<uint4 *>(qt + (c >> 3) * (kPfRows * 128) + sw128(lr, c & 7)) = h;
            }
        }
        // K: a task is 8 dims of one key (8 FP8 bytes in, one 16-byte f16 chunk out); eight
        // consecutive threads take the eight chunks of one 64-dim block row, so each
        // quarter-warp's stores cover all 32 banks
        constexpr int kKT = kPfKeys * (HD / 8) / kCT;                    // K tasks per thread
        constexpr int kVB = (kPfKeys / 8) * (HD / 32) / kP2ConvWarps;    // V^T blocks per warp
        constexpr int kVG = kVB < 4 ? kVB : 4;                           // V^T blocks per round
        const int w8 = warp - 8;
        const uint32_t vsel = static_cast<uint32_t>(2 * (lane & 3)) | static_cast<uint32_t>(2 * (lane & 3) + 1) << 4;
        bool ok = true;
        for (int h = 0; h < 2 * ntiles && ok; ++h) {
            const int st = h % L::kNS, i = h >> 1, hf = h & 1, b = i & 1;
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kFull, st), (h / L::kNS) & 1, abort_flag));
            // the K buffer's previous tile (i-2) is through both S products
            if (ok && hf == 0)
                ok = __all_sync(0xFFFFFFFFu,
                                mbar_wait(bar(L::kKFree, b), ((i >> 1) & 1) ^ 1u, abort_flag));
            if (!ok) break;
            const uint64_t mask = meta[st];
            const uint8_t *kst = bp + L::kStage + st * L::kStageBytes;
            const uint8_t *vst = kst + kPfKeys * HD;
            // this half's 64 keys: rows 64*hf.. of every 64-dim block of the K buffer
            uint8_t *kdst0 = bp + L::kK + b * L::kKBuf + hf * (kPfKeys * 128);
            // and key block hf of the V^T buffer
            const uint32_t vbase = base + L::kV + b * L::kVBuf + hf * (HD * 128);
            uint4 vw[kVG][2];
            auto v_load = [&](int g0) {
#pragma unroll
                for (int q = 0; q < kVG; ++q) {
                    const int blk = w8 + (g0 + q) * kP2ConvWarps;
                    const int ko = blk % (kPfKeys / 8), dg = blk / (kPfKeys / 8);
                    const int key = ko * 8 + (lane >> 2);
                    const int sgi = (32 * dg) / L::kSeg, cc = ((32 * dg) % L::kSeg) >> 4;
                    const uint8_t *vrow = vst + sgi * kPfKeys * L::kSeg;
                    vw[q][0] = *reinterpret_cast<const uint4 *>(vrow + swz<L::kSeg>(key, cc));
                    vw[q][1] = *reinterpret_cast<const uint4 *>(vrow + swz<L::kSeg>(key, cc + 1));
                    if (!((mask >> key) & 1ull)) vw[q][0] = vw[q][1] = make_uint4(0u, 0u, 0u, 0u);
                }
            };
            auto v_store = [&](int g0) {
#pragma unroll
                for (int q = 0; q < kVG; ++q) {
                    const int blk = w8 + (g0 + q) * kP2ConvWarps;
                    const int ko = blk % (kPfKeys / 8), dg = blk / (kPfKeys / 8);
                    const uint4 lo = vw[q][0], hi = vw[q][1];
                    const uint32_t wd[8] = {lo.x, lo.y, lo.z, lo.w, hi.x, hi.y, hi.z, hi.w};
                    uint32_t rv[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e)  // bytes 8e + 2(t%4), +1 of the key's 32
                        rv[e] = f16x2_from_e4m3x2(__byte_perm(wd[2 * e], wd[2 * e + 1], vsel));
                    const int n = 32 * dg + 8 * (lane >> 3) + (lane & 7);
                    stsm_x4_t(vbase + sw128(n, ko), rv[0], rv[1], rv[2], rv[3]);
                }
            };
            // K: every load of the half before its conversions
            uint2 kw[kKT];
#pragma unroll
            for (int q = 0; q < kKT; ++q) {
                const int task = ct + q * kCT;
                const int key = task / (HD / 8), c = task % (HD / 8);
                const int sgi = (8 * c) / L::kSeg, within = (8 * c) % L::kSeg;
                kw[q] = *reinterpret_cast<const uint2 *>(kst + sgi * kPfKeys * L::kSeg +
                                                         swz<L::kSeg>(key, within >> 4) + (within & 8));
                if (!((mask >> key) & 1ull)) kw[q] = make_uint2(0u, 0u);
            }
#pragma unroll
            for (int q = 0; q < kKT; ++q) {
                const int task = ct + q * kCT;
                const int key = task / (HD / 8), c = task % (HD / 8);
                const uint2 w = kw[q];
                uint4 h;
                h.x = f16x2_from_e4m3x2(w.x);
                h.y = f16x2_from_e4m3x2_hi(w.x);
                h.z = f16x2_from_e4m3x2(w.y);
                h.w = f16x2_from_e4m3x2_hi(w.y);
                *reinterpret_cast<uint4 *>(kdst0 + (c >> 3) * (kP2Keys * 128) + sw128(key, c & 7)) = h;
            }
            if (hf == 1) {  // both halves of the tile's K are in place
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar(L::kKReady, b));
            }
            // the V^T buffer's previous tile (i-2) is through both O products
            if (hf == 0)
                ok = __all_sync(0xFFFFFFFFu,
                                mbar_wait(bar(L::kVFree, b), ((i >> 1) & 1) ^ 1u, abort_flag));
            if (!ok) break;
            v_load(0);
            v_store(0);
#pragma unroll
            for (int g0 = kVG; g0 < kVB; g0 += kVG) {
                v_load(g0);
                v_store(g0);
            }
            if (ct == 0) buf_mask[2 * b + hf] = mask;  // for the softmax warps, released with v_ready
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(bar(L::kEmpty, st));
                if (hf == 1) mbar_arrive(bar(L::kVReady, b));
            }
        }
        if (!ok && lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    else {
        // ------------------------------------------------------------ softmax warps
        const int rt = warp >> 2;                   // row tile 0 or 1
        const int r = row0 + tid;                   // this thread's score row
        const bool row_ok = r < nb * G;
        const int jq = row_ok ? r / G : 0, gq = row_ok ? r % G : 0;
        const int pos = Ls - nb + jq;               // last key position the row may see
        const float score_scale = a.sm_scale * sk * 1.4426950408889634f;  // log2(e)
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>((warp & 3) * 32) << 16);
        const uint32_t scol = lane_addr + L::col_s(rt);
        float m_used = -INFINITY;
        uint64_t lsum2 = pk2(0.f, 0.f);  // the row sum, in two fp32 halves
        bool ok = true;
        for (int i = 0; i < ntiles && ok; ++i) {
            const int b = i & 1;
            // S(rt, i) is done, and with it O(rt, i-1)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kSReady, rt), i & 1, abort_flag));
            // the tile's valid-key masks (stored with its V^T)
            if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kVReady, b), (i >> 1) & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            const int k0 = key_tile(i) * kP2Keys;
            const int vis_n = row_ok ? min(kP2Keys, max(0, pos - k0 + 1)) : 0;
            const uint64_t vis0 = buf_mask[2 * b] & (vis_n >= 64 ? ~0ull : ((1ull << vis_n) - 1));
            const uint64_t vis1 = buf_mask[2 * b + 1] &
                                  (vis_n >= 128 ? ~0ull : vis_n <= 64 ? 0ull : ((1ull << (vis_n - 64)) - 1));
            const bool whole = __all_sync(0xFFFFFFFFu, (vis0 & vis1) == ~0ull);
            auto vis_bits = [&](int c) {  // the visible keys among columns 32c..32c+31
                return static_cast<uint32_t>((c < 2 ? vis0 : vis1) >> (32 * (c & 1)));
            };
            // pass 1: the row's maximum over the tile (raw extreme, scaled once, on a whole
            // tile).  Chunks 0 and 1, then 2 and 3, each pair loaded together; 2 and 3 stay in
            // registers for pass 2.
            uint32_t sa[32], sb[32];
            float mx = -INFINITY, ext = score_scale >= 0.f ? -INFINITY : INFINITY;
            auto chunk_max = [&](const uint32_t (&sc)[32], int c) {
                if (whole) {
                    ext = score_scale >= 0.f ? fmaxf(ext, extreme32<true>(sc)) : fminf(ext, extreme32<false>(sc));
                } else {
                    const uint32_t bits = vis_bits(c);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if ((bits >> e) & 1u) mx = fmaxf(mx, __uint_as_float(sc[e]) * score_scale);
                }
            };
            tmem_ld32(scol, sa);
            tmem_ld32(scol + 32, sb);
            tmem_wait_ld();
            chunk_max(sa, 0);
            chunk_max(sb, 1);
            tmem_ld32(scol + 64, sa);
            tmem_ld32(scol + 96, sb);
            tmem_wait_ld();
            chunk_max(sa, 2);
            chunk_max(sb, 3);
            if (whole) mx = ext * score_scale;
            float factor = 1.f;
            if (mx > -INFINITY) {
                if (m_used == -INFINITY) {
                    m_used = mx;
                } else if (mx > m_used + 8.f) {
                    factor = ex2(m_used - mx);
                    m_used = mx;
                }
            }
            if (__any_sync(0xFFFFFFFFu, factor != 1.f)) {
                // O(rt, i-1) is complete (covered by the commit of S(rt, i))
                lsum2 = mul_f32x2(lsum2, pk2(factor, factor));
#pragma unroll 1
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + L::col_o(rt) + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * factor);
                    tmem_st32(lane_addr + L::col_o(rt) + c0, o);
                }
            }
            // pass 2: P = 2^(score - m) as f16 pairs, written over the first half of each
            // chunk's own scores; chunks 2 and 3 from registers, each followed by the reload
            // of chunk 0 or 1 into its registers
            const float msub = m_used == -INFINITY ? 0.f : m_used;
            const uint64_t sub2 = pk2(-msub, -msub);
            const float mult = whole ? score_scale : 1.f;
            const uint64_t mul2 = pk2(mult, mult);
            auto chunk_p = [&](uint32_t (&sc)[32], int c) {
                if (!whole) {
                    const uint32_t bits = vis_bits(c);
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        sc[e] = __float_as_uint(((bits >> e) & 1u) ? __uint_as_float(sc[e]) * score_scale
                                                                    : -INFINITY);
                }
                // P = 2^x in fp32, rounded to f16 pairs for the product; the row sum adds the
                // fp32 values in packed pairs
                uint32_t p[16];
#pragma unroll
                for (int w = 0; w < 16; ++w) {
                    const float2 x = upk2(fma_f32x2(pk2u(sc[2 * w], sc[2 * w + 1]), mul2, sub2));
                    const float e0 = ex2(x.x), e1 = ex2(x.y);
                    p[w] = f16x2_from_f32(e0, e1);
                    lsum2 = add_f32x2(lsum2, pk2(e0, e1));
                }
                tmem_st16(scol + 32 * c, p);
            };
            chunk_p(sa, 2);
            tmem_ld32(scol, sa);       // chunk 0's scores: its columns are not written yet
            chunk_p(sb, 3);
            tmem_ld32(scol + 32, sb);  // chunk 1's
            tmem_wait_ld();
            chunk_p(sa, 0);
            chunk_p(sb, 1);
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(L::kPReady, rt));
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar(L::kODone, rt), 0, abort_flag));
        if (ok) {
            tc_fence_after();
            const float2 ls = upk2(lsum2);
            const float lsum = ls.x + ls.y;
            const float inv = lsum > 0.f ? sv / lsum : 0.f;
            uint4 *orow = reinterpret_cast<uint4 *>(
                a.out + ((static_cast<int64_t>(qr.q0) + jq) * a.n_q + kvh * G + gq) * HD);
#pragma unroll 1
            for (int c0 = 0; c0 < HD; c0 += 32) {
                uint32_t o[32];
                tmem_ld32(lane_addr + L::col_o(rt) + c0, o);
                tmem_wait_ld();
                if (row_ok) {
#pragma unroll
                    for (int c = 0; c < 32; c += 8) {
                        uint4 w;
                        w.x = bf16x2_from_f32(__uint_as_float(o[c]) * inv, __uint_as_float(o[c + 1]) * inv);
                        w.y = bf16x2_from_f32(__uint_as_float(o[c + 2]) * inv, __uint_as_float(o[c + 3]) * inv);
                        w.z = bf16x2_from_f32(__uint_as_float(o[c + 4]) * inv, __uint_as_float(o[c + 5]) * inv);
                        w.w = bf16x2_from_f32(__uint_as_float(o[c + 6]) * inv, __uint_as_float(o[c + 7]) * inv);
                        orow[(c0 + c) / 8] = w;
                    }
                }
            }
        } else if (lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kP2MmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int HD>
cudaError_t run_prefill(const DecodeArgs &d, cudaStream_t stream) {
    using L = PfSmem<HD>;
    const int row_bytes = d.n_kv * HD;
    const int box_rows = d.block_size >= kPfKeys ? kPfKeys : d.block_size;  // whole tile when one block holds it
    const int64_t rows = static_cast<int64_t>(d.num_blocks) * d.block_size;
    CUtensorMap tmk, tmv;
    cudaError_t err;
    if ((err = encode_cache_map(&tmk, d.key_cache, rows, row_bytes, L::kSeg, box_rows)) != cudaSuccess)
        return err;
    if ((err = encode_cache_map(&tmv, d.value_cache, rows, row_bytes, L::kSeg, box_rows)) != cudaSuccess)
        return err;
    PrefillArgs a;
    a.out = static_cast<__nv_bfloat16 *>(d.out);
    a.query = static_cast<const __nv_bfloat16 *>(d.query);
    a.qsl = d.qsl;
    a.qmax = d.qmax;
    a.qrows = d.qrows;
    a.block_tables = d.block_tables;
    a.max_blocks_per_seq = d.max_blocks_per_seq;
    a.seq_lens = d.seq_lens;
    a.num_seqs = d.num_seqs;
    a.n_q = d.n_q;
    a.n_kv = d.n_kv;
    a.group = d.n_q / d.n_kv;
    a.block_size = d.block_size;
    a.num_blocks = d.num_blocks;
    a.max_len = d.max_blocks_per_seq * d.block_size;
    a.sm_scale = d.sm_scale;
    a.k_scale = d.k_scale;
    a.v_scale = d.v_scale;
    a.scale_dtype = d.scale_dtype;
    a.status = d.status;
    a.box_rows = box_rows;
    // more than one tile of 128 rows per kv head (a multi-query call): 256 rows per CTA
    if constexpr (HD <= 128) {
        if (d.qsl != nullptr && d.qmax * a.group > kPfRows) {
            const size_t smem2 = Pf2Smem<HD>::kTotal + 1024;
            auto kern2 = prefill2_kernel<HD>;
            int occ2 = 0;  // also raises the kernel's shared memory limit, once per device
            if ((err = kernel_occupancy(kern2, kP2Warps * 32, smem2, &occ2)) != cudaSuccess)
                return err;
            a.row_tiles = (d.qmax * a.group + kP2Rows - 1) / kP2Rows;
            const int64_t ctas = static_cast<int64_t>(d.num_seqs) * a.row_tiles * d.n_kv;
            kern2<<<static_cast<unsigned>(ctas), kP2Warps * 32, smem2, stream>>>(tmk, tmv, a);
            return cudaGetLastError();
        }
    }
    const size_t smem = L::kTotal + 1024;
    auto kern = prefill_kernel<HD>;
    int occ = 0;  // also raises the kernel's shared memory limit, once per device
    if ((err = kernel_occupancy(kern, kPfWarps * 32, smem, &occ)) != cudaSuccess) return err;
    a.row_tiles = (d.qmax * a.group + kPfRows - 1) / kPfRows;
    const int64_t ctas = static_cast<int64_t>(d.num_seqs) * a.row_tiles * d.n_kv;
    kern<<<static_cast<unsigned>(ctas), kPfWarps * 32, smem, stream>>>(tmk, tmv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_attention(const DecodeArgs &d, cudaStream_t stream) {
    if (d.num_seqs == 0) return cudaSuccess;
    if (d.k_bf16 || d.v_bf16) return cudaErrorNotSupported;
    if (d.n_q / d.n_kv > kPfRows) return cudaErrorNotSupported;
    const int64_t row_tiles = (static_cast<int64_t>(d.qmax) * (d.n_q / d.n_kv) + kPfRows - 1) / kPfRows;
    if (row_tiles * d.n_kv * d.num_seqs > 0x7FFFFFFF) return cudaErrorNotSupported;
    switch (d.head_dim) {
        case 64: return run_prefill<64>(d, stream);
        case 128: return run_prefill<128>(d, stream);
        case 256: return run_prefill<256>(d, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace kvfp8
