// Causal multi-query attention over the FP8 (E4M3) cache for long query chunks (prefill),
// sm_103a tensor cores (tcgen05) with accumulators in tensor memory.
//
// What it computes is kvfp8_paged_attention_multi (llama.cpp "llama : Add FP8 KV-cache
// support (#28392)", tests/test-fp8.cpp check_fp8_attention: a batch of new tokens, each
// attending to every cached token up to its own position, on K/V rounded through the cache
// format).  The decode kernel covers up to 16 (query token, head) score columns per kv
// head; past that the rows form a real M dimension and the contraction is dense, so:
//
//  * Work unit: one CTA per (sequence, kv head, tile of 128 score rows).  A row is a
//    (query token j, head g of the kv head's group) pair, row = j*G + g, so all rows of a
//    tile share one K/V stream.  Keys are visited in tiles of 64 up to the tile's last
//    causal position.
//  * Warps 0-3 (one TMEM lane quarter each, one score row per thread):
//      - convert the tile's q rows bf16 -> f16 once, and each K tile e4m3 -> f16, into the
//        K-major 128-byte-swizzled operand layout; each V tile e4m3 -> f16 transposed
//        (V^T: head dims as rows, keys along K), so both products take K-major operands;
//      - thread 0 issues S = Q.K^T (tcgen05.mma kind::f16, M = 128, N = 64, fp32 in TMEM);
//      - every thread reads its row of S from TMEM, applies the causal mask and the online
//        softmax (log2 domain), writes P (f16) back over S in TMEM;
//      - thread 0 issues O += P.V (A = P from TMEM, B = V^T from shared memory, M = 128,
//        N = head_dim, fp32 in TMEM).  O is rescaled in TMEM only when a row's running
//        maximum grows by more than 2^8 (then P <= 2^8 stays well inside fp16);
//      - the epilogue reads O, divides by the row sum, applies v_scale and stores bf16.
//  * Warp 4 issues the TMA loads of the FP8 K/V tiles (the per-head-segment boxes of the
//    decode kernel's cache map) into a two-stage ring.
//  * All waits are bounded (mbarriers with a clock64 limit); a wait that runs out sets
//    KVFP8_DEV_TIMEOUT.  Tensor memory is always released before the CTA exits.
#include "paged_decode_kernel.cuh"

namespace kvfp8 {
namespace {

constexpr int kPfRows = 128;   // score rows per CTA (TMEM lanes)
constexpr int kPfKeys = 64;    // keys per tile
constexpr int kPfThreads = 160;  // 4 compute warps + 1 producer warp

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
// Instruction descriptor, kind::f16: f16 A and B, fp32 D, both K-major, M x N.
__host__ __device__ constexpr uint32_t f16_idesc(int m, int n) {
    return (1u << 4) | (static_cast<uint32_t>(n >> 3) << 17) | (static_cast<uint32_t>(m >> 4) << 24);
}
// byte offset of 16-byte chunk c of row r in a 128-byte-swizzled K-major block
__device__ __forceinline__ uint32_t sw128(int r, int c) {
    return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
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
};

// Shared-memory plan (byte offsets from a 1024-aligned base).
template <int HD>
struct PfSmem {
    static constexpr int kSeg = HD >= 128 ? 128 : 64;             // fp8 TMA box row (swizzle span)
    static constexpr int kSegs = HD / kSeg;
    static constexpr int kQ = 0;                                   // Q f16: HD/64 blocks x 128 rows x 128 B
    static constexpr int kK = kQ + HD * 256;                       // K f16: HD/64 blocks x 64 rows x 128 B
    static constexpr int kV = kK + HD * 128;                       // V^T f16: HD rows x 128 B
    static constexpr int kStage = kV + HD * 128;                   // fp8 K then V, per stage
    static constexpr int kStageBytes = 2 * kPfKeys * HD;
    static constexpr int kBars = kStage + 2 * kStageBytes;         // full[2], empty[2], s, o, wg
    static constexpr int kMeta = kBars + 8 * 8;                    // valid-key mask per stage
    static constexpr int kMisc = kMeta + 16;                       // tmem base, abort flag
    static constexpr int kTotal = kMisc + 16;
    static constexpr uint32_t kTmemCols = HD + 64 <= 128 ? 128 : (HD + 64 <= 256 ? 256 : 512);
    static constexpr uint32_t kColS = 0;   // S (64 fp32 columns); P (f16) reuses its first 32
    static constexpr uint32_t kColO = 64;  // O (HD fp32 columns)
};

template <int HD>
__global__ void __launch_bounds__(kPfThreads)
prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
               const PrefillArgs a) {
    using L = PfSmem<HD>;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *bp = smem_raw + (base - raw);
    const uint32_t bar_full = base + L::kBars, bar_empty = bar_full + 16;
    const uint32_t bar_s = bar_full + 32, bar_o = bar_full + 40, bar_wg = bar_full + 48;
    volatile uint64_t *meta = reinterpret_cast<volatile uint64_t *>(bp + L::kMeta);
    volatile uint32_t *tmem_slot = reinterpret_cast<volatile uint32_t *>(bp + L::kMisc);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(bp + L::kMisc + 4);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int seq = blockIdx.x, tile = blockIdx.y, kvh = blockIdx.z;

    const float sk = load_scale(a.k_scale, a.scale_dtype);
    const float sv = load_scale(a.v_scale, a.scale_dtype);
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (seq == 0 && tile == 0 && kvh == 0 && tid == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    // this sequence's query rows and cached length (flagged once, by its first CTA)
    const int raw_nq = a.qsl[seq + 1] - a.qsl[seq];
    const QueryRange qr = query_range(a.qsl, seq, a.qmax, a.qrows);
    int Lraw = a.seq_lens[seq];
    const int Ls = min(max(Lraw, 0), a.max_len);
    if (tile == 0 && kvh == 0 && tid == 0 &&
        (qr.count != raw_nq || Lraw < 0 || Lraw > a.max_len || qr.count > Ls))
        flag(a.status, KVFP8_DEV_BAD_BLOCK);
    const int nb = qr.count, G = a.group;
    const int row0 = tile * kPfRows;                 // first score row of this tile
    if (row0 >= nb * G) return;                      // no rows here
    const int j_last = min(nb, (row0 + kPfRows + G - 1) / G) - 1;
    const int kend = Ls - nb + j_last + 1;           // keys the tile's last row may see
    const int ntiles = kend > 0 ? (kend + kPfKeys - 1) / kPfKeys : 0;

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
        mbar_init(bar_full, 1);
        mbar_init(bar_full + 8, 1);
        mbar_init(bar_empty, 4);
        mbar_init(bar_empty + 8, 4);
        mbar_init(bar_s, 1);
        mbar_init(bar_o, 1);
        mbar_init(bar_wg, 128);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0) {
        tmem_alloc(base + L::kMisc, L::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 4 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 4) {
        // ------------------------------------------------------------ producer warp
        const int32_t *bt = a.block_tables + static_cast<int64_t>(seq) * a.max_blocks_per_seq;
        const int bs = a.block_size, br = a.box_rows;
        bool aborted = false;
        int issued = 0;
        for (int i = 0; i < ntiles && !aborted; ++i) {
            const int stage = i & 1;
            const uint32_t full = bar_full + 8 * stage;
            if (lane == 0) {
                if (!mbar_wait(bar_empty + 8 * stage, ((i >> 1) & 1) ^ 1u, abort_flag)) {
                    aborted = true;
                } else {
                    // one box per head segment and box_rows keys; keys past kend or in a bad
                    // block are left out of the load and of the valid mask
                    uint64_t mask = 0;
                    int boxes = 0;
                    const int nbox = kPfKeys / br;
                    int rows[kPfKeys / 8];
                    for (int p = 0; p < nbox; ++p) {
                        const int t = i * kPfKeys + p * br;
                        rows[p] = -1;
                        if (t >= kend) continue;
                        const int e = t / bs;
                        const int blk = e < a.max_blocks_per_seq ? bt[e] : -1;
                        if (blk < 0 || blk >= a.num_blocks) {
                            flag(a.status, KVFP8_DEV_BAD_BLOCK);
                            continue;
                        }
                        rows[p] = blk * bs + t % bs;
                        ++boxes;
                        const int nk = min(br, kend - t);
                        mask |= (nk >= 64 ? ~0ull : ((1ull << nk) - 1)) << (p * br);
                    }
                    meta[stage] = mask;
                    if (boxes > 0) {
                        mbar_arrive_tx(full, static_cast<uint32_t>(boxes * L::kSegs * 2 * br * L::kSeg));
                        const uint32_t kst = base + L::kStage + stage * L::kStageBytes;
                        const uint32_t vst = kst + kPfKeys * HD;
                        for (int p = 0; p < nbox; ++p) {
                            if (rows[p] < 0) continue;
                            for (int sgi = 0; sgi < L::kSegs; ++sgi) {
                                const uint32_t off = static_cast<uint32_t>(sgi * kPfKeys * L::kSeg + p * br * L::kSeg);
                                tma_load_3d(kst + off, &tmk, 0, kvh * L::kSegs + sgi, rows[p], full);
                                tma_load_3d(vst + off, &tmv, 0, kvh * L::kSegs + sgi, rows[p], full);
                            }
                        }
                    } else {
                        mbar_arrive(full);
                    }
                    ++issued;
                }
            }
            aborted = __shfl_sync(0xFFFFFFFFu, aborted, 0);
        }
        if (aborted && lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
            // let copies already issued land before the CTA's shared memory goes away
            const volatile int32_t never = 0;
            for (int k = max(0, issued - 2); k < issued; ++k)
                mbar_wait(bar_full + 8 * (k & 1), (k >> 1) & 1, &never);
        }
    } else {
        // ------------------------------------------------------------ compute warps
        const int r = row0 + tid;                   // this thread's score row (TMEM lane tid)
        const bool row_ok = r < nb * G;
        const int jq = row_ok ? r / G : 0, gq = row_ok ? r % G : 0;
        const int pos = Ls - nb + jq;               // last key position the row may see
        const float score_scale = a.sm_scale * sk * 1.4426950408889634f;  // log2(e)
        const uint32_t lane_addr = tmem + (static_cast<uint32_t>(warp * 32) << 16);
        uint32_t wg_phase = 0;
        bool ok = true;
        // warp-group barrier with a bounded wait
        auto wg_sync = [&]() {
            mbar_arrive(bar_wg);
            const bool done = mbar_wait(bar_wg, wg_phase, abort_flag);
            wg_phase ^= 1u;
            return done;
        };

        // q row -> f16, 128-byte-swizzled K-major blocks of 64 head dims
        {
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
                *reinterpret_cast<uint4 *>(bp + L::kQ + (c >> 3) * (kPfRows * 128) + sw128(tid, c & 7)) = h;
            }
        }

        float m_used = -INFINITY, lsum = 0.f;
        int i = 0;
        for (; i < ntiles && ok; ++i) {
            const int stage = i & 1;
            // the tile's FP8 bytes have landed; the previous tile's products are done (its
            // K, V^T and P may be overwritten)
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_full + 8 * stage, (i >> 1) & 1, abort_flag));
            if (ok && i > 0) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o, (i - 1) & 1, abort_flag));
            if (!ok) break;
            const uint64_t mask = meta[stage];
            const uint8_t *kst = bp + L::kStage + stage * L::kStageBytes;
            const uint8_t *vst = kst + kPfKeys * HD;
            // K: 64 keys x HD/16 chunks of 16 fp8 -> f16 (invalid keys: zeros)
            for (int task = tid; task < kPfKeys * (HD / 16); task += 128) {
                const int key = task / (HD / 16), c = task % (HD / 16);  // dims 16c .. 16c+15
                const int sgi = (16 * c) / L::kSeg, within = (16 * c) % L::kSeg;
                uint4 w = *reinterpret_cast<const uint4 *>(kst + sgi * kPfKeys * L::kSeg +
                                                           swz<L::kSeg>(key, within >> 4));
                if (!((mask >> key) & 1ull)) w = make_uint4(0u, 0u, 0u, 0u);
                uint4 h0, h1;
                h0.x = f16x2_from_e4m3x2(w.x);
                h0.y = f16x2_from_e4m3x2_hi(w.x);
                h0.z = f16x2_from_e4m3x2(w.y);
                h0.w = f16x2_from_e4m3x2_hi(w.y);
                h1.x = f16x2_from_e4m3x2(w.z);
                h1.y = f16x2_from_e4m3x2_hi(w.z);
                h1.z = f16x2_from_e4m3x2(w.w);
                h1.w = f16x2_from_e4m3x2_hi(w.w);
                const int kb = (16 * c) / 64, c8 = ((16 * c) % 64) / 8;
                uint8_t *kdst = bp + L::kK + kb * (kPfKeys * 128);
                *reinterpret_cast<uint4 *>(kdst + sw128(key, c8)) = h0;
                *reinterpret_cast<uint4 *>(kdst + sw128(key, c8 + 1)) = h1;
            }
            // V^T: key pairs x HD/16 chunks; dim n of keys (2kp, 2kp+1) -> row n, K index 2kp
            for (int task = tid; task < (kPfKeys / 2) * (HD / 16); task += 128) {
                const int kp = task / (HD / 16), c = task % (HD / 16);
                const int sgi = (16 * c) / L::kSeg, within = (16 * c) % L::kSeg;
                const uint8_t *vseg = vst + sgi * kPfKeys * L::kSeg;
                uint4 va = *reinterpret_cast<const uint4 *>(vseg + swz<L::kSeg>(2 * kp, within >> 4));
                uint4 vb = *reinterpret_cast<const uint4 *>(vseg + swz<L::kSeg>(2 * kp + 1, within >> 4));
                if (!((mask >> (2 * kp)) & 1ull)) va = make_uint4(0u, 0u, 0u, 0u);
                if (!((mask >> (2 * kp + 1)) & 1ull)) vb = make_uint4(0u, 0u, 0u, 0u);
                const uint32_t aw[4] = {va.x, va.y, va.z, va.w}, bw[4] = {vb.x, vb.y, vb.z, vb.w};
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                    // bytes (a_d, b_d) for dims d = 4*q4 .. 4*q4+3 of the chunk
                    const uint32_t lo = __byte_perm(aw[q4], bw[q4], 0x5140);  // a0 b0 a1 b1
                    const uint32_t hi = __byte_perm(aw[q4], bw[q4], 0x7362);  // a2 b2 a3 b3
                    const uint32_t pv[4] = {f16x2_from_e4m3x2(lo), f16x2_from_e4m3x2_hi(lo),
                                            f16x2_from_e4m3x2(hi), f16x2_from_e4m3x2_hi(hi)};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int n = 16 * c + 4 * q4 + e;   // head dim = row of V^T
                        *reinterpret_cast<uint32_t *>(bp + L::kV + sw128(n, (2 * kp) >> 3) +
                                                      ((2 * kp) & 7) * 2) = pv[e];
                    }
                }
            }
            fence_proxy_async();
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + 8 * stage);  // the FP8 stage may be refilled
            ok = __all_sync(0xFFFFFFFFu, wg_sync());
            if (!ok) break;
            if (tid == 0) {  // S = Q . K^T over HD/16 k-steps
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < HD / 16; ++k) {
                    const uint64_t ad = sw128_desc(base + L::kQ + (k >> 2) * (kPfRows * 128) + (k & 3) * 32);
                    const uint64_t bd = sw128_desc(base + L::kK + (k >> 2) * (kPfKeys * 128) + (k & 3) * 32);
                    umma_ss(tmem + L::kColS, ad, bd, f16_idesc(kPfRows, kPfKeys), k > 0 ? 1u : 0u);
                }
                umma_commit(bar_s);
            }
            ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_s, i & 1, abort_flag));
            if (!ok) break;
            tc_fence_after();
            uint32_t s[2][32];
            tmem_ld32(lane_addr + L::kColS, s[0]);
            tmem_ld32(lane_addr + L::kColS + 32, s[1]);
            tmem_wait_ld();
            // causal mask, scale, running maximum
            const int k0 = i * kPfKeys;
            float mx = -INFINITY;
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
                for (int c = 0; c < 32; ++c) {
                    const int key = 32 * h + c;
                    const bool vis = row_ok && k0 + key <= pos && ((mask >> key) & 1ull);
                    const float v = vis ? __uint_as_float(s[h][c]) * score_scale : -INFINITY;
                    s[h][c] = __float_as_uint(v);
                    mx = fmaxf(mx, v);
                }
            // rescale O only when the maximum grew by more than 2^8 (first visible keys: O
            // is still zero for this row, nothing to rescale)
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
                lsum *= factor;
#pragma unroll 1
                for (int c0 = 0; c0 < HD; c0 += 32) {
                    uint32_t o[32];
                    tmem_ld32(lane_addr + L::kColO + c0, o);
                    tmem_wait_ld();
#pragma unroll
                    for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * factor);
                    tmem_st32(lane_addr + L::kColO + c0, o);
                }
            }
            // P = 2^(s - m), f16 pairs over the first 32 columns of S
            uint32_t p[32];
            const float msub = m_used == -INFINITY ? 0.f : m_used;
#pragma unroll
            for (int c = 0; c < 32; ++c) {
                const int h = c >> 4, e = (2 * c) & 31;
                const float p0 = ex2(__uint_as_float(s[h][e]) - msub);
                const float p1 = ex2(__uint_as_float(s[h][e + 1]) - msub);
                lsum += p0 + p1;
                p[c] = f16x2_from_f32(p0, p1);
            }
            tmem_st32(lane_addr + L::kColS, p);
            tmem_wait_st();
            tc_fence_before();
            ok = __all_sync(0xFFFFFFFFu, wg_sync());
            if (!ok) break;
            if (tid == 0) {  // O += P . V over 64/16 k-steps; A from TMEM, B = V^T
                tc_fence_after();
#pragma unroll
                for (int k = 0; k < kPfKeys / 16; ++k) {
                    const uint64_t bd = sw128_desc(base + L::kV + k * 32);
                    umma_ts(tmem + L::kColO, tmem + L::kColS + 8 * k, bd, f16_idesc(kPfRows, HD),
                            (i > 0 || k > 0) ? 1u : 0u);
                }
                umma_commit(bar_o);
            }
        }
        if (ok) ok = __all_sync(0xFFFFFFFFu, mbar_wait(bar_o, (ntiles - 1) & 1, abort_flag));
        if (ok) {
            tc_fence_after();
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
            // let products already issued finish before tensor memory is released
            const volatile int32_t never = 0;
            if (i > 0) mbar_wait(bar_o, (i - 1) & 1, &never);
            mbar_wait(bar_s, i & 1, &never);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, L::kTmemCols);
    }
}

template <int HD>
cudaError_t run_prefill(const DecodeArgs &d, cudaStream_t stream) {
    using L = PfSmem<HD>;
    const int row_bytes = d.n_kv * HD;
    const int box_rows = d.block_size >= kChunkTokens ? kChunkTokens : d.block_size;
    const int64_t rows = static_cast<int64_t>(d.num_blocks) * d.block_size;
    CUtensorMap tmk, tmv;
    cudaError_t err;
    if ((err = encode_cache_map(&tmk, d.key_cache, rows, row_bytes, L::kSeg, box_rows)) != cudaSuccess)
        return err;
    if ((err = encode_cache_map(&tmv, d.value_cache, rows, row_bytes, L::kSeg, box_rows)) != cudaSuccess)
        return err;
    const size_t smem = L::kTotal + 1024;
    auto kern = prefill_kernel<HD>;
    if ((err = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    static_cast<int>(smem))) != cudaSuccess)
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
    const int tiles = (d.qmax * a.group + kPfRows - 1) / kPfRows;
    dim3 grid(d.num_seqs, tiles, d.n_kv);
    kern<<<grid, kPfThreads, smem, stream>>>(tmk, tmv, a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prefill_attention(const DecodeArgs &d, cudaStream_t stream) {
    if (d.num_seqs == 0) return cudaSuccess;
    if (d.qsl == nullptr || d.k_bf16 || d.v_bf16) return cudaErrorNotSupported;
    if (d.n_q / d.n_kv > kPfRows) return cudaErrorNotSupported;
    if ((d.qmax * (d.n_q / d.n_kv) + kPfRows - 1) / kPfRows > 65535) return cudaErrorNotSupported;
    switch (d.head_dim) {
        case 64: return run_prefill<64>(d, stream);
        case 128: return run_prefill<128>(d, stream);
        case 256: return run_prefill<256>(d, stream);
        default: return cudaErrorNotSupported;
    }
}

}  // namespace kvfp8
