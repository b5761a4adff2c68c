// Single-query (decode) paged attention over an FP8 (E4M3) KV cache, sm_103a.
//
// What it computes (llama.cpp "llama : Add FP8 KV-cache support (#28392)",
// tests/test-fp8.cpp check_fp8_attention and llama-graph.cpp
// build_attn_scale_kv_inputs/_output): for every sequence b and query head h,
//   s_t = sm_scale * k_scale * q[b,h] . dec(K_t[h/G]),  out = v_scale * softmax(s) . dec(V[h/G])
// over the seq_lens[b] tokens reached through block_tables[b].
//
// Design (HBM-bound: 1 byte of K and 1 of V per element, G = n_q/n_kv flops per byte):
//  * Work split: the cache is cut into 16-token chunks; the chunks of all sequences are
//    laid end to end and each CTA of a fixed grid (one to three per SM; fewer when there
//    are fewer chunks than CTAs) takes an equal contiguous, non-empty range, whatever
//    the length mix.  A sequence that lies inside one CTA is finished there; otherwise
//    each CTA writes a partial (normalized o, log2-sum-exp) and a combine kernel merges
//    them.  Partial (seq, cta) pairs are stored at index seq+cta, which is unique because
//    both grow monotonically along the chunk order.  A one-CTA plan kernel computes the
//    chunk prefix over the sequences first, and one record per CTA (its chunk range and
//    first sequence, so a CTA starts with one read).  Plan -> decode -> combine are chained
//    as programmatic dependent launches, so each grid's launch and prologue overlap its
//    predecessor; while a decode CTA waits for the plan it prefetches its slice of the
//    block tables into L2, and its producer prefetches each next sequence's query rows.
//  * One CTA = one producer warp + one consumer warp per kv head of its head group (the
//    kv heads split into equal groups of at most 8, or 4 for 16 FP8 score columns at head_dim
//    128, a second grid dimension; one group when n_kv is at most that).  A 16-token chunk of a block holds all kv heads of those tokens (16
//    contiguous rows of n_kv*head_dim bytes), and a CTA fetches its group's part of them,
//    so the producer issues TMA tensor loads of [16 rows x 128 B] boxes (one per head and
//    128-byte segment of head_dim) with 128-byte swizzle into a multi-stage ring, on an
//    mbarrier per stage; the block-table entries come in 32 at a time, one per lane.
//  * Consumer warp (one kv head, all G query heads of its group) per chunk:
//      S^T[16 tok x 8 heads]  = K[16 x d] . q^T     mma.sync m16n8k16 f16 -> f32
//        K fragments: ldmatrix of the fp8 bytes as b16 pairs, cvt e4m3x2 -> f16x2;
//        the head-dim order inside a k-step is permuted identically for q.
//      online softmax (exp2, log2-scaled scores) per head column
//      P^T -> movmatrix.trans -> B fragments (tokens x heads) without shared memory
//      O^T[d x 8 heads]      += V^T[d x 16 tok] . P^T    mma.sync m16n8k16
//        V fragments: ldmatrix.trans gives two tokens' byte pairs, one prmt regroups them
//        into token pairs per head-dim, cvt e4m3x2 -> f16x2; output dims are permuted
//        and undone at the store.
//    The cache bytes convert to fp16 exactly; q (bf16) converts exactly inside the fp16
//    range; accumulation is fp32.  The scales are folded: k_scale * sm_scale * log2(e)
//    into the scores, v_scale into the final normalization.
//  * Every wait is bounded; a wait that runs out sets KVFP8_DEV_TIMEOUT, the CTA drains
//    its outstanding copies (again bounded) and returns.
//  * Mixed cache dtypes (one side E4M3, the other bf16 without a scale): the bf16 side's
//    chunk is twice as wide in shared memory and its fragments feed bf16 mma.sync directly
//    (K against bf16 q; V against p split into two bf16 parts).
//
// This header holds the kernels and the templated launcher; paged_decode.cu instantiates
// the all-E4M3 variants, paged_decode_mixed.cu the mixed ones.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdlib>
#include <mutex>

#include "kvfp8_device.cuh"
#include "kvfp8_internal.h"

namespace kvfp8 {
namespace {

constexpr int kMaxKvHeads = 8;                 // consumer warps per CTA
constexpr int kThreadsMax = 32 * (kMaxKvHeads + 1);
#ifdef KVFP8_TEST_WITHHOLD_FIRST_CHUNK
// Test-only build (a separate library file, never the package's): every CTA's producer
// withholds the copy of its first chunk and every wait gives up after ~1e5 cycles, so the
// consumers' bounded waits run out while no copy is in flight, driving the timeout path.
constexpr long long kWaitCycles = 100000LL;
constexpr bool kWithholdFirstChunk = true;
#else
constexpr long long kWaitCycles = 4000000000LL;  // ~2 s at 2 GHz
constexpr bool kWithholdFirstChunk = false;
#endif

struct ChunkMeta {
    int32_t seq;
    int32_t tok0;
    int32_t nvalid;
    int32_t flags;
};
enum : int32_t { kFirst = 1, kLast = 2, kDirect = 4, kDone = 8 };

// The plan's record for one decode CTA: chunk range [lo, hi) (empty past the effective
// grid), the sequence s holding chunk lo, its chunk range [cs, ce) and length L.
struct CtaPlan {
    int32_t lo, hi, s, cs, ce, L, pad0, pad1;
};

struct KernelArgs {
    __nv_bfloat16 *out;
    const __nv_bfloat16 *query;
    const int32_t *block_tables;
    int32_t max_blocks_per_seq;
    const int32_t *seq_lens;
    int32_t num_seqs;
    int32_t n_q, n_kv, group, block_size, num_blocks;
    int32_t hpc;  // kv heads per CTA (head group size); blockIdx.y is the head group
    int32_t max_len;  // max_blocks_per_seq * block_size
    float sm_scale;
    const void *k_scale;
    const void *v_scale;
    int32_t scale_dtype;
    const int32_t *cstart;
    const CtaPlan *cta_plan;  // one record per CTA (from the plan kernel)
    float *part_lse;
    float *part_o;
    uint32_t *status;
    int32_t num_ctas;
    int32_t stages;
    int32_t box_rows;  // 16, or 8 for 8-token blocks
    int32_t whole_box;  // 1: one TMA box covers a chunk's rows for all heads (see host)
    // multi-query (causal) form: sequence b's query rows start at qsl[b] (nullptr: one
    // query per sequence, row b); rows_per_seq = max query count * n_q
    const int32_t *qsl;
    int32_t rows_per_seq;
    int32_t qrows;  // rows of query and out (multi-query form)
    // mixed cache dtypes: 1 = that side's cache is bf16 and carries no scale
    int32_t k_bf16, v_bf16;
};

// Query rows [q0, q0 + count) of sequence b in the multi-query form, or count 0 when the
// sequence's query_start_loc entries are out of range (flagged by the plan kernel).
struct QueryRange {
    int q0, count;
};
__device__ __forceinline__ QueryRange query_range(const int32_t *qsl, int b, int qmax, int qrows) {
    const int q0 = qsl[b], n = qsl[b + 1] - q0;
    if (q0 < 0 || n < 0 || n > qmax || q0 + n > qrows) return QueryRange{0, 0};
    return QueryRange{q0, n};
}

// ---------------------------------------------------------------- PTX wrappers


__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for the phase of the given parity.  Gives up when *abort is raised by
// another warp, or after kWaitCycles.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          const volatile int32_t *abort) {
    if (mbar_try(bar, parity)) return true;
    const long long t0 = clock64();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (mbar_try(bar, parity)) return true;
        if ((it & 15u) == 15u) {
            if (*abort) return false;
            if (clock64() - t0 > kWaitCycles) return false;
        }
    }
    return false;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap *map, int c0, int c1,
                                            int c2, uint32_t bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ uint32_t movm_t(uint32_t x) {
    uint32_t r;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(r) : "r"(x));
    return r;
}

__device__ __forceinline__ void mma16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void mma16816_bf16(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// Byte offset of 16-byte chunk cc of row `row` inside a [16 rows x SEG bytes] box that
// TMA wrote with SEG-byte swizzle (box base aligned to the swizzle span).
template <int SEG>
__device__ __forceinline__ uint32_t swz(int row, int cc) {
    const int x = (SEG == 128) ? (row & 7) : ((row >> 1) & 3);
    return static_cast<uint32_t>(row * SEG + ((cc ^ x) << 4));
}

// ---------------------------------------------------------------- kernels

// Running merge of split-KV partials (lse_c in log2 units, o_c normalized):
// sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M) with M the running maximum; a part with no
// visible token (lse = -inf) adds nothing.
struct PartMerge {
    float M = -INFINITY, den = 0.f;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    __device__ __forceinline__ void add(float l, const float4 &v) {
        if (l == -INFINITY) return;
        if (l > M) {  // rescale what has been summed so far
            const float r = ex2(M - l);  // 0 while M is still -inf
            den *= r;
            acc.x *= r;
            acc.y *= r;
            acc.z *= r;
            acc.w *= r;
            M = l;
        }
        const float w = ex2(l - M);
        den += w;
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
    }
    // four bf16 outputs: scale * acc / den (zeros when no part saw a token)
    __device__ __forceinline__ uint2 result(float scale) const {
        const float inv = den > 0.f ? scale / den : 0.f;
        return make_uint2(bf16x2_from_f32(acc.x * inv, acc.y * inv),
                          bf16x2_from_f32(acc.z * inv, acc.w * inv));
    }
};

__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Per-call plan, one CTA of 1024 threads:
//  * cstart[s] = first chunk of sequence s (exclusive prefix of its 16-token chunk
//    counts), cstart[num_seqs] = total;
//  * the output rows of empty sequences are zeroed (no CTA visits them);
//  * one CtaPlan record per decode CTA (the prefix and the clamped lengths are kept in
//    shared memory when they fit, else read back from global memory).
constexpr int kPlanSmemSeqs = 4096;

__global__ void __launch_bounds__(1024)
plan_kernel(const int32_t *seq_lens, const int32_t *qsl, int32_t qmax, int32_t qrows,
            int32_t num_seqs, int32_t max_len, int32_t num_ctas, int32_t *cstart,
            CtaPlan *cta_plan, __nv_bfloat16 *out, int32_t out_row_elems, uint32_t *status) {
    pdl_trigger();  // the decode grid may start its prologue; it waits for this grid's writes
    __shared__ int32_t warp_tot[32];
    __shared__ int32_t carry;
    __shared__ int32_t cs_smem[kPlanSmemSeqs + 1];
    __shared__ int32_t len_smem[kPlanSmemSeqs];
    const bool in_smem = num_seqs <= kPlanSmemSeqs;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) carry = 0;
    __syncthreads();
    for (int base = 0; base < num_seqs; base += 1024) {
        const int i = base + tid;
        int n = 0;
        if (i < num_seqs) {
            int L = seq_lens[i];
            if (L < 0 || L > max_len) {
                flag(status, KVFP8_DEV_BAD_BLOCK);
                L = L < 0 ? 0 : max_len;
            }
            int nq = 1;  // query rows of the sequence
            if (qsl) {
                const int raw = qsl[i + 1] - qsl[i];
                nq = query_range(qsl, i, qmax, qrows).count;
                if (nq != raw) flag(status, KVFP8_DEV_BAD_BLOCK);  // rows out of range: skipped
                if (nq > L) flag(status, KVFP8_DEV_BAD_BLOCK);     // positions below zero
            }
            n = nq > 0 ? (L + kChunkTokens - 1) / kChunkTokens : 0;
            if (in_smem) len_smem[i] = L;
        }
        unsigned empty = __ballot_sync(0xFFFFFFFFu, i < num_seqs && n == 0);
        while (empty) {  // this warp zeroes the output rows of its empty sequences
            const int b = base + warp * 32 + __ffs(empty) - 1;
            empty &= empty - 1;
            const QueryRange qr = qsl ? query_range(qsl, b, qmax, qrows) : QueryRange{b, 1};
            const int64_t r0 = qr.q0, nr = qr.count;
            uint4 *rows = reinterpret_cast<uint4 *>(out + r0 * out_row_elems);
            for (int64_t k = lane; k < nr * out_row_elems / 8; k += 32)
                rows[k] = make_uint4(0u, 0u, 0u, 0u);
        }
        int x = n;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xFFFFFFFFu, x, o);
            if (lane >= o) x += y;
        }
        if (lane == 31) warp_tot[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = warp_tot[lane];
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xFFFFFFFFu, w, o);
                if (lane >= o) w += y;
            }
            warp_tot[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int before = carry + (warp > 0 ? warp_tot[warp - 1] : 0) + x - n;
        if (i < num_seqs) {
            cstart[i] = before;
            if (in_smem) cs_smem[i] = before;
        }
        __syncthreads();
        if (tid == 0) carry += warp_tot[31];
        __syncthreads();
    }
    const int32_t total = carry;
    if (tid == 0) {
        cstart[num_seqs] = total;
        if (in_smem) cs_smem[num_seqs] = total;
    }
    __syncthreads();  // cstart complete (block-visible)
    // Each decode CTA's record: its chunk range and the sequence holding its first chunk,
    // the last s with cstart[s] <= lo.
    const int32_t *cs_tab = in_smem ? cs_smem : cstart;
    const int64_t T = total;
    const int64_t P = T < num_ctas ? T : num_ctas;
    for (int c = tid; c < num_ctas; c += blockDim.x) {
        CtaPlan r = {0, 0, 0, 0, 0, 0, 0, 0};
        if (c < P) {
            r.lo = static_cast<int32_t>(static_cast<int64_t>(c) * T / P);
            r.hi = static_cast<int32_t>(static_cast<int64_t>(c + 1) * T / P);
            int lo = 0, hi = num_seqs;  // invariant: cs_tab[lo] <= r.lo < cs_tab[hi]
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (cs_tab[mid] <= r.lo) lo = mid; else hi = mid;
            }
            r.s = lo;
            r.cs = cs_tab[lo];
            r.ce = cs_tab[lo + 1];
            r.L = in_smem ? len_smem[lo] : min(max(seq_lens[lo], 0), max_len);
        }
        cta_plan[c] = r;
    }
}

// Chunks of sequence i (and its clamped length): 16-token chunks of its L cached tokens, or
// none when it has no query rows.  The same rule the plan kernel applies.
__device__ __forceinline__ int seq_chunks(const KernelArgs &a, int i, int &L) {
    L = min(max(a.seq_lens[i], 0), a.max_len);
    const int nq = a.qsl ? query_range(a.qsl, i, a.rows_per_seq / a.n_q, a.qrows).count : 1;
    return nq > 0 ? (L + kChunkTokens - 1) / kChunkTokens : 0;
}

// Bring the query rows a CTA's consumers will read for sequence s (its head group's rows,
// or the sequence's query tokens in the multi-query form, at most 32 KiB) into L2 ahead of
// their first chunk: the producer runs up to a ring of chunks ahead of the consumers, so a
// consumer starting a sequence finds its q in L2 instead of waiting on HBM.
template <int HD>
__device__ __forceinline__ void prefetch_q(const KernelArgs &a, int s, int h0, int lane) {
    const __nv_bfloat16 *q;
    int64_t bytes;
    if (a.qsl != nullptr) {
        const QueryRange qr = query_range(a.qsl, s, a.rows_per_seq / a.n_q, a.qrows);
        q = a.query + static_cast<int64_t>(qr.q0) * a.n_q * HD;
        bytes = static_cast<int64_t>(qr.count) * a.n_q * HD * 2;
        bytes = bytes < 32768 ? bytes : 32768;
    } else {
        q = a.query + (static_cast<int64_t>(s) * a.n_q + h0 * a.group) * HD;
        bytes = static_cast<int64_t>(a.hpc) * a.group * HD * 2;
    }
    const char *p = reinterpret_cast<const char *>(q);
    for (int64_t off = static_cast<int64_t>(lane) * 128; off < bytes; off += 32 * 128)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p + off));
}

// The CTA whose chunk range contains chunk x (ranges are [c*T/P, (c+1)*T/P), P <= T).
__device__ __forceinline__ int cta_of(int64_t x, int64_t T, int64_t P) {
    return static_cast<int>(((x + 1) * P - 1) / T);
}

// Merge the partials (seq, c), c in [cf, cl], of every sequence that crossed CTA ranges:
// out = v_scale * sum_c 2^(lse_c - M) o_c / sum_c 2^(lse_c - M).  One thread per four output
// dims of one head.  A single pass with a running maximum: the loads of all partials are
// independent of one another (the loop is unrolled), so they are in flight together.
// Launched as a programmatic dependent of the decode grid.
// kCombineSlices slices of a sequence's parts are merged side by side (256 threads each),
// then the slices' running states are merged: sequences cut into many parts (few, long
// sequences over a full grid) get several loads in flight per output element.
template <int HD, int kCombineSlices>
__global__ void __launch_bounds__(256 * kCombineSlices) combine_kernel(const KernelArgs a) {
    constexpr int TPH = HD / 4;     // threads per head
    constexpr int HPB = 256 / TPH;  // heads per CTA
    __shared__ float sm_m[kCombineSlices][256], sm_den[kCombineSlices][256];
    __shared__ float4 sm_acc[kCombineSlices][256];
    const int seq = blockIdx.x;
    const int slice = threadIdx.x / 256, t = threadIdx.x % 256;
    const int row = blockIdx.y * HPB + t / TPH;  // row of the sequence
    const int d = (t % TPH) * 4;
    pdl_wait();  // the decode grid's partials are visible from here on
    const float sk = a.k_bf16 ? 1.f : load_scale(a.k_scale, a.scale_dtype);
    const float sv = a.v_bf16 ? 1.f : load_scale(a.v_scale, a.scale_dtype);
    const int64_t cs = a.cstart[seq], ce = a.cstart[seq + 1], T = a.cstart[a.num_seqs];
    if (!scale_ok(sk) || !scale_ok(sv)) return;  // uniform over the CTA
    if (ce == cs) return;                        // empty: zeroed by the plan kernel
    const int64_t P = min(static_cast<int64_t>(a.num_ctas), T);  // the effective grid
    const int cf = cta_of(cs, T, P), cl = cta_of(ce - 1, T, P);
    if (cf == cl) return;  // finished inside one CTA
    bool valid = row < a.rows_per_seq;
    int64_t out_row = static_cast<int64_t>(seq) * a.n_q + row;
    if (valid && a.qsl != nullptr) {
        const QueryRange qr = query_range(a.qsl, seq, a.rows_per_seq / a.n_q, a.qrows);
        valid = row / a.n_q < qr.count;  // past this sequence's queries otherwise
        out_row = static_cast<int64_t>(qr.q0) * a.n_q + row;
    }
    // this slice's parts [c_lo, c_hi) of the sequence's k, eight per batch, every load of a
    // batch issued before the first is used
    const int k = cl - cf + 1;
    const int c_lo = slice * k / kCombineSlices, c_hi = (slice + 1) * k / kCombineSlices;
    PartMerge mg;
    if (valid) {
        const int64_t p0 = static_cast<int64_t>(seq) + cf;
        const float *lse = a.part_lse + p0 * a.rows_per_seq + row;
        const float *o = a.part_o + (p0 * a.rows_per_seq + row) * HD + d;
        const int64_t lse_stride = a.rows_per_seq, o_stride = static_cast<int64_t>(a.rows_per_seq) * HD;
        for (int c0 = c_lo; c0 < c_hi; c0 += 8) {
            float l[8];
            float4 v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                l[i] = -INFINITY;
                if (c0 + i < c_hi) {
                    l[i] = lse[(c0 + i) * lse_stride];
                    v[i] = *reinterpret_cast<const float4 *>(o + (c0 + i) * o_stride);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) mg.add(l[i], v[i]);
        }
    }
    sm_m[slice][t] = mg.M;
    sm_den[slice][t] = mg.den;
    sm_acc[slice][t] = mg.acc;
    __syncthreads();
    if (slice != 0 || !valid) return;
    // merge the slices' running states (a slice that saw no part has M = -inf, den = 0)
    PartMerge all;
#pragma unroll
    for (int sl = 0; sl < kCombineSlices; ++sl) {
        const float m = sm_m[sl][t];
        if (m == -INFINITY) continue;
        if (m > all.M) {
            const float r = ex2(all.M - m);  // 0 while all.M is still -inf
            all.den *= r;
            all.acc.x *= r;
            all.acc.y *= r;
            all.acc.z *= r;
            all.acc.w *= r;
            all.M = m;
        }
        const float w = ex2(m - all.M);
        const float4 v = sm_acc[sl][t];
        all.den += w * sm_den[sl][t];
        all.acc.x += w * v.x;
        all.acc.y += w * v.y;
        all.acc.z += w * v.z;
        all.acc.w += w * v.w;
    }
    *reinterpret_cast<uint2 *>(a.out + out_row * HD + d) = all.result(sv);
}

// Two CTAs per SM where the accumulators fit in the resulting 96 registers per thread
// (head_dim * query tiles <= 128, and not the bf16-V form with two query tiles, whose extra
// probability fragments do not fit); three for the form below; one otherwise.
// 16 FP8 score columns at head_dim 128 keep q in shared memory instead of 32 registers a
// lane, take at most 4 kv heads per CTA (5 warps) and run 3 CTAs per SM: 12 consumer warps per
// SM instead of 8, for a consumer that is bound by its own dependency chains.
template <int HD, int NT, bool KT16, bool VT16>
__host__ __device__ constexpr bool q_in_smem() { return HD == 128 && NT == 2 && !KT16 && !VT16; }

// kv heads (consumer warps) per CTA at most
template <int HD, int NT, bool KT16, bool VT16>
__host__ __device__ constexpr int max_heads() { return q_in_smem<HD, NT, KT16, VT16>() ? 4 : kMaxKvHeads; }

template <int HD, int NT, bool KT16, bool VT16>
__host__ __device__ constexpr int min_ctas_per_sm() {
    return q_in_smem<HD, NT, KT16, VT16>() ? 3 : HD * NT <= 128 && !(VT16 && NT == 2) ? 2 : 1;
}

// bytes of one consumer warp's q fragments in shared memory: per 16-dim k-step, each lane's
// words of both n-tiles (16 bytes)
template <int HD>
__host__ __device__ constexpr int q_smem_bytes_per_warp() { return (HD / 16) * 32 * 16; }

// KT16 / VT16: that side's cache holds bf16 (mixed cache dtypes) instead of E4M3 bytes; its
// fragments go to bf16 mma.sync without a convert and its scale is not applied.
template <int HD, int NT, bool kMulti, bool KT16, bool VT16>
__global__ void __launch_bounds__(32 * (max_heads<HD, NT, KT16, VT16>() + 1),
                                  min_ctas_per_sm<HD, NT, KT16, VT16>())
decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
              const KernelArgs a) {
    constexpr int KB = KT16 ? 2 : 1, VB = VT16 ? 2 : 1;  // bytes per element of each side
    // bytes per TMA box row (the swizzle span), boxes per head, 16-byte chunks per box row
    constexpr int SEGK = HD * KB >= 128 ? 128 : 64, SEGV = HD * VB >= 128 ? 128 : 64;
    constexpr int SEGSK = HD * KB / SEGK, SEGSV = HD * VB / SEGV;
    constexpr int CPSK = SEGK / 16, CPSV = SEGV / 16;
    constexpr int KP = HD / 32;  // pairs of 16-dim k-steps / m-tiles

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);

    const int S = a.stages;
    const int hpc = a.hpc, h0 = static_cast<int>(blockIdx.y) * hpc;  // this CTA's kv heads
    const int RK = hpc * HD * KB, RV = hpc * HD * VB;  // bytes of a cache row this CTA holds
    const uint32_t kchunk_bytes = static_cast<uint32_t>(kChunkTokens * RK);
    const uint32_t stage_bytes = kchunk_bytes + static_cast<uint32_t>(kChunkTokens * RV);
    const uint32_t bars = base + static_cast<uint32_t>(S) * stage_bytes;  // full[S], empty[S]
    ChunkMeta *meta = reinterpret_cast<ChunkMeta *>(base_ptr + S * stage_bytes + 16 * S);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(meta + S);
    constexpr bool kQS = q_in_smem<HD, NT, KT16, VT16>();
    // q fragments (kQS): after the ring's barriers, records and abort flag, 16-byte aligned
    const uint32_t q_smem = (smem_u32(const_cast<int32_t *>(abort_flag)) + 16u + 15u) & ~15u;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < S; ++i) {
            mbar_init(bars + 8 * i, 1);
            mbar_init(bars + 8 * (S + i), hpc);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == hpc && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmk)) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&tmv)) : "memory");
    }
    if (warp == hpc && blockIdx.y == 0) {
        // This CTA's slice of the block tables into L2 while the plan grid runs, so the
        // table read after the plan hits L2.  The tables are inputs written before this call
        // (the plan kernel was launched behind that work), and a prefetch returns no data,
        // so it needs no ordering with the plan.
        const int64_t bytes = static_cast<int64_t>(a.num_seqs) * a.max_blocks_per_seq * 4;
        const int64_t per = (bytes + gridDim.x - 1) / gridDim.x;
        const char *tb = reinterpret_cast<const char *>(a.block_tables);
        for (int64_t off = blockIdx.x * per + lane * 128; off < min(bytes, (blockIdx.x + 1) * per);
             off += 32 * 128)
            asm volatile("prefetch.global.L2 [%0];" ::"l"(tb + off));
    }
    pdl_wait();     // the plan grid's records and zeroed rows are visible from here on
    pdl_trigger();  // let the combine grid get launched; it waits for this grid to finish

    const float sk = KT16 ? 1.f : load_scale(a.k_scale, a.scale_dtype);
    const float sv = VT16 ? 1.f : load_scale(a.v_scale, a.scale_dtype);
    if (!scale_ok(sk) || !scale_ok(sv)) {
        if (blockIdx.x == 0 && threadIdx.x == 0) flag(a.status, KVFP8_DEV_BAD_SCALE);
        return;
    }
    // Effective grid: at most one CTA per chunk, so that every active CTA's range is
    // non-empty and the CTAs between a sequence's first and last one all hold a part of it;
    // the plan leaves CTAs past it an empty range.
    const CtaPlan *rec = a.cta_plan + blockIdx.x;
    const int32_t pl_lo = rec->lo, pl_hi = rec->hi;
    if (pl_lo >= pl_hi) return;
    const int64_t chunk_lo = pl_lo, chunk_hi = pl_hi;
    __syncthreads();

    if (warp == hpc) {
        // ------------------------------------------------------------ producer warp
        int64_t issued = 0;
        int stage = 0;
        uint32_t phase = 0;
        bool aborted = false;
        if (chunk_lo < chunk_hi) {
            int s = rec->s;  // sequence holding chunk_lo, its chunks and length (from the plan)
            int64_t cs = rec->cs, ce = rec->ce;
            int L = rec->L;
            int wbase = -1 << 30;  // first block-table entry held in the lane window
            int32_t win = 0;
            prefetch_q<HD>(a, s, h0, lane);
            for (int64_t x = chunk_lo; x < chunk_hi; ++x) {
                if (x >= ce) {
                    while (x >= ce) {
                        ++s;
                        cs = ce;
                        ce = cs + seq_chunks(a, s, L);
                    }
                    wbase = -1 << 30;
                    prefetch_q<HD>(a, s, h0, lane);
                }
                const int j = static_cast<int>(x - cs);
                const int tok0 = j * kChunkTokens;
                int nvalid = min(kChunkTokens, L - tok0);
                const int nloads = (nvalid + a.box_rows - 1) / a.box_rows;
                const int e0 = tok0 / a.block_size;  // first block-table entry of the chunk
                if (e0 < wbase || e0 + nloads - 1 >= wbase + 32) {
                    wbase = e0;
                    const int e = wbase + lane;
                    win = (e < a.max_blocks_per_seq)
                              ? a.block_tables[static_cast<int64_t>(s) * a.max_blocks_per_seq + e]
                              : -1;
                }
                int rows0[2];
                bool ok = true;
#pragma unroll
                for (int p = 0; p < 2; ++p) {
                    const int t = tok0 + p * a.box_rows;
                    const int blk = __shfl_sync(0xFFFFFFFFu, win, (t / a.block_size - wbase) & 31);
                    if (p < nloads) {
                        ok = ok && blk >= 0 && blk < a.num_blocks;
                        rows0[p] = blk * a.block_size + t % a.block_size;
                    }
                }
                int32_t flags = 0;
                if (x == chunk_lo || x == cs) flags |= kFirst;
                if (x == chunk_hi - 1 || x == ce - 1) flags |= kLast;
                if (cs >= chunk_lo && ce <= chunk_hi) flags |= kDirect;
                if (lane == 0) {
                    if (!mbar_wait(bars + 8 * (S + stage), phase ^ 1u, abort_flag)) {
                        aborted = true;
                    } else {
                        if (!ok) {
                            flag(a.status, KVFP8_DEV_BAD_BLOCK);
                            nvalid = 0;
                        }
                        meta[stage] = ChunkMeta{s, tok0, nvalid, flags};
                        const uint32_t full = bars + 8 * stage;
                        if (kWithholdFirstChunk && issued == 0) {
                            // test build: neither a copy nor an arrival for this stage
                        } else if (nvalid > 0) {
                            const uint32_t rows_bytes = static_cast<uint32_t>(a.box_rows * (RK + RV));
                            mbar_arrive_tx(full, nloads * rows_bytes);
                            const uint32_t kst = base + static_cast<uint32_t>(stage) * stage_bytes;
                            const uint32_t vst = kst + kchunk_bytes;
                            if (a.whole_box) {  // one box: the group's head segments, 16 rows
                                tma_load_3d(kst, &tmk, 0, rows0[0], h0 * SEGSK, full);
                                tma_load_3d(vst, &tmv, 0, rows0[0], h0 * SEGSV, full);
                            } else {
                                for (int p = 0; p < nloads; ++p) {
                                    for (int g = 0; g < hpc * SEGSK; ++g) {
                                        const uint32_t off = static_cast<uint32_t>(
                                            g * kChunkTokens * SEGK + p * a.box_rows * SEGK);
                                        tma_load_3d(kst + off, &tmk, 0, h0 * SEGSK + g, rows0[p], full);
                                    }
                                    for (int g = 0; g < hpc * SEGSV; ++g) {
                                        const uint32_t off = static_cast<uint32_t>(
                                            g * kChunkTokens * SEGV + p * a.box_rows * SEGV);
                                        tma_load_3d(vst + off, &tmv, 0, h0 * SEGSV + g, rows0[p], full);
                                    }
                                }
                            }
                        } else {
                            mbar_arrive(full);
                        }
                    }
                }
                aborted = __shfl_sync(0xFFFFFFFFu, aborted, 0);
                if (aborted) break;
                ++issued;
                if (++stage == S) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
        }
        if (!aborted) {
            if (lane == 0) {
                if (!mbar_wait(bars + 8 * (S + stage), phase ^ 1u, abort_flag)) {
                    aborted = true;
                } else {
                    meta[stage] = ChunkMeta{0, 0, 0, kDone};
                    mbar_arrive(bars + 8 * stage);
                }
            }
            aborted = __shfl_sync(0xFFFFFFFFu, aborted, 0);
        }
        if (aborted && lane == 0) {
            flag(a.status, KVFP8_DEV_TIMEOUT);
            *abort_flag = 1;
            // let copies already issued land before the CTA's shared memory goes away
            const int64_t first = issued > S ? issued - S : 0;
            for (int64_t k = first; k < issued; ++k) {
                const volatile int32_t never = 0;
                mbar_wait(bars + 8 * static_cast<int>(k % S), static_cast<uint32_t>((k / S) & 1),
                          &never);
            }
        }
    } else if (warp < hpc) {
        // ------------------------------------------------------------ consumer warp
        const int kvh = h0 + warp;  // its kv head; warp is the head's place in the group
        const int gid = lane >> 2, tig = lane & 3;
        const float score_scale = a.sm_scale * sk * 1.4426950408889634f;  // log2(e)

        float o[KP][2][NT][4];
        float m[NT][2], l[NT][2];
        uint32_t qb[kQS ? 1 : 2 * KP][NT][2];
        // kQS: this lane's words of k-step c at q_lane + 512 c
        const uint32_t q_lane = q_smem + static_cast<uint32_t>(warp * q_smem_bytes_per_warp<HD>() + lane * 16);
        // multi-query form: per score column (query token j, head g) the last cache
        // position it may see, and its row within the sequence (-1: a padding column)
        int plim[NT][2], crow[NT][2];
        int q0 = 0;
#pragma unroll
        for (int e = 0; e < KP; ++e)
#pragma unroll
            for (int j = 0; j < 2; ++j)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int r = 0; r < 4; ++r) o[e][j][nt][r] = 0.f;
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) m[nt][0] = m[nt][1] = -INFINITY, l[nt][0] = l[nt][1] = 0.f;

        // per-lane shared-memory offsets inside one head's [SEGS][16][SEG] region
        const int krow = (lane & 7) + (((lane >> 3) & 1) << 3);
        const int kchunk_hi = lane >> 4;          // +1 chunk for lanes 16..31
        const int vtok = (lane & 7) + ((lane >> 4) << 3);
        const int vchunk_hi = (lane >> 3) & 1;    // +1 chunk for lanes 8..15 and 24..31

        int stage = 0;
        uint32_t phase = 0;
        for (;;) {
            // every lane waits (acquire on the TMA bytes); the outcome is made warp-uniform
            if (!__all_sync(0xFFFFFFFFu, mbar_wait(bars + 8 * stage, phase, abort_flag))) {
                if (lane == 0) {
                    flag(a.status, KVFP8_DEV_TIMEOUT);
                    *abort_flag = 1;
                }
                break;
            }
            const ChunkMeta mt = meta[stage];
            if (mt.flags & kDone) break;

            if (mt.flags & kFirst) {
                int nq = 1;
                if (kMulti) {
                    const QueryRange qr = query_range(a.qsl, mt.seq, a.rows_per_seq / a.n_q, a.qrows);
                    q0 = qr.q0;
                    nq = qr.count;
                    const int L = min(max(a.seq_lens[mt.seq], 0), a.max_len);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int c = 0; c < 2; ++c) {
                            const int n = nt * 8 + 2 * tig + c;
                            const int j = n / a.group, g = n % a.group;
                            plim[nt][c] = j < nq ? L - nq + j : -1;
                            crow[nt][c] = j < nq ? j * a.n_q + kvh * a.group + g : -1;
                        }
                }
                // column gid of n-tile nt: query token jq, head gq of the group
                auto q_row = [&](int nt, bool &qv) {
                    const int n = nt * 8 + gid;
                    const int jq = kMulti ? n / a.group : 0;
                    const int gq = kMulti ? n % a.group : n;
                    qv = kMulti ? jq < nq : n < a.group;
                    return a.query +
                           ((static_cast<int64_t>(kMulti ? q0 + jq : mt.seq)) * a.n_q + kvh * a.group + gq) * HD;
                };
                if constexpr (kQS) {
                    // each lane's B fragment words, converted once per sequence, into its own
                    // 16-byte slots (read back only by the same lane: no warp sync needed)
                    bool qv[NT];
                    const __nv_bfloat16 *qrow[NT];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) qrow[nt] = q_row(nt, qv[nt]);
#pragma unroll
                    for (int c = 0; c < 2 * KP; ++c) {
                        uint32_t wd[2 * NT];
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            uint2 w = make_uint2(0u, 0u);
                            if (qv[nt]) w = *reinterpret_cast<const uint2 *>(qrow[nt] + 16 * c + 4 * tig);
                            wd[2 * nt] = f16x2_from_f32(bf16lo(w.x), bf16hi(w.x));
                            wd[2 * nt + 1] = f16x2_from_f32(bf16lo(w.y), bf16hi(w.y));
                        }
                        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(q_lane + 512u * c),
                                     "r"(wd[0]), "r"(wd[1]), "r"(wd[2]), "r"(wd[3])
                                     : "memory");
                    }
                } else {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        bool qv;
                        const __nv_bfloat16 *qrow = q_row(nt, qv);
#pragma unroll
                        for (int c = 0; c < 2 * KP; ++c) {
                            if constexpr (KT16) {  // bf16 as it is, in the natural k order
                                const uint32_t *qw = reinterpret_cast<const uint32_t *>(qrow + 16 * c);
                                qb[c][nt][0] = qv ? qw[tig] : 0u;
                                qb[c][nt][1] = qv ? qw[4 + tig] : 0u;
                            } else {
                                uint2 w = make_uint2(0u, 0u);
                                if (qv) w = *reinterpret_cast<const uint2 *>(qrow + 16 * c + 4 * tig);
                                qb[c][nt][0] = f16x2_from_f32(bf16lo(w.x), bf16hi(w.x));
                                qb[c][nt][1] = f16x2_from_f32(bf16lo(w.y), bf16hi(w.y));
                            }
                        }
                    }
                }
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    m[nt][0] = m[nt][1] = -INFINITY;
                    l[nt][0] = l[nt][1] = 0.f;
                }
#pragma unroll
                for (int e = 0; e < KP; ++e)
#pragma unroll
                    for (int j = 0; j < 2; ++j)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int r = 0; r < 4; ++r) o[e][j][nt][r] = 0.f;
            }

            const int nvalid = mt.nvalid;
            if (nvalid > 0) {
                const uint32_t sbase = base + static_cast<uint32_t>(stage) * stage_bytes;
                const uint32_t kbase = sbase + warp * (kChunkTokens * HD * KB);
                const uint32_t vbase = sbase + kchunk_bytes + warp * (kChunkTokens * HD * VB);

                // ---- scores S^T[token][head] = K . q^T
                float sacc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    sacc[nt][0] = sacc[nt][1] = sacc[nt][2] = sacc[nt][3] = 0.f;
                if constexpr (KT16) {
                    // bf16 K: a 16-byte chunk is 8 dims, so k-step c spans chunks 2c, 2c+1;
                    // ldmatrix gives the A fragments in the natural layout
#pragma unroll
                    for (int c = 0; c < 2 * KP; ++c) {
                        const int ch = 2 * c + kchunk_hi;
                        const uint32_t addr = kbase + (ch / CPSK) * (kChunkTokens * SEGK) +
                                              swz<SEGK>(krow, ch % CPSK);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4(addr, r0, r1, r2, r3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816_bf16(sacc[nt], r0, r1, r2, r3, qb[c][nt][0], qb[c][nt][1]);
                    }
                } else
#pragma unroll
                for (int kk = 0; kk < KP; ++kk) {
                    const int ch = 2 * kk + kchunk_hi;
                    const uint32_t addr = kbase + (ch / CPSK) * (kChunkTokens * SEGK) +
                                          swz<SEGK>(krow, ch % CPSK);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4(addr, r0, r1, r2, r3);
                    const uint32_t a0 = f16x2_from_e4m3x2(r0), a1 = f16x2_from_e4m3x2(r1);
                    const uint32_t a2 = f16x2_from_e4m3x2_hi(r0), a3 = f16x2_from_e4m3x2_hi(r1);
                    const uint32_t b0 = f16x2_from_e4m3x2(r2), b1 = f16x2_from_e4m3x2(r3);
                    const uint32_t b2 = f16x2_from_e4m3x2_hi(r2), b3 = f16x2_from_e4m3x2_hi(r3);
                    if constexpr (kQS) {
                        uint32_t qa[4], qc[4];  // k-steps 2kk, 2kk+1: (n-tile 0 b0, b1, n-tile 1 b0, b1)
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(qa[0]), "=r"(qa[1]), "=r"(qa[2]), "=r"(qa[3])
                                     : "r"(q_lane + 1024u * kk));
                        asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                                     : "=r"(qc[0]), "=r"(qc[1]), "=r"(qc[2]), "=r"(qc[3])
                                     : "r"(q_lane + 1024u * kk + 512u));
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816(sacc[nt], a0, a1, a2, a3, qa[2 * nt], qa[2 * nt + 1]);
                            mma16816(sacc[nt], b0, b1, b2, b3, qc[2 * nt], qc[2 * nt + 1]);
                        }
                    } else {
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816(sacc[nt], a0, a1, a2, a3, qb[2 * kk][nt][0], qb[2 * kk][nt][1]);
                            mma16816(sacc[nt], b0, b1, b2, b3, qb[2 * kk + 1][nt][0],
                                     qb[2 * kk + 1][nt][1]);
                        }
                    }
                }

                // ---- online softmax per head column (log2 domain)
                const bool lo_ok = gid < nvalid, hi_ok = gid + 8 < nvalid;
                uint32_t pb[NT][2];
                uint32_t pbl[NT][2];  // bf16 V: the low parts of p (p = high + low)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float p[4];
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        bool lo_c = lo_ok, hi_c = hi_ok;
                        if (kMulti) {  // causal: token tok0+row is visible up to plim
                            lo_c = lo_c && mt.tok0 + gid <= plim[nt][c];
                            hi_c = hi_c && mt.tok0 + gid + 8 <= plim[nt][c];
                        }
                        const float s_lo = lo_c ? sacc[nt][c] * score_scale : -INFINITY;
                        const float s_hi = hi_c ? sacc[nt][c + 2] * score_scale : -INFINITY;
                        float mx = fmaxf(s_lo, s_hi);
                        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 4));
                        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 8));
                        mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, 16));
                        const float m_old = m[nt][c];
                        float m_new = fmaxf(m_old, mx);
                        const float alpha = (m_old == -INFINITY) ? 0.f : ex2(m_old - m_new);
                        // a column that has seen no visible token yet keeps weight 0
                        const float m_sub = (kMulti && m_new == -INFINITY) ? 0.f : m_new;
                        p[c] = ex2(s_lo - m_sub);
                        p[c + 2] = ex2(s_hi - m_sub);
                        l[nt][c] = l[nt][c] * alpha + p[c] + p[c + 2];
                        m[nt][c] = m_new;
                        if (alpha != 1.f) {
#pragma unroll
                            for (int e = 0; e < KP; ++e)
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    o[e][j][nt][c] *= alpha;
                                    o[e][j][nt][c + 2] *= alpha;
                                }
                        }
                    }
                    if constexpr (VT16) {
                        // bf16 operands for the bf16 V: p as a sum of two bf16 numbers keeps
                        // 16 significant bits (one bf16 would keep 8)
                        const uint32_t h0 = bf16x2_from_f32(p[0], p[1]);
                        const uint32_t h1 = bf16x2_from_f32(p[2], p[3]);
                        pb[nt][0] = movm_t(h0);
                        pb[nt][1] = movm_t(h1);
                        pbl[nt][0] = movm_t(bf16x2_from_f32(p[0] - bf16lo(h0), p[1] - bf16hi(h0)));
                        pbl[nt][1] = movm_t(bf16x2_from_f32(p[2] - bf16lo(h1), p[3] - bf16hi(h1)));
                    } else {
                        pb[nt][0] = movm_t(f16x2_from_f32(p[0], p[1]));  // tokens 0-7
                        pb[nt][1] = movm_t(f16x2_from_f32(p[2], p[3]));  // tokens 8-15
                        pbl[nt][0] = pbl[nt][1] = 0u;
                    }
                }

                // ---- O^T[dim][head] += V^T . P^T
                uint32_t mlo = 0xFFFFFFFFu, mhi = 0xFFFFFFFFu;
                if (nvalid < kChunkTokens) {  // zero the bytes of tokens past the end
                    mlo = (2 * tig < nvalid ? 0x0000FFFFu : 0u) |
                          (2 * tig + 1 < nvalid ? 0xFFFF0000u : 0u);
                    mhi = (2 * tig + 8 < nvalid ? 0x0000FFFFu : 0u) |
                          (2 * tig + 9 < nvalid ? 0xFFFF0000u : 0u);
                }
                if constexpr (VT16) {
                    // bf16 V: m-tile t covers dims 16t..16t+15 (chunks 2t, 2t+1); ldmatrix.trans
                    // gives V^T's A fragments with tokens along k, no permutation
#pragma unroll
                    for (int t = 0; t < 2 * KP; ++t) {
                        const int ch = 2 * t + vchunk_hi;
                        const uint32_t addr = vbase + (ch / CPSV) * (kChunkTokens * SEGV) +
                                              swz<SEGV>(vtok, ch % CPSV);
                        uint32_t r0, r1, r2, r3;
                        ldsm_x4_t(addr, r0, r1, r2, r3);
                        r0 &= mlo;
                        r1 &= mlo;
                        r2 &= mhi;
                        r3 &= mhi;
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt) {
                            mma16816_bf16(o[t >> 1][t & 1][nt], r0, r1, r2, r3, pb[nt][0], pb[nt][1]);
                            mma16816_bf16(o[t >> 1][t & 1][nt], r0, r1, r2, r3, pbl[nt][0], pbl[nt][1]);
                        }
                    }
                } else
#pragma unroll
                for (int e = 0; e < KP; ++e) {
                    const int ch = 2 * e + vchunk_hi;
                    const uint32_t addr = vbase + (ch / CPSV) * (kChunkTokens * SEGV) +
                                          swz<SEGV>(vtok, ch % CPSV);
                    uint32_t r0, r1, r2, r3;
                    ldsm_x4_t(addr, r0, r1, r2, r3);
                    r0 = __byte_perm(r0 & mlo, 0u, 0x3120);
                    r1 = __byte_perm(r1 & mlo, 0u, 0x3120);
                    r2 = __byte_perm(r2 & mhi, 0u, 0x3120);
                    r3 = __byte_perm(r3 & mhi, 0u, 0x3120);
                    {
                        const uint32_t a0 = f16x2_from_e4m3x2(r0), a1 = f16x2_from_e4m3x2(r1);
                        const uint32_t a2 = f16x2_from_e4m3x2(r2), a3 = f16x2_from_e4m3x2(r3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(o[e][0][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    }
                    {
                        const uint32_t a0 = f16x2_from_e4m3x2_hi(r0), a1 = f16x2_from_e4m3x2_hi(r1);
                        const uint32_t a2 = f16x2_from_e4m3x2_hi(r2), a3 = f16x2_from_e4m3x2_hi(r3);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            mma16816(o[e][1][nt], a0, a1, a2, a3, pb[nt][0], pb[nt][1]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(bars + 8 * (S + stage));
            if (++stage == S) {
                stage = 0;
                phase ^= 1u;
            }

            if (mt.flags & kLast) {
                const bool direct = (mt.flags & kDirect) != 0;
                const int64_t pidx = static_cast<int64_t>(mt.seq) + blockIdx.x;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
                    for (int c = 0; c < 2; ++c) {
                        float lt = l[nt][c];
                        lt += __shfl_xor_sync(0xFFFFFFFFu, lt, 4);
                        lt += __shfl_xor_sync(0xFFFFFFFFu, lt, 8);
                        lt += __shfl_xor_sync(0xFFFFFFFFu, lt, 16);
                        const int g = nt * 8 + 2 * tig + c;
                        if (kMulti ? crow[nt][c] < 0 : g >= a.group) continue;  // padding column
                        // the row of this column within the sequence's rows, and in out
                        const int srow = kMulti ? crow[nt][c] : kvh * a.group + g;
                        const int64_t orow_idx = kMulti ? static_cast<int64_t>(q0) * a.n_q + srow
                                                        : static_cast<int64_t>(mt.seq) * a.n_q + srow;
                        if (VT16) {
                            // o[e][j] holds dims 32e+16j+gid (c) and +8 (c+2): one element each
                            const float inv = lt > 0.f ? (direct ? sv : 1.f) / lt : 0.f;
#pragma unroll
                            for (int e = 0; e < KP; ++e)
#pragma unroll
                                for (int j = 0; j < 2; ++j) {
                                    const int d = 32 * e + 16 * j + gid;
                                    const float x0 = o[e][j][nt][c] * inv, x1 = o[e][j][nt][c + 2] * inv;
                                    if (direct) {
                                        __nv_bfloat16 *orow = a.out + orow_idx * HD;
                                        orow[d] = __float2bfloat16_rn(x0);
                                        orow[d + 8] = __float2bfloat16_rn(x1);
                                    } else {
                                        float *prow = a.part_o + (pidx * a.rows_per_seq + srow) * HD;
                                        prow[d] = x0;
                                        prow[d + 8] = x1;
                                    }
                                }
                            if (!direct && gid == 0)
                                a.part_lse[pidx * a.rows_per_seq + srow] =
                                    lt > 0.f ? m[nt][c] + __log2f(lt) : -INFINITY;
                        } else if (direct) {
                            const float inv = lt > 0.f ? sv / lt : 0.f;
                            __nv_bfloat16 *orow = a.out + orow_idx * HD;
#pragma unroll
                            for (int e = 0; e < KP; ++e) {
                                const int d = 32 * e + 2 * gid;
                                *reinterpret_cast<uint32_t *>(orow + d) =
                                    bf16x2_from_f32(o[e][0][nt][c] * inv, o[e][1][nt][c] * inv);
                                *reinterpret_cast<uint32_t *>(orow + d + 16) = bf16x2_from_f32(
                                    o[e][0][nt][c + 2] * inv, o[e][1][nt][c + 2] * inv);
                            }
                        } else {
                            const float inv = lt > 0.f ? 1.f / lt : 0.f;
                            float *prow = a.part_o + (pidx * a.rows_per_seq + srow) * HD;
#pragma unroll
                            for (int e = 0; e < KP; ++e) {
                                const int d = 32 * e + 2 * gid;
                                *reinterpret_cast<float2 *>(prow + d) =
                                    make_float2(o[e][0][nt][c] * inv, o[e][1][nt][c] * inv);
                                *reinterpret_cast<float2 *>(prow + d + 16) = make_float2(
                                    o[e][0][nt][c + 2] * inv, o[e][1][nt][c + 2] * inv);
                            }
                            if (gid == 0)
                                a.part_lse[pidx * a.rows_per_seq + srow] =
                                    lt > 0.f ? m[nt][c] + __log2f(lt) : -INFINITY;
                        }
                    }
                }
            }
        }
    }
    __syncthreads();
}

// ---------------------------------------------------------------- host side

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        cudaDriverEntryPointQueryResult q;
        void *p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// The cache as a 3-D byte tensor (SEG bytes, n_kv*head_dim/SEG segments, rows) read in
// [box_rows x SEG] boxes with SEG-byte swizzle.
cudaError_t encode_cache_map(CUtensorMap *map, const uint8_t *cache, int64_t rows, int row_bytes,
                             int seg, int box_rows) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(seg),
                                static_cast<cuuint64_t>(row_bytes / seg),
                                static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(seg),
                                   static_cast<cuuint64_t>(row_bytes)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(seg), 1u, static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(cache),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           seg == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// The same bytes as a 3-D tensor ordered (SEG bytes, rows, segments) -- the segment
// stride (SEG) below the row stride -- so that one [SEG x 16 rows x box_segs] box fetches
// a head group's part of a 16-token chunk into the same [segment][row][SEG] swizzled
// layout that the per-segment boxes produce, with one TMA instruction instead of one per
// segment.
cudaError_t encode_cache_map_whole(CUtensorMap *map, const uint8_t *cache, int64_t rows,
                                   int row_bytes, int seg, int box_segs) {
    auto enc = tensor_map_encoder();
    if (enc == nullptr) return cudaErrorNotSupported;
    const int segs = row_bytes / seg;
    if (segs > (1 << 20) || box_segs > 256) return cudaErrorNotSupported;
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(seg), static_cast<cuuint64_t>(rows),
                                static_cast<cuuint64_t>(segs)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes),
                                   static_cast<cuuint64_t>(seg)};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(seg), static_cast<cuuint32_t>(kChunkTokens),
                               static_cast<cuuint32_t>(box_segs)};
    const cuuint32_t estr[3] = {1u, 1u, 1u};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t *>(cache),
                           dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                           seg == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}


template <int HD, int NT, bool kMulti, bool KT16, bool VT16>
cudaError_t run(const DecodeArgs &d, const DecodeWorkspace &ws, cudaStream_t stream) {
    DeviceFacts facts;
    cudaError_t err = device_facts(&facts);
    if (err != cudaSuccess) return err;
    const int sms = facts.sms, smem_optin = facts.smem_optin;

    constexpr int KB = KT16 ? 2 : 1, VB = VT16 ? 2 : 1;
    constexpr int SEGK = HD * KB >= 128 ? 128 : 64, SEGV = HD * VB >= 128 ? 128 : 64;
    const int kbytes = d.n_kv * HD * KB, vbytes = d.n_kv * HD * VB;  // cache row bytes
    // kv heads per CTA: the largest divisor of n_kv up to 8; the groups are a grid dimension
    int hpc = std::min(d.n_kv, max_heads<HD, NT, KT16, VT16>());
    while (d.n_kv % hpc != 0) --hpc;
    const int groups = d.n_kv / hpc;
    const int stage_bytes = kChunkTokens * hpc * HD * (KB + VB);
    const int ctas_per_sm = std::max(
        1, std::min(min_ctas_per_sm<HD, NT, KT16, VT16>(), env_int("KVFP8_DECODE_CTAS_PER_SM", 3)));
    const int max_stages = std::max(2, std::min(8, env_int("KVFP8_DECODE_MAX_STAGES", 8)));
    // per stage: the K and V chunk, two mbarriers and one ChunkMeta; then the abort flag
    // and up to 1 KiB to align the ring to the 128-byte swizzle span; 1 KiB of the SM's
    // shared memory goes to each CTA's system use
    // (and the consumers' q fragments where they live in shared memory)
    constexpr size_t q_bytes =
        q_in_smem<HD, NT, KT16, VT16>() ? 4 * q_smem_bytes_per_warp<HD>() + 16 : 0;
    auto smem_for = [&](int st) { return static_cast<size_t>(st) * (stage_bytes + 32) + 16 + 1024 + q_bytes; };
    const size_t sm_budget = static_cast<size_t>(smem_optin) + 1024;
    int stages = max_stages;
    while (stages > 2 && (smem_for(stages) + 1024) * ctas_per_sm > sm_budget) --stages;
    const size_t smem = smem_for(stages);
    if (smem > static_cast<size_t>(smem_optin)) return cudaErrorNotSupported;

    auto kern = decode_kernel<HD, NT, kMulti, KT16, VT16>;
    const int threads = 32 * (hpc + 1);
    int occ = 0;
    if ((err = kernel_occupancy(kern, threads, smem, &occ)) != cudaSuccess) return err;
    occ = std::max(1, std::min(occ, ctas_per_sm));
    // about one resident wave over all head groups
    const int num_ctas = std::max(1, std::min(sms * occ / groups, kMaxDecodeCtas));

    CUtensorMap tmk, tmv;
    const int box_rows = d.block_size >= kChunkTokens ? kChunkTokens : d.block_size;
    const int64_t rows = static_cast<int64_t>(d.num_blocks) * d.block_size;
    // whole-chunk boxes when a chunk never straddles blocks (and the driver accepts the
    // map); otherwise one box per head segment
    bool whole = box_rows == kChunkTokens && env_int("KVFP8_DECODE_SEGMENT_BOXES", 0) == 0 &&
                 encode_cache_map_whole(&tmk, d.key_cache, rows, kbytes, SEGK, hpc * HD * KB / SEGK) ==
                     cudaSuccess &&
                 encode_cache_map_whole(&tmv, d.value_cache, rows, vbytes, SEGV, hpc * HD * VB / SEGV) ==
                     cudaSuccess;
    if (!whole) {
        if ((err = encode_cache_map(&tmk, d.key_cache, rows, kbytes, SEGK, box_rows)) != cudaSuccess)
            return err;
        if ((err = encode_cache_map(&tmv, d.value_cache, rows, vbytes, SEGV, box_rows)) !=
            cudaSuccess)
            return err;
    }

    uint8_t *w = static_cast<uint8_t *>(d.workspace);
    KernelArgs k;
    k.out = static_cast<__nv_bfloat16 *>(d.out);
    k.query = static_cast<const __nv_bfloat16 *>(d.query);
    k.block_tables = d.block_tables;
    k.max_blocks_per_seq = d.max_blocks_per_seq;
    k.seq_lens = d.seq_lens;
    k.num_seqs = d.num_seqs;
    k.n_q = d.n_q;
    k.n_kv = d.n_kv;
    k.group = d.n_q / d.n_kv;
    k.hpc = hpc;
    k.block_size = d.block_size;
    k.num_blocks = d.num_blocks;
    k.max_len = d.max_blocks_per_seq * d.block_size;
    k.sm_scale = d.sm_scale;
    k.k_scale = d.k_scale;
    k.v_scale = d.v_scale;
    k.scale_dtype = d.scale_dtype;
    k.cstart = reinterpret_cast<const int32_t *>(w + ws.cstart_off);
    k.cta_plan = reinterpret_cast<const CtaPlan *>(w + ws.cta_off);
    k.part_lse = reinterpret_cast<float *>(w + ws.lse_off);
    k.part_o = reinterpret_cast<float *>(w + ws.o_off);
    k.status = d.status;
    k.num_ctas = num_ctas;
    k.stages = stages;
    k.box_rows = box_rows;
    k.whole_box = whole ? 1 : 0;
    k.qsl = d.qsl;
    k.rows_per_seq = d.qmax * d.n_q;
    k.qrows = d.qrows;
    k.k_bf16 = KT16 ? 1 : 0;
    k.v_bf16 = VT16 ? 1 : 0;

    plan_kernel<<<1, 1024, 0, stream>>>(d.seq_lens, d.qsl, d.qmax, d.qrows, d.num_seqs, k.max_len,
                                        num_ctas, reinterpret_cast<int32_t *>(w + ws.cstart_off),
                                        reinterpret_cast<CtaPlan *>(w + ws.cta_off), k.out,
                                        d.n_q * HD, d.status);
    if ((err = cudaGetLastError()) != cudaSuccess) return err;

    // Programmatic dependent launch: the decode grid starts its prologue while the plan
    // grid runs and waits (griddepcontrol.wait) before touching any data.
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(num_ctas, groups);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if ((err = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, k)) != cudaSuccess) return err;

    constexpr int kHeadsPerCta = 256 / (HD / 4);
    cudaLaunchConfig_t ccfg = cfg;
    ccfg.gridDim = dim3(d.num_seqs, (k.rows_per_seq + kHeadsPerCta - 1) / kHeadsPerCta);
    ccfg.dynamicSmemBytes = 0;
    // parts per sequence on average: every CTA's sequences plus one per sequence
    const int64_t parts = (static_cast<int64_t>(num_ctas) + d.num_seqs) / std::max(1, d.num_seqs);
    if (parts >= 32) {
        ccfg.blockDim = dim3(256 * 4);
        return cudaLaunchKernelEx(&ccfg, combine_kernel<HD, 4>, k);
    }
    if (parts >= 16) {
        ccfg.blockDim = dim3(256 * 2);
        return cudaLaunchKernelEx(&ccfg, combine_kernel<HD, 2>, k);
    }
    ccfg.blockDim = dim3(256);
    return cudaLaunchKernelEx(&ccfg, combine_kernel<HD, 1>, k);
}

}  // namespace
}  // namespace kvfp8
