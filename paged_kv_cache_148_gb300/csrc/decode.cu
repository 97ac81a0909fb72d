// pa_decode: paged decode attention with split-KV partitions and a merge.
//
// Semantics: the pseudo-kernel and backend rules of "03｜PagedAttention 与 KV
// Cache 内存系统" §4 — for every (sequence, query head) walk the visible logical
// blocks, look the physical block up in the table, attend to the page and
// combine blockwise softmax states (max, exp_sum, weighted value); the lookup
// is fused into the kernel, long contexts are split into partitions whose
// states are merged by a second kernel.
//
// Design (sm_103a, HBM-bound):
//  * One CTA = (sequence, kv-head, partition).  All G = H_q / H_kv query heads
//    of the group share every K/V byte read (GQA mapping g -> g / G).
//  * A warp owns every W-th 16-token chunk of the partition and streams them
//    through its own S-stage ring in shared memory with 1-D bulk copies (TMA
//    engine) completing on an mbarrier: 4 KiB of K and 4 KiB of V per chunk,
//    one contiguous run of a (block, kv-head) page.  Lane 0 is the producer;
//    block-table entries for the next 32 chunks are prefetched one per lane.
//  * Scores: lanes split the 256-byte row into 16-byte columns (16 lanes per
//    row, two rows per warp access, conflict-free LDS.128).  The partial dot
//    products of 8 tokens x G heads are finished by a transpose-reduction
//    over 4 shuffle rounds in which every round halves the live values; each
//    lane's token/head order is permuted (by XOR with its lane bits) so the
//    rounds need no selects.  Afterwards a lane holds G/2 finished scores.
//  * Softmax in base 2 (scores carry scale*log2 e); the running max is only
//    raised when a score exceeds it by more than 2^8, so rescaling the
//    accumulators is rare; the result is unchanged because the shift cancels
//    in the final division.
//  * P*V: probabilities go through a 16xG shared buffer; lanes accumulate
//    acc[g][d] over their 8 rows for their 16-byte column; the two row halves
//    are added at the end.
//  * The CTA's warps combine in shared memory; a single-partition sequence
//    writes the normalised output directly, otherwise (m, l, acc) partials go
//    to the workspace and decode_merge_kernel finishes.
//  * FP8 pages (Row<uint8_t>): 128-byte code rows, 8-byte lane columns, and
//    each chunk's 16 K and 16 V row scales in the same ring stage; the K
//    scale multiplies the finished score, the V scale is folded into the
//    probability pair (the running sum keeps the plain probability).
//  * Sliding window (pa_decode_window): partitions start at the window's
//    first chunk and rows before it are masked.
//  * Fused step (pa_decode_step): the same kernel also writes the new token
//    of (sequence, kv-head) into its slot, and into the shared-memory copy of
//    the chunk that holds it (P1 §4.1), and the last partition CTA of each
//    (sequence, kv-head) to finish -- counted by a semaphore in the
//    workspace -- merges the group's partials, so a decode step is one
//    launch.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include "common.cuh"
#include "host_common.h"
#include "tcgen05.cuh"

namespace pa {

constexpr int kChunk = 16;                        // tokens per ring stage
constexpr int kRowBytes = 256;                    // bf16 / f32 rows (FP8 rows: 128)
constexpr float kRescaleThreshold = 8.0f;         // log2 units: rescale when max grows > 256x
constexpr unsigned kFull = 0xffffffffu;

struct DecodeParams {
    const unsigned char* k_pool;
    const unsigned char* v_pool;
    int32_t num_blocks;
    int32_t log2_bp;
    int32_t num_kv_heads;
    const void* q;
    int32_t num_q_heads;
    const int32_t* block_tables;
    int32_t max_blocks;
    const int32_t* context_lens;
    float scale_log2;
    int32_t part_chunks;
    int32_t max_parts;
    int32_t max_context;
    int32_t window;               // sliding window in positions (0: the whole context)
    float* out;
    float* ws_m;
    float* ws_l;
    float* ws_acc;
    int32_t* d_err;
    // fused step only
    const unsigned char* k_new;   // [B][H_kv][D] new rows
    const unsigned char* v_new;
    const int64_t* slot_mapping;  // [B] slot of position context_lens[s] - 1
    int32_t* sem;                 // [B][H_kv] partitions finished (zero between calls)
    // FP8 pages: float row scales [num_blocks][H_kv][B_p]
    const float* k_scale;
    const float* v_scale;
    // shared-prefix decode only: declared pairs (nullptr otherwise)
    const int32_t* partner;       // [B] the other member of a pair, or -1
    const int32_t* shared_lens;   // [B] tokens on the pair's shared leading pages
    int32_t num_seqs;
};

// Storage types of a pool row.  A lane owns one column of kColBytes bytes of a
// row (16 lanes cover a row), which load2 turns into element pairs (float2).
// Q is read with Row<Q>.  kScaled: the pool carries one float scale per row
// (FP8 pages), applied to the finished score (K) and folded into the
// probability (V).
template <typename T>
struct Row;
template <>
struct Row<float> {
    static constexpr int N = 4;  // elements per 16-byte column
    static constexpr int kRowBytes = 256, kColBytes = 16;
    static constexpr bool kScaled = false;
    using Q = float;
    static PA_DEVICE void load2(const unsigned char* p, float2 (&f)[2]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        f[0] = make_float2(__uint_as_float(u.x), __uint_as_float(u.y));
        f[1] = make_float2(__uint_as_float(u.z), __uint_as_float(u.w));
    }
};
template <>
struct Row<uint16_t> {  // bf16 bit patterns
    static constexpr int N = 8;
    static constexpr int kRowBytes = 256, kColBytes = 16;
    static constexpr bool kScaled = false;
    using Q = uint16_t;
    static PA_DEVICE void load2(const unsigned char* p, float2 (&f)[4]) {
        const uint4 u = *reinterpret_cast<const uint4*>(p);
        f[0] = make_float2(bf16_lo(u.x), bf16_hi(u.x));
        f[1] = make_float2(bf16_lo(u.y), bf16_hi(u.y));
        f[2] = make_float2(bf16_lo(u.z), bf16_hi(u.z));
        f[3] = make_float2(bf16_lo(u.w), bf16_hi(u.w));
    }
};
// two E4M3 codes (low byte first) -> their values, exactly (through f16x2)
PA_DEVICE float2 e4m3x2_to_float2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
    float2 f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
        "cvt.f32.f16 %0, lo;\n\tcvt.f32.f16 %1, hi;\n\t}"
        : "=f"(f.x), "=f"(f.y) : "r"(h2));
    return f;
}
template <>
struct Row<uint8_t> {  // FP8 E4M3 codes, one float scale per row
    static constexpr int N = 8;  // elements per 8-byte column
    static constexpr int kRowBytes = 128, kColBytes = 8;
    static constexpr bool kScaled = true;
    using Q = uint16_t;  // queries stay bf16
    static PA_DEVICE void load2(const unsigned char* p, float2 (&f)[4]) {
        const uint2 u = *reinterpret_cast<const uint2*>(p);
        f[0] = e4m3x2_to_float2(u.x & 0xffffu);
        f[1] = e4m3x2_to_float2(u.x >> 16);
        f[2] = e4m3x2_to_float2(u.y & 0xffffu);
        f[3] = e4m3x2_to_float2(u.y >> 16);
    }
};

// Shared memory of a CTA: per warp S ring stages of [K chunk | V chunk |
// K row scales | V row scales] (the scales only for scaled rows), then the
// stages' mbarriers and valid-row masks, then the (p, p) probability pairs.
template <int W, int S, int G, typename R>
struct DecodeSmem {
    static constexpr int chunk = kChunk * R::kRowBytes;          // K (or V) bytes per stage
    static constexpr int scales = R::kScaled ? 2 * kChunk * 4 : 0;
    static constexpr int stage = 2 * chunk + scales;
    static constexpr size_t ring = (size_t)W * S * stage;
    static constexpr size_t bars = ring;
    static constexpr size_t masks = bars + (size_t)W * S * 8;
    static constexpr size_t probs = masks + (size_t)W * S * 4;
    static constexpr size_t total = probs + (size_t)W * kChunk * G * 8;  // (p, p) pairs
    // the CTA combine reuses the ring: per warp 2G + G*D floats
    static_assert((size_t)W * (4 * G + G * 128) * 4 <= ring, "combine area must fit in the ring");
    static_assert(stage % 16 == 0, "bulk copy destinations stay 16-byte aligned");
};

// Producer side: lane 0 of a warp fetches chunk `c` (16 tokens starting at
// c*16) of sequence s, kv-head h, into the ring stage at `kst`: K rows, V rows
// and, for scaled rows, the 16 K and 16 V row scales.  Writes the mask of rows
// in [lo, n), then arms the barrier with the bytes in flight.
template <int W, typename R>
PA_DEVICE void issue_chunk(const DecodeParams& p, int s, int h, int n, int lo, int c,
                           int32_t id_first, unsigned char* kst, uint64_t* bar,
                           uint32_t* mask_slot) {
    constexpr int RB = R::kRowBytes, CB = kChunk * RB;
    constexpr uint32_t kScaleBytes = R::kScaled ? 4 : 0;  // per row, for K and for V
    const int t0 = c * kChunk;
    const int bp = 1 << p.log2_bp;
    const int valid = min(kChunk, n - t0);
    uint32_t mask = 0, bytes = 0;
    const int64_t page_rows = (int64_t)bp;
    if (bp >= kChunk) {
        const int32_t id = id_first;
        if (id < 0 || id >= p.num_blocks) {
            set_error(p.d_err, id < 0 ? PA_ERR_NEGATIVE_BLOCK : PA_ERR_OUT_OF_RANGE);
            *mask_slot = 0;
            mbar_arrive_expect_tx(bar, 0);
            return;
        }
        mask = (1u << valid) - 1u;  // valid <= 16
        if (lo > t0) mask &= ~((1u << (lo - t0)) - 1u);  // rows before the window
        bytes = 2 * CB + 2 * kChunk * kScaleBytes;
        const int64_t row0 = ((int64_t)id * p.num_kv_heads + h) * page_rows + (t0 & (bp - 1));
        *mask_slot = mask;
        mbar_arrive_expect_tx(bar, bytes);
        bulk_g2s(kst, p.k_pool + row0 * RB, CB, bar);
        bulk_g2s(kst + CB, p.v_pool + row0 * RB, CB, bar);
        if constexpr (R::kScaled) {
            bulk_g2s(kst + 2 * CB, p.k_scale + row0, kChunk * 4, bar);
            bulk_g2s(kst + 2 * CB + kChunk * 4, p.v_scale + row0, kChunk * 4, bar);
        }
        return;
    }
    // block size below the chunk: 16 / bp pages per chunk
    const int pages = kChunk >> p.log2_bp;
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks;
    const int e0 = t0 >> p.log2_bp;
    int32_t ids[kChunk];
#pragma unroll 1
    for (int pp = 0; pp < pages; ++pp) {
        ids[pp] = -1;
        const int tok = t0 + pp * bp;
        if (tok >= n) break;
        if (tok + bp <= lo) continue;  // the whole page is before the window
        const int e = e0 + pp;
        const int32_t id = (e < p.max_blocks) ? __ldg(table + e) : -1;
        if (e >= p.max_blocks || id >= p.num_blocks) {
            set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
            continue;
        }
        if (id < 0) {
            set_error(p.d_err, PA_ERR_NEGATIVE_BLOCK);
            continue;
        }
        ids[pp] = id;
        const int rows = min(bp, n - tok);
        mask |= ((1u << rows) - 1u) << (pp * bp);
        bytes += 2u * (uint32_t)bp * (RB + kScaleBytes);
    }
    if (lo > t0) mask &= ~((1u << (lo - t0)) - 1u);  // rows before the window
    *mask_slot = mask;
    mbar_arrive_expect_tx(bar, bytes);
#pragma unroll 1
    for (int pp = 0; pp < pages; ++pp) {
        if (t0 + pp * bp >= n) break;
        if (ids[pp] < 0) continue;
        const int64_t row0 = ((int64_t)ids[pp] * p.num_kv_heads + h) * page_rows;
        const uint32_t nb = (uint32_t)bp * RB;
        bulk_g2s(kst + pp * bp * RB, p.k_pool + row0 * RB, nb, bar);
        bulk_g2s(kst + CB + pp * bp * RB, p.v_pool + row0 * RB, nb, bar);
        if constexpr (R::kScaled) {  // bp >= 4: 16-byte pieces
            bulk_g2s(kst + 2 * CB + pp * bp * 4, p.k_scale + row0, (uint32_t)bp * 4, bar);
            bulk_g2s(kst + 2 * CB + kChunk * 4 + pp * bp * 4, p.v_scale + row0, (uint32_t)bp * 4,
                     bar);
        }
    }
}

// atomicAdd with release-acquire semantics at GPU scope
PA_DEVICE int atom_add_acq_rel_gpu(int32_t* p, int v) {
    int old;
    asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// Fused step: merge of the (m, l, acc) partials of the G heads of (s, h),
// run by the last partition CTA of the group (same math as
// decode_merge_kernel).  `sm` is free shared memory (the ring).
template <int G, int D, int W>
PA_DEVICE void merge_group(const DecodeParams& p, int s, int h, int n_parts, float* sm) {
    constexpr int kCap = 1024;                // partitions per pass through shared memory
    constexpr int NV = G * D / 4;             // float4 outputs of the group
    constexpr int NO = (NV + W * 32 - 1) / (W * 32);
    constexpr int U = 4;                      // partitions per batch of independent loads
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t qh0 = (int64_t)s * p.num_q_heads + (int64_t)h * G;
    float* Mh = sm;
    float* Lh = sm + G;
    float* wts = sm + 2 * G;
    // maxima over the partitions, one warp per head
    for (int g = warp; g < G; g += W) {
        const float* mrow = p.ws_m + (qh0 + g) * p.max_parts;
        float M = -INFINITY;
        for (int i = lane; i < n_parts; i += 32) M = fmaxf(M, __ldcg(mrow + i));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
        if (lane == 0) {
            Mh[g] = M;
            Lh[g] = 0.f;
        }
    }
    float4 a[NO];
#pragma unroll
    for (int k = 0; k < NO; ++k) a[k] = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int p0 = 0; p0 < n_parts; p0 += kCap) {
        const int cnt = min(kCap, n_parts - p0);
        __syncthreads();  // maxima ready / previous weights consumed
        for (int g = warp; g < G; g += W) {
            const int64_t r0 = (qh0 + g) * p.max_parts + p0;
            float ls = 0.f;
            for (int i = lane; i < cnt; i += 32) {
                const float w = ex2(__ldcg(p.ws_m + r0 + i) - Mh[g]);
                wts[g * kCap + i] = w;
                ls = fmaf(__ldcg(p.ws_l + r0 + i), w, ls);
            }
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) ls += __shfl_xor_sync(kFull, ls, off);
            if (lane == 0) Lh[g] += ls;
        }
        __syncthreads();
        // every thread's outputs advance together over U partitions at a time,
        // so U * NO independent 16-byte loads are in flight
        for (int i0 = 0; i0 < cnt; i0 += U) {
            float4 v[NO][U];
#pragma unroll
            for (int k = 0; k < NO; ++k) {
                const int idx = threadIdx.x + k * W * 32;
                const int g = idx / (D / 4), d4 = idx - g * (D / 4);
                const float4* ar = reinterpret_cast<const float4*>(
                    p.ws_acc + ((qh0 + g) * p.max_parts + p0) * D) + d4;
#pragma unroll
                for (int u = 0; u < U; ++u)
                    v[k][u] = (idx < NV && i0 + u < cnt) ? __ldcg(ar + (int64_t)(i0 + u) * (D / 4))
                                                         : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int k = 0; k < NO; ++k) {
                const int idx = threadIdx.x + k * W * 32;
                const int g = min(idx / (D / 4), G - 1);
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float w = i0 + u < cnt ? wts[g * kCap + i0 + u] : 0.f;
                    a[k].x = fmaf(v[k][u].x, w, a[k].x);
                    a[k].y = fmaf(v[k][u].y, w, a[k].y);
                    a[k].z = fmaf(v[k][u].z, w, a[k].z);
                    a[k].w = fmaf(v[k][u].w, w, a[k].w);
                }
            }
        }
    }
    __syncthreads();
#pragma unroll
    for (int k = 0; k < NO; ++k) {
        const int idx = threadIdx.x + k * W * 32;
        if (idx < NV) {
            const int g = idx / (D / 4), d4 = idx - g * (D / 4);
            const float inv = 1.f / Lh[g];
            reinterpret_cast<float4*>(p.out + (qh0 + g) * D)[d4] =
                make_float4(a[k].x * inv, a[k].y * inv, a[k].z * inv, a[k].w * inv);
        }
    }
}

template <typename T, int G, int W, int S, bool kFused>
PA_DEVICE void decode_partition_body(const DecodeParams& p) {
    using R = Row<T>;
    constexpr int EPL = R::N;                 // elements of a row per lane
    constexpr int D = EPL * 16;               // head_dim
    constexpr int NS = 8 * G;                 // partial scores per lane: 8 rows x G heads
    constexpr int ROUNDS = G == 1 ? 3 : 4;    // halving rounds of the transpose-reduce
    constexpr int NSF = G == 1 ? 1 : G / 2;   // finished scores per lane
    using L = DecodeSmem<W, S, G, R>;
    constexpr int RB = R::kRowBytes;          // bytes of a stored row
    static_assert(G == 1 || G == 2 || G == 4 || G == 8, "group size");
    static_assert(!kFused || RB == 256, "the fused new-row write moves 16 bytes per lane");

    const int s = blockIdx.x, h = blockIdx.y, part = blockIdx.z;
    griddep_wait();  // K/V rows, tables and lengths may come from the previous kernel
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool big_pages = p.log2_bp >= 4;
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks;
    auto table_id_at = [&](int c) -> int32_t {
        const int e = (c * kChunk) >> p.log2_bp;
        return e < p.max_blocks ? __ldg(table + e) : -1;
    };
    // With a sliding window only positions lo .. n-1 are visible (the window of
    // the query at n - 1); partitions then start at chunk c_lo = lo / 16.
    // Block-table prefetch: lane j holds the id of this warp's local chunk j;
    // without a window it goes out together with the length load.
    int32_t id_reg = -1;
    if (p.window <= 0 && big_pages) id_reg = table_id_at(part * p.part_chunks + warp + lane * W);
    int n = __ldg(p.context_lens + s);
    if (n > p.max_context) {  // longer than the plan allows
        if (part == 0 && h == 0 && threadIdx.x == 0) set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
        n = p.max_context;
    }
    int c_lo = 0;
    if (p.window > 0) {
        if (n > p.window) c_lo = (n - p.window) / kChunk;
        if (big_pages) id_reg = table_id_at(c_lo + part * p.part_chunks + warp + lane * W);
    }
    const int lo = (p.window > 0 && n > p.window) ? n - p.window : 0;
    const int c_begin = c_lo + part * p.part_chunks;
    const int first = c_begin + warp;  // this warp's chunks: first + i*W
    auto table_id = [&](int i) -> int32_t { return table_id_at(first + i * W); };
    const int n_chunks = (n + kChunk - 1) / kChunk;
    if (n <= 0 || c_begin >= n_chunks) return;
    const int c_end = min(c_begin + p.part_chunks, n_chunks);
    const int n_parts = (n_chunks - c_lo + p.part_chunks - 1) / p.part_chunks;

    extern __shared__ __align__(128) unsigned char smem[];
    unsigned char* ring = smem + (size_t)warp * S * L::stage;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::bars) + warp * S;
    uint32_t* masks = reinterpret_cast<uint32_t*>(smem + L::masks) + warp * S;
    float2* ps = reinterpret_cast<float2*>(smem + L::probs) + warp * kChunk * G;
    __shared__ int aborted;
    if (threadIdx.x == 0) aborted = 0;

    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < S; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    const int my_n = first < c_end ? (c_end - first + W - 1) / W : 0;
    int id_base = 0;

    // the error check for the table width happens at issue time
    auto issue = [&](int i, int32_t id) {
        const int stage = i % S;
        const int c = first + i * W;
        if (big_pages && ((c * kChunk) >> p.log2_bp) >= p.max_blocks) id = p.num_blocks;  // flagged
        issue_chunk<W, R>(p, s, h, n, lo, c, id, ring + (size_t)stage * L::stage, &bars[stage],
                          &masks[stage]);
    };

    // fused step: the warp that streams the chunk holding position n - 1 loads
    // the new token's row of (s, h) now (K in lanes 0-15, V in lanes 16-31,
    // 16 bytes each) and, once that chunk is in shared memory, stores it both
    // to its slot in the pool and over the chunk's copy of the row -- the bulk
    // copy may have read the slot before or after the store, the attention
    // uses the new row either way
    const int last_chunk = n_chunks - 1;
    const bool owner = kFused && c_end == n_chunks && last_chunk >= first &&
                       (last_chunk - first) % W == 0;
    // kept in shared memory so that no registers stay live through the main loop
    __shared__ uint4 new_row[32];
    __shared__ int64_t new_slot;
    __shared__ int32_t last_pid;  // table entry of the page holding position n - 1
    uint4 row_reg = make_uint4(0, 0, 0, 0);
    if (owner) {
        const int64_t src = ((int64_t)s * p.num_kv_heads + h) * kRowBytes + (lane & 15) * 16;
        row_reg = __ldg(reinterpret_cast<const uint4*>((lane < 16 ? p.k_new : p.v_new) + src));
        if (lane == 0) {
            new_slot = __ldg(p.slot_mapping + s);
            const int e = (n - 1) >> p.log2_bp;
            last_pid = e < p.max_blocks ? __ldg(table + e) : -1;
        }
    }

    // prologue: first S chunks in flight
#pragma unroll
    for (int i = 0; i < S; ++i) {
        const int32_t id = __shfl_sync(kFull, id_reg, i & 31);
        if (lane == 0 && i < my_n) issue(i, id);
    }
    if (owner) new_row[lane] = row_reg;  // the loads completed behind the prologue's copies

    // per-lane constants of the transpose-reduce layout
    const int half = lane >> 4;               // which row of a row pair
    const int col = lane & 15;                // 16-byte column of the row
    const int jx = (lane >> 1) & 7;           // local row j holds row 2*(j^jx)+half
    const int gx = G == 1 ? 0 : (lane & 1) * (G / 2);  // local head g holds head g^gx
    const int t_mine = 2 * jx + half;         // row of this lane's finished scores

    // query registers (element pairs), permuted by gx, pre-scaled into base-2 logits
    constexpr int EP = EPL / 2;
    float2 q2[G][EP];
    {
        using QT = typename R::Q;  // the query's storage type (bf16 for FP8 pages)
        const QT* qb = reinterpret_cast<const QT*>(p.q) +
                       ((int64_t)s * p.num_q_heads + (int64_t)h * G) * D + col * EPL;
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float2 f[EP];
            Row<QT>::load2(reinterpret_cast<const unsigned char*>(qb + (int64_t)(g ^ gx) * D), f);
#pragma unroll
            for (int e = 0; e < EP; ++e)
                q2[g][e] = make_float2(f[e].x * p.scale_log2, f[e].y * p.scale_log2);
        }
    }

    // P*V accumulators: element pairs of this lane's column, for every head
    float2 acc[G][EP];
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < EP; ++e) acc[g][e] = make_float2(0.f, 0.f);
    float m[G];
#pragma unroll
    for (int g = 0; g < G; ++g) m[g] = -INFINITY;
    float l_lane[NSF];
#pragma unroll
    for (int x = 0; x < NSF; ++x) l_lane[x] = 0.f;

    bool ok = true;
#pragma unroll 1
    for (int i = 0; i < my_n; ++i) {
        const int stage = i % S;
        const uint32_t parity = (uint32_t)(i / S) & 1u;
        ok = mbar_wait(&bars[stage], parity, p.d_err);
        if (!__all_sync(kFull, ok)) {
            ok = false;
            break;
        }
        const uint32_t vmask = masks[stage];
        const bool masked = vmask != 0xffffu;
        const unsigned char* kst = ring + (size_t)stage * L::stage;
        const unsigned char* vst = kst + L::chunk;
        const float* ksc = reinterpret_cast<const float*>(kst + 2 * L::chunk);  // scaled rows only
        const float* vsc = ksc + kChunk;
        if (owner && first + i * W == last_chunk) {
            const int pos = n - 1;
            const int64_t bpm = (1 << p.log2_bp) - 1;
            const int64_t slot = new_slot;
            const int32_t pid = last_pid;
            int err = 0;
            if (slot < 0 || slot >= ((int64_t)p.num_blocks << p.log2_bp))
                err = PA_ERR_OUT_OF_RANGE;
            else if (pid < 0 || (slot >> p.log2_bp) != pid || (slot & bpm) != (pos & bpm))
                err = PA_ERR_INVALID_ARG;  // not the slot of the last position
            if (err != 0) {
                if (lane == 0) set_error(p.d_err, err);
            } else {
                const uint4 v = new_row[lane];
                const int64_t row = ((int64_t)pid * p.num_kv_heads + h) * (bpm + 1) + (pos & bpm);
                unsigned char* pool = const_cast<unsigned char*>(lane < 16 ? p.k_pool : p.v_pool);
                *reinterpret_cast<uint4*>(pool + row * kRowBytes + (lane & 15) * 16) = v;
                unsigned char* st = const_cast<unsigned char*>(lane < 16 ? kst : vst);
                *reinterpret_cast<uint4*>(st + (pos & (kChunk - 1)) * kRowBytes + (lane & 15) * 16) = v;
                fence_proxy_async_smem();  // before a later bulk copy refills this stage
            }
            __syncwarp();
        }

        // ---- scores: partial dots over this lane's column, then transpose-reduce
        float part[NS];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = 2 * (j ^ jx) + half;
            float2 k[EP];
            R::load2(kst + row * RB + col * R::kColBytes, k);
#pragma unroll
            for (int g = 0; g < G; ++g) {
                // even and odd elements accumulate in the two halves of a packed FMA
                float2 a = make_float2(0.f, 0.f);
#pragma unroll
                for (int e = 0; e < EP; ++e) a = __ffma2_rn(q2[g][e], k[e], a);
                part[j * G + g] = a.x + a.y;
            }
        }
#pragma unroll
        for (int r = 0; r < ROUNDS; ++r) {
            const int hn = NS >> (r + 1);
#pragma unroll
            for (int x = 0; x < hn; ++x)
                part[x] += __shfl_xor_sync(kFull, part[x + hn], 8 >> r);
        }
        if (G == 1) part[0] += __shfl_xor_sync(kFull, part[0], 1);

        // ---- online softmax (base 2) with rare rescaling
        const bool tvalid = !masked || ((vmask >> t_mine) & 1u);
        float sc[NSF], mm[NSF];
        // scaled rows: the K row scale multiplies the finished score
        const float kscale = (R::kScaled && tvalid) ? ksc[t_mine] : 1.f;
#pragma unroll
        for (int x = 0; x < NSF; ++x) {
            sc[x] = tvalid ? part[x] * kscale : -INFINITY;
            mm[x] = G == 1 ? m[0] : ((lane & 1) ? m[G / 2 + x] : m[x]);
        }
        bool need = false;
#pragma unroll
        for (int x = 0; x < NSF; ++x) need |= sc[x] > mm[x] + kRescaleThreshold;
        if (__any_sync(kFull, need)) {
            float cm[NSF];
#pragma unroll
            for (int x = 0; x < NSF; ++x) cm[x] = sc[x];
#pragma unroll
            for (int off = 2; off <= 16; off <<= 1)
#pragma unroll
                for (int x = 0; x < NSF; ++x) cm[x] = fmaxf(cm[x], __shfl_xor_sync(kFull, cm[x], off));
            float cmax[G];
            if (G == 1) {
                cmax[0] = cm[0];
            } else {
#pragma unroll
                for (int x = 0; x < NSF; ++x) {
                    const float o = __shfl_xor_sync(kFull, cm[x], 1);
                    cmax[x] = (lane & 1) ? o : cm[x];
                    cmax[G / 2 + x] = (lane & 1) ? cm[x] : o;
                }
            }
            float corr[G];
#pragma unroll
            for (int g = 0; g < G; ++g) {
                const float mn = fmaxf(m[g], cmax[g]);
                corr[g] = ex2(m[g] - mn);
                m[g] = mn;
                const float2 c2 = make_float2(corr[g], corr[g]);
#pragma unroll
                for (int e = 0; e < EP; ++e) acc[g][e] = __fmul2_rn(acc[g][e], c2);
            }
#pragma unroll
            for (int x = 0; x < NSF; ++x) {
                l_lane[x] *= G == 1 ? corr[0] : ((lane & 1) ? corr[G / 2 + x] : corr[x]);
                mm[x] = G == 1 ? m[0] : ((lane & 1) ? m[G / 2 + x] : m[x]);
            }
        }
        float pr[NSF];
#pragma unroll
        for (int x = 0; x < NSF; ++x) {
            pr[x] = tvalid ? ex2(sc[x] - mm[x]) : 0.f;
            l_lane[x] += pr[x];
        }

        // ---- broadcast probabilities of the 16 rows x G heads, each stored as a
        //      (p, p) pair so the P*V packed FMAs read their operand directly
        //      (scaled rows: the V row scale is folded into the pair; l keeps p)
        const float vscale = R::kScaled ? (tvalid ? vsc[t_mine] : 0.f) : 1.f;
        if (G == 1) {
            if ((lane & 1) == 0) ps[t_mine] = make_float2(pr[0] * vscale, pr[0] * vscale);
        } else {
#pragma unroll
            for (int x = 0; x < NSF; ++x) {
                const float pv = pr[x] * vscale;
                ps[t_mine * G + gx + x] = make_float2(pv, pv);
            }
        }
        __syncwarp();

        // ---- P * V over this lane's 8 rows and 16-byte column
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const int row = 2 * j + half;
            float2 pg[G];
#pragma unroll
            for (int g = 0; g < G; ++g) pg[g] = ps[row * G + g];
            float2 v[EP];
            R::load2(vst + row * RB + col * R::kColBytes, v);
            if (masked && !((vmask >> row) & 1u)) {
#pragma unroll
                for (int e = 0; e < EP; ++e) v[e] = make_float2(0.f, 0.f);  // unwritten rows may hold NaN
            }
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < EP; ++e) acc[g][e] = __ffma2_rn(pg[g], v[e], acc[g][e]);
        }
        __syncwarp();

        // ---- refill this stage with chunk i + S
        const int nxt = i + S;
        if (big_pages && nxt - id_base >= 32) {
            id_base += 32;
            id_reg = (id_base + lane < my_n) ? table_id(id_base + lane) : -1;
        }
        const int32_t nid = big_pages ? __shfl_sync(kFull, id_reg, (nxt - id_base) & 31) : -1;
        if (lane == 0 && nxt < my_n) issue(nxt, nid);
    }
    if (!ok) aborted = 1;
    griddep_launch();  // the merge may start launching; it waits for this grid to finish

    // ---- finish this warp's state
#pragma unroll
    for (int g = 0; g < G; ++g)
#pragma unroll
        for (int e = 0; e < EP; ++e) {
            acc[g][e].x += __shfl_xor_sync(kFull, acc[g][e].x, 16);
            acc[g][e].y += __shfl_xor_sync(kFull, acc[g][e].y, 16);
        }
#pragma unroll
    for (int off = 2; off <= 16; off <<= 1)
#pragma unroll
        for (int x = 0; x < NSF; ++x) l_lane[x] += __shfl_xor_sync(kFull, l_lane[x], off);
    float lsum[G];
    if (G == 1) {
        lsum[0] = l_lane[0];
    } else {
#pragma unroll
        for (int x = 0; x < NSF; ++x) {
            const float o = __shfl_xor_sync(kFull, l_lane[x], 1);
            lsum[x] = (lane & 1) ? o : l_lane[x];
            lsum[G / 2 + x] = (lane & 1) ? l_lane[x] : o;
        }
    }

    // ---- combine the CTA's warps (reusing the ring) and write
    __syncthreads();
    if (aborted) {
        if constexpr (!kFused) return;
        // a fused step still counts this partition, so the group's semaphore
        // returns to zero (the merged result is flagged invalid by *d_err)
        if (n_parts > 1) {
            __shared__ int last_aborted;
            if (threadIdx.x == 0) {
                const int old = atom_add_acq_rel_gpu(p.sem + (int64_t)s * p.num_kv_heads + h, 1);
                last_aborted = old == n_parts - 1;
                if (last_aborted) atomicExch(p.sem + (int64_t)s * p.num_kv_heads + h, 0);
            }
            __syncthreads();
        }
        return;
    }
    // per warp: acc [G][D], then m [G], l [G]; the stride keeps float4 alignment
    float* cw = reinterpret_cast<float*>(smem);
    constexpr int MOFF = G * D, LOFF = G * D + G;
    constexpr int WSTRIDE = G * D + ((2 * G + 3) / 4) * 4;
    float* mine = cw + warp * WSTRIDE;
    if (lane == 0) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            mine[MOFF + g] = m[g];
            mine[LOFF + g] = lsum[g];
        }
    }
    if (lane < 16) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < EP; e += 2)
                *reinterpret_cast<float4*>(mine + g * D + col * EPL + 2 * e) =
                    make_float4(acc[g][e].x, acc[g][e].y, acc[g][e + 1].x, acc[g][e + 1].y);
    }
    __syncthreads();
    const int64_t qh0 = (int64_t)s * p.num_q_heads + (int64_t)h * G;
    for (int idx = threadIdx.x; idx < G * D; idx += W * 32) {
        const int g = idx / D, d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < W; ++w) M = fmaxf(M, cw[w * WSTRIDE + MOFF + g]);
        float Lsum = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < W; ++w) {
            const float c = ex2(cw[w * WSTRIDE + MOFF + g] - M);
            Lsum = fmaf(cw[w * WSTRIDE + LOFF + g], c, Lsum);
            A = fmaf(cw[w * WSTRIDE + g * D + d], c, A);
        }
        if (n_parts == 1) {
            p.out[(qh0 + g) * D + d] = A / Lsum;
        } else {
            const int64_t wi = (qh0 + g) * p.max_parts + part;
            p.ws_acc[wi * D + d] = A;
            if (d == 0) {
                p.ws_m[wi] = M;
                p.ws_l[wi] = Lsum;
            }
        }
    }
    if constexpr (kFused) {
        if (n_parts > 1) {
            // publish this partition's partials and count it: the barrier orders
            // the CTA's stores before thread 0's release-acquire add, which makes
            // them visible to whichever CTA of the group counts last; that one
            // merges (its acquire orders the reads of the others' partials)
            __shared__ int is_last;
            __syncthreads();
            if (threadIdx.x == 0) {
                int32_t* sem = p.sem + (int64_t)s * p.num_kv_heads + h;
                const int old = atom_add_acq_rel_gpu(sem, 1);
                is_last = old == n_parts - 1;
                if (is_last) atomicExch(sem, 0);  // every partition of the group has counted
            }
            __syncthreads();
            if (is_last) merge_group<G, D, W>(p, s, h, n_parts, cw);
        }
    }
}

// The partition kernel.  FP8 rows at G <= 4 need half the shared memory of
// 16-bit rows, so their variant caps registers for 4 resident CTAs per SM;
// the others keep the compiler's own register choice (3 CTAs per SM by
// shared memory, 2 at G = 8).
template <typename T, int G, int W, int S, bool kFused>
__global__ void __launch_bounds__(W * 32) decode_partition_kernel(const DecodeParams p) {
    decode_partition_body<T, G, W, S, kFused>(p);
}

template <typename T, int G, int W, int S>
__global__ void __launch_bounds__(W * 32, 4) decode_partition_kernel_4ctas(const DecodeParams p) {
    decode_partition_body<T, G, W, S, false>(p);
}

}  // namespace pa
#include "decode_mma.cuh"
#include "decode_mma_fp8.cuh"
namespace pa {

// Merge of split-KV partials (P1 §4): M = max m_p, L = sum l_p 2^(m_p - M),
// out = sum acc_p 2^(m_p - M) / L.  One CTA per (sequence, q-head): the
// partition maxima and sums are loaded in parallel (one per thread) into
// shared memory; for head_dim 64 or 128 and up to 128 partitions each thread
// sums one float4 column over a quarter (an eighth) of the partitions with
// all of its loads issued up front, otherwise every thread sums its output
// element over all partitions.
constexpr int kMergeThreads = 128;
constexpr int kMergeMaxParts = 1024;  // partitions handled per pass through shared memory

template <int kPre>
__global__ void __launch_bounds__(kMergeThreads) decode_merge_kernel(const DecodeParams p, int D) {
    const int s = blockIdx.x / p.num_q_heads;
    const int g = blockIdx.x - s * p.num_q_heads;
    griddep_wait();  // partials come from the partition kernel
    const int n = min(__ldg(p.context_lens + s), p.max_context);
    if (n <= 0) return;
    const int n_chunks = (n + kChunk - 1) / kChunk;
    const int c_lo = (p.window > 0 && n > p.window) ? (n - p.window) / kChunk : 0;
    int n_parts = (n_chunks - c_lo + p.part_chunks - 1) / p.part_chunks;
    if (p.partner != nullptr) {  // shared-prefix decode: pair slots, then own partitions
        const mma::Pairing pr = mma::pairing_of(p, s, false);
        n_parts = pr.np_shared + pr.np_priv;
    }
    n_parts = min(n_parts, p.max_parts);
    if (n_parts <= 1) return;
    __shared__ float wts[kMergeMaxParts];
    __shared__ float red[kMergeThreads / 32];
    const int64_t base = ((int64_t)s * p.num_q_heads + g) * p.max_parts;
    const int tid = threadIdx.x;
    if (n_parts <= kMergeThreads && (D == 64 || D == 128)) {
        // thread t owns float4 column t % (D/4) of the output and the partitions
        // grp, grp + ngrp, ... (grp = t / (D/4)); the first kPre of them are
        // loaded up front together with the maxima and sums, so the CTA spends
        // about one round of load latency; the groups are added at the end
        const int nvec = D >> 2, ngrp = kMergeThreads / nvec;
        const int col = tid % nvec, grp = tid / nvec;
        const float4* a4 = reinterpret_cast<const float4*>(p.ws_acc + base * D) + col;
        float4 pre[kPre];
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int i = grp + u * ngrp;
            pre[u] = i < n_parts ? __ldcg(a4 + (int64_t)i * nvec) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
        const float mi = tid < n_parts ? __ldcg(p.ws_m + base + tid) : -INFINITY;
        const float li = tid < n_parts ? __ldcg(p.ws_l + base + tid) : 0.f;
        float M = mi;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
        if ((tid & 31) == 0) red[tid >> 5] = M;
        __syncthreads();
        M = red[0];
#pragma unroll
        for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red[w]);
        const float wi = tid < n_parts ? ex2(mi - M) : 0.f;
        wts[tid] = wi;
        float L = li * wi;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
        __syncthreads();  // everyone has read red[] for M; wts complete
        if ((tid & 31) == 0) red[tid >> 5] = L;
        __syncthreads();
        L = 0.f;
#pragma unroll
        for (int w = 0; w < kMergeThreads / 32; ++w) L += red[w];
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kPre; ++u) {
            const int i = grp + u * ngrp;
            const float w = i < n_parts ? wts[i] : 0.f;
            acc.x = fmaf(pre[u].x, w, acc.x);
            acc.y = fmaf(pre[u].y, w, acc.y);
            acc.z = fmaf(pre[u].z, w, acc.z);
            acc.w = fmaf(pre[u].w, w, acc.w);
        }
        for (int i = grp + kPre * ngrp; i < n_parts; i += ngrp) {
            const float4 v = __ldcg(a4 + (int64_t)i * nvec);
            const float w = wts[i];
            acc.x = fmaf(v.x, w, acc.x);
            acc.y = fmaf(v.y, w, acc.y);
            acc.z = fmaf(v.z, w, acc.z);
            acc.w = fmaf(v.w, w, acc.w);
        }
        __shared__ float4 grp_acc[kMergeThreads];
        grp_acc[tid] = acc;
        __syncthreads();
        if (tid < nvec) {
            float4 t = grp_acc[tid];
            for (int g2 = 1; g2 < ngrp; ++g2) {
                const float4 o = grp_acc[g2 * nvec + tid];
                t.x += o.x;
                t.y += o.y;
                t.z += o.z;
                t.w += o.w;
            }
            const float inv = 1.f / L;
            reinterpret_cast<float4*>(p.out + ((int64_t)s * p.num_q_heads + g) * D)[tid] =
                make_float4(t.x * inv, t.y * inv, t.z * inv, t.w * inv);
        }
        return;
    }
    // global max over partitions
    float M = -INFINITY;
    for (int i = tid; i < n_parts; i += kMergeThreads) M = fmaxf(M, p.ws_m[base + i]);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    if ((tid & 31) == 0) red[tid >> 5] = M;
    __syncthreads();
    M = red[0];
#pragma unroll
    for (int w = 1; w < kMergeThreads / 32; ++w) M = fmaxf(M, red[w]);
    float acc[2] = {0.f, 0.f}, L = 0.f;
    for (int p0 = 0; p0 < n_parts; p0 += kMergeMaxParts) {
        const int cnt = min(kMergeMaxParts, n_parts - p0);
        __syncthreads();
        for (int i = tid; i < cnt; i += kMergeThreads) wts[i] = ex2(p.ws_m[base + p0 + i] - M);
        for (int i = tid; i < cnt; i += kMergeThreads) L = fmaf(p.ws_l[base + p0 + i], wts[i], L);
        __syncthreads();
        const float* a = p.ws_acc + (base + p0) * D;
#pragma unroll 4
        for (int i = 0; i < cnt; ++i) {
            const float w = wts[i];
            if (tid < D) acc[0] = fmaf(a[(int64_t)i * D + tid], w, acc[0]);
            if (tid + kMergeThreads < D) acc[1] = fmaf(a[(int64_t)i * D + tid + kMergeThreads], w, acc[1]);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
    __syncthreads();
    if ((tid & 31) == 0) red[tid >> 5] = L;
    __syncthreads();
    L = 0.f;
#pragma unroll
    for (int w = 0; w < kMergeThreads / 32; ++w) L += red[w];
    float* o = p.out + ((int64_t)s * p.num_q_heads + g) * D;
    if (tid < D) o[tid] = acc[0] / L;
    if (tid + kMergeThreads < D) o[tid + kMergeThreads] = acc[1] / L;
}

// ---------------------------------------------------------------- host side
constexpr int kWarps = 4;
constexpr int kStages = 2;
// The automatic plan sizes partitions so that a batch whose every sequence
// had max_context tokens would fill kWaves rounds of resident CTAs; real
// batches are shorter on average, so they run about half as many.  Fewer,
// longer partitions measured faster on long contexts (less partial traffic,
// fewer CTA start-ups, whole rounds): 3072 tokens gave 224 us against 237 us
// at 1728 on 8 sequences of 32K-107K tokens at G = 8, while 4- to 16-way
// splits of U[128, 4096] contexts at G = 4 all lay within 90-94 us.
constexpr int kWaves = 5;

// The tensor-core partition kernel (decode_mma.cuh) serves bf16 pools with
// head_dim 128 and pages of >= 16 tokens (a chunk then lies in one page),
// when the pool's rows fit the int32 row coordinate of its TMA boxes, at
// G >= 2 query heads per kv-head; MHA (G = 1) and everything else run on
// the CUDA-core kernel.
static bool use_mma(const pa_kv_pool* pool, int32_t Hq) {
    const int G = pool->num_kv_heads > 0 ? Hq / pool->num_kv_heads : 1;
    return pool->dtype == PA_DTYPE_BF16 && pool->head_dim == mma::kD && pool->block_size >= 16 &&
           (int64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size <= INT32_MAX &&
           (G == 2 || G == 4 || G == 8);
}

static bool use_mma_fp8(const pa_kv_pool* pool, int32_t Hq);

// Partition CTAs per SM the plan counts on: 3 (the shared-memory limit of
// both tensor-core kernels and of 16-bit and f32 rows on the CUDA-core one),
// 2 for the CUDA-core kernel at G = 8, where registers allow only two.  (FP8
// rows at G <= 4 run 4 per SM, but measured fastest with the 3-per-SM plan:
// more partitions cost more in the merge than they gain in balance.)
static int ctas_per_sm(const pa_kv_pool* pool, int32_t Hq) {
    const int G = pool->num_kv_heads > 0 ? Hq / pool->num_kv_heads : 1;
    if (use_mma(pool, Hq) || use_mma_fp8(pool, Hq)) return 3;
    return G >= 8 ? 2 : 3;
}

struct Plan {
    int32_t part_chunks;
    int32_t max_parts;
    size_t ws_bytes;
    size_t off_l, off_acc;
};

static size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

static pa_status make_plan(const pa_kv_pool* pool, int32_t B, int32_t Hq, int32_t max_ctx,
                           int32_t partition_tokens, Plan* plan, int32_t window = 0,
                           int waves = kWaves) {
    if (B < 0 || Hq <= 0 || max_ctx < 0 || window < 0) return PA_ERR_INVALID_ARG;
    int64_t chunks_max = ((int64_t)max_ctx + kChunk - 1) / kChunk;
    // a window of w positions starting anywhere touches at most ceil(w/16) + 1 chunks
    if (window > 0) chunks_max = std::min<int64_t>(chunks_max, ((int64_t)window + kChunk - 1) / kChunk + 1);
    int64_t pc;
    if (partition_tokens > 0) {
        if (partition_tokens % kChunk != 0) return PA_ERR_INVALID_ARG;
        pc = partition_tokens / kChunk;
    } else if (partition_tokens == 0) {
        const int64_t units = (int64_t)B * pool->num_kv_heads;
        const int64_t target = (int64_t)device_sm_count() * ctas_per_sm(pool, Hq) * waves;
        pc = (units * chunks_max + target - 1) / (target > 0 ? target : 1);
        if (pc < 2 * kWarps) pc = 2 * kWarps;
        pc = (pc + kWarps - 1) / kWarps * kWarps;
    } else {
        return PA_ERR_INVALID_ARG;
    }
    if (chunks_max > 0 && (chunks_max + pc - 1) / pc > 65535) pc = (chunks_max + 65534) / 65535;
    if (pc > (int64_t)1 << 26) pc = (int64_t)1 << 26;
    plan->part_chunks = (int32_t)pc;
    plan->max_parts = (int32_t)(chunks_max > 0 ? (chunks_max + pc - 1) / pc : 1);
    if (plan->max_parts <= 1) {
        plan->ws_bytes = plan->off_l = plan->off_acc = 0;
        return PA_OK;
    }
    const size_t rows = (size_t)B * Hq * plan->max_parts;
    plan->off_l = align256(rows * 4);
    plan->off_acc = plan->off_l + align256(rows * 4);
    plan->ws_bytes = plan->off_acc + rows * (size_t)pool->head_dim * 4;
    return PA_OK;
}

// Plan of the shared-prefix decode: partitions sized for 9 rounds of resident
// CTAs (its pair units carry 2G query columns, so their CTAs run longer; on 8
// sequences of 32K-107K tokens at G = 8 the coarser plan gained nothing:
// 231-236 us per step at 1728 tokens, 235 us at 3072); splitting a context
// at the shared length adds at most one slot per sequence.
constexpr int kSharedWaves = 9;
static pa_status make_shared_plan(const pa_kv_pool* pool, int32_t B, int32_t Hq, int32_t max_ctx,
                                  int32_t partition_tokens, Plan* plan) {
    pa_status st = make_plan(pool, B, Hq, max_ctx, partition_tokens, plan, 0, kSharedWaves);
    if (st != PA_OK) return st;
    plan->max_parts += 1;
    const size_t rows = (size_t)B * Hq * plan->max_parts;
    plan->off_l = align256(rows * 4);
    plan->off_acc = plan->off_l + align256(rows * 4);
    plan->ws_bytes = plan->off_acc + rows * (size_t)pool->head_dim * 4;
    return PA_OK;
}

template <typename T, int G, bool kFused>
static pa_status launch_partial(const DecodeParams& prm, int32_t B, int32_t Hkv, int32_t max_parts,
                                cudaStream_t stream) {
    using Lay = DecodeSmem<kWarps, kStages, G, Row<T>>;
    void (*kern)(const DecodeParams);
    if constexpr (Row<T>::kScaled && G <= 4 && !kFused)
        kern = decode_partition_kernel_4ctas<T, G, kWarps, kStages>;
    else
        kern = decode_partition_kernel<T, G, kWarps, kStages, kFused>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)Lay::total);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    dim3 grid((unsigned)B, (unsigned)Hkv, (unsigned)max_parts);
    cudaError_t e = launch_pdl(kern, grid, dim3(kWarps * 32), Lay::total, stream, prm);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return launch_status();
}

// Tensor maps of the K and V pools viewed as [rows][head_dim] bf16, boxes of
// 16 rows x 64 dims in the 128-byte swizzle.
static pa_status pool_maps(const pa_kv_pool* pool, CUtensorMap* mk, CUtensorMap* mv) {
    const uint64_t rows = (uint64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size;
    const uint64_t dims[2] = {(uint64_t)mma::kD, rows};
    const uint64_t strides[1] = {(uint64_t)mma::kD * 2};
    const uint32_t box[2] = {64, (uint32_t)kChunk};
    if (!encode_bf16_map_sw128(mk, pool->k_pool, 2, dims, strides, box) ||
        !encode_bf16_map_sw128(mv, pool->v_pool, 2, dims, strides, box))
        return PA_ERR_CUDA;
    return PA_OK;
}

template <typename K>
static pa_status launch_mma(K kern, const pa_kv_pool* pool, const DecodeParams& prm, int32_t B,
                            int32_t max_parts, bool* attr_done, cudaStream_t stream) {
    CUtensorMap mk, mv;
    pa_status st = pool_maps(pool, &mk, &mv);
    if (st != PA_OK) return st;
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)mma::kSmem);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    cudaError_t e = launch_pdl(kern, dim3((unsigned)B, (unsigned)pool->num_kv_heads, (unsigned)max_parts),
                               dim3(mma::kW * 32), mma::kSmem, stream, prm, mk, mv);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return launch_status();
}

template <int G, bool kFused = false>
static pa_status launch_partial_mma(const pa_kv_pool* pool, const DecodeParams& prm, int32_t B,
                                    int32_t max_parts, cudaStream_t stream) {
    static bool attr_done[64] = {false};
    return launch_mma(mma::decode_mma_kernel<G, kFused>, pool, prm, B, max_parts, attr_done, stream);
}

// FP8 pages at G = 8 run on the tensor-core FP8 kernel (decode_mma_fp8.cuh):
// pages of >= 16 tokens, head_dim 128.
static bool use_mma_fp8(const pa_kv_pool* pool, int32_t Hq) {
    const int G = pool->num_kv_heads > 0 ? Hq / pool->num_kv_heads : 1;
    return pool->dtype == PA_DTYPE_FP8_E4M3 && pool->head_dim == mma8::kD &&
           pool->block_size >= 16 && G == 8 &&
           (int64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size <= INT32_MAX;
}

static pa_status launch_partial_mma_fp8(const pa_kv_pool* pool, const DecodeParams& prm,
                                        int32_t B, int32_t Hkv, int32_t max_parts,
                                        cudaStream_t stream) {
    // the pools as [rows][128] codes, boxes of 16 rows in the 128-byte swizzle
    CUtensorMap mk, mv;
    const uint64_t rows = (uint64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size;
    const uint64_t dims[2] = {(uint64_t)mma8::kD, rows};
    const uint64_t strides[1] = {(uint64_t)mma8::kD};
    const uint32_t box[2] = {(uint32_t)mma8::kD, (uint32_t)kChunk};
    if (!encode_u8_map_sw128(&mk, pool->k_pool, 2, dims, strides, box) ||
        !encode_u8_map_sw128(&mv, pool->v_pool, 2, dims, strides, box))
        return PA_ERR_CUDA;
    auto kern = mma8::decode_fp8_mma_kernel<8>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)mma8::kSmem);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    cudaError_t e = launch_pdl(kern, dim3((unsigned)B, (unsigned)Hkv, (unsigned)max_parts),
                               dim3(mma8::kW * 32), mma8::kSmem, stream, prm, mk, mv);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return launch_status();
}

template <int G>
static pa_status launch_shared_mma(const pa_kv_pool* pool, const DecodeParams& prm, int32_t B,
                                   int32_t max_parts, cudaStream_t stream) {
    static bool attr_done[64] = {false};
    return launch_mma(mma::decode_shared_kernel<G>, pool, prm, B, max_parts, attr_done, stream);
}

template <typename T, bool kFused>
static pa_status dispatch_group(int G, const DecodeParams& prm, int32_t B, int32_t Hkv,
                                int32_t max_parts, cudaStream_t st) {
    switch (G) {
        case 1: return launch_partial<T, 1, kFused>(prm, B, Hkv, max_parts, st);
        case 2: return launch_partial<T, 2, kFused>(prm, B, Hkv, max_parts, st);
        case 4: return launch_partial<T, 4, kFused>(prm, B, Hkv, max_parts, st);
        case 8: return launch_partial<T, 8, kFused>(prm, B, Hkv, max_parts, st);
        default: return PA_ERR_UNSUPPORTED;
    }
}

static void bind_workspace(const Plan& plan, void* workspace, DecodeParams* prm) {
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    prm->ws_m = plan.ws_bytes ? reinterpret_cast<float*>(ws) : nullptr;
    prm->ws_l = plan.ws_bytes ? reinterpret_cast<float*>(ws + plan.off_l) : nullptr;
    prm->ws_acc = plan.ws_bytes ? reinterpret_cast<float*>(ws + plan.off_acc) : nullptr;
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_decode_partition_tokens(const pa_kv_pool* pool, int32_t num_seqs,
                                                int32_t num_q_heads, int32_t max_context,
                                                int32_t* partition_tokens) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (!partition_tokens) return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(pool, num_seqs, num_q_heads, max_context, 0, &plan);
    if (st != PA_OK) return st;
    *partition_tokens = plan.part_chunks * kChunk;
    return PA_OK;
}

extern "C" pa_status pa_decode_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                               int32_t num_q_heads, int32_t max_context,
                                               int32_t partition_tokens, size_t* bytes) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (!bytes) return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan);
    if (st != PA_OK) return st;
    *bytes = plan.ws_bytes;
    return PA_OK;
}

static pa_status decode_partial_impl(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                                     const int32_t* block_tables, int32_t max_blocks_per_seq,
                                     const int32_t* context_lens, int32_t num_seqs,
                                     int32_t max_context, int32_t window, float scale,
                                     int32_t partition_tokens, float* out, void* workspace,
                                     size_t workspace_bytes, int32_t* d_err, pa_stream_t stream) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq < 0 || max_context < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!q || !block_tables || !context_lens || !out) return PA_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / pool->num_kv_heads;
    const bool fp8 = pool->dtype == PA_DTYPE_FP8_E4M3;
    if (fp8) {  // bf16 queries against E4M3 rows of D = 128 with float row scales
        if (pool->head_dim != 128 || pool->block_size < 4) return PA_ERR_UNSUPPORTED;
        if (!aligned16(pool->k_scale) || !aligned16(pool->v_scale)) return PA_ERR_INVALID_ARG;
    } else if ((int64_t)pool->head_dim * dtype_bytes(pool->dtype) != kRowBytes) {
        return PA_ERR_UNSUPPORTED;
    }
    if (!is_pow2(pool->block_size)) return PA_ERR_UNSUPPORTED;
    if (pool->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned16(pool->k_pool) || !aligned16(pool->v_pool))
        return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan, window);
    if (st != PA_OK) return st;
    if (plan.max_parts > 65535) return PA_ERR_UNSUPPORTED;
    if (plan.ws_bytes > 0 && (workspace == nullptr || workspace_bytes < plan.ws_bytes ||
                              !aligned16(workspace)))
        return PA_ERR_INVALID_ARG;

    DecodeParams prm = {};
    prm.k_pool = static_cast<const unsigned char*>(pool->k_pool);
    prm.v_pool = static_cast<const unsigned char*>(pool->v_pool);
    prm.num_blocks = pool->num_blocks;
    prm.log2_bp = ilog2(pool->block_size);
    prm.num_kv_heads = pool->num_kv_heads;
    prm.q = q;
    prm.num_q_heads = num_q_heads;
    prm.block_tables = block_tables;
    prm.max_blocks = max_blocks_per_seq;
    prm.context_lens = context_lens;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.part_chunks = plan.part_chunks;
    prm.max_parts = plan.max_parts;
    prm.max_context = max_context;
    prm.window = window;
    prm.out = out;
    bind_workspace(plan, workspace, &prm);
    prm.d_err = d_err;
    prm.k_scale = fp8 ? static_cast<const float*>(pool->k_scale) : nullptr;
    prm.v_scale = fp8 ? static_cast<const float*>(pool->v_scale) : nullptr;
    cudaStream_t cs = (cudaStream_t)stream;
    if (use_mma(pool, num_q_heads)) {
        switch (G) {
            case 2: return launch_partial_mma<2>(pool, prm, num_seqs, plan.max_parts, cs);
            case 4: return launch_partial_mma<4>(pool, prm, num_seqs, plan.max_parts, cs);
            case 8: return launch_partial_mma<8>(pool, prm, num_seqs, plan.max_parts, cs);
            default: return PA_ERR_UNSUPPORTED;
        }
    }
    if (use_mma_fp8(pool, num_q_heads))
        return launch_partial_mma_fp8(pool, prm, num_seqs, pool->num_kv_heads, plan.max_parts, cs);
    if (fp8)
        return dispatch_group<uint8_t, false>(G, prm, num_seqs, pool->num_kv_heads, plan.max_parts, cs);
    if (pool->dtype == PA_DTYPE_F32)
        return dispatch_group<float, false>(G, prm, num_seqs, pool->num_kv_heads, plan.max_parts, cs);
    return dispatch_group<uint16_t, false>(G, prm, num_seqs, pool->num_kv_heads, plan.max_parts, cs);
}

static pa_status decode_merge_impl(const pa_kv_pool* pool, int32_t num_q_heads,
                                   const int32_t* context_lens, int32_t num_seqs,
                                   int32_t max_context, int32_t window, int32_t partition_tokens,
                                   float* out, void* workspace, size_t workspace_bytes,
                                   pa_stream_t stream, const int32_t* partner = nullptr,
                                   const int32_t* shared_lens = nullptr) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || max_context < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!context_lens || !out) return PA_ERR_INVALID_ARG;
    Plan plan;
    st = partner ? make_shared_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan)
                 : make_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan, window);
    if (st != PA_OK) return st;
    if (plan.max_parts <= 1) return PA_OK;
    if (workspace == nullptr || workspace_bytes < plan.ws_bytes || !aligned16(workspace))
        return PA_ERR_INVALID_ARG;
    DecodeParams prm = {};
    prm.num_q_heads = num_q_heads;
    prm.context_lens = context_lens;
    prm.part_chunks = plan.part_chunks;
    prm.max_parts = plan.max_parts;
    prm.max_context = max_context;
    prm.window = window;
    prm.out = out;
    bind_workspace(plan, workspace, &prm);
    prm.log2_bp = ilog2(pool->block_size);
    prm.partner = partner;
    prm.shared_lens = shared_lens;
    prm.num_seqs = num_seqs;
    const int D = pool->head_dim;
    // partials prefetched per thread: enough for every partition of the plan
    // with D/4 threads per partition group; few registers keep more CTAs resident
    const int groups = kMergeThreads / std::max(1, D / 4);
    auto kern = plan.max_parts <= 4 * groups ? decode_merge_kernel<4> : decode_merge_kernel<16>;
    cudaError_t e = launch_pdl(kern, dim3((unsigned)((int64_t)num_seqs * num_q_heads)),
                               dim3(kMergeThreads), 0, (cudaStream_t)stream, prm, D);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return launch_status();
}

extern "C" pa_status pa_decode_partial(const pa_kv_pool* pool, const void* q,
                                       int32_t num_q_heads, const int32_t* block_tables,
                                       int32_t max_blocks_per_seq, const int32_t* context_lens,
                                       int32_t num_seqs, int32_t max_context, float scale,
                                       int32_t partition_tokens, float* out, void* workspace,
                                       size_t workspace_bytes, int32_t* d_err,
                                       pa_stream_t stream) {
    return decode_partial_impl(pool, q, num_q_heads, block_tables, max_blocks_per_seq,
                               context_lens, num_seqs, max_context, 0, scale, partition_tokens,
                               out, workspace, workspace_bytes, d_err, stream);
}

extern "C" pa_status pa_decode_merge(const pa_kv_pool* pool, int32_t num_q_heads,
                                     const int32_t* context_lens, int32_t num_seqs,
                                     int32_t max_context, int32_t partition_tokens, float* out,
                                     void* workspace, size_t workspace_bytes,
                                     pa_stream_t stream) {
    return decode_merge_impl(pool, num_q_heads, context_lens, num_seqs, max_context, 0,
                             partition_tokens, out, workspace, workspace_bytes, stream);
}

extern "C" pa_status pa_decode(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                               const int32_t* block_tables, int32_t max_blocks_per_seq,
                               const int32_t* context_lens, int32_t num_seqs, int32_t max_context,
                               float scale, int32_t partition_tokens, float* out, void* workspace,
                               size_t workspace_bytes, int32_t* d_err, pa_stream_t stream) {
    pa_status st = pa_decode_partial(pool, q, num_q_heads, block_tables, max_blocks_per_seq,
                                     context_lens, num_seqs, max_context, scale, partition_tokens,
                                     out, workspace, workspace_bytes, d_err, stream);
    if (st != PA_OK) return st;
    return pa_decode_merge(pool, num_q_heads, context_lens, num_seqs, max_context,
                           partition_tokens, out, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- fused step
// Workspace of pa_decode_step: pa_decode's partials, then one int32 semaphore
// per (sequence, kv-head), 256-byte aligned.
static size_t step_sem_offset(const Plan& plan) { return align256(plan.ws_bytes); }

static size_t step_workspace_bytes(const Plan& plan, int32_t B, int32_t Hkv) {
    if (plan.max_parts <= 1) return 0;
    return step_sem_offset(plan) + (size_t)B * Hkv * 4;
}

extern "C" pa_status pa_decode_step_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                                    int32_t num_q_heads, int32_t max_context,
                                                    int32_t partition_tokens, size_t* bytes) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (!bytes) return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan);
    if (st != PA_OK) return st;
    *bytes = step_workspace_bytes(plan, num_seqs, pool->num_kv_heads);
    return PA_OK;
}

extern "C" pa_status pa_decode_step(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                                    const int64_t* slot_mapping, const void* q,
                                    int32_t num_q_heads, const int32_t* block_tables,
                                    int32_t max_blocks_per_seq, const int32_t* context_lens,
                                    int32_t num_seqs, int32_t max_context, float scale,
                                    int32_t partition_tokens, float* out, void* workspace,
                                    size_t workspace_bytes, int32_t* d_err, pa_stream_t stream) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq < 0 || max_context < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!q || !block_tables || !context_lens || !out || !k_new || !v_new || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / pool->num_kv_heads;
    if (pool->dtype == PA_DTYPE_FP8_E4M3) return PA_ERR_UNSUPPORTED;  // the step writes raw rows
    if ((int64_t)pool->head_dim * dtype_bytes(pool->dtype) != kRowBytes) return PA_ERR_UNSUPPORTED;
    if (!is_pow2(pool->block_size)) return PA_ERR_UNSUPPORTED;
    if (pool->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned16(pool->k_pool) || !aligned16(pool->v_pool) ||
        !aligned16(k_new) || !aligned16(v_new))
        return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan);
    if (st != PA_OK) return st;
    if (plan.max_parts > 65535) return PA_ERR_UNSUPPORTED;
    const size_t need = step_workspace_bytes(plan, num_seqs, pool->num_kv_heads);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !aligned16(workspace)))
        return PA_ERR_INVALID_ARG;

    DecodeParams prm = {};
    prm.k_pool = static_cast<const unsigned char*>(pool->k_pool);
    prm.v_pool = static_cast<const unsigned char*>(pool->v_pool);
    prm.num_blocks = pool->num_blocks;
    prm.log2_bp = ilog2(pool->block_size);
    prm.num_kv_heads = pool->num_kv_heads;
    prm.q = q;
    prm.num_q_heads = num_q_heads;
    prm.block_tables = block_tables;
    prm.max_blocks = max_blocks_per_seq;
    prm.context_lens = context_lens;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.part_chunks = plan.part_chunks;
    prm.max_parts = plan.max_parts;
    prm.max_context = max_context;
    prm.out = out;
    bind_workspace(plan, workspace, &prm);
    prm.d_err = d_err;
    prm.k_new = static_cast<const unsigned char*>(k_new);
    prm.v_new = static_cast<const unsigned char*>(v_new);
    prm.slot_mapping = slot_mapping;
    prm.sem = need > 0 ? reinterpret_cast<int32_t*>(static_cast<unsigned char*>(workspace) +
                                                    step_sem_offset(plan))
                       : nullptr;
    cudaStream_t cs = (cudaStream_t)stream;
    if (use_mma(pool, num_q_heads)) {
        switch (G) {
            case 2: return launch_partial_mma<2, true>(pool, prm, num_seqs, plan.max_parts, cs);
            case 4: return launch_partial_mma<4, true>(pool, prm, num_seqs, plan.max_parts, cs);
            case 8: return launch_partial_mma<8, true>(pool, prm, num_seqs, plan.max_parts, cs);
            default: return PA_ERR_UNSUPPORTED;
        }
    }
    if (pool->dtype == PA_DTYPE_F32)
        return dispatch_group<float, true>(G, prm, num_seqs, pool->num_kv_heads, plan.max_parts, cs);
    return dispatch_group<uint16_t, true>(G, prm, num_seqs, pool->num_kv_heads, plan.max_parts, cs);
}

// ---------------------------------------------------------------- sliding window
extern "C" pa_status pa_decode_window_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                                      int32_t num_q_heads, int32_t max_context,
                                                      int32_t window, int32_t partition_tokens,
                                                      size_t* bytes) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (!bytes || window <= 0) return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan, window);
    if (st != PA_OK) return st;
    *bytes = plan.ws_bytes;
    return PA_OK;
}

extern "C" pa_status pa_decode_window(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t max_context, int32_t window, float scale,
                                      int32_t partition_tokens, float* out, void* workspace,
                                      size_t workspace_bytes, int32_t* d_err, pa_stream_t stream) {
    if (window <= 0) return PA_ERR_INVALID_ARG;
    pa_status st = decode_partial_impl(pool, q, num_q_heads, block_tables, max_blocks_per_seq,
                                       context_lens, num_seqs, max_context, window, scale,
                                       partition_tokens, out, workspace, workspace_bytes, d_err,
                                       stream);
    if (st != PA_OK) return st;
    return decode_merge_impl(pool, num_q_heads, context_lens, num_seqs, max_context, window,
                             partition_tokens, out, workspace, workspace_bytes, stream);
}

// ---------------------------------------------------------------- shared prefixes
static bool shared_supported(const pa_kv_pool* pool, int32_t Hq) {
    const int G = Hq / pool->num_kv_heads;
    return pool->dtype == PA_DTYPE_BF16 && pool->head_dim == mma::kD && pool->block_size >= 16 &&
           is_pow2(pool->block_size) &&
           (int64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size <= INT32_MAX &&
           (G == 1 || G == 2 || G == 4 || G == 8);
}

extern "C" pa_status pa_decode_shared_workspace_bytes(const pa_kv_pool* pool, int32_t num_seqs,
                                                      int32_t num_q_heads, int32_t max_context,
                                                      int32_t partition_tokens, size_t* bytes) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (!bytes) return PA_ERR_INVALID_ARG;
    Plan plan;
    st = make_shared_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan);
    if (st != PA_OK) return st;
    *bytes = plan.ws_bytes;
    return PA_OK;
}

extern "C" pa_status pa_decode_shared(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                                      const int32_t* block_tables, int32_t max_blocks_per_seq,
                                      const int32_t* context_lens, int32_t num_seqs,
                                      int32_t max_context, const int32_t* partner,
                                      const int32_t* shared_lens, float scale,
                                      int32_t partition_tokens, float* out, void* workspace,
                                      size_t workspace_bytes, int32_t* d_err, pa_stream_t stream) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || num_q_heads <= 0 || max_blocks_per_seq < 0 || max_context < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!q || !block_tables || !context_lens || !out || !partner || !shared_lens)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    if (!shared_supported(pool, num_q_heads)) return PA_ERR_UNSUPPORTED;
    if (pool->num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned16(pool->k_pool) || !aligned16(pool->v_pool))
        return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / pool->num_kv_heads;
    Plan plan;
    st = make_shared_plan(pool, num_seqs, num_q_heads, max_context, partition_tokens, &plan);
    if (st != PA_OK) return st;
    if (plan.max_parts > 65535) return PA_ERR_UNSUPPORTED;
    if (workspace == nullptr || workspace_bytes < plan.ws_bytes || !aligned16(workspace))
        return PA_ERR_INVALID_ARG;
    DecodeParams prm = {};
    prm.k_pool = static_cast<const unsigned char*>(pool->k_pool);
    prm.v_pool = static_cast<const unsigned char*>(pool->v_pool);
    prm.num_blocks = pool->num_blocks;
    prm.log2_bp = ilog2(pool->block_size);
    prm.num_kv_heads = pool->num_kv_heads;
    prm.q = q;
    prm.num_q_heads = num_q_heads;
    prm.block_tables = block_tables;
    prm.max_blocks = max_blocks_per_seq;
    prm.context_lens = context_lens;
    prm.scale_log2 = scale * 1.4426950408889634f;
    prm.part_chunks = plan.part_chunks;
    prm.max_parts = plan.max_parts;
    prm.max_context = max_context;
    prm.out = out;
    bind_workspace(plan, workspace, &prm);
    prm.d_err = d_err;
    prm.partner = partner;
    prm.shared_lens = shared_lens;
    prm.num_seqs = num_seqs;
    cudaStream_t cs = (cudaStream_t)stream;
    switch (G) {
        case 1: st = launch_shared_mma<1>(pool, prm, num_seqs, plan.max_parts, cs); break;
        case 2: st = launch_shared_mma<2>(pool, prm, num_seqs, plan.max_parts, cs); break;
        case 4: st = launch_shared_mma<4>(pool, prm, num_seqs, plan.max_parts, cs); break;
        case 8: st = launch_shared_mma<8>(pool, prm, num_seqs, plan.max_parts, cs); break;
        default: return PA_ERR_UNSUPPORTED;
    }
    if (st != PA_OK) return st;
    return decode_merge_impl(pool, num_q_heads, context_lens, num_seqs, max_context, 0,
                             partition_tokens, out, workspace, workspace_bytes, stream, partner,
                             shared_lens);
}
