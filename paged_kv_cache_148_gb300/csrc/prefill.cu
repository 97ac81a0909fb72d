// pa_prefill: paged chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators and P in TMEM, operands staged by TMA).
//
// Semantics: "03｜PagedAttention 与 KV Cache 内存系统" §4 — prefill reuses a
// flash-style tiled attention kernel that is handed the paged block table
// (paging decides where K/V live, tiling decides how one attention pass moves
// through them).  New token i of a sequence sits at position
// context_len - n_new + i and, with a causal mask, sees positions 0..itself.
//
// CTA = (pair of q-tiles, kv-head, sequence).  A q-tile is 128 rows =
// (128/G) queries x the G query heads that share one kv-head; the CTA runs
// two consecutive q-tiles (A, B) against every K/V tile it stages, so each
// staged byte feeds 256 rows.  Key tiles are 128 keys = 128/B_p pages, each
// page half (64 dims) fetched by one tiled TMA load straight from the pool
// through the block table.
//
// Roles (320 threads, one CTA per SM):
//   warp 0      TMA producer: both Q tiles once; K tiles into a 2-stage ring
//               (a stage frees when the S MMAs of both q-tiles complete) and
//               V tiles into a 3-stage ring (freed when both P*V MMAs
//               complete).  Lane k handles page k of a tile.
//   warp 1      MMA issuer (the whole warp; elect.sync picks the lane that
//               issues each MMA): S_X = Q_X K_j^T into TMEM, then
//               O_X += P_X V_j with P_X read from TMEM, alternating A and B so
//               one q-tile's softmax overlaps the other's MMAs.
//   warps 2-5   softmax of q-tile A, warps 6-9 softmax of q-tile B: thread r
//               owns row r (TMEM lane r): two passes over S_j in TMEM (row max,
//               then exponentials), base-2 online softmax with lazy rescaling
//               of O (only when the row max grows by more than 2^8), P_j
//               written as fp16 pairs into TMEM over the S columns already
//               read, and finally O / l to global memory.
//               Between tiles the softmax warps of one q-tile also turn the
//               next V tile from bf16 into fp16 in place (thread r converts
//               row r; rows past the written keys become zeros): after
//               publishing P_X(j) they wait ~half a tile for S_X(j+1), and the
//               conversion fills that wait on all four SM sub-partitions.  V
//               tiles alternate between the two q-tiles (the one that still
//               has tiles takes them all).
// Q K^T runs on bf16 operands; P V runs on fp16 operands: P in [0, 2^8]
// keeps 11 significant bits in fp16 against 8 in bf16, which the stated
// accuracy needs (bf16 P alone leaves ~1.6e-3 relative L2 error at 2.5K
// keys).  bf16 -> fp16 is exact for |v| <= 65504 (the fp16 range) apart from
// fp16 subnormals below 2^-14, whose absolute error stays under 2^-25.  Larger
// magnitudes saturate to +-65504; the threads that convert V track the
// largest |v| they convert and store PA_ERR_UNSUPPORTED in *d_err when one
// was out of range, so such a result never passes silently.
// All mbarrier waits are bounded; a wait that runs out sets PA_ERR_TIMEOUT
// and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "tcgen05.cuh"

namespace pa {

constexpr int kPfRows = 128;            // M: rows of a q-tile (queries x heads)
constexpr int kPfKeys = 128;            // N: keys per KV tile
constexpr int kPfDim = 128;             // head_dim
constexpr int kHalf = 128 * 128;        // bytes of one 64-column half of a 128-row 16-bit tile
constexpr int kTile = 2 * kHalf;        // 32 KiB
constexpr int kPfThreads = 320;
constexpr uint32_t kTmemCols = 512;     // S_A | S_B | O_A | O_B
constexpr float kPfRescale = 8.0f;

// shared-memory map (offsets from a 1024-aligned base)
constexpr int kKStages = 2;
constexpr int kVStages = 3;
constexpr int kOffQ = 0;                             // Q_A, Q_B
constexpr int kOffK = 2 * kTile;                     // kKStages stages
constexpr int kOffV = kOffK + kKStages * kTile;      // kVStages stages
constexpr int kOffBar = kOffV + kVStages * kTile;
constexpr int kPfSmem = kOffBar + 1024 + 1024;       // + barriers and page ids, + alignment slack

struct PrefillParams {
    const int32_t* cu_seqlens_q;
    const int32_t* context_lens;
    const int32_t* block_tables;
    int32_t max_blocks;
    int32_t num_blocks;
    int32_t num_kv_heads;
    int32_t num_q_heads;
    int32_t log2_bp;
    int32_t causal;
    float scale_log2;
    int32_t max_qtiles;
    float* out;
    int32_t* d_err;
};

struct PfBars {
    uint64_t q_full;
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages];
    uint64_t v_empty[kVStages];
    uint64_t v_ready[kVStages];     // V converted to fp16 (one q-tile's 128 softmax threads)
    uint64_t s_full[2];             // per q-tile: S_j in TMEM
    uint64_t p_full[2][2];          // per q-tile and half of the keys: P_j in TMEM (128 threads)
    uint64_t o_done[2];             // per q-tile: P_j V_j accumulated into O
    uint32_t tmem_base;
    int32_t abort;
};

PA_DEVICE void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
}

PA_DEVICE uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// two floats -> fp16 pair (lo in the low half)
PA_DEVICE uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// running magnitude maximum of bf16 pairs: |result| = max(|a|, |b|) per half
// (the sign bits are not used)
PA_DEVICE uint32_t bf16x2_absmax(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.xorsign.abs.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// bf16 pair -> fp16 pair (round to nearest even, saturating at the fp16 range)
PA_DEVICE uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r) : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}

PA_DEVICE float fmax3(float a, float b, float c) {
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

PA_DEVICE void tmem_ld16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

PA_DEVICE void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
          "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
          "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}

// bounded wait that also honours a CTA-wide abort flag
PA_DEVICE bool pf_wait(uint64_t* bar, uint32_t parity, PfBars* b, int32_t* d_err) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    uint32_t spins = 0;
    while (!mbar_try_wait(bar, parity)) {
        if ((++spins & 255u) == 0) {
            if (*(volatile int32_t*)&b->abort) return false;
            if (global_timer_ns() - t0 > kWaitLimitNs) {
                set_error(d_err, PA_ERR_TIMEOUT);
                *(volatile int32_t*)&b->abort = 1;
                return false;
            }
        }
    }
    return true;
}

// A warp-uniform bounded wait (all lanes wait; the result is agreed by vote).
PA_DEVICE bool pf_wait_warp(uint64_t* bar, uint32_t parity, PfBars* b, int32_t* d_err) {
    const bool ok = pf_wait(bar, parity, b, d_err);
    return __all_sync(0xffffffffu, ok);
}

template <int G>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    constexpr int QT = kPfRows / G;  // queries per q-tile
    const int n_pairs = (p.max_qtiles + 1) / 2;
    const int qp = n_pairs - 1 - (int)blockIdx.x;  // longest tiles first
    const int h = blockIdx.y, s = blockIdx.z;
    const int q_begin = __ldg(p.cu_seqlens_q + s);
    const int n_new = __ldg(p.cu_seqlens_q + s + 1) - q_begin;
    const int q0 = 2 * qp * QT;  // first query of q-tile A; q-tile B starts at q0 + QT
    if (n_new <= 0 || q0 >= n_new) {
        if (qp == 0 && h == 0 && threadIdx.x == 0 && n_new > p.max_qtiles * QT)
            set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int ctx = __ldg(p.context_lens + s);
    const int base_pos = ctx - n_new;  // position of new token 0
    if (base_pos < 0) {
        if (threadIdx.x == 0) set_error(p.d_err, PA_ERR_INVALID_ARG);
        return;
    }
    const bool has_b = q0 + QT < n_new;
    // keys each q-tile needs: [0, kv_end_X)
    const int last_a = min(q0 + QT, n_new) - 1, last_b = min(q0 + 2 * QT, n_new) - 1;
    const int kv_end_a = p.causal ? base_pos + last_a + 1 : ctx;
    const int kv_end_b = has_b ? (p.causal ? base_pos + last_b + 1 : ctx) : 0;
    const int kv_end = max(kv_end_a, kv_end_b);
    const int nt_a = (kv_end_a + kPfKeys - 1) / kPfKeys;
    const int nt_b = (kv_end_b + kPfKeys - 1) / kPfKeys;
    const int n_tiles = max(nt_a, nt_b);
    const int bp = 1 << p.log2_bp;
    const int pages_per_tile = kPfKeys >> p.log2_bp;
    // keys at or past `zlim` may be unwritten or not loaded: V rows there are zeroed
    const int zlim = min(ctx, ((kv_end + bp - 1) >> p.log2_bp) << p.log2_bp);

    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    PfBars* bars = reinterpret_cast<PfBars*>(smem + kOffBar);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        mbar_init(&bars->q_full, 1);
        for (int i = 0; i < kKStages; ++i) {
            mbar_init(&bars->k_full[i], 1);
            mbar_init(&bars->k_empty[i], 1);
        }
        for (int i = 0; i < kVStages; ++i) {
            mbar_init(&bars->v_full[i], 1);
            mbar_init(&bars->v_empty[i], 1);
            mbar_init(&bars->v_ready[i], 128);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->p_full[i][0], 128);
            mbar_init(&bars->p_full[i][1], 128);
            mbar_init(&bars->o_done[i], 1);
        }
        bars->abort = 0;
        fence_mbar_init();
    }
    if (warp == 1) {
        tc::tmem_alloc(&bars->tmem_base, kTmemCols);
        tc::tmem_relinquish();
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = bars->tmem_base;
    // per q-tile X: S_X at columns [128 X, 128 X + 128); P_X (fp16 pairs) over its
    // first 64 columns; O_X at [256 + 128 X, 256 + 128 X + 128)
    auto tS = [&](int x) { return tmem + 128u * x; };
    auto tO = [&](int x) { return tmem + 256u + 128u * x; };

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks;
        // this lane's page of tile j: the table read is issued one tile ahead
        // (fetch_id) and checked only when the tile is loaded (tile_row), so the
        // warp never stalls on it
        auto lane_page = [&](int j) {
            const int e = j * pages_per_tile + lane;
            return (lane < pages_per_tile && (e << p.log2_bp) < kv_end) ? e : -1;
        };
        auto fetch_id = [&](int j) -> int32_t {
            const int e = lane_page(j);
            return (e >= 0 && e < p.max_blocks) ? __ldg(table + e) : -1;
        };
        auto tile_row = [&](int j, int32_t id) -> int32_t {
            if (lane_page(j) < 0) return -1;
            if (id < 0 || id >= p.num_blocks) {
                set_error(p.d_err, id < 0 ? PA_ERR_NEGATIVE_BLOCK : PA_ERR_OUT_OF_RANGE);
                id = 0;  // stay in bounds; the result is flagged as invalid
            }
            return (id * p.num_kv_heads + h) << p.log2_bp;
        };
        auto loaded_pages = [&](int j) {
            const int rem = kv_end - j * kPfKeys;
            return min(pages_per_tile, (rem + bp - 1) >> p.log2_bp);
        };
        if (lane == 0) {
            tc::prefetch_tmap(&tmap_q);
            tc::prefetch_tmap(&tmap_k);
            tc::prefetch_tmap(&tmap_v);
            mbar_arrive_expect_tx(&bars->q_full, has_b ? 2 * kTile : kTile);
            tc::tma_load_3d(smem + kOffQ, &tmap_q, 0, h * G, q_begin + q0, &bars->q_full);
            tc::tma_load_3d(smem + kOffQ + kHalf, &tmap_q, 64, h * G, q_begin + q0, &bars->q_full);
            if (has_b) {
                tc::tma_load_3d(smem + kOffQ + kTile, &tmap_q, 0, h * G, q_begin + q0 + QT,
                                &bars->q_full);
                tc::tma_load_3d(smem + kOffQ + kTile + kHalf, &tmap_q, 64, h * G,
                                q_begin + q0 + QT, &bars->q_full);
            }
        }
        // K_j then V_j for every tile, each as soon as its stage is released: K_j
        // once Q K_{j-2}^T has completed, V_j once P V_{j-3} has.  Both releases
        // come from the same MMA commit point, so blocking on them in this order
        // never holds back a load that could already go.
        int32_t next_id = fetch_id(0);  // prefetched table entry of tile j
        for (int j = 0; j < n_tiles; ++j) {
            if (j >= kKStages &&
                !pf_wait_warp(&bars->k_empty[j % kKStages], ((j / kKStages) - 1) & 1, bars, p.d_err))
                break;
            const int row = tile_row(j, next_id);
            if (j + 1 < n_tiles) next_id = fetch_id(j + 1);
            const int loaded = loaded_pages(j);
            const uint32_t bytes = (uint32_t)loaded * bp * 128 * 2;
            uint64_t* kbar = &bars->k_full[j % kKStages];
            if (lane == 0) mbar_arrive_expect_tx(kbar, bytes);
            __syncwarp();
            if (lane < loaded) {
                unsigned char* dst = smem + kOffK + (j % kKStages) * kTile + lane * bp * 128;
                tc::tma_load_2d(dst, &tmap_k, 0, row, kbar);
                tc::tma_load_2d(dst + kHalf, &tmap_k, 64, row, kbar);
            }
            if (j >= kVStages &&
                !pf_wait_warp(&bars->v_empty[j % kVStages], ((j / kVStages) - 1) & 1, bars, p.d_err))
                break;
            uint64_t* vbar = &bars->v_full[j % kVStages];
            if (lane == 0) mbar_arrive_expect_tx(vbar, bytes);
            __syncwarp();
            if (lane < loaded) {
                unsigned char* dst = smem + kOffV + (j % kVStages) * kTile + lane * bp * 128;
                tc::tma_load_2d(dst, &tmap_v, 0, row, vbar);
                tc::tma_load_2d(dst + kHalf, &tmap_v, 64, row, vbar);
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // The whole warp runs the issue loop (waits are warp-wide votes) and one
        // elected lane issues each tcgen05 instruction.
        constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, 128, 0, 0);
        constexpr uint32_t idesc_pv = tc::idesc_f16_f32(128, 128, 0, 1);
        const uint32_t q_addr = smem_u32(smem + kOffQ);
        const int nt[2] = {nt_a, nt_b};
        bool ok = pf_wait_warp(&bars->q_full, 0, bars, p.d_err);
        // Shared-memory descriptors are built once; an MMA step only adds the
        // byte offset (>> 4) of its sub-tile to the start-address field.
        const uint64_t dq = tc::smem_desc_sw128(q_addr, 16, 1024);
        const uint64_t dk = tc::smem_desc_sw128(smem_u32(smem + kOffK), 16, 1024);
        const uint64_t dv = tc::smem_desc_sw128(smem_u32(smem + kOffV), kHalf, 1024);
        // S_X(j) = Q_X K_j^T
        auto qk = [&](int x, int j) {
            const uint64_t a0 = dq + (uint64_t)((x * kTile) >> 4);
            const uint64_t b0 = dk + (uint64_t)(((j % kKStages) * kTile) >> 4);
            const uint32_t d = tS(x);
#pragma unroll
            for (int kk = 0; kk < 8; ++kk) {
                const uint64_t koff = (uint64_t)(((kk >> 2) * kHalf + (kk & 3) * 32) >> 4);
                tc::mma_ss_warp(d, a0 + koff, b0 + koff, idesc_qk, kk > 0 ? 1u : 0u);
            }
            tc::commit_warp(&bars->s_full[x]);
        };
        // O_X += P_X(j) V_j, P_X in TMEM (8 columns of fp16 pairs per 16 keys);
        // the softmax publishes P in two halves of 64 keys
        auto pv = [&](int x, int j) -> bool {
            const uint64_t b0 = dv + (uint64_t)(((j % kVStages) * kTile) >> 4);
            const uint32_t d = tO(x), a = tS(x);
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                if (!pf_wait_warp(&bars->p_full[x][hf], j & 1, bars, p.d_err)) return false;
                tc::fence_after_sync();
#pragma unroll
                for (int kk = 4 * hf; kk < 4 * hf + 4; ++kk)
                    tc::mma_ts_warp(d, a + kk * 8, b0 + (uint64_t)((kk * 2048) >> 4), idesc_pv,
                                    (j > 0 || kk > 0) ? 1u : 0u);
            }
            tc::commit_warp(&bars->o_done[x]);
            return true;
        };
        if (ok) ok = pf_wait_warp(&bars->k_full[0], 0, bars, p.d_err);
        if (ok) {
            tc::fence_after_sync();
            for (int x = 0; x < 2; ++x)
                if (nt[x] > 0) qk(x, 0);
            tc::commit_warp(&bars->k_empty[0]);
        }
        for (int j = 0; ok && j < n_tiles; ++j) {
            const bool more = j + 1 < n_tiles;
            bool k_next = false;
            if (!pf_wait_warp(&bars->v_ready[j % kVStages], (j / kVStages) & 1, bars, p.d_err)) {
                ok = false;
                break;
            }
            for (int x = 0; x < 2; ++x) {
                if (j >= nt[x]) continue;
                // P_X(j) published by its softmax (which read S_X(j) first)
                if (!pv(x, j)) { ok = false; break; }
                if (j + 1 < nt[x]) {
                    if (!k_next) {
                        if (!pf_wait_warp(&bars->k_full[(j + 1) % kKStages],
                                          ((j + 1) / kKStages) & 1, bars, p.d_err)) {
                            ok = false;
                            break;
                        }
                        tc::fence_after_sync();
                        k_next = true;
                    }
                    qk(x, j + 1);  // overwrites P_X(j) after the P*V above consumed it
                }
            }
            if (!ok) break;
            tc::commit_warp(&bars->v_empty[j % kVStages]);
            if (more) {
                if (!k_next) {  // neither q-tile uses K_{j+1}: still release its stage
                    if (!pf_wait_warp(&bars->k_full[(j + 1) % kKStages], ((j + 1) / kKStages) & 1,
                                      bars, p.d_err)) { ok = false; break; }
                }
                tc::commit_warp(&bars->k_empty[(j + 1) % kKStages]);
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int x = warp >= 6 ? 1 : 0;           // q-tile A or B
        const int nt_x = x ? nt_b : nt_a;
        // V_jv is converted by a q-tile that runs tile jv - 1 (tile 0: by A):
        // A for even jv, B for odd jv, or whichever of them still has tiles
        auto v_owner = [&](int jv) -> int {
            const bool a_has = jv == 0 ? nt_a > 0 : jv - 1 < nt_a;
            const bool b_has = jv == 0 ? false : jv - 1 < nt_b;
            return (a_has && ((jv & 1) == 0 || !b_has)) ? 0 : 1;
        };
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;         // tile row == TMEM lane
        const int i = r / G, g = r - i * G;
        const int qi = q0 + x * QT + i;
        const bool live = qi < n_new;
        int lim = p.causal ? base_pos + qi : ctx - 1;  // last visible key
        if (!live) lim = 0;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t sX = tS(x) + lane_addr, oX = tO(x) + lane_addr;
        const float sc = p.scale_log2;
        float m_used = -INFINITY, l = 0.f;  // m_used in scaled base-2 units
        uint32_t vmax = 0;  // largest |V| this thread converted, as a bf16 pair
        // row r of V tile jv from bf16 to fp16 in place (zeros past the
        // written keys), then this thread's arrival on v_ready
        auto convert_v = [&](int jv) -> bool {
            if (!pf_wait_warp(&bars->v_full[jv % kVStages], (jv / kVStages) & 1, bars, p.d_err))
                return false;
            const uint32_t vrow = smem_u32(smem + kOffV + (jv % kVStages) * kTile) + r * 128;
            if (jv * kPfKeys + r < zlim) {
                // chunk order rotated by the row: the 8 threads of a 128-bit phase
                // hit 8 different bank groups; eight loads go out before the
                // first store so their latencies overlap
#pragma unroll
                for (int hb = 0; hb < 2; ++hb) {
                    uint4 xv[8];
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        xv[c] = ld_shared_v4(vrow + hb * kHalf + ((c + r) & 7) * 16);
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        vmax = bf16x2_absmax(vmax, bf16x2_absmax(bf16x2_absmax(xv[c].x, xv[c].y),
                                                                 bf16x2_absmax(xv[c].z, xv[c].w)));
#pragma unroll
                    for (int c = 0; c < 8; ++c)
                        st_shared_v4(vrow + hb * kHalf + ((c + r) & 7) * 16,
                                     bf16x2_to_f16x2(xv[c].x), bf16x2_to_f16x2(xv[c].y),
                                     bf16x2_to_f16x2(xv[c].z), bf16x2_to_f16x2(xv[c].w));
                }
            } else {
#pragma unroll
                for (int c = 0; c < 16; ++c)
                    st_shared_v4(vrow + (c >> 3) * kHalf + ((c + r) & 7) * 16, 0, 0, 0, 0);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->v_ready[jv % kVStages]);
            return true;
        };
        bool ok = true;
        if (n_tiles > 0 && v_owner(0) == x) ok = convert_v(0);
        for (int j = 0; ok && j < nt_x; ++j) {
            if (!pf_wait_warp(&bars->s_full[x], j & 1, bars, p.d_err)) { ok = false; break; }
            tc::fence_after_sync();
            const int key0 = j * kPfKeys;
            const bool full = key0 + kPfKeys - 1 <= lim;
            // the whole S row with one TMEM wait
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::tmem_ld32(sX + c * 32, sr[c]);
            tc::tmem_wait_ld();
            if (!full) {
#pragma unroll
                for (int c = 0; c < 4; ++c)
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                        if (key0 + c * 32 + e > lim) sr[c][e] = __float_as_uint(-INFINITY);
            }
            // row max as 8 independent chains (the 128 values are all in registers)
            float mx[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) mx[q] = -INFINITY;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const int q = ((c * 32 + e) >> 1) & 7;
                    mx[q] = fmax3(mx[q], __uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1]));
                }
            const float tmax = fmaxf(fmax3(mx[0], mx[1], mx[2]), fmax3(mx[3], mx[4], fmax3(mx[5], mx[6], mx[7])));
            const float tmax_s = tmax * sc;
            if (j == 0) {
                m_used = tmax_s;
            } else {
                // rescale O and l only when the row max grew by more than 2^8
                const bool need = tmax_s > m_used + kPfRescale;
                if (__any_sync(0xffffffffu, need)) {
                    if (!pf_wait_warp(&bars->o_done[x], (j - 1) & 1, bars, p.d_err)) { ok = false; break; }
                    tc::fence_after_sync();
                    const float m_new = need ? tmax_s : m_used;
                    const float f = ex2(m_used - m_new);
#pragma unroll 1
                    for (int c = 0; c < 8; ++c) {  // 16 columns at a time: S is still live
                        uint32_t o[16];
                        tmem_ld16(oX + c * 16, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 16; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tmem_st16(oX + c * 16, o);
                    }
                    tc::tmem_wait_st();
                    l *= f;
                    m_used = m_new;
                }
            }
            // P = 2^(s*scale - m) as fp16 pairs over the S columns already read;
            // each half of 64 keys is published as soon as it is stored
            const float2 sc2 = make_float2(sc, sc), negm2 = make_float2(-m_used, -m_used);
            float2 ls[2] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f)};  // partial row sums
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t pk[16];
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float2 xx = __ffma2_rn(
                        make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sc2,
                        negm2);
                    const float2 pp = make_float2(ex2(xx.x), ex2(xx.y));
                    ls[(e >> 1) & 1] = __fadd2_rn(ls[(e >> 1) & 1], pp);
                    pk[e >> 1] = pack_f16(pp.x, pp.y);
                }
                tmem_st16(sX + c * 16, pk);
                if (c & 1) {
                    tc::tmem_wait_st();
                    tc::fence_before_sync();
                    mbar_arrive(&bars->p_full[x][c >> 1]);
                }
            }
            l += (ls[0].x + ls[1].x) + (ls[0].y + ls[1].y);
            // the wait for S_X(j+1) is this q-tile's share of the V conversion
            if (j + 1 < n_tiles && v_owner(j + 1) == x && !convert_v(j + 1)) { ok = false; break; }
        }
        // a V element beyond the fp16 range (|v| >= 65536, the first bf16 magnitude
        // above 65504, or an infinity) was saturated by the conversion: the result
        // is not the attention over the stored values, so say so
        if ((vmax & 0x7fffu) >= 0x4780u || ((vmax >> 16) & 0x7fffu) >= 0x4780u)
            set_error(p.d_err, PA_ERR_UNSUPPORTED);
        // epilogue: O / l -> out
        if (ok && nt_x > 0) ok = pf_wait_warp(&bars->o_done[x], (nt_x - 1) & 1, bars, p.d_err);
        if (ok && nt_x > 0) {
            tc::fence_after_sync();
            const float inv = live ? 1.f / l : 0.f;
            float* orow = p.out + ((int64_t)(q_begin + qi) * p.num_q_heads + h * G + g) * kPfDim;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tc::tmem_ld32(oX + c * 32, o);
                tc::tmem_wait_ld();
                if (live) {
#pragma unroll
                    for (int e = 0; e < 32; e += 4)
                        *reinterpret_cast<float4*>(orow + c * 32 + e) =
                            make_float4(__uint_as_float(o[e]) * inv, __uint_as_float(o[e + 1]) * inv,
                                        __uint_as_float(o[e + 2]) * inv,
                                        __uint_as_float(o[e + 3]) * inv);
                }
            }
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side
static bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box) {
    uint64_t d[3], st[2];
    uint32_t bx[3];
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        if (i > 0) st[i - 1] = strides[i - 1];
    }
    return encode_bf16_map_sw128(m, base, rank, d, st, bx);
}

template <int G>
static pa_status launch_prefill(const pa_kv_pool* pool, const void* q, int32_t total_q,
                                int32_t Hq, int32_t B, const PrefillParams& prm,
                                cudaStream_t stream) {
    constexpr int QT = kPfRows / G;
    CUtensorMap mq, mk, mv;
    const cuuint64_t qdims[3] = {(cuuint64_t)kPfDim, (cuuint64_t)Hq, (cuuint64_t)total_q};
    const cuuint64_t qstr[2] = {(cuuint64_t)kPfDim * 2, (cuuint64_t)Hq * kPfDim * 2};
    const cuuint32_t qbox[3] = {64, (cuuint32_t)G, (cuuint32_t)QT};
    const cuuint64_t rows = (cuuint64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size;
    const cuuint64_t kdims[2] = {(cuuint64_t)kPfDim, rows};
    const cuuint64_t kstr[1] = {(cuuint64_t)kPfDim * 2};
    const cuuint32_t kbox[2] = {64, (cuuint32_t)pool->block_size};
    if (!make_map(&mq, q, 3, qdims, qstr, qbox) || !make_map(&mk, pool->k_pool, 2, kdims, kstr, kbox) ||
        !make_map(&mv, pool->v_pool, 2, kdims, kstr, kbox))
        return PA_ERR_CUDA;
    auto kern = prefill_kernel<G>;
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64 || !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPfSmem);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        if (dev >= 0 && dev < 64) attr_done[dev] = true;
    }
    dim3 grid((unsigned)((prm.max_qtiles + 1) / 2), (unsigned)pool->num_kv_heads, (unsigned)B);
    kern<<<grid, kPfThreads, kPfSmem, stream>>>(mq, mk, mv, prm);
    return launch_status();
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_prefill(const pa_kv_pool* pool, const void* q, int32_t total_q,
                                int32_t num_q_heads, const int32_t* cu_seqlens_q,
                                const int32_t* context_lens, const int32_t* block_tables,
                                int32_t max_blocks_per_seq, int32_t num_seqs, int32_t max_q_len,
                                int32_t max_context, float scale, int32_t causal, float* out,
                                int32_t* d_err, pa_stream_t stream) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (num_seqs < 0 || total_q < 0 || num_q_heads <= 0 || max_q_len < 0 || max_context < 0 ||
        max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || total_q == 0 || max_q_len == 0) return PA_OK;
    if (!q || !cu_seqlens_q || !context_lens || !block_tables || !out) return PA_ERR_INVALID_ARG;
    if (num_q_heads % pool->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;
    const int G = num_q_heads / pool->num_kv_heads;
    if (pool->dtype != PA_DTYPE_BF16 || pool->head_dim != kPfDim) return PA_ERR_UNSUPPORTED;
    if (!is_pow2(pool->block_size) || pool->block_size < 8 || pool->block_size > 128)
        return PA_ERR_UNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    if (pool->num_kv_heads > 65535 || num_seqs > 65535) return PA_ERR_UNSUPPORTED;
    if ((int64_t)pool->num_blocks * pool->num_kv_heads * pool->block_size > INT32_MAX)
        return PA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(out) || !aligned16(pool->k_pool) || !aligned16(pool->v_pool))
        return PA_ERR_INVALID_ARG;
    PrefillParams prm;
    prm.cu_seqlens_q = cu_seqlens_q;
    prm.context_lens = context_lens;
    prm.block_tables = block_tables;
    prm.max_blocks = max_blocks_per_seq;
    prm.num_blocks = pool->num_blocks;
    prm.num_kv_heads = pool->num_kv_heads;
    prm.num_q_heads = num_q_heads;
    prm.log2_bp = ilog2(pool->block_size);
    prm.causal = causal ? 1 : 0;
    prm.scale_log2 = scale * 1.4426950408889634f;
    const int QT = kPfRows / G;
    prm.max_qtiles = (max_q_len + QT - 1) / QT;
    prm.out = out;
    prm.d_err = d_err;
    cudaStream_t cs = (cudaStream_t)stream;
    switch (G) {
        case 1: return launch_prefill<1>(pool, q, total_q, num_q_heads, num_seqs, prm, cs);
        case 2: return launch_prefill<2>(pool, q, total_q, num_q_heads, num_seqs, prm, cs);
        case 4: return launch_prefill<4>(pool, q, total_q, num_q_heads, num_seqs, prm, cs);
        default: return launch_prefill<8>(pool, q, total_q, num_q_heads, num_seqs, prm, cs);
    }
}
