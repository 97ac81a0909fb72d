// pa_prefill: paged chunked-prefill attention on the 5th-generation tensor
// cores (tcgen05, accumulators in TMEM, operands staged by TMA).
//
// Semantics: "03｜PagedAttention 与 KV Cache 内存系统" §4 — prefill reuses a
// flash-style tiled attention kernel that is handed the paged block table
// (paging decides where K/V live, tiling decides how one attention pass moves
// through them).  New token i of a sequence sits at position
// context_len - n_new + i and, with a causal mask, sees positions 0..itself.
//
// CTA = (q-tile, kv-head, sequence).  A tile is 128 rows = (128/G) queries x
// the G query heads that share one kv-head, so every K/V byte staged in
// shared memory feeds all G heads.  Key tiles are 128 keys = 128/B_p pages,
// each page half (64 dims) fetched by one tiled TMA load straight from the
// pool through the block table.
//
// Roles (192 threads):
//   warp 0  TMA producer: Q tile once, then K tiles into a 3-stage ring
//           (a stage frees when its S MMA completes) and V tiles into a
//           2-stage ring (freed when its P*V MMA completes), issuing
//           whichever load has a free stage.
//   warp 1  MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//           buffers, then O += P_{j-1} V_{j-1} once the softmax published
//           P_{j-1}; tcgen05.commit signals completion on mbarriers.
//   warps 2-5  softmax: thread r owns row r (TMEM lane r): loads S_j, masks,
//           online softmax in base 2 with lazy rescaling of O (only when the
//           row max grows by more than 2^8), converts its key row of the V
//           tile from bf16 to fp16 in place, writes P_j as fp16 into a
//           128-byte-swizzled K-major tile, and finally normalises O.
// Q K^T runs on bf16 operands; P V runs on fp16 operands: P in [0, 2^8]
// keeps 11 significant bits in fp16 against 8 in bf16, which the stated
// accuracy needs (bf16 P alone leaves ~1.6e-3 relative L2 error at 2.5K
// keys).  bf16 -> fp16 is exact for |v| <= 65504 (the fp16 range; larger
// magnitudes saturate to +-65504) apart from fp16 subnormals below 2^-14,
// whose absolute error stays under 2^-25.
// All mbarrier waits are bounded; a wait that runs out sets PA_ERR_TIMEOUT
// and the CTA winds down.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include <cmath>
#include <mutex>

#include "common.cuh"
#include "host_common.h"
#include "tcgen05.cuh"

namespace pa {

constexpr int kPfRows = 128;            // M: rows of a tile (queries x heads)
constexpr int kPfKeys = 128;            // N: keys per KV tile
constexpr int kPfDim = 128;             // head_dim
constexpr int kHalf = 128 * 128;        // bytes of one 64-column half of a 128-row bf16 tile
constexpr int kTile = 2 * kHalf;        // 32 KiB
constexpr int kPfThreads = 192;
constexpr uint32_t kTmemCols = 512;     // S0 | S1 | O (| unused)
constexpr float kPfRescale = 8.0f;

// shared-memory map (offsets from a 1024-aligned base)
constexpr int kKStages = 3;
constexpr int kVStages = 2;
constexpr int kOffQ = 0;
constexpr int kOffK = kTile;                         // kKStages stages
constexpr int kOffV = kOffK + kKStages * kTile;      // kVStages stages
constexpr int kOffP = kOffV + kVStages * kTile;
constexpr int kOffBar = kOffP + kTile;
constexpr int kPfSmem = kOffBar + 1024 + 1024;  // + barriers and page ids, + alignment slack

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

constexpr int kIdRing = 4;  // tiles of page ids kept for the V loads (K runs <= 3 tiles ahead)

struct PfBars {
    int32_t page_row[kIdRing][32];  // pool row of each page of a tile (128 / B_p <= 16 used)
    uint64_t q_full;
    uint64_t k_full[kKStages];
    uint64_t k_empty[kKStages];
    uint64_t v_full[kVStages];
    uint64_t v_empty[kVStages];
    uint64_t s_full[2];
    uint64_t s_empty[2];
    uint64_t p_full;
    uint64_t o_done;
    uint32_t tmem_base;
    int32_t abort;
};

// two floats -> fp16 pair (lo in the low half)
PA_DEVICE uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// bf16 pair -> fp16 pair (saturating at the fp16 range)
PA_DEVICE uint32_t bf16x2_to_f16x2(uint32_t w) {
    uint32_t r;
    asm("cvt.rn.satfinite.f16x2.f32 %0, %1, %2;"
        : "=r"(r) : "f"(__uint_as_float(w & 0xffff0000u)), "f"(__uint_as_float(w << 16)));
    return r;
}

// acc + lo + hi of an fp16 pair, accumulated in fp32
PA_DEVICE float add_f16x2_to(float acc, uint32_t h2) {
    float r;
    asm("{ .reg .b16 a, b; mov.b32 {a, b}, %1; add.rn.f32.f16 %0, a, %2; add.rn.f32.f16 %0, b, %0; }"
        : "=f"(r) : "r"(h2), "f"(acc));
    return r;
}

PA_DEVICE uint4 ld_shared_v4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

PA_DEVICE void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};"
                 ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d) : "memory");
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

template <int G>
__global__ void __launch_bounds__(kPfThreads, 1)
prefill_kernel(const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_k,
               const __grid_constant__ CUtensorMap tmap_v, const PrefillParams p) {
    constexpr int QT = kPfRows / G;  // queries per tile
    const int qt = p.max_qtiles - 1 - (int)blockIdx.x;  // longest tiles first
    const int h = blockIdx.y, s = blockIdx.z;
    const int q_begin = __ldg(p.cu_seqlens_q + s);
    const int n_new = __ldg(p.cu_seqlens_q + s + 1) - q_begin;
    const int q0 = qt * QT;
    if (n_new <= 0 || q0 >= n_new) {
        if (qt == 0 && h == 0 && threadIdx.x == 0 && n_new > p.max_qtiles * QT)
            set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    const int ctx = __ldg(p.context_lens + s);
    const int base_pos = ctx - n_new;  // position of new token 0
    if (base_pos < 0) {
        if (threadIdx.x == 0) set_error(p.d_err, PA_ERR_INVALID_ARG);
        return;
    }
    const int q_last = min(q0 + QT, n_new) - 1;
    const int kv_end = p.causal ? base_pos + q_last + 1 : ctx;  // keys [0, kv_end)
    const int n_tiles = (kv_end + kPfKeys - 1) / kPfKeys;
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
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bars->s_full[i], 1);
            mbar_init(&bars->s_empty[i], 128);
        }
        mbar_init(&bars->p_full, 128);
        mbar_init(&bars->o_done, 1);
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
    const uint32_t tS = tmem;             // columns [0, 256): two S buffers
    const uint32_t tO = tmem + 256;       // columns [256, 384): O

    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        // The whole warp works: lane k handles page k of a tile (one coalesced
        // table load per tile, prefetched a tile ahead, then its own TMA loads);
        // lane 0 arms the barriers and decides when a stage is free.
        const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks;
        auto load_rows = [&](int j) -> int32_t {  // this lane's page of tile j
            const int e = j * pages_per_tile + lane;
            if (lane >= pages_per_tile || (e << p.log2_bp) >= kv_end) return -1;
            int32_t id = e < p.max_blocks ? __ldg(table + e) : -1;
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
            mbar_arrive_expect_tx(&bars->q_full, kTile);
            tc::tma_load_3d(smem + kOffQ, &tmap_q, 0, h * G, q_begin + q0, &bars->q_full);
            tc::tma_load_3d(smem + kOffQ + kHalf, &tmap_q, 64, h * G, q_begin + q0, &bars->q_full);
        }
        int32_t next_row = load_rows(0);  // prefetched ids of tile kn
        int kn = 0, vn = 0;
        uint64_t t_idle = 0;
        uint32_t spins = 0;
        while (kn < n_tiles || vn < n_tiles) {
            bool moved = false;
            // K tile kn into its stage once the S MMA of tile kn - 3 has completed
            int go = 0;
            if (lane == 0)
                go = kn < n_tiles && kn < vn + kIdRing &&  // page ids of tiles vn..kn stay live
                     (kn < kKStages || mbar_try_wait(&bars->k_empty[kn % kKStages],
                                                     ((kn / kKStages) - 1) & 1));
            if (__shfl_sync(0xffffffffu, go, 0)) {
                const int row = next_row;
                if (kn + 1 < n_tiles) next_row = load_rows(kn + 1);
                bars->page_row[kn % kIdRing][lane] = row;
                const int loaded = loaded_pages(kn);
                uint64_t* bar = &bars->k_full[kn % kKStages];
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)loaded * bp * 128 * 2);
                __syncwarp();
                if (lane < loaded) {
                    unsigned char* dst = smem + kOffK + (kn % kKStages) * kTile + lane * bp * 128;
                    tc::tma_load_2d(dst, &tmap_k, 0, row, bar);
                    tc::tma_load_2d(dst + kHalf, &tmap_k, 64, row, bar);
                }
                ++kn;
                moved = true;
            }
            // V tile vn once the P*V MMA of tile vn - 2 has completed
            go = 0;
            if (lane == 0)
                go = vn < n_tiles && vn < kn &&
                     (vn < kVStages || mbar_try_wait(&bars->v_empty[vn % kVStages],
                                                     ((vn / kVStages) - 1) & 1));
            if (__shfl_sync(0xffffffffu, go, 0)) {
                const int row = bars->page_row[vn % kIdRing][lane];
                const int loaded = loaded_pages(vn);
                uint64_t* bar = &bars->v_full[vn % kVStages];
                if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)loaded * bp * 128 * 2);
                __syncwarp();
                if (lane < loaded) {
                    unsigned char* dst = smem + kOffV + (vn % kVStages) * kTile + lane * bp * 128;
                    tc::tma_load_2d(dst, &tmap_v, 0, row, bar);
                    tc::tma_load_2d(dst + kHalf, &tmap_v, 64, row, bar);
                }
                ++vn;
                moved = true;
            }
            if (moved) {
                t_idle = 0;
                continue;
            }
            int stop = 0;
            if (lane == 0 && (++spins & 255u) == 0) {
                if (*(volatile int32_t*)&bars->abort) stop = 1;
                const uint64_t now = global_timer_ns();
                if (t_idle == 0) {
                    t_idle = now;
                } else if (now - t_idle > kWaitLimitNs) {
                    set_error(p.d_err, PA_ERR_TIMEOUT);
                    *(volatile int32_t*)&bars->abort = 1;
                    stop = 1;
                }
            }
            if (__shfl_sync(0xffffffffu, stop, 0)) break;
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc_qk = tc::idesc_bf16_f32(128, 128, 0, 0);
            constexpr uint32_t idesc_pv = tc::idesc_f16_f32(128, 128, 0, 1);
            const uint32_t q_addr = smem_u32(smem + kOffQ);
            const uint32_t p_addr = smem_u32(smem + kOffP);
            bool ok = pf_wait(&bars->q_full, 0, bars, p.d_err);
            auto pv = [&](int t) -> bool {
                if (!pf_wait(&bars->p_full, t & 1, bars, p.d_err)) return false;
                tc::fence_after_sync();
                const uint32_t v_addr = smem_u32(smem + kOffV + (t % kVStages) * kTile);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t poff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    const uint64_t b = tc::smem_desc_sw128(v_addr + kk * 2048, kHalf, 1024);
                    tc::mma_bf16(tO, tc::smem_desc_sw128(p_addr + poff, 16, 1024), b, idesc_pv,
                                 (t > 0 || kk > 0) ? 1u : 0u);
                }
                tc::commit(&bars->o_done);
                tc::commit(&bars->v_empty[t % kVStages]);
                return true;
            };
            for (int j = 0; ok && j < n_tiles; ++j) {
                const int st = j & 1;
                const int ks = j % kKStages;
                if (!pf_wait(&bars->k_full[ks], (j / kKStages) & 1, bars, p.d_err)) { ok = false; break; }
                if (j >= 2 && !pf_wait(&bars->s_empty[st], ((j >> 1) - 1) & 1, bars, p.d_err)) { ok = false; break; }
                tc::fence_after_sync();
                const uint32_t k_addr = smem_u32(smem + kOffK + ks * kTile);
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk >> 2) * kHalf + (kk & 3) * 32;
                    const uint64_t a = tc::smem_desc_sw128(q_addr + koff, 16, 1024);
                    const uint64_t b = tc::smem_desc_sw128(k_addr + koff, 16, 1024);
                    tc::mma_bf16(tS + st * 128, a, b, idesc_qk, kk > 0 ? 1u : 0u);
                }
                tc::commit(&bars->s_full[st]);
                tc::commit(&bars->k_empty[ks]);
                if (j >= 1 && !pv(j - 1)) { ok = false; break; }
            }
            if (ok) pv(n_tiles - 1);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;        // tile row == TMEM lane
        const int i = r / G, g = r - i * G;
        const int qi = q0 + i;
        const bool live = qi < n_new;
        int lim = p.causal ? base_pos + qi : ctx - 1;  // last visible key
        if (!live) lim = 0;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        const uint32_t p_row = smem_u32(smem + kOffP) + r * 128;
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < n_tiles; ++j) {
            const int sb = j & 1;
            ok = pf_wait(&bars->s_full[sb], (j >> 1) & 1, bars, p.d_err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            tc::fence_after_sync();
            uint32_t sr[4][32];
#pragma unroll
            for (int c = 0; c < 4; ++c) tc::tmem_ld32(tS + lane_addr + sb * 128 + c * 32, sr[c]);
            tc::tmem_wait_ld();
            tc::fence_before_sync();
            mbar_arrive(&bars->s_empty[sb]);

            const int key0 = j * kPfKeys;
            float tmax = -INFINITY;
            const bool full = key0 + kPfKeys - 1 <= lim;
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                    float x = __uint_as_float(sr[c][e]) * p.scale_log2;
                    if (!full && key0 + c * 32 + e > lim) x = -INFINITY;
                    sr[c][e] = __float_as_uint(x);
                    tmax = fmaxf(tmax, x);
                }
            bool o_ready = false;
            if (j == 0) {
                m_used = tmax;
            } else {
                const float m_new = fmaxf(m_used, tmax);
                const bool need = m_new > m_used + kPfRescale;
                if (__any_sync(0xffffffffu, need)) {
                    // O holds tiles < j at scale m_used: wait for PV_{j-1}, then rescale
                    ok = pf_wait(&bars->o_done, (j - 1) & 1, bars, p.d_err);
                    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
                    o_ready = true;
                    tc::fence_after_sync();
                    const float f = need ? ex2(m_used - m_new) : 1.f;
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        uint32_t o[32];
                        tc::tmem_ld32(tO + lane_addr + c * 32, o);
                        tc::tmem_wait_ld();
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                        tc::tmem_st32(tO + lane_addr + c * 32, o);
                    }
                    tc::tmem_wait_st();
                    tc::fence_before_sync();
                    l *= f;
                    if (need) m_used = m_new;
                }
            }
            // probabilities (masked keys give exactly 0)
            // probabilities in fp16; the row sum adds the rounded values the
            // tensor cores multiply with
            float lsum = 0.f;
            uint32_t pk[64];
#pragma unroll
            for (int c = 0; c < 4; ++c)
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float a = ex2(__uint_as_float(sr[c][e]) - m_used);
                    const float b2 = ex2(__uint_as_float(sr[c][e + 1]) - m_used);
                    const uint32_t w = pack_f16(a, b2);
                    lsum = add_f16x2_to(lsum, w);
                    pk[(c * 32 + e) >> 1] = w;
                }
            l += lsum;
            // the P tile is single-buffered: PV_{j-1} must have finished reading it
            if (j >= 1 && !o_ready) {
                ok = pf_wait(&bars->o_done, (j - 1) & 1, bars, p.d_err);
                if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            }
            // this thread's key row of V_j: bf16 -> fp16 in place (16-byte chunks keep
            // their swizzled positions); rows past the written keys become zeros
            ok = pf_wait(&bars->v_full[j % kVStages], (j / kVStages) & 1, bars, p.d_err);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
            {
                const uint32_t vrow = smem_u32(smem + kOffV + (j % kVStages) * kTile) + r * 128;
                // chunk order rotated by the row so the 8 threads of a 128-bit access
                // phase touch 8 different bank groups
                if (key0 + r < zlim) {
#pragma unroll
                    for (int c = 0; c < 16; ++c) {
                        const uint32_t a = vrow + (c >> 3) * kHalf + ((c + r) & 7) * 16;
                        const uint4 x = ld_shared_v4(a);
                        st_shared_v4(a, bf16x2_to_f16x2(x.x), bf16x2_to_f16x2(x.y),
                                     bf16x2_to_f16x2(x.z), bf16x2_to_f16x2(x.w));
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < 16; ++c)
                        st_shared_v4(vrow + (c >> 3) * kHalf + ((c + r) & 7) * 16, 0, 0, 0, 0);
                }
            }
            // P row r: 16-byte chunk c (keys 8c..8c+7) at chunk (c mod 8) ^ (r mod 8) of half c/8
#pragma unroll
            for (int c = 0; c < 16; ++c) {
                const uint32_t addr = p_row + (c >> 3) * kHalf + (((c & 7) ^ (r & 7)) << 4);
                st_shared_v4(addr, pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
            }
            fence_proxy_async_smem();
            mbar_arrive(&bars->p_full);
        }
        // epilogue: O / l -> out
        if (ok) ok = pf_wait(&bars->o_done, (n_tiles - 1) & 1, bars, p.d_err);
        if (__all_sync(0xffffffffu, ok)) {
            tc::fence_after_sync();
            const float inv = live ? 1.f / l : 0.f;
            float* orow = p.out + ((int64_t)(q_begin + qi) * p.num_q_heads + h * G + g) * kPfDim;
#pragma unroll
            for (int c = 0; c < 4; ++c) {
                uint32_t o[32];
                tc::tmem_ld32(tO + lane_addr + c * 32, o);
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
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

static bool make_map(CUtensorMap* m, const void* base, int rank, const cuuint64_t* dims,
                     const cuuint64_t* strides, const cuuint32_t* box) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                    strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
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
    dim3 grid((unsigned)prm.max_qtiles, (unsigned)pool->num_kv_heads, (unsigned)B);
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
