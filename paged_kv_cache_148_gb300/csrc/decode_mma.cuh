// Tensor-core form of the decode partition work for bf16 pools with
// head_dim 128 and pages of >= 16 tokens, and the shared-prefix pair units
// built on it.  Included by decode.cu after DecodeParams.
//
// Semantics are those of the CUDA-core partition kernel ("03｜PagedAttention
// 与 KV Cache 内存系统" §4: walk the visible blocks through the table, combine
// blockwise softmax states); only the arithmetic moves to warp-level
// mma.sync m16n8k16 (bf16 operands, fp32 accumulation):
//  * a warp streams every W-th 16-token chunk of its unit through a 2-stage
//    ring; a chunk is four 2-D TMA boxes of 16 rows x 64 dims (K low, K high,
//    V low, V high) taken from the pool viewed as [rows][128] bf16 with the
//    128-byte swizzle: row r of a box holds its 16-byte unit u at u ^ (r & 7);
//  * S^T = K Q^T: the 16 tokens are the M rows, the query heads of the unit
//    the N columns (8 per n-tile), head_dim the K dimension.  Tile row r
//    stands for token (r >> 1) + 4 (r & 1) (+8 for the upper half), so that
//    each 8-lane phase of the K loads and of the ldmatrix V loads touches
//    rows whose swizzle keys differ and no bank is hit twice;
//  * one 16-byte K load feeds two k-steps: the dims a lane holds are the same
//    permutation of k on the K and the Q side, so the dot products are
//    unchanged;
//  * online softmax in base 2 on the accumulator fragments (maxima over the
//    16 tokens by shuffles; lazy rescaling only when a maximum grows by more
//    than 2^8);
//  * O^T += V^T P^T: V^T fragments by ldmatrix.trans straight from the
//    swizzled boxes; P^T comes from the S^T accumulator layout through
//    movmatrix.trans, split into a bf16 high part and a bf16 low part (two
//    MMAs) so the probabilities keep about 16 significant bits;
//  * the warps combine in shared memory and write the output (a single
//    partition) or (max, exp_sum, weighted V) partials for the merge.
//
// Shared-prefix pair units ("03｜PagedAttention 与 KV Cache 内存系统" §5 and
// "PagedAttention 的原理是什么？…" §四: forked sequences hold the same
// physical blocks of their common prefix, refcount 2).  A unit may score each
// staged page against the heads of two sequences at once: head columns
// 0..G-1 belong to sequence A, G..2G-1 to sequence B, so a shared page is
// read from HBM once for both.  Each sequence's partials go to its own slots
// and the ordinary merge combines them; the result equals the plain decode of
// each sequence.
#pragma once

namespace pa {
namespace mma {

constexpr int kD = 128;
constexpr int kBox = 64 * kChunk * 2;                       // 2 KiB: 16 rows x 64 dims
constexpr int kStageBytes = 4 * kBox;                        // K lo | K hi | V lo | V hi
constexpr int kW = 4;                                        // warps per CTA
constexpr int kS = 2;                                        // ring stages per warp
constexpr size_t kRing = (size_t)kW * kS * kStageBytes;      // 64 KiB
constexpr size_t kSmem = 1024 + kRing + kW * kS * 8 + kW * kS * 4;

PA_DEVICE void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                              uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

PA_DEVICE void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                             uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

PA_DEVICE uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// two floats -> bf16 pair (lo in the low half), round to nearest even
PA_DEVICE uint32_t pack_bf16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

PA_DEVICE uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

// token held by tile row r (r < 8); row r + 8 holds token 8 + pi_tok(r)
PA_DEVICE int pi_tok(int r) { return (r >> 1) + 4 * (r & 1); }

// One unit of work: chunks [cb, ce) of sequence seq_a's table, for kv-head h.
struct Unit {
    int h;
    int seq_a, seq_b;  // head columns 0..G-1: seq_a's q-heads; G..2G-1: seq_b's (pair units)
    int cb, ce;
    int n;             // positions < n are visible
    int lo;            // first visible position (sliding window), else 0
    int slot;          // partial slot written for both sequences
    int np_a, np_b;    // slots (partitions) of each sequence; 1: write the output directly
};

// One-launch step (pa_decode_step): the new token's K and V rows of (s, h),
// kept in shared memory from the kernel's start until the chunk that holds
// position n - 1 has landed.
struct StepRow {
    uint4 row[32];   // lanes 0-15: K row, 16-31: V row (16 bytes each)
    int64_t slot;    // slot_mapping[s]
    int32_t pid;     // table entry of the page holding position n - 1
};

// Unit body for NH head columns (NH = G: one sequence; NH = 2G: a pair).  The
// caller has set *aborted = 0 and every thread of the CTA enters.  With
// kFused (pa_decode_step, NH = G) the warp that streams the chunk holding
// position n - 1 also writes the new token's row into the pool and into that
// chunk's staged copy, and the last partition of (s, h) to finish merges the
// partials (n_parts > 1).
template <int G, int NH, bool kFused = false>
PA_DEVICE void unit_body(const DecodeParams& p, const CUtensorMap* mk, const CUtensorMap* mv,
                         unsigned char* smem, int* aborted, const Unit& u,
                         StepRow* step = nullptr) {
    static_assert(!kFused || NH == G, "the one-launch step decodes single sequences");
    constexpr int NT = (NH + 7) / 8;  // n-tiles of 8 head columns
    static_assert(NH == G || NH == 2 * G, "one sequence or a pair");
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int32_t* table = p.block_tables + (int64_t)u.seq_a * p.max_blocks;
    const int32_t* table_b = NH > G ? p.block_tables + (int64_t)u.seq_b * p.max_blocks : nullptr;
    const int first = u.cb + warp;  // this warp's chunks: first + i * kW
    const int my_n = first < u.ce ? (u.ce - first + kW - 1) / kW : 0;
    // page id of this warp's local chunk i (an entry past the table is flagged
    // at issue); a pair unit checks that both tables name the same page
    auto table_id = [&](int i) -> int32_t {
        const int e = ((first + i * kW) * kChunk) >> p.log2_bp;
        if (e >= p.max_blocks) return p.num_blocks;
        const int32_t id = __ldg(table + e);
        if (NH > G && __ldg(table_b + e) != id) set_error(p.d_err, PA_ERR_INVALID_ARG);
        return id;
    };
    int32_t id_reg = lane < my_n ? table_id(lane) : -1;  // lane j: local chunk id_base + j
    int id_base = 0;

    unsigned char* ring = smem + (size_t)warp * kS * kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kRing) + warp * kS;
    uint32_t* masks = reinterpret_cast<uint32_t*>(smem + kRing + kW * kS * 8) + warp * kS;
    if (lane == 0) {
#pragma unroll
        for (int i = 0; i < kS; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // lane 0 issues local chunk i: four boxes of 16 rows x 64 dims; with pages
    // of >= 16 tokens a chunk lies within one page
    auto issue = [&](int i, int32_t id) {
        const int stage = i % kS;
        const int t0 = (first + i * kW) * kChunk;
        const bool page_ok = id >= 0 && id < p.num_blocks;
        if (!page_ok) set_error(p.d_err, id < 0 ? PA_ERR_NEGATIVE_BLOCK : PA_ERR_OUT_OF_RANGE);
        const int valid = min(kChunk, u.n - t0);
        uint32_t mask = page_ok ? ((1u << valid) - 1u) : 0u;
        if (u.lo > t0) mask &= ~((1u << min(u.lo - t0, kChunk)) - 1u);  // before the window
        uint64_t* bar = &bars[stage];
        masks[stage] = mask;
        if (!page_ok) {
            mbar_arrive_expect_tx(bar, 0);
            return;
        }
        mbar_arrive_expect_tx(bar, (uint32_t)kStageBytes);
        const int32_t y = (int32_t)((((int64_t)id * p.num_kv_heads + u.h) << p.log2_bp) +
                                    (t0 & ((1 << p.log2_bp) - 1)));
        unsigned char* dst = ring + (size_t)stage * kStageBytes;
        tc::tma_load_2d(dst, mk, 0, y, bar);
        tc::tma_load_2d(dst + kBox, mk, 64, y, bar);
        tc::tma_load_2d(dst + 2 * kBox, mv, 0, y, bar);
        tc::tma_load_2d(dst + 3 * kBox, mv, 64, y, bar);
    };

    // one-launch step: the owner warp streams the chunk of position n - 1 and
    // loads the new row now (the loads complete behind the prologue's copies)
    const int n_chunks = (u.n + kChunk - 1) / kChunk;
    const int last_chunk = n_chunks - 1;
    const bool owner = kFused && u.ce == n_chunks && last_chunk >= first &&
                       (last_chunk - first) % kW == 0;
    uint4 row_reg = make_uint4(0, 0, 0, 0);
    if (owner) {
        const int64_t src = ((int64_t)u.seq_a * p.num_kv_heads + u.h) * kRowBytes + (lane & 15) * 16;
        row_reg = __ldg(reinterpret_cast<const uint4*>((lane < 16 ? p.k_new : p.v_new) + src));
        if (lane == 0) {
            step->slot = __ldg(p.slot_mapping + u.seq_a);
            const int e = (u.n - 1) >> p.log2_bp;
            step->pid = e < p.max_blocks ? __ldg(table + e) : -1;
        }
    }

    // Q^T columns: n-tile t, column 8t + gid; lane (gid, tig) holds dims
    // 32q + 8tig .. +7 of that head for q = 0..3 (zeros for padding columns)
    uint4 qa[NT][4];
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        const int hh = 8 * t + gid;
        const int seq = hh < G ? u.seq_a : u.seq_b;
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(p.q) +
                             ((int64_t)seq * p.num_q_heads + (int64_t)u.h * G + (hh % G)) * kD;
#pragma unroll
        for (int q = 0; q < 4; ++q)
            qa[t][q] = hh < NH ? __ldg(reinterpret_cast<const uint4*>(qb + 32 * q + 8 * tig))
                               : make_uint4(0, 0, 0, 0);
    }

#pragma unroll
    for (int i = 0; i < kS; ++i) {
        const int32_t id = __shfl_sync(kFull, id_reg, i & 31);
        if (lane == 0 && i < my_n) issue(i, id);
    }
    if (owner) {
        step->row[lane] = row_reg;  // kept in shared memory through the loop
        __syncwarp();               // lane 0's slot and page id are visible to the warp
    }

    // O^T accumulators: o[mt][t] = dims 16 mt + gid (0, 1) and + 8 (2, 3) of
    // head columns 8t + 2tig (0, 2) and 8t + 2tig + 1 (1, 3)
    float o[8][NT][4];
#pragma unroll
    for (int mt = 0; mt < 8; ++mt)
#pragma unroll
        for (int t = 0; t < NT; ++t) o[mt][t][0] = o[mt][t][1] = o[mt][t][2] = o[mt][t][3] = 0.f;
    float m[NT][2], l[NT][2];  // running maxima (base 2) and this lane's share of the sums
#pragma unroll
    for (int t = 0; t < NT; ++t) {
        m[t][0] = m[t][1] = -INFINITY;
        l[t][0] = l[t][1] = 0.f;
    }
    const int ta = pi_tok(gid), tb = 8 + pi_tok(gid);  // tokens of tile rows gid, gid + 8
    // K: k-step pair q reads unit 4(q & 1) + tig of box q >> 1; rows ta and tb
    // share the swizzle key ta
    const uint32_t k_lane0 = ta * 128 + ((tig ^ ta) << 4);
    const uint32_t k_lane1 = ta * 128 + (((tig ^ ta) ^ 4) << 4);
    // ldmatrix row addresses: matrices 0 / 1 hold tokens pi(r) / 8 + pi(r) of
    // dims 16mt .. +7 (unit 2(mt & 3) of box mt >> 2), matrices 2 / 3 the same
    // tokens of dims 16mt + 8 .. +15 (the next unit)
    const int v_tok = ((lane >> 3) & 1) * 8 + pi_tok(lane & 7);
    const uint32_t v_row = v_tok * 128;
    const uint32_t v_key = (uint32_t)((lane >> 4) ^ (v_tok & 7));

    bool ok = true;
#pragma unroll 1
    for (int i = 0; i < my_n; ++i) {
        const int stage = i % kS;
        const uint32_t parity = (uint32_t)(i / kS) & 1u;
        ok = mbar_wait(&bars[stage], parity, p.d_err);
        if (!__all_sync(kFull, ok)) {
            ok = false;
            break;
        }
        const uint32_t vmask = masks[stage];
        unsigned char* kst = ring + (size_t)stage * kStageBytes;
        unsigned char* vst = kst + 2 * kBox;
        if (vmask != 0xffffu) {
            // rows no copy wrote or that are not visible may hold any bits
            // (NaN times a zero weight is NaN): clear their V rows
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int idx = j * 32 + lane, r = idx >> 4;
                if (!((vmask >> r) & 1u))
                    *reinterpret_cast<uint4*>(vst + ((idx >> 3) & 1) * kBox + r * 128 + (idx & 7) * 16) =
                        make_uint4(0, 0, 0, 0);
            }
            fence_proxy_async_smem();  // before a later copy refills this stage
            __syncwarp();
        }
        if (owner && first + i * kW == last_chunk) {
            // the new token: check that its slot is that of position n - 1 under
            // the table, then store its row to the pool and over the staged
            // chunk's row (the copy may have read the slot before or after the
            // store; the attention uses the new row either way)
            const int pos = u.n - 1;
            const int64_t bpm = (1 << p.log2_bp) - 1;
            const int64_t slot = step->slot;
            const int32_t pid = step->pid;
            int err = 0;
            if (slot < 0 || slot >= ((int64_t)p.num_blocks << p.log2_bp))
                err = PA_ERR_OUT_OF_RANGE;
            else if (pid < 0 || (slot >> p.log2_bp) != pid || (slot & bpm) != (pos & bpm))
                err = PA_ERR_INVALID_ARG;  // not the slot of the last position
            if (err != 0) {
                if (lane == 0) set_error(p.d_err, err);
            } else {
                const uint4 v = step->row[lane];
                const int64_t prow = ((int64_t)pid * p.num_kv_heads + u.h) * (bpm + 1) + (pos & bpm);
                unsigned char* pool = const_cast<unsigned char*>(lane < 16 ? p.k_pool : p.v_pool);
                *reinterpret_cast<uint4*>(pool + prow * kRowBytes + (lane & 15) * 16) = v;
                // 16-byte unit w of row r of a box sits at w ^ (r & 7) (128-byte swizzle)
                const int r = pos & (kChunk - 1), unit = lane & 15;
                unsigned char* box = kst + (lane < 16 ? 0 : 2 * kBox) + (unit >> 3) * kBox;
                *reinterpret_cast<uint4*>(box + r * 128 + (((unit & 7) ^ (r & 7)) << 4)) = v;
                fence_proxy_async_smem();  // before a later copy refills this stage
            }
            __syncwarp();
        }

        // ---- S^T = K Q^T per n-tile, even and odd k-steps in separate chains
        const uint32_t kb = smem_u32(kst);
        float sc[NT][2][4];
#pragma unroll
        for (int t = 0; t < NT; ++t)
#pragma unroll
            for (int e = 0; e < 2; ++e) sc[t][e][0] = sc[t][e][1] = sc[t][e][2] = sc[t][e][3] = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint32_t ka = kb + (q >> 1) * kBox + ((q & 1) ? k_lane1 : k_lane0);
            const uint4 ra = lds128(ka);            // token ta
            const uint4 rb = lds128(ka + 8 * 128);  // token tb
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                mma_bf16_16816(sc[t][0], ra.x, rb.x, ra.y, rb.y, qa[t][q].x, qa[t][q].y);
                mma_bf16_16816(sc[t][1], ra.z, rb.z, ra.w, rb.w, qa[t][q].z, qa[t][q].w);
            }
        }
        const bool va = (vmask >> ta) & 1u, vb = (vmask >> tb) & 1u;
        uint32_t bh0[NT], bh1[NT], bl0[NT], bl1[NT];
#pragma unroll
        for (int t = 0; t < NT; ++t) {
            // s[token][head]: tokens ta, tb; head columns 8t + 2tig (+1), base-2 logits
            float s2[2][2];
            s2[0][0] = va ? (sc[t][0][0] + sc[t][1][0]) * p.scale_log2 : -INFINITY;
            s2[0][1] = va ? (sc[t][0][1] + sc[t][1][1]) * p.scale_log2 : -INFINITY;
            s2[1][0] = vb ? (sc[t][0][2] + sc[t][1][2]) * p.scale_log2 : -INFINITY;
            s2[1][1] = vb ? (sc[t][0][3] + sc[t][1][3]) * p.scale_log2 : -INFINITY;
            float cm[2] = {fmaxf(s2[0][0], s2[1][0]), fmaxf(s2[0][1], s2[1][1])};
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                cm[0] = fmaxf(cm[0], __shfl_xor_sync(kFull, cm[0], off));
                cm[1] = fmaxf(cm[1], __shfl_xor_sync(kFull, cm[1], off));
            }
            // lazy rescale: the lanes that share a head column hold the same m and cm
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                if (cm[x] > m[t][x] + kRescaleThreshold) {
                    const float corr = ex2(m[t][x] - cm[x]);
                    m[t][x] = cm[x];
                    l[t][x] *= corr;
#pragma unroll
                    for (int mt = 0; mt < 8; ++mt) {
                        o[mt][t][x] *= corr;
                        o[mt][t][x + 2] *= corr;
                    }
                }
            }
            float pr[2][2];
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                pr[0][x] = va ? ex2(s2[0][x] - m[t][x]) : 0.f;
                pr[1][x] = vb ? ex2(s2[1][x] - m[t][x]) : 0.f;
                l[t][x] += pr[0][x] + pr[1][x];
            }
            // P^T in the accumulator layout (row = token, column pair = this
            // lane's heads), high and low bf16 parts, transposed into the B
            // layout (k = token, n = head)
            const uint32_t h0 = pack_bf16(pr[0][0], pr[0][1]);
            const uint32_t h1 = pack_bf16(pr[1][0], pr[1][1]);
            const uint32_t l0 = pack_bf16(pr[0][0] - bf16_lo(h0), pr[0][1] - bf16_hi(h0));
            const uint32_t l1 = pack_bf16(pr[1][0] - bf16_lo(h1), pr[1][1] - bf16_hi(h1));
            bh0[t] = movmatrix_trans(h0);
            bh1[t] = movmatrix_trans(h1);
            bl0[t] = movmatrix_trans(l0);
            bl1[t] = movmatrix_trans(l1);
        }

        // ---- O^T += V^T P^T over 8 tiles of 16 dims, every n-tile
        const uint32_t vaddr = smem_u32(vst) + v_row;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vaddr + (mt >> 2) * kBox + (((2u * (mt & 3)) ^ v_key) << 4), r0, r1, r2, r3);
#pragma unroll
            for (int t = 0; t < NT; ++t) {
                mma_bf16_16816(o[mt][t], r0, r2, r1, r3, bh0[t], bh1[t]);
                mma_bf16_16816(o[mt][t], r0, r2, r1, r3, bl0[t], bl1[t]);
            }
        }
        __syncwarp();

        // ---- refill this stage with local chunk i + kS
        const int nxt = i + kS;
        if (nxt - id_base >= 32) {
            id_base += 32;
            id_reg = (id_base + lane < my_n) ? table_id(id_base + lane) : -1;
        }
        const int32_t nid = __shfl_sync(kFull, id_reg, (nxt - id_base) & 31);
        if (lane == 0 && nxt < my_n) issue(nxt, nid);
    }
    if (!ok) *aborted = 1;
    griddep_launch();  // the merge may start launching; it waits for this grid to finish

#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
            l[t][0] += __shfl_xor_sync(kFull, l[t][0], off);
            l[t][1] += __shfl_xor_sync(kFull, l[t][1], off);
        }

    // ---- combine the CTA's warps (reusing the ring) and write
    __syncthreads();
    if (*aborted) {
        if constexpr (kFused) {
            // the step still counts this partition so the group's semaphore
            // returns to zero (the result is flagged invalid by *d_err)
            if (u.np_a > 1 && threadIdx.x == 0) {
                int32_t* sem = p.sem + (int64_t)u.seq_a * p.num_kv_heads + u.h;
                if (atom_add_acq_rel_gpu(sem, 1) == u.np_a - 1) atomicExch(sem, 0);
            }
        }
        return;
    }
    constexpr int MOFF = NH * kD, LOFF = NH * kD + NH;
    constexpr int WSTRIDE = NH * kD + ((2 * NH + 3) / 4) * 4;
    static_assert((size_t)kW * WSTRIDE * 4 <= kRing, "the warps' combine fits in the ring");
    float* cw = reinterpret_cast<float*>(smem);
    float* mine = cw + warp * WSTRIDE;
#pragma unroll
    for (int t = 0; t < NT; ++t)
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            const int hh = 8 * t + 2 * tig + x;
            if (hh < NH) {
#pragma unroll
                for (int mt = 0; mt < 8; ++mt) {
                    mine[hh * kD + 16 * mt + gid] = o[mt][t][x];
                    mine[hh * kD + 16 * mt + 8 + gid] = o[mt][t][x + 2];
                }
                if (gid == 0) {
                    mine[MOFF + hh] = m[t][x];
                    mine[LOFF + hh] = l[t][x];
                }
            }
        }
    __syncthreads();
    for (int idx = threadIdx.x; idx < NH * kD; idx += kW * 32) {
        const int hh = idx / kD, d = idx - hh * kD;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kW; ++w) M = fmaxf(M, cw[w * WSTRIDE + MOFF + hh]);
        float Lsum = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            const float c = ex2(cw[w * WSTRIDE + MOFF + hh] - M);
            Lsum = fmaf(cw[w * WSTRIDE + LOFF + hh], c, Lsum);
            A = fmaf(cw[w * WSTRIDE + hh * kD + d], c, A);
        }
        const int seq = hh < G ? u.seq_a : u.seq_b;
        const int np = hh < G ? u.np_a : u.np_b;
        const int64_t qh = (int64_t)seq * p.num_q_heads + (int64_t)u.h * G + (hh % G);
        if (np == 1) {
            p.out[qh * kD + d] = A / Lsum;
        } else {
            const int64_t wi = qh * p.max_parts + u.slot;
            p.ws_acc[wi * kD + d] = A;
            if (d == 0) {
                p.ws_m[wi] = M;
                p.ws_l[wi] = Lsum;
            }
        }
    }
    if constexpr (kFused) {
        if (u.np_a > 1) {
            // publish this partition's partials and count it: the barrier orders
            // the CTA's stores before thread 0's release-acquire add; the CTA
            // that counts last merges (its acquire orders the reads of the
            // others' partials) and returns the semaphore to zero
            __shared__ int is_last;
            __syncthreads();
            if (threadIdx.x == 0) {
                int32_t* sem = p.sem + (int64_t)u.seq_a * p.num_kv_heads + u.h;
                is_last = atom_add_acq_rel_gpu(sem, 1) == u.np_a - 1;
                if (is_last) atomicExch(sem, 0);
            }
            __syncthreads();
            if (is_last) merge_group<G, kD, kW>(p, u.seq_a, u.h, u.np_a, cw);
        }
    }
}

// 1024-aligned dynamic shared memory of a CTA (the 128-byte swizzle wants its
// boxes on 1024-byte boundaries)
PA_DEVICE unsigned char* aligned_smem(unsigned char* raw) {
    return reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(raw) + 1023) &
                                            ~uintptr_t(1023));
}

// The partition kernel: CTA = (sequence, kv-head, partition), as the
// CUDA-core form, same plan and partials.  kFused: the one-launch step.
template <int G, bool kFused = false>
__global__ void __launch_bounds__(kW * 32, 3)
    decode_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mk,
                      const __grid_constant__ CUtensorMap mv) {
    const int s = blockIdx.x, h = blockIdx.y, part = blockIdx.z;
    griddep_wait();  // K/V rows, tables and lengths may come from the previous kernel
    int n = __ldg(p.context_lens + s);
    if (n > p.max_context) {  // longer than the plan allows
        if (part == 0 && h == 0 && threadIdx.x == 0) set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
        n = p.max_context;
    }
    const int lo = (p.window > 0 && n > p.window) ? n - p.window : 0;
    const int c_lo = lo / kChunk;
    const int c_begin = c_lo + part * p.part_chunks;
    const int n_chunks = (n + kChunk - 1) / kChunk;
    if (n <= 0 || c_begin >= n_chunks) return;
    const int n_parts = (n_chunks - c_lo + p.part_chunks - 1) / p.part_chunks;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ int aborted;
    if (threadIdx.x == 0) {
        aborted = 0;
        tc::prefetch_tmap(&mk);
        tc::prefetch_tmap(&mv);
    }
    Unit u;
    u.h = h;
    u.seq_a = u.seq_b = s;
    u.cb = c_begin;
    u.ce = min(c_begin + p.part_chunks, n_chunks);
    u.n = n;
    u.lo = lo;
    u.slot = part;
    u.np_a = u.np_b = n_parts;
    if constexpr (kFused) {
        __shared__ StepRow step;
        unit_body<G, G, true>(p, &mk, &mv, aligned_smem(smem_raw), &aborted, u, &step);
    } else {
        unit_body<G, G>(p, &mk, &mv, aligned_smem(smem_raw), &aborted, u);
    }
}

// ---------------------------------------------------------------- shared prefixes
// The pairing of sequence s as both members see it.  A declaration counts
// only if it is mutual: partner[s] = q, partner[q] = s, the same shared
// length on both sides, a positive multiple of the block size and of 16
// tokens, no longer than either context.  Anything else is reported (once,
// by `report`) as PA_ERR_INVALID_ARG and both are decoded on their own.
struct Pairing {
    int partner;    // -1: decoded on its own
    int shared;     // shared chunks
    int n;          // visible positions of s
    int np_shared;  // pair units (run by the lower member's CTAs)
    int np_priv;    // partitions over s's own chunks
};

PA_DEVICE int visible_len(const DecodeParams& p, int s) {
    return min(__ldg(p.context_lens + s), p.max_context);
}

PA_DEVICE Pairing pairing_of(const DecodeParams& p, int s, bool report) {
    Pairing r;
    r.partner = -1;
    r.shared = 0;
    r.n = visible_len(p, s);
    const int q = __ldg(p.partner + s);
    if (q >= 0) {
        bool ok = q < p.num_seqs && q != s && __ldg(p.partner + q) == s;
        const int P = __ldg(p.shared_lens + s);
        ok = ok && __ldg(p.shared_lens + q) == P && P > 0 && (P & ((1 << p.log2_bp) - 1)) == 0 &&
             (P & (kChunk - 1)) == 0;
        ok = ok && P <= r.n && P <= visible_len(p, q);
        if (ok) {
            r.partner = q;
            r.shared = P / kChunk;
        } else if (report) {
            set_error(p.d_err, PA_ERR_INVALID_ARG);
        }
    }
    const int pc = p.part_chunks;
    const int nc = (max(r.n, 0) + kChunk - 1) / kChunk;
    r.np_shared = (r.shared + pc - 1) / pc;
    r.np_priv = (nc - r.shared + pc - 1) / pc;
    return r;
}

// Grid (sequence s, kv-head h, z).  z < np_shared: the lower member of a pair
// runs pair unit z over the shared chunks (slot z of both members);
// np_shared <= z < np_shared + np_priv: partition z - np_shared of s's own
// chunks (slot z).
template <int G>
__global__ void __launch_bounds__(kW * 32, 3)
    decode_shared_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mk,
                         const __grid_constant__ CUtensorMap mv) {
    const int s = blockIdx.x, h = blockIdx.y, z = blockIdx.z;
    griddep_wait();
    const bool reporter = z == 0 && h == 0 && threadIdx.x == 0;
    if (reporter && __ldg(p.context_lens + s) > p.max_context) set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
    const Pairing me = pairing_of(p, s, reporter);
    if (me.n <= 0) return;
    const int pc = p.part_chunks;
    const int nc = (me.n + kChunk - 1) / kChunk;
    Unit u;
    u.h = h;
    u.n = me.n;
    u.lo = 0;
    u.slot = z;
    u.np_a = me.np_shared + me.np_priv;
    if (z < me.np_shared) {
        if (s > me.partner) return;  // the lower member's CTAs run the pair units
        const Pairing other = pairing_of(p, me.partner, false);
        u.seq_a = s;
        u.seq_b = me.partner;
        u.cb = z * pc;
        u.ce = min(u.cb + pc, me.shared);
        u.np_b = other.np_shared + other.np_priv;
    } else {
        const int zp = z - me.np_shared;
        if (zp >= me.np_priv) return;
        u.seq_a = u.seq_b = s;
        u.cb = me.shared + zp * pc;
        u.ce = min(u.cb + pc, nc);
        u.np_b = u.np_a;
    }
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    __shared__ int aborted;
    if (threadIdx.x == 0) {
        aborted = 0;
        tc::prefetch_tmap(&mk);
        tc::prefetch_tmap(&mv);
    }
    if (z < me.np_shared)
        unit_body<G, 2 * G>(p, &mk, &mv, aligned_smem(smem_raw), &aborted, u);
    else
        unit_body<G, G>(p, &mk, &mv, aligned_smem(smem_raw), &aborted, u);
}

}  // namespace mma
}  // namespace pa
