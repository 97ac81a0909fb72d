// Tensor-core form of the decode partition work for FP8 (E4M3) pages with one
// float32 scale per (token, kv-head) row, head_dim 128, pages of >= 16
// tokens and bf16 queries.  Included by decode.cu after DecodeParams; used
// where the CUDA-core FP8 kernel is bound by its arithmetic (G = 8).  Same
// unit of work, plan, partials and merge as decode_partition_kernel
// ("03｜PagedAttention 与 KV Cache 内存系统" §4: paged decode with split-KV
// partitions; "KV Cache：容量、布局与生命周期": quantised pages count their
// bytes per element in the page budget).
//
// Per warp and 16-token chunk, all MMAs are mma.sync m16n8k16 with f16
// operands and fp32 accumulation (E4M3 -> f16 is exact):
//   * staging: one 2-D TMA box of 16 rows x 128 codes for K and one for V,
//     from the pools viewed as [rows][128] bytes with the 128-byte swizzle
//     (row r holds its 16-byte unit u at u ^ (r & 7)), and two 64-byte bulk
//     copies of the chunk's K and V row scales; tile row r stands for token
//     ((r & 3) << 1) | (r >> 2) (+8 for the upper half), so the rows one
//     half-warp reads with the 8-byte K fragment loads have swizzle keys that
//     differ in bits 1-2 and touch distinct banks;
//   * S^T = K Q^T: M = 16 tokens, N = 8 heads, K = 16 dims; a lane converts
//     8 codes of each of its two rows per pair of k-steps
//     (cvt.rn.f16x2.e4m3x2) straight into its A fragment; Q is converted to
//     f16 once;
//   * score = acc * k_scale[token] in fp32; the V row scale enters through
//     the exponent: O accumulates p_o = 2^(s + lg2 v_scale - m') with its own
//     running max m', the sum l uses p = 2^(s - m), so the f16 P operand holds
//     values near 1 for the terms that matter whatever the scale's magnitude;
//   * the warp converts the chunk's V codes into a per-warp f16 buffer, each
//     token into its tile row (rows of 272 bytes, rows outside the visible
//     range zeroed), and O^T += V^T P^T
//     runs as in the bf16 kernel (ldmatrix.x4.trans for V^T, movmatrix for
//     P^T, P split into f16 high + low parts);
//   * at the end acc = o * 2^(m' - m), so the CTA combine and the merge see
//     the usual (m, l, acc) partials.
#pragma once

namespace pa {
namespace mma8 {

constexpr int kD = 128;
constexpr int kBox = kChunk * 128;                 // one TMA box: 16 rows x 128 codes
constexpr int kScaleOff = 2 * kBox;                // K box | V box | K scales | V scales
constexpr int kStageBytes = 5 * 1024;              // 4224 used, 1024-aligned boxes
constexpr int kVPad = 272;                         // f16 V row stride in shared memory
constexpr int kVBuf = kChunk * kVPad;              // per-warp f16 V buffer, 4352
constexpr int kW = 4, kS = 2;
constexpr size_t kRing = (size_t)kW * kS * kStageBytes;
constexpr size_t kBufs = kRing;                    // kW f16 V buffers
constexpr size_t kBars = kBufs + (size_t)kW * kVBuf;
constexpr size_t kMasks = kBars + (size_t)kW * kS * 8;
constexpr size_t kSmem = 1024 + kMasks + (size_t)kW * kS * 4;
static_assert(kVBuf % 16 == 0, "ldmatrix alignment");

// token held by tile row r (r < 8); row r + 8 holds token 8 + tile_tok(r).  The
// rows an 8-byte K fragment load reads in one half-warp (r = 0-3 or 4-7) then
// have swizzle keys that differ in bits 1-2, so its 8 units hit distinct banks
PA_DEVICE int tile_tok(int r) { return ((r & 3) << 1) | (r >> 2); }
PA_DEVICE int tok_tile(int t) { return (t >> 1) | ((t & 1) << 2); }

PA_DEVICE void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                             uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

PA_DEVICE void ldsm_x4_trans(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                             uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

PA_DEVICE uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

PA_DEVICE uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// two E4M3 codes (low byte first) -> f16x2 (exact)
PA_DEVICE uint32_t e4m3x2_f16x2(uint32_t two) {
    uint32_t h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((uint16_t)two));
    return h2;
}

// two floats -> f16 pair (lo in the low half), round to nearest even
PA_DEVICE uint32_t pack_f16(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

PA_DEVICE float f16_lo(uint32_t w) {
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, lo;\n\t}"
        : "=f"(f) : "r"(w));
    return f;
}
PA_DEVICE float f16_hi(uint32_t w) {
    float f;
    asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %1;\n\tcvt.f32.f16 %0, hi;\n\t}"
        : "=f"(f) : "r"(w));
    return f;
}

// bf16 pair -> f16 pair (through f32)
PA_DEVICE uint32_t bf16x2_to_f16x2(uint32_t w) { return pack_f16(bf16_lo(w), bf16_hi(w)); }

PA_DEVICE uint32_t movmatrix_trans(uint32_t a) {
    uint32_t d;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

PA_DEVICE float lg2_approx(float x) {
    float y;
    asm("lg2.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

template <int G>
__global__ void __launch_bounds__(kW * 32)
    decode_fp8_mma_kernel(const DecodeParams p, const __grid_constant__ CUtensorMap mk,
                          const __grid_constant__ CUtensorMap mv) {
    static_assert(G >= 1 && G <= 8, "the heads of a group are the N columns of one tile");
    const int s = blockIdx.x, h = blockIdx.y, part = blockIdx.z;
    griddep_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tig = lane & 3;
    const int32_t* table = p.block_tables + (int64_t)s * p.max_blocks;
    int n = __ldg(p.context_lens + s);
    if (n > p.max_context) {
        if (part == 0 && h == 0 && threadIdx.x == 0) set_error(p.d_err, PA_ERR_OUT_OF_RANGE);
        n = p.max_context;
    }
    const int c_lo = (p.window > 0 && n > p.window) ? (n - p.window) / kChunk : 0;
    const int lo = (p.window > 0 && n > p.window) ? n - p.window : 0;
    const int c_begin = c_lo + part * p.part_chunks;
    const int first = c_begin + warp;
    const int n_chunks = (n + kChunk - 1) / kChunk;
    if (n <= 0 || c_begin >= n_chunks) return;
    const int c_end = min(c_begin + p.part_chunks, n_chunks);
    const int n_parts = (n_chunks - c_lo + p.part_chunks - 1) / p.part_chunks;
    const int my_n = first < c_end ? (c_end - first + kW - 1) / kW : 0;
    auto table_id = [&](int i) -> int32_t {
        const int e = ((first + i * kW) * kChunk) >> p.log2_bp;
        return e < p.max_blocks ? __ldg(table + e) : p.num_blocks;  // flagged at issue
    };
    int32_t id_reg = table_id(lane);
    int id_base = 0;

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    unsigned char* ring = smem + (size_t)warp * kS * kStageBytes;
    unsigned char* vbuf = smem + kBufs + (size_t)warp * kVBuf;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kBars) + warp * kS;
    uint32_t* masks = reinterpret_cast<uint32_t*>(smem + kMasks) + warp * kS;
    __shared__ int aborted;
    if (threadIdx.x == 0) {
        aborted = 0;
        tc::prefetch_tmap(&mk);
        tc::prefetch_tmap(&mv);
    }
    if (lane == 0) {
        for (int i = 0; i < kS; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    __syncthreads();

    // lane 0 issues chunk i (a chunk lies in one page): one box of 16 K code
    // rows, one of 16 V code rows, and the chunk's K and V row scales
    auto issue = [&](int i, int32_t id) {
        const int stage = i % kS;
        const int t0 = (first + i * kW) * kChunk;
        const int bp = 1 << p.log2_bp;
        const bool page_ok = id >= 0 && id < p.num_blocks;
        if (!page_ok) set_error(p.d_err, id < 0 ? PA_ERR_NEGATIVE_BLOCK : PA_ERR_OUT_OF_RANGE);
        const int valid = min(kChunk, n - t0);
        uint32_t mask = page_ok ? ((1u << valid) - 1u) : 0u;
        if (lo > t0) mask &= ~((1u << min(lo - t0, kChunk)) - 1u);
        uint64_t* bar = &bars[stage];
        masks[stage] = mask;
        if (!page_ok) {
            mbar_arrive_expect_tx(bar, 0);
            return;
        }
        mbar_arrive_expect_tx(bar, (uint32_t)(2 * kBox + 2 * kChunk * 4));
        const int64_t row0 = ((int64_t)id * p.num_kv_heads + h) * bp + (t0 & (bp - 1));
        unsigned char* st = ring + (size_t)stage * kStageBytes;
        tc::tma_load_2d(st, &mk, 0, (int32_t)row0, bar);
        tc::tma_load_2d(st + kBox, &mv, 0, (int32_t)row0, bar);
        bulk_g2s(st + kScaleOff, p.k_scale + row0, kChunk * 4, bar);
        bulk_g2s(st + kScaleOff + kChunk * 4, p.v_scale + row0, kChunk * 4, bar);
    };

    // Q^T columns in f16: lane (gid, tig) holds dims 32 q + 8 tig .. + 7 of head gid
    uint4 qa[4];
    {
        const uint16_t* qb = reinterpret_cast<const uint16_t*>(p.q) +
                             ((int64_t)s * p.num_q_heads + (int64_t)h * G + gid) * kD;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            uint4 w = gid < G ? __ldg(reinterpret_cast<const uint4*>(qb + 32 * q + 8 * tig))
                              : make_uint4(0, 0, 0, 0);
            qa[q] = make_uint4(bf16x2_to_f16x2(w.x), bf16x2_to_f16x2(w.y), bf16x2_to_f16x2(w.z),
                               bf16x2_to_f16x2(w.w));
        }
    }

#pragma unroll
    for (int i = 0; i < kS; ++i) {
        const int32_t id = __shfl_sync(kFull, id_reg, i & 31);
        if (lane == 0 && i < my_n) issue(i, id);
    }

    float o[8][4];
#pragma unroll
    for (int t = 0; t < 8; ++t) o[t][0] = o[t][1] = o[t][2] = o[t][3] = 0.f;
    float m[2] = {-INFINITY, -INFINITY};   // running maxima of s (for l), heads 2 tig, 2 tig + 1
    float mo[2] = {-INFINITY, -INFINITY};  // running maxima of s + lg2 v_scale (for o)
    float l[2] = {0.f, 0.f};
    const int ta = tile_tok(gid), tb = 8 + tile_tok(gid);  // tokens of tile rows gid, gid + 8
    // K fragment: k-step pair q reads codes 32q + 8tig .. +7 of rows ta and tb:
    // 16-byte unit 2q + (tig >> 1) at (unit ^ (ta & 7)), byte 8 (tig & 1) in it
    uint32_t k_off[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
        k_off[q] = ta * 128 + ((((2 * q) + (tig >> 1)) ^ (ta & 7)) << 4) + 8 * (tig & 1);
    // ldmatrix: matrices 0 / 1 = tokens r / 8 + r of dims 16 mt .. + 7, 2 / 3 the next 8 dims
    const uint32_t v_lane = (((lane >> 3) & 1) * 8 + (lane & 7)) * kVPad + (lane >> 4) * 16;

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
        const unsigned char* vst = kst + kBox;
        const float* ksc = reinterpret_cast<const float*>(kst + kScaleOff);
        const float* vsc = ksc + kChunk;

        // ---- V codes -> f16 buffer (rows outside the mask zeroed: unwritten
        //      slots may hold NaN codes); 8 lanes per row, 16 codes each
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            // token r's codes c*16 .. +15 (swizzled unit), to its tile row
            const int idx = j * 32 + lane, r = idx >> 3, c = idx & 7;
            uint4 w0 = make_uint4(0, 0, 0, 0), w1 = make_uint4(0, 0, 0, 0);
            if ((vmask >> r) & 1u) {
                const uint4 u = lds128(smem_u32(vst) + r * 128 + ((c ^ (r & 7)) << 4));
                w0 = make_uint4(e4m3x2_f16x2(u.x & 0xffffu), e4m3x2_f16x2(u.x >> 16),
                                e4m3x2_f16x2(u.y & 0xffffu), e4m3x2_f16x2(u.y >> 16));
                w1 = make_uint4(e4m3x2_f16x2(u.z & 0xffffu), e4m3x2_f16x2(u.z >> 16),
                                e4m3x2_f16x2(u.w & 0xffffu), e4m3x2_f16x2(u.w >> 16));
            }
            const int tr = (r & 8) | tok_tile(r & 7);
            *reinterpret_cast<uint4*>(vbuf + tr * kVPad + c * 32) = w0;
            *reinterpret_cast<uint4*>(vbuf + tr * kVPad + c * 32 + 16) = w1;
        }

        // ---- S^T = K Q^T: codes -> f16 A fragments, 8 k-steps in two chains
        const uint32_t kb = smem_u32(kst);
        float sc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint2 ua = lds64(kb + k_off[q]);            // token ta, codes 32 q + 8 tig ..
            const uint2 ub = lds64(kb + k_off[q] + 8 * 128);  // token tb (same swizzle key)
            const uint32_t a0 = e4m3x2_f16x2(ua.x & 0xffffu), a1 = e4m3x2_f16x2(ua.x >> 16);
            const uint32_t a2 = e4m3x2_f16x2(ua.y & 0xffffu), a3 = e4m3x2_f16x2(ua.y >> 16);
            const uint32_t b0 = e4m3x2_f16x2(ub.x & 0xffffu), b1 = e4m3x2_f16x2(ub.x >> 16);
            const uint32_t b2 = e4m3x2_f16x2(ub.y & 0xffffu), b3 = e4m3x2_f16x2(ub.y >> 16);
            mma_f16_16816(sc[0], a0, b0, a1, b1, qa[q].x, qa[q].y);
            mma_f16_16816(sc[1], a2, b2, a3, b3, qa[q].z, qa[q].w);
        }
        const bool va = (vmask >> ta) & 1u, vb = (vmask >> tb) & 1u;
        const float ksa = va ? ksc[ta] * p.scale_log2 : 0.f, ksb = vb ? ksc[tb] * p.scale_log2 : 0.f;
        const float lva = va ? lg2_approx(vsc[ta]) : -INFINITY;
        const float lvb = vb ? lg2_approx(vsc[tb]) : -INFINITY;
        // s[token][head] (base-2 logits) for tokens ta, tb and heads 2 tig (+ 1)
        float s2[2][2];
        s2[0][0] = va ? (sc[0][0] + sc[1][0]) * ksa : -INFINITY;
        s2[0][1] = va ? (sc[0][1] + sc[1][1]) * ksa : -INFINITY;
        s2[1][0] = vb ? (sc[0][2] + sc[1][2]) * ksb : -INFINITY;
        s2[1][1] = vb ? (sc[0][3] + sc[1][3]) * ksb : -INFINITY;
        float cm[2] = {fmaxf(s2[0][0], s2[1][0]), fmaxf(s2[0][1], s2[1][1])};
        float co[2] = {fmaxf(s2[0][0] + lva, s2[1][0] + lvb), fmaxf(s2[0][1] + lva, s2[1][1] + lvb)};
#pragma unroll
        for (int off = 4; off <= 16; off <<= 1) {
#pragma unroll
            for (int x = 0; x < 2; ++x) {
                cm[x] = fmaxf(cm[x], __shfl_xor_sync(kFull, cm[x], off));
                co[x] = fmaxf(co[x], __shfl_xor_sync(kFull, co[x], off));
            }
        }
        // lazy rescale of l (by m) and of o (by m'), separately
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            if (cm[x] > m[x] + kRescaleThreshold) {
                l[x] *= ex2(m[x] - cm[x]);
                m[x] = cm[x];
            }
            if (co[x] > mo[x] + kRescaleThreshold) {
                const float corr = ex2(mo[x] - co[x]);
                mo[x] = co[x];
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    o[t][x] *= corr;
                    o[t][x + 2] *= corr;
                }
            }
        }
        __syncwarp();
        float po[2][2];
#pragma unroll
        for (int x = 0; x < 2; ++x) {
            l[x] += (va ? ex2(s2[0][x] - m[x]) : 0.f) + (vb ? ex2(s2[1][x] - m[x]) : 0.f);
            // an all-zero V row (scale 0) contributes nothing; mo is finite
            // whenever some exponent is
            const float ea = s2[0][x] + lva, eb = s2[1][x] + lvb;
            po[0][x] = ea > -INFINITY ? ex2(ea - mo[x]) : 0.f;
            po[1][x] = eb > -INFINITY ? ex2(eb - mo[x]) : 0.f;
        }
        // P^T (with the V scale) in the accumulator layout, f16 hi + lo, transposed
        const uint32_t h0 = pack_f16(po[0][0], po[0][1]);
        const uint32_t h1 = pack_f16(po[1][0], po[1][1]);
        const uint32_t l0 = pack_f16(po[0][0] - f16_lo(h0), po[0][1] - f16_hi(h0));
        const uint32_t l1 = pack_f16(po[1][0] - f16_lo(h1), po[1][1] - f16_hi(h1));
        const uint32_t bh0 = movmatrix_trans(h0), bh1 = movmatrix_trans(h1);
        const uint32_t bl0 = movmatrix_trans(l0), bl1 = movmatrix_trans(l1);

        // ---- O^T += V^T P^T from the f16 buffer
        const uint32_t vaddr = smem_u32(vbuf) + v_lane;
#pragma unroll
        for (int mt = 0; mt < 8; ++mt) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_trans(vaddr + mt * 32, r0, r1, r2, r3);
            mma_f16_16816(o[mt], r0, r2, r1, r3, bh0, bh1);
            mma_f16_16816(o[mt], r0, r2, r1, r3, bl0, bl1);
        }
        __syncwarp();  // every lane is done with the stage and the f16 buffer

        // ---- refill this stage with chunk i + kS
        const int nxt = i + kS;
        if (nxt - id_base >= 32) {
            id_base += 32;
            id_reg = (id_base + lane < my_n) ? table_id(id_base + lane) : -1;
        }
        const int32_t nid = __shfl_sync(kFull, id_reg, (nxt - id_base) & 31);
        if (lane == 0 && nxt < my_n) issue(nxt, nid);
    }
    if (!ok) aborted = 1;
    griddep_launch();

#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        l[0] += __shfl_xor_sync(kFull, l[0], off);
        l[1] += __shfl_xor_sync(kFull, l[1], off);
    }
    // o is in units of 2^m', l of 2^m: bring o to 2^m (no tokens: o is zero)
    float fo[2];
#pragma unroll
    for (int x = 0; x < 2; ++x) fo[x] = mo[x] == -INFINITY ? 0.f : ex2(mo[x] - m[x]);

    // ---- combine the CTA's warps (reusing the ring) and write
    __syncthreads();
    if (aborted) return;
    constexpr int D = kD;
    constexpr int MOFF = G * D, LOFF = G * D + G;
    constexpr int WSTRIDE = G * D + ((2 * G + 3) / 4) * 4;
    static_assert((size_t)kW * WSTRIDE * 4 <= kRing, "combine fits the ring");
    float* cw = reinterpret_cast<float*>(smem);
    float* mine = cw + warp * WSTRIDE;
#pragma unroll
    for (int x = 0; x < 2; ++x) {
        const int g = 2 * tig + x;
        if (g < G) {
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                mine[g * D + 16 * t + gid] = o[t][x] * fo[x];
                mine[g * D + 16 * t + 8 + gid] = o[t][x + 2] * fo[x];
            }
            if (gid == 0) {
                mine[MOFF + g] = m[x];
                mine[LOFF + g] = l[x];
            }
        }
    }
    __syncthreads();
    const int64_t qh0 = (int64_t)s * p.num_q_heads + (int64_t)h * G;
    for (int idx = threadIdx.x; idx < G * D; idx += kW * 32) {
        const int g = idx / D, d = idx - g * D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kW; ++w) M = fmaxf(M, cw[w * WSTRIDE + MOFF + g]);
        float Lsum = 0.f, A = 0.f;
#pragma unroll
        for (int w = 0; w < kW; ++w) {
            const float mw = cw[w * WSTRIDE + MOFF + g];
            const float c = mw == -INFINITY ? 0.f : ex2(mw - M);
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
}

}  // namespace mma8
}  // namespace pa
