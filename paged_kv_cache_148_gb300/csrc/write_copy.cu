// pa_write_kv and pa_copy_blocks: the scatter write of new K/V rows through
// slot_mapping (P1 §4.1 of "03｜PagedAttention 与 KV Cache 内存系统") and the
// whole-block copy used for copy-on-write of a shared tail block (P1 §5;
// "KV Cache：容量、布局与生命周期", section 引用计数与尾块 COW).
//
// Both are pure HBM copies.  Each thread moves 16-byte vectors, consecutive
// threads touch consecutive vectors of one row or page, so every warp access
// is a fully used 512-byte span on both the read and the write side.  FP8
// pages are written by a separate kernel that quantises each bf16 row (one
// warp per row) and stores its codes and scale; the copy moves the scales
// along with the code pages.
#include "common.cuh"
#include "host_common.h"

namespace pa {

// A thread moves U consecutive 16-byte vectors of one (token, kv-head) row of
// K and of V (U divides the row's vectors), all loads issued before the stores.
template <int U>
__global__ void __launch_bounds__(256) write_kv_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const uint4* __restrict__ k_new,
    const uint4* __restrict__ v_new, const int64_t* __restrict__ slot_mapping, int64_t total_vecs,
    int32_t row_vecs, int32_t num_kv_heads, int32_t block_size, int64_t num_slots,
    int32_t* d_err) {
    griddep_wait();
    griddep_launch();  // the attention kernel that follows may start launching
    const int64_t per_token = (int64_t)row_vecs * num_kv_heads;
    for (int64_t i = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) * U; i < total_vecs;
         i += (int64_t)gridDim.x * blockDim.x * U) {
        const int64_t t = i / per_token;
        const int64_t r = i - t * per_token;          // h * row_vecs + vec
        const int64_t slot = __ldg(slot_mapping + t);
        uint4 kx[U], vx[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            kx[u] = __ldg(k_new + i + u);
            vx[u] = __ldg(v_new + i + u);
        }
        if (slot < 0 || slot >= num_slots) {
            if (r == 0) set_error(d_err, PA_ERR_OUT_OF_RANGE);
            continue;
        }
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        const int64_t h = r / row_vecs, vec = r - h * row_vecs;
        const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * row_vecs + vec;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            k_pool[dst + u] = kx[u];
            v_pool[dst + u] = vx[u];
        }
    }
}

// FP8 pages: one warp per (token, kv-head, K or V) row of D = 128 bf16 inputs;
// lane l quantises elements 4l .. 4l+3.  amax over the row by shuffles, scale =
// amax / 448 and inv = 448 / amax with IEEE division, codes = E4M3(x * inv)
// rounded to nearest even and saturated (cvt ... satfinite).
PA_DEVICE uint32_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

__global__ void __launch_bounds__(256) write_kv_fp8_kernel(
    uint8_t* __restrict__ k_pool, uint8_t* __restrict__ v_pool, float* __restrict__ k_scale,
    float* __restrict__ v_scale, const uint2* __restrict__ k_new, const uint2* __restrict__ v_new,
    const int64_t* __restrict__ slot_mapping, int64_t rows, int32_t num_kv_heads,
    int32_t block_size, int64_t num_slots, int32_t* d_err) {
    griddep_wait();
    griddep_launch();
    const int lane = threadIdx.x & 31;
    const int64_t step = ((int64_t)gridDim.x * blockDim.x) >> 5;
    for (int64_t r = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5; r < rows; r += step) {
        const int which = (int)(r & 1);             // 0: K, 1: V
        const int64_t th = r >> 1;                  // token * H_kv + head
        const int64_t t = th / num_kv_heads;
        const int64_t h = th - t * num_kv_heads;
        const int64_t slot = __ldg(slot_mapping + t);
        if (slot < 0 || slot >= num_slots) {
            if (lane == 0 && which == 0 && h == 0) set_error(d_err, PA_ERR_OUT_OF_RANGE);
            continue;
        }
        const uint2 x = __ldg((which ? v_new : k_new) + th * 32 + lane);
        const float f0 = bf16_lo(x.x), f1 = bf16_hi(x.x), f2 = bf16_lo(x.y), f3 = bf16_hi(x.y);
        float a = fmaxf(fmaxf(fabsf(f0), fabsf(f1)), fmaxf(fabsf(f2), fabsf(f3)));
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, off));
        const float scale = __fdiv_rn(a, 448.f);
        const float inv = a > 0.f ? __fdiv_rn(448.f, a) : 0.f;
        const uint32_t codes = e4m3x2(__fmul_rn(f0, inv), __fmul_rn(f1, inv)) |
                               (e4m3x2(__fmul_rn(f2, inv), __fmul_rn(f3, inv)) << 16);
        const int64_t blk = slot / block_size, off = slot - blk * block_size;
        const int64_t row = (blk * num_kv_heads + h) * block_size + off;
        reinterpret_cast<uint32_t*>((which ? v_pool : k_pool) + row * 128)[lane] = codes;
        if (lane == 0) (which ? v_scale : k_scale)[row] = scale;
    }
}

// grid.x = pair, grid.y = slices of the page; each thread copies kCopyU
// vectors of K and kCopyU of V per round (stride: the slice width), all eight
// loads issued before the stores.
constexpr int kCopyU = 4;

__global__ void __launch_bounds__(256) copy_blocks_kernel(
    uint4* __restrict__ k_pool, uint4* __restrict__ v_pool, const int32_t* __restrict__ src,
    const int32_t* __restrict__ dst, int64_t page_vecs, int32_t num_blocks, float* k_scale,
    float* v_scale, int32_t scales_per_page, int32_t* d_err) {
    const int32_t s = __ldg(src + blockIdx.x), d = __ldg(dst + blockIdx.x);
    if (s < 0 || s >= num_blocks || d < 0 || d >= num_blocks) {
        if (blockIdx.y == 0 && threadIdx.x == 0) set_error(d_err, PA_ERR_OUT_OF_RANGE);
        return;
    }
    if (blockIdx.y == 0) {  // FP8 pages: the block's row scales travel with it
        for (int i = threadIdx.x; i < scales_per_page; i += blockDim.x) {
            k_scale[(int64_t)d * scales_per_page + i] = k_scale[(int64_t)s * scales_per_page + i];
            v_scale[(int64_t)d * scales_per_page + i] = v_scale[(int64_t)s * scales_per_page + i];
        }
    }
    const uint4* ks = k_pool + (int64_t)s * page_vecs;
    const uint4* vs = v_pool + (int64_t)s * page_vecs;
    uint4* kd = k_pool + (int64_t)d * page_vecs;
    uint4* vd = v_pool + (int64_t)d * page_vecs;
    const int64_t step = (int64_t)gridDim.y * blockDim.x;
    for (int64_t v = (int64_t)blockIdx.y * blockDim.x + threadIdx.x; v < page_vecs;
         v += kCopyU * step) {
        uint4 a[kCopyU], c[kCopyU];
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const int64_t w = v + u * step;
            if (w < page_vecs) {
                a[u] = ks[w];
                c[u] = vs[w];
            }
        }
#pragma unroll
        for (int u = 0; u < kCopyU; ++u) {
            const int64_t w = v + u * step;
            if (w < page_vecs) {
                kd[w] = a[u];
                vd[w] = c[u];
            }
        }
    }
}

}  // namespace pa

using namespace pa;

extern "C" pa_status pa_write_kv(const pa_kv_pool* pool, const void* k_new, const void* v_new,
                                 const int64_t* slot_mapping, int32_t num_tokens, int32_t* d_err,
                                 pa_stream_t stream) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (num_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!k_new || !v_new || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (pool->dtype == PA_DTYPE_FP8_E4M3) {  // bf16 rows in, E4M3 rows and scales out
        if (pool->head_dim != 128) return PA_ERR_UNSUPPORTED;
        if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(pool->k_pool) ||
            !aligned16(pool->v_pool) || !aligned16(pool->k_scale) || !aligned16(pool->v_scale))
            return PA_ERR_INVALID_ARG;
        const int64_t rows = (int64_t)num_tokens * pool->num_kv_heads * 2;
        int64_t blocks = (rows * 32 + 255) / 256;
        if (blocks > 1048576) blocks = 1048576;
        cudaError_t e = launch_pdl(
            write_kv_fp8_kernel, dim3((unsigned)blocks), dim3(256), 0, (cudaStream_t)stream,
            (uint8_t*)pool->k_pool, (uint8_t*)pool->v_pool, (float*)pool->k_scale,
            (float*)pool->v_scale, (const uint2*)k_new, (const uint2*)v_new, slot_mapping, rows,
            pool->num_kv_heads, pool->block_size, (int64_t)pool->num_blocks * pool->block_size,
            d_err);
        if (e != cudaSuccess) {
            record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        return launch_status();
    }
    const int64_t row_bytes = (int64_t)pool->head_dim * dtype_bytes(pool->dtype);
    if (row_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(pool->k_pool) ||
        !aligned16(pool->v_pool))
        return PA_ERR_INVALID_ARG;
    const int32_t row_vecs = (int32_t)(row_bytes / 16);
    const int64_t total = (int64_t)num_tokens * pool->num_kv_heads * row_vecs;
    const int threads = 256;
    const int U = row_vecs % 4 == 0 ? 4 : 1;  // vectors per thread, within one row
    int64_t blocks = (total / U + threads - 1) / threads;
    if (blocks > 1048576) blocks = 1048576;
    // dependent launch: the kernel waits (griddep_wait) for the previous kernel
    // in the stream before it writes, but its launch overlaps that kernel's tail
    cudaError_t e = launch_pdl(
        U == 4 ? write_kv_kernel<4> : write_kv_kernel<1>, dim3((unsigned)blocks), dim3(threads), 0,
        (cudaStream_t)stream,
        (uint4*)pool->k_pool, (uint4*)pool->v_pool, (const uint4*)k_new, (const uint4*)v_new,
        slot_mapping, total, row_vecs, pool->num_kv_heads, pool->block_size,
        (int64_t)pool->num_blocks * pool->block_size, d_err);
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return launch_status();
}

extern "C" pa_status pa_copy_blocks(const pa_kv_pool* pool, const int32_t* src,
                                    const int32_t* dst, int32_t n, int32_t* d_err,
                                    pa_stream_t stream) {
    pa_status st = check_pool(pool);
    if (st != PA_OK) return st;
    if (n < 0) return PA_ERR_INVALID_ARG;
    if (n == 0) return PA_OK;
    if (!src || !dst) return PA_ERR_INVALID_ARG;
    const int64_t page_bytes = (int64_t)pool->num_kv_heads * pool->block_size * pool->head_dim *
                               dtype_bytes(pool->dtype);
    if (page_bytes % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (!aligned16(pool->k_pool) || !aligned16(pool->v_pool)) return PA_ERR_INVALID_ARG;
    const int64_t page_vecs = page_bytes / 16;
    const int threads = 256;
    int64_t slices = (page_vecs + threads * kCopyU - 1) / (threads * kCopyU);
    if (slices < 1) slices = 1;
    if (slices > 65535) slices = 65535;
    dim3 grid((unsigned)n, (unsigned)slices);
    const bool fp8 = pool->dtype == PA_DTYPE_FP8_E4M3;
    copy_blocks_kernel<<<grid, threads, 0, (cudaStream_t)stream>>>(
        (uint4*)pool->k_pool, (uint4*)pool->v_pool, src, dst, page_vecs, pool->num_blocks,
        fp8 ? (float*)pool->k_scale : nullptr, fp8 ? (float*)pool->v_scale : nullptr,
        fp8 ? pool->num_kv_heads * pool->block_size : 0, d_err);
    return launch_status();
}
