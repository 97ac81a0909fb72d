// Host-side helpers shared by the entry points of libpagedkv.so.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/pagedkv.h"

namespace pa {

// Last CUDA error text seen by this library on the calling thread.
void record_cuda_error(cudaError_t e);

inline int32_t dtype_bytes(int32_t dtype) {
    return dtype == PA_DTYPE_F32 ? 4 : dtype == PA_DTYPE_FP8_E4M3 ? 1 : 2;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

inline bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

inline int ilog2(int64_t x) {
    int l = 0;
    while ((int64_t(1) << (l + 1)) <= x) ++l;
    return l;
}

inline pa_status check_pool(const pa_kv_pool* p) {
    if (p == nullptr || p->k_pool == nullptr || p->v_pool == nullptr) return PA_ERR_INVALID_ARG;
    if (p->num_blocks <= 0 || p->block_size <= 0 || p->num_kv_heads <= 0 || p->head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (p->dtype != PA_DTYPE_F32 && p->dtype != PA_DTYPE_BF16 && p->dtype != PA_DTYPE_FP8_E4M3)
        return PA_ERR_INVALID_ARG;
    if (p->dtype == PA_DTYPE_FP8_E4M3 && (p->k_scale == nullptr || p->v_scale == nullptr))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

// Status of the launch just made (cudaGetLastError).
inline pa_status launch_status() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    return PA_OK;
}

// Streaming multiprocessors of the current device (cached per device).
int device_sm_count();

// Tiled TMA descriptor of a bf16 tensor of rank 2 or 3 with the 128-byte
// swizzle (dims innermost first, strides in bytes for dims 1.., box in
// elements), encoded through the driver's cuTensorMapEncodeTiled.  false if
// the driver entry point is missing or refuses the description.
bool encode_bf16_map_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides, const uint32_t* box);
// The same for byte elements (FP8 codes).
bool encode_u8_map_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box);

// Launch with programmatic stream serialization (the kernel must call
// griddep_wait() before touching memory its predecessor may write).
template <typename Kern, typename... Args>
inline cudaError_t launch_pdl(Kern kern, dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace pa
