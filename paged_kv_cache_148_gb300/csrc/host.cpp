// Host half of libpagedkv.so: status strings, slot arithmetic and the block
// allocator (refcounts, free list, fork, copy-on-write tail).
//
// Slot arithmetic follows "KV Cache：容量、布局与生命周期" (section Page-table
// 寻址) and "03｜PagedAttention 与 KV Cache 内存系统" §3.  The allocator follows
// the same page's sections 生命周期与所有权 and 引用计数与尾块 COW, and §5 of the
// latter (a freed block without a prefix hash is the next one reused, so the
// free list is a stack).
#include <algorithm>
#include <cstring>
#include <mutex>
#include <new>
#include <string>
#include <vector>

#include <cudaTypedefs.h>

#include "host_common.h"

namespace pa {

static thread_local std::string g_last_cuda_error = "no CUDA error recorded";

void record_cuda_error(cudaError_t e) {
    g_last_cuda_error = std::string(cudaGetErrorName(e)) + ": " + cudaGetErrorString(e);
}

int device_sm_count() {
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 152;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0)
            n = 152;
        cached[dev] = n;
    }
    return cached[dev];
}

static bool encode_map_sw128(CUtensorMap* map, CUtensorMapDataType type, const void* base,
                             int rank, const uint64_t* dims, const uint64_t* strides,
                             const uint32_t* box) {
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
    if (fn == nullptr || rank < 1 || rank > 3) return false;
    cuuint64_t d[3];
    cuuint64_t st[2];
    cuuint32_t bx[3];
    const cuuint32_t es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        d[i] = dims[i];
        bx[i] = box[i];
        if (i > 0) st[i - 1] = strides[i - 1];
    }
    CUresult r = fn(map, type, (cuuint32_t)rank, const_cast<void*>(base),
                    d, st, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_bf16_map_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                           const uint64_t* strides, const uint32_t* box) {
    return encode_map_sw128(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, base, rank, dims, strides, box);
}

bool encode_u8_map_sw128(CUtensorMap* map, const void* base, int rank, const uint64_t* dims,
                         const uint64_t* strides, const uint32_t* box) {
    return encode_map_sw128(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, base, rank, dims, strides, box);
}

// Refcounted pool of block ids with a LIFO free list.
struct Allocator {
    std::vector<int32_t> refcount;
    std::vector<int32_t> free_list;  // pop from the back
};

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_str(int32_t s) {
    switch (s) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
        case PA_ERR_OUT_OF_RANGE: return "PA_ERR_OUT_OF_RANGE: logical block not allocated or id/slot outside the pool";
        case PA_ERR_NEGATIVE_BLOCK: return "PA_ERR_NEGATIVE_BLOCK: negative physical block id";
        case PA_ERR_NO_FREE_BLOCK: return "PA_ERR_NO_FREE_BLOCK: free list is empty";
        case PA_ERR_REFCOUNT: return "PA_ERR_REFCOUNT: release of a block nobody holds";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: shape or dtype not implemented";
        case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime error";
        case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: bounded device wait ran out";
        default: return "unknown pa_status";
    }
}

const char* pa_last_cuda_error(void) { return g_last_cuda_error.c_str(); }

int32_t pa_abi_version(void) { return 2; }

pa_status pa_page_size_bytes(const pa_kv_pool* pool, int64_t* bytes) {
    if (!pool || !bytes) return PA_ERR_INVALID_ARG;
    if (pool->block_size <= 0 || pool->num_kv_heads <= 0 || pool->head_dim <= 0)
        return PA_ERR_INVALID_ARG;
    if (pool->dtype != PA_DTYPE_F32 && pool->dtype != PA_DTYPE_BF16 &&
        pool->dtype != PA_DTYPE_FP8_E4M3)
        return PA_ERR_INVALID_ARG;
    *bytes = 2ll * pool->block_size * pool->num_kv_heads * pool->head_dim *
             dtype_bytes(pool->dtype);
    if (pool->dtype == PA_DTYPE_FP8_E4M3) *bytes += 2ll * pool->block_size * pool->num_kv_heads * 4;
    return PA_OK;
}

pa_status pa_physical_slot(const int32_t* table, int32_t n_entries, int32_t block_size,
                           int64_t pos, int64_t* slot) {
    if (block_size <= 0 || pos < 0 || !slot || n_entries < 0) return PA_ERR_INVALID_ARG;
    const int64_t logical = pos / block_size;
    const int64_t offset = pos - logical * block_size;
    if (logical >= n_entries) return PA_ERR_OUT_OF_RANGE;
    if (!table) return PA_ERR_INVALID_ARG;
    const int64_t phys = table[logical];
    if (phys < 0) return PA_ERR_NEGATIVE_BLOCK;
    *slot = phys * block_size + offset;
    return PA_OK;
}

pa_status pa_slot_mapping(const int32_t* table, int32_t n_entries, int32_t block_size,
                          const int64_t* positions, int64_t count, int64_t* slots) {
    if (count < 0 || (count > 0 && (!positions || !slots))) return PA_ERR_INVALID_ARG;
    for (int64_t i = 0; i < count; ++i) {
        pa_status st = pa_physical_slot(table, n_entries, block_size, positions[i], slots + i);
        if (st != PA_OK) return st;
    }
    return PA_OK;
}

pa_status pa_alloc_create(int32_t num_blocks, const int32_t* free_order, void** handle) {
    if (num_blocks <= 0 || !handle) return PA_ERR_INVALID_ARG;
    Allocator* a = new (std::nothrow) Allocator();
    if (!a) return PA_ERR_INVALID_ARG;
    a->refcount.assign((size_t)num_blocks, 0);
    a->free_list.resize((size_t)num_blocks);
    if (free_order) {
        std::vector<char> seen((size_t)num_blocks, 0);
        for (int32_t i = 0; i < num_blocks; ++i) {
            const int32_t b = free_order[i];
            if (b < 0 || b >= num_blocks || seen[(size_t)b]) {
                delete a;
                return PA_ERR_INVALID_ARG;  // not a permutation
            }
            seen[(size_t)b] = 1;
            a->free_list[(size_t)i] = b;
        }
    } else {
        for (int32_t i = 0; i < num_blocks; ++i) a->free_list[(size_t)i] = i;
    }
    *handle = a;
    return PA_OK;
}

void pa_alloc_destroy(void* handle) { delete static_cast<Allocator*>(handle); }

pa_status pa_alloc_append(void* handle, int32_t* table, int32_t* n, int32_t capacity) {
    Allocator* a = static_cast<Allocator*>(handle);
    if (!a || !table || !n || *n < 0 || *n >= capacity) return PA_ERR_INVALID_ARG;
    if (a->free_list.empty()) return PA_ERR_NO_FREE_BLOCK;
    const int32_t b = a->free_list.back();
    a->free_list.pop_back();
    a->refcount[(size_t)b] = 1;
    table[(*n)++] = b;
    return PA_OK;
}

pa_status pa_alloc_fork(void* handle, const int32_t* table, int32_t n) {
    Allocator* a = static_cast<Allocator*>(handle);
    if (!a || n < 0 || (n > 0 && !table)) return PA_ERR_INVALID_ARG;
    const int32_t nb = (int32_t)a->refcount.size();
    for (int32_t i = 0; i < n; ++i)
        if (table[i] < 0 || table[i] >= nb || a->refcount[(size_t)table[i]] <= 0)
            return PA_ERR_OUT_OF_RANGE;  // only held blocks can be shared
    for (int32_t i = 0; i < n; ++i) a->refcount[(size_t)table[i]] += 1;
    return PA_OK;
}

pa_status pa_alloc_writable_tail(void* handle, int32_t* table, int32_t* n, int32_t capacity,
                                 int64_t logical_length, int32_t block_size, int32_t* block,
                                 int32_t* offset, int32_t* cow_src) {
    Allocator* a = static_cast<Allocator*>(handle);
    if (!a || !table || !n || !block || !offset || !cow_src) return PA_ERR_INVALID_ARG;
    if (block_size <= 0 || logical_length < 0 || *n < 0) return PA_ERR_INVALID_ARG;
    const int64_t logical = logical_length / block_size;
    const int32_t off = (int32_t)(logical_length - logical * block_size);
    int32_t cow = -1;
    if (off == 0) {
        if (logical != *n) return PA_ERR_INVALID_ARG;
        pa_status st = pa_alloc_append(handle, table, n, capacity);
        if (st != PA_OK) return st;
    } else {
        if (logical >= *n) return PA_ERR_OUT_OF_RANGE;
        const int32_t cur = table[logical];
        if (cur < 0 || cur >= (int32_t)a->refcount.size()) return PA_ERR_OUT_OF_RANGE;
        if (a->refcount[(size_t)cur] > 1) {
            if (a->free_list.empty()) return PA_ERR_NO_FREE_BLOCK;
            const int32_t fresh = a->free_list.back();
            a->free_list.pop_back();
            a->refcount[(size_t)cur] -= 1;
            a->refcount[(size_t)fresh] = 1;
            table[logical] = fresh;
            cow = cur;
        }
    }
    *block = table[logical];
    *offset = off;
    *cow_src = cow;
    return PA_OK;
}

pa_status pa_alloc_reserve(void* handle, int32_t* table, int32_t* n, int32_t capacity,
                           int64_t logical_length, int64_t count, int32_t block_size,
                           int64_t* slots, int32_t* cow_src, int32_t* cow_dst,
                           int32_t cow_capacity, int32_t* n_cow) {
    if (count < 0 || (count > 0 && !slots) || !n_cow || *n_cow < 0) return PA_ERR_INVALID_ARG;
    for (int64_t i = 0; i < count; ++i) {
        int32_t blk, off, cow;
        pa_status st = pa_alloc_writable_tail(handle, table, n, capacity, logical_length + i,
                                              block_size, &blk, &off, &cow);
        if (st != PA_OK) return st;
        if (cow >= 0) {
            if (!cow_src || !cow_dst || *n_cow >= cow_capacity) return PA_ERR_INVALID_ARG;
            cow_src[*n_cow] = cow;
            cow_dst[*n_cow] = blk;
            *n_cow += 1;
        }
        slots[i] = (int64_t)blk * block_size + off;
    }
    return PA_OK;
}

pa_status pa_alloc_release(void* handle, const int32_t* table, int32_t n) {
    Allocator* a = static_cast<Allocator*>(handle);
    if (!a || n < 0 || (n > 0 && !table)) return PA_ERR_INVALID_ARG;
    const int32_t nb = (int32_t)a->refcount.size();
    // validate first so a failed release changes nothing; an id listed k
    // times needs at least k holders
    std::vector<int32_t> ids(table, table + n);
    std::sort(ids.begin(), ids.end());
    for (int32_t i = 0; i < n;) {
        const int32_t b = ids[(size_t)i];
        if (b < 0 || b >= nb) return PA_ERR_OUT_OF_RANGE;
        int32_t j = i;
        while (j < n && ids[(size_t)j] == b) ++j;
        if (a->refcount[(size_t)b] < j - i) return PA_ERR_REFCOUNT;
        i = j;
    }
    for (int32_t i = 0; i < n; ++i) {
        const int32_t b = table[i];
        if (--a->refcount[(size_t)b] == 0) a->free_list.push_back(b);
    }
    return PA_OK;
}

int32_t pa_alloc_refcount(void* handle, int32_t block) {
    Allocator* a = static_cast<Allocator*>(handle);
    if (!a || block < 0 || block >= (int32_t)a->refcount.size()) return -1;
    return a->refcount[(size_t)block];
}

int32_t pa_alloc_num_free(void* handle) {
    Allocator* a = static_cast<Allocator*>(handle);
    return a ? (int32_t)a->free_list.size() : -1;
}

}  // extern "C"
