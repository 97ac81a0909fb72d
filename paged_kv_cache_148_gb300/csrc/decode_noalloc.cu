// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory when they need to run it.
//
// pa_decode keeps its split-KV partials in a workspace the caller allocates.
// Some callers have no way to do that: a plugin or custom-op host may hand
// the op raw device pointers and no allocator, and a serving process usually
// gives nearly all HBM to the block pool and keeps no allocator headroom.
// This variant runs the same kernels with the same partition plan, with the
// workspace taken from a file-scope device array of kNoAllocScratchBytes.
// The array is part of the library's device image: every GPU that loads the
// library's kernels holds it until the process exits.
//
// Set-up: the first call in a CUDA context (the current device's, made
// current by the caller) looks up the array's device address with
// cudaGetSymbolAddress and caches it under the context's unique id; a later
// call in another context (another device, or the primary context created
// again after cudaDeviceReset) looks it up again.  Make the first call on
// each device before any stream capture.
//
// Every call shares the one array, so calls that overlap on the GPU
// (different streams, no ordering between them) race on it.  Nothing in it
// needs to start at zero: a call that completes without error writes every
// partial it later reads.  After PA_ERR_TIMEOUT (a partition gave up waiting
// for its copies) the merge may read partials left by an earlier call, so
// that output must be discarded.
#include <cuda.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "host_common.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
struct Cached {
    unsigned long long ctx_id;  // cuCtxGetId of the context the address belongs to
    void* ptr;
};
Cached g_scratch[kMaxDevices] = {};

// Unique id of the calling thread's current context (driver entry points,
// found through the runtime so the library needs no link to libcuda).
pa_status current_context_id(unsigned long long* id) {
    static PFN_cuCtxGetCurrent_v4000 get_current = nullptr;
    static PFN_cuCtxGetId_v12000 get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault,
                                             &q) == cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(p);
    });
    if (get_current == nullptr || get_id == nullptr) return PA_ERR_CUDA;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS) return PA_ERR_CUDA;
    if (ctx == nullptr) {
        // no context on this thread yet: cudaSetDevice makes the device's
        // primary context current (it initialises it, allocating nothing)
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaSetDevice(dev);
        if (e != cudaSuccess) {
            pa::record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        if (get_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) return PA_ERR_CUDA;
    }
    return get_id(ctx, id) == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// Device address of g_decode_scratch in the current context (looked up once
// per context).
pa_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        pa::record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    unsigned long long id = 0;
    pa_status st = current_context_id(&id);
    if (st != PA_OK) return st;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch[dev].ptr == nullptr || g_scratch[dev].ctx_id != id) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            pa::record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        g_scratch[dev] = Cached{id, ptr};
    }
    *out = g_scratch[dev].ptr;
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_noalloc(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                                       const int32_t* block_tables, int32_t max_blocks_per_seq,
                                       const int32_t* context_lens, int32_t num_seqs,
                                       int32_t max_context, float scale, int32_t partition_tokens,
                                       float* out, int32_t* d_err, pa_stream_t stream) {
    size_t need = 0;
    pa_status st = pa_decode_workspace_bytes(pool, num_seqs, num_q_heads, max_context,
                                             partition_tokens, &need);
    if (st != PA_OK) return st;
    if (need > kNoAllocScratchBytes) return PA_ERR_UNSUPPORTED;  // beyond the static maximum
    void* ws = nullptr;
    st = scratch_address(&ws);
    if (st != PA_OK) return st;
    return pa_decode(pool, q, num_q_heads, block_tables, max_blocks_per_seq, context_lens,
                     num_seqs, max_context, scale, partition_tokens, out, ws,
                     kNoAllocScratchBytes, d_err, stream);
}
