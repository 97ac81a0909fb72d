// pa_decode_noalloc: paged decode for callers that cannot allocate device
// memory when they need to run it.
//
// pa_decode keeps its split-KV partials in a workspace the caller allocates.
// Some callers have no way to do that: code recorded into a CUDA graph must
// not call cudaMalloc while the capture is open; a plugin or custom-op host
// may hand the op raw pointers and no allocator; a serving process usually
// gives nearly all HBM to the block pool and keeps no allocator headroom.
// This variant runs the same kernels, with the workspace taken from a
// file-scope device array of kNoAllocScratchBytes.  The array is part of the
// library's device image: every GPU that loads the library holds it until
// the process exits.
//
// Set-up: the first call on a device (with that device current) looks up the
// array's device address with cudaGetSymbolAddress and caches it; make that
// first call before any stream capture.  Every call shares the one array, so
// calls that overlap on the GPU (different streams, no ordering between them)
// race on it.  Nothing in it needs to start at zero: each call writes every
// partial it later reads.
#include <mutex>

#include "host_common.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;  // 16 MiB per device
static __device__ __align__(256) unsigned char g_decode_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device (looked up once).
pa_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        pa::record_cuda_error(e);
        return PA_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_decode_scratch);
        if (e != cudaSuccess || ptr == nullptr) {
            pa::record_cuda_error(e);
            return PA_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    }
    *out = g_scratch_ptr[dev];
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
