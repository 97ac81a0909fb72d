// pa_prefill: paged chunked-prefill attention (tensor-core kernel pending).
#include "common.cuh"
#include "host_common.h"

extern "C" pa_status pa_prefill(const pa_kv_pool* pool, const void* q, int32_t num_q_heads,
                                const int32_t* cu_seqlens_q, const int32_t* context_lens,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                int32_t num_seqs, int32_t max_q_len, int32_t max_context,
                                float scale, int32_t causal, float* out, int32_t* d_err,
                                pa_stream_t stream) {
    (void)pool; (void)q; (void)num_q_heads; (void)cu_seqlens_q; (void)context_lens;
    (void)block_tables; (void)max_blocks_per_seq; (void)num_seqs; (void)max_q_len;
    (void)max_context; (void)scale; (void)causal; (void)out; (void)d_err; (void)stream;
    return PA_ERR_UNSUPPORTED;
}
