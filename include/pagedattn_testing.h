/*
 * pagedattn_testing.h -- test hooks of libpagedattn.so. Not for production
 * use: these entry points exist so that tests can drive paths that correct
 * operation never reaches. Same conventions as pagedattn.h.
 */
#ifndef PAGEDATTN_TESTING_H_
#define PAGEDATTN_TESTING_H_

#include "pagedattn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * pa_prefill with every CTA's product-issuing thread first waiting on a
 * shared-memory barrier that nothing ever signals. That wait gives up after
 * its limit (about one second), so no product is issued; the warps waiting on
 * products then give up in turn, every CTA winds down (its copies in flight
 * land and its tensor memory is freed) and the launch ends. Each wait that
 * gave up is counted by pa_wait_timeout_count; `out` is left unwritten.
 * Arguments, checks and errors as for pa_prefill. It exercises the bounded
 * waits' give-up path without any fault or hang.
 */
int pa_testing_prefill_stalled(void* out, const void* query, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               const int32_t* seq_lens, const int32_t* query_start,
                               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                               int block_size, float scale, int max_blocks_per_seq,
                               int num_blocks, int max_query_len, pa_dtype dtype,
                               pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
                               cudaStream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* PAGEDATTN_TESTING_H_ */
