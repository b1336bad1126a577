// Internal interface between the C-ABI layer (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime_api.h>
#include <stddef.h>
#include <stdint.h>

namespace pa {

// Default split-K partition: 512 tokens, 1024 when the table can address
// kLongContextTokens or more (long rows: half the pieces and merges, and
// rows still have several partitions to balance).
constexpr int kDefaultPartitionTokens = 512;
constexpr int kLongPartitionTokens = 1024;
constexpr long long kLongContextTokens = 4096;
constexpr int kMaxPartitionTokens = 1 << 20;
constexpr int kMaxGroup = 16;  // query heads per kv head (rows of one mma tile)

struct DecodeArgs {
  void* out;
  const void* query;
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;          // num_q_heads / num_kv_heads
  int heads_per_cta;  // kv heads one CTA works on together (4, 2 or 1; divides num_kv_heads)
  int block_shift;    // log2(block_size)
  int max_blocks_per_seq;
  int num_blocks;
  int partition_tokens;
  int max_partitions;  // ceil(max_blocks_per_seq * block_size / partition_tokens)
  float scale_log2;    // scale * log2(e): scores are kept in base-2 units
  int out_f32;         // 1: out is fp32; 0: out has the input element type
  const void* new_key;    // [S, Hkv, d] newest token's K/V rows, or null (plain decode)
  const void* new_value;
  float* ws_out;       // [S, Hq, max_partitions, d] fp32 partial outputs (normalised)
  float* ws_lse;       // [S, Hq, max_partitions] fp32 base-2 log-sum-exp
  int* ws_count;       // [S * Hkv] arrival counters (zero between calls)
  unsigned long long* ws_claim;  // dynamic partitions claimed so far (zero between calls), or null
  unsigned* ws_done;             // CTAs finished (zero between calls)
  int dyn_percent;     // share (%) of each row's partitions handed out at run time
  unsigned long long* bad;  // device counter of rejected indices
};

struct PrefillArgs {
  void* out;                  // [total_q, Hq, d]
  const void* query;          // [total_q, Hq, d]
  const void* key_cache;
  const void* value_cache;
  const int32_t* block_tables;
  const int32_t* seq_lens;
  const int32_t* query_start;  // [S + 1]
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int block_shift;
  int max_blocks_per_seq;
  int num_blocks;
  float scale_log2;
  int out_f32;
  unsigned long long* bad;
  unsigned long long* timeouts;  // bounded waits that gave up (tensor-core kernel)
  int stall_for_test;  // 1: the product thread waits on a barrier nothing signals
  void* v16;           // bf16 caches: fp16 copy of the value rows [S * MB * B, Hkv, d], or null
};

// Bytes of the fp16 copy of the value rows the bf16 prefill can use (0 when
// it does not apply: fp16 caches, or a copy of 2^31 slots or more).
size_t prefill_v16_bytes(int num_seqs, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                         int block_size, bool bf16);

// Tensor-core (tcgen05) prefill: block sizes 1..64 (TMA block copies from 8
// up, 16-byte row copies below), fewer than 2^31 slots.
bool prefill_tc_supported(int block_size, long long num_slots);
cudaError_t launch_prefill_tc(const PrefillArgs& a, int head_dim, bool bf16, int max_query_len,
                              cudaStream_t stream);

// Records `msg` as the calling thread's last error and returns `code`;
// clear_error() empties it (entry points call it first).
int set_error(int code, const char* msg);
void clear_error();

// Workspace carve-up shared by pa_decode_workspace_bytes and pa_decode.
// Layout: a 256-byte header (the dynamic-partition claim counter and the
// count of finished CTAs), the per-(sequence, kv head) arrival counters, then
// the fp32 partial results.
struct WorkspaceLayout {
  size_t count_off, lse_off, out_off, total;
};
constexpr size_t kWorkspaceHeader = 256;
// Percentage of each row's partitions the decode kernel hands out at run time.
constexpr int kDynamicPercent = 8;
WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_dim, int max_partitions);

// Scheduling of the persistent decode kernel: a partition weighs its tokens
// plus kUnitCost; a CTA keeps at most kMaxSegments segment records at a time.
constexpr int kUnitCost = 64;
constexpr int kMaxSegments = 64;

// Launchers: return a cudaError_t from the launch (cudaSuccess on success).
// `num_sms` is the device's multiprocessor count (the persistent grid is a
// multiple of it).
cudaError_t launch_decode(const DecodeArgs& a, int head_dim, bool bf16, int num_sms,
                          cudaStream_t stream);

cudaError_t launch_copy_blocks(void* key_cache, void* value_cache, const int32_t* src,
                               const int32_t* dst, int num_copies, long long block_bytes,
                               int num_blocks, unsigned long long* bad, cudaStream_t stream);

cudaError_t launch_reshape_and_cache(const void* key, const void* value, void* key_cache,
                                     void* value_cache, const int64_t* slot_mapping,
                                     int num_tokens, int row_bytes, long long num_slots,
                                     unsigned long long* bad, cudaStream_t stream);

}  // namespace pa
