// C-ABI layer of libpagedattn.so: argument checks, workspace carve-up,
// dispatch to the kernels, and error reporting. Declarations and the
// contract of every entry point are in include/pagedattn.h.
#include <cuda_runtime.h>
#include <math.h>
#include <stdarg.h>
#include <stdio.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"
#include "pagedattn.h"
#include "pagedattn_testing.h"

// Share (%) of every row's partitions that the decode kernel hands out at run
// time, for 512-token partitions, scaled with the partition length (0: the
// whole split is static).
#ifndef PA_DECODE_DYNAMIC_PERCENT
#define PA_DECODE_DYNAMIC_PERCENT pa::kDynamicPercent
#endif

namespace {

thread_local std::string g_error;

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof(buf), fmt, ap);
  va_end(ap);
  g_error = buf;
  return code;
}

int cuda_fail(cudaError_t e, const char* what) {
  return fail(PA_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorString(e), cudaGetErrorName(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

int log2_pow2(int b) {  // -1 unless b is a power of two in [1, 64]
  for (int k = 0; k <= 6; ++k)
    if (b == (1 << k)) return k;
  return -1;
}

// Device-resident counters: out-of-range indices the kernels skipped, and
// bounded waits (tensor-core prefill) that gave up.
__device__ unsigned long long g_bad_index_count;
__device__ unsigned long long g_wait_timeout_count;

constexpr int kMaxDevices = 64;
std::atomic<unsigned long long*> g_bad_ptr[kMaxDevices];
std::atomic<unsigned long long*> g_timeout_ptr[kMaxDevices];
std::atomic<int> g_num_sms[kMaxDevices];

int num_sms(int* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device index %d", dev);
  int n = g_num_sms[dev].load(std::memory_order_acquire);
  if (n <= 0) {
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceGetAttribute(multiprocessor count)");
    g_num_sms[dev].store(n, std::memory_order_release);
  }
  *out = n;
  return PA_OK;
}

// Device address of one of the two counters on the current device (cached).
int counter(bool timeouts, unsigned long long** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_fail(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PA_ERR_UNSUPPORTED, "device index %d", dev);
  std::atomic<unsigned long long*>& slot = timeouts ? g_timeout_ptr[dev] : g_bad_ptr[dev];
  unsigned long long* p = slot.load(std::memory_order_acquire);
  if (p == nullptr) {
    e = timeouts ? cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_wait_timeout_count)
                 : cudaGetSymbolAddress(reinterpret_cast<void**>(&p), g_bad_index_count);
    if (e != cudaSuccess) return cuda_fail(e, "cudaGetSymbolAddress(counter)");
    slot.store(p, std::memory_order_release);
  }
  *out = p;
  return PA_OK;
}

int bad_counter(unsigned long long** out) { return counter(false, out); }

int read_counter(bool timeouts, unsigned long long* count, int clear) {
  if (count == nullptr) return fail(PA_ERR_INVALID, "count is NULL");
  unsigned long long* p = nullptr;
  int rc = counter(timeouts, &p);
  if (rc != PA_OK) return rc;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_fail(e, "cudaDeviceSynchronize");
  e = cudaMemcpy(count, p, sizeof(*count), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return cuda_fail(e, "cudaMemcpy(counter)");
  if (clear) {
    e = cudaMemset(p, 0, sizeof(*p));
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemset(counter)");
  }
  return PA_OK;
}

int check_dtype(pa_dtype dtype) {
  if (dtype != PA_FLOAT16 && dtype != PA_BFLOAT16)
    return fail(PA_ERR_INVALID, "dtype %d is neither PA_FLOAT16 nor PA_BFLOAT16", (int)dtype);
  return PA_OK;
}

int resolve_partition(int partition_tokens, int block_size, int max_blocks_per_seq, int* pt) {
  int p = partition_tokens;
  if (p == 0)
    p = static_cast<long long>(max_blocks_per_seq) * block_size >= pa::kLongContextTokens
            ? pa::kLongPartitionTokens
            : pa::kDefaultPartitionTokens;
  if (p < 0) return fail(PA_ERR_INVALID, "partition_tokens %d < 0", partition_tokens);
  if (p % 16 != 0 || p % block_size != 0)
    return fail(PA_ERR_INVALID, "partition_tokens %d must be a multiple of 16 and of block_size %d",
                p, block_size);
  if (p > pa::kMaxPartitionTokens)
    return fail(PA_ERR_UNSUPPORTED, "partition_tokens %d > %d", p, pa::kMaxPartitionTokens);
  *pt = p;
  return PA_OK;
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Split-K workspaces: how many leading bytes of each are known to be zero.
// Every pa_decode leaves the arrival counters it used at zero and writes fp32
// partial results from lse_off on. A later call whose counters reach past the
// known-zero prefix (more rows, or after a call whose partial results started
// earlier) would find partial-result bytes there, so it clears its counter
// region on the stream first. Kept per workspace address, most recent last; an
// address not in the list counts as unknown and is cleared once.
struct WsZero {
  const void* ptr;
  size_t zero_prefix;
};
std::mutex g_ws_mu;
std::vector<WsZero> g_ws_zero;
constexpr size_t kWsRecords = 64;

// Clears [0, lse_off) of `ws` on `stream` unless its counters
// [0, counter_bytes) are already known to be zero; records the zero prefix
// this call leaves behind.
cudaError_t prepare_workspace(void* ws, size_t counter_bytes, size_t lse_off,
                              cudaStream_t stream) {
  std::lock_guard<std::mutex> lock(g_ws_mu);
  size_t zp = 0;
  size_t i = 0;
  for (; i < g_ws_zero.size(); ++i)
    if (g_ws_zero[i].ptr == ws) break;
  if (i < g_ws_zero.size()) {
    zp = g_ws_zero[i].zero_prefix;
    g_ws_zero.erase(g_ws_zero.begin() + static_cast<long>(i));
  }
  if (counter_bytes > zp) {
    cudaError_t e = cudaMemsetAsync(ws, 0, lse_off, stream);
    if (e != cudaSuccess) return e;
    zp = lse_off;
  } else if (lse_off < zp) {
    zp = lse_off;  // this call's partial results start inside the old prefix
  }
  if (g_ws_zero.size() >= kWsRecords) g_ws_zero.erase(g_ws_zero.begin());
  g_ws_zero.push_back({ws, zp});
  return cudaSuccess;
}

}  // namespace

namespace pa {
int set_error(int code, const char* msg) { return fail(code, "%s", msg); }
void clear_error() { g_error.clear(); }

size_t prefill_v16_bytes(int num_seqs, int num_kv_heads, int head_dim, int max_blocks_per_seq,
                         int block_size, bool bf16) {
  if (!bf16 || num_seqs < 1 || num_kv_heads < 1 || (head_dim != 64 && head_dim != 128) ||
      max_blocks_per_seq < 1 || log2_pow2(block_size) < 0)
    return 0;
  const long long slots = static_cast<long long>(num_seqs) * max_blocks_per_seq * block_size;
  if (slots > 0x7fffffffll) return 0;  // slot numbers are 32-bit in the kernel
  return round_up(static_cast<size_t>(slots) * num_kv_heads * head_dim * 2, 256);
}

WorkspaceLayout workspace_layout(int num_seqs, int num_q_heads, int head_dim, int max_partitions) {
  WorkspaceLayout w{};
  const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads;
  if (max_partitions <= 1) return w;
  w.count_off = kWorkspaceHeader;
  w.lse_off = round_up(kWorkspaceHeader + rows * sizeof(int), 256);
  w.out_off = w.lse_off + round_up(rows * max_partitions * sizeof(float), 256);
  w.total = w.out_off + rows * max_partitions * static_cast<size_t>(head_dim) * sizeof(float);
  return w;
}
}  // namespace pa

extern "C" {

const char* pa_last_error(void) { return g_error.c_str(); }

int pa_bad_index_count(unsigned long long* count, int clear) {
  g_error.clear();
  return read_counter(false, count, clear);
}

int pa_wait_timeout_count(unsigned long long* count, int clear) {
  g_error.clear();
  return read_counter(true, count, clear);
}

int pa_reshape_and_cache(const void* key, const void* value, void* key_cache, void* value_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int num_blocks, pa_dtype dtype,
                         cudaStream_t stream) {
  g_error.clear();
  int rc = check_dtype(dtype);
  if (rc != PA_OK) return rc;
  if (num_tokens < 0) return fail(PA_ERR_INVALID, "num_tokens %d < 0", num_tokens);
  if (num_kv_heads < 1) return fail(PA_ERR_INVALID, "num_kv_heads %d < 1", num_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (log2_pow2(block_size) < 0)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: powers of two up to 64)", block_size);
  if (num_blocks < 1) return fail(PA_ERR_INVALID, "num_blocks %d < 1", num_blocks);
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !key_cache || !value_cache || !slot_mapping)
    return fail(PA_ERR_INVALID, "a pointer argument is NULL");
  if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID, "key, value and the caches must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return fail(PA_ERR_INVALID, "slot_mapping must be 8-byte aligned");
  const long long row_bytes = static_cast<long long>(num_kv_heads) * head_dim * 2;
  if (row_bytes > (1ll << 30)) return fail(PA_ERR_UNSUPPORTED, "a token row of %lld bytes", row_bytes);
  unsigned long long* bad = nullptr;
  rc = bad_counter(&bad);
  if (rc != PA_OK) return rc;
  cudaError_t e = pa::launch_reshape_and_cache(
      key, value, key_cache, value_cache, slot_mapping, num_tokens, static_cast<int>(row_bytes),
      static_cast<long long>(num_blocks) * block_size, bad, stream);
  if (e != cudaSuccess) return cuda_fail(e, "reshape_and_cache launch");
  return PA_OK;
}

int pa_copy_blocks(void* key_cache, void* value_cache, const int32_t* src, const int32_t* dst,
                   int num_copies, int num_kv_heads, int head_dim, int block_size, int num_blocks,
                   pa_dtype dtype, cudaStream_t stream) {
  g_error.clear();
  int rc = check_dtype(dtype);
  if (rc != PA_OK) return rc;
  if (num_copies < 0) return fail(PA_ERR_INVALID, "num_copies %d < 0", num_copies);
  if (num_kv_heads < 1) return fail(PA_ERR_INVALID, "num_kv_heads %d < 1", num_kv_heads);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  if (log2_pow2(block_size) < 0)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: powers of two up to 64)", block_size);
  if (num_blocks < 1) return fail(PA_ERR_INVALID, "num_blocks %d < 1", num_blocks);
  if (num_copies == 0) return PA_OK;
  if (!key_cache || !value_cache || !src || !dst) return fail(PA_ERR_INVALID, "a pointer argument is NULL");
  if (!aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID, "the caches must be 16-byte aligned");
  if (!aligned4(src) || !aligned4(dst)) return fail(PA_ERR_INVALID, "src and dst must be 4-byte aligned");
  unsigned long long* bad = nullptr;
  rc = bad_counter(&bad);
  if (rc != PA_OK) return rc;
  const long long block_bytes = static_cast<long long>(block_size) * num_kv_heads * head_dim * 2;
  cudaError_t e = pa::launch_copy_blocks(key_cache, value_cache, src, dst, num_copies, block_bytes,
                                         num_blocks, bad, stream);
  if (e != cudaSuccess) return cuda_fail(e, "copy_blocks launch");
  return PA_OK;
}

}  // extern "C"

namespace {

int prefill_impl(void* out, const void* query, const void* key_cache, const void* value_cache,
                 const int32_t* block_tables, const int32_t* seq_lens, const int32_t* query_start,
                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                 float scale, int max_blocks_per_seq, int num_blocks, int max_query_len,
                 pa_dtype dtype, pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
                 int stall_for_test, cudaStream_t stream) {
  g_error.clear();
  int rc = check_dtype(dtype);
  if (rc != PA_OK) return rc;
  if (out_dtype != dtype && out_dtype != PA_FLOAT32)
    return fail(PA_ERR_INVALID, "out_dtype %d must equal dtype %d or be PA_FLOAT32", (int)out_dtype,
                (int)dtype);
  if (num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs %d < 0", num_seqs);
  if (num_q_heads < 1 || num_kv_heads < 1 || num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "num_q_heads %d must be a positive multiple of num_kv_heads %d",
                num_q_heads, num_kv_heads);
  const int group = num_q_heads / num_kv_heads;
  if (group > pa::kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "%d query heads per kv head (> %d)", group, pa::kMaxGroup);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  const int shift = log2_pow2(block_size);
  if (shift < 0)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: powers of two up to 64)", block_size);
  if (max_blocks_per_seq < 1 || num_blocks < 1)
    return fail(PA_ERR_INVALID, "max_blocks_per_seq and num_blocks must be >= 1");
  if (static_cast<long long>(max_blocks_per_seq) * block_size > 0x7fffffffll)
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq * block_size overflows int");
  if (!pa::prefill_tc_supported(block_size, static_cast<long long>(num_blocks) * block_size))
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * block_size is 2^31 slots or more");
  if (!isfinite(scale)) return fail(PA_ERR_INVALID, "scale is not finite");
  if (max_query_len < 0) return fail(PA_ERR_INVALID, "max_query_len %d < 0", max_query_len);
  if (num_seqs > 65535 || num_kv_heads > 65535)
    return fail(PA_ERR_UNSUPPORTED, "num_seqs %d / num_kv_heads %d above 65535", num_seqs, num_kv_heads);
  // bf16 with a workspace: the fp16 copy of the value rows (one P.V product)
  const size_t v16_need = pa::prefill_v16_bytes(num_seqs, num_kv_heads, head_dim,
                                                max_blocks_per_seq, block_size,
                                                dtype == PA_BFLOAT16);
  void* v16 = nullptr;
  if (workspace != nullptr && v16_need > 0) {
    if (workspace_bytes < v16_need)
      return fail(PA_ERR_WORKSPACE, "prefill workspace of %zu bytes needed, %zu given", v16_need,
                  workspace_bytes);
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
    v16 = workspace;
  }
  if (num_seqs == 0 || max_query_len == 0) return PA_OK;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !seq_lens || !query_start)
    return fail(PA_ERR_INVALID, "a pointer argument is NULL");
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID, "out, query and the caches must be 16-byte aligned");
  if (!aligned4(block_tables) || !aligned4(seq_lens) || !aligned4(query_start))
    return fail(PA_ERR_INVALID, "block_tables, seq_lens and query_start must be 4-byte aligned");
  unsigned long long* bad = nullptr;
  rc = bad_counter(&bad);
  if (rc != PA_OK) return rc;
  pa::PrefillArgs a{};
  a.out = out;
  a.query = query;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.query_start = query_start;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.block_shift = shift;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.out_f32 = out_dtype == PA_FLOAT32 ? 1 : 0;
  a.bad = bad;
  a.stall_for_test = stall_for_test;
  a.v16 = v16;
  rc = counter(true, &a.timeouts);
  if (rc != PA_OK) return rc;
  cudaError_t e = pa::launch_prefill_tc(a, head_dim, dtype == PA_BFLOAT16, max_query_len, stream);
  if (e != cudaSuccess) return cuda_fail(e, "paged prefill launch");
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_prefill(void* out, const void* query, const void* key_cache, const void* value_cache,
               const int32_t* block_tables, const int32_t* seq_lens, const int32_t* query_start,
               int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
               float scale, int max_blocks_per_seq, int num_blocks, int max_query_len,
               pa_dtype dtype, pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
               cudaStream_t stream) {
  return prefill_impl(out, query, key_cache, value_cache, block_tables, seq_lens, query_start,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                      max_blocks_per_seq, num_blocks, max_query_len, dtype, out_dtype, workspace,
                      workspace_bytes, 0, stream);
}

size_t pa_prefill_workspace_bytes(int num_seqs, int num_kv_heads, int head_dim,
                                  int max_blocks_per_seq, int block_size, pa_dtype dtype) {
  return pa::prefill_v16_bytes(num_seqs, num_kv_heads, head_dim, max_blocks_per_seq, block_size,
                               dtype == PA_BFLOAT16);
}

int pa_testing_prefill_stalled(void* out, const void* query, const void* key_cache,
                               const void* value_cache, const int32_t* block_tables,
                               const int32_t* seq_lens, const int32_t* query_start, int num_seqs,
                               int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                               float scale, int max_blocks_per_seq, int num_blocks,
                               int max_query_len, pa_dtype dtype, pa_dtype out_dtype,
                               void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return prefill_impl(out, query, key_cache, value_cache, block_tables, seq_lens, query_start,
                      num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, scale,
                      max_blocks_per_seq, num_blocks, max_query_len, dtype, out_dtype, workspace,
                      workspace_bytes, 1, stream);
}

int pa_decode_partition_tokens(int partition_tokens, int block_size, int max_blocks_per_seq) {
  g_error.clear();
  if (log2_pow2(block_size) < 0)
    return fail(PA_ERR_INVALID, "block_size %d is not a power of two in [1, 64]", block_size);
  if (max_blocks_per_seq < 1)
    return fail(PA_ERR_INVALID, "max_blocks_per_seq %d < 1", max_blocks_per_seq);
  int pt = 0;
  const int rc = resolve_partition(partition_tokens, block_size, max_blocks_per_seq, &pt);
  return rc == PA_OK ? pt : rc;
}

size_t pa_decode_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_tokens) {
  if (num_seqs < 0 || num_q_heads < 1 || (head_dim != 64 && head_dim != 128) ||
      max_blocks_per_seq < 1 || log2_pow2(block_size) < 0)
    return 0;
  int pt = 0;
  std::string saved = g_error;
  if (resolve_partition(partition_tokens, block_size, max_blocks_per_seq, &pt) != PA_OK) {
    g_error = saved;
    return 0;
  }
  const long long lmax = static_cast<long long>(max_blocks_per_seq) * block_size;
  const long long parts = (lmax + pt - 1) / pt;
  return pa::workspace_layout(num_seqs, num_q_heads, head_dim, static_cast<int>(parts)).total;
}

}  // extern "C"

namespace {

int decode_impl(void* out, const void* query, const void* key_cache, const void* value_cache,
                const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
                int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
                int max_blocks_per_seq, int num_blocks, int partition_tokens, pa_dtype dtype,
                pa_dtype out_dtype, void* workspace, size_t workspace_bytes,
                const void* new_key, const void* new_value, cudaStream_t stream) {
  g_error.clear();
  int rc = check_dtype(dtype);
  if (rc != PA_OK) return rc;
  if (out_dtype != dtype && out_dtype != PA_FLOAT32)
    return fail(PA_ERR_INVALID, "out_dtype %d must equal dtype %d or be PA_FLOAT32", (int)out_dtype,
                (int)dtype);
  if (num_seqs < 0) return fail(PA_ERR_INVALID, "num_seqs %d < 0", num_seqs);
  if (num_q_heads < 1 || num_kv_heads < 1)
    return fail(PA_ERR_INVALID, "num_q_heads %d / num_kv_heads %d must be >= 1", num_q_heads,
                num_kv_heads);
  if (num_q_heads % num_kv_heads != 0)
    return fail(PA_ERR_INVALID, "num_q_heads %d is not a multiple of num_kv_heads %d", num_q_heads,
                num_kv_heads);
  const int group = num_q_heads / num_kv_heads;
  if (group > pa::kMaxGroup)
    return fail(PA_ERR_UNSUPPORTED, "%d query heads per kv head (> %d)", group, pa::kMaxGroup);
  if (head_dim != 64 && head_dim != 128)
    return fail(PA_ERR_UNSUPPORTED, "head_dim %d (supported: 64, 128)", head_dim);
  const int shift = log2_pow2(block_size);
  if (shift < 0)
    return fail(PA_ERR_UNSUPPORTED, "block_size %d (supported: powers of two up to 64)", block_size);
  if (max_blocks_per_seq < 1) return fail(PA_ERR_INVALID, "max_blocks_per_seq %d < 1", max_blocks_per_seq);
  if (num_blocks < 1) return fail(PA_ERR_INVALID, "num_blocks %d < 1", num_blocks);
  // cache slots travel as 32-bit values in the kernel (all ones = none)
  if ((static_cast<long long>(num_blocks) << shift) > 0xfffffffeLL)
    return fail(PA_ERR_UNSUPPORTED, "num_blocks * block_size is 2^32 - 1 slots or more");
  if (!isfinite(scale)) return fail(PA_ERR_INVALID, "scale is not finite");
  int pt = 0;
  rc = resolve_partition(partition_tokens, block_size, max_blocks_per_seq, &pt);
  if (rc != PA_OK) return rc;
  const long long lmax = static_cast<long long>(max_blocks_per_seq) * block_size;
  if (lmax > 0x7fffffffll)
    return fail(PA_ERR_UNSUPPORTED, "max_blocks_per_seq * block_size = %lld overflows int", lmax);
  if (num_seqs > 65535 || num_kv_heads > 65535)
    return fail(PA_ERR_UNSUPPORTED, "num_seqs %d / num_kv_heads %d above 65535", num_seqs,
                num_kv_heads);
  if (num_seqs == 0) return PA_OK;
  if (!out || !query || !key_cache || !value_cache || !block_tables || !seq_lens)
    return fail(PA_ERR_INVALID, "a pointer argument is NULL");
  if (!aligned16(out) || !aligned16(query) || !aligned16(key_cache) || !aligned16(value_cache))
    return fail(PA_ERR_INVALID, "out, query and the caches must be 16-byte aligned");
  if (!aligned4(block_tables) || !aligned4(seq_lens))
    return fail(PA_ERR_INVALID, "block_tables and seq_lens must be 4-byte aligned");

  const int parts = static_cast<int>((lmax + pt - 1) / pt);
  const pa::WorkspaceLayout wl = pa::workspace_layout(num_seqs, num_q_heads, head_dim, parts);
  if (wl.total > 0) {
    if (workspace == nullptr || workspace_bytes < wl.total)
      return fail(PA_ERR_WORKSPACE, "workspace of %zu bytes needed, %zu given", wl.total,
                  workspace == nullptr ? (size_t)0 : workspace_bytes);
    if (!aligned16(workspace)) return fail(PA_ERR_INVALID, "workspace must be 16-byte aligned");
  }
  int sms = 0;
  rc = num_sms(&sms);
  if (rc != PA_OK) return rc;
  // the persistent schedule works in 64-bit positions: the total weight times
  // the grid size (at most 32 CTAs per SM) must stay below 2^62
  {
    const double wmax = static_cast<double>(num_seqs) * num_kv_heads *
                        (static_cast<double>(lmax) + static_cast<double>(parts) * pa::kUnitCost);
    if (wmax * 32.0 * sms >= 4.0e18)
      return fail(PA_ERR_UNSUPPORTED, "num_seqs * num_kv_heads * max sequence length too large");
  }
  unsigned long long* bad = nullptr;
  rc = bad_counter(&bad);
  if (rc != PA_OK) return rc;
  if (wl.total > 0) {
    const size_t counter_bytes =
        pa::kWorkspaceHeader + static_cast<size_t>(num_seqs) * num_kv_heads * sizeof(int);
    cudaError_t e = prepare_workspace(workspace, counter_bytes, wl.lse_off, stream);
    if (e != cudaSuccess) return cuda_fail(e, "cudaMemsetAsync(workspace counters)");
  }

  pa::DecodeArgs a{};
  a.out = out;
  a.query = query;
  a.key_cache = key_cache;
  a.value_cache = value_cache;
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  // One kv head per scheduling unit: grouping 2 or 4 heads per CTA (warps on
  // adjacent heads) made the units coarser and was never faster at 512-token
  // partitions on GB300; the kernel keeps the grouping as a parameter.
  a.heads_per_cta = 1;
  a.block_shift = shift;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.partition_tokens = pt;
  a.max_partitions = parts;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.out_f32 = out_dtype == PA_FLOAT32 ? 1 : 0;
  a.new_key = new_key;
  a.new_value = new_value;
  char* ws = static_cast<char*>(workspace);
  a.ws_count = wl.total ? reinterpret_cast<int*>(ws + wl.count_off) : nullptr;
  // the trailing partitions of rows are handed out at run time only with a
  // workspace (its header holds the claim counter)
  a.ws_claim = wl.total ? reinterpret_cast<unsigned long long*>(ws) : nullptr;
  a.ws_done = wl.total ? reinterpret_cast<unsigned*>(ws + 8) : nullptr;
  // the share grows with the partition length (fewer, larger units per row)
  a.dyn_percent = wl.total ? std::min(50, PA_DECODE_DYNAMIC_PERCENT * pt / 512) : 0;
  a.ws_lse = wl.total ? reinterpret_cast<float*>(ws + wl.lse_off) : nullptr;
  a.ws_out = wl.total ? reinterpret_cast<float*>(ws + wl.out_off) : nullptr;
  a.bad = bad;
  cudaError_t e = pa::launch_decode(a, head_dim, dtype == PA_BFLOAT16, sms, stream);
  if (e != cudaSuccess) return cuda_fail(e, "paged decode launch");
  return PA_OK;
}

}  // namespace

extern "C" {

int pa_decode(void* out, const void* query, const void* key_cache, const void* value_cache,
              const int32_t* block_tables, const int32_t* seq_lens, int num_seqs,
              int num_q_heads, int num_kv_heads, int head_dim, int block_size, float scale,
              int max_blocks_per_seq, int num_blocks, int partition_tokens, pa_dtype dtype,
              pa_dtype out_dtype, void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  return decode_impl(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, scale, max_blocks_per_seq,
                     num_blocks, partition_tokens, dtype, out_dtype, workspace, workspace_bytes,
                     nullptr, nullptr, stream);
}

int pa_decode_append(void* out, const void* query, const void* new_key, const void* new_value,
                     void* key_cache, void* value_cache, const int32_t* block_tables,
                     const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, float scale, int max_blocks_per_seq,
                     int num_blocks, int partition_tokens, pa_dtype dtype, pa_dtype out_dtype,
                     void* workspace, size_t workspace_bytes, cudaStream_t stream) {
  g_error.clear();
  if (num_seqs > 0) {
    if (!new_key || !new_value) return fail(PA_ERR_INVALID, "new_key / new_value is NULL");
    if (!aligned16(new_key) || !aligned16(new_value))
      return fail(PA_ERR_INVALID, "new_key and new_value must be 16-byte aligned");
  }
  return decode_impl(out, query, key_cache, value_cache, block_tables, seq_lens, num_seqs,
                     num_q_heads, num_kv_heads, head_dim, block_size, scale, max_blocks_per_seq,
                     num_blocks, partition_tokens, dtype, out_dtype, workspace, workspace_bytes,
                     new_key, new_value, stream);
}

}  // extern "C"
