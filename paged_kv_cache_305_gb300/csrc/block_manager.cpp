// Host-side block manager of the paged KV cache (C ABI in include/pagedattn.h).
//
// Semantics ("PagedAttention by hand", What is PagedAttention / Why divide
// memory into physical blocks?; "PagedAttention" glossary, How It Works):
// free blocks are a stack of interchangeable ids; a sequence's block table
// grows by one block only when its last block is full; forking a sequence
// shares all its blocks (reference counts + 1); writing into a block whose
// reference count is above 1 first copies that one block into a fresh block
// (copy-on-write); freeing a sequence returns the blocks whose count drops to 0.
//
// Free-stack order (the pages fix none): the stack starts with block 0 on top
// (a fresh pool hands out 0, 1, 2, ...), a freed sequence pushes its blocks in
// table order, allocation pops the top. Freed sequence ids are reused last in,
// first out. Not thread-safe: calls on one manager must be serialised.
#include <stdint.h>

#include <new>
#include <string>
#include <vector>

#include "internal.h"
#include "pagedattn.h"

struct pa_block_manager {
  int num_blocks = 0;
  int block_size = 0;
  int max_blocks_per_seq = 0;
  std::vector<int32_t> free_stack;  // top = back()
  std::vector<int32_t> refs;        // per physical block
  struct Seq {
    bool live = false;
    int64_t len = 0;
    std::vector<int32_t> blocks;
  };
  std::vector<Seq> seqs;
  std::vector<int> free_ids;  // reusable sequence ids, top = back()
};

namespace {

int bad(const char* msg) { return pa::set_error(PA_ERR_INVALID, msg); }

bool live(const pa_block_manager* bm, int id) {
  return id >= 0 && id < static_cast<int>(bm->seqs.size()) && bm->seqs[id].live;
}

int take_id(pa_block_manager* bm) {
  if (!bm->free_ids.empty()) {
    const int id = bm->free_ids.back();
    bm->free_ids.pop_back();
    return id;
  }
  bm->seqs.emplace_back();
  return static_cast<int>(bm->seqs.size()) - 1;
}

}  // namespace

extern "C" {

int pa_bm_create(int num_blocks, int block_size, int max_blocks_per_seq, pa_block_manager** out) {
  pa::clear_error();
  if (out == nullptr) return bad("out is NULL");
  *out = nullptr;
  if (num_blocks < 1 || block_size < 1 || max_blocks_per_seq < 1)
    return bad("num_blocks, block_size and max_blocks_per_seq must be >= 1");
  pa_block_manager* bm = new (std::nothrow) pa_block_manager;
  if (bm == nullptr) return pa::set_error(PA_ERR_CAPACITY, "host allocation failed");
  bm->num_blocks = num_blocks;
  bm->block_size = block_size;
  bm->max_blocks_per_seq = max_blocks_per_seq;
  bm->free_stack.resize(num_blocks);
  for (int i = 0; i < num_blocks; ++i) bm->free_stack[i] = num_blocks - 1 - i;
  bm->refs.assign(num_blocks, 0);
  *out = bm;
  return PA_OK;
}

void pa_bm_destroy(pa_block_manager* bm) { delete bm; }

int pa_bm_new_sequence(pa_block_manager* bm, int* seq_id) {
  pa::clear_error();
  if (bm == nullptr || seq_id == nullptr) return bad("a pointer argument is NULL");
  const int id = take_id(bm);
  pa_block_manager::Seq& s = bm->seqs[id];
  s.live = true;
  s.len = 0;
  s.blocks.clear();
  *seq_id = id;
  return PA_OK;
}

int pa_bm_fork(pa_block_manager* bm, int parent, int* child) {
  pa::clear_error();
  if (bm == nullptr || child == nullptr) return bad("a pointer argument is NULL");
  if (!live(bm, parent)) return bad("parent is not a live sequence");
  const int id = take_id(bm);
  pa_block_manager::Seq& p = bm->seqs[parent];  // after take_id: seqs may have grown
  pa_block_manager::Seq& c = bm->seqs[id];
  c.live = true;
  c.len = p.len;
  c.blocks = p.blocks;
  for (int32_t b : c.blocks) ++bm->refs[b];
  *child = id;
  return PA_OK;
}

int pa_bm_free_sequence(pa_block_manager* bm, int seq_id) {
  pa::clear_error();
  if (bm == nullptr) return bad("bm is NULL");
  if (!live(bm, seq_id)) return bad("seq_id is not a live sequence");
  pa_block_manager::Seq& s = bm->seqs[seq_id];
  for (int32_t b : s.blocks) {
    if (--bm->refs[b] == 0) bm->free_stack.push_back(b);
  }
  s.blocks.clear();
  s.len = 0;
  s.live = false;
  bm->free_ids.push_back(seq_id);
  return PA_OK;
}

int pa_bm_append(pa_block_manager* bm, const int* seq_ids, const int* num_new, int count,
                 int64_t* slot_mapping, int slot_capacity, int32_t* copy_src, int32_t* copy_dst,
                 int copy_capacity, int* num_copies) {
  pa::clear_error();
  if (bm == nullptr || num_copies == nullptr) return bad("a pointer argument is NULL");
  *num_copies = 0;
  if (count < 0) return bad("count < 0");
  if (count == 0) return PA_OK;
  if (seq_ids == nullptr || num_new == nullptr || slot_mapping == nullptr || copy_src == nullptr ||
      copy_dst == nullptr)
    return bad("a pointer argument is NULL");
  if (copy_capacity < count) return bad("copy_capacity must be >= count (one copy per sequence at most)");
  const int64_t B = bm->block_size;
  // validate, and count the blocks this append takes, in request order
  int64_t total = 0, need = 0;
  std::vector<int32_t> drop;  // shared blocks already copied away earlier in this call
  for (int i = 0; i < count; ++i) {
    const int id = seq_ids[i];
    if (!live(bm, id)) return bad("a seq_id is not a live sequence");
    if (num_new[i] < 0) return bad("num_new must be >= 0");
    for (int j = 0; j < i; ++j)
      if (seq_ids[j] == id) return bad("a sequence may appear once per append");
    const pa_block_manager::Seq& s = bm->seqs[id];
    const int64_t end = s.len + num_new[i];
    if ((end + B - 1) / B > bm->max_blocks_per_seq)
      return pa::set_error(PA_ERR_CAPACITY, "a block table would exceed max_blocks_per_seq");
    total += num_new[i];
    if (num_new[i] == 0) continue;
    const int64_t first_new_blocks = (end + B - 1) / B - (s.len + B - 1) / B;
    need += first_new_blocks;
    if (s.len % B != 0) {
      const int32_t blk = s.blocks[s.len / B];
      int32_t r = bm->refs[blk];
      for (int32_t d : drop)
        if (d == blk) --r;
      if (r > 1) {
        ++need;
        drop.push_back(blk);
      }
    }
  }
  if (total > slot_capacity) return bad("slot_capacity is smaller than the number of new tokens");
  if (need > static_cast<int64_t>(bm->free_stack.size()))
    return pa::set_error(PA_ERR_CAPACITY, "not enough free blocks");
  // apply
  int64_t k = 0;
  int nc = 0;
  for (int i = 0; i < count; ++i) {
    pa_block_manager::Seq& s = bm->seqs[seq_ids[i]];
    for (int n = 0; n < num_new[i]; ++n) {
      const int64_t t = s.len;
      const int64_t lb = t / B, off = t % B;
      int32_t blk;
      if (off == 0) {
        blk = bm->free_stack.back();
        bm->free_stack.pop_back();
        bm->refs[blk] = 1;
        s.blocks.push_back(blk);
      } else {
        blk = s.blocks[lb];
        if (bm->refs[blk] > 1) {  // copy-on-write of this one block
          const int32_t fresh = bm->free_stack.back();
          bm->free_stack.pop_back();
          bm->refs[fresh] = 1;
          --bm->refs[blk];
          copy_src[nc] = blk;
          copy_dst[nc] = fresh;
          ++nc;
          s.blocks[lb] = fresh;
          blk = fresh;
        }
      }
      slot_mapping[k++] = static_cast<int64_t>(blk) * B + off;
      s.len = t + 1;
    }
  }
  *num_copies = nc;
  return PA_OK;
}

int pa_bm_block_tables(const pa_block_manager* bm, const int* seq_ids, int count,
                       int32_t* block_tables, int32_t* seq_lens) {
  pa::clear_error();
  if (bm == nullptr) return bad("bm is NULL");
  if (count < 0) return bad("count < 0");
  if (count == 0) return PA_OK;
  if (seq_ids == nullptr || block_tables == nullptr || seq_lens == nullptr)
    return bad("a pointer argument is NULL");
  const int MB = bm->max_blocks_per_seq;
  for (int i = 0; i < count; ++i) {
    if (!live(bm, seq_ids[i])) return bad("a seq_id is not a live sequence");
    const pa_block_manager::Seq& s = bm->seqs[seq_ids[i]];
    if (s.len > 0x7fffffff) return pa::set_error(PA_ERR_UNSUPPORTED, "a sequence is longer than 2^31-1");
    int32_t* row = block_tables + static_cast<int64_t>(i) * MB;
    const int n = static_cast<int>(s.blocks.size());
    for (int j = 0; j < MB; ++j) row[j] = j < n ? s.blocks[j] : 0;
    seq_lens[i] = static_cast<int32_t>(s.len);
  }
  return PA_OK;
}

int pa_bm_num_free_blocks(const pa_block_manager* bm, int* n) {
  pa::clear_error();
  if (bm == nullptr || n == nullptr) return bad("a pointer argument is NULL");
  *n = static_cast<int>(bm->free_stack.size());
  return PA_OK;
}

int pa_bm_ref_count(const pa_block_manager* bm, int block, int* count) {
  pa::clear_error();
  if (bm == nullptr || count == nullptr) return bad("a pointer argument is NULL");
  if (block < 0 || block >= bm->num_blocks) return bad("block out of range");
  *count = bm->refs[block];
  return PA_OK;
}

}  // extern "C"
