// Host-side KV block management: how many pages fit, and which are free.
//
// swiftLLM's engine (architecture section) asks its worker to profile the
// number of GPU blocks, then allocates the KV cache and a KV swap space of
// that many blocks; every step it swaps blocks in and out before computing.
// Here a block is one page of the pools: 16 tokens of every KV head.
//
// pa_profile_num_blocks turns free device bytes into a page count;
// pa_block_allocator_* is the free list that hands pages to sequences;
// pa_block_table_grow extends one sequence's block-table row as it grows.
// The allocator is a LIFO stack of free pages (fresh pages come out in
// ascending order), guarded by a mutex, with an ownership bit per page so
// that a double free or a stray index is refused instead of corrupting it.
#include <stdint.h>
#include <stdlib.h>

#include <mutex>
#include <new>
#include <vector>

#include "pa_internal.h"

struct pa_block_allocator {
  std::mutex mu;
  std::vector<int32_t> free_stack;  // top = back
  std::vector<uint8_t> used;        // 1 = handed out
};

namespace {

// Bytes of one page in every layer's K and V pools (16-bit elements), or in
// an 8-bit cache (INT8 or E4M3 codes plus one fp32 scale per row).
int64_t page_bytes(const pa_shape_t* s, int32_t num_layers, int32_t kv_kind) {
  const int64_t rows = (int64_t)s->num_kv_heads * s->page_size;
  const int64_t d = s->head_dim;
  const int64_t per_row = kv_kind == PA_KV_16BIT ? 2 * d : d + 4;
  return 2 * rows * per_row * num_layers;
}

}  // namespace

extern "C" int64_t pa_profile_num_blocks(const pa_shape_t* shape, int32_t num_layers,
                                         int32_t kv_kind, size_t free_bytes,
                                         size_t reserve_bytes) {
  if (!shape || shape->num_kv_heads <= 0 || shape->head_dim <= 0 || shape->page_size <= 0 ||
      num_layers <= 0 ||
      (kv_kind != PA_KV_16BIT && kv_kind != PA_KV_INT8 && kv_kind != PA_KV_FP8))
    return -1;
  if (free_bytes <= reserve_bytes) return 0;
  const size_t per_page = (size_t)page_bytes(shape, num_layers, kv_kind);
  const int64_t n = (int64_t)((free_bytes - reserve_bytes) / per_page);
  return n > INT32_MAX ? INT32_MAX : n;
}

extern "C" pa_status_t pa_block_allocator_create(int32_t num_blocks, pa_block_allocator_t** out) {
  if (!out || num_blocks < 0) return PA_ERR_INVALID_ARG;
  *out = nullptr;
  pa_block_allocator* a = new (std::nothrow) pa_block_allocator;
  if (!a) return PA_ERR_NO_MEMORY;
  try {
    a->free_stack.resize((size_t)num_blocks);
    a->used.assign((size_t)num_blocks, 0);
  } catch (...) {
    delete a;
    return PA_ERR_NO_MEMORY;
  }
  for (int32_t i = 0; i < num_blocks; ++i) a->free_stack[(size_t)i] = num_blocks - 1 - i;
  *out = a;
  return PA_OK;
}

extern "C" void pa_block_allocator_destroy(pa_block_allocator_t* a) { delete a; }

extern "C" int32_t pa_block_num_free(pa_block_allocator_t* a) {
  if (!a) return -1;
  std::lock_guard<std::mutex> g(a->mu);
  return (int32_t)a->free_stack.size();
}

extern "C" pa_status_t pa_block_alloc(pa_block_allocator_t* a, int32_t n, int32_t* blocks_out) {
  if (!a || n < 0 || (n > 0 && !blocks_out)) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(a->mu);
  if ((size_t)n > a->free_stack.size()) return PA_ERR_NO_MEMORY;  // all or nothing
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = a->free_stack.back();
    a->free_stack.pop_back();
    a->used[(size_t)b] = 1;
    blocks_out[i] = b;
  }
  return PA_OK;
}

extern "C" pa_status_t pa_block_free(pa_block_allocator_t* a, const int32_t* blocks, int32_t n) {
  if (!a || n < 0 || (n > 0 && !blocks)) return PA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> g(a->mu);
  // Validate first, marking each listed page 2 so a page listed twice is
  // caught; a refused call restores the marks and frees nothing.
  const size_t nb = a->used.size();
  for (int32_t i = 0; i < n; ++i) {
    const int32_t b = blocks[i];
    if (b < 0 || (size_t)b >= nb || a->used[(size_t)b] != 1) {
      for (int32_t k = 0; k < i; ++k) a->used[(size_t)blocks[k]] = 1;
      return PA_ERR_INVALID_ARG;
    }
    a->used[(size_t)b] = 2;
  }
  for (int32_t i = 0; i < n; ++i) {
    a->used[(size_t)blocks[i]] = 0;
    a->free_stack.push_back(blocks[i]);
  }
  return PA_OK;
}

extern "C" pa_status_t pa_block_table_grow(pa_block_allocator_t* a, int32_t* row,
                                           int32_t max_pages, int32_t page_size,
                                           int32_t old_len, int32_t new_len) {
  if (!a || !row || max_pages <= 0 || page_size <= 0 || old_len < 0 || new_len < old_len)
    return PA_ERR_INVALID_ARG;
  const int64_t have = ((int64_t)old_len + page_size - 1) / page_size;
  const int64_t need = ((int64_t)new_len + page_size - 1) / page_size;
  if (need > max_pages) return PA_ERR_INVALID_ARG;
  if (need == have) return PA_OK;
  return pa_block_alloc(a, (int32_t)(need - have), row + have);
}
