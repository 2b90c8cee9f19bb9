// Host-side tile list of the multi-token attention kernel.
//
// A tile is a block of query rows of one (sequence, KV head): rows / G
// consecutive query tokens times the G query heads that share the KV head.
// Its time is set by the causal length it streams (the position of its last
// query + 1): every stage of keys costs about the same whether the tile has
// all its rows or a single decode token's G.  Tiles are issued longest
// stream first (more rows first among equals), so the tail of the grid
// holds the short ones.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <vector>

#include "pa_internal.h"

namespace pa {
namespace {

std::atomic<uint64_t> g_prefill_ids{1};

struct Tile {
  int32_t b, g, tok0, ntok;
  int64_t work;
};

}  // namespace
}  // namespace pa

extern "C" pa_status_t pa_prefill_plan_ex(const pa_shape_t* shape, const int32_t* seq_lens_host,
                                          const int32_t* q_lens_host,
                                          const pa_prefill_options_t* options,
                                          pa_prefill_plan_t* plan_out) {
  using namespace pa;
  if (!plan_out) return PA_ERR_INVALID_ARG;
  memset(plan_out, 0, sizeof(*plan_out));
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  const pa_prefill_options_t o = options ? *options : pa_prefill_options_t{};
  // rows per tile: the tcgen05 kernel's 128 by default, 64 for the mma.sync kernel
  if (o.rows_per_tile != 0 && o.rows_per_tile != kPrefillRowsTc5 && o.rows_per_tile != kPrefillRows)
    return PA_ERR_INVALID_ARG;
  const int B = shape->batch, Hkv = shape->num_kv_heads, D = shape->head_dim;
  const int G = shape->num_q_heads / Hkv;
  const int rows = o.rows_per_tile == 0 ? kPrefillRowsTc5 : o.rows_per_tile;
  const int tok_per_tile = rows / G;
  if (B > 0 && (!seq_lens_host || !q_lens_host)) return PA_ERR_INVALID_ARG;

  std::vector<int32_t> cu((size_t)B + 1, 0);
  std::vector<Tile> tiles;
  for (int b = 0; b < B; ++b) {
    const int32_t L = seq_lens_host[b], n = q_lens_host[b];
    if (L < 0 || n < 0 || n > L || (int64_t)L > (int64_t)shape->max_pages_per_seq * shape->page_size)
      return PA_ERR_INVALID_ARG;
    if ((int64_t)cu[(size_t)b] + n > INT32_MAX) return PA_ERR_INVALID_ARG;
    cu[(size_t)b + 1] = cu[(size_t)b] + n;
    for (int tok0 = 0; tok0 < n; tok0 += tok_per_tile) {
      const int ntok = std::min(tok_per_tile, n - tok0);
      const int64_t span = (int64_t)(L - n + tok0 + ntok);  // keys the tile's last query sees
      for (int g = 0; g < Hkv; ++g) tiles.push_back({b, g, tok0, ntok, span});
    }
  }
  std::stable_sort(tiles.begin(), tiles.end(), [](const Tile& x, const Tile& y) {
    return x.work != y.work ? x.work > y.work : x.ntok > y.ntok;
  });
  const PrefillLayout lay = prefill_layout((int)tiles.size(), B);
  int32_t* blob = (int32_t*)malloc(lay.blob_bytes);
  if (!blob) return PA_ERR_NO_MEMORY;
  memset(blob, 0, lay.blob_bytes);
  const uint64_t id = g_prefill_ids.fetch_add(1);
  blob[0] = (int32_t)kPrefillMagic;
  blob[1] = (int32_t)tiles.size();
  blob[2] = B;
  blob[3] = cu[(size_t)B];
  blob[4] = (int32_t)(id & 0xffffffffu);
  blob[5] = (int32_t)(id >> 32);
  blob[6] = G;
  blob[7] = D;
  blob[8] = rows;
  int32_t* t = blob + lay.tiles_off / 4;
  for (size_t i = 0; i < tiles.size(); ++i) {
    t[4 * i + 0] = tiles[i].b;
    t[4 * i + 1] = tiles[i].g;
    t[4 * i + 2] = tiles[i].tok0;
    t[4 * i + 3] = tiles[i].ntok;
  }
  memcpy(blob + lay.cu_off / 4, cu.data(), sizeof(int32_t) * cu.size());

  plan_out->shape = *shape;
  plan_out->num_tiles = (int32_t)tiles.size();
  plan_out->total_q = cu[(size_t)B];
  plan_out->owns_blob = 1;
  plan_out->plan_id = id;
  plan_out->blob_bytes = lay.blob_bytes;
  plan_out->workspace_bytes = lay.blob_bytes;
  plan_out->host_blob = blob;
  plan_out->rows_per_tile = rows;
  plan_out->wait_limit_ns = o.wait_limit_ns;
  return PA_OK;
}

extern "C" pa_status_t pa_prefill_plan(const pa_shape_t* shape, const int32_t* seq_lens_host,
                                       const int32_t* q_lens_host, pa_prefill_plan_t* plan_out) {
  return pa_prefill_plan_ex(shape, seq_lens_host, q_lens_host, nullptr, plan_out);
}

extern "C" void pa_prefill_plan_free(pa_prefill_plan_t* plan) {
  if (!plan) return;
  if (plan->owns_blob && plan->host_blob) free(plan->host_blob);
  plan->host_blob = nullptr;
  plan->blob_bytes = 0;
}
