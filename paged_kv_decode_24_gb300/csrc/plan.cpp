// Host-side split planner: turns host seq_lens into the warp task list that
// the split-decode kernel walks, plus the split groups it merges.
//
// Flash-Decoding (swiftLLM, feature list: paged attention v2) cuts a long
// sequence into chunks processed in parallel, each producing a partial
// output and log-sum-exp, merged afterwards.  The planner decides where to
// cut: each sequence is split into near-equal page ranges no longer than
// the average load of one resident CTA, so that no task outlasts the rest of
// the grid, and tasks are issued longest first so the tail of the grid holds
// the short ones.  A batch whose sequences are already shorter than that is
// not split: a split costs a partial write, a merge and a CTA start, and
// balances nothing there.
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <vector>

#include "pa_internal.h"

namespace pa {

pa_status_t check_shape(const pa_shape_t* s) {
  if (!s) return PA_ERR_INVALID_ARG;
  if (s->batch < 0 || s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->head_dim <= 0 ||
      s->page_size <= 0 || s->max_pages_per_seq <= 0 || s->num_pages <= 0)
    return PA_ERR_INVALID_ARG;
  if (s->num_q_heads % s->num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  const int g = s->num_q_heads / s->num_kv_heads;
  if (g != 1 && g != 2 && g != 4 && g != 8) return PA_ERR_UNSUPPORTED;
  if (s->head_dim != 64 && s->head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (s->page_size != kPageSize) return PA_ERR_UNSUPPORTED;
  if (s->num_kv_heads > (int)kItemHeadMask) return PA_ERR_UNSUPPORTED;
  if (s->dtype != PA_DTYPE_F16 && s->dtype != PA_DTYPE_BF16) return PA_ERR_UNSUPPORTED;
  if ((int64_t)s->max_pages_per_seq * s->page_size > INT32_MAX) return PA_ERR_INVALID_ARG;
  return PA_OK;
}

namespace {

uint64_t next_plan_id() {
  static std::atomic<uint64_t> counter{
      (uint64_t)std::chrono::high_resolution_clock::now().time_since_epoch().count() * 2654435761u};
  return counter.fetch_add(0x9e3779b97f4a7c15ull) | 1ull;
}

}  // namespace
}  // namespace pa

namespace pa {
namespace {

// Page stages per warp of the 8-bit-cache kernel at head_dim 128.  Three
// when every CTA of the plan is resident at once (one wave); otherwise two
// when the tasks average at most kQ8ShortPagesPerWarp pages per warp, else
// three.  Over several waves, a warp that streams few pages gains nothing
// from a third page in flight: two stages measured faster on short tasks
// (workloads of many short sequences, the short tasks of a skewed mix),
// three on long ones; in one wave of short tasks three measured faster.
int q8_stages_for(int n_tasks, int n_shared, int64_t total_pages, int64_t n_ctas,
                  int64_t cta_slots) {
  if (n_ctas <= cta_slots) return 3;
  const int64_t warps = (int64_t)n_shared * kWarpsPerCta + (n_tasks - n_shared);
  return warps > 0 && total_pages <= (int64_t)kQ8ShortPagesPerWarp * warps ? 2 : 3;
}

// Fill *plan_out and, when dst is non-null, write the task list into dst
// (dst_bytes long).  With dst == nullptr and alloc set, the list goes into a
// fresh malloc'ed block owned by the plan.  opt may be null (defaults).
pa_status_t plan_impl(const pa_shape_t* shape, const int32_t* seq_lens_host, int32_t num_sms,
                      int32_t forced_splits, const pa_plan_options_t* opt, void* dst,
                      size_t dst_bytes, bool alloc, pa_plan_t* plan_out) {
  if (!plan_out) return PA_ERR_INVALID_ARG;
  memset(plan_out, 0, sizeof(*plan_out));
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  if (num_sms <= 0 || forced_splits < 0) return PA_ERR_INVALID_ARG;
  const pa_plan_options_t o = opt ? *opt : pa_plan_options_t{};
  if (o.min_chunk_pages < 0 || o.waves < 0 || o.waves > 64 || o.bundle_waves > 64 ||
      (o.merge != PA_MERGE_IN_SPLIT_KERNEL && o.merge != PA_MERGE_COMBINE_KERNEL) ||
      o.l2_prefetch_pages > 32 || (o.q8_stages != 0 && o.q8_stages != 2 && o.q8_stages != 3) ||
      (o.early_kv != 0 && o.early_kv != 1))
    return PA_ERR_INVALID_ARG;
  const int B = shape->batch, Hkv = shape->num_kv_heads, D = shape->head_dim;
  const int G = shape->num_q_heads / Hkv, S = shape->page_size;
  if (B > 0 && !seq_lens_host) return PA_ERR_INVALID_ARG;

  std::vector<int32_t> pages(B), nsplit(B);
  int64_t total_units = 0, total_pages = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t L = seq_lens_host[b];
    if (L < 0 || (int64_t)L > (int64_t)shape->max_pages_per_seq * S) return PA_ERR_INVALID_ARG;
    pages[b] = (L + S - 1) / S;
    total_units += (int64_t)std::max(pages[b], 1) * Hkv;
    total_pages += (int64_t)pages[b] * Hkv;
  }

  // Split counts.  Forced: min(forced, pages).  Auto: pages per split such
  // that the task count is about `waves` times the CTAs the GPU holds at
  // once (one CTA per task), never finer than min_chunk pages.  The default
  // of one wave caps a task at the average page load of a CTA slot.
  const int min_chunk = o.min_chunk_pages > 0 ? o.min_chunk_pages : kMinChunkPages;
  const int bundle_max = o.bundle_max_pages > 0 ? o.bundle_max_pages
                                                : (o.bundle_max_pages < 0 ? 0 : kBundleMaxPages);
  const int waves = o.waves > 0 ? o.waves : kPlanWaves;
  int32_t chunk = 0;
  if (forced_splits == 0) {
    const int64_t slots = (int64_t)num_sms * resident_ctas_per_sm(D, G);
    const int64_t target_tasks = (int64_t)waves * slots;
    chunk = (int32_t)std::max<int64_t>((total_units + target_tasks - 1) / target_tasks, min_chunk);
  }
  int64_t W64 = 0;
  int32_t max_splits = 1, max_size = 0, C = 0, nidx = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t np = pages[b];
    int32_t n = forced_splits > 0 ? std::max(1, std::min(forced_splits, np))
                                  : std::max(1, (np + chunk - 1) / chunk);
    n = std::min(n, (int32_t)kMaxSplits);
    nsplit[b] = n;
    max_splits = std::max(max_splits, n);
    max_size = std::max(max_size, (np + n - 1) / n);
    W64 += (int64_t)n * Hkv;
    if (n > 1) {
      C += Hkv;
      nidx += n * Hkv;
    }
  }
  if (W64 > INT32_MAX / 4) return PA_ERR_UNSUPPORTED;
  const int W = (int)W64;

  // CTAs: tasks longer than bundle_max get a CTA each (its warps share the
  // pages).  When there are many more tasks than CTA slots, the shorter ones,
  // which come last in longest-first order, go four to a CTA, one per warp.
  // That costs latency (a warp walks a whole task) but saves a CTA start per
  // task, which only pays off when the GPU runs several waves of them.
  const int64_t cta_slots = (int64_t)num_sms * resident_ctas_per_sm(D, G);
  const bool several = o.bundle_waves < 0 ||
                       W64 > (o.bundle_waves > 0 ? o.bundle_waves : kBundleWhenOver) * cta_slots;
  const int bundle_pages = several ? bundle_max : 0;
  int n_small = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t np = pages[b], n = nsplit[b];
    for (int j = 0; j < n; ++j) {
      const int32_t sz = (int32_t)((int64_t)np * (j + 1) / n - (int64_t)np * j / n);
      if (sz <= bundle_pages) n_small += Hkv;
    }
  }
  const int n_shared = W - n_small;  // longest first: the small tasks are the last ones
  const int NC = n_shared + (n_small + kWarpsPerCta - 1) / kWarpsPerCta;
  const Layout lay = layout(W, C, nidx, G, D);
  char* blob = nullptr;
  if (dst) {
    if (dst_bytes < lay.blob_bytes) {
      plan_out->blob_bytes = lay.blob_bytes;  // tells the caller how much is needed
      return PA_ERR_WORKSPACE;
    }
    blob = (char*)dst;
  } else if (alloc) {
    blob = (char*)malloc(lay.blob_bytes);
    if (!blob) return PA_ERR_NO_MEMORY;
  } else {
    return PA_ERR_INVALID_ARG;
  }

  // Tasks in (sequence, head, split) order are placed longest first with a
  // counting sort on their page count: deterministic, O(W + max_size).
  // Split j of a sequence with np pages and n splits covers
  // [floor(np*j/n), floor(np*(j+1)/n)).
  std::vector<int32_t> count(max_size + 2, 0);
  for (int b = 0; b < B; ++b) {
    const int32_t np = pages[b], n = nsplit[b];
    for (int j = 0; j < n; ++j) {
      const int32_t sz = (int32_t)((int64_t)np * (j + 1) / n - (int64_t)np * j / n);
      count[max_size - sz] += Hkv;
    }
  }
  std::vector<int32_t> start(max_size + 2, 0);
  for (int k = 1; k <= max_size + 1; ++k) start[k] = start[k - 1] + count[k - 1];

  int32_t* hdr = (int32_t*)blob;
  memset(blob, 0, lay.items_off);
  const uint64_t id = next_plan_id();
  hdr[0] = (int32_t)kMagic;
  hdr[1] = W;
  hdr[2] = C;
  hdr[3] = nidx;
  hdr[4] = (int32_t)(uint32_t)(id & 0xffffffffu);
  hdr[5] = (int32_t)(uint32_t)(id >> 32);
  hdr[6] = G;
  hdr[7] = D;
  hdr[8] = NC;
  hdr[9] = n_shared;
  int32_t* items = (int32_t*)(blob + lay.items_off);
  int32_t* slots = (int32_t*)(blob + lay.slots_off);
  int32_t* groups = (int32_t*)(blob + lay.groups_off);
  int32_t gcount = 0, icount = 0;
  for (int b = 0; b < B; ++b) {
    const int32_t np = pages[b], n = nsplit[b];
    for (int h = 0; h < Hkv; ++h) {
      if (n > 1) {
        groups[4 * gcount + 0] = b;
        groups[4 * gcount + 1] = h;
        groups[4 * gcount + 2] = n;
        groups[4 * gcount + 3] = icount;
        ++gcount;
      }
      for (int j = 0; j < n; ++j) {
        const int32_t lo = (int32_t)((int64_t)np * j / n);
        const int32_t hi = (int32_t)((int64_t)np * (j + 1) / n);
        const int32_t pos = start[max_size - (hi - lo)]++;
        uint32_t hw = (uint32_t)h;
        if (n > 1) hw |= kItemSplit;
        if (j == n - 1) hw |= kItemLast;
        items[4 * pos + 0] = b;
        items[4 * pos + 1] = (int32_t)hw;
        items[4 * pos + 2] = lo;
        items[4 * pos + 3] = hi;
        slots[2 * pos + 0] = n > 1 ? icount++ : -1;
        slots[2 * pos + 1] = n > 1 ? gcount - 1 : -1;
      }
    }
  }
  // zero the alignment gaps and the group counters, so the blob bytes are
  // fully defined
  const size_t used = lay.slots_off + 8 * (size_t)W;
  if (lay.groups_off > used) memset(blob + used, 0, lay.groups_off - used);
  memset(blob + lay.counters_off, 0, lay.blob_bytes - lay.counters_off);

  plan_out->shape = *shape;
  plan_out->num_work_items = W;
  plan_out->num_groups = C;
  plan_out->num_split_items = nidx;
  plan_out->max_splits = max_splits;
  plan_out->chunk_pages = forced_splits > 0 ? max_size : chunk;
  plan_out->warps_per_cta = kWarpsPerCta;
  plan_out->num_ctas = NC;
  plan_out->num_shared_ctas = n_shared;
  plan_out->owns_blob = dst ? 0 : 1;
  plan_out->plan_id = id;
  plan_out->blob_bytes = lay.blob_bytes;
  plan_out->workspace_bytes = lay.total;
  plan_out->host_blob = blob;
  plan_out->merge = o.merge;
  plan_out->l2_prefetch_pages = o.l2_prefetch_pages;
  plan_out->l2_prefetch_ctas = o.l2_prefetch_ctas;
  plan_out->q8_stages =
      o.q8_stages != 0 ? o.q8_stages : q8_stages_for(W, n_shared, total_pages, NC, cta_slots);
  plan_out->wait_limit_ns = o.wait_limit_ns;
  plan_out->early_kv = o.early_kv;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status_t pa_plan(const pa_shape_t* shape, const int32_t* seq_lens_host,
                               int32_t num_sms, int32_t forced_splits, pa_plan_t* plan_out) {
  return pa::plan_impl(shape, seq_lens_host, num_sms, forced_splits, nullptr, nullptr, 0, true,
                       plan_out);
}

extern "C" pa_status_t pa_plan_in(const pa_shape_t* shape, const int32_t* seq_lens_host,
                                  int32_t num_sms, int32_t forced_splits, void* host_buffer,
                                  size_t host_buffer_bytes, pa_plan_t* plan_out) {
  if (!host_buffer) return PA_ERR_INVALID_ARG;
  return pa::plan_impl(shape, seq_lens_host, num_sms, forced_splits, nullptr, host_buffer,
                       host_buffer_bytes, false, plan_out);
}

extern "C" pa_status_t pa_plan_ex(const pa_shape_t* shape, const int32_t* seq_lens_host,
                                  int32_t num_sms, int32_t forced_splits,
                                  const pa_plan_options_t* options, void* host_buffer,
                                  size_t host_buffer_bytes, pa_plan_t* plan_out) {
  return pa::plan_impl(shape, seq_lens_host, num_sms, forced_splits, options, host_buffer,
                       host_buffer_bytes, host_buffer == nullptr, plan_out);
}

extern "C" void pa_plan_free(pa_plan_t* plan) {
  if (!plan) return;
  if (plan->owns_blob) free(plan->host_blob);
  plan->owns_blob = 0;
  plan->host_blob = nullptr;
  plan->blob_bytes = 0;
}
