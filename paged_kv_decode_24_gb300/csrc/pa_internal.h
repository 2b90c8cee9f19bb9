// Internal constants and layouts shared by the planner and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "pagedattn.h"

#if defined(__CUDACC__)
#define PA_HD __host__ __device__
#else
#define PA_HD
#endif

namespace pa {

constexpr int kPageSize = 16;        // tokens per page (the only size built)
constexpr int kWarpsPerCta = 4;      // independent warp tasks per CTA
constexpr int kMaxSplits = 1024;     // per (sequence, KV head); the combine keeps weights in smem
constexpr int kMinChunkPages = 4;    // auto planner never cuts finer than this
constexpr uint32_t kMagic = 0x564b4150u;  // "PAKV"
constexpr size_t kSmemPerSm = 227 * 1024;
constexpr int kMaxCtaSmem = 227 * 1024;

// Item flags live in the top bits of the kv_head word.
constexpr uint32_t kItemSplit = 0x80000000u;  // writes a partial (o, lse) instead of out
constexpr uint32_t kItemLast = 0x40000000u;   // last page range of its sequence
constexpr uint32_t kItemHeadMask = 0x0000ffffu;

// Page-copy pipeline depth per warp.
PA_HD constexpr int stages_for(int head_dim) { return head_dim == 64 ? 6 : 3; }

// Shared memory of one warp's pipeline; the kernel carves exactly this.
struct WarpSmem {
  int tile, k_off, v_off, bar_off, page_off, p_off, a_off, bytes;
};

PA_HD constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

PA_HD constexpr WarpSmem warp_smem(int head_dim, int group, int stages) {
  WarpSmem w{};
  w.tile = kPageSize * head_dim * 2;
  w.k_off = 0;
  w.v_off = stages * w.tile;
  w.bar_off = 2 * stages * w.tile;
  w.page_off = w.bar_off + 2 * stages * 8;
  w.p_off = align_up(w.page_off + stages * 4, 16);
  w.a_off = w.p_off + kPageSize * group * 4;
  w.bytes = align_up(w.a_off + (group < 4 ? 4 : group) * 4, 128);
  return w;
}

inline int cta_smem_bytes(int head_dim, int group) {
  return kWarpsPerCta * warp_smem(head_dim, group, stages_for(head_dim)).bytes;
}

inline int resident_warps_per_sm(int head_dim, int group) {
  int ctas = (int)(kSmemPerSm / (size_t)(cta_smem_bytes(head_dim, group) + 1024));
  if (ctas < 1) ctas = 1;
  if (ctas * kWarpsPerCta > 64) ctas = 64 / kWarpsPerCta;
  return ctas * kWarpsPerCta;
}

// Workspace = [plan blob | lse partials | o partials].
// Blob = header (16 x int32) | items (int4 each) | groups (int4 each) | split index list (int32).
// header: [0] magic [1] items [2] groups [3] index entries [4] plan_id lo [5] plan_id hi
//         [6] group size [7] head_dim.  Kernels check words 0..3 against their launch.
struct Layout {
  size_t items_off, groups_off, idx_off, blob_bytes, lse_off, o_off, total;
};

inline size_t align_sz(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline Layout layout(int items, int groups, int nidx, int group, int head_dim) {
  Layout l{};
  l.items_off = 64;
  l.groups_off = l.items_off + 16 * (size_t)items;
  l.idx_off = l.groups_off + 16 * (size_t)groups;
  l.blob_bytes = align_sz(l.idx_off + 4 * (size_t)nidx, 16);
  l.lse_off = align_sz(l.blob_bytes, 256);
  l.o_off = align_sz(l.lse_off + 4 * (size_t)items * group, 256);
  l.total = align_sz(l.o_off + 4 * (size_t)items * group * head_dim, 256);
  return l;
}

// Validation shared by every entry point.
pa_status_t check_shape(const pa_shape_t* s);

}  // namespace pa
