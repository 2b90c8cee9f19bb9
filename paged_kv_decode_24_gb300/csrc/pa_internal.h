// Internal constants and layouts shared by the planner and the kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>

#include "pagedattn.h"

#if defined(__CUDACC__)
#define PA_HD __host__ __device__
#else
#define PA_HD
#endif

namespace pa {

constexpr int kPageSize = 16;        // tokens per page (the only size built)
constexpr int kWarpsPerCta = 4;      // warps sharing one task's pages
constexpr int kMaxSplits = 1024;     // per (sequence, KV head)
constexpr int kMinChunkPages = 48;   // auto planner never cuts finer than this
constexpr int kBundleMaxPages = 8;   // tasks this short are bundled one per warp
constexpr int kPlanWaves = 1;        // auto planner: tasks ~ waves x resident CTAs
constexpr int kL2PrefetchPages = 2;  // pages per warp asked of L2 before the wait on the previous kernel
constexpr int kBundleWhenOver = 3;   // bundle short tasks only past this many tasks per CTA slot
constexpr int kQ8ShortPagesPerWarp = 12;  // 8-bit kernel: two page stages up to this mean
constexpr uint32_t kMagic = 0x564b4150u;  // "PAKV"
constexpr size_t kSmemPerSm = 227 * 1024;
constexpr int kMaxCtaSmem = 227 * 1024;

constexpr uint64_t kDefaultWaitNs = 1000000000ull;  // a plan's wait limit of 0 means ~1 s

// The wait limit a kernel uses for a plan's wait_limit_ns (0: the default).
inline uint64_t wait_limit_or_default(uint64_t ns) { return ns ? ns : kDefaultWaitNs; }

// Code formats of the 8-bit caches (per-row fp32 scales in both).
constexpr int kCodeInt8 = 0;  // two's-complement int8 codes
constexpr int kCodeE4m3 = 1;  // OCP E4M3 bytes

// Item flags live in the top bits of the kv_head word.
constexpr uint32_t kItemSplit = 0x80000000u;  // writes a partial (o, lse) instead of out
constexpr uint32_t kItemLast = 0x40000000u;   // last page range of its sequence
constexpr uint32_t kItemHeadMask = 0x0000ffffu;

// Per-warp ring depth in half-stages (one K or V tile of one page each).
PA_HD constexpr int half_stages_for(int head_dim) { return head_dim == 64 ? 6 : 3; }
// The 8-bit caches' ring holds whole pages (K and V code tiles and their
// row scales on one barrier): 3 pages of D = 128 or 6 of D = 64 keep about
// 12 KB per warp in flight, as the fp16 ring does.
// At D = 128 a plan may ask for 2 (pa_plan_t.q8_stages) when its tasks are
// short.
PA_HD constexpr int q8_page_stages_for(int head_dim) { return head_dim == 64 ? 6 : 3; }

// Shared memory of one warp of the split-decode kernel; the kernel carves
// exactly this, and the CTA holds kWarpsPerCta of them.
struct WarpSmem {
  int tile, ring, bar, page, p, a, nrow, bytes;
};

PA_HD constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

PA_HD constexpr WarpSmem warp_smem(int head_dim, int group, int nsh) {
  WarpSmem w{};
  w.tile = kPageSize * head_dim * 2;         // one K or V tile of one (page, head)
  w.ring = 0;                                // nsh tiles
  w.bar = nsh * w.tile;                      // nsh mbarriers
  w.page = w.bar + 8 * nsh;                  // nsh physical page ids
  w.p = align_up(w.page + 4 * nsh, 16);      // [16][group] softmax weights, stored as (p, p)
  w.a = w.p + kPageSize * group * 8;         // [group] rescale factors
  w.nrow = align_up(w.a + 4 * (group < 4 ? 4 : group), 16);  // new K row, new V row (append)
  w.bytes = align_up(w.nrow + 2 * head_dim * 2, 128);
  return w;
}

inline int cta_smem_bytes(int head_dim, int group) {
  return kWarpsPerCta * warp_smem(head_dim, group, half_stages_for(head_dim)).bytes;
}

// Resident split-decode CTAs per SM, from shared memory and the registers
// per thread the kernels compile to (the planner runs on the host without a
// GPU): 108 for the CUDA-core kernel (G = 1), 128 for the tensor-core and
// 8-bit kernels, whose launch bounds ask for four CTAs per SM.
inline int resident_ctas_per_sm(int head_dim, int group) {
  int by_smem = (int)(kSmemPerSm / (size_t)(cta_smem_bytes(head_dim, group) + 1024));
  const int regs = group <= 1 ? 108 : 128;
  int by_regs = 65536 / (kWarpsPerCta * 32 * regs);
  int n = by_smem < by_regs ? by_smem : by_regs;
  if (n * kWarpsPerCta > 64) n = 64 / kWarpsPerCta;
  return n < 1 ? 1 : n;
}

// Workspace = [plan blob | lse partials | o partials].
// Blob = header (16 x int32) | tasks (int4 each) | task slots (int2 each:
// partial slot, -1 = direct output, and the task's group) | groups (int4
// each: seq, kv head, splits, first slot) | group counters (int32 each,
// zero in the plan: split tasks of the group finished so far in a launch;
// the task that completes the group merges it and sets it back to zero).
// header: [0] magic [1] tasks [2] groups [3] partial slots [4] plan_id lo
//         [5] plan_id hi [6] group size [7] head_dim [8] CTAs [9] shared CTAs.
// Kernels check words 0..3 and 8..9 against their launch.  The partials of a
// group's splits occupy consecutive slots, in split order.  CTA i < shared
// CTAs runs task i with all its warps; the CTAs after it run the remaining
// (short) tasks four at a time, one per warp, in task order.
struct Layout {
  size_t items_off, slots_off, groups_off, counters_off, blob_bytes, lse_off, o_off, total;
};

inline size_t align_sz(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline Layout layout(int items, int groups, int nslots, int group, int head_dim) {
  Layout l{};
  l.items_off = 64;
  l.slots_off = l.items_off + 16 * (size_t)items;
  l.groups_off = align_sz(l.slots_off + 8 * (size_t)items, 16);
  l.counters_off = l.groups_off + 16 * (size_t)groups;
  l.blob_bytes = align_sz(l.counters_off + 4 * (size_t)groups, 16);
  l.lse_off = align_sz(l.blob_bytes, 256);
  l.o_off = align_sz(l.lse_off + 4 * (size_t)nslots * group, 256);
  l.total = align_sz(l.o_off + 4 * (size_t)nslots * group * head_dim, 256);
  return l;
}

// Multi-token attention: a tile is a number of query rows (tokens x heads of
// one KV head): 128 for the tcgen05 kernel (one TMEM lane per row), 64 for
// the mma.sync kernel.  Blob = header (16 x int32: [0] magic [1] tiles [2] B
// [3] T [4,5] plan_id [6] G [7] D [8] rows per tile) | tiles (int4:
// sequence, KV head, first token, tokens) | cu (int32 [B+1], row offsets).
constexpr int kPrefillRows = 64;
constexpr int kPrefillRowsTc5 = 128;
constexpr uint32_t kPrefillMagic = 0x564b4650u;  // "PFKV"

struct PrefillLayout {
  size_t tiles_off, cu_off, blob_bytes;
};

inline PrefillLayout prefill_layout(int tiles, int batch) {
  PrefillLayout l{};
  l.tiles_off = 64;
  l.cu_off = l.tiles_off + 16 * (size_t)tiles;
  l.blob_bytes = align_sz(l.cu_off + 4 * ((size_t)batch + 1), 256);
  return l;
}

// Validation shared by every entry point.
pa_status_t check_shape(const pa_shape_t* s);

// Every host-side check of pa_decode_attention (shape, plan against shape,
// pointers, scale, workspace size), in the order that call makes them.
// Returns PA_OK for a call that would launch, and also for batch == 0, which
// launches nothing (*launches is then false).
pa_status_t check_decode_call(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                              const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* seq_lens, float scale,
                              const void* out, const void* workspace, size_t workspace_bytes,
                              const int32_t* dev_status, bool* launches);

}  // namespace pa
