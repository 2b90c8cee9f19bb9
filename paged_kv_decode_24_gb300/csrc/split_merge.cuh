// The merge step of split decoding (Flash-Decoding; the reduce step of
// swiftLLM's paged attention v2), run by the split task that finishes its
// group last, at the end of the split kernel itself.
//
// A group is one (sequence, KV head) whose pages are cut into ns splits.
// Each split task writes a normalised partial output o_s and its
// log2-sum-exp lse_s into the group's consecutive workspace slots, then adds
// one to the group's counter.  The task that brings the counter to ns
// merges, for each query head of the KV head,
//     M = max_s lse_s,   w_s = 2^(lse_s - M),   out = sum_s w_s o_s / sum_s w_s
// (out = 0 when every split is empty), and sets the counter back to 0, so
// the next launch on the same uploaded plan starts from zero.  Nothing else
// touches a counter during a launch once it reaches ns, and the next launch
// reads it only after the kernel boundary.
//
// Memory order: the task's threads write its partial, meet at a barrier
// (__syncthreads or __syncwarp), and one thread adds to the counter with
// atom.acq_rel.gpu: a release that covers the writes the barrier ordered
// before it, and an acquire of every earlier release on the counter.  The
// merging task's threads meet that thread at a barrier again and read the
// partials with ld.global.cg (from L2, never a stale L1 line).
//
// Which task merges depends on timing, and a group may mix tasks that a CTA
// shares with tasks run by one warp.  Both merge with the same function, one
// 4-float chunk (a head, four dims) at a time over all splits in split
// order, so the output is the same bits whichever task merges.
#pragma once

#include <math.h>

#include "device_common.cuh"
#include "elem.cuh"

namespace pa {

// What the merge of one group reads and writes.
struct MergeTarget {
  const float* lse;  // workspace partial lse, [slot][G]
  const float* o;    // workspace partial outputs, [slot][G][D]
  void* out;         // [B][Hq][D], the kernel's output element type
  int* counter;      // this group's counter
  int4 grp;          // {sequence, KV head, splits, first slot}
  int G, num_q_heads;
};

// A split task that gave up (a bounded wait ran out) writes no partial.  It
// marks its slot's log-sum-exps NaN instead, so that a separate combine
// kernel leaves the group's output unwritten rather than merging what an
// earlier call left in the slot.  (The merge inside the split kernel never
// runs for such a group: the task does not count itself finished.)  Lanes
// 0 .. G-1 of one warp call it.
__device__ __forceinline__ void mark_split_missing(float* part_lse, int slot, int G, int lane) {
  if (slot >= 0 && lane < G) part_lse[(size_t)slot * G + lane] = __int_as_float(0x7fc00000);
}

// Splits whose partials one thread loads at once: 16, or 4 for a group of
// at most 4 splits (fewer predicated-off loads).  A group always takes the
// same batch, so its output bits never depend on which task merges.
constexpr int kMergeBatch = 16;
constexpr int kMergeBatchSmall = 4;

__device__ __forceinline__ int atom_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// The merged chunk (head h, dims d0 .. d0+3) of the group: a running
// (max, sum, accumulator) over batches of NB splits.
template <int D, int NB>
__device__ __forceinline__ float4 merge_chunk(const MergeTarget& t, int h, int d0) {
  const int ns = t.grp.z, off = t.grp.w;
  const float* lb = t.lse + (size_t)off * t.G + h;
  const float* ob = t.o + ((size_t)off * t.G + h) * D + d0;
  const size_t sstride = (size_t)t.G * D;
  float m = -INFINITY, z = 0.f;
  float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int s0 = 0; s0 < ns; s0 += NB) {
    float l[NB];
    float4 x[NB];
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const int s = s0 + u;
      l[u] = -INFINITY;
      x[u] = make_float4(0.f, 0.f, 0.f, 0.f);
      if (s < ns) {
        l[u] = __ldcg(lb + (size_t)s * t.G);
        x[u] = __ldcg(reinterpret_cast<const float4*>(ob + (size_t)s * sstride));
      }
    }
    float mn = m;
#pragma unroll
    for (int u = 0; u < NB; ++u) mn = fmaxf(mn, l[u]);
    if (mn == -INFINITY) continue;  // every split so far is empty
    const float sc = ex2(m - mn);   // 0 while m is still -inf
    z *= sc;
    a.x *= sc;
    a.y *= sc;
    a.z *= sc;
    a.w *= sc;
#pragma unroll
    for (int u = 0; u < NB; ++u) {
      const float e = ex2(l[u] - mn);  // 0 for an empty or absent split
      z += e;
      a.x = fmaf(e, x[u].x, a.x);
      a.y = fmaf(e, x[u].y, a.y);
      a.z = fmaf(e, x[u].z, a.z);
      a.w = fmaf(e, x[u].w, a.w);
    }
    m = mn;
  }
  if (!(z > 0.f)) return make_float4(0.f, 0.f, 0.f, 0.f);
  return make_float4(a.x / z, a.y / z, a.z / z, a.w / z);
}

// Chunks u = first, first + stride, ... of the group's G * D / 4.
template <typename T, int D>
__device__ __forceinline__ void merge_chunks(const MergeTarget& t, int first, int stride) {
  constexpr int CPH = D / 4;  // chunks per head
  for (int u = first; u < t.G * CPH; u += stride) {
    const int h = u / CPH, d0 = (u % CPH) * 4;
    const float4 r = t.grp.z <= kMergeBatchSmall ? merge_chunk<D, kMergeBatchSmall>(t, h, d0)
                                                 : merge_chunk<D, kMergeBatch>(t, h, d0);
    uint2 v;
    v.x = Elem<T>::from_f2(r.x, r.y);
    v.y = Elem<T>::from_f2(r.z, r.w);
    *reinterpret_cast<uint2*>(static_cast<T*>(t.out) +
                              ((size_t)t.grp.x * t.num_q_heads + (size_t)t.grp.y * t.G + h) * D +
                              d0) = v;
  }
}

// A split task run by one warp, after every lane has written its share of
// the partial.  Warp-uniform; merges the group if this task completes it.
template <typename T, int D>
__device__ __forceinline__ void split_finish_warp(const MergeTarget& t, int lane) {
  __syncwarp();
  int last = 0;
  if (lane == 0) last = atom_add_acq_rel_gpu(t.counter, 1) == t.grp.z - 1;
  last = __shfl_sync(kFull, last, 0);
  if (!last) return;
  __syncwarp();
  merge_chunks<T, D>(t, lane, 32);
  if (lane == 0) *t.counter = 0;
}

// A split task shared by the NW warps of a CTA, after every thread has
// written its share of the partial.  CTA-uniform; `flag` is one shared int.
template <typename T, int D, int NW>
__device__ __forceinline__ void split_finish_cta(const MergeTarget& t, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) *flag = atom_add_acq_rel_gpu(t.counter, 1) == t.grp.z - 1;
  __syncthreads();
  if (!*flag) return;
  merge_chunks<T, D>(t, threadIdx.x, NW * 32);
  if (threadIdx.x == 0) *t.counter = 0;
}

}  // namespace pa
