// Split decode attention over a paged KV cache, on CUDA cores.  Used for MHA
// (G = 1), where one multiply-add per K or V element keeps up with HBM;
// decode_tc.cuh holds the tensor-core form used for G >= 2.
//
// A task is (sequence b, KV head g, page range [pg0, pg1)).  A CTA either
// shares one task among its NW warps (warp w takes pages w, w+NW, ...) or,
// for short tasks, runs up to NW of them, one per warp.  Each warp streams
// its pages through a private ring of NSH
// shared-memory half-stages: a K tile or a V tile of one page, each one
// contiguous (page, head) slice of S*D halves.  Lane 0 fills a half-stage
// with a single 1-D bulk copy that completes on that stage's mbarrier.
// Separate K and V stages let the V copy of a page land while the page's
// scores are being computed, without doubling the ring.
//
// The warp serves all G query heads of its KV head from that single read of
// K and V (GQA: MonadKai/xLLM, KV cache with GQA).  It keeps an online softmax
// per query head (xLLM introduction, SoftMax with an online normalizer):
// running max m, running sum l, and an accumulator rescaled whenever m grows.
// At the end the NW warp states (m, l, acc) meet in shared memory and merge
// with the same log-sum-exp rule the split merge uses.  No atomics touch
// data, and every reduction has a fixed order, so reruns are bit-identical.
// This follows the from-scratch engine article, section 3.4: shared memory
// instead of atomicAdd.
//
// Lane roles on a page of 16 tokens:
//   QK: lane = (row group rg = lane/8, chunk c = lane%8).  Lane (rg, c) takes
//       tokens rg, rg+4, rg+8, rg+12 and, in each row, dims [8c, 8c+8) (and
//       [64+8c, 64+8c+8) when D = 128).  Eight lanes read one 128-byte run
//       per shared-memory load, conflict-free.  The 4*G partial dot products
//       are summed over the 8 chunk lanes by a reduce-scatter: 3 shuffle
//       rounds, halving the values each round.
//   PV: lane owns output dims [D/32*lane, D/32*(lane+1)) of every head and
//       walks the 16 rows.  The weights are read from shared memory as
//       broadcasts, stored twice over (p, p) so that one 64-bit load is a
//       whole operand.
// The multiply-adds of both products use the packed two-wide FP32 FMA
// (fma.rn.f32x2) on pairs of adjacent dims, so each instruction does two.
//
// With k_new/v_new given (pa_append_decode_attention), the warp whose pages
// include position L-1 also appends the new token.  It overwrites that row of
// the K and V tiles in shared memory before computing on them, and writes
// both rows to the pool once its copies of that page have landed.  No other
// task touches that page, so the write races with nothing.
//
// A task whose sequence has more than one split writes its normalised output
// and log2-sum-exp to the workspace; the group's last task to finish merges
// them into the output (split_merge.cuh; swiftLLM, paged attention v2 /
// Flash-Decoding), or, with fuse_merge off, combine_kernel does after this
// kernel.  Otherwise the task writes its output directly.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math.h>

#include "device_common.cuh"
#include "elem.cuh"
#include "pa_internal.h"
#include "split_merge.cuh"

namespace pa {

// Element pointers (q, pools, new rows, out) hold the kernel's element type
// (fp16 or bf16; fp16 for the 8-bit-cache kernel's q, new rows and out).
struct SplitParams {
  const void* q;
  const void* k_pages;
  const void* v_pages;
  const void* k_new;  // non-null: append the new token (fused pa_kv_append)
  const void* v_new;
  const int32_t* block_table;
  const int32_t* seq_lens;
  void* out;
  const int32_t* ws_header;
  const int4* items;
  const int2* item_slots;  // {partial slot (-1 = direct output), group} of each task
  const int4* groups;      // {sequence, KV head, splits, first slot} of each split group
  int* counters;           // per group: its split tasks finished so far (split_merge.cuh)
  float* part_lse;
  float* part_o;
  int32_t* status;
  float qscale;  // scale * log2(e): scores are kept in base 2
  int32_t batch, num_q_heads, num_kv_heads, max_pages, num_pages;
  int32_t num_items, num_groups, num_split_items, num_ctas;  // must match the header
  int32_t num_shared;  // CTAs [0, num_shared) share a task; the rest run up to NW short tasks
  CUtensorMap tmap_k;  // pools as 4-D tensors [P][Hkv][16][D] for the TMA tensor copies
  CUtensorMap tmap_v;
  // 8-bit cache (split_decode_q8_kernel only): INT8 codes or E4M3 bytes
  // [P][Hkv][16][D] and per-row scales [P][Hkv][16]; the fused append
  // writes them.
  const int8_t* k_codes;
  const int8_t* v_codes;
  const float* k_scales;
  const float* v_scales;
  // L2 prefetch before the wait on the previous kernel: CTAs [0, pf_ctas)
  // prefetch the first pf_pages (<= 32) pages of each warp's share.
  int32_t pf_pages, pf_ctas;
  // 1: the last split task of each group merges it (split_merge.cuh);
  // 0: split tasks only write partials, and combine_kernel merges them.
  int32_t fuse_merge;
  uint64_t wait_ns;  // bound of each wait on a page copy (the plan's wait_limit_ns)
  // 1: seq_lens, the block table and the first page copies come before the
  // wait on the previous kernel (the plan's early_kv); 0: after it.
  int32_t early_kv;
};

// A split task's slot and group agree with each other and with the task.
__device__ __forceinline__ bool split_slot_ok(const SplitParams& p, int2 sg, int4 grp, int b,
                                              int kvh) {
  return sg.x >= 0 && sg.x < p.num_split_items && sg.y >= 0 && sg.y < p.num_groups &&
         grp.x == b && grp.y == kvh && grp.z >= 2 && grp.z <= kMaxSplits && grp.w >= 0 &&
         sg.x >= grp.w && sg.x < grp.w + grp.z && grp.w + grp.z <= p.num_split_items;
}

// The merge target of split group gi (its record grp) of this launch.
__device__ __forceinline__ MergeTarget merge_target(const SplitParams& p, int gi, int4 grp, int G) {
  MergeTarget t;
  t.lse = p.part_lse;
  t.o = p.part_o;
  t.out = p.out;
  t.counter = p.counters + gi;
  t.grp = grp;
  t.G = G;
  t.num_q_heads = p.num_q_heads;
  return t;
}

// Before the wait on the previous kernel, lane k of a warp may prefetch page
// k of the warp's share of task `it` (page j = warp + k * NW of a shared
// task, j = k of a warp's own task) into L2.  Returns that page's physical
// index, or -1.  The prefetch is only a hint: the previous kernel may still
// rewrite the block table, so the entry is read through L2 (ld.global.cg
// leaves no stale line in L1 for the reads after the wait), every index is
// bounded to its buffer, and nothing depends on the prefetched bytes.
template <int NW>
__device__ __forceinline__ int prefetch_page_of_lane(const SplitParams& p, int4 it, bool coop,
                                                     int warp, int lane) {
  if (lane >= p.pf_pages) return -1;
  const int b = it.x, kvh = (int)((uint32_t)it.y & kItemHeadMask), pg0 = it.z, pg1 = it.w;
  if (b < 0 || b >= p.batch || kvh >= p.num_kv_heads || pg0 < 0 || pg1 < pg0 || pg1 > p.max_pages)
    return -1;
  const int j = coop ? warp + lane * NW : lane;
  if (j >= pg1 - pg0) return -1;
  const int phys = __ldcg(p.block_table + (size_t)b * p.max_pages + pg0 + j);
  return (phys >= 0 && phys < p.num_pages) ? phys : -1;
}

template <int D, int G>
struct Geometry {
  static constexpr int CH = D / 64;                   // 16-byte K chunks per lane per row
  static constexpr int DPL = D / 32;                  // output dims per lane
  static constexpr int NV = 4 * G;                    // partial scores per lane
  static constexpr int NVL = NV >= 8 ? NV / 8 : 1;    // scores per lane after reduce-scatter
  static constexpr int HEAD_LANES = 8 / G;            // chunk lanes that share one head
};

// d = a * b + c on two fp32 lanes with one instruction.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "mov.b64 rc, {%6, %7};\n\t"
      "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
  return d;
}

// Sum the N values held by each of the 8 lanes of a row group (lane bits
// 0..2) so that afterwards lane c holds complete sums.  Each round sends
// half of the remaining values to the partner lane and keeps the other
// half: bit set -> keep the upper half.  After the rounds lane c holds value
// indices [c*N/8, c*N/8 + N/8) when N >= 8.  With N = 4 the last round has one
// value left and both partners end with the same sum.
template <int N, int MASK>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
  if constexpr (MASK >= 1) {
    if constexpr (N >= 2) {
      const bool up = (lane & MASK) != 0;
#pragma unroll
      for (int k = 0; k < N / 2; ++k) {
        const float lo = v[k], hi = v[k + N / 2];
        const float send = up ? lo : hi;
        const float keep = up ? hi : lo;
        v[k] = keep + __shfl_xor_sync(kFull, send, MASK);
      }
      reduce_scatter<N / 2, MASK / 2>(v, lane);
    } else {
      v[0] += __shfl_xor_sync(kFull, v[0], MASK);
      reduce_scatter<1, MASK / 2>(v, lane);
    }
  }
}

// d = a * (s, s) on two fp32 lanes with one instruction.
__device__ __forceinline__ float2 fmul2s(float2 a, float s) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %4};\n\t"
      "mul.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(s));
  return d;
}

// Shared memory of one warp (bytes); the CTA holds NW of these.
template <int D, int G, int NSH>
struct WarpLayout {
  static constexpr WarpSmem W = warp_smem(D, G, NSH);
  static constexpr int TILE = W.tile;
  static constexpr int RING = W.ring;
  static constexpr int BAR = W.bar;
  static constexpr int PAGE = W.page;
  static constexpr int P = W.p;
  static constexpr int A = W.a;
  static constexpr int NROW = W.nrow;
  static constexpr int BYTES = W.bytes;
};

// Four CTAs (16 warps) per SM for G <= 4: the register cap is 128.
template <int G>
struct MinCtas {
  static constexpr int value = G <= 4 ? 4 : 2;
};

template <typename T, int D, int G, int NW, int NSH, bool EARLY>
__global__ void __launch_bounds__(NW * 32, MinCtas<G>::value)
    split_decode_kernel(const SplitParams p) {
  using Geo = Geometry<D, G>;
  using L = WarpLayout<D, G, NSH>;
  extern __shared__ __align__(128) unsigned char smem_raw[];
  __shared__ int cta_failed, cta_last;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rg = lane >> 3;
  const int c = lane & 7;
  unsigned char* ws = smem_raw + warp * L::BYTES;
  const uint32_t ws_u32 = smem_u32(ws);
  int* page_ids = reinterpret_cast<int*>(ws + L::PAGE);
  float* p_s = reinterpret_cast<float*>(ws + L::P);
  float* a_s = reinterpret_cast<float*>(ws + L::A);

  if ((int)blockIdx.x >= p.num_ctas) return;  // whole CTA
  // The task list is written only by pa_plan_upload (a copy, which the
  // programmatic launch does not overlap), so it may be read before the
  // wait on the previous kernel.
  const int4 hdr = *reinterpret_cast<const int4*>(p.ws_header);
  const int2 hdr_ctas = *reinterpret_cast<const int2*>(p.ws_header + 8);
  // CTA -> task(s) by arithmetic: no descriptor load on the startup path
  const bool coop = (int)blockIdx.x < p.num_shared;  // CTA-uniform
  const int first = coop ? (int)blockIdx.x : p.num_shared + ((int)blockIdx.x - p.num_shared) * NW;
  const int count = coop ? 1 : min(NW, p.num_items - first);
  const int task = coop ? first : (warp < count ? first + warp : -1);
  int4 it = make_int4(0, 0, 0, 0);
  int2 sg = make_int2(-1, -1);  // {partial slot, group}
  int4 grp = make_int4(-1, -1, 0, 0);
  if (task >= 0 && task < p.num_items) {
    it = p.items[task];
    sg = p.item_slots[task];
    if (sg.y >= 0 && sg.y < p.num_groups) grp = p.groups[sg.y];
  }
  const int slot = sg.x;

  if (task >= 0 && task < p.num_items && (int)blockIdx.x < p.pf_ctas) {
    const int phys = prefetch_page_of_lane<NW>(p, it, coop, warp, lane);
    if (phys >= 0) {
      const size_t off = ((size_t)phys * p.num_kv_heads + ((uint32_t)it.y & kItemHeadMask)) *
                         (kPageSize * D);
      prefetch_l2_bulk(static_cast<const T*>(p.k_pages) + off, L::TILE);
      prefetch_l2_bulk(static_cast<const T*>(p.v_pages) + off, L::TILE);
    }
  }
  if (threadIdx.x == 0) cta_failed = 0;
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSH; ++s) mbar_init(ws_u32 + L::BAR + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();

  pdl_launch_dependents();
  // Everything the previous kernel wrote is visible after the wait.  With
  // early_kv the task's seq_len, block-table entries and first page copies
  // come before it (nothing still running writes them); q and the new rows
  // always come after it.
  if constexpr (!EARLY) pdl_wait_primary();

  if (hdr.x != (int)kMagic || hdr.y != p.num_items || hdr.z != p.num_groups ||
      hdr.w != p.num_split_items || hdr_ctas.x != p.num_ctas || hdr_ctas.y != p.num_shared ||
      count < 1 || first < 0 || first + count > p.num_items) {
    if (threadIdx.x == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;  // CTA-uniform
  }
  if (task < 0) return;  // idle warp of a partial bundle; bundles never sync the CTA
  const int b = it.x;
  const uint32_t hw = (uint32_t)it.y;
  const int kvh = (int)(hw & kItemHeadMask);
  const bool is_split = (hw & kItemSplit) != 0;
  const bool is_last = (hw & kItemLast) != 0;
  const int pg0 = it.z, pg1 = it.w;
  if (b < 0 || b >= p.batch || kvh >= p.num_kv_heads || pg0 < 0 || pg1 < pg0 ||
      pg1 > p.max_pages || (is_split && !split_slot_ok(p, sg, grp, b, kvh))) {
    if (lane == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;  // all warps of a shared task see the same task
  }
  const int Lmax = p.max_pages * kPageSize;
  int seq_len = p.seq_lens[b];
  if (seq_len < 0 || seq_len > Lmax) {
    if (lane == 0) set_status(p.status, PA_DEV_BAD_SEQ_LEN);
    seq_len = min(max(seq_len, 0), Lmax);
  }
  if (is_last && seq_len > pg1 * kPageSize && lane == 0)
    set_status(p.status, PA_DEV_PLAN_MISMATCH);
  const int npg = pg1 - pg0;
  // this warp's pages of the task: j = pstart + k * pstride, k < npk
  const int pstart = coop ? warp : 0;
  const int pstride = coop ? NW : 1;
  const int npk = coop ? (warp < npg ? (npg - warp + NW - 1) / NW : 0) : npg;

  // What the previous kernel may write (the new rows, q) is read by
  // load_inputs: here, after the wait, or with early_kv after the first
  // page copies and the wait.
  int k_app = -1;
  T* nrow = reinterpret_cast<T*>(ws + L::NROW);  // [2][D]: K row, V row
  float2 qf[G][Geo::CH * 4];
  auto load_inputs = [&]() {
    // Fused append: k_app is this warp's page index that holds position L-1,
    // or -1.  The new K and V rows are staged in this warp's shared memory now.
    if (p.k_new != nullptr && seq_len > 0) {
      const int j_app = (seq_len - 1) / kPageSize - pg0;
      if (j_app >= pstart && j_app < npg && (j_app - pstart) % pstride == 0) {
        k_app = (j_app - pstart) / pstride;
        const size_t src = ((size_t)b * p.num_kv_heads + kvh) * D;
        for (int i = lane; i < D / 8; i += 32) {
          reinterpret_cast<uint4*>(nrow)[i] =
              __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.k_new) + src) + i);
          reinterpret_cast<uint4*>(nrow + D)[i] =
              __ldg(reinterpret_cast<const uint4*>(static_cast<const T*>(p.v_new) + src) + i);
        }
        __syncwarp();
      }
    }

    // q for the G heads of this KV head, pre-scaled by scale*log2(e), as pairs.
    {
      const T* qb = static_cast<const T*>(p.q) + ((size_t)b * p.num_q_heads + (size_t)kvh * G) * D;
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int ch = 0; ch < Geo::CH; ++ch) {
          const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qb + h * D + ch * 64 + c * 8));
          float2 f[4];
          elem8_to_float2x4<T>(raw, f);
#pragma unroll
          for (int e = 0; e < 4; ++e)
            qf[h][ch * 4 + e] = make_float2(f[e].x * p.qscale, f[e].y * p.qscale);
        }
    }
  };
  if constexpr (!EARLY) load_inputs();

  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages + pg0;
  const size_t page_stride = (size_t)p.num_kv_heads * kPageSize * D;  // halves
  const T* kbase = static_cast<const T*>(p.k_pages) + (size_t)kvh * kPageSize * D;
  const T* vbase = static_cast<const T*>(p.v_pages) + (size_t)kvh * kPageSize * D;
  const uint64_t policy = l2_evict_first_policy();

  // Block-table entries of the task, 32 per window: lane k of the current
  // window holds entry 32*w + k.  The next window is loaded one window ahead.
  int bt_cur = lane < npg ? __ldg(bt_row + lane) : -1;
  int bt_nxt = 32 + lane < npg ? __ldg(bt_row + 32 + lane) : -1;
  int bt_w = 0;

  // Issue half-tile hi of this warp: page k = hi/2 of the warp (task page
  // j = pstart + k*pstride), K tile for even hi, V tile for odd hi, into stage
  // hi % NSH.  Warp-collective (the block-table entry comes by shuffle);
  // lane 0 issues.  hi grows by one per call.  A page past the sequence end
  // or with an invalid index is not copied: its barrier is released empty and
  // the page is masked.
  auto issue = [&](int hi) {
    const int j = pstart + (hi >> 1) * pstride;
    if ((j >> 5) != bt_w) {  // j grows by at most NW <= 32 between calls
      ++bt_w;
      bt_cur = bt_nxt;
      const int idx = 32 * (bt_w + 1) + lane;
      bt_nxt = idx < npg ? __ldg(bt_row + idx) : -1;
    }
    int phys = __shfl_sync(kFull, bt_cur, j & 31);
    if (lane == 0) {
      const int s = hi % NSH;
      const uint32_t bar = ws_u32 + L::BAR + 8 * s;
      if ((pg0 + j) * kPageSize >= seq_len) {
        phys = -1;
      } else if (phys < 0 || phys >= p.num_pages) {
        if ((hi & 1) == 0) set_status(p.status, PA_DEV_BAD_PAGE);
        phys = -1;
      }
      page_ids[s] = phys;
      fence_proxy_async_smem();
      if (phys >= 0) {
        const T* src = ((hi & 1) ? vbase : kbase) + (size_t)phys * page_stride;
        mbar_arrive_expect_tx(bar, L::TILE);
        bulk_g2s(ws_u32 + L::RING + s * L::TILE, src, L::TILE, bar, policy);
      } else {
        mbar_arrive(bar);
      }
    }
  };

  const int nhalf = 2 * npk;
  const int npre = nhalf < NSH ? nhalf : NSH;
  for (int hi = 0; hi < npre; ++hi) issue(hi);

  if constexpr (EARLY) {
    pdl_wait_primary();
    load_inputs();
  }

  // Softmax state of this lane's head: m is shared by the lanes of a head,
  // l_part is this lane's own share of the running sum.
  float m_run = -INFINITY, l_part = 0.f;
  const int myh = (G == 1) ? 0 : ((c * Geo::NVL) >> 2);
  // acc[h][e] = output dims lane*DPL + 2e, +2e+1 of head h
  float2 acc[G][Geo::DPL / 2];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < Geo::DPL / 2; ++e) acc[h][e] = make_float2(0.f, 0.f);

  bool failed = false;
  int hfail = 0;
  for (int k = 0; k < npk; ++k) {
    const int hk = 2 * k;
    const int sk = hk % NSH;
    if (!__all_sync(kFull, mbar_wait_bounded(ws_u32 + L::BAR + 8 * sk, (hk / NSH) & 1, p.wait_ns))) {
      failed = true;
      hfail = hk;
      break;
    }
    const int phys = page_ids[sk];
    const int j = pstart + k * pstride;
    const int nvalid = phys < 0 ? 0 : min(kPageSize, seq_len - (pg0 + j) * kPageSize);
    const bool append_here = (k == k_app) && phys >= 0;
    const int r_app = (seq_len - 1) % kPageSize;
    if (append_here) {
      T* row = reinterpret_cast<T*>(ws + L::RING + sk * L::TILE) + r_app * D;
      for (int i = lane; i < D / 8; i += 32)
        reinterpret_cast<uint4*>(row)[i] = reinterpret_cast<const uint4*>(nrow)[i];
      __syncwarp();
    }

    if (nvalid > 0) {
      // ---- scores of the page's 16 tokens for the G heads
      const T* Ks = reinterpret_cast<const T*>(ws + L::RING + sk * L::TILE);
      float v[Geo::NV];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = rg + 4 * i;
        float2 a2[G];
#pragma unroll
        for (int h = 0; h < G; ++h) a2[h] = make_float2(0.f, 0.f);
#pragma unroll
        for (int ch = 0; ch < Geo::CH; ++ch) {
          const uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * D + ch * 64 + c * 8);
          float2 kf[4];
          elem8_to_float2x4<T>(raw, kf);
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int e = 0; e < 4; ++e) a2[h] = ffma2(qf[h][ch * 4 + e], kf[e], a2[h]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) v[h * 4 + i] = a2[h].x + a2[h].y;
      }
      reduce_scatter<Geo::NV, 4>(v, lane);

      // ---- online softmax update for this lane's head
      float pmax = -INFINITY;
#pragma unroll
      for (int e = 0; e < Geo::NVL; ++e) {
        const int vi = (Geo::NV >= 8) ? c * Geo::NVL + e : (c >> 1);
        const int t = rg + 4 * (vi & 3);
        if (t >= nvalid) v[e] = -INFINITY;
        pmax = fmaxf(pmax, v[e]);
      }
#pragma unroll
      for (int m = 1; m < Geo::HEAD_LANES; m <<= 1)
        pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, m));
      pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 8));
      pmax = fmaxf(pmax, __shfl_xor_sync(kFull, pmax, 16));
      const float m_new = fmaxf(m_run, pmax);
      const bool dead = (m_new == -INFINITY);
      const float alpha = dead ? 1.f : ex2(m_run - m_new);
      float psum = 0.f;
#pragma unroll
      for (int e = 0; e < Geo::NVL; ++e) {
        const int vi = (Geo::NV >= 8) ? c * Geo::NVL + e : (c >> 1);
        const int t = rg + 4 * (vi & 3);
        const float pk = dead ? 0.f : ex2(v[e] - m_new);
        *reinterpret_cast<float2*>(p_s + (t * G + (vi >> 2)) * 2) = make_float2(pk, pk);
        psum += pk;
      }
      l_part = l_part * alpha + psum;
      m_run = m_new;
      if (rg == 0 && (c & (Geo::HEAD_LANES - 1)) == 0) a_s[myh] = alpha;
      __syncwarp();
    }
    // the K stage is free: refill it with the half-tile NSH ahead
    if (hk + NSH < nhalf) issue(hk + NSH);

    const int hv = hk + 1;
    const int sv = hv % NSH;
    if (!__all_sync(kFull, mbar_wait_bounded(ws_u32 + L::BAR + 8 * sv, (hv / NSH) & 1, p.wait_ns))) {
      failed = true;
      hfail = hv;
      break;
    }
    if (append_here) {
      T* row = reinterpret_cast<T*>(ws + L::RING + sv * L::TILE) + r_app * D;
      for (int i = lane; i < D / 8; i += 32)
        reinterpret_cast<uint4*>(row)[i] = reinterpret_cast<const uint4*>(nrow + D)[i];
      // both copies of this page have landed, so the pool rows can be written
      const size_t dst = (((size_t)phys * p.num_kv_heads + kvh) * kPageSize + r_app) * D;
      uint4* kw = reinterpret_cast<uint4*>(static_cast<T*>(const_cast<void*>(p.k_pages)) + dst);
      uint4* vw = reinterpret_cast<uint4*>(static_cast<T*>(const_cast<void*>(p.v_pages)) + dst);
      for (int i = lane; i < D / 8; i += 32) {
        kw[i] = reinterpret_cast<const uint4*>(nrow)[i];
        vw[i] = reinterpret_cast<const uint4*>(nrow + D)[i];
      }
      __syncwarp();
    }
    if (nvalid > 0) {
      // ---- rescale and accumulate p . V
      float al[G];
      bool rescale = false;
#pragma unroll
      for (int h = 0; h < G; ++h) {
        al[h] = a_s[h];
        rescale |= (al[h] != 1.f);
      }
      if (rescale) {
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < Geo::DPL / 2; ++e) acc[h][e] = fmul2s(acc[h][e], al[h]);
      }
      const T* Vs = reinterpret_cast<const T*>(ws + L::RING + sv * L::TILE);
      auto pv_row = [&](int t) {
        float2 pp[G];
        if constexpr (G >= 2) {
#pragma unroll
          for (int h = 0; h < G; h += 2) {
            const float4 w4 = *reinterpret_cast<const float4*>(p_s + (t * G + h) * 2);
            pp[h] = make_float2(w4.x, w4.y);
            pp[h + 1] = make_float2(w4.z, w4.w);
          }
        } else {
          pp[0] = *reinterpret_cast<const float2*>(p_s + t * 2);
        }
        float2 vf[Geo::DPL / 2];
        if constexpr (Geo::DPL == 4) {
          const uint2 raw = *reinterpret_cast<const uint2*>(Vs + t * D + lane * 4);
          vf[0] = Elem<T>::to_f2(raw.x);
          vf[1] = Elem<T>::to_f2(raw.y);
        } else {
          vf[0] = Elem<T>::to_f2(*reinterpret_cast<const uint32_t*>(Vs + t * D + lane * 2));
        }
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int e = 0; e < Geo::DPL / 2; ++e) acc[h][e] = ffma2(pp[h], vf[e], acc[h][e]);
      };
      // rows past nvalid are skipped: their weight is 0, but the row may hold
      // anything, NaN included
      if (nvalid == kPageSize) {
#pragma unroll
        for (int t = 0; t < kPageSize; ++t) pv_row(t);
      } else {
#pragma unroll
        for (int t = 0; t < kPageSize; ++t)
          if (t < nvalid) pv_row(t);
      }
    }
    __syncwarp();
    if (hv + NSH < nhalf) issue(hv + NSH);
  }

  if (failed) {
    // A copy did not land in time.  Report it and let the copies already
    // issued finish (bounded).  The task writes nothing.
    if (lane == 0) {
      set_status(p.status, PA_DEV_TIMEOUT);
      const int last = min(nhalf, hfail + NSH);
      for (int h = hfail; h < last; ++h)
        mbar_wait_bounded(ws_u32 + L::BAR + 8 * (h % NSH), (h / NSH) & 1, kDrainWaitNs);
      cta_failed = 1;
    }
    __syncwarp();
  } else if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSH; ++s) mbar_inval(ws_u32 + L::BAR + 8 * s);
  }

  // l: sum this lane's share over the lanes of its head (G == 1: lanes c and
  // c^1 hold the same values, so bit 0 is not summed).
#pragma unroll
  for (int m = (G == 1 ? 2 : 1); m < Geo::HEAD_LANES; m <<= 1)
    l_part += __shfl_xor_sync(kFull, l_part, m);
  l_part += __shfl_xor_sync(kFull, l_part, 8);
  l_part += __shfl_xor_sync(kFull, l_part, 16);
  float o[G][Geo::DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int e = 0; e < Geo::DPL / 2; ++e) {
      o[h][2 * e] = acc[h][e].x;
      o[h][2 * e + 1] = acc[h][e].y;
    }

  if (!coop) {
    // ---- a task of its own: normalise and write from registers
    if (failed) {
      if (is_split) mark_split_missing(p.part_lse, slot, G, lane);
      return;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const int rep = h * Geo::HEAD_LANES;  // lane (rg 0, c = h*HEAD_LANES) holds head h's state
      const float lh = __shfl_sync(kFull, l_part, rep);
      const float mh = __shfl_sync(kFull, m_run, rep);
      const float inv = lh > 0.f ? 1.f / lh : 0.f;
      if (!is_split) {
        T* dst = static_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)kvh * G + h) * D +
                 lane * Geo::DPL;
        if constexpr (Geo::DPL == 4) {
          uint2 wv;
          wv.x = Elem<T>::from_f2(o[h][0] * inv, o[h][1] * inv);
          wv.y = Elem<T>::from_f2(o[h][2] * inv, o[h][3] * inv);
          *reinterpret_cast<uint2*>(dst) = wv;
        } else {
          *reinterpret_cast<uint32_t*>(dst) = Elem<T>::from_f2(o[h][0] * inv, o[h][1] * inv);
        }
      } else {
        float* dst = p.part_o + ((size_t)slot * G + h) * D + lane * Geo::DPL;
        if constexpr (Geo::DPL == 4) {
          *reinterpret_cast<float4*>(dst) =
              make_float4(o[h][0] * inv, o[h][1] * inv, o[h][2] * inv, o[h][3] * inv);
        } else {
          *reinterpret_cast<float2*>(dst) = make_float2(o[h][0] * inv, o[h][1] * inv);
        }
        if (lane == 0) p.part_lse[(size_t)slot * G + h] = lh > 0.f ? mh + lg2(lh) : -INFINITY;
      }
    }
    if (is_split && p.fuse_merge) split_finish_warp<T, D>(merge_target(p, sg.y, grp, G), lane);
    return;
  }

  // ---- shared task: merge the NW warp states in shared memory (rings are free)
  __syncthreads();
  if (cta_failed) {
    if (is_split && warp == 0) mark_split_missing(p.part_lse, slot, G, lane);
    return;
  }
  float* st = reinterpret_cast<float*>(smem_raw);  // [NW][2G + G*D]
  constexpr int SLOT = 2 * G + G * D;
  float* mine = st + warp * SLOT;
  if (rg == 0 && (c & (Geo::HEAD_LANES - 1)) == 0) {
    mine[myh] = m_run;
    mine[G + myh] = l_part;
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float* dst = mine + 2 * G + h * D + lane * Geo::DPL;
#pragma unroll
    for (int d = 0; d < Geo::DPL; ++d) dst[d] = o[h][d];
  }
  __syncthreads();

  for (int idx = threadIdx.x; idx < G * D; idx += NW * 32) {
    const int h = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < NW; ++w) M = fmaxf(M, st[w * SLOT + h]);
    float Z = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < NW; ++w) {
        const float sc = ex2(st[w * SLOT + h] - M);  // 0 for an empty warp (m = -inf)
        Z = fmaf(st[w * SLOT + G + h], sc, Z);
        O = fmaf(st[w * SLOT + 2 * G + h * D + d], sc, O);
      }
    }
    const float r = Z > 0.f ? O / Z : 0.f;
    if (!is_split) {
      static_cast<T*>(p.out)[((size_t)b * p.num_q_heads + (size_t)kvh * G + h) * D + d] =
          Elem<T>::from_f(r);
    } else {
      p.part_o[((size_t)slot * G + h) * D + d] = r;
      if (d == 0) p.part_lse[(size_t)slot * G + h] = Z > 0.f ? M + lg2(Z) : -INFINITY;
    }
  }
  if (is_split && p.fuse_merge)  // CTA-uniform: one task
    split_finish_cta<T, D, NW>(merge_target(p, sg.y, grp, G), &cta_last);
}

}  // namespace pa
