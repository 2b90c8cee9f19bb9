// Split decode attention with the two per-page products on tensor cores.
//
// Same tasks, CTA shapes, pipeline and merge as decode_kernel.cuh (see there
// for the task / bundle / split scheme).  What differs is how a page is moved
// and multiplied.
//
// Page copies: each K or V tile of a (page, KV head) arrives by TMA tensor
// copies (cp.async.bulk.tensor.4d) from a tensor map over the pool
// [P][Hkv][16][D].  The map's coordinate is the physical page, so the
// block-table gather is the copy's own address computation.  Boxes are
// 16 rows x 64 halves with the 128-byte swizzle: 16-byte chunk c of row r
// lands at chunk c ^ (r % 8).  That makes every ldmatrix below
// conflict-free.
//
// Products, for the 16 tokens of a page and the G <= 8 query heads of the
// KV head (padded to 8):
//   S^T[16 tok x 8 heads]  = K[16 x D] . Q^T[D x 8]
//       D/16 mma.m16n8k16 (A = K tile by ldmatrix, B = q held in registers)
//   O^T[D x 8 heads]      += V^T[D x 16 tok] . P^T[16 tok x 8]
//       D/16 m-tiles x 2 (A = V tile by ldmatrix.trans).  B = P^T in fp16 is
//       split into hi = fp16(p) and lo = fp16(p - hi), so the product keeps
//       about 22 bits of p.  Accumulation is fp32 throughout.
// The online softmax runs on the S^T fragments.  A thread holds tokens g and
// g+8 of heads 2t and 2t+1 (g = lane/4, t = lane%4), so a head's page max is
// a 3-shuffle reduction over g.  P^T reaches the B-fragment layout with four
// shuffles and two byte permutes per hi/lo half.  Per page and warp this
// is 3*D/16 mma and 2*D/16 ldmatrix in place of about 512 FMAs per lane on
// CUDA cores.  The rows of a partial page past the sequence end are zeroed in
// the V fragments (their weight is 0, but they may hold anything, NaN too).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "decode_kernel.cuh"
#include "device_common.cuh"
#include "pa_internal.h"

namespace pa {

__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap* map, int c0, int c1,
                                            int c2, int c3, uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3, %4, %5}], [%6], %7;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3), "r"(bar),
      "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                        uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2,
                                          uint32_t& r3) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
               : "r"(addr));
}

// D += A . B for one m16n8k16 tile, fp32 accumulators; A and B both fp16
// (T = __half) or both bf16 (T = __nv_bfloat16).
template <typename T = __half>
__device__ __forceinline__ void mma_16816(float* d, uint32_t a0, uint32_t a1, uint32_t a2,
                                          uint32_t a3, uint32_t b0, uint32_t b1) {
  if constexpr (std::is_same<T, __half>::value) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
  }
}

__device__ __forceinline__ uint32_t pack_half2(float lo, float hi) {
  const __half2 h = __floats2half2_rn(lo, hi);
  return *reinterpret_cast<const uint32_t*>(&h);
}

__device__ __forceinline__ float2 unpack_half2(uint32_t v) {
  return __half22float2(*reinterpret_cast<const __half2*>(&v));
}

// Byte offset of 16-byte chunk `chunk` (of 8 per 128-byte row) of row `row`
// in a 128-byte-swizzled box of 16 rows.
__device__ __forceinline__ uint32_t swz(int row, int chunk) {
  return (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
}

// Shared memory of the tensor-core kernel, per CTA: NW rings of NSH tiles
// (1024-aligned for the swizzle), then per-warp bookkeeping.
template <int D, int NW, int NSH>
struct TcLayout {
  static constexpr int TILE = kPageSize * D * 2;      // a multiple of 1024
  static constexpr int RING = NSH * TILE;             // per warp
  static constexpr int RINGS = NW * RING;
  static constexpr int BARS = 0;                      // NSH mbarriers
  static constexpr int PAGES = align_up(8 * NSH, 16); // NSH page ids
  static constexpr int NROW = PAGES + align_up(4 * NSH, 16);  // new K row, new V row
  static constexpr int EXTRA = align_up(NROW + 2 * D * 2, 16);
  static constexpr int FLAG = RINGS + NW * EXTRA;
  static constexpr int BYTES = FLAG + 16 + 1024;      // + slack to align the base to 1024
};

template <typename T, int D, int G, int NW, int NSH, bool EARLY>
__global__ void __launch_bounds__(NW * 32, 4)
    split_decode_tc_kernel(const __grid_constant__ SplitParams p) {
  static_assert(G <= 8, "the mma tile holds at most 8 query heads");
  using L = TcLayout<D, NW, NSH>;
  constexpr int KSTEPS = D / 16;  // QK k-steps, also PV m-tiles
  constexpr int BOXES = D / 64;
  extern __shared__ unsigned char smem_dyn[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int g = lane >> 2;
  const int t = lane & 3;
  const uint32_t ring = smem_u32(base) + warp * L::RING;
  unsigned char* extra = base + L::RINGS + warp * L::EXTRA;
  const uint32_t bars = smem_u32(extra) + L::BARS;
  int* page_ids = reinterpret_cast<int*>(extra + L::PAGES);
  T* nrow = reinterpret_cast<T*>(extra + L::NROW);
  int* cta_failed = reinterpret_cast<int*>(base + L::FLAG);
  int* cta_last = cta_failed + 1;

  if ((int)blockIdx.x >= p.num_ctas) return;  // whole CTA
  // Plan data is written only by pa_plan_upload (a copy, which the
  // programmatic launch does not overlap): it may be read before the wait.
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
  if (threadIdx.x == 0) {
    *cta_failed = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSH; ++s) mbar_init(bars + 8 * s, 1);
    fence_barrier_init();
  }
  __syncthreads();

  pdl_launch_dependents();
  // Everything the previous kernel wrote is visible after the wait.  With
  // early_kv the task's seq_len, block-table entries and first page copies
  // come before it; q and the new rows always come after it.
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
  const int pstart = coop ? warp : 0;
  const int pstride = coop ? NW : 1;
  const int npk = coop ? (warp < npg ? (npg - warp + NW - 1) / NW : 0) : npg;

  // What the previous kernel may write (the new rows, q) is read by
  // load_inputs: here, after the wait, or with early_kv after the first
  // page copies and the wait.
  int k_app = -1;
  uint32_t qb[KSTEPS][2];
  auto load_inputs = [&]() {
    // Fused append: k_app is this warp's page index that holds position L-1,
    // or -1.  The new K and V rows are staged in this warp's shared memory.
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

    // Q^T fragments (B operand of S^T = K Q^T): column n = head g of the group,
    // rows = dims.  Heads past G are zero.
    {
      const T* qrow =
          static_cast<const T*>(p.q) + ((size_t)b * p.num_q_heads + (size_t)kvh * G + g) * D;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        if (g < G) {
          qb[kk][0] = __ldg(reinterpret_cast<const unsigned int*>(qrow + kk * 16 + 2 * t));
          qb[kk][1] = __ldg(reinterpret_cast<const unsigned int*>(qrow + kk * 16 + 2 * t + 8));
        } else {
          qb[kk][0] = qb[kk][1] = 0u;
        }
      }
    }
  };
  if constexpr (!EARLY) load_inputs();

  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages + pg0;
  const uint64_t policy = l2_evict_first_policy();
  int bt_cur = lane < npg ? __ldg(bt_row + lane) : -1;
  int bt_nxt = 32 + lane < npg ? __ldg(bt_row + 32 + lane) : -1;
  int bt_w = 0;

  // Issue half-tile hi of this warp (K tile of its page hi/2 for even hi, V
  // tile for odd hi) into stage hi % NSH; warp-collective, lane 0 issues.
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
      const uint32_t bar = bars + 8 * s;
      if ((pg0 + j) * kPageSize >= seq_len) {
        phys = -1;
      } else if (phys < 0 || phys >= p.num_pages) {
        if ((hi & 1) == 0) set_status(p.status, PA_DEV_BAD_PAGE);
        phys = -1;
      }
      page_ids[s] = phys;
      fence_proxy_async_smem();
      if (phys >= 0) {
        const CUtensorMap* map = (hi & 1) ? &p.tmap_v : &p.tmap_k;
        mbar_arrive_expect_tx(bar, L::TILE);
#pragma unroll
        for (int bx = 0; bx < BOXES; ++bx)
          tma_load_4d(ring + s * L::TILE + bx * 2048, map, bx * 64, 0, kvh, phys, bar, policy);
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

  // Online softmax state of heads 2t and 2t+1 (identical across the 8 lanes
  // of a t), and this lane's share of their running sums.
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_part[2] = {0.f, 0.f};
  float o[KSTEPS][4];  // O^T: dims 16*mt + g (+8), heads 2t, 2t+1
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  const float qs = p.qscale;
  // lanes whose P^T entries this lane needs (see the header comment)
  const int src1 = (2 * t) * 4 + (g >> 1);
  const int src2 = (2 * t + 1) * 4 + (g >> 1);
  const unsigned int perm = (g & 1) ? 0x7632u : 0x5410u;

  bool failed = false;
  int hfail = 0;
  for (int k = 0; k < npk; ++k) {
    const int hk = 2 * k;
    const int sk = hk % NSH;
    if (!__all_sync(kFull, mbar_wait_bounded(bars + 8 * sk, (hk / NSH) & 1, p.wait_ns))) {
      failed = true;
      hfail = hk;
      break;
    }
    const int phys = page_ids[sk];
    const int j = pstart + k * pstride;
    const int nvalid = phys < 0 ? 0 : min(kPageSize, seq_len - (pg0 + j) * kPageSize);
    const bool append_here = (k == k_app) && phys >= 0;
    const int r_app = (seq_len - 1) % kPageSize;
    const uint32_t ktile = ring + sk * L::TILE;
    if (append_here) {
      // 16-byte chunk i of the new row: box i/8, chunk i%8, swizzled by the row
      for (int i = lane; i < D / 8; i += 32) {
        const uint4 v = reinterpret_cast<const uint4*>(nrow)[i];
        *reinterpret_cast<uint4*>(base + (ktile - smem_u32(base)) + (i >> 3) * 2048 +
                                  swz(r_app, i & 7)) = v;
      }
      __syncwarp();
    }

    uint32_t pb_hi0 = 0, pb_hi1 = 0, pb_lo0 = 0, pb_lo1 = 0;
    float al0 = 1.f, al1 = 1.f;
    bool rescale = false;
    if (nvalid > 0) {
      // ---- S^T = K . Q^T
      float c[4] = {0.f, 0.f, 0.f, 0.f};
      const int kr = (lane & 7) + 8 * ((lane >> 3) & 1);  // token row this lane addresses
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        const int chunk = (kk & 3) * 2 + (lane >> 4);
        uint32_t a0, a1, a2, a3;
        ldsm_x4(ktile + (kk >> 2) * 2048 + swz(kr, chunk), a0, a1, a2, a3);
        mma_16816<T>(c, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
      }
      float s0 = c[0] * qs, s1 = c[1] * qs, s2 = c[2] * qs, s3 = c[3] * qs;
      if (g >= nvalid) s0 = s1 = -INFINITY;
      if (g + 8 >= nvalid) s2 = s3 = -INFINITY;
      // ---- online softmax for heads 2t (s0, s2) and 2t+1 (s1, s3)
      float mA = fmaxf(s0, s2), mB = fmaxf(s1, s3);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(kFull, mA, m));
        mB = fmaxf(mB, __shfl_xor_sync(kFull, mB, m));
      }
      const float nA = fmaxf(m_run[0], mA), nB = fmaxf(m_run[1], mB);
      const bool deadA = nA == -INFINITY, deadB = nB == -INFINITY;
      al0 = deadA ? 1.f : ex2(m_run[0] - nA);
      al1 = deadB ? 1.f : ex2(m_run[1] - nB);
      const float p0 = deadA ? 0.f : ex2(s0 - nA);
      const float p2 = deadA ? 0.f : ex2(s2 - nA);
      const float p1 = deadB ? 0.f : ex2(s1 - nB);
      const float p3 = deadB ? 0.f : ex2(s3 - nB);
      l_part[0] = l_part[0] * al0 + (p0 + p2);
      l_part[1] = l_part[1] * al1 + (p1 + p3);
      m_run[0] = nA;
      m_run[1] = nB;
      rescale = __any_sync(kFull, al0 != 1.f || al1 != 1.f);
      // ---- P^T into B fragments, hi and lo parts in the element type
      const uint32_t h01 = Elem<T>::from_f2(p0, p1);  // token g: heads 2t, 2t+1
      const uint32_t h23 = Elem<T>::from_f2(p2, p3);  // token g+8
      const float2 f01 = Elem<T>::to_f2(h01), f23 = Elem<T>::to_f2(h23);
      const uint32_t l01 = Elem<T>::from_f2(p0 - f01.x, p1 - f01.y);
      const uint32_t l23 = Elem<T>::from_f2(p2 - f23.x, p3 - f23.y);
      pb_hi0 = __byte_perm(__shfl_sync(kFull, h01, src1), __shfl_sync(kFull, h01, src2), perm);
      pb_hi1 = __byte_perm(__shfl_sync(kFull, h23, src1), __shfl_sync(kFull, h23, src2), perm);
      pb_lo0 = __byte_perm(__shfl_sync(kFull, l01, src1), __shfl_sync(kFull, l01, src2), perm);
      pb_lo1 = __byte_perm(__shfl_sync(kFull, l23, src1), __shfl_sync(kFull, l23, src2), perm);
    }
    // the K stage is free: refill it
    __syncwarp();
    if (hk + NSH < nhalf) issue(hk + NSH);

    const int hv = hk + 1;
    const int sv = hv % NSH;
    if (!__all_sync(kFull, mbar_wait_bounded(bars + 8 * sv, (hv / NSH) & 1, p.wait_ns))) {
      failed = true;
      hfail = hv;
      break;
    }
    const uint32_t vtile = ring + sv * L::TILE;
    if (append_here) {
      for (int i = lane; i < D / 8; i += 32) {
        const uint4 v = reinterpret_cast<const uint4*>(nrow + D)[i];
        *reinterpret_cast<uint4*>(base + (vtile - smem_u32(base)) + (i >> 3) * 2048 +
                                  swz(r_app, i & 7)) = v;
      }
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
      if (rescale) {
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
      }
      // ---- O^T += V^T . P^T (hi and lo)
      // masks for tokens 2t, 2t+1 and 2t+8, 2t+9 (zero the rows past nvalid)
      const uint32_t mk0 = (2 * t < nvalid ? 0x0000ffffu : 0u) | (2 * t + 1 < nvalid ? 0xffff0000u : 0u);
      const uint32_t mk8 =
          (2 * t + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * t + 9 < nvalid ? 0xffff0000u : 0u);
      const int q4 = lane >> 3;
      const int vr = (q4 >> 1) * 8 + (lane & 7);  // token row this lane addresses
#pragma unroll
      for (int mt = 0; mt < KSTEPS; ++mt) {
        const int chunk = (mt & 3) * 2 + (q4 & 1);
        uint32_t a0, a1, a2, a3;
        ldsm_x4_t(vtile + (mt >> 2) * 2048 + swz(vr, chunk), a0, a1, a2, a3);
        if (nvalid < kPageSize) {
          a0 &= mk0;
          a1 &= mk0;
          a2 &= mk8;
          a3 &= mk8;
        }
        mma_16816<T>(o[mt], a0, a1, a2, a3, pb_hi0, pb_hi1);
        mma_16816<T>(o[mt], a0, a1, a2, a3, pb_lo0, pb_lo1);
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
        mbar_wait_bounded(bars + 8 * (h % NSH), (h / NSH) & 1, kDrainWaitNs);
      *cta_failed = 1;
    }
    __syncwarp();
  } else if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NSH; ++s) mbar_inval(bars + 8 * s);
  }

  // full running sums of heads 2t, 2t+1: add the shares of the 8 lanes of t
#pragma unroll
  for (int m = 4; m <= 16; m <<= 1) {
    l_part[0] += __shfl_xor_sync(kFull, l_part[0], m);
    l_part[1] += __shfl_xor_sync(kFull, l_part[1], m);
  }

  if (!coop) {
    // ---- a task of its own: normalise into this warp's (now free) ring,
    // then write coalesced
    if (failed) {
      if (is_split) mark_split_missing(p.part_lse, slot, G, lane);
      return;
    }
    float* stage = reinterpret_cast<float*>(base + warp * L::RING);  // [G][D]
    const float inv0 = l_part[0] > 0.f ? 1.f / l_part[0] : 0.f;
    const float inv1 = l_part[1] > 0.f ? 1.f / l_part[1] : 0.f;
#pragma unroll
    for (int mt = 0; mt < KSTEPS; ++mt) {
      const int d0 = 16 * mt + g;
      if (2 * t < G) {
        stage[(2 * t) * D + d0] = o[mt][0] * inv0;
        stage[(2 * t) * D + d0 + 8] = o[mt][2] * inv0;
      }
      if (2 * t + 1 < G) {
        stage[(2 * t + 1) * D + d0] = o[mt][1] * inv1;
        stage[(2 * t + 1) * D + d0 + 8] = o[mt][3] * inv1;
      }
    }
    if (is_split && g == 0) {
      if (2 * t < G)
        p.part_lse[(size_t)slot * G + 2 * t] = l_part[0] > 0.f ? m_run[0] + lg2(l_part[0]) : -INFINITY;
      if (2 * t + 1 < G)
        p.part_lse[(size_t)slot * G + 2 * t + 1] =
            l_part[1] > 0.f ? m_run[1] + lg2(l_part[1]) : -INFINITY;
    }
    __syncwarp();
    if (!is_split) {
      T* dst = static_cast<T*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)kvh * G) * D;
      for (int i = lane * 2; i < G * D; i += 64)
        *reinterpret_cast<uint32_t*>(dst + i) = Elem<T>::from_f2(stage[i], stage[i + 1]);
    } else {
      float* dst = p.part_o + (size_t)slot * G * D;
      for (int i = lane * 4; i < G * D; i += 128)
        *reinterpret_cast<float4*>(dst + i) = *reinterpret_cast<const float4*>(stage + i);
      if (p.fuse_merge) split_finish_warp<T, D>(merge_target(p, sg.y, grp, G), lane);
    }
    return;
  }

  // ---- shared task: merge the NW warp states in shared memory (rings are free)
  __syncthreads();
  if (*cta_failed) {
    if (is_split && warp == 0) mark_split_missing(p.part_lse, slot, G, lane);
    return;
  }
  float* st = reinterpret_cast<float*>(base);  // [NW][2G + G*D]
  constexpr int SLOT = 2 * G + G * D;
  float* mine = st + warp * SLOT;
  if (g == 0) {
    if (2 * t < G) {
      mine[2 * t] = m_run[0];
      mine[G + 2 * t] = l_part[0];
    }
    if (2 * t + 1 < G) {
      mine[2 * t + 1] = m_run[1];
      mine[G + 2 * t + 1] = l_part[1];
    }
  }
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) {
    const int d0 = 16 * mt + g;
    if (2 * t < G) {
      mine[2 * G + (2 * t) * D + d0] = o[mt][0];
      mine[2 * G + (2 * t) * D + d0 + 8] = o[mt][2];
    }
    if (2 * t + 1 < G) {
      mine[2 * G + (2 * t + 1) * D + d0] = o[mt][1];
      mine[2 * G + (2 * t + 1) * D + d0 + 8] = o[mt][3];
    }
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
    split_finish_cta<T, D, NW>(merge_target(p, sg.y, grp, G), cta_last);
}

}  // namespace pa
