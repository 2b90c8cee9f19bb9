// Split decode attention over a paged KV cache.
//
// One warp = one task (sequence b, KV head g, page range [pg0, pg1)).  The
// warp streams its pages through a private ring of NS shared-memory stages.
// Lane 0 issues one 1-D bulk copy per (page, head) slice of K and of V; each
// slice is one contiguous run of S*D halves, so one copy moves a whole tile
// with no address math per row.  Copies complete on an mbarrier.  The warp
// serves all G query heads of its KV head from that single read of K and V
// (GQA: MonadKai/xLLM, KV cache with GQA).  It keeps an online softmax
// (xLLM introduction, SoftMax with an online normalizer): a running max m, a
// running sum l and a rescaled accumulator per query head.
//
// Lane roles on a page of 16 tokens:
//   QK: lane = (row group rg = lane/8, chunk c = lane%8).  Lane (rg, c) takes
//       tokens rg, rg+4, rg+8, rg+12 and, in each row, dims [8c, 8c+8) (and
//       [64+8c, 64+8c+8) when D = 128).  Eight lanes read one 128-byte run
//       per shared-memory load, so the loads are conflict-free.  The 4*G
//       partial dot products are summed over the 8 chunk lanes by a
//       reduce-scatter (3 shuffle rounds, halving the values each round)
//       instead of 4*G separate butterflies.
//   PV: lane owns output dims [D/32*lane, D/32*(lane+1)) of every head and
//       walks the 16 rows; the softmax weights come from shared memory as
//       broadcasts.
// All reductions are shuffles or shared memory in a fixed order, with no
// atomics on data, so a rerun is bit-identical.  This follows the
// from-scratch engine article, section 3.4: shared memory instead of
// atomicAdd.
//
// A task whose sequence has more than one split writes its normalised
// output and log2-sum-exp to the workspace.  combine_kernel merges those
// (swiftLLM, paged attention v2 / Flash-Decoding).  Otherwise the task
// writes the fp16 output directly.
#pragma once

#include <cuda_fp16.h>
#include <math.h>

#include "device_common.cuh"
#include "pa_internal.h"

namespace pa {

struct SplitParams {
  const __half* q;
  const __half* k_pages;
  const __half* v_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  __half* out;
  const int32_t* ws_header;
  const int4* items;
  float* part_lse;
  float* part_o;
  int32_t* status;
  float qscale;  // scale * log2(e): scores are kept in base 2
  int32_t batch, num_q_heads, num_kv_heads, max_pages, num_pages;
  int32_t num_items, num_groups, num_split_items;  // must match the workspace header
};

template <int D, int G>
struct Geometry {
  static constexpr int CH = D / 64;                   // 16-byte K chunks per lane per row
  static constexpr int DPL = D / 32;                  // output dims per lane
  static constexpr int NV = 4 * G;                    // partial scores per lane
  static constexpr int NVL = NV >= 8 ? NV / 8 : 1;    // scores per lane after reduce-scatter
  static constexpr int HEAD_LANES = 8 / G;            // chunk lanes that share one head
};

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

__device__ __forceinline__ void half8_to_float(const uint4& raw, float* f) {
  const __half2* h2 = reinterpret_cast<const __half2*>(&raw);
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 x = __half22float2(h2[e]);
    f[2 * e] = x.x;
    f[2 * e + 1] = x.y;
  }
}

template <int D, int G, int NS>
__global__ void __launch_bounds__(kWarpsPerCta * 32)
    split_decode_kernel(const SplitParams p) {
  using Geo = Geometry<D, G>;
  constexpr WarpSmem L = warp_smem(D, G, NS);
  extern __shared__ __align__(128) unsigned char smem_raw[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int rg = lane >> 3;
  const int c = lane & 7;
  unsigned char* ws = smem_raw + warp * L.bytes;
  const uint32_t ws_u32 = smem_u32(ws);
  int* page_ids = reinterpret_cast<int*>(ws + L.page_off);
  float* p_s = reinterpret_cast<float*>(ws + L.p_off);  // [16][G] softmax weights of a page
  float* a_s = reinterpret_cast<float*>(ws + L.a_off);  // [G] rescale factors of a page

  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(ws_u32 + L.bar_off + 16 * s, 1);
      mbar_init(ws_u32 + L.bar_off + 16 * s + 8, 1);
    }
    fence_barrier_init();
  }
  __syncwarp();

  pdl_launch_dependents();
  pdl_wait_primary();  // everything the previous kernel wrote is visible after this

  const int item_idx = blockIdx.x * kWarpsPerCta + warp;
  if (item_idx >= p.num_items) return;

  const int4 hdr = *reinterpret_cast<const int4*>(p.ws_header);
  if (hdr.x != (int)kMagic || hdr.y != p.num_items || hdr.z != p.num_groups ||
      hdr.w != p.num_split_items) {
    if (lane == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;
  }
  const int4 it = p.items[item_idx];
  const int b = it.x;
  const uint32_t hw = (uint32_t)it.y;
  const int kvh = (int)(hw & kItemHeadMask);
  const bool is_split = (hw & kItemSplit) != 0;
  const bool is_last = (hw & kItemLast) != 0;
  const int pg0 = it.z, pg1 = it.w;
  if (b < 0 || b >= p.batch || kvh >= p.num_kv_heads || pg0 < 0 || pg1 < pg0 ||
      pg1 > p.max_pages) {
    if (lane == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;
  }
  const int Lmax = p.max_pages * kPageSize;
  int seq_len = p.seq_lens[b];
  if (seq_len < 0 || seq_len > Lmax) {
    if (lane == 0) set_status(p.status, PA_DEV_BAD_SEQ_LEN);
    seq_len = min(max(seq_len, 0), Lmax);
  }
  if (is_last && seq_len > pg1 * kPageSize && lane == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
  const int npg = pg1 - pg0;

  // q for the G heads of this KV head, pre-scaled by scale*log2(e).
  float qf[G][Geo::CH * 8];
  {
    const __half* qb = p.q + ((size_t)b * p.num_q_heads + (size_t)kvh * G) * D;
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int ch = 0; ch < Geo::CH; ++ch) {
        const uint4 raw = __ldg(reinterpret_cast<const uint4*>(qb + h * D + ch * 64 + c * 8));
        float f[8];
        half8_to_float(raw, f);
#pragma unroll
        for (int e = 0; e < 8; ++e) qf[h][ch * 8 + e] = f[e] * p.qscale;
      }
  }

  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages + pg0;
  const size_t page_stride = (size_t)p.num_kv_heads * kPageSize * D;  // halves
  const __half* kbase = p.k_pages + (size_t)kvh * kPageSize * D;
  const __half* vbase = p.v_pages + (size_t)kvh * kPageSize * D;
  const uint64_t policy = l2_evict_first_policy();

  // Block-table entries of the task, 32 per window: lane k of the current
  // window holds entry 32*w + k; the next window is loaded one window ahead
  // so the copy issue never waits on it.
  int bt_cur = lane < npg ? __ldg(bt_row + lane) : -1;
  int bt_nxt = 32 + lane < npg ? __ldg(bt_row + 32 + lane) : -1;
  int bt_w = 0;

  // Issue page j of the task into stage j % NS.  Warp-collective (the entry
  // comes by shuffle); lane 0 issues.  j grows by one per call.  A page past
  // the sequence end or with an invalid index is not copied: its barriers
  // are released empty and the page is masked.
  auto issue = [&](int j) {
    if ((j >> 5) != bt_w) {
      ++bt_w;
      bt_cur = bt_nxt;
      const int idx = 32 * (bt_w + 1) + lane;
      bt_nxt = idx < npg ? __ldg(bt_row + idx) : -1;
    }
    int phys = __shfl_sync(kFull, bt_cur, j & 31);
    if (lane == 0) {
      const int s = j % NS;
      const uint32_t kb = ws_u32 + L.bar_off + 16 * s;
      if ((pg0 + j) * kPageSize >= seq_len) {
        phys = -1;
      } else if (phys < 0 || phys >= p.num_pages) {
        set_status(p.status, PA_DEV_BAD_PAGE);
        phys = -1;
      }
      page_ids[s] = phys;
      fence_proxy_async_smem();
      if (phys >= 0) {
        mbar_arrive_expect_tx(kb, L.tile);
        bulk_g2s(ws_u32 + L.k_off + s * L.tile, kbase + (size_t)phys * page_stride, L.tile, kb,
                 policy);
        mbar_arrive_expect_tx(kb + 8, L.tile);
        bulk_g2s(ws_u32 + L.v_off + s * L.tile, vbase + (size_t)phys * page_stride, L.tile, kb + 8,
                 policy);
      } else {
        mbar_arrive(kb);
        mbar_arrive(kb + 8);
      }
    }
  };

  const int npre = npg < NS ? npg : NS;
  for (int j = 0; j < npre; ++j) issue(j);

  // Softmax state of this lane's head (lanes of one head hold equal copies).
  float m_run = -INFINITY, l_run = 0.f;
  const int myh = (G == 1) ? 0 : ((c * Geo::NVL) >> 2);
  float acc[G][Geo::DPL];
#pragma unroll
  for (int h = 0; h < G; ++h)
#pragma unroll
    for (int d = 0; d < Geo::DPL; ++d) acc[h][d] = 0.f;

  int jfail = -1;
  for (int j = 0; j < npg; ++j) {
    const int s = j % NS;
    const uint32_t kb = ws_u32 + L.bar_off + 16 * s;
    const uint32_t par = (uint32_t)(j / NS) & 1u;
    if (!__all_sync(kFull, mbar_wait_bounded(kb, par))) {
      jfail = j;
      break;
    }
    const int phys = page_ids[s];
    const int nvalid = phys < 0 ? 0 : min(kPageSize, seq_len - (pg0 + j) * kPageSize);

    if (nvalid > 0) {
      // ---- scores of the page's 16 tokens for the G heads
      const __half* Ks = reinterpret_cast<const __half*>(ws + L.k_off + s * L.tile);
      float v[Geo::NV];
#pragma unroll
      for (int k = 0; k < Geo::NV; ++k) v[k] = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int t = rg + 4 * i;
#pragma unroll
        for (int ch = 0; ch < Geo::CH; ++ch) {
          const uint4 raw = *reinterpret_cast<const uint4*>(Ks + t * D + ch * 64 + c * 8);
          float kf[8];
          half8_to_float(raw, kf);
#pragma unroll
          for (int h = 0; h < G; ++h) {
            float a = v[h * 4 + i];
#pragma unroll
            for (int e = 0; e < 8; ++e) a = fmaf(qf[h][ch * 8 + e], kf[e], a);
            v[h * 4 + i] = a;
          }
        }
      }
      reduce_scatter<Geo::NV, 4>(v, lane);

      // ---- online softmax update for this lane's head
      float pmax = -INFINITY;
#pragma unroll
      for (int k = 0; k < Geo::NVL; ++k) {
        const int vi = (Geo::NV >= 8) ? c * Geo::NVL + k : (c >> 1);
        const int t = rg + 4 * (vi & 3);
        if (t >= nvalid) v[k] = -INFINITY;
        pmax = fmaxf(pmax, v[k]);
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
      for (int k = 0; k < Geo::NVL; ++k) {
        const int vi = (Geo::NV >= 8) ? c * Geo::NVL + k : (c >> 1);
        const int t = rg + 4 * (vi & 3);
        const float pk = dead ? 0.f : ex2(v[k] - m_new);
        p_s[t * G + (vi >> 2)] = pk;
        psum += pk;
      }
      // G == 1: lanes c and c^1 hold the same value, so bit 0 is not summed.
#pragma unroll
      for (int m = (G == 1 ? 2 : 1); m < Geo::HEAD_LANES; m <<= 1)
        psum += __shfl_xor_sync(kFull, psum, m);
      psum += __shfl_xor_sync(kFull, psum, 8);
      psum += __shfl_xor_sync(kFull, psum, 16);
      l_run = l_run * alpha + psum;
      m_run = m_new;
      if (rg == 0 && (c & (Geo::HEAD_LANES - 1)) == 0) a_s[myh] = alpha;
      __syncwarp();
    }

    if (!__all_sync(kFull, mbar_wait_bounded(kb + 8, par))) {
      jfail = j;
      break;
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
          for (int d = 0; d < Geo::DPL; ++d) acc[h][d] *= al[h];
      }
      const __half* Vs = reinterpret_cast<const __half*>(ws + L.v_off + s * L.tile);
#pragma unroll
      for (int t = 0; t < kPageSize; ++t) {
        if (t < nvalid) {
          float pp[G];
#pragma unroll
          for (int h = 0; h < G; ++h) pp[h] = p_s[t * G + h];
          float vf[Geo::DPL];
          if constexpr (Geo::DPL == 4) {
            const uint2 raw = *reinterpret_cast<const uint2*>(Vs + t * D + lane * 4);
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&raw.x));
            const float2 bb = __half22float2(*reinterpret_cast<const __half2*>(&raw.y));
            vf[0] = a.x;
            vf[1] = a.y;
            vf[2] = bb.x;
            vf[3] = bb.y;
          } else {
            const float2 a = __half22float2(*reinterpret_cast<const __half2*>(Vs + t * D + lane * 2));
            vf[0] = a.x;
            vf[1] = a.y;
          }
#pragma unroll
          for (int h = 0; h < G; ++h)
#pragma unroll
            for (int d = 0; d < Geo::DPL; ++d) acc[h][d] = fmaf(pp[h], vf[d], acc[h][d]);
        }
      }
    }
    __syncwarp();
    if (j + NS < npg) issue(j + NS);
  }

  if (jfail >= 0) {
    // A copy did not land in time.  Report, let the copies already issued
    // finish (bounded), and leave without writing.
    if (lane == 0) {
      set_status(p.status, PA_DEV_TIMEOUT);
      const int last = min(npg, jfail + NS);
      for (int j = jfail; j < last; ++j) {
        const uint32_t kb = ws_u32 + L.bar_off + 16 * (j % NS);
        const uint32_t par = (uint32_t)(j / NS) & 1u;
        mbar_wait_bounded(kb, par, 10000000ull);
        mbar_wait_bounded(kb + 8, par, 10000000ull);
      }
    }
    __syncwarp();
    return;
  }

  // ---- epilogue: normalise and write
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const int rep = h * Geo::HEAD_LANES;  // lane (rg 0, c = h*HEAD_LANES) owns head h's state
    const float lh = __shfl_sync(kFull, l_run, rep);
    const float mh = __shfl_sync(kFull, m_run, rep);
    const float inv = lh > 0.f ? 1.f / lh : 0.f;
    if (!is_split) {
      __half* o = p.out + ((size_t)b * p.num_q_heads + (size_t)kvh * G + h) * D + lane * Geo::DPL;
      if constexpr (Geo::DPL == 4) {
        const __half2 a = __floats2half2_rn(acc[h][0] * inv, acc[h][1] * inv);
        const __half2 bb = __floats2half2_rn(acc[h][2] * inv, acc[h][3] * inv);
        uint2 w;
        w.x = *reinterpret_cast<const uint32_t*>(&a);
        w.y = *reinterpret_cast<const uint32_t*>(&bb);
        *reinterpret_cast<uint2*>(o) = w;
      } else {
        *reinterpret_cast<__half2*>(o) = __floats2half2_rn(acc[h][0] * inv, acc[h][1] * inv);
      }
    } else {
      float* o = p.part_o + ((size_t)item_idx * G + h) * D + lane * Geo::DPL;
      if constexpr (Geo::DPL == 4) {
        *reinterpret_cast<float4*>(o) =
            make_float4(acc[h][0] * inv, acc[h][1] * inv, acc[h][2] * inv, acc[h][3] * inv);
      } else {
        *reinterpret_cast<float2*>(o) = make_float2(acc[h][0] * inv, acc[h][1] * inv);
      }
      if (lane == 0) p.part_lse[(size_t)item_idx * G + h] = lh > 0.f ? mh + lg2(lh) : -INFINITY;
    }
  }
}

}  // namespace pa
