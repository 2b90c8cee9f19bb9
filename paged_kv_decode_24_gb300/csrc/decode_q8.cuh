// Split decode attention over an 8-bit paged KV cache with per-row fp32
// scales: INT8 codes (MonadKai/xLLM, introduction: KV-cache quantisation,
// per-row INT8) or E4M3 bytes ("Eine LLM-Inferenz-Engine von Grund auf mit
// C++ und CUDA bauen", section 4: FP8 quantisation of the cache), the FMT
// template parameter (kCodeInt8, kCodeE4m3).
//
// Tasks, CTA shapes, the per-warp copy ring, the fused append, the in-CTA
// merge and the split partials are those of decode_tc.cuh; what differs is
// what a page holds and how it is multiplied.  The K half-stage of a
// (page, KV head) brings its 16 x D int8 K code tile by one TMA tensor copy
// and the 16 fp32 K scales and 16 fp32 V scales of its rows by two 64-byte
// bulk copies; the V half-stage brings the V code tile.  Tiles land with the
// 128-byte swizzle (D = 128) or the 64-byte swizzle (D = 64), so every
// ldmatrix below is free of bank conflicts.  A row costs D + 4 bytes per
// tensor against 2 D for fp16.
//
// The int8 codes become fp16 in registers: with its sign bit flipped a byte
// is b + 128, and placed under the fp16 exponent of 1024 it reads
// 1152 + b, exactly.  One byte permute makes two such halves.  E4M3 bytes
// become fp16 by the hardware conversion of a byte pair (exact: every E4M3
// value is an fp16 value); they carry no bias.
//
// Products, for the 16 tokens of a page and the G <= 8 query heads of the KV
// head (padded to 8), g = lane / 4 and t = lane % 4:
//
//   S^T[16 tok x 8 heads] = (K_codes + 1152)[16 x D] . Q^T[D x 8]
//       D/16 mma.m16n8k16; ldmatrix (not transposed) of the row-major code
//       tile gives a thread the 4 codes of dims 4t..4t+3 of token g (and
//       g+8) per 16-dim step, so the reduction order is permuted to logical
//       k (2t, 2t+1) = dims 4t, 4t+1 and (2t+8, 2t+9) = dims 4t+2, 4t+3, and
//       q is loaded the same way.  The bias 1152 * sum_d q_d of each head is
//       one product of the same shape, made once per task and subtracted
//       (INT8 only); then row t of S^T is multiplied by its K scale.
//
//   O^T[D x 8] += V_codes^T[D x 16 tok] . P'^T[16 tok x 8]
//       D/16 m-tiles x 2 mma.m16n8k16.  ldmatrix.trans on 2-byte elements
//       of the row-major V tile gives a thread tokens 2t, 2t+1 of dims 2g,
//       2g+1; one byte permute per dim pairs the two tokens, so m-tile row
//       g is dim 2g and row g+8 is dim 2g+1 of its 16 dims.  The V codes
//       are exact fp16 integers after subtracting 1152 (INT8).  An E4M3 byte
//       may be NaN, so on a page the sequence ends in, the E4M3 V codes of
//       rows past the end are zeroed before the conversion.
//
// P' = p * s_v / R carries each token's V scale: R is the largest V scale
// the warp has met so far, so P' <= 1 stays in the normal fp16 range, and
// the accumulator is kept in units of 1/R (rescaled when R grows, together
// with the online-softmax rescale).  P' is split into fp16 hi + lo, so the
// product keeps about 22 bits of it.  Rows past the sequence end get
// P' = 0 whatever their scales hold (NaN too).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <math.h>

#include <type_traits>

#include "decode_tc.cuh"
#include "quant_common.cuh"

namespace pa {

__device__ __forceinline__ void ldsm_x4_addr(uint32_t addr, uint32_t* r) {
  ldsm_x4(addr, r[0], r[1], r[2], r[3]);
}

__device__ __forceinline__ void ldsm_x4_t_addr(uint32_t addr, uint32_t* r) {
  ldsm_x4_t(addr, r[0], r[1], r[2], r[3]);
}

// Bytes (i, j) of w, each as 1152 + code, into one half2 (byte i low).
// The selector puts byte i and byte j of w ^ 0x80808080 under the fp16
// exponent byte 0x64.
template <unsigned SEL>
__device__ __forceinline__ uint32_t biased_pair(uint32_t u) {
  return __byte_perm(u, 0x64646464u, SEL);
}

__device__ __forceinline__ uint32_t sub1152(uint32_t h) {
  const __half2 bias = __halves2half2(__ushort_as_half(0x6480), __ushort_as_half(0x6480));
  const __half2 r = __hsub2(*reinterpret_cast<const __half2*>(&h), bias);
  return *reinterpret_cast<const uint32_t*>(&r);
}

// Byte offset of byte `x` of row `row` in a swizzled code tile of 16 rows of
// D bytes: 128-byte swizzle (chunk ^= row % 8) for D = 128, 64-byte swizzle
// (chunk ^= (row / 2) % 4) for D = 64, as the TMA copy lays them out.
template <int D>
__device__ __forceinline__ uint32_t q8_swz(int row, int x) {
  if constexpr (D == 128)
    return (uint32_t)(row * 128 + (((x >> 4) ^ (row & 7)) << 4) + (x & 15));
  else
    return (uint32_t)(row * 64 + (((x >> 4) ^ ((row >> 1) & 3)) << 4) + (x & 15));
}

// Shared memory of the 8-bit kernel, per CTA: NW rings of NS page stages
// (K code tile, then V code tile; 1024-aligned for the swizzle), then per
// warp NS mbarriers, NS page ids, NS scale blocks (16 K then 16 V row
// scales) and the new row's codes and scales (fused append).
template <int D, int NW, int NS>
struct Q8Layout {
  static constexpr int TILE = kPageSize * D;          // 1024 or 2048 bytes
  static constexpr int STAGE = 2 * TILE;
  static constexpr int RING = NS * STAGE;
  static constexpr int RINGS = NW * RING;
  static constexpr int BARS = 0;
  static constexpr int PAGES = align_up(8 * NS, 16);
  static constexpr int SCALES = PAGES + align_up(4 * NS, 16);
  static constexpr int NROW = SCALES + 128 * NS;      // K codes, V codes, K scale, V scale
  static constexpr int EXTRA = align_up(NROW + 2 * D + 16, 16);
  static constexpr int FLAG = RINGS + NW * EXTRA;
  static constexpr int BYTES = FLAG + 16 + 1024;      // + slack to align the base to 1024
};

// Lazy rescaling: a running maximum (softmax, in log2 units) is replaced
// only when a page exceeds it by more than this, so weights stay below
// 2^kLazyLog2 and the accumulator is rarely rescaled.  The V-scale reference
// R is replaced only when a page's largest V scale exceeds 2 R.
constexpr float kLazyLog2 = 8.f;

template <int D, int G, int NW, int NS, int FMT, bool EARLY>
__global__ void __launch_bounds__(NW * 32, 4)
    split_decode_q8_kernel(const __grid_constant__ SplitParams p) {
  static_assert(G <= 8, "the mma tile holds at most 8 query heads");
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  using L = Q8Layout<D, NW, NS>;
  constexpr int KSTEPS = D / 16;  // QK k-steps; also PV m-tiles
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
  const uint32_t page_ids = smem_u32(extra) + L::PAGES;     // [NS] int
  const uint32_t scl = smem_u32(extra) + L::SCALES;         // [NS][32] fp32: K, V row scales
  unsigned char* nrow = extra + L::NROW;                      // [2][D] codes, then 2 scales
  float* nscale = reinterpret_cast<float*>(nrow + 2 * D);
  int* cta_failed = reinterpret_cast<int*>(base + L::FLAG);
  int* cta_last = cta_failed + 1;

  if ((int)blockIdx.x >= p.num_ctas) return;  // whole CTA
  // Plan data is written only by pa_plan_upload (a copy, which the
  // programmatic launch does not overlap): it may be read before the wait.
  const int4 hdr = *reinterpret_cast<const int4*>(p.ws_header);
  const int2 hdr_ctas = *reinterpret_cast<const int2*>(p.ws_header + 8);
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
      const size_t row0 = ((size_t)phys * p.num_kv_heads + ((uint32_t)it.y & kItemHeadMask)) *
                          kPageSize;
      prefetch_l2_bulk(p.k_codes + row0 * D, kPageSize * D);
      prefetch_l2_bulk(p.v_codes + row0 * D, kPageSize * D);
      prefetch_l2_bulk(p.k_scales + row0, kPageSize * 4);
      prefetch_l2_bulk(p.v_scales + row0, kPageSize * 4);
    }
  }
  if (threadIdx.x == 0) {
    *cta_failed = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
  }
  if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_init(bars + 8 * s, 1);
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

  // ldmatrix row addresses of this lane, as an offset inside a tile: lane l
  // addresses row (l & 7) + 8 ((l >> 3) & 1) of 16-byte chunk (l >> 4) (+ the
  // step's chunk pair), swizzled like the TMA copy.  Chunk pairs start at
  // even chunks, so the step is an XOR of the chunk bits.
  uint32_t lm_off;
  {
    const int row = (lane & 7) + 8 * ((lane >> 3) & 1);
    const int chunk = lane >> 4;
    if constexpr (D == 128)
      lm_off = (uint32_t)(row * 128 + ((chunk ^ (row & 7)) << 4));
    else
      lm_off = (uint32_t)(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
  }

  // What the previous kernel may write (the new rows, q) is read by
  // load_inputs: here, after the wait, or with early_kv after the first
  // page copies and the wait.
  int k_app = -1;
  uint32_t qb[KSTEPS][2];
  float cb0, cb1;
  auto load_inputs = [&]() {
    // Fused append: the warp whose pages hold position L-1 quantises the new
    // K and V rows into its shared memory now and patches them in later.
    if (p.k_new != nullptr && seq_len > 0) {
      const int j_app = (seq_len - 1) / kPageSize - pg0;
      if (j_app >= pstart && j_app < npg && (j_app - pstart) % pstride == 0) {
        k_app = (j_app - pstart) / pstride;
        const size_t src = ((size_t)b * p.num_kv_heads + kvh) * D;
        float sk, sv;
        const uint32_t ck =
            quantize_row_warp<D, FMT>(static_cast<const __half*>(p.k_new) + src, lane, sk);
        const uint32_t cv =
            quantize_row_warp<D, FMT>(static_cast<const __half*>(p.v_new) + src, lane, sv);
        if constexpr (D == 128) {
          reinterpret_cast<uint32_t*>(nrow)[lane] = ck;
          reinterpret_cast<uint32_t*>(nrow + D)[lane] = cv;
        } else {
          reinterpret_cast<uint16_t*>(nrow)[lane] = (uint16_t)ck;
          reinterpret_cast<uint16_t*>(nrow + D)[lane] = (uint16_t)cv;
        }
        if (lane == 0) {
          nscale[0] = sk;
          nscale[1] = sv;
        }
        __syncwarp();
      }
    }

    // Q^T fragments with the permuted reduction order: b0 = dims 4t, 4t+1 and
    // b1 = dims 4t+2, 4t+3 of each 16-dim step, column n = head g.  Heads past
    // G are zero.  cb = the same product with every K code at its bias 1152.
    {
      const __half* qrow =
          static_cast<const __half*>(p.q) + ((size_t)b * p.num_q_heads + (size_t)kvh * G + g) * D;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; ++kk) {
        if (g < G) {
          const uint2 v = __ldg(reinterpret_cast<const uint2*>(qrow + kk * 16 + 4 * t));
          qb[kk][0] = v.x;
          qb[kk][1] = v.y;
        } else {
          qb[kk][0] = qb[kk][1] = 0u;
        }
      }
      float cb[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (FMT == kCodeInt8) {
        const uint32_t k1152 = 0x64806480u;
#pragma unroll
        for (int kk = 0; kk < KSTEPS; ++kk)
          mma_16816(cb, k1152, k1152, k1152, k1152, qb[kk][0], qb[kk][1]);
      }
      cb0 = cb[0];
      cb1 = cb[1];
    }
  };
  if constexpr (!EARLY) load_inputs();

  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages + pg0;
  const uint64_t policy = l2_evict_first_policy();
  int bt_cur = lane < npg ? __ldg(bt_row + lane) : -1;
  int bt_nxt = 32 + lane < npg ? __ldg(bt_row + 32 + lane) : -1;
  int bt_w = 0;
  const size_t head_rows = (size_t)kvh * kPageSize;  // row offset of this head in a page

  // Issue this warp's page k into stage k % NS: both code tiles and both
  // scale blocks on one mbarrier; warp-collective, lane 0 issues.
  auto issue = [&](int k) {
    const int j = pstart + k * pstride;
    if ((j >> 5) != bt_w) {  // j grows by at most NW <= 32 between calls
      ++bt_w;
      bt_cur = bt_nxt;
      const int idx = 32 * (bt_w + 1) + lane;
      bt_nxt = idx < npg ? __ldg(bt_row + idx) : -1;
    }
    int phys = __shfl_sync(kFull, bt_cur, j & 31);
    if (lane == 0) {
      const int s = k % NS;
      const uint32_t bar = bars + 8 * s;
      if ((pg0 + j) * kPageSize >= seq_len) {
        phys = -1;
      } else if (phys < 0 || phys >= p.num_pages) {
        set_status(p.status, PA_DEV_BAD_PAGE);
        phys = -1;
      }
      asm volatile("st.shared.s32 [%0], %1;" ::"r"(page_ids + 4 * s), "r"(phys) : "memory");
      fence_proxy_async_smem();
      if (phys >= 0) {
        const size_t row0 = (size_t)phys * p.num_kv_heads * kPageSize + head_rows;
        const uint32_t dst = ring + s * L::STAGE;
        mbar_arrive_expect_tx(bar, 2 * L::TILE + 128);
        tma_load_4d(dst, &p.tmap_k, 0, 0, kvh, phys, bar, policy);
        tma_load_4d(dst + L::TILE, &p.tmap_v, 0, 0, kvh, phys, bar, policy);
        bulk_g2s(scl + 128 * s, p.k_scales + row0, 64, bar, policy);
        bulk_g2s(scl + 128 * s + 64, p.v_scales + row0, 64, bar, policy);
      } else {
        mbar_arrive(bar);
      }
    }
  };

  const int npre = npk < NS ? npk : NS;
  for (int k = 0; k < npre; ++k) issue(k);

  if constexpr (EARLY) {
    pdl_wait_primary();
    load_inputs();
  }

  // Running state.  m_run: per-head reference maximum (log2 units, lazy);
  // l_part: this lane's share of the running sums; R (vref): V-scale
  // reference; o: O^T in units of 2^-m_run / R, dims 16mt+2g (+1), heads
  // 2t, 2t+1.
  float m_run[2] = {-INFINITY, -INFINITY};
  float l_part[2] = {0.f, 0.f};
  float vref = 0.f, vref_inv = 0.f;
  float o[KSTEPS][4];
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
  const float qs = p.qscale;
  // lanes whose P'^T entries this lane needs (as in decode_tc.cuh)
  const int src1 = (2 * t) * 4 + (g >> 1);
  const int src2 = (2 * t + 1) * 4 + (g >> 1);
  const unsigned int perm = (g & 1) ? 0x7632u : 0x5410u;

  bool failed = false;
  int kfail = 0;
  for (int k = 0; k < npk; ++k) {
    const int s = k % NS;
    if (!__all_sync(kFull, mbar_wait_bounded(bars + 8 * s, (k / NS) & 1, p.wait_ns))) {
      failed = true;
      kfail = k;
      break;
    }
    const int phys = lds_s32(page_ids + 4 * s);
    const int j = pstart + k * pstride;
    const int nvalid = phys < 0 ? 0 : min(kPageSize, seq_len - (pg0 + j) * kPageSize);
    const uint32_t ktile = ring + s * L::STAGE;
    const uint32_t vtile = ktile + L::TILE;
    const uint32_t ksc = scl + 128 * s;  // 16 K scales, then 16 V scales
    if (k == k_app && phys >= 0) {
      // Both copies of the page have landed: patch the new row into the
      // staged tiles and scales, then write it to the pools.  No other task
      // reads this page.
      const int r = (seq_len - 1) % kPageSize;
      for (int i = lane; i < D / 16; i += 32) {
        const uint4 kv = reinterpret_cast<const uint4*>(nrow)[i];
        const uint4 vv = reinterpret_cast<const uint4*>(nrow + D)[i];
        unsigned char* kt = base + (ktile - smem_u32(base));
        *reinterpret_cast<uint4*>(kt + q8_swz<D>(r, 16 * i)) = kv;
        *reinterpret_cast<uint4*>(kt + L::TILE + q8_swz<D>(r, 16 * i)) = vv;
      }
      const size_t row = ((size_t)phys * p.num_kv_heads + kvh) * kPageSize + r;
      uint4* kw = reinterpret_cast<uint4*>(const_cast<int8_t*>(p.k_codes) + row * D);
      uint4* vw = reinterpret_cast<uint4*>(const_cast<int8_t*>(p.v_codes) + row * D);
      for (int i = lane; i < D / 16; i += 32) {
        kw[i] = reinterpret_cast<const uint4*>(nrow)[i];
        vw[i] = reinterpret_cast<const uint4*>(nrow + D)[i];
      }
      if (lane == 0) {
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(ksc + 4 * r), "f"(nscale[0]) : "memory");
        asm volatile("st.shared.f32 [%0], %1;" ::"r"(ksc + 64 + 4 * r), "f"(nscale[1]) : "memory");
        const_cast<float*>(p.k_scales)[row] = nscale[0];
        const_cast<float*>(p.v_scales)[row] = nscale[1];
      }
      __syncwarp();
    }

    if (nvalid > 0) {
      // ---- S^T = (K_codes + 1152) . Q^T - bias, then the K row scales
      // two accumulators (even and odd k-steps) halve the dependent mma chain
      float c[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
      const uint32_t kaddr = ktile + lm_off;
#pragma unroll
      for (int kk = 0; kk < KSTEPS; kk += 2) {
        uint32_t r[4];
        ldsm_x4_addr(kaddr ^ (uint32_t)(kk << 4), r);
        // r[0], r[1]: tokens g, g+8 of step kk; r[2], r[3]: of step kk+1
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          if constexpr (FMT == kCodeE4m3) {
            // bytes 0, 1: dims 4t, 4t+1 (logical k 2t, 2t+1); bytes 2, 3: dims
            // 4t+2, 4t+3 (logical k 2t+8, 2t+9)
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_half2x2(r[2 * h], a0, a2);
            e4m3x4_to_half2x2(r[2 * h + 1], a1, a3);
            mma_16816(c[h], a0, a1, a2, a3, qb[kk + h][0], qb[kk + h][1]);
          } else {
            const uint32_t u0 = r[2 * h] ^ 0x80808080u, u1 = r[2 * h + 1] ^ 0x80808080u;
            mma_16816(c[h], biased_pair<0x4140u>(u0), biased_pair<0x4140u>(u1),
                      biased_pair<0x4342u>(u0), biased_pair<0x4342u>(u1), qb[kk + h][0],
                      qb[kk + h][1]);
          }
        }
      }
      const float ks0 = lds_f32(ksc + 4 * g) * qs, ks8 = lds_f32(ksc + 4 * (g + 8)) * qs;
      float s0 = ((c[0][0] + c[1][0]) - cb0) * ks0, s1 = ((c[0][1] + c[1][1]) - cb1) * ks0;
      float s2 = ((c[0][2] + c[1][2]) - cb0) * ks8, s3 = ((c[0][3] + c[1][3]) - cb1) * ks8;
      if (g >= nvalid) s0 = s1 = -INFINITY;
      if (g + 8 >= nvalid) s2 = s3 = -INFINITY;
      // ---- V scales of rows g, g+8 (0 past nvalid) and the reference R
      const float vs0 = g < nvalid ? lds_f32(ksc + 64 + 4 * g) : 0.f;
      const float vs8 = g + 8 < nvalid ? lds_f32(ksc + 64 + 4 * (g + 8)) : 0.f;
      float vmax = fmaxf(vs0, vs8);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) vmax = fmaxf(vmax, __shfl_xor_sync(kFull, vmax, m));
      float fr = 1.f;
      if (vmax > 2.f * vref) {  // warp-uniform; always true on the first nonzero page
        fr = vref / vmax;
        vref = vmax;
        vref_inv = 1.f / vmax;
      }
      // ---- online softmax for heads 2t (s0, s2) and 2t+1 (s1, s3), lazy max
      float mA = fmaxf(s0, s2), mB = fmaxf(s1, s3);
#pragma unroll
      for (int m = 4; m <= 16; m <<= 1) {
        mA = fmaxf(mA, __shfl_xor_sync(kFull, mA, m));
        mB = fmaxf(mB, __shfl_xor_sync(kFull, mB, m));
      }
      float al0 = 1.f, al1 = 1.f;
      if (mA > m_run[0] + kLazyLog2) {  // uniform across the 8 lanes of a head
        al0 = ex2(m_run[0] - mA);       // 0 on the first live page
        m_run[0] = mA;
      }
      if (mB > m_run[1] + kLazyLog2) {
        al1 = ex2(m_run[1] - mB);
        m_run[1] = mB;
      }
      const bool deadA = m_run[0] == -INFINITY, deadB = m_run[1] == -INFINITY;
      const float p0 = deadA ? 0.f : ex2(s0 - m_run[0]);
      const float p2 = deadA ? 0.f : ex2(s2 - m_run[0]);
      const float p1 = deadB ? 0.f : ex2(s1 - m_run[1]);
      const float p3 = deadB ? 0.f : ex2(s3 - m_run[1]);
      l_part[0] = l_part[0] * al0 + (p0 + p2);
      l_part[1] = l_part[1] * al1 + (p1 + p3);
      if (__any_sync(kFull, al0 != 1.f || al1 != 1.f) || fr != 1.f) {
        al0 *= fr;
        al1 *= fr;
#pragma unroll
        for (int mt = 0; mt < KSTEPS; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
      }
      // ---- P'^T = (p * s_v / R)^T into B fragments, hi and lo fp16 parts
      const float w0 = vs0 * vref_inv, w8 = vs8 * vref_inv;
      const float q0 = p0 * w0, q1 = p1 * w0, q2 = p2 * w8, q3 = p3 * w8;
      const uint32_t h01 = pack_half2(q0, q1);  // token g: heads 2t, 2t+1
      const uint32_t h23 = pack_half2(q2, q3);  // token g+8
      const float2 f01 = unpack_half2(h01), f23 = unpack_half2(h23);
      const uint32_t l01 = pack_half2(q0 - f01.x, q1 - f01.y);
      const uint32_t l23 = pack_half2(q2 - f23.x, q3 - f23.y);
      const uint32_t pb_hi0 =
          __byte_perm(__shfl_sync(kFull, h01, src1), __shfl_sync(kFull, h01, src2), perm);
      const uint32_t pb_hi1 =
          __byte_perm(__shfl_sync(kFull, h23, src1), __shfl_sync(kFull, h23, src2), perm);
      const uint32_t pb_lo0 =
          __byte_perm(__shfl_sync(kFull, l01, src1), __shfl_sync(kFull, l01, src2), perm);
      const uint32_t pb_lo1 =
          __byte_perm(__shfl_sync(kFull, l23, src1), __shfl_sync(kFull, l23, src2), perm);
      // ---- O^T += V_codes^T . P'^T (hi and lo); rows past nvalid have P' = 0
      const uint32_t vaddr = vtile + lm_off;
      // r[0], r[1] of an m-tile: tokens 0-7, 8-15; each holds tokens 2t, 2t+1
      // (byte pairs 0,1 and 2,3) of dims 2g, 2g+1.  tail: E4M3 bytes of rows
      // past nvalid (which may be NaN) are zeroed first.
      auto pv = [&](auto tail) {
        uint32_t vm0 = 0xffffffffu, vm1 = 0xffffffffu;
        if constexpr (decltype(tail)::value) {
          vm0 = (2 * t < nvalid ? 0x0000ffffu : 0u) | (2 * t + 1 < nvalid ? 0xffff0000u : 0u);
          vm1 = (2 * t + 8 < nvalid ? 0x0000ffffu : 0u) | (2 * t + 9 < nvalid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < KSTEPS; mt += 2) {
          uint32_t r[4];
          ldsm_x4_t_addr(vaddr ^ (uint32_t)(mt << 4), r);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            uint32_t a0, a1, a2, a3;
            if constexpr (FMT == kCodeE4m3) {
              uint32_t w0 = r[2 * h], w1 = r[2 * h + 1];
              if constexpr (decltype(tail)::value) {
                w0 &= vm0;
                w1 &= vm1;
              }
              // bytes (0, 2) are dim 2g of tokens 2t, 2t+1; bytes (1, 3) dim 2g+1
              // a0: dim 2g, tokens 2t, 2t+1; a1: dim 2g+1; a2, a3: tokens 2t+8, 2t+9
              e4m3x4_to_half2x2(__byte_perm(w0, 0u, 0x3120u), a0, a1);
              e4m3x4_to_half2x2(__byte_perm(w1, 0u, 0x3120u), a2, a3);
            } else {
              const uint32_t u0 = r[2 * h] ^ 0x80808080u, u1 = r[2 * h + 1] ^ 0x80808080u;
              a0 = sub1152(biased_pair<0x4240u>(u0));  // dim 2g, tokens 2t, 2t+1
              a1 = sub1152(biased_pair<0x4341u>(u0));  // dim 2g+1
              a2 = sub1152(biased_pair<0x4240u>(u1));  // dim 2g, tokens 2t+8, 2t+9
              a3 = sub1152(biased_pair<0x4341u>(u1));
            }
            mma_16816(o[mt + h], a0, a1, a2, a3, pb_hi0, pb_hi1);
            mma_16816(o[mt + h], a0, a1, a2, a3, pb_lo0, pb_lo1);
          }
        }
      };
      if constexpr (FMT == kCodeE4m3) {
        if (nvalid < kPageSize)
          pv(std::true_type{});
        else
          pv(std::false_type{});
      } else {
        pv(std::false_type{});
      }
    }
    // the stage is free: refill it
    __syncwarp();
    if (k + NS < npk) issue(k + NS);
  }

  if (failed) {
    // A copy did not land in time.  Report it and let the copies already
    // issued finish (bounded).  The task writes nothing.
    if (lane == 0) {
      set_status(p.status, PA_DEV_TIMEOUT);
      const int last = min(npk, kfail + NS);
      for (int k = kfail; k < last; ++k)
        mbar_wait_bounded(bars + 8 * (k % NS), (k / NS) & 1, kDrainWaitNs);
      *cta_failed = 1;
    }
    __syncwarp();
  } else if (lane == 0) {
#pragma unroll
    for (int s = 0; s < NS; ++s) mbar_inval(bars + 8 * s);
  }

#pragma unroll
  for (int m = 4; m <= 16; m <<= 1) {
    l_part[0] += __shfl_xor_sync(kFull, l_part[0], m);
    l_part[1] += __shfl_xor_sync(kFull, l_part[1], m);
  }
  // back from units of 1/R (m_run stays the reference of o and l)
#pragma unroll
  for (int mt = 0; mt < KSTEPS; ++mt) {
    o[mt][0] *= vref;
    o[mt][1] *= vref;
    o[mt][2] *= vref;
    o[mt][3] *= vref;
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
      const int d0 = 16 * mt + 2 * g;
      if (2 * t < G)
        *reinterpret_cast<float2*>(stage + (2 * t) * D + d0) =
            make_float2(o[mt][0] * inv0, o[mt][2] * inv0);
      if (2 * t + 1 < G)
        *reinterpret_cast<float2*>(stage + (2 * t + 1) * D + d0) =
            make_float2(o[mt][1] * inv1, o[mt][3] * inv1);
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
      __half* dst = static_cast<__half*>(p.out) + ((size_t)b * p.num_q_heads + (size_t)kvh * G) * D;
      for (int i = lane * 2; i < G * D; i += 64)
        *reinterpret_cast<__half2*>(dst + i) = __floats2half2_rn(stage[i], stage[i + 1]);
    } else {
      float* dst = p.part_o + (size_t)slot * G * D;
      for (int i = lane * 4; i < G * D; i += 128)
        *reinterpret_cast<float4*>(dst + i) = *reinterpret_cast<const float4*>(stage + i);
      if (p.fuse_merge) split_finish_warp<__half, D>(merge_target(p, sg.y, grp, G), lane);
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
    const int d0 = 16 * mt + 2 * g;
    if (2 * t < G) {
      mine[2 * G + (2 * t) * D + d0] = o[mt][0];
      mine[2 * G + (2 * t) * D + d0 + 1] = o[mt][2];
    }
    if (2 * t + 1 < G) {
      mine[2 * G + (2 * t + 1) * D + d0] = o[mt][1];
      mine[2 * G + (2 * t + 1) * D + d0 + 1] = o[mt][3];
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
      static_cast<__half*>(p.out)[((size_t)b * p.num_q_heads + (size_t)kvh * G + h) * D + d] =
          __float2half_rn(r);
    } else {
      p.part_o[((size_t)slot * G + h) * D + d] = r;
      if (d == 0) p.part_lse[(size_t)slot * G + h] = Z > 0.f ? M + lg2(Z) : -INFINITY;
    }
  }
  if (is_split && p.fuse_merge)  // CTA-uniform: one task
    split_finish_cta<__half, D, NW>(merge_target(p, sg.y, grp, G), cta_last);
}

}  // namespace pa
