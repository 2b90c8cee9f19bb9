// Attention of several query tokens per sequence over the paged KV cache
// (chunked prefill; prefill and decode tokens in one batch), FlashAttention-
// style on tensor cores.  The from-scratch engine article (section 4) names
// processing several prompt tokens at once with a fused FlashAttention-style
// kernel as the step after decode; swiftLLM lists piggybacked prefill and
// decode and Flash Attention.
//
// A CTA owns a tile of 64 query rows of one (sequence, KV head): 64 / G
// consecutive query tokens times the G query heads of the KV head.  Warp w
// takes rows 16w .. 16w+15 (row r is token r / G, head r % G).  The CTA
// streams the causal part of the sequence, positions 0 .. (its last
// query's position), in stages of 32 tokens (two pages): thread 0 issues
// each stage's K and V page tiles as TMA tensor copies (coordinate = the
// physical page) onto the stage's "full" mbarrier, and refills a stage once
// all four warps have arrived on its "empty" mbarrier.  Every wait is
// bounded; a CTA that gives up drains the copies it issued before leaving.
//
// Per warp and stage, on mma.sync.m16n8k16 (fp16 or bf16, fp32 accumulate):
//   S[16 rows x 32 tok] = Q[16 x D] . K^T      Q held in registers as A
//       fragments; K by ldmatrix (rows = tokens), 4 n-tiles x D/16 k-steps;
//   masking: token j is visible to the row whose query sits at position p
//       iff j <= p (and its page was copied);
//   online softmax per row in base 2, with lazy rescaling: the running max
//       moves only when a stage beats it by more than 2^8;
//   O[16 x D] += P[16 x 32] . V                P repacked from the S
//       fragments into A fragments in the element type, as hi + lo parts
//       (split_hi_lo: about twice the type's bits of p, as in the decode
//       kernels), each multiplied into O; V by ldmatrix.trans, D/8 n-tiles
//       x 2 k-steps.
// The output is O / l, rounded to the element type.
#pragma once

#include <cuda.h>
#include <math.h>

#include "decode_tc.cuh"
#include "elem.cuh"

namespace pa {

// Lazy rescaling threshold (log2 units): weights stay below 2^8.
constexpr float kLazyLog2Prefill = 8.f;

struct PrefillParams {
  const void* q;
  void* out;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* ws;  // the uploaded plan blob
  const int32_t* cu;  // its row offsets [B+1]
  int32_t* status;
  float qscale;       // scale * log2(e)
  int32_t batch, num_q_heads, num_kv_heads, max_pages, num_pages, num_tiles, total_q;
  uint64_t wait_ns;   // bound of each barrier wait (the plan's wait_limit_ns)
  CUtensorMap tmap_k;
  CUtensorMap tmap_v;
};

template <int D, int NS>
struct PfLayout {
  static constexpr int TILE = kPageSize * D * 2;   // one page of one head
  static constexpr int PAGES = 2;                  // pages per stage: 32 tokens
  static constexpr int STAGE = 2 * PAGES * TILE;   // K pages, then V pages
  static constexpr int RING = NS * STAGE;
  static constexpr int FULL = RING;                // NS mbarriers
  static constexpr int EMPTY = FULL + 8 * NS;      // NS mbarriers
  static constexpr int PIDS = EMPTY + 8 * NS;      // NS x PAGES page ids
  static constexpr int FLAG = align_up(PIDS + 4 * NS * PAGES, 16);
  static constexpr int BYTES = FLAG + 16 + 1024;   // + slack to align the base to 1024
};

template <typename T, int D, int G, int NS>
__global__ void __launch_bounds__(128, 2) prefill_kernel(const __grid_constant__ PrefillParams p) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  using L = PfLayout<D, NS>;
  constexpr int KSTEPS = D / 16;  // QK k-steps
  constexpr int NTD = D / 8;      // PV n-tiles (8 dims each)
  constexpr int BOXES = D / 64;
  constexpr int TOKS = kPrefillRows / G;
  constexpr int BN = kPageSize * L::PAGES;
  extern __shared__ unsigned char smem_dyn[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int lg = lane >> 2;
  const int t = lane & 3;
  const uint32_t ring = smem_u32(base);
  const uint32_t full = ring + L::FULL;
  const uint32_t empty = ring + L::EMPTY;
  const uint32_t pids = ring + L::PIDS;
  int* cta_flag = reinterpret_cast<int*>(base + L::FLAG);

  if ((int)blockIdx.x >= p.num_tiles) return;  // whole CTA
  // The plan is written only by its upload (a copy the programmatic launch
  // does not overlap): it may be read before the wait.
  const int4 hdr = *reinterpret_cast<const int4*>(p.ws);
  const int4 tile = reinterpret_cast<const int4*>(p.ws + 16)[blockIdx.x];
  if (threadIdx.x == 0) {
    *cta_flag = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      mbar_init(full + 8 * s, 1);
      mbar_init(empty + 8 * s, 4);
    }
    fence_barrier_init();
  }
  __syncthreads();
  pdl_launch_dependents();
  pdl_wait_primary();

  const int b = tile.x, g = tile.y, tok0 = tile.z, ntok = tile.w;
  if (hdr.x != (int)kPrefillMagic || hdr.y != p.num_tiles || hdr.z != p.batch ||
      hdr.w != p.total_q || b < 0 || b >= p.batch || g < 0 || g >= p.num_kv_heads || tok0 < 0 ||
      ntok < 1 || ntok > TOKS) {
    if (threadIdx.x == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;  // CTA-uniform, nothing issued yet
  }
  const int32_t* cu = p.cu;
  const int cu0 = cu[b], qn = cu[b + 1] - cu0;
  const int Lseq = p.seq_lens[b];
  if (cu0 < 0 || qn < tok0 + ntok || cu[b + 1] > p.total_q || Lseq < qn ||
      Lseq > p.max_pages * kPageSize) {
    if (threadIdx.x == 0)
      set_status(p.status, Lseq > p.max_pages * kPageSize ? PA_DEV_BAD_SEQ_LEN : PA_DEV_PLAN_MISMATCH);
    return;  // CTA-uniform, nothing issued yet
  }
  const int pos0 = Lseq - qn + tok0;  // position of the tile's first query
  const int span = pos0 + ntok;       // keys 0 .. span-1
  const int nkt = (span + BN - 1) / BN;
  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages;
  const uint64_t policy = l2_evict_first_policy();

  // Stage kt: pages 2kt, 2kt+1 of the sequence (those below span) for K and
  // V; thread 0 only.
  auto issue = [&](int kt) {
    const int s = kt % NS;
    int phys[L::PAGES];
    int nvalid = 0;
#pragma unroll
    for (int u = 0; u < L::PAGES; ++u) {
      const int j = L::PAGES * kt + u;
      int ph = -1;
      if (j * kPageSize < span) {
        ph = __ldg(bt_row + j);
        if (ph < 0 || ph >= p.num_pages) {
          set_status(p.status, PA_DEV_BAD_PAGE);
          ph = -1;
        }
      }
      phys[u] = ph;
      nvalid += ph >= 0;
      asm volatile("st.shared.s32 [%0], %1;" ::"r"(pids + 4 * (s * L::PAGES + u)), "r"(ph)
                   : "memory");
    }
    fence_proxy_async_smem();
    const uint32_t bar = full + 8 * s;
    if (nvalid == 0) {
      mbar_arrive(bar);
      return;
    }
    mbar_arrive_expect_tx(bar, (uint32_t)(nvalid * 2 * L::TILE));
    const uint32_t dst = ring + s * L::STAGE;
#pragma unroll
    for (int u = 0; u < L::PAGES; ++u) {
      if (phys[u] < 0) continue;
#pragma unroll
      for (int bx = 0; bx < BOXES; ++bx) {
        tma_load_4d(dst + u * L::TILE + bx * 2048, &p.tmap_k, bx * 64, 0, g, phys[u], bar, policy);
        tma_load_4d(dst + (L::PAGES + u) * L::TILE + bx * 2048, &p.tmap_v, bx * 64, 0, g, phys[u],
                    bar, policy);
      }
    }
  };

  int issued = 0;
  if (threadIdx.x == 0) {
    for (; issued < nkt && issued < NS; ++issued) issue(issued);
  }

  // This thread's two rows: r0 = 16 warp + lg, r1 = r0 + 8.
  const int r0 = 16 * warp + lg, r1 = r0 + 8;
  const int tt0 = r0 / G, tt1 = r1 / G;
  const bool ok0 = tt0 < ntok, ok1 = tt1 < ntok;
  const int qp0 = pos0 + tt0, qp1 = pos0 + tt1;  // query positions
  const size_t row0 = ((size_t)(cu0 + tok0 + tt0) * p.num_q_heads + (size_t)g * G + r0 % G) * D;
  const size_t row1 = ((size_t)(cu0 + tok0 + tt1) * p.num_q_heads + (size_t)g * G + r1 % G) * D;

  // Q as A fragments: a0 = row r0, dims 16kk+2t..+1; a1 = row r1; a2, a3 = +8 dims.
  uint32_t qa[KSTEPS][4];
  {
    const T* q = static_cast<const T*>(p.q);
#pragma unroll
    for (int kk = 0; kk < KSTEPS; ++kk) {
      const int d = 16 * kk + 2 * t;
      qa[kk][0] = ok0 ? __ldg(reinterpret_cast<const unsigned int*>(q + row0 + d)) : 0u;
      qa[kk][1] = ok1 ? __ldg(reinterpret_cast<const unsigned int*>(q + row1 + d)) : 0u;
      qa[kk][2] = ok0 ? __ldg(reinterpret_cast<const unsigned int*>(q + row0 + d + 8)) : 0u;
      qa[kk][3] = ok1 ? __ldg(reinterpret_cast<const unsigned int*>(q + row1 + d + 8)) : 0u;
    }
  }

  // ldmatrix lane offsets (128-byte swizzle, chunk ^= row % 8).  K: lane l
  // addresses token row (l & 7) (+8 for the n-tile's second half, added per
  // n-tile) of 16-byte chunk 4kq + (l >> 3); V: token row (l & 7) + 8 ((l >> 3)
  // & 1) of chunk 2nd + (l >> 4).  The per-step chunk bits are XORed in.
  const int rr = lane & 7;
  const uint32_t k_off = (uint32_t)(rr * 128 + (((lane >> 3) ^ rr) << 4));
  const uint32_t v_off = (uint32_t)((rr + 8 * ((lane >> 3) & 1)) * 128 + (((lane >> 4) ^ rr) << 4));

  float m_run[2] = {-INFINITY, -INFINITY};
  float l_part[2] = {0.f, 0.f};
  float o[NTD][4];
#pragma unroll
  for (int n = 0; n < NTD; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  const float qs = p.qscale;

  bool failed = false;
  for (int kt = 0; kt < nkt; ++kt) {
    const int s = kt % NS;
    const uint32_t parity = (uint32_t)((kt / NS) & 1);
    if (!__all_sync(kFull, mbar_wait_bounded(full + 8 * s, parity, p.wait_ns))) {
      failed = true;
      break;
    }
    const uint32_t ktile = ring + s * L::STAGE;
    const uint32_t vtile = ktile + L::PAGES * L::TILE;
    const int kv0 = BN * kt;
    bool page_ok[L::PAGES];
#pragma unroll
    for (int u = 0; u < L::PAGES; ++u) page_ok[u] = lds_s32(pids + 4 * (s * L::PAGES + u)) >= 0;

    // ---- S = Q K^T over the stage's 4 n-tiles of 8 tokens
    float sc[4][4];
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const uint32_t kb = ktile + (nt >> 1) * L::TILE + (nt & 1) * 1024 + k_off;
#pragma unroll
      for (int kq = 0; kq < KSTEPS / 2; ++kq) {
        uint32_t r[4];
        ldsm_x4(((kb + (kq >> 1) * 2048) ^ (uint32_t)((kq & 1) << 6)), r[0], r[1], r[2], r[3]);
        mma_16816<T>(sc[nt], qa[2 * kq][0], qa[2 * kq][1], qa[2 * kq][2], qa[2 * kq][3], r[0], r[1]);
        mma_16816<T>(sc[nt], qa[2 * kq + 1][0], qa[2 * kq + 1][1], qa[2 * kq + 1][2],
                     qa[2 * kq + 1][3], r[2], r[3]);
      }
    }
    // ---- scale and mask (causal, and pages not copied)
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const int j = kv0 + 8 * nt + 2 * t;
      const bool pg = page_ok[nt >> 1];
      sc[nt][0] = (pg && ok0 && j <= qp0) ? sc[nt][0] * qs : -INFINITY;
      sc[nt][1] = (pg && ok0 && j + 1 <= qp0) ? sc[nt][1] * qs : -INFINITY;
      sc[nt][2] = (pg && ok1 && j <= qp1) ? sc[nt][2] * qs : -INFINITY;
      sc[nt][3] = (pg && ok1 && j + 1 <= qp1) ? sc[nt][3] * qs : -INFINITY;
      mx0 = fmaxf(mx0, fmaxf(sc[nt][0], sc[nt][1]));
      mx1 = fmaxf(mx1, fmaxf(sc[nt][2], sc[nt][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(kFull, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(kFull, mx1, 2));
    float al0 = 1.f, al1 = 1.f;
    if (mx0 > m_run[0] + kLazyLog2Prefill) {  // uniform across the 4 lanes of a row
      al0 = ex2(m_run[0] - mx0);              // 0 on the row's first live stage
      m_run[0] = mx0;
    }
    if (mx1 > m_run[1] + kLazyLog2Prefill) {
      al1 = ex2(m_run[1] - mx1);
      m_run[1] = mx1;
    }
    if (__any_sync(kFull, al0 != 1.f || al1 != 1.f)) {
#pragma unroll
      for (int n = 0; n < NTD; ++n) {
        o[n][0] *= al0;
        o[n][1] *= al0;
        o[n][2] *= al1;
        o[n][3] *= al1;
      }
    }
    const bool dead0 = m_run[0] == -INFINITY, dead1 = m_run[1] == -INFINITY;
    float ps0 = 0.f, ps1 = 0.f;
    uint32_t pa[L::PAGES][4], pl[L::PAGES][4];  // P hi and lo parts
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
      const float p0 = dead0 ? 0.f : ex2(sc[nt][0] - m_run[0]);
      const float p1 = dead0 ? 0.f : ex2(sc[nt][1] - m_run[0]);
      const float p2 = dead1 ? 0.f : ex2(sc[nt][2] - m_run[1]);
      const float p3 = dead1 ? 0.f : ex2(sc[nt][3] - m_run[1]);
      ps0 += p0 + p1;
      ps1 += p2 + p3;
      // n-tile 2u is tokens 0-7 (a0, a1) of page u's k-step, 2u+1 tokens 8-15 (a2, a3)
      split_hi_lo<T>(make_float2(p0, p1), pa[nt >> 1][(nt & 1) * 2 + 0], pl[nt >> 1][(nt & 1) * 2 + 0]);
      split_hi_lo<T>(make_float2(p2, p3), pa[nt >> 1][(nt & 1) * 2 + 1], pl[nt >> 1][(nt & 1) * 2 + 1]);
    }
    l_part[0] = l_part[0] * al0 + ps0;
    l_part[1] = l_part[1] * al1 + ps1;

    // ---- O += P V, one k-step per page.  V rows at or past the span (or of
    // a page not copied) have P = 0 but may hold anything, NaN too: their
    // halves of the fragments are zeroed.
#pragma unroll
    for (int u = 0; u < L::PAGES; ++u) {
      const uint32_t vb = vtile + u * L::TILE + v_off;
      const int vlim = page_ok[u] ? span - (kv0 + kPageSize * u) : 0;  // valid tokens of page u
      const uint32_t mk0 = (2 * t < vlim ? 0x0000ffffu : 0u) | (2 * t + 1 < vlim ? 0xffff0000u : 0u);
      const uint32_t mk8 =
          (2 * t + 8 < vlim ? 0x0000ffffu : 0u) | (2 * t + 9 < vlim ? 0xffff0000u : 0u);
#pragma unroll
      for (int nd = 0; nd < NTD / 2; ++nd) {
        uint32_t r[4];
        ldsm_x4_t((vb + (nd >> 2) * 2048) ^ (uint32_t)((nd & 3) << 5), r[0], r[1], r[2], r[3]);
        if (vlim < kPageSize) {
          r[0] &= mk0;
          r[1] &= mk8;
          r[2] &= mk0;
          r[3] &= mk8;
        }
        mma_16816<T>(o[2 * nd], pa[u][0], pa[u][1], pa[u][2], pa[u][3], r[0], r[1]);
        mma_16816<T>(o[2 * nd + 1], pa[u][0], pa[u][1], pa[u][2], pa[u][3], r[2], r[3]);
        mma_16816<T>(o[2 * nd], pl[u][0], pl[u][1], pl[u][2], pl[u][3], r[0], r[1]);
        mma_16816<T>(o[2 * nd + 1], pl[u][0], pl[u][1], pl[u][2], pl[u][3], r[2], r[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(empty + 8 * s);
    // ---- refill this stage once every warp is done with it
    if (warp == 0) {
      bool ok = true;
      if (lane == 0 && issued < nkt && issued == kt + NS) {
        ok = mbar_wait_bounded(empty + 8 * s, parity, p.wait_ns);
        if (ok) issue(issued++);
      }
      if (!__all_sync(kFull, ok)) {
        failed = true;
        break;
      }
    }
  }

  if (failed && lane == 0) {
    set_status(p.status, PA_DEV_TIMEOUT);
    *cta_flag = 1;
  }
  __syncthreads();  // every warp is done with the ring
  if (threadIdx.x == 0) {
    // the last NS stages issued may still be in flight after a failure
    for (int kt = issued - NS < 0 ? 0 : issued - NS; kt < issued; ++kt)
      mbar_wait_bounded(full + 8 * (kt % NS), (uint32_t)((kt / NS) & 1), kDrainWaitNs);
  }
  if (*cta_flag) return;

  // ---- normalise and write the rows
  l_part[0] += __shfl_xor_sync(kFull, l_part[0], 1);
  l_part[0] += __shfl_xor_sync(kFull, l_part[0], 2);
  l_part[1] += __shfl_xor_sync(kFull, l_part[1], 1);
  l_part[1] += __shfl_xor_sync(kFull, l_part[1], 2);
  const float inv0 = l_part[0] > 0.f ? 1.f / l_part[0] : 0.f;
  const float inv1 = l_part[1] > 0.f ? 1.f / l_part[1] : 0.f;
  T* out = static_cast<T*>(p.out);
#pragma unroll
  for (int n = 0; n < NTD; ++n) {
    const int d = 8 * n + 2 * t;
    if (ok0) *reinterpret_cast<uint32_t*>(out + row0 + d) = Elem<T>::from_f2(o[n][0] * inv0, o[n][1] * inv0);
    if (ok1) *reinterpret_cast<uint32_t*>(out + row1 + d) = Elem<T>::from_f2(o[n][2] * inv1, o[n][3] * inv1);
  }
}

}  // namespace pa
