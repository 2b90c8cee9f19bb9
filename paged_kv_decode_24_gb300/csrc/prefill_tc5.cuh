// Multi-token attention on the fifth-generation tensor cores (tcgen05):
// the same operation as prefill.cuh, on 128-row tiles, with MMAs issued by
// one thread from shared-memory descriptors and tensor memory (TMEM) into
// TMEM.
//
// A CTA owns 128 query rows of one (sequence, KV head): 128 / G query tokens
// times the G heads of the KV head.  Thread r of warps 0-3 owns row r, which
// is TMEM lane r, so a row's softmax needs no shuffles.  Warp 4 issues the
// MMAs, warp 5 the key copies and warp 6 the value copies; the warps meet
// only on mbarriers.
// Shared memory (1024-aligned, 128-byte swizzle everywhere, the layout the
// TMA copies and the row threads write and the MMA descriptors read):
//   a ring of NK key stages of 64 tokens (four pages), each
//     K [D/64 boxes][64 tokens][128 B]        B operand of S, K-major
//   a ring of NV value stages of 64 tokens, each
//     V [D/64 boxes][64 tokens][128 B]        B operand of P.V, MN-major
//   Q   [D/64 boxes][128 rows][128 B]         A operand of S, K-major
// TMEM: two buffers of 64 columns and O of D columns.  Stage kt uses buffer
// kt & 1: S(kt) lands there, and once the row threads have read it P(kt)
// takes its place, P_hi then P_lo, keys 2j and 2j+1 in column j, the A
// operand of P.V (row m in lane m).
// The weights p are kept as two 16-bit parts, hi = p rounded to the element
// type and lo = the remainder rounded, and O accumulates P_hi V + P_lo V:
// about twice the element type's bits of p, as in the decode kernels, so
// the result stays within the decode path's tolerance.  Keeping P in TMEM
// spares the shared-memory traffic of storing and reading it (twice the
// bytes with the lo part) for that of reading Q.
//
// Per stage kt:
//   S(kt) = Q K^T  (D/16 MMAs, M = 128, N = 64) into buffer kt & 1,
//     issued once P.V(kt-2) has finished reading that buffer;  committed to s_done[kt & 1]
//   the row threads load S(kt) into registers; row softmax, lazy rescaling
//   P(kt) hi and lo into the same columns, with no wait on P.V(kt-1),
//     which reads the other buffer
//   O += P_hi V + P_lo V   (8 MMAs, M = 128, N = D, K = 16 each)   committed to pv_done
// Keys and values have rings of their own: a key stage is refilled as soon
// as S has read it, a value stage once P.V has.  Sixty-four keys per stage
// spread each stage's fixed costs (waits, fences, TMEM loads) over twice the
// keys of a two-page stage.  Waiting warps sleep on their barriers
// (mbar_wait_bounded_sleep) so that they take no issue slots from the row
// warps.
// Every wait is bounded; on failure the CTA waits (bounded) for its copies
// and MMAs, frees its TMEM and writes nothing.
#pragma once

#include <cuda.h>
#include <math.h>

#include "decode_tc.cuh"
#include "elem.cuh"
#include "prefill.cuh"

namespace pa {

namespace tc5 {

// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets, the fixed version bits and the swizzle mode (2: 128-byte, 4:
// 64-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo,
                                              uint32_t swizzle = 2) {
  uint64_t d = 0;
  d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
  d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
  d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
  d |= (uint64_t)1 << 46;
  d |= (uint64_t)swizzle << 61;
  return d;
}

// Instruction descriptor of kind::f16: fp32 accumulator, A and B of the
// element type, major-ness of A and B, N and M.
template <typename T>
__device__ __forceinline__ uint32_t instr_desc(int m, int n, bool b_mn_major) {
  const uint32_t ty = std::is_same<T, __half>::value ? 0u : 1u;
  return (1u << 4) | (ty << 7) | (ty << 10) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(n >> 3) << 17) | ((uint32_t)(m >> 4) << 24);
}

__device__ __forceinline__ void mma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                    uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

// The same with A (M x K, K-major) read from TMEM: row m in lane m, two
// 16-bit elements per 32-bit column.
__device__ __forceinline__ void mma_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b,
                                           uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void commit(uint32_t bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ void fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void ld16(uint32_t taddr, float* v) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void st16u(uint32_t taddr, const uint32_t* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
      "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
}

__device__ __forceinline__ void st16(uint32_t taddr, const float* v) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, "
      "%11, %12, %13, %14, %15, %16};" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15]))
      : "memory");
}

// L2 policy for the keys and values: the other tiles of the sequence read
// them again.
__device__ __forceinline__ uint64_t l2_evict_normal_policy() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_normal.b64 %0, 1.0;" : "=l"(p));
  return p;
}

}  // namespace tc5

// d = a + b on two fp32 lanes with one instruction.
__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
  float2 d;
  asm("{\n\t.reg .b64 ra, rb, rd;\n\t"
      "mov.b64 ra, {%2, %3};\n\t"
      "mov.b64 rb, {%4, %5};\n\t"
      "add.rn.f32x2 rd, ra, rb;\n\t"
      "mov.b64 {%0, %1}, rd;\n\t}"
      : "=f"(d.x), "=f"(d.y)
      : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y));
  return d;
}

namespace tc5 {

__device__ __forceinline__ void wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

}  // namespace tc5

constexpr int kTc5Rows = 128;                        // query rows per CTA (one TMEM lane each)
constexpr int kTc5Tokens = 64;                       // keys per stage
constexpr int kTc5Pages = kTc5Tokens / kPageSize;    // pages per stage
constexpr int kTc5Threads = 224;  // row warps 0-3, MMA warp 4, key copies 5, value copies 6

// Two CTAs share an SM (113 KB of shared memory and 256 TMEM columns each).
template <int D>
struct Tc5Layout {
  static constexpr int BOXES = D / 64;
  static constexpr int NK = D == 128 ? 3 : 6;                   // key stages
  static constexpr int NV = D == 128 ? 2 : 4;                   // value stages
  // An idle row warp waits for the last stage's value copies without having
  // waited for P.V of the stage before.  With one value slot that stage's
  // copy may still be in flight, and the parity wait would then read the
  // phase before it as complete.  With two or more slots the slot's earlier
  // phases are always complete.  A single value slot was measured to
  // corrupt exactly those tiles.
  static_assert(NV >= 2, "value ring needs two slots");
  static constexpr int KVBOX = kTc5Tokens * 128;                // 8 KB per box
  static constexpr int STAGE = BOXES * KVBOX;                   // one K or V stage
  static constexpr int K0 = 0;
  static constexpr int V0 = K0 + NK * STAGE;
  static constexpr int QBOX = kTc5Rows * 128;                   // 16 KB: 64 dims of 128 rows
  static constexpr int Q = V0 + NV * STAGE;                     // Q [D/64 boxes][128 rows][128 B]
  static constexpr int BUFS = Q + BOXES * QBOX;                 // the 1024-aligned buffers
  // SMALL bytes hold the mbarriers (k_full[NK], k_free[NK], v_full[NV],
  // v_free[NV], s_done[2], pv_done[2], p_ready[2], drain), the TMEM
  // address and a flag.  The buffers start at the first 1024-byte boundary
  // of the allocation (the 128-byte swizzle needs it); the small area goes
  // before them when the gap is wide enough, else after them, so BUFS + 1024
  // bytes always hold both.
  static constexpr int SMALL = 256;
  static constexpr int BARS = 0;
  static constexpr int TMEM_SLOT = align_up(BARS + 8 * (2 * NK + 2 * NV + 7), 16);
  static constexpr int FLAG = TMEM_SLOT + 16;
  static_assert(FLAG + 16 <= SMALL, "barriers overflow their area");
  static constexpr int BYTES = BUFS + 1024;
  static constexpr uint32_t TMEM_COLS = 256;                    // two S/P buffers (64 each), O (D)
};

template <typename T, int D, int G>
__global__ void __launch_bounds__(kTc5Threads, 2)
    prefill_tc5_kernel(const __grid_constant__ PrefillParams p) {
  static_assert(D == 64 || D == 128, "head_dim 64 or 128");
  using L = Tc5Layout<D>;
  constexpr int NK = L::NK;
  constexpr int NV = L::NV;
  constexpr int BN = kTc5Tokens;
  constexpr int TOKS = kTc5Rows / G;
  extern __shared__ __align__(16) unsigned char smem_dyn[];
  unsigned char* base = reinterpret_cast<unsigned char*>(
      (reinterpret_cast<uintptr_t>(smem_dyn) + 1023) & ~uintptr_t(1023));
  unsigned char* small = base - smem_dyn >= L::SMALL ? smem_dyn : base + L::BUFS;
  const uint32_t sbase = smem_u32(base);
  const uint32_t ssmall = smem_u32(small);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int lane = tid & 31;
  const bool mma_warp = warp == 4;
  const bool copy_warp = warp == 5 || warp == 6;
  const bool row_warp = warp < 4;
  const uint32_t k_full = ssmall + L::BARS;     // NK: a key stage's copies landed
  const uint32_t k_free = k_full + 8 * NK;      // NK: S has read a key stage
  const uint32_t v_full = k_free + 8 * NK;      // NV: a value stage's copies landed
  const uint32_t v_free = v_full + 8 * NV;      // NV: P.V has read a value stage
  const uint32_t s_done = v_free + 8 * NV;      // 2: S(kt) computed, into buffer kt & 1
  const uint32_t pv_done = s_done + 16;         // 2: P.V(kt) computed
  // 2: P(kt) written and O rescaled by the 4 row warps.  Two phases of one
  // barrier could complete before the MMA warp looks at the first.
  const uint32_t p_ready = pv_done + 16;
  const uint32_t drain = p_ready + 16;          // every MMA issued has finished
  int* cta_flag = reinterpret_cast<int*>(small + L::FLAG);

  if ((int)blockIdx.x >= p.num_tiles) return;  // whole CTA
  const int4 hdr = *reinterpret_cast<const int4*>(p.ws);
  const int4 tile = reinterpret_cast<const int4*>(p.ws + 16)[blockIdx.x];
  if (tid == 0) {
    *cta_flag = 0;
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_k)) : "memory");
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&p.tmap_v)) : "memory");
    for (int s = 0; s < NK; ++s) {
      mbar_init(k_full + 8 * s, 1);
      mbar_init(k_free + 8 * s, 1);
    }
    for (int s = 0; s < NV; ++s) {
      mbar_init(v_full + 8 * s, 1);
      mbar_init(v_free + 8 * s, 1);
    }
    mbar_init(s_done, 1);
    mbar_init(s_done + 8, 1);
    mbar_init(pv_done, 1);
    mbar_init(pv_done + 8, 1);
    mbar_init(p_ready, 4);
    mbar_init(p_ready + 8, 4);
    mbar_init(drain, 1);
    fence_barrier_init();
  }
  if (mma_warp) {  // TMEM for this CTA, freed by this warp at the end
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     ssmall + L::TMEM_SLOT),
                 "r"(L::TMEM_COLS)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc5::fence_before();
  __syncthreads();
  tc5::fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(small + L::TMEM_SLOT);
  // columns: S, O, then P: hi (keys 2j, 2j+1 in column j) and lo, 32 each
  const uint32_t t_x = tmem, t_o = tmem + 2 * BN;
  const uint32_t lane_off = (uint32_t)(32 * (warp & 3)) << 16;  // a row warp's TMEM lanes

  pdl_launch_dependents();
  pdl_wait_primary();

  const int b = tile.x, g = tile.y, tok0 = tile.z, ntok = tile.w;
  bool bad = hdr.x != (int)kPrefillMagic || hdr.y != p.num_tiles || hdr.z != p.batch ||
             hdr.w != p.total_q || b < 0 || b >= p.batch || g < 0 || g >= p.num_kv_heads ||
             tok0 < 0 || ntok < 1 || ntok > TOKS;
  int cu0 = 0, qn = 0, Lseq = 0;
  if (!bad) {
    cu0 = p.cu[b];
    qn = p.cu[b + 1] - cu0;
    Lseq = p.seq_lens[b];
    if (cu0 < 0 || qn < tok0 + ntok || p.cu[b + 1] > p.total_q || Lseq < qn ||
        Lseq > p.max_pages * kPageSize) {
      if (tid == 0)
        set_status(p.status, Lseq > p.max_pages * kPageSize ? PA_DEV_BAD_SEQ_LEN : PA_DEV_PLAN_MISMATCH);
      bad = true;
    }
  } else if (tid == 0) {
    set_status(p.status, PA_DEV_PLAN_MISMATCH);
  }
  const int pos0 = Lseq - qn + tok0;
  const int span = pos0 + ntok;
  const int nkt = bad ? 0 : (span + BN - 1) / BN;
  const int32_t* bt_row = p.block_table + (size_t)b * p.max_pages;

  // ---- Q tile into shared memory (row = thread of warps 0-3), zero past
  // ntok: K-major with the 128-byte swizzle, [D/64 boxes][128 rows][128 B],
  // 16-byte chunk c of a row's box at chunk c ^ (row % 8)
  const int row = tid & 127;
  const int tt = row / G;                 // query token of this row within the tile
  const bool ok = !bad && row_warp && tt < ntok;
  const int qpos = pos0 + tt;             // its position
  const size_t qrow = ((size_t)(cu0 + tok0 + tt) * p.num_q_heads + (size_t)g * G + row % G) * D;
  if (row_warp) {
    const uint4* src = reinterpret_cast<const uint4*>(static_cast<const T*>(p.q) + qrow);
#pragma unroll
    for (int c = 0; c < D / 8; ++c) {
      const uint4 v = ok ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
      *reinterpret_cast<uint4*>(base + L::Q + (c >> 3) * L::QBOX + row * 128 +
                                (((c & 7) ^ (row & 7)) << 4)) = v;
    }
    fence_proxy_async_smem();  // the tensor core reads it (async proxy)
  }
  // Q is in shared memory for the MMA warp: the row warps and the MMA warp
  // meet on a named barrier; the copy warps, which do not read Q, start at once.
  if (!copy_warp) {
    tc5::fence_before();
    asm volatile("bar.sync 1, %0;" ::"n"(5 * 32) : "memory");
    tc5::fence_after();
  }

  if (copy_warp) {
    // ================= copies (lane 0 of warp 5: keys, of warp 6: values) =================
    // Stage kt holds pages 4kt .. 4kt+3 of the sequence; a page past the
    // span or with an invalid index is not copied (its keys are masked, and
    // the row warps zero its value rows before P.V reads them).  Each ring
    // runs as far ahead as its own slots allow: a key slot is free once S
    // has read it, a value slot once P.V has.  (With one warp for both, the
    // keys would wait behind the value ring, which frees a stage later.)
    if (lane == 0 && nkt > 0) {
      const bool keys = warp == 5;
      const int NR = keys ? NK : NV;
      const uint32_t ring = sbase + (keys ? L::K0 : L::V0);
      const uint32_t full_bar = keys ? k_full : v_full;
      const uint32_t free_bar = keys ? k_free : v_free;
      const CUtensorMap* map = keys ? &p.tmap_k : &p.tmap_v;
      const uint64_t policy = tc5::l2_evict_normal_policy();
      const uint32_t kv_bytes = (uint32_t)(D * kPageSize * 2);
      // The block-table entries of stage kt+1 are loaded while the slot of
      // stage kt is awaited, so their latency is off the copy path.  The
      // loads are volatile asm, which the compiler keeps in place.
      int nxt[kTc5Pages];
      auto load_entries = [&](int kt) {
#pragma unroll
        for (int u = 0; u < kTc5Pages; ++u) {
          const int j = kTc5Pages * kt + u;
          nxt[u] = -1;
          if (j * kPageSize < span)
            asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(nxt[u]) : "l"(bt_row + j));
        }
      };
      load_entries(0);
      int n = 0;  // stages issued
      bool good = true;
      for (int kt = 0; kt < nkt; ++kt) {
        int phys[kTc5Pages];
#pragma unroll
        for (int u = 0; u < kTc5Pages; ++u) phys[u] = nxt[u];
        if (kt + 1 < nkt) load_entries(kt + 1);
        const int slot = kt % NR;
        good = kt < NR || mbar_wait_bounded_sleep(free_bar + 8 * slot, (uint32_t)((kt / NR - 1) & 1), p.wait_ns);
        if (!good) break;
        int nvalid = 0;
        bool zeroed = false;
#pragma unroll
        for (int u = 0; u < kTc5Pages; ++u) {
          const int j = kTc5Pages * kt + u;
          if (j * kPageSize < span && (phys[u] < 0 || phys[u] >= p.num_pages)) {
            if (keys) {
              set_status(p.status, PA_DEV_BAD_PAGE);
            } else {
              // a page inside the span that is not copied: its keys are
              // masked, and its value rows (which may hold anything from
              // earlier stages) become zeros before P.V reads them
              for (int bx = 0; bx < L::BOXES; ++bx)
                for (int c = 0; c < kPageSize * 8; ++c)
                  *reinterpret_cast<uint4*>(base + L::V0 + slot * L::STAGE + bx * L::KVBOX +
                                            u * 2048 + c * 16) =
                      make_uint4(0u, 0u, 0u, 0u);
              zeroed = true;
            }
            phys[u] = -1;
          }
          nvalid += phys[u] >= 0;
        }
        if (zeroed) fence_proxy_async_smem();  // the tensor core reads them (async proxy)
        const uint32_t bar = full_bar + 8 * slot;
        if (nvalid == 0) {
          mbar_arrive(bar);
        } else {
          mbar_arrive_expect_tx(bar, (uint32_t)nvalid * kv_bytes);
#pragma unroll
          for (int u = 0; u < kTc5Pages; ++u)
            if (phys[u] >= 0)
              for (int bx = 0; bx < L::BOXES; ++bx)
                tma_load_4d(ring + slot * L::STAGE + bx * L::KVBOX + u * 2048, map, bx * 64, 0,
                            g, phys[u], bar, policy);
        }
        ++n;
      }
      if (!good) {
        set_status(p.status, PA_DEV_TIMEOUT);
        *reinterpret_cast<volatile int*>(cta_flag) = 1;
      }
      // copies in flight land before the CTA exits: the last stage issued
      // into each slot (on success all of them have been consumed already)
      for (int k = n - NR < 0 ? 0 : n - NR; k < n; ++k)
        mbar_wait_bounded_sleep(full_bar + 8 * (k % NR), (uint32_t)((k / NR) & 1), kDrainWaitNs);
    }
    __syncwarp();
  } else if (mma_warp) {
    // ================= MMAs (lane 0) =================
    if (lane == 0 && nkt > 0) {
      const uint32_t idesc_s = tc5::instr_desc<T>(128, BN, false);
      const uint32_t idesc_o = tc5::instr_desc<T>(128, D, true);
      auto issue_s = [&](int kt) -> bool {  // S(kt) = Q K^T
        const int sk = kt % NK;
        if (!mbar_wait_bounded_sleep(k_full + 8 * sk, (uint32_t)((kt / NK) & 1), p.wait_ns)) return false;
        tc5::fence_after();
        const uint32_t kst = sbase + L::K0 + sk * L::STAGE;
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint64_t ad = tc5::smem_desc(sbase + L::Q + (k >> 2) * L::QBOX + (k & 3) * 32, 16, 1024);
          const uint64_t bd = tc5::smem_desc(kst + (k >> 2) * L::KVBOX + (k & 3) * 32, 16, 1024);
          tc5::mma(t_x + (uint32_t)(BN * (kt & 1)), ad, bd, idesc_s, k > 0 ? 1u : 0u);
        }
        tc5::commit(k_free + 8 * sk);
        tc5::commit(s_done + 8 * (kt & 1));
        return true;
      };
      bool good = issue_s(0);
      for (int kt = 0; kt < nkt && good; ++kt) {
        if (kt + 1 < nkt) {
          // buffer (kt + 1) & 1 holds P(kt - 1) until P.V(kt - 1) has read it
          good = (kt < 1 || mbar_wait_bounded_sleep(pv_done + 8 * ((kt - 1) & 1),
                                                    (uint32_t)(((kt - 1) >> 1) & 1), p.wait_ns)) &&
                 issue_s(kt + 1);
          if (!good) break;
        }
        const int sv = kt % NV;
        good = mbar_wait_bounded_sleep(p_ready + 8 * (kt & 1), (uint32_t)((kt >> 1) & 1), p.wait_ns) &&
               mbar_wait_bounded_sleep(v_full + 8 * sv, (uint32_t)((kt / NV) & 1), p.wait_ns);
        if (!good) break;
        tc5::fence_after();
        const uint32_t vst = sbase + L::V0 + sv * L::STAGE;
#pragma unroll
        for (int k = 0; k < BN / 16; ++k) {
          const uint64_t bd = tc5::smem_desc(vst + k * 2048, L::KVBOX, 1024);
          const uint32_t t_p = t_x + (uint32_t)(BN * (kt & 1));
          tc5::mma_tmem_a(t_o, t_p + (uint32_t)(8 * k), bd, idesc_o, (kt > 0 || k > 0) ? 1u : 0u);
          tc5::mma_tmem_a(t_o, t_p + 32u + (uint32_t)(8 * k), bd, idesc_o, 1u);
        }
        tc5::commit(v_free + 8 * sv);
        tc5::commit(pv_done + 8 * (kt & 1));
      }
      if (!good) {
        set_status(p.status, PA_DEV_TIMEOUT);
        *reinterpret_cast<volatile int*>(cta_flag) = 1;
      }
      // every MMA issued finishes before TMEM is freed: one more commit
      // covers them all
      tc5::commit(drain);
      mbar_wait_bounded_sleep(drain, 0u, kDrainWaitNs);
    }
    __syncwarp();
  } else {
    // ================= rows: softmax and output (warps 0-3) =================
    float m_run = -INFINITY, l_run = 0.f;
    bool good = true;
    // Value rows past the span (which may hold anything) become zeros in the
    // last stage, after its value copies have landed (they would overwrite).
    // Each of the 128 row threads takes its share.
    auto zero_value_tail = [&](int kt) -> bool {
      const int sv_slot = kt % NV;
      if (!__all_sync(kFull, mbar_wait_bounded_sleep(v_full + 8 * sv_slot, (uint32_t)((kt / NV) & 1), p.wait_ns)))
        return false;
      const int first_bad = span - BN * kt;  // tokens [first_bad, BN) of this stage
      unsigned char* vsm = base + L::V0 + sv_slot * L::STAGE;
      for (int i = row; i < L::BOXES * BN * 8; i += 128) {  // 16-byte chunks
        const int bx = i / (BN * 8), r = (i / 8) % BN, ch = i % 8;
        if (r >= first_bad)
          *reinterpret_cast<uint4*>(vsm + bx * L::KVBOX + r * 128 + (ch << 4)) =
              make_uint4(0u, 0u, 0u, 0u);
      }
      return true;
    };
    // A warp without a query row in the tile (a short tile: fewer than 32 /
    // G tokens per 32 rows) computes nothing.  It keeps its place in the
    // barrier counts and zeroes its share of value rows; its P rows feed O
    // rows that are never written.
    const bool idle = !__any_sync(kFull, ok);
    for (int kt = 0; idle && kt < nkt; ++kt) {
      good = __all_sync(kFull, mbar_wait_bounded_sleep(s_done + 8 * (kt & 1), (uint32_t)((kt >> 1) & 1), p.wait_ns));
      if (!good) break;
      __syncwarp();
      if (BN * kt + BN > span && !zero_value_tail(kt)) {
        good = false;
        break;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready + 8 * (kt & 1));
    }
    // block-table entries of the stage, loaded one stage ahead (page checks
    // mask the keys of a page that was not copied)
    int nph[kTc5Pages];
#pragma unroll
    for (int u = 0; u < kTc5Pages; ++u)
      nph[u] = !idle && nkt > 0 && u * kPageSize < span ? __ldg(bt_row + u) : -1;
    for (int kt = 0; !idle && kt < nkt; ++kt) {
      bool pgv[kTc5Pages];
      bool all_pages = true;
#pragma unroll
      for (int u = 0; u < kTc5Pages; ++u) {
        pgv[u] = nph[u] >= 0 && nph[u] < p.num_pages;
        all_pages = all_pages && pgv[u];
      }
      if (kt + 1 < nkt) {  // volatile asm loads stay here, a stage ahead of their use
#pragma unroll
        for (int u = 0; u < kTc5Pages; ++u) {
          const int j = kTc5Pages * (kt + 1) + u;
          nph[u] = -1;
          if (j * kPageSize < span)
            asm volatile("ld.global.nc.s32 %0, [%1];" : "=r"(nph[u]) : "l"(bt_row + j));
        }
      }
      good = __all_sync(kFull, mbar_wait_bounded_sleep(s_done + 8 * (kt & 1), (uint32_t)((kt >> 1) & 1), p.wait_ns));
      if (!good) break;
      tc5::fence_after();
      const uint32_t t_sp = t_x + (uint32_t)(BN * (kt & 1));  // S(kt), then P(kt)
      float sv[BN];
#pragma unroll
      for (int c = 0; c < BN; c += 16) tc5::ld16(t_sp + (uint32_t)c + lane_off, sv + c);
      tc5::wait_ld();

      // ---- mask, row max (lazy), weights
      const int kv0 = BN * kt;
      // visible iff the page was copied and the key is not after the query;
      // a stage every lane of the warp sees whole skips the per-key test
      const int lim = ok ? qpos - kv0 : -1;  // last visible column of the stage
      if (!__all_sync(kFull, all_pages && lim >= BN - 1)) {
#pragma unroll
        for (int c = 0; c < BN; ++c) {
          const bool vis = pgv[c / kPageSize] && c <= lim;
          sv[c] = vis ? sv[c] : -INFINITY;
        }
      }
      // row max of the raw scores (the scale is positive), tree-reduced
      float mx;
      {
        float t[BN / 2];
#pragma unroll
        for (int c = 0; c < BN / 2; ++c) t[c] = fmaxf(sv[c], sv[c + BN / 2]);
#pragma unroll
        for (int w = BN / 4; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) t[c] = fmaxf(t[c], t[c + w]);
        mx = t[0] * p.qscale;  // in scaled (log2) units
      }
      float al = 1.f;
      bool resc = false;
      if (mx > m_run + kLazyLog2Prefill) {
        al = ex2(m_run - mx);  // 0 when the row had no weight yet
        resc = m_run != -INFINITY;
        m_run = mx;
      }
      // p = 2^(s * scale - m): one ex2 per key, the arguments and the row
      // sum on packed pairs (fma.rn.f32x2, add.rn.f32x2); p is kept as hi
      // (pk) + lo (pl)
      uint32_t pk[BN / 2], pl[BN / 2];
      float ps;
      {
        float2 t[BN / 4];
        // a row with no weight yet has only masked (-inf) scores: 2^-inf = 0
        const float nm = m_run == -INFINITY ? -INFINITY : -m_run;
        const float2 qs2 = make_float2(p.qscale, p.qscale), nm2 = make_float2(nm, nm);
#pragma unroll
        for (int c = 0; c < BN; c += 4) {
          const float2 x0 = ffma2(make_float2(sv[c], sv[c + 1]), qs2, nm2);
          const float2 x1 = ffma2(make_float2(sv[c + 2], sv[c + 3]), qs2, nm2);
          const float2 a0 = make_float2(ex2(x0.x), ex2(x0.y));
          const float2 a1 = make_float2(ex2(x1.x), ex2(x1.y));
          t[c / 4] = fadd2(a0, a1);
          split_hi_lo<T>(a0, pk[c / 2], pl[c / 2]);
          split_hi_lo<T>(a1, pk[c / 2 + 1], pl[c / 2 + 1]);
        }
#pragma unroll
        for (int w = BN / 8; w >= 1; w >>= 1)
#pragma unroll
          for (int c = 0; c < w; ++c) t[c] = fadd2(t[c], t[c + w]);
        ps = t[0].x + t[0].y;
      }
      l_run = l_run * al + ps;

      // ---- P(kt) goes over S(kt) in its buffer, which P.V(kt - 2) has
      // finished reading before S(kt) was issued; O may be rescaled only
      // once P.V(kt-1) is done
      const bool any_resc = __any_sync(kFull, resc);
      if (any_resc && kt >= 1) {
        good = __all_sync(kFull, mbar_wait_bounded_sleep(pv_done + 8 * ((kt - 1) & 1),
                                                   (uint32_t)(((kt - 1) >> 1) & 1), p.wait_ns));
        if (!good) break;
      }
      tc5::fence_after();
      // ---- P(kt) row, hi and lo, into TMEM (lane = row, column j = keys
      // 2j, 2j+1), before the rescale so that their registers are free for it
      tc5::st16u(t_sp + lane_off, pk);
      tc5::st16u(t_sp + 16u + lane_off, pk + 16);
      tc5::st16u(t_sp + 32u + lane_off, pl);
      tc5::st16u(t_sp + 48u + lane_off, pl + 16);
      tc5::wait_st();
      if (any_resc && kt >= 1) {  // rare: rescale this warp's O rows in TMEM
        const float f = resc ? al : 1.f;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          float ov[16];
          tc5::ld16(t_o + (uint32_t)c + lane_off, ov);
          tc5::wait_ld();
#pragma unroll
          for (int i = 0; i < 16; ++i) ov[i] *= f;
          tc5::st16(t_o + (uint32_t)c + lane_off, ov);
        }
        tc5::wait_st();
      }
      // value rows past the span (which may hold anything) become zeros
      if (kv0 + BN > span && !zero_value_tail(kt)) {
        good = false;
        break;
      }
      fence_proxy_async_smem();
      tc5::fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(p_ready + 8 * (kt & 1));
    }
    if (!idle && nkt > 0 && good) {
      good = __all_sync(kFull, mbar_wait_bounded_sleep(pv_done + 8 * ((nkt - 1) & 1),
                                                 (uint32_t)(((nkt - 1) >> 1) & 1), p.wait_ns));
      // a copy or MMA warp that gave up leaves O incomplete: write nothing
      good = good && *reinterpret_cast<volatile int*>(cta_flag) == 0;
      good = __all_sync(kFull, good);
      if (good) {
        tc5::fence_after();
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
        T* out = static_cast<T*>(p.out) + qrow;
#pragma unroll
        for (int c = 0; c < D; c += 16) {
          float ov[16];
          tc5::ld16(t_o + (uint32_t)c + lane_off, ov);
          tc5::wait_ld();
          if (ok) {
            uint4 w0, w1;
            w0.x = Elem<T>::from_f2(ov[0] * inv, ov[1] * inv);
            w0.y = Elem<T>::from_f2(ov[2] * inv, ov[3] * inv);
            w0.z = Elem<T>::from_f2(ov[4] * inv, ov[5] * inv);
            w0.w = Elem<T>::from_f2(ov[6] * inv, ov[7] * inv);
            w1.x = Elem<T>::from_f2(ov[8] * inv, ov[9] * inv);
            w1.y = Elem<T>::from_f2(ov[10] * inv, ov[11] * inv);
            w1.z = Elem<T>::from_f2(ov[12] * inv, ov[13] * inv);
            w1.w = Elem<T>::from_f2(ov[14] * inv, ov[15] * inv);
            reinterpret_cast<uint4*>(out + c)[0] = w0;
            reinterpret_cast<uint4*>(out + c)[1] = w1;
          }
        }
      }
    }
    if (!good && lane == 0) set_status(p.status, PA_DEV_TIMEOUT);
  }

  // ---- free TMEM once every warp is done with it
  tc5::fence_before();
  __syncthreads();
  if (mma_warp) {
    tc5::fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                 "r"(L::TMEM_COLS)
                 : "memory");
  }
}

}  // namespace pa
