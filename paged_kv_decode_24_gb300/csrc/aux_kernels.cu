// The stand-alone split combine, KV append (fp16, INT8 and FP8 caches), the
// multi-token append, the block copy and the debug gather-index export.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "device_common.cuh"
#include "elem.cuh"
#include "launch.h"
#include "quant_common.cuh"

namespace pa {

// ---------------------------------------------------------------------------
// Combine: one CTA per (sequence, KV head, query head in the group) whose
// sequence was split.  With partials (o_s, lse_s) in base 2:
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s
// (swiftLLM, paged attention v2 / Flash-Decoding).  The group's partials sit
// in consecutive slots.  Warp w takes splits w, w+8, ... in batches of four
// with their loads in flight together.  It keeps a running (max, sum,
// rescaled accumulator) like the online softmax.  The 8 warp states then
// merge in shared memory in warp order.  The order is fixed, so the result
// is deterministic.  The plan (groups) is read before the wait on the split
// kernel; after it, one round of loads brings every partial a warp needs.
constexpr int kCombineWarps = 8;

template <typename T, int D>
__global__ void __launch_bounds__(kCombineWarps * 32) combine_kernel(const CombineParams p) {
  constexpr int DPL = D / 32;
  __shared__ float sm_m[kCombineWarps], sm_z[kCombineWarps];
  __shared__ float sm_acc[kCombineWarps][D];
  __shared__ int sm_missing;

  const int G = p.group_size;
  const int gi = blockIdx.x / G;
  const int j = blockIdx.x % G;
  const int4 hdr = *reinterpret_cast<const int4*>(p.ws_header);
  const int4 grp = gi < p.num_groups ? p.groups[gi] : make_int4(0, 0, 0, 0);

  // The next kernel in the stream may become resident now; it waits for this
  // grid before it touches anything this kernel reads or writes.
  pdl_launch_dependents();
  pdl_wait_primary();  // partials of the split kernel are visible after this

  if (hdr.x != (int)kMagic || hdr.y != p.num_items || hdr.z != p.num_groups ||
      hdr.w != p.num_split_items || gi >= p.num_groups) {
    if (threadIdx.x == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;
  }
  const int ns = grp.z, off = grp.w;  // {seq, kv head, splits, first slot}
  if (ns < 1 || ns > kMaxSplits || off < 0 || off + ns > p.num_split_items) {
    if (threadIdx.x == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const float* ob = p.part_o + ((size_t)off * G + j) * D + lane * DPL;
  const float* lb = p.part_lse + (size_t)off * G + j;
  const size_t sstride = (size_t)G * D;

  if (threadIdx.x == 0) sm_missing = 0;
  __syncthreads();
  float m = -INFINITY, z = 0.f, acc[DPL];
  bool missing = false;  // a split task that gave up marked its slot NaN
#pragma unroll
  for (int d = 0; d < DPL; ++d) acc[d] = 0.f;
  for (int s0 = warp; s0 < ns; s0 += 4 * kCombineWarps) {
    float lse[4], x[4][DPL];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int s = s0 + u * kCombineWarps;
      lse[u] = -INFINITY;
#pragma unroll
      for (int d = 0; d < DPL; ++d) x[u][d] = 0.f;
      if (s < ns) {
        lse[u] = lb[(size_t)s * G];
        if constexpr (DPL == 4) {
          const float4 v = *reinterpret_cast<const float4*>(ob + (size_t)s * sstride);
          x[u][0] = v.x; x[u][1] = v.y; x[u][2] = v.z; x[u][3] = v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(ob + (size_t)s * sstride);
          x[u][0] = v.x; x[u][1] = v.y;
        }
      }
    }
#pragma unroll
    for (int u = 0; u < 4; ++u) missing |= isnan(lse[u]);
    const float mb = fmaxf(fmaxf(lse[0], lse[1]), fmaxf(lse[2], lse[3]));
    const float mn = fmaxf(m, mb);
    if (mn == -INFINITY) continue;  // every split so far is empty
    const float sc = ex2(m - mn);   // 0 while m is still -inf
    z *= sc;
#pragma unroll
    for (int d = 0; d < DPL; ++d) acc[d] *= sc;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const float e = ex2(lse[u] - mn);  // 0 for an empty or absent split
      z += e;
#pragma unroll
      for (int d = 0; d < DPL; ++d) acc[d] = fmaf(e, x[u][d], acc[d]);
    }
    m = mn;
  }
  if (lane == 0) {
    sm_m[warp] = m;
    sm_z[warp] = z;
  }
  if (missing) sm_missing = 1;
#pragma unroll
  for (int d = 0; d < DPL; ++d) sm_acc[warp][lane * DPL + d] = acc[d];
  __syncthreads();
  if (sm_missing) return;  // a split gave up: the group's output stays unwritten
  if (threadIdx.x < D) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kCombineWarps; ++w) M = fmaxf(M, sm_m[w]);
    float Z = 0.f, O = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kCombineWarps; ++w) {
        const float sc = ex2(sm_m[w] - M);
        Z = fmaf(sm_z[w], sc, Z);
        O = fmaf(sm_acc[w][threadIdx.x], sc, O);
      }
    }
    const float r = Z > 0.f ? O / Z : 0.f;
    static_cast<T*>(p.out)[((size_t)grp.x * p.num_q_heads + (size_t)grp.y * G + j) * D +
                           threadIdx.x] = Elem<T>::from_f(r);
  }
}

// ---------------------------------------------------------------------------
// Append: k_new[b][h] -> k_pages[block_table[b][(L-1)/S]][h][(L-1)%S], same
// for V; one thread per 16-byte chunk.
__global__ void append_kernel(const AppendParams p) {
  const int chunks = p.head_dim / 8;
  const long long total = (long long)p.batch * p.num_kv_heads * chunks;
  const int Lmax = p.max_pages * kPageSize;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ch = (int)(i % chunks);
    const int h = (int)((i / chunks) % p.num_kv_heads);
    const int b = (int)(i / chunks / p.num_kv_heads);
    const int L = p.seq_lens[b];
    if (L < 0 || L > Lmax) {
      if (ch == 0 && h == 0) set_status(p.status, PA_DEV_BAD_SEQ_LEN);
      continue;
    }
    if (L == 0) continue;
    const int pos = L - 1;
    const int page = p.block_table[(size_t)b * p.max_pages + pos / kPageSize];
    if (page < 0 || page >= p.num_pages) {
      if (ch == 0 && h == 0) set_status(p.status, PA_DEV_BAD_PAGE);
      continue;
    }
    const size_t dst =
        (((size_t)page * p.num_kv_heads + h) * kPageSize + pos % kPageSize) * p.head_dim + ch * 8;
    const size_t src = ((size_t)b * p.num_kv_heads + h) * p.head_dim + ch * 8;
    *reinterpret_cast<uint4*>(p.k_pages + dst) = *reinterpret_cast<const uint4*>(p.k_new + src);
    *reinterpret_cast<uint4*>(p.v_pages + dst) = *reinterpret_cast<const uint4*>(p.v_new + src);
  }
}

// ---------------------------------------------------------------------------
// Append into an 8-bit cache: one warp per (sequence, KV head) quantises the
// new K and V rows (per-row INT8 or E4M3, quant_common.cuh) and writes their
// codes and scales at position L-1.
constexpr int kAppendWarps = 8;

template <int D, int FMT>
__global__ void __launch_bounds__(kAppendWarps * 32) append_q8_kernel(const AppendQ8Params p) {
  constexpr int PER = D / 32;
  const int lane = threadIdx.x & 31;
  const long long total = (long long)p.batch * p.num_kv_heads;
  const int Lmax = p.max_pages * kPageSize;
  for (long long r = (long long)blockIdx.x * kAppendWarps + (threadIdx.x >> 5); r < total;
       r += (long long)gridDim.x * kAppendWarps) {
    const int h = (int)(r % p.num_kv_heads);
    const int b = (int)(r / p.num_kv_heads);
    const int L = p.seq_lens[b];
    if (L < 0 || L > Lmax) {
      if (h == 0 && lane == 0) set_status(p.status, PA_DEV_BAD_SEQ_LEN);
      continue;
    }
    if (L == 0) continue;
    const int pos = L - 1;
    const int page = p.block_table[(size_t)b * p.max_pages + pos / kPageSize];
    if (page < 0 || page >= p.num_pages) {
      if (h == 0 && lane == 0) set_status(p.status, PA_DEV_BAD_PAGE);
      continue;
    }
    const size_t row = ((size_t)page * p.num_kv_heads + h) * kPageSize + pos % kPageSize;
    const size_t src = ((size_t)b * p.num_kv_heads + h) * D;
    float sk, sv;
    const uint32_t ck = quantize_row_warp<D, FMT>(p.k_new + src, lane, sk);
    const uint32_t cv = quantize_row_warp<D, FMT>(p.v_new + src, lane, sv);
    if constexpr (PER == 4) {
      reinterpret_cast<uint32_t*>(p.k_codes + row * D)[lane] = ck;
      reinterpret_cast<uint32_t*>(p.v_codes + row * D)[lane] = cv;
    } else {
      reinterpret_cast<uint16_t*>(p.k_codes + row * D)[lane] = (uint16_t)ck;
      reinterpret_cast<uint16_t*>(p.v_codes + row * D)[lane] = (uint16_t)cv;
    }
    if (lane == 0) {
      p.k_scales[row] = sk;
      p.v_scales[row] = sv;
    }
  }
}

// ---------------------------------------------------------------------------
// Block copy (KV swap in/out, copy within a pool): CTA i takes pairs i, i +
// grid, ...; its threads move a block in 16-byte words, four loads in flight
// per thread before the four stores.  Either side may be mapped host memory.
constexpr int kCopyThreads = 256;

__global__ void __launch_bounds__(kCopyThreads) copy_blocks_kernel(const CopyBlocksParams p) {
  const int64_t words = p.block_bytes / 16;
  for (int i = blockIdx.x; i < p.n; i += gridDim.x) {
    const int2 pr = p.pairs[i];
    if (pr.x < 0 || pr.x >= p.src_blocks || pr.y < 0 || pr.y >= p.dst_blocks) {
      if (threadIdx.x == 0) set_status(p.status, PA_DEV_BAD_PAGE);
      continue;  // CTA-uniform
    }
    const uint4* s = reinterpret_cast<const uint4*>(static_cast<const char*>(p.src) +
                                                     (size_t)pr.x * (size_t)p.block_bytes);
    uint4* d = reinterpret_cast<uint4*>(static_cast<char*>(p.dst) +
                                        (size_t)pr.y * (size_t)p.block_bytes);
    int64_t w = threadIdx.x;
    for (; w + 3 * kCopyThreads < words; w += 4 * kCopyThreads) {
      const uint4 a = s[w], b = s[w + kCopyThreads], c = s[w + 2 * kCopyThreads],
                  e = s[w + 3 * kCopyThreads];
      d[w] = a;
      d[w + kCopyThreads] = b;
      d[w + 2 * kCopyThreads] = c;
      d[w + 3 * kCopyThreads] = e;
    }
    for (; w < words; w += kCopyThreads) d[w] = s[w];
  }
}

// ---------------------------------------------------------------------------
// Append of several rows per sequence (multi-token step): one thread per
// 16-byte chunk of a (row, KV head); a row finds its sequence by binary
// search in cu.
__global__ void append_tokens_kernel(const AppendTokensParams p) {
  const int chunks = p.head_dim / 8;
  const long long total = (long long)p.total_q * p.num_kv_heads * chunks;
  const int Lmax = p.max_pages * kPageSize;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int ch = (int)(i % chunks);
    const int h = (int)((i / chunks) % p.num_kv_heads);
    const int r = (int)(i / chunks / p.num_kv_heads);
    int lo = 0, hi = p.batch;  // largest b with cu[b] <= r
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (p.cu[mid] <= r) lo = mid; else hi = mid;
    }
    const int b = lo, n = p.cu[b + 1] - p.cu[b];
    const int L = p.seq_lens[b];
    if (L < n || L > Lmax) {
      if (ch == 0 && h == 0) set_status(p.status, L > Lmax ? PA_DEV_BAD_SEQ_LEN : PA_DEV_PLAN_MISMATCH);
      continue;
    }
    const int pos = L - n + (r - p.cu[b]);
    const int page = p.block_table[(size_t)b * p.max_pages + pos / kPageSize];
    if (page < 0 || page >= p.num_pages) {
      if (ch == 0 && h == 0) set_status(p.status, PA_DEV_BAD_PAGE);
      continue;
    }
    const size_t dst =
        (((size_t)page * p.num_kv_heads + h) * kPageSize + pos % kPageSize) * p.head_dim + ch * 8;
    const size_t src = ((size_t)r * p.num_kv_heads + h) * p.head_dim + ch * 8;
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.k_pages) + dst) =
        *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.k_new) + src);
    *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.v_pages) + dst) =
        *reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.v_new) + src);
  }
}

// ---------------------------------------------------------------------------
// Debug export of the gather map: slot = page * S + t % S, -1 past the end,
// -2 for an invalid page index.
__global__ void gather_slots_kernel(const int32_t* block_table, const int32_t* seq_lens,
                                    int32_t* out, int32_t* status, int batch, int max_pages,
                                    int num_pages) {
  const long long width = (long long)max_pages * kPageSize;
  const long long total = width * batch;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int b = (int)(i / width);
    const int t = (int)(i % width);
    int L = seq_lens[b];
    if (L < 0 || L > width) {
      if (t == 0) set_status(status, PA_DEV_BAD_SEQ_LEN);
      L = L < 0 ? 0 : (int)width;
    }
    int v = -1;
    if (t < L) {
      const int page = block_table[(size_t)b * max_pages + t / kPageSize];
      if (page < 0 || page >= num_pages) {
        set_status(status, PA_DEV_BAD_PAGE);
        v = -2;
      } else {
        v = page * kPageSize + t % kPageSize;
      }
    }
    out[i] = v;
  }
}

// ---------------------------------------------------------------------------
// Launchers

static int grid_for(long long work, int threads) {
  long long g = (work + threads - 1) / threads;
  if (g < 1) g = 1;
  if (g > 152 * 16) g = 152 * 16;
  return (int)g;
}

cudaError_t launch_combine(const CombineParams& p, int head_dim, int dtype, int grid,
                           cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kCombineWarps * 32);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == PA_DTYPE_BF16) {
    if (head_dim == 64) return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 64>, p);
    return cudaLaunchKernelEx(&cfg, combine_kernel<__nv_bfloat16, 128>, p);
  }
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, combine_kernel<__half, 64>, p);
  return cudaLaunchKernelEx(&cfg, combine_kernel<__half, 128>, p);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const long long work = (long long)p.batch * p.num_kv_heads * (p.head_dim / 8);
  append_kernel<<<grid_for(work, 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append_q8(const AppendQ8Params& p, cudaStream_t stream) {
  const long long rows = (long long)p.batch * p.num_kv_heads;
  long long g = (rows + kAppendWarps - 1) / kAppendWarps;
  const int grid = (int)(g < 1 ? 1 : g > 152 * 16 ? 152 * 16 : g);
  if (p.fmt == kCodeE4m3) {
    if (p.head_dim == 64)
      append_q8_kernel<64, kCodeE4m3><<<grid, kAppendWarps * 32, 0, stream>>>(p);
    else
      append_q8_kernel<128, kCodeE4m3><<<grid, kAppendWarps * 32, 0, stream>>>(p);
  } else {
    if (p.head_dim == 64)
      append_q8_kernel<64, kCodeInt8><<<grid, kAppendWarps * 32, 0, stream>>>(p);
    else
      append_q8_kernel<128, kCodeInt8><<<grid, kAppendWarps * 32, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_copy_blocks(const CopyBlocksParams& p, cudaStream_t stream) {
  const int grid = p.n < 152 * 8 ? p.n : 152 * 8;
  copy_blocks_kernel<<<grid, kCopyThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_append_tokens(const AppendTokensParams& p, cudaStream_t stream) {
  const long long work = (long long)p.total_q * p.num_kv_heads * (p.head_dim / 8);
  append_tokens_kernel<<<grid_for(work, 256), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gather(const int32_t* block_table, const int32_t* seq_lens, int32_t* out,
                          int32_t* status, int batch, int max_pages, int num_pages,
                          cudaStream_t stream) {
  const long long work = (long long)batch * max_pages * kPageSize;
  gather_slots_kernel<<<grid_for(work, 256), 256, 0, stream>>>(block_table, seq_lens, out, status,
                                                                batch, max_pages, num_pages);
  return cudaGetLastError();
}

}  // namespace pa
