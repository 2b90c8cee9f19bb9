// Combine (log-sum-exp merge of split partials), KV append and the debug
// gather-index export.
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "device_common.cuh"
#include "launch.h"

namespace pa {

// ---------------------------------------------------------------------------
// Combine: one CTA per (sequence, KV head, query head in the group) whose
// sequence was split.  With partials (o_s, lse_s) in base 2:
//   M = max_s lse_s,  w_s = 2^(lse_s - M),  out = sum_s w_s o_s / sum_s w_s
// (swiftLLM, paged attention v2 / Flash-Decoding).  One thread per output
// dim; the split weights sit in shared memory.  Summation order is the split
// order, so the result is deterministic.
template <int D>
__global__ void __launch_bounds__(D) combine_kernel(const CombineParams p) {
  __shared__ float w[kMaxSplits];
  __shared__ int ix[kMaxSplits];
  __shared__ float red[D / 32];
  __shared__ float bcast;

  pdl_wait_primary();  // partials of the split kernel are visible after this

  const int4 hdr = *reinterpret_cast<const int4*>(p.ws_header);
  if (hdr.x != (int)kMagic || hdr.y != p.num_items || hdr.z != p.num_groups ||
      hdr.w != p.num_split_items) {
    if (threadIdx.x == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;
  }
  const int gi = blockIdx.x / p.group_size;
  const int j = blockIdx.x % p.group_size;
  const int4 grp = p.groups[gi];  // {seq, kv_head, nsplit, index offset}
  const int ns = grp.z;
  if (ns < 1 || ns > kMaxSplits) {
    if (threadIdx.x == 0) set_status(p.status, PA_DEV_PLAN_MISMATCH);
    return;
  }
  const int tid = threadIdx.x;
  const int G = p.group_size;

  float mx = -INFINITY;
  for (int s = tid; s < ns; s += D) {
    const int it = p.idx[grp.w + s];
    ix[s] = it;
    const float v = p.part_lse[(size_t)it * G + j];
    w[s] = v;
    mx = fmaxf(mx, v);
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, m));
  if ((tid & 31) == 0) red[tid >> 5] = mx;
  __syncthreads();
  if (tid == 0) {
    float a = red[0];
    for (int k = 1; k < D / 32; ++k) a = fmaxf(a, red[k]);
    bcast = a;
  }
  __syncthreads();
  mx = bcast;

  float z = 0.f;
  for (int s = tid; s < ns; s += D) {
    const float e = (mx == -INFINITY) ? 0.f : ex2(w[s] - mx);
    w[s] = e;
    z += e;
  }
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) z += __shfl_xor_sync(kFull, z, m);
  __syncthreads();  // all reads of bcast done
  if ((tid & 31) == 0) red[tid >> 5] = z;
  __syncthreads();
  if (tid == 0) {
    float a = 0.f;
    for (int k = 0; k < D / 32; ++k) a += red[k];
    bcast = a;
  }
  __syncthreads();
  z = bcast;

  float a = 0.f;
  for (int s = 0; s < ns; ++s) a = fmaf(w[s], p.part_o[((size_t)ix[s] * G + j) * D + tid], a);
  const float r = z > 0.f ? a / z : 0.f;
  p.out[((size_t)grp.x * p.num_q_heads + (size_t)grp.y * G + j) * D + tid] = __float2half_rn(r);
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

cudaError_t launch_combine(const CombineParams& p, int head_dim, int grid, cudaStream_t stream) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(head_dim);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (head_dim == 64) return cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
  return cudaLaunchKernelEx(&cfg, combine_kernel<128>, p);
}

cudaError_t launch_append(const AppendParams& p, cudaStream_t stream) {
  const long long work = (long long)p.batch * p.num_kv_heads * (p.head_dim / 8);
  append_kernel<<<grid_for(work, 256), 256, 0, stream>>>(p);
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
