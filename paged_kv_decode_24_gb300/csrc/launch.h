// Kernel parameter blocks and launchers (host <-> device glue, internal).
// Append and combine work for both 16-bit element types: the append copies
// rows bit for bit, and the combine's output type is chosen at launch.
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "pa_internal.h"

namespace pa {

struct SplitParams;  // decode_kernel.cuh

struct CombineParams {
  const int32_t* ws_header;
  const int4* groups;
  const float* part_lse;
  const float* part_o;
  void* out;  // fp16 or bf16, as the launch's dtype
  int32_t* status;
  int32_t group_size;
  int32_t num_q_heads;
  int32_t num_items, num_groups, num_split_items;  // must match the workspace header
};

struct AppendParams {
  const __half* k_new;
  const __half* v_new;
  __half* k_pages;
  __half* v_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t* status;
  int32_t batch, num_kv_heads, head_dim, max_pages, num_pages;
};

// Append into an 8-bit cache: INT8 codes or E4M3 bytes (fmt: kCodeInt8 or
// kCodeE4m3, quant_common.cuh), with their per-row fp32 scales.
struct AppendQ8Params {
  const __half* k_new;
  const __half* v_new;
  int8_t* k_codes;
  int8_t* v_codes;
  float* k_scales;
  float* v_scales;
  const int32_t* block_table;
  const int32_t* seq_lens;
  int32_t* status;
  int32_t batch, num_kv_heads, head_dim, max_pages, num_pages;
  int32_t fmt;
};

struct CopyBlocksParams {
  void* dst;
  const void* src;
  const int2* pairs;  // (src block, dst block)
  int64_t block_bytes;
  int32_t n, src_blocks, dst_blocks;
  int32_t* status;
};

cudaError_t launch_copy_blocks(const CopyBlocksParams& p, cudaStream_t stream);

// Append of several rows per sequence: row cu[b] + i goes to position
// seq_lens[b] - (cu[b+1] - cu[b]) + i.  Rows are 16-bit elements, copied
// bit for bit.
struct AppendTokensParams {
  const void* k_new;
  const void* v_new;
  void* k_pages;
  void* v_pages;
  const int32_t* block_table;
  const int32_t* seq_lens;
  const int32_t* cu;  // [B+1], in the uploaded multi-token plan
  int32_t* status;
  int32_t batch, total_q, num_kv_heads, head_dim, max_pages, num_pages;
};

cudaError_t launch_append_tokens(const AppendTokensParams& p, cudaStream_t stream);

struct PrefillParams;  // prefill.cuh
cudaError_t launch_prefill_d64(const PrefillParams& p, int group, int dtype, cudaStream_t stream);
cudaError_t launch_prefill_d128(const PrefillParams& p, int group, int dtype, cudaStream_t stream);
cudaError_t launch_prefill_tc5_d64(const PrefillParams& p, int group, int dtype,
                                   cudaStream_t stream);
cudaError_t launch_prefill_tc5_d128(const PrefillParams& p, int group, int dtype,
                                    cudaStream_t stream);
cudaError_t launch_split(const SplitParams& p, int head_dim, int group, int dtype, int grid,
                         cudaStream_t stream);
cudaError_t launch_split_q8(const SplitParams& p, int head_dim, int group, int fmt, int stages,
                            int grid, cudaStream_t stream);
cudaError_t launch_append_q8(const AppendQ8Params& p, cudaStream_t stream);
cudaError_t launch_combine(const CombineParams& p, int head_dim, int dtype, int grid,
                           cudaStream_t stream);
cudaError_t launch_append(const AppendParams& p, cudaStream_t stream);
cudaError_t launch_gather(const int32_t* block_table, const int32_t* seq_lens, int32_t* out,
                          int32_t* status, int batch, int max_pages, int num_pages,
                          cudaStream_t stream);

}  // namespace pa
