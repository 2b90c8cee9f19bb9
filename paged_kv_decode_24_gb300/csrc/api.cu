// C-ABI entry points of libpagedattn: argument checks, then launches.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#include <atomic>
#include <mutex>

#include "decode_kernel.cuh"
#include "launch.h"
#include "pa_internal.h"
#include "prefill.cuh"
#include "prefill_tc5.cuh"

namespace pa {

cudaError_t launch_split_d64(const SplitParams& p, int group, int dtype, int grid,
                             cudaStream_t stream);
cudaError_t launch_split_d128(const SplitParams& p, int group, int dtype, int grid,
                              cudaStream_t stream);
cudaError_t launch_split_tc_d64(const SplitParams& p, int group, int dtype, int grid,
                                cudaStream_t stream);
cudaError_t launch_split_tc_d128(const SplitParams& p, int group, int dtype, int grid,
                                 cudaStream_t stream);
cudaError_t launch_split_q8_d64(const SplitParams& p, int group, int grid, cudaStream_t stream);
cudaError_t launch_split_q8_d128(const SplitParams& p, int group, int stages, int grid,
                                 cudaStream_t stream);
cudaError_t launch_split_f8_d64(const SplitParams& p, int group, int grid, cudaStream_t stream);
cudaError_t launch_split_f8_d128(const SplitParams& p, int group, int stages, int grid,
                                 cudaStream_t stream);

// MHA (G = 1) does one multiply-add per K or V element: the CUDA-core kernel
// keeps up with HBM.  With G >= 2 query heads per KV head the CUDA-core kernel
// becomes issue-bound (about 900 instructions per page at G = 4), so those
// groups go to the tensor-core kernel.
cudaError_t launch_split(const SplitParams& p, int head_dim, int group, int dtype, int grid,
                         cudaStream_t stream) {
  if (group == 1) {
    if (head_dim == 64) return launch_split_d64(p, group, dtype, grid, stream);
    if (head_dim == 128) return launch_split_d128(p, group, dtype, grid, stream);
  } else {
    if (head_dim == 64) return launch_split_tc_d64(p, group, dtype, grid, stream);
    if (head_dim == 128) return launch_split_tc_d128(p, group, dtype, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// The 8-bit caches (INT8 codes or E4M3 bytes) have one kernel for every group
// size: its products run on tensor cores, which the padding of G = 1 to 8
// heads does not slow down.  At head_dim 128 the plan picks 2 or 3 page
// stages per warp (pa_plan_t.q8_stages).
cudaError_t launch_split_q8(const SplitParams& p, int head_dim, int group, int fmt, int stages,
                            int grid, cudaStream_t stream) {
  if (fmt == kCodeE4m3) {
    if (head_dim == 64) return launch_split_f8_d64(p, group, grid, stream);
    if (head_dim == 128) return launch_split_f8_d128(p, group, stages, grid, stream);
  } else {
    if (head_dim == 64) return launch_split_q8_d64(p, group, grid, stream);
    if (head_dim == 128) return launch_split_q8_d128(p, group, stages, grid, stream);
  }
  return cudaErrorInvalidValue;
}

// cuTensorMapEncodeTiled, reached through the runtime's driver entry point.
static PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      (void)cudaGetLastError();
  });
  return fn;
}

// A pool [P][Hkv][16][D] of 16-bit elements as a 4-D tensor, innermost
// first, with boxes of 64 elements x 16 rows and the 128-byte swizzle.
static bool encode_pool_map(CUtensorMap* map, const void* pool, const pa_shape_t& s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t D = (cuuint64_t)s.head_dim;
  cuuint64_t dims[4] = {D, (cuuint64_t)kPageSize, (cuuint64_t)s.num_kv_heads,
                        (cuuint64_t)s.num_pages};
  cuuint64_t strides[3] = {D * 2, D * 2 * kPageSize, D * 2 * kPageSize * s.num_kv_heads};
  cuuint32_t box[4] = {64, (cuuint32_t)kPageSize, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapDataType ty = s.dtype == PA_DTYPE_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return enc(map, ty, 4, const_cast<void*>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// An 8-bit code pool (INT8 or E4M3) [P][Hkv][16][D] as a 4-D tensor with one box per
// (page, head) tile: D bytes x 16 rows, 128-byte swizzle for D = 128 and
// 64-byte swizzle for D = 64 (a row is never wider than its swizzle span).
static bool encode_code_map(CUtensorMap* map, const void* pool, const pa_shape_t& s) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t D = (cuuint64_t)s.head_dim;
  cuuint64_t dims[4] = {D, (cuuint64_t)kPageSize, (cuuint64_t)s.num_kv_heads,
                        (cuuint64_t)s.num_pages};
  cuuint64_t strides[3] = {D, D * kPageSize, D * kPageSize * s.num_kv_heads};
  cuuint32_t box[4] = {(cuuint32_t)D, (cuuint32_t)kPageSize, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  const CUtensorMapSwizzle sw = D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 4, const_cast<void*>(pool), dims, strides, box,
             estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

bool aligned(const void* p, uintptr_t a) { return p && ((uintptr_t)p % a) == 0; }

bool same_plan_shape(const pa_shape_t& a, const pa_shape_t& b) {
  return a.batch == b.batch && a.num_q_heads == b.num_q_heads && a.num_kv_heads == b.num_kv_heads &&
         a.head_dim == b.head_dim && a.page_size == b.page_size &&
         a.max_pages_per_seq == b.max_pages_per_seq;
}

pa_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return PA_OK;
  (void)cudaGetLastError();  // clear a sticky launch error so later calls report their own
  return PA_ERR_CUDA;
}

// CTAs in the split kernel's first wave on the current device: its SMs (read
// once per device) times the CTAs one SM holds (the planner's estimate).
int first_wave_ctas(int head_dim, int group) {
  static std::atomic<int> sms[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  int n = sms[dev & 63].load(std::memory_order_relaxed);
  if (n <= 0) {
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
      (void)cudaGetLastError();
      return 0;
    }
    sms[dev & 63].store(n, std::memory_order_relaxed);
  }
  return n * resident_ctas_per_sm(head_dim, group);
}

}  // namespace
}  // namespace pa

extern "C" const char* pa_status_string(pa_status_t status) {
  switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED:
      return "unsupported shape (head_dim 64/128, page_size 16, Hq/Hkv in 1,2,4,8, "
             "dtype f16/bf16; 8-bit caches f16 only)";
    case PA_ERR_WORKSPACE: return "workspace smaller than the plan requires";
    case PA_ERR_CUDA: return "CUDA runtime error";
    case PA_ERR_DEVICE_OOB: return "device detected an out-of-range index";
    case PA_ERR_TIMEOUT: return "device wait timed out";
    case PA_ERR_NO_MEMORY: return "host allocation failed";
    case PA_ERR_PLAN: return "plan does not match the shape";
  }
  return "unknown status";
}

extern "C" const char* pa_version(void) { return "libpagedattn 0.1 (sm_103a)"; }

extern "C" pa_status_t pa_kv_append(const pa_shape_t* shape, const void* k_new, const void* v_new,
                                    void* k_pages, void* v_pages, const int32_t* block_table,
                                    const int32_t* seq_lens, int32_t* dev_status, void* stream) {
  using namespace pa;
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  if (shape->batch == 0) return PA_OK;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pages, 16) ||
      !aligned(v_pages, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(dev_status, 4))
    return PA_ERR_INVALID_ARG;
  AppendParams p{};
  p.k_new = (const __half*)k_new;
  p.v_new = (const __half*)v_new;
  p.k_pages = (__half*)k_pages;
  p.v_pages = (__half*)v_pages;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.status = dev_status;
  p.batch = shape->batch;
  p.num_kv_heads = shape->num_kv_heads;
  p.head_dim = shape->head_dim;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pages = shape->num_pages;
  return cuda_status(launch_append(p, (cudaStream_t)stream));
}

namespace pa {
namespace {

// pa_kv_append_q8 and pa_kv_append_fp8: the same checks and launch, codes of
// format fmt.
pa_status_t append8_impl(const pa_shape_t* shape, const void* k_new, const void* v_new,
                         void* k_codes, void* v_codes, float* k_scales, float* v_scales,
                         const int32_t* block_table, const int32_t* seq_lens,
                         int32_t* dev_status, void* stream, int fmt) {
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  if (shape->dtype != PA_DTYPE_F16) return PA_ERR_UNSUPPORTED;
  if (shape->batch == 0) return PA_OK;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_codes, 16) ||
      !aligned(v_codes, 16) || !aligned(k_scales, 16) || !aligned(v_scales, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(dev_status, 4))
    return PA_ERR_INVALID_ARG;
  AppendQ8Params p{};
  p.k_new = (const __half*)k_new;
  p.v_new = (const __half*)v_new;
  p.k_codes = (int8_t*)k_codes;
  p.v_codes = (int8_t*)v_codes;
  p.k_scales = k_scales;
  p.v_scales = v_scales;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.status = dev_status;
  p.batch = shape->batch;
  p.num_kv_heads = shape->num_kv_heads;
  p.head_dim = shape->head_dim;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pages = shape->num_pages;
  p.fmt = fmt;
  return cuda_status(launch_append_q8(p, (cudaStream_t)stream));
}

}  // namespace
}  // namespace pa

extern "C" pa_status_t pa_kv_append_q8(const pa_shape_t* shape, const void* k_new,
                                       const void* v_new, void* k_codes, void* v_codes,
                                       float* k_scales, float* v_scales,
                                       const int32_t* block_table, const int32_t* seq_lens,
                                       int32_t* dev_status, void* stream) {
  return pa::append8_impl(shape, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table,
                          seq_lens, dev_status, stream, pa::kCodeInt8);
}

extern "C" pa_status_t pa_kv_append_fp8(const pa_shape_t* shape, const void* k_new,
                                        const void* v_new, void* k_codes, void* v_codes,
                                        float* k_scales, float* v_scales,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int32_t* dev_status, void* stream) {
  return pa::append8_impl(shape, k_new, v_new, k_codes, v_codes, k_scales, v_scales, block_table,
                          seq_lens, dev_status, stream, pa::kCodeE4m3);
}

extern "C" pa_status_t pa_plan_upload(const pa_plan_t* plan, void* workspace,
                                      size_t workspace_bytes, void* stream) {
  if (!plan || !plan->host_blob || plan->blob_bytes == 0) return PA_ERR_INVALID_ARG;
  if (!pa::aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return PA_ERR_WORKSPACE;
  return pa::cuda_status(cudaMemcpyAsync(workspace, plan->host_blob, plan->blob_bytes,
                                         cudaMemcpyHostToDevice, (cudaStream_t)stream));
}

namespace pa {
namespace {

// The cache a decode reads: 16-bit pools, or 8-bit code pools (INT8 codes or
// E4M3 bytes, fmt) with their row scales (scales non-null).
struct KvCache {
  const void* k;
  const void* v;
  const float* k_scales;
  const float* v_scales;
  int fmt;
  bool int8() const { return k_scales != nullptr; }
};

pa_status_t decode_impl(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                        const void* k_new, const void* v_new, const KvCache& kv,
                        const int32_t* block_table, const int32_t* seq_lens, float scale,
                        void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream);

}  // namespace
}  // namespace pa

namespace pa {

pa_status_t check_decode_call(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                              const void* k_pages, const void* v_pages,
                              const int32_t* block_table, const int32_t* seq_lens, float scale,
                              const void* out, const void* workspace, size_t workspace_bytes,
                              const int32_t* dev_status, bool* launches) {
  *launches = false;
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  if (!plan) return PA_ERR_INVALID_ARG;
  if (!same_plan_shape(plan->shape, *shape)) return PA_ERR_PLAN;
  if (shape->batch == 0) return PA_OK;
  if (plan->num_work_items <= 0 || plan->num_ctas <= 0 || plan->num_shared_ctas < 0 ||
      plan->num_shared_ctas > plan->num_ctas || plan->l2_prefetch_pages > 32 ||
      (plan->merge != PA_MERGE_IN_SPLIT_KERNEL && plan->merge != PA_MERGE_COMBINE_KERNEL) ||
      (plan->q8_stages != 2 && plan->q8_stages != 3) || (plan->early_kv != 0 && plan->early_kv != 1))
    return PA_ERR_PLAN;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(dev_status, 4) ||
      !aligned(workspace, 256))
    return PA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return PA_ERR_WORKSPACE;
  *launches = true;
  return PA_OK;
}

}  // namespace pa

extern "C" pa_status_t pa_decode_attention(const pa_shape_t* shape, const pa_plan_t* plan,
                                           const void* q, const void* k_pages, const void* v_pages,
                                           const int32_t* block_table, const int32_t* seq_lens,
                                           float scale, void* out, void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           void* stream) {
  const pa::KvCache kv{k_pages, v_pages, nullptr, nullptr, -1};
  return pa::decode_impl(shape, plan, q, nullptr, nullptr, kv, block_table, seq_lens, scale, out,
                         workspace, workspace_bytes, dev_status, stream);
}

extern "C" pa_status_t pa_append_decode_attention(
    const pa_shape_t* shape, const pa_plan_t* plan, const void* q, const void* k_new,
    const void* v_new, void* k_pages, void* v_pages, const int32_t* block_table,
    const int32_t* seq_lens, float scale, void* out, void* workspace, size_t workspace_bytes,
    int32_t* dev_status, void* stream) {
  if (shape && shape->batch > 0 && (!pa::aligned(k_new, 16) || !pa::aligned(v_new, 16)))
    return PA_ERR_INVALID_ARG;
  const pa::KvCache kv{k_pages, v_pages, nullptr, nullptr, -1};
  return pa::decode_impl(shape, plan, q, k_new, v_new, kv, block_table, seq_lens, scale, out,
                         workspace, workspace_bytes, dev_status, stream);
}

namespace pa {
namespace {

// The decode calls of the 8-bit caches: scales must be 16-byte aligned.
pa_status_t decode8(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                    const void* k_new, const void* v_new, const void* k_codes,
                    const void* v_codes, const float* k_scales, const float* v_scales,
                    const int32_t* block_table, const int32_t* seq_lens, float scale, void* out,
                    void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream,
                    int fmt) {
  if (shape && shape->batch > 0 &&
      (!aligned(k_scales, 16) || !aligned(v_scales, 16) ||
       (k_new != nullptr && (!aligned(k_new, 16) || !aligned(v_new, 16)))))
    return PA_ERR_INVALID_ARG;
  const KvCache kv{k_codes, v_codes, k_scales, v_scales, fmt};
  return decode_impl(shape, plan, q, k_new, v_new, kv, block_table, seq_lens, scale, out,
                     workspace, workspace_bytes, dev_status, stream);
}

}  // namespace
}  // namespace pa

extern "C" pa_status_t pa_decode_attention_q8(const pa_shape_t* shape, const pa_plan_t* plan,
                                              const void* q, const void* k_codes,
                                              const void* v_codes, const float* k_scales,
                                              const float* v_scales, const int32_t* block_table,
                                              const int32_t* seq_lens, float scale, void* out,
                                              void* workspace, size_t workspace_bytes,
                                              int32_t* dev_status, void* stream) {
  return pa::decode8(shape, plan, q, nullptr, nullptr, k_codes, v_codes, k_scales, v_scales,
                     block_table, seq_lens, scale, out, workspace, workspace_bytes, dev_status,
                     stream, pa::kCodeInt8);
}

extern "C" pa_status_t pa_append_decode_attention_q8(
    const pa_shape_t* shape, const pa_plan_t* plan, const void* q, const void* k_new,
    const void* v_new, void* k_codes, void* v_codes, float* k_scales, float* v_scales,
    const int32_t* block_table, const int32_t* seq_lens, float scale, void* out, void* workspace,
    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (shape && shape->batch > 0 && (k_new == nullptr || v_new == nullptr))
    return PA_ERR_INVALID_ARG;
  return pa::decode8(shape, plan, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales,
                     block_table, seq_lens, scale, out, workspace, workspace_bytes, dev_status,
                     stream, pa::kCodeInt8);
}

extern "C" pa_status_t pa_decode_attention_fp8(const pa_shape_t* shape, const pa_plan_t* plan,
                                               const void* q, const void* k_codes,
                                               const void* v_codes, const float* k_scales,
                                               const float* v_scales, const int32_t* block_table,
                                               const int32_t* seq_lens, float scale, void* out,
                                               void* workspace, size_t workspace_bytes,
                                               int32_t* dev_status, void* stream) {
  return pa::decode8(shape, plan, q, nullptr, nullptr, k_codes, v_codes, k_scales, v_scales,
                     block_table, seq_lens, scale, out, workspace, workspace_bytes, dev_status,
                     stream, pa::kCodeE4m3);
}

extern "C" pa_status_t pa_append_decode_attention_fp8(
    const pa_shape_t* shape, const pa_plan_t* plan, const void* q, const void* k_new,
    const void* v_new, void* k_codes, void* v_codes, float* k_scales, float* v_scales,
    const int32_t* block_table, const int32_t* seq_lens, float scale, void* out, void* workspace,
    size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (shape && shape->batch > 0 && (k_new == nullptr || v_new == nullptr))
    return PA_ERR_INVALID_ARG;
  return pa::decode8(shape, plan, q, k_new, v_new, k_codes, v_codes, k_scales, v_scales,
                     block_table, seq_lens, scale, out, workspace, workspace_bytes, dev_status,
                     stream, pa::kCodeE4m3);
}

namespace pa {
namespace {

pa_status_t decode_impl(const pa_shape_t* shape, const pa_plan_t* plan, const void* q,
                        const void* k_new, const void* v_new, const KvCache& kv,
                        const int32_t* block_table, const int32_t* seq_lens, float scale,
                        void* out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                        void* stream) {
  bool launches = false;
  pa_status_t st = check_decode_call(shape, plan, q, kv.k, kv.v, block_table, seq_lens, scale, out,
                                     workspace, workspace_bytes, dev_status, &launches);
  if (st != PA_OK || !launches) return st;
  if (kv.int8() && shape->dtype != PA_DTYPE_F16) return PA_ERR_UNSUPPORTED;

  const int G = shape->num_q_heads / shape->num_kv_heads;
  const int D = shape->head_dim;
  const Layout lay = layout(plan->num_work_items, plan->num_groups, plan->num_split_items, G, D);
  char* ws = (char*)workspace;
  cudaStream_t s = (cudaStream_t)stream;

  SplitParams p{};
  p.q = q;
  if (kv.int8()) {
    p.k_codes = (const int8_t*)kv.k;
    p.v_codes = (const int8_t*)kv.v;
    p.k_scales = kv.k_scales;
    p.v_scales = kv.v_scales;
  } else {
    p.k_pages = kv.k;
    p.v_pages = kv.v;
  }
  p.k_new = k_new;
  p.v_new = v_new;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.out = out;
  p.ws_header = (const int32_t*)ws;
  p.items = (const int4*)(ws + lay.items_off);
  p.item_slots = (const int2*)(ws + lay.slots_off);
  p.groups = (const int4*)(ws + lay.groups_off);
  p.counters = (int*)(ws + lay.counters_off);
  p.part_lse = (float*)(ws + lay.lse_off);
  p.part_o = (float*)(ws + lay.o_off);
  p.status = dev_status;
  p.qscale = (float)((double)scale * 1.4426950408889634);  // log2(e)
  p.batch = shape->batch;
  p.num_q_heads = shape->num_q_heads;
  p.num_kv_heads = shape->num_kv_heads;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pages = shape->num_pages;
  p.num_items = plan->num_work_items;
  p.num_groups = plan->num_groups;
  p.num_split_items = plan->num_split_items;
  p.num_ctas = plan->num_ctas;
  p.num_shared = plan->num_shared_ctas;
  // Only the first wave's CTAs can start before the previous kernel ends, so
  // by default only they prefetch; the plan's options may say otherwise.
  p.pf_pages = plan->l2_prefetch_pages == 0 ? kL2PrefetchPages
                                            : (plan->l2_prefetch_pages < 0 ? 0 : plan->l2_prefetch_pages);
  p.pf_ctas = plan->l2_prefetch_ctas == 0 ? first_wave_ctas(D, G)
                                          : (plan->l2_prefetch_ctas < 0 ? 0 : plan->l2_prefetch_ctas);
  // Split groups are merged by their last split task inside the split kernel,
  // or, for a plan made with PA_MERGE_COMBINE_KERNEL, by a separate combine
  // kernel launched after the split kernel.
  p.fuse_merge = plan->merge == PA_MERGE_COMBINE_KERNEL ? 0 : 1;
  p.wait_ns = wait_limit_or_default(plan->wait_limit_ns);
  p.early_kv = plan->early_kv;
  if (kv.int8()) {
    if (!encode_code_map(&p.tmap_k, kv.k, *shape) || !encode_code_map(&p.tmap_v, kv.v, *shape))
      return PA_ERR_CUDA;
    st = cuda_status(launch_split_q8(p, D, G, kv.fmt, plan->q8_stages, plan->num_ctas, s));
  } else {
    if (!encode_pool_map(&p.tmap_k, kv.k, *shape) || !encode_pool_map(&p.tmap_v, kv.v, *shape))
      return PA_ERR_CUDA;
    st = cuda_status(launch_split(p, D, G, shape->dtype, plan->num_ctas, s));
  }
  if (st != PA_OK || p.fuse_merge || plan->num_groups == 0) return st;

  CombineParams c{};
  c.ws_header = (const int32_t*)ws;
  c.groups = (const int4*)(ws + lay.groups_off);
  c.part_lse = p.part_lse;
  c.part_o = p.part_o;
  c.out = out;
  c.status = dev_status;
  c.group_size = G;
  c.num_q_heads = shape->num_q_heads;
  c.num_items = p.num_items;
  c.num_groups = p.num_groups;
  c.num_split_items = p.num_split_items;
  return cuda_status(launch_combine(c, D, shape->dtype, plan->num_groups * G, s));
}

}  // namespace
}  // namespace pa

// ---- several query tokens per sequence

extern "C" pa_status_t pa_prefill_plan_upload(const pa_prefill_plan_t* plan, void* workspace,
                                              size_t workspace_bytes, void* stream) {
  if (!plan || !plan->host_blob || plan->blob_bytes == 0) return PA_ERR_INVALID_ARG;
  if (!pa::aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return PA_ERR_WORKSPACE;
  return pa::cuda_status(cudaMemcpyAsync(workspace, plan->host_blob, plan->blob_bytes,
                                         cudaMemcpyHostToDevice, (cudaStream_t)stream));
}

namespace pa {
namespace {

pa_status_t check_prefill_call(const pa_shape_t* shape, const pa_prefill_plan_t* plan,
                               const void* workspace, size_t workspace_bytes) {
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  if (!plan) return PA_ERR_INVALID_ARG;
  if (!same_plan_shape(plan->shape, *shape)) return PA_ERR_PLAN;
  if (plan->num_tiles < 0 || plan->total_q < 0) return PA_ERR_PLAN;
  if (plan->total_q > 0 && !aligned(workspace, 256)) return PA_ERR_INVALID_ARG;
  if (workspace_bytes < plan->workspace_bytes) return PA_ERR_WORKSPACE;
  return PA_OK;
}

}  // namespace
}  // namespace pa

extern "C" pa_status_t pa_kv_append_tokens(const pa_shape_t* shape, const pa_prefill_plan_t* plan,
                                           const void* k_new, const void* v_new, void* k_pages,
                                           void* v_pages, const int32_t* block_table,
                                           const int32_t* seq_lens, const void* workspace,
                                           size_t workspace_bytes, int32_t* dev_status,
                                           void* stream) {
  using namespace pa;
  pa_status_t st = check_prefill_call(shape, plan, workspace, workspace_bytes);
  if (st != PA_OK) return st;
  if (shape->batch == 0 || plan->total_q == 0) return PA_OK;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_pages, 16) ||
      !aligned(v_pages, 16) || !aligned(block_table, 4) || !aligned(seq_lens, 4) ||
      !aligned(dev_status, 4))
    return PA_ERR_INVALID_ARG;
  AppendTokensParams p{};
  p.k_new = k_new;
  p.v_new = v_new;
  p.k_pages = k_pages;
  p.v_pages = v_pages;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.cu = (const int32_t*)((const char*)workspace + prefill_layout(plan->num_tiles, shape->batch).cu_off);
  p.status = dev_status;
  p.batch = shape->batch;
  p.total_q = plan->total_q;
  p.num_kv_heads = shape->num_kv_heads;
  p.head_dim = shape->head_dim;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pages = shape->num_pages;
  return cuda_status(launch_append_tokens(p, (cudaStream_t)stream));
}

extern "C" pa_status_t pa_prefill_attention(const pa_shape_t* shape, const pa_prefill_plan_t* plan,
                                            const void* q, const void* k_pages,
                                            const void* v_pages, const int32_t* block_table,
                                            const int32_t* seq_lens, float scale, void* out,
                                            void* workspace, size_t workspace_bytes,
                                            int32_t* dev_status, void* stream) {
  using namespace pa;
  pa_status_t st = check_prefill_call(shape, plan, workspace, workspace_bytes);
  if (st != PA_OK) return st;
  if (shape->batch == 0 || plan->num_tiles == 0) return PA_OK;
  if (!plan->host_blob) return PA_ERR_PLAN;
  if (!aligned(q, 16) || !aligned(k_pages, 16) || !aligned(v_pages, 16) || !aligned(out, 16) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(dev_status, 4))
    return PA_ERR_INVALID_ARG;
  if (!isfinite(scale)) return PA_ERR_INVALID_ARG;
  PrefillParams p{};
  p.q = q;
  p.out = out;
  p.block_table = block_table;
  p.seq_lens = seq_lens;
  p.ws = (const int32_t*)workspace;
  p.cu = (const int32_t*)((const char*)workspace +
                          prefill_layout(plan->num_tiles, shape->batch).cu_off);
  p.status = dev_status;
  p.qscale = (float)((double)scale * 1.4426950408889634);  // log2(e)
  p.batch = shape->batch;
  p.num_q_heads = shape->num_q_heads;
  p.num_kv_heads = shape->num_kv_heads;
  p.max_pages = shape->max_pages_per_seq;
  p.num_pages = shape->num_pages;
  p.num_tiles = plan->num_tiles;
  p.total_q = plan->total_q;
  p.wait_ns = wait_limit_or_default(plan->wait_limit_ns);
  if (!encode_pool_map(&p.tmap_k, k_pages, *shape) || !encode_pool_map(&p.tmap_v, v_pages, *shape))
    return PA_ERR_CUDA;
  const int G = shape->num_q_heads / shape->num_kv_heads;
  const int rows = ((const int32_t*)plan->host_blob)[8];  // the kernel the tiles were cut for
  cudaStream_t s = (cudaStream_t)stream;
  cudaError_t e;
  if (rows == kPrefillRowsTc5)
    e = shape->head_dim == 64 ? launch_prefill_tc5_d64(p, G, shape->dtype, s)
                              : launch_prefill_tc5_d128(p, G, shape->dtype, s);
  else if (rows == kPrefillRows)
    e = shape->head_dim == 64 ? launch_prefill_d64(p, G, shape->dtype, s)
                              : launch_prefill_d128(p, G, shape->dtype, s);
  else
    return PA_ERR_PLAN;
  return cuda_status(e);
}

extern "C" pa_status_t pa_copy_blocks(void* dst_pool, int32_t dst_blocks, const void* src_pool,
                                      int32_t src_blocks, size_t block_bytes, const int32_t* pairs,
                                      int32_t n, int32_t* dev_status, void* stream) {
  using namespace pa;
  if (n < 0 || dst_blocks < 0 || src_blocks < 0) return PA_ERR_INVALID_ARG;
  if (block_bytes == 0 || block_bytes % 16 != 0) return PA_ERR_INVALID_ARG;
  if (n == 0) return PA_OK;
  if (!aligned(dst_pool, 16) || !aligned(src_pool, 16) || !aligned(pairs, 8) ||
      !aligned(dev_status, 4))
    return PA_ERR_INVALID_ARG;
  CopyBlocksParams p{};
  p.dst = dst_pool;
  p.src = src_pool;
  p.pairs = reinterpret_cast<const int2*>(pairs);
  p.block_bytes = (int64_t)block_bytes;
  p.n = n;
  p.src_blocks = src_blocks;
  p.dst_blocks = dst_blocks;
  p.status = dev_status;
  return cuda_status(launch_copy_blocks(p, (cudaStream_t)stream));
}

extern "C" pa_status_t pa_debug_gather_indices(const pa_shape_t* shape, const int32_t* block_table,
                                               const int32_t* seq_lens, int32_t* out_slots,
                                               int32_t* dev_status, void* stream) {
  using namespace pa;
  pa_status_t st = check_shape(shape);
  if (st != PA_OK) return st;
  if (shape->batch == 0) return PA_OK;
  if ((int64_t)shape->num_pages * shape->page_size > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!aligned(block_table, 4) || !aligned(seq_lens, 4) || !aligned(out_slots, 4) ||
      !aligned(dev_status, 4))
    return PA_ERR_INVALID_ARG;
  return cuda_status(launch_gather(block_table, seq_lens, out_slots, dev_status, shape->batch,
                                   shape->max_pages_per_seq, shape->num_pages,
                                   (cudaStream_t)stream));
}
