// pa_decode_attention_static: decode attention that allocates nothing.
//
// For callers that cannot allocate device memory: code embedded in another
// runtime that hands it only its input and output buffers and owns all
// device memory itself, or a latency-critical loop where a cudaMalloc could
// stall on device synchronisation.  The split partials and the uploaded task
// list live in one file-scope __device__ array instead of a caller workspace.
// Every GPU that loads this library holds the array until the process exits.
//
// The array is shared by all calls on a device and keeps the previous call's
// contents.  Calls that overlap on the GPU (two streams, or concurrent host
// threads) race on it.  Nothing in it has to start at zero: each call
// uploads its own task list, and every partial is written before it is read.
#include <cuda_runtime.h>

#include "pa_internal.h"

namespace {

// PA_STATIC_WORKSPACE_BYTES (include/pagedattn.h) bytes of device scratch.
static __device__ __align__(256) unsigned char g_static_workspace[PA_STATIC_WORKSPACE_BYTES];

// Device address of the array on the current device.  In host code
// g_static_workspace names a host-side stand-in, not device memory, so the
// address must come from the runtime, with the device current.  It is looked
// up on every call, not cached: once the module is loaded the lookup
// allocates nothing, and a context rebuilt after cudaDeviceReset may place
// the array elsewhere.
pa_status_t static_workspace_address(void** out) {
  void* p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_static_workspace);
  if (e != cudaSuccess || p == nullptr) {
    (void)cudaGetLastError();
    return PA_ERR_CUDA;
  }
  *out = p;
  return PA_OK;
}

}  // namespace

extern "C" pa_status_t pa_decode_attention_static(const pa_shape_t* shape, const pa_plan_t* plan,
                                                  const void* q, const void* k_pages,
                                                  const void* v_pages, const int32_t* block_table,
                                                  const int32_t* seq_lens, float scale, void* out,
                                                  int32_t* dev_status, void* stream) {
  // Every check pa_decode_attention makes, in its order, before anything is
  // queued into the shared array; the array's size stands in for the
  // workspace size, so a plan too big for it is PA_ERR_WORKSPACE.
  const void* ws_check = reinterpret_cast<const void*>(uintptr_t(256));  // alignment only
  bool launches = false;
  pa_status_t st = pa::check_decode_call(shape, plan, q, k_pages, v_pages, block_table, seq_lens,
                                         scale, out, ws_check, (size_t)PA_STATIC_WORKSPACE_BYTES,
                                         dev_status, &launches);
  if (st != PA_OK || !launches) return st;
  if (!plan->host_blob || plan->blob_bytes == 0) return PA_ERR_INVALID_ARG;
  void* ws = nullptr;
  st = static_workspace_address(&ws);
  if (st != PA_OK) return st;
  st = pa_plan_upload(plan, ws, (size_t)PA_STATIC_WORKSPACE_BYTES, stream);
  if (st != PA_OK) return st;
  return pa_decode_attention(shape, plan, q, k_pages, v_pages, block_table, seq_lens, scale, out,
                             ws, (size_t)PA_STATIC_WORKSPACE_BYTES, dev_status, stream);
}
