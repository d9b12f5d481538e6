// Backward without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the moment they run the
// backward: a runtime whose memory pool already owns the whole device, or a
// latency-critical loop where a cudaMalloc would synchronize the device. This
// entry point runs the same backward as tree_attn_bwd with its scratch (the
// per-row -lse*log2(e) and -Delta rows) taken from a fixed array compiled into
// the library instead of from a workspace argument. It allocates nothing.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "plan_internal.h"

namespace treeattn {
namespace {

// The scratch array. Every GPU that loads the library holds it until the
// process exits. In host code its name is only a stand-in for the device
// symbol, so kernels get the address found by cudaGetSymbolAddress below.
__device__ __align__(256) unsigned char g_static_scratch[TREE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
tree_status_t scratch_address(void** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(TREE_ERR_CUDA, std::string("cudaGetDevice: ") + cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(TREE_ERR_UNSUPPORTED, "device ordinal out of range");
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || !p)
      return fail(TREE_ERR_CUDA,
                  std::string("cudaGetSymbolAddress of the scratch array: ") + cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return TREE_OK;
}

}  // namespace
}  // namespace treeattn

using namespace treeattn;

extern "C" tree_status_t tree_attn_bwd_static_scratch(
    const tree_plan_t* plan, const void* dout, const void* q, const void* k, const void* v,
    const void* o, const float* lse, void* dq, void* dk, void* dv, int32_t hq, int32_t hkv,
    int32_t head_dim, tree_dtype_t dtype, tree_dtype_t grad_dtype, float softmax_scale,
    tree_stream_t stream) {
  if (!plan) return fail(TREE_ERR_INVALID_ARG, "NULL plan");
  const size_t need = tree_attn_bwd_workspace_bytes(plan, hq, head_dim, dtype);
  if (need > TREE_STATIC_SCRATCH_BYTES)
    return fail(TREE_ERR_UNSUPPORTED,
                "this backward needs " + std::to_string(need) +
                    " bytes of scratch; the built-in array holds " +
                    std::to_string(static_cast<size_t>(TREE_STATIC_SCRATCH_BYTES)) +
                    " (use tree_attn_bwd with a workspace)");
  void* scratch = nullptr;
  tree_status_t st = scratch_address(&scratch);
  if (st != TREE_OK) return st;
  // The kernels write every scratch entry they later read, so stale contents
  // from an earlier call need no clearing.
  return tree_attn_bwd(plan, dout, q, k, v, o, lse, dq, dk, dv, hq, hkv, head_dim, dtype,
                       grad_dtype, softmax_scale, scratch, TREE_STATIC_SCRATCH_BYTES, stream);
}
