// gdn_static_ws.cu -- gdn_mixed_batch for callers that cannot allocate device memory.
//
// Some callers have no way to obtain device scratch: a plain C host or a plugin embedded in a
// framework that owns every device allocation and exposes no allocation hook, or a serving
// loop that must never call cudaMalloc/cudaFree because those calls can synchronise the device
// and stall unrelated streams.  For them this file keeps the scratch of gdn_mixed_batch (the
// fp32 post-conv q|k|v of every token, then the chunked prefill's per-chunk records) in a fixed
// device array compiled into the library, so the call needs nothing beyond the caller's own
// inputs and outputs.
//
// Costs and rules of the fixed array:
//   - its GDN_STATIC_WORKSPACE_BYTES are reserved on every GPU that loads this part of the
//     library and stay reserved until the process exits;
//   - a batch fits when gdn_workspace_bytes() + gdn_prefill_workspace_bytes() is at most that
//     size; larger batches are refused with GDN_ERR_WORKSPACE before anything is enqueued;
//   - every call on a device shares the one array, so calls that may overlap on the GPU
//     (different streams, or different host threads without ordering) race on it;
//   - the array keeps whatever the previous call left; nothing in it needs to start at zero,
//     because every element a call reads was written earlier by that same call;
//   - in host code the array's name is only a host-side stand-in, so the device address is
//     looked up with cudaGetSymbolAddress, with the device current, on the first call made in
//     each CUDA context (in practice the device's primary context, so once per device); make
//     that first call before any stream capture.  A context that replaces an earlier one at the
//     same handle value (after cudaDeviceReset) cannot be told apart, so do not use this entry
//     point across cudaDeviceReset.
// The paper has no counterpart to this entry point.
#include <mutex>

#include "gdn_internal.cuh"

static __device__ __align__(256) unsigned char g_gdn_static_workspace[GDN_STATIC_WORKSPACE_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// The driver's cuCtxGetCurrent, reached through the runtime so the library needs no link
// against the driver library.
typedef int (*CtxGetCurrentFn)(void** ctx);

std::mutex g_mutex;
void* g_address[kMaxDevices] = {};
void* g_context[kMaxDevices] = {};
CtxGetCurrentFn g_ctx_get_current = nullptr;
bool g_ctx_fn_looked_up = false;

// The current context's handle, or NULL when it cannot be determined (then only the device
// ordinal keys the cache).  Called with g_mutex held.
void* current_context() {
  if (!g_ctx_fn_looked_up) {
    g_ctx_fn_looked_up = true;
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &fn, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_ctx_get_current = reinterpret_cast<CtxGetCurrentFn>(fn);
  }
  void* ctx = nullptr;
  if (g_ctx_get_current && g_ctx_get_current(&ctx) != 0) ctx = nullptr;
  return ctx;
}

// Device address of the array in the current device's context, or NULL.
void* static_workspace_address() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  // cudaFree(0) is not used to force context creation here: it is one of the calls this entry
  // point exists to avoid.  cudaGetSymbolAddress below creates the context if needed.
  std::lock_guard<std::mutex> lock(g_mutex);
  void* ctx = current_context();
  if (!g_address[dev] || ctx != g_context[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_gdn_static_workspace) != cudaSuccess) return nullptr;
    g_address[dev] = p;
    g_context[dev] = ctx ? ctx : current_context();
  }
  return g_address[dev];
}

}  // namespace

extern "C" int gdn_mixed_batch_static_workspace(const gdn_layer_desc* layer, const gdn_layer_params* params,
                                                const gdn_pools* pools, const void* x, const void* a, const void* b,
                                                int32_t num_actual_tokens, const gdn_rows* non_spec,
                                                int32_t num_decodes, int32_t num_prefills, const gdn_rows* spec,
                                                void* out, uint32_t* d_status, void* stream) {
  // The whole scratch gdn_mixed_batch will use: the post-conv q|k|v plus, when prefill rows take
  // the tensor-core path, one record per (64-token chunk, v-head) (0 otherwise).
  const size_t need = gdn_workspace_bytes(layer, non_spec, spec) +
                      gdn_prefill_workspace_bytes(layer, non_spec, num_prefills);
  if (need > (size_t)GDN_STATIC_WORKSPACE_BYTES) return GDN_ERR_WORKSPACE;
  void* ws = static_workspace_address();
  if (!ws) return GDN_ERR_CUDA;
  return gdn_mixed_batch(layer, params, pools, x, a, b, num_actual_tokens, non_spec, num_decodes, num_prefills, spec,
                         out, ws, (size_t)GDN_STATIC_WORKSPACE_BYTES, d_status, stream);
}
