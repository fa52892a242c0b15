// static_ws.cu -- sa_decode for callers that cannot allocate device memory.
//
// A split decode needs scratch for the per-chunk partial states.  sa_decode
// takes that scratch from the caller.  Some callers have no way to provide it:
// a plugin loaded into a host program that owns every device allocation and
// hands out only the tensors it passes in, or a caller on a latency-critical
// path that must not call cudaMalloc (which can synchronise the device).  For
// them this file keeps the scratch in one file-scope device array of fixed
// size, created when the library's device code is loaded on a GPU and held by
// every GPU that loads the library until the process exits.
//
// The array's name is only a host-side stand-in for the device symbol, so the
// host code below never passes it to a kernel: it looks up the array's device
// address with cudaGetSymbolAddress once per device (with that device
// current) and hands that address to sa_decode as its workspace.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/sink_attn.h"
#include "sa_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_static_workspace[SA_STATIC_WORKSPACE_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_static_mu;
void *g_static_ptr[kMaxDevices] = {nullptr};

// Device address of the array on the current device (looked up on first use).
cudaError_t static_workspace_ptr(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess)
        return e;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_static_mu);
    if (!g_static_ptr[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_workspace);
        if (e != cudaSuccess)
            return e;
        g_static_ptr[dev] = p;
    }
    *out = g_static_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" sa_status_t sa_decode_static_workspace(const void *q, const sa_kv_desc_t *kv, const int32_t *seqlens,
                                                  int32_t batch, int32_t num_qo_heads, int32_t max_kv_len,
                                                  const float *sinks, int32_t window, float sm_scale, void *out,
                                                  float *lse, int32_t num_splits, cudaStream_t stream)
{
    if (!kv)  // sa_decode rejects it before any launch, with its own message
        return sa_decode(q, kv, seqlens, batch, num_qo_heads, max_kv_len, sinks, window, sm_scale, out, lse,
                         nullptr, 0, num_splits, stream);
    const size_t need = sa_decode_workspace_size(batch, num_qo_heads, kv->num_kv_heads, kv->head_dim, max_kv_len,
                                                 window, num_splits);
    if (need > SA_STATIC_WORKSPACE_BYTES)
        return sa::set_last_error(SA_ERR_WORKSPACE,
                                  "sa_decode_static_workspace: this split needs %zu bytes of scratch, the static "
                                  "array holds %zu; pass fewer num_splits or call sa_decode with a workspace",
                                  need, static_cast<size_t>(SA_STATIC_WORKSPACE_BYTES));
    void *ws = nullptr;
    if (need > 0) {
        const cudaError_t e = static_workspace_ptr(&ws);
        if (e != cudaSuccess)
            return sa::set_last_error(SA_ERR_CUDA, "sa_decode_static_workspace: cudaGetSymbolAddress: %s",
                                      cudaGetErrorString(e));
    }
    return sa_decode(q, kv, seqlens, batch, num_qo_heads, max_kv_len, sinks, window, sm_scale, out, lse, ws,
                     need > 0 ? static_cast<size_t>(SA_STATIC_WORKSPACE_BYTES) : 0, num_splits, stream);
}
