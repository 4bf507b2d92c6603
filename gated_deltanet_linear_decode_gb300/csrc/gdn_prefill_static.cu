// gdn_prefill_static.cu -- gdn_prefill_chunked_static (include/gdn.h): the
// chunked prefill with its scratch in one fixed, statically declared device
// area instead of a caller-provided workspace, for callers that cannot
// allocate device memory.  It looks up the area's device address and hands it
// to gdn_prefill_chunked as the workspace; nothing else differs.
#include <cuda_runtime.h>

#include "gdn.h"

namespace {

constexpr size_t kScratchBytes = GDN_PREFILL_STATIC_SCRATCH_BYTES;

// The scratch area: one per device for the life of the process, shared by every
// call.  In host code this name is only a stand-in for the symbol, never a
// device address; the kernels get the address looked up below.
static __device__ __align__(256) unsigned char g_prefill_scratch[kScratchBytes];

// Device address of the area on the current device.  Looked up on every call
// (a host-side query): a cached address would go stale if the device's
// context were destroyed and created again (cudaDeviceReset, or the primary
// context released), which loads the module anew, possibly elsewhere.
cudaError_t scratch_address(void** addr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_prefill_scratch);
    if (e != cudaSuccess) return e;
    *addr = p;
    return cudaSuccess;
}

}  // namespace

extern "C" gdn_status gdn_prefill_chunked_static(const gdn_dims* dims, const gdn_weights* w, int32_t n_seq,
                                                 const int32_t* cu_seqlens_host, const int32_t* cu_seqlens_dev,
                                                 const void* x, const void* z, const void* a_raw, const void* b_raw,
                                                 void* conv_state, void* S, int32_t zero_init, void* out,
                                                 float* prenorm_out, int32_t* dev_status, gdn_stream_t stream) {
    if (!dims || n_seq < 0 || !cu_seqlens_host) return GDN_E_INVALID_ARG;
    const size_t need = gdn_prefill_workspace_bytes(dims, n_seq, cu_seqlens_host[n_seq]);
    if (need > kScratchBytes) return GDN_E_WORKSPACE;
    void* ws = nullptr;
    if (need > 0 && scratch_address(&ws) != cudaSuccess) return GDN_E_CUDA;
    return gdn_prefill_chunked(dims, w, n_seq, cu_seqlens_host, cu_seqlens_dev, x, z, a_raw, b_raw, conv_state, S,
                               zero_init, out, prenorm_out, ws, need > 0 ? kScratchBytes : 0, dev_status, stream);
}
