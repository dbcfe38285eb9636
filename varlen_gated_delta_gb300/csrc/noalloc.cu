// noalloc.cu - gdn_layer_varlen_noalloc: the layer call for callers that
// cannot allocate device memory.
//
// Some callers have no way to call cudaMalloc for the layer's workspace: a
// plain-C host runtime with no device allocator of its own, an inference
// plugin whose host framework owns every byte of device memory and forbids
// side allocations, or a latency-critical loop where cudaMalloc's implicit
// device synchronisation is not acceptable.  This entry point takes the same
// inputs and outputs as gdn_layer_varlen but uses, as its workspace, a
// file-scope device array of fixed size (GDN_NOALLOC_SCRATCH_BYTES).  Every
// GPU that loads the library holds that array until the process exits.
//
// Host code cannot use the array's name as a device address (in host code it
// names a host-side stand-in), so on the first call on each device, with that
// device current, the address is looked up once with cudaGetSymbolAddress and
// cached.  That first call should therefore come before any stream capture.
// The array is shared by every call and keeps the previous call's contents;
// the header the kernels read back is cleared on the stream before each use.
// Calls that overlap on the GPU (e.g. on two streams) race on the array.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gdn.h"
#include "internal.h"

namespace gdn {
namespace {

__device__ __align__(256) unsigned char g_noalloc_scratch[GDN_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
void *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array on the current device (set up once).
int scratch_address(void **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return set_error(GDN_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return set_error(GDN_ERR_UNSUPPORTED, "device %d beyond the %d devices this entry point tracks",
                         dev, kMaxDevices);
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || ptr == nullptr)
            return set_error(GDN_ERR_CUDA, "cudaGetSymbolAddress of the static scratch: %s",
                             cudaGetErrorString(e));
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return GDN_OK;
}

}  // namespace
}  // namespace gdn

extern "C" int gdn_layer_varlen_noalloc(
    const void *qkv, const void *w, const void *bias, const float *a, const float *b,
    const float *A_log, const float *dt_bias, const int32_t *offsets,
    const int32_t *offsets_host, const void *conv_init, void *conv_fin, const float *state_init,
    void *out, float *state_fin, int B, int N, int H, int HQ, int K, int V, int Kc, int D,
    int act, float scale, int dtype, void *stream) {
    const size_t need = gdn_workspace_bytes(B, N, H, HQ, K, V, Kc, D, dtype);
    if (need == 0) {
        // invalid geometry: let the regular entry point report the exact reason
        return gdn_layer_varlen(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host,
                                conv_init, conv_fin, state_init, out, state_fin, B, N, H, HQ, K,
                                V, Kc, D, act, scale, dtype, nullptr, 0, stream);
    }
    if (need > GDN_NOALLOC_SCRATCH_BYTES)
        return gdn::set_error(GDN_ERR_WORKSPACE,
                              "gdn_layer_varlen_noalloc: this call needs %zu bytes of scratch but "
                              "the static scratch holds %zu bytes (N=%d tokens is too many for "
                              "this head geometry); use gdn_layer_varlen with a workspace",
                              need, (size_t)GDN_NOALLOC_SCRATCH_BYTES, N);
    void *scratch = nullptr;
    int rc = gdn::scratch_address(&scratch);
    if (rc != GDN_OK) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemsetAsync(scratch, 0, sizeof(gdn::WsHeader), s);
    if (e != cudaSuccess)
        return gdn::set_error(GDN_ERR_CUDA, "clearing the static scratch header: %s",
                              cudaGetErrorString(e));
    // (the regular layer path, without its side stream: this call creates nothing)
    return gdn::layer_varlen_nofork(qkv, w, bias, a, b, A_log, dt_bias, offsets, offsets_host,
                                    conv_init, conv_fin, state_init, out, state_fin, B, N, H, HQ,
                                    K, V, Kc, D, act, scale, dtype, scratch,
                                    GDN_NOALLOC_SCRATCH_BYTES, stream);
}
