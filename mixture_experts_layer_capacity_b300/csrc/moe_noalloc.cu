// moe_noalloc.cu -- moe_forward_no_alloc: the forward pass for callers that
// cannot allocate device memory, with its scratch in a fixed array that the
// library itself places in device memory when the module loads.
//
// The scratch is a file-scope __device__ array.  Its name in host code is
// only a host-side stand-in, so the device address is looked up with
// cudaGetSymbolAddress (with the device current) and passed on; nothing here
// calls cudaMalloc, cudaFree or any allocating routine.  The lookup is
// repeated on every call made outside stream capture, so a device reset
// (which reloads the module and may move the array) is picked up by the next
// such call; calls made while the stream is capturing use the address found
// by the last call outside capture on that device.
#include <mutex>

#include "moe_internal.h"

namespace {

// Every GPU that loads this library holds this array until the process exits.
static __device__ __align__(256) unsigned char g_static_scratch[MOE_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void *g_scratch_ptr[kMaxDevices] = {nullptr};

// Device address of g_static_scratch on the current device: looked up
// afresh when `stream` is not capturing (and remembered per device), taken
// from that memory while it is.  Returns cudaSuccess or the lookup's error.
cudaError_t scratch_address(cudaStream_t stream, void **ptr)
{
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess)
        return err;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    err = cudaStreamIsCapturing(stream, &cs);
    if (err != cudaSuccess)
        return err;
    if (dev < 0 || dev >= kMaxDevices)
        return cudaGetSymbolAddress(ptr, g_static_scratch);
    std::lock_guard<std::mutex> lock(g_mu);
    if (cs == cudaStreamCaptureStatusNone || !g_scratch_ptr[dev]) {
        void *p = nullptr;
        err = cudaGetSymbolAddress(&p, g_static_scratch);
        if (err != cudaSuccess)
            return err;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_forward_no_alloc(
    const moe_config *cfg, const void *x, const void *W_r, const float *router_bias,
    const void *W_gate, const void *W_up, const void *W_down, const void *Ws_gate,
    const void *Ws_up, const void *Ws_down, void *y, float *router_logits, int32_t *topk_idx,
    float *topk_w, uint8_t *dropped_mask, int32_t *expert_counts, int32_t *kept_counts,
    float *aux_loss, cudaStream_t stream)
{
    size_t need = 0;
    const moe_status st = moe_workspace_size(cfg, &need);
    if (st != MOE_OK)
        return st;
    if (need > (size_t)MOE_STATIC_SCRATCH_BYTES)
        return MOE_ERR_WORKSPACE;  // the layer needs more scratch than the static array holds
    void *scratch = nullptr;
    if (scratch_address(stream, &scratch) != cudaSuccess || !scratch)
        return MOE_ERR_CUDA;
    // moe_forward clears the parts of its workspace that must start at zero
    // (status word and counters) on the stream before its first kernel.
    return moe_forward(cfg, x, W_r, router_bias, W_gate, W_up, W_down, Ws_gate, Ws_up, Ws_down, y,
                       router_logits, topk_idx, topk_w, dropped_mask, expert_counts, kept_counts,
                       aux_loss, scratch, (size_t)MOE_STATIC_SCRATCH_BYTES, stream);
}
