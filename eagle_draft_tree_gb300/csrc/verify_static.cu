// verify_static.cu -- eagle_tree_verify_static: eagle_tree_verify with its scratch in static device
// storage, for callers that cannot hand the library a device workspace (see include/eagle.h).
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"

namespace {

constexpr size_t kVerifyScratchBytes = size_t(256) << 10;  // 256 KB: e.g. 113 sequences of 64 nodes
constexpr int kMaxDevices = 64;

// The scratch itself: file-scope device storage, zero-filled when the module is loaded.  Only its
// header (the device status word and the per-call failure tag) is ever read before this call
// writes it, and both start at zero; every other byte is written by a kernel of the call before
// another reads it.  A call whose waits ran out is recognised by its own failure tag, so what an
// earlier call left never reaches the outputs.
static __device__ __align__(256) unsigned char g_verify_scratch[kVerifyScratchBytes];

// Per-device address of the scratch, looked up by the first call on each device.
std::atomic<void *> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" eagle_status eagle_tree_verify_static(const eagle_verify_cfg *cfg, const float *target_logits,
                                                 const float *draft_logits, const int32_t *tokens,
                                                 const int32_t *parents, const int32_t *node_row,
                                                 const float *uniforms, int32_t *out_tokens, int32_t *out_len,
                                                 int32_t *out_path, float *out_ratio, cudaStream_t stream) {
    if (!cfg) return EAGLE_ERR_INVALID_ARG;
    const size_t need = eagle_tree_verify_workspace_size(cfg);
    if (need == 0)  // an invalid configuration: the regular entry point reports why, launching nothing
        return eagle_tree_verify(cfg, target_logits, draft_logits, tokens, parents, node_row, uniforms, out_tokens,
                                 out_len, out_path, out_ratio, nullptr, 0, stream);
    if (need > kVerifyScratchBytes) return EAGLE_ERR_UNSUPPORTED;  // more nodes than the scratch holds
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return EAGLE_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return EAGLE_ERR_UNSUPPORTED;
    // the scratch address below is the current device's: the stream must belong to that device
    int sdev = -1;
    if (cudaStreamGetDevice(stream, &sdev) != cudaSuccess) return EAGLE_ERR_INVALID_ARG;
    if (sdev != dev) return EAGLE_ERR_INVALID_ARG;
    void *scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!scratch) {
        if (cudaGetSymbolAddress(&scratch, g_verify_scratch) != cudaSuccess || !scratch) return EAGLE_ERR_CUDA;
        g_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    return eagle_tree_verify(cfg, target_logits, draft_logits, tokens, parents, node_row, uniforms, out_tokens,
                             out_len, out_path, out_ratio, scratch, kVerifyScratchBytes, stream);
}
