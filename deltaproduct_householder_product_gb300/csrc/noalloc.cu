// dp_forward_noalloc: the whole-sequence forward for callers that cannot
// allocate device memory. Some embedders own every byte of HBM through their
// own allocator or a fixed memory budget (an inference server that
// pre-partitions the GPU, a framework plugin whose host forbids raw
// cudaMalloc, a latency-critical path that cannot afford cudaMalloc's
// implicit synchronisation), so they cannot hand dp_forward the workspace it
// asks for. This entry point takes the same inputs and outputs as dp_forward
// but keeps its scratch (the device status word and any per-call scratch the
// forward kernels need) in a fixed array inside libdp.so.
//
// The array is a file-scope __device__ object: every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits. All
// calls on a device share it, so calls whose kernels overlap on the GPU
// (different streams without ordering between them) race on it; calls on one
// stream are ordered and safe. Problems whose workspace (as reported by
// dp_forward_workspace_size) exceeds kNoAllocScratchBytes are rejected with
// DP_ERR_WORKSPACE.
#include <mutex>

#include "internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = 64 * 1024;
constexpr int kMaxDevices = 64;

// In host code this name is only a host-side stand-in for the device array;
// its device address comes from cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

void *g_scratch_addr[kMaxDevices];
std::mutex g_scratch_lock;

// Device address of the scratch array on the current device. Outside stream
// capture it is looked up on every call (cheap), so a context rebuilt after
// cudaDeviceReset never receives the old context's address; a call made while
// `stream` is capturing uses the address cached by the last uncaptured call
// on that device and fails with DP_ERR_CUDA if there was none.
dp_status scratch_for_current_device(cudaStream_t stream, void **out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return DP_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return DP_ERR_UNSUPPORTED;
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        cudaGetLastError();
        return DP_ERR_CUDA;
    }
    std::lock_guard<std::mutex> guard(g_scratch_lock);
    if (cap == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return DP_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    if (!g_scratch_addr[dev]) return DP_ERR_CUDA;
    *out = g_scratch_addr[dev];
    return DP_OK;
}

}  // namespace

extern "C" dp_status dp_forward_noalloc(const dp_dims *dims, const void *q, const void *k,
                                        const void *v, const void *beta, const void *g,
                                        const float *h0, void *o, float *h_final,
                                        dp_stream_t stream)
{
    size_t need = 0;
    dp_status s = dp_forward_workspace_size(dims, &need);
    if (s != DP_OK) return s;
    if (need > kNoAllocScratchBytes) return DP_ERR_WORKSPACE;
    void *scratch = nullptr;
    s = scratch_for_current_device((cudaStream_t)stream, &scratch);
    if (s != DP_OK) return s;
    // The array is zero at load. The kernels write the status word only on a
    // device-side error, and this call clears it again behind its own kernel,
    // so the next call's kernel starts from zero. The rest of the array holds
    // whatever the last call left: per-chunk records (rewritten by every call
    // before they are read) and the cooperative mode's flags (cleared by
    // dp_forward before each cooperative launch), so calls of different
    // shapes may follow one another on a stream.
    s = dp_forward(dims, q, k, v, beta, g, h0, o, h_final, scratch, kNoAllocScratchBytes, stream);
    if (s != DP_OK) return s;
    if (cudaMemsetAsync(scratch, 0, need, (cudaStream_t)stream) != cudaSuccess) return DP_ERR_CUDA;
    return DP_OK;
}
