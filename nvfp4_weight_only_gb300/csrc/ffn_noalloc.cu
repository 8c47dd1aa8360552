// ffn_noalloc.cu -- ffn_swiglu_nvfp4 on a library-owned, fixed workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// FFN: a serving process that reserves the device's memory for its own pool at
// start-up and forbids any later cudaMalloc, or code that must not risk the
// implicit device-wide synchronisation an allocation can cause.  This entry
// point gives them the FFN without a caller-provided workspace: the workspace
// is one file-scope device array of kNoAllocWorkspaceBytes, which every GPU
// that loads the library holds until the process exits.
//
// The array follows the workspace contract of ffn_swiglu_nvfp4: zero-filled
// once (here, at the first call on each device), then left reusable by every
// successful call.  A call that abandons a bounded wait leaves a nonzero
// status word and possibly inconsistent split-K counters; nvfp4_noalloc_status
// reports that and zero-fills the array again.
#include <cstdint>
#include <mutex>

#include "internal.h"
#include "nvfp4ffn.h"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = 24u << 20;  // 24 MiB
constexpr int kMaxDevices = 64;

// The workspace itself.  In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_ffn_workspace[kNoAllocWorkspaceBytes];

std::mutex g_setup_mutex;
void* g_workspace_ptr[kMaxDevices] = {nullptr};

// Device address of g_ffn_workspace on the current device.  The first request
// on a device (with that device current) resolves the address and zero-fills
// the array on `stream`, waiting for the fill to finish; later requests
// return the cached address and touch nothing.
nvfp4_status workspace_address(cudaStream_t stream, void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_workspace_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ffn_workspace) != cudaSuccess || p == nullptr)
            return NVFP4_ERR_CUDA;
        if (cudaMemsetAsync(p, 0, kNoAllocWorkspaceBytes, stream) != cudaSuccess ||
            cudaStreamSynchronize(stream) != cudaSuccess)
            return NVFP4_ERR_CUDA;
        g_workspace_ptr[dev] = p;
    }
    *out = g_workspace_ptr[dev];
    return NVFP4_OK;
}

}  // namespace

extern "C" nvfp4_status ffn_swiglu_nvfp4_noalloc(const void* x, int M, int H, int I,
                                                 const void* gate_up_packed, float gate_scale2,
                                                 float up_scale2, const void* down_packed,
                                                 float down_scale2, nvfp4_act act, void* out,
                                                 cudaStream_t stream) {
    // Every argument check comes first: a rejected call changes nothing.
    const int v = nvf::validate_ffn_args(x, M, H, I, gate_up_packed, down_packed, (int)act, out);
    if (v != NVFP4_OK) return (nvfp4_status)v;
    if (M > 16) return NVFP4_ERR_RANGE;  // one kernel group: the array is sized for it
    const size_t need = ffn_swiglu_nvfp4_workspace_bytes(M, H, I);
    if (need == 0 || need > kNoAllocWorkspaceBytes) return NVFP4_ERR_WORKSPACE;
    void* ws = nullptr;
    const nvfp4_status st = workspace_address(stream, &ws);
    if (st != NVFP4_OK) return st;
    return ffn_swiglu_nvfp4(x, M, H, I, gate_up_packed, gate_scale2, up_scale2, down_packed,
                            down_scale2, act, out, ws, kNoAllocWorkspaceBytes, stream);
}

extern "C" nvfp4_status nvfp4_noalloc_status(cudaStream_t stream) {
    void* ws = nullptr;
    nvfp4_status st = workspace_address(stream, &ws);
    if (st != NVFP4_OK) return st;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (word == 0) return NVFP4_OK;
    // A timed-out call may leave split-K counters off zero: start over.
    if (cudaMemsetAsync(ws, 0, kNoAllocWorkspaceBytes, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    return NVFP4_ERR_TIMEOUT;
}
