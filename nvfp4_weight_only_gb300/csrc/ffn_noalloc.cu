// ffn_noalloc.cu -- ffn_swiglu_nvfp4 on a library-owned, fixed workspace.
//
// Some callers cannot allocate device memory at the point where they run the
// FFN: a serving process that reserves the device's memory for its own pool at
// start-up and forbids any later cudaMalloc, or code that must not risk the
// implicit device-wide synchronisation an allocation can cause.  This entry
// point gives them the FFN without a caller-provided workspace: the workspace
// is one file-scope device array of kNoAllocWorkspaceBytes, which every GPU
// that loads the library holds until the process exits.
#include <cstdint>
#include <mutex>

#include "nvfp4ffn.h"

namespace {

constexpr size_t kNoAllocWorkspaceBytes = 24u << 20;  // 24 MiB
constexpr int kMaxDevices = 64;

// The workspace itself.  In host code this name is only a stand-in for the
// symbol; the device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_ffn_workspace[kNoAllocWorkspaceBytes];

std::mutex g_setup_mutex;
void* g_workspace_ptr[kMaxDevices] = {nullptr};

// Device address of g_ffn_workspace on the current device, resolved once per
// device (with that device current) and cached.
nvfp4_status workspace_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return NVFP4_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (g_workspace_ptr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_ffn_workspace) != cudaSuccess || p == nullptr)
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
    if (!x || !gate_up_packed || !down_packed || !out) return NVFP4_ERR_NULL;
    if (M < 1 || M > 16) return NVFP4_ERR_RANGE;
    if (H < 16 || I < 16 || H % 16 != 0 || I % 16 != 0) return NVFP4_ERR_SHAPE;
    void* ws = nullptr;
    nvfp4_status st = workspace_address(&ws);
    if (st != NVFP4_OK) return st;
    const size_t need = ffn_swiglu_nvfp4_workspace_bytes(M, H, I);
    if (need == 0 || need > kNoAllocWorkspaceBytes) return NVFP4_ERR_WORKSPACE;
    // The array keeps whatever the previous call left; start from zero.
    if (cudaMemsetAsync(ws, 0, need, stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    return ffn_swiglu_nvfp4(x, M, H, I, gate_up_packed, gate_scale2, up_scale2, down_packed,
                            down_scale2, act, out, ws, kNoAllocWorkspaceBytes, stream);
}
