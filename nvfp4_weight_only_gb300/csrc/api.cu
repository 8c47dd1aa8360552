// api.cu -- the C ABI declared in include/nvfp4ffn.h: host-side argument
// validation, workspace carving and launch of the sm_103a kernels.  No
// arithmetic of the method lives here.
#include <cstdint>
#include <cstring>

#include "internal.h"
#include "layout.h"
#include "nvfp4ffn.h"
#include "nvfp4ffn_testing.h"

namespace {

constexpr size_t kQuantizeScratch = 256;
// Size assumed for workspace queries when no device is visible.
constexpr int kFallbackSms = 160;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool overlap(const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

int sms_for_sizing() {
    const int n = nvf::device_sm_count();
    return n > 0 ? n : kFallbackSms;
}

nvfp4_status cuda_status(cudaError_t e) { return e == cudaSuccess ? NVFP4_OK : NVFP4_ERR_CUDA; }

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// Token rows per call: up to kMaxTokens; the kernels take groups of up to
// kGroupTokens rows, so a larger batch runs as consecutive groups, each of
// which streams the weights once.
constexpr int kMaxTokens = 64;
constexpr int kGroupTokens = 16;

int group_count(int M) { return (M + kGroupTokens - 1) / kGroupTokens; }
int group_rows(int M, int g) {
    const int left = M - g * kGroupTokens;
    return left < kGroupTokens ? left : kGroupTokens;
}

// Partial-sum bytes of the largest launch among M's groups (they run one
// after another on the same stream, so they share one area).
size_t group_partial_bytes(int streams, int M, int N, int K, int sms, bool f8 = false) {
    size_t most = nvf::gemv_partial_bytes(streams, group_rows(M, 0), N, K, sms, f8);
    const int last = group_rows(M, group_count(M) - 1);
    const size_t b = nvf::gemv_partial_bytes(streams, last, N, K, sms, f8);
    return b > most ? b : most;
}

// GEMV workspace: [status][counter region][partials].  0 if N has more row
// blocks than the counter region holds.
size_t gemv_ws_bytes(int streams, int M, int N, int K, int sms, bool f8 = false) {
    if (nvf::gemv_counter_bytes(N) > nvf::kCounterRegionBytes) return 0;
    return nvf::kDataOffset + round256(group_partial_bytes(streams, M, N, K, sms, f8));
}

// FFN workspace: [status][counter region: dual's counters, then down's]
// [h (M x I bf16)][dual-kernel partials][down-kernel partials]
struct FfnLayout {
    size_t down_cnt_off, h_off, dual_off, dual_bytes, down_off, down_bytes, total;
    bool fits;  // both kernels' counters fit the counter region
};

FfnLayout ffn_layout(int M, int H, int I, int sms, bool f8 = false) {
    FfnLayout l;
    l.down_cnt_off = nvf::gemv_counter_bytes(I);
    l.fits = l.down_cnt_off + nvf::gemv_counter_bytes(H) <= nvf::kCounterRegionBytes;
    l.h_off = nvf::kDataOffset;
    l.dual_off = l.h_off + round256((size_t)M * I * 2);
    l.dual_bytes = round256(group_partial_bytes(2, M, I, H, sms, f8));
    l.down_off = l.dual_off + l.dual_bytes;
    l.down_bytes = round256(group_partial_bytes(1, M, H, I, sms, f8));
    l.total = l.down_off + l.down_bytes;
    return l;
}

}  // namespace

namespace nvf {

int validate_ffn_args(const void* x, int M, int H, int I, const void* gate_up_packed,
                      const void* down_packed, int act, const void* out) {
    if (!x || !gate_up_packed || !down_packed || !out) return NVFP4_ERR_NULL;
    if (M < 1 || M > kMaxTokens) return NVFP4_ERR_RANGE;
    if (act != NVFP4_ACT_SILU && act != NVFP4_ACT_GELU_TANH) return NVFP4_ERR_RANGE;
    if (H < 16 || I < 16 || H % 16 != 0 || I % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gate_up_packed) || !aligned16(down_packed) ||
        !aligned16(out))
        return NVFP4_ERR_ALIGN;
    if (overlap(x, (size_t)M * H * 2, out, (size_t)M * H * 2)) return NVFP4_ERR_ALIAS;
    return NVFP4_OK;
}

}  // namespace nvf

extern "C" {

size_t nvfp4_quantize_scratch_bytes(int N, int K) {
    (void)N;
    (void)K;
    return kQuantizeScratch;
}

nvfp4_status nvfp4_quantize(const void* w, nvfp4_src_dtype dtype, int N, int K, uint8_t* codes,
                            uint8_t* scales, float* scale2_out, void* scratch,
                            size_t scratch_bytes, cudaStream_t stream) {
    if (!w || !codes || !scales || !scale2_out || !scratch) return NVFP4_ERR_NULL;
    if (dtype != NVFP4_SRC_F32 && dtype != NVFP4_SRC_BF16) return NVFP4_ERR_RANGE;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(w) || !aligned16(codes) || !aligned16(scratch)) return NVFP4_ERR_ALIGN;
    if (scratch_bytes < kQuantizeScratch) return NVFP4_ERR_WORKSPACE;
    cudaError_t e = nvf::launch_quantize(w, dtype == NVFP4_SRC_BF16 ? 1 : 0, N, K, codes, scales,
                                         scratch, stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    float s2 = 0.0f;
    e = cudaMemcpyAsync(&s2, reinterpret_cast<char*>(scratch) + 4, 4, cudaMemcpyDeviceToHost,
                        stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    *scale2_out = s2;
    return NVFP4_OK;
}

size_t nvfp4_repacked_bytes(int N, int K) {
    if (N < 1 || K < 16) return 0;
    return nvf::repacked_bytes(N, K, 1);
}

size_t nvfp4_repacked_gate_up_bytes(int I, int H) {
    if (I < 1 || H < 16) return 0;
    return nvf::repacked_bytes(I, H, 2);
}

nvfp4_status nvfp4_repack(const uint8_t* codes, const uint8_t* scales, int N, int K, void* packed,
                          cudaStream_t stream) {
    if (!codes || !scales || !packed) return NVFP4_ERR_NULL;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(packed)) return NVFP4_ERR_ALIGN;
    return cuda_status(
        nvf::launch_repack(codes, scales, N, K, reinterpret_cast<uint8_t*>(packed), 1, 0, stream));
}

nvfp4_status nvfp4_repack_gate_up(const uint8_t* gate_codes, const uint8_t* gate_scales,
                                  const uint8_t* up_codes, const uint8_t* up_scales, int I, int H,
                                  void* packed, cudaStream_t stream) {
    if (!gate_codes || !gate_scales || !up_codes || !up_scales || !packed) return NVFP4_ERR_NULL;
    if (I < 1 || H < 16 || H % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(packed)) return NVFP4_ERR_ALIGN;
    uint8_t* p = reinterpret_cast<uint8_t*>(packed);
    cudaError_t e = nvf::launch_repack(gate_codes, gate_scales, I, H, p, 2, 0, stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    return cuda_status(nvf::launch_repack(up_codes, up_scales, I, H, p, 2, 1, stream));
}

nvfp4_status nvfp4_unpack(const void* packed, int N, int K, uint8_t* codes, uint8_t* scales,
                          cudaStream_t stream) {
    if (!packed || !codes || !scales) return NVFP4_ERR_NULL;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(packed)) return NVFP4_ERR_ALIGN;
    return cuda_status(nvf::launch_unpack(reinterpret_cast<const uint8_t*>(packed), N, K, codes,
                                          scales, stream));
}

size_t nvfp4_gemv_workspace_bytes(int M, int N, int K) {
    if (M < 1 || M > kMaxTokens || N < 1 || K < 16) return 0;
    return gemv_ws_bytes(1, M, N, K, sms_for_sizing());
}

nvfp4_status nvfp4_gemv(const void* x, int M, int K, const void* packed_w, float scale2, int N,
                        void* y, void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!x || !packed_w || !y || !ws) return NVFP4_ERR_NULL;
    if (M < 1 || M > kMaxTokens) return NVFP4_ERR_RANGE;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(packed_w) || !aligned16(y) || !aligned16(ws))
        return NVFP4_ERR_ALIGN;
    if (overlap(x, (size_t)M * K * 2, y, (size_t)M * N * 2)) return NVFP4_ERR_ALIAS;
    const int sms = nvf::device_sm_count();
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const size_t need = gemv_ws_bytes(1, M, N, K, sms);
    if (need == 0) return NVFP4_ERR_SHAPE;
    if (ws_bytes < need) return NVFP4_ERR_WORKSPACE;
    char* w = reinterpret_cast<char*>(ws);
    for (int g = 0; g < group_count(M); ++g) {
        const size_t r0 = (size_t)g * kGroupTokens;
        const cudaError_t e = nvf::launch_stream_gemv(
            1, reinterpret_cast<const char*>(x) + r0 * K * 2, group_rows(M, g), K, packed_w, N,
            scale2, scale2, 0, reinterpret_cast<char*>(y) + r0 * N * 2, reinterpret_cast<int*>(w),
            reinterpret_cast<int*>(w + nvf::kStatusBytes), w + nvf::kDataOffset,
            need - nvf::kDataOffset, sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

size_t ffn_swiglu_nvfp4_workspace_bytes(int M, int H, int I) {
    if (M < 1 || M > kMaxTokens || H < 16 || I < 16) return 0;
    const FfnLayout l = ffn_layout(M, H, I, sms_for_sizing());
    return l.fits ? l.total : 0;
}

size_t ffn_swiglu_nvfp4_hidden_offset(void) { return nvf::kDataOffset; }

nvfp4_status ffn_swiglu_nvfp4(const void* x, int M, int H, int I, const void* gate_up_packed,
                              float gate_scale2, float up_scale2, const void* down_packed,
                              float down_scale2, nvfp4_act act, void* out, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
    if (!ws) return NVFP4_ERR_NULL;
    const int v = nvf::validate_ffn_args(x, M, H, I, gate_up_packed, down_packed, (int)act, out);
    if (v != NVFP4_OK) return (nvfp4_status)v;
    if (!aligned16(ws)) return NVFP4_ERR_ALIGN;
    const int sms = nvf::device_sm_count();
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const FfnLayout l = ffn_layout(M, H, I, sms);
    if (!l.fits) return NVFP4_ERR_SHAPE;
    if (ws_bytes < l.total) return NVFP4_ERR_WORKSPACE;
    char* w = reinterpret_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* counters = reinterpret_cast<int*>(w + nvf::kStatusBytes);
    void* h = w + l.h_off;
    for (int g = 0; g < group_count(M); ++g) {
        const size_t r0 = (size_t)g * kGroupTokens;
        const int mg = group_rows(M, g);
        char* hg = reinterpret_cast<char*>(h) + r0 * I * 2;
        cudaError_t e = nvf::launch_stream_gemv(
            2, reinterpret_cast<const char*>(x) + r0 * H * 2, mg, H, gate_up_packed, I,
            gate_scale2, up_scale2, (int)act, hg, status, counters, w + l.dual_off, l.dual_bytes,
            sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
        e = nvf::launch_stream_gemv(1, hg, mg, I, down_packed, H, down_scale2, down_scale2, 0,
                                    reinterpret_cast<char*>(out) + r0 * H * 2, status,
                                    counters + l.down_cnt_off / sizeof(int), w + l.down_off,
                                    l.down_bytes, sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

// LoRA FFN workspace: the FFN's, then the fp32 slice sums of A_gate x, A_up x
// (lora_partial_bytes each), the bf16 gate and up deltas [M, I] each, and the
// slice sums of A_down h.
struct LoraLayout {
    FfnLayout ffn;
    size_t xa_g, xa_u, d_g, d_u, xa_d, total;
};

LoraLayout lora_layout(int M, int H, int I, int r, int sms) {
    LoraLayout l;
    l.ffn = ffn_layout(M, H, I, sms);
    const size_t xr = round256(nvf::lora_partial_bytes(M, r)), xi = round256((size_t)M * I * 2);
    l.xa_g = l.ffn.total;
    l.xa_u = l.xa_g + xr;
    l.d_g = l.xa_u + xr;
    l.d_u = l.d_g + xi;
    l.xa_d = l.d_u + xi;
    l.total = l.xa_d + xr;
    return l;
}

size_t ffn_swiglu_nvfp4_lora_workspace_bytes(int M, int H, int I, int rank) {
    if (M < 1 || M > 16 || H < 16 || I < 16 || rank < 1 || rank > nvf::kLoraMaxRank) return 0;
    const LoraLayout l = lora_layout(M, H, I, rank, sms_for_sizing());
    return l.ffn.fits ? l.total : 0;
}

nvfp4_status ffn_swiglu_nvfp4_lora(const void* x, int M, int H, int I, const void* gate_up_packed,
                                   float gate_scale2, float up_scale2, const void* down_packed,
                                   float down_scale2, nvfp4_act act, int rank, const void* gate_a,
                                   const void* gate_b, const void* up_a, const void* up_b,
                                   const void* down_a, const void* down_b, void* out, void* ws,
                                   size_t ws_bytes, cudaStream_t stream) {
    if (!ws) return NVFP4_ERR_NULL;
    const int v = nvf::validate_ffn_args(x, M, H, I, gate_up_packed, down_packed, (int)act, out);
    if (v != NVFP4_OK) return (nvfp4_status)v;
    if (M > kGroupTokens || rank < 1 || rank > nvf::kLoraMaxRank) return NVFP4_ERR_RANGE;
    const void* pa[3] = {gate_a, up_a, down_a};
    const void* pb[3] = {gate_b, up_b, down_b};
    for (int p = 0; p < 3; ++p) {
        if ((pa[p] == nullptr) != (pb[p] == nullptr)) return NVFP4_ERR_NULL;
        if (pa[p] && (!aligned16(pa[p]) || !aligned16(pb[p]))) return NVFP4_ERR_ALIGN;
    }
    if (!aligned16(ws)) return NVFP4_ERR_ALIGN;
    const int sms = nvf::device_sm_count();
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const LoraLayout l = lora_layout(M, H, I, rank, sms);
    if (!l.ffn.fits) return NVFP4_ERR_SHAPE;
    if (ws_bytes < l.total) return NVFP4_ERR_WORKSPACE;
    char* w = reinterpret_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* counters = reinterpret_cast<int*>(w + nvf::kStatusBytes);
    void* h = w + l.ffn.h_off;
    cudaError_t e = cudaSuccess;
    // gate/up deltas of x, before the gate/up kernel
    const void* A[2];
    const void* B[2];
    void* xa[2];
    void* d[2];
    int np = 0;
    const void* deltas[2] = {nullptr, nullptr};
    for (int p = 0; p < 2; ++p)
        if (pa[p]) {
            A[np] = pa[p];
            B[np] = pb[p];
            xa[np] = w + (p == 0 ? l.xa_g : l.xa_u);
            d[np] = w + (p == 0 ? l.d_g : l.d_u);
            deltas[p] = d[np];
            ++np;
        }
    if (np > 0) {
        e = nvf::launch_lora_xa(x, M, H, A, xa, np, rank, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
        e = nvf::launch_lora_delta(xa, H, B, d, np, M, I, rank, false, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    e = nvf::launch_stream_gemv(2, x, M, H, gate_up_packed, I, gate_scale2, up_scale2, (int)act, h,
                                status, counters, w + l.ffn.dual_off, l.ffn.dual_bytes, sms, true,
                                stream, np > 0 ? deltas : nullptr);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    // The down kernel follows the gate/up kernel directly, so that it streams
    // its weights while the gate/up kernel finishes; A_down h comes after it.
    e = nvf::launch_stream_gemv(1, h, M, I, down_packed, H, down_scale2, down_scale2, 0, out,
                                status, counters + l.ffn.down_cnt_off / sizeof(int),
                                w + l.ffn.down_off, l.ffn.down_bytes, sms, true, stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    void* xad = w + l.xa_d;
    if (down_a) {  // out = bf16(out + B_down bf16(A_down h))
        e = nvf::launch_lora_xa(h, M, I, &down_a, &xad, 1, rank, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
        const void* xac = xad;
        e = nvf::launch_lora_delta(&xac, I, &down_b, &out, 1, M, H, rank, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

size_t nvfp4_lora_apply_scratch_bytes(int M, int rank) {
    if (M < 1 || M > 16 || rank < 1 || rank > nvf::kLoraMaxRank) return 0;
    return round256(nvf::lora_partial_bytes(M, rank));
}

nvfp4_status nvfp4_lora_apply(const void* v, int M, int K, const void* a, const void* b, int rank,
                              int N, void* base, void* scratch, size_t scratch_bytes,
                              cudaStream_t stream) {
    if (!v || !a || !b || !base || !scratch) return NVFP4_ERR_NULL;
    if (M < 1 || M > 16 || rank < 1 || rank > nvf::kLoraMaxRank) return NVFP4_ERR_RANGE;
    if (K < 2 || K % 2 != 0 || N < 1) return NVFP4_ERR_SHAPE;
    if (!aligned16(v) || !aligned16(a) || !aligned16(b) || !aligned16(base) || !aligned16(scratch))
        return NVFP4_ERR_ALIGN;
    if (overlap(v, (size_t)M * K * 2, base, (size_t)M * N * 2)) return NVFP4_ERR_ALIAS;
    if (scratch_bytes < nvfp4_lora_apply_scratch_bytes(M, rank)) return NVFP4_ERR_WORKSPACE;
    cudaError_t e = nvf::launch_lora_xa(v, M, K, &a, &scratch, 1, rank, stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    const void* xa = scratch;
    return cuda_status(nvf::launch_lora_delta(&xa, K, &b, &base, 1, M, N, rank, true, stream));
}

size_t ffn_gate_up_nvfp4_workspace_bytes(int M, int H, int I) {
    if (M < 1 || M > kMaxTokens || H < 16 || I < 16) return 0;
    return gemv_ws_bytes(2, M, I, H, sms_for_sizing());
}

nvfp4_status ffn_gate_up_nvfp4(const void* x, int M, int H, int I, const void* gate_up_packed,
                               float gate_scale2, float up_scale2, nvfp4_act act, void* h,
                               void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!x || !gate_up_packed || !h || !ws) return NVFP4_ERR_NULL;
    if (M < 1 || M > kMaxTokens) return NVFP4_ERR_RANGE;
    if (act != NVFP4_ACT_SILU && act != NVFP4_ACT_GELU_TANH) return NVFP4_ERR_RANGE;
    if (H < 16 || I < 16 || H % 16 != 0 || I % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(gate_up_packed) || !aligned16(h) || !aligned16(ws))
        return NVFP4_ERR_ALIGN;
    if (overlap(x, (size_t)M * H * 2, h, (size_t)M * I * 2)) return NVFP4_ERR_ALIAS;
    const int sms = nvf::device_sm_count();
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const size_t need = gemv_ws_bytes(2, M, I, H, sms);
    if (need == 0) return NVFP4_ERR_SHAPE;
    if (ws_bytes < need) return NVFP4_ERR_WORKSPACE;
    char* w = reinterpret_cast<char*>(ws);
    for (int g = 0; g < group_count(M); ++g) {
        const size_t r0 = (size_t)g * kGroupTokens;
        const cudaError_t e = nvf::launch_stream_gemv(
            2, reinterpret_cast<const char*>(x) + r0 * H * 2, group_rows(M, g), H, gate_up_packed,
            I, gate_scale2, up_scale2, (int)act, reinterpret_cast<char*>(h) + r0 * I * 2,
            reinterpret_cast<int*>(w), reinterpret_cast<int*>(w + nvf::kStatusBytes),
            w + nvf::kDataOffset, need - nvf::kDataOffset, sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

nvfp4_status nvfp4_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!ws) return NVFP4_ERR_NULL;
    return cuda_status(cudaMemsetAsync(ws, 0, ws_bytes, stream));
}

nvfp4_status nvfp4_workspace_status(void* ws, cudaStream_t stream) {
    if (!ws) return NVFP4_ERR_NULL;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return NVFP4_ERR_CUDA;
    int st = 0;
    if (cudaMemcpy(&st, ws, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
        return NVFP4_ERR_CUDA;
    if (st == 0) return NVFP4_OK;
    if (cudaMemset(ws, 0, sizeof(int)) != cudaSuccess) return NVFP4_ERR_CUDA;
    return NVFP4_ERR_TIMEOUT;
}

nvfp4_status nvfp4_testing_inject_stall(int enable, unsigned long long wait_limit_ns) {
    if (!enable) {
        nvf::set_test_stall(0, 1000000000ull);
        return NVFP4_OK;
    }
    if (wait_limit_ns < 1000ull || wait_limit_ns > 1000000000ull) return NVFP4_ERR_RANGE;
    nvf::set_test_stall(1, wait_limit_ns);
    return NVFP4_OK;
}

int nvfp4_testing_plan_aligned(int streams, int M, int N, int K, int num_sms) {
    if ((streams != 1 && streams != 2) || M < 1 || M > 16 || N < 1 || K < 16 || num_sms < 1)
        return -1;
    return nvf::gemv_plan_aligned(streams, M, N, K, num_sms) ? 1 : 0;
}

int nvfp4_testing_plan_aligned_w8a16(int streams, int M, int N, int K, int num_sms) {
    if ((streams != 1 && streams != 2) || M < 1 || M > 16 || N < 1 || K < 16 || num_sms < 1)
        return -1;
    return nvf::gemv_plan_aligned(streams, M, N, K, num_sms, true) ? 1 : 0;
}

/* ------------------------------------------------------------ block-scaled FP8 */

size_t w8a16_repacked_bytes(int N, int K) {
    if (N < 1 || K < 16) return 0;
    return nvf::repacked_bytes_f8(N, K, 1);
}

size_t w8a16_repacked_gate_up_bytes(int I, int H) {
    if (I < 1 || H < 16) return 0;
    return nvf::repacked_bytes_f8(I, H, 2);
}

static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

nvfp4_status w8a16_repack(const uint8_t* codes, const float* grid, int N, int K, void* packed,
                          cudaStream_t stream) {
    if (!codes || !grid || !packed) return NVFP4_ERR_NULL;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(packed) || !aligned4(grid)) return NVFP4_ERR_ALIGN;
    return cuda_status(nvf::launch_repack_f8(codes, grid, N, K,
                                             reinterpret_cast<uint8_t*>(packed), 1, 0, stream));
}

nvfp4_status w8a16_repack_gate_up(const uint8_t* gate_codes, const float* gate_grid,
                                  const uint8_t* up_codes, const float* up_grid, int I, int H,
                                  void* packed, cudaStream_t stream) {
    if (!gate_codes || !gate_grid || !up_codes || !up_grid || !packed) return NVFP4_ERR_NULL;
    if (I < 1 || H < 16 || H % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(packed) || !aligned4(gate_grid) || !aligned4(up_grid)) return NVFP4_ERR_ALIGN;
    uint8_t* p = reinterpret_cast<uint8_t*>(packed);
    cudaError_t e = nvf::launch_repack_f8(gate_codes, gate_grid, I, H, p, 2, 0, stream);
    if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    return cuda_status(nvf::launch_repack_f8(up_codes, up_grid, I, H, p, 2, 1, stream));
}

nvfp4_status w8a16_unpack(const void* packed, int N, int K, uint8_t* codes, float* grid,
                          cudaStream_t stream) {
    if (!packed || !codes || !grid) return NVFP4_ERR_NULL;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(packed) || !aligned4(grid)) return NVFP4_ERR_ALIGN;
    return cuda_status(nvf::launch_unpack_f8(reinterpret_cast<const uint8_t*>(packed), N, K,
                                             codes, grid, stream));
}

size_t w8a16_gemv_workspace_bytes(int M, int N, int K) {
    if (M < 1 || M > kMaxTokens || N < 1 || K < 16) return 0;
    return gemv_ws_bytes(1, M, N, K, sms_for_sizing(), true);
}

nvfp4_status w8a16_gemv(const void* x, int M, int K, const void* packed_w, int N, void* y,
                        void* ws, size_t ws_bytes, cudaStream_t stream) {
    if (!x || !packed_w || !y || !ws) return NVFP4_ERR_NULL;
    if (M < 1 || M > kMaxTokens) return NVFP4_ERR_RANGE;
    if (N < 1 || K < 16 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (!aligned16(x) || !aligned16(packed_w) || !aligned16(y) || !aligned16(ws))
        return NVFP4_ERR_ALIGN;
    if (overlap(x, (size_t)M * K * 2, y, (size_t)M * N * 2)) return NVFP4_ERR_ALIAS;
    const int sms = nvf::device_sm_count();
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const size_t need = gemv_ws_bytes(1, M, N, K, sms, true);
    if (need == 0) return NVFP4_ERR_SHAPE;
    if (ws_bytes < need) return NVFP4_ERR_WORKSPACE;
    char* w = reinterpret_cast<char*>(ws);
    for (int g = 0; g < group_count(M); ++g) {
        const size_t r0 = (size_t)g * kGroupTokens;
        const cudaError_t e = nvf::launch_stream_gemv_f8(
            1, reinterpret_cast<const char*>(x) + r0 * K * 2, group_rows(M, g), K, packed_w, N, 0,
            reinterpret_cast<char*>(y) + r0 * N * 2, reinterpret_cast<int*>(w),
            reinterpret_cast<int*>(w + nvf::kStatusBytes), w + nvf::kDataOffset,
            need - nvf::kDataOffset, sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

size_t ffn_swiglu_w8a16_workspace_bytes(int M, int H, int I) {
    if (M < 1 || M > kMaxTokens || H < 16 || I < 16) return 0;
    const FfnLayout l = ffn_layout(M, H, I, sms_for_sizing(), true);
    return l.fits ? l.total : 0;
}

nvfp4_status ffn_swiglu_w8a16(const void* x, int M, int H, int I, const void* gate_up_packed,
                              const void* down_packed, nvfp4_act act, void* out, void* ws,
                              size_t ws_bytes, cudaStream_t stream) {
    if (!ws) return NVFP4_ERR_NULL;
    const int v = nvf::validate_ffn_args(x, M, H, I, gate_up_packed, down_packed, (int)act, out);
    if (v != NVFP4_OK) return (nvfp4_status)v;
    if (!aligned16(ws)) return NVFP4_ERR_ALIGN;
    const int sms = nvf::device_sm_count();
    if (sms <= 0) return NVFP4_ERR_CUDA;
    const FfnLayout l = ffn_layout(M, H, I, sms, true);
    if (!l.fits) return NVFP4_ERR_SHAPE;
    if (ws_bytes < l.total) return NVFP4_ERR_WORKSPACE;
    char* w = reinterpret_cast<char*>(ws);
    int* status = reinterpret_cast<int*>(w);
    int* counters = reinterpret_cast<int*>(w + nvf::kStatusBytes);
    char* h = w + l.h_off;
    for (int g = 0; g < group_count(M); ++g) {
        const size_t r0 = (size_t)g * kGroupTokens;
        const int mg = group_rows(M, g);
        char* hg = h + r0 * I * 2;
        cudaError_t e = nvf::launch_stream_gemv_f8(
            2, reinterpret_cast<const char*>(x) + r0 * H * 2, mg, H, gate_up_packed, I, (int)act,
            hg, status, counters, w + l.dual_off, l.dual_bytes, sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
        e = nvf::launch_stream_gemv_f8(1, hg, mg, I, down_packed, H, 0,
                                       reinterpret_cast<char*>(out) + r0 * H * 2, status,
                                       counters + l.down_cnt_off / sizeof(int), w + l.down_off,
                                       l.down_bytes, sms, true, stream);
        if (e != cudaSuccess) return NVFP4_ERR_CUDA;
    }
    return NVFP4_OK;
}

const char* nvfp4_status_string(nvfp4_status status) {
    switch (status) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_NULL: return "null pointer argument";
        case NVFP4_ERR_SHAPE: return "invalid shape (sizes must be positive, K/H/I multiples of 16)";
        case NVFP4_ERR_ALIGN: return "device pointer not 16-byte aligned";
        case NVFP4_ERR_RANGE: return "argument out of range (M outside the call's range, or an unknown enum value)";
        case NVFP4_ERR_WORKSPACE: return "workspace too small";
        case NVFP4_ERR_CUDA: return "CUDA runtime error";
        case NVFP4_ERR_TIMEOUT: return "kernel abandoned a bounded wait";
        case NVFP4_ERR_ALIAS: return "input and output buffers overlap";
    }
    return "unknown status";
}

}  // extern "C"
