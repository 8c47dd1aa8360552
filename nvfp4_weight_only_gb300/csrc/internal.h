// internal.h -- launchers shared between the kernel files and the C ABI.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime_api.h>

namespace nvf {

// quantize.cu
cudaError_t launch_quantize(const void* w, int src_bf16, int N, int K, uint8_t* codes,
                            uint8_t* scales, void* scratch, cudaStream_t s);

// repack.cu
cudaError_t launch_repack(const uint8_t* codes, const uint8_t* scales, int N, int K,
                          uint8_t* packed, int streams, int stream_index, cudaStream_t s);
cudaError_t launch_unpack(const uint8_t* packed, int N, int K, uint8_t* codes, uint8_t* scales,
                          cudaStream_t s);
// Block-scaled FP8: E4M3 bytes [N, K] + FP32 grid [ceil(N/128), ceil(K/128)]
// <-> the FP8 fragment layout (layout.h); stream_index of `streams`.
cudaError_t launch_repack_f8(const uint8_t* codes, const float* grid, int N, int K,
                             uint8_t* packed, int streams, int stream_index, cudaStream_t s);
cudaError_t launch_unpack_f8(const uint8_t* packed, int N, int K, uint8_t* codes, float* grid,
                             cudaStream_t s);

// stream_gemv.cu
// Every GEMV/FFN workspace starts with a status word area, then one fixed
// region that holds nothing but split-K counters (one int per (row block,
// tile) of each kernel).  Successful calls leave every counter at zero, and no
// call writes anything else there, so a workspace zero-filled once serves any
// sequence of shapes.  Partial sums (and the FFN's h) follow the region.
constexpr size_t kStatusBytes = 256;
constexpr size_t kCounterRegionBytes = 128u << 10;
constexpr size_t kDataOffset = kStatusBytes + kCounterRegionBytes;

// fp32 partial-sum bytes of one launch (f8: block-scaled FP8 weights), and
// the counter bytes for N rows.
size_t gemv_partial_bytes(int streams, int M, int N, int K, int num_sms, bool f8 = false);
size_t gemv_counter_bytes(int N);
// lora_deltas (streams == 2, may be null): bf16 [M, N] deltas added to the
// rounded gate and up values before the activation, g = bf16(g + delta_g);
// either entry may be null.
cudaError_t launch_stream_gemv(int streams, const void* x, int M, int K, const void* packed, int N,
                               float scale_a, float scale_b, int act, void* out, int* status,
                               int* counters, void* partials, size_t partial_bytes, int num_sms,
                               bool early_weights, cudaStream_t s,
                               const void* const* lora_deltas = nullptr);

int device_sm_count();

// stream_gemv_fp8.cu: the same kernels on block-scaled FP8 weights (repacked
// by launch_repack_f8); no per-tensor scale, no adapter deltas.
cudaError_t launch_stream_gemv_f8(int streams, const void* x, int M, int K, const void* packed,
                                  int N, int act, void* out, int* status, int* counters,
                                  void* partials, size_t partial_bytes, int num_sms,
                                  bool early_weights, cudaStream_t s);

// The testing switch's current values (set_test_stall).
unsigned long long test_wait_ns();
int test_stall();

// lora.cu: the adapter overlay, dW = B A (A [r, K], B [N, r], bf16).
constexpr int kLoraMaxRank = 64;
constexpr int kLoraMaxSplit = 32;  // K slices of the A v partial sums
// Slices the A v sums over K take (the same for both launches below).
int lora_split(int K);
// fp32 bytes of one pair's partial sums [r][split][M] (split at its maximum).
size_t lora_partial_bytes(int M, int r);
// part[p] = per-slice fp32 sums of A[p] v for each of `pairs` (1 or 2)
// matrices A[p] [r, K]; v is [M, K].
cudaError_t launch_lora_xa(const void* v, int M, int K, const void* const* A, void* const* part,
                           int pairs, int r, cudaStream_t s);
// xa = bf16(sum of the slices of part[p]) (K as given to launch_lora_xa), then
// d = bf16(B[p] xa) [M, N]: stored in out[p] (add false) or added to it as
// out[p] = bf16(out[p] + d) (add true).
cudaError_t launch_lora_delta(const void* const* part, int K, const void* const* B,
                              void* const* out, int pairs, int M, int N, int r, bool add,
                              cudaStream_t s);

// Whether the kernel's shared-memory plan for this problem has the alignment
// its accesses assume (the launcher refuses plans that do not).
bool gemv_plan_aligned(int streams, int M, int N, int K, int num_sms, bool f8 = false);

// Testing only: with stall != 0 every later GEMV/FFN launch runs with a
// producer that issues no copies and bounded waits of wait_ns, so each
// launch abandons its first wait and reports NVFP4_ERR_TIMEOUT.
void set_test_stall(int stall, unsigned long long wait_ns);

// Host-side argument checks of ffn_swiglu_nvfp4 that do not involve the
// workspace (shared by the fixed-workspace entry point); 0 = OK, else an
// nvfp4_status value.
int validate_ffn_args(const void* x, int M, int H, int I, const void* gate_up_packed,
                      const void* down_packed, int act, const void* out);

}  // namespace nvf
