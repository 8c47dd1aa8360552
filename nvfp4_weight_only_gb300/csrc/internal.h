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

// stream_gemv.cu
// Byte layout of a GEMV/FFN workspace: [status word area][...].
constexpr size_t kStatusBytes = 256;

size_t gemv_scratch_bytes(int streams, int M, int N, int K, int num_sms);
cudaError_t launch_stream_gemv(int streams, const void* x, int M, int K, const void* packed, int N,
                               float scale_a, float scale_b, int act, void* out, int* status,
                               void* scratch, size_t scratch_bytes, int num_sms, bool early_weights,
                               cudaStream_t s);

int device_sm_count();

}  // namespace nvf
