// quantize.cu -- load-time NVFP4 quantisation of an fp32/bf16 weight.
//
// Follows "spark_model/weight_loader/qwen35_dense.rs", load_layers: a global
// absmax kernel, then a quantize kernel (quantize_to_nvfp4).  The arithmetic
// is IEEE fp32 in a fixed order, with the rounding done by the hardware's
// round-to-nearest-even saturating converts:
//   scale2 = amax / 2688 (1 when amax == 0)
//   s      = E4M3(bamax / 6 / scale2)            per 16-element block
//   code   = E2M1(w / (E4M3value(s) * scale2))   per element, sign kept
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "internal.h"

namespace nvf {
namespace {

constexpr int kThreads = 256;

__device__ __forceinline__ float bf16_bits_to_f32(uint32_t b) { return __uint_as_float(b << 16); }

__device__ __forceinline__ void load16(const void* w, int src_bf16, size_t block, float (&v)[16]) {
    if (src_bf16) {
        const uint4* p = reinterpret_cast<const uint4*>(w) + block * 2;
        uint4 q[2] = {__ldg(p), __ldg(p + 1)};
        const uint32_t* u = reinterpret_cast<const uint32_t*>(q);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            v[2 * i] = bf16_bits_to_f32(u[i] & 0xFFFFu);
            v[2 * i + 1] = bf16_bits_to_f32(u[i] >> 16);
        }
    } else {
        const float4* p = reinterpret_cast<const float4*>(w) + block * 4;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float4 q = __ldg(p + i);
            v[4 * i] = q.x;
            v[4 * i + 1] = q.y;
            v[4 * i + 2] = q.z;
            v[4 * i + 3] = q.w;
        }
    }
}

// max |W| over all 16-element blocks, as fp32 bits (non-negative floats order
// like their bit patterns), folded into *amax_bits with atomicMax.
__global__ void __launch_bounds__(kThreads) absmax_kernel(const void* w, int src_bf16,
                                                          size_t nblocks, unsigned* amax_bits) {
    float m = 0.0f;
    for (size_t b = blockIdx.x * (size_t)kThreads + threadIdx.x; b < nblocks;
         b += (size_t)gridDim.x * kThreads) {
        float v[16];
        load16(w, src_bf16, b, v);
#pragma unroll
        for (int i = 0; i < 16; ++i) m = fmaxf(m, fabsf(v[i]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    __shared__ float wm[kThreads / 32];
    if ((threadIdx.x & 31) == 0) wm[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x == 0) {
        float r = 0.0f;
        for (int i = 0; i < kThreads / 32; ++i) r = fmaxf(r, wm[i]);
        atomicMax(amax_bits, __float_as_uint(r));
    }
}

// One thread per 16-element block b: canonical codes at bytes [8b, 8b+8),
// scale at byte b (the blocks of a row are contiguous in both arrays).
__global__ void __launch_bounds__(kThreads) quantize_kernel(const void* w, int src_bf16,
                                                            size_t nblocks, uint8_t* codes,
                                                            uint8_t* scales,
                                                            const unsigned* amax_bits,
                                                            float* scale2_out) {
    const float amax = __uint_as_float(*amax_bits);
    const float scale2 = (amax == 0.0f) ? 1.0f : __fdiv_rn(amax, 2688.0f);
    if (blockIdx.x == 0 && threadIdx.x == 0) *scale2_out = scale2;
    for (size_t b = blockIdx.x * (size_t)kThreads + threadIdx.x; b < nblocks;
         b += (size_t)gridDim.x * kThreads) {
        float v[16];
        load16(w, src_bf16, b, v);
        float bamax = 0.0f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bamax = fmaxf(bamax, fabsf(v[i]));
        const float t = __fdiv_rn(__fdiv_rn(bamax, 6.0f), scale2);
        const uint32_t s = f32_to_e4m3(t);
        const float denom = __fmul_rn(e4m3_to_f32(s), scale2);
        uint32_t word[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            uint32_t c;
            if (s == 0u) {
                c = signbit(v[i]) ? 8u : 0u;
            } else {
                const float q = __fdiv_rn(v[i], denom);
                c = f32_to_e2m1(q) | (signbit(q) ? 8u : 0u);
            }
            word[i >> 3] |= c << (4 * (i & 7));
        }
        *reinterpret_cast<uint2*>(codes + 8 * b) = make_uint2(word[0], word[1]);
        scales[b] = (uint8_t)s;
    }
    // Make the codes visible GPU-wide before this block exits: the GEMV kernels
    // may be launched as soon as every block of this grid has exited.
    __threadfence();
}

}  // namespace

cudaError_t launch_quantize(const void* w, int src_bf16, int N, int K, uint8_t* codes,
                            uint8_t* scales, void* scratch, cudaStream_t s) {
    unsigned* amax = reinterpret_cast<unsigned*>(scratch);
    float* scale2 = reinterpret_cast<float*>(reinterpret_cast<char*>(scratch) + 4);
    const size_t nblocks = (size_t)N * (K / 16);
    cudaError_t e = cudaMemsetAsync(amax, 0, 4, s);
    if (e != cudaSuccess) return e;
    const int sms = device_sm_count();
    long long want = (long long)((nblocks + kThreads - 1) / kThreads);
    int grid = (int)(want < 8LL * sms ? (want > 0 ? want : 1) : 8LL * sms);
    absmax_kernel<<<grid, kThreads, 0, s>>>(w, src_bf16, nblocks, amax);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    quantize_kernel<<<grid, kThreads, 0, s>>>(w, src_bf16, nblocks, codes, scales, amax, scale2);
    return cudaGetLastError();
}

}  // namespace nvf
