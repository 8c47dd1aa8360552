// lora.cu -- the LoRA overlay of the dense FFN ("spark_model/layers/
// dense_ffn.rs", DenseFfnLayer::apply_lora_gate_up / apply_lora_down: gate and
// up take dW x before the activation, the output takes dW h after the down
// projection), dW = B A with A [r, in] and B [out, r] in bf16.
//
//   lora_xa_kernel:    xa[m][j]   = bf16(sum_k A[j][k] v[m][k])        (A v)
//   lora_delta_kernel: d[m][n]    = bf16(sum_j B[n][j] xa[m][j])       (B xa)
//                      and either stores d or base[m][n] = bf16(base + d)
//
// Both are small next to the FFN's weight stream (r rows of A, r columns of
// B); they sum in a fixed order, so results are deterministic.
#include <cuda_bf16.h>

#include <cstdint>

#include "internal.h"

namespace nvf {

constexpr int kLoraThreads = 256;
constexpr int kLoraMaxM = 16;

struct LoraXaArgs {
    const __nv_bfloat16* v;  // [M, K]
    const __nv_bfloat16* A[2];
    __nv_bfloat16* xa[2];    // [M, r]
    int M, K, r;
};

// One block per (row j of A, pair): every thread accumulates its K stride for
// all M tokens in fp32, then the block sums in a fixed order (warp butterfly,
// then the warps in index order).
__global__ void __launch_bounds__(kLoraThreads) lora_xa_kernel(const LoraXaArgs a) {
    const int j = blockIdx.x, p = blockIdx.y;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const __nv_bfloat162* arow = reinterpret_cast<const __nv_bfloat162*>(a.A[p] + (size_t)j * a.K);
    float acc[kLoraMaxM];
#pragma unroll
    for (int m = 0; m < kLoraMaxM; ++m) acc[m] = 0.0f;
    const int K2 = a.K / 2;
    for (int k2 = tid; k2 < K2; k2 += kLoraThreads) {
        const float2 w = __bfloat1622float2(arow[k2]);
#pragma unroll
        for (int m = 0; m < kLoraMaxM; ++m) {
            if (m < a.M) {
                const float2 x = __bfloat1622float2(
                    reinterpret_cast<const __nv_bfloat162*>(a.v + (size_t)m * a.K)[k2]);
                acc[m] = fmaf(w.x, x.x, acc[m]);
                acc[m] = fmaf(w.y, x.y, acc[m]);
            }
        }
    }
    __shared__ float red[kLoraThreads / 32][kLoraMaxM];
#pragma unroll
    for (int m = 0; m < kLoraMaxM; ++m) {
        float s = acc[m];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) red[warp][m] = s;
    }
    __syncthreads();
    if (tid < a.M) {
        float s = 0.0f;
#pragma unroll
        for (int w = 0; w < kLoraThreads / 32; ++w) s += red[w][tid];
        a.xa[p][(size_t)tid * a.r + j] = __float2bfloat16_rn(s);
    }
}

struct LoraDeltaArgs {
    const __nv_bfloat16* xa[2];  // [M, r]
    const __nv_bfloat16* B[2];   // [N, r]
    __nv_bfloat16* out[2];       // [M, N]: the delta, or the base it is added to
    int M, N, r, add;
};

// One thread per output row n: d = bf16(sum_j B[n][j] xa[m][j]) for every m,
// then stored (add == 0) or added to the base as bf16(base + d).  A bf16 plus
// a bf16 is exact in fp32 whenever the smaller term can move the rounding, so
// one rounding of the fp32 sum is the bf16 rounding of the exact sum.
__global__ void __launch_bounds__(kLoraThreads) lora_delta_kernel(const LoraDeltaArgs a) {
    const int p = blockIdx.y;
    __shared__ float xs[kLoraMaxM * 64];
    for (int i = threadIdx.x; i < a.M * a.r; i += kLoraThreads)
        xs[i] = __bfloat162float(a.xa[p][i]);
    __syncthreads();
    const int n = blockIdx.x * kLoraThreads + threadIdx.x;
    if (n >= a.N) return;
    const __nv_bfloat16* brow = a.B[p] + (size_t)n * a.r;
    for (int m = 0; m < a.M; ++m) {
        float s = 0.0f;
        for (int j = 0; j < a.r; ++j) s = fmaf(__bfloat162float(brow[j]), xs[m * a.r + j], s);
        const __nv_bfloat16 d = __float2bfloat16_rn(s);
        __nv_bfloat16* o = a.out[p] + (size_t)m * a.N + n;
        *o = a.add ? __float2bfloat16_rn(__bfloat162float(*o) + __bfloat162float(d)) : d;
    }
}

cudaError_t launch_lora_xa(const void* v, int M, int K, const void* const* A, void* const* xa,
                           int pairs, int r, cudaStream_t s) {
    if (M < 1 || M > kLoraMaxM || r < 1 || r > kLoraMaxRank || pairs < 1 || pairs > 2 || K % 2)
        return cudaErrorInvalidValue;
    LoraXaArgs a{};
    a.v = reinterpret_cast<const __nv_bfloat16*>(v);
    for (int p = 0; p < pairs; ++p) {
        a.A[p] = reinterpret_cast<const __nv_bfloat16*>(A[p]);
        a.xa[p] = reinterpret_cast<__nv_bfloat16*>(xa[p]);
    }
    a.M = M;
    a.K = K;
    a.r = r;
    lora_xa_kernel<<<dim3(r, pairs), kLoraThreads, 0, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_lora_delta(const void* const* xa, const void* const* B, void* const* out,
                              int pairs, int M, int N, int r, bool add, cudaStream_t s) {
    if (M < 1 || M > kLoraMaxM || r < 1 || r > kLoraMaxRank || pairs < 1 || pairs > 2 || N < 1)
        return cudaErrorInvalidValue;
    LoraDeltaArgs a{};
    for (int p = 0; p < pairs; ++p) {
        a.xa[p] = reinterpret_cast<const __nv_bfloat16*>(xa[p]);
        a.B[p] = reinterpret_cast<const __nv_bfloat16*>(B[p]);
        a.out[p] = reinterpret_cast<__nv_bfloat16*>(out[p]);
    }
    a.M = M;
    a.N = N;
    a.r = r;
    a.add = add ? 1 : 0;
    lora_delta_kernel<<<dim3((N + kLoraThreads - 1) / kLoraThreads, pairs), kLoraThreads, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace nvf
