// lora.cu -- the LoRA overlay of the dense FFN ("spark_model/layers/
// dense_ffn.rs", DenseFfnLayer::apply_lora_gate_up / apply_lora_down: gate and
// up take dW x before the activation, the output takes dW h after the down
// projection), dW = B A with A [r, in] and B [out, r] in bf16.
//
//   lora_xa_partial_kernel: part[j][s][m] = sum over K slice s of A[j][k] v[m][k]
//   lora_delta_kernel:      xa[m][j] = bf16(sum_s part[j][s][m])         (A v)
//                           d[m][n]  = bf16(sum_j B[n][j] xa[m][j])      (B xa)
//                           then stores d or base[m][n] = bf16(base + d)
//
// Both are small next to the FFN's weight stream (r rows of A, r columns of
// B), so what costs time is latency: the K sum is cut into slices that each
// CTA covers with one vector load per thread, every thread issues its loads
// before the first multiply, and code that each thread runs once is kept
// small (its first execution fetches every instruction line from L2).  Both
// kernels are launched as programmatic dependents: they load their adapter
// matrix (never written by the kernel before them) before waiting for that
// kernel, and read v, the partials and the base only after it.  Sums run in a
// fixed order, so results are deterministic.
#include <cuda_bf16.h>

#include <cstdint>

#include "internal.h"

namespace nvf {

constexpr int kLoraThreads = 256;
constexpr int kLoraMaxM = 16;

int lora_split(int K) {
    const int kv = (K % 8 == 0) ? K / 8 : K / 2;  // vectors of the partial kernel
    const int s = (kv + kLoraThreads - 1) / kLoraThreads;
    return s < 1 ? 1 : (s > kLoraMaxSplit ? kLoraMaxSplit : s);
}

size_t lora_partial_bytes(int M, int r) {
    return (size_t)M * r * kLoraMaxSplit * sizeof(float);
}

struct LoraXaArgs {
    const __nv_bfloat16* v;  // [M, K]
    const __nv_bfloat16* A[2];
    float* part[2];          // [r][split][M]
    int M, K, split;
};

template <typename Vec>
__device__ __forceinline__ float dot_acc(const Vec& w, const Vec& x, float acc) {
    constexpr int kPairs = sizeof(Vec) / 4;
    const uint32_t* wp = reinterpret_cast<const uint32_t*>(&w);
    const uint32_t* xp = reinterpret_cast<const uint32_t*>(&x);
#pragma unroll
    for (int i = 0; i < kPairs; ++i) {
        __nv_bfloat162 wb, xb;
        *reinterpret_cast<uint32_t*>(&wb) = wp[i];
        *reinterpret_cast<uint32_t*>(&xb) = xp[i];
        const float2 wf = __bfloat1622float2(wb), xf = __bfloat1622float2(xb);
        acc = fmaf(wf.x, xf.x, acc);
        acc = fmaf(wf.y, xf.y, acc);
    }
    return acc;
}

// One block per (K slice s, row j of A, pair p).  Vec is uint4 (8 bf16) when
// K % 8 == 0, else uint32_t (2 bf16).  A thread loads its A vector and the M
// matching token vectors together, then multiplies; the block sums each token
// in a fixed order (warp butterfly, then the warps in index order).
template <typename Vec>
__global__ void __launch_bounds__(kLoraThreads) lora_xa_partial_kernel(const LoraXaArgs a) {
    constexpr int kElems = sizeof(Vec) / 2;
    const int s = blockIdx.x, j = blockIdx.y, p = blockIdx.z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kv = a.K / kElems;
    const int per = (kv + a.split - 1) / a.split;
    const int v0 = s * per;
    const int v1 = min(kv, v0 + per);
    const __nv_bfloat16* A = p ? a.A[1] : a.A[0];  // no dynamic index into the parameters
    const Vec* arow = reinterpret_cast<const Vec*>(A + (size_t)j * a.K);
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int i0 = v0 + tid;
    Vec w0{};
    if (i0 < v1) w0 = arow[i0];
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float acc[kLoraMaxM];
#pragma unroll
    for (int m = 0; m < kLoraMaxM; ++m) acc[m] = 0.0f;
    for (int i = i0; i < v1; i += kLoraThreads) {
        const Vec w = i == i0 ? w0 : arow[i];
        Vec xv[kLoraMaxM];
#pragma unroll
        for (int m = 0; m < kLoraMaxM; ++m)
            if (m < a.M) xv[m] = reinterpret_cast<const Vec*>(a.v + (size_t)m * a.K)[i];
#pragma unroll
        for (int m = 0; m < kLoraMaxM; ++m)
            if (m < a.M) acc[m] = dot_acc(w, xv[m], acc[m]);
    }
    __shared__ float red[kLoraThreads / 32][kLoraMaxM];
#pragma unroll
    for (int m = 0; m < kLoraMaxM; ++m) {
        if (m < a.M) {
            float t = acc[m];
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
            if (lane == 0) red[warp][m] = t;
        }
    }
    __syncthreads();
    if (tid < a.M) {
        float t = 0.0f;
#pragma unroll
        for (int w = 0; w < kLoraThreads / 32; ++w) t += red[w][tid];
        (p ? a.part[1] : a.part[0])[((size_t)j * a.split + s) * a.M + tid] = t;
    }
}

struct LoraDeltaArgs {
    const float* part[2];        // [r][split][M]
    const __nv_bfloat16* B[2];   // [N, r]
    __nv_bfloat16* out[2];       // [M, N]: the delta, or the base it is added to
    int M, N, r, split, add;
};

// xs[m*r + j] = bf16(sum of part[j][s][m] over the slices s, in slice order),
// read from L2; the loads of one sum go out eight at a time.
__device__ __forceinline__ void fill_xa(const float* part, int M, int r, int split, float* xs) {
    for (int i = threadIdx.x; i < M * r; i += kLoraThreads) {
        const int m = i / r, j = i - m * r;
        const float* q = part + (size_t)j * split * M + m;
        float t = 0.0f;
#pragma unroll 8
        for (int sl = 0; sl < split; ++sl) t += __ldcg(q + (size_t)sl * M);
        xs[i] = __bfloat162float(__float2bfloat16_rn(t));
    }
}

// Row n of every token's delta: d = bf16(sum_j B[n][j] xa[m][j]), stored at
// ocol[m*N] (add false) or added to the base there as bf16(base + d).  bv: the
// row of B (r % 8 == 0), else brow is read.  base0: token 0's base, loaded by
// the caller ahead of time.  The token loop stays rolled: this code runs once
// per row, so its size, not its issue count, is what costs (every first
// execution of an instruction line is a fetch from L2).
template <bool kVec>
__device__ __forceinline__ void delta_row(const uint4 (&bv)[kLoraMaxRank / 8],
                                          const __nv_bfloat16* brow, const float* xs, int M,
                                          int r, int N, bool add, float base0,
                                          __nv_bfloat16* ocol) {
    for (int m = 0; m < M; ++m) {
        __nv_bfloat16* const o = ocol + (size_t)m * N;
        const float base = !add ? 0.0f : m == 0 ? base0 : __bfloat162float(*o);
        const float* xm = xs + m * r;
        float acc = 0.0f;
        if constexpr (kVec) {
            const int nv = r / 8;
#pragma unroll
            for (int c = 0; c < kLoraMaxRank / 8; ++c) {
                if (c < nv) {
                    const uint32_t words[4] = {bv[c].x, bv[c].y, bv[c].z, bv[c].w};
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const uint32_t wd = words[e >> 1];  // element 2i in the low half
                        const float bj =
                            __uint_as_float((e & 1) ? (wd & 0xffff0000u) : (wd << 16));
                        acc = fmaf(bj, xm[8 * c + e], acc);
                    }
                }
            }
        } else {
#pragma unroll 4
            for (int j = 0; j < r; ++j) acc = fmaf(__bfloat162float(brow[j]), xm[j], acc);
        }
        const __nv_bfloat16 d = __float2bfloat16_rn(acc);
        *o = add ? __float2bfloat16_rn(base + __bfloat162float(d)) : d;
    }
}

// One thread per output row n.  Each thread loads its whole B row (r % 8 == 0)
// before the wait on the preceding kernel, and token 0's base value right
// after it; the block meanwhile completes xa = bf16(sum of the slice
// partials, in slice order) into shared memory.  The thread then forms
// d = bf16(sum_j B[n][j] xa[m][j]) for every m and stores it (add == 0) or
// adds it to the base as bf16(base + d).  A bf16 plus a bf16 is exact in fp32
// whenever the smaller term can move the rounding, so one rounding of the
// fp32 sum is the bf16 rounding of the exact sum.
template <bool kVec>
__global__ void __launch_bounds__(kLoraThreads) lora_delta_kernel(const LoraDeltaArgs a) {
    const int p = blockIdx.y;
    const int n = blockIdx.x * kLoraThreads + threadIdx.x;
    const bool live = n < a.N;
    const __nv_bfloat16* brow = (p ? a.B[1] : a.B[0]) + (size_t)(live ? n : 0) * a.r;
    __nv_bfloat16* const ocol = (p ? a.out[1] : a.out[0]) + n;
    constexpr int kMaxV = kLoraMaxRank / 8;
    uint4 bv[kMaxV];
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if constexpr (kVec) {  // r % 8 == 0: at most 8 16-byte loads
        const int nv = a.r / 8;
#pragma unroll
        for (int c = 0; c < kMaxV; ++c)
            if (live && c < nv) bv[c] = reinterpret_cast<const uint4*>(brow)[c];
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");
    const float base0 = live && a.add ? __bfloat162float(ocol[0]) : 0.0f;
    __shared__ float xs[kLoraMaxM * kLoraMaxRank];  // [m][j]
    fill_xa(p ? a.part[1] : a.part[0], a.M, a.r, a.split, xs);
    __syncthreads();
    if (live) delta_row<kVec>(bv, brow, xs, a.M, a.r, a.N, a.add != 0, base0, ocol);
}

// A launch that may begin while the preceding kernel on the stream finishes
// (programmatic stream serialisation); the kernel orders itself after that
// kernel with griddepcontrol.wait.
template <typename Args>
cudaError_t launch_dependent(void (*kernel)(Args), dim3 grid, cudaStream_t s, const Args& a) {
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kLoraThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, a);
}

cudaError_t launch_lora_xa(const void* v, int M, int K, const void* const* A, void* const* part,
                           int pairs, int r, cudaStream_t s) {
    if (M < 1 || M > kLoraMaxM || r < 1 || r > kLoraMaxRank || pairs < 1 || pairs > 2 || K < 2 ||
        K % 2)
        return cudaErrorInvalidValue;
    LoraXaArgs a{};
    a.v = reinterpret_cast<const __nv_bfloat16*>(v);
    for (int p = 0; p < pairs; ++p) {
        a.A[p] = reinterpret_cast<const __nv_bfloat16*>(A[p]);
        a.part[p] = reinterpret_cast<float*>(part[p]);
    }
    a.M = M;
    a.K = K;
    a.split = lora_split(K);
    const dim3 grid(a.split, r, pairs);
    return K % 8 == 0 ? launch_dependent(lora_xa_partial_kernel<uint4>, grid, s, a)
                      : launch_dependent(lora_xa_partial_kernel<uint32_t>, grid, s, a);
}

cudaError_t launch_lora_delta(const void* const* part, int K, const void* const* B,
                              void* const* out, int pairs, int M, int N, int r, bool add,
                              cudaStream_t s) {
    if (M < 1 || M > kLoraMaxM || r < 1 || r > kLoraMaxRank || pairs < 1 || pairs > 2 || N < 1 ||
        K < 2)
        return cudaErrorInvalidValue;
    LoraDeltaArgs a{};
    for (int p = 0; p < pairs; ++p) {
        a.part[p] = reinterpret_cast<const float*>(part[p]);
        a.B[p] = reinterpret_cast<const __nv_bfloat16*>(B[p]);
        a.out[p] = reinterpret_cast<__nv_bfloat16*>(out[p]);
    }
    a.M = M;
    a.N = N;
    a.r = r;
    a.split = lora_split(K);
    a.add = add ? 1 : 0;
    const dim3 grid((N + kLoraThreads - 1) / kLoraThreads, pairs);
    return r % 8 == 0 ? launch_dependent(lora_delta_kernel<true>, grid, s, a)
                      : launch_dependent(lora_delta_kernel<false>, grid, s, a);
}

}  // namespace nvf
