// repack.cu -- canonical NVFP4 <-> fragment layout (a byte permutation).
//
// The principle is that of DenseFfnLayer::ensure_nvfp4_mmq_weight on
// "spark_model/layers/dense_ffn.rs": a raw shuffle of the checkpoint's E2M1
// code bytes and E4M3 scale bytes into the layout a kernel wants, with no
// numerics.  The target layout is this library's own (see layout.h).
#include "internal.h"
#include "layout.h"

namespace nvf {
namespace {

constexpr int kThreads = 256;

// Canonical position of byte p of lane `lane`'s 16 code bytes in a unit.
__device__ __forceinline__ void code_pos(int lane, int p, int& row_in_tile, int& k) {
    const int g = lane >> 2, t = lane & 3, j = p >> 2, r = p & 3;
    row_in_tile = g + 8 * (r & 1);
    k = 16 * j + 2 * t + 8 * (r >> 1);
}

// Canonical position of scale byte q (0..63) of a unit.
__device__ __forceinline__ void scale_pos(int q, int& row_in_tile, int& block) {
    const int g = q >> 3, r = q & 7;
    row_in_tile = g + 8 * (r & 1);
    block = r >> 1;
}

// One thread per (unit, lane): 16 code bytes; lanes 0..7 also 8 scale bytes.
__global__ void __launch_bounds__(kThreads) repack_kernel(const uint8_t* __restrict__ codes,
                                                          const uint8_t* __restrict__ scales,
                                                          int N, int K, int C, int RB,
                                                          uint8_t* __restrict__ out, int unit_stride,
                                                          int stream_off) {
    const long long total = (long long)RB * C * kBlockTiles * 32;
    for (long long idx = blockIdx.x * (long long)kThreads + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * kThreads) {
        const int lane = (int)(idx & 31);
        const long long unit = idx >> 5;  // ((rb*C + c)*8 + ti)
        const int ti = (int)(unit % kBlockTiles);
        const int c = (int)((unit / kBlockTiles) % C);
        const int rb = (int)(unit / ((long long)kBlockTiles * C));
        const int row0 = rb * kBlockRows + ti * kTileRows;
        uint8_t* dst = out + unit * unit_stride + stream_off;
        uint32_t w[4] = {0u, 0u, 0u, 0u};
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            int rr, kk;
            code_pos(lane, p, rr, kk);
            const int row = row0 + rr, k = c * kChunkK + kk;
            uint32_t b = 0;
            if (row < N && k < K) b = codes[(long long)row * (K / 2) + k / 2];
            w[p >> 2] |= b << (8 * (p & 3));
        }
        *reinterpret_cast<uint4*>(dst + 16 * lane) = make_uint4(w[0], w[1], w[2], w[3]);
        if (lane < 8) {
            uint32_t sw[2] = {0u, 0u};
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                int rr, jb;
                scale_pos(lane * 8 + q8, rr, jb);
                const int row = row0 + rr, blk = c * 4 + jb;
                uint32_t b = 0;
                if (row < N && blk < K / 16) b = scales[(long long)row * (K / 16) + blk];
                sw[q8 >> 2] |= b << (8 * (q8 & 3));
            }
            *reinterpret_cast<uint2*>(dst + kUnitCodeBytes + 8 * lane) = make_uint2(sw[0], sw[1]);
        }
    }
    // Make the repacked weight visible GPU-wide before this block exits: the
    // GEMV kernels may start streaming it as soon as every block has exited.
    __threadfence();
}

__global__ void __launch_bounds__(kThreads) unpack_kernel(const uint8_t* __restrict__ in, int N,
                                                          int K, int C, int RB,
                                                          uint8_t* __restrict__ codes,
                                                          uint8_t* __restrict__ scales) {
    const long long total = (long long)RB * C * kBlockTiles * 32;
    for (long long idx = blockIdx.x * (long long)kThreads + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * kThreads) {
        const int lane = (int)(idx & 31);
        const long long unit = idx >> 5;
        const int ti = (int)(unit % kBlockTiles);
        const int c = (int)((unit / kBlockTiles) % C);
        const int rb = (int)(unit / ((long long)kBlockTiles * C));
        const int row0 = rb * kBlockRows + ti * kTileRows;
        const uint8_t* src = in + unit * kUnitBytes;
        const uint4 v = *reinterpret_cast<const uint4*>(src + 16 * lane);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int p = 0; p < 16; ++p) {
            int rr, kk;
            code_pos(lane, p, rr, kk);
            const int row = row0 + rr, k = c * kChunkK + kk;
            if (row < N && k < K)
                codes[(long long)row * (K / 2) + k / 2] = (uint8_t)(w[p >> 2] >> (8 * (p & 3)));
        }
        if (lane < 8) {
            const uint2 s = *reinterpret_cast<const uint2*>(src + kUnitCodeBytes + 8 * lane);
            const uint32_t sw[2] = {s.x, s.y};
#pragma unroll
            for (int q8 = 0; q8 < 8; ++q8) {
                int rr, jb;
                scale_pos(lane * 8 + q8, rr, jb);
                const int row = row0 + rr, blk = c * 4 + jb;
                if (row < N && blk < K / 16)
                    scales[(long long)row * (K / 16) + blk] = (uint8_t)(sw[q8 >> 2] >> (8 * (q8 & 3)));
            }
        }
    }
}

int grid_for(long long total) {
    long long want = (total + kThreads - 1) / kThreads;
    long long cap = 16LL * device_sm_count();
    if (want < 1) want = 1;
    return (int)(want < cap ? want : cap);
}

}  // namespace

cudaError_t launch_repack(const uint8_t* codes, const uint8_t* scales, int N, int K,
                          uint8_t* packed, int streams, int stream_index, cudaStream_t s) {
    const Geometry g = geometry(N, K);
    const long long total = (long long)g.RB * g.C * kBlockTiles * 32;
    repack_kernel<<<grid_for(total), kThreads, 0, s>>>(codes, scales, N, K, g.C, g.RB, packed,
                                                       kUnitBytes * streams,
                                                       kUnitBytes * stream_index);
    return cudaGetLastError();
}

cudaError_t launch_unpack(const uint8_t* packed, int N, int K, uint8_t* codes, uint8_t* scales,
                          cudaStream_t s) {
    const Geometry g = geometry(N, K);
    const long long total = (long long)g.RB * g.C * kBlockTiles * 32;
    unpack_kernel<<<grid_for(total), kThreads, 0, s>>>(packed, N, K, g.C, g.RB, codes, scales);
    return cudaGetLastError();
}

}  // namespace nvf
