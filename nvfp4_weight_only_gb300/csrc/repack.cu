// repack.cu -- canonical NVFP4 / block-scaled FP8 <-> fragment layouts (byte
// permutations; the FP8 grid entries are copied, one per tile and chunk).
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

// ---- block-scaled FP8 (layout.h)

// Canonical position of byte p (0..31) of lane `lane`'s 32 code bytes in a tile.
__device__ __forceinline__ void f8_code_pos(int lane, int p, int& row_in_tile, int& k) {
    const int g = lane >> 2, t = lane & 3, j = p >> 3, r = (p >> 1) & 3, e = p & 1;
    row_in_tile = g + 8 * (r & 1);
    k = 16 * j + 2 * t + 8 * (r >> 1) + e;
}

// One thread per (group, tile, lane): 32 code bytes of one stream; lane 0
// also writes the tile's scale.  Group g = rb*C + c.
__global__ void __launch_bounds__(kThreads) repack_f8_kernel(const uint8_t* __restrict__ codes,
                                                             const float* __restrict__ grid,
                                                             int N, int K, int C, int RB,
                                                             uint8_t* __restrict__ out,
                                                             int streams, int si) {
    const long long total = (long long)RB * C * kBlockTiles * 32;
    const int KB = (K + 127) / 128;
    const long long gbytes = (long long)streams * (kBlockTiles * kF8TileBytes + kBlockTiles * 4);
    for (long long idx = blockIdx.x * (long long)kThreads + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * kThreads) {
        const int lane = (int)(idx & 31);
        const int ti = (int)((idx >> 5) % kBlockTiles);
        const long long grp = (idx >> 5) / kBlockTiles;
        const int c = (int)(grp % C);
        const int rb = (int)(grp / C);
        const int row0 = rb * kBlockRows + ti * kTileRows;
        uint8_t* gdst = out + grp * gbytes;
        uint32_t w[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            int rr, kk;
            f8_code_pos(lane, p, rr, kk);
            const int row = row0 + rr, k = c * kChunkK + kk;
            uint32_t b = 0;
            if (row < N && k < K) b = codes[(long long)row * K + k];
            w[p >> 2] |= b << (8 * (p & 3));
        }
        uint8_t* dst = gdst + (ti * streams + si) * kF8TileBytes + 32 * lane;
        *reinterpret_cast<uint4*>(dst) = make_uint4(w[0], w[1], w[2], w[3]);
        *reinterpret_cast<uint4*>(dst + 16) = make_uint4(w[4], w[5], w[6], w[7]);
        if (lane == 0) {
            const int k0 = c * kChunkK;
            const float sc = (row0 < N && k0 < K) ? grid[(long long)(row0 / 128) * KB + k0 / 128]
                                                  : 0.0f;
            *reinterpret_cast<float*>(gdst + (long long)streams * kBlockTiles * kF8TileBytes +
                                      4 * (ti * streams + si)) = sc;
        }
    }
    // visible GPU-wide before the block exits (the GEMV may stream it next)
    __threadfence();
}

// Inverse of repack_f8_kernel for one stream (streams == 1): codes, and each
// grid entry from the first tile and chunk of its 128 x 128 block.
__global__ void __launch_bounds__(kThreads) unpack_f8_kernel(const uint8_t* __restrict__ in,
                                                             int N, int K, int C, int RB,
                                                             uint8_t* __restrict__ codes,
                                                             float* __restrict__ grid) {
    const long long total = (long long)RB * C * kBlockTiles * 32;
    const int KB = (K + 127) / 128;
    const long long gbytes = kBlockTiles * kF8TileBytes + kBlockTiles * 4;
    for (long long idx = blockIdx.x * (long long)kThreads + threadIdx.x; idx < total;
         idx += (long long)gridDim.x * kThreads) {
        const int lane = (int)(idx & 31);
        const int ti = (int)((idx >> 5) % kBlockTiles);
        const long long grp = (idx >> 5) / kBlockTiles;
        const int c = (int)(grp % C);
        const int rb = (int)(grp / C);
        const int row0 = rb * kBlockRows + ti * kTileRows;
        const uint8_t* gsrc = in + grp * gbytes;
        const uint8_t* src = gsrc + ti * kF8TileBytes + 32 * lane;
        const uint4 v0 = *reinterpret_cast<const uint4*>(src);
        const uint4 v1 = *reinterpret_cast<const uint4*>(src + 16);
        const uint32_t w[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
        for (int p = 0; p < 32; ++p) {
            int rr, kk;
            f8_code_pos(lane, p, rr, kk);
            const int row = row0 + rr, k = c * kChunkK + kk;
            if (row < N && k < K) codes[(long long)row * K + k] = (uint8_t)(w[p >> 2] >> (8 * (p & 3)));
        }
        const int k0 = c * kChunkK;
        if (lane == 0 && row0 < N && k0 < K && row0 % 128 == 0 && k0 % 128 == 0)
            grid[(long long)(row0 / 128) * KB + k0 / 128] =
                *reinterpret_cast<const float*>(gsrc + kBlockTiles * kF8TileBytes + 4 * ti);
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

cudaError_t launch_repack_f8(const uint8_t* codes, const float* grid, int N, int K,
                             uint8_t* packed, int streams, int stream_index, cudaStream_t s) {
    const Geometry g = geometry(N, K);
    const long long total = (long long)g.RB * g.C * kBlockTiles * 32;
    repack_f8_kernel<<<grid_for(total), kThreads, 0, s>>>(codes, grid, N, K, g.C, g.RB, packed,
                                                          streams, stream_index);
    return cudaGetLastError();
}

cudaError_t launch_unpack_f8(const uint8_t* packed, int N, int K, uint8_t* codes, float* grid,
                             cudaStream_t s) {
    const Geometry g = geometry(N, K);
    const long long total = (long long)g.RB * g.C * kBlockTiles * 32;
    unpack_f8_kernel<<<grid_for(total), kThreads, 0, s>>>(packed, N, K, g.C, g.RB, codes, grid);
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
