// layout.h -- geometry of the repacked ("fragment") NVFP4 weight layout.
//
// The canonical NVFP4 projection (packed E2M1 codes [N, K/2], element 2j in the
// low nibble of byte j, plus E4M3 scales [N, K/16]; "spark_model/layers/
// dense_ffn.rs", doc comment of DenseFfnLayer::ensure_int8_weight) is permuted
// byte by byte, with no change to any value, into units that one warp feeds
// straight into mma.sync.m16n8k16 A fragments:
//
//   unit   = 16 weight rows x 64 K elements = 512 code bytes + 64 scale bytes
//   codes  : lane L = 4g + t (g = L/4, t = L%4) owns bytes [16L, 16L+16);
//            byte 4j + r (j = k16 block 0..3 of the chunk, r = 0..3) holds the
//            canonical byte of row g + 8*(r&1) at K pair 16j + 2t + 8*(r>>1),
//            i.e. exactly the A-fragment registers a0..a3 of block j.
//   scales : byte 8g + 2j + (r&1) holds the E4M3 scale of row g + 8*(r&1),
//            block j.
//   row block = 16 units of consecutive 16-row tiles (256 rows), for one chunk;
//   order  = [row block][chunk][tile in block], so one row block's data for
//            a run of chunks is one contiguous byte range.
//
// Rows are zero-padded to a multiple of 256 and K to a multiple of 256 (four
// chunks; zero codes with zero scales contribute nothing).  The gate/up variant stores the
// gate unit and the up unit of the same tile back to back (1152 bytes), so the
// dual kernel streams both projections of its rows from one range.
#pragma once
#include <cstddef>
#include <cstdint>

namespace nvf {

constexpr int kTileRows = 16;
constexpr int kBlockTiles = 16;
constexpr int kBlockRows = kTileRows * kBlockTiles;  // 256
constexpr int kChunkK = 64;
constexpr int kChunkAlign = 4;  // chunks per row block are a multiple of this
constexpr int kUnitCodeBytes = 512;
constexpr int kUnitScaleBytes = 64;
constexpr int kUnitBytes = kUnitCodeBytes + kUnitScaleBytes;  // 576

inline __host__ __device__ long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

struct Geometry {
    int N, K;    // logical rows, columns
    int RB;      // row blocks of 256 rows
    int C;       // chunks of 64 K elements (a multiple of kChunkAlign)
};

inline __host__ __device__ Geometry geometry(int N, int K) {
    Geometry g;
    g.N = N;
    g.K = K;
    g.RB = (int)ceil_div(N, kBlockRows);
    g.C = (int)(ceil_div(ceil_div(K, kChunkK), kChunkAlign) * kChunkAlign);
    return g;
}

// Bytes of one repacked projection (streams = 1) or gate/up pair (streams = 2).
inline size_t repacked_bytes(int N, int K, int streams) {
    Geometry g = geometry(N, K);
    return (size_t)g.RB * g.C * kBlockTiles * kUnitBytes * streams;
}

// ---- block-scaled FP8 (the dense-FFN page's DenseFfnWeightsFp8: E4M3 bytes
// [N, K] row-major and an FP32 grid [ceil(N/128), ceil(K/128)], weight =
// e4m3(q[n][k]) * grid[n/128][k/128]) in the same row blocks and chunks:
//
//   tile   = 16 rows x 64 K = 1024 code bytes; lane L = 4g + t owns bytes
//            [32L, 32L+32), byte 8j + 2r + e (j = k16 block 0..3, r = 0..3,
//            e = 0, 1) holding the canonical byte of row g + 8*(r&1) at
//            K = 16j + 2t + 8*(r>>1) + e: registers a0..a3 of block j, two
//            E4M3 per f16x2 register;
//   group  = one (row block, chunk): the 16 tiles' codes (tile-major, the
//            streams of a tile back to back), then one fp32 per tile and
//            stream: the grid entry of the tile's 128-row block at the
//            chunk's 128-K block (every 16-row tile lies inside one 128-row
//            block, and every 64-K chunk inside one 128-K block);
//   order  = [row block][chunk], like the NVFP4 layout.
// Padding rows and K carry zero codes and a zero scale.
constexpr int kF8TileBytes = 1024;

inline size_t f8_group_bytes_host(int streams) {
    return (size_t)streams * (kBlockTiles * kF8TileBytes + kBlockTiles * 4);
}

// Bytes of one repacked FP8 projection (streams = 1) or gate/up pair (2).
inline size_t repacked_bytes_f8(int N, int K, int streams) {
    Geometry g = geometry(N, K);
    return (size_t)g.RB * g.C * f8_group_bytes_host(streams);
}

}  // namespace nvf
