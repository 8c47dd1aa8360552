// stream_gemv.cu -- the NVFP4 decode GEMV family for GB300 (sm_103a).
//
// One kernel template serves
//   * the standalone projection  y = bf16(scale2 * W x)               (NS = 1)
//   * the dual gate+up projection with the activation epilogue        (NS = 2)
//       h = bf16( act(bf16(scale_g * Wg x)) * bf16(scale_u * Wu x) )
// for M = 1..8 (NT = 1) or 9..16 (NT = 2) token rows.  The pages' decode path
// ("spark_model/layers/dense_ffn.rs", DenseFfnLayer::forward: dual gate+up
// GEMV, activation, down GEMV; forward_km: each weight read once for all M
// rows) is the prior art; the structure here is GB300's own:
//
//   * persistent grid, one CTA per SM: 8 consumer warps + 1 producer warp;
//   * the producer streams contiguous runs of repacked weight units through a
//     ring of shared-memory stages with the bulk-copy (TMA) engine, completion
//     tracked by mbarriers;
//   * each consumer warp owns one 16-row tile of every 128-row block and turns
//     its 16 code bytes per 64-K chunk into exact f16 weights
//     (E2M1 -> f16 by cvt, times the E4M3 scale by an exact f16 multiply) fed
//     as the A operand of mma.sync m16n8k16 with fp32 accumulators; the token
//     rows (x) are the B operand, staged once per CTA range in shared memory
//     as f16 after a per-token power-of-two scaling (exact; keeps any finite
//     bf16 input inside the f16 range);
//   * work = (row block, chunk) steps in row-major order, split into equal
//     contiguous ranges; a row block whose K range spans several ranges is
//     finished by the last range to arrive (atomic counter), which sums the
//     fp32 partial slots in range order, so results are deterministic.
//
// Every mbarrier wait is bounded (device status word + abort flag), and a CTA
// drains its own bulk copies before it exits.
#include <cuda_bf16.h>

#include "device_util.cuh"
#include "internal.h"
#include "layout.h"

namespace nvf {

constexpr int kConsumerWarps = kBlockTiles;  // one warp per 16-row tile
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kThreads = kConsumerThreads + 32;
constexpr int kSmemMax = 227 * 1024;
constexpr int kXBudget = 96 * 1024;
constexpr int kRingBudget = 96 * 1024;
constexpr int kMaxStages = 16;
constexpr int kMiscBytes = 512;
constexpr int kConsumerBarrier = 1;

struct Plan {
    int NS, NT, G;
    int RB, C, SRB;
    long long L;
    int grid, R;
    long long Pmax;
    int xcap, stage_bytes, stages, s_max, slot_floats;
    int x_off, bar_off, misc_off;
    size_t smem;
    size_t counters_off, partials_off, total;
};

static Plan make_plan(int NS, int M, int N, int K, int num_sms) {
    Plan p{};
    p.NS = NS;
    p.NT = (M <= 8) ? 1 : 2;
    p.G = (p.NT == 1) ? 1 : 2;
    const Geometry g = geometry(N, K);
    p.RB = g.RB;
    p.C = g.C;
    p.SRB = (int)ceil_div(p.RB, p.G);
    p.L = (long long)p.SRB * p.C;
    const int xchunk = p.NT * 1024;
    const int xcap_max = kXBudget / xchunk;
    p.grid = num_sms > 0 ? num_sms : 1;
    if (p.L < p.grid) p.grid = (int)p.L;
    for (int rpc = 1;; ++rpc) {
        long long R = (long long)p.grid * rpc;
        if (R > p.L) R = p.L;
        p.R = (int)R;
        p.Pmax = ceil_div(p.L, p.R);
        const long long need = p.Pmax < p.C ? p.Pmax : p.C;
        if (need <= xcap_max || p.R == p.L) break;
    }
    p.xcap = (int)(p.Pmax < p.C ? p.Pmax : p.C);
    p.stage_bytes = p.G * kBlockTiles * kUnitBytes * NS;
    const int x_bytes = p.xcap * xchunk;
    int ring = kSmemMax - x_bytes - kMiscBytes - 16 * kMaxStages;
    if (ring > kRingBudget) ring = kRingBudget;
    p.stages = ring / p.stage_bytes;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) p.stages = 2;
    p.x_off = (int)(ceil_div((long long)p.stages * p.stage_bytes, 128) * 128);
    p.bar_off = p.x_off + x_bytes;
    p.misc_off = p.bar_off + 16 * p.stages;
    p.smem = (size_t)p.misc_off + kMiscBytes;
    long long smax = ceil_div(p.Pmax, p.C) + 1;
    if (smax > p.SRB) smax = p.SRB;
    p.s_max = (int)smax;
    p.slot_floats = p.G * kBlockTiles * NS * kTileRows * (p.NT * 8);
    p.counters_off = 0;
    p.partials_off = (size_t)ceil_div((long long)p.SRB * 4, 256) * 256;
    p.total = p.partials_off + (size_t)p.R * p.s_max * p.slot_floats * sizeof(float);
    return p;
}

struct KArgs {
    const __nv_bfloat16* x;
    const uint8_t* blob;
    __nv_bfloat16* out;
    float* partials;
    int* counters;
    int* status;
    long long L;
    int M, K, N, C, RB, R, grid;
    int stages, stage_bytes, x_off, bar_off, misc_off, s_max;
    float scale_a, scale_b;
    int act;
};

__device__ __forceinline__ long long range_start(const KArgs& a, long long r) {
    return r * a.L / a.R;
}

// Index of the range that contains step s (inverse of range_start).
__device__ __forceinline__ int range_of(const KArgs& a, long long s) {
    return (int)(((s + 1) * (long long)a.R - 1) / a.L);
}

// SiLU(t) = t / (1 + e^-t).  GeLU (tanh form) 0.5 t (1 + tanh(z)) with
// z = sqrt(2/pi) (t + 0.044715 t^3) is evaluated through the identity
// 1 + tanh(z) = 2 / (1 + e^-2z), i.e. t / (1 + e^-2z): the same full-accuracy
// expf as SiLU and no cancellation in 1 + tanh(z) for negative t.
__device__ __forceinline__ float act_fn(int act, float t) {
    if (act == 0) return t / (1.0f + expf(-t));
    const float two_c = 1.5957691216057308f;  // 2 * sqrt(2/pi)
    return t / (1.0f + expf(-two_c * (t + 0.044715f * t * t * t)));
}

template <int NS>
__device__ __forceinline__ void store_output(const KArgs& a, int row, int token, float va,
                                             float vb) {
    if (NS == 1) {
        a.out[(size_t)token * a.N + row] = __float2bfloat16_rn(va * a.scale_a);
    } else {
        const float gb = __bfloat162float(__float2bfloat16_rn(va * a.scale_a));
        const float ub = __bfloat162float(__float2bfloat16_rn(vb * a.scale_b));
        a.out[(size_t)token * a.N + row] = __float2bfloat16_rn(act_fn(a.act, gb) * ub);
    }
}

// Stage the token rows for chunks c_start .. c_start+nx-1 (mod C) into shared
// memory as f16 B fragments, after scaling token m by tok_scale[m] = 2^e_m.
template <int NT>
__device__ void stage_x(const KArgs& a, uint8_t* xs, int c_start, int nx, float* tok_scale,
                        float* tok_unscale, unsigned* amax_u) {
    const int ctid = threadIdx.x, lane = ctid & 31;
    if (ctid < 16) amax_u[ctid] = 0u;
    named_barrier_sync(kConsumerBarrier, kConsumerThreads);
    const int groups = nx * 8;  // groups of 8 consecutive K elements
    for (int m = 0; m < a.M; ++m) {
        const __nv_bfloat16* xr = a.x + (size_t)m * a.K;
        float mx = 0.0f;
        for (int q = ctid; q < groups; q += kConsumerThreads) {
            int c = c_start + (q >> 3);
            if (c >= a.C) c -= a.C;
            const int k = c * kChunkK + (q & 7) * 8;
            if (k < a.K) {
                const uint4 v = __ldg(reinterpret_cast<const uint4*>(xr + k));
                const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    mx = fmaxf(mx, fabsf(__uint_as_float(w[i] << 16)));
                    mx = fmaxf(mx, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
                }
            }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        if (lane == 0 && mx > 0.0f) atomicMax(&amax_u[m], __float_as_uint(mx));
    }
    named_barrier_sync(kConsumerBarrier, kConsumerThreads);
    if (ctid < 16) {
        const float am = __uint_as_float(amax_u[ctid]);
        int e = 0;
        if (am > 0.0f) {
            int ex;
            frexpf(am, &ex);  // am < 2^ex, so am * 2^(15-ex) lies in [2^14, 2^15)
            e = 15 - ex;
            e = e < -100 ? -100 : (e > 100 ? 100 : e);
        }
        tok_scale[ctid] = __int_as_float((127 + e) << 23);
        tok_unscale[ctid] = __int_as_float((127 - e) << 23);
    }
    named_barrier_sync(kConsumerBarrier, kConsumerThreads);
    const int items = nx * NT * 64;
    for (int it = ctid; it < items; it += kConsumerThreads) {
        const int ln = it & 31, h = (it >> 5) & 1, q = it >> 6;
        const int nt = q % NT, ci = q / NT;
        int c = c_start + ci;
        if (c >= a.C) c -= a.C;
        const int token = nt * 8 + (ln >> 2), tq = ln & 3;
        uint32_t o[4] = {0u, 0u, 0u, 0u};
        if (token < a.M) {
            const float sc = tok_scale[token];
            const __nv_bfloat16* xr = a.x + (size_t)token * a.K;
#pragma unroll
            for (int jj = 0; jj < 2; ++jj) {
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    const int k = c * kChunkK + 16 * (2 * h + jj) + 2 * tq + 8 * hf;
                    if (k < a.K) {
                        const uint32_t pr = __ldg(reinterpret_cast<const unsigned*>(xr + k));
                        const __half2 hv = __floats2half2_rn(__uint_as_float(pr << 16) * sc,
                                                             __uint_as_float(pr & 0xFFFF0000u) * sc);
                        o[2 * jj + hf] = *reinterpret_cast<const uint32_t*>(&hv);
                    }
                }
            }
        }
        *reinterpret_cast<uint4*>(xs + ((ci * NT + nt) * 2 + h) * 512 + ln * 16) =
            make_uint4(o[0], o[1], o[2], o[3]);
    }
    named_barrier_sync(kConsumerBarrier, kConsumerThreads);
}

template <int NS, int NT>
__global__ void __launch_bounds__(kThreads, 1) stream_gemv_kernel(const KArgs a) {
    constexpr int G = (NT == 1) ? 1 : 2;
    constexpr int UB = kUnitBytes * NS;
    constexpr int TOK = NT * 8;
    constexpr int SLOT = G * kBlockTiles * NS * kTileRows * TOK;

    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t ring_s = smem_addr(smem);
    uint8_t* xs = smem + a.x_off;
    const uint32_t full0 = smem_addr(smem + a.bar_off);
    const uint32_t empty0 = full0 + 8u * a.stages;
    float* tok_scale = reinterpret_cast<float*>(smem + a.misc_off);
    float* tok_unscale = tok_scale + 16;
    unsigned* amax_u = reinterpret_cast<unsigned*>(tok_unscale + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(amax_u + 16);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, kConsumerWarps);
        }
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == kConsumerWarps) {
        // ---------------- producer: one lane issues every bulk copy ----------------
        if (lane != 0) return;
        long long i = 0;
        bool ok = true;
        for (int r = blockIdx.x; r < a.R; r += a.grid) {
            const long long s0 = range_start(a, r), s1 = range_start(a, r + 1);
            for (long long s = s0; s < s1; ++s, ++i) {
                const int st = (int)(i % a.stages);
                const uint32_t ph = (uint32_t)((i / a.stages) & 1);
                if (ok && !mbar_wait_bounded(empty0 + 8u * st, ph ^ 1u, abort_flag)) {
                    ok = false;
                    *abort_flag = 1;
                    atomicOr(a.status, 1);
                }
                if (!ok) continue;
                const int srb = (int)(s / a.C), c = (int)(s % a.C);
                const int rb0 = srb * G;
                const int np = (a.RB - rb0) < G ? (a.RB - rb0) : G;
                mbar_arrive_expect_tx(full0 + 8u * st, (uint32_t)(np * kBlockTiles * UB));
                for (int gi = 0; gi < np; ++gi) {
                    bulk_copy_g2s(ring_s + (uint32_t)(st * a.stage_bytes + gi * kBlockTiles * UB),
                                  a.blob + ((size_t)(rb0 + gi) * a.C + c) * kBlockTiles * UB,
                                  (uint32_t)(kBlockTiles * UB), full0 + 8u * st);
                }
            }
        }
        // Drain: wait (bounded) until every copy issued by this CTA has landed.
        const int zero = 0;
        const long long first = i > a.stages ? i - a.stages : 0;
        for (long long j = first; j < i; ++j)
            mbar_wait_bounded(full0 + 8u * (int)(j % a.stages), (uint32_t)((j / a.stages) & 1),
                              &zero);
        return;
    }

    // ---------------- consumers ----------------
    const int g = lane >> 2, tq = lane & 3;
    float acc[G][NS][NT][2][4];
#pragma unroll
    for (int gi = 0; gi < G; ++gi)
#pragma unroll
        for (int si = 0; si < NS; ++si)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int ch = 0; ch < 2; ++ch)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[gi][si][nt][ch][e] = 0.0f;

    long long i = 0;
    bool ok = true;
    for (int r = blockIdx.x; r < a.R; r += a.grid) {
        const long long s0 = range_start(a, r), s1 = range_start(a, r + 1);
        const int c_start = (int)(s0 % a.C);
        const int nx = (int)((s1 - s0) < a.C ? (s1 - s0) : a.C);
        named_barrier_sync(kConsumerBarrier, kConsumerThreads);  // x buffer is free
        stage_x<NT>(a, xs, c_start, nx, tok_scale, tok_unscale, amax_u);
        float unscale[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e) unscale[nt][e] = tok_unscale[nt * 8 + 2 * tq + e];

        for (long long s = s0; s < s1; ++s, ++i) {
            const int st = (int)(i % a.stages);
            const uint32_t ph = (uint32_t)((i / a.stages) & 1);
            if (ok && !mbar_wait_bounded(full0 + 8u * st, ph, abort_flag)) {
                ok = false;
                *abort_flag = 1;
                atomicOr(a.status, 1);
            }
            const int srb = (int)(s / a.C), c = (int)(s % a.C);
            if (ok) {
                int ci = c - c_start;
                if (ci < 0) ci += a.C;
                uint32_t b[NT][8];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int h = 0; h < 2; ++h) {
                        const uint4 v = *reinterpret_cast<const uint4*>(
                            xs + ((ci * NT + nt) * 2 + h) * 512 + lane * 16);
                        b[nt][4 * h + 0] = v.x;
                        b[nt][4 * h + 1] = v.y;
                        b[nt][4 * h + 2] = v.z;
                        b[nt][4 * h + 3] = v.w;
                    }
                const uint8_t* stage = smem + (size_t)st * a.stage_bytes;
#pragma unroll
                for (int gi = 0; gi < G; ++gi) {
                    if (G > 1 && srb * G + gi >= a.RB) continue;
                    const uint8_t* unit = stage + (gi * kBlockTiles + warp) * UB;
#pragma unroll
                    for (int si = 0; si < NS; ++si) {
                        const uint4 cw =
                            *reinterpret_cast<const uint4*>(unit + si * kUnitBytes + lane * 16);
                        const uint2 sw = *reinterpret_cast<const uint2*>(
                            unit + si * kUnitBytes + kUnitCodeBytes + g * 8);
                        const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            uint32_t a0, a1, a2, a3;
                            e2m1x8_to_f16x2x4(cws[j], a0, a1, a2, a3);
                            const uint32_t sp = ((j < 2 ? sw.x : sw.y) >> (16 * (j & 1))) & 0xFFFFu;
                            const uint32_t s2 = e4m3x2_to_f16x2(sp);
                            const uint32_t sg = prmt(s2, s2, 0x1010u);
                            const uint32_t sg8 = prmt(s2, s2, 0x3232u);
                            a0 = hmul2(a0, sg);
                            a2 = hmul2(a2, sg);
                            a1 = hmul2(a1, sg8);
                            a3 = hmul2(a3, sg8);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt)
                                mma_f16_16816(acc[gi][si][nt][j & 1], a0, a1, a2, a3,
                                              b[nt][2 * j], b[nt][2 * j + 1]);
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty0 + 8u * st);

            if (c != a.C - 1 && s != s1 - 1) continue;
            // ---------------- end of a segment of row block srb ----------------
            const long long seg_lo = s0 > (long long)srb * a.C ? s0 : (long long)srb * a.C;
            const bool full_cover = (seg_lo == (long long)srb * a.C) && (c == a.C - 1);
            float v[G][NS][NT][4];
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
#pragma unroll
                for (int si = 0; si < NS; ++si)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            v[gi][si][nt][e] = (acc[gi][si][nt][0][e] + acc[gi][si][nt][1][e]) *
                                               unscale[nt][e & 1];
                            acc[gi][si][nt][0][e] = 0.0f;
                            acc[gi][si][nt][1][e] = 0.0f;
                        }
            if (full_cover) {
#pragma unroll
                for (int gi = 0; gi < G; ++gi)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int row = (srb * G + gi) * kBlockRows + warp * kTileRows + g +
                                            8 * (e >> 1);
                            const int token = nt * 8 + 2 * tq + (e & 1);
                            if (ok && row < a.N && token < a.M)
                                store_output<NS>(a, row, token, v[gi][0][nt][e],
                                                 v[gi][NS - 1][nt][e]);
                        }
                continue;
            }
            // Partial: write this range's slot, then let the last range finish.
            const int si_slot = srb - (int)(s0 / a.C);
            float* slot = a.partials + ((size_t)r * a.s_max + si_slot) * SLOT;
#pragma unroll
            for (int gi = 0; gi < G; ++gi)
#pragma unroll
                for (int si = 0; si < NS; ++si)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const int idx =
                                (((gi * kBlockTiles + warp) * NS + si) * kTileRows + g + 8 * (e >> 1)) *
                                    TOK +
                                nt * 8 + 2 * tq + (e & 1);
                            slot[idx] = v[gi][si][nt][e];
                        }
            __threadfence();
            named_barrier_sync(kConsumerBarrier, kConsumerThreads);
            const long long p_lo = (long long)srb * a.C;
            const int r_first = range_of(a, p_lo), r_last = range_of(a, p_lo + a.C - 1);
            if (threadIdx.x == 0) {
                const int nparts = r_last - r_first + 1;
                const int old = atomicAdd(&a.counters[srb], 1);
                const int last = (old == nparts - 1) ? 1 : 0;
                if (last) {
                    a.counters[srb] = 0;  // ready for the next call
                    __threadfence();
                }
                *last_flag = last;
            }
            named_barrier_sync(kConsumerBarrier, kConsumerThreads);
            if (*last_flag) {
                const int elems = G * kBlockTiles * kTileRows * a.M;
                for (int e = threadIdx.x; e < elems; e += kConsumerThreads) {
                    const int token = e % a.M;
                    const int rest = e / a.M;
                    const int row16 = rest % kTileRows;
                    const int tis = rest / kTileRows;  // tile within the super row block
                    const int row = srb * G * kBlockRows + tis * kTileRows + row16;
                    if (row >= a.N) continue;
                    float sum[NS];
#pragma unroll
                    for (int si = 0; si < NS; ++si) sum[si] = 0.0f;
                    for (int rr = r_first; rr <= r_last; ++rr) {
                        const int ss = srb - (int)(range_start(a, rr) / a.C);
                        const float* sl = a.partials + ((size_t)rr * a.s_max + ss) * SLOT;
#pragma unroll
                        for (int si = 0; si < NS; ++si)
                            sum[si] += __ldcg(sl + ((tis * NS + si) * kTileRows + row16) * TOK + token);
                    }
                    if (ok) store_output<NS>(a, row, token, sum[0], sum[NS - 1]);
                }
            }
            named_barrier_sync(kConsumerBarrier, kConsumerThreads);
        }
    }
}

int device_sm_count() {
    static int cache[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        cudaGetLastError();
        return 0;
    }
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev] = n;
    }
    return cache[dev];
}

size_t gemv_scratch_bytes(int streams, int M, int N, int K, int num_sms) {
    return make_plan(streams, M, N, K, num_sms).total;
}

template <int NS, int NT>
static cudaError_t launch_t(const Plan& p, const KArgs& a, cudaStream_t s) {
    static bool attr_done[64] = {false};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(stream_gemv_kernel<NS, NT>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    stream_gemv_kernel<NS, NT><<<p.grid, kThreads, p.smem, s>>>(a);
    return cudaGetLastError();
}

cudaError_t launch_stream_gemv(int streams, const void* x, int M, int K, const void* packed, int N,
                               float scale_a, float scale_b, int act, void* out, int* status,
                               void* scratch, size_t scratch_bytes, int num_sms, cudaStream_t s) {
    const Plan p = make_plan(streams, M, N, K, num_sms);
    if (scratch_bytes < p.total) return cudaErrorInvalidValue;
    KArgs a;
    a.x = reinterpret_cast<const __nv_bfloat16*>(x);
    a.blob = reinterpret_cast<const uint8_t*>(packed);
    a.out = reinterpret_cast<__nv_bfloat16*>(out);
    a.counters = reinterpret_cast<int*>(reinterpret_cast<char*>(scratch) + p.counters_off);
    a.partials = reinterpret_cast<float*>(reinterpret_cast<char*>(scratch) + p.partials_off);
    a.status = status;
    a.L = p.L;
    a.M = M;
    a.K = K;
    a.N = N;
    a.C = p.C;
    a.RB = p.RB;
    a.R = p.R;
    a.grid = p.grid;
    a.stages = p.stages;
    a.stage_bytes = p.stage_bytes;
    a.x_off = p.x_off;
    a.bar_off = p.bar_off;
    a.misc_off = p.misc_off;
    a.s_max = p.s_max;
    a.scale_a = scale_a;
    a.scale_b = scale_b;
    a.act = act;
    if (streams == 1)
        return p.NT == 1 ? launch_t<1, 1>(p, a, s) : launch_t<1, 2>(p, a, s);
    return p.NT == 1 ? launch_t<2, 1>(p, a, s) : launch_t<2, 2>(p, a, s);
}

}  // namespace nvf
