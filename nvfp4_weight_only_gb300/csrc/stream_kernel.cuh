// stream_kernel.cuh -- the decode GEMV kernel template for GB300 (sm_103a),
// shared by the NVFP4 launcher (stream_gemv.cu) and the block-scaled FP8
// launcher (stream_gemv_fp8.cu), which compile in parallel.
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
//   * persistent grid, one CTA of 16 warps per SM; warp w owns the 16-row
//     tile w of every 256-row block of the repacked weight (layout.h);
//   * weights stream through a ring of shared-memory stages filled by the
//     bulk-copy (TMA) engine: one lane of a producer warpgroup issues every
//     copy, a "full" mbarrier per stage completes on the copy's bytes and an
//     "empty" mbarrier on the 512 consumer lanes' release, so the consumers
//     never issue copies and never wait for one another;
//   * per k16 block a warp turns its 4 code bytes into exact f16 A fragments
//     (one cvt per E2M1 pair), runs mma.sync m16n8k16 against the token rows
//     (B operand, staged once per range in shared memory as f16 after an exact
//     per-token power-of-two scaling that keeps any finite bf16 row inside the
//     f16 range), and applies the two E4M3 row scales to the fp32 block sums;
//   * work = (row block, step of chunks) in row-major order, split into equal
//     contiguous ranges; a row block whose K range spans several ranges is
//     finished either by the last range to arrive (atomic counter) or, where
//     the final sums are heavy (use_coop), by all ranges that end in it, each
//     taking a share of the outputs (coop_finish).  Either way every output
//     sums the fp32 partials in range order, so results are deterministic.
//
// The block-scaled FP8 weights of the dense-FFN page's native FP8 arm
// (DenseFfnWeightsFp8: E4M3 bytes [N, K] with an FP32 scale per 128 x 128
// block) run through the same grid, ring, token staging and split-K machinery
// (template flag F8): per k16 block a warp converts 8 code bytes into four
// exact f16 A fragments (two E4M3 per cvt), the chunk's four MMAs chain into
// one fp32 tile, and the tile's block scale is applied to it with FFMAs.
//
// Every mbarrier wait is bounded (device status word + abort flag), and a CTA
// that gave up waits (bounded) for its own bulk copies before it exits.
#pragma once
#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include "device_util.cuh"
#include "internal.h"
#include "layout.h"

namespace nvf {

constexpr int kWarps = kBlockTiles;  // consumer warps: one per 16-row tile of a row block
constexpr int kConsumerThreads = kWarps * 32;
// + one producer warpgroup, whose first lane issues every bulk copy.  The
// register file is re-split at entry (setmaxnreg): launched at 96 per thread
// (640 x 96 = 61440), the producer warpgroup drops to 24 and the consumers
// rise to 112 (512 x 112 + 128 x 24 = 60416 <= 61440).
constexpr int kThreads = kConsumerThreads + 128;
constexpr int kLaunchRegs = 96, kProducerRegs = 24, kConsumerRegs = 112;
static_assert(kConsumerThreads * kConsumerRegs + 128 * kProducerRegs <= kThreads * kLaunchRegs,
              "setmaxnreg split exceeds the launch allocation");
constexpr int kSmemMax = 227 * 1024;
constexpr int kXBudget = 96 * 1024;
constexpr int kRingBudget = 200 * 1024;
constexpr int kMaxStages = 8;
constexpr int kMinStages = 3;  // fewest ring stages a widened token area may leave
// Up to this many tokens (one MMA token group) the split-K partials are
// element-major: each output element's parts are contiguous, and the last
// range reads them in 16-byte vectors.  With two token groups (M > 8) each
// range writes one contiguous slot instead.
constexpr int kElemMajorMaxM = 8;
static_assert(kElemMajorMaxM >= 2, "the diagonal layout (M <= 2) writes element-major partials");
// The misc area: token scales and amax (0..), the abort flag, the per-stage
// copy counts (kMiscIssuesOff), then the publication area (kMiscPubOff):
// kMaxEvents "segment stored" mbarriers (count kWarps), kMaxEvents
// "published" mbarriers (count 1) and the returned counts, kWarps per event.
constexpr int kMaxEvents = 8;
constexpr int kMiscIssuesOff = 256;  // per-stage copy counts (kMaxStages ints)
constexpr int kMiscPubOff = 512;
constexpr int kMiscBytes = kMiscPubOff + 16 * kMaxEvents + 4 * 16 * kMaxEvents;
// Chunks (of 64 K elements) summed in plain fp32 before the sum is folded into
// the exact hi/lo pair.
constexpr int kFoldChunks = 8;
// Weight units (16 rows x 64 K) each warp handles per pipeline step; a step
// spans kUnitsPerStep / streams chunks (a divisor of kChunkAlign).
#ifndef NVF_UNITS_PER_STEP
#define NVF_UNITS_PER_STEP 4
#endif
constexpr int kUnitsPerStep = NVF_UNITS_PER_STEP;
// FP8 tiles are 1024 bytes per chunk: two units per warp per step keep a stage
// near the NVFP4 one (32.9 KB).
constexpr int kF8UnitsPerStep = 2;

// Bytes of one (row block, chunk) group of the weight layout for `streams`.
__host__ __device__ constexpr int group_bytes(int streams, bool f8) {
    return f8 ? streams * (kBlockTiles * kF8TileBytes + kBlockTiles * 4)
              : kBlockTiles * kUnitBytes * streams;
}

struct Plan {
    int NS, NT, RB, C, CS;  // CS: steps per row block
    long long L;            // steps in the whole problem
    int grid, R;
    long long Pmax;         // steps per range (max)
    int cps, xcap, x_stride, stage_bytes, stages, s_max, slot_floats;
    int part_stride;  // M <= kElemMajorMaxM: element-major partials, parts per element
                      // padded to 4 (0: range-major slots)
    int x_off, bar_off, cnt_off, misc_off;
    size_t smem;
    size_t counter_bytes;  // split-K counters: one int per (row block, tile)
    size_t total;          // fp32 partial sums
};

static Plan make_plan(int NS, int M, int N, int K, int num_sms, bool f8) {
    Plan p{};
    p.NS = NS;
    p.NT = (M <= 8) ? 1 : 2;
    p.cps = (f8 ? kF8UnitsPerStep : kUnitsPerStep) / NS;
    const Geometry g = geometry(N, K);
    p.RB = g.RB;
    p.C = g.C;
    p.CS = p.C / p.cps;
    p.L = (long long)p.RB * p.CS;
    // x lives in shared memory as f16, token-major: per token 128 bytes per
    // chunk (+16 bytes of row padding that keeps the B-fragment loads free of
    // bank conflicts).
    // NVFP4 with M <= 2 uses the diagonal layout: 1024 bytes per chunk for
    // both tokens.
    const bool diag = M <= 2 && !f8;
    auto xcap_for = [&](int budget) {
        return diag ? budget / 1024 : (budget - 16 * M) / (128 * M);
    };
    int xcap_max = xcap_for(kXBudget);
    p.grid = num_sms > 0 ? num_sms : 1;
    if (p.L < p.grid) p.grid = (int)p.L;
    {
        // One range per CTA saves a second staging, tail and set of partials;
        // when the token rows of such a range just miss the budget, let them
        // take ring space as long as kMinStages stages remain.
        const long long need1 = ceil_div(p.L, p.grid) * p.cps < p.C ? ceil_div(p.L, p.grid) * p.cps
                                                                     : p.C;
        const int stage = p.cps * group_bytes(NS, f8);
        const int wide = kSmemMax - kMiscBytes - 32 * kMaxStages - 512 - kMinStages * stage;
        if (need1 > xcap_max && need1 <= xcap_for(wide)) xcap_max = xcap_for(wide);
    }
    for (int rpc = 1;; ++rpc) {
        long long R = (long long)p.grid * rpc;
        if (R > p.L) R = p.L;
        p.R = (int)R;
        p.Pmax = ceil_div(p.L, p.R);
        const long long need = p.Pmax * p.cps < p.C ? p.Pmax * p.cps : p.C;
        if (need <= xcap_max || p.R == p.L) break;
    }
    p.xcap = (int)(p.Pmax * p.cps < p.C ? p.Pmax * p.cps : p.C);
    p.x_stride = diag ? 0 : p.xcap * 128 + 16;
    p.stage_bytes = p.cps * group_bytes(NS, f8);
    const int x_bytes = diag ? p.xcap * 1024 : M * p.x_stride;
    int ring = kSmemMax - x_bytes - kMiscBytes - 32 * kMaxStages - 256;
    if (ring > kRingBudget) ring = kRingBudget;
    p.stages = ring / p.stage_bytes;
    if (p.stages > kMaxStages) p.stages = kMaxStages;
    if (p.stages < 2) p.stages = 2;
    p.x_off = (int)(ceil_div((long long)p.stages * p.stage_bytes, 128) * 128);
    p.bar_off = (int)(ceil_div((long long)p.x_off + x_bytes, 16) * 16);
    p.cnt_off = p.bar_off + 8 * p.stages;
    p.misc_off = (int)(ceil_div((long long)p.cnt_off + 8LL * p.stages, 128) * 128);
    p.smem = (size_t)p.misc_off + kMiscBytes;
    long long smax = ceil_div(p.Pmax, p.CS) + 1;
    if (smax > p.RB) smax = p.RB;
    p.s_max = (int)smax;
    p.slot_floats = kBlockTiles * NS * kTileRows * M;
    p.counter_bytes = (size_t)ceil_div((long long)p.RB * kBlockTiles * 4, 256) * 256;
    p.part_stride = 0;
    if (M <= kElemMajorMaxM) {
        // element-major: the parts of one output element are contiguous, so the
        // last range to arrive reads them with a few 16-byte loads
        long long most = 1;
        for (long long rb = 0; rb < p.RB; ++rb) {
            const long long lo = rb * p.CS, hi = lo + p.CS - 1;
            const long long parts = ((hi + 1) * p.R - 1) / p.L - ((lo + 1) * p.R - 1) / p.L + 1;
            if (parts > most) most = parts;
        }
        p.part_stride = (int)ceil_div(most, 4) * 4;
        p.total = (size_t)p.RB * p.slot_floats * (size_t)p.part_stride * sizeof(float);
    } else {
        p.total = (size_t)p.R * p.s_max * p.slot_floats * sizeof(float);
    }
    return p;
}

// Whether the shared-memory carve-up has the alignment every access assumes:
// bulk-copy destinations (ring stages) and 16-byte vector loads (token rows,
// x_stride) on 16 bytes, mbarriers on 8, the misc area (float, int and
// mbarrier words, read as vectors nowhere today) on 128, and the whole inside
// the per-CTA limit.  The launcher refuses a plan that fails it.
static bool plan_aligned(const Plan& p) {
    return p.stage_bytes % 128 == 0 && p.x_off % 128 == 0 && p.x_stride % 16 == 0 &&
           p.bar_off % 16 == 0 && p.cnt_off % 8 == 0 && p.misc_off % 128 == 0 &&
           kMiscIssuesOff % 16 == 0 && kMiscPubOff % 16 == 0 && p.smem <= (size_t)kSmemMax &&
           p.stages >= 2 && p.stages <= kMaxStages;
}

// Division by a fixed divisor d >= 1 of numerators below 2^32, by a multiply:
// with m = floor((2^64 - 1) / d) + 1, floor(n / d) = high 64 bits of n * m for
// every n < 2^32 (the product overshoots n / d by less than n / 2^64 < 1 / d,
// which never crosses the next integer).  d == 1 is passed through.
struct FastDiv {
    unsigned long long m;
    unsigned d;
    static FastDiv make(unsigned d) {
        FastDiv f;
        f.d = d;
        f.m = d > 1 ? ~0ull / d + 1 : 0;
        return f;
    }
    __device__ __forceinline__ unsigned div(unsigned n) const {
        return d > 1 ? (unsigned)__umul64hi((unsigned long long)n, m) : n;
    }
};

struct KArgs {
    const __nv_bfloat16* x;
    const uint8_t* blob;
    __nv_bfloat16* out;
    float* partials;
    int* counters;
    int* status;
    long long L;
    int M, K, N, C, CS, RB, R, grid;
    int stages, stage_bytes, x_off, x_stride, bar_off, cnt_off, misc_off, s_max;
    int part_stride;  // element-major partials: parts per element, padded to 4 (0: slots)
    float scale_a, scale_b;
    int act;
    int early_weights;  // stream weights before waiting on the preceding kernel
    // Longest bounded wait (ns).  `stall` (testing only) makes the producer
    // issue no copies, so the consumers' first wait runs out after wait_ns.
    unsigned long long wait_ns;
    int stall;
    // L * R < 2^32: the range arithmetic below runs on FastDiv multiplies
    int fast;
    FastDiv div_R, div_L, div_CS;
    // adapter deltas for gate and up (bf16 [M, N], null when absent)
    const __nv_bfloat16* lora_dg;
    const __nv_bfloat16* lora_du;
};

__device__ __forceinline__ long long range_start(const KArgs& a, long long r) {
    if (a.fast) return a.div_R.div((unsigned)(r * a.L));
    return r * a.L / a.R;
}

// Index of the range that contains step q (inverse of range_start).
__device__ __forceinline__ int range_of(const KArgs& a, long long q) {
    if (a.fast) return (int)a.div_L.div((unsigned)((q + 1) * a.R - 1));
    return (int)(((q + 1) * (long long)a.R - 1) / a.L);
}

// Row block of step q.
__device__ __forceinline__ int rb_of_step(const KArgs& a, int q) {
    return a.fast ? (int)a.div_CS.div((unsigned)q) : q / a.CS;
}

// Position in this CTA's step sequence: ranges blockIdx.x, +grid, +2*grid, ...
struct StepCursor {
    int r, q, q_end, rb, cb;  // range, step, range end, row block, step within row block
    __device__ __forceinline__ void start_range(const KArgs& a) {
        if (r < a.R) {
            q = (int)range_start(a, r);
            q_end = (int)range_start(a, r + 1);
            rb = rb_of_step(a, q);
            cb = q - rb * a.CS;
        }
    }
    __device__ __forceinline__ void init(const KArgs& a) {
        r = blockIdx.x;
        start_range(a);
    }
    __device__ __forceinline__ bool valid(const KArgs& a) const { return r < a.R; }
    __device__ __forceinline__ void advance(const KArgs& a) {
        if (r >= a.R) return;
        ++q;
        if (++cb == a.CS) {
            cb = 0;
            ++rb;
        }
        if (q == q_end) {
            r += a.grid;
            start_range(a);
        }
    }
};

// h = bf16(act(g) * u) for bf16-valued g, u, with act(t) = t * sigmoid(y):
// SiLU has y = t; GeLU (tanh form) 0.5 t (1 + tanh(z)) has y = 2z,
// z = sqrt(2/pi) (t + 0.044715 t^3), by the identity 1 + tanh(z) = 2 sigmoid(2z).
// sigmoid(y) is 1 / (1 + e^-y) for y >= 0 and e^y / (1 + e^y) for y < 0, so
// neither branch overflows and the far negative tail keeps its (subnormal)
// value instead of collapsing to zero.  When 1 + e^-y rounds to exactly 1 in
// fp32, act(g) = g to fp32 precision while the exact act(g) is slightly
// smaller in magnitude; g*u is then exact in fp32, and an exact bf16 tie of
// it must round toward zero, as the exact product (strictly inside) does.
// Not inlined: the last range's epilogue runs it for several elements per lane
// right after the stream, and one shared copy of its code costs one round of
// instruction fetch misses instead of one per unrolled element.
__device__ __forceinline__ __nv_bfloat16 gated_product_inline(int act, float g, float u) {
    const float y = (act == 0) ? g : 1.5957691216057308f * (g + 0.044715f * g * g * g);
    if (y < 0.0f) {
        const float e = expf(y);
        return __float2bfloat16_rn(g * (e / (1.0f + e)) * u);
    }
    const float den = 1.0f + expf(-y);
    const float p = (g / den) * u;
    if (den == 1.0f) {
        const uint32_t bits = __float_as_uint(p);
        if ((bits & 0xFFFFu) == 0x8000u) return __ushort_as_bfloat16((unsigned short)(bits >> 16));
    }
    return __float2bfloat16_rn(p);
}

static __device__ __noinline__ __nv_bfloat16 gated_product(int act, float g, float u) {
    return gated_product_inline(act, g, u);
}

template <int NS>
__device__ __forceinline__ void store_output(const KArgs& a, int row, int token, float va,
                                             float vb) {
    if (NS == 1) {
        a.out[(size_t)token * a.N + row] = __float2bfloat16_rn(va * a.scale_a);
    } else {
        float gb = __bfloat162float(__float2bfloat16_rn(va * a.scale_a));
        float ub = __bfloat162float(__float2bfloat16_rn(vb * a.scale_b));
        // adapter deltas land on the rounded projections, before the
        // activation; a bf16 plus a bf16 rounds once, exactly, through fp32
        if (a.lora_dg != nullptr)
            gb = __bfloat162float(__float2bfloat16_rn(
                gb + __bfloat162float(a.lora_dg[(size_t)token * a.N + row])));
        if (a.lora_du != nullptr)
            ub = __bfloat162float(__float2bfloat16_rn(
                ub + __bfloat162float(a.lora_du[(size_t)token * a.N + row])));
        a.out[(size_t)token * a.N + row] = gated_product(a.act, gb, ub);
    }
}

// Error-free addition (Knuth's TwoSum): hi + lo gains b exactly.
__device__ __forceinline__ void two_sum_acc(float& hi, float& lo, float b) {
    const float s = hi + b;
    const float bb = s - hi;
    const float err = (hi - (s - bb)) + (b - bb);
    hi = s;
    lo += err;
}

// Barrier over the consumer warps only (the producer warp never joins).
__device__ __forceinline__ void consumer_sync() { named_barrier_sync(1, kConsumerThreads); }

// The exponent e of a token with absolute maximum amax (bit pattern): amax *
// 2^e lies in [2^14, 2^15), clamped to +-100; 0 for an all-zero token.
__device__ __forceinline__ int token_exponent(unsigned amax_bits) {
    const float am = __uint_as_float(amax_bits);
    int e = 0;
    if (am > 0.0f) {
        int ex;
        frexpf(am, &ex);  // am < 2^ex, so am * 2^(15-ex) lies in [2^14, 2^15)
        e = 15 - ex;
        e = e < -100 ? -100 : (e > 100 ? 100 : e);
    }
    return e;
}

__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// bf16 pair -> f16 pair scaled by sc = 2^e (exact for the range kept).
__device__ __forceinline__ uint32_t scale_pair_to_f16(uint32_t pr, float sc) {
    const __half2 hv = __floats2half2_rn(__uint_as_float(pr << 16) * sc,
                                         __uint_as_float(pr & 0xFFFF0000u) * sc);
    return *reinterpret_cast<const uint32_t*>(&hv);
}

__device__ __forceinline__ void track_amax(float& mx, const uint4& v) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        mx = fmaxf(mx, fabsf(__uint_as_float(w[i] << 16)));
        mx = fmaxf(mx, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
    }
}

// The 16-byte group q (8 k values) of token m's rows for chunks c_start ...
// (mod C), or zeros past K.
__device__ __forceinline__ uint4 load_x_group(const KArgs& a, int m, int c_start, int q) {
    int c = c_start + (q >> 3);
    if (c >= a.C) c -= a.C;
    const int k0 = c * kChunkK + (q & 7) * 8;
    if (k0 >= a.K) return make_uint4(0u, 0u, 0u, 0u);
    return __ldg(reinterpret_cast<const uint4*>(a.x + (size_t)m * a.K + k0));
}

// Stage the token rows for chunks c_start .. c_start+nx-1 (mod C) into shared
// memory as f16, token-major, in the order the B fragments are read: for token
// m and chunk ci, 128 bytes at m*x_stride + ci*128, where lane quarter t owns
// 32 bytes = the k pairs (16j+2t, +1) and (16j+2t+8, +9) of blocks j = 0..3.
// One coalesced global pass (16-byte loads) scatters the bf16 values into
// place and tracks each token's amax; after one barrier a shared-memory-only
// pass scales token m by 2^e_m (amax * 2^e_m in [2^14, 2^15)) and rounds to
// f16, which is exact for every bf16 value within 2^-24 of the row's amax.
// (The scattered 4-byte stores conflict on banks; issued before the barrier
// they hide behind the other warps' loads, and the conversion pass is
// conflict-free 16-byte accesses.)  The consumers wait for the preceding grid
// (griddepcontrol.wait) only here, just before the first token load, so that
// their set-up overlaps that grid's tail.  amax_u[0..15] is zero on entry and
// left zero.
template <int NT>
__device__ void stage_x(const KArgs& a, uint8_t* xs, int c_start, int nx, float* tok_unscale,
                        unsigned* amax_u) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    // Warps are dealt to tokens, wpt per token, so that every index below is
    // a shift or an add and a token's amax is one warp reduction.
    const int wpt = kWarps / a.M;
    const int m = warp / wpt, wi = warp - m * wpt;
    const int per_token = nx * 8;  // 16-byte groups of 8 k per token
    const int stride = wpt * 32;
    float mx_local = 0.0f;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (m < a.M) {
        uint8_t* row = xs + m * a.x_stride;
        // A lane's groups go in rounds of kLoads: all loads of a round are in
        // flight together before any value is used.
        constexpr int kLoads = 8;
        for (int base = wi * 32 + lane; base < per_token; base += kLoads * stride) {
            uint4 v[kLoads];
#pragma unroll
            for (int u = 0; u < kLoads; ++u) {
                const int q = base + u * stride;
                v[u] = q < per_token ? load_x_group(a, m, c_start, q) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int u = 0; u < kLoads; ++u) {
                const int q = base + u * stride;
                if (q >= per_token) break;
                track_amax(mx_local, v[u]);
                // pair i (k = k0 + 2i, +1) belongs to lane quarter t = i, block
                // j = grp/2, half = grp&1 (b0 for k%16 < 8, b1 otherwise)
                const int ci = q >> 3, grp = q & 7;
                uint8_t* dst = row + ci * 128 + (grp >> 1) * 8 + (grp & 1) * 4;
                const uint32_t w[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int i = 0; i < 4; ++i) *reinterpret_cast<uint32_t*>(dst + i * 32) = w[i];
            }
        }
    }
    // amax >= 0, so its bit pattern orders like its value
    const unsigned wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(mx_local));
    if (lane == 0 && m < a.M && wmax != 0u) atomicMax(&amax_u[m], wmax);
    consumer_sync();
    if (tid < 16) tok_unscale[tid] = pow2f(-token_exponent(amax_u[tid]));
    if (m < a.M) {  // exact power-of-two f16 conversion, 16 bytes per lane
        uint4* row = reinterpret_cast<uint4*>(xs + m * a.x_stride);
        const float sc = pow2f(token_exponent(amax_u[m]));
        for (int i = wi * 32 + lane; i < per_token; i += stride) {
            uint4 w = row[i];
            w.x = scale_pair_to_f16(w.x, sc);
            w.y = scale_pair_to_f16(w.y, sc);
            w.z = scale_pair_to_f16(w.z, sc);
            w.w = scale_pair_to_f16(w.w, sc);
            row[i] = w;
        }
    }
    consumer_sync();
    if (tid < 16) amax_u[tid] = 0u;  // for the next range (after its opening barrier)
}

// Token rows for one or two tokens ("diagonal" B operand).  The 8 columns of
// an m16n8k16 tile hold (scale block j of the chunk, token m) at column
// 2j + m: the MMA of block j sees the token rows only in its own two columns,
// so the four MMAs of a chunk can accumulate into one tile and lane quarter t
// ends up holding block t's sums, which it alone scales.  Per chunk ci the
// 1024 bytes at ci*1024 hold, for lane L = 4g + t, the B registers of the four
// MMAs: bytes h*512 + 16L + 4r (h = j/2, r = 2(j%2) + b) are the pair
// (x[m][16j + 2t + 8b], +1) when g = 2j + m with m < M, and zero otherwise.
// The area is zero-filled before the wait for the preceding grid; then, as in
// stage_x, the loads are issued together, and after the amax barrier each
// lane converts its groups and writes their words over the zeros.
static __device__ void stage_x_diag(const KArgs& a, uint8_t* xs, int c_start, int nx, float* tok_unscale,
                             unsigned* amax_u) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int wpt = kWarps / a.M;  // warps per token (M <= 2)
    const int m = warp / wpt, wi = warp - m * wpt;
    const int per_token = nx * 8;  // 16-byte groups of 8 k per token
    const int stride = wpt * 32;
    const int q0 = wi * 32 + lane;
    constexpr int kLoads = 2;  // 64 chunks of 8 groups over 256 lanes (M = 2)
    const bool in_regs = per_token <= kLoads * stride;
    float mx_local = 0.0f;
    for (int i = tid; i < nx * 64; i += kConsumerThreads)  // before the grid wait
        reinterpret_cast<uint4*>(xs)[i] = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("griddepcontrol.wait;" ::: "memory");
    uint4 v[kLoads];
#pragma unroll
    for (int u = 0; u < kLoads; ++u) {
        const int q = q0 + u * stride;
        v[u] = q < per_token ? load_x_group(a, m, c_start, q) : make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int u = 0; u < kLoads; ++u) track_amax(mx_local, v[u]);
    for (int q = q0 + kLoads * stride; q < per_token; q += stride)  // beyond the registers
        track_amax(mx_local, load_x_group(a, m, c_start, q));
    const unsigned wmax = __reduce_max_sync(0xffffffffu, __float_as_uint(mx_local));
    if (lane == 0 && wmax != 0u) atomicMax(&amax_u[m], wmax);
    consumer_sync();  // amax complete; zero fill ordered before the data words
    if (tid < 16) tok_unscale[tid] = pow2f(-token_exponent(amax_u[tid]));
    const float sc = pow2f(token_exponent(amax_u[m]));
    for (int base = q0; base < per_token; base += kLoads * stride) {
#pragma unroll
        for (int u = 0; u < kLoads; ++u) {
            const int q = base + u * stride;
            if (q >= per_token) break;
            const uint4 w4 = in_regs ? v[u] : load_x_group(a, m, c_start, q);
            const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
            // pair i (k = 8*grp + 2i): block j = grp/2, half b = grp&1, quarter t = i
            const int ci = q >> 3, grp = q & 7;
            const int j = grp >> 1, b = grp & 1;
            uint8_t* dst =
                xs + ci * 1024 + (j >> 1) * 512 + (4 * (2 * j + m)) * 16 + 4 * (2 * (j & 1) + b);
#pragma unroll
            for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint32_t*>(dst + 16 * i) = scale_pair_to_f16(w[i], sc);
        }
    }
    consumer_sync();
    if (tid < 16) amax_u[tid] = 0u;  // for the next range (after its opening barrier)
}

// Split-K bookkeeping of one warp's tile.  Slot (range r, segment index) holds,
// per tile, that range's fp32 partial sums of the tile's 16 rows x TOK tokens
// for each stream; a per-(row block, tile) counter names the last range to
// arrive, which sums all parts in range order.
template <int NS>
__device__ __forceinline__ float* tile_slot(const KArgs& a, int r, int rb, int warp) {
    const size_t slot = (size_t)kBlockTiles * NS * kTileRows * a.M;
    const int si_slot = rb - rb_of_step(a, (int)range_start(a, r));
    return a.partials + ((size_t)r * a.s_max + si_slot) * slot + (size_t)warp * NS * kTileRows * a.M;
}

// Count this warp's partial of (row block rb, tile) as arrived.  The
// increment is acquire-release at GPU scope: the slot stores of every lane,
// ordered before it by the caller's __syncwarp, are visible to the range that
// observes the final count, and that range sees the others' slots.  The warp
// does not wait for the returned count here: a segment that closes in the
// middle of a range keeps streaming, and the count is examined after the
// range's last step (resolve_tile).
__device__ __forceinline__ int publish_tile(const KArgs& a, int rb, int warp, int lane) {
    int old = 0;
    if (lane == 0) old = atom_add_acq_rel_gpu(a.counters + rb * kBlockTiles + warp, 1);
    return old;  // lane 0 only; consumed later by resolve_tile
}

// The counter's old value for a pending publication `p` of this warp (lane 0):
// p >= 0 is the value itself; p <= -2 is publisher event -2 - p, whose value is
// read once the publisher has marked the event done.  Returns -1 (and flags
// the call) if that wait is abandoned.
__device__ __forceinline__ int pending_old_value(const KArgs& a, int p, int warp,
                                                 uint32_t pub_done0, const int* pub_old,
                                                 const volatile int* abort_flag) {
    if (p >= 0) return p;
    const int e = -2 - p;
    if (!mbar_wait_bounded(pub_done0 + 8u * e, 0, abort_flag, a.wait_ns)) {
        atomicOr(a.status, 1);
        return -1;
    }
    return pub_old[e * kWarps + warp];
}

// Whether the publication that returned `old` (lane 0) was the last of the
// ranges covering rb; the last one resets the counter for the next call.
__device__ __forceinline__ bool resolve_tile(const KArgs& a, int rb, int warp, int lane, int old) {
    int last = 0;
    if (lane == 0) {
        const long long p_lo = (long long)rb * a.CS;
        const int nparts = range_of(a, p_lo + a.CS - 1) - range_of(a, p_lo) + 1;
        last = (old >= 0 && old == nparts - 1) ? 1 : 0;
        if (last) a.counters[rb * kBlockTiles + warp] = 0;  // ready for the next call
    }
    last = __shfl_sync(0xffffffffu, last, 0);
    __syncwarp();  // the other lanes' slot loads follow lane 0's acquire
    return last != 0;
}

// End of the segment of row block rb (last step cb_last) that range r covers,
// for this warp's tile; no CTA-wide synchronisation.  A segment spanning the
// whole K range is stored at once (returns -1).  Otherwise the fp32 partial
// goes to the range's slot and is counted in on the tile's counter: for the
// CTA's first kMaxEvents such segments (event evt) by the publisher warp,
// asynchronously (returns -2 - evt), later ones by this warp (returns the
// counter's old value, lane 0).  Whether this range arrived last, and so must
// reduce the tile, is resolved after the stream (resolve_pending).  With
// coop_last (a range's last segment in the cooperative kernels) the partial is
// stored and kSegCoop returned: the caller then finishes the tile with
// coop_finish.  (Publisher events return -2 .. -1 - kMaxEvents.)
constexpr int kSegCoop = -1000;
static_assert(kSegCoop < -1 - kMaxEvents, "kSegCoop must not be a publisher event code");
template <int NS, int NT, bool DIAG, bool EM>
__device__ __forceinline__ int finish_segment(const KArgs& a, float (&hi)[NS][NT][4],
                                               float (&lo)[NS][NT][4],
                                               const float (&unscale)[NT][2], int r, int q0,
                                               int rb, int cb_last, int warp, int lane, bool ok,
                                               int evt, uint32_t seg_done0, bool coop_last) {
    const int g = lane >> 2, tq = lane & 3;
    const int seg_lo = q0 > rb * a.CS ? q0 : rb * a.CS;
    const bool full_cover = (seg_lo == rb * a.CS) && (cb_last == a.CS - 1);
    float v[NS][NT][4];
#pragma unroll
    for (int si = 0; si < NS; ++si)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                v[si][nt][e] = (hi[si][nt][e] + lo[si][nt][e]) * unscale[nt][e & 1];
                hi[si][nt][e] = 0.0f;
                lo[si][nt][e] = 0.0f;
                if (DIAG) {  // lane quarters hold blocks 0..3: sum them (fixed order)
                    v[si][nt][e] += __shfl_xor_sync(0xffffffffu, v[si][nt][e], 1);
                    v[si][nt][e] += __shfl_xor_sync(0xffffffffu, v[si][nt][e], 2);
                }
            }
    // Element e of lane (g, tq) is row g + 8*(e>>1) and token nt*8 + 2*tq + (e&1);
    // with the diagonal layout every quarter holds the same sums, token e&1,
    // and quarter 0 stores them.
    const bool lane_stores = !DIAG || tq == 0;
    if (full_cover) {
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int row = rb * kBlockRows + warp * kTileRows + g + 8 * (e >> 1);
                const int token = DIAG ? (e & 1) : nt * 8 + 2 * tq + (e & 1);
                if (ok && lane_stores && row < a.N && token < a.M)
                    store_output<NS>(a, row, token, v[0][nt][e], v[NS - 1][nt][e]);
            }
        return -1;
    }
    if (EM) {
        // element-major: element (si, row, token) of the tile, part r - r_first
        float* base = a.partials + (size_t)(rb * kBlockTiles + warp) * (NS * kTileRows * a.M) *
                                       a.part_stride +
                      (r - range_of(a, (long long)rb * a.CS));
#pragma unroll
        for (int si = 0; si < NS; ++si)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int token = DIAG ? (e & 1) : 2 * tq + (e & 1);
                if (lane_stores && token < a.M)
                    base[(size_t)((si * kTileRows + g + 8 * (e >> 1)) * a.M + token) *
                         a.part_stride] = v[si][0][e];
            }
    } else {
        float* slot = tile_slot<NS>(a, r, rb, warp);
#pragma unroll
        for (int si = 0; si < NS; ++si)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int token = nt * 8 + 2 * tq + (e & 1);
                    if (lane_stores && token < a.M)
                        slot[(si * kTileRows + g + 8 * (e >> 1)) * a.M + token] = v[si][nt][e];
                }
    }
    __syncwarp();
    if (coop_last) return kSegCoop;
    if (evt < kMaxEvents) {
        // the publisher warp counts the tile in once every warp has stored;
        // this warp streams on (the arrive releases the lanes' slot stores to
        // the CTA, and the publisher's GPU-scope release carries them on)
        if (lane == 0) mbar_arrive(seg_done0 + 8u * evt);
        return -2 - evt;
    }
    return publish_tile(a, rb, warp, lane);
}

// The last range to arrive for (row block rb, this warp's tile): sum every
// range's partial in range order and store the tile's outputs.  Each lane owns
// up to kIter of the tile's 16 x M elements; the slot loads of all of them for
// kB ranges are issued before any is used, so a tile costs one load latency
// per kB ranges whatever M is.
template <int NS, int NT>
__device__ __forceinline__ void reduce_tile(const KArgs& a, int rb, int warp, int lane, bool ok,
                                            int e_begin, int e_end) {
    constexpr int kIter = kTileRows * 8 * NT / 32;  // elements per lane at M = 8 NT
    constexpr int kB = 32 / (kIter * NS);           // ranges per batch (32 loads in flight)
    const long long p_lo = (long long)rb * a.CS;
    const int r_first = range_of(a, p_lo), r_last = range_of(a, p_lo + a.CS - 1);
    const int n_el = kTileRows * a.M;
    float sum[kIter][NS];
#pragma unroll
    for (int i = 0; i < kIter; ++i)
#pragma unroll
        for (int si = 0; si < NS; ++si) sum[i][si] = 0.0f;
    for (int r0 = r_first; r0 <= r_last; r0 += kB) {
        float part[kB][kIter][NS];
#pragma unroll
        for (int b = 0; b < kB; ++b) {
            const int rr = r0 + b;
            const float* sl = rr <= r_last ? tile_slot<NS>(a, rr, rb, warp) : nullptr;
#pragma unroll
            for (int i = 0; i < kIter; ++i) {
                const int e = e_begin + lane + 32 * i;
#pragma unroll
                for (int si = 0; si < NS; ++si)
                    part[b][i][si] = (sl != nullptr && e < e_end) ? __ldcg(sl + si * n_el + e) : 0.0f;
            }
        }
#pragma unroll
        for (int b = 0; b < kB; ++b)
#pragma unroll
            for (int i = 0; i < kIter; ++i)
#pragma unroll
                for (int si = 0; si < NS; ++si) sum[i][si] += part[b][i][si];
    }
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
        const int e = e_begin + lane + 32 * i;
        if (e >= e_end) continue;
        const int token = e % a.M, row16 = e / a.M;
        const int row = rb * kBlockRows + warp * kTileRows + row16;
        if (ok && row < a.N) store_output<NS>(a, row, token, sum[i][0], sum[i][NS - 1]);
    }
}

// Where the E4M3 row scales are applied.  With one n8 token tile: to the fp32
// block sums of independent zero-initialised MMAs, by FFMA (measured faster
// than chained MMAs on GB300).  With two token tiles: folded into the A
// fragments by an exact f16 multiply, so the MMAs accumulate directly and the
// scaling is shared by both tiles.
// reduce_tile for the element-major partials (M <= MAXM): lane l owns elements
// l, l+32, ... (< 16*M) of each stream and reads each element's parts in
// 16-byte vectors, kPB parts per batch with every load of the batch in flight
// together, summing them in range order.
template <int NS, int MAXM>
__device__ __forceinline__ void reduce_tile_em(const KArgs& a, int rb, int warp, int lane,
                                               bool ok, int e_begin, int e_end) {
    constexpr int kIter = (kTileRows * MAXM + 31) / 32;  // elements per lane at the largest M
    constexpr int kPB = 32 / (kIter * NS);                 // parts per batch (32 in flight)
    static_assert(kPB % 4 == 0, "parts are read in 16-byte vectors");
    const long long p_lo = (long long)rb * a.CS;
    const int nparts = range_of(a, p_lo + a.CS - 1) - range_of(a, p_lo) + 1;
    const int n_el = kTileRows * a.M;
    const float* base = a.partials + (size_t)(rb * kBlockTiles + warp) * (NS * n_el) * a.part_stride;
    float sum[kIter][NS];
#pragma unroll
    for (int i = 0; i < kIter; ++i)
#pragma unroll
        for (int si = 0; si < NS; ++si) sum[i][si] = 0.0f;
    for (int p0 = 0; p0 < nparts; p0 += kPB) {
        float part[kIter][NS][kPB];
#pragma unroll
        for (int i = 0; i < kIter; ++i) {
            const int e = e_begin + lane + 32 * i;
#pragma unroll
            for (int si = 0; si < NS; ++si) {
                const float4* src = reinterpret_cast<const float4*>(
                    base + (size_t)(si * n_el + e) * a.part_stride + p0);
#pragma unroll
                for (int q = 0; q < kPB / 4; ++q) {
                    const float4 v4 = (e < e_end && p0 + 4 * q < nparts)
                                          ? __ldcg(src + q)
                                          : make_float4(0.f, 0.f, 0.f, 0.f);
                    part[i][si][4 * q] = v4.x;
                    part[i][si][4 * q + 1] = v4.y;
                    part[i][si][4 * q + 2] = v4.z;
                    part[i][si][4 * q + 3] = v4.w;
                }
            }
        }
#pragma unroll
        for (int i = 0; i < kIter; ++i)
#pragma unroll
            for (int si = 0; si < NS; ++si)
#pragma unroll
                for (int q = 0; q < kPB; ++q)
                    if (p0 + q < nparts) sum[i][si] += part[i][si][q];
    }
#pragma unroll
    for (int i = 0; i < kIter; ++i) {
        const int e = e_begin + lane + 32 * i;
        if (e >= e_end) continue;
        const int token = e % a.M, row16 = e / a.M;
        const int row = rb * kBlockRows + warp * kTileRows + row16;
        if (ok && row < a.N) store_output<NS>(a, row, token, sum[i][0], sum[i][NS - 1]);
    }
}

// Final sums and outputs of elements [e_begin, e_end) of (row block rb, this
// warp's tile), every part read in range order.
template <int NS, int NT, bool DIAG, bool EM>
__device__ __forceinline__ void reduce_any(const KArgs& a, int rb, int warp, int lane, bool ok,
                                           int e_begin, int e_end) {
    if constexpr (EM)
        reduce_tile_em<NS, DIAG ? 2 : kElemMajorMaxM>(a, rb, warp, lane, ok, e_begin, e_end);
    else
        reduce_tile<NS, NT>(a, rb, warp, lane, ok, e_begin, e_end);
}

// Cooperative finish of a split row block (the non-diagonal kernels).  The
// ranges whose last segment lies in row block rb -- every range covering rb
// except one whose range continues into the next row block -- are its
// participants.  Each publishes its own partial (acquire-release add on the
// tile's counter; the lanes' partial stores are ordered before it by the
// caller's __syncwarp), waits (bounded) until all nparts parts are counted in,
// and then sums and stores its own share of the tile's elements, reading every
// part in range order -- so the results do not depend on which range arrives
// last.  The remaining range counts its part in during its stream and never
// reduces.  Every participant adds 1 more once it has seen the full count; the
// one that brings the counter to nparts + participants resets it to zero for
// the next call.  A warp that gave up a wait earlier (!ok) or whose CTA
// aborted skips all of this; the others then give up their wait after the
// time limit and report it.
template <int NS, int NT, bool DIAG, bool EM>
__device__ __forceinline__ void coop_finish(const KArgs& a, int r, int rb, int warp, int lane,
                                            bool ok, volatile int* abort_flag) {
    if (!ok || *abort_flag) return;
    const long long p_lo = (long long)rb * a.CS;
    const int r_first = range_of(a, p_lo), r_last = range_of(a, p_lo + a.CS - 1);
    const int nparts = r_last - r_first + 1;
    const int P = r_last - r_first + (range_start(a, r_last + 1) <= p_lo + a.CS ? 1 : 0);
    int* cnt = a.counters + rb * kBlockTiles + warp;
    int done = 0;
    if (lane == 0) {
        atom_add_acq_rel_gpu(cnt, 1);
        done = wait_count_bounded(cnt, nparts, abort_flag, a.wait_ns) ? 1 : 0;
        if (!done) {
            *abort_flag = 1;
            atomicOr(a.status, 1);
        }
    }
    done = __shfl_sync(0xffffffffu, done, 0);
    __syncwarp();  // the other lanes' part loads follow lane 0's acquire
    if (!done) return;
    const int n_el = kTileRows * a.M;
    const int per = (n_el + P - 1) / P;
    const int j = r - r_first;
    const int e0 = min(n_el, j * per), e1 = min(n_el, e0 + per);
    reduce_any<NS, NT, DIAG, EM>(a, rb, warp, lane, ok, e0, e1);
    if (lane == 0) {
        const int old = atomicAdd(cnt, 1);
        if (old == nparts + P - 1) *cnt = 0;  // every participant has seen the full count
    }
}

template <int NT>
__device__ __forceinline__ constexpr bool kScaleInA() {
    return NT == 2;
}

// One chunk (64 K elements) of the current step for this warp.  Per k16
// block: the E2M1 codes become exact f16 A fragments (one cvt per byte), the
// MMA forms the block's dot products against the staged token fragments from
// a zero accumulator, and the two row scales (E4M3 -> f16 -> f32, exact) are
// applied to those fp32 block sums with FFMAs.  Every MMA is independent; the
// FMA pipe takes the scaling, which leaves the ALU pipe to the decode.
// wl: this lane's 16 code bytes of the chunk's unit; sl: the scale bytes of
// its row pair (g, g+8); xl[nt]: its B fragments of token tile nt (32 bytes).
// The second stream's unit follows the first's (gate/up interleave).
template <int NS, int NT, bool ONE>
__device__ __forceinline__ void process_chunk(const uint8_t* wl, const uint8_t* sl,
                                              const uint8_t* const (&xl)[NT],
                                              float (&acc)[NS][NT][4]) {
    uint32_t b[NT][8];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(xl[nt]);
        const uint4 v1 = *reinterpret_cast<const uint4*>(xl[nt] + 16);
        b[nt][0] = v0.x;
        b[nt][1] = v0.y;
        b[nt][2] = v0.z;
        b[nt][3] = v0.w;
        b[nt][4] = v1.x;
        b[nt][5] = v1.y;
        b[nt][6] = v1.z;
        b[nt][7] = v1.w;
    }
#pragma unroll
    for (int si = 0; si < NS; ++si) {
        const uint4 cw = *reinterpret_cast<const uint4*>(wl + si * kUnitBytes);
        const uint2 sw = *reinterpret_cast<const uint2*>(sl + si * kUnitBytes);
        const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
            uint32_t a0, a1, a2, a3;
            e2m1x8_to_f16x2x4(cws[jb], a0, a1, a2, a3);
            const uint32_t sword = jb < 2 ? sw.x : sw.y;
            const uint32_t s2 = (jb & 1) ? e4m3x2_hi_to_f16x2(sword)
                                         : e4m3x2_to_f16x2(sword);  // (row g, row g+8) scales
            if (kScaleInA<NT>()) {
                // (s_g, s_g) and (s_g8, s_g8) as f16x2; an E4M3 value times an
                // E2M1 value is exact in f16 (at most 6 significant bits,
                // magnitudes from 2^-10 to 2688).
                const uint32_t sg = prmt(s2, 0u, 0x1010u);
                const uint32_t sg8 = prmt(s2, 0u, 0x3232u);
                a0 = hmul2(a0, sg);
                a2 = hmul2(a2, sg);
                a1 = hmul2(a1, sg8);
                a3 = hmul2(a3, sg8);
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
                    mma_f16_16816(acc[si][nt], a0, a1, a2, a3, b[nt][2 * jb], b[nt][2 * jb + 1]);
            } else {
                const float sgf = __half2float(__ushort_as_half((unsigned short)(s2 & 0xFFFFu)));
                const float sg8f = __half2float(__ushort_as_half((unsigned short)(s2 >> 16)));
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    float d[4];
                    mma_f16_16816_zero(d, a0, a1, a2, a3, b[nt][2 * jb], b[nt][2 * jb + 1]);
                    acc[si][nt][0] = fmaf(d[0], sgf, acc[si][nt][0]);
                    acc[si][nt][2] = fmaf(d[2], sg8f, acc[si][nt][2]);
                    if (!ONE) {  // columns 2t+1 hold token 1 and up
                        acc[si][nt][1] = fmaf(d[1], sgf, acc[si][nt][1]);
                        acc[si][nt][3] = fmaf(d[3], sg8f, acc[si][nt][3]);
                    }
                }
            }
        }
    }
}

// One chunk with the diagonal token layout (M <= 2, stage_x_diag): the four
// MMAs of the chunk accumulate into one tile, whose columns 2j, 2j+1 hold
// block j's sums for tokens 0, 1; lane quarter t then applies block t's two
// row scales (rows g, g+8) with FFMAs.  Per k16 block: 4 cvt + 1 MMA; per
// chunk and lane: one scale-pair select and conversion and 2 (ONE) or 4 FFMAs.
// wl, sl as for process_chunk; xl: this lane's 16 bytes of the chunk's first
// 512-byte half of the diagonal token area (the second half follows).
template <int NS, bool ONE>
__device__ __forceinline__ void process_chunk_diag(const uint8_t* wl, const uint8_t* sl,
                                                   const uint8_t* xl, uint32_t scale_sel,
                                                   float (&acc)[NS][1][4]) {
    const uint4 v0 = *reinterpret_cast<const uint4*>(xl);
    const uint4 v1 = *reinterpret_cast<const uint4*>(xl + 512);
    const uint32_t b[8] = {v0.x, v0.y, v0.z, v0.w, v1.x, v1.y, v1.z, v1.w};
#pragma unroll
    for (int si = 0; si < NS; ++si) {
        const uint4 cw = *reinterpret_cast<const uint4*>(wl + si * kUnitBytes);
        const uint2 sw = *reinterpret_cast<const uint2*>(sl + si * kUnitBytes);
        const uint32_t cws[4] = {cw.x, cw.y, cw.z, cw.w};
        float d[4];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
            uint32_t a0, a1, a2, a3;
            e2m1x8_to_f16x2x4(cws[jb], a0, a1, a2, a3);
            if (jb == 0)
                mma_f16_16816_zero(d, a0, a1, a2, a3, b[0], b[1]);
            else
                mma_f16_16816(d, a0, a1, a2, a3, b[2 * jb], b[2 * jb + 1]);
        }
        // bytes 2t, 2t+1 of the row pair's 8 scale bytes: block t of rows g, g+8
        const uint32_t s2 = e4m3x2_to_f16x2(prmt(sw.x, sw.y, scale_sel));
        const float sgf = __half2float(__ushort_as_half((unsigned short)(s2 & 0xFFFFu)));
        const float sg8f = __half2float(__ushort_as_half((unsigned short)(s2 >> 16)));
        acc[si][0][0] = fmaf(d[0], sgf, acc[si][0][0]);
        acc[si][0][2] = fmaf(d[2], sg8f, acc[si][0][2]);
        if (!ONE) {
            acc[si][0][1] = fmaf(d[1], sgf, acc[si][0][1]);
            acc[si][0][3] = fmaf(d[3], sg8f, acc[si][0][3]);
        }
    }
}

// One chunk (64 K elements) of block-scaled FP8 weights for this warp.  Per
// k16 block: the lane's 8 code bytes become the four f16 A fragments (one cvt
// per E4M3 pair, exact), and the chunk's four MMAs chain into one fp32 tile
// from a zero accumulator; the tile's block scale (one fp32 per 128 rows x
// 128 K, the same for all 16 rows of the tile) is then applied with FFMAs.
// wl: this lane's 32 code bytes of the chunk's tile; sl: the tile's scales
// (one fp32 per stream); xl[nt] as for process_chunk.  The second stream's
// tile follows the first's.
template <int NS, int NT, bool ONE>
__device__ __forceinline__ void process_chunk_f8(const uint8_t* wl, const uint8_t* sl,
                                                 const uint8_t* const (&xl)[NT],
                                                 float (&acc)[NS][NT][4]) {
    uint32_t b[NT][8];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const uint4 v0 = *reinterpret_cast<const uint4*>(xl[nt]);
        const uint4 v1 = *reinterpret_cast<const uint4*>(xl[nt] + 16);
        b[nt][0] = v0.x;
        b[nt][1] = v0.y;
        b[nt][2] = v0.z;
        b[nt][3] = v0.w;
        b[nt][4] = v1.x;
        b[nt][5] = v1.y;
        b[nt][6] = v1.z;
        b[nt][7] = v1.w;
    }
#pragma unroll
    for (int si = 0; si < NS; ++si) {
        const uint4 c0 = *reinterpret_cast<const uint4*>(wl + si * kF8TileBytes);
        const uint4 c1 = *reinterpret_cast<const uint4*>(wl + si * kF8TileBytes + 16);
        const float scale = *reinterpret_cast<const float*>(sl + 4 * si);
        // word 2j: (row g, k pair 16j+2t) and (row g+8, same k); word 2j+1:
        // the same rows at k pair 16j+2t+8
        const uint32_t cw[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
        float d[NT][4];
#pragma unroll
        for (int jb = 0; jb < 4; ++jb) {
            const uint32_t a0 = e4m3x2_to_f16x2(cw[2 * jb]);
            const uint32_t a1 = e4m3x2_hi_to_f16x2(cw[2 * jb]);
            const uint32_t a2 = e4m3x2_to_f16x2(cw[2 * jb + 1]);
            const uint32_t a3 = e4m3x2_hi_to_f16x2(cw[2 * jb + 1]);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                if (jb == 0)
                    mma_f16_16816_zero(d[nt], a0, a1, a2, a3, b[nt][0], b[nt][1]);
                else
                    mma_f16_16816(d[nt], a0, a1, a2, a3, b[nt][2 * jb], b[nt][2 * jb + 1]);
            }
        }
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
            acc[si][nt][0] = fmaf(d[nt][0], scale, acc[si][nt][0]);
            acc[si][nt][2] = fmaf(d[nt][2], scale, acc[si][nt][2]);
            if (!ONE) {
                acc[si][nt][1] = fmaf(d[nt][1], scale, acc[si][nt][1]);
                acc[si][nt][3] = fmaf(d[nt][3], scale, acc[si][nt][3]);
            }
        }
    }
}

// First byte of the step at `cur` in the repacked blob.
template <int NS, bool F8>
__device__ __forceinline__ const uint8_t* step_src(const KArgs& a, const StepCursor& cur) {
    constexpr int CPS = (F8 ? kF8UnitsPerStep : kUnitsPerStep) / NS;
    return a.blob + ((size_t)cur.rb * a.C + (size_t)cur.cb * CPS) * group_bytes(NS, F8);
}

// Issue the bulk copy of the step at `cur` into ring stage st (one thread).
// The weights are read exactly once per call, so their lines are marked for
// early eviction: L2 keeps the token rows, h and the split-K partials instead.
template <int NS, bool F8>
__device__ __forceinline__ void issue_step(const KArgs& a, const StepCursor& cur, int st,
                                           uint32_t ring_s, uint32_t full0, int* issues) {
    constexpr int CPS = (F8 ? kF8UnitsPerStep : kUnitsPerStep) / NS;
    const uint32_t bytes = (uint32_t)(CPS * group_bytes(NS, F8));
    mbar_arrive_expect_tx(full0 + 8u * st, bytes);
    bulk_copy_g2s_hint(ring_s + (uint32_t)(st * a.stage_bytes), step_src<NS, F8>(a, cur), bytes,
                       full0 + 8u * st, l2_evict_first_policy());
    ++issues[st];
}

// The row blocks (and counter values) a warp must still resolve, oldest
// first, up to four.  PendRegs keeps them in registers with compile-time
// indexing (a dynamically indexed array lives in local memory, whose L1 share
// is small next to the shared-memory carve-out); PendArray is the plain array.
// Measured: the registers win for the diagonal layout (M <= 2), the array for
// the others, whose register budget the scalars crowd.
struct PendRegs {
    int rb0 = 0, rb1 = 0, rb2 = 0, rb3 = 0, o0 = 0, o1 = 0, o2 = 0, o3 = 0;
    __device__ __forceinline__ void set(int n, int rb, int old) {
        rb0 = n == 0 ? rb : rb0;
        rb1 = n == 1 ? rb : rb1;
        rb2 = n == 2 ? rb : rb2;
        rb3 = n == 3 ? rb : rb3;
        o0 = n == 0 ? old : o0;
        o1 = n == 1 ? old : o1;
        o2 = n == 2 ? old : o2;
        o3 = n == 3 ? old : o3;
    }
    __device__ __forceinline__ void pop_front() {
        rb0 = rb1;
        rb1 = rb2;
        rb2 = rb3;
        o0 = o1;
        o1 = o2;
        o2 = o3;
    }
    template <int I>
    __device__ __forceinline__ int rb() const {
        return I == 0 ? rb0 : I == 1 ? rb1 : I == 2 ? rb2 : rb3;
    }
    template <int I>
    __device__ __forceinline__ int old() const {
        return I == 0 ? o0 : I == 1 ? o1 : I == 2 ? o2 : o3;
    }
};

struct PendArray {
    int rb_[4], o_[4];
    __device__ __forceinline__ void set(int n, int rb, int old) {
        rb_[n] = rb;
        o_[n] = old;
    }
    __device__ __forceinline__ void pop_front() {
        for (int i = 1; i < 4; ++i) {
            rb_[i - 1] = rb_[i];
            o_[i - 1] = o_[i];
        }
    }
    template <int I>
    __device__ __forceinline__ int rb() const {
        return rb_[I];
    }
    template <int I>
    __device__ __forceinline__ int old() const {
        return o_[I];
    }
};

// A consumer's wait on a stage that was not full at the first test: bounded,
// and kept out of line so that the step loop stays small.  On giving up it
// raises the CTA's abort flag and the device status word.
static __device__ __noinline__ bool wait_stage_slow(uint32_t bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned long long limit_ns,
                                             int* status) {
    if (mbar_wait_bounded(bar, parity, abort_flag, limit_ns)) return true;
    *abort_flag = 1;
    atomicOr(status, 1);
    return false;
}

// ONE: a single token row (M == 1), which needs only the even MMA columns.
// DIAG: M <= 2 with the diagonal token layout (stage_x_diag; NVFP4 only).
// EM: element-major split-K partials (M <= kElemMajorMaxM).
// F8: block-scaled FP8 weights (process_chunk_f8) instead of NVFP4.
// COOP: split row blocks finished cooperatively (coop_finish) instead of by the
// last range to arrive; a compile-time choice, since a kernel holding both
// finishing paths runs slower than either (register pressure).
template <int NS, int NT, bool ONE, bool DIAG, bool EM, bool F8, bool COOP>
__global__ void __launch_bounds__(kThreads, 1) stream_gemv_kernel(const KArgs a) {
    static_assert(!(F8 && DIAG), "the diagonal token layout is for NVFP4 block scales");
    static_assert(!(COOP && DIAG), "the diagonal kernels finish by the last range to arrive");
    constexpr bool coop = COOP;
    constexpr int CPS = (F8 ? kF8UnitsPerStep : kUnitsPerStep) / NS;  // chunks per step
    constexpr int GB = group_bytes(NS, F8);                             // bytes per chunk

    extern __shared__ __align__(128) uint8_t smem[];
    const uint32_t ring_s = smem_addr(smem);
    uint8_t* xs = smem + a.x_off;
    const uint32_t full0 = smem_addr(smem + a.bar_off);   // stage filled (tx bytes)
    const uint32_t empty0 = smem_addr(smem + a.cnt_off);  // stage released by all consumers
    float* tok_unscale = reinterpret_cast<float*>(smem + a.misc_off);
    unsigned* amax_u = reinterpret_cast<unsigned*>(tok_unscale + 16);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(amax_u + 16);
    int* issues = reinterpret_cast<int*>(smem + a.misc_off + kMiscIssuesOff);  // copies per stage
    const uint32_t seg_done0 = smem_addr(smem + a.misc_off + kMiscPubOff);  // per event
    const uint32_t pub_done0 = seg_done0 + 8u * kMaxEvents;
    int* pub_old = reinterpret_cast<int*>(smem + a.misc_off + kMiscPubOff + 16 * kMaxEvents);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tq = lane & 3;
    // diagonal layout: PRMT selector of scale bytes 2tq, 2tq+1 (block tq)
    const uint32_t scale_sel = (uint32_t)(2 * tq) | ((uint32_t)(2 * tq + 1) << 4);
    (void)scale_sel;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(full0 + 8u * s, 1);
            mbar_init(empty0 + 8u * s, kConsumerThreads);  // every consumer lane arrives
            issues[s] = 0;
        }
        for (int e = 0; e < kMaxEvents; ++e) {
            mbar_init(seg_done0 + 8u * e, kWarps);
            mbar_init(pub_done0 + 8u * e, 1);
        }
        for (int t = 0; t < 16; ++t) amax_u[t] = 0u;  // staging's token maxima
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    // Let the next kernel on the stream launch as SMs free up; it will wait
    // for this grid before it touches anything this grid writes.
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

    if (warp >= kWarps) {
        // ---- producer warpgroup: lane 0 of its first warp streams every step
        // of this CTA's ranges through the ring.  Weights are never written by
        // the preceding kernel when early_weights is set, so the ring fills
        // before the wait on it.
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducerRegs));
        if (warp == kWarps && lane == 0) {
            if (!a.early_weights) asm volatile("griddepcontrol.wait;" ::: "memory");
            StepCursor ahead;
            ahead.init(a);
            int pst = 0, round = 0;
            while (!a.stall && ahead.valid(a) && !*abort_flag) {
                // refilling a stage: wait until all consumer warps released it
                if (round > 0 && !mbar_wait_bounded(empty0 + 8u * pst, (uint32_t)((round - 1) & 1),
                                                    abort_flag, a.wait_ns)) {
                    *abort_flag = 1;
                    atomicOr(a.status, 1);
                    break;
                }
                asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
                issue_step<NS, F8>(a, ahead, pst, ring_s, full0, issues);
                ahead.advance(a);
                if (++pst == a.stages) {
                    pst = 0;
                    ++round;
                }
            }
            // Every copy must have landed before the CTA (and its shared
            // memory) goes away; the consumers wait for all of them unless a
            // wait was abandoned, so this only waits in that case, and always
            // with the full limit whatever wait_ns is.
            const int zero = 0;
            for (int s = 0; s < a.stages; ++s)
                if (issues[s] > 0)
                    mbar_wait_bounded(full0 + 8u * s, (uint32_t)((issues[s] - 1) & 1), &zero);
        } else if (warp == kWarps + 1) {
            // ---- publisher: counts the consumer warps' partial tiles in on the
            // split-K counters, so that the GPU-scope release of the slot
            // stores (which waits for them to reach L2) holds up this warp and
            // not the stream.  The segments are enumerated as the consumers
            // walk them; lane t < kWarps handles tile t.
            int e = 0;
            for (int r = blockIdx.x; r < a.R && e < kMaxEvents; r += a.grid) {
                const int q0 = (int)range_start(a, r), q1 = (int)range_start(a, r + 1);
                int rb = rb_of_step(a, q0);
                int cb = q0 - rb * a.CS;
                for (int q = q0; q < q1 && e < kMaxEvents; q += a.CS - cb, ++rb, cb = 0) {
                    const int seg_n = q1 - q < a.CS - cb ? q1 - q : a.CS - cb;
                    if (cb == 0 && seg_n == a.CS) continue;  // whole row block: stored directly
                    if (coop && q + seg_n == q1) continue;   // last segment: coop_finish
                    if (!mbar_wait_bounded(seg_done0 + 8u * e, 0, abort_flag, a.wait_ns)) {
                        *abort_flag = 1;
                        atomicOr(a.status, 1);
                        return;
                    }
                    if (lane < kWarps)
                        pub_old[e * kWarps + lane] =
                            atom_add_acq_rel_gpu(a.counters + rb * kBlockTiles + lane, 1);
                    __syncwarp();
                    if (lane == 0) mbar_arrive(pub_done0 + 8u * e);
                    ++e;
                }
            }
        }
        return;
    }
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumerRegs));
    // (The consumers wait for the preceding grid in the token staging, just
    // before the first token load.)
    // The ring as seen by this lane: the offset of the current stage, its
    // "full" barrier (its "empty" barrier lies bar_gap further) and phase, and
    // the lane's code and scale addresses in stage 0.
    // NVFP4: unit pairs (codes then scales) tile by tile.  FP8: the tiles'
    // codes, then one fp32 scale per tile and stream after all of them.
    const uint8_t* const wl0 =
        F8 ? smem + warp * (NS * kF8TileBytes) + lane * 32 : smem + warp * (NS * kUnitBytes) + lane * 16;
    const uint8_t* const sl0 =
        F8 ? smem + NS * kBlockTiles * kF8TileBytes + warp * (4 * NS)
           : smem + warp * (NS * kUnitBytes) + kUnitCodeBytes + (lane >> 2) * 8;
    const uint32_t stage_bytes = (uint32_t)a.stage_bytes;
    const uint32_t ring_bytes = stage_bytes * (uint32_t)a.stages;
    const uint32_t bar_gap = empty0 - full0;
    uint32_t st_off = 0, bar_f = full0, ph = 0;
    bool ok = true;
    // row blocks whose tile this warp must still reduce (it arrived last)
    constexpr int kMaxPending = 4;
    static_assert(kMaxPending == 4, "the pending FIFO holds four entries");
    using Pend = typename std::conditional<DIAG, PendRegs, PendArray>::type;
    Pend pend;
    int n_pending = 0;
    int evt = 0;  // partial segments so far (publisher events)
    constexpr int kFoldSteps = kFoldChunks / CPS;  // steps between folds
    static_assert(kFoldSteps * CPS == kFoldChunks, "fold period is a whole number of steps");
    // Token fragments: this lane's bytes of chunk 0 of the staged rows, and
    // the distance between consecutive chunks.
    constexpr int kXChunk = DIAG ? 1024 : 128;
    const uint8_t* xl0[NT];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
        const int token = min(nt * 8 + (lane >> 2), a.M - 1);
        xl0[nt] = DIAG ? xs + lane * 16 : xs + token * a.x_stride + tq * 32;
    }
    const int C = a.C;
    for (int r = blockIdx.x; r < a.R; r += a.grid) {
        // ---- a new range: steps q0 .. q1-1; stage its token rows
        const int q0 = (int)range_start(a, r), q1 = (int)range_start(a, r + 1);
        int rb = rb_of_step(a, q0);
        int cb = q0 - rb * a.CS;
        const int c_start = cb * CPS;
        const int nx = (q1 - q0) * CPS < C ? (q1 - q0) * CPS : C;
        consumer_sync();  // every warp is done with the previous range's x
        if (DIAG)
            stage_x_diag(a, xs, c_start, nx, tok_unscale, amax_u);
        else
            stage_x<NT>(a, xs, c_start, nx, tok_unscale, amax_u);
        float unscale[NT][2];
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 2; ++e)
                unscale[nt][e] = tok_unscale[DIAG ? e : nt * 8 + 2 * tq + e];
        // the range's sums (every segment leaves them at zero again)
        float acc[NS][NT][4], hi[NS][NT][4], lo[NS][NT][4];
#pragma unroll
        for (int si = 0; si < NS; ++si)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[si][nt][e] = 0.0f;
                    hi[si][nt][e] = 0.0f;
                    lo[si][nt][e] = 0.0f;
                }
        int ci = 0;  // staged chunk of the current step
        // ---- the range's segments: the run of its steps inside one row block
        for (int q = q0; q < q1; q += a.CS - cb, ++rb, cb = 0) {
            const int seg_n = q1 - q < a.CS - cb ? q1 - q : a.CS - cb;
            // the steps in groups of kFoldSteps, the sums folded after each
#pragma unroll 1
            for (int k0 = 0; k0 < seg_n; k0 += kFoldSteps) {
                const int kn = seg_n - k0 < kFoldSteps ? seg_n - k0 : kFoldSteps;
#pragma unroll 1
                for (int k = 0; k < kn; ++k) {
                    // A warp that gave up a wait keeps walking the steps (every
                    // consumer warp must reach each range's barriers) but waits
                    // no more; its results are discarded.
                    if (!mbar_try_wait(bar_f, ph) && ok)
                        ok = wait_stage_slow(bar_f, ph, abort_flag, a.wait_ns, a.status);
                    const uint8_t* wl = wl0 + st_off;
                    const uint8_t* sl = sl0 + st_off;
                    const int xo = ci * kXChunk;
#pragma unroll
                    for (int j = 0; j < CPS; ++j) {
                        if constexpr (DIAG) {
                            process_chunk_diag<NS, ONE>(wl + j * GB, sl + j * GB,
                                                        xl0[0] + xo + j * kXChunk, scale_sel, acc);
                        } else {
                            const uint8_t* xj[NT];
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) xj[nt] = xl0[nt] + xo + j * kXChunk;
                            if constexpr (F8)
                                process_chunk_f8<NS, NT, ONE>(wl + j * GB, sl + j * GB, xj, acc);
                            else
                                process_chunk<NS, NT, ONE>(wl + j * GB, sl + j * GB, xj, acc);
                        }
                    }
                    // Release the stage to the producer (each lane for itself).
                    mbar_arrive(bar_f + bar_gap);
                    st_off += stage_bytes;
                    bar_f += 8u;
                    if (st_off == ring_bytes) {
                        st_off = 0;
                        bar_f = full0;
                        ph ^= 1u;
                    }
                    ci += CPS;
                    if (ci >= C) ci -= C;
                }
#pragma unroll
                for (int si = 0; si < NS; ++si)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; e += ONE ? 2 : 1) {
                            two_sum_acc(hi[si][nt][e], lo[si][nt][e], acc[si][nt][e]);
                            acc[si][nt][e] = 0.0f;
                        }
            }
            const bool coop_last = coop && q + seg_n == q1;
            const int old = finish_segment<NS, NT, DIAG, EM>(a, hi, lo, unscale, r, q0, rb,
                                                             cb + seg_n - 1, warp, lane, ok, evt,
                                                             seg_done0, coop_last);
            if constexpr (COOP) {
                if (old == kSegCoop)
                    coop_finish<NS, NT, DIAG, EM>(a, r, rb, warp, lane, ok, abort_flag);
                else if (old != -1)
                    ++evt;  // counted in by the publisher or this warp; a participant reduces
            } else if (old != -1) {
                ++evt;
                if (n_pending == kMaxPending) {  // resolve the oldest now
                    const int o = pending_old_value(a, pend.template old<0>(), warp, pub_done0,
                                                    pub_old, abort_flag);
                    if (resolve_tile(a, pend.template rb<0>(), warp, lane, o))
                        reduce_any<NS, NT, DIAG, EM>(a, pend.template rb<0>(), warp, lane, ok, 0,
                                                     kTileRows * a.M);
                    pend.pop_front();
                    --n_pending;
                }
                pend.set(n_pending, rb, old);
                ++n_pending;
            }
        }
    }
    // Resolve what is still pending, oldest first, in a rolled loop: this code
    // runs once per kernel, so one copy of it (fewer instruction lines to
    // fetch from L2) is what counts, not its issue count.
#pragma unroll 1
    for (; n_pending > 0; --n_pending) {
        const int o = pending_old_value(a, pend.template old<0>(), warp, pub_done0, pub_old,
                                        abort_flag);
        if (resolve_tile(a, pend.template rb<0>(), warp, lane, o))
            reduce_any<NS, NT, DIAG, EM>(a, pend.template rb<0>(), warp, lane, ok, 0,
                                         kTileRows * a.M);
        pend.pop_front();
    }
}

template <int NS, int NT, bool ONE, bool DIAG, bool EM, bool F8, bool COOP>
static cudaError_t launch_t(const Plan& p, const KArgs& a, cudaStream_t s) {
    // set once per device; a second thread racing here sets it again, harmlessly
    static std::atomic<bool> attr_done[64];
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64 && !attr_done[dev]) {
        cudaError_t e = cudaFuncSetAttribute(stream_gemv_kernel<NS, NT, ONE, DIAG, EM, F8, COOP>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemMax);
        if (e != cudaSuccess) return e;
        attr_done[dev] = true;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = p.smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, stream_gemv_kernel<NS, NT, ONE, DIAG, EM, F8, COOP>, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}


// Whether a launch finishes split row blocks cooperatively (the COOP kernels).
// It pays where the final reduction is heavy; below that its extra round trip
// (publish, wait for the full count, then load) costs more than the shared
// work saves.  Measured on GB300 (5120 x 17408 and 4096 x 12288 layers): the
// gate/up kernel, whose epilogue evaluates the activation, gains from M = 7;
// a single projection gains from M = 4 when its row blocks are split into at
// least four parts and its ranges are at least four steps long (a 4096 x
// 4096 projection, two steps per range, lost 1 us at M = 4), and from M = 9
// (two token tiles) at any split.  It needs
// one range per CTA: a CTA that waits at the end of each of several ranges
// would tie every CTA's progress to its neighbours'.
static bool use_coop(const Plan& p, int M) {
    if (p.R != p.grid) return false;
    if (p.NS == 2) return M >= 7;
    return M >= 9 || (M >= 4 && p.R >= 4 * p.RB && p.Pmax >= 4);
}

// Kernel arguments for a plan (the adapter deltas are left null).
static KArgs make_kargs(const Plan& p, const void* x, int M, int K, const void* packed, int N,
                        float scale_a, float scale_b, int act, void* out, int* status,
                        int* counters, void* partials, bool early_weights) {
    KArgs a;
    a.x = reinterpret_cast<const __nv_bfloat16*>(x);
    a.blob = reinterpret_cast<const uint8_t*>(packed);
    a.out = reinterpret_cast<__nv_bfloat16*>(out);
    a.counters = counters;
    a.partials = reinterpret_cast<float*>(partials);
    a.status = status;
    a.L = p.L;
    a.M = M;
    a.K = K;
    a.N = N;
    a.C = p.C;
    a.CS = p.CS;
    a.RB = p.RB;
    a.R = p.R;
    a.grid = p.grid;
    a.stages = p.stages;
    a.stage_bytes = p.stage_bytes;
    a.x_off = p.x_off;
    a.x_stride = p.x_stride;
    a.bar_off = p.bar_off;
    a.cnt_off = p.cnt_off;
    a.misc_off = p.misc_off;
    a.s_max = p.s_max;
    a.part_stride = p.part_stride;
    a.scale_a = scale_a;
    a.scale_b = scale_b;
    a.act = act;
    a.early_weights = early_weights ? 1 : 0;
    a.wait_ns = test_wait_ns();
    a.stall = test_stall();
    a.lora_dg = nullptr;
    a.lora_du = nullptr;
    a.fast = (unsigned long long)p.L * (unsigned long long)p.R < (1ull << 32) ? 1 : 0;
    a.div_R = FastDiv::make((unsigned)p.R);
    a.div_L = FastDiv::make((unsigned)(p.L < (1LL << 32) ? p.L : 1));
    a.div_CS = FastDiv::make((unsigned)p.CS);
    return a;
}

}  // namespace nvf
