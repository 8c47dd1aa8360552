// stream_gemv.cu -- host side of the decode GEMV family: the SM count, the
// plan queries, the testing switch for the bounded waits and the NVFP4
// launcher.  The kernel template itself is in stream_kernel.cuh.
#include "stream_kernel.cuh"

namespace nvf {

int device_sm_count() {
    static std::atomic<int> cache[64];
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

size_t gemv_partial_bytes(int streams, int M, int N, int K, int num_sms, bool f8) {
    return make_plan(streams, M, N, K, num_sms, f8).total;
}

size_t gemv_counter_bytes(int N) {
    return (size_t)ceil_div((long long)geometry(N, kChunkK).RB * kBlockTiles * 4, 256) * 256;
}

bool gemv_plan_aligned(int streams, int M, int N, int K, int num_sms, bool f8) {
    return plan_aligned(make_plan(streams, M, N, K, num_sms, f8));
}

namespace {
std::atomic<int> g_test_stall{0};
std::atomic<unsigned long long> g_test_wait_ns{kWaitLimitNs};
}  // namespace

void set_test_stall(int stall, unsigned long long wait_ns) {
    g_test_wait_ns.store(wait_ns);
    g_test_stall.store(stall);
}

unsigned long long test_wait_ns() { return g_test_wait_ns.load(); }
int test_stall() { return g_test_stall.load(); }

cudaError_t launch_stream_gemv(int streams, const void* x, int M, int K, const void* packed, int N,
                               float scale_a, float scale_b, int act, void* out, int* status,
                               int* counters, void* partials, size_t partial_bytes, int num_sms,
                               bool early_weights, cudaStream_t s,
                               const void* const* lora_deltas) {
    const Plan p = make_plan(streams, M, N, K, num_sms, false);
    if (partial_bytes < p.total || !plan_aligned(p)) return cudaErrorInvalidValue;
    if (streams != 2 && lora_deltas != nullptr) return cudaErrorInvalidValue;
    KArgs a = make_kargs(p, x, M, K, packed, N, scale_a, scale_b, act, out, status, counters,
                         partials, early_weights);
    a.lora_dg = lora_deltas ? reinterpret_cast<const __nv_bfloat16*>(lora_deltas[0]) : nullptr;
    a.lora_du = lora_deltas ? reinterpret_cast<const __nv_bfloat16*>(lora_deltas[1]) : nullptr;
    // one token tile (M <= 8) always takes element-major partials
    static_assert(kElemMajorMaxM == 8, "element-major partials exactly when NT == 1");
    if ((p.part_stride != 0) != (p.NT == 1)) return cudaErrorInvalidValue;
    const bool coop = use_coop(p, M);
    if (streams == 1) {
        if (M == 1) return launch_t<1, 1, true, true, true, false, false>(p, a, s);
        if (M == 2) return launch_t<1, 1, false, true, true, false, false>(p, a, s);
        if (p.NT == 1)
            return coop ? launch_t<1, 1, false, false, true, false, true>(p, a, s)
                        : launch_t<1, 1, false, false, true, false, false>(p, a, s);
        return coop ? launch_t<1, 2, false, false, false, false, true>(p, a, s)
                    : launch_t<1, 2, false, false, false, false, false>(p, a, s);
    }
    if (M == 1) return launch_t<2, 1, true, true, true, false, false>(p, a, s);
    if (M == 2) return launch_t<2, 1, false, true, true, false, false>(p, a, s);
    if (p.NT == 1)
        return coop ? launch_t<2, 1, false, false, true, false, true>(p, a, s)
                    : launch_t<2, 1, false, false, true, false, false>(p, a, s);
    return coop ? launch_t<2, 2, false, false, false, false, true>(p, a, s)
                : launch_t<2, 2, false, false, false, false, false>(p, a, s);
}

}  // namespace nvf
