// stream_gemv_fp8.cu -- launcher of the decode GEMV kernels on block-scaled
// FP8 weights (the dense-FFN page's native FP8 arm: w8a16_gemv_dual for gate
// and up with the activation, then the down projection on h).  The kernel
// template is in stream_kernel.cuh; this translation unit instantiates its F8
// variants, so they compile beside the NVFP4 ones.
#include "stream_kernel.cuh"

namespace nvf {

cudaError_t launch_stream_gemv_f8(int streams, const void* x, int M, int K, const void* packed,
                                  int N, int act, void* out, int* status, int* counters,
                                  void* partials, size_t partial_bytes, int num_sms,
                                  bool early_weights, cudaStream_t s) {
    const Plan p = make_plan(streams, M, N, K, num_sms, true);
    if (partial_bytes < p.total || !plan_aligned(p)) return cudaErrorInvalidValue;
    // no per-tensor scale: the block scales are applied inside the sum
    const KArgs a = make_kargs(p, x, M, K, packed, N, 1.0f, 1.0f, act, out, status, counters,
                               partials, early_weights);
    // one token tile (M <= 8) always takes element-major partials
    static_assert(kElemMajorMaxM == 8, "element-major partials exactly when NT == 1");
    if ((p.part_stride != 0) != (p.NT == 1)) return cudaErrorInvalidValue;
    const bool coop = use_coop(p, M);
    if (streams == 1) {
        if (M == 1) return launch_t<1, 1, true, false, true, true, false>(p, a, s);
        if (p.NT == 1)
            return coop ? launch_t<1, 1, false, false, true, true, true>(p, a, s)
                        : launch_t<1, 1, false, false, true, true, false>(p, a, s);
        return coop ? launch_t<1, 2, false, false, false, true, true>(p, a, s)
                    : launch_t<1, 2, false, false, false, true, false>(p, a, s);
    }
    if (M == 1) return launch_t<2, 1, true, false, true, true, false>(p, a, s);
    if (p.NT == 1)
        return coop ? launch_t<2, 1, false, false, true, true, true>(p, a, s)
                    : launch_t<2, 1, false, false, true, true, false>(p, a, s);
    return coop ? launch_t<2, 2, false, false, false, true, true>(p, a, s)
                : launch_t<2, 2, false, false, false, true, false>(p, a, s);
}

}  // namespace nvf
