/*
 * nvfp4ffn.h -- C ABI of libnvfp4ffn.so: NVFP4 weight-only SwiGLU FFN decode
 * on one NVIDIA GB300 (sm_103a).
 *
 *   out[M, H] = down( act( gate(x) ) * up(x) ),   M = 1..16 per kernel pass
 *   (up to 64 rows per call, in passes of 16),
 *   x, out BF16;  gate [I, H], up [I, H], down [H, I] NVFP4;  act = SiLU | GeLU-tanh.
 *
 * Beside it: a LoRA delta overlay on the same FFN, and the FFN and GEMV on
 * block-scaled FP8 weights (the w8a16 calls near the end of this header).
 *
 * What the calls restate (Atlas engine pages):
 *  - "spark_model/layers/dense_ffn.rs", module doc comment: the dense SwiGLU
 *    FFN, the gated product of the gate and up projections of x fed to the
 *    down projection, with the weights dequantised inside the dot product.
 *  - same page, doc comment of DenseFfnLayer::ensure_int8_weight: an NVFP4
 *    projection is packed E2M1 codes [N, K/2], one E4M3 scale per 16 K
 *    elements [N, K/16], and one FP32 `weight_scale_2` per tensor.
 *  - same page, DenseFfnLayer::forward: the decode FFN as a dual gate+up GEMV
 *    followed by the activation and a down GEMV; forward_km / forward_k2 /
 *    forward_k3: the same for M verify rows, each weight read once for all M.
 *  - same page, DenseFfnLayer::ensure_nvfp4_mmq_weight: a load-time repack of
 *    the checkpoint NVFP4 into a kernel layout that is a raw bit shuffle of the
 *    same codes and scale bytes.
 *  - "spark_model/weight_loader/qwen35_dense.rs", load_layers: BF16/FP32
 *    weights become NVFP4 at load time through a global-absmax kernel and a
 *    quantize kernel (quantize_to_nvfp4).
 *
 * Conventions for every call:
 *  - Pointers marked (device) are device pointers owned by the caller; the
 *    library never frees them and keeps no reference after the call returns.
 *  - Calls are asynchronous on `stream` unless marked "synchronises".
 *  - The return value is a status; nothing aborts or throws across the ABI.
 *    Argument errors are detected on the host before any launch; a failed
 *    launch is reported as NVFP4_ERR_CUDA with the CUDA error left readable
 *    through cudaGetLastError().
 *  - BF16 tensors are row-major with a row stride equal to their width.
 *  - Device pointers must be 16-byte aligned.
 *  - Every GEMV/FFN pass (up to 16 rows) reads its weights once and sums
 *    split-K partials in a fixed order, so results are bit-reproducible.
 *  - The GEMV/FFN and LoRA kernels use programmatic dependent launch: they
 *    may start while the preceding kernel on `stream` is still finishing and
 *    begin reading their (repacked) weights or adapter matrices at once; they
 *    read x and write every output only after that kernel has completed.  So
 *    the weight and adapter buffers must not be written by the kernel issued
 *    immediately before the call on the same stream.  This library's
 *    quantise and repack calls are safe predecessors (their blocks fence
 *    their stores before exiting).
 *  - The GEMV/FFN kernels launch one block per SM.  With 4 or more token rows
 *    a launch may finish its split row blocks cooperatively: its blocks then
 *    wait for one another, which assumes that every block of the launch can
 *    be resident at once.  Two such calls overlapping on the GPU (issued on
 *    different streams or from different threads or processes sharing the
 *    SMs) can each hold SMs that the other's blocks need; their waits then
 *    give up after about a second and the call reports NVFP4_ERR_TIMEOUT
 *    (nvfp4_workspace_status).  Issue the calls for one device on one stream,
 *    or order the streams with events.
 */
#ifndef NVFP4FFN_H
#define NVFP4FFN_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_NULL = 1,      /* a required pointer is NULL */
    NVFP4_ERR_SHAPE = 2,     /* a size is <= 0, or K/H/I is not a multiple of 16 */
    NVFP4_ERR_ALIGN = 3,     /* a device pointer is not 16-byte aligned */
    NVFP4_ERR_RANGE = 4,     /* M outside the call's range, or an unknown enum value */
    NVFP4_ERR_WORKSPACE = 5, /* workspace smaller than the size query returns */
    NVFP4_ERR_CUDA = 6,      /* a CUDA runtime call or launch failed */
    NVFP4_ERR_TIMEOUT = 7,   /* a kernel gave up on a bounded wait (device status word) */
    NVFP4_ERR_ALIAS = 8      /* input and output buffers overlap */
} nvfp4_status;

/* Gating nonlinearity (enum FfnActivation on the dense-FFN page).
 * SiLU(t) = t / (1 + e^-t); GeLU-tanh(t) = 0.5 t (1 + tanh(sqrt(2/pi)(t + 0.044715 t^3))). */
typedef enum { NVFP4_ACT_SILU = 0, NVFP4_ACT_GELU_TANH = 1 } nvfp4_act;

/* Element type of the weight handed to nvfp4_quantize. */
typedef enum { NVFP4_SRC_F32 = 0, NVFP4_SRC_BF16 = 1 } nvfp4_src_dtype;

/* ------------------------------------------------------------------ quantise */

/* Bytes of scratch nvfp4_quantize needs (a few words; independent of N, K). */
size_t nvfp4_quantize_scratch_bytes(int N, int K);

/*
 * Quantise a weight W [N, K] (row-major, fp32 or bf16, device) to NVFP4 in the
 * canonical checkpoint layout ("spark_model/weight_loader/qwen35_dense.rs",
 * load_layers: global absmax, then quantize):
 *   amax   = max |W|;  scale2 = amax / 2688 (= 6 * 448), or 1 when amax == 0
 *   per 16-element block b of a row:  s_b = E4M3(bamax_b / 6 / scale2)
 *   per element:  code = E2M1(w / (E4M3value(s_b) * scale2))   (code 0 with
 *   the element's sign when s_b == 0)
 * in IEEE fp32 with that operation order; both conversions round to nearest,
 * ties to even, saturate at the largest finite value and keep the sign.
 *   codes  (device, out) u8 [N, K/2]: element 2j in the low nibble of byte j.
 *   scales (device, out) u8 [N, K/16]: E4M3 ("fn": bias 7, max 448).
 *   scale2_out (host, out): the per-tensor FP32 scale.  A device copy is left
 *   at byte offset 4 of `scratch`.
 *   scratch (device) >= nvfp4_quantize_scratch_bytes(N, K).
 * Requirements: N >= 1, K >= 16, K % 16 == 0, W finite.
 * Synchronises `stream` (it reads scale2 back to the host): a load-time call.
 */
nvfp4_status nvfp4_quantize(const void* w, nvfp4_src_dtype dtype, int N, int K,
                            uint8_t* codes, uint8_t* scales, float* scale2_out,
                            void* scratch, size_t scratch_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ repack */

/*
 * Kernel layout ("fragment layout"): a byte permutation of the canonical codes
 * and scales (the principle of DenseFfnLayer::ensure_nvfp4_mmq_weight: same
 * codes, same scale bytes, no numerics), zero-padded to N' = roundup(N, 256)
 * rows and K' = roundup(K, 256) columns.  For N % 256 == 0 and K % 256 == 0 it
 * holds exactly the canonical byte count N*K*9/16.  The layout is opaque to
 * callers; nvfp4_unpack inverts it.
 */
size_t nvfp4_repacked_bytes(int N, int K);

/* codes [N, K/2], scales [N, K/16] (device, canonical) -> packed (device,
 * nvfp4_repacked_bytes(N, K) bytes).  N >= 1, K % 16 == 0. */
nvfp4_status nvfp4_repack(const uint8_t* codes, const uint8_t* scales, int N, int K,
                          void* packed, cudaStream_t stream);

/* Gate and up projections ([I, H] each) interleaved so that one kernel reads
 * gate row n and up row n together: 2 * nvfp4_repacked_bytes(I, H) bytes. */
size_t nvfp4_repacked_gate_up_bytes(int I, int H);
nvfp4_status nvfp4_repack_gate_up(const uint8_t* gate_codes, const uint8_t* gate_scales,
                                  const uint8_t* up_codes, const uint8_t* up_scales,
                                  int I, int H, void* packed, cudaStream_t stream);

/* Inverse of nvfp4_repack (a test and inspection aid): packed -> canonical
 * codes [N, K/2] and scales [N, K/16] (device). */
nvfp4_status nvfp4_unpack(const void* packed, int N, int K, uint8_t* codes,
                          uint8_t* scales, cudaStream_t stream);

/* ------------------------------------------------------------------ GEMV */

/*
 * Workspace bytes for nvfp4_gemv on the current device (cross-CTA partial
 * sums and their counters); 0 for invalid sizes or N > 524288.
 * Workspace contract (all GEMV/FFN calls): zero-fill the workspace once after
 * it is allocated (cudaMemset or nvfp4_workspace_init).  Every call that
 * completes normally leaves it ready for the next one, whatever the next
 * call's entry point and shape, provided the workspace is large enough for
 * that call.  Calls sharing one workspace must be ordered (one stream).
 */
size_t nvfp4_gemv_workspace_bytes(int M, int N, int K);

/*
 * One NVFP4 projection (the w4a16 decode GEMV of "spark_model/layers/
 * dense_ffn.rs", DenseFfnLayer::forward / forward_km):
 *   y[m, n] = bf16( scale2 * sum_k x[m, k] * E2M1(c[n, k]) * E4M3(s[n, k/16]) )
 *   x (device) bf16 [M, K];  packed_w (device) from nvfp4_repack(N, K);
 *   y (device, out) bf16 [M, N];  ws (device) >= nvfp4_gemv_workspace_bytes.
 * Requirements: 1 <= M <= 64, N >= 1, K >= 16, K % 16 == 0, x and y disjoint.
 * Accumulation is fp32 on exactly dequantised weights; every x row is scaled
 * by a power of two into the fp16 operand range, so any finite bf16 x works.
 * The kernels take up to 16 token rows at a time: M > 16 (a verify batch or a
 * small prefill, the page's forward_prefill range M <= 64) runs as groups of
 * 16 rows and a remainder, each group streaming the weights once.
 */
nvfp4_status nvfp4_gemv(const void* x, int M, int K, const void* packed_w, float scale2,
                        int N, void* y, void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ FFN */

/* Workspace bytes for ffn_swiglu_nvfp4 on the current device: the bf16
 * activation h [M, I] plus the partial sums of both kernels (0 for invalid
 * sizes or I + H above about 524288).  Contract as for nvfp4_gemv. */
size_t ffn_swiglu_nvfp4_workspace_bytes(int M, int H, int I);

/* Byte offset inside an ffn_swiglu_nvfp4 workspace of the bf16 activation
 * h [M, I] (row-major) that the call leaves there (an inspection aid). */
size_t ffn_swiglu_nvfp4_hidden_offset(void);

/*
 * The decode FFN (DenseFfnLayer::forward and forward_km on the dense-FFN
 * page), in two launches:
 *   1. g = bf16(gate_scale2 * gate.x),  u = bf16(up_scale2 * up.x),
 *      h = bf16(act(g) * u)                      [M, I] bf16, in ws
 *   2. out = bf16(down_scale2 * down.h)          [M, H] bf16
 *   x (device) bf16 [M, H];  gate_up_packed (device) from
 *   nvfp4_repack_gate_up(I, H);  down_packed (device) from nvfp4_repack(H, I);
 *   out (device, out) bf16 [M, H];  ws (device) >= ffn_swiglu_nvfp4_workspace_bytes.
 * Requirements: 1 <= M <= 64, H and I >= 16 and multiples of 16, x and out
 * disjoint, act a nvfp4_act value.  M > 16 runs in groups of 16 rows, as for
 * nvfp4_gemv.
 */
nvfp4_status ffn_swiglu_nvfp4(const void* x, int M, int H, int I,
                              const void* gate_up_packed, float gate_scale2, float up_scale2,
                              const void* down_packed, float down_scale2, nvfp4_act act,
                              void* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes for ffn_gate_up_nvfp4 on the current device (zero-fill once). */
size_t ffn_gate_up_nvfp4_workspace_bytes(int M, int H, int I);

/*
 * The gate/up half of the FFN alone (step 1 of ffn_swiglu_nvfp4; the fused
 * dual GEMV + activation of DenseFfnLayer::forward on the dense-FFN page):
 *   h[m, i] = bf16( act(bf16(gate_scale2 * gate.x)) * bf16(up_scale2 * up.x) )
 *   x (device) bf16 [M, H];  gate_up_packed (device) from nvfp4_repack_gate_up;
 *   h (device, out) bf16 [M, I];  ws (device) >= ffn_gate_up_nvfp4_workspace_bytes.
 * A caller that adds its own terms to h (an adapter) finishes the layer with
 * nvfp4_gemv on the down projection.  Requirements as for ffn_swiglu_nvfp4.
 */
nvfp4_status ffn_gate_up_nvfp4(const void* x, int M, int H, int I, const void* gate_up_packed,
                               float gate_scale2, float up_scale2, nvfp4_act act, void* h,
                               void* ws, size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ LoRA overlay */

/*
 * The adapter overlay of the dense-FFN page (DenseFfnLayer::apply_lora_gate_up
 * and apply_lora_down): gate and up take dW x after their projections and
 * before the activation, the output takes dW h after the down projection,
 * contracted over the activation h.  dW = B A with A [r, in] and B [out, r]
 * bf16 row-major (device), 1 <= r <= 64; any alpha/r is folded into B.  Each
 * intermediate is bf16: xa = bf16(A v), d = bf16(B xa), base = bf16(base + d).
 */

/* Workspace bytes for ffn_swiglu_nvfp4_lora (the FFN's plus the adapter
 * intermediates); contract as for nvfp4_gemv. */
size_t ffn_swiglu_nvfp4_lora_workspace_bytes(int M, int H, int I, int rank);

/*
 * ffn_swiglu_nvfp4 with the overlay:
 *   g = bf16(bf16(gate_scale2 * gate.x) + bf16(Bg bf16(Ag x)))   (likewise u)
 *   h = bf16(act(g) * u),  out = bf16(bf16(down_scale2 * down.h) + bf16(Bd bf16(Ad h)))
 * gate_a [r, H] / gate_b [I, r], up_a [r, H] / up_b [I, r], down_a [r, I] /
 * down_b [H, r] (device, bf16); a pair given as two NULL pointers is absent
 * (its delta is zero).  A pair with one NULL pointer is NVFP4_ERR_NULL; rank
 * outside [1, 64] is NVFP4_ERR_RANGE.  Other arguments and requirements as
 * ffn_swiglu_nvfp4, except 1 <= M <= 16.  Up to four small launches join the
 * FFN's two.
 */
nvfp4_status ffn_swiglu_nvfp4_lora(const void* x, int M, int H, int I,
                                   const void* gate_up_packed, float gate_scale2,
                                   float up_scale2, const void* down_packed,
                                   float down_scale2, nvfp4_act act, int rank,
                                   const void* gate_a, const void* gate_b, const void* up_a,
                                   const void* up_b, const void* down_a, const void* down_b,
                                   void* out, void* ws, size_t ws_bytes, cudaStream_t stream);

/* Scratch bytes for nvfp4_lora_apply (fp32 partial sums of a v over K slices;
 * independent of K). */
size_t nvfp4_lora_apply_scratch_bytes(int M, int rank);

/*
 * The page's apply_lora_delta on its own: base[m][n] = bf16(base[m][n] +
 * bf16(sum_j b[n][j] xa[m][j])) with xa = bf16(a v):  v (device) bf16 [M, K],
 * a [rank, K], b [N, rank] (device, bf16), base (device, in/out) bf16 [M, N],
 * scratch (device) >= nvfp4_lora_apply_scratch_bytes.  1 <= M <= 16, K even,
 * v and base disjoint.
 */
nvfp4_status nvfp4_lora_apply(const void* v, int M, int K, const void* a, const void* b,
                              int rank, int N, void* base, void* scratch, size_t scratch_bytes,
                              cudaStream_t stream);

/*
 * ffn_swiglu_nvfp4 (1 <= M <= 16) for callers that cannot allocate device
 * memory where they run the FFN (a process that reserves the device's memory for its own pool at
 * start-up and forbids later cudaMalloc, or code that must not risk the
 * implicit device synchronisation of an allocation).  The pages have no
 * counterpart of this call; it exists for such callers.
 *   Same arguments and results as ffn_swiglu_nvfp4, without ws/ws_bytes: the
 *   workspace is one library-owned device array of 24 MiB, held by every GPU
 *   that loads the library until the process exits.  Shapes whose
 *   ffn_swiglu_nvfp4_workspace_bytes exceeds 24 MiB are rejected with
 *   NVFP4_ERR_WORKSPACE (M = 16 at H = 5376, I = 21504 needs about 21 MiB).
 *   Every argument is checked before anything is touched: a rejected call
 *   changes nothing on the device.
 *   The first call on each device (with that device current) resolves the
 *   array's device address (cudaGetSymbolAddress) and zero-fills the array on
 *   `stream`, synchronising it; make that first call before any stream
 *   capture.  Later calls only enqueue the two FFN kernels on `stream`: like
 *   ffn_swiglu_nvfp4's workspace, the array is left ready for the next call by
 *   every call that completes normally.  The call allocates nothing.
 *   Every call shares the one array, so calls that overlap on the GPU
 *   (different streams without ordering between them) race and corrupt each
 *   other's results.
 *   A call whose kernel abandoned a bounded wait is reported only by
 *   nvfp4_noalloc_status, which also repairs the array; until it is called,
 *   later calls may return wrong results.
 */
nvfp4_status ffn_swiglu_nvfp4_noalloc(const void* x, int M, int H, int I,
                                      const void* gate_up_packed, float gate_scale2,
                                      float up_scale2, const void* down_packed, float down_scale2,
                                      nvfp4_act act, void* out, cudaStream_t stream);

/*
 * Status of ffn_swiglu_nvfp4_noalloc calls on the current device, the
 * counterpart of nvfp4_workspace_status for the library's fixed array (no
 * counterpart on the pages).  Synchronises `stream`, reads and clears the
 * array's status word: NVFP4_OK, or NVFP4_ERR_TIMEOUT when a kernel abandoned
 * a bounded wait since the last check, in which case the whole array is
 * zero-filled again (on `stream`, synchronised) so the next call starts clean.
 * Performs the first-call set-up if no call has yet run on this device.
 */
nvfp4_status nvfp4_noalloc_status(cudaStream_t stream);

/* ------------------------------------------------------ block-scaled FP8 (w8a16) */

/*
 * The dense-FFN page's native FP8 arm (DenseFfnWeightsFp8 and set_fp8_weights;
 * the FP8 dispatch of DenseFfnLayer::forward: w8a16_gemv_dual for gate and up,
 * then w8a16_gemv_silu_input for the down projection on the activation),
 * weights used as loaded, with no NVFP4 requantisation.  A projection [N, K]:
 *   codes (device) E4M3 bytes [N, K] row-major, the "fn" variant (0x7F/0xFF
 *         are NaN, outside the contract);
 *   grid  (device) fp32 [ceil(N/128), ceil(K/128)] row-major, 4-byte aligned;
 *   W[n][k] = e4m3(codes[n][k]) * grid[n/128][k/128]  (the block grid the
 *   weight loader's proj_is_fp8_any_scale accepts; a per-tensor scalar scale
 *   is the uniform grid).
 * The roundings are those of the NVFP4 path: g, u, h and out are bf16.  Every
 * call below follows the conventions of its NVFP4 counterpart (status codes,
 * validation before any launch, asynchronous on `stream`, the workspace
 * contract, M up to 64 in groups of 16, K/H/I multiples of 16).
 */

/* Bytes of a repacked FP8 projection [N, K] / gate+up pair [I, H] (0 for
 * invalid sizes): the codes, padded to 256 rows and 256 K, plus one fp32
 * scale per 16 rows and 64 K. */
size_t w8a16_repacked_bytes(int N, int K);
size_t w8a16_repacked_gate_up_bytes(int I, int H);

/* Canonical FP8 -> kernel layout (codes permuted, grid entries copied per
 * 16-row tile and 64-K chunk; no arithmetic).  packed (device, out) >=
 * w8a16_repacked_bytes(N, K), 16-byte aligned. */
nvfp4_status w8a16_repack(const uint8_t* codes, const float* grid, int N, int K, void* packed,
                          cudaStream_t stream);

/* Gate and up [I, H] into one blob (each tile's gate and up codes back to
 * back), >= w8a16_repacked_gate_up_bytes(I, H). */
nvfp4_status w8a16_repack_gate_up(const uint8_t* gate_codes, const float* gate_grid,
                                  const uint8_t* up_codes, const float* up_grid, int I, int H,
                                  void* packed, cudaStream_t stream);

/* Inverse of w8a16_repack (a test aid): codes [N, K] and grid. */
nvfp4_status w8a16_unpack(const void* packed, int N, int K, uint8_t* codes, float* grid,
                          cudaStream_t stream);

/* Workspace bytes for w8a16_gemv; contract as for nvfp4_gemv. */
size_t w8a16_gemv_workspace_bytes(int M, int N, int K);

/*
 * y[m][n] = bf16(sum_k x[m][k] * W[n][k]) for the FP8 projection (the page's
 * w8a16_gemv):  x (device) bf16 [M, K];  packed_w from w8a16_repack(N, K);
 * y (device, out) bf16 [M, N];  ws >= w8a16_gemv_workspace_bytes.
 */
nvfp4_status w8a16_gemv(const void* x, int M, int K, const void* packed_w, int N, void* y,
                        void* ws, size_t ws_bytes, cudaStream_t stream);

/* Workspace bytes for ffn_swiglu_w8a16; h [M, I] lies at
 * ffn_swiglu_nvfp4_hidden_offset() in it, as for ffn_swiglu_nvfp4. */
size_t ffn_swiglu_w8a16_workspace_bytes(int M, int H, int I);

/*
 * The decode FFN on FP8 weights, in two launches:
 *   1. g = bf16(gate.x), u = bf16(up.x), h = bf16(act(g) * u)   [M, I] in ws
 *   2. out = bf16(down.h)                                        [M, H]
 *   gate_up_packed from w8a16_repack_gate_up(I, H); down_packed from
 *   w8a16_repack(H, I); other arguments as ffn_swiglu_nvfp4.
 */
nvfp4_status ffn_swiglu_w8a16(const void* x, int M, int H, int I, const void* gate_up_packed,
                              const void* down_packed, nvfp4_act act, void* out, void* ws,
                              size_t ws_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------ utilities */

/* Zero-fill a workspace (asynchronous memset on `stream`). */
nvfp4_status nvfp4_workspace_init(void* ws, size_t ws_bytes, cudaStream_t stream);

/*
 * Synchronises `stream`, then reads and clears the device status word at the
 * start of a GEMV/FFN workspace: NVFP4_OK, or NVFP4_ERR_TIMEOUT when a kernel
 * abandoned a bounded wait since the last check.  A kernel that gave up may
 * leave the workspace's split-K counters off zero: after NVFP4_ERR_TIMEOUT,
 * zero-fill the workspace again (nvfp4_workspace_init) before reusing it.
 */
nvfp4_status nvfp4_workspace_status(void* ws, cudaStream_t stream);

/* Static, human-readable name of a status code. */
const char* nvfp4_status_string(nvfp4_status status);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4FFN_H */
