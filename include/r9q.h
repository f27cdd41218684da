/*
 * r9q.h — C ABI of libr9q.so: block-scaled fp8 (e4m3) GEMMs for GB300 (sm_103a).
 *
 * The operation: a GEMM y[M][N] = x[M][K] * w[N][K]^T whose weights are OCP
 * FP8 E4M3 codes with one fp32 scale per 128x128 block, accumulated in fp32
 * and written as bf16.  Two modes:
 *   W8A8        — each token's activations are quantised per 128-wide K group
 *                 (scale = amax/448 in fp32, q = e4m3(x/scale) rounded to
 *                 nearest even, saturating to +-448) inside the GEMM's A-load,
 *                 byte-identical to a separate quantisation pass
 *                 (r9700-stack v0.3.1 release notes, "What changed for someone
 *                 running it": fused activation quant in the dense fp8 block
 *                 GEMM, whose off setting restores the separate pass);
 *   weight-only — the fp8 weights against the unquantised bf16 activations
 *                 (same notes: fp8 hyper-connection decode GEMMs, bf16 MMA
 *                 against the unquantised activations).
 * Plus a fused expert MLP: silu(gate)*up in the gate_up GEMM's epilogue and the
 * fp8 row quantisation of that result in the down GEMM's A-load (releases page,
 * v0.3.3 "What changed": the fused MoE decode path).
 *
 * Conventions for every entry point:
 *  - All data pointers are DEVICE pointers owned by the caller.  The library
 *    never allocates device memory and keeps no caller pointer after a call
 *    returns.  Its own device state is two file-scope device arrays: a 4-byte
 *    error word (r9q_last_device_error) and the 1 MiB scratch of
 *    r9q_gate_up_swiglu_down_noalloc.  Their device addresses are looked up
 *    once per device and cached; after cudaDeviceReset those cached
 *    addresses are stale, so the library must not be called on that device
 *    again in the same process.
 *  - Matrices are row-major and contiguous.  bf16 is passed as void* (16-bit
 *    IEEE bfloat16).  e4m3 codes are uint8_t.
 *  - Data pointers (bf16 / e4m3 / outputs) must be 16-byte aligned; fp32
 *    scale pointers 4-byte aligned.
 *  - N, K (and H, I, H_out) must be positive multiples of 128; M >= 1.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Calls are asynchronous: a return of 0 means "enqueued".
 *  - Outputs never alias inputs.  Outputs are fully overwritten.
 *  - Errors are negative return codes (below); on an error nothing has been
 *    enqueued and no CUDA state is changed.  A device-side wait that times out
 *    (it never should) sets a device error word readable with
 *    r9q_last_device_error.
 *  - Calls on one stream are ordered; a workspace may not be shared by calls
 *    that can run concurrently on different streams.
 */
#ifndef R9Q_H_
#define R9Q_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define R9Q_VERSION 1

/* return codes */
#define R9Q_OK              0
#define R9Q_ERR_NULL       -1   /* a required pointer is NULL */
#define R9Q_ERR_DIM        -2   /* bad or unsupported dimensions */
#define R9Q_ERR_ALIGN      -3   /* pointer misaligned */
#define R9Q_ERR_WORKSPACE  -4   /* workspace missing or too small */
#define R9Q_ERR_LAUNCH     -5   /* CUDA launch / runtime error */
#define R9Q_ERR_TIMEOUT    -6   /* a bounded device wait gave up */
#define R9Q_ERR_DEVICE     -7   /* current device is not sm_103 */
#define R9Q_ERR_ARG        -8   /* other invalid argument (flags, op) */

/* Library version (R9Q_VERSION). */
int r9q_version(void);

/* Human-readable text for a return code; never NULL. */
const char* r9q_strerror(int code);

/* Reads and clears the device error word after synchronising `stream`.
 * Returns 0 when no kernel has reported an error since the last call,
 * otherwise the recorded negative code (R9Q_ERR_TIMEOUT). */
int r9q_last_device_error(void* stream);

/* Grouped block-fp8 GEMM: several experts in one launch, for the MoE decode
 * path (releases page, v0.3.3 "What changed": the fused MoE decode path),
 * where each expert's GEMM has only a few tokens.  Expert g multiplies its
 * token rows a[offsets[g] .. offsets[g+1]) by its own weights and writes the
 * same rows of y; experts with no token cost nothing.  Per expert the
 * operation is that of r9q_gemm_fp8_block_qa (W8A8 with the group-128
 * activation quant in the A-load) or, with
 * R9Q_GROUPED_WEIGHT_ONLY, that of r9q_gemm_fp8w_bf16a; with
 * R9Q_GROUPED_SWIGLU the epilogue is that of the gate_up GEMM of
 * r9q_gate_up_swiglu_down (gate/up rows interleaved per 128, h = silu(g)*u).
 *   a_bf16   bf16 [offsets[E]][K], tokens sorted by expert (device)
 *   offsets  int64 [E + 1] on the HOST: offsets[0] = 0, non-decreasing
 *   E        1..128 experts
 *   w        e4m3 [E][N][K] (device), expert g's weights at g*N*K
 *   ws       fp32 [E][N/128][K/128] (device)
 *   y_bf16   bf16 [offsets[E]][N], or [offsets[E]][N/2] with R9Q_GROUPED_SWIGLU
 * N and K multiples of 128 (N of 256 with R9Q_GROUPED_SWIGLU); the fused quant
 * writes no codes out.  Errors: R9Q_ERR_NULL, R9Q_ERR_DIM (sizes, E),
 * R9Q_ERR_ARG (offsets not starting at 0 or decreasing, unknown flags, y
 * overlapping an input), R9Q_ERR_ALIGN, R9Q_ERR_LAUNCH.  offsets[E] = 0 is a
 * no-op.  Allocates nothing; asynchronous on `stream`. */
#define R9Q_GROUPED_WEIGHT_ONLY 1
#define R9Q_GROUPED_SWIGLU      2
int r9q_grouped_gemm_fp8(const void* a_bf16, const int64_t* offsets, int64_t E, const uint8_t* w, const float* ws,
                         void* y_bf16, int64_t N, int64_t K, int flags, void* stream);

/* Failure-detection self-test; the pages have no counterpart.  Launches one
 * small kernel on `stream` whose bounded device waits run out, each on an
 * mbarrier or a counter that nothing ever completes: `which` is a bit set of
 * 1 = the spinning mbarrier wait of the GEMM pipelines, 2 = the sleeping one,
 * 4 = the cluster-scope wait of the split-K reduction, 8 = the counter wait on
 * the prefill kernel's quantised-row counters.  Each selected wait gives up
 * after its bound (up to about a second), the kernel records R9Q_ERR_TIMEOUT
 * in the device error word and returns, and the context stays usable; read
 * the word with r9q_last_device_error.  which = 0 runs the kernel with no
 * wait (nothing is recorded).  Returns R9Q_ERR_ARG for `which` outside 0..15,
 * R9Q_ERR_LAUNCH if the launch fails, else R9Q_OK. */
int r9q_selftest_wait_timeout(int which, void* stream);

/* Programmatic dependent launch of the GEMM entry points (default: off).
 * When on, a GEMM kernel may begin while the kernel launched just before it on
 * the same stream is still running: it starts streaming its weights w at once
 * and waits for that kernel to finish before it reads anything else
 * (activations, scales) or writes anything.  Turn it on only where the kernel
 * launched immediately before each GEMM never writes that GEMM's weights (a
 * decode step: the weights are constant).  Process-wide; returns the previous
 * setting.  The down GEMM inside r9q_gate_up_swiglu_down always uses it (its
 * predecessor is the library's own gate_up kernel). */
int r9q_set_pdl(int enable);

/* fp32 -> e4m3 conversion used by every quantiser: round to nearest even,
 * saturating to +-448 (OCP FP8 E4M3; the saturation rule of the operation's
 * statement).  x: n floats, q: n bytes.  n >= 0 (0 is a no-op). */
int r9q_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, void* stream);

/* Per-token-group-128 activation quantisation (the separate pass of the
 * unfused W8A8 path; r9700-stack v0.3.1 notes: what runs when the fused
 * activation quant is switched off).  x_bf16[M][K] -> xq[M][K] e4m3 codes and
 * xs[M][K/128] fp32 scales, s = amax/448 (fp32 division), q = e4m3(x/s) with
 * one fp32 division per element; an all-zero group gives s = 0 and codes 0. */
int r9q_quant_group128(const void* x_bf16, int64_t M, int64_t K,
                       uint8_t* xq, float* xs, void* stream);

/* The SwiGLU step of the expert MLP as a separate pass (what
 * r9q_gate_up_swiglu_down runs with R9Q_MLP_UNFUSED, and what its fused
 * epilogue reproduces bit for bit; releases page, v0.3.3 "What changed": the
 * fused MoE decode path, silu(gate)*up on the interleaved gate_up output).
 *   gu_bf16[M][2I]: gate and up interleaved per 128 columns, columns
 *     [256j, 256j+128) gate block j, [256j+128, 256j+256) up block j;
 *   h_bf16[M][I]:   h[m][128j+c] = bf16( silu(g) * u ), g = gu[m][256j+c],
 *     u = gu[m][256j+128+c], evaluated in fp32 as e = exp(-g), g / (1 + e),
 *     times u, one IEEE rounding per step; exp is the library's own (Cody and
 *     Waite's reduction with a degree-7 Taylor polynomial, under 1 ulp), so
 *     the result is the same on every GPU and driver.
 * I a positive multiple of 128, M >= 1; both pointers 16-byte aligned, h
 * not overlapping gu.  Errors: R9Q_ERR_NULL, R9Q_ERR_DIM, R9Q_ERR_ALIGN,
 * R9Q_ERR_ARG (overlap), R9Q_ERR_DEVICE, R9Q_ERR_LAUNCH. */
int r9q_swiglu_interleaved(const void* gu_bf16, int64_t M, int64_t I, void* h_bf16, void* stream);

/* Weight quantisation with one fp32 scale per 128x128 block (set-up, not the
 * hot path): w[N][K] fp32 -> wq[N][K] e4m3, ws[N/128][K/128] fp32,
 * s = amax/448 over the block, q = e4m3(w/s). */
int r9q_quant_weight_block128(const float* w, int64_t N, int64_t K,
                              uint8_t* wq, float* ws, void* stream);

/* W8A8 block-fp8 GEMM (r9700-stack v0.3.1 notes: r9k_gemm_fp8_block_qa;
 * v0.3.0 notes: exact block-scaled fp8 GEMM).
 *   y[m][n] = bf16( sum_kb P[m][n][kb] * as[m][kb] * ws[n/128][kb] ),
 *   P[m][n][kb] = sum_{k in block kb} e4m3(aq[m][k]) * e4m3(w[n][k]) in fp32.
 * Fused mode (a_bf16 != NULL): the activations are quantised per token and
 *   128-wide K group inside the kernel; aq[M][K] / as[M][K/128] are then
 *   OPTIONAL outputs (either both NULL or both set) that receive exactly the
 *   bytes and scales r9q_quant_group128 produces.
 * Unfused mode (a_bf16 == NULL): aq / as are required inputs.
 * w[N][K] e4m3, ws[N/128][K/128] fp32, y_bf16[M][N].
 * workspace: query r9q_workspace_bytes(R9Q_OP_GEMM_W8A8, ...); when it
 *   reports 0 bytes, workspace may be NULL.  From M = 33 on (the tensor-core
 *   path) the workspace holds the quantised A, the split-K partials of shapes
 *   with few 128x256 tiles, and a 64 KiB header of counters: zero the whole
 *   workspace once before its first use (cudaMemset); every call that
 *   returns R9Q_OK and whose kernel completes leaves the header at zero again,
 *   so one workspace can serve any sequence of shapes on one stream.  After a
 *   call that recorded a device error (r9q_last_device_error), zero it again.
 *   Calls that may run at the same time on the GPU need separate workspaces. */
int r9q_gemm_fp8_block_qa(const void* a_bf16, uint8_t* aq, float* as,
                          const uint8_t* w, const float* ws, void* y_bf16,
                          int64_t M, int64_t N, int64_t K,
                          void* workspace, size_t workspace_bytes, void* stream);

/* Weight-only fp8 GEMM: y[m][n] = bf16( sum_kb (sum_{k in kb} x[m][k] * e4m3(w[n][k])) * ws[n/128][kb] )
 * with x the unquantised bf16 activations (r9700-stack v0.3.1 notes: fp8
 * hyper-connection decode GEMMs).  Products are exact in fp32 (the e4m3
 * weights are converted exactly to bf16 in registers). */
int r9q_gemm_fp8w_bf16a(const void* a_bf16, const uint8_t* w, const float* ws, void* y_bf16,
                        int64_t M, int64_t N, int64_t K,
                        void* workspace, size_t workspace_bytes, void* stream);

/* Flags of r9q_gate_up_swiglu_down. */
#define R9Q_MLP_WEIGHT_ONLY 1   /* both GEMMs weight-only (no quant of x or h) */
#define R9Q_MLP_UNFUSED     2   /* run the separate-launch chain instead of the fused one */

/* Expert MLP at decode (releases page, v0.3.3 "What changed": fused MoE decode
 * path, silu(gate)*up in the gate_up GEMM's epilogue, the fp8 row quant inside
 * the down GEMM's A-load, outputs bit-identical to the separate-launch path).
 *   gu = GEMM(x, w_gu) with w_gu[2I][H] holding gate and up interleaved per
 *        128 rows: rows [256j, 256j+128) are gate block j, rows
 *        [256j+128, 256j+256) up block j; s_gu[2I/128][H/128];
 *   h[m][128j+c] = bf16( silu(g) * u ), g = bf16(gu[m][256j+c]),
 *        u = bf16(gu[m][256j+128+c]);
 *   y = GEMM(h, w_dn) with w_dn[H_out][I], s_dn[H_out/128][I/128],
 *        h quantised per token and 128-wide group in the A-load (W8A8).
 * Both GEMMs are W8A8 (x quantised in the gate_up A-load) unless
 * R9Q_MLP_WEIGHT_ONLY.  h_bf16_out[M][I], hq_out[M][I], hs_out[M][I/128] are
 * optional outputs (hq/hs only in W8A8 mode; both or neither).  R9Q_MLP_UNFUSED
 * runs gate_up GEMM -> SwiGLU -> quant -> down GEMM as separate launches and
 * gives bit-identical outputs.  workspace: r9q_workspace_bytes(
 * R9Q_OP_GATE_UP_SWIGLU_DOWN, M, I, H, H_out, flags, &bytes). */
int r9q_gate_up_swiglu_down(const void* x_bf16,
                            const uint8_t* w_gu, const float* s_gu,
                            const uint8_t* w_dn, const float* s_dn,
                            void* y_bf16, int64_t M, int64_t H, int64_t I, int64_t H_out,
                            void* h_bf16_out, uint8_t* hq_out, float* hs_out, int flags,
                            void* workspace, size_t workspace_bytes, void* stream);

/* Allocation-free variant of r9q_gate_up_swiglu_down, for callers that cannot
 * allocate device memory where they run the MLP (an arena or pool owner that
 * hands out no scratch, a plug-in that only receives its input and output
 * buffers, code that must not call cudaMalloc).  The pages have no counterpart:
 * this is a library convenience.  Same arguments and results as the fused path
 * of r9q_gate_up_swiglu_down (flags may hold R9Q_MLP_WEIGHT_ONLY; R9Q_MLP_UNFUSED
 * is rejected with R9Q_ERR_ARG) except that there is no h output and no
 * workspace: h lives in a scratch array inside the library, 1 MiB per GPU held
 * from load until process exit, so M * I must not exceed 524288 (larger sizes
 * return R9Q_ERR_WORKSPACE).  The call allocates nothing.  The first call on a
 * device looks up that device's scratch address (cudaGetSymbolAddress with the
 * device current), so make that first call before capturing a stream.  All
 * calls share the one scratch array, which is fully rewritten by each call:
 * calls that can overlap on the GPU (different streams) race on it. */
int r9q_gate_up_swiglu_down_noalloc(const void* x_bf16,
                                    const uint8_t* w_gu, const float* s_gu,
                                    const uint8_t* w_dn, const float* s_dn,
                                    void* y_bf16, int64_t M, int64_t H, int64_t I, int64_t H_out,
                                    uint8_t* hq_out, float* hs_out, int flags, void* stream);

/* Workspace query. */
#define R9Q_OP_GEMM_W8A8            1   /* (M, N, K) */
#define R9Q_OP_GEMM_W8BF16          2   /* (M, N, K) */
#define R9Q_OP_GATE_UP_SWIGLU_DOWN  3   /* (M, N=I, K=H, N2=H_out, flags) */
/* Writes the bytes of device workspace the call needs (0 = none) to *bytes. */
int r9q_workspace_bytes(int op, int64_t M, int64_t N, int64_t K, int64_t N2, int flags,
                        size_t* bytes);

#ifdef __cplusplus
}
#endif
#endif /* R9Q_H_ */
