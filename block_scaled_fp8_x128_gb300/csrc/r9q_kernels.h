// Internal launch interface between the C ABI (r9q_api.cu) and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>

namespace r9q {

// ---- stream (decode-width) GEMM ----
enum AMode : int { A_QUANT = 0, A_PREQ = 1, A_BF16 = 2 };
enum Epi : int { EPI_STORE = 0, EPI_SWIGLU = 1 };

constexpr int kMaxStages = 4;                    // weight ring depth (runtime 2..4)
constexpr int kCWarps = 8;                       // MMA (mma.sync) or promotion (tcgen05) warps, split-K reduction
constexpr int kStreamThreads = (kCWarps + 2) * 32;   // tcgen05 body: + the TMA producer warp + the MMA warp
// Body of the stream GEMM for a token tile: tcgen05 (r9q_stream.cuh) for
// W8A8 tiles of 16+ rows, where it measured faster; mma.sync
// (r9q_stream_sync.cuh, (kCWarps + 1) * 32 threads) for 8-row W8A8 tiles,
// where the tcgen05 issue/commit/wait round trips cost more than the small
// contraction itself, and for weight-only calls (bf16 activations: the fp8
// tensor cores would need them re-encoded, which measured slower).
constexpr bool stream_uses_tc(int MT, int amode) { return amode != A_BF16 && MT >= 16; }
constexpr int stream_threads(int MT, int amode) {
    return stream_uses_tc(MT, amode) ? kStreamThreads : (kCWarps + 1) * 32;
}
constexpr int kStageBytes = 128 * 128;           // 128 weight rows x 128 k (e4m3)
constexpr int kBarBytes = 256;                   // mbarriers, TMEM address, flags
constexpr int kMaxSplits = 8;                    // cluster size limit (portable)
constexpr int kAccBufs = 4;                      // TMEM k-block partial buffers
constexpr int kMaxRing = 8;                      // tcgen05 body: ring stages incl. the reused activation area
// tcgen05 body barrier area: full/empty per ring stage, the activation copy,
// rfull[2], rfree[2], mdone/tfree per TMEM buffer; then the TMEM address and
// three flags.
static_assert((2 * kMaxRing + 5 + 2 * kAccBufs) * 8 + 8 + 12 <= kBarBytes, "stream barrier area");
// MMA width N of the token tile (tcgen05 at M = 128 takes N a multiple of 16)
// and the TMEM columns a CTA allocates (kAccBufs partials, a power of two).
constexpr int stream_mma_n(int MT) { return MT < 16 ? 16 : MT; }
constexpr int stream_tmem_cols(int MT) { return kAccBufs * stream_mma_n(MT); }
// CTAs per SM that the stream kernel's register budget is compiled for, and
// that the planner counts on (tcgen05 body, 320 threads: 3 CTAs allow 64
// registers a thread, 2 allow 96; mma.sync body, 288 threads: 72 and 112).  W8A8 plans are the same for fused and pre-quantised
// activations (same summation order), so both use the A_QUANT figure.  The
// register budget also bounds the TMEM a SM's resident CTAs hold: at most
// 3 x 64, 2 x 128 or 1 x 256 columns.
constexpr int stream_min_blocks(int MT, int amode) {
    return MT >= 64 ? 1 : MT >= 32 ? 2 : (MT >= 16 && amode == A_BF16) ? 2 : 3;
}

// Split-K exchange of the stream kernel: every rank of a cluster owns a slice
// of each 128-row tile's outputs and receives every rank's partial of that
// slice, [S][stream_recv_rows(S)][MT] fp32 per buffer.  Slices are whole pairs
// of adjacent output columns (so every bf16x2 store is 4-byte aligned): the 64
// row pairs of a tile (plain store), or its 32 pairs of h columns, each with
// its gate and up row (SwiGLU epilogue), split as evenly as the integer
// division q * S / pairs gives.
constexpr int stream_recv_rows(int S) {
    return 2 * ((64 + S - 1) / S) > 4 * ((32 + S - 1) / S) ? 2 * ((64 + S - 1) / S) : 4 * ((32 + S - 1) / S);
}

struct StreamParams {
    const uint16_t* a;   // bf16 activations [M][K]          (A_QUANT, A_BF16)
    uint8_t* aq;         // e4m3 [M][K]: input (A_PREQ) / optional output (A_QUANT)
    float* as;           // fp32 [M][KB]: input (A_PREQ) / optional output (A_QUANT)
    const float* ws;     // fp32 [NB][KB] weight block scales
    uint16_t* y;         // bf16 output [M][ldy] (EPI_STORE: y, EPI_SWIGLU: h)
    int M, K, KB, ldy;
    int splits;          // K splits = cluster size S
    int groups;          // tile groups G: cluster g owns tiles g, g+G, ...
    int ntiles;          // 128-row weight tiles
    int stages;          // ring depth
    int* err;            // device error word
};

// Expert table of the grouped launch (passed by value with the launch).
constexpr int kMaxGroups = 128;
struct GroupTable {
    int zchunks;                 // token chunks (of MT rows) per expert in grid.z
    int wrows;                   // weight rows per expert (N; 2I for the SwiGLU epilogue)
    int off[kMaxGroups + 1];     // expert g's token rows: [off[g], off[g+1])
};

struct StreamPlan {
    int MT;              // token tile: 8, 16, 32 or 64
    int splits;          // cluster size along K
    int groups;          // tile groups
    int ntiles;          // 128-row weight tiles
    int mchunks;         // ceil(M / MT)
    int stages;          // ring depth
    size_t smem;         // dynamic shared memory bytes
};

size_t stream_smem_bytes(int MT, int amode, int S, int kbs_max, int ntl_max, int stages);
// Chooses MT and the split count; returns false when no configuration fits.
bool plan_stream(int64_t M, int64_t N, int64_t K, int amode, int sms, StreamPlan* plan);

cudaError_t launch_stream(const StreamPlan& plan, int amode, int epi, const CUtensorMap& wmap,
                          const StreamParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_stream_a_quant(const StreamPlan& plan, int epi, const CUtensorMap& wmap,
                                  const StreamParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_stream_a_preq(const StreamPlan& plan, int epi, const CUtensorMap& wmap,
                                 const StreamParams& p, cudaStream_t st, bool pdl);
cudaError_t launch_stream_a_bf16(const StreamPlan& plan, int epi, const CUtensorMap& wmap,
                                 const StreamParams& p, cudaStream_t st, bool pdl);

// Grouped launch (A_QUANT or A_BF16 A-loads): grid.z = experts x zchunks.
cudaError_t launch_stream_grouped(const StreamPlan& plan, int amode, int epi, const CUtensorMap& wmap,
                                  const StreamParams& p, const GroupTable& gt, int nexperts, cudaStream_t st,
                                  bool pdl);

// Raises a kernel's dynamic shared memory limit once per device (the attribute
// is not touched again afterwards, so launches can be captured in graphs).
cudaError_t ensure_dynamic_smem(const void* kernel, size_t bytes);

// ---- tcgen05 prefill GEMM (W8A8, M > 64) ----
constexpr int kTcMinM = 33;
size_t tc_smem_bytes();
int tc_max_kb();            // largest K/128 the tensor-core path takes
// Split-K ranks per 128x256 tile for (M, N, K) on `sms` SMs (1 = persistent tiles).
int tc_plan_splits(int64_t M, int64_t N, int64_t K, int sms);
cudaError_t launch_tc_gemm(const CUtensorMap& amap, const CUtensorMap& bmap, const CUtensorMap& ymap,
                           const uint16_t* a, uint8_t* aq, float* as, const float* ws, int* ready, uint16_t* y,
                           int splits, float* part, int* done, int* exits, int M, int N, int K, int* err, int sms,
                           cudaStream_t st);

// The current device's error word (kernels record bounded-wait timeouts there).
int device_error_word(int** out);

// ---- elementwise / quantisation ----
cudaError_t launch_e4m3_from_f32(const float* x, int64_t n, uint8_t* q, cudaStream_t st, int sms);
cudaError_t launch_quant_group128(const uint16_t* x, int64_t M, int64_t K, uint8_t* xq, float* xs,
                                  cudaStream_t st, int sms);
cudaError_t launch_quant_weight_block128(const float* w, int64_t N, int64_t K, uint8_t* wq, float* ws,
                                         cudaStream_t st);
cudaError_t launch_swiglu_interleaved(const uint16_t* gu, int64_t M, int64_t I, uint16_t* h,
                                      cudaStream_t st, int sms);

}  // namespace r9q
