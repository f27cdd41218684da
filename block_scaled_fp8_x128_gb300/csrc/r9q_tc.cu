// Prefill-width block-scaled fp8 GEMM on the 5th-generation tensor cores
// (tcgen05 + TMEM), sm_103a.  W8A8 only; r9q_gemm_fp8_block_qa sends every
// call with M >= 33 here (split-K over the grid while the tiles are few).
//
// The contraction is dense here (r9700-stack v0.3.0 notes: fp8 GEMMs on the
// tiled tensor-core kernel at prefill sizes, and the exact block-scaled fp8
// variant), so it runs on tcgen05:
//  * persistent CTAs (one per SM) walk 128x256 output tiles in m-major order;
//  * warp 0 streams A (128x128 e4m3) and B (256x128 e4m3) k-blocks with 2-D
//    TMA, 128-byte swizzle, into a 3-stage shared-memory ring;
//  * warp 1 issues tcgen05.mma.kind::f8f6f4 (M=128, N=256, K=32; four per
//    128-wide k-block) into one of two TMEM partial buffers (2 x 256 fp32
//    columns) and commits the stage and the buffer to mbarriers;
//  * warps 4..11 (two warpgroups, 128 columns each) tcgen05.ld every k-block's
//    partial and promote it into register accumulators with
//    as[m][kb] * ws[nb][kb] -- the fp32 block scales cannot enter the MMA, so
//    they are applied per k-block exactly as the block-scaled definition reads,
//    while the tensor cores fill the other buffer;
//  * the finished tile goes out as bf16 through a swizzled shared-memory
//    staging area and TMA stores.
// Fused activation quant (a_bf16 given): before taking up their roles, all
// warps of the grid quantise each A row exactly once, per 128-wide group, into
// a global scratch copy (aq/as) that the A loads read, dealing rows out in
// global order and counting finished rows per m-tile; the A loads (and the
// scale reads) of an m-tile wait (bounded) until its rows are all in.  The
// codes and scales are those of the standalone quant kernel, bit for bit.
// Split-K mode (few tiles, e.g. M of a few hundred rows): the grid holds S CTAs
// per tile, each owning a contiguous range of k-blocks; a CTA writes its fp32
// partial tile to scratch and publishes it on the tile's counter (release);
// once all S are in (acquire), CTA rank r sums rows [r*128/S, (r+1)*128/S) of
// the S partials in rank order (deterministic) and stores bf16.  The grid is
// cooperative, so every CTA a tile waits for is resident.
// All waits are bounded: a timeout records R9Q_ERR_TIMEOUT, the kernel drains
// what it issued, frees its TMEM and returns.
#include "r9q_device.cuh"
#include "r9q_kernels.h"

namespace r9q {

namespace tc {

constexpr int BM = 128, BN = 256, BK = 128;
constexpr int kStages = 3;
constexpr int kABytes = BM * BK;                 // 16 KB
constexpr int kBBytes = BN * BK;                 // 32 KB
constexpr int kTcStageBytes = kABytes + kBBytes; // 48 KB
constexpr int kOutBytes = 2 * 128 * 128;         // 2 warpgroups x one box (128 rows x 128 B)
constexpr int kMaxKB = 96;                       // K <= 12288 on this path (scale staging)
constexpr int kAsBytes = BM * (kMaxKB + 1) * 4;  // activation scales of a tile: [KB][BM + 1] fp32
constexpr int kWsBytes = 2 * kMaxKB * 4;         // weight scales of a tile
// With KB <= 48 the scale areas hold two tiles, so the staging warps fill the
// next tile's scales while the epilogue works on the current one.
constexpr int kAsDoubleMaxKB = (BM * (kMaxKB + 1)) / (2 * (BM + 1));
static_assert(kMaxKB * (BM + 1) <= BM * (kMaxKB + 1), "one buffer of the largest KB fits");
constexpr int kThreads = 384;                   // producer, MMA, 2 spare, 8 epilogue warps
constexpr int kEpiWarp0 = 4;                     // warps 4..11
// Registers a thread: at launch, and after the quant phase for warpgroup 0
// (producer, MMA, two spare warps) and the two epilogue warpgroups.  The split
// must add up to what the block was launched with, else setmaxnreg.inc would
// wait for registers that never come free; the launcher checks the launch
// count against the compiled kernel.
constexpr int kLaunchRegs = 168, kRegsWg0 = 56, kRegsEpi = 224;
static_assert(kRegsWg0 * 128 + kRegsEpi * 256 == kLaunchRegs * kThreads, "register split");
constexpr uint32_t kTmemCols = 512;
constexpr int kMaxSplitK = 8;                    // split-K ranks per tile
constexpr int kRedU = 4;                         // split-K reduction: float4 outputs in flight a thread

struct Params {
    const uint16_t* a;        // bf16 activations [M][K] (fused) or nullptr
    uint8_t* aq;              // e4m3 scratch / input [M][K]
    float* as;                // fp32 scales [M][KB]
    const float* ws;          // [NB][KB]
    int* ready;               // [m-tiles] quantised-chunk counters (fused), zero at launch
    int M, N, K, KB, NB;
    int mtiles, ntiles;
    uint16_t* y;              // bf16 [M][N] (split-K stores; otherwise the TMA map)
    int splits;               // S > 1: CTA u owns tile u / S, k-blocks of rank u % S (split-K)
    float* part;              // split-K: fp32 partial tiles [tiles][S][BM][BN]
    int* done;                // split-K: [tiles] partials published, zero at launch
    int* exits;               // CTAs finished; the last one returns ready, done and exits to
                              // zero (nullptr: the host zeroes the counters before each launch)
    int* err;
};

// kind::f8f6f4 instruction descriptor of the 128 x 256 tile (D fp32, A and B
// e4m3, both K-major); the shared-memory descriptors, the MMA issue, the
// commits and the tcgen05 fences are r9q_device.cuh's umma_* helpers.
constexpr uint32_t kIdesc = umma_idesc_e4m3(BM, BN);

// 32 consecutive TMEM columns of this thread's lane.  The load is asynchronous:
// its registers may be used only after a tmem_wait that names them.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
}
// Waits for every TMEM load of this thread; the registers of the loads named
// (r, and s through the empty statement that follows) count as written here,
// so no use of them moves above the wait.
__device__ __forceinline__ void tmem_wait(uint32_t (&r)[32], uint32_t (&s)[32]) {
    asm volatile("tcgen05.wait::ld.sync.aligned;"
                 : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                   "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]),
                   "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]),
                   "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]),
                   "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
                 :
                 : "memory");
    asm volatile(""
                 : "+r"(s[0]), "+r"(s[1]), "+r"(s[2]), "+r"(s[3]), "+r"(s[4]), "+r"(s[5]), "+r"(s[6]), "+r"(s[7]),
                   "+r"(s[8]), "+r"(s[9]), "+r"(s[10]), "+r"(s[11]), "+r"(s[12]), "+r"(s[13]), "+r"(s[14]),
                   "+r"(s[15]), "+r"(s[16]), "+r"(s[17]), "+r"(s[18]), "+r"(s[19]), "+r"(s[20]), "+r"(s[21]),
                   "+r"(s[22]), "+r"(s[23]), "+r"(s[24]), "+r"(s[25]), "+r"(s[26]), "+r"(s[27]), "+r"(s[28]),
                   "+r"(s[29]), "+r"(s[30]), "+r"(s[31])
                 :
                 : "memory");
}

// acc[i] += v[i] * sc for 32 columns, two lanes of packed fp32 FMA at a time
// (each lane is an IEEE fma, rounded to nearest: the same as fmaf).
__device__ __forceinline__ void promote32(float* acc, const uint32_t (&v)[32], float sc) {
    const float2 s2 = make_float2(sc, sc);
#pragma unroll
    for (int i = 0; i < 32; i += 2) {
        const float2 r = __ffma2_rn(make_float2(__uint_as_float(v[i]), __uint_as_float(v[i + 1])), s2,
                                    make_float2(acc[i], acc[i + 1]));
        acc[i] = r.x;
        acc[i + 1] = r.y;
    }
}

__device__ __forceinline__ void tma_store_2d(const void* tmap, int c0, int c1, const void* src) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%1, %2}], [%3];" ::"l"(
                     reinterpret_cast<uint64_t>(tmap)),
                 "r"(c0), "r"(c1), "r"(smem_u32(src))
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void named_sync(int id, int n) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

__device__ __forceinline__ void red_release_add(int* p, int v) {
    asm volatile("red.release.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// A tile's scales into shared memory, by `nthr` threads (this one is `idx`):
// the activation scales of its `rows` rows ([rows][KB], contiguous at src)
// kb-major with rows padded to BM + 1 (so the epilogue's reads, [kb][its row],
// hit distinct banks; rows past M read as 0), and the weight-block scales of
// its two 128-column blocks nb0, nb0 + 1 ([2][KB]).  Coalesced 16-byte loads,
// four in flight a thread, when the scale array is 16-byte aligned.
__device__ __forceinline__ void stage_scales(float* asb, float* wsb, const float* src, int rows, const float* ws,
                                             int nb0, int NB, int KB, int idx, int nthr) {
    const int nv = rows * KB;
    const int nv4 = ((reinterpret_cast<uintptr_t>(src) & 15) == 0) ? nv / 4 : 0;
    for (int i0 = 0; i0 < nv4; i0 += 4 * nthr) {
        float4 v[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * nthr + idx;
            v[u] = (i < nv4) ? reinterpret_cast<const float4*>(src)[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const int i = i0 + u * nthr + idx;
            if (i < nv4) {
                const float f[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
                for (int c = 0; c < 4; ++c) {
                    const int e = 4 * i + c, r = e / KB;
                    asb[(e - r * KB) * (BM + 1) + r] = f[c];
                }
            }
        }
    }
    for (int e = nv4 * 4 + idx; e < BM * KB; e += nthr) {      // the rest, then rows past M
        const int r = e / KB;
        asb[(e - r * KB) * (BM + 1) + r] = (e < nv) ? src[e] : 0.0f;
    }
    for (int e = idx; e < 2 * KB; e += nthr) {
        const int h = e / KB, nb = nb0 + h;
        wsb[e] = (nb < NB) ? ws[(int64_t)nb * KB + (e - h * KB)] : 0.0f;
    }
}

// bounded wait for `need` quantised rows of m-tile mt
__device__ __forceinline__ bool wait_rows(const int* ready, int need) { return wait_count(ready, need); }

}  // namespace tc

using namespace tc;

// 12 warps: each SM sub-partition holds 3 of them, so up to 168 registers a thread.
// SPLIT: split-K mode (p.splits > 1); otherwise persistent whole-K tiles.
template <bool SPLIT>
__global__ void __launch_bounds__(kThreads, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap amap, const __grid_constant__ CUtensorMap bmap,
                   const __grid_constant__ CUtensorMap ymap, const Params p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* ring = smem;                                        // kStages x 48 KB
    uint8_t* outst = smem + kStages * kTcStageBytes;             // output staging
    float* as_s = reinterpret_cast<float*>(outst + kOutBytes);   // [BM][KB + 1]
    float* ws_s = as_s + BM * (kMaxKB + 1);                      // [nsbuf][2][KB]
    uint64_t* bars = reinterpret_cast<uint64_t*>(ws_s + 2 * kMaxKB);
    uint64_t* full = bars;                                       // [kStages]
    uint64_t* empty = bars + kStages;                            // [kStages]
    uint64_t* tfull = bars + 2 * kStages;                        // [2] partial ready in TMEM
    uint64_t* tempty = bars + 2 * kStages + 2;                   // [2] partial consumed
    uint64_t* staged = bars + 2 * kStages + 4;                   // [2] a tile's scales are in smem
    uint64_t* consumed = bars + 2 * kStages + 6;                 // [2] ... and no longer needed
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 8);
    int* flags = reinterpret_cast<int*>(tmem_slot + 2);          // [0] error, [1] ring issued, [2] mma k-blocks,
                                                                 // [3] last CTA out

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int total = p.mtiles * p.ntiles;
    const int KB = p.KB;
    // Work of this CTA: tiles t_first, t_first + t_step, ... and k-blocks
    // [kb_lo, kb_hi) of each (split-K: one tile, the rank's k-range).
    const int S = SPLIT ? p.splits : 1;
    constexpr bool split = SPLIT;
    const int rank = split ? (int)blockIdx.x % S : 0;
    const int t_first = split ? (int)blockIdx.x / S : (int)blockIdx.x;
    const int t_step = split ? total : (int)gridDim.x;
    const int kb_lo = rank * KB / S, kb_hi = (rank + 1) * KB / S;
    // fused quant: a row is nch chunks of CH groups; an m-tile is ready when
    // its rows * nch chunks are published
    constexpr int CH = 16;
    const int nch = (KB + CH - 1) / CH;
    const int64_t nunits = (int64_t)p.M * nch;
    const bool fused = p.a != nullptr;
    const int nsbuf = KB <= kAsDoubleMaxKB ? 2 : 1;             // scale buffers
    volatile int* vflags = flags;
    auto fail = [&]() {
        record_error(p.err, kErrTimeout);
        atomicExch(&flags[0], 1);
    };

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&tfull[b], 1);
            mbar_init(&tempty[b], 8);                            // one arrive per epilogue warp
            mbar_init(&staged[b], 2);                            // one arrive per staging warp
            mbar_init(&consumed[b], 8);                          // one arrive per epilogue warp
        }
        flags[0] = flags[1] = flags[2] = 0;
        fence_proxy_async_smem();
    }
    if (warp == 1) tmem_alloc(tmem_slot, kTmemCols);
    umma_fence_before();
    __syncthreads();
    umma_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (fused) {
        // ---------------- quant phase: every warp of the grid ----------------
        // A row is a sequence of chunks of 16 groups; chunks are dealt out in
        // global order, consecutive chunks to consecutive CTAs (warp w of CTA
        // c takes chunks c + grid*w, c + grid*(w + 12), ...), so m-tiles fill
        // up from the top and a few rows still spread over many SMs.  Each finished chunk is published to its m-tile's ready
        // counter (an m-tile is complete at rows * chunks-per-row).  A warp
        // issues its next chunk's loads before quantising the current one.
        // Lane l holds 16 values of group 4j + (l >> 3) of the chunk.
        const int gw = blockIdx.x + gridDim.x * warp;         // first chunk of this warp
        const int GW = gridDim.x * (kThreads / 32);
        const int gl = lane >> 3, el = (lane & 7) * 16;
        auto load = [&](uint4 (&v)[CH / 4][2], int64_t row, int c) {
            const uint16_t* src = p.a + row * p.K;
#pragma unroll
            for (int j = 0; j < CH / 4; ++j) {
                const int g = c * CH + 4 * j + gl;
                if (g < KB) {
                    const uint4* q = reinterpret_cast<const uint4*>(src + (int64_t)g * BK + el);
                    v[j][0] = q[0];
                    v[j][1] = q[1];
                } else {
                    v[j][0] = v[j][1] = make_uint4(0u, 0u, 0u, 0u);
                }
            }
        };
        auto quant = [&](const uint4 (&v)[CH / 4][2], int64_t row, int c) {
            uint8_t* dq = p.aq + row * p.K;
#pragma unroll
            for (int j = 0; j < CH / 4; ++j) {
                if (c * CH + 4 * j < KB) {
                    const int g = c * CH + 4 * j + gl;
                    float sc;
                    const uint4 codes = quant_group128_lane8(v[j], sc);
                    if (g < KB) {
                        *reinterpret_cast<uint4*>(dq + (int64_t)g * BK + el) = codes;
                        if ((lane & 7) == 0) p.as[row * KB + g] = sc;
                    }
                }
            }
            // the chunk is done: publish it to its m-tile's ready counter
            __syncwarp();
            if (lane == 0) {
                fence_proxy_async_global();
                red_release_add(p.ready + row / BM, 1);
            }
        };
        // the chunk after the next one goes to L2 while this one is quantised
        auto prefetch = [&](int64_t u) {
            if (lane == 0 && u < nunits) {
                const int64_t row = u / nch;
                const int c = (int)(u - row * nch);
                const int groups = min(CH, KB - c * CH);
                bulk_prefetch_l2(p.a + row * p.K + (int64_t)c * CH * BK, (uint32_t)(groups * BK * 2));
            }
        };
        uint4 va[CH / 4][2], vb[CH / 4][2];
        int64_t u = gw;
        if (u < nunits) load(va, u / nch, (int)(u % nch));
        while (u < nunits) {
            prefetch(u + 2 * (int64_t)GW);
            int64_t u2 = u + GW;
            if (u2 < nunits) load(vb, u2 / nch, (int)(u2 % nch));
            quant(va, u / nch, (int)(u % nch));
            u = u2;
            if (u >= nunits) break;
            prefetch(u + 2 * (int64_t)GW);
            u2 = u + GW;
            if (u2 < nunits) load(va, u2 / nch, (int)(u2 % nch));
            quant(vb, u / nch, (int)(u % nch));
            u = u2;
        }
    }

    // Registers move from warpgroup 0 (short loops) to the epilogue warpgroups
    // (128 fp32 accumulators a thread).  Every warp gets to its setmaxnreg:
    // the quant phase above has no waits.
    if (warp < kEpiWarp0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kRegsWg0));
        if (warp == 0) {
            // ---------------- TMA producer ----------------
            if (lane == 0) {
                int it = 0;
                for (int t = t_first; t < total && *vflags == 0; t += t_step) {
                    const int mt = t / p.ntiles, nt = t % p.ntiles;
                    if (fused) {
                        const int need = min(BM, p.M - mt * BM) * nch;
                        if (!wait_rows(p.ready + mt, need)) {
                            fail();
                            break;
                        }
                        fence_proxy_async_global();     // the TMA reads what generic stores wrote
                    }
                    for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
                        const int st = it % kStages;
                        if (it >= kStages && !mbar_wait_sleep(&empty[st], ((uint32_t)(it / kStages) & 1u) ^ 1u)) {
                            fail();
                            break;
                        }
                        uint8_t* sa = ring + st * kTcStageBytes;
                        mbar_expect_tx(&full[st], kTcStageBytes);
                        tma_load_2d(sa, &amap, kb * BK, mt * BM, &full[st]);
                        tma_load_2d(sa + kABytes, &bmap, kb * BK, nt * BN, &full[st]);
                        flags[1] = it + 1;
                    }
                    if (*vflags) break;
                }
            }
        } else if (warp == 1) {
            // ---------------- MMA issuer ----------------
            if (lane == 0) {
                int it = 0;
                for (int t = t_first; t < total && *vflags == 0; t += t_step) {
                    for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
                        const int st = it % kStages;
                        const int ab = it & 1;
                        if (!mbar_wait_sleep(&full[st], (uint32_t)(it / kStages) & 1u)) {
                            fail();
                            break;
                        }
                        if (it >= 2 && !mbar_wait_sleep(&tempty[ab], ((uint32_t)(it >> 1) & 1u) ^ 1u)) {
                            fail();
                            break;
                        }
                        umma_fence_after();
                        const uint32_t sa = smem_u32(ring + st * kTcStageBytes);
                        const uint32_t sb = sa + kABytes;
                        const uint32_t td = tmem_base + (uint32_t)(ab * BN);
#pragma unroll
                        for (int k = 0; k < BK / 32; ++k)
                            umma_e4m3(td, umma_sdesc_sw128(sa + k * 32), umma_sdesc_sw128(sb + k * 32), kIdesc,
                                      k > 0 ? 1u : 0u);
                        umma_commit(&empty[st]);      // stage free once these MMAs have read it
                        umma_commit(&tfull[ab]);      // partial ready for the epilogue
                        flags[2] = it + 1;
                    }
                    if (*vflags) break;
                }
            }
        }
        if (warp >= 2) {
            // ---------------- scale staging (warps 2..3) ----------------
            // From this CTA's second tile on (the epilogue stages the first
            // itself): once a tile's rows are quantised and its buffer is
            // free, copy its scales into that buffer.
            int j = 1;
            for (int t = t_first + t_step; t < total; t += t_step, ++j) {
                const int b = j % nsbuf;
                const int mt = t / p.ntiles, nt = t % p.ntiles;
                if (j >= nsbuf && *vflags == 0 &&
                    !mbar_wait_sleep(&consumed[b], (uint32_t)(j / nsbuf - 1) & 1u))
                    fail();
                const int rows = min(BM, p.M - mt * BM);
                if (fused && *vflags == 0 && !wait_rows(p.ready + mt, rows * nch)) fail();
                stage_scales(as_s + b * KB * (BM + 1), ws_s + b * 2 * KB, p.as + (int64_t)mt * BM * KB, rows, p.ws,
                             nt * 2, p.NB, KB, (warp - 2) * 32 + lane, 64);
                __syncwarp();
                if (lane == 0) mbar_arrive(&staged[b]);
            }
        }
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kRegsEpi));
        // ---------------- epilogue: promotion + store ----------------
        const int ew = warp - kEpiWarp0;          // 0..7
        const int wg = ew >> 2;                   // column half
        const int q = warp & 3;                   // TMEM lane quarter of this warp
        const int rl = q * 32 + lane;             // row within the tile
        const bool leader = (ew & 3) == 0 && lane == 0;
        uint8_t* stg = outst + wg * (128 * 128);
        int it = 0, j = 0;
        for (int t = t_first; t < total; t += t_step, ++j) {
            const int mt = t / p.ntiles, nt = t % p.ntiles;
            const int sb = j % nsbuf;
            if (j == 0) {
                // the first tile's scales: all 256 epilogue threads copy them
                // (one round of loads), then stand in for the staging warps
                const int rows = min(BM, p.M - mt * BM);
                if (fused && *vflags == 0 && !wait_rows(p.ready + mt, rows * nch)) fail();
                stage_scales(as_s, ws_s, p.as + (int64_t)mt * BM * KB, rows, p.ws, nt * 2, p.NB, KB, ew * 32 + lane,
                             256);
                named_sync(3, 256);
                if ((ew == 0 || ew == 4) && lane == 0) mbar_arrive(&staged[0]);
            }
            // this tile's scales, from the staging warps
            if (*vflags == 0 && !mbar_wait_sleep(&staged[sb], (uint32_t)(j / nsbuf) & 1u)) fail();
            const float* as_col = as_s + sb * KB * (BM + 1) + rl;     // [kb * (BM + 1)]
            const float* ws_wg = ws_s + sb * 2 * KB + wg * KB;
            float acc[128];
#pragma unroll
            for (int i = 0; i < 128; ++i) acc[i] = 0.0f;
            for (int kb = kb_lo; kb < kb_hi; ++kb, ++it) {
                const int ab = it & 1;
                const float sc = as_col[kb * (BM + 1)] * ws_wg[kb];
                if (*vflags == 0 && !mbar_wait_sleep(&tfull[ab], (uint32_t)(it >> 1) & 1u)) fail();
                umma_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(ab * BN + wg * 128);
                // Two 32-column loads in flight at a time: the FMAs of one
                // pair overlap the TMEM latency of the next.
                uint32_t ra[32], rb[32];
                tmem_ld32(taddr, ra);
                tmem_ld32(taddr + 32, rb);
                tmem_wait(ra, rb);
                promote32(acc, ra, sc);
                tmem_ld32(taddr + 64, ra);
                promote32(acc + 32, rb, sc);
                tmem_ld32(taddr + 96, rb);
                tmem_wait(ra, rb);
                // the whole partial is in registers: free the buffer for the
                // MMA two k-blocks ahead before the last FMAs
                umma_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&tempty[ab]);
                promote32(acc + 64, ra, sc);
                promote32(acc + 96, rb, sc);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&consumed[sb]);     // scale buffer free for a later tile
            if (SPLIT) {
                // ---- split-K: this rank's partial goes to scratch (reduced below) ----
                // layout [tile][rank][column quad q][row] of float4: a warp's
                // 32 rows of one quad are 512 contiguous bytes
                float4* dst = reinterpret_cast<float4*>(p.part) + ((int64_t)(t * S + rank) * (BN / 4) + wg * 32) * BM + rl;
#pragma unroll
                for (int c = 0; c < 32; ++c)
                    __stcg(dst + c * BM, make_float4(acc[4 * c], acc[4 * c + 1], acc[4 * c + 2], acc[4 * c + 3]));
                continue;
            }
            // ---- bf16 out: two 64-column boxes through the swizzled staging, TMA stores ----
            const int col0 = nt * BN + wg * 128;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (leader) bulk_wait_read0();    // the previous store has read the staging
                named_sync(1 + wg, 128);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    uint4 o;
                    o.x = pack_bf16x2(acc[h * 64 + c * 8 + 0], acc[h * 64 + c * 8 + 1]);
                    o.y = pack_bf16x2(acc[h * 64 + c * 8 + 2], acc[h * 64 + c * 8 + 3]);
                    o.z = pack_bf16x2(acc[h * 64 + c * 8 + 4], acc[h * 64 + c * 8 + 5]);
                    o.w = pack_bf16x2(acc[h * 64 + c * 8 + 6], acc[h * 64 + c * 8 + 7]);
                    *reinterpret_cast<uint4*>(stg + rl * 128 + ((c ^ (rl & 7)) << 4)) = o;
                }
                fence_proxy_async_smem();
                named_sync(1 + wg, 128);
                if (leader) {
                    if (col0 + 64 * h < p.N) tma_store_2d(&ymap, col0 + 64 * h, mt * BM, stg);
                    bulk_commit();
                }
            }
        }
        if (leader) bulk_wait0();
        if (SPLIT && t_first < total) {
            // ---- split-K: publish the partial; once all S are in, rank r sums
            // rows [r*RB, (r+1)*RB) over ranks 0..S-1 in order (threads take
            // consecutive rows of one column quad: coalesced partial reads) ----
            const int t = t_first, mt = t / p.ntiles, nt = t % p.ntiles;
            __threadfence();
            named_sync(3, 256);
            const int et = ew * 32 + lane;          // 0..255
            if (et == 0) {
                red_release_add(p.done + t, 1);
                if (*vflags == 0 && !wait_count(p.done + t, S)) fail();
            }
            named_sync(3, 256);
            const int RB = BM / S;                  // rows reduced by this rank
            const float4* src = reinterpret_cast<const float4*>(p.part) + (int64_t)t * S * (BN / 4) * BM;
            for (int u0 = 0; u0 < RB * (BN / 4); u0 += kRedU * 256) {
                float4 v[kRedU][kMaxSplitK];
#pragma unroll
                for (int i = 0; i < kRedU; ++i) {
                    const int u = u0 + i * 256 + et;
                    if (u < RB * (BN / 4)) {
                        const int row = rank * RB + u % RB, c4 = u / RB;
#pragma unroll
                        for (int r = 0; r < kMaxSplitK; ++r)
                            if (r < S) v[i][r] = __ldcg(src + ((int64_t)r * (BN / 4) + c4) * BM + row);
                    }
                }
#pragma unroll
                for (int i = 0; i < kRedU; ++i) {
                    const int u = u0 + i * 256 + et;
                    if (u >= RB * (BN / 4)) continue;
                    const int row = rank * RB + u % RB, c4 = u / RB;
                    float4 a = v[i][0];
#pragma unroll
                    for (int r = 1; r < kMaxSplitK; ++r)
                        if (r < S) {
                            a.x = __fadd_rn(a.x, v[i][r].x);
                            a.y = __fadd_rn(a.y, v[i][r].y);
                            a.z = __fadd_rn(a.z, v[i][r].z);
                            a.w = __fadd_rn(a.w, v[i][r].w);
                        }
                    const int m = mt * BM + row, n = nt * BN + 4 * c4;
                    if (m < p.M && n < p.N)
                        *reinterpret_cast<uint2*>(p.y + (int64_t)m * p.N + n) =
                            make_uint2(pack_bf16x2(a.x, a.y), pack_bf16x2(a.z, a.w));
                }
            }
        }
    }

    // ---------------- teardown ----------------
    umma_fence_before();
    __syncthreads();
    if (flags[0] != 0 && tid == 0) {
        // drain what was issued: ring copies, then the MMAs' last commits
        const int issued = flags[1];
        for (int i = max(0, issued - kStages); i < issued; ++i)
            (void)mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u);
        const int mmas = flags[2];
        for (int i = max(0, mmas - 2); i < mmas; ++i) (void)mbar_wait(&tfull[i & 1], (uint32_t)(i >> 1) & 1u);
    }
    if (p.exits != nullptr) {
        // Every counter access of this CTA is behind the barrier above; the
        // last CTA of the grid to get here returns the counters to zero for
        // the next call on the same scratch.
        if (tid == 0) {
            int prev;
            asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], 1;" : "=r"(prev) : "l"(p.exits) : "memory");
            flags[3] = (prev == (int)gridDim.x - 1) ? 1 : 0;
        }
        __syncthreads();
        if (flags[3]) {
            if (p.ready) for (int i = tid; i < p.mtiles; i += kThreads) p.ready[i] = 0;
            if (SPLIT && p.done) for (int i = tid; i < total; i += kThreads) p.done[i] = 0;
            if (tid == 0) *p.exits = 0;
        }
    }
    __syncthreads();
    umma_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, kTmemCols);
}

size_t tc_smem_bytes() { return 1024 + (size_t)kStages * kTcStageBytes + kOutBytes + kAsBytes + kWsBytes + 256; }
int tc_max_kb() { return kMaxKB; }

int tc_plan_splits(int64_t M, int64_t N, int64_t K, int sms) {
    const int64_t tiles = ((M + BM - 1) / BM) * ((N + BN - 1) / BN);
    const int64_t KB = K / BK;
    for (int S = kMaxSplitK; S >= 2; S >>= 1)
        if (tiles * S <= sms && KB >= S) return S;
    return 1;
}

cudaError_t launch_tc_gemm(const CUtensorMap& amap, const CUtensorMap& bmap, const CUtensorMap& ymap,
                           const uint16_t* a, uint8_t* aq, float* as, const float* ws, int* ready, uint16_t* y,
                           int splits, float* part, int* done, int* exits, int M, int N, int K, int* err, int sms,
                           cudaStream_t st) {
    Params p;
    p.a = a;
    p.aq = aq;
    p.as = as;
    p.ws = ws;
    p.ready = ready;
    p.M = M;
    p.N = N;
    p.K = K;
    p.KB = K / BK;
    p.NB = N / 128;
    p.mtiles = (M + BM - 1) / BM;
    p.ntiles = (N + BN - 1) / BN;
    p.y = y;
    p.splits = splits;
    p.part = part;
    p.done = done;
    p.exits = exits;
    p.err = err;
    if (splits < 1 || splits > kMaxSplitK || (BM % splits) != 0 || p.KB < splits) return cudaErrorInvalidValue;
    if (splits > 1 && (part == nullptr || done == nullptr || y == nullptr)) return cudaErrorInvalidValue;
    const size_t smem = tc_smem_bytes();
    void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const Params) =
        splits > 1 ? tc_gemm_kernel<true> : tc_gemm_kernel<false>;
    // The kernel's register split assumes the compiled launch count.
    static const int launch_regs[2] = {[]() {
                                           cudaFuncAttributes fa = {};
                                           return cudaFuncGetAttributes(&fa, tc_gemm_kernel<false>) == cudaSuccess
                                                      ? fa.numRegs
                                                      : -1;
                                       }(),
                                       []() {
                                           cudaFuncAttributes fa = {};
                                           return cudaFuncGetAttributes(&fa, tc_gemm_kernel<true>) == cudaSuccess
                                                      ? fa.numRegs
                                                      : -1;
                                       }()};
    if (launch_regs[splits > 1 ? 1 : 0] != kLaunchRegs) return cudaErrorInvalidConfiguration;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorLaunchOutOfResources;
    const int total = p.mtiles * p.ntiles;
    // split-K: one CTA per (tile, rank), all resident (the ranks of a tile wait
    // for each other); otherwise persistent CTAs, at most one per SM
    const int grid = splits > 1 ? total * splits : (total < sms ? total : sms);
    if (grid > sms * per_sm) return cudaErrorInvalidConfiguration;
    // Every CTA quantises rows other CTAs wait for, so all CTAs must be
    // resident at once: a cooperative launch guarantees it (one CTA per SM).
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, amap, bmap, ymap, p);
}

}  // namespace r9q
