// Decode-width block-scaled fp8 GEMM ("stream" kernel), sm_103a.
//
// At decode widths the GEMM is a weight stream: every weight byte is used by a
// few tokens, so HBM bandwidth bounds it (r9700-stack v0.3.1 notes: the decode
// GEMMs' weights are the step's largest stream, and fp8 halves it).  This
// kernel serves W8A8 calls with M <= 32 (larger W8A8 calls go to the tcgen05
// kernel), and every weight-only and expert-MLP call, in token chunks of up
// to 64 rows.
// Design:
//  * grid (S, G, ceil(M/MT)) launched as clusters of S CTAs along K.  Cluster
//    g owns the 128-row weight tiles t = g, g+G, g+2G, ... (one scale block
//    row, or 64 gate + 64 up rows for the SwiGLU epilogue); CTA s of the
//    cluster owns a contiguous range of 128-wide k-blocks of every such tile.
//  * one producer thread streams the CTA's 128x128 e4m3 weight tiles with 2-D
//    TMA (128-byte swizzle) through a shared-memory ring guarded by full/empty
//    mbarriers, running ahead across tile boundaries.
//  * the CTA's activation slice arrives in shared memory with one bulk copy
//    per token row, issued right after the first weight stages, and serves
//    every tile of the CTA.  W8A8: each 128-wide group is quantised in place
//    once per CTA at the A-load (shuffle amax, fp32-division-exact quotient,
//    cvt.rn.satfinite.e4m3x2), byte-identical to the standalone quant kernel.
//    Weight-only: the bf16 rows are the B operand, their pairs swapped in
//    registers to match the in-register e4m3 -> bf16 conversion.
//  * eight MMA warps (16 weight rows each) run swap-AB mma.sync (weights are
//    the 16-row A operand, tokens the 8-column B operand): m16n8k32 e4m3 for
//    W8A8, m16n8k16 bf16 for weight-only.  Each k-block's fp32 partial is
//    promoted into register accumulators with as[m][kb] * ws[nb][kb] (the
//    exact block-scaled form: v0.3.0 notes, exact block-scaled fp8 variant).
//  * split-K is reduced through distributed shared memory: each CTA parks its
//    tile partial in one of two shared buffers and signals every peer with a
//    cluster-scope mbarrier arrive; CTA r then sums slice r of the tile over
//    ranks 0..S-1 in that fixed order (deterministic, no global workspace)
//    and tells the peers when it has finished reading.
//  * the epilogue writes bf16 y, or (SwiGLU) rounds gate and up to bf16 and
//    writes h = bf16(silu(g) * u).
// Every mbarrier wait is bounded; a timeout records R9Q_ERR_TIMEOUT in the
// device error word and the kernel drains its copies and returns.
#pragma once

#include "r9q_device.cuh"
#include "r9q_kernels.h"

namespace r9q {

__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity) {
    for (uint32_t i = 0; i < kSpinLimit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(ok)
            : "r"(smem_u32(bar)), "r"(parity)
            : "memory");
        if (ok) return true;
    }
    return false;
}

// Arrive on the barrier at the same shared-memory offset in every CTA of the
// cluster.  One cluster-scope fence releases everything this CTA did before
// (the caller synchronises the CTA's writers first); the arrives themselves
// are relaxed, so the release is paid once rather than once per peer.
__device__ __forceinline__ void mbar_arrive_all_ranks(uint64_t* local_bar, int S) {
    asm volatile("fence.acq_rel.cluster;" ::: "memory");
    const uint32_t a = smem_u32(local_bar);
    for (int r = 0; r < S; ++r) {
        const uint32_t addr = dsmem_addr(a, (uint32_t)r);
        asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(addr) : "memory");
    }
}

__device__ __forceinline__ void consumer_sync() {
    asm volatile("bar.sync 1, %0;" ::"n"(kCWarps * 32) : "memory");
}

template <int EPI>
__device__ __forceinline__ void tile_rows(int t, int& r0, int& r1, int& nb0, int& nb1) {
    if (EPI == EPI_SWIGLU) {
        const int j = t >> 1, hh = t & 1;
        r0 = 2 * kBlock * j + 64 * hh;       // gate rows
        r1 = r0 + kBlock;                    // up rows
        nb0 = 2 * j;
        nb1 = 2 * j + 1;
    } else {
        r0 = kBlock * t;
        r1 = r0 + 64;
        nb0 = nb1 = t;
    }
}

// The kernel body for the token rows [m0, m0 + mvalid) (mvalid >= 1) of one
// problem whose weight rows start at wrow0 and whose block-scale rows start at
// nbase (both 0 for a single GEMM; an expert's offsets in the grouped launch).
template <int MT, int AMODE, int EPI>
__device__ __forceinline__ void stream_gemm_body(const CUtensorMap& wmap, const StreamParams& p, const int m0,
                                                 const int mvalid, const int wrow0, const int nbase) {
    constexpr int NT = MT / 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    // The next kernel in the stream may start launching at once: it waits for
    // this grid's completion itself before it reads anything this grid writes.
    pdl_trigger();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.splits, G = p.groups, nst = p.stages;
    const int split = (int)cluster_ctarank();
    const int group = blockIdx.y;
    const int KB = p.KB;
    const int kbase = KB / S, krem = KB % S;
    const int kb0 = split * kbase + min(split, krem);
    const int nkb = kbase + (split < krem ? 1 : 0);
    const int kbs_max = kbase + (krem ? 1 : 0);
    const int kslice = kbs_max * kBlock;
    const int ntl = (p.ntiles - group + G - 1) / G;       // tiles of this cluster
    const int ntl_max = (p.ntiles + G - 1) / G;
    const int iters = ntl * nkb;

    // shared memory carve-up (must match stream_smem_bytes)
    uint8_t* ring = smem;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + nst * kStageBytes);
    uint64_t* full = bars;                       // [kMaxStages]
    uint64_t* empty = bars + kMaxStages;         // [kMaxStages]
    uint64_t* abar = bars + 2 * kMaxStages;      // activation bulk copies
    uint64_t* pfull = abar + 1;                  // [2] every rank's partial is parked
    uint64_t* pfree = abar + 3;                  // [2] every rank has read my partial
    int* flags = reinterpret_cast<int*>(bars + 2 * kMaxStages + 5);   // [0] error, [1] issued
    float* P = reinterpret_cast<float*>(smem + nst * kStageBytes + kBarBytes);   // [npbuf][MT][kPStride]
    const int npbuf = ntl_max > 1 ? 2 : 1;                            // partial buffers
    float* ws_s = P + npbuf * MT * kPStride;                          // [ntl_max][2][kbs_max]
    float* as_s = ws_s + ntl_max * 2 * kbs_max;                       // [MT][kbs_max]
    uintptr_t act_addr = reinterpret_cast<uintptr_t>(as_s + MT * kbs_max);
    uint8_t* act = reinterpret_cast<uint8_t*>((act_addr + 15) & ~static_cast<uintptr_t>(15));
    // Row stride of the activation slice.  W8A8 (fused): bf16 rows whose first
    // kslice bytes are overwritten in place by the e4m3 codes; +16 keeps the
    // code rows on distinct banks for the B-fragment loads.  Weight-only: bf16
    // rows, +32 for the 8-byte B-fragment loads.  Unfused: e4m3 rows.
    const int act_ld = (AMODE == A_QUANT) ? (2 * kslice + 16) : (AMODE == A_BF16) ? (2 * kslice + 32) : (kslice + 16);
    const int row_bytes = (AMODE == A_PREQ) ? nkb * kBlock : 2 * nkb * kBlock;   // bytes copied per token

    if (tid == 0) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCWarps);
        }
        mbar_init(abar, 1);
        flags[0] = 0;
        flags[1] = 0;
        fence_proxy_async_smem();     // the TMA unit sees the initialised ring barriers
    }
    if (tid == 32) {
        mbar_init(&pfull[0], S);
        mbar_init(&pfull[1], S);
        mbar_init(&pfree[0], S);
        mbar_init(&pfree[1], S);
        fence_mbar_init();            // peers see them once the cluster barrier below completes
    }
    // the producer and the MMA warps use the barriers just initialised
    __syncthreads();
    // Every peer's barriers must exist before anyone arrives on them remotely:
    // arrive on the cluster barrier now, wait for it only just before the
    // first remote arrive, so the weight stream starts at once.
    cluster_arrive();

    // ---- producer prologue: fill the ring, then fetch the activations ----
    const bool producer = (warp == kCWarps && lane == 0);
    const int npro = min(iters, nst);
    if (producer) {
        tma_prefetch_desc(&wmap);
        for (int it = 0; it < npro; ++it) {
            const int tl = it / nkb, i = it - tl * nkb;
            int r0, r1, nb0, nb1;
            tile_rows<EPI>(group + tl * G, r0, r1, nb0, nb1);
            r0 += wrow0;
            r1 += wrow0;
            mbar_expect_tx(&full[it], kStageBytes);
            tma_load_2d(ring + it * kStageBytes, &wmap, (kb0 + i) * kBlock, r0, &full[it]);
            tma_load_2d(ring + it * kStageBytes + kStageBytes / 2, &wmap, (kb0 + i) * kBlock, r1, &full[it]);
        }
        flags[1] = npro;
        // the rest of this CTA's weight slice goes to L2 now, so that the ring
        // refills from L2 and the DRAM stream does not wait for the MMAs
        for (int it = npro; it < iters; ++it) {
            const int tl = it / nkb, i = it - tl * nkb;
            int r0, r1, nb0, nb1;
            tile_rows<EPI>(group + tl * G, r0, r1, nb0, nb1);
            tma_prefetch_l2_2d(&wmap, (kb0 + i) * kBlock, wrow0 + r0);
            tma_prefetch_l2_2d(&wmap, (kb0 + i) * kBlock, wrow0 + r1);
        }
    }
    // Weights and their block scales never come from the preceding kernel:
    // load the scales now.  The activation rows may: prefetch them into L2
    // only (no stale data can result) and copy them after the wait.
    if (producer) {
        for (int tok = 0; tok < mvalid; ++tok) {
            const uint8_t* src = (AMODE == A_PREQ)
                ? p.aq + (int64_t)(m0 + tok) * p.K + (int64_t)kb0 * kBlock
                : reinterpret_cast<const uint8_t*>(p.a + (int64_t)(m0 + tok) * p.K + (int64_t)kb0 * kBlock);
            bulk_prefetch_l2(src, (uint32_t)row_bytes);
        }
    }
    for (int c = tid; c < ntl * nkb; c += kStreamThreads) {
        const int tl = c / nkb, i = c - tl * nkb;
        int r0, r1, nb0, nb1;
        tile_rows<EPI>(group + tl * G, r0, r1, nb0, nb1);
        ws_s[(tl * 2 + 0) * kbs_max + i] = p.ws[(int64_t)(nbase + nb0) * KB + kb0 + i];
        ws_s[(tl * 2 + 1) * kbs_max + i] = p.ws[(int64_t)(nbase + nb1) * KB + kb0 + i];
    }
    pdl_wait();
    if (producer) {
        mbar_expect_tx(abar, (uint32_t)(mvalid * row_bytes));
        for (int tok = 0; tok < mvalid; ++tok) {
            const uint8_t* src = (AMODE == A_PREQ)
                ? p.aq + (int64_t)(m0 + tok) * p.K + (int64_t)kb0 * kBlock
                : reinterpret_cast<const uint8_t*>(p.a + (int64_t)(m0 + tok) * p.K + (int64_t)kb0 * kBlock);
            bulk_load(act + tok * act_ld, src, (uint32_t)row_bytes, abar);
        }
    }

    // rows past the last token: zero codes / activations and zero scales
    for (int c = tid; c < (MT - mvalid) * (row_bytes / 16); c += kStreamThreads) {
        const int tok = mvalid + c / (row_bytes / 16), ch = c % (row_bytes / 16);
        *reinterpret_cast<uint4*>(act + tok * act_ld + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (AMODE == A_PREQ) {
        for (int c = tid; c < MT * nkb; c += kStreamThreads) {
            const int tok = c / nkb, kbl = c - tok * nkb;
            as_s[tok * kbs_max + kbl] = (tok < mvalid) ? p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] : 0.0f;
        }
    } else if (AMODE == A_QUANT) {
        // only the padding rows: the scales of rows < mvalid are written by the
        // quant loop below, which other warps may already be running
        for (int c = tid; c < (MT - mvalid) * nkb; c += kStreamThreads)
            as_s[(mvalid + c / nkb) * kbs_max + c % nkb] = 0.0f;
    }
    if (!mbar_wait(abar, 0)) {
        record_error(p.err, kErrTimeout);
        atomicExch(&flags[0], 1);
    }

    if (AMODE == A_QUANT) {
        // In-place group quantisation: one warp walks a token row's groups in
        // increasing order, so the codes of group g (bytes [128g, 128g+128))
        // only overwrite bf16 data of groups <= g that it has already read.
        for (int tok = warp; tok < mvalid; tok += kCWarps + 1) {
            uint8_t* row = act + tok * act_ld;
            for (int kbl = 0; kbl < nkb; ++kbl) {
                const uint2 v = *reinterpret_cast<const uint2*>(row + kbl * 2 * kBlock + 8 * lane);
                float s;
                const uint32_t codes =
                    quant_group128_warp(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), s);
                __syncwarp();
                *reinterpret_cast<uint32_t*>(row + kbl * kBlock + 4 * lane) = codes;
                if (lane == 0) as_s[tok * kbs_max + kbl] = s;
                if (p.aq != nullptr && group == 0) {
                    const int64_t off = (int64_t)(m0 + tok) * p.K + (int64_t)(kb0 + kbl) * kBlock + 4 * lane;
                    *reinterpret_cast<uint32_t*>(p.aq + off) = codes;
                    if (lane == 0) p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] = s;
                }
            }
        }
    }
    __syncthreads();

    const int g = lane >> 2, t = lane & 3;
    if (warp < kCWarps) {
        cluster_wait();
        // ---- MMA warps: rows [16*warp, 16*warp + 16) of every tile ----
        const int box = warp >> 2;
        const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int lchk = lane >> 4;
        const int row = warp * 16 + lrow;
        // A failed wait sets flags[0]; from then on every wait is skipped but
        // all MMA warps keep walking the same loop and barrier sequence, so no
        // warp is left waiting at a named barrier.
        volatile int* vflags = flags;
        auto fail = [&]() {
            record_error(p.err, kErrTimeout);
            atomicExch(&flags[0], 1);
        };
        // Tile tl's partial is parked and announced, then tile tl-1 is reduced:
        // the wait for the peers' partials of one tile overlaps the MMAs of the next.
        for (int tl = 0; tl <= ntl; ++tl) {
            if (tl < ntl) {
                float acc[NT][4];
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[nt][e] = 0.0f;
                const float* wsv_s = ws_s + (tl * 2 + box) * kbs_max;
                for (int i = 0; i < nkb; ++i) {
                    const int it = tl * nkb + i;
                    const int st = it % nst;
                    if (*vflags == 0 && !mbar_wait(&full[st], (uint32_t)(it / nst) & 1u)) fail();
                    const uint32_t tbase = smem_u32(ring + st * kStageBytes);
                    float d[NT][4];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) d[nt][e] = 0.0f;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        uint32_t a[4];
                        const int chunk = ks * 2 + lchk;
                        ldmatrix_x4(tbase + row * 128 + ((chunk ^ (row & 7)) << 4), a[0], a[1], a[2], a[3]);
                        if (AMODE != A_BF16) {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint8_t* bp = act + (nt * 8 + g) * act_ld + i * kBlock + ks * 32 + 4 * t;
                                mma_e4m3_16832(d[nt], a, *reinterpret_cast<const uint32_t*>(bp),
                                               *reinterpret_cast<const uint32_t*>(bp + 16));
                            }
                        } else {
                            uint32_t ev[4], od[4];
#pragma unroll
                            for (int r = 0; r < 4; ++r) e4m3x4_to_bf16x2x2(a[r], ev[r], od[r]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint8_t* bp = act + (nt * 8 + g) * act_ld + 2 * (i * kBlock + ks * 32 + 4 * t);
                                // (x0,x1),(x2,x3) -> (x0,x2),(x1,x3): the pairing of e4m3x4_to_bf16x2x2
                                const uint2 bv = *reinterpret_cast<const uint2*>(bp);
                                const uint2 cv = *reinterpret_cast<const uint2*>(bp + 32);
                                mma_bf16_16816(d[nt], ev[0], ev[1], od[0], od[1], __byte_perm(bv.x, bv.y, 0x5410),
                                               __byte_perm(bv.x, bv.y, 0x7632));
                                mma_bf16_16816(d[nt], ev[2], ev[3], od[2], od[3], __byte_perm(cv.x, cv.y, 0x5410),
                                               __byte_perm(cv.x, cv.y, 0x7632));
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&empty[st]);
                    // block-scale promotion of this k-block's partial
                    const float wsv = wsv_s[i];
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        float sc0 = wsv, sc1 = wsv;
                        if (AMODE != A_BF16) {
                            sc0 = as_s[(nt * 8 + 2 * t) * kbs_max + i] * wsv;
                            sc1 = as_s[(nt * 8 + 2 * t + 1) * kbs_max + i] * wsv;
                        }
                        acc[nt][0] = fmaf(d[nt][0], sc0, acc[nt][0]);
                        acc[nt][1] = fmaf(d[nt][1], sc1, acc[nt][1]);
                        acc[nt][2] = fmaf(d[nt][2], sc0, acc[nt][2]);
                        acc[nt][3] = fmaf(d[nt][3], sc1, acc[nt][3]);
                    }
                }

                // ---- park the partial in buffer b = tl & 1 (after its last readers are done) ----
                const int b = tl & 1;
                const uint32_t use = (uint32_t)(tl >> 1);
                if (tl >= 2 && *vflags == 0 && !mbar_wait_cluster(&pfree[b], (use - 1) & 1u)) fail();
                float* Pb = P + b * MT * kPStride;
#pragma unroll
                for (int nt = 0; nt < NT; ++nt) {
                    const int r = warp * 16 + g;
                    const int tok = nt * 8 + 2 * t;
                    Pb[tok * kPStride + r] = acc[nt][0];
                    Pb[(tok + 1) * kPStride + r] = acc[nt][1];
                    Pb[tok * kPStride + r + 8] = acc[nt][2];
                    Pb[(tok + 1) * kPStride + r + 8] = acc[nt][3];
                }
                consumer_sync();
                if (tid == 0) mbar_arrive_all_ranks(&pfull[b], S);
            }
            if (tl >= 1) {
                const int rt = tl - 1;
                const int tile = group + rt * G;
                const int b = rt & 1;
                const uint32_t use = (uint32_t)(rt >> 1);
                if (*vflags == 0 && !mbar_wait_cluster(&pfull[b], use & 1u)) fail();
                const float* Pb = P + b * MT * kPStride;
                // ---- split-K reduction of tile rt, slice `split`, over ranks 0..S-1 + epilogue ----
                // Sums go to registers first; the peers are told their partials are
                // free before the global stores, so the release never waits on them.
                const uint32_t pbase = smem_u32(Pb);
                constexpr int UPT = (EPI == EPI_SWIGLU) ? 32 : 64;   // units per token
                constexpr int MAXU = (MT * UPT + kCWarps * 32 - 1) / (kCWarps * 32);   // units per thread, S = 1
                const int U = MT * UPT;
                const int u_lo = (split * U) / S, u_hi = ((split + 1) * U) / S;
                uint32_t outv[MAXU];
#pragma unroll
                for (int j = 0; j < MAXU; ++j) {
                    const int u = u_lo + tid + j * kCWarps * 32;
                    outv[j] = 0u;
                    if (u >= u_hi) continue;
                    const int tok = u / UPT, up = u - tok * UPT;
                    if (tok >= mvalid) continue;
                    // all ranks' partials are loaded first (independent remote
                    // loads in flight together), then summed in rank order
                    if (EPI == EPI_STORE) {
                        const uint32_t off = (uint32_t)((tok * kPStride + 2 * up) * 4);
                        float2 v[kMaxSplits];
#pragma unroll
                        for (int r = 0; r < kMaxSplits; ++r)
                            if (r < S) v[r] = ld_dsmem_f32x2(dsmem_addr(pbase + off, (uint32_t)r));
                        float2 sum = v[0];
#pragma unroll
                        for (int r = 1; r < kMaxSplits; ++r)
                            if (r < S) {
                                sum.x = __fadd_rn(sum.x, v[r].x);
                                sum.y = __fadd_rn(sum.y, v[r].y);
                            }
                        outv[j] = pack_bf16x2(sum.x, sum.y);
                    } else {
                        const uint32_t offg = (uint32_t)((tok * kPStride + 2 * up) * 4);
                        const uint32_t offu = offg + 64 * 4;
                        float2 gv[kMaxSplits], uv[kMaxSplits];
#pragma unroll
                        for (int r = 0; r < kMaxSplits; ++r)
                            if (r < S) {
                                gv[r] = ld_dsmem_f32x2(dsmem_addr(pbase + offg, (uint32_t)r));
                                uv[r] = ld_dsmem_f32x2(dsmem_addr(pbase + offu, (uint32_t)r));
                            }
                        float2 gs = gv[0], us = uv[0];
#pragma unroll
                        for (int r = 1; r < kMaxSplits; ++r)
                            if (r < S) {
                                gs.x = __fadd_rn(gs.x, gv[r].x);
                                gs.y = __fadd_rn(gs.y, gv[r].y);
                                us.x = __fadd_rn(us.x, uv[r].x);
                                us.y = __fadd_rn(us.y, uv[r].y);
                            }
                        const float h0 = silu_mul(bf16_round(gs.x), bf16_round(us.x));
                        const float h1 = silu_mul(bf16_round(gs.y), bf16_round(us.y));
                        outv[j] = pack_bf16x2(h0, h1);
                    }
                }
                consumer_sync();
                if (tid == 0) mbar_arrive_all_ranks(&pfree[b], S);
#pragma unroll
                for (int j = 0; j < MAXU; ++j) {
                    const int u = u_lo + tid + j * kCWarps * 32;
                    if (u >= u_hi) continue;
                    const int tok = u / UPT, up = u - tok * UPT;
                    if (tok >= mvalid) continue;
                    const int64_t col = (EPI == EPI_STORE) ? (int64_t)kBlock * tile + 2 * up : (int64_t)64 * tile + 2 * up;
                    *reinterpret_cast<uint32_t*>(p.y + (int64_t)(m0 + tok) * p.ldy + col) = outv[j];
                }
            }
        }
        // Peers stop touching this CTA's shared memory once every rank has
        // arrived on its pfree barriers for their last use: wait for those
        // instead of a cluster-wide barrier at exit.
        for (int b2 = 0; b2 < 2 && b2 < ntl; ++b2) {
            const uint32_t last_use = (uint32_t)((ntl - 1 - b2) >> 1);
            if (!mbar_wait_cluster(&pfree[b2], last_use & 1u)) fail();   // also after an error
        }
    } else {
        cluster_wait();
    }
    if (warp == kCWarps && lane == 0) {
        // ---- producer steady state (runs ahead across tiles) ----
        int issued = npro;
        int cur_tl = -1, r0 = 0, r1 = 0, nb0, nb1;
        for (int it = nst; it < iters; ++it) {
            const int st = it % nst;
            if (!mbar_wait(&empty[st], ((uint32_t)(it / nst) & 1u) ^ 1u)) {
                record_error(p.err, kErrTimeout);
                atomicExch(&flags[0], 1);
                break;
            }
            const int tl = it / nkb, i = it - tl * nkb;
            if (tl != cur_tl) {
                tile_rows<EPI>(group + tl * G, r0, r1, nb0, nb1);
                r0 += wrow0;
                r1 += wrow0;
                cur_tl = tl;
            }
            mbar_expect_tx(&full[st], kStageBytes);
            tma_load_2d(ring + st * kStageBytes, &wmap, (kb0 + i) * kBlock, r0, &full[st]);
            tma_load_2d(ring + st * kStageBytes + kStageBytes / 2, &wmap, (kb0 + i) * kBlock, r1, &full[st]);
            issued = it + 1;
        }
        flags[1] = issued;
    }
    __syncthreads();

    // After an error, wait (bounded) for every copy still in flight before the
    // CTA exits.
    if (flags[0] != 0 && tid == 0) {
        const int issued = flags[1];
        for (int it = max(0, issued - nst); it < issued; ++it)
            (void)mbar_wait(&full[it % nst], (uint32_t)(it / nst) & 1u);
    }
}

template <int MT, int AMODE, int EPI>
__global__ void __launch_bounds__(kStreamThreads)
    stream_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const StreamParams p) {
    const int m0 = blockIdx.z * MT;
    stream_gemm_body<MT, AMODE, EPI>(wmap, p, m0, min(MT, p.M - m0), 0, 0);
}

// Grouped launch: grid.z = expert x token chunk; expert g owns the token rows
// [off[g], off[g+1]), weight rows [g * wrows, (g+1) * wrows) and block-scale
// rows [g * wrows/128, ...).  Chunks past an expert's tokens leave at once: the
// cluster shares blockIdx.z, so all its CTAs leave together, before any
// cluster barrier.
template <int MT, int AMODE, int EPI>
__global__ void __launch_bounds__(kStreamThreads)
    stream_grouped_kernel(const __grid_constant__ CUtensorMap wmap, const StreamParams p,
                          const __grid_constant__ GroupTable gt) {
    const int g = (int)blockIdx.z / gt.zchunks;
    const int m0 = gt.off[g] + ((int)blockIdx.z - g * gt.zchunks) * MT;
    const int mvalid = min(MT, gt.off[g + 1] - m0);
    if (mvalid <= 0) return;
    stream_gemm_body<MT, AMODE, EPI>(wmap, p, m0, mvalid, g * gt.wrows, g * (gt.wrows / kBlock));
}

template <int AMODE>
cudaError_t launch_stream_impl(const StreamPlan& plan, int epi, const CUtensorMap& wmap,
                               const StreamParams& p, cudaStream_t st, bool pdl) {
    void (*kern)(const CUtensorMap, const StreamParams) = nullptr;
    if (epi == EPI_STORE) {
        switch (plan.MT) {
            case 8: kern = stream_gemm_kernel<8, AMODE, EPI_STORE>; break;
            case 16: kern = stream_gemm_kernel<16, AMODE, EPI_STORE>; break;
            case 32: kern = stream_gemm_kernel<32, AMODE, EPI_STORE>; break;
            case 64: kern = stream_gemm_kernel<64, AMODE, EPI_STORE>; break;
            default: return cudaErrorInvalidValue;
        }
    } else {
        if (AMODE == A_PREQ) return cudaErrorInvalidValue;
        switch (plan.MT) {
            case 8: kern = stream_gemm_kernel<8, AMODE, EPI_SWIGLU>; break;
            case 16: kern = stream_gemm_kernel<16, AMODE, EPI_SWIGLU>; break;
            case 32: kern = stream_gemm_kernel<32, AMODE, EPI_SWIGLU>; break;
            case 64: kern = stream_gemm_kernel<64, AMODE, EPI_SWIGLU>; break;
            default: return cudaErrorInvalidValue;
        }
    }
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), plan.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.splits, (unsigned)plan.groups, (unsigned)plan.mchunks);
    cfg.blockDim = dim3(kStreamThreads, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = st;
    cudaLaunchAttribute attrs[2];
    attrs[0].id = cudaLaunchAttributeClusterDimension;
    attrs[0].val.clusterDim.x = (unsigned)plan.splits;
    attrs[0].val.clusterDim.y = 1;
    attrs[0].val.clusterDim.z = 1;
    int nattr = 1;
    if (pdl) {
        attrs[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[1].val.programmaticStreamSerializationAllowed = 1;
        nattr = 2;
    }
    cfg.attrs = attrs;
    cfg.numAttrs = nattr;
    return cudaLaunchKernelEx(&cfg, kern, wmap, p);
}

}  // namespace r9q
