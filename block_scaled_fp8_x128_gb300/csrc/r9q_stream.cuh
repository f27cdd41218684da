// Decode-width block-scaled fp8 GEMM ("stream" kernel), sm_103a.
//
// At M <= 64 tokens the GEMM is a weight stream: every weight byte is used by
// at most 64 tokens, so HBM bandwidth bounds it (r9700-stack v0.3.1 notes: the
// decode GEMMs' weights are the step's largest stream, and fp8 halves it).
// Design:
//  * grid (S, N/128, ceil(M/MT)), launched as clusters of S CTAs along K.  A
//    CTA owns 128 weight rows (one scale block row, or 64 gate + 64 up rows
//    for the SwiGLU epilogue) and a contiguous range of 128-wide k-blocks.
//  * one producer thread streams 128x128 e4m3 weight tiles with 2-D TMA
//    (128-byte swizzle) into a 4-stage shared-memory ring guarded by
//    full/empty mbarriers; the whole ring is issued before anything else.
//  * the CTA's activation slice arrives in shared memory with one bulk copy
//    per token row, issued right after the weight ring.  W8A8: each 128-wide
//    group is then quantised in place by one warp at the A-load (shuffle amax,
//    fp32 division-exact quotient, cvt.rn.satfinite.e4m3x2), byte-identical
//    to the standalone quant kernel.  Weight-only: the bf16 rows are the B
//    operand, their pairs swapped in registers to match the in-register
//    e4m3 -> bf16 conversion.
//  * four MMA warps run swap-AB mma.sync (weights are the 16-row A operand,
//    tokens the 8-column B operand): m16n8k32 e4m3 for W8A8, m16n8k16 bf16
//    for weight-only.  Each k-block's fp32 partial is promoted into register
//    accumulators with as[m][kb] * ws[nb][kb] (the exact block-scaled form:
//    v0.3.0 notes, exact block-scaled fp8 variant).
//  * split-K is reduced through distributed shared memory: each CTA parks its
//    fp32 partial in its own shared memory, the cluster synchronises, and CTA
//    r sums slice r of the tile over ranks 0..S-1 in that fixed order, so the
//    result is deterministic and no global workspace or counter is needed.
//  * the epilogue writes bf16 y, or (SwiGLU) rounds gate and up to bf16 and
//    writes h = bf16(silu(g) * u).
// Every mbarrier wait is bounded; a timeout records R9Q_ERR_TIMEOUT in the
// device error word, drains the copies in flight and finishes the cluster
// protocol so the kernel always returns.
#pragma once

#include "r9q_device.cuh"
#include "r9q_kernels.h"

namespace r9q {

template <int MT, int AMODE, int EPI>
__global__ void __launch_bounds__(kStreamThreads)
    stream_gemm_kernel(const __grid_constant__ CUtensorMap wmap, const StreamParams p) {
    constexpr int NT = MT / 8;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = p.splits;
    const int split = (int)cluster_ctarank();
    const int tile = blockIdx.y;
    const int m0 = blockIdx.z * MT;
    const int mvalid = min(MT, p.M - m0);
    const int KB = p.KB;
    const int kbase = KB / S, krem = KB % S;
    const int kb0 = split * kbase + min(split, krem);
    const int nkb = kbase + (split < krem ? 1 : 0);
    const int kbs_max = kbase + (krem ? 1 : 0);
    const int kslice = kbs_max * kBlock;

    int r0, r1, nb0, nb1;
    if (EPI == EPI_SWIGLU) {
        const int j = tile >> 1, hh = tile & 1;
        r0 = 2 * kBlock * j + 64 * hh;       // gate rows
        r1 = r0 + kBlock;                    // up rows
        nb0 = 2 * j;
        nb1 = 2 * j + 1;
    } else {
        r0 = kBlock * tile;
        r1 = r0 + 64;
        nb0 = nb1 = tile;
    }

    // shared memory carve-up (must match stream_smem_bytes)
    uint8_t* ring = smem;
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
    uint64_t* empty = full + kStages;
    uint64_t* abar = empty + kStages;                           // activation bulk copies
    int* flags = reinterpret_cast<int*>(abar + 2);              // [0] error, [1] issued
    float* ws_s = reinterpret_cast<float*>(flags + 4);          // [2][kbs_max]
    float* as_s = ws_s + 2 * kbs_max;                           // [MT][kbs_max]
    uintptr_t act_addr = reinterpret_cast<uintptr_t>(as_s + MT * kbs_max);
    uint8_t* act = reinterpret_cast<uint8_t*>((act_addr + 15) & ~static_cast<uintptr_t>(15));
    // Row stride of the activation slice.  W8A8 (fused): bf16 rows whose first
    // kslice bytes are overwritten in place by the e4m3 codes; +16 keeps the
    // code rows on distinct banks for the B-fragment loads.  Weight-only: bf16
    // rows, +32 for the 8-byte B-fragment loads.  Unfused: e4m3 rows.
    const int act_ld = (AMODE == A_QUANT) ? (2 * kslice + 16) : (AMODE == A_BF16) ? (2 * kslice + 32) : (kslice + 16);
    const int row_bytes = (AMODE == A_PREQ) ? nkb * kBlock : 2 * nkb * kBlock;   // bytes copied per token

    if (tid == 0) {
#pragma unroll
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCWarps);
        }
        mbar_init(abar, 1);
        flags[0] = 0;
        flags[1] = 0;
        fence_mbar_init();
    }
    __syncthreads();

    // ---- producer prologue: fill the whole ring, then fetch the activations ----
    const int npro = min(nkb, kStages);
    const bool producer = (warp == kCWarps && lane == 0);
    if (producer) {
        tma_prefetch_desc(&wmap);
        for (int i = 0; i < npro; ++i) {
            mbar_expect_tx(&full[i], kStageBytes);
            tma_load_2d(ring + i * kStageBytes, &wmap, (kb0 + i) * kBlock, r0, &full[i]);
            tma_load_2d(ring + i * kStageBytes + kStageBytes / 2, &wmap, (kb0 + i) * kBlock, r1, &full[i]);
        }
        flags[1] = npro;
    }
    // Weights never come from the preceding kernel; activations and scales may.
    pdl_trigger();
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

    for (int i = tid; i < nkb; i += kStreamThreads) {
        ws_s[i] = p.ws[(int64_t)nb0 * KB + kb0 + i];
        ws_s[kbs_max + i] = p.ws[(int64_t)nb1 * KB + kb0 + i];
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
                if (p.aq != nullptr && tile == 0) {
                    const int64_t off = (int64_t)(m0 + tok) * p.K + (int64_t)(kb0 + kbl) * kBlock + 4 * lane;
                    *reinterpret_cast<uint32_t*>(p.aq + off) = codes;
                    if (lane == 0) p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] = s;
                }
            }
        }
    }
    __syncthreads();

    float acc[2][NT][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][nt][e] = 0.0f;

    const int g = lane >> 2, t = lane & 3;
    if (warp < kCWarps) {
        // ---- MMA warps: rows [32*warp, 32*warp + 32) of the tile ----
        const float* wsv_s = ws_s + (warp >> 1) * kbs_max;
        const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int lchk = lane >> 4;
        for (int i = 0; i < nkb; ++i) {
            const int st = i % kStages;
            if (!mbar_wait(&full[st], (uint32_t)(i / kStages) & 1u)) {
                record_error(p.err, kErrTimeout);
                atomicExch(&flags[0], 1);
                break;
            }
            const uint32_t tbase = smem_u32(ring + st * kStageBytes);
            float d[2][NT][4];
#pragma unroll
            for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                    for (int e = 0; e < 4; ++e) d[mt][nt][e] = 0.0f;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
                uint32_t a[2][4];
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    const int row = warp * 32 + mt * 16 + lrow;
                    const int chunk = ks * 2 + lchk;
                    ldmatrix_x4(tbase + row * 128 + ((chunk ^ (row & 7)) << 4), a[mt][0], a[mt][1], a[mt][2],
                                a[mt][3]);
                }
                if (AMODE != A_BF16) {
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint8_t* bp = act + (nt * 8 + g) * act_ld + i * kBlock + ks * 32 + 4 * t;
                        const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp);
                        const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + 16);
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) mma_e4m3_16832(d[mt][nt], a[mt], b0, b1);
                    }
                } else {
                    uint32_t ev[2][4], od[2][4];
#pragma unroll
                    for (int mt = 0; mt < 2; ++mt)
#pragma unroll
                        for (int r = 0; r < 4; ++r) e4m3x4_to_bf16x2x2(a[mt][r], ev[mt][r], od[mt][r]);
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt) {
                        const uint8_t* bp = act + (nt * 8 + g) * act_ld + 2 * (i * kBlock + ks * 32 + 4 * t);
                        // (x0,x1),(x2,x3) -> (x0,x2),(x1,x3): the pairing of e4m3x4_to_bf16x2x2
                        const uint2 bv = *reinterpret_cast<const uint2*>(bp);
                        const uint2 cv = *reinterpret_cast<const uint2*>(bp + 32);
                        const uint32_t b0 = __byte_perm(bv.x, bv.y, 0x5410), b1 = __byte_perm(bv.x, bv.y, 0x7632);
                        const uint32_t c0 = __byte_perm(cv.x, cv.y, 0x5410), c1 = __byte_perm(cv.x, cv.y, 0x7632);
#pragma unroll
                        for (int mt = 0; mt < 2; ++mt) {
                            mma_bf16_16816(d[mt][nt], ev[mt][0], ev[mt][1], od[mt][0], od[mt][1], b0, b1);
                            mma_bf16_16816(d[mt][nt], ev[mt][2], ev[mt][3], od[mt][2], od[mt][3], c0, c1);
                        }
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
#pragma unroll
                for (int mt = 0; mt < 2; ++mt) {
                    acc[mt][nt][0] = fmaf(d[mt][nt][0], sc0, acc[mt][nt][0]);
                    acc[mt][nt][1] = fmaf(d[mt][nt][1], sc1, acc[mt][nt][1]);
                    acc[mt][nt][2] = fmaf(d[mt][nt][2], sc0, acc[mt][nt][2]);
                    acc[mt][nt][3] = fmaf(d[mt][nt][3], sc1, acc[mt][nt][3]);
                }
            }
        }
    } else if (lane == 0) {
        // ---- producer steady state ----
        int issued = npro;
        for (int i = kStages; i < nkb; ++i) {
            const int st = i % kStages;
            if (!mbar_wait(&empty[st], ((uint32_t)(i / kStages) & 1u) ^ 1u)) {
                record_error(p.err, kErrTimeout);
                atomicExch(&flags[0], 1);
                break;
            }
            mbar_expect_tx(&full[st], kStageBytes);
            tma_load_2d(ring + st * kStageBytes, &wmap, (kb0 + i) * kBlock, r0, &full[st]);
            tma_load_2d(ring + st * kStageBytes + kStageBytes / 2, &wmap, (kb0 + i) * kBlock, r1, &full[st]);
            issued = i + 1;
        }
        flags[1] = issued;
    }
    __syncthreads();

    // After an error, wait (bounded) for every copy still in flight before the
    // ring is reused or the CTA exits.
    if (flags[0] != 0 && tid == 0) {
        const int issued = flags[1];
        for (int i = max(0, issued - kStages); i < issued; ++i)
            (void)mbar_wait(&full[i % kStages], (uint32_t)(i / kStages) & 1u);
    }
    __syncthreads();

    // ---- park the fp32 partial: P[tok][row] in the (now idle) ring ----
    float* P = reinterpret_cast<float*>(ring);
    if (warp < kCWarps) {
#pragma unroll
        for (int mt = 0; mt < 2; ++mt)
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) {
                const int row = warp * 32 + mt * 16 + g;
                const int tok = nt * 8 + 2 * t;
                P[tok * kPStride + row] = acc[mt][nt][0];
                P[(tok + 1) * kPStride + row] = acc[mt][nt][1];
                P[tok * kPStride + row + 8] = acc[mt][nt][2];
                P[(tok + 1) * kPStride + row + 8] = acc[mt][nt][3];
            }
    }
    cluster_sync();

    // ---- split-K reduction over the cluster (fixed rank order) + epilogue ----
    const uint32_t pbase = smem_u32(P);
    constexpr int UPT = (EPI == EPI_SWIGLU) ? 32 : 64;   // units per token
    const int U = MT * UPT;
    const int u_lo = (split * U) / S, u_hi = ((split + 1) * U) / S;
    for (int u = u_lo + tid; u < u_hi; u += kStreamThreads) {
        const int tok = u / UPT, up = u - tok * UPT;
        if (tok >= mvalid) continue;
        if (EPI == EPI_STORE) {
            const uint32_t off = (uint32_t)((tok * kPStride + 2 * up) * 4);
            float2 sum = ld_dsmem_f32x2(dsmem_addr(pbase + off, 0));
            for (int r = 1; r < S; ++r) {
                const float2 v = ld_dsmem_f32x2(dsmem_addr(pbase + off, (uint32_t)r));
                sum.x = __fadd_rn(sum.x, v.x);
                sum.y = __fadd_rn(sum.y, v.y);
            }
            *reinterpret_cast<uint32_t*>(p.y + (int64_t)(m0 + tok) * p.ldy + kBlock * tile + 2 * up) =
                pack_bf16x2(sum.x, sum.y);
        } else {
            const uint32_t offg = (uint32_t)((tok * kPStride + 2 * up) * 4);
            const uint32_t offu = offg + 64 * 4;
            float2 gs = ld_dsmem_f32x2(dsmem_addr(pbase + offg, 0));
            float2 us = ld_dsmem_f32x2(dsmem_addr(pbase + offu, 0));
            for (int r = 1; r < S; ++r) {
                const float2 gv = ld_dsmem_f32x2(dsmem_addr(pbase + offg, (uint32_t)r));
                const float2 uv = ld_dsmem_f32x2(dsmem_addr(pbase + offu, (uint32_t)r));
                gs.x = __fadd_rn(gs.x, gv.x);
                gs.y = __fadd_rn(gs.y, gv.y);
                us.x = __fadd_rn(us.x, uv.x);
                us.y = __fadd_rn(us.y, uv.y);
            }
            const float h0 = silu_mul(bf16_round(gs.x), bf16_round(us.x));
            const float h1 = silu_mul(bf16_round(gs.y), bf16_round(us.y));
            *reinterpret_cast<uint32_t*>(p.y + (int64_t)(m0 + tok) * p.ldy + 64 * tile + 2 * up) =
                pack_bf16x2(h0, h1);
        }
    }
    cluster_sync();   // keep every CTA's shared memory alive until all ranks have read it
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
    cfg.gridDim = dim3((unsigned)plan.splits, (unsigned)plan.ntiles, (unsigned)plan.mchunks);
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
