// Decode-width block-scaled fp8 GEMM ("stream" kernel), mma.sync body, sm_103a.
// Serves the token tiles the tcgen05 body (r9q_stream.cuh) does not take
// (stream_uses_tc): 8-row W8A8 tiles and weight-only tiles of up to 16 rows.
// At those sizes the contraction is a few mma.sync per warp and k-block, and
// the tcgen05 round trip (issue, commit, mbarrier wait, TMEM load) costs more
// than it saves.
//
// At decode widths the GEMM is a weight stream: every weight byte is used by a
// few tokens, so HBM bandwidth bounds it (r9700-stack v0.3.1 notes: the decode
// GEMMs' weights are the step's largest stream, and fp8 halves it).
// Design:
//  * grid (S, G, ceil(M/MT)) launched as clusters of S CTAs along K.  Cluster
//    g owns the 128-row weight tiles t = g, g+G, g+2G, ... (one scale block
//    row, or 64 gate + 64 up rows for the SwiGLU epilogue); CTA s of the
//    cluster owns a contiguous range of 128-wide k-blocks of every such tile.
//  * one producer thread streams the CTA's 128x128 e4m3 weight tiles with 2-D
//    TMA (128-byte swizzle) through a shared-memory ring guarded by full/empty
//    mbarriers, running ahead across tile boundaries.
//  * the producer thread initialises the ring barriers and issues the weight
//    stages as its first act, before any block or cluster barrier; the cluster
//    barrier and the dependency wait (griddepcontrol.wait) come after.  The
//    CTA's activation slice then arrives in shared memory with one bulk copy
//    per token row and serves every tile of the CTA.  W8A8: each 128-wide
//    group is quantised in place once per CTA at the A-load, spread over all
//    warps (shuffle amax, fp32-division-exact quotient,
//    cvt.rn.satfinite.e4m3x2), byte-identical to the standalone quant kernel.
//    Weight-only: the bf16 rows are the B operand, their pairs swapped in
//    registers to match the in-register e4m3 -> bf16 conversion.
//  * eight MMA warps (16 weight rows each; the row-group count kSyncRowGroups
//    lets a warp hold several 16-row groups that share its activation
//    fragments, measured slower) run swap-AB mma.sync (weights are the 16-row
//    A operand, tokens the 8-column B operand): m16n8k32 e4m3 for W8A8,
//    m16n8k16 bf16 for weight-only.  Each k-block's fp32 partial is
//    promoted into register accumulators with as[m][kb] * ws[nb][kb] (the
//    exact block-scaled form: v0.3.0 notes, exact block-scaled fp8 variant).
//  * split-K is reduced through distributed shared memory, pushed: every rank
//    owns a slice of each tile's output columns (whole column pairs), and each
//    MMA warp stores its accumulators straight from registers into the owners'
//    receive buffers with st.async, whose bytes complete on the owner's
//    mbarrier (no fence or arrive by the pushers); the owner sums its slice
//    over ranks 0..S-1 in that fixed order (deterministic, no global
//    workspace).  With several tiles per CTA the receive buffers alternate,
//    and an owner tells the pushers when a buffer may be refilled.
//  * the epilogue writes bf16 y, or (SwiGLU) rounds gate and up to bf16 and
//    writes h = bf16(silu(g) * u).
// Every mbarrier wait is bounded; a timeout records R9Q_ERR_TIMEOUT in the
// device error word and the kernel drains its copies and returns.
#pragma once

#include "r9q_stream_common.cuh"

namespace r9q {

constexpr int kSyncRowGroups = 1;                 // 16-row mma groups a consumer warp holds
constexpr int kSyncThreads = (kCWarps + 1) * 32;  // consumer warps + the producer warp

// The kernel body for the token rows [m0, m0 + mvalid) (mvalid >= 1) of one
// problem whose weight rows start at wrow0 and whose block-scale rows start at
// nbase (both 0 for a single GEMM; an expert's offsets in the grouped launch).
template <int MT, int AMODE, int EPI>
__device__ __forceinline__ void stream_sync_body(const CUtensorMap& wmap, const StreamParams& p, const int m0,
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
    uint64_t* rfull = abar + 1;                  // [2] every rank's slice of a tile has landed in buffer b
    uint64_t* rfree = abar + 3;                  // [2] every rank has summed what I pushed into its buffer b
    int* flags = reinterpret_cast<int*>(bars + 2 * kMaxStages + 5);   // [0] error, [1] issued
    const int rr = stream_recv_rows(S);                               // receive rows per source rank
    float* R = reinterpret_cast<float*>(smem + nst * kStageBytes + kBarBytes);   // [npbuf][S][rr][MT]
    const int npbuf = ntl_max > 1 ? 2 : 1;                            // receive buffers
    float* ws_s = R + npbuf * S * rr * MT;                            // [ntl_max][2][kbs_max]
    float* as_s = ws_s + ntl_max * 2 * kbs_max;                       // [MT][kbs_max]
    uintptr_t act_addr = reinterpret_cast<uintptr_t>(as_s + MT * kbs_max);
    uint8_t* act = reinterpret_cast<uint8_t*>((act_addr + 15) & ~static_cast<uintptr_t>(15));
    // Row stride of the activation slice.  W8A8 (fused): bf16 rows whose first
    // kslice bytes are overwritten in place by the e4m3 codes; +16 keeps the
    // code rows on distinct banks for the B-fragment loads.  Weight-only: bf16
    // rows, +32 for the 8-byte B-fragment loads.  Unfused: e4m3 rows.
    const int act_ld = (AMODE == A_QUANT) ? (2 * kslice + 16) : (AMODE == A_BF16) ? (2 * kslice + 32) : (kslice + 16);
    const int row_bytes = (AMODE == A_PREQ) ? nkb * kBlock : 2 * nkb * kBlock;   // bytes copied per token

    // ---- producer prologue: its barriers, then the weight ring at once ----
    const bool producer = (warp == kCWarps && lane == 0);
    const int npro = min(iters, nst);
    if (producer) {
        for (int s = 0; s < nst; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCWarps);
        }
        mbar_init(abar, 1);
        flags[0] = 0;
        flags[1] = npro;
        fence_proxy_async_smem();     // the TMA unit sees the initialised ring barriers
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
    // Bytes this rank receives per tile: every rank's values (all MT tokens)
    // of the rows of my slice (plain store: 2 rows a column pair; SwiGLU: a
    // gate and an up row per h column).
    const int q_lo = slice_first_pair<EPI>(split, S), q_hi = slice_first_pair<EPI>(split + 1, S);
    const uint32_t recv_bytes = (uint32_t)(S * (EPI == EPI_SWIGLU ? 4 : 2) * (q_hi - q_lo) * MT * 4);
    if (tid == 0) {
        // rfull: one arrival (mine, with the byte count) plus the peers' bytes
        mbar_init(&rfull[0], 1);
        mbar_init(&rfull[1], 1);
        mbar_init(&rfree[0], S);
        mbar_init(&rfree[1], S);
        fence_mbar_init();            // peers see them once the cluster barrier below completes
        // arm the receive barriers of my first two tiles (peers' bytes may land
        // before or after; the phase completes when both are in)
        if (ntl > 0) mbar_expect_tx(&rfull[0], recv_bytes);
        if (ntl > 1) mbar_expect_tx(&rfull[1], recv_bytes);
    }
    // the MMA warps use the barriers just initialised
    __syncthreads();
    // Every peer's barriers must exist before anyone arrives on them remotely:
    // arrive on the cluster barrier now, wait for it only just before the
    // first remote access.  Peers touch nothing of this CTA but those barriers
    // and the receive buffers they write, so the arrive is relaxed: the
    // initialisation is released by fence_mbar_init above.
    cluster_arrive_relaxed();

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
    for (int c = tid; c < ntl * nkb; c += kSyncThreads) {
        const int tl = c / nkb, i = c - tl * nkb;
        int r0, r1, nb0, nb1;
        tile_rows<EPI>(group + tl * G, r0, r1, nb0, nb1);
        ws_s[(tl * 2 + 0) * kbs_max + i] = p.ws[(int64_t)(nbase + nb0) * KB + kb0 + i];
        ws_s[(tl * 2 + 1) * kbs_max + i] = p.ws[(int64_t)(nbase + nb1) * KB + kb0 + i];
    }
    // every peer's barriers exist (before any remote access below)
    cluster_wait();
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
    for (int c = tid; c < (MT - mvalid) * (row_bytes / 16); c += kSyncThreads) {
        const int tok = mvalid + c / (row_bytes / 16), ch = c % (row_bytes / 16);
        *reinterpret_cast<uint4*>(act + tok * act_ld + ch * 16) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (AMODE == A_PREQ) {
        for (int c = tid; c < MT * nkb; c += kSyncThreads) {
            const int tok = c / nkb, kbl = c - tok * nkb;
            as_s[tok * kbs_max + kbl] = (tok < mvalid) ? p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] : 0.0f;
        }
    } else if (AMODE == A_QUANT) {
        // only the padding rows: the scales of rows < mvalid are written by the
        // quant loop below, which other warps may already be running
        for (int c = tid; c < (MT - mvalid) * nkb; c += kSyncThreads)
            as_s[(mvalid + c / nkb) * kbs_max + c % nkb] = 0.0f;
    }
    if (!mbar_wait(abar, 0)) {
        record_error(p.err, kErrTimeout);
        atomicExch(&flags[0], 1);
    }

    if (AMODE == A_QUANT) {
        // In-place group quantisation.  At most one group per warp: each warp
        // reads one group, the CTA synchronises (the warp alone when a row has
        // one group), each warp writes that group's codes over the start of
        // its data.  More groups: each warp walks its
        // rows, four groups (eight lanes a group) a pass; pass j reads bytes
        // [1024j, 1024j + 1024) of the row and writes the codes to bytes
        // [512j, 512j + 512), which only this pass or earlier ones have read,
        // with all the warp's reads of a pass before its writes.
        constexpr int W = kCWarps + 1;
        if (mvalid * nkb <= W) {
            const bool on = warp < mvalid * nkb;
            const int tok = on ? warp / nkb : 0, kbl = on ? warp - tok * nkb : 0;
            uint8_t* row = act + tok * act_ld;
            uint2 v = make_uint2(0u, 0u);
            if (on) v = *reinterpret_cast<const uint2*>(row + kbl * 2 * kBlock + 8 * lane);
            if (nkb > 1) __syncthreads();   // one group a row: no other warp touches the row
            else __syncwarp();
            if (on) {
                float sc;
                const uint32_t codes = quant_group128_warp(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), sc);
                *reinterpret_cast<uint32_t*>(row + kbl * kBlock + 4 * lane) = codes;
                if (lane == 0) as_s[tok * kbs_max + kbl] = sc;
                if (p.aq != nullptr && group == 0) {
                    const int64_t off = (int64_t)(m0 + tok) * p.K + (int64_t)(kb0 + kbl) * kBlock + 4 * lane;
                    *reinterpret_cast<uint32_t*>(p.aq + off) = codes;
                    if (lane == 0) p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] = sc;
                }
            }
        } else {
            const int gl = lane >> 3, el = (lane & 7) * 16;
            for (int tok = warp; tok < mvalid; tok += W) {
                uint8_t* row = act + tok * act_ld;
                for (int kb4 = 0; kb4 < nkb; kb4 += 4) {
                    const int kbl = kb4 + gl;
                    uint4 v[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                    if (kbl < nkb) {
                        v[0] = *reinterpret_cast<const uint4*>(row + kbl * 2 * kBlock + 2 * el);
                        v[1] = *reinterpret_cast<const uint4*>(row + kbl * 2 * kBlock + 2 * el + 16);
                    }
                    __syncwarp();
                    float sc;
                    const uint4 codes = quant_group128_lane8(v, sc);
                    if (kbl < nkb) {
                        *reinterpret_cast<uint4*>(row + kbl * kBlock + el) = codes;
                        if ((lane & 7) == 0) as_s[tok * kbs_max + kbl] = sc;
                        if (p.aq != nullptr && group == 0) {
                            const int64_t off = (int64_t)(m0 + tok) * p.K + (int64_t)(kb0 + kbl) * kBlock + el;
                            *reinterpret_cast<uint4*>(p.aq + off) = codes;
                            if ((lane & 7) == 0) p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] = sc;
                        }
                    }
                    __syncwarp();
                }
            }
        }
    }
    __syncthreads();

    const int g = lane >> 2, t = lane & 3;
    if (warp < kCWarps) {
        // ---- MMA warps: rows [16*RG*warp, 16*RG*(warp + 1)) of every tile, as
        // RG 16-row groups that share every activation fragment the warp loads ----
        constexpr int RG = kSyncRowGroups;
        const int box = (warp * 16 * RG) >> 6;           // 64-row half: scale row nb0 or nb1
        const int lrow = (lane & 7) + ((lane >> 3) & 1) * 8;
        const int lchk = lane >> 4;
        // A failed wait sets flags[0]; from then on every wait is skipped but
        // all MMA warps keep walking the same loop and barrier sequence, so no
        // warp is left waiting at a named barrier.
        volatile int* vflags = flags;
        auto fail = [&]() {
            record_error(p.err, kErrTimeout);
            atomicExch(&flags[0], 1);
        };
        // Tile tl's partial is pushed, then tile tl-1 is reduced: the wait for
        // the peers' partials of one tile overlaps the MMAs of the next.
        for (int tl = 0; tl <= ntl; ++tl) {
            if (tl < ntl) {
                float acc[RG][NT][4];
#pragma unroll
                for (int rg = 0; rg < RG; ++rg)
#pragma unroll
                    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[rg][nt][e] = 0.0f;
                const float* wsv_s = ws_s + (tl * 2 + box) * kbs_max;
                for (int i = 0; i < nkb; ++i) {
                    const int it = tl * nkb + i;
                    const int st = it % nst;
                    if (*vflags == 0 && !mbar_wait(&full[st], (uint32_t)(it / nst) & 1u)) fail();
                    const uint32_t tbase = smem_u32(ring + st * kStageBytes);
                    float d[RG][NT][4];
#pragma unroll
                    for (int rg = 0; rg < RG; ++rg)
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
#pragma unroll
                            for (int e = 0; e < 4; ++e) d[rg][nt][e] = 0.0f;
#pragma unroll
                    for (int ks = 0; ks < 4; ++ks) {
                        const int chunk = ks * 2 + lchk;
                        uint32_t a[RG][4];
#pragma unroll
                        for (int rg = 0; rg < RG; ++rg) {
                            const int row = warp * 16 * RG + rg * 16 + lrow;
                            ldmatrix_x4(tbase + row * 128 + ((chunk ^ (row & 7)) << 4), a[rg][0], a[rg][1], a[rg][2],
                                        a[rg][3]);
                        }
                        if (AMODE != A_BF16) {
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint8_t* bp = act + (nt * 8 + g) * act_ld + i * kBlock + ks * 32 + 4 * t;
                                const uint32_t b0 = *reinterpret_cast<const uint32_t*>(bp);
                                const uint32_t b1 = *reinterpret_cast<const uint32_t*>(bp + 16);
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg) mma_e4m3_16832(d[rg][nt], a[rg], b0, b1);
                            }
                        } else {
                            uint32_t ev[RG][4], od[RG][4];
#pragma unroll
                            for (int rg = 0; rg < RG; ++rg)
#pragma unroll
                                for (int r = 0; r < 4; ++r) e4m3x4_to_bf16x2x2(a[rg][r], ev[rg][r], od[rg][r]);
#pragma unroll
                            for (int nt = 0; nt < NT; ++nt) {
                                const uint8_t* bp = act + (nt * 8 + g) * act_ld + 2 * (i * kBlock + ks * 32 + 4 * t);
                                // (x0,x1),(x2,x3) -> (x0,x2),(x1,x3): the pairing of e4m3x4_to_bf16x2x2
                                const uint2 bv = *reinterpret_cast<const uint2*>(bp);
                                const uint2 cv = *reinterpret_cast<const uint2*>(bp + 32);
                                const uint32_t b0 = __byte_perm(bv.x, bv.y, 0x5410), b1 = __byte_perm(bv.x, bv.y, 0x7632);
                                const uint32_t c0 = __byte_perm(cv.x, cv.y, 0x5410), c1 = __byte_perm(cv.x, cv.y, 0x7632);
#pragma unroll
                                for (int rg = 0; rg < RG; ++rg) {
                                    mma_bf16_16816(d[rg][nt], ev[rg][0], ev[rg][1], od[rg][0], od[rg][1], b0, b1);
                                    mma_bf16_16816(d[rg][nt], ev[rg][2], ev[rg][3], od[rg][2], od[rg][3], c0, c1);
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
                        for (int rg = 0; rg < RG; ++rg) {
                            acc[rg][nt][0] = fmaf(d[rg][nt][0], sc0, acc[rg][nt][0]);
                            acc[rg][nt][1] = fmaf(d[rg][nt][1], sc1, acc[rg][nt][1]);
                            acc[rg][nt][2] = fmaf(d[rg][nt][2], sc0, acc[rg][nt][2]);
                            acc[rg][nt][3] = fmaf(d[rg][nt][3], sc1, acc[rg][nt][3]);
                        }
                    }
                }

                // ---- push the tile's partial to the ranks that own its rows ----
                // into buffer b = tl & 1 of each owner, once every owner has
                // summed what was pushed there two tiles ago; the stores count
                // their bytes on the owner's rfull[b]
                const int b = tl & 1;
                const uint32_t use = (uint32_t)(tl >> 1);
                if (tl >= 2 && *vflags == 0 && !mbar_wait_cluster(&rfree[b], (use - 1) & 1u)) fail();
                const uint32_t rbase = smem_u32(R + (size_t)b * S * rr * MT) + (uint32_t)(split * rr * MT * 4);
                const uint32_t rbar = smem_u32(&rfull[b]);
#pragma unroll
                for (int rg = 0; rg < RG; ++rg)
#pragma unroll
                    for (int h8 = 0; h8 < 2; ++h8) {
                        int owner, u;
                        slice_of<EPI>(warp * 16 * RG + rg * 16 + g + 8 * h8, S, owner, u);
                        const uint32_t dst = dsmem_addr(rbase + (uint32_t)(u * MT * 4), (uint32_t)owner);
                        const uint32_t dbar = dsmem_addr(rbar, (uint32_t)owner);
#pragma unroll
                        for (int nt = 0; nt < NT; ++nt)
                            st_async_f32x2(dst + (uint32_t)((nt * 8 + 2 * t) * 4), acc[rg][nt][2 * h8],
                                           acc[rg][nt][2 * h8 + 1], dbar);
                    }
            }
            if (tl >= 1) {
                // ---- tile rt: sum my slice over the ranks 0..S-1, in that order ----
                const int rt = tl - 1;
                const int tile = group + rt * G;
                const int b = rt & 1;
                const uint32_t use = (uint32_t)(rt >> 1);
                if (*vflags == 0 && !mbar_wait_cluster(&rfull[b], use & 1u)) fail();
                const float* Rb = R + (size_t)b * S * rr * MT;
                const int q0 = slice_first_pair<EPI>(split, S), q1 = slice_first_pair<EPI>(split + 1, S);
                const int units = (q1 - q0) * MT;                   // (column pair, token), token fastest
                constexpr int MAXU = (64 * MT + kCWarps * 32 - 1) / (kCWarps * 32);   // S = 1 holds the most
                const int cap = 2 * ((32 + S - 1) / S);              // SwiGLU: up rows follow `cap` gate rows
                uint32_t outv[MAXU];
#pragma unroll
                for (int jj = 0; jj < MAXU; ++jj) {
                    const int q = tid + jj * kCWarps * 32;
                    outv[jj] = 0u;
                    if (q >= units) continue;
                    const int pr = q / MT, tok = q - pr * MT;
                    if (tok >= mvalid) continue;
                    const int u = 2 * pr;
                    if (EPI == EPI_STORE) {
                        float s0 = Rb[u * MT + tok], s1 = Rb[(u + 1) * MT + tok];
                        for (int r = 1; r < S; ++r) {
                            s0 = __fadd_rn(s0, Rb[(r * rr + u) * MT + tok]);
                            s1 = __fadd_rn(s1, Rb[(r * rr + u + 1) * MT + tok]);
                        }
                        outv[jj] = pack_bf16x2(s0, s1);
                    } else {
                        float g0 = Rb[u * MT + tok], g1 = Rb[(u + 1) * MT + tok];
                        float u0 = Rb[(cap + u) * MT + tok], u1 = Rb[(cap + u + 1) * MT + tok];
                        for (int r = 1; r < S; ++r) {
                            const float* Rr = Rb + r * rr * MT;
                            g0 = __fadd_rn(g0, Rr[u * MT + tok]);
                            g1 = __fadd_rn(g1, Rr[(u + 1) * MT + tok]);
                            u0 = __fadd_rn(u0, Rr[(cap + u) * MT + tok]);
                            u1 = __fadd_rn(u1, Rr[(cap + u + 1) * MT + tok]);
                        }
                        outv[jj] = pack_bf16x2(silu_mul(bf16_round(g0), bf16_round(u0)),
                                               silu_mul(bf16_round(g1), bf16_round(u1)));
                    }
                }
                // the pushers may reuse buffer b (tile rt + 2) once every owner has read it
                if (rt + 2 < ntl) {
                    consumer_sync();
                    if (tid == 0) {
                        mbar_expect_tx(&rfull[b], recv_bytes);      // armed for tile rt + 2
                        mbar_arrive_all_ranks(&rfree[b], S);
                    }
                }
#pragma unroll
                for (int jj = 0; jj < MAXU; ++jj) {
                    const int q = tid + jj * kCWarps * 32;
                    if (q >= units) continue;
                    const int pr = q / MT, tok = q - pr * MT;
                    if (tok >= mvalid) continue;
                    const int64_t col = (EPI == EPI_STORE ? (int64_t)kBlock * tile : (int64_t)64 * tile) + 2 * (q0 + pr);
                    *reinterpret_cast<uint32_t*>(p.y + (int64_t)(m0 + tok) * p.ldy + col) = outv[jj];
                }
            }
        }
        // Peers touch my shared memory with their pushes (the last tile's have
        // landed once its rfull wait above completed) and with their arrives on
        // my rfree barriers, the last of which completes the last round of each
        // buffer: wait for those rounds before leaving (bounded, also after an
        // error, when the waits above may have been skipped).
        if (*vflags != 0 && ntl > 0)
            (void)mbar_wait_cluster(&rfull[(ntl - 1) & 1], (uint32_t)((ntl - 1) >> 1) & 1u);
        for (int b2 = 0; b2 < 2; ++b2) {
            const int rounds = (ntl - 2 - b2 + 1) / 2;       // tiles rt = b2, b2 + 2, ... with rt + 2 < ntl
            if (rounds > 0 && !mbar_wait_cluster(&rfree[b2], (uint32_t)(rounds - 1) & 1u)) fail();
        }
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
__global__ void __launch_bounds__(kSyncThreads, stream_min_blocks(MT, AMODE == A_BF16 ? A_BF16 : A_QUANT))
    stream_sync_kernel(const __grid_constant__ CUtensorMap wmap, const StreamParams p) {
    const int m0 = blockIdx.z * MT;
    stream_sync_body<MT, AMODE, EPI>(wmap, p, m0, min(MT, p.M - m0), 0, 0);
}

// Grouped launch: grid.z = expert x token chunk; expert g owns the token rows
// [off[g], off[g+1]), weight rows [g * wrows, (g+1) * wrows) and block-scale
// rows [g * wrows/128, ...).  Chunks past an expert's tokens leave at once: the
// cluster shares blockIdx.z, so all its CTAs leave together, before any
// cluster barrier.
template <int MT, int AMODE, int EPI>
__global__ void __launch_bounds__(kSyncThreads, stream_min_blocks(MT, AMODE == A_BF16 ? A_BF16 : A_QUANT))
    stream_sync_grouped_kernel(const __grid_constant__ CUtensorMap wmap, const StreamParams p,
                          const __grid_constant__ GroupTable gt) {
    const int g = (int)blockIdx.z / gt.zchunks;
    const int m0 = gt.off[g] + ((int)blockIdx.z - g * gt.zchunks) * MT;
    const int mvalid = min(MT, gt.off[g + 1] - m0);
    if (mvalid <= 0) return;
    stream_sync_body<MT, AMODE, EPI>(wmap, p, m0, mvalid, g * gt.wrows, g * (gt.wrows / kBlock));
}

}  // namespace r9q
