// Decode-width block-scaled fp8 GEMM ("stream" kernel), tcgen05 body, sm_103a.
//
// At decode widths the GEMM is a weight stream: every weight byte is used by a
// few tokens, so HBM bandwidth bounds it (r9700-stack v0.3.1 notes: the decode
// GEMMs' weights are the step's largest stream, and fp8 halves it).  This body
// serves W8A8 token tiles of 16 to 64 rows (stream_uses_tc); 8-row tiles and
// weight-only calls run the mma.sync body (r9q_stream_sync.cuh), which shares
// the grid, the weight ring and the split-K exchange described here.
// Design:
//  * grid (S, G, ceil(M/MT)) launched as clusters of S CTAs along K.  Cluster
//    g owns the 128-row weight tiles t = g, g+G, g+2G, ... (one scale block
//    row, or 64 gate + 64 up rows for the SwiGLU epilogue); CTA s of the
//    cluster owns a contiguous range of 128-wide k-blocks of every such tile.
//  * warp 8, lane 0 streams the CTA's 128x128 e4m3 weight tiles with 2-D TMA
//    (128-byte swizzle) through a shared-memory ring guarded by full/empty
//    mbarriers, running ahead across tile boundaries; it initialises the ring
//    barriers and issues the first stages as its first act, before any block
//    or cluster barrier.  The cluster barrier and the dependency wait
//    (griddepcontrol.wait) come after; the CTA's activation slice then arrives
//    with one bulk copy per token row.
//  * the B operand: every warp turns the activation slice into e4m3 rows of a
//    128-byte-swizzled K-major tile in shared memory (MMA width N = max(MT,
//    16) rows, zero past the last token), with one scale per (token, k-block).
//    W8A8: the group-128 quantisation (shuffle amax, fp32-division-exact
//    quotient, cvt.rn.satfinite.e4m3x2), byte-identical to the standalone
//    quant kernel; pre-quantised activations are copied into the layout.
//  * warp 9: TMEM allocation (kAccBufs partial buffers of N fp32 columns) and,
//    lane 0, the MMAs: per k-block four tcgen05.mma.kind::f8f6f4
//    M=128 x N x K=32 straight from the TMA stage
//    and the B tile, committed to the stage's empty barrier and to the
//    buffer's mdone barrier.
//  * warps 0..7 (TMEM lane quarter = warp % 4, token columns by warp / 4)
//    tcgen05.ld each k-block's partial and promote it into register
//    accumulators with as[m][kb] * ws[nb][kb] (the exact block-scaled form:
//    v0.3.0 notes, exact block-scaled fp8 variant).
//  * split-K is reduced through distributed shared memory, pushed: every rank
//    owns a slice of each tile's output columns (whole column pairs), and each
//    promoting thread stores its row's accumulators straight from registers
//    into the owner's receive buffer with st.async, whose bytes complete on
//    the owner's mbarrier (no fence or arrive by the pushers); the owner sums
//    its slice over ranks 0..S-1 in that fixed order (deterministic, no
//    global workspace).  With several tiles per CTA the receive buffers
//    alternate, and an owner tells the pushers when a buffer may be refilled.
//  * the epilogue writes bf16 y, or (SwiGLU) rounds gate and up to bf16 and
//    writes h = bf16(silu(g) * u).
// Every mbarrier wait is bounded; a timeout records R9Q_ERR_TIMEOUT in the
// device error word and the kernel drains its copies and MMAs, frees its TMEM
// and returns.
#pragma once

#include "r9q_stream_common.cuh"

namespace r9q {

// Byte offset of 16-byte chunk ch (k = 16*ch .. 16*ch + 15) of token row tok in
// k-block kbl of the B operand: per k-block N rows of 128 bytes, 8-row atoms
// of 1024 bytes with the 128-byte swizzle (chunk index XOR row within the
// atom), the layout the tensor cores read through umma_sdesc_sw128.
template <int N>
__device__ __forceinline__ uint32_t b_offset(int tok, int kbl, int ch) {
    return (uint32_t)(kbl * (N * 128) + (tok >> 3) * 1024 + (tok & 7) * 128 + ((ch ^ (tok & 7)) << 4));
}

// The kernel body for the token rows [m0, m0 + mvalid) (mvalid >= 1) of one
// problem whose weight rows start at wrow0 and whose block-scale rows start at
// nbase (both 0 for a single GEMM; an expert's offsets in the grouped launch).
template <int MT, int AMODE, int EPI>
__device__ __forceinline__ void stream_gemm_body(const CUtensorMap& wmap, const StreamParams& p, const int m0,
                                                 const int mvalid, const int wrow0, const int nbase) {
    constexpr int N = stream_mma_n(MT);                   // MMA width (token columns, zero rows past MT)
    constexpr int TPW = MT >= 16 ? MT / 2 : 8;            // token columns a promoting thread holds
    constexpr int NPROMO = MT >= 16 ? kCWarps : 4;        // promoting warps (columns [TPW*(w/4), +TPW))
    static_assert(AMODE != A_BF16, "weight-only calls run the mma.sync body");
    constexpr uint32_t kIdesc = umma_idesc_e4m3(128, N);
    constexpr uint32_t kTmemCols = (uint32_t)stream_tmem_cols(MT);
    constexpr int kMmaWarp = kCWarps + 1;
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

    // Activation rows as copied: bf16 (fused quant) or e4m3 codes.
    const int act_ld = (AMODE == A_PREQ) ? kslice : 2 * kslice;
    const int act_bytes = MT * act_ld;                           // a multiple of 1024
    // shared memory carve-up (must match stream_smem_bytes)
    uint8_t* ring = smem;                                        // [nst][128 rows x 128 B] weights
    uint8_t* act = smem + nst * kStageBytes;                     // [MT][act_ld] activation rows
    uint8_t* bop = act + act_bytes;                              // [kbs_max][N rows x 128 B]
    // Once the B tile is built the activation rows are dead: their space
    // continues the ring (stages nst .. ntot-1, used from the first refill on).
    const int ntot = min(nst + act_bytes / kStageBytes, kMaxRing);
    const int bterm = kbs_max * N * 128;
    uint64_t* bars = reinterpret_cast<uint64_t*>(bop + bterm);
    uint64_t* full = bars;                       // [kMaxRing] weight stage landed
    uint64_t* empty = bars + kMaxRing;           // [kMaxRing] the MMAs reading the stage are done
    uint64_t* abar = bars + 2 * kMaxRing;        // activation bulk copies
    uint64_t* rfull = abar + 1;                  // [2] every rank's slice of a tile has landed in buffer b
    uint64_t* rfree = abar + 3;                  // [2] every rank has summed what I pushed into its buffer b
    uint64_t* mdone = abar + 5;                  // [kAccBufs] TMEM partial buffer holds a finished k-block
    uint64_t* tfree = mdone + kAccBufs;          // [kAccBufs] the promoting warps have read the buffer
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tfree + kAccBufs);
    int* flags = reinterpret_cast<int*>(tmem_slot + 2);   // [0] error, [1] stages issued, [2] k-blocks committed
    const int rr = stream_recv_rows(S);                               // receive rows per source rank
    float* R = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + kBarBytes);   // [npbuf][S][rr][MT]
    const int npbuf = ntl_max > 1 ? 2 : 1;                            // receive buffers
    float* ws_s = R + npbuf * S * rr * MT;                            // [ntl_max][2][kbs_max]
    float* as_s = ws_s + ntl_max * 2 * kbs_max;                       // [MT][kbs_max]
    const int row_bytes = (AMODE == A_PREQ) ? nkb * kBlock : 2 * nkb * kBlock;   // bytes copied per token

    // ---- producer prologue: its barriers, then the weight ring at once ----
    const bool producer = (warp == kCWarps && lane == 0);
    const int npro = min(iters, nst);
    if (producer) {
        for (int s = 0; s < ntot; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        mbar_init(abar, 1);
        for (int b = 0; b < kAccBufs; ++b) {
            mbar_init(&mdone[b], 1);
            mbar_init(&tfree[b], NPROMO);
        }
        flags[0] = 0;
        flags[1] = npro;
        flags[2] = 0;
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
    if (warp == kMmaWarp) tmem_alloc(tmem_slot, kTmemCols);
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
    // the barriers just initialised and the TMEM address are used below
    umma_fence_before();
    __syncthreads();
    umma_fence_after();
    const uint32_t tmem_base = *tmem_slot;
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
    const int nws = ntl * nkb;
    for (int c = tid; c < nws; c += kStreamThreads) {
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
    // B rows past the last token: zero codes; their scales: zero
    for (int c = tid; c < nkb * (N - mvalid) * 8; c += kStreamThreads) {
        const int kbl = c / ((N - mvalid) * 8), r2 = c - kbl * ((N - mvalid) * 8);
        const int tok = mvalid + (r2 >> 3), ch = r2 & 7;
        *reinterpret_cast<uint4*>(bop + b_offset<N>(tok, kbl, ch)) = make_uint4(0u, 0u, 0u, 0u);
    }
    if (AMODE == A_PREQ) {
        for (int c = tid; c < MT * nkb; c += kStreamThreads) {
            const int tok = c / nkb, kbl = c - tok * nkb;
            as_s[tok * kbs_max + kbl] = (tok < mvalid) ? p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] : 0.0f;
        }
    } else {
        // only the padding rows: the scales of rows < mvalid are written below
        for (int c = tid; c < (MT - mvalid) * nkb; c += kStreamThreads)
            as_s[(mvalid + c / nkb) * kbs_max + c % nkb] = 0.0f;
    }
    if (!mbar_wait(abar, 0)) {
        record_error(p.err, kErrTimeout);
        atomicExch(&flags[0], 1);
    }

    // ---- the B operand: the CTA's activation slice as e4m3, in the swizzled
    // layout, with its scale per (token, k-block) in as_s ----
    constexpr int W = kCWarps + 2;
    if (AMODE == A_QUANT) {
        // Group-128 quantisation.  At most one group per warp: each warp takes
        // one group; otherwise four groups a warp pass, eight lanes a group.
        if (mvalid * nkb <= W) {
            if (warp < mvalid * nkb) {
                const int tok = warp / nkb, kbl = warp - tok * nkb;
                const uint2 v = *reinterpret_cast<const uint2*>(act + tok * act_ld + kbl * 2 * kBlock + 8 * lane);
                float sc;
                const uint32_t codes = quant_group128_warp(bf16_lo(v.x), bf16_hi(v.x), bf16_lo(v.y), bf16_hi(v.y), sc);
                *reinterpret_cast<uint32_t*>(bop + b_offset<N>(tok, kbl, lane >> 2) + 4 * (lane & 3)) = codes;
                if (lane == 0) as_s[tok * kbs_max + kbl] = sc;
                if (p.aq != nullptr && group == 0) {
                    const int64_t off = (int64_t)(m0 + tok) * p.K + (int64_t)(kb0 + kbl) * kBlock + 4 * lane;
                    *reinterpret_cast<uint32_t*>(p.aq + off) = codes;
                    if (lane == 0) p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] = sc;
                }
            }
        } else {
            const int gl = lane >> 3, el = (lane & 7) * 16;
            const int ngroups = mvalid * nkb, nquads = (ngroups + 3) >> 2;
            for (int qd = warp; qd < nquads; qd += W) {
                const int gi = qd * 4 + gl;
                const bool on = gi < ngroups;
                const int tok = on ? gi / nkb : 0, kbl = on ? gi - tok * nkb : 0;
                uint4 v[2] = {make_uint4(0u, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u)};
                if (on) {
                    v[0] = *reinterpret_cast<const uint4*>(act + tok * act_ld + kbl * 2 * kBlock + 2 * el);
                    v[1] = *reinterpret_cast<const uint4*>(act + tok * act_ld + kbl * 2 * kBlock + 2 * el + 16);
                }
                float sc;
                const uint4 codes = quant_group128_lane8(v, sc);
                if (on) {
                    *reinterpret_cast<uint4*>(bop + b_offset<N>(tok, kbl, lane & 7)) = codes;
                    if ((lane & 7) == 0) as_s[tok * kbs_max + kbl] = sc;
                    if (p.aq != nullptr && group == 0) {
                        const int64_t off = (int64_t)(m0 + tok) * p.K + (int64_t)(kb0 + kbl) * kBlock + el;
                        *reinterpret_cast<uint4*>(p.aq + off) = codes;
                        if ((lane & 7) == 0) p.as[(int64_t)(m0 + tok) * KB + kb0 + kbl] = sc;
                    }
                }
            }
        }
    } else {
        // pre-quantised codes: copied rows -> swizzled layout
        for (int c = tid; c < mvalid * nkb * 8; c += kStreamThreads) {
            const int tok = c / (nkb * 8), r = c - tok * (nkb * 8), kbl = r >> 3, ch = r & 7;
            *reinterpret_cast<uint4*>(bop + b_offset<N>(tok, kbl, ch)) =
                *reinterpret_cast<const uint4*>(act + tok * act_ld + kbl * kBlock + ch * 16);
        }
    }
    // the tensor cores read B through the async proxy
    fence_proxy_async_smem();
    __syncthreads();

    volatile int* vflags = flags;
    auto fail = [&]() {
        record_error(p.err, kErrTimeout);
        atomicExch(&flags[0], 1);
    };

    if (warp == kMmaWarp) {
        // ---- MMA issuer: k-block it of tile it / nkb into TMEM buffer it % kAccBufs ----
        if (lane == 0) {
            int committed = 0;
            for (int it = 0; it < iters; ++it) {
                if (*vflags != 0) break;
                const int tl = it / nkb, i = it - tl * nkb, st = it % ntot, b = it % kAccBufs;
                (void)tl;
                if (!mbar_wait(&full[st], (uint32_t)(it / ntot) & 1u)) {
                    fail();
                    break;
                }
                if (it >= kAccBufs && !mbar_wait(&tfree[b], (uint32_t)(it / kAccBufs - 1) & 1u)) {
                    fail();
                    break;
                }
                umma_fence_after();
                const uint32_t td = tmem_base + (uint32_t)(b * N);
                const uint32_t sa = smem_u32(ring + st * kStageBytes);
                const uint32_t sb = smem_u32(bop + i * (N * 128));
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    umma_e4m3(td, umma_sdesc_sw128(sa + 32 * k), umma_sdesc_sw128(sb + 32 * k), kIdesc, k ? 1u : 0u);
                umma_commit(&empty[st]);      // the stage may be refilled once these MMAs are done
                umma_commit(&mdone[b]);
                committed = it + 1;
            }
            flags[2] = committed;
            // After an error the promoting warps stop waiting: let the MMAs
            // issued finish before the TMEM is released (bounded).
            if (*vflags != 0 && committed > 0) {
                const int last = committed - 1;
                (void)mbar_wait(&mdone[last % kAccBufs], (uint32_t)(last / kAccBufs) & 1u);
            }
        }
        __syncwarp();
    }

    if (warp < kCWarps) {
        // ---- promotion: warp w reads TMEM lanes 32*(w%4) .. +31 (tile rows)
        // and token columns [TPW*(w/4), +TPW); each k-block's partial is
        // promoted into register accumulators with as[m][kb] * ws[nb][kb] ----
        const bool promo = warp < NPROMO;
        const int row = 32 * (warp & 3) + lane;                 // weight tile row = TMEM lane
        const int cb = (warp >> 2) * TPW;                       // first token column
        const int box = row >> 6;                               // 64-row half: scale row nb0 or nb1
        const uint32_t tlane = (uint32_t)(32 * (warp & 3)) << 16;
        // A failed wait sets flags[0]; from then on every wait is skipped but
        // all warps keep walking the same loop and barrier sequence, so no
        // warp is left waiting at a named barrier.
        // Tile tl's partial is pushed, then tile tl-1 is reduced: the wait for
        // the peers' partials of one tile overlaps the MMAs of the next.
        for (int tl = 0; tl <= ntl; ++tl) {
            if (tl < ntl && promo) {
                float acc[TPW];
#pragma unroll
                for (int j = 0; j < TPW; ++j) acc[j] = 0.0f;
                const float* wsv_s = ws_s + (tl * 2 + box) * kbs_max;
                for (int i = 0; i < nkb; ++i) {
                    const int it = tl * nkb + i, b = it % kAccBufs;
                    if (*vflags == 0 && !mbar_wait(&mdone[b], (uint32_t)(it / kAccBufs) & 1u)) fail();
                    umma_fence_after();
                    float d[TPW];
                    tmem_ld<TPW>(tmem_base + tlane + (uint32_t)(b * N + cb), d);
                    tmem_wait_ld(d);
                    umma_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(&tfree[b]);
                    const float wsv = wsv_s[i];
#pragma unroll
                    for (int j = 0; j < TPW; ++j)
                        acc[j] = fmaf(d[j], as_s[(cb + j) * kbs_max + i] * wsv, acc[j]);
                }

                // ---- push the row's partial to the rank that owns it ----
                // into buffer b = tl & 1 of the owner, once every owner has
                // summed what was pushed there two tiles ago; the stores count
                // their bytes on the owner's rfull[b]
                const int b = tl & 1;
                const uint32_t use = (uint32_t)(tl >> 1);
                if (tl >= 2 && *vflags == 0 && !mbar_wait_cluster(&rfree[b], (use - 1) & 1u)) fail();
                const uint32_t rbase = smem_u32(R + (size_t)b * S * rr * MT) + (uint32_t)(split * rr * MT * 4);
                int owner, u;
                slice_of<EPI>(row, S, owner, u);
                const uint32_t dst = dsmem_addr(rbase + (uint32_t)((u * MT + cb) * 4), (uint32_t)owner);
                const uint32_t dbar = dsmem_addr(smem_u32(&rfull[b]), (uint32_t)owner);
#pragma unroll
                for (int c4 = 0; c4 < TPW / 4; ++c4)
                    st_async_f32x4(dst + (uint32_t)(16 * c4), acc[4 * c4], acc[4 * c4 + 1], acc[4 * c4 + 2],
                                   acc[4 * c4 + 3], dbar);
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
        // (after the B tile is built: the stages past nst are free from here on)
        int issued = npro;
        int cur_tl = -1, r0 = 0, r1 = 0, nb0, nb1;
        for (int it = npro; it < iters; ++it) {
            const int st = it % ntot;
            if (it >= ntot && !mbar_wait(&empty[st], ((uint32_t)(it / ntot) & 1u) ^ 1u)) {
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
    umma_fence_before();
    __syncthreads();
    // After an error, wait (bounded) for every copy still in flight before the
    // CTA exits.
    if (flags[0] != 0 && tid == 0) {
        const int issued = flags[1];
        for (int it = max(0, issued - ntot); it < issued; ++it)
            (void)mbar_wait(&full[it % ntot], (uint32_t)(it / ntot) & 1u);
    }
    if (warp == kMmaWarp) {
        umma_fence_after();
        tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int MT, int AMODE, int EPI>
__global__ void __launch_bounds__(kStreamThreads, stream_min_blocks(MT, A_QUANT))
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
__global__ void __launch_bounds__(kStreamThreads, stream_min_blocks(MT, A_QUANT))
    stream_grouped_kernel(const __grid_constant__ CUtensorMap wmap, const StreamParams p,
                          const __grid_constant__ GroupTable gt) {
    const int g = (int)blockIdx.z / gt.zchunks;
    const int m0 = gt.off[g] + ((int)blockIdx.z - g * gt.zchunks) * MT;
    const int mvalid = min(MT, gt.off[g + 1] - m0);
    if (mvalid <= 0) return;
    stream_gemm_body<MT, AMODE, EPI>(wmap, p, m0, mvalid, g * gt.wrows, g * (gt.wrows / kBlock));
}

}  // namespace r9q
