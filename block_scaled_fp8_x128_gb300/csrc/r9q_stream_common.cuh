// Pieces shared by the two bodies of the decode-width stream GEMM
// (r9q_stream.cuh: tcgen05; r9q_stream_sync.cuh: mma.sync): cluster-scope
// barrier waits, the weight rows of a tile and the split-K slice ownership.
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

// Split-K slices (see stream_recv_rows): pair q of the tile's output columns
// belongs to rank q * S / NP (NP = 64 row pairs for the plain store, 32 pairs
// of h columns for SwiGLU); rank r's first pair is ceil(r * NP / S).
template <int EPI>
__device__ __forceinline__ int slice_pairs() { return EPI == EPI_SWIGLU ? 32 : 64; }
template <int EPI>
__device__ __forceinline__ int slice_first_pair(int r, int S) {
    return (r * slice_pairs<EPI>() + S - 1) / S;
}
// Owner rank of tile row j (0..127) and the row's index in the owner's receive
// area: plain store, rows 2*first .. in order; SwiGLU, gate rows (j < 64) of
// the owner's h columns first, then their up rows (index cap + c, where cap =
// 2 * ceil(32 / S) columns is the most a slice holds).
template <int EPI>
__device__ __forceinline__ void slice_of(int j, int S, int& owner, int& u) {
    if (EPI == EPI_SWIGLU) {
        const int c = j & 63;
        owner = (c >> 1) * S / 32;
        u = (j >> 6) * (2 * ((32 + S - 1) / S)) + c - 2 * slice_first_pair<EPI>(owner, S);
    } else {
        owner = (j >> 1) * S / 64;
        u = j - 2 * slice_first_pair<EPI>(owner, S);
    }
}

}  // namespace r9q
