// Launch side of the decode-width stream GEMM: picks the body for the token
// tile (stream_uses_tc: tcgen05 or mma.sync) and launches it as clusters of
// S CTAs along K, with programmatic dependent launch when asked.
#pragma once

#include "r9q_stream.cuh"
#include "r9q_stream_sync.cuh"

namespace r9q {

template <int AMODE, int EPI>
using StreamKernel = void (*)(const CUtensorMap, const StreamParams);
template <int AMODE, int EPI>
using StreamGroupedKernel = void (*)(const CUtensorMap, const StreamParams, const GroupTable);

// The body's kernel for a token tile (only the chosen one is instantiated).
template <int MT, int AMODE, int EPI>
StreamKernel<AMODE, EPI> stream_kernel_for() {
    if constexpr (stream_uses_tc(MT, AMODE)) return stream_gemm_kernel<MT, AMODE, EPI>;
    else return stream_sync_kernel<MT, AMODE, EPI>;
}
template <int MT, int AMODE, int EPI>
StreamGroupedKernel<AMODE, EPI> stream_grouped_kernel_for() {
    if constexpr (stream_uses_tc(MT, AMODE)) return stream_grouped_kernel<MT, AMODE, EPI>;
    else return stream_sync_grouped_kernel<MT, AMODE, EPI>;
}

template <int AMODE, int EPI>
StreamKernel<AMODE, EPI> pick_stream(int MT) {
    switch (MT) {
        case 8: return stream_kernel_for<8, AMODE, EPI>();
        case 16: return stream_kernel_for<16, AMODE, EPI>();
        case 32: return stream_kernel_for<32, AMODE, EPI>();
        case 64: return stream_kernel_for<64, AMODE, EPI>();
        default: return nullptr;
    }
}

template <int AMODE, int EPI>
StreamGroupedKernel<AMODE, EPI> pick_stream_grouped(int MT) {
    switch (MT) {
        case 8: return stream_grouped_kernel_for<8, AMODE, EPI>();
        case 16: return stream_grouped_kernel_for<16, AMODE, EPI>();
        case 32: return stream_grouped_kernel_for<32, AMODE, EPI>();
        case 64: return stream_grouped_kernel_for<64, AMODE, EPI>();
        default: return nullptr;
    }
}

// Cluster launch of S CTAs along K; `nz` token chunks (times experts) in z.
template <typename Kernel, typename... Args>
cudaError_t launch_stream_clusters(Kernel kern, const StreamPlan& plan, int amode, unsigned nz, cudaStream_t st,
                                   bool pdl, Args... args) {
    if (!kern) return cudaErrorInvalidValue;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), plan.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.splits, (unsigned)plan.groups, nz);
    cfg.blockDim = dim3((unsigned)stream_threads(plan.MT, amode), 1, 1);
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
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

template <int AMODE>
cudaError_t launch_stream_impl(const StreamPlan& plan, int epi, const CUtensorMap& wmap,
                               const StreamParams& p, cudaStream_t st, bool pdl) {
    if (epi == EPI_STORE)
        return launch_stream_clusters(pick_stream<AMODE, EPI_STORE>(plan.MT), plan, AMODE, (unsigned)plan.mchunks, st,
                                      pdl, wmap, p);
    if (AMODE == A_PREQ) return cudaErrorInvalidValue;
    return launch_stream_clusters(pick_stream<AMODE, EPI_SWIGLU>(plan.MT), plan, AMODE, (unsigned)plan.mchunks, st, pdl,
                                  wmap, p);
}

}  // namespace r9q
