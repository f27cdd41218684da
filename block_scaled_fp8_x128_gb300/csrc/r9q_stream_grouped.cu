// Grouped (several experts per launch) instantiations of the decode stream
// kernel: W8A8 with the fused activation quant, and weight-only.
#include "r9q_stream.cuh"

namespace r9q {

namespace {

template <int AMODE, int EPI>
using GroupedKernel = void (*)(const CUtensorMap, const StreamParams, const GroupTable);

template <int AMODE, int EPI>
GroupedKernel<AMODE, EPI> pick_grouped(int MT) {
    switch (MT) {
        case 8: return stream_grouped_kernel<8, AMODE, EPI>;
        case 16: return stream_grouped_kernel<16, AMODE, EPI>;
        case 32: return stream_grouped_kernel<32, AMODE, EPI>;
        case 64: return stream_grouped_kernel<64, AMODE, EPI>;
        default: return nullptr;
    }
}

}  // namespace

cudaError_t launch_stream_grouped(const StreamPlan& plan, int amode, int epi, const CUtensorMap& wmap,
                                  const StreamParams& p, const GroupTable& gt, int nexperts, cudaStream_t st,
                                  bool pdl) {
    void (*kern)(const CUtensorMap, const StreamParams, const GroupTable) = nullptr;
    if (amode == A_QUANT)
        kern = (epi == EPI_STORE) ? pick_grouped<A_QUANT, EPI_STORE>(plan.MT) : pick_grouped<A_QUANT, EPI_SWIGLU>(plan.MT);
    else if (amode == A_BF16)
        kern = (epi == EPI_STORE) ? pick_grouped<A_BF16, EPI_STORE>(plan.MT) : pick_grouped<A_BF16, EPI_SWIGLU>(plan.MT);
    if (!kern) return cudaErrorInvalidValue;
    cudaError_t e = ensure_dynamic_smem(reinterpret_cast<const void*>(kern), plan.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.splits, (unsigned)plan.groups, (unsigned)(nexperts * gt.zchunks));
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
    return cudaLaunchKernelEx(&cfg, kern, wmap, p, gt);
}

}  // namespace r9q
