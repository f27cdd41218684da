// Grouped (several experts per launch) instantiations of the decode stream
// kernel: W8A8 with the fused activation quant, and weight-only.
#include "r9q_stream_launch.cuh"

namespace r9q {

cudaError_t launch_stream_grouped(const StreamPlan& plan, int amode, int epi, const CUtensorMap& wmap,
                                  const StreamParams& p, const GroupTable& gt, int nexperts, cudaStream_t st,
                                  bool pdl) {
    const unsigned nz = (unsigned)(nexperts * gt.zchunks);
    if (amode == A_QUANT)
        return epi == EPI_STORE
            ? launch_stream_clusters(pick_stream_grouped<A_QUANT, EPI_STORE>(plan.MT), plan, A_QUANT, nz, st, pdl, wmap, p, gt)
            : launch_stream_clusters(pick_stream_grouped<A_QUANT, EPI_SWIGLU>(plan.MT), plan, A_QUANT, nz, st, pdl, wmap, p, gt);
    if (amode == A_BF16)
        return epi == EPI_STORE
            ? launch_stream_clusters(pick_stream_grouped<A_BF16, EPI_STORE>(plan.MT), plan, A_BF16, nz, st, pdl, wmap, p, gt)
            : launch_stream_clusters(pick_stream_grouped<A_BF16, EPI_SWIGLU>(plan.MT), plan, A_BF16, nz, st, pdl, wmap, p, gt);
    return cudaErrorInvalidValue;
}

}  // namespace r9q
