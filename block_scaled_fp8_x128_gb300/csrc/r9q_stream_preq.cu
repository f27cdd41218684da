// Instantiations of the decode-width stream GEMM for the A_PREQ A-load
// (one translation unit per A-load mode so the library builds in parallel).
#include "r9q_stream_launch.cuh"

namespace r9q {

cudaError_t launch_stream_a_preq(const StreamPlan& plan, int epi, const CUtensorMap& wmap,
                              const StreamParams& p, cudaStream_t st, bool pdl) {
    return launch_stream_impl<A_PREQ>(plan, epi, wmap, p, st, pdl);
}

}  // namespace r9q
