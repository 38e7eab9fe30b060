// tc_gemm_f16.cu -- instantiations of the tensor-core kernel for fp16 inputs, fp16 output
// (one CTA per tile and the cta_group::2 pair).  Split per input type so the
// build compiles the instantiations in parallel.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_f16(bool pair, const TcLaunch& L) {
    return pair ? tc_launch_impl<InKind::F16, __half, true>(L)
                : tc_launch_impl<InKind::F16, __half, false>(L);
}

TcGeometry tc_geometry_f16(bool pair) {
    return pair ? tc_geometry_impl<InKind::F16, true>() : tc_geometry_impl<InKind::F16, false>();
}

}  // namespace gb300
