// tc_gemm_fp8.cu -- instantiations of the tensor-core kernel for e4m3 inputs, bf16 output
// (one CTA per tile and the cta_group::2 pair).  Split per input type so the
// build compiles the instantiations in parallel.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_fp8(bool pair, const TcLaunch& L) {
    return pair ? tc_launch_impl<InKind::E4M3, __nv_bfloat16, true>(L)
                : tc_launch_impl<InKind::E4M3, __nv_bfloat16, false>(L);
}

TcGeometry tc_geometry_fp8(bool pair) {
    return pair ? tc_geometry_impl<InKind::E4M3, true>() : tc_geometry_impl<InKind::E4M3, false>();
}

}  // namespace gb300
