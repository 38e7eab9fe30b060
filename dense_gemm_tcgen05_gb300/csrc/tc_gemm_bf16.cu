// tc_gemm_bf16.cu -- instantiations of the tensor-core kernel for bf16 inputs, bf16 output
// (one CTA per tile and the cta_group::2 pair).  Split per input type so the
// build compiles the instantiations in parallel.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_bf16(bool pair, const TcLaunch& L) {
    return pair ? tc_launch_impl<InKind::BF16, __nv_bfloat16, true>(L)
                : tc_launch_impl<InKind::BF16, __nv_bfloat16, false>(L);
}

TcGeometry tc_geometry_bf16(bool pair) {
    return pair ? tc_geometry_impl<InKind::BF16, true>() : tc_geometry_impl<InKind::BF16, false>();
}

}  // namespace gb300
