// tc_gemm_bf16.cu -- instantiations of the tensor-core kernel for bf16 inputs, bf16 output
// (TMA producer with one CTA per tile or a cta_group::2 pair, and the
// load-based producer).  Split per input type so the build compiles the
// instantiations in parallel.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_bf16(bool pair, Producer prod, const TcLaunch& L) {
    return tc_launch_impl<InKind::BF16, __nv_bfloat16>(pair, prod, L);
}

TcGeometry tc_geometry_bf16(bool pair, bool half) {
    return tc_geometry_impl<InKind::BF16>(pair, half);
}

}  // namespace gb300
