// tc_gemm_f16.cu -- instantiations of the tensor-core kernel for fp16 inputs, fp16 output
// (TMA producer with one CTA per tile or a cta_group::2 pair, and the
// load-based producer).  Split per input type so the build compiles the
// instantiations in parallel.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_f16(bool pair, Producer prod, const TcLaunch& L) {
    return tc_launch_impl<InKind::F16, __half>(pair, prod, L);
}

TcGeometry tc_geometry_f16(bool pair, bool half) {
    return tc_geometry_impl<InKind::F16>(pair, half);
}

}  // namespace gb300
