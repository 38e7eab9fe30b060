// tc_gemm_fp8.cu -- instantiations of the tensor-core kernel for e4m3 inputs with a
// bf16 or an fp32 output
// (TMA producer with one CTA per tile or a cta_group::2 pair, and the
// load-based producer).  Split per input type so the build compiles the
// instantiations in parallel.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_fp8(bool pair, Producer prod, bool out_f32, const TcLaunch& L) {
    return out_f32 ? tc_launch_impl<InKind::E4M3, float>(pair, prod, L)
                   : tc_launch_impl<InKind::E4M3, __nv_bfloat16>(pair, prod, L);
}

TcGeometry tc_geometry_fp8(bool pair, bool half) {
    return tc_geometry_impl<InKind::E4M3>(pair, half);
}

}  // namespace gb300
