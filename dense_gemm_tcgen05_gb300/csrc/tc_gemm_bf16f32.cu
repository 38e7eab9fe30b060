// tc_gemm_bf16f32.cu -- instantiations of the tensor-core kernel for bf16 inputs with an
// fp32 output, the GEMM of the tensor-core FP32 path (gemm_f32_bf16x6).  A
// translation unit of its own, so that the build compiles it in parallel and
// the bf16-output kernels are untouched by it.
#include "tc_gemm.cuh"

namespace gb300 {

cudaError_t tc_launch_bf16_f32(bool pair, Producer prod, const TcLaunch& L) {
    return tc_launch_impl<InKind::BF16, float>(pair, prod, L);
}

}  // namespace gb300
