// tc_gemm_mc.cu -- instantiations of the cluster-of-two-pairs tensor-core
// kernel (tc_gemm_mc.cuh) for every input type and output type.
#include "launch.h"
#include "tc_gemm_mc.cuh"

namespace gb300 {

cudaError_t tc_mc_launch(InKind in, bool out_f32, const TcLaunch& L) {
    switch (in) {
        case InKind::F16: return tc_mc_launch_impl<InKind::F16, __half>(L);
        case InKind::BF16: return tc_mc_launch_impl<InKind::BF16, __nv_bfloat16>(L);
        default:
            return out_f32 ? tc_mc_launch_impl<InKind::E4M3, float>(L)
                           : tc_mc_launch_impl<InKind::E4M3, __nv_bfloat16>(L);
    }
}

cudaError_t tc_mc_max_clusters(InKind in, bool out_f32, int* n) {
    switch (in) {
        case InKind::F16: return tc_mc_max_clusters_impl<InKind::F16, __half>(n);
        case InKind::BF16: return tc_mc_max_clusters_impl<InKind::BF16, __nv_bfloat16>(n);
        default:
            return out_f32 ? tc_mc_max_clusters_impl<InKind::E4M3, float>(n)
                           : tc_mc_max_clusters_impl<InKind::E4M3, __nv_bfloat16>(n);
    }
}

}  // namespace gb300
