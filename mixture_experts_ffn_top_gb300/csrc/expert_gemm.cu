// expert_gemm.cu -- tensor-core grouped expert GEMM (placeholder until the
// tcgen05 kernels land: the tensor path reports itself unavailable).
#include "moe_internal.cuh"

namespace moe {

bool tensor_path_supported(const moe_weights_s *) { return false; }
int prepare_tensor_maps(moe_weights_s *) { return MOE_OK; }
int launch_plan_and_gather(const moe_weights_s *, const int8_t *, const float *, const int32_t *, const int32_t *,
                           const int32_t *, int, int, bool, void *, const WsLayout &, cudaStream_t) {
    return MOE_ERR_UNSUPPORTED_SHAPE;
}
int launch_gemm_gate_up(const moe_weights_s *, int, int, bool, void *, const WsLayout &, int32_t *, int,
                        cudaStream_t) {
    return MOE_ERR_UNSUPPORTED_SHAPE;
}
int launch_gemm_down(const moe_weights_s *, int, int, bool, const float *, float *, float *, void *,
                     const WsLayout &, cudaStream_t) {
    return MOE_ERR_UNSUPPORTED_SHAPE;
}
int launch_h16_to_q8(const moe_weights_s *, int, int, void *, const WsLayout &, int8_t *, float *, cudaStream_t) {
    return MOE_ERR_UNSUPPORTED_SHAPE;
}
int launch_q8_to_h16(const moe_weights_s *, int, int, void *, const WsLayout &, const int8_t *, const float *,
                     cudaStream_t) {
    return MOE_ERR_UNSUPPORTED_SHAPE;
}

}  // namespace moe
