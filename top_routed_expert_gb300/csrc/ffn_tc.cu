// Tensor-core (tcgen05) grouped expert FFN -- placeholder until implemented.
#include "common.cuh"

namespace moe {

bool ffn_tc_supported(const moe_config_t&) { return false; }
size_t ffn_tc_ws_bytes(const moe_config_t&) { return 0; }
cudaError_t launch_ffn_tc(const moe_config_t&, const void*, const float*, const int32_t*, const int32_t*,
                          const moe_weights_t*, float*, float*, void*, unsigned*, int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace moe
