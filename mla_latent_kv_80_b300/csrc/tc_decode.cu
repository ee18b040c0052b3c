// Tensor-core decode attention (placeholder until the tcgen05 kernel lands).
#include "tc_decode.cuh"

namespace mla {

bool tc_decode_supported(const mla_dims_t&) { return false; }

cudaError_t launch_tc_decode(const mla_dims_t&, const mla_cache_t&, int, int,
                             const __nv_bfloat16*, const int32_t*, int, const int32_t*, int,
                             float*, float*, __nv_bfloat16*, float*, int32_t*, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace mla
