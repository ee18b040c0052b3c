// Tensor-core (tcgen05 / TMEM / TMA) decode attention over the latent cache.
#pragma once
#include "mla_internal.cuh"

namespace mla {

constexpr int kTcTileN = 64;  // tokens per KV tile of the tensor-core kernel

// True when the dims match the tensor-core kernel (n_h = 128, d_c = 512,
// d_rope = 64, bf16 activations, bf16 or fp8 cache) and the device is sm_103.
bool tc_decode_supported(const mla_dims_t& d);

// Clusters of the decode kernel that can be resident at once on the current
// device (one worker each): the default split count, so that no worker waits
// for a second wave.
int tc_decode_max_workers();

cudaError_t launch_tc_decode(const mla_dims_t& d, const mla_cache_t& c, int B, int q_per_seq,
                             const __nv_bfloat16* q_abs, const int32_t* bt, int max_pages,
                             const int32_t* plan, int workers, float* o_part, float* lse_part,
                             __nv_bfloat16* o_lat, float* lse, int32_t* status, cudaStream_t st);

}  // namespace mla
