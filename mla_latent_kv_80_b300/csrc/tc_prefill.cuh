// Chunked prefill in the explicit form: gather the latent rows, form each
// head's keys and values with a tensor-core GEMM, and attend causally with a
// tcgen05 flash-attention kernel.
#pragma once
#include "mla_internal.cuh"

namespace mla {

// bf16 activations, d_h = d_v = 128, d_rope = 64, d_c % 64 == 0, bf16 or fp8
// cache, sm_103 device.
bool tc_prefill_supported(const mla_dims_t& d);

struct PrefillWs {
  int l_pad;               // rows per sequence in the gathered / formed buffers (multiple of 128)
  size_t lat_off, k_off, v_off, rope_off, total;
};
PrefillWs prefill_ws_layout(const mla_dims_t& d, int B, int C, int max_seq_len);

// Flops of the explicit and absorbed forms for C queries at the end of a
// sequence of L tokens (the cost model of mla_prefill_form).
double prefill_flops_explicit(const mla_dims_t& d, int C, int64_t L);
double prefill_flops_absorbed(const mla_dims_t& d, int C, int64_t L);

cudaError_t launch_prefill(const mla_dims_t& d, const mla_cache_t& c, int B, int C, int max_seq_len,
                           const __nv_bfloat16* q, const __nv_bfloat16* w_uk, const __nv_bfloat16* w_uv,
                           const int32_t* bt, int max_pages, const int32_t* seq_lens, const int32_t* seq_start,
                           void* ws, __nv_bfloat16* o, float* lse, int32_t* status, cudaStream_t st);

}  // namespace mla
