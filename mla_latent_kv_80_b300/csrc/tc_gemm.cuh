// Tensor-core skinny GEMMs of the decode step (append, absorb, out-proj, W_O).
#pragma once
#include "mla_internal.cuh"

#include <cuda.h>

namespace mla {

// 2-D bf16 tensor map with the 128-byte swizzle: rows of `row_elems` elements,
// `inner` of them addressed, boxes of 64 elements x box_rows rows.
bool tc_map2d_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t row_elems,
                   uint32_t box_rows);

// bf16 activations and tile-friendly dims (d_c % 128, d_h % 64, d_model % 64, d_v = 128) on sm_103.
bool tc_gemm_supported(const mla_dims_t& d);
// K splits of the append GEMM for T tokens (its workspace holds ksplit * T * (d_c + d_rope) fp32).
int tc_append_ksplit(const mla_dims_t& d, int T);

cudaError_t launch_tc_append_gemm(const mla_dims_t& d, int T, const __nv_bfloat16* h,
                                  const __nv_bfloat16* w_dkv, const __nv_bfloat16* w_kr, float* ws,
                                  int ksplit, int32_t* status, cudaStream_t st);
cudaError_t launch_tc_absorb(const mla_dims_t& d, int T, const __nv_bfloat16* q, const int32_t* pos,
                             const __nv_bfloat16* w_uk, __nv_bfloat16* q_abs, cudaStream_t st);
cudaError_t launch_tc_out_proj(const mla_dims_t& d, int T, const __nv_bfloat16* o_lat,
                               const __nv_bfloat16* w_uv, __nv_bfloat16* o, cudaStream_t st);
// K splits of the W_O GEMM for T tokens (its workspace holds ksplit * T * d_model fp32).
int tc_wo_ksplit(const mla_dims_t& d, int T);
// Split-K partial sums of out = W_O . o (o as [T][n_h * d_v]) into ws[ksplit][T][d_model].
cudaError_t launch_tc_wo_gemm(const mla_dims_t& d, int T, const __nv_bfloat16* o, const __nv_bfloat16* w_o,
                              float* ws, int ksplit, int32_t* status, cudaStream_t st);

}  // namespace mla
