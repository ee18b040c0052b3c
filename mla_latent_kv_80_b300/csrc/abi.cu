// C ABI of libmla: argument validation, workspace sizing and kernel dispatch.
#include "mla_internal.cuh"
#include "tc_decode.cuh"
#include "tc_gemm.cuh"
#include "tc_prefill.cuh"

#include <cmath>
#include <mutex>

namespace mla {

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 148;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 148;
  return n > 0 ? n : 148;
}

static bool valid_dims(const mla_dims_t* d) {
  if (d == nullptr) return false;
  if (d->n_h < 1 || d->d_h < 1 || d->d_v < 1 || d->d_c < 16 || d->d_rope < 0 || d->d_model < 8)
    return false;
  if (d->d_c > kMaxDc || d->d_c % 16 != 0) return false;
  if (d->d_rope > kMaxDrope || d->d_rope % 2 != 0) return false;
  if (d->d_h > kMaxDh || d->d_v > 512 || d->d_model % 8 != 0) return false;
  if (!(d->page_size == 16 || d->page_size == 32 || d->page_size == 64 || d->page_size == 128))
    return false;
  // The attention kernels take the maximum of the raw scores and scale it
  // afterwards, which is the maximum of the scaled scores only for a positive
  // scale; the RoPE frequencies theta^(-2i/d) need a positive base.
  if (!(d->softmax_scale > 0.f) || !std::isfinite(d->softmax_scale)) return false;
  if (!(d->rope_theta > 0.f) || !std::isfinite(d->rope_theta)) return false;
  return true;
}

static bool supported_types(const mla_dims_t* d) {
  if (d->act_dtype == MLA_F32) return d->cache_dtype == MLA_F32;
  if (d->act_dtype == MLA_BF16) return d->cache_dtype == MLA_BF16 || d->cache_dtype == MLA_FP8_E4M3;
  return false;
}

static int check_dims(const mla_dims_t* d) {
  if (!valid_dims(d)) return MLA_ERR_INVALID_ARG;
  if (!supported_types(d)) return MLA_ERR_UNSUPPORTED;
  return MLA_OK;
}

static int check_cache(const mla_dims_t* d, const mla_cache_t* c) {
  if (c == nullptr || c->ckv == nullptr || c->num_pages < 0) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(c->ckv) & 15) != 0) return MLA_ERR_INVALID_ARG;
  if (d->cache_dtype == MLA_FP8_E4M3) {
    if (c->kr == nullptr || c->scale == nullptr) return MLA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(c->kr) & 15) != 0) return MLA_ERR_INVALID_ARG;
  }
  return MLA_OK;
}

static int cuda_status(cudaError_t e) { return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA; }

// Worker count of the decode split (num_splits = 0 picks per path).
static int decode_workers(const mla_dims_t* d, int num_splits) {
  if (num_splits > 0) return num_splits;
  return tc_decode_supported(*d) ? tc_decode_max_workers() : sm_count();
}

struct DecodeWs {
  size_t plan_bytes, opart_bytes, lse_bytes, total;
  int max_partials;
};

static DecodeWs decode_ws_layout(const mla_dims_t* d, int B, int q, int workers) {
  DecodeWs w;
  const int P = B * q;
  w.max_partials = 2 * workers;
  w.plan_bytes = align256(plan_ints(P, workers) * sizeof(int32_t));
  w.opart_bytes = align256((size_t)w.max_partials * d->n_h * d->d_c * sizeof(float));
  w.lse_bytes = align256((size_t)w.max_partials * d->n_h * sizeof(float));
  w.total = w.plan_bytes + w.opart_bytes + w.lse_bytes;
  return w;
}

}  // namespace mla

using namespace mla;

extern "C" {

int mla_abi_version(void) { return MLA_ABI_VERSION; }

const char* mla_status_string(int s) {
  switch (s) {
    case MLA_OK: return "ok";
    case MLA_ERR_INVALID_ARG: return "invalid argument";
    case MLA_ERR_UNSUPPORTED: return "unsupported dimensions or dtypes";
    case MLA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MLA_ERR_CUDA: return "CUDA launch error";
    case MLA_ERR_BAD_PAGE: return "block-table entry outside the page pool";
    case MLA_ERR_DEVICE_TIMEOUT: return "bounded device wait gave up";
    case MLA_ERR_NO_DEVICE: return "no CUDA device";
    case MLA_ERR_NO_PAGES: return "page pool exhausted";
    default: return "unknown status";
  }
}

int mla_cache_append_workspace_size(const mla_dims_t* dims, int32_t T, size_t* bytes) {
  if (bytes == nullptr || T < 0) return MLA_ERR_INVALID_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  const int n_out = dims->d_c + dims->d_rope;
  const int ks = tc_gemm_supported(*dims) ? tc_append_ksplit(*dims, T)
                                          : append_ksplit(T, n_out, dims->d_model);
  *bytes = T == 0 ? 0 : align256((size_t)ks * T * n_out * sizeof(float));
  return MLA_OK;
}

int mla_cache_append(const mla_dims_t* dims, const mla_cache_t* cache, int32_t T, const void* h,
                     const void* w_dkv, const void* w_kr, const int32_t* seq_idx,
                     const int32_t* pos, const int32_t* block_table, int32_t max_pages_per_seq,
                     void* workspace, size_t workspace_bytes, int32_t* status,
                     mla_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (T < 0 || max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if ((rc = check_cache(dims, cache))) return rc;
  if (T == 0) return MLA_OK;
  if (!h || !w_dkv || !w_kr || !seq_idx || !pos || !block_table) return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_cache_append_workspace_size(dims, T, &need);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if (need > 0 && workspace == nullptr) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tc_gemm_supported(*dims)) {
    const int ks = tc_append_ksplit(*dims, T);
    e = launch_tc_append_gemm(*dims, T, (const __nv_bfloat16*)h, (const __nv_bfloat16*)w_dkv,
                              (const __nv_bfloat16*)w_kr, (float*)workspace, ks, status, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    return cuda_status(launch_append_epilogue<__nv_bfloat16>(*dims, *cache, T, seq_idx, pos,
                                                             block_table, max_pages_per_seq,
                                                             (const float*)workspace, ks, status, st));
  }
  const int ks = append_ksplit(T, dims->d_c + dims->d_rope, dims->d_model);
  if (dims->act_dtype == MLA_F32)
    e = launch_append_simt<float>(*dims, *cache, T, (const float*)h, (const float*)w_dkv,
                                  (const float*)w_kr, seq_idx, pos, block_table,
                                  max_pages_per_seq, (float*)workspace, ks, status, st);
  else
    e = launch_append_simt<__nv_bfloat16>(*dims, *cache, T, (const __nv_bfloat16*)h,
                                          (const __nv_bfloat16*)w_dkv, (const __nv_bfloat16*)w_kr,
                                          seq_idx, pos, block_table, max_pages_per_seq,
                                          (float*)workspace, ks, status, st);
  return cuda_status(e);
}

int mla_absorb_q(const mla_dims_t* dims, int32_t T, const void* q, const int32_t* pos,
                 const void* w_uk, void* q_abs, mla_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!q || !pos || !w_uk || !q_abs) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tc_gemm_supported(*dims))
    e = launch_tc_absorb(*dims, T, (const __nv_bfloat16*)q, pos, (const __nv_bfloat16*)w_uk,
                         (__nv_bfloat16*)q_abs, st);
  else if (dims->act_dtype == MLA_F32)
    e = launch_absorb_simt<float>(*dims, T, (const float*)q, pos, (const float*)w_uk,
                                  (float*)q_abs, st);
  else
    e = launch_absorb_simt<__nv_bfloat16>(*dims, T, (const __nv_bfloat16*)q, pos,
                                          (const __nv_bfloat16*)w_uk, (__nv_bfloat16*)q_abs, st);
  return cuda_status(e);
}

int mla_decode_default_splits(const mla_dims_t* dims, int32_t* splits) {
  if (splits == nullptr) return MLA_ERR_INVALID_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  *splits = decode_workers(dims, 0);
  return MLA_OK;
}

int mla_decode_workspace_size(const mla_dims_t* dims, int32_t B, int32_t q_per_seq,
                              int32_t num_splits, size_t* bytes) {
  if (bytes == nullptr || B < 0 || q_per_seq < 1 || num_splits < 0) return MLA_ERR_INVALID_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  *bytes = decode_ws_layout(dims, B, q_per_seq, decode_workers(dims, num_splits)).total;
  return MLA_OK;
}

int mla_decode_attn(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                    int32_t q_per_seq, const void* q_abs, const int32_t* block_table,
                    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t num_splits,
                    void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                    int32_t* status, mla_stream_t stream) {
  return mla_decode_attn_window(dims, cache, B, q_per_seq, q_abs, block_table, max_pages_per_seq, seq_lens,
                                nullptr, num_splits, workspace, workspace_bytes, o_lat, lse, status, stream);
}

int mla_decode_attn_window(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B, int32_t q_per_seq,
                           const void* q_abs, const int32_t* block_table, int32_t max_pages_per_seq,
                           const int32_t* seq_lens, const int32_t* seq_start, int32_t num_splits,
                           void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                           int32_t* status, mla_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (B < 0 || q_per_seq < 1 || num_splits < 0 || max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if ((rc = check_cache(dims, cache))) return rc;
  if (B == 0) return MLA_OK;
  if (!q_abs || !block_table || !seq_lens || !o_lat || !lse || !workspace)
    return MLA_ERR_INVALID_ARG;
  const int workers = decode_workers(dims, num_splits);
  const DecodeWs L = decode_ws_layout(dims, B, q_per_seq, workers);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  char* ws = static_cast<char*>(workspace);
  int32_t* plan = reinterpret_cast<int32_t*>(ws);
  float* o_part = reinterpret_cast<float*>(ws + L.plan_bytes);
  float* lse_part = reinterpret_cast<float*>(ws + L.plan_bytes + L.opart_bytes);
  const bool tc = tc_decode_supported(*dims);
  // The tensor-core kernel pays about four tiles' time to start on a problem
  // (Q slice load, pipeline fill, epilogue); the SIMT kernel's start is cheap.
  cudaError_t e = launch_plan(B, q_per_seq, seq_lens, seq_start, tc ? kTcTileN : 32, tc ? 4 : 0, workers, plan, st);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  if (tc) {
    e = launch_tc_decode(*dims, *cache, B, q_per_seq, (const __nv_bfloat16*)q_abs, block_table,
                         max_pages_per_seq, plan, workers, o_part, lse_part,
                         (__nv_bfloat16*)o_lat, lse, status, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_combine<__nv_bfloat16>(*dims, B * q_per_seq, plan, o_part, lse_part,
                                      (__nv_bfloat16*)o_lat, lse, st, /*blocked=*/true, workers);
  } else if (dims->act_dtype == MLA_F32) {
    e = launch_decode_simt<float>(*dims, *cache, B, q_per_seq, (const float*)q_abs, block_table,
                                  max_pages_per_seq, plan, workers, o_part, lse_part,
                                  (float*)o_lat, lse, status, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_combine<float>(*dims, B * q_per_seq, plan, o_part, lse_part, (float*)o_lat, lse, st);
  } else {
    e = launch_decode_simt<__nv_bfloat16>(*dims, *cache, B, q_per_seq,
                                          (const __nv_bfloat16*)q_abs, block_table,
                                          max_pages_per_seq, plan, workers, o_part, lse_part,
                                          (__nv_bfloat16*)o_lat, lse, status, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_combine<__nv_bfloat16>(*dims, B * q_per_seq, plan, o_part, lse_part,
                                      (__nv_bfloat16*)o_lat, lse, st);
  }
  return cuda_status(e);
}

int mla_prefill_form(const mla_dims_t* dims, int32_t q_per_seq, int64_t seq_len, int32_t* explicit_form) {
  if (explicit_form == nullptr || q_per_seq < 1 || seq_len < 0) return MLA_ERR_INVALID_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  *explicit_form =
      prefill_flops_explicit(*dims, q_per_seq, seq_len) < prefill_flops_absorbed(*dims, q_per_seq, seq_len) ? 1 : 0;
  return MLA_OK;
}

int mla_prefill_workspace_size(const mla_dims_t* dims, int32_t B, int32_t q_per_seq, int32_t max_seq_len,
                               size_t* bytes) {
  if (bytes == nullptr || B < 0 || q_per_seq < 1 || max_seq_len < 0) return MLA_ERR_INVALID_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  *bytes = prefill_ws_layout(*dims, B, q_per_seq, max_seq_len).total;
  return MLA_OK;
}

int mla_prefill_attn(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B, int32_t q_per_seq,
                     int32_t max_seq_len, const void* q, const void* w_uk, const void* w_uv,
                     const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                     void* workspace, size_t workspace_bytes, void* o, float* lse, int32_t* status,
                     mla_stream_t stream) {
  return mla_prefill_attn_window(dims, cache, B, q_per_seq, max_seq_len, q, w_uk, w_uv, block_table,
                                 max_pages_per_seq, seq_lens, nullptr, workspace, workspace_bytes, o, lse, status,
                                 stream);
}

int mla_prefill_attn_window(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B, int32_t q_per_seq,
                            int32_t max_seq_len, const void* q, const void* w_uk, const void* w_uv,
                            const int32_t* block_table, int32_t max_pages_per_seq, const int32_t* seq_lens,
                            const int32_t* seq_start, void* workspace, size_t workspace_bytes, void* o, float* lse,
                            int32_t* status, mla_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (B < 0 || q_per_seq < 1 || max_seq_len < 0 || max_pages_per_seq < 1) return MLA_ERR_INVALID_ARG;
  if ((rc = check_cache(dims, cache))) return rc;
  if (!tc_prefill_supported(*dims)) return MLA_ERR_UNSUPPORTED;
  if (B == 0) return MLA_OK;
  if (!q || !w_uk || !w_uv || !block_table || !seq_lens || !workspace || !o || !lse || !status)
    return MLA_ERR_INVALID_ARG;
  // Vector loads and stores of q and o, tensor maps over the workspace and weights.
  auto misaligned = [](const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) != 0; };
  if (misaligned(q, 16) || misaligned(o, 16) || misaligned(w_uk, 16) || misaligned(w_uv, 16) ||
      misaligned(workspace, 256))
    return MLA_ERR_INVALID_ARG;
  const PrefillWs L = prefill_ws_layout(*dims, B, q_per_seq, max_seq_len);
  // Tensor-map row coordinates are 32-bit; sequences and heads index the
  // attention kernel's grid (z and y, at most 65535 each).
  if ((int64_t)B * L.l_pad >= (int64_t)1 << 31 || (int64_t)B * q_per_seq * dims->n_h >= (int64_t)1 << 31 ||
      B > 65535 || dims->n_h > 65535)
    return MLA_ERR_INVALID_ARG;
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE_TOO_SMALL;
  cudaError_t e = launch_prefill(*dims, *cache, B, q_per_seq, max_seq_len, (const __nv_bfloat16*)q,
                                 (const __nv_bfloat16*)w_uk, (const __nv_bfloat16*)w_uv, block_table,
                                 max_pages_per_seq, seq_lens, seq_start, workspace, (__nv_bfloat16*)o, lse, status,
                                 reinterpret_cast<cudaStream_t>(stream));
  return cuda_status(e);
}

int mla_out_proj(const mla_dims_t* dims, int32_t T, const void* o_lat, const void* w_uv, void* o,
                 mla_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!o_lat || !w_uv || !o) return MLA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (tc_gemm_supported(*dims))
    e = launch_tc_out_proj(*dims, T, (const __nv_bfloat16*)o_lat, (const __nv_bfloat16*)w_uv,
                           (__nv_bfloat16*)o, st);
  else if (dims->act_dtype == MLA_F32)
    e = launch_out_proj_simt<float>(*dims, T, (const float*)o_lat, (const float*)w_uv, (float*)o, st);
  else
    e = launch_out_proj_simt<__nv_bfloat16>(*dims, T, (const __nv_bfloat16*)o_lat,
                                            (const __nv_bfloat16*)w_uv, (__nv_bfloat16*)o, st);
  return cuda_status(e);
}

int mla_out_proj_wo_workspace_size(const mla_dims_t* dims, int32_t T, size_t* bytes) {
  if (bytes == nullptr || T < 0) return MLA_ERR_INVALID_ARG;
  int rc = check_dims(dims);
  if (rc) return rc;
  const int ks = tc_gemm_supported(*dims) ? tc_wo_ksplit(*dims, T) : wo_ksplit_simt(*dims, T);
  *bytes = T == 0 ? 0 : align256((size_t)ks * T * dims->d_model * sizeof(float));
  return MLA_OK;
}

int mla_out_proj_wo(const mla_dims_t* dims, int32_t T, const void* o_lat, const void* w_uv, const void* w_o,
                    void* o, void* out, void* workspace, size_t workspace_bytes, int32_t* status,
                    mla_stream_t stream) {
  int rc = check_dims(dims);
  if (rc) return rc;
  if (T < 0) return MLA_ERR_INVALID_ARG;
  if (T == 0) return MLA_OK;
  if (!o_lat || !w_uv || !w_o || !o || !out || !workspace) return MLA_ERR_INVALID_ARG;
  size_t need = 0;
  mla_out_proj_wo_workspace_size(dims, T, &need);
  if (workspace_bytes < need) return MLA_ERR_WORKSPACE_TOO_SMALL;
  if ((rc = mla_out_proj(dims, T, o_lat, w_uv, o, stream)) != MLA_OK) return rc;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  float* ws = static_cast<float*>(workspace);
  cudaError_t e;
  if (tc_gemm_supported(*dims)) {
    const int ks = tc_wo_ksplit(*dims, T);
    e = launch_tc_wo_gemm(*dims, T, (const __nv_bfloat16*)o, (const __nv_bfloat16*)w_o, ws, ks, status, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_reduce_splits<__nv_bfloat16>(T, dims->d_model, ks, ws, (__nv_bfloat16*)out, st);
  } else if (dims->act_dtype == MLA_F32) {
    const int ks = wo_ksplit_simt(*dims, T);
    e = launch_wo_gemm_simt<float>(*dims, T, (const float*)o, (const float*)w_o, ws, ks, st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_reduce_splits<float>(T, dims->d_model, ks, ws, (float*)out, st);
  } else {
    const int ks = wo_ksplit_simt(*dims, T);
    e = launch_wo_gemm_simt<__nv_bfloat16>(*dims, T, (const __nv_bfloat16*)o, (const __nv_bfloat16*)w_o, ws, ks,
                                           st);
    if (e != cudaSuccess) return MLA_ERR_CUDA;
    e = launch_reduce_splits<__nv_bfloat16>(T, dims->d_model, ks, ws, (__nv_bfloat16*)out, st);
  }
  return cuda_status(e);
}

int mla_quantize_fp8_rows(const float* x, int32_t rows, int32_t cols, uint8_t* codes,
                          float* scales, mla_stream_t stream) {
  if (rows < 0 || cols < 1 || cols > 4096) return MLA_ERR_INVALID_ARG;
  if (rows == 0) return MLA_OK;
  if (!x || !codes || !scales) return MLA_ERR_INVALID_ARG;
  return cuda_status(launch_quantize_rows(x, rows, cols, codes, scales,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"
