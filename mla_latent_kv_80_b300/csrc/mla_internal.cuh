// Internal declarations shared by the libmla translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>
#include <utility>

#include "../../include/mla.h"

namespace mla {

constexpr int kMaxDc = 512;
constexpr int kMaxDrope = 64;
constexpr int kMaxDh = 512;

enum class CacheKind { F32 = 0, BF16 = 1, FP8 = 2 };

// ------------------------------------------------------------------ scalar helpers
__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

template <typename T> __device__ __forceinline__ T from_f32(float x);
template <> __device__ __forceinline__ float from_f32<float>(float x) { return x; }
template <> __device__ __forceinline__ __nv_bfloat16 from_f32<__nv_bfloat16>(float x) {
  return __float2bfloat16_rn(x);
}

// Programmatic dependent launch. Every kernel of the library is launched with
// programmatic stream serialization (launch_pdl below): it signals at its start
// that the next kernel may be scheduled, does its set-up, and waits for the
// previous kernel's completion (and memory) before touching anything written
// in the stream. The next kernel can only start once every block of this one
// has started, so the early signal cannot starve this kernel of SMs; every
// kernel waits on all paths, so completion stays transitive along the stream.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ void set_status(int32_t* status, int code) {
  if (status != nullptr) atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

// RoPE inverse frequencies theta^(-2i/d_rope) for the pairs i < d_rope/2,
// computed once on the host in double and passed to kernels by value as a
// float pair hi + lo, so that the angle keeps its low bits in single precision.
struct RopeFreqs {
  float hi[kMaxDrope / 2];
  float lo[kMaxDrope / 2];
};
RopeFreqs rope_freqs(int d_rope, float theta);

// cos/sin of the angle pos * (hi + lo), all in single precision. The product
// is carried as p + e with e = fma(pos, hi, -p) (exact) plus pos * lo; it is
// reduced by k = round(p / 2 pi) with 2 pi split into three parts (Cody-Waite):
// 6 (k * 6 is exact for |k| < 2^21), then the fp32 value of 2 pi - 6, then the
// remainder. The reduced angle is within about 4e-7 rad of the exact one for
// |pos| < 2^23; its sine and cosine come from the special-function unit, whose
// absolute error on [-pi, pi] is about 2^-21.
__device__ __forceinline__ void rope_cos_sin(int pos, float hi, float lo, float* c, float* s) {
  const float kTwoPiMid = 0x1.21fb54p-2f;   // fp32(2 pi - 6)
  const float kTwoPiLow = 0x1.10b462p-28f;  // 2 pi - 6 - kTwoPiMid
  const float x = (float)pos;               // exact for |pos| < 2^24
  const float p = x * hi;
  const float e = fmaf(x, hi, -p) + x * lo;
  const float k = rintf(p * 0.159154943091895335768883763372514362f);
  float r = fmaf(-k, 6.0f, p);
  r = fmaf(-k, kTwoPiMid, r);
  r = fmaf(-k, kTwoPiLow, r);
  __sincosf(r + e, s, c);
}

// E4M3 with saturation, round to nearest even (CUDA conversion intrinsic).
__device__ __forceinline__ uint8_t f32_to_e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_f32(uint8_t code) {
  __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)code, __NV_E4M3);
  return __half2float(__half(hr));
}

// Per-token scale of the fp8 cache recipe: amax/448, 1 when amax = 0, at least FLT_MIN.
__device__ __forceinline__ float e4m3_row_scale(float amax) {
  if (amax == 0.0f) return 1.0f;
  float s = amax / 448.0f;
  return s < 1.17549435e-38f ? 1.17549435e-38f : s;
}

// ------------------------------------------------------------------ decode plan
// Device-built split plan, stored at the start of the decode workspace.
// Problem p = b * q + j sees the keys at positions [lo_p, len_p): len_p is
// seq_lens[b] - q + j + 1 and lo_p the sequence's first visible position (0
// unless a window start is given), clamped to [0, len_p]. Its tiles are the
// tile_n-wide key blocks that meet that range, from block tf_p = lo_p / tile_n
// on. The tiles of all problems, in problem order, are cut into G contiguous
// worker ranges of equal cost, where a range costs its tiles plus `seg_cost`
// for each problem it touches (the fixed cost of starting on a problem), so
// that a worker whose range spans two problems gets fewer tiles. Layout (int32):
//   hdr[0] problems P (= B * q_per_seq), hdr[1] total tiles, hdr[2] seg_cost,
//   hdr[3] workers G; cum[P+1] (tile prefix sums), pbase[P+1] (prefix sums of
//   partial slots of the problems cut between workers), len[P] (len_p),
//   first[G] (the problem holding each worker's first tile, P for none),
//   wstart[G+1] (each worker's first tile; its range ends at the next worker's
//   start), pw0[P] (the first worker of each problem), pcnt[P] (workers per
//   problem), vcum[P+1] (prefix sums of tiles plus start costs), lo[P] (lo_p)
//   and tf[P] (tf_p).
struct PlanView {
  const int32_t* hdr;
  const int32_t* cum;
  const int32_t* pbase;
  const int32_t* len;
  const int32_t* first;
  const int32_t* wstart;
  const int32_t* pw0;
  const int32_t* pcnt;
  const int32_t* lo;
  const int32_t* tf;
};

__host__ __device__ __forceinline__ size_t plan_ints(int problems, int workers) {
  return 8 + 8 * (size_t)problems + 2 * (size_t)workers;
}

__device__ __forceinline__ PlanView plan_view(const int32_t* plan) {
  const int P = plan[0];
  PlanView v;
  v.hdr = plan;
  v.cum = plan + 4;
  v.pbase = v.cum + (P + 1);
  v.len = v.pbase + (P + 1);
  v.first = v.len + P;
  v.wstart = v.first + plan[3];
  v.pw0 = v.wstart + plan[3] + 1;
  v.pcnt = v.pw0 + P;
  v.lo = v.pcnt + P + (P + 1);  // after vcum
  v.tf = v.lo + P;
  return v;
}
__host__ __device__ __forceinline__ size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// Workers that touch problem p and its partial base slot.
__device__ __forceinline__ void problem_workers(const PlanView& pv, int p, int* first, int* count) {
  *first = pv.pw0[p];
  *count = pv.pcnt[p];
}

// ------------------------------------------------------------------ launchers
// seq_start (device [B], may be NULL for all zeros): each sequence's first visible key position.
cudaError_t launch_plan(int B, int q_per_seq, const int32_t* seq_lens, const int32_t* seq_start, int tile_n,
                        int seg_cost, int workers, int32_t* plan, cudaStream_t st);

template <typename A>
cudaError_t launch_append_simt(const mla_dims_t& d, const mla_cache_t& c, int T, const A* h,
                               const A* w_dkv, const A* w_kr, const int32_t* seq_idx,
                               const int32_t* pos, const int32_t* bt, int max_pages,
                               float* ws, int ksplit, int32_t* status, cudaStream_t st);

template <typename A>
cudaError_t launch_absorb_simt(const mla_dims_t& d, int T, const A* q, const int32_t* pos,
                               const A* w_uk, A* q_abs, cudaStream_t st);

template <typename A>
cudaError_t launch_out_proj_simt(const mla_dims_t& d, int T, const A* o_lat, const A* w_uv,
                                 A* o, cudaStream_t st);

template <typename A>
cudaError_t launch_decode_simt(const mla_dims_t& d, const mla_cache_t& c, int B, int q_per_seq,
                               const A* q_abs, const int32_t* bt, int max_pages,
                               const int32_t* plan, int workers, float* o_part, float* lse_part,
                               A* o_lat, float* lse, int32_t* status, cudaStream_t st);

// Merges the split partials of each problem. Partial rows are [slot][head][d_c]
// row-major, or, with `blocked` (the tensor-core decode, d_c = 512, n_h = 128),
// piece-major: [slot][32-column chunk][4-column piece][head][4]; `workers` (the
// decode's worker count) then picks the combine's form.
template <typename A>
cudaError_t launch_combine(const mla_dims_t& d, int problems, const int32_t* plan,
                           const float* o_part, const float* lse_part, A* o_lat, float* lse,
                           cudaStream_t st, bool blocked = false, int workers = 0);

cudaError_t launch_quantize_rows(const float* x, int rows, int cols, uint8_t* codes, float* scales,
                                 cudaStream_t st);

// out[t][i] = sum over k < ksplit of ws[k][t][i], rounded to A (T rows of n).
template <typename A>
cudaError_t launch_reduce_splits(int T, int n, int ksplit, const float* ws, A* out, cudaStream_t st);
// Split-K partial sums of out = W_O . o on CUDA cores (o as [T][n_h * d_v]) into ws[ksplit][T][d_model].
template <typename A>
cudaError_t launch_wo_gemm_simt(const mla_dims_t& d, int T, const A* o, const A* w_o, float* ws, int ksplit,
                                cudaStream_t st);
int wo_ksplit_simt(const mla_dims_t& d, int T);

int append_ksplit(int T, int n_out, int d_model);
int sm_count();

// Launches `k` with programmatic stream serialization (see pdl_wait above).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*k)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, std::forward<Args>(args)...);
}
// True when the current device is an sm_103 part (B300), the only target the
// tensor-core kernels are built for.
bool tc_device_ok();

template <typename A>
cudaError_t launch_append_epilogue(const mla_dims_t& d, const mla_cache_t& c, int T,
                                   const int32_t* seq_idx, const int32_t* pos, const int32_t* bt,
                                   int max_pages, const float* ws, int ksplit, int32_t* status,
                                   cudaStream_t st);

}  // namespace mla
