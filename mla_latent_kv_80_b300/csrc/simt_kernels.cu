// CUDA-core kernels for every step of MLA decode: the fp32 path, and the
// reference-shaped path for dims the tensor-core kernels do not cover.
//
// Method: DeepSeek-V2 MLA as the pages state it ("MLA 之后，KV cache 确实得重新
// 理解一遍": c_kv = W_DKV x, k_R = RoPE(W_KR x), score = (W_UK^T q)^T c_kv +
// q_R^T k_R, o = W_UV (sum_j a_j c_kv(j))).
#include "mla_internal.cuh"

#include <math.h>

#include <cmath>
#include <mutex>

namespace mla {

RopeFreqs rope_freqs(int d_rope, float theta) {
  // A small cache: decode steps call this with the same (d_rope, theta).
  static std::mutex mu;
  static int cached_d = -1;
  static float cached_theta = 0.f;
  static RopeFreqs cached;
  std::lock_guard<std::mutex> lock(mu);
  if (d_rope != cached_d || theta != cached_theta) {
    for (int i = 0; i < kMaxDrope / 2; ++i) {
      const double f = i < d_rope / 2 ? std::pow((double)theta, -2.0 * i / (double)d_rope) : 0.0;
      cached.hi[i] = (float)f;
      cached.lo[i] = (float)(f - (double)cached.hi[i]);
    }
    cached_d = d_rope;
    cached_theta = theta;
  }
  return cached;
}

// ====================================================================== plan
// One block builds the split plan: problem p = b * q + j has
// len_p = seq_lens[b] - q + j + 1 visible keys and ceil(len_p / tile_n) tiles.
// Prefix sums run in shared memory in chunks of blockDim.x problems.
__device__ __forceinline__ int block_exclusive_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5, nw = blockDim.x >> 5;
  int x = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(0xffffffffu, x, o);
    if (lane >= o) x += n;
  }
  if (lane == 31) warp_tot[wid] = x;
  __syncthreads();
  if (wid == 0) {
    int t = lane < nw ? warp_tot[lane] : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int n = __shfl_up_sync(0xffffffffu, t, o);
      if (lane >= o) t += n;
    }
    if (lane < nw) warp_tot[lane] = t;
  }
  __syncthreads();
  const int excl = x - v + (wid > 0 ? warp_tot[wid - 1] : 0);
  *total = warp_tot[nw - 1];
  __syncthreads();
  return excl;
}

__global__ void __launch_bounds__(1024) plan_kernel(int B, int q, const int32_t* __restrict__ seq_lens,
                                                    const int32_t* __restrict__ seq_start, int tile_n, int seg_cost,
                                                    int workers, int32_t* __restrict__ plan) {
  pdl_trigger();
  pdl_wait();
  const int P = B * q, G = workers;
  int32_t* cum = plan + 4;
  int32_t* pbase = cum + (P + 1);
  int32_t* lens = pbase + (P + 1);
  int32_t* first = lens + P;
  int32_t* wstart = first + G;
  int32_t* pw0 = wstart + G + 1;
  int32_t* pcnt = pw0 + P;
  int32_t* vcum = pcnt + P;
  int32_t* los = vcum + (P + 1);
  int32_t* tfs = los + P;
  __shared__ int warp_tot[32];
  // Pass 1: tiles, their prefix sums, and the prefix sums of tiles plus start costs.
  int carry = 0, vcarry = 0;
  for (int base = 0; base < P; base += blockDim.x) {
    const int p = base + threadIdx.x;
    int tiles = 0;
    if (p < P) {
      int len = seq_lens[p / q] - q + (p % q) + 1;
      len = len < 0 ? 0 : len;
      int lo = seq_start != nullptr ? seq_start[p / q] : 0;
      lo = lo < 0 ? 0 : (lo > len ? len : lo);
      const int tf = lo / tile_n;
      tiles = lo < len ? (len + tile_n - 1) / tile_n - tf : 0;
      lens[p] = len;
      los[p] = lo;
      tfs[p] = tf;
    }
    int total, vtotal;
    const int excl = block_exclusive_scan(tiles, warp_tot, &total);
    const int vexcl = block_exclusive_scan(tiles > 0 ? tiles + seg_cost : 0, warp_tot, &vtotal);
    if (p < P) {
      cum[p] = carry + excl;
      vcum[p] = vcarry + vexcl;
    }
    carry += total;
    vcarry += vtotal;
  }
  const int total_tiles = carry, total_v = vcarry;
  int per_v = G > 0 ? (total_v + G - 1) / G : total_v;
  per_v = per_v < 1 ? 1 : per_v;
  for (int w = threadIdx.x; w <= G; w += blockDim.x) {
    wstart[w] = total_tiles;
    if (w < G) first[w] = P;
  }
  __syncthreads();  // cum[], vcum[] and the initial wstart[] are read below
  // Pass 2: worker w starts at cost position w * per_v; inside problem p (cost
  // range [vcum[p], vcum[p+1]), its first seg_cost units standing for the start
  // cost) that is tile cum[p] + max(0, position - vcum[p] - seg_cost).
  for (int p = threadIdx.x; p < P; p += blockDim.x) {
    const int v0 = vcum[p];
    const int v1 = (p + 1 < P) ? vcum[p + 1] : total_v;
    if (v1 > v0) {
      for (int w = (v0 + per_v - 1) / per_v; w <= (v1 - 1) / per_v && w < G; ++w) {
        const int into = w * per_v - v0 - seg_cost;
        wstart[w] = cum[p] + (into > 0 ? into : 0);
        first[w] = p;
      }
    }
  }
  __syncthreads();  // wstart[] is searched below
  // Pass 3: the workers of each problem and the partial slots of the problems
  // cut between workers.
  carry = 0;
  for (int base = 0; base < P; base += blockDim.x) {
    const int p = base + threadIdx.x;
    int cnt = 0;
    if (p < P) {
      const int c0 = cum[p];
      const int c1 = (p + 1 < P) ? cum[p + 1] : total_tiles;
      int w0 = 0, n = 0;
      if (c1 > c0 && G > 0) {
        // first worker whose range ends past c0, first worker whose range ends past c1 - 1
        int lo = 0, hi = G - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (wstart[mid + 1] > c0) hi = mid; else lo = mid + 1;
        }
        w0 = lo;
        hi = G - 1;
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (wstart[mid + 1] > c1 - 1) hi = mid; else lo = mid + 1;
        }
        n = lo - w0 + 1;
      }
      pw0[p] = w0;
      pcnt[p] = n;
      cnt = n >= 2 ? n : 0;
    }
    int total;
    const int excl = block_exclusive_scan(cnt, warp_tot, &total);
    if (p < P) pbase[p] = carry + excl;
    carry += total;
  }
  if (threadIdx.x == 0) {
    cum[P] = total_tiles;
    pbase[P] = carry;
    vcum[P] = total_v;
    plan[0] = P;
    plan[1] = total_tiles;
    plan[2] = seg_cost;
    plan[3] = G;
  }
}

cudaError_t launch_plan(int B, int q_per_seq, const int32_t* seq_lens, const int32_t* seq_start, int tile_n,
                        int seg_cost, int workers, int32_t* plan, cudaStream_t st) {
  int threads = B * q_per_seq;
  threads = threads < 32 ? 32 : (threads > 1024 ? 1024 : ((threads + 31) / 32) * 32);
  return launch_pdl(plan_kernel, dim3(1), dim3(threads), 0, st, B, q_per_seq, seq_lens, seq_start, tile_n, seg_cost,
                    workers, plan);
}

// ====================================================================== append
// Split-K GEMM: ws[ks][t][n] = sum over k in split ks of h[t][k] * W[n][k], where
// W = [W_DKV ; W_KR] (n < d_c from W_DKV, else W_KR).
constexpr int AP_TOK = 16, AP_OUT = 64, AP_K = 64;

template <typename A>
__global__ void __launch_bounds__(256) append_gemm_kernel(int T, int d_c, int d_rope, int d_model,
                                                          const A* __restrict__ h,
                                                          const A* __restrict__ w_dkv,
                                                          const A* __restrict__ w_kr, int k_per_split,
                                                          float* __restrict__ ws) {
  pdl_trigger();
  pdl_wait();
  __shared__ float hs[AP_TOK][AP_K + 1];
  __shared__ float wsm[AP_K][AP_OUT + 1];
  const int n_out = d_c + d_rope;
  const int n0 = blockIdx.x * AP_OUT, t0 = blockIdx.y * AP_TOK, ks = blockIdx.z;
  const int k_begin = ks * k_per_split;
  const int k_end = min(d_model, k_begin + k_per_split);
  const int col = threadIdx.x % AP_OUT, grp = threadIdx.x / AP_OUT;  // 4 groups of 4 tokens
  float acc[4] = {0.f, 0.f, 0.f, 0.f};
  for (int k0 = k_begin; k0 < k_end; k0 += AP_K) {
    for (int i = threadIdx.x; i < AP_TOK * AP_K; i += blockDim.x) {
      int tt = i / AP_K, kk = i % AP_K;
      int t = t0 + tt, k = k0 + kk;
      hs[tt][kk] = (t < T && k < k_end) ? to_f32(h[(size_t)t * d_model + k]) : 0.f;
    }
    for (int i = threadIdx.x; i < AP_OUT * AP_K; i += blockDim.x) {
      int nn = i / AP_K, kk = i % AP_K;
      int n = n0 + nn, k = k0 + kk;
      float v = 0.f;
      if (n < n_out && k < k_end)
        v = n < d_c ? to_f32(w_dkv[(size_t)n * d_model + k])
                    : to_f32(w_kr[(size_t)(n - d_c) * d_model + k]);
      wsm[kk][nn] = v;
    }
    __syncthreads();
#pragma unroll 8
    for (int kk = 0; kk < AP_K; ++kk) {
      float wv = wsm[kk][col];
#pragma unroll
      for (int i = 0; i < 4; ++i) acc[i] = fmaf(hs[grp * 4 + i][kk], wv, acc[i]);
    }
    __syncthreads();
  }
  int n = n0 + col;
  if (n < n_out) {
    for (int i = 0; i < 4; ++i) {
      int t = t0 + grp * 4 + i;
      if (t < T) ws[((size_t)ks * T + t) * n_out + n] = acc[i];
    }
  }
}

// Epilogue per token: reduce the K splits, rotate k_R, quantise, write the slot.
template <typename A, CacheKind CK>
__global__ void __launch_bounds__(256) append_epilogue_kernel(
    int T, int d_c, int d_rope, int page_size, RopeFreqs freqs, int ksplit,
    const float* __restrict__ ws, const int32_t* __restrict__ seq_idx,
    const int32_t* __restrict__ pos, const int32_t* __restrict__ bt, int max_pages,
    int64_t num_pages, void* __restrict__ ckv, void* __restrict__ kr, float* __restrict__ scale,
    int32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ float x[kMaxDc + kMaxDrope];
  __shared__ float red[32];
  const int t = blockIdx.x;
  const int n_out = d_c + d_rope;
  // The token's slot is looked up first, so that these dependent loads overlap
  // the loads of the partial sums below.
  const int p = pos[t], b = seq_idx[t];
  const int pg = p / page_size;
  int page = -1;
  if (p >= 0 && pg < max_pages) page = bt[(size_t)b * max_pages + pg];
  for (int n = threadIdx.x; n < n_out; n += blockDim.x) {
    // Up to 8 K-split partials are loaded before they are summed.
    float s = 0.f;
    int k = 0;
    for (; k + 8 <= ksplit; k += 8) {
      float v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) v[u] = ws[((size_t)(k + u) * T + t) * n_out + n];
#pragma unroll
      for (int u = 0; u < 8; ++u) s += v[u];
    }
    for (; k < ksplit; ++k) s += ws[((size_t)k * T + t) * n_out + n];
    x[n] = s;
  }
  __syncthreads();
  // RoPE on the decoupled key, pairs (2i, 2i+1).
  for (int i = threadIdx.x; i < d_rope / 2; i += blockDim.x) {
    float c, s;
    rope_cos_sin(p, freqs.hi[i], freqs.lo[i], &c, &s);
    float x0 = x[d_c + 2 * i], x1 = x[d_c + 2 * i + 1];
    float r0 = x0 * c - x1 * s;
    float r1 = x0 * s + x1 * c;
    x[d_c + 2 * i] = r0;
    x[d_c + 2 * i + 1] = r1;
  }
  __syncthreads();
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0) set_status(status, MLA_ERR_BAD_PAGE);
    return;
  }
  const int64_t slot = (int64_t)page * page_size + p % page_size;
  if constexpr (CK == CacheKind::FP8) {
    float m = 0.f;
    for (int n = threadIdx.x; n < d_c; n += blockDim.x) m = fmaxf(m, fabsf(x[n]));
    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
    __syncthreads();
    if (threadIdx.x < 32) {
      float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
      for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
      if (threadIdx.x == 0) red[0] = v;
    }
    __syncthreads();
    const float sc = e4m3_row_scale(red[0]);
    uint8_t* dst = reinterpret_cast<uint8_t*>(ckv) + slot * d_c;
    for (int n = threadIdx.x; n < d_c; n += blockDim.x) dst[n] = f32_to_e4m3(x[n] / sc);
    __nv_bfloat16* kd = reinterpret_cast<__nv_bfloat16*>(kr) + slot * d_rope;
    for (int n = threadIdx.x; n < d_rope; n += blockDim.x) kd[n] = __float2bfloat16_rn(x[d_c + n]);
    if (threadIdx.x == 0) scale[slot] = sc;
  } else {
    using C = typename std::conditional<CK == CacheKind::F32, float, __nv_bfloat16>::type;
    C* dst = reinterpret_cast<C*>(ckv) + slot * n_out;
    for (int n = threadIdx.x; n < n_out; n += blockDim.x) dst[n] = from_f32<C>(x[n]);
  }
}

int append_ksplit(int T, int n_out, int d_model) {
  if (T <= 0) return 1;
  int tiles = ((n_out + AP_OUT - 1) / AP_OUT) * ((T + AP_TOK - 1) / AP_TOK);
  int kchunks = (d_model + AP_K - 1) / AP_K;
  int ks = (2 * 148 + tiles - 1) / tiles;
  ks = ks < 1 ? 1 : ks;
  ks = ks > kchunks ? kchunks : ks;
  ks = ks > 32 ? 32 : ks;
  return ks;
}

template <typename A>
cudaError_t launch_append_simt(const mla_dims_t& d, const mla_cache_t& c, int T, const A* h,
                               const A* w_dkv, const A* w_kr, const int32_t* seq_idx,
                               const int32_t* pos, const int32_t* bt, int max_pages, float* ws,
                               int ksplit, int32_t* status, cudaStream_t st) {
  const int n_out = d.d_c + d.d_rope;
  int kchunks = (d.d_model + AP_K - 1) / AP_K;
  int k_per_split = ((kchunks + ksplit - 1) / ksplit) * AP_K;
  dim3 grid((n_out + AP_OUT - 1) / AP_OUT, (T + AP_TOK - 1) / AP_TOK, ksplit);
  cudaError_t e = launch_pdl(append_gemm_kernel<A>, grid, dim3(256), 0, st, T, d.d_c, d.d_rope, d.d_model, h,
                             w_dkv, w_kr, k_per_split, ws);
  if (e != cudaSuccess) return e;
  return launch_append_epilogue<A>(d, c, T, seq_idx, pos, bt, max_pages, ws, ksplit, status, st);
}

// The same for fp32 and bf16 caches, spread wider: one block per (token, 128
// outputs) and one output per thread, with all of an output's split-K partials
// requested before they are summed (no whole-row reduction is needed without
// the fp8 scale). A RoPE pair (2i, 2i+1) never straddles two blocks (d_c is
// even), so the k_R part is rotated through shared memory within its block.
template <typename A, CacheKind CK>
__global__ void __launch_bounds__(128) append_epilogue_wide_kernel(
    int T, int d_c, int d_rope, int page_size, RopeFreqs freqs, int ksplit,
    const float* __restrict__ ws, const int32_t* __restrict__ seq_idx,
    const int32_t* __restrict__ pos, const int32_t* __restrict__ bt, int max_pages,
    int64_t num_pages, void* __restrict__ ckv, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  __shared__ float x[128];
  const int t = blockIdx.x, n = blockIdx.y * 128 + threadIdx.x;
  const int n_out = d_c + d_rope;
  const int p = pos[t], b = seq_idx[t];
  const int pg = p / page_size;
  int page = -1;
  if (p >= 0 && pg < max_pages) page = bt[(size_t)b * max_pages + pg];
  float sum = 0.f;
  if (n < n_out) {
    int k = 0;
    for (; k + 16 <= ksplit; k += 16) {
      float v[16];
#pragma unroll
      for (int u = 0; u < 16; ++u) v[u] = ws[((size_t)(k + u) * T + t) * n_out + n];
#pragma unroll
      for (int u = 0; u < 16; ++u) sum += v[u];
    }
    for (; k < ksplit; ++k) sum += ws[((size_t)k * T + t) * n_out + n];
  }
  x[threadIdx.x] = sum;
  __syncthreads();
  if (n >= d_c && n < n_out && ((n - d_c) & 1) == 0) {
    const int i = (n - d_c) / 2;
    float c, sn;
    rope_cos_sin(p, freqs.hi[i], freqs.lo[i], &c, &sn);
    const float x0 = x[threadIdx.x], x1 = x[threadIdx.x + 1];
    x[threadIdx.x] = x0 * c - x1 * sn;
    x[threadIdx.x + 1] = x0 * sn + x1 * c;
  }
  __syncthreads();
  if (page < 0 || page >= num_pages) {
    if (threadIdx.x == 0 && blockIdx.y == 0) set_status(status, MLA_ERR_BAD_PAGE);
    return;
  }
  using C = typename std::conditional<CK == CacheKind::F32, float, __nv_bfloat16>::type;
  const int64_t slot = (int64_t)page * page_size + p % page_size;
  if (n < n_out) reinterpret_cast<C*>(ckv)[slot * n_out + n] = from_f32<C>(x[threadIdx.x]);
}

template <typename A>
cudaError_t launch_append_epilogue(const mla_dims_t& d, const mla_cache_t& c, int T,
                                   const int32_t* seq_idx, const int32_t* pos, const int32_t* bt,
                                   int max_pages, const float* ws, int ksplit, int32_t* status,
                                   cudaStream_t st) {
  switch (d.cache_dtype) {
    case MLA_F32:
      return launch_pdl(append_epilogue_wide_kernel<A, CacheKind::F32>, dim3(T, (d.d_c + d.d_rope + 127) / 128),
                        dim3(128), 0, st, T, d.d_c, d.d_rope, d.page_size, rope_freqs(d.d_rope, d.rope_theta), ksplit,
                        ws, seq_idx, pos, bt, max_pages, c.num_pages, c.ckv, status);
    case MLA_BF16:
      return launch_pdl(append_epilogue_wide_kernel<A, CacheKind::BF16>, dim3(T, (d.d_c + d.d_rope + 127) / 128),
                        dim3(128), 0, st, T, d.d_c, d.d_rope, d.page_size, rope_freqs(d.d_rope, d.rope_theta), ksplit,
                        ws, seq_idx, pos, bt, max_pages, c.num_pages, c.ckv, status);
    default:
      return launch_pdl(append_epilogue_kernel<A, CacheKind::FP8>, dim3(T), dim3(256), 0, st, T, d.d_c, d.d_rope,
                        d.page_size, rope_freqs(d.d_rope, d.rope_theta), ksplit, ws, seq_idx, pos, bt, max_pages,
                        c.num_pages, c.ckv, c.kr, c.scale, status);
  }
}

// ====================================================================== absorb
constexpr int AB_TOK = 16;

template <typename A>
__global__ void __launch_bounds__(256) absorb_kernel(int T, int n_h, int d_h, int d_rope, int d_c,
                                                     RopeFreqs freqs, const A* __restrict__ q,
                                                     const int32_t* __restrict__ pos,
                                                     const A* __restrict__ w_uk,
                                                     A* __restrict__ q_abs) {
  pdl_trigger();
  pdl_wait();
  __shared__ float qs[AB_TOK][kMaxDh];
  const int h = blockIdx.x, t0 = blockIdx.y * AB_TOK;
  const int dq = d_h + d_rope, dqa = d_c + d_rope;
  for (int i = threadIdx.x; i < AB_TOK * d_h; i += blockDim.x) {
    int tt = i / d_h, k = i % d_h, t = t0 + tt;
    qs[tt][k] = t < T ? to_f32(q[((size_t)t * n_h + h) * dq + k]) : 0.f;
  }
  __syncthreads();
  const A* W = w_uk + (size_t)h * d_h * d_c;
  for (int col = threadIdx.x; col < d_c; col += blockDim.x) {
    float acc[AB_TOK];
#pragma unroll
    for (int i = 0; i < AB_TOK; ++i) acc[i] = 0.f;
    for (int k = 0; k < d_h; ++k) {
      float w = to_f32(W[(size_t)k * d_c + col]);
#pragma unroll
      for (int i = 0; i < AB_TOK; ++i) acc[i] = fmaf(qs[i][k], w, acc[i]);
    }
#pragma unroll
    for (int i = 0; i < AB_TOK; ++i) {
      int t = t0 + i;
      if (t < T) q_abs[((size_t)t * n_h + h) * dqa + col] = from_f32<A>(acc[i]);
    }
  }
  const int half = d_rope / 2;
  for (int i = threadIdx.x; i < AB_TOK * half; i += blockDim.x) {
    int tt = i / half, pr = i % half, t = t0 + tt;
    if (t >= T) continue;
    const A* src = q + ((size_t)t * n_h + h) * dq + d_h;
    float x0 = to_f32(src[2 * pr]), x1 = to_f32(src[2 * pr + 1]);
    float c, s;
    rope_cos_sin(pos[t], freqs.hi[pr], freqs.lo[pr], &c, &s);
    A* dst = q_abs + ((size_t)t * n_h + h) * dqa + d_c;
    dst[2 * pr] = from_f32<A>(x0 * c - x1 * s);
    dst[2 * pr + 1] = from_f32<A>(x0 * s + x1 * c);
  }
}

template <typename A>
cudaError_t launch_absorb_simt(const mla_dims_t& d, int T, const A* q, const int32_t* pos,
                               const A* w_uk, A* q_abs, cudaStream_t st) {
  dim3 grid(d.n_h, (T + AB_TOK - 1) / AB_TOK);
  return launch_pdl(absorb_kernel<A>, grid, dim3(256), 0, st, T, d.n_h, d.d_h, d.d_rope, d.d_c,
                    rope_freqs(d.d_rope, d.rope_theta), q, pos, w_uk, q_abs);
}

// ====================================================================== out projection
constexpr int OP_TOK = 8;

template <typename A>
__global__ void __launch_bounds__(256) out_proj_kernel(int T, int n_h, int d_c, int d_v,
                                                       const A* __restrict__ o_lat,
                                                       const A* __restrict__ w_uv,
                                                       A* __restrict__ o) {
  pdl_trigger();
  pdl_wait();
  __shared__ float xs[OP_TOK][kMaxDc];
  const int h = blockIdx.x, t0 = blockIdx.y * OP_TOK;
  for (int i = threadIdx.x; i < OP_TOK * d_c; i += blockDim.x) {
    int tt = i / d_c, k = i % d_c, t = t0 + tt;
    xs[tt][k] = t < T ? to_f32(o_lat[((size_t)t * n_h + h) * d_c + k]) : 0.f;
  }
  __syncthreads();
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
  const A* W = w_uv + (size_t)h * d_v * d_c;
  for (int row = warp; row < d_v; row += nwarps) {
    float acc[OP_TOK];
#pragma unroll
    for (int i = 0; i < OP_TOK; ++i) acc[i] = 0.f;
    for (int k = lane; k < d_c; k += 32) {
      float w = to_f32(W[(size_t)row * d_c + k]);
#pragma unroll
      for (int i = 0; i < OP_TOK; ++i) acc[i] = fmaf(w, xs[i][k], acc[i]);
    }
#pragma unroll
    for (int i = 0; i < OP_TOK; ++i) {
      float v = acc[i];
      for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
      int t = t0 + i;
      if (lane == 0 && t < T) o[((size_t)t * n_h + h) * d_v + row] = from_f32<A>(v);
    }
  }
}

template <typename A>
cudaError_t launch_out_proj_simt(const mla_dims_t& d, int T, const A* o_lat, const A* w_uv, A* o,
                                 cudaStream_t st) {
  dim3 grid(d.n_h, (T + OP_TOK - 1) / OP_TOK);
  return launch_pdl(out_proj_kernel<A>, grid, dim3(256), 0, st, T, d.n_h, d.d_c, d.d_v, o_lat, w_uv, o);
}

// ====================================================================== decode (CUDA cores)
// Grid (workers, head groups). Each block walks its worker's share of the tile
// sequence, keeping for HG heads the running max m, the running sum l and the
// unnormalised latent sum O (online softmax), and writes either the final
// o_lat / lse or a partial for the combine kernel.
constexpr int DS_HG = 8;     // heads per block
constexpr int DS_TILE = 32;  // tokens per tile (one lane per token in the softmax)

__host__ __device__ inline size_t decode_simt_smem(int d_qk) {
  return sizeof(float) * ((size_t)DS_HG * d_qk + (size_t)DS_TILE * (d_qk + 1) + DS_HG * DS_TILE +
                          3 * DS_HG);
}

template <typename A, CacheKind CK>
__global__ void __launch_bounds__(256) decode_simt_kernel(
    int n_h, int d_c, int d_rope, int page_size, float scale, int q_per_seq,
    const A* __restrict__ q_abs, const void* __restrict__ ckv, const void* __restrict__ kr,
    const float* __restrict__ cscale, int64_t num_pages, const int32_t* __restrict__ bt,
    int max_pages, const int32_t* __restrict__ plan, float* __restrict__ o_part,
    float* __restrict__ lse_part, A* __restrict__ o_lat, float* __restrict__ lse_out,
    int32_t* status) {
  pdl_trigger();
  pdl_wait();
  extern __shared__ float smem[];
  const int d_qk = d_c + d_rope;
  float* qs = smem;                          // [HG][d_qk]
  float* cs = qs + DS_HG * d_qk;             // [TILE][d_qk + 1]
  float* ps = cs + DS_TILE * (d_qk + 1);     // [HG][TILE]
  float* ms = ps + DS_HG * DS_TILE;          // [HG] running max
  float* ls = ms + DS_HG;                    // [HG] running sum
  float* cr = ls + DS_HG;                    // [HG] rescale factor of this tile

  PlanView pv = plan_view(plan);
  const int w = blockIdx.x;
  const int h0 = blockIdx.y * DS_HG;
  const int nh_blk = min(DS_HG, n_h - h0);
  int g0 = pv.wstart[w];
  const int g1 = pv.wstart[w + 1];
  if (g0 >= g1) return;
  int p = pv.first[w];  // the problem holding this worker's first tile
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int cols_per_thread = (d_c + blockDim.x - 1) / blockDim.x;  // <= 2 for d_c <= 512
  while (g0 < g1) {
    while (pv.cum[p + 1] <= g0) ++p;
    const int b = p / q_per_seq, j = p % q_per_seq;
    const int t_lo = g0 - pv.cum[p];
    const int t_hi = min(g1, pv.cum[p + 1]) - pv.cum[p];
    const int len = pv.len[p], lo = pv.lo[p], tf = pv.tf[p];
    (void)j;
    // Load q for the block's heads.
    const A* qsrc = q_abs + (size_t)p * n_h * d_qk;
    for (int i = threadIdx.x; i < DS_HG * d_qk; i += blockDim.x) {
      int hh = i / d_qk, k = i % d_qk;
      qs[i] = hh < nh_blk ? to_f32(qsrc[(size_t)(h0 + hh) * d_qk + k]) : 0.f;
    }
    if (threadIdx.x < DS_HG) { ms[threadIdx.x] = -INFINITY; ls[threadIdx.x] = 0.f; }
    float acc[DS_HG][2];
#pragma unroll
    for (int hh = 0; hh < DS_HG; ++hh) { acc[hh][0] = 0.f; acc[hh][1] = 0.f; }
    __syncthreads();
    for (int tile = t_lo; tile < t_hi; ++tile) {
      const int tok0 = (tf + tile) * DS_TILE;
      // Stage the tile (fp32), zero past the sequence end.
      for (int i = threadIdx.x; i < DS_TILE * d_qk; i += blockDim.x) {
        int tt = i / d_qk, k = i % d_qk, t = tok0 + tt;
        float v = 0.f;
        if (t >= lo && t < len) {
          int pg = t / page_size;
          int page = pg < max_pages ? bt[(size_t)b * max_pages + pg] : -1;
          if (page < 0 || page >= num_pages) {
            set_status(status, MLA_ERR_BAD_PAGE);
          } else {
            int64_t slot = (int64_t)page * page_size + t % page_size;
            if constexpr (CK == CacheKind::FP8) {
              if (k < d_c)
                v = e4m3_to_f32(reinterpret_cast<const uint8_t*>(ckv)[slot * d_c + k]) * cscale[slot];
              else
                v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(kr)[slot * d_rope + (k - d_c)]);
            } else if constexpr (CK == CacheKind::F32) {
              v = reinterpret_cast<const float*>(ckv)[slot * d_qk + k];
            } else {
              v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(ckv)[slot * d_qk + k]);
            }
          }
        }
        cs[tt * (d_qk + 1) + k] = v;
      }
      __syncthreads();
      // Scores: warp = head, lane = token.
      for (int hh = warp; hh < DS_HG; hh += blockDim.x / 32) {
        const int t = tok0 + lane;
        float s = 0.f;
        const float* qh = qs + hh * d_qk;
        const float* ct = cs + lane * (d_qk + 1);
        for (int k = 0; k < d_qk; ++k) s = fmaf(qh[k], ct[k], s);
        s = (t >= lo && t < len && hh < nh_blk) ? s * scale : -INFINITY;
        float mx = s;
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        const float m_old = ms[hh];
        const float m_new = fmaxf(m_old, mx);
        const float pr = (s == -INFINITY) ? 0.f : expf(s - m_new);
        float sum = pr;
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        ps[hh * DS_TILE + lane] = pr;
        if (lane == 0) {
          const float c = (m_old == -INFINITY) ? 0.f : expf(m_old - m_new);
          cr[hh] = c;
          ls[hh] = ls[hh] * c + sum;
          ms[hh] = m_new;
        }
      }
      __syncthreads();
      // O = O * c + P . C over the latent columns.
      for (int ci = 0; ci < cols_per_thread; ++ci) {
        const int col = threadIdx.x + ci * blockDim.x;
        if (col >= d_c) break;
#pragma unroll
        for (int hh = 0; hh < DS_HG; ++hh) {
          float a = acc[hh][ci] * cr[hh];
          for (int tt = 0; tt < DS_TILE; ++tt) a = fmaf(ps[hh * DS_TILE + tt], cs[tt * (d_qk + 1) + col], a);
          acc[hh][ci] = a;
        }
      }
      __syncthreads();
    }
    // Write the final result or a partial.
    int first, count;
    problem_workers(pv, p, &first, &count);
    const bool whole = count <= 1;
    const int slot = pv.pbase[p] + (w - first);
    for (int ci = 0; ci < cols_per_thread; ++ci) {
      const int col = threadIdx.x + ci * blockDim.x;
      if (col >= d_c) break;
      for (int hh = 0; hh < nh_blk; ++hh) {
        const float l = ls[hh];
        const float v = l > 0.f ? acc[hh][ci] / l : 0.f;
        const size_t row = (size_t)p * n_h + h0 + hh;
        if (whole) o_lat[row * d_c + col] = from_f32<A>(v);
        else o_part[((size_t)slot * n_h + h0 + hh) * d_c + col] = v;
      }
    }
    if (threadIdx.x < nh_blk) {
      const int hh = threadIdx.x;
      const float l = ls[hh];
      const float lse = l > 0.f ? ms[hh] + logf(l) : -INFINITY;
      if (whole) lse_out[(size_t)p * n_h + h0 + hh] = lse;
      else lse_part[(size_t)slot * n_h + h0 + hh] = lse;
    }
    __syncthreads();
    g0 = pv.cum[p] + t_hi;
    ++p;
  }
}

template <typename A>
cudaError_t launch_decode_simt(const mla_dims_t& d, const mla_cache_t& c, int B, int q_per_seq,
                               const A* q_abs, const int32_t* bt, int max_pages,
                               const int32_t* plan, int workers, float* o_part, float* lse_part,
                               A* o_lat, float* lse, int32_t* status, cudaStream_t st) {
  const int d_qk = d.d_c + d.d_rope;
  const size_t smem = decode_simt_smem(d_qk);
  dim3 grid(workers, (d.n_h + DS_HG - 1) / DS_HG);
  cudaError_t e;
#define MLA_LAUNCH_DS(CKV)                                                                      \
  do {                                                                                          \
    auto k = decode_simt_kernel<A, CKV>;                                                        \
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);        \
    if (e != cudaSuccess) return e;                                                             \
    e = launch_pdl(k, grid, dim3(256), smem, st, d.n_h, d.d_c, d.d_rope, d.page_size,          \
                   d.softmax_scale, q_per_seq, q_abs, c.ckv, c.kr, c.scale, c.num_pages, bt,     \
                   max_pages, plan, o_part, lse_part, o_lat, lse, status);                      \
    if (e != cudaSuccess) return e;                                                             \
  } while (0)
  switch (d.cache_dtype) {
    case MLA_F32: MLA_LAUNCH_DS(CacheKind::F32); break;
    case MLA_BF16: MLA_LAUNCH_DS(CacheKind::BF16); break;
    default: MLA_LAUNCH_DS(CacheKind::FP8); break;
  }
#undef MLA_LAUNCH_DS
  return cudaGetLastError();
}

// ====================================================================== combine
// One warp per (problem, head) row. Problems without keys get o_lat = 0 and
// lse = -inf; problems done by one worker are already final; the others merge
// their partials: lse = log sum_s exp(lse_s), o = sum_s exp(lse_s - lse) o_s.
// Each lane owns VEC-wide column groups and issues the loads of several
// partials before using them, so many loads are in flight per warp.
template <typename A, int VEC>
__global__ void __launch_bounds__(256) combine_kernel(int n_h, int d_c, const int32_t* __restrict__ plan,
                                                      const float* __restrict__ o_part,
                                                      const float* __restrict__ lse_part,
                                                      A* __restrict__ o_lat, float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
  constexpr int kMaxGroups = 512 / (32 * VEC) > 0 ? 512 / (32 * VEC) : 1;
  const int P = plan[0];
  PlanView pv = plan_view(plan);
  const int row = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= P * n_h) return;
  const int p = row / n_h, h = row % n_h;
  int first, count;
  problem_workers(pv, p, &first, &count);
  if (count == 1) return;
  A* dst = o_lat + (size_t)row * d_c;
  if (count == 0) {
    for (int c = lane; c < d_c; c += 32) dst[c] = from_f32<A>(0.f);
    if (lane == 0) lse[row] = -INFINITY;
    return;
  }
  const int base = pv.pbase[p];
  // Max and weight sum of the partial lse values, 32 partials at a time.
  float m = -INFINITY;
  for (int s0 = 0; s0 < count; s0 += 32) {
    const float l = (s0 + lane < count) ? lse_part[(size_t)(base + s0 + lane) * n_h + h] : -INFINITY;
    m = fmaxf(m, l);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float wsum = 0.f;
  for (int s0 = 0; s0 < count; s0 += 32) {
    const float l = (s0 + lane < count) ? lse_part[(size_t)(base + s0 + lane) * n_h + h] : -INFINITY;
    wsum += (l == -INFINITY || m == -INFINITY) ? 0.f : expf(l - m);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) wsum += __shfl_xor_sync(0xffffffffu, wsum, o);
  const float lse_all = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
  const int groups = d_c / (32 * VEC);
  float acc[kMaxGroups][VEC];
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g)
#pragma unroll
    for (int e = 0; e < VEC; ++e) acc[g][e] = 0.f;
  for (int s0 = 0; s0 < count; s0 += 32) {
    const float l = (s0 + lane < count) ? lse_part[(size_t)(base + s0 + lane) * n_h + h] : -INFINITY;
    const float wl = (l == -INFINITY || lse_all == -INFINITY) ? 0.f : expf(l - lse_all);
    const int n = min(32, count - s0);
    for (int i = 0; i < n; ++i) {
      const float wgt = __shfl_sync(0xffffffffu, wl, i);
      const float* src = o_part + ((size_t)(base + s0 + i) * n_h + h) * d_c;
      float v[kMaxGroups][VEC];
#pragma unroll
      for (int g = 0; g < kMaxGroups; ++g) {
        if (g < groups) {
          if constexpr (VEC == 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + (g * 32 + lane) * 4);
            v[g][0] = x.x; v[g][1] = x.y; v[g][2] = x.z; v[g][3] = x.w;
          } else {
            v[g][0] = src[g * 32 + lane];
          }
        }
      }
#pragma unroll
      for (int g = 0; g < kMaxGroups; ++g)
        if (g < groups)
#pragma unroll
          for (int e = 0; e < VEC; ++e) acc[g][e] = fmaf(wgt, v[g][e], acc[g][e]);
    }
  }
#pragma unroll
  for (int g = 0; g < kMaxGroups; ++g) {
    if (g >= groups) break;
#pragma unroll
    for (int e = 0; e < VEC; ++e) {
      const int c = (VEC == 4) ? (g * 32 + lane) * 4 + e : g * 32 + lane;
      dst[c] = from_f32<A>(acc[g][e]);
    }
  }
  if (lane == 0) lse[row] = lse_all;
}

// Combine for d_c = 512: 128 threads per row, one float4 of columns each. The
// problem count comes in as an argument so that the plan lookups are issued
// together, and the first partial rows are requested before their weights are
// known, which keeps the number of dependent memory round trips small.
template <typename A>
__global__ void __launch_bounds__(256) combine_wide_kernel(int P, int n_h, const int32_t* __restrict__ plan,
                                                           const float* __restrict__ o_part,
                                                           const float* __restrict__ lse_part,
                                                           A* __restrict__ o_lat, float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
  constexpr int D = 512;
  constexpr int kPre = 4;  // partial rows fetched before the weights
  const int row = blockIdx.x * 2 + (threadIdx.x >> 7);
  const int tid = threadIdx.x & 127;
  if (row >= P * n_h) return;
  const int p = row / n_h, h = row % n_h;
  const PlanView pv = plan_view(plan);
  const int base = pv.pbase[p], count = pv.pcnt[p];
  if (count == 1) return;
  A* dst = o_lat + (size_t)row * D + tid * 4;
  if (count == 0) {
#pragma unroll
    for (int e = 0; e < 4; ++e) dst[e] = from_f32<A>(0.f);
    if (tid == 0) lse[row] = -INFINITY;
    return;
  }
  const float* lp = lse_part + (size_t)base * n_h + h;
  const float* op = o_part + ((size_t)base * n_h + h) * D + tid * 4;
  const size_t stride = (size_t)n_h * D;
  float4 pre[kPre];
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    pre[u] = u < count ? *reinterpret_cast<const float4*>(op + (size_t)u * stride) : make_float4(0.f, 0.f, 0.f, 0.f);
  // Online maximum and weight sum of the partial lse values in one pass.
  float m = -INFINITY, wsum = 0.f;
  for (int s = 0; s < count; ++s) {
    const float l = lp[(size_t)s * n_h];
    if (l == -INFINITY) continue;
    if (l > m) {
      wsum = wsum * expf(m - l) + 1.f;
      m = l;
    } else {
      wsum += expf(l - m);
    }
  }
  const float lse_all = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  auto add = [&](const float4& v, float l) {
    const float wgt = (l == -INFINITY || lse_all == -INFINITY) ? 0.f : expf(l - lse_all);
    acc.x = fmaf(wgt, v.x, acc.x);
    acc.y = fmaf(wgt, v.y, acc.y);
    acc.z = fmaf(wgt, v.z, acc.z);
    acc.w = fmaf(wgt, v.w, acc.w);
  };
#pragma unroll
  for (int u = 0; u < kPre; ++u)
    if (u < count) add(pre[u], lp[(size_t)u * n_h]);
  int s = kPre;
  for (; s + 4 <= count; s += 4) {
    float4 v[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) v[u] = *reinterpret_cast<const float4*>(op + (size_t)(s + u) * stride);
#pragma unroll
    for (int u = 0; u < 4; ++u) add(v[u], lp[(size_t)(s + u) * n_h]);
  }
  for (; s < count; ++s) add(*reinterpret_cast<const float4*>(op + (size_t)s * stride), lp[(size_t)s * n_h]);
  dst[0] = from_f32<A>(acc.x);
  dst[1] = from_f32<A>(acc.y);
  dst[2] = from_f32<A>(acc.z);
  dst[3] = from_f32<A>(acc.w);
  if (tid == 0) lse[row] = lse_all;
}

// Combine for the piece-major partials of the tensor-core decode (d_c = 512,
// 128 heads). Block (problem, 32-column chunk, part): two threads per head
// row, each merging kSub 4-column pieces; for a given split and piece the loads
// of 128 threads cover 2 KB contiguously. Splits are merged kBatch at a time:
// their lse values and pieces are all requested before any is used, so their
// latencies overlap. Many problems with few splits each take the narrow form
// (kSub = 2, kBatch = 4): few registers, four blocks per SM, many loads in
// flight. Few problems with many splits each take the wide form (kSub = 4,
// kBatch = 8): fewer, longer threads with deep batches.
template <typename A, int kSub, int kBatch, int kMinBlocks>
__global__ void __launch_bounds__(256, kMinBlocks) combine_blocked_kernel(int P, const int32_t* __restrict__ plan,
                                                                          const float* __restrict__ o_part,
                                                                          const float* __restrict__ lse_part,
                                                                          A* __restrict__ o_lat,
                                                                          float* __restrict__ lse) {
  pdl_trigger();
  pdl_wait();
  constexpr int H = 128, D = 512, kParts = 8 / (2 * kSub), kCols = 4 * kSub;
  const int p = blockIdx.x / (16 * kParts), ch = (blockIdx.x / kParts) % 16, part = blockIdx.x % kParts;
  const int h = threadIdx.x & (H - 1), qh = threadIdx.x >> 7;
  const int sub0 = part * 2 * kSub + qh * kSub;  // first 4-column piece of this thread in the chunk
  const PlanView pv = plan_view(plan);
  const int base = pv.pbase[p], count = pv.pcnt[p];
  if (count == 1) return;
  const size_t row = (size_t)p * H + h;
  A* dst = o_lat + row * D + ch * 32 + sub0 * 4;
  const bool lead = (ch == 0 && sub0 == 0);
  float acc[kCols];
#pragma unroll
  for (int e = 0; e < kCols; ++e) acc[e] = 0.f;
  float lse_all = -INFINITY;
  if (count > 0) {
    float m = -INFINITY, wsum = 0.f;
    for (int s0 = 0; s0 < count; s0 += kBatch) {
      float lb[kBatch];
      float4 v[kBatch][kSub];
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        lb[u] = -INFINITY;
#pragma unroll
        for (int q4 = 0; q4 < kSub; ++q4) v[u][q4] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (s0 + u < count) {
          const int s = s0 + u;
          lb[u] = lse_part[(size_t)(base + s) * H + h];
          const float4* src =
              reinterpret_cast<const float4*>(o_part) + ((size_t)(base + s) * 16 + ch) * 8 * H + sub0 * H + h;
#pragma unroll
          for (int q4 = 0; q4 < kSub; ++q4) v[u][q4] = src[q4 * H];
        }
      }
      // Rescale what is accumulated so far to the new running maximum.
      float mb = m;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) mb = fmaxf(mb, lb[u]);
      if (mb == -INFINITY) continue;
      const float r = (m == -INFINITY) ? 0.f : expf(m - mb);
      wsum *= r;
#pragma unroll
      for (int e = 0; e < kCols; ++e) acc[e] *= r;
      m = mb;
#pragma unroll
      for (int u = 0; u < kBatch; ++u) {
        const float wgt = (lb[u] == -INFINITY) ? 0.f : expf(lb[u] - m);
        wsum += wgt;
#pragma unroll
        for (int q4 = 0; q4 < kSub; ++q4) {
          acc[4 * q4] = fmaf(wgt, v[u][q4].x, acc[4 * q4]);
          acc[4 * q4 + 1] = fmaf(wgt, v[u][q4].y, acc[4 * q4 + 1]);
          acc[4 * q4 + 2] = fmaf(wgt, v[u][q4].z, acc[4 * q4 + 2]);
          acc[4 * q4 + 3] = fmaf(wgt, v[u][q4].w, acc[4 * q4 + 3]);
        }
      }
    }
    // o = sum_s e^{lse_s - m} o_s / sum_s e^{lse_s - m};  lse = m + log sum_s e^{lse_s - m}
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
#pragma unroll
    for (int e = 0; e < kCols; ++e) acc[e] *= inv;
    lse_all = (wsum > 0.f) ? m + logf(wsum) : -INFINITY;
  }
  if constexpr (sizeof(A) == 2 && kCols == 4) {
    const A c0 = from_f32<A>(acc[0]), c1 = from_f32<A>(acc[1]), c2 = from_f32<A>(acc[2]), c3 = from_f32<A>(acc[3]);
    *reinterpret_cast<uint2*>(dst) =
        make_uint2((uint32_t)*reinterpret_cast<const uint16_t*>(&c0) |
                       ((uint32_t)*reinterpret_cast<const uint16_t*>(&c1) << 16),
                   (uint32_t)*reinterpret_cast<const uint16_t*>(&c2) |
                       ((uint32_t)*reinterpret_cast<const uint16_t*>(&c3) << 16));
  } else if constexpr (sizeof(A) == 2) {
    uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
    for (int q = 0; q < kCols / 8; ++q) {
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const A lo = from_f32<A>(acc[8 * q + 2 * e]), hi = from_f32<A>(acc[8 * q + 2 * e + 1]);
        w[e] = (uint32_t)*reinterpret_cast<const uint16_t*>(&lo) |
               ((uint32_t)*reinterpret_cast<const uint16_t*>(&hi) << 16);
      }
      d4[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
  } else {
#pragma unroll
    for (int e = 0; e < kCols; ++e) dst[e] = from_f32<A>(acc[e]);
  }
  if (lead) lse[row] = lse_all;
}

template <typename A>
cudaError_t launch_combine(const mla_dims_t& d, int problems, const int32_t* plan,
                           const float* o_part, const float* lse_part, A* o_lat, float* lse,
                           cudaStream_t st, bool blocked, int workers) {
  const int rows = problems * d.n_h;
  if (rows == 0) return cudaSuccess;
  if (blocked) {
    if (d.d_c != 512 || d.n_h != 128) return cudaErrorInvalidValue;
    // A problem holds at most 1 + workers / problems pieces on average.
    if (workers <= 2 * problems)
      return launch_pdl(combine_blocked_kernel<A, 2, 4, 4>, dim3(problems * 32), dim3(256), 0, st, problems, plan,
                        o_part, lse_part, o_lat, lse);
    return launch_pdl(combine_blocked_kernel<A, 1, 8, 4>, dim3(problems * 64), dim3(256), 0, st, problems, plan,
                      o_part, lse_part, o_lat, lse);
  } else if (d.d_c == 512) {
    return launch_pdl(combine_wide_kernel<A>, dim3((rows + 1) / 2), dim3(256), 0, st, problems, d.n_h, plan, o_part,
                      lse_part, o_lat, lse);
  } else if (d.d_c % 128 == 0) {
    return launch_pdl(combine_kernel<A, 4>, dim3((rows + 7) / 8), dim3(256), 0, st, d.n_h, d.d_c, plan, o_part,
                      lse_part, o_lat, lse);
  } else {
    return launch_pdl(combine_kernel<A, 1>, dim3((rows + 7) / 8), dim3(256), 0, st, d.n_h, d.d_c, plan, o_part,
                      lse_part, o_lat, lse);
  }
  return cudaGetLastError();
}

// ====================================================================== W_O output projection
// The W_O GEMM reuses the append's split-K kernel with [W_DKV ; W_KR] = W_O
// (d_model rows, no k_R rows) and h = o viewed as [T][n_h * d_v]; the K splits
// are summed by the kernel below.
template <typename A>
__global__ void __launch_bounds__(256) reduce_splits_kernel(int total, int ksplit, const float* __restrict__ ws,
                                                            A* __restrict__ out) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= total) return;
  float s = 0.f;
  int k = 0;
  for (; k + 4 <= ksplit; k += 4) {
    const float a = ws[(size_t)k * total + i], b = ws[(size_t)(k + 1) * total + i];
    const float c = ws[(size_t)(k + 2) * total + i], d = ws[(size_t)(k + 3) * total + i];
    s += (a + b) + (c + d);
  }
  for (; k < ksplit; ++k) s += ws[(size_t)k * total + i];
  out[i] = from_f32<A>(s);
}

template <typename A>
cudaError_t launch_reduce_splits(int T, int n, int ksplit, const float* ws, A* out, cudaStream_t st) {
  const int total = T * n;
  if (total == 0) return cudaSuccess;
  return launch_pdl(reduce_splits_kernel<A>, dim3((total + 255) / 256), dim3(256), 0, st, total, ksplit, ws, out);
}

int wo_ksplit_simt(const mla_dims_t& d, int T) { return append_ksplit(T, d.d_model, d.n_h * d.d_v); }

template <typename A>
cudaError_t launch_wo_gemm_simt(const mla_dims_t& d, int T, const A* o, const A* w_o, float* ws, int ksplit,
                                cudaStream_t st) {
  const int K = d.n_h * d.d_v;
  const int kchunks = (K + AP_K - 1) / AP_K;
  const int k_per_split = ((kchunks + ksplit - 1) / ksplit) * AP_K;
  dim3 grid((d.d_model + AP_OUT - 1) / AP_OUT, (T + AP_TOK - 1) / AP_TOK, ksplit);
  return launch_pdl(append_gemm_kernel<A>, grid, dim3(256), 0, st, T, d.d_model, 0, K, o, w_o, w_o, k_per_split, ws);
}

// ====================================================================== fp8 codec
__global__ void __launch_bounds__(256) quantize_rows_kernel(const float* __restrict__ x, int cols,
                                                            uint8_t* __restrict__ codes,
                                                            float* __restrict__ scales) {
  pdl_trigger();
  pdl_wait();
  __shared__ float red[32];
  const int r = blockIdx.x;
  const float* xr = x + (size_t)r * cols;
  float m = 0.f;
  for (int c = threadIdx.x; c < cols; c += blockDim.x) m = fmaxf(m, fabsf(xr[c]));
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    float v = threadIdx.x < (blockDim.x >> 5) ? red[threadIdx.x] : 0.f;
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (threadIdx.x == 0) red[0] = v;
  }
  __syncthreads();
  const float sc = e4m3_row_scale(red[0]);
  for (int c = threadIdx.x; c < cols; c += blockDim.x) codes[(size_t)r * cols + c] = f32_to_e4m3(xr[c] / sc);
  if (threadIdx.x == 0) scales[r] = sc;
}

cudaError_t launch_quantize_rows(const float* x, int rows, int cols, uint8_t* codes, float* scales,
                                 cudaStream_t st) {
  if (rows == 0) return cudaSuccess;
  return launch_pdl(quantize_rows_kernel, dim3(rows), dim3(256), 0, st, x, cols, codes, scales);
}

// ====================================================================== instantiations
#define MLA_INST(A)                                                                               \
  template cudaError_t launch_append_simt<A>(const mla_dims_t&, const mla_cache_t&, int, const A*, \
                                             const A*, const A*, const int32_t*, const int32_t*,   \
                                             const int32_t*, int, float*, int, int32_t*,           \
                                             cudaStream_t);                                        \
  template cudaError_t launch_absorb_simt<A>(const mla_dims_t&, int, const A*, const int32_t*,     \
                                             const A*, A*, cudaStream_t);                          \
  template cudaError_t launch_out_proj_simt<A>(const mla_dims_t&, int, const A*, const A*, A*,     \
                                               cudaStream_t);                                      \
  template cudaError_t launch_decode_simt<A>(const mla_dims_t&, const mla_cache_t&, int, int,      \
                                             const A*, const int32_t*, int, const int32_t*, int,   \
                                             float*, float*, A*, float*, int32_t*, cudaStream_t);  \
  template cudaError_t launch_combine<A>(const mla_dims_t&, int, const int32_t*, const float*,     \
                                         const float*, A*, float*, cudaStream_t, bool, int);       \
  template cudaError_t launch_append_epilogue<A>(const mla_dims_t&, const mla_cache_t&, int,       \
                                                 const int32_t*, const int32_t*, const int32_t*,   \
                                                 int, const float*, int, int32_t*, cudaStream_t);  \
  template cudaError_t launch_reduce_splits<A>(int, int, int, const float*, A*, cudaStream_t);     \
  template cudaError_t launch_wo_gemm_simt<A>(const mla_dims_t&, int, const A*, const A*, float*,  \
                                              int, cudaStream_t);
MLA_INST(float)
MLA_INST(__nv_bfloat16)
#undef MLA_INST

}  // namespace mla
