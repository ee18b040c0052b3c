// Chunked prefill in the explicit (non-absorbed) form.
//
// A chunk of C query tokens per sequence attends causally over the sequence's
// cache. The pages form every token's per-head key [W_UK[h] c_t ; k_R,t] and
// value W_UV[h] c_t from the cached latent for training ("MLA 之后，KV cache
// 确实得重新理解一遍", "第一步，训练时"; "MLA 是什么 | dg's Blog", "完整代码"): with
// many queries per sequence that form costs less than absorbing W_UK and W_UV
// into every query (the cost model is mla_prefill_form's). Three steps:
//   1. prefill_gather_kernel: each sequence's cached rows [c_KV | k_R] into a
//      dense bf16 buffer of l_pad rows per sequence (fp8 entries dequantised;
//      the rows up to the next multiple of 128 zeroed), and the queries with
//      their RoPE part rotated at their positions;
//   2. the expansion GEMM (tc_gemm.cu): keys W_UK[h] c_t and values W_UV[h] c_t
//      for every gathered row, bf16 [row][head][128];
//   3. prefill_attn_kernel: flash attention over the formed keys and values,
//      one CTA per (128 queries, head, sequence), S = Q K^T and O += P V on the
//      tensor cores with S and O in tensor memory.
#include "tc_prefill.cuh"
#include "tc_gemm.cuh"
#include "sm100_ptx.cuh"

#include <cuda.h>
#include <math.h>
#include <mutex>

namespace mla {
using namespace ptx;

namespace tcp {
constexpr int kRows = 128;                      // queries per CTA (one per TMEM lane)
constexpr int kTile = 128;                      // keys per tile
constexpr int kDh = 128, kDr = 64, kDv = 128;   // the dims the kernel is built for
constexpr uint32_t kBox = 128 * 128;            // [128 rows x 64 bf16], 128-byte swizzle: 16 KB
constexpr uint32_t OFF_Q = 0;                   // Q: q_nope (2 boxes) and q_rope (1 box)
constexpr uint32_t OFF_K = OFF_Q + 3 * kBox;    // 2 stages of K: k_nope (2 boxes), k_R (1 box)
constexpr uint32_t OFF_V = OFF_K + 6 * kBox;    // V (2 boxes: value columns 0-63, 64-127)
constexpr uint32_t OFF_P = OFF_V + 2 * kBox;    // P bf16 (2 boxes: keys 0-63, 64-127)
constexpr uint32_t OFF_BAR = OFF_P + 2 * kBox;
constexpr uint32_t kSmem = OFF_BAR + 256 + 1024;  // barriers, TMEM address, alignment slack
static_assert(kSmem <= 232448, "shared memory of the prefill attention kernel");
// Tensor memory: two S buffers (128 columns each), then O (128 columns).
constexpr uint32_t TM_S = 0, TM_O = 256, kTmemCols = 512;
enum Bar {
  B_QFULL = 0,
  B_KFULL,                 // + stage
  B_KEMPTY = B_KFULL + 2,  // + stage
  B_VFULL = B_KEMPTY + 2,
  B_VEMPTY,
  B_SFULL,                 // + S buffer
  B_SFREE = B_SFULL + 2,   // + S buffer
  B_PFULL = B_SFREE + 2,
  B_PVDONE,
  B_MMADONE,
  B_COUNT
};
static_assert(B_COUNT * 8 + 8 <= 256, "barrier area");
constexpr uint64_t kWaitNs = 2000000000ull;
// The running maximum is only raised (and O rescaled) when a tile's maximum
// exceeds it by more than this many binary orders: P then stays below 2^8.
constexpr float kRescaleLog2 = 8.f;
}  // namespace tcp

namespace {

__device__ __forceinline__ bool pwait(uint32_t bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && globaltimer() - t0 > tcp::kWaitNs) {
      set_status(status, MLA_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

// Keys visible to the last query of sequence b, clamped to what the buffers hold.
__device__ __forceinline__ int prefill_len(const int32_t* seq_lens, int b, int max_len) {
  return min(max(seq_lens[b], 0), max_len);
}

// Byte offset of 16-byte unit u (8 bf16) of row r in a [rows x 64] bf16 box
// with the 128-byte swizzle (8-row groups of 1024 bytes, unit index XOR row % 8).
__device__ __forceinline__ uint32_t swz128(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

}  // namespace

// One warp per gathered row (sequence blockIdx.y, position blockIdx.x * 8 + warp).
// Rows [len, roundup(len, 128)) are zeroed so that the last key tile holds
// finite values; rows past that are never read and not written.
__global__ void __launch_bounds__(256) prefill_gather_kernel(int l_pad, int max_len, int d_c, int d_rope,
                                                             int page_size, int max_pages, int64_t num_pages,
                                                             int fp8, const void* __restrict__ ckv,
                                                             const __nv_bfloat16* __restrict__ kr,
                                                             const float* __restrict__ scale,
                                                             const int32_t* __restrict__ bt,
                                                             const int32_t* __restrict__ seq_lens,
                                                             __nv_bfloat16* __restrict__ lat, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int b = blockIdx.y, t = blockIdx.x * 8 + warp;
  if (t == 0 && lane == 0 && seq_lens[b] > max_len) set_status(status, MLA_ERR_INVALID_ARG);
  const int len = prefill_len(seq_lens, b, max_len);
  if (t >= ((len + tcp::kTile - 1) & ~(tcp::kTile - 1))) return;
  const int row_elems = d_c + d_rope, chunks = row_elems / 8;
  uint4* dst = reinterpret_cast<uint4*>(lat + ((size_t)b * l_pad + t) * row_elems);
  int64_t slot = -1;
  if (t < len) {
    const int pg = bt[(size_t)b * max_pages + t / page_size];
    if (pg < 0 || pg >= num_pages) {
      if (lane == 0) set_status(status, MLA_ERR_BAD_PAGE);
    } else {
      slot = (int64_t)pg * page_size + t % page_size;
    }
  }
  if (slot < 0) {
    for (int i = lane; i < chunks; i += 32) dst[i] = make_uint4(0, 0, 0, 0);
    return;
  }
  if (!fp8) {
    const uint4* src = reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(ckv) + slot * row_elems);
    for (int i = lane; i < chunks; i += 32) dst[i] = src[i];
    return;
  }
  // fp8 cache: c = code * scale, rounded to bf16; k_R copied.
  const float sc = scale[slot];
  const uint8_t* codes = reinterpret_cast<const uint8_t*>(ckv) + slot * d_c;
  for (int i = lane; i < d_c / 8; i += 32) {
    const uint2 cw = *reinterpret_cast<const uint2*>(codes + i * 8);
    const uint32_t w2[2] = {cw.x, cw.y};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
#pragma unroll
      for (int hf = 0; hf < 2; ++hf) {
        const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(w2[k] >> (16 * hf)), __NV_E4M3);
        const float2 f2 = __half22float2(__half2(hr));
        const __nv_bfloat162 b2 = __floats2bfloat162_rn(f2.x * sc, f2.y * sc);
        o[2 * k + hf] = *reinterpret_cast<const uint32_t*>(&b2);
      }
    }
    dst[i] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  const uint4* ksrc = reinterpret_cast<const uint4*>(kr + slot * d_rope);
  for (int i = lane; i < d_rope / 8; i += 32) dst[d_c / 8 + i] = ksrc[i];
}

// One warp per (query row, head): q_nope copied, q_rope rotated at the query's
// position seq_lens[b] - C + j (RoPE of interleaved pairs, as the cache's k_R).
// A query at a negative position sees no key; its rotation uses position 0.
__global__ void __launch_bounds__(256) prefill_rope_q_kernel(int T, int C, int n_h, int max_len, RopeFreqs freqs,
                                                             const int32_t* __restrict__ seq_lens,
                                                             const __nv_bfloat16* __restrict__ q,
                                                             __nv_bfloat16* __restrict__ q_rot) {
  pdl_trigger();
  pdl_wait();
  const int item = blockIdx.x * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (item >= T * n_h) return;
  const int row = item / n_h;
  const int b = row / C, j = row % C;
  const int pos = max(prefill_len(seq_lens, b, max_len) - C + j, 0);
  constexpr int dq = tcp::kDh + tcp::kDr;
  const __nv_bfloat16* src = q + (size_t)item * dq;
  __nv_bfloat16* dst = q_rot + (size_t)item * dq;
  if (lane < tcp::kDh / 8)
    reinterpret_cast<uint4*>(dst)[lane] = reinterpret_cast<const uint4*>(src)[lane];
  // 32 pairs of the RoPE part, one per lane.
  const __nv_bfloat162 x = reinterpret_cast<const __nv_bfloat162*>(src + tcp::kDh)[lane];
  float c, s;
  rope_cos_sin(pos, freqs.hi[lane], freqs.lo[lane], &c, &s);
  const float x0 = __low2float(x), x1 = __high2float(x);
  reinterpret_cast<__nv_bfloat162*>(dst + tcp::kDh)[lane] = __floats2bfloat162_rn(x0 * c - x1 * s, x0 * s + x1 * c);
}

namespace {
struct PrefillArgs {
  int C, n_h, l_pad, max_len;
  float scale_log2;  // softmax_scale * log2(e)
  const int32_t* seq_lens;
  __nv_bfloat16* o;
  float* lse;
  int32_t* status;
};
}  // namespace

// Flash attention of 128 queries of one head of one sequence over the formed
// keys and values, causal. Roles (256 threads):
//   warp 0 lane 0  TMA: Q once, then per key tile j K_j (two stages, k_nope from
//                  the formed keys and k_R from the gathered rows) and V_j (one
//                  stage; V_j is requested once P.V of tile j-1 has completed)
//   warp 1         TMEM allocation; lane 0 issues the MMAs: S_j = Q K_j^T into
//                  S buffer j % 2, then O += P_{j-1} V_{j-1}, so that S_{j}
//                  runs while the softmax of tile j-1 is computed
//   warps 4-7      softmax, one query row per thread (TMEM lane = row): scores
//                  of tile j scaled to base 2 and masked past the row's
//                  position; the running maximum is raised only when a tile
//                  exceeds it by more than 2^8, and then O is rescaled in
//                  TMEM; P (bf16) goes to shared memory as the A operand of
//                  P.V. At the end O / l and the log-sum-exp are stored.
// Every wait is bounded (2 s); a timeout sets MLA_ERR_DEVICE_TIMEOUT in the
// status word and every role leaves its loop.
__global__ void __launch_bounds__(256, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_v,
                    PrefillArgs a) {
  using namespace tcp;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto BAR = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 8 * B_COUNT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qb = (int)gridDim.x - 1 - (int)blockIdx.x;  // the longest query blocks start first
  const int h = blockIdx.y, b = blockIdx.z;
  pdl_trigger();
  if (threadIdx.x == 0) {
    mbar_init(BAR(B_QFULL), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(B_KFULL + s), 1);
      mbar_init(BAR(B_KEMPTY + s), 1);
      mbar_init(BAR(B_SFULL + s), 1);
      mbar_init(BAR(B_SFREE + s), 4);
    }
    mbar_init(BAR(B_VFULL), 1);
    mbar_init(BAR(B_VEMPTY), 1);
    mbar_init(BAR(B_PFULL), 4);
    mbar_init(BAR(B_PVDONE), 1);
    mbar_init(BAR(B_MMADONE), 1);
    fence_mbar_init_cluster();
    prefetch_tmap(&tm_q);
    prefetch_tmap(&tm_k);
    prefetch_tmap(&tm_kr);
    prefetch_tmap(&tm_v);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  pdl_wait();  // the gathered rows, formed keys/values and rotated queries come from the previous kernels

  const int len = prefill_len(a.seq_lens, b, a.max_len);
  const int q0 = qb * kRows;                 // this CTA's first query of the chunk
  const int nq = min(kRows, a.C - q0);       // its valid queries
  const int pos0 = len - a.C + q0;           // position of its first query
  const int pos_max = pos0 + nq - 1;
  const int n = pos_max < 0 ? 0 : pos_max / kTile + 1;  // key tiles any of its queries sees
  const int krow0 = b * a.l_pad;

  if (warp == 0 && lane == 0 && n > 0) {
    // ------------------------------------------------------------ TMA producer
    bool ok = true;
    const int qy = b * a.C + q0;
    mbar_arrive_expect_tx(BAR(B_QFULL), 3 * kBox);
    for (int c = 0; c < 3; ++c) tma_load_2d(base + OFF_Q + c * kBox, &tm_q, h * (kDh + kDr) + 64 * c, qy, BAR(B_QFULL));
    auto load_k = [&](int j) {
      const int s = j & 1, y = krow0 + j * kTile;
      const uint32_t dst = base + OFF_K + s * 3 * kBox;
      mbar_arrive_expect_tx(BAR(B_KFULL + s), 3 * kBox);
      tma_load_2d(dst, &tm_k, h * kDh, y, BAR(B_KFULL + s));
      tma_load_2d(dst + kBox, &tm_k, h * kDh + 64, y, BAR(B_KFULL + s));
      tma_load_2d(dst + 2 * kBox, &tm_kr, 0, y, BAR(B_KFULL + s));
    };
    load_k(0);
    int k_issued = 1, v_issued = 0;
    for (int j = 0; j < n; ++j) {
      if (j + 1 < n) {
        if (j + 1 >= 2 && !pwait(BAR(B_KEMPTY + ((j + 1) & 1)), (((j + 1) >> 1) - 1) & 1, a.status)) {
          ok = false;
          break;
        }
        load_k(j + 1);
        ++k_issued;
      }
      if (j >= 1 && !pwait(BAR(B_VEMPTY), (j - 1) & 1, a.status)) {
        ok = false;
        break;
      }
      mbar_arrive_expect_tx(BAR(B_VFULL), 2 * kBox);
      tma_load_2d(base + OFF_V, &tm_v, h * kDv, krow0 + j * kTile, BAR(B_VFULL));
      tma_load_2d(base + OFF_V + kBox, &tm_v, h * kDv + 64, krow0 + j * kTile, BAR(B_VFULL));
      ++v_issued;
    }
    (void)ok;
    // Every copy issued has landed before this thread leaves (instant on the
    // normal path, where the MMAs consumed them all).
    pwait(BAR(B_QFULL), 0, a.status);
    for (int s = 0; s < 2; ++s) {
      const int cnt = (k_issued - s + 1) / 2;  // loads into stage s: tiles s, s + 2, ...
      if (cnt > 0) pwait(BAR(B_KFULL + s), (cnt - 1) & 1, a.status);
    }
    if (v_issued > 0) pwait(BAR(B_VFULL), (v_issued - 1) & 1, a.status);
  } else if (warp == 1 && lane == 0 && n > 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kDv, false, true);
    auto pv = [&](int i) -> bool {
      if (!pwait(BAR(B_PFULL), i & 1, a.status) || !pwait(BAR(B_VFULL), i & 1, a.status)) return false;
      tc_fence_after();
      // A = P [128 queries x 128 keys] (K-major, two 64-key boxes); B = V
      // [128 keys x 128 values], MN-major (two 64-value boxes, 16 KB apart).
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_f16(tmem + TM_O, smem_desc(base + OFF_P + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024, kSwizzle128B),
                smem_desc(base + OFF_V + kk * 2048, kBox, 1024, kSwizzle128B), idesc_pv,
                (i > 0 || kk > 0) ? 1u : 0u);
      mma_commit(BAR(B_VEMPTY));
      mma_commit(BAR(B_PVDONE));
      return true;
    };
    bool ok = pwait(BAR(B_QFULL), 0, a.status);
    for (int j = 0; ok && j < n; ++j) {
      const int s = j & 1;
      if (!pwait(BAR(B_KFULL + s), (j >> 1) & 1, a.status) ||
          (j >= 2 && !pwait(BAR(B_SFREE + s), ((j >> 1) - 1) & 1, a.status))) {
        ok = false;
        break;
      }
      tc_fence_after();
      const uint32_t kb = base + OFF_K + s * 3 * kBox;
      // S_j = Q K_j^T over 192 = three 64-wide boxes (q_nope . k_nope, then q_R . k_R).
#pragma unroll
      for (int c = 0; c < 3; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem + TM_S + s * kTile, smem_desc(base + OFF_Q + c * kBox + kk * 32, 16, 1024, kSwizzle128B),
                  smem_desc(kb + c * kBox + kk * 32, 16, 1024, kSwizzle128B), idesc_s, (c | kk) ? 1u : 0u);
      mma_commit(BAR(B_KEMPTY + s));
      mma_commit(BAR(B_SFULL + s));
      if (j >= 1 && !pv(j - 1)) ok = false;
    }
    if (ok) pv(n - 1);
    // Every MMA issued has completed before TMEM is released.
    mma_commit(BAR(B_MMADONE));
    pwait(BAR(B_MMADONE), 0, a.status);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax and epilogue
    const int qd = warp - 4, r = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const int pos = pos0 + r;
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      const int s = j & 1;
      ok = __all_sync(0xffffffffu, pwait(BAR(B_SFULL + s), (j >> 1) & 1, a.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_base + TM_S + s * kTile + cc * 32, v[cc]);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_SFREE + s));
      // Base-2 scores; keys past the row's position are masked (only tiles
      // that reach past the warp's first position need the test).
      const int kbase = j * kTile;
      const bool need_mask = kbase + kTile - 1 > pos0 + qd * 32;
      float mx = -INFINITY;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          float t = __uint_as_float(v[cc][x]) * a.scale_log2;
          if (need_mask && kbase + cc * 32 + x > pos) t = -INFINITY;
          v[cc][x] = __float_as_uint(t);
          mx = fmaxf(mx, t);
        }
      const bool upd = mx > m_run + kRescaleLog2;
      const float m_new = upd ? mx : m_run;
      const float fac = upd ? ex2_approx(m_run - m_new) : 1.f;  // 0 while nothing was seen
      const float mref = (m_new == -INFINITY) ? 0.f : m_new;
      uint32_t pk[64];
      float sum = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc)
#pragma unroll
        for (int x2 = 0; x2 < 16; ++x2) {
          const float p0 = ex2_approx(__uint_as_float(v[cc][2 * x2]) - mref);
          const float p1 = ex2_approx(__uint_as_float(v[cc][2 * x2 + 1]) - mref);
          sum += p0 + p1;
          const __nv_bfloat162 p2 = __floats2bfloat162_rn(p0, p1);
          pk[cc * 16 + x2] = *reinterpret_cast<const uint32_t*>(&p2);
        }
      l = l * fac + sum;
      m_run = m_new;
      if (j >= 1) {
        // P.V of tile j-1 has completed: P's buffer is free and O may be rescaled.
        ok = __all_sync(0xffffffffu, pwait(BAR(B_PVDONE), (j - 1) & 1, a.status));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, upd)) {
#pragma unroll 1
          for (int cc = 0; cc < 4; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + TM_O + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * fac);
            tmem_st32(tmem + lane_base + TM_O + cc * 32, o);
          }
          tmem_wait_st();
        }
      }
      uint8_t* pbuf = gbase + OFF_P;
#pragma unroll
      for (int u = 0; u < 16; ++u)
        *reinterpret_cast<uint4*>(pbuf + (u >> 3) * kBox + swz128(r, u & 7)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PFULL));
    }
    if (ok && n > 0) ok = __all_sync(0xffffffffu, pwait(BAR(B_PVDONE), (n - 1) & 1, a.status));
    if (ok) {
      tc_fence_after();
      const bool valid = r < nq;
      const size_t row = (size_t)b * a.C + q0 + r;
      const float inv = l > 0.f ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(a.o + (row * a.n_h + h) * kDv);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(tmem + lane_base + TM_O + cc * 32, o);
          tmem_wait_ld();
        } else {
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = 0u;
        }
        uint32_t w[16];
#pragma unroll
        for (int x2 = 0; x2 < 16; ++x2) {
          const __nv_bfloat162 h2 =
              __floats2bfloat162_rn(__uint_as_float(o[2 * x2]) * inv, __uint_as_float(o[2 * x2 + 1]) * inv);
          w[x2] = *reinterpret_cast<const uint32_t*>(&h2);
        }
        if (valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[cc * 4 + u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if (valid) a.lse[row * a.n_h + h] = l > 0.f ? (m_run + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ====================================================================== host side
bool tc_prefill_supported(const mla_dims_t& d) {
  return d.act_dtype == MLA_BF16 && (d.cache_dtype == MLA_BF16 || d.cache_dtype == MLA_FP8_E4M3) &&
         d.d_h == tcp::kDh && d.d_v == tcp::kDv && d.d_rope == tcp::kDr && d.d_c >= 64 && d.d_c % 64 == 0 &&
         tc_device_ok();
}


PrefillWs prefill_ws_layout(const mla_dims_t& d, int B, int C, int max_seq_len) {
  PrefillWs w = {};
  w.l_pad = (max_seq_len > 0 ? (max_seq_len + tcp::kTile - 1) / tcp::kTile : 1) * tcp::kTile;
  const size_t rows = (size_t)B * w.l_pad;
  w.lat_off = 0;
  w.k_off = w.lat_off + align256(rows * (d.d_c + d.d_rope) * 2);
  w.v_off = w.k_off + align256(rows * d.n_h * d.d_h * 2);
  w.q_off = w.v_off + align256(rows * d.n_h * d.d_v * 2);
  w.total = w.q_off + align256((size_t)B * C * d.n_h * (d.d_h + d.d_rope) * 2);
  return w;
}

// Visible (query, key) pairs of C queries at the end of a sequence of L tokens.
static double prefill_pairs(int C, int64_t L) {
  double pairs = 0;
  for (int j = 0; j < C; ++j) {
    const int64_t vis = L - C + j + 1;
    if (vis > 0) pairs += (double)vis;
  }
  return pairs;
}

double prefill_flops_explicit(const mla_dims_t& d, int C, int64_t L) {
  return 2.0 * d.n_h * (d.d_h + d.d_v) * d.d_c * (double)L +
         2.0 * d.n_h * (d.d_h + d.d_rope + d.d_v) * prefill_pairs(C, L);
}

double prefill_flops_absorbed(const mla_dims_t& d, int C, int64_t L) {
  return 2.0 * d.n_h * (d.d_h + d.d_v) * d.d_c * (double)C +
         2.0 * d.n_h * (2.0 * d.d_c + d.d_rope) * prefill_pairs(C, L);
}

cudaError_t launch_prefill(const mla_dims_t& d, const mla_cache_t& c, int B, int C, int max_seq_len,
                           const __nv_bfloat16* q, const __nv_bfloat16* w_uk, const __nv_bfloat16* w_uv,
                           const int32_t* bt, int max_pages, const int32_t* seq_lens, void* ws,
                           __nv_bfloat16* o, float* lse, int32_t* status, cudaStream_t st) {
  using namespace tcp;
  const PrefillWs L = prefill_ws_layout(d, B, C, max_seq_len);
  uint8_t* w8 = reinterpret_cast<uint8_t*>(ws);
  __nv_bfloat16* lat = reinterpret_cast<__nv_bfloat16*>(w8 + L.lat_off);
  __nv_bfloat16* kbuf = reinterpret_cast<__nv_bfloat16*>(w8 + L.k_off);
  __nv_bfloat16* vbuf = reinterpret_cast<__nv_bfloat16*>(w8 + L.v_off);
  __nv_bfloat16* q_rot = reinterpret_cast<__nv_bfloat16*>(w8 + L.q_off);
  const int max_len = std::min<int64_t>(max_seq_len, (int64_t)max_pages * d.page_size);
  const int rows = B * L.l_pad, T = B * C;
  const int fp8 = d.cache_dtype == MLA_FP8_E4M3 ? 1 : 0;

  cudaError_t e = launch_pdl(prefill_gather_kernel, dim3(L.l_pad / 8, B), dim3(256), 0, st, L.l_pad, max_len, d.d_c,
                             d.d_rope, d.page_size, max_pages, (int64_t)c.num_pages, fp8, (const void*)c.ckv,
                             (const __nv_bfloat16*)c.kr, (const float*)c.scale, bt, seq_lens, lat, status);
  if (e != cudaSuccess) return e;
  const int items = T * d.n_h;
  e = launch_pdl(prefill_rope_q_kernel, dim3((items + 7) / 8), dim3(256), 0, st, T, C, d.n_h, max_len,
                 rope_freqs(d.d_rope, d.rope_theta), seq_lens, q, q_rot);
  if (e != cudaSuccess) return e;
  e = launch_tc_expand_kv(d, rows, L.l_pad, max_len, seq_lens, lat, w_uk, w_uv, kbuf, vbuf, status, st);
  if (e != cudaSuccess) return e;

  CUtensorMap tm_q, tm_k, tm_kr, tm_v;
  const uint64_t dq = (uint64_t)d.n_h * (kDh + kDr), dkv = (uint64_t)d.n_h * kDh;
  if (!tc_map2d_bf16(&tm_q, q_rot, dq, (uint64_t)T, dq, kRows) ||
      !tc_map2d_bf16(&tm_k, kbuf, dkv, (uint64_t)rows, dkv, kTile) ||
      !tc_map2d_bf16(&tm_kr, lat + d.d_c, kDr, (uint64_t)rows, (uint64_t)(d.d_c + d.d_rope), kTile) ||
      !tc_map2d_bf16(&tm_v, vbuf, dkv, (uint64_t)rows, dkv, kTile))
    return cudaErrorInvalidValue;
  PrefillArgs a;
  a.C = C;
  a.n_h = d.n_h;
  a.l_pad = L.l_pad;
  a.max_len = max_len;
  a.scale_log2 = d.softmax_scale * 1.4426950408889634f;
  a.seq_lens = seq_lens;
  a.o = o;
  a.lse = lse;
  a.status = status;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)kSmem);
  });
  if (attr != cudaSuccess) return attr;
  return launch_pdl(prefill_attn_kernel, dim3((C + kRows - 1) / kRows, d.n_h, B), dim3(256), kSmem, st, tm_q, tm_k,
                    tm_kr, tm_v, a);
}

}  // namespace mla
