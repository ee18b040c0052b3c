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
//      the rows up to the next multiple of 128 zeroed);
//   2. prefill_expand_kernel: keys W_UK[h] c_t and values W_UV[h] c_t for every
//      gathered row, bf16 [row][head][128], on the tensor cores;
//   3. prefill_attn_kernel: flash attention over the formed keys and values,
//      one CTA per (256 queries, head, sequence) as two tiles of 128 whose
//      softmaxes take turns: the queries' RoPE part is rotated in shared
//      memory, S = Q K^T and O += P V run on the tensor cores with S, P and O
//      in tensor memory.
#include "tc_prefill.cuh"
#include "tc_gemm.cuh"
#include "sm100_ptx.cuh"

#include <cuda.h>
#include <math.h>
#include <algorithm>
#include <atomic>
#include <mutex>

namespace mla {
using namespace ptx;

namespace tcp {
constexpr int kRows = 128;                      // queries per tile (one per TMEM lane)
constexpr int kTile = 128;                      // keys per tile
constexpr int kDh = 128, kDr = 64, kDv = 128;   // the dims the kernels are built for
constexpr uint32_t kBox = 128 * 128;            // [128 rows x 64 bf16], 128-byte swizzle: 16 KB
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

__device__ __forceinline__ float max3f(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (d0, d1) = (a0, a1) * b + c, one instruction on the paired fp32 pipe.
__device__ __forceinline__ void fma_x2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n"
      " mov.b64 rc, {%5, %5};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) += (a0, a1), one instruction on the paired fp32 pipe.
__device__ __forceinline__ void add_x2(float& d0, float& d1, float a0, float a1) {
  asm("{\n .reg .b64 ra, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rd, {%0, %1};\n"
      " add.rn.f32x2 rd, rd, ra;\n mov.b64 {%0, %1}, rd;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}
// Maximum of 32 raw scores by three-input max instructions.
__device__ __forceinline__ float max_of32(const uint32_t (&v)[32]) {
  float m[12];
#pragma unroll
  for (int x = 0; x < 10; ++x)
    m[x] = max3f(__uint_as_float(v[3 * x]), __uint_as_float(v[3 * x + 1]), __uint_as_float(v[3 * x + 2]));
  m[10] = __uint_as_float(v[30]);
  m[11] = __uint_as_float(v[31]);
#pragma unroll
  for (int x = 0; x < 4; ++x) m[x] = max3f(m[3 * x], m[3 * x + 1], m[3 * x + 2]);
  return max3f(m[0], m[1], fmaxf(m[2], m[3]));
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
                                                             const int32_t* __restrict__ seq_start,
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
  // Positions before the window are never read from the cache (their pages
  // may be gone): they stay zero, like the rows past the end.
  const int lo = seq_start != nullptr ? min(max(seq_start[b], 0), len) : 0;
  int64_t slot = -1;
  if (t < len && t >= lo) {
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

// cos/sin of RoPE angle pos * theta^(-2i/d_rope) for every position below
// max_len and pair i (one thread each), for the queries' rotation.
__global__ void __launch_bounds__(256) prefill_rope_table_kernel(int max_len, int pairs, RopeFreqs freqs,
                                                                 float2* __restrict__ tab) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= max_len * pairs) return;
  const int pos = i / pairs, pr = i % pairs;
  float c, sn;
  rope_cos_sin(pos, freqs.hi[pr], freqs.lo[pr], &c, &sn);
  tab[i] = make_float2(c, sn);
}

namespace tce {
constexpr int kTok = 128;                   // gathered rows per CTA (MMA M, TMEM lanes)
constexpr int kN = 256;                     // outputs per head: W_UK[h] rows, then W_UV[h] rows
constexpr int kMaxChunks = 8;               // d_c / 64 <= 8
constexpr int kStages = 3;                  // weight ring
constexpr uint32_t kABox = 128 * 128;       // [128 rows x 64 bf16], 128-byte swizzle: 16 KB
constexpr uint32_t kWChunk = 256 * 128;     // [256 weight rows x 64 bf16]: 32 KB
constexpr uint32_t OFF_A = 0;
constexpr uint32_t OFF_W = OFF_A + kMaxChunks * kABox;
constexpr uint32_t OFF_BAR = OFF_W + kStages * kWChunk;
constexpr uint32_t kSmem = OFF_BAR + 128 + 1024;
static_assert(kSmem <= 232448, "shared memory of the expansion kernel");
enum Bar { B_AFULL = 0, B_WFULL, B_WEMPTY = B_WFULL + kStages, B_DFULL = B_WEMPTY + kStages, B_DEMPTY = B_DFULL + 2,
           B_MMADONE = B_DEMPTY + 2, B_COUNT };
static_assert(B_COUNT * 8 + 8 <= 128, "barrier area");
}  // namespace tce

// Keys and values of `hpc` heads for 128 gathered rows:
//   out[r][h] = [W_UK[h] c_r | W_UV[h] c_r]  (D[128 rows x 256] = C[128 x d_c] . [W_UK[h]; W_UV[h]]^T)
// Two CTAs of a cluster take adjacent 128-row tiles of one sequence and the
// same heads. Each row tile's latent stays in its CTA's shared memory for all
// heads; the weight rows stream through a 3-stage ring, each CTA loading one
// half of every chunk (W_UK's rows or W_UV's) by TMA multicast into both CTAs,
// so the weights cross from L2 once per pair. A stage is reused once both
// CTAs' MMAs have released it (a multicast commit to both). Two TMEM
// accumulators of 256 columns alternate between heads, so the store of one
// head's results (warps 4-7, one row per thread) overlaps the MMAs of the
// next. A pair whose first tile starts at or past its sequence's length is
// skipped; a second tile past the length computes but stores nothing.
__global__ void __launch_bounds__(256, 1)
prefill_expand_kernel(const __grid_constant__ CUtensorMap tm_lat, const __grid_constant__ CUtensorMap tm_wuk,
                      const __grid_constant__ CUtensorMap tm_wuv, int n_h, int hpc, int k_chunks, int l_pad,
                      int max_len, const int32_t* __restrict__ seq_lens, const int32_t* __restrict__ seq_start,
                      __nv_bfloat16* __restrict__ k_out, __nv_bfloat16* __restrict__ v_out, int32_t* status) {
  using namespace tce;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  auto BAR = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 8 * B_COUNT);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int row0 = blockIdx.x * kTok, h0 = blockIdx.y * hpc;
  pdl_trigger();
  pdl_wait();  // the gathered rows come from the previous kernel
  const int b = row0 / l_pad;
  const int len = prefill_len(seq_lens, b, max_len);
  // Cluster-uniform: the pair's tiles decide (both lie in one sequence); a pair
  // wholly past the end or wholly before the window holds nothing that is read.
  const int pair0 = (int)(blockIdx.x & ~1u) * kTok - b * l_pad;
  const int lo = seq_start != nullptr ? min(max(seq_start[b], 0), len) : 0;
  if (pair0 >= len || pair0 + 2 * kTok <= lo) return;
  const bool store_rows = row0 - b * l_pad < len;
  const int nh = min(hpc, n_h - h0);
  if (threadIdx.x == 0) {
    mbar_init(BAR(B_AFULL), 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(BAR(B_WFULL + s), 1);
      mbar_init(BAR(B_WEMPTY + s), 2);  // released by both CTAs' MMAs
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(B_DFULL + i), 1);
      mbar_init(BAR(B_DEMPTY + i), 4);
    }
    mbar_init(BAR(B_MMADONE), 1);
    fence_mbar_init_cluster();
    prefetch_tmap(&tm_lat);
    prefetch_tmap(&tm_wuk);
    prefetch_tmap(&tm_wuv);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();  // both CTAs' barriers exist before any multicast or remote commit
  cluster_wait();
  const uint32_t tmem = *tmem_slot;
  const int n_chunks = nh * k_chunks;

  if (warp == 0 && lane == 0) {
    // ------------------------------------------------------------ TMA producer
    mbar_arrive_expect_tx(BAR(B_AFULL), k_chunks * kABox);
    for (int kc = 0; kc < k_chunks; ++kc) tma_load_2d(base + OFF_A + kc * kABox, &tm_lat, kc * 64, row0, BAR(B_AFULL));
    int issued = 0;
    for (int i = 0; i < n_chunks; ++i) {
      const int s = i % kStages, h = h0 + i / k_chunks, kc = i % k_chunks;
      if (i >= kStages && !pwait(BAR(B_WEMPTY + s), ((i / kStages) - 1) & 1, status)) break;
      const uint32_t dst = base + OFF_W + s * kWChunk;
      mbar_arrive_expect_tx(BAR(B_WFULL + s), kWChunk);
      if (rank == 0) tma_load_2d_mc(dst, &tm_wuk, kc * 64, h * tcp::kDh, BAR(B_WFULL + s), 0x3);
      else tma_load_2d_mc(dst + kWChunk / 2, &tm_wuv, kc * 64, h * tcp::kDv, BAR(B_WFULL + s), 0x3);
      ++issued;
    }
    // Every copy into this CTA has landed before it leaves.
    pwait(BAR(B_AFULL), 0, status);
    for (int s = 0; s < kStages; ++s) {
      const int cnt = (issued - s + kStages - 1) / kStages;
      if (cnt > 0) pwait(BAR(B_WFULL + s), (cnt - 1) & 1, status);
    }
  } else if (warp == 1 && lane == 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc = idesc_bf16_f32(kTok, kN, false, false);
    bool ok = pwait(BAR(B_AFULL), 0, status);
    for (int hi = 0; ok && hi < nh; ++hi) {
      const int buf = hi & 1;
      if (hi >= 2 && !pwait(BAR(B_DEMPTY + buf), ((hi >> 1) - 1) & 1, status)) break;
      tc_fence_after();
      for (int kc = 0; kc < k_chunks; ++kc) {
        const int i = hi * k_chunks + kc, s = i % kStages;
        if (!pwait(BAR(B_WFULL + s), (i / kStages) & 1, status)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = base + OFF_A + kc * kABox, w = base + OFF_W + s * kWChunk;
#pragma unroll
        for (int k16 = 0; k16 < 4; ++k16)
          mma_f16(tmem + buf * kN, smem_desc(a + k16 * 32, 16, 1024, kSwizzle128B),
                  smem_desc(w + k16 * 32, 16, 1024, kSwizzle128B), idesc, (kc | k16) ? 1u : 0u);
        mma_commit_multicast(BAR(B_WEMPTY + s), 0x3);  // the stage is free in both CTAs' view
      }
      if (ok) mma_commit(BAR(B_DFULL + buf));
    }
    mma_commit(BAR(B_MMADONE));
    pwait(BAR(B_MMADONE), 0, status);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ epilogue: one gathered row per thread
    const int qd = warp - 4, r = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const size_t orow = ((size_t)row0 + r) * n_h;
    for (int hi = 0; hi < nh; ++hi) {
      const int buf = hi & 1, h = h0 + hi;
      if (!__all_sync(0xffffffffu, pwait(BAR(B_DFULL + buf), (hi >> 1) & 1, status))) break;
      tc_fence_after();
      // Each half (keys, then values: 128 columns) is read with four loads in
      // flight and one wait; the accumulator is released as soon as the second
      // half is in registers, before its stores.
#pragma unroll 1
      for (int half = 0; half < 2; ++half) {
        uint4* dst = reinterpret_cast<uint4*>((half ? v_out : k_out) + (orow + h) * tcp::kDh);
        uint32_t v[4][32];
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) tmem_ld32(tmem + lane_base + buf * kN + half * 128 + cc * 32, v[cc]);
        tmem_wait_ld();
        if (half == 1) {
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(BAR(B_DEMPTY + buf));
        }
        if (!store_rows) continue;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t w[16];
#pragma unroll
          for (int x2 = 0; x2 < 16; ++x2) {
            const __nv_bfloat162 b2 =
                __floats2bfloat162_rn(__uint_as_float(v[cc][2 * x2]), __uint_as_float(v[cc][2 * x2 + 1]));
            w[x2] = *reinterpret_cast<const uint32_t*>(&b2);
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) dst[cc * 4 + u] = make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
  // Neither CTA leaves while the other may still deliver a weight half or a
  // stage release into it.
  cluster_arrive();
  cluster_wait();
}

namespace {
struct PrefillArgs {
  int C, n_h, l_pad, max_len;
  float scale_log2;  // softmax_scale * log2(e)
  const int32_t* seq_start;  // first visible position per sequence, or null
  const float2* rope;  // [max_len][d_rope / 2] (cos, sin) of each position and pair
  const int32_t* seq_lens;
  __nv_bfloat16* o;
  float* lse;
  int32_t* status;
};
}  // namespace

namespace tcq {
// Two query tiles per CTA (256 queries of one head of one sequence), each with
// its own S and O accumulators and softmax warps, sharing every key and value
// tile: while one tile's softmax runs, the tensor pipe works on the other's
// MMAs.
constexpr int kRows = tcp::kRows, kTile = tcp::kTile, kDh = tcp::kDh, kDr = tcp::kDr, kDv = tcp::kDv;
constexpr uint32_t kBox = tcp::kBox;
constexpr uint32_t OFF_Q = 0;                   // Q of tile g at OFF_Q + 3 g kBox: q_nope (2 boxes), q_rope (1 box)
constexpr uint32_t OFF_K = OFF_Q + 6 * kBox;    // 2 stages of K: k_nope (2 boxes), k_R (1 box)
constexpr uint32_t OFF_V = OFF_K + 6 * kBox;    // V (2 boxes: value columns 0-63, 64-127)
constexpr uint32_t OFF_BAR = OFF_V + 2 * kBox;
constexpr uint32_t kSmem = OFF_BAR + 256 + 1024;
static_assert(kSmem <= 232448, "shared memory of the two-tile prefill attention kernel");
// Tensor memory: S of tile g at 128 g (P of tile g, bf16, over its first 64
// columns once the scores are read), O of tile g at 256 + 128 g.
constexpr uint32_t TM_S = 0, TM_O = 256, kTmemCols = 512;
constexpr int kThreads = 384;
enum Bar {
  B_QFULL = 0,
  B_QROT,                  // both tiles' RoPE parts are rotated (count: the 10 rotating warps)
  B_KFULL,                 // + stage
  B_KEMPTY = B_KFULL + 2,  // + stage: S of both tiles for the stage's key tile is done
  B_VFULL = B_KEMPTY + 2,
  B_VEMPTY,
  B_SFULL,                 // + tile
  B_PFULL = B_SFULL + 2,   // + tile (count 4)
  B_PVDONE = B_PFULL + 2,  // + tile
  B_MMADONE = B_PVDONE + 2,
  B_COUNT
};
static_assert(B_COUNT * 8 + 8 <= 256, "barrier area");
}  // namespace tcq

// Flash attention of 256 queries (two tiles of 128, A and B) of one head of one
// sequence over the formed keys and values, causal. Roles (384 threads):
//   warp 0 lane 0  TMA: Q of both tiles once, then per key tile j K_j (two
//                  stages) and V_j (one stage, requested once P.V of both tiles
//                  for tile j-1 is done)
//   warp 1         TMEM allocation; lane 0 issues the MMAs in the order S_A(0),
//                  S_B(0), then per j: P_A(j) V_j, S_A(j+1), P_B(j) V_j,
//                  S_B(j+1). S_g(j+1) waits for P_g(j) V_j, since P_g lives in
//                  S_g's tensor memory; P.V reads P from tensor memory.
//   warps 2-11     rotate both tiles' RoPE parts in shared memory first
//   warps 4-7, 8-11  softmax of tile A, of tile B: one query row per thread
//                  (TMEM lane = row); scores in base 2, masked past the row's
//                  position and before the window; the running maximum is
//                  raised only when a tile exceeds it by more than 2^8, and
//                  then O is rescaled in TMEM; P (bf16) is written over the
//                  scores in tensor memory. At the end O / l and the
//                  log-sum-exp are stored.
// Every wait is bounded (2 s); a timeout sets MLA_ERR_DEVICE_TIMEOUT in the
// status word and every role leaves its loop.
__global__ void __launch_bounds__(tcq::kThreads, 1)
prefill_attn_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                     const __grid_constant__ CUtensorMap tm_kr, const __grid_constant__ CUtensorMap tm_v,
                     PrefillArgs a) {
  using namespace tcq;
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
    mbar_init(BAR(B_QROT), 10);
    for (int s = 0; s < 2; ++s) {
      mbar_init(BAR(B_KFULL + s), 1);
      mbar_init(BAR(B_KEMPTY + s), 1);
      mbar_init(BAR(B_SFULL + s), 1);
      mbar_init(BAR(B_PFULL + s), 4);
      mbar_init(BAR(B_PVDONE + s), 1);
    }
    mbar_init(BAR(B_VFULL), 1);
    mbar_init(BAR(B_VEMPTY), 1);
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
  pdl_wait();  // the gathered rows and the formed keys and values come from the previous kernels

  const int len = prefill_len(a.seq_lens, b, a.max_len);
  const int q0 = qb * 2 * kRows;                // this CTA's first query of the chunk
  const int nq = min(2 * kRows, a.C - q0);      // its valid queries (tile A's, then tile B's)
  const int pos0 = len - a.C + q0;              // position of its first query
  const int pos_max = pos0 + nq - 1;
  const int lo = a.seq_start != nullptr ? min(max(a.seq_start[b], 0), len) : 0;  // first visible position
  const int j0 = lo / kTile;                                 // first key tile with a visible key
  const int n_end = pos_max < 0 ? 0 : pos_max / kTile + 1;   // one past the last such tile
  const int n = n_end > j0 ? n_end - j0 : 0;                 // key tiles processed: j0 .. n_end - 1
  const int krow0 = b * a.l_pad + j0 * kTile;                // row of the first of them

  if (warp >= 2 && n > 0) {
    // Warps 2-11 rotate the RoPE part of both tiles' Q (box 2 of each: [128
    // rows x 64], 128-byte swizzle) at each row's position, interleaved pairs.
    const int t = threadIdx.x - 64;  // 0..319
    const bool got = __all_sync(0xffffffffu, pwait(BAR(B_QFULL), 0, a.status));
    if (got) {
#pragma unroll 1
      for (int k = t; k < 2 * kRows * 8; k += kThreads - 64) {
        const int row = k >> 3, u = k & 7, g = row >> 7, rr = row & (kRows - 1);
        const int pos = min(max(pos0 + row, 0), a.max_len - 1);  // rows past the chunk are not stored
        const float4* cs = reinterpret_cast<const float4*>(a.rope + (size_t)pos * (kDr / 2) + u * 4);
        const float4 cs01 = __ldg(cs), cs23 = __ldg(cs + 1);
        const float cz[4] = {cs01.x, cs01.z, cs23.x, cs23.z}, sz[4] = {cs01.y, cs01.w, cs23.y, cs23.w};
        uint4* cell = reinterpret_cast<uint4*>(gbase + OFF_Q + (3 * g + 2) * kBox + swz128(rr, u));
        const uint4 v = *cell;
        uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const __nv_bfloat162 x = *reinterpret_cast<const __nv_bfloat162*>(&w[e]);
          const float x0 = __low2float(x), x1 = __high2float(x);
          const __nv_bfloat162 y = __floats2bfloat162_rn(x0 * cz[e] - x1 * sz[e], x0 * sz[e] + x1 * cz[e]);
          w[e] = *reinterpret_cast<const uint32_t*>(&y);
        }
        *cell = make_uint4(w[0], w[1], w[2], w[3]);
      }
      fence_proxy_async_smem();
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(BAR(B_QROT));
  }

  if (warp == 0 && lane == 0 && n > 0) {
    // ------------------------------------------------------------ TMA producer
    const int qy = b * a.C + q0;
    mbar_arrive_expect_tx(BAR(B_QFULL), 6 * kBox);
    for (int g = 0; g < 2; ++g)
      for (int c = 0; c < 3; ++c)
        tma_load_2d(base + OFF_Q + (3 * g + c) * kBox, &tm_q, h * (kDh + kDr) + 64 * c, qy + g * kRows,
                    BAR(B_QFULL));
    auto load_k = [&](int j) {
      const int s = j & 1, y = krow0 + j * kTile;
      const uint32_t dst = base + OFF_K + s * 3 * kBox;
      mbar_arrive_expect_tx(BAR(B_KFULL + s), 3 * kBox);
      tma_load_2d(dst, &tm_k, h * kDh, y, BAR(B_KFULL + s));
      tma_load_2d(dst + kBox, &tm_k, h * kDh + 64, y, BAR(B_KFULL + s));
      tma_load_2d(dst + 2 * kBox, &tm_kr, 0, y, BAR(B_KFULL + s));
    };
    auto load_v = [&](int j) {
      mbar_arrive_expect_tx(BAR(B_VFULL), 2 * kBox);
      tma_load_2d(base + OFF_V, &tm_v, h * kDv, krow0 + j * kTile, BAR(B_VFULL));
      tma_load_2d(base + OFF_V + kBox, &tm_v, h * kDv + 64, krow0 + j * kTile, BAR(B_VFULL));
    };
    // V has one stage: V_{j+1} is requested only when P.V of tile j is done,
    // so it is first brought into L2 with K_{j+1}, two tiles ahead.
    auto prefetch_v = [&](int j) {
      tma_prefetch_2d(&tm_v, h * kDv, krow0 + j * kTile);
      tma_prefetch_2d(&tm_v, h * kDv + 64, krow0 + j * kTile);
    };
    load_k(0);
    int k_issued = 1, v_issued = 1;
    if (n > 1) {
      load_k(1);
      prefetch_v(1);
      ++k_issued;
    }
    load_v(0);
    for (int j = 0; j < n; ++j) {
      // K_{j+2} into stage j % 2 once both tiles' S of key tile j are done;
      // V_{j+1} once both tiles' P.V of key tile j are done.
      if (j + 2 < n) {
        if (!pwait(BAR(B_KEMPTY + (j & 1)), (j >> 1) & 1, a.status)) break;
        load_k(j + 2);
        prefetch_v(j + 2);
        ++k_issued;
      }
      if (j + 1 < n) {
        if (!pwait(BAR(B_VEMPTY), j & 1, a.status)) break;
        load_v(j + 1);
        ++v_issued;
      }
    }
    // Every copy issued has landed before this thread leaves (instant on the
    // normal path, where the MMAs consumed them all).
    pwait(BAR(B_QFULL), 0, a.status);
    for (int s = 0; s < 2; ++s) {
      const int cnt = (k_issued - s + 1) / 2;  // loads into stage s: tiles s, s + 2, ...
      if (cnt > 0) pwait(BAR(B_KFULL + s), (cnt - 1) & 1, a.status);
    }
    pwait(BAR(B_VFULL), (v_issued - 1) & 1, a.status);
  } else if (warp == 1 && lane == 0 && n > 0) {
    // ------------------------------------------------------------ MMA issuer
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false, false);
    constexpr uint32_t idesc_pv = idesc_bf16_f32(128, kDv, false, true);
    // S_g(j) = Q_g K_j^T over 192 = three 64-wide boxes.
    auto issue_s = [&](int g, int j) {
      const uint32_t kb = base + OFF_K + (j & 1) * 3 * kBox, qb_ = base + OFF_Q + 3 * g * kBox;
#pragma unroll
      for (int c = 0; c < 3; ++c)
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_f16(tmem + TM_S + g * kTile, smem_desc(qb_ + c * kBox + kk * 32, 16, 1024, kSwizzle128B),
                  smem_desc(kb + c * kBox + kk * 32, 16, 1024, kSwizzle128B), idesc_s, (c | kk) ? 1u : 0u);
      mma_commit(BAR(B_SFULL + g));
    };
    // O_g += P_g(j) V_j: A = P_g in tensor memory (columns TM_S + 128 g + 8 kk
    // hold keys 16 kk .. 16 kk + 15), B = V [128 keys x 128 values] MN-major.
    auto issue_pv = [&](int g, int j) {
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk)
        mma_f16_ts(tmem + TM_O + g * kDv, tmem + TM_S + g * kTile + kk * 8,
                   smem_desc(base + OFF_V + kk * 2048, kBox, 1024, kSwizzle128B), idesc_pv,
                   (j > 0 || kk > 0) ? 1u : 0u);
      mma_commit(BAR(B_PVDONE + g));
    };
    bool ok = pwait(BAR(B_QFULL), 0, a.status) && pwait(BAR(B_QROT), 0, a.status) &&
              pwait(BAR(B_KFULL), 0, a.status);
    if (ok) {
      tc_fence_after();
      issue_s(0, 0);
      issue_s(1, 0);
      mma_commit(BAR(B_KEMPTY));
    }
    for (int j = 0; ok && j < n; ++j) {
      const bool more = j + 1 < n;
      const int s1 = (j + 1) & 1;
      // Tile A: P_A(j) V_j, then S_A(j+1) once that P.V is done.
      if (!pwait(BAR(B_PFULL), j & 1, a.status) || !pwait(BAR(B_VFULL), j & 1, a.status)) break;
      tc_fence_after();
      issue_pv(0, j);
      if (more) {
        if (!pwait(BAR(B_PVDONE), j & 1, a.status) || !pwait(BAR(B_KFULL + s1), ((j + 1) >> 1) & 1, a.status)) break;
        tc_fence_after();
        issue_s(0, j + 1);
      }
      // Tile B: P_B(j) V_j (V_j is then free), then S_B(j+1).
      if (!pwait(BAR(B_PFULL + 1), j & 1, a.status)) break;
      tc_fence_after();
      issue_pv(1, j);
      mma_commit(BAR(B_VEMPTY));
      if (more) {
        if (!pwait(BAR(B_PVDONE + 1), j & 1, a.status)) break;
        tc_fence_after();
        issue_s(1, j + 1);
        mma_commit(BAR(B_KEMPTY + s1));
      }
    }
    // Every MMA issued has completed before TMEM is released.
    mma_commit(BAR(B_MMADONE));
    pwait(BAR(B_MMADONE), 0, a.status);
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax and epilogue of tile g
    const int g = (warp - 4) >> 2, qd = warp & 3, r = qd * 32 + lane;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    const uint32_t ts = tmem + lane_base + TM_S + g * kTile, to = tmem + lane_base + TM_O + g * kDv;
    const int pos = pos0 + g * kRows + r;
    const int wpos0 = pos0 + g * kRows + qd * 32;  // the warp's first position
    float m_run = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      ok = __all_sync(0xffffffffu, pwait(BAR(B_SFULL + g), j & 1, a.status));
      if (!ok) break;
      tc_fence_after();
      uint32_t v[4][32];
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) tmem_ld32(ts + cc * 32, v[cc]);
      tmem_wait_ld();
      const int kbase = (j0 + j) * kTile;
      if (kbase + kTile - 1 > wpos0 || kbase < lo) {
        // Key k of the tile (0..127) is visible for lo <= kbase + k <= pos.
        const int k_hi = pos - kbase, k_lo = lo - kbase;
#pragma unroll
        for (int cc = 0; cc < 4; ++cc)
#pragma unroll
          for (int x = 0; x < 32; ++x)
            if (cc * 32 + x > k_hi || cc * 32 + x < k_lo) v[cc][x] = __float_as_uint(-INFINITY);
      }
      const float mx =
          fmaxf(fmaxf(max_of32(v[0]), max_of32(v[1])), fmaxf(max_of32(v[2]), max_of32(v[3]))) * a.scale_log2;
      const bool upd = mx > m_run + tcp::kRescaleLog2;
      const float m_new = upd ? mx : m_run;
      const float fac = upd ? ex2_approx(m_run - m_new) : 1.f;  // 0 while nothing was seen
      const float neg_mref = (m_new == -INFINITY) ? 0.f : -m_new;
      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t pk[16];
#pragma unroll
        for (int x2 = 0; x2 < 16; ++x2) {
          float p0, p1;
          fma_x2(p0, p1, __uint_as_float(v[cc][2 * x2]), __uint_as_float(v[cc][2 * x2 + 1]), a.scale_log2,
                 neg_mref);
          p0 = ex2_approx(p0);
          p1 = ex2_approx(p1);
          if (x2 & 1) add_x2(s2, s3, p0, p1);
          else add_x2(s0, s1, p0, p1);
          const __nv_bfloat162 p2 = __floats2bfloat162_rn(p0, p1);
          pk[x2] = *reinterpret_cast<const uint32_t*>(&p2);
        }
        // P of keys 32 cc .. 32 cc + 31 over columns 16 cc .. 16 cc + 15: the
        // scores there are already in registers.
        tmem_st16(ts + cc * 16, pk);
      }
      const float sum = (s0 + s1) + (s2 + s3);
      l = l * fac + sum;
      m_run = m_new;
      // P.V of tile j-1 completed before S of tile j was issued: O may be
      // rescaled now.
      if (__any_sync(0xffffffffu, upd) && j >= 1) {
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          tmem_ld32(to + cc * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * fac);
          tmem_st32(to + cc * 32, o);
        }
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PFULL + g));
    }
    if (ok && n > 0) ok = __all_sync(0xffffffffu, pwait(BAR(B_PVDONE + g), (n - 1) & 1, a.status));
    if (ok) {
      tc_fence_after();
      const int qi = g * kRows + r;  // query index within the CTA
      const bool valid = qi < nq;
      const size_t row = (size_t)b * a.C + q0 + qi;
      // A row that saw no key is empty: o = 0 and lse = -inf.
      const bool seen = m_run != -INFINITY && l > 0.f;
      const float inv = seen ? 1.f / l : 0.f;
      uint4* dst = reinterpret_cast<uint4*>(a.o + (row * a.n_h + h) * kDv);
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        if (n > 0) {
          tmem_ld32(to + cc * 32, o);
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
      if (valid) a.lse[row * a.n_h + h] = seen ? (m_run + log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

bool tc_prefill_supported(const mla_dims_t& d) {
  return d.act_dtype == MLA_BF16 && (d.cache_dtype == MLA_BF16 || d.cache_dtype == MLA_FP8_E4M3) &&
         d.d_h == tcp::kDh && d.d_v == tcp::kDv && d.d_rope == tcp::kDr && d.d_c >= 64 && d.d_c % 64 == 0 &&
         tc_device_ok();
}


PrefillWs prefill_ws_layout(const mla_dims_t& d, int B, int C, int max_seq_len) {
  PrefillWs w = {};
  // Rows per sequence: a multiple of 256, so that the expansion kernel's CTA
  // pairs (two 128-row tiles) never straddle two sequences.
  w.l_pad = (max_seq_len > 0 ? (max_seq_len + 255) / 256 : 1) * 256;
  const size_t rows = (size_t)B * w.l_pad;
  w.lat_off = 0;
  w.k_off = w.lat_off + align256(rows * (d.d_c + d.d_rope) * 2);
  w.v_off = w.k_off + align256(rows * d.n_h * d.d_h * 2);
  w.rope_off = w.v_off + align256(rows * d.n_h * d.d_v * 2);
  w.total = w.rope_off + align256((size_t)w.l_pad * (d.d_rope / 2) * sizeof(float2));
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

// Resident 2-CTA clusters of the expansion kernel per device, computed once.
static int64_t expand_resident_clusters() {
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int clusters = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256, 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = tce::kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaOccupancyMaxActiveClusters(&clusters, prefill_expand_kernel, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      clusters = std::max(1, sm_count() / 2);
    }
    v = clusters;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

cudaError_t launch_prefill(const mla_dims_t& d, const mla_cache_t& c, int B, int C, int max_seq_len,
                           const __nv_bfloat16* q, const __nv_bfloat16* w_uk, const __nv_bfloat16* w_uv,
                           const int32_t* bt, int max_pages, const int32_t* seq_lens, const int32_t* seq_start,
                           void* ws, __nv_bfloat16* o, float* lse, int32_t* status, cudaStream_t st) {
  using namespace tcp;
  const PrefillWs L = prefill_ws_layout(d, B, C, max_seq_len);
  uint8_t* w8 = reinterpret_cast<uint8_t*>(ws);
  __nv_bfloat16* lat = reinterpret_cast<__nv_bfloat16*>(w8 + L.lat_off);
  __nv_bfloat16* kbuf = reinterpret_cast<__nv_bfloat16*>(w8 + L.k_off);
  __nv_bfloat16* vbuf = reinterpret_cast<__nv_bfloat16*>(w8 + L.v_off);
  const int max_len = std::min<int64_t>(max_seq_len, (int64_t)max_pages * d.page_size);
  const int rows = B * L.l_pad, T = B * C;
  const int fp8 = d.cache_dtype == MLA_FP8_E4M3 ? 1 : 0;

  cudaError_t e = launch_pdl(prefill_gather_kernel, dim3(L.l_pad / 8, B), dim3(256), 0, st, L.l_pad, max_len, d.d_c,
                             d.d_rope, d.page_size, max_pages, (int64_t)c.num_pages, fp8, (const void*)c.ckv,
                             (const __nv_bfloat16*)c.kr, (const float*)c.scale, bt, seq_lens, seq_start, lat,
                             status);
  if (e != cudaSuccess) return e;
  float2* rope_tab = reinterpret_cast<float2*>(w8 + L.rope_off);
  if (max_len > 0) {
    const int items = max_len * (d.d_rope / 2);
    e = launch_pdl(prefill_rope_table_kernel, dim3((items + 255) / 256), dim3(256), 0, st, max_len, d.d_rope / 2,
                   rope_freqs(d.d_rope, d.rope_theta), rope_tab);
    if (e != cudaSuccess) return e;
  }
  {
    CUtensorMap tm_lat, tm_wuk, tm_wuv;
    if (!tc_map2d_bf16(&tm_lat, lat, d.d_c, (uint64_t)rows, (uint64_t)(d.d_c + d.d_rope), tce::kTok) ||
        !tc_map2d_bf16(&tm_wuk, w_uk, d.d_c, (uint64_t)d.n_h * kDh, d.d_c, 128) ||
        !tc_map2d_bf16(&tm_wuv, w_uv, d.d_c, (uint64_t)d.n_h * kDv, d.d_c, 128))
      return cudaErrorInvalidValue;
    static std::once_flag once_e;
    static cudaError_t attr_e = cudaSuccess;
    std::call_once(once_e, [] {
      attr_e = cudaFuncSetAttribute(prefill_expand_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)tce::kSmem);
    });
    if (attr_e != cudaSuccess) return attr_e;
    // Heads per CTA: every cluster holds one pair of row tiles and hpc heads,
    // and runs for a time proportional to hpc plus its latent tiles' load
    // (about half a head's weights); the clusters run in waves of the resident
    // count. The split of the heads into groups minimises waves x (hpc + 1/2),
    // the fewest groups among equals.
    const int tiles = rows / tce::kTok;  // even: l_pad is a multiple of 256
    const int64_t resident = expand_resident_clusters();
    int groups = 1, hpc = d.n_h;
    int64_t best = -1;
    for (int g = 1; g <= d.n_h; ++g) {
      const int per = (d.n_h + g - 1) / g;
      if ((d.n_h + per - 1) / per != g) continue;  // the same split as a smaller g
      const int64_t waves = ((int64_t)(tiles / 2) * g + resident - 1) / resident;
      if (best < 0 || waves * (2 * per + 1) < best) {
        best = waves * (2 * per + 1);
        groups = g;
        hpc = per;
      }
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(tiles, groups);
    cfg.blockDim = dim3(256);
    cfg.dynamicSmemBytes = tce::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, prefill_expand_kernel, tm_lat, tm_wuk, tm_wuv, d.n_h, hpc, d.d_c / 64, L.l_pad,
                           max_len, seq_lens, seq_start, kbuf, vbuf, status);
    if (e != cudaSuccess) return e;
  }

  CUtensorMap tm_q, tm_k, tm_kr, tm_v;
  const uint64_t dq = (uint64_t)d.n_h * (kDh + kDr), dkv = (uint64_t)d.n_h * kDh;
  if (!tc_map2d_bf16(&tm_q, q, dq, (uint64_t)T, dq, kRows) ||
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
  a.rope = rope_tab;
  a.seq_lens = seq_lens;
  a.seq_start = seq_start;
  a.o = o;
  a.lse = lse;
  a.status = status;
  static std::once_flag once;
  static cudaError_t attr = cudaSuccess;
  std::call_once(once, [] {
    attr = cudaFuncSetAttribute(prefill_attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcq::kSmem);
  });
  if (attr != cudaSuccess) return attr;
  return launch_pdl(prefill_attn_kernel, dim3((C + 2 * kRows - 1) / (2 * kRows), d.n_h, B), dim3(tcq::kThreads),
                    tcq::kSmem, st, tm_q, tm_k, tm_kr, tm_v, a);
}

}  // namespace mla
