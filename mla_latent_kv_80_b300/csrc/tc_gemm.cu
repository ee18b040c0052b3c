// Tensor-core (tcgen05) skinny GEMMs of one MLA decode step. Each streams a
// weight matrix once through TMA and multiplies it with the few token rows of
// the step, D^T[M x N] = W[M x K] . X^T[K x N] with M = weight rows (tile 128),
// N = tokens (tile <= 128), fp32 accumulation in TMEM:
//   append   x_t = [W_DKV ; W_KR] h_t          ("MLA 之后，KV cache 确实得重新理解一遍",
//                                               "第一步": c_kv = W_DKV x; k_R = W_KR x)
//            split over K; fp32 partial sums go to the append workspace and the
//            epilogue kernel reduces them, rotates k_R and writes the slot.
//   absorb   q_lat[t,h] = W_UK[h]^T q_nope[t,h]  (same page, "第二步": W_UK
//            pre-multiplied into the query); A is W_UK[h] read MN-major.
//   out-proj o[t,h] = W_UV[h] o_lat[t,h]        (same page, "第二步": W_UV applied
//            once to the latent weighted sum).
// One CTA (4 warps) computes one 128 x BN tile: warp 0 lane 0 issues TMA into
// a 6-stage ring, warp 1 lane 0 issues the MMAs, all four warps (one thread
// per TMEM lane) run the epilogue.
#include "tc_gemm.cuh"
#include "sm100_ptx.cuh"

#include <cuda.h>
#include <math.h>
#include <mutex>

namespace mla {
using namespace ptx;

namespace tcg {
// Ring stages per kernel: the absorb GEMM (two K chunks per CTA) uses two, so
// that four CTAs fit on an SM; the others stream eight or more chunks per CTA.
// W_O (K split eight ways, 320 CTAs for DeepSeek-V2) uses three, three CTAs per
// SM. With 256-token tiles (the out-proj of more than 128 rows) a stage is
// 48 KB: the out-proj then keeps four.
__host__ __device__ constexpr int stages_for(int epi, int bn = 128) {
  return epi == 1 ? 2 : (epi == 3 ? 3 : (bn > 128 ? 4 : 6));
}
constexpr int kBK = 64;                        // K per stage (one 128-byte swizzle atom)
constexpr uint32_t kABytes = 128 * kBK * 2;    // 16 KB
constexpr uint64_t kWaitNs = 2000000000ull;
enum Epi { EPI_APPEND_PARTIAL = 0, EPI_ABSORB = 1, EPI_OUTPROJ = 2, EPI_WO_PARTIAL = 3 };
__host__ __device__ constexpr uint32_t b_bytes(int bn) { return (uint32_t)bn * kBK * 2; }
__host__ __device__ constexpr uint32_t smem_bytes(int epi, int bn) {
  return stages_for(epi, bn) * (kABytes + b_bytes(bn)) + 256 + 1024;
}
}  // namespace tcg

namespace {

__device__ __forceinline__ bool gwait(uint32_t bar, uint32_t parity, int32_t* status) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63) == 0 && globaltimer() - t0 > tcg::kWaitNs) {
      set_status(status, MLA_ERR_DEVICE_TIMEOUT);
      return false;
    }
  }
}

struct GemmArgs {
  int T;           // token rows
  int n_h;         // heads (absorb / out-proj)
  int k_chunks;    // K chunks of 64 per 128-row tile
  int m_per_cta;   // consecutive 128-row tiles handled by one CTA (each its own TMEM columns)
  int m_valid;     // valid output rows of the whole GEMM (append: d_c + d_rope)
  int d_c, d_rope, d_h, d_v;
  RopeFreqs freqs;
  const int32_t* pos;
  const __nv_bfloat16* q;   // absorb: source of the RoPE part
  void* out;                // append: fp32 workspace; absorb: q_abs; out-proj: o
  int32_t* status;
};

}  // namespace

// grid: x = M tile, y = N tile, z = head (absorb / out-proj) or K split (append)
template <int EPI, bool A_MN, int BN>
__global__ void __launch_bounds__(128)
tc_gemm_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_a2,
               const __grid_constant__ CUtensorMap tm_b, GemmArgs g) {
  using namespace tcg;
  constexpr int kStages = stages_for(EPI, BN);
  static_assert(smem_bytes(EPI, BN) <= 232448, "shared memory of the GEMM");
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t OFF_B = kStages * kABytes;
  const uint32_t OFF_BAR = OFF_B + kStages * b_bytes(BN);
  auto FULL = [&](int s) { return base + OFF_BAR + 8u * s; };
  auto EMPTY = [&](int s) { return base + OFF_BAR + 8u * (kStages + s); };
  const uint32_t DONE = base + OFF_BAR + 8u * (2 * kStages);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 8 * (2 * kStages + 1));
  uint32_t tmem_cols = 32;
  while (tmem_cols < (uint32_t)(g.m_per_cta * BN)) tmem_cols <<= 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int mt0 = blockIdx.x * g.m_per_cta, nt = blockIdx.y, z = blockIdx.z;
  const int n_chunks = g.m_per_cta * g.k_chunks;
  pdl_trigger();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), 1);
    }
    mbar_init(DONE, 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    prefetch_tmap(&tm_a);
    prefetch_tmap(&tm_b);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  bool ok = true;
  if (!(warp == 0 && lane == 0)) pdl_wait();  // the producer waits after its first weight loads

  // Coordinates of this CTA's operands.
  //   append:   A rows mt*128 of [W_DKV ; W_KR] (tm_a2 = W_KR for the last tile), K from z*k_chunks
  //   absorb:   A = W_UK[z] viewed [d_h rows][d_c cols], MN-major: x = c, y = z*d_h + k
  //   out-proj: A = W_UV[z] viewed [n_h*d_v rows][d_c cols], K-major: x = k, y = z*d_v
  const int k0 = (EPI == EPI_APPEND_PARTIAL || EPI == EPI_WO_PARTIAL) ? z * g.k_chunks * kBK : 0;
  if (warp == 0 && lane == 0) {
    // Weights do not depend on earlier kernels: the first ring stages' weight
    // tiles are requested before waiting for the previous kernel, the token rows
    // (written by it) only after.
    auto load_a = [&](int ci) {
      const int s = ci % kStages;
      const int mt = mt0 + ci / g.k_chunks, kc = ci % g.k_chunks;
      const uint32_t a_dst = base + s * kABytes;
      const int kk = k0 + kc * kBK;
      if (EPI == EPI_APPEND_PARTIAL) {
        if (mt * 128 >= g.d_c) tma_load_2d(a_dst, &tm_a2, kk, 0, FULL(s));
        else tma_load_2d(a_dst, &tm_a, kk, mt * 128, FULL(s));
      } else if (EPI == EPI_WO_PARTIAL) {
        tma_load_2d(a_dst, &tm_a, kk, mt * 128, FULL(s));
      } else if (EPI == EPI_ABSORB) {
        tma_load_2d(a_dst, &tm_a, mt * 128, z * g.d_h + kk, FULL(s));
        tma_load_2d(a_dst + 8192, &tm_a, mt * 128 + 64, z * g.d_h + kk, FULL(s));
      } else {
        tma_load_2d(a_dst, &tm_a, kk, mt * 128 + z * g.d_v, FULL(s));
      }
    };
    auto load_b = [&](int ci) {
      const int s = ci % kStages;
      const int kc = ci % g.k_chunks;
      const uint32_t b_dst = base + OFF_B + s * b_bytes(BN);
      const int kk = k0 + kc * kBK;
      if (EPI == EPI_APPEND_PARTIAL || EPI == EPI_WO_PARTIAL) tma_load_2d(b_dst, &tm_b, kk, nt * BN, FULL(s));
      else if (EPI == EPI_ABSORB) tma_load_2d(b_dst, &tm_b, z * (g.d_h + g.d_rope) + kk, nt * BN, FULL(s));
      else tma_load_2d(b_dst, &tm_b, z * g.d_c + kk, nt * BN, FULL(s));
    };
    const int pre = n_chunks < kStages ? n_chunks : kStages;
    for (int ci = 0; ci < pre; ++ci) {
      mbar_arrive_expect_tx(FULL(ci), kABytes + b_bytes(BN));
      load_a(ci);
    }
    pdl_wait();
    for (int ci = 0; ci < pre; ++ci) load_b(ci);
    int issued = pre;
    for (int ci = pre; ci < n_chunks; ++ci) {
      const int s = ci % kStages;
      if (!gwait(EMPTY(s), ((ci / kStages) - 1) & 1, g.status)) { ok = false; break; }
      mbar_arrive_expect_tx(FULL(s), kABytes + b_bytes(BN));
      load_a(ci);
      load_b(ci);
      ++issued;
    }
    if (!ok) {
      // The copies still in flight land (bounded wait) before the CTA's shared
      // memory is released: the last phase issued on each stage.
      for (int s = 0; s < kStages && s < issued; ++s) gwait(FULL(s), ((issued - 1 - s) / kStages) & 1, g.status);
    }
  } else if (warp == 1 && lane == 0) {
    constexpr uint32_t idesc = idesc_bf16_f32(128, BN, A_MN, false);
    for (int ci = 0; ci < n_chunks; ++ci) {
      const int s = ci % kStages;
      const int mi = ci / g.k_chunks, kc = ci % g.k_chunks;
      if (!gwait(FULL(s), (ci / kStages) & 1, g.status)) { ok = false; break; }
      tc_fence_after();
      const uint32_t a_base = base + s * kABytes;
      const uint32_t b_base = base + OFF_B + s * b_bytes(BN);
#pragma unroll
      for (int k16 = 0; k16 < kBK / 16; ++k16) {
        const uint64_t a = A_MN ? smem_desc(a_base + k16 * 2048, 8192, 1024, kSwizzle128B)
                                : smem_desc(a_base + k16 * 32, 16, 1024, kSwizzle128B);
        const uint64_t b = smem_desc(b_base + k16 * 32, 16, 1024, kSwizzle128B);
        mma_f16(tmem + mi * BN, a, b, idesc, (kc | k16) ? 1u : 0u);
      }
      mma_commit(EMPTY(s));
    }
    mma_commit(DONE);
  }
  __syncwarp();

  if (EPI == EPI_ABSORB && warp >= 2) {
    // RoPE part of q_abs for this head and these tokens, by the two warps that
    // are idle while the MMAs run, shared among the head's M-tile CTAs.
    const int half = g.d_rope / 2;
    const int dq = g.d_h + g.d_rope, dqa = g.d_c + g.d_rope;
    // A batch of (token, pair) items per thread: every input is loaded before
    // the first result is stored (the output may alias nothing, but the
    // compiler cannot know that), so the loads' latencies overlap.
    constexpr int kItems = 8;
    const int step = 64 * (int)gridDim.x;
    for (int i0 = threadIdx.x - 64 + 64 * (int)blockIdx.x; i0 < BN * half; i0 += step * kItems) {
      __nv_bfloat162 xv[kItems];
      int tp[kItems];
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        const int i = i0 + step * u;
        const int t = nt * BN + i / half, pr = i % half;
        tp[u] = -1;
        if (i < BN * half && t < g.T) {
          xv[u] = *reinterpret_cast<const __nv_bfloat162*>(g.q + ((size_t)t * g.n_h + z) * dq + g.d_h + 2 * pr);
          tp[u] = g.pos[t];
        }
      }
#pragma unroll
      for (int u = 0; u < kItems; ++u) {
        const int i = i0 + step * u;
        const int t = nt * BN + i / half, pr = i % half;
        if (i >= BN * half || t >= g.T) continue;
        float c, s;
        rope_cos_sin(tp[u], g.freqs.hi[pr], g.freqs.lo[pr], &c, &s);
        const float x0 = __low2float(xv[u]), x1 = __high2float(xv[u]);
        *reinterpret_cast<__nv_bfloat162*>(reinterpret_cast<__nv_bfloat16*>(g.out) + ((size_t)t * g.n_h + z) * dqa +
                                          g.d_c + 2 * pr) = __floats2bfloat162_rn(x0 * c - x1 * s, x0 * s + x1 * c);
      }
    }
  }
  // ------------------------------------------------------------ epilogue
  // CTA-uniform: the TMEM loads below are warp-collective and the staged
  // outputs need a block barrier.
  const bool done = __syncthreads_and(gwait(DONE, 0, g.status) && ok);
  tc_fence_after();
  const int m = threadIdx.x;  // TMEM lane = output row within the tile
  const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
  if (done && (EPI == EPI_APPEND_PARTIAL || EPI == EPI_WO_PARTIAL)) {
#pragma unroll 1
    for (int mi = 0; mi < g.m_per_cta; ++mi) {
      const int row = (mt0 + mi) * 128 + m;
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + mi * BN + c0, v);
        tmem_wait_ld();
        for (int x = 0; x < 32; ++x) {
          const int t = nt * BN + c0 + x;
          if (t >= g.T) break;
          if (row < g.m_valid)
            reinterpret_cast<float*>(g.out)[((size_t)z * g.T + t) * g.m_valid + row] = __uint_as_float(v[x]);
        }
      }
    }
  } else if (done) {
    // absorb / out-proj: the tile is staged in shared memory (the ring is idle
    // once every MMA has completed) as [token][row] bf16, then each token's
    // contiguous output row (d_c or d_v values) is written with 16-byte stores.
    const int wcols = g.m_per_cta * 128;
    __nv_bfloat16* stage = reinterpret_cast<__nv_bfloat16*>(gbase);
#pragma unroll 1
    for (int mi = 0; mi < g.m_per_cta; ++mi) {
#pragma unroll 1
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t v[32];
        tmem_ld32(tmem + lane_base + mi * BN + c0, v);
        tmem_wait_ld();
#pragma unroll
        for (int x = 0; x < 32; ++x) stage[(c0 + x) * wcols + mi * 128 + m] = __float2bfloat16_rn(__uint_as_float(v[x]));
      }
    }
    __syncthreads();
    const int ntok = min(BN, g.T - nt * BN);
    const int chunks = wcols / 8;
    const size_t row_elems = (EPI == EPI_ABSORB) ? (size_t)(g.d_c + g.d_rope) : (size_t)g.d_v;
    __nv_bfloat16* out = reinterpret_cast<__nv_bfloat16*>(g.out);
    const int head = z;
    for (int i = threadIdx.x; i < ntok * chunks; i += blockDim.x) {
      const int tt = i / chunks, ch = i % chunks;
      const size_t t = (size_t)(nt * BN + tt);
      *reinterpret_cast<uint4*>(out + (t * g.n_h + head) * row_elems + mt0 * 128 + ch * 8) =
          *reinterpret_cast<const uint4*>(stage + tt * wcols + ch * 8);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, tmem_cols);
  }
}

// ====================================================================== host side
namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

}  // namespace

// bf16 2-D map, 128-byte swizzle, inner box 64 elements.
bool tc_map2d_bf16(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t row_elems,
                   uint32_t box_rows) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_elems * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {
bool map2d(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t row_elems, uint32_t box_rows) {
  return tc_map2d_bf16(m, ptr, inner, rows, row_elems, box_rows);
}

template <int EPI, bool A_MN, int BN>
cudaError_t launch(dim3 grid, const CUtensorMap& a, const CUtensorMap& a2, const CUtensorMap& b,
                   const GemmArgs& g, cudaStream_t st) {
  auto k = tc_gemm_kernel<EPI, A_MN, BN>;
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [&] {
    err = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)tcg::smem_bytes(EPI, BN));
  });
  if (err != cudaSuccess) return err;
  return launch_pdl(k, grid, dim3(128), tcg::smem_bytes(EPI, BN), st, a, a2, b, g);
}

// Token tile: 16..128 in steps of 16.
int pick_bn(int T) {
  if (T <= 16) return 16;
  if (T <= 32) return 32;
  if (T <= 64) return 64;
  return 128;
}

// Token tile of the out-proj GEMM: up to 256 rows, so that more than 128 rows
// read each W_UV tile once (MMA N = 256). The absorb GEMM (two K chunks per
// CTA) gains more from more CTAs and keeps at most 64; W_O keeps 128, whose K
// split then keeps more CTAs streaming (measured on 256 rows).
int pick_bn_wide(int T) { return T > 128 ? 256 : pick_bn(T); }

template <int EPI, bool A_MN>
cudaError_t launch_bn(int bn, dim3 grid, const CUtensorMap& a, const CUtensorMap& a2,
                      const CUtensorMap& b, const GemmArgs& g, cudaStream_t st) {
  switch (bn) {
    case 16: return launch<EPI, A_MN, 16>(grid, a, a2, b, g, st);
    case 32: return launch<EPI, A_MN, 32>(grid, a, a2, b, g, st);
    case 64: return launch<EPI, A_MN, 64>(grid, a, a2, b, g, st);
    case 128: return launch<EPI, A_MN, 128>(grid, a, a2, b, g, st);
    default: return launch<EPI, A_MN, 256>(grid, a, a2, b, g, st);
  }
}

}  // namespace

bool tc_gemm_supported(const mla_dims_t& d) {
  return d.act_dtype == MLA_BF16 && d.d_c % 128 == 0 && d.d_h % 64 == 0 && d.d_v == 128 &&
         d.d_model % 64 == 0 && d.d_rope <= 128 && d.d_rope % 2 == 0 && tc_device_ok();
}

int tc_append_ksplit(const mla_dims_t& d, int T) {
  if (T <= 0) return 1;
  const int m_tiles = (d.d_c + d.d_rope + 127) / 128;
  const int n_tiles = (T + pick_bn(T) - 1) / pick_bn(T);
  const int k_chunks = d.d_model / tcg::kBK;
  // At most 16 K splits (80 weight-streaming CTAs for the 576-row weight, five
  // 64-wide K chunks each); the epilogue sums the fp32 partials eight at a time.
  // More splits measured no faster and only grow the partial workspace.
  int ks = (sm_count() + m_tiles * n_tiles - 1) / (m_tiles * n_tiles);
  if (ks > 16) ks = 16;
  if (ks < 1) ks = 1;
  while (ks > 1 && k_chunks % ks != 0) --ks;  // equal K per split
  return ks;
}

cudaError_t launch_tc_append_gemm(const mla_dims_t& d, int T, const __nv_bfloat16* h,
                                  const __nv_bfloat16* w_dkv, const __nv_bfloat16* w_kr, float* ws,
                                  int ksplit, int32_t* status, cudaStream_t st) {
  const int bn = pick_bn(T);
  CUtensorMap a, a2, b;
  if (!map2d(&a, w_dkv, d.d_model, d.d_c, d.d_model, 128) ||
      !map2d(&a2, w_kr, d.d_model, d.d_rope, d.d_model, 128) ||
      !map2d(&b, h, d.d_model, T, d.d_model, bn))
    return cudaErrorInvalidValue;
  GemmArgs g = {};
  g.T = T;
  g.k_chunks = d.d_model / tcg::kBK / ksplit;
  g.m_per_cta = 1;
  g.m_valid = d.d_c + d.d_rope;
  g.d_c = d.d_c;
  g.d_rope = d.d_rope;
  g.out = ws;
  g.status = status;
  dim3 grid((d.d_c + d.d_rope + 127) / 128, (T + bn - 1) / bn, ksplit);
  return launch_bn<tcg::EPI_APPEND_PARTIAL, false>(bn, grid, a, a2, b, g, st);
}

cudaError_t launch_tc_absorb(const mla_dims_t& d, int T, const __nv_bfloat16* q, const int32_t* pos,
                             const __nv_bfloat16* w_uk, __nv_bfloat16* q_abs, cudaStream_t st) {
  // At most 64 tokens per tile: a CTA holds only two K chunks, and more, smaller
  // CTAs hide the load and store latencies better (256 rows: 41.0 -> 34.8 us).
  const int bn = pick_bn(T) > 64 ? 64 : pick_bn(T);
  const int dq = d.d_h + d.d_rope;
  CUtensorMap a, b;
  // W_UK as [n_h * d_h rows][d_c]: read MN-major (c contiguous) with 64-row K boxes.
  if (!map2d(&a, w_uk, d.d_c, (uint64_t)d.n_h * d.d_h, d.d_c, 64) ||
      !map2d(&b, q, (uint64_t)d.n_h * dq, T, (uint64_t)d.n_h * dq, bn))
    return cudaErrorInvalidValue;
  GemmArgs g = {};
  g.T = T;
  g.n_h = d.n_h;
  g.k_chunks = d.d_h / tcg::kBK;
  g.m_per_cta = 1;  // one CTA per (128-row tile of W_UK[h]^T, head)
  g.d_c = d.d_c;
  g.d_rope = d.d_rope;
  g.d_h = d.d_h;
  g.freqs = rope_freqs(d.d_rope, d.rope_theta);
  g.pos = pos;
  g.q = q;
  g.out = q_abs;
  dim3 grid(d.d_c / 128, (T + bn - 1) / bn, d.n_h);
  return launch_bn<tcg::EPI_ABSORB, true>(bn, grid, a, a, b, g, st);
}

cudaError_t launch_tc_out_proj(const mla_dims_t& d, int T, const __nv_bfloat16* o_lat,
                               const __nv_bfloat16* w_uv, __nv_bfloat16* o, cudaStream_t st) {
  const int bn = pick_bn_wide(T);
  CUtensorMap a, b;
  if (!map2d(&a, w_uv, d.d_c, (uint64_t)d.n_h * d.d_v, d.d_c, 128) ||
      !map2d(&b, o_lat, (uint64_t)d.n_h * d.d_c, T, (uint64_t)d.n_h * d.d_c, bn))
    return cudaErrorInvalidValue;
  GemmArgs g = {};
  g.T = T;
  g.n_h = d.n_h;
  g.k_chunks = d.d_c / tcg::kBK;
  g.m_per_cta = 1;
  g.d_c = d.d_c;
  g.d_v = d.d_v;
  g.out = o;
  dim3 grid(1, (T + bn - 1) / bn, d.n_h);
  return launch_bn<tcg::EPI_OUTPROJ, false>(bn, grid, a, a, b, g, st);
}

int tc_wo_ksplit(const mla_dims_t& d, int T) {
  // K = n_h * d_v in 64-wide chunks, split so that about two CTAs per SM stream
  // W_O (each split a whole number of chunks).
  const int m_tiles = (d.d_model + 127) / 128;
  const int n_tiles = (T + pick_bn(T) - 1) / pick_bn(T);
  const int k_chunks = d.n_h * d.d_v / tcg::kBK;
  int ks = (2 * sm_count() + m_tiles * n_tiles - 1) / (m_tiles * n_tiles);
  if (ks > 16) ks = 16;
  if (ks < 1) ks = 1;
  while (ks > 1 && k_chunks % ks != 0) --ks;
  return ks;
}

cudaError_t launch_tc_wo_gemm(const mla_dims_t& d, int T, const __nv_bfloat16* o, const __nv_bfloat16* w_o,
                              float* ws, int ksplit, int32_t* status, cudaStream_t st) {
  const int bn = pick_bn(T);
  const uint64_t K = (uint64_t)d.n_h * d.d_v;
  CUtensorMap a, b;
  if (!map2d(&a, w_o, K, d.d_model, K, 128) || !map2d(&b, o, K, T, K, bn)) return cudaErrorInvalidValue;
  GemmArgs g = {};
  g.T = T;
  g.k_chunks = (int)(K / tcg::kBK) / ksplit;
  g.m_per_cta = 1;
  g.m_valid = d.d_model;
  g.out = ws;
  g.status = status;
  dim3 grid((d.d_model + 127) / 128, (T + bn - 1) / bn, ksplit);
  return launch_bn<tcg::EPI_WO_PARTIAL, false>(bn, grid, a, a, b, g, st);
}

}  // namespace mla
