// Tensor-core MLA decode attention for B300 (sm_103a): tcgen05 MMAs with TMEM
// accumulators, TMA-staged cache tiles, and a 2-CTA cluster per worker.
//
// What it computes (per problem p = (sequence, query) and head h, the absorbed
// form of the page "MLA 之后，KV cache 确实得重新理解一遍", "第二步" and "RoPE
// 为什么必须解耦"):
//   s_t   = scale * q_abs[p,h] . [c_KV,t | k_R,t]   over the 576-wide cached entry
//   o_lat = sum_t softmax(s)_t c_KV,t               (latent weighted sum)
//   lse   = log sum_t exp(s_t)
//
// Layout of the work (one cluster of two CTAs per worker, 128 heads = MMA M):
//   * CTA r owns latent columns [256r, 256r+256) of c_KV and k_R columns
//     [32r, 32r+32). Every 64-token cache tile is loaded once: each CTA fetches
//     only its 288 columns, so HBM bytes are read exactly once.
//   * S_r = Q[:, cols_r] . K[:, cols_r]^T (M=128, N=64, K=288) lands in TMEM
//     (two S buffers, so Q.K^T of the next tile overlaps the softmax).
//   * Each CTA owns the softmax of half of the head rows: CTA r owns TMEM lanes
//     [16r, 16r+16) of every 32-lane quadrant. For the other half it sends its
//     partial scores to the peer (16-bit fixed point per half row, one bulk
//     copy per quadrant); for its own half it adds the peer's partial to its
//     own exact one, runs the online softmax (running max with lazy rescale,
//     exp2) and writes bf16 P for those rows into its own P buffer in shared
//     memory and, by bulk copy, into the peer's, with the rows' rescale
//     factors.
//   * P (all 128 rows, shared memory, two buffers) is the A operand of
//     O += P . V (M=128, N=256): each CTA accumulates its 256 latent columns of
//     O for every head in TMEM. O for 128 heads x 512 columns in fp32 would fill
//     one SM's tensor memory, which is why O is split across the pair.
//   * With an fp8 cache the tile's E4M3 codes and per-token scales are staged
//     by TMA and four converter warps write code * scale as bf16 into the same
//     tile layout, so the MMAs are those of the bf16 cache.
// Roles per CTA: warp 0 lane 0 issues TMA; warp 1 lane 0 copies the Q slice
// into TMEM and issues Q.K^T; warp 3 lane 0 issues P.V; warps 4-7 (one per
// TMEM lane quadrant) run the softmax of the CTA's own rows; warps 8-11 encode
// and send the partial scores of the peer's rows, apply the peer's rescale
// factors to those rows of O and write their output; warps 12-15 (fp8 cache
// only) convert tiles. Every wait is bounded: after 2 s the kernel records
// MLA_ERR_DEVICE_TIMEOUT in *status and unwinds.
#include "tc_decode.cuh"
#include "sm100_ptx.cuh"

#include <cuda.h>
#include <math.h>
#include <atomic>
#include <mutex>

namespace mla {
using namespace ptx;

namespace tcd {
constexpr int kRows = 128;
constexpr int kTile = kTcTileN;                          // 64 tokens
constexpr uint32_t kKvChunk = 64 * 128;                  // [64 tokens x 64 bf16], 128B swizzle
constexpr uint32_t kKvKrOff = 4 * kKvChunk;
constexpr uint32_t kKrBytes = 64 * 64;                   // [64 tokens x 32 bf16], 64B swizzle
constexpr uint32_t kSlotBytes = 4 * kKvChunk + kKrBytes;  // 36 KB
constexpr uint32_t kQChunk = 128 * 128;                  // [128 rows x 64 bf16]; two per ring slot
constexpr uint32_t kQkrBytes = 128 * 64;                 // [128 rows x 32 bf16], 64B swizzle
constexpr uint32_t kPBytes = 128 * 128;                  // P [128 rows x 64 tokens] bf16, 128B swizzle
// Partial scores travel as 16-bit fixed point: each half row (32 scores, one
// thread) is sent as its maximum mx, a power-of-two step q chosen from the half
// row's range (mx - min < 2^15 q), and 32 unsigned offsets e = round((mx - s)/q),
// decoded as mx - e q. The error is at most q/2, under range * 2^-15. A quadrant
// sends 32 threads x 64 bytes of offsets ([k][thread][16 B]) then 32 x 8 bytes
// of references.
constexpr uint32_t kXRefOff = 32 * 64;
constexpr uint32_t kXQuad = kXRefOff + 32 * 8;           // 2304
constexpr uint32_t kXTile = 4 * kXQuad;                  // 9216 per tile
constexpr int kRecvBufs = 2;                             // tile j lands in buffer j % 2
constexpr int kPBufs = 1;                                // P buffers (tile j in buffer j % kPBufs)
constexpr uint32_t kPRemoteBytes = 4 * 2048 + 64 * 4;    // the peer's 64 P rows + their factors
// fp8 staging: E4M3 codes [64 tokens x 256] then per-token scales [64].
constexpr uint32_t kStCodes = 64 * 256;
constexpr uint32_t kStBytes = 17 * 1024;
constexpr int kStages8 = 2;

constexpr int kMaxSlots = 6;

template <bool FP8>
struct Cfg {
  static constexpr int kSlots = FP8 ? 4 : 5;
  static constexpr uint32_t OFF_SLOTS = 0;
  static constexpr uint32_t OFF_P = OFF_SLOTS + kSlots * kSlotBytes;
  static constexpr uint32_t OFF_QKR = OFF_P + kPBufs * kPBytes;
  static constexpr uint32_t OFF_RECV = OFF_QKR + kQkrBytes;
  static constexpr uint32_t OFF_FACT = OFF_RECV + kRecvBufs * kXTile;  // [kPBufs][128] fp32 rescale factors from the peer
  static constexpr uint32_t OFF_LREC = OFF_FACT + kPBufs * 512;        // [2][128] fp32 1/l from the peer
  static constexpr uint32_t OFF_STAGE = (OFF_LREC + 2 * 512 + 1023) & ~1023u;
  static constexpr uint32_t OFF_BAR = OFF_STAGE + (FP8 ? kStages8 * kStBytes : 0);
  static constexpr uint32_t kSmemBytes = OFF_BAR + 512 + 1024;  // barriers, flags, alignment slack
  static constexpr int kWarps = FP8 ? 16 : 12;
  static constexpr int kThreads = 32 * kWarps;
  static_assert(OFF_P % 1024 == 0 && OFF_QKR % 1024 == 0 && OFF_STAGE % 1024 == 0, "alignment");
  static_assert(kSmemBytes <= 232448, "shared memory");
  static_assert(kSlots <= kMaxSlots, "barrier slots");
};

enum Bar {
  B_KVFULL = 0,                   // + slot
  B_KVEMPTY = kMaxSlots,          // + slot
  B_QKRFULL = 2 * kMaxSlots,
  B_QKREMPTY,
  B_SFULL,            // + S buffer: Q.K^T of a tile committed
  B_SFREE = B_SFULL + 2,   // + S buffer: the softmax and exchange warps have read it
  B_RECV = B_SFREE + 2,    // + receive buffer: the peer's partial scores have landed
  B_PREM = B_RECV + kRecvBufs,  // + P buffer: the peer's P rows and factors have landed
  B_OWNP = B_PREM + kPBufs,       // + P buffer: this CTA's P rows are written
  B_RESC = B_OWNP + kPBufs,       // + P buffer: the peer's rescale factors are applied to O
  B_PVDONE = B_RESC + kPBufs,     // + P buffer: this CTA's P.V of the buffer's tile is done
  B_PVPEER = B_PVDONE + kPBufs,   // + P buffer: the peer's P.V of the buffer's tile is done
  B_OFREE = B_PVPEER + kPBufs,    // O has been read out (segment end)
  B_LFULL,                 // + segment parity: the peer's 1/l for its rows has landed
  B_STFULL = B_LFULL + 2,  // + fp8 stage
  B_STEMPTY = B_STFULL + kStages8,
  NBAR = B_STEMPTY + kStages8
};
static_assert(8 * NBAR + 16 <= 512, "barrier area");
// TMEM columns: O (this CTA's 256 latent columns), two S buffers, the Q slice's c_KV part.
constexpr uint32_t TM_O = 0, TM_S = 256, TM_Q = 384, kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by 2^8
}  // namespace tcd

namespace {

struct Ctl {
  int32_t* status;
  volatile int* abort;
};

__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctl& c,
                                         bool cluster_scope = false) {
  auto probe = [&]() {
    return cluster_scope ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
  };
  if (probe()) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t i = 1;; ++i) {
    if (probe()) return true;
    if ((i & 63) == 0) {
      if (*c.abort) return false;
      if (globaltimer() - t0 > tcd::kWaitNs) {
        set_status(c.status, MLA_ERR_DEVICE_TIMEOUT);
        *c.abort = 1;
        return false;
      }
    }
  }
}
// Warp-wide bounded wait: every lane gets the same answer.
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctl& c, bool cluster_scope = false) {
  return __all_sync(0xffffffffu, wait_bar(bar, parity, c, cluster_scope));
}

// Walks one worker's share of the tile sequence as segments (problem, tile range).
struct SegIter {
  const int32_t* cum;
  const int32_t* pbase;
  const int32_t* lens;
  const int32_t* pw0;
  const int32_t* pcnt;
  const int32_t* los;
  const int32_t* tfs;
  int w, g0, g1, p;
  __device__ void init(const int32_t* plan, int worker) {
    PlanView pv = plan_view(plan);
    cum = pv.cum;
    pbase = pv.pbase;
    lens = pv.len;
    pw0 = pv.pw0;
    pcnt = pv.pcnt;
    los = pv.lo;
    tfs = pv.tf;
    w = worker;
    g0 = pv.wstart[worker];
    g1 = pv.wstart[worker + 1];
    p = pv.first[worker];  // the problem holding the first tile (one load, no search)
  }
  // Tiles [t_lo, t_hi) of problem `prob`, counted from its first tile (key
  // block tf); its visible keys are the positions [lo, len).
  __device__ bool next(int& prob, int& t_lo, int& t_hi, int& len, int& whole, int& slot, int& lo, int& tf) {
    if (g0 >= g1) return false;
    while (cum[p + 1] <= g0) ++p;
    t_lo = g0 - cum[p];
    t_hi = min(g1, cum[p + 1]) - cum[p];
    len = lens[p];
    lo = los[p];
    tf = tfs[p];
    whole = (pcnt[p] == 1);
    slot = pbase[p] + (w - pw0[p]);
    prob = p;
    g0 = cum[p] + t_hi;
    ++p;
    return true;
  }
};

// A tile of the worker's sequence with everything the softmax needs about it.
struct TileCursor {
  SegIter it;
  bool valid_tile;
  int p, t_lo, t_hi, len, whole, pslot, lo, tf;  // segment
  int k;                                         // position in the segment
  uint32_t entry;                                // ring entry that holds the tile
  __device__ void start(const int32_t* plan, int worker) {
    it.init(plan, worker);
    valid_tile = it.next(p, t_lo, t_hi, len, whole, pslot, lo, tf);
    k = 0;
    entry = 2;  // the segment's two Q entries come first
  }
  __device__ void advance() {
    ++k;
    ++entry;
    if (t_lo + k >= t_hi) {
      valid_tile = it.next(p, t_lo, t_hi, len, whole, pslot, lo, tf);
      k = 0;
      entry += 2;
    }
  }
  __device__ bool first() const { return k == 0; }
  __device__ bool last() const { return t_lo + k == t_hi - 1; }
  // Visible columns [vlo(), vhi()) of the current tile.
  __device__ int vhi() const { return min(tcd::kTile, len - (tf + t_lo + k) * tcd::kTile); }
  __device__ int vlo() const { return max(0, lo - (tf + t_lo + k) * tcd::kTile); }
};

// The next tile to stage in a worker's share: only whether it exists and how
// many of its tokens are inside its sequence (a light cursor, few registers).
struct TileAhead {
  const int32_t* cum;
  const int32_t* lens;
  const int32_t* los;
  const int32_t* tfs;
  int g, g1, p, c0, c1, len, lo, tf;  // tile index; problem p holds tiles [c0, c1)
  __device__ void start(const int32_t* plan, int worker) {
    const PlanView pv = plan_view(plan);
    cum = pv.cum;
    lens = pv.len;
    los = pv.lo;
    tfs = pv.tf;
    g = pv.wstart[worker];
    g1 = pv.wstart[worker + 1];
    p = pv.first[worker];
    c0 = c1 = 0;
    len = 0;
    locate();
  }
  __device__ void locate() {
    if (g >= g1 || g < c1) return;
    while (cum[p + 1] <= g) ++p;
    c0 = cum[p];
    c1 = cum[p + 1];
    len = lens[p];
    lo = los[p];
    tf = tfs[p];
  }
  __device__ bool valid_tile() const { return g < g1; }
  __device__ int vhi() const { return min(tcd::kTile, len - (tf + g - c0) * tcd::kTile); }
  __device__ int vlo() const { return max(0, lo - (tf + g - c0) * tcd::kTile); }
  __device__ void advance() {
    ++g;
    locate();
  }
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
__device__ __forceinline__ float fmin3(float a, float b, float c) {
  float d;
  asm("min.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}
// (d0, d1) = (a0, a1) * b + c on the paired fp32 pipe.
__device__ __forceinline__ void ffma2(float& d0, float& d1, float a0, float a1, float b, float c) {
  asm("{\n .reg .b64 ra, rb, rc, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rb, {%4, %4};\n"
      " mov.b64 rc, {%5, %5};\n fma.rn.f32x2 rd, ra, rb, rc;\n mov.b64 {%0, %1}, rd;\n}"
      : "=f"(d0), "=f"(d1)
      : "f"(a0), "f"(a1), "f"(b), "f"(c));
}
// (d0, d1) += (a0, a1) on the paired fp32 pipe.
__device__ __forceinline__ void fadd2(float& d0, float& d1, float a0, float a1) {
  asm("{\n .reg .b64 ra, rd;\n mov.b64 ra, {%2, %3};\n mov.b64 rd, {%0, %1};\n"
      " add.rn.f32x2 rd, rd, ra;\n mov.b64 {%0, %1}, rd;\n}"
      : "+f"(d0), "+f"(d1)
      : "f"(a0), "f"(a1));
}

// Maximum and minimum of the scores in columns [vlo, vhi) of 32 (all 32 when
// vlo <= 0 and vhi >= 32).
__device__ __forceinline__ void range32(const uint32_t (&sv)[32], int vlo, int vhi, float& mx, float& mn) {
  if (vlo <= 0 && vhi >= 32) {
    float a[11], c[11];
#pragma unroll
    for (int x = 0; x < 10; ++x) {
      const float v0 = __uint_as_float(sv[3 * x]), v1 = __uint_as_float(sv[3 * x + 1]),
                  v2 = __uint_as_float(sv[3 * x + 2]);
      a[x] = fmax3(v0, v1, v2);
      c[x] = fmin3(v0, v1, v2);
    }
    a[10] = fmaxf(__uint_as_float(sv[30]), __uint_as_float(sv[31]));
    c[10] = fminf(__uint_as_float(sv[30]), __uint_as_float(sv[31]));
    mx = fmax3(fmax3(a[0], a[1], a[2]), fmax3(a[3], a[4], a[5]), fmax3(a[6], a[7], fmax3(a[8], a[9], a[10])));
    mn = fmin3(fmin3(c[0], c[1], c[2]), fmin3(c[3], c[4], c[5]), fmin3(c[6], c[7], fmin3(c[8], c[9], c[10])));
  } else {
    mx = -INFINITY;
    mn = INFINITY;
#pragma unroll
    for (int x = 0; x < 32; ++x) {
      if (x >= vlo && x < vhi) {
        mx = fmaxf(mx, __uint_as_float(sv[x]));
        mn = fminf(mn, __uint_as_float(sv[x]));
      }
    }
  }
}

// Byte offset of 16-byte unit u (8 bf16) of row r in a [rows x 64] bf16 tile
// with the 128-byte swizzle (8-row groups of 1024 bytes, unit index XOR row % 8).
__device__ __forceinline__ uint32_t sw128_off(int r, int u) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((u ^ (r & 7)) << 4));
}

// Writes 32 fp32 values of one O row (times inv) to o_lat (bf16, whole problem)
// or to a piece-major partial slot. `col` is the row's first latent column.
__device__ __forceinline__ void store_o_row(const uint32_t (&o)[32], float inv, bool whole, size_t grow, int r,
                                            int pslot, int col, __nv_bfloat16* o_lat, float* o_part) {
  if (whole) {
    uint4* dst = reinterpret_cast<uint4*>(o_lat + grow * 512 + col);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      uint32_t w4[4];
#pragma unroll
      for (int e2 = 0; e2 < 4; ++e2) {
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[q4 * 8 + 2 * e2]) * inv,
                                                        __uint_as_float(o[q4 * 8 + 2 * e2 + 1]) * inv);
        w4[e2] = *reinterpret_cast<const uint32_t*>(&h2);
      }
      dst[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
  } else {
    // Partials are piece-major: [slot][32-column chunk][4-column piece][row][4].
    float4* dst = reinterpret_cast<float4*>(o_part + ((size_t)pslot * 16 + col / 32) * 8 * tcd::kRows * 4) + r;
#pragma unroll
    for (int q4 = 0; q4 < 8; ++q4)
      dst[q4 * tcd::kRows] = make_float4(__uint_as_float(o[4 * q4]) * inv, __uint_as_float(o[4 * q4 + 1]) * inv,
                                         __uint_as_float(o[4 * q4 + 2]) * inv, __uint_as_float(o[4 * q4 + 3]) * inv);
  }
}
}  // namespace

template <bool FP8>
__global__ void __launch_bounds__(tcd::Cfg<FP8>::kThreads, 1)
tc_decode_kernel(const __grid_constant__ CUtensorMap tm_q64, const __grid_constant__ CUtensorMap tm_q32,
                 const __grid_constant__ CUtensorMap tm_kv, const __grid_constant__ CUtensorMap tm_kr,
                 const __grid_constant__ CUtensorMap tm_sc, const int32_t* __restrict__ plan,
                 const int32_t* __restrict__ bt, int max_pages, int page_size, int box_rows, int64_t num_pages,
                 int oob_row, int q_per_seq, float scale_log2, float* __restrict__ o_part,
                 float* __restrict__ lse_part, __nv_bfloat16* __restrict__ o_lat, float* __restrict__ lse_out,
                 int32_t* status) {
  using namespace tcd;
  using C = Cfg<FP8>;
  constexpr int S = C::kSlots;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int worker = (int)cluster_id_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto BAR = [&](int i) { return base + C::OFF_BAR + 8u * (uint32_t)i; };
  auto SLOT = [&](uint32_t e) { return base + C::OFF_SLOTS + (e % S) * kSlotBytes; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + C::OFF_BAR + 8 * NBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + C::OFF_BAR + 8 * NBAR + 8);

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      uint32_t count = 1;
      if (i >= B_KVFULL && i < B_KVFULL + kMaxSlots) count = FP8 ? 5 : 1;
      if (i == B_SFREE || i == B_SFREE + 1 || i == B_OFREE) count = 8;
      if ((i >= B_RECV && i < B_PVDONE) || i == B_LFULL || i == B_LFULL + 1 ||
          (i >= B_STEMPTY && i < B_STEMPTY + kStages8))
        count = 4;  // receive buffers, the peer's P, own P, applied factors, 1/l, fp8 stages
      mbar_init(BAR(i), count);
    }
    // Buffers filled by the peer start armed for their first uses; each of the
    // four consuming warps re-arms its share once it has read a buffer.
    for (int w = 0; w < 4; ++w) {
      for (int b = 0; b < kRecvBufs; ++b) mbar_arrive_expect_tx(BAR(B_RECV + b), kXQuad);
      for (int b = 0; b < kPBufs; ++b) mbar_arrive_expect_tx(BAR(B_PREM + b), kPRemoteBytes / 4);
      for (int b = 0; b < 2; ++b) mbar_arrive_expect_tx(BAR(B_LFULL + b), 16 * 4);
    }
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q64);
    prefetch_tmap(&tm_q32);
    prefetch_tmap(&tm_kv);
    prefetch_tmap(&tm_kr);
    if (FP8) prefetch_tmap(&tm_sc);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  cluster_arrive();
  cluster_wait();
  const uint32_t tmem = *tmem_slot;
  const Ctl ctl{status, abort_flag};
  pdl_wait();  // set-up above overlaps the previous kernel; its outputs are read below

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot, lo, tf;
      uint32_t seg = 0, e = 0, jt = 0;
      bool ok = true;
      auto acquire = [&](uint32_t ee) -> bool {
        return ee < (uint32_t)S || wait_bar(BAR(B_KVEMPTY + ee % S), ((ee / S) - 1) & 1, ctl);
      };
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot, lo, tf)) {
        const int row0 = p * kRows;
        // The c_KV part of the Q slice, staged in two ring slots on its way to TMEM.
        for (int h = 0; h < 2 && ok; ++h, ++e) {
          if (!acquire(e)) { ok = false; break; }
          const uint32_t full = BAR(B_KVFULL + e % S);
          mbar_arrive_expect_tx(full, 2 * kQChunk);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(SLOT(e) + c * kQChunk, &tm_q64, (int)rank * 256 + (2 * h + c) * 64, row0, full);
        }
        if (!ok) break;
        // The k_R part of the Q slice stays in shared memory.
        if (seg > 0 && !wait_bar(BAR(B_QKREMPTY), (seg - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(BAR(B_QKRFULL), kQkrBytes);
        tma_load_2d(base + C::OFF_QKR, &tm_q32, 512 + (int)rank * 32, row0, BAR(B_QKRFULL));
        const int b = p / q_per_seq;
        // Pool row of the box of tokens [tok, tok + box_rows) of this problem, or
        // -1 when none of them is visible (past the end, or wholly before the
        // window, whose pages may be gone) / -2 on a bad page.
        auto box_row = [&](int tok) -> int {
          if (tok >= len || tok + box_rows <= lo) return -1;
          const int pg = tok / page_size;
          const int page = pg < max_pages ? bt[(size_t)b * max_pages + pg] : -1;
          if (page < 0 || page >= num_pages) return -2;
          return page * page_size + tok % page_size;
        };
        for (int t = t_lo; t < t_hi; ++t, ++e, ++jt) {
          if (!acquire(e)) { ok = false; break; }
          const uint32_t full = BAR(B_KVFULL + e % S);
          const uint32_t st = SLOT(e);
          if (!FP8) {
            mbar_arrive_expect_tx(full, kSlotBytes);
            for (int r0 = 0; r0 < kTile; r0 += box_rows) {
              int y = box_row((tf + t) * kTile + r0);
              if (y == -2) set_status(status, MLA_ERR_BAD_PAGE);
              if (y < 0) y = oob_row;  // fully out of range: the copy fills zeros
              for (int c = 0; c < 4; ++c)
                tma_load_2d(st + c * kKvChunk + r0 * 128, &tm_kv, (int)rank * 256 + c * 64, y, full);
              tma_load_2d(st + kKvKrOff + r0 * 64, &tm_kr, 512 + (int)rank * 32, y, full);
            }
          } else {
            // k_R straight into the tile; codes and scales into a staging buffer.
            if (jt >= (uint32_t)kStages8 &&
                !wait_bar(BAR(B_STEMPTY + jt % kStages8), ((jt / kStages8) - 1) & 1, ctl)) {
              ok = false;
              break;
            }
            const uint32_t sfull = BAR(B_STFULL + jt % kStages8);
            const uint32_t stg = base + C::OFF_STAGE + (jt % kStages8) * kStBytes;
            mbar_arrive_expect_tx(full, kKrBytes);
            mbar_arrive_expect_tx(sfull, kStCodes + kTile * 4);
            for (int r0 = 0; r0 < kTile; r0 += box_rows) {
              int y = box_row((tf + t) * kTile + r0);
              if (y == -2) set_status(status, MLA_ERR_BAD_PAGE);
              if (y < 0) y = oob_row;
              tma_load_2d(st + kKvKrOff + r0 * 64, &tm_kr, (int)rank * 32, y, full);
              tma_load_2d(stg + r0 * 256, &tm_kv, (int)rank * 256, y, sfull);
              tma_load_1d(stg + kStCodes + r0 * 4, &tm_sc, y, sfull);
            }
          }
        }
        ++seg;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ Q.K^T issuer
    // Copies a segment's Q slice into TMEM, then issues Q.K^T for each tile into
    // S buffer j % 2 once its tile, the buffer and the Q slice are ready.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false, false);
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot, lo, tf;
      uint32_t e = 0, j = 0, sidx = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot, lo, tf)) {
        if (!wait_bar(BAR(B_KVFULL + e % S), (e / S) & 1, ctl) ||
            !wait_bar(BAR(B_KVFULL + (e + 1) % S), ((e + 1) / S) & 1, ctl))
          break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h) {
          const uint32_t st = SLOT(e + h);
          for (int c = 0; c < 2; ++c)
            for (int kk = 0; kk < 4; ++kk)
              tmem_cp_128x256b(tmem + TM_Q + (2 * h + c) * 32 + kk * 8,
                               smem_desc(st + c * kQChunk + kk * 32, 16, 1024, kSwizzle128B));
          mma_commit(BAR(B_KVEMPTY + (e + h) % S));
        }
        e += 2;
        if (!wait_bar(BAR(B_QKRFULL), sidx & 1, ctl)) break;
        for (int t = t_lo; t < t_hi; ++t, ++e, ++j) {
          const uint32_t sb = j & 1;
          if (!wait_bar(BAR(B_KVFULL + e % S), (e / S) & 1, ctl) ||
              (j >= 2 && !wait_bar(BAR(B_SFREE + sb), ((j - 2) >> 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = SLOT(e), d = tmem + TM_S + 64 * sb;
          for (int c = 0; c < 4; ++c)
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(d, tmem + TM_Q + c * 32 + kk * 8,
                         smem_desc(st + c * kKvChunk + kk * 32, 16, 1024, kSwizzle128B), idesc_s, (c | kk) ? 1u : 0u);
          for (int kk = 0; kk < 2; ++kk)
            mma_f16(d, smem_desc(base + C::OFF_QKR + kk * 32, 16, 512, kSwizzle64B),
                    smem_desc(st + kKvKrOff + kk * 32, 16, 512, kSwizzle64B), idesc_s, 1u);
          mma_commit(BAR(B_SFULL + sb));
          if (t == t_hi - 1) mma_commit(BAR(B_QKREMPTY));
        }
        ++sidx;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ P.V issuer
    // O += P . V for tile j once both halves of P (this CTA's rows and the
    // peer's) are in P buffer j % 2 and the peer's rescale factors are applied;
    // the first tile of a segment also waits until the previous O was read out.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot, lo, tf;
      uint32_t e = 0, j = 0, sidx = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot, lo, tf)) {
        e += 2;  // the segment's Q entries
        for (int t = t_lo; t < t_hi; ++t, ++e, ++j) {
          const bool first = (t == t_lo);
          const uint32_t pb = j % kPBufs, pph = (j / kPBufs) & 1;
          if (!wait_bar(BAR(B_OWNP + pb), pph, ctl) || !wait_bar(BAR(B_RESC + pb), pph, ctl) ||
              (first && sidx > 0 && !wait_bar(BAR(B_OFREE), (sidx - 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = SLOT(e), pa = base + C::OFF_P + pb * kPBytes;
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_f16(tmem + TM_O, smem_desc(pa + kk * 32, 16, 1024, kSwizzle128B),
                    smem_desc(st + kk * 2048, kKvChunk, 1024, kSwizzle128B), idesc_pv, (first && kk == 0) ? 0u : 1u);
          mma_commit(BAR(B_KVEMPTY + e % S));
          mma_commit(BAR(B_PVDONE + pb));
          // The peer learns of it on a barrier of its own: one arrival source
          // per barrier keeps its phases in order.
          mma_commit_multicast(BAR(B_PVPEER + pb), (uint16_t)(1u << peer));
        }
        ++sidx;
      }
    }
  } else if (warp >= 4 && warp < 8) {
    // ------------------------------------------------------------ softmax of this CTA's rows
    // Warp qd owns TMEM lanes [32qd + 16 rank, +16): thread t holds head row
    // 32qd + 16 rank + t % 16 and score columns 32 (t / 16) .. + 32 of each tile.
    const int qd = warp & 3, hh = lane >> 4;
    const int row = qd * 32 + 16 * (int)rank + (lane & 15);
    const uint32_t lane_off = (uint32_t)(qd * 32 + 16 * (int)rank) << 16;
    const uint32_t p_rows = (uint32_t)(qd * 32 + 16 * (int)rank) * 128;  // this warp's 2 KB of each P buffer
    const uint32_t p_peer = mapa(base + C::OFF_P, peer);
    const uint32_t prem_peer = mapa(BAR(B_PREM), peer);
    const uint32_t fact_peer = mapa(base + C::OFF_FACT, peer);
    const uint32_t lrec_peer = mapa(base + C::OFF_LREC, peer);
    const uint32_t lfull_peer = mapa(BAR(B_LFULL), peer);
    TileCursor cur;
    cur.start(plan, worker);
    float m_ref = -INFINITY, l = 0.f;
    uint32_t seg = 0;
    bool ok = true;
    uint32_t j = 0;
    for (; ok && cur.valid_tile; ++j) {
      const uint32_t sb = j & 1;
      // a. This CTA's exact partial scores of its rows.
      if (!wait_warp(BAR(B_SFULL + sb), (j >> 1) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld16x2_32<32>(tmem + lane_off + TM_S + 64 * sb, sv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_SFREE + sb));
      // b. Add the peer's partial: mx - e q = (2^23 + e) (-q) + (mx + 2^23 q),
      //    the offset becoming a float by putting 0x4B00 above its 16 bits.
      const uint32_t rb = j % kRecvBufs;
      if (!wait_warp(BAR(B_RECV + rb), (j / kRecvBufs) & 1, ctl, true)) { ok = false; break; }
      float s[32];
      {
        const uint8_t* recv = gbase + C::OFF_RECV + rb * kXTile + qd * kXQuad;
        const uint2 ref = *reinterpret_cast<const uint2*>(recv + kXRefOff + lane * 8);
        const float peer_mx = __uint_as_float(ref.x), peer_q = __uint_as_float(ref.y);
        const float k_peer = fmaf(8388608.f, peer_q, peer_mx);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(recv + k * 512 + lane * 16);
          const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int x = 8 * k + 2 * i;
            float b0, b1;
            ffma2(b0, b1, __uint_as_float(__byte_perm(pw[i], 0x4B000000u, 0x7610)),
                  __uint_as_float(__byte_perm(pw[i], 0x4B000000u, 0x7632)), -peer_q, k_peer);
            s[x] = __uint_as_float(sv[x]);
            s[x + 1] = __uint_as_float(sv[x + 1]);
            fadd2(s[x], s[x + 1], b0, b1);
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(BAR(B_RECV + rb), kXQuad);
      const bool first = cur.first(), last = cur.last();
      const int vlo = cur.vlo(), vhi = cur.vhi();
      const uint32_t tile_entry = cur.entry;
      const int p = cur.p, whole = cur.whole, pslot = cur.pslot;
      cur.advance();
      // c. Online softmax in log2 units. Tokens past the end (only in a
      //    sequence's last tile) or before the window (only in its first) are
      //    masked; the maximum is taken on the raw scores and the scale is
      //    folded into the exponent's multiply-add.
      if (vlo > 0 || vhi < kTile) {
#pragma unroll
        for (int x = 0; x < 32; ++x)
          if (32 * hh + x < vlo || 32 * hh + x >= vhi) s[x] = -INFINITY;
      }
      if (first) {
        m_ref = -INFINITY;
        l = 0.f;
      }
      float mx[12];
#pragma unroll
      for (int x = 0; x < 10; ++x) mx[x] = fmax3(s[3 * x], s[3 * x + 1], s[3 * x + 2]);
      mx[10] = s[30];
      mx[11] = s[31];
#pragma unroll
      for (int x = 0; x < 4; ++x) mx[x] = fmax3(mx[3 * x], mx[3 * x + 1], mx[3 * x + 2]);
      float mrow = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      mrow = fmaxf(mrow, __shfl_xor_sync(0xffffffffu, mrow, 16));
      const float mt = mrow * scale_log2;
      const bool need = (m_ref == -INFINITY) || (mt > m_ref + kRescaleThreshold);
      const float m_new = need ? fmaxf(mt, m_ref) : m_ref;
      const float factor = need ? ex2_approx(m_ref - m_new) : 1.f;
      uint32_t pk[16];
      float ps0 = 0.f, ps1 = 0.f, ps2 = 0.f, ps3 = 0.f;
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float e0, e1;
        ffma2(e0, e1, s[2 * x], s[2 * x + 1], scale_log2, -m_new);
        e0 = ex2_approx(e0);
        e1 = ex2_approx(e1);
        const __nv_bfloat162 h2 = __floats2bfloat162_rn(e0, e1);
        pk[x] = *reinterpret_cast<const uint32_t*>(&h2);
        if (x & 1) fadd2(ps2, ps3, e0, e1);
        else fadd2(ps0, ps1, e0, e1);
      }
      l = l * factor + ((ps0 + ps1) + (ps2 + ps3));
      m_ref = m_new;
      const bool rescale = need && !first;
      // d. P buffer pb is free once P.V of tile j - kPBufs has completed in
      //    both CTAs; O can be rescaled once this CTA's P.V of tile j - 1 has.
      const uint32_t pb = j % kPBufs;
      if (j >= (uint32_t)kPBufs &&
          (!wait_warp(BAR(B_PVDONE + pb), ((j - kPBufs) / kPBufs) & 1, ctl) ||
           !wait_warp(BAR(B_PVPEER + pb), ((j - kPBufs) / kPBufs) & 1, ctl, true))) { ok = false; break; }
      if (__any_sync(0xffffffffu, rescale)) {
        if (!wait_warp(BAR(B_PVDONE + (j - 1) % kPBufs), ((j - 1) / kPBufs) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
        const float f = rescale ? factor : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t ta = tmem + lane_off + TM_O + 32 * cc;
          tmem_ld16x2_32<128>(ta, o);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
          tmem_st16x2_32<128>(ta, o);
        }
        tmem_wait_st();
      }
      // e. P of this warp's rows into buffer pb: here for this CTA's P.V, and by
      //    bulk copy into the peer's buffer with the rows' rescale factors.
      if (lane == 0) {  // the copy of tile j - kPBufs has read this buffer
        if (kPBufs == 1) bulk_wait_read_all();
        else bulk_wait_read_1();
      }
      __syncwarp();
      uint8_t* pbuf = gbase + C::OFF_P + pb * kPBytes;
#pragma unroll
      for (int u = 0; u < 4; ++u)
        *reinterpret_cast<uint4*>(pbuf + sw128_off(row, 4 * hh + u)) =
            make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
      if (vlo > 0 || vhi < kTile) {
        // Rows past the sequence end or before the window may hold anything
        // (NaN): zero their latent part so that P = 0 times V cannot poison O.
        uint8_t* st = gbase + C::OFF_SLOTS + (tile_entry % S) * kSlotBytes;
        const int n_lo = vlo, words = (n_lo + (kTile - vhi)) * 32;
        for (int i = qd * 32 + lane; i < words; i += 128) {
          const int k = i / 32, wd = i % 32;
          const int r = k < n_lo ? k : vhi + (k - n_lo);
          *reinterpret_cast<uint4*>(st + (wd >> 3) * kKvChunk + r * 128 + (wd & 7) * 16) = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(BAR(B_OWNP + pb));
        bulk_copy_to_peer(p_peer + pb * kPBytes + p_rows, base + C::OFF_P + pb * kPBytes + p_rows, 2048,
                          prem_peer + 8u * pb);
        bulk_commit();
      }
      if (hh == 0)
        st_async_b32(fact_peer + pb * 512 + row * 4, __float_as_uint(rescale ? factor : 1.f), prem_peer + 8u * pb);
      if (!last) continue;
      // f. Segment end: 1/l of this CTA's rows to the peer, then O of these rows out.
      const float l_row = l + __shfl_xor_sync(0xffffffffu, l, 16);
      const float inv_l = 1.f / l_row;
      if (hh == 0)
        st_async_b32(lrec_peer + (seg & 1) * 512 + row * 4, __float_as_uint(inv_l), lfull_peer + 8u * (seg & 1));
      if (!wait_warp(BAR(B_PVDONE + pb), (j / kPBufs) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const size_t grow = (size_t)p * kRows + row;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld16x2_32<128>(tmem + lane_off + TM_O + 32 * cc, o);
        tmem_wait_ld();
        store_o_row(o, inv_l, whole, grow, row, pslot, (int)rank * 256 + hh * 128 + 32 * cc, o_lat, o_part);
      }
      if (hh == 0) {
        const float lse = (m_ref + log2f(l_row)) * 0.69314718055994531f;
        if (whole) lse_out[grow] = lse;
        else lse_part[(size_t)pslot * kRows + row] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_OFREE));
      ++seg;
    }
    // The peer's completions of its last P.V tiles have not been waited for:
    // consume them (in phase order) so that none is still arriving when this
    // CTA exits.
    for (uint32_t t = (j > (uint32_t)kPBufs ? j - kPBufs : 0); ok && t < j; ++t)
      ok = wait_warp(BAR(B_PVPEER + t % kPBufs), (t / kPBufs) & 1, ctl, true);
    if (lane == 0) bulk_wait_read_all();
  } else if (warp >= 8 && warp < 12) {
    // ------------------------------------------------------------ the peer's rows
    // Warp 8 + qd holds TMEM lanes [32qd + 16 peer, +16) (rows whose softmax
    // the peer runs): it encodes this CTA's partial scores of those rows for
    // the peer, applies the peer's rescale factors to those rows of O, and
    // writes their output at segment ends.
    const int qd = warp & 3, hh = lane >> 4;
    const int row = qd * 32 + 16 * (int)peer + (lane & 15);
    const uint32_t lane_off = (uint32_t)(qd * 32 + 16 * (int)peer) << 16;
    const uint32_t recv_peer = mapa(base + C::OFF_RECV, peer) + qd * kXQuad;
    const uint32_t bar_recv_peer = mapa(BAR(B_RECV), peer);
    // Stage tile jj: load, encode (columns outside the visible [vlo, vhi) are
    // left out of the range) and store this quadrant's part straight into the peer's
    // receive buffer jj % kRecvBufs. The tile that buffer held before
    // (jj - kRecvBufs) the peer had consumed before it sent the P of that tile,
    // which this warp has already waited for.
    auto stage = [&](uint32_t jj, int vlo, int vhi) -> bool {
      const uint32_t sb = jj & 1;
      if (!wait_warp(BAR(B_SFULL + sb), (jj >> 1) & 1, ctl)) return false;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld16x2_32<32>(tmem + lane_off + TM_S + 64 * sb, sv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_SFREE + sb));
      float mx, mn;
      range32(sv, vlo - 32 * hh, vhi - 32 * hh, mx, mn);
      // Step q = 2^-k with range < 2^(E+1) <= 2^15 q, E the range's exponent;
      // k is capped at 60 for (near) constant half rows.
      const int eb = max((int)((__float_as_uint(mx - mn) >> 23) & 0xFFu), 81);
      const float enc = __uint_as_float((uint32_t)(268 - eb) << 23);  // 2^k
      const float q = __uint_as_float((uint32_t)(eb - 14) << 23);    // 2^-k
      // y = 2^23 + round((mx - s) 2^k): its low 16 bits are the offset.
      uint32_t w[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float d0, d1, y0, y1;
        ffma2(d0, d1, __uint_as_float(sv[2 * x]), __uint_as_float(sv[2 * x + 1]), -1.f, mx);
        ffma2(y0, y1, d0, d1, enc, 8388608.f);
        w[x] = __byte_perm(__float_as_uint(y0), __float_as_uint(y1), 0x5410);
      }
      const uint32_t b = jj % kRecvBufs;
      const uint32_t dst = recv_peer + b * kXTile, dbar = bar_recv_peer + 8u * b;
#pragma unroll
      for (int k = 0; k < 4; ++k)
        st_async_v4(dst + k * 512 + lane * 16, w[4 * k], w[4 * k + 1], w[4 * k + 2], w[4 * k + 3], dbar);
      st_async_b32(dst + kXRefOff + lane * 8, __float_as_uint(mx), dbar);
      st_async_b32(dst + kXRefOff + lane * 8 + 4, __float_as_uint(q), dbar);
      return true;
    };
    TileCursor cur;
    TileAhead ahead;  // the next tile to stage
    cur.start(plan, worker);
    ahead.start(plan, worker);
    bool ok = true;
    if (ahead.valid_tile()) {
      ok = stage(0, ahead.vlo(), ahead.vhi());
      ahead.advance();
    }
    uint32_t seg = 0;
    for (uint32_t j = 0; ok && cur.valid_tile; ++j) {
      const uint32_t pb = j % kPBufs;
      // Tile j + 1 is staged before this tile's factors are applied, so that
      // its exchange overlaps the peer's softmax of tile j. With a 3-slot ring
      // the first tile of a new segment (two Q entries after tile j) reuses
      // tile j's slot, which P.V of tile j frees only after this warp's
      // RESC(j): there the order is reversed.
      const bool stage_late = (S < 4) && cur.last();
      if (ahead.valid_tile() && !stage_late) {
        if (!stage(j + 1, ahead.vlo(), ahead.vhi())) { ok = false; break; }
        ahead.advance();
      }
      // The peer's P rows of tile j and their rescale factors.
      if (!wait_warp(BAR(B_PREM + pb), (j / kPBufs) & 1, ctl, true)) { ok = false; break; }
      const float f = *reinterpret_cast<const float*>(gbase + C::OFF_FACT + pb * 512 + row * 4);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(BAR(B_PREM + pb), kPRemoteBytes / 4);
      const bool last = cur.last();
      const int p = cur.p, whole = cur.whole, pslot = cur.pslot;
      cur.advance();
      if (__any_sync(0xffffffffu, f != 1.f)) {
        // Only after a segment's first tile: P.V of tile j - 1 must be done.
        if (!wait_warp(BAR(B_PVDONE + (j - 1) % kPBufs), ((j - 1) / kPBufs) & 1, ctl)) { ok = false; break; }
        tc_fence_after();
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t ta = tmem + lane_off + TM_O + 32 * cc;
          tmem_ld16x2_32<128>(ta, o);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
          tmem_st16x2_32<128>(ta, o);
        }
        tmem_wait_st();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_RESC + pb));
      if (stage_late && ahead.valid_tile()) {
        if (!stage(j + 1, ahead.vlo(), ahead.vhi())) { ok = false; break; }
        ahead.advance();
      }
      if (!last) continue;
      // Segment end: the peer's 1/l for these rows, then O of these rows out.
      const uint32_t lb = seg & 1;
      if (!wait_warp(BAR(B_LFULL + lb), (seg >> 1) & 1, ctl, true)) { ok = false; break; }
      const float inv_l = *reinterpret_cast<const float*>(gbase + C::OFF_LREC + lb * 512 + row * 4);
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(BAR(B_LFULL + lb), 16 * 4);
      if (!wait_warp(BAR(B_PVDONE + pb), (j / kPBufs) & 1, ctl)) { ok = false; break; }
      tc_fence_after();
      const size_t grow = (size_t)p * kRows + row;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld16x2_32<128>(tmem + lane_off + TM_O + 32 * cc, o);
        tmem_wait_ld();
        store_o_row(o, inv_l, whole, grow, row, pslot, (int)rank * 256 + hh * 128 + 32 * cc, o_lat, o_part);
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_OFREE));
      ++seg;
    }
  } else if (FP8 && warp >= 12) {
    // ------------------------------------------------------------ fp8 tile converter
    // Writes code * scale as bf16 into the tile's c_KV chunks (128-byte swizzle),
    // 16 codes (one token, 16 columns) per thread and step.
    const int ct = threadIdx.x - 384;
    SegIter it;
    it.init(plan, worker);
    int p, t_lo, t_hi, len, whole, slot, lo, tf;
    uint32_t e = 0, jt = 0;
    bool ok = true;
    auto slot_free = [&](uint32_t ee) -> bool {
      return ee < (uint32_t)S || wait_warp(BAR(B_KVEMPTY + ee % S), ((ee / S) - 1) & 1, ctl);
    };
    while (ok && it.next(p, t_lo, t_hi, len, whole, slot, lo, tf)) {
      for (int h = 0; h < 2; ++h, ++e) {  // Q entries: nothing to convert
        if (!slot_free(e)) { ok = false; break; }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_KVFULL + e % S));
      }
      for (int t = t_lo; ok && t < t_hi; ++t, ++e, ++jt) {
        const uint32_t sg = jt % kStages8;
        if (!slot_free(e) || !wait_warp(BAR(B_STFULL + sg), (jt / kStages8) & 1, ctl)) { ok = false; break; }
        const uint8_t* stg = gbase + C::OFF_STAGE + sg * kStBytes;
        uint8_t* dst_slot = gbase + C::OFF_SLOTS + (e % S) * kSlotBytes;
#pragma unroll 2
        for (int n = 0; n < 8; ++n) {
          const int k = ct + 128 * n, r = k >> 4, ch = k & 15;
          const uint4 v = *reinterpret_cast<const uint4*>(stg + r * 256 + ch * 16);
          const float sc = *reinterpret_cast<const float*>(stg + kStCodes + r * 4);
          const uint32_t cw[4] = {v.x, v.y, v.z, v.w};
          uint32_t o[8];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
              const __half2_raw hr =
                  __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(cw[i] >> (16 * hf)), __NV_E4M3);
              const float2 f2 = __half22float2(__half2(hr));
              const __nv_bfloat162 b2 = __floats2bfloat162_rn(f2.x * sc, f2.y * sc);
              o[2 * i + hf] = *reinterpret_cast<const uint32_t*>(&b2);
            }
          }
          uint8_t* dst = dst_slot + (ch >> 2) * kKvChunk;
          const int u0 = 2 * (ch & 3);
          *reinterpret_cast<uint4*>(dst + sw128_off(r, u0)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(dst + sw128_off(r, u0 + 1)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(BAR(B_STEMPTY + sg));
          mbar_arrive(BAR(B_KVFULL + e % S));
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (*abort_flag) {
    // After an abort, copies and MMAs this CTA issued may still be in flight:
    // they complete within microseconds, and the CTA waits a bounded 1 ms for
    // them before its tensor and shared memory are released.
    const uint64_t t0 = globaltimer();
    while (globaltimer() - t0 < 1000000ull) {
    }
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  cluster_arrive();
  cluster_wait();
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

// 2-D tensor map: rows of `inner` elements of `dtype`, `row_bytes` apart.
bool make_map(CUtensorMap* m, CUtensorMapDataType dtype, const void* ptr, uint64_t inner, uint64_t rows,
              uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 1-D fp32 tensor map of n elements, boxes of `box` elements.
bool make_map_1d_f32(CUtensorMap* m, const void* ptr, uint64_t n, uint32_t box) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[1] = {n};
  cuuint64_t strides[1] = {4};  // unused at rank 1, but the encoder rejects a null array
  cuuint32_t boxd[1] = {box};
  cuuint32_t estr[1] = {1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 1, const_cast<void*>(ptr), dims, strides, boxd, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool FP8>
cudaError_t set_smem_attr() {
  static std::once_flag once;
  static cudaError_t err = cudaSuccess;
  std::call_once(once, [] {
    err = cudaFuncSetAttribute(tc_decode_kernel<FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)tcd::Cfg<FP8>::kSmemBytes);
  });
  return err;
}

}  // namespace

bool tc_device_ok() {
  // Per-device answer, computed once; concurrent first calls compute the same value.
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    v = (major == 10 && minor == 3) ? 1 : 2;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v == 1;
}

int tc_decode_max_workers() {
  // Resident 2-CTA clusters of the decode kernel per device, computed once.
  static std::atomic<int> cached[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  int v = cached[dev].load(std::memory_order_relaxed);
  if (v == 0) {
    int clusters = 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2 * 256, 1, 1);
    cfg.blockDim = dim3(tcd::Cfg<false>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = tcd::Cfg<false>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (set_smem_attr<false>() != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&clusters, tc_decode_kernel<false>, &cfg) != cudaSuccess || clusters < 1) {
      cudaGetLastError();
      clusters = sm_count() / 2;
    }
    v = clusters;
    cached[dev].store(v, std::memory_order_relaxed);
  }
  return v;
}

bool tc_decode_supported(const mla_dims_t& d) {
  return d.n_h == 128 && d.d_c == 512 && d.d_rope == 64 && d.act_dtype == MLA_BF16 &&
         (d.cache_dtype == MLA_BF16 || d.cache_dtype == MLA_FP8_E4M3) && tc_device_ok();
}

cudaError_t launch_tc_decode(const mla_dims_t& d, const mla_cache_t& c, int B, int q_per_seq,
                             const __nv_bfloat16* q_abs, const int32_t* bt, int max_pages,
                             const int32_t* plan, int workers, float* o_part, float* lse_part,
                             __nv_bfloat16* o_lat, float* lse, int32_t* status, cudaStream_t st) {
  using namespace tcd;
  const bool fp8 = d.cache_dtype == MLA_FP8_E4M3;
  const uint64_t rows = (uint64_t)B * q_per_seq * kRows;
  const uint64_t slots = (uint64_t)c.num_pages * d.page_size;
  if (slots == 0 || slots > 0x7FFFFFF0ull || rows > 0x7FFFFFF0ull) return cudaErrorInvalidValue;
  const uint32_t box_rows = d.page_size < kTile ? (uint32_t)d.page_size : (uint32_t)kTile;
  CUtensorMap mq64, mq32, mkv, mkr, msc;
  const uint64_t qrow = 576 * 2;
  if (!make_map(&mq64, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_abs, 576, rows, qrow, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mq32, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, q_abs, 576, rows, qrow, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  if (!fp8) {
    if (!make_map(&mkv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.ckv, 576, slots, qrow, 64, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_128B) ||
        !make_map(&mkr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.ckv, 576, slots, qrow, 32, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_64B))
      return cudaErrorInvalidValue;
    msc = mkr;  // unused
  } else {
    if ((reinterpret_cast<uintptr_t>(c.scale) & 15) != 0) return cudaErrorInvalidValue;
    if (!make_map(&mkv, CU_TENSOR_MAP_DATA_TYPE_UINT8, c.ckv, 512, slots, 512, 256, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_NONE) ||
        !make_map(&mkr, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, c.kr, 64, slots, 128, 32, box_rows,
                  CU_TENSOR_MAP_SWIZZLE_64B) ||
        !make_map_1d_f32(&msc, c.scale, slots, box_rows))
      return cudaErrorInvalidValue;
  }
  cudaError_t err = fp8 ? set_smem_attr<true>() : set_smem_attr<false>();
  if (err != cudaSuccess) return err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * workers, 1, 1);
  cfg.blockDim = dim3(fp8 ? Cfg<true>::kThreads : Cfg<false>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = fp8 ? Cfg<true>::kSmemBytes : Cfg<false>::kSmemBytes;
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
  const float scale_log2 = d.softmax_scale * 1.4426950408889634f;
  auto kern = fp8 ? tc_decode_kernel<true> : tc_decode_kernel<false>;
  return cudaLaunchKernelEx(&cfg, kern, mq64, mq32, mkv, mkr, msc, plan, bt, max_pages, d.page_size, (int)box_rows,
                            (int64_t)c.num_pages, (int)slots, q_per_seq, scale_log2, o_part, lse_part, o_lat, lse,
                            status);
}

}  // namespace mla
