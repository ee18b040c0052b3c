// Tensor-core MLA decode attention for B300 (sm_103a): tcgen05 MMAs with TMEM
// operands and accumulators, TMA-staged cache tiles, and a 2-CTA cluster per
// worker.
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
//     [32r, 32r+32). Every 64-token cache tile is TMA-loaded once: each CTA
//     fetches only its 288 columns, so HBM bytes are read exactly once.
//   * S_r = Q[:, cols_r] . K[:, cols_r]^T (M=128, N=64, K=288) lands in TMEM.
//     The two partial scores are summed through distributed shared memory
//     (16-bit fixed point per half row, part bulk copy, part st.async), so both
//     CTAs hold the identical S without doing the QK^T work twice.
//   * Both CTAs run the same online softmax (running max with lazy rescale,
//     exp2, bf16 P) and each accumulates its half of O = P . V (M=128, N=256)
//     in TMEM. O for 128 heads x 512 latent columns in fp32 would fill one SM's
//     TMEM; split across the pair it leaves room for S, P and Q.
//   * Tensor memory holds O (256 columns), S (64), P (32, the A operand of P.V)
//     and the c_KV part of the Q slice (128, the A operand of Q.K^T), so shared
//     memory holds a 4-slot ring of cache tiles. The Q slice reaches TMEM
//     through two ring slots and tcgen05.cp at every problem change.
// Roles per CTA (384 threads): warp 0 lane 0 issues TMA into the ring; warp 1
// lane 0 the Q copies and Q.K^T MMAs; warp 3 lane 0 the P.V MMAs; warp 2 lane 0
// the bulk copies of staged partial scores to the peer; warps 4-11 (two per
// TMEM lane quadrant, one head row per thread, 32 score columns per warp) run
// the softmax. They stage tile j+1's partial scores for the exchange before
// working on tile j when those are ready, so the exchange overlaps the softmax.
// Every wait is bounded: after 2 s the kernel records MLA_ERR_DEVICE_TIMEOUT in
// *status and unwinds.
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
constexpr int kTile = kTcTileN;  // 64 tokens
constexpr int kSlots = 4;
constexpr int kPrefetch = 0;                        // tiles ahead warmed in L2
constexpr uint32_t kKvChunk = 64 * 128;             // [64 tokens x 64 bf16], 128B swizzle
constexpr uint32_t kKvKrOff = 4 * kKvChunk;
constexpr uint32_t kSlotBytes = 4 * kKvChunk + 64 * 64;  // + [64 x 32] k_R part, 64B swizzle
constexpr uint32_t kQChunk = 128 * 128;             // [128 rows x 64 bf16]; two per ring slot
constexpr uint32_t kQkrBytes = 128 * 64;            // [128 rows x 32 bf16], 64B swizzle
// Partial scores travel as 16-bit fixed point: each half row (32 scores, one
// softmax thread) is sent as its maximum mx, a power-of-two step q chosen from
// the half row's range (mx - min < 2^15 q), and 32 unsigned offsets
// e = round((mx - s) / q), decoded as mx - e q. The error is at most q / 2, under
// range * 2^-15 for every score, and both CTAs decode the same numbers. A row is
// 16 bytes of references (mx and q of both halves) plus 8 chunks of 16 bytes.
// Exchange buffers are chunk-major ([chunk][row]), the references in chunk 0.
// The first kBulkChunks chunks of every row go in one bulk copy, the rest as
// st.async stores from the softmax threads, so the exchange uses both the copy
// engine and the SM's own path to the peer.
constexpr int kXchgChunks = 9;
constexpr uint32_t kXchgBytes = kXchgChunks * 128 * 16;  // one tile of partial scores
constexpr int kBulkChunks = 7;
constexpr uint32_t kBulkBytes = kBulkChunks * 128 * 16;
// Data chunk k (0..3) of half h goes to position xchg_pos(h, k): each half sends
// the same number of chunks with st.async.
constexpr int kRemoteHalf = (kXchgChunks - kBulkChunks) / 2;
constexpr int kLocalHalf = 4 - kRemoteHalf;
static_assert(kXchgChunks == 9 && 2 * kRemoteHalf == kXchgChunks - kBulkChunks, "chunk split");
__device__ __forceinline__ int xchg_pos(int h, int k) {
  return k < kLocalHalf ? 1 + h * kLocalHalf + k : kBulkChunks + h * kRemoteHalf + (k - kLocalHalf);
}
constexpr uint32_t OFF_SLOTS = 0;
constexpr uint32_t OFF_SEND = OFF_SLOTS + kSlots * kSlotBytes;
// Tile j of the peer's partial scores lands in receive buffer j % kRecvBufs.
constexpr int kRecvBufs = 3;
constexpr uint32_t OFF_RECV = OFF_SEND + kBulkBytes;
constexpr uint32_t OFF_QKR = OFF_RECV + kRecvBufs * kXchgBytes;
constexpr uint32_t OFF_RED = OFF_QKR + kQkrBytes;  // row maxima [2][2][128] and sums [2][128]
constexpr uint32_t OFF_BAR = OFF_RED + 3 * 2 * 128 * 4;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
constexpr int kSoftWarps = 8;  // two per TMEM lane quadrant, 32 score columns each
constexpr int kThreads = 128 + 32 * kSoftWarps;
enum Bar {
  B_KVFULL = 0,            // + slot
  B_KVEMPTY = kSlots,      // + slot
  B_QKRFULL = 2 * kSlots, B_QKREMPTY, B_SFULL, B_SFREE, B_PFULL, B_PVDONE, B_OFREE,
  B_RECV,                  // + buffer: the peer's partial scores for a tile have landed
  B_STAGED = B_RECV + kRecvBufs,  // softmax warps staged a tile's partial scores
  B_SENDFREE,              // the bulk copy has read the staging buffer
  B_PAIR,                  // + quadrant: the quadrant's two softmax warps have posted a row value
  NBAR = B_PAIR + 4
};
// TMEM columns: O, S, P, the Q slice's c_KV part, and the offsets of the last
// staged tile's partial scores (16 per half row), kept until that tile's combine.
constexpr uint32_t TM_O = 0, TM_S = 256, TM_P = 320, TM_Q = 352, TM_X = 480, kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by 2^8
static_assert(kSlotBytes % 1024 == 0 && OFF_SEND % 1024 == 0 && OFF_RECV % 1024 == 0 && OFF_QKR % 512 == 0,
              "swizzle atoms");
static_assert(2 * kQChunk <= kSlotBytes, "a ring slot holds two Q chunks");
static_assert(kSlots >= 3, "the Q slice takes two ring slots");
static_assert(kSmemBytes <= 232448, "shared memory");
static_assert(8 * NBAR + 16 <= 256, "barrier area");
static_assert(TM_Q + 128 <= kTmemCols, "tensor memory");
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

// Walks one worker's share of the tile sequence as segments (problem, tile range).
struct SegIter {
  const int32_t* cum;
  const int32_t* pbase;
  const int32_t* lens;
  const int32_t* pw0;
  const int32_t* pcnt;
  int w, g0, g1, p;
  __device__ void init(const int32_t* plan, int worker) {
    PlanView pv = plan_view(plan);
    cum = pv.cum;
    pbase = pv.pbase;
    lens = pv.len;
    pw0 = pv.pw0;
    pcnt = pv.pcnt;
    w = worker;
    g0 = pv.wstart[worker];
    g1 = pv.wstart[worker + 1];
    p = pv.first[worker];  // the problem holding the first tile (one load, no search)
  }
  __device__ bool next(int& prob, int& t_lo, int& t_hi, int& len, int& whole, int& slot) {
    if (g0 >= g1) return false;
    while (cum[p + 1] <= g0) ++p;
    t_lo = g0 - cum[p];
    t_hi = min(g1, cum[p + 1]) - cum[p];
    len = lens[p];
    whole = (pcnt[p] == 1);
    slot = pbase[p] + (w - pw0[p]);
    prob = p;
    g0 = cum[p] + t_hi;
    ++p;
    return true;
  }
};

// Number of tiles in a worker's share of the tile sequence.
__device__ __forceinline__ int worker_tiles(const int32_t* plan, int worker) {
  const PlanView pv = plan_view(plan);
  return pv.wstart[worker + 1] - pv.wstart[worker];
}

// A tile of the worker's sequence with everything the softmax needs about it.
struct TileCursor {
  SegIter it;
  bool valid_tile;
  int p, t_lo, t_hi, len, whole, pslot;  // segment
  int k;                                 // position in the segment
  uint32_t entry;                        // ring entry that holds the tile
  uint32_t seg;                          // segment index
  __device__ void start(const int32_t* plan, int worker) {
    it.init(plan, worker);
    entry = 0;
    seg = 0;
    valid_tile = it.next(p, t_lo, t_hi, len, whole, pslot);
    k = 0;
    entry = 2;  // the segment's two Q entries come first
  }
  __device__ void advance() {
    ++k;
    ++entry;
    if (t_lo + k >= t_hi) {
      valid_tile = it.next(p, t_lo, t_hi, len, whole, pslot);
      k = 0;
      ++seg;
      entry += 2;
    }
  }
  __device__ bool first() const { return k == 0; }
  __device__ bool last() const { return t_lo + k == t_hi - 1; }
  __device__ int tile() const { return t_lo + k; }
};

// The next tile to stage in a worker's share: only whether it exists and how
// many of its tokens are inside its sequence (a light cursor, few registers).
struct TileAhead {
  const int32_t* cum;
  const int32_t* lens;
  int g, g1, p, c0, c1, len;  // tile index; problem p holds tiles [c0, c1)
  __device__ void start(const int32_t* plan, int worker) {
    const PlanView pv = plan_view(plan);
    cum = pv.cum;
    lens = pv.len;
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
  }
  __device__ bool valid_tile() const { return g < g1; }
  __device__ int valid() const { return min(tcd::kTile, len - (g - c0) * tcd::kTile); }
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
}  // namespace

__global__ void __launch_bounds__(tcd::kThreads, 1)
tc_decode_kernel(const __grid_constant__ CUtensorMap tm_q64, const __grid_constant__ CUtensorMap tm_q32,
                 const __grid_constant__ CUtensorMap tm_kv64, const __grid_constant__ CUtensorMap tm_kv32,
                 const int32_t* __restrict__ plan, const int32_t* __restrict__ bt, int max_pages,
                 int page_size, int box_rows, int64_t num_pages, int oob_row, int q_per_seq,
                 float scale_log2, float* __restrict__ o_part, float* __restrict__ lse_part,
                 __nv_bfloat16* __restrict__ o_lat, float* __restrict__ lse_out, int32_t* status) {
  using namespace tcd;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* gbase = smem_raw + (base - raw);
  const uint32_t rank = cluster_ctarank(), peer = rank ^ 1u;
  const int worker = (int)cluster_id_x();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  auto BAR = [&](int i) { return base + OFF_BAR + 8u * (uint32_t)i; };
  auto SLOT = [&](uint32_t e) { return base + OFF_SLOTS + (e % kSlots) * kSlotBytes; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_BAR + 8 * NBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 8 * NBAR + 8);

  pdl_trigger();
  if (threadIdx.x == 0) {
    for (int i = 0; i < NBAR; ++i) {
      const bool per_warp = (i == B_SFREE || i == B_PFULL || i == B_OFREE || i == B_STAGED ||
                             (i >= B_RECV && i < B_RECV + kRecvBufs));
      mbar_init(BAR(i), per_warp ? kSoftWarps : (i >= B_PAIR ? 2 : 1));
    }
    // The receive buffers start armed for the peer's first tiles; each softmax
    // warp re-arms its share of a buffer once it has read it.
    for (int b = 0; b < kRecvBufs; ++b)
      for (int w = 0; w < kSoftWarps; ++w) mbar_arrive_expect_tx(BAR(B_RECV + b), kXchgBytes / kSoftWarps);
    *abort_flag = 0;
    fence_mbar_init_cluster();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tm_q64);
    prefetch_tmap(&tm_q32);
    prefetch_tmap(&tm_kv64);
    prefetch_tmap(&tm_kv32);
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
      int p, t_lo, t_hi, len, whole, slot;
      uint32_t seg = 0, e = 0;
      bool ok = true;
      auto acquire = [&](uint32_t ee) -> bool {
        return ee < (uint32_t)kSlots || wait_bar(BAR(B_KVEMPTY + ee % kSlots), ((ee / kSlots) - 1) & 1, ctl);
      };
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
        const int row0 = p * kRows;
        // The c_KV part of the Q slice, staged in two ring slots on its way to TMEM.
        for (int h = 0; h < 2 && ok; ++h, ++e) {
          if (!acquire(e)) { ok = false; break; }
          const uint32_t full = BAR(B_KVFULL + e % kSlots);
          mbar_arrive_expect_tx(full, 2 * kQChunk);
          for (int c = 0; c < 2; ++c)
            tma_load_2d(SLOT(e) + c * kQChunk, &tm_q64, (int)rank * 256 + (2 * h + c) * 64, row0, full);
        }
        if (!ok) break;
        // The k_R part of the Q slice stays in shared memory.
        if (seg > 0 && !wait_bar(BAR(B_QKREMPTY), (seg - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(BAR(B_QKRFULL), kQkrBytes);
        tma_load_2d(base + OFF_QKR, &tm_q32, 512 + (int)rank * 32, row0, BAR(B_QKRFULL));
        const int b = p / q_per_seq;
        // Page-box row of token `tok` of this problem, or -1 past its end / -2 on a bad page.
        auto box_row = [&](int tok) -> int {
          if (tok >= len) return -1;
          const int pg = tok / page_size;
          const int page = pg < max_pages ? bt[(size_t)b * max_pages + pg] : -1;
          if (page < 0 || page >= num_pages) return -2;
          return page * page_size + tok % page_size;
        };
        auto prefetch_tile = [&](int t) {
          for (int r0 = 0; r0 < kTile; r0 += box_rows) {
            const int y = box_row(t * kTile + r0);
            if (y < 0) continue;
            for (int c = 0; c < 4; ++c) tma_prefetch_2d(&tm_kv64, (int)rank * 256 + c * 64, y);
            tma_prefetch_2d(&tm_kv32, 512 + (int)rank * 32, y);
          }
        };
        for (int t = t_lo; t < min(t_hi, t_lo + kPrefetch); ++t) prefetch_tile(t);
        for (int t = t_lo; t < t_hi; ++t, ++e) {
          if (t + kPrefetch < t_hi) prefetch_tile(t + kPrefetch);
          if (!acquire(e)) { ok = false; break; }
          const uint32_t full = BAR(B_KVFULL + e % kSlots);
          mbar_arrive_expect_tx(full, kSlotBytes);
          const uint32_t st = SLOT(e);
          for (int r0 = 0; r0 < kTile; r0 += box_rows) {
            int y = box_row(t * kTile + r0);
            if (y == -2) set_status(status, MLA_ERR_BAD_PAGE);
            if (y < 0) y = oob_row;  // fully out of range: the copy fills zeros
            for (int c = 0; c < 4; ++c)
              tma_load_2d(st + c * kKvChunk + r0 * 128, &tm_kv64, (int)rank * 256 + c * 64, y, full);
            tma_load_2d(st + kKvKrOff + r0 * 64, &tm_kv32, 512 + (int)rank * 32, y, full);
          }
        }
        ++seg;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ Q.K^T issuer
    // Copies a segment's Q slice into TMEM, then issues Q.K^T for each tile once
    // its tile, the S buffer and the Q slice are ready. P.V has its own issuer
    // (warp 3): an issuing thread blocks while the tensor pipe's short queue is
    // full, and P.V, which releases a ring slot, must not wait behind a whole
    // Q.K^T issued just before its P became ready.
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false, false);
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot;
      uint32_t e = 0, j = 0, sidx = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
        if (!wait_bar(BAR(B_KVFULL + e % kSlots), (e / kSlots) & 1, ctl) ||
            !wait_bar(BAR(B_KVFULL + (e + 1) % kSlots), ((e + 1) / kSlots) & 1, ctl))
          break;
        tc_fence_after();
        for (int h = 0; h < 2; ++h) {
          const uint32_t st = SLOT(e + h);
          for (int c = 0; c < 2; ++c)
            for (int kk = 0; kk < 4; ++kk)
              tmem_cp_128x256b(tmem + TM_Q + (2 * h + c) * 32 + kk * 8,
                               smem_desc(st + c * kQChunk + kk * 32, 16, 1024, kSwizzle128B));
          mma_commit(BAR(B_KVEMPTY + (e + h) % kSlots));
        }
        e += 2;
        if (!wait_bar(BAR(B_QKRFULL), sidx & 1, ctl)) break;
        for (int t = t_lo; t < t_hi; ++t, ++e, ++j) {
          if (!wait_bar(BAR(B_KVFULL + e % kSlots), (e / kSlots) & 1, ctl) ||
              (j >= 1 && !wait_bar(BAR(B_SFREE), (j - 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = SLOT(e);
          for (int c = 0; c < 4; ++c)
            for (int kk = 0; kk < 4; ++kk)
              mma_f16_ts(tmem + TM_S, tmem + TM_Q + c * 32 + kk * 8,
                         smem_desc(st + c * kKvChunk + kk * 32, 16, 1024, kSwizzle128B), idesc_s,
                         (c | kk) ? 1u : 0u);
          for (int kk = 0; kk < 2; ++kk)
            mma_f16(tmem + TM_S, smem_desc(base + OFF_QKR + kk * 32, 16, 512, kSwizzle64B),
                    smem_desc(st + kKvKrOff + kk * 32, 16, 512, kSwizzle64B), idesc_s, 1u);
          mma_commit(BAR(B_SFULL));
          if (t == t_hi - 1) mma_commit(BAR(B_QKREMPTY));
        }
        ++sidx;
      }
    }
  } else if (warp == 3) {
    // ------------------------------------------------------------ P.V issuer
    // O += P . V for each tile as soon as its P is in TMEM; the first tile of a
    // segment also waits until the previous segment's O has been read out.
    if (lane == 0) {
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot;
      uint32_t e = 0, j = 0, sidx = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
        e += 2;  // the segment's Q entries
        for (int t = t_lo; t < t_hi; ++t, ++e, ++j) {
          const bool first = (t == t_lo);
          if (!wait_bar(BAR(B_PFULL), j & 1, ctl) ||
              (first && sidx > 0 && !wait_bar(BAR(B_OFREE), (sidx - 1) & 1, ctl))) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t st = SLOT(e);
          for (int kk = 0; kk < kTile / 16; ++kk)
            mma_f16_ts(tmem + TM_O, tmem + TM_P + kk * 8,
                       smem_desc(st + kk * 2048, kKvChunk, 1024, kSwizzle128B), idesc_pv,
                       (first && kk == 0) ? 0u : 1u);
          mma_commit(BAR(B_KVEMPTY + e % kSlots));
          mma_commit(BAR(B_PVDONE));
        }
        ++sidx;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ score exchange
    // Moves the bulk part of each staged tile of partial scores into the peer's
    // receive buffer j % kRecvBufs. The softmax warps stage a tile only once the
    // peer has freed that buffer (see the softmax loop), so no handshake is
    // needed here.
    if (lane == 0) {
      const uint32_t recv_peer = mapa(base + OFF_RECV, peer);
      const uint32_t bar_recv_peer = mapa(BAR(B_RECV), peer);
      const int n = worker_tiles(plan, worker);
      for (int j = 0; j < n; ++j) {
        if (!wait_bar(BAR(B_STAGED), j & 1, ctl)) break;
        const uint32_t b = (uint32_t)j % kRecvBufs;
        bulk_copy_to_peer(recv_peer + b * kXchgBytes, base + OFF_SEND, kBulkBytes, bar_recv_peer + 8u * b);
        bulk_commit();
        bulk_wait_read_all();
        mbar_arrive(BAR(B_SENDFREE));
      }
      bulk_wait_read_all();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    // Warp pair (qd, h): TMEM lane quadrant qd (head rows 32qd..32qd+31, one per
    // thread) and score columns 32h..32h+31 of each tile. The two warps of a
    // quadrant agree on each row's maximum through shared memory; each keeps a
    // partial row sum and owns half of the O columns for rescaling and output.
    const int qd = warp & 3, h = (warp - 4) >> 2;
    const int r = qd * 32 + lane;  // head row == TMEM lane
    const int t256 = threadIdx.x - 128;
    const uint32_t lane_base = (uint32_t)(qd * 32) << 16;
    // The quadrant's two warps meet on an mbarrier (bounded waits, unlike bar.sync).
    const uint32_t pair_bar = BAR(B_PAIR + qd);
    uint32_t pair_uses = 0;
    auto pair_sync = [&]() -> bool {
      __syncwarp();
      if (lane == 0) mbar_arrive(pair_bar);
      const bool done = __all_sync(0xffffffffu, wait_bar(pair_bar, pair_uses & 1, ctl));
      ++pair_uses;
      return done;
    };
    float* red = reinterpret_cast<float*>(gbase + OFF_RED);
    // Byte offset in an exchange buffer of 16-byte chunk c of row r (chunk-major).
    auto xchg_off = [&](int c) { return (uint32_t)(c * 128 + r) * 16u; };
    const uint32_t recv_peer = mapa(base + OFF_RECV, peer);
    const uint32_t bar_recv_peer = mapa(BAR(B_RECV), peer);
    // This thread's half row as sent, for the tile to combine next (own_*) and
    // the last one staged (nxt_*, its offsets parked in TMEM): offsets (two per
    // word), maximum and step.
    uint32_t own_w[16];
    float own_mx = 0.f, own_q = 0.f, nxt_mx = 0.f, nxt_q = 0.f;
    const uint32_t tm_x = tmem + lane_base + TM_X + 16 * h;
    auto rotate = [&]() {
      tmem_wait_st();
      tmem_ld16(tm_x, own_w);
      tmem_wait_ld();
      own_mx = nxt_mx;
      own_q = nxt_q;
    };
    // Load this warp's 32 columns of S(j) from TMEM, free the buffer, encode them
    // (columns at or past `valid` are left out of the range) and send them: the
    // references and most chunks through the staging buffer and the bulk copy,
    // the rest stored straight into the peer's receive buffer.
    auto take_and_stage = [&](uint32_t j, int valid) -> bool {
      if (!__all_sync(0xffffffffu, wait_bar(BAR(B_SFULL), j & 1, ctl))) return false;
      tc_fence_after();
      uint32_t sv[32];
      tmem_ld32(tmem + lane_base + TM_S + 32 * h, sv);
      tmem_wait_ld();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_SFREE));
      const uint32_t dst = recv_peer + (j % kRecvBufs) * kXchgBytes, dbar = bar_recv_peer + 8u * (j % kRecvBufs);
      if (j >= 1 && !__all_sync(0xffffffffu, wait_bar(BAR(B_SENDFREE), (j - 1) & 1, ctl))) return false;
      float mx, mn;
      if (32 * h + 32 <= valid) {
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
          if (32 * h + x < valid) {
            mx = fmaxf(mx, __uint_as_float(sv[x]));
            mn = fminf(mn, __uint_as_float(sv[x]));
          }
        }
      }
      // Step q = 2^-k with range < 2^(E+1) <= 2^15 q, E the range's exponent;
      // k is capped at 60 for (near) constant half rows.
      const int eb = max((int)((__float_as_uint(mx - mn) >> 23) & 0xFFu), 81);
      const float enc = __uint_as_float((uint32_t)(268 - eb) << 23);  // 2^k
      const float q = __uint_as_float((uint32_t)(eb - 14) << 23);    // 2^-k
      // y = 2^23 + round((mx - s) 2^k): its low 16 bits are the offset.
      uint32_t nxt_w[16];
#pragma unroll
      for (int x = 0; x < 16; ++x) {
        float d0, d1, y0, y1;
        ffma2(d0, d1, __uint_as_float(sv[2 * x]), __uint_as_float(sv[2 * x + 1]), -1.f, mx);
        ffma2(y0, y1, d0, d1, enc, 8388608.f);
        nxt_w[x] = __byte_perm(__float_as_uint(y0), __float_as_uint(y1), 0x5410);
      }
      nxt_mx = mx;
      nxt_q = q;
      tmem_st16(tm_x, nxt_w);
      *reinterpret_cast<uint2*>(gbase + OFF_SEND + xchg_off(0) + 8 * h) =
          make_uint2(__float_as_uint(mx), __float_as_uint(q));
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = xchg_pos(h, k);
        if (c < kBulkChunks)
          *reinterpret_cast<uint4*>(gbase + OFF_SEND + xchg_off(c)) =
              make_uint4(nxt_w[4 * k], nxt_w[4 * k + 1], nxt_w[4 * k + 2], nxt_w[4 * k + 3]);
        else
          st_async_v4(dst + xchg_off(c), nxt_w[4 * k], nxt_w[4 * k + 1], nxt_w[4 * k + 2], nxt_w[4 * k + 3], dbar);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_STAGED));
      return true;
    };
    // Each iteration j first waits for the peer's tile j, then stages tile j + 1
    // (so that its exchange overlaps this tile's combine, softmax and P), then
    // combines tile j. Tile j + 1 goes into the peer's buffer that held its tile
    // j - 2: the peer staged the tile j that has just arrived after it had
    // combined its tile j - 2, so the buffer is free without a handshake.
    TileCursor cur;
    TileAhead ahead;  // the next tile to stage
    cur.start(plan, worker);
    ahead.start(plan, worker);
    bool ok = true;
    if (ahead.valid_tile()) {
      ok = take_and_stage(0, ahead.valid());
      ahead.advance();
    }
    float m_ref = -INFINITY, l = 0.f;
    for (uint32_t j = 0; ok && cur.valid_tile; ++j) {
      // a. This thread's half of tile j as sent, then the peer's half (buffer
      //    j % kRecvBufs); then stage tile j + 1.
      rotate();
      const uint32_t rb = j % kRecvBufs;
      if (!__all_sync(0xffffffffu, wait_bar(BAR(B_RECV + rb), (j / kRecvBufs) & 1, ctl, true))) { ok = false; break; }
      if (ahead.valid_tile()) {
        if (!take_and_stage(j + 1, ahead.valid())) { ok = false; break; }
        ahead.advance();
      }
      float s[32];
      {
        // Each half row decodes as mx - e q = (2^23 + e) (-q) + (mx + 2^23 q):
        // the offset becomes a float by putting 0x4B00 above its 16 bits.
        const uint8_t* recv = gbase + OFF_RECV + rb * kXchgBytes;
        const uint2 ref = *reinterpret_cast<const uint2*>(recv + xchg_off(0) + 8 * h);
        const float peer_mx = __uint_as_float(ref.x), peer_q = __uint_as_float(ref.y);
        const float k_own = fmaf(8388608.f, own_q, own_mx), k_peer = fmaf(8388608.f, peer_q, peer_mx);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint4 v = *reinterpret_cast<const uint4*>(recv + xchg_off(xchg_pos(h, k)));
          const uint32_t pw[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const int x = 8 * k + 2 * i;
            const uint32_t ow = own_w[4 * k + i];
            float a0, a1, b0, b1;
            ffma2(a0, a1, __uint_as_float(__byte_perm(ow, 0x4B000000u, 0x7610)),
                  __uint_as_float(__byte_perm(ow, 0x4B000000u, 0x7632)), -own_q, k_own);
            ffma2(b0, b1, __uint_as_float(__byte_perm(pw[i], 0x4B000000u, 0x7610)),
                  __uint_as_float(__byte_perm(pw[i], 0x4B000000u, 0x7632)), -peer_q, k_peer);
            fadd2(a0, a1, b0, b1);
            s[x] = a0;
            s[x + 1] = a1;
          }
        }
      }
      // b. Re-arm this warp's share of the buffer for tile j + kRecvBufs.
      __syncwarp();
      if (lane == 0) mbar_arrive_expect_tx(BAR(B_RECV + rb), kXchgBytes / kSoftWarps);
      const bool first = cur.first(), last = cur.last();
      // Scores at or past column `valid` are past the sequence end.
      const int valid = min(kTile, cur.len - cur.tile() * kTile);
      const uint32_t tile_entry = cur.entry;
      const int p = cur.p, whole = cur.whole, pslot = cur.pslot;
      cur.advance();
      // c. Online softmax in log2 units. Tokens past the end (only in a sequence's
      //    last tile) are masked; the maximum is taken on the raw scores and the
      //    scale is folded into the exponent's multiply-add.
      if (valid < kTile) {
#pragma unroll
        for (int x = 0; x < 32; ++x)
          if (32 * h + x >= valid) s[x] = -INFINITY;
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
      // The row's maximum over both column halves, through shared memory.
      red[((j & 1) * 2 + h) * 128 + r] = fmax3(mx[0], mx[1], fmaxf(mx[2], mx[3]));
      if (!pair_sync()) { ok = false; break; }
      const float mt = fmaxf(red[((j & 1) * 2) * 128 + r], red[((j & 1) * 2 + 1) * 128 + r]) * scale_log2;
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
      // P (TMEM) and O are free once the previous P . V has completed.
      if (j >= 1 && !__all_sync(0xffffffffu, wait_bar(BAR(B_PVDONE), (j - 1) & 1, ctl))) { ok = false; break; }
      tc_fence_after();
      // Rows decide independently whether their running max moved; the TMEM
      // accesses are warp-collective, so the whole warp rescales its half of O
      // when any row needs it (rows that do not use a factor of 1).
      const bool rescale = need && !first;
      if (__any_sync(0xffffffffu, rescale)) {
        const float f = rescale ? factor : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < 4; ++cc) {
          uint32_t o[32];
          const uint32_t ta = tmem + lane_base + TM_O + (4 * h + cc) * 32;
          tmem_ld32(ta, o);
          tmem_wait_ld();
#pragma unroll
          for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
          tmem_st32(ta, o);
        }
      }
      tmem_st16(tmem + lane_base + TM_P + 16 * h, pk);  // 32 tokens of bf16 P in 16 columns
      tmem_wait_st();
      if (valid < kTile) {
        // Rows past the sequence end may hold anything (NaN): zero them so that
        // P = 0 times V cannot poison O.
        uint8_t* st = gbase + OFF_SLOTS + (tile_entry % kSlots) * kSlotBytes;
        const int words = (kTile - valid) * 36;
        for (int i = t256; i < words; i += 32 * kSoftWarps) {
          const int row = valid + i / 36, wd = i % 36;
          uint8_t* dst = wd < 32 ? st + (wd >> 3) * kKvChunk + row * 128 + (wd & 7) * 16
                                 : st + kKvKrOff + row * 64 + (wd - 32) * 16;
          *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
        }
        fence_proxy_async_smem();
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_PFULL));
      if (!last) continue;
      // d. Segment epilogue: O / l to o_lat (whole problem) or to a partial slot;
      //    this warp writes O columns 128h..128h+127 of its rows.
      red[(4 + h) * 128 + r] = l;
      if (!pair_sync()) { ok = false; break; }
      const float l_row = red[4 * 128 + r] + red[5 * 128 + r];
      if (!__all_sync(0xffffffffu, wait_bar(BAR(B_PVDONE), j & 1, ctl))) { ok = false; break; }
      tc_fence_after();
      const float inv_l = 1.f / l_row;
      const size_t row = (size_t)p * kRows + r;
#pragma unroll 1
      for (int cc = 0; cc < 4; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + TM_O + (4 * h + cc) * 32, o);
        tmem_wait_ld();
        const int col = (int)rank * 256 + (4 * h + cc) * 32;
        if (whole) {
          uint4* dst = reinterpret_cast<uint4*>(o_lat + row * 512 + col);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w4[4];
#pragma unroll
            for (int e2 = 0; e2 < 4; ++e2) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[q4 * 8 + 2 * e2]) * inv_l,
                                                              __uint_as_float(o[q4 * 8 + 2 * e2 + 1]) * inv_l);
              w4[e2] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        } else {
          // Partials go out piece-major ([slot][32-column chunk][4-column piece]
          // [row][4]): each warp store covers 512 contiguous bytes.
          float4* dst = reinterpret_cast<float4*>(o_part + ((size_t)pslot * 16 + col / 32) * 8 * kRows * 4) + r;
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4 * kRows] = make_float4(__uint_as_float(o[4 * q4]) * inv_l, __uint_as_float(o[4 * q4 + 1]) * inv_l,
                                  __uint_as_float(o[4 * q4 + 2]) * inv_l, __uint_as_float(o[4 * q4 + 3]) * inv_l);
        }
      }
      if (rank == 0 && h == 0) {
        const float lse = (m_ref + log2f(l_row)) * 0.69314718055994531f;
        if (whole) lse_out[row] = lse;
        else lse_part[(size_t)pslot * kRows + r] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_OFREE));
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
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

// 2-D bf16 tensor map: rows of `inner` elements, `row_bytes` apart.
bool make_map(CUtensorMap* m, const void* ptr, uint64_t inner, uint64_t rows, uint64_t row_bytes,
              uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t dims[2] = {inner, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {box_inner, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(ptr), dims, strides, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
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
    cfg.blockDim = dim3(tcd::kThreads, 1, 1);
    cfg.dynamicSmemBytes = tcd::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaFuncSetAttribute(tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)tcd::kSmemBytes) != cudaSuccess ||
        cudaOccupancyMaxActiveClusters(&clusters, tc_decode_kernel, &cfg) != cudaSuccess ||
        clusters < 1) {
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
         d.cache_dtype == MLA_BF16 && tc_device_ok();
}

cudaError_t launch_tc_decode(const mla_dims_t& d, const mla_cache_t& c, int B, int q_per_seq,
                             const __nv_bfloat16* q_abs, const int32_t* bt, int max_pages,
                             const int32_t* plan, int workers, float* o_part, float* lse_part,
                             __nv_bfloat16* o_lat, float* lse, int32_t* status, cudaStream_t st) {
  using namespace tcd;
  const uint64_t rows = (uint64_t)B * q_per_seq * kRows;
  const uint64_t slots = (uint64_t)c.num_pages * d.page_size;
  if (slots == 0 || slots > 0x7FFFFFF0ull || rows > 0x7FFFFFF0ull) return cudaErrorInvalidValue;
  const uint32_t box_rows = d.page_size < kTile ? (uint32_t)d.page_size : (uint32_t)kTile;
  CUtensorMap mq64, mq32, mkv64, mkv32;
  const uint64_t row_bytes = 576 * 2;
  if (!make_map(&mq64, q_abs, 576, rows, row_bytes, 64, 128, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mq32, q_abs, 576, rows, row_bytes, 32, 128, CU_TENSOR_MAP_SWIZZLE_64B) ||
      !make_map(&mkv64, c.ckv, 576, slots, row_bytes, 64, box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !make_map(&mkv32, c.ckv, 576, slots, row_bytes, 32, box_rows, CU_TENSOR_MAP_SWIZZLE_64B))
    return cudaErrorInvalidValue;
  static std::once_flag attr_once;
  static cudaError_t attr_err = cudaSuccess;
  std::call_once(attr_once, [] {
    attr_err = cudaFuncSetAttribute(tc_decode_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    (int)kSmemBytes);
  });
  if (attr_err != cudaSuccess) return attr_err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * workers, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = kSmemBytes;
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
  return cudaLaunchKernelEx(&cfg, tc_decode_kernel, mq64, mq32, mkv64, mkv32, plan, bt, max_pages,
                            d.page_size, (int)box_rows, (int64_t)c.num_pages, (int)slots, q_per_seq,
                            scale_log2, o_part, lse_part, o_lat, lse, status);
}

}  // namespace mla

