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
//     [32r, 32r+32). Every 64-token cache tile is TMA-loaded once: each CTA
//     fetches only its 288 columns, so HBM bytes are read exactly once.
//   * S_r = Q[:, cols_r] . K[:, cols_r]^T (M=128, N=64, K=288) lands in the
//     CTA's TMEM. The two partial scores are summed through distributed shared
//     memory (st.async into the peer, completion on the peer's mbarrier), so
//     both CTAs hold the identical S without doing the QK^T work twice.
//   * Both CTAs run the same online softmax (running max with lazy rescale,
//     exp2, bf16 P) and each accumulates its half of O = P . V (M=128, N=256)
//     in TMEM columns [0, 256). O for 128 heads x 512 latent columns in fp32
//     would fill one SM's TMEM; split across the pair it leaves room for S.
// Roles per CTA (256 threads): warp 0 lane 0 issues TMA, warp 1 lane 0 issues
// MMAs, warp 2 lane 0 moves the partial scores to the peer (one bulk copy per
// tile from a staging buffer), warps 4-7 (one thread per head row = TMEM lane)
// run the softmax, rescale and epilogue. The softmax warps never wait on each
// other: they hand off through mbarriers only. Every wait is bounded: after 2 s
// the kernel records MLA_ERR_DEVICE_TIMEOUT in *status and unwinds.
#include "tc_decode.cuh"
#include "sm100_ptx.cuh"

#include <cuda.h>
#include <math.h>
#include <mutex>

namespace mla {
using namespace ptx;

namespace tcd {
constexpr int kRows = 128;
constexpr int kTile = kTcTileN;  // 64 tokens
constexpr int kStages = 2;
constexpr int kPrefetch = 6;  // tiles ahead warmed in L2 (includes the kStages in shared memory)
constexpr uint32_t kQChunk = 128 * 128;           // [128 rows x 64 bf16], 128B swizzle
constexpr uint32_t kQBytes = 4 * kQChunk + 128 * 64;  // + [128 x 32] k_R part, 64B swizzle
constexpr uint32_t kKvChunk = 64 * 128;            // [64 tokens x 64 bf16]
constexpr uint32_t kKvKrOff = 4 * kKvChunk;
constexpr uint32_t kKvStage = 4 * kKvChunk + 64 * 64;
constexpr uint32_t kPBytes = 128 * 128;            // [128 rows x 64 tokens] bf16
constexpr uint32_t kXchgBytes = 128 * 64 * 4;      // one tile of partial scores, fp32
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_KV = OFF_Q + kQBytes;
constexpr uint32_t OFF_P = OFF_KV + kStages * kKvStage;
constexpr uint32_t OFF_SEND = OFF_P + kPBytes;      // own partial, staged for the bulk copy
constexpr uint32_t OFF_RECV = OFF_SEND + kXchgBytes;  // the peer's partial
constexpr uint32_t OFF_BAR = OFF_RECV + kXchgBytes;
constexpr uint32_t kSmemBytes = OFF_BAR + 256 + 1024;  // + alignment slack
// warp 0: TMA, warp 1: MMA, warp 2: score exchange, warp 3: idle, warps 4-7: softmax
constexpr int kThreads = 256;
enum Bar {
  B_QFULL, B_QEMPTY, B_KVFULL, B_KVFULL1, B_KVEMPTY, B_KVEMPTY1, B_SFULL, B_SFULL1,
  B_SFREE, B_SFREE1, B_PFULL, B_PVDONE, B_OFREE, B_RECV, B_SENDOK,
  B_STAGED,    // softmax warps staged this tile's partial scores
  B_SENDFREE,  // the bulk copy has read the staging buffer
  B_CONSUMED,  // softmax warps have read the peer's partial
  NBAR
};
constexpr uint32_t TM_O = 0, TM_S = 256, kTmemCols = 512;
constexpr uint64_t kWaitNs = 2000000000ull;
constexpr float kRescaleThreshold = 8.0f;  // log2 units: rescale O only when the max grows by 2^8
static_assert(OFF_KV % 1024 == 0 && OFF_P % 1024 == 0 && kKvStage % 1024 == 0, "swizzle atoms");
static_assert(kSmemBytes <= 232448, "shared memory");
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
  int per, w, g0, g1, p;
  __device__ void init(const int32_t* plan, int worker) {
    PlanView pv = plan_view(plan);
    cum = pv.cum;
    pbase = pv.pbase;
    lens = pv.len;
    const int P = plan[0], total = plan[1];
    per = plan[2];
    w = worker;
    g0 = worker * per;
    g1 = min(total, g0 + per);
    int lo = 0, hi = P > 0 ? P - 1 : 0;
    while (lo < hi) {
      int mid = (lo + hi) >> 1;
      if (cum[mid + 1] > g0) hi = mid; else lo = mid + 1;
    }
    p = lo;
  }
  __device__ bool next(int& prob, int& t_lo, int& t_hi, int& len, int& whole, int& slot) {
    if (g0 >= g1) return false;
    while (cum[p + 1] <= g0) ++p;
    t_lo = g0 - cum[p];
    t_hi = min(g1, cum[p + 1]) - cum[p];
    len = lens[p];
    const int c0 = cum[p], c1 = cum[p + 1];
    const int first = c0 / per, last = (c1 - 1) / per;
    whole = (last == first);
    slot = pbase[p] + (w - first);
    prob = p;
    g0 = cum[p] + t_hi;
    ++p;
    return true;
  }
};

__device__ __forceinline__ float bf16lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

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
  volatile int* abort_flag = reinterpret_cast<volatile int*>(gbase + OFF_BAR + 8 * NBAR);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(gbase + OFF_BAR + 8 * NBAR + 8);

  if (threadIdx.x == 0) {
    const uint32_t counts[NBAR] = {1, 1, 1, 1, 1, 1, 1, 1, 4, 4, 4, 1, 4, 1, 1, 4, 1, 4};
    for (int i = 0; i < NBAR; ++i) mbar_init(BAR(i), counts[i]);
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

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot;
      uint32_t seg = 0, j = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
        if (seg > 0 && !wait_bar(BAR(B_QEMPTY), (seg - 1) & 1, ctl)) break;
        mbar_arrive_expect_tx(BAR(B_QFULL), kQBytes);
        const int row0 = p * kRows;
        for (int c = 0; c < 4; ++c)
          tma_load_2d(base + OFF_Q + c * kQChunk, &tm_q64, (int)rank * 256 + c * 64, row0, BAR(B_QFULL));
        tma_load_2d(base + OFF_Q + 4 * kQChunk, &tm_q32, 512 + (int)rank * 32, row0, BAR(B_QFULL));
        const int b = p / q_per_seq;
        // Page-box row of token `tok` of this problem, or -1 past its end / on a bad page.
        auto box_row = [&](int tok) -> int {
          if (tok >= len) return -1;
          const int pg = tok / page_size;
          const int page = pg < max_pages ? bt[(size_t)b * max_pages + pg] : -1;
          if (page < 0 || page >= num_pages) return -2;
          return page * page_size + tok % page_size;
        };
        // Warm L2 with tiles ahead of the shared-memory ring so that HBM latency
        // overlaps the tiles being computed.
        auto prefetch_tile = [&](int t) {
          for (int r0 = 0; r0 < kTile; r0 += box_rows) {
            const int y = box_row(t * kTile + r0);
            if (y < 0) continue;
            for (int c = 0; c < 4; ++c) tma_prefetch_2d(&tm_kv64, (int)rank * 256 + c * 64, y);
            tma_prefetch_2d(&tm_kv32, 512 + (int)rank * 32, y);
          }
        };
        for (int t = t_lo + kStages; t < min(t_hi, t_lo + kPrefetch); ++t) prefetch_tile(t);
        for (int t = t_lo; t < t_hi; ++t, ++j) {
          if (t + kPrefetch < t_hi) prefetch_tile(t + kPrefetch);
          const int s = j % kStages;
          if (j >= (uint32_t)kStages &&
              !wait_bar(BAR(B_KVEMPTY + s), ((j / kStages) - 1) & 1, ctl)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(BAR(B_KVFULL + s), kKvStage);
          const uint32_t st = base + OFF_KV + s * kKvStage;
          for (int r0 = 0; r0 < kTile; r0 += box_rows) {
            int y = box_row(t * kTile + r0);
            if (y == -2) set_status(status, MLA_ERR_BAD_PAGE);
            if (y < 0) y = oob_row;  // fully out of range: the copy fills zeros
            for (int c = 0; c < 4; ++c)
              tma_load_2d(st + c * kKvChunk + r0 * 128, &tm_kv64, (int)rank * 256 + c * 64, y,
                          BAR(B_KVFULL + s));
            tma_load_2d(st + kKvKrOff + r0 * 64, &tm_kv32, 512 + (int)rank * 32, y, BAR(B_KVFULL + s));
          }
        }
        ++seg;
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(128, kTile, false, false);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(128, 256, false, true);
      auto issue_pv = [&](uint32_t jj, bool first, uint32_t segi) -> bool {
        if (!wait_bar(BAR(B_PFULL), jj & 1, ctl)) return false;
        if (first && segi > 0 && !wait_bar(BAR(B_OFREE), (segi - 1) & 1, ctl)) return false;
        tc_fence_after();
        const uint32_t st = base + OFF_KV + (jj % kStages) * kKvStage;
        for (int kk = 0; kk < kTile / 16; ++kk) {
          const uint64_t a = smem_desc(base + OFF_P + kk * 32, 16, 1024, kSwizzle128B);
          const uint64_t bdesc = smem_desc(st + kk * 2048, kKvChunk, 1024, kSwizzle128B);
          mma_f16(tmem + TM_O, a, bdesc, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
        mma_commit(BAR(B_KVEMPTY + (jj % kStages)));
        mma_commit(BAR(B_PVDONE));
        return true;
      };
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot;
      uint32_t seg = 0, j0 = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
        if (!wait_bar(BAR(B_QFULL), seg & 1, ctl)) break;
        tc_fence_after();
        const int n = t_hi - t_lo;
        for (int k = 0; k < n; ++k) {
          const uint32_t j = j0 + k;
          const int s = j % kStages, sb = j & 1;
          if (!wait_bar(BAR(B_KVFULL + s), (j / kStages) & 1, ctl)) { ok = false; break; }
          if (j >= 2 && !wait_bar(BAR(B_SFREE + sb), ((j >> 1) - 1) & 1, ctl)) { ok = false; break; }
          tc_fence_after();
          const uint32_t st = base + OFF_KV + s * kKvStage;
          const uint32_t d = tmem + TM_S + sb * kTile;
          for (int c = 0; c < 4; ++c)
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t a = smem_desc(base + OFF_Q + c * kQChunk + kk * 32, 16, 1024, kSwizzle128B);
              const uint64_t bdesc = smem_desc(st + c * kKvChunk + kk * 32, 16, 1024, kSwizzle128B);
              mma_f16(d, a, bdesc, idesc_s, (c | kk) ? 1u : 0u);
            }
          for (int kk = 0; kk < 2; ++kk) {
            const uint64_t a = smem_desc(base + OFF_Q + 4 * kQChunk + kk * 32, 16, 512, kSwizzle64B);
            const uint64_t bdesc = smem_desc(st + kKvKrOff + kk * 32, 16, 512, kSwizzle64B);
            mma_f16(d, a, bdesc, idesc_s, 1u);
          }
          mma_commit(BAR(B_SFULL + sb));
          if (k == n - 1) mma_commit(BAR(B_QEMPTY));
          if (k >= 1 && !issue_pv(j - 1, k == 1, seg)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(j0 + n - 1, n == 1, seg)) break;
        j0 += n;
        ++seg;
      }
    }
  } else if (warp == 2) {
    // ------------------------------------------------------------ score exchange
    // Moves this CTA's staged partial scores into the peer's receive buffer with
    // one bulk copy per tile and tells the peer when its data has been read, so
    // that neither the copy's completion nor the cluster-scope release waits on
    // the softmax warps' path.
    if (lane == 0) {
      const uint32_t recv_peer = mapa(base + OFF_RECV, peer);
      const uint32_t bar_recv_peer = mapa(BAR(B_RECV), peer);
      const uint32_t bar_sendok_peer = mapa(BAR(B_SENDOK), peer);
      SegIter it;
      it.init(plan, worker);
      int p, t_lo, t_hi, len, whole, slot;
      uint32_t j = 0;
      bool ok = true;
      while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
        for (int t = t_lo; t < t_hi; ++t, ++j) {
          if (!wait_bar(BAR(B_STAGED), j & 1, ctl)) { ok = false; break; }
          if (j >= 1 && !wait_bar(BAR(B_SENDOK), (j - 1) & 1, ctl, true)) { ok = false; break; }
          mbar_arrive_expect_tx(BAR(B_RECV), kXchgBytes);
          bulk_copy_to_peer(recv_peer, base + OFF_SEND, kXchgBytes, bar_recv_peer);
          bulk_commit();
          bulk_wait_read_all();
          mbar_arrive(BAR(B_SENDFREE));
          if (!wait_bar(BAR(B_CONSUMED), j & 1, ctl)) { ok = false; break; }
          mbar_arrive_remote(bar_sendok_peer);
        }
      }
      bulk_wait_read_all();
    }
  } else if (warp >= 4) {
    // ------------------------------------------------------------ softmax / epilogue
    const int r = threadIdx.x - 128;  // head row == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t row_off = (uint32_t)r * 256u;
    // Byte offset in an exchange buffer of 16-byte chunk c (of 16) of row r.
    auto xchg_off = [&](int c) { return row_off + (uint32_t)((c ^ (r & 7)) * 16); };
    SegIter it;
    it.init(plan, worker);
    int p, t_lo, t_hi, len, whole, slot;
    uint32_t seg = 0, j0 = 0;
    bool ok = true;
    while (ok && it.next(p, t_lo, t_hi, len, whole, slot)) {
      float m_ref = -INFINITY, l = 0.f;
      const int n = t_hi - t_lo;
      for (int k = 0; k < n; ++k) {
        const uint32_t j = j0 + k;
        const int sb = j & 1;
        if (!__all_sync(0xffffffffu, wait_bar(BAR(B_SFULL + sb), (j >> 1) & 1, ctl))) { ok = false; break; }
        tc_fence_after();
        uint32_t sv[64];
        {
          uint32_t (&lo)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[0]);
          uint32_t (&hi)[32] = *reinterpret_cast<uint32_t(*)[32]>(&sv[32]);
          tmem_ld32(tmem + lane_base + TM_S + sb * kTile, lo);
          tmem_ld32(tmem + lane_base + TM_S + sb * kTile + 32, hi);
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_SFREE + sb));
        // Stage the partial for the exchange warp once the previous copy has read it.
        if (j >= 1 && !__all_sync(0xffffffffu, wait_bar(BAR(B_SENDFREE), (j - 1) & 1, ctl))) { ok = false; break; }
#pragma unroll
        for (int c = 0; c < 16; ++c)
          *reinterpret_cast<uint4*>(gbase + OFF_SEND + xchg_off(c)) =
              make_uint4(sv[4 * c], sv[4 * c + 1], sv[4 * c + 2], sv[4 * c + 3]);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_STAGED));
        if (!__all_sync(0xffffffffu, wait_bar(BAR(B_RECV), j & 1, ctl, true))) { ok = false; break; }
        float s[64];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const uint4 v = *reinterpret_cast<const uint4*>(gbase + OFF_RECV + xchg_off(c));
          s[4 * c] = __uint_as_float(sv[4 * c]) + __uint_as_float(v.x);
          s[4 * c + 1] = __uint_as_float(sv[4 * c + 1]) + __uint_as_float(v.y);
          s[4 * c + 2] = __uint_as_float(sv[4 * c + 2]) + __uint_as_float(v.z);
          s[4 * c + 3] = __uint_as_float(sv[4 * c + 3]) + __uint_as_float(v.w);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_CONSUMED));
        // Online softmax in log2 units: scale, mask past the end, tree maximum.
        const int valid = min(kTile, len - (t_lo + k) * kTile);
#pragma unroll
        for (int x = 0; x < 64; ++x) s[x] = x < valid ? s[x] * scale_log2 : -INFINITY;
        float mx[16];
#pragma unroll
        for (int x = 0; x < 16; ++x) mx[x] = fmaxf(fmaxf(s[x], s[x + 16]), fmaxf(s[x + 32], s[x + 48]));
#pragma unroll
        for (int x = 0; x < 8; ++x) mx[x] = fmaxf(mx[x], mx[x + 8]);
#pragma unroll
        for (int x = 0; x < 4; ++x) mx[x] = fmaxf(mx[x], mx[x + 4]);
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        const bool need = (m_ref == -INFINITY) || (mt > m_ref + kRescaleThreshold);
        const float m_new = need ? fmaxf(mt, m_ref) : m_ref;
        const float factor = need ? ex2_approx(m_ref - m_new) : 1.f;
        uint32_t pk[32];
        float ps[8];
#pragma unroll
        for (int x = 0; x < 8; ++x) ps[x] = 0.f;
#pragma unroll
        for (int x = 0; x < 32; ++x) {
          const __nv_bfloat162 h2 = __floats2bfloat162_rn(ex2_approx(s[2 * x] - m_new), ex2_approx(s[2 * x + 1] - m_new));
          pk[x] = *reinterpret_cast<const uint32_t*>(&h2);
          ps[x & 7] += bf16lo(pk[x]) + bf16hi(pk[x]);
        }
        l = l * factor + (((ps[0] + ps[1]) + (ps[2] + ps[3])) + ((ps[4] + ps[5]) + (ps[6] + ps[7])));
        m_ref = m_new;
        // The P buffer and O are free once the previous P . V has completed.
        if (j >= 1 && !__all_sync(0xffffffffu, wait_bar(BAR(B_PVDONE), (j - 1) & 1, ctl))) { ok = false; break; }
        tc_fence_after();
        // Rows decide independently whether their running max moved; the TMEM
        // accesses are warp-collective, so the whole warp rescales when any
        // row needs it (rows that do not use a factor of 1).
        const bool rescale = need && k > 0;
        if (__any_sync(0xffffffffu, rescale)) {
          const float f = rescale ? factor : 1.f;
#pragma unroll 1
          for (int cc = 0; cc < 8; ++cc) {
            uint32_t o[32];
            tmem_ld32(tmem + lane_base + TM_O + cc * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int x = 0; x < 32; ++x) o[x] = __float_as_uint(__uint_as_float(o[x]) * f);
            tmem_st32(tmem + lane_base + TM_O + cc * 32, o);
          }
          tmem_wait_st();
        }
        uint8_t* prow = gbase + OFF_P + r * 128;
#pragma unroll
        for (int c = 0; c < 8; ++c)
          *reinterpret_cast<uint4*>(prow + ((c ^ (r & 7)) * 16)) =
              make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        if (valid < kTile) {
          // Rows past the sequence end may hold anything (NaN): zero them so that
          // P = 0 times V cannot poison O.
          uint8_t* st = gbase + OFF_KV + (j % kStages) * kKvStage;
          const int words = (kTile - valid) * 36;
          for (int i = r; i < words; i += 128) {
            const int row = valid + i / 36, wd = i % 36;
            uint8_t* dst = wd < 32 ? st + (wd >> 3) * kKvChunk + row * 128 + (wd & 7) * 16
                                   : st + kKvKrOff + row * 64 + (wd - 32) * 16;
            *reinterpret_cast<uint4*>(dst) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(B_PFULL));
      }
      if (!ok) break;
      // Segment epilogue: O / l to o_lat (whole problem) or to a partial slot.
      const uint32_t jl = j0 + n - 1;
      if (!__all_sync(0xffffffffu, wait_bar(BAR(B_PVDONE), jl & 1, ctl))) break;
      tc_fence_after();
      const float inv_l = 1.f / l;
      const size_t row = (size_t)p * kRows + r;
#pragma unroll 1
      for (int cc = 0; cc < 8; ++cc) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + TM_O + cc * 32, o);
        tmem_wait_ld();
        const int col = (int)rank * 256 + cc * 32;
        if (whole) {
          uint4* dst = reinterpret_cast<uint4*>(o_lat + row * 512 + col);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const __nv_bfloat162 h2 = __floats2bfloat162_rn(__uint_as_float(o[q4 * 8 + 2 * e]) * inv_l,
                                                              __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv_l);
              w4[e] = *reinterpret_cast<const uint32_t*>(&h2);
            }
            dst[q4] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        } else {
          float4* dst = reinterpret_cast<float4*>(o_part + ((size_t)slot * kRows + r) * 512 + col);
#pragma unroll
          for (int q4 = 0; q4 < 8; ++q4)
            dst[q4] = make_float4(__uint_as_float(o[4 * q4]) * inv_l, __uint_as_float(o[4 * q4 + 1]) * inv_l,
                                  __uint_as_float(o[4 * q4 + 2]) * inv_l, __uint_as_float(o[4 * q4 + 3]) * inv_l);
        }
      }
      if (rank == 0) {
        const float lse = (m_ref + log2f(l)) * 0.69314718055994531f;
        if (whole) lse_out[row] = lse;
        else lse_part[(size_t)slot * kRows + r] = lse;
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(B_OFREE));
      j0 += n;
      ++seg;
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
  static int cached[64];
  static std::once_flag once;
  std::call_once(once, [] {
    for (int i = 0; i < 64; ++i) cached[i] = -1;
  });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
  if (cached[dev] < 0) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return false;
    cached[dev] = (major == 10 && minor == 3) ? 1 : 0;
  }
  return cached[dev] == 1;
}


int tc_decode_max_workers() {
  static int cached[64];
  static std::once_flag once;
  std::call_once(once, [] {
    for (int i = 0; i < 64; ++i) cached[i] = 0;
  });
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
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
    cached[dev] = clusters;
  }
  return cached[dev];
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
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const float scale_log2 = d.softmax_scale * 1.4426950408889634f;
  return cudaLaunchKernelEx(&cfg, tc_decode_kernel, mq64, mq32, mkv64, mkv32, plan, bt, max_pages,
                            d.page_size, (int)box_rows, (int64_t)c.num_pages, (int)slots, q_per_seq,
                            scale_log2, o_part, lse_part, o_lat, lse, status);
}

}  // namespace mla
