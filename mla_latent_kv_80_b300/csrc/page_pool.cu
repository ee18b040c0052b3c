// Host-side page pool of the paged latent cache, and the device copy of pages.
//
// The cache is paged by token, and sequences that share a prefix share its
// latent vectors ("MLA 之后，KV cache 确实得重新理解一遍", "所以 cache 逻辑到底哪里
// 要重写": prefix sharing and prefix caching share the latent vectors; sliding
// windows and per-token eviction keep working). This pool hands out page ids
// for the block table:
//  * pages are reference counted; a forked sequence shares every full page of
//    its parent's shared prefix, and a partially filled last page is copied
//    (the copy is queued for mla_copy_pages) so that neither side ever appends
//    into a page the other can see;
//  * evicting a sequence's positions before p releases the pages that hold
//    only such positions (their table entries become -1) and raises the
//    sequence's first visible position, which mla_decode_attn_window takes;
//  * a page returns to the free list when no sequence refers to it.
// All pool calls are host-only and serialised by the pool's mutex.
#include "mla_internal.cuh"

#include <mutex>
#include <new>
#include <vector>

struct mla_pool {
  std::mutex mu;
  int64_t num_pages = 0;
  int32_t page_size = 0, max_seqs = 0, max_pages = 0;
  std::vector<int32_t> refs;        // per page
  std::vector<int32_t> free_list;   // pages with refs == 0 (a stack)
  std::vector<uint8_t> live;        // per sequence slot
  std::vector<int32_t> capacity;    // positions [0, capacity) have pages (or were evicted)
  std::vector<int32_t> start;       // first visible position
  std::vector<int32_t> table;       // [max_seqs][max_pages], -1 = none
  std::vector<int32_t> copy_src, copy_dst;  // pending page copies
};

namespace {

int32_t* row_of(mla_pool* p, int32_t seq) { return p->table.data() + (size_t)seq * p->max_pages; }

bool valid_seq(const mla_pool* p, int32_t seq) {
  return seq >= 0 && seq < p->max_seqs && p->live[(size_t)seq];
}

int32_t take_page(mla_pool* p) {
  if (p->free_list.empty()) return -1;
  const int32_t pg = p->free_list.back();
  p->free_list.pop_back();
  p->refs[(size_t)pg] = 1;
  return pg;
}

void drop_page(mla_pool* p, int32_t pg) {
  if (pg < 0) return;
  if (--p->refs[(size_t)pg] == 0) p->free_list.push_back(pg);
}

int32_t new_slot(mla_pool* p) {
  for (int32_t s = 0; s < p->max_seqs; ++s)
    if (!p->live[(size_t)s]) {
      p->live[(size_t)s] = 1;
      p->capacity[(size_t)s] = 0;
      p->start[(size_t)s] = 0;
      int32_t* r = row_of(p, s);
      for (int32_t i = 0; i < p->max_pages; ++i) r[i] = -1;
      return s;
    }
  return -1;
}

}  // namespace

extern "C" {

int mla_pool_create(int64_t num_pages, int32_t page_size, int32_t max_seqs, int32_t max_pages_per_seq,
                    mla_pool_t** pool) {
  if (pool == nullptr || num_pages < 1 || num_pages > 0x7FFFFFFF || page_size < 1 || max_seqs < 1 ||
      max_pages_per_seq < 1)
    return MLA_ERR_INVALID_ARG;
  mla_pool* p = new (std::nothrow) mla_pool;
  if (p == nullptr) return MLA_ERR_NO_PAGES;
  p->num_pages = num_pages;
  p->page_size = page_size;
  p->max_seqs = max_seqs;
  p->max_pages = max_pages_per_seq;
  p->refs.assign((size_t)num_pages, 0);
  p->free_list.reserve((size_t)num_pages);
  for (int64_t i = num_pages - 1; i >= 0; --i) p->free_list.push_back((int32_t)i);  // page 0 first
  p->live.assign((size_t)max_seqs, 0);
  p->capacity.assign((size_t)max_seqs, 0);
  p->start.assign((size_t)max_seqs, 0);
  p->table.assign((size_t)max_seqs * max_pages_per_seq, -1);
  *pool = p;
  return MLA_OK;
}

void mla_pool_destroy(mla_pool_t* pool) { delete pool; }

int mla_pool_new_seq(mla_pool_t* p, int32_t* seq) {
  if (p == nullptr || seq == nullptr) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  const int32_t s = new_slot(p);
  if (s < 0) return MLA_ERR_NO_PAGES;
  *seq = s;
  return MLA_OK;
}

int mla_pool_reserve(mla_pool_t* p, int32_t seq, int32_t len) {
  if (p == nullptr || len < 0) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!valid_seq(p, seq)) return MLA_ERR_INVALID_ARG;
  const int32_t need = (len + p->page_size - 1) / p->page_size;
  if (need > p->max_pages) return MLA_ERR_INVALID_ARG;
  int32_t* r = row_of(p, seq);
  const int32_t have = (p->capacity[(size_t)seq] + p->page_size - 1) / p->page_size;
  int32_t missing = 0;
  for (int32_t i = have; i < need; ++i) missing += (r[i] < 0);
  if ((size_t)missing > p->free_list.size()) return MLA_ERR_NO_PAGES;
  for (int32_t i = have; i < need; ++i)
    if (r[i] < 0) r[i] = take_page(p);
  if (len > p->capacity[(size_t)seq]) p->capacity[(size_t)seq] = len;
  return MLA_OK;
}

int mla_pool_fork(mla_pool_t* p, int32_t parent, int32_t shared_tokens, int32_t* child) {
  if (p == nullptr || child == nullptr || shared_tokens < 0) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!valid_seq(p, parent) || shared_tokens > p->capacity[(size_t)parent]) return MLA_ERR_INVALID_ARG;
  const int32_t full = shared_tokens / p->page_size;
  const bool partial = shared_tokens % p->page_size != 0;
  const int32_t* pr = row_of(p, parent);
  if (partial && p->free_list.empty()) return MLA_ERR_NO_PAGES;
  const int32_t c = new_slot(p);
  if (c < 0) return MLA_ERR_NO_PAGES;
  int32_t* cr = row_of(p, c);
  for (int32_t i = 0; i < full; ++i) {
    cr[i] = pr[i];
    if (pr[i] >= 0) ++p->refs[(size_t)pr[i]];
  }
  if (partial) {
    const int32_t src = pr[full];
    const int32_t dst = take_page(p);
    cr[full] = dst;
    if (src >= 0) {
      p->copy_src.push_back(src);
      p->copy_dst.push_back(dst);
    }
  }
  p->capacity[(size_t)c] = shared_tokens;
  p->start[(size_t)c] = p->start[(size_t)parent] < shared_tokens ? p->start[(size_t)parent] : shared_tokens;
  *child = c;
  return MLA_OK;
}

int mla_pool_evict_before(mla_pool_t* p, int32_t seq, int32_t pos) {
  if (p == nullptr || pos < 0) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!valid_seq(p, seq)) return MLA_ERR_INVALID_ARG;
  if (pos > p->capacity[(size_t)seq]) pos = p->capacity[(size_t)seq];
  int32_t* r = row_of(p, seq);
  for (int32_t i = 0; i < pos / p->page_size; ++i) {
    drop_page(p, r[i]);
    r[i] = -1;
  }
  if (pos > p->start[(size_t)seq]) p->start[(size_t)seq] = pos;
  return MLA_OK;
}

int mla_pool_free_seq(mla_pool_t* p, int32_t seq) {
  if (p == nullptr) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!valid_seq(p, seq)) return MLA_ERR_INVALID_ARG;
  int32_t* r = row_of(p, seq);
  for (int32_t i = 0; i < p->max_pages; ++i) {
    drop_page(p, r[i]);
    r[i] = -1;
  }
  p->live[(size_t)seq] = 0;
  return MLA_OK;
}

int mla_pool_block_table(mla_pool_t* p, int32_t* table) {
  if (p == nullptr || table == nullptr) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  for (size_t i = 0; i < p->table.size(); ++i) table[i] = p->table[i];
  return MLA_OK;
}

int mla_pool_seq_info(mla_pool_t* p, int32_t seq, int32_t* capacity, int32_t* start) {
  if (p == nullptr || capacity == nullptr || start == nullptr) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  if (!valid_seq(p, seq)) return MLA_ERR_INVALID_ARG;
  *capacity = p->capacity[(size_t)seq];
  *start = p->start[(size_t)seq];
  return MLA_OK;
}

int mla_pool_page_refs(mla_pool_t* p, int32_t page, int32_t* refs) {
  if (p == nullptr || refs == nullptr || page < 0 || page >= p->num_pages) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  *refs = p->refs[(size_t)page];
  return MLA_OK;
}

int mla_pool_free_pages(mla_pool_t* p, int64_t* n) {
  if (p == nullptr || n == nullptr) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  *n = (int64_t)p->free_list.size();
  return MLA_OK;
}

int mla_pool_take_copies(mla_pool_t* p, int32_t* src, int32_t* dst, int32_t max, int32_t* n) {
  if (p == nullptr || n == nullptr || max < 0) return MLA_ERR_INVALID_ARG;
  std::lock_guard<std::mutex> lock(p->mu);
  const int32_t k = (int32_t)p->copy_src.size();
  if (k > max || (k > 0 && (src == nullptr || dst == nullptr))) {
    *n = k;
    return MLA_ERR_WORKSPACE_TOO_SMALL;
  }
  for (int32_t i = 0; i < k; ++i) {
    src[i] = p->copy_src[(size_t)i];
    dst[i] = p->copy_dst[(size_t)i];
  }
  p->copy_src.clear();
  p->copy_dst.clear();
  *n = k;
  return MLA_OK;
}

}  // extern "C"

// ====================================================================== device page copy
namespace mla {
namespace {

// One block per page copy; the page's bytes of every cache array move in
// 16-byte words (page rows are contiguous in each array).
__global__ void __launch_bounds__(256) copy_pages_kernel(int n, const int32_t* __restrict__ src,
                                                         const int32_t* __restrict__ dst, int64_t num_pages,
                                                         uint4* a0, size_t w0, uint4* a1, size_t w1, uint4* a2,
                                                         size_t w2, int32_t* status) {
  pdl_trigger();
  pdl_wait();
  const int i = blockIdx.x;
  if (i >= n) return;
  const int64_t s = src[i], d = dst[i];
  if (s < 0 || s >= num_pages || d < 0 || d >= num_pages) {
    if (threadIdx.x == 0) set_status(status, MLA_ERR_BAD_PAGE);
    return;
  }
  uint4* arr[3] = {a0, a1, a2};
  const size_t words[3] = {w0, w1, w2};
  for (int k = 0; k < 3; ++k) {
    if (arr[k] == nullptr) continue;
    const uint4* from = arr[k] + (size_t)s * words[k];
    uint4* to = arr[k] + (size_t)d * words[k];
    for (size_t x = threadIdx.x; x < words[k]; x += blockDim.x) to[x] = from[x];
  }
}

}  // namespace
}  // namespace mla

extern "C" int mla_copy_pages(const mla_dims_t* dims, const mla_cache_t* cache, int32_t n, const int32_t* src,
                              const int32_t* dst, int32_t* status, mla_stream_t stream) {
  using namespace mla;
  if (dims == nullptr || cache == nullptr || cache->ckv == nullptr || n < 0) return MLA_ERR_INVALID_ARG;
  if (n == 0) return MLA_OK;
  if (src == nullptr || dst == nullptr) return MLA_ERR_INVALID_ARG;
  const size_t ps = (size_t)dims->page_size;
  size_t w0, w1 = 0, w2 = 0;
  void *a1 = nullptr, *a2 = nullptr;
  if (dims->cache_dtype == MLA_FP8_E4M3) {
    if (cache->kr == nullptr || cache->scale == nullptr) return MLA_ERR_INVALID_ARG;
    w0 = ps * dims->d_c;                     // E4M3 codes
    w1 = ps * dims->d_rope * 2;              // bf16 k_R
    w2 = ps * 4;                             // fp32 scales
    a1 = cache->kr;
    a2 = cache->scale;
  } else {
    w0 = ps * (size_t)(dims->d_c + dims->d_rope) * (dims->cache_dtype == MLA_F32 ? 4 : 2);
  }
  if (w0 % 16 || w1 % 16 || w2 % 16) return MLA_ERR_UNSUPPORTED;  // pages must be whole 16-byte words
  const uintptr_t align = reinterpret_cast<uintptr_t>(cache->ckv) | reinterpret_cast<uintptr_t>(a1) |
                          reinterpret_cast<uintptr_t>(a2);
  if (align & 15) return MLA_ERR_INVALID_ARG;
  cudaError_t e = launch_pdl(copy_pages_kernel, dim3(n), dim3(256), 0, reinterpret_cast<cudaStream_t>(stream), n, src,
                             dst, (int64_t)cache->num_pages, static_cast<uint4*>(cache->ckv), w0 / 16,
                             static_cast<uint4*>(a1), w1 / 16, static_cast<uint4*>(a2), w2 / 16, status);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
