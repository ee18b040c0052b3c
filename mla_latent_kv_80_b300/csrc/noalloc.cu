// Decode attention for callers that cannot allocate device memory.
//
// mla_decode_attn needs a caller-provided scratch workspace (the split plan
// and the split-KV partials). Some callers cannot call cudaMalloc at the point
// where they run a decode step: code running inside a region that the
// application's memory manager owns, plugins that are handed only their
// input and output buffers, or paths that must not touch the allocator at all.
// mla_decode_attn_noalloc gives them the same computation with the scratch in
// a fixed-size array that lives in this library's device image instead.
#include "mla_internal.cuh"

#include <mutex>

namespace mla {
namespace {

// Scratch for mla_decode_attn_noalloc: 48 MiB. It holds the split plan and the
// partials of the tensor-core path's default worker count (one per resident
// 2-SM cluster: 74 on a 148-SM GPU, about 39 MB at n_h = 128, d_c = 512). When
// num_splits = 0 and the default worker count of a path needs more (the
// CUDA-core path defaults to one worker per SM), the call uses the largest
// worker count whose scratch fits. Every GPU that loads the library keeps this
// array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(48) << 20;
__device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

// Device address of the scratch array on the current device. In host code the
// array's name is only a host-side stand-in, so the address is looked up once
// per device (with that device current) and cached for the lifetime of the
// device's primary context (a cudaDeviceReset invalidates it).
int scratch_address(void** out) {
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_NO_DEVICE;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
      cudaGetLastError();
      return MLA_ERR_CUDA;
    }
    addr[dev] = p;
  }
  *out = addr[dev];
  return MLA_OK;
}

}  // namespace
}  // namespace mla

extern "C" {

size_t mla_decode_noalloc_scratch_bytes(void) { return mla::kNoAllocScratchBytes; }

int mla_decode_attn_noalloc(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                            int32_t q_per_seq, const void* q_abs, const int32_t* block_table,
                            int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t num_splits,
                            void* o_lat, float* lse, int32_t* status, mla_stream_t stream) {
  size_t need = 0;
  int rc = mla_decode_workspace_size(dims, B, q_per_seq, num_splits, &need);
  if (rc != MLA_OK) return rc;
  if (num_splits == 0 && need > mla::kNoAllocScratchBytes) {
    // The default worker count does not fit: take the largest count that does.
    int32_t hi = 0;
    if ((rc = mla_decode_default_splits(dims, &hi)) != MLA_OK) return rc;
    int32_t lo = 0;  // largest count known to fit (0 = none yet)
    while (hi - lo > 1) {
      const int32_t mid = lo + (hi - lo) / 2;
      if ((rc = mla_decode_workspace_size(dims, B, q_per_seq, mid, &need)) != MLA_OK) return rc;
      if (need <= mla::kNoAllocScratchBytes) lo = mid;
      else hi = mid;
    }
    if (lo == 0) return MLA_ERR_WORKSPACE_TOO_SMALL;
    num_splits = lo;
    if ((rc = mla_decode_workspace_size(dims, B, q_per_seq, num_splits, &need)) != MLA_OK) return rc;
  }
  if (need > mla::kNoAllocScratchBytes) return MLA_ERR_WORKSPACE_TOO_SMALL;
  void* scratch = nullptr;
  rc = mla::scratch_address(&scratch);
  if (rc != MLA_OK) return rc;
  return mla_decode_attn(dims, cache, B, q_per_seq, q_abs, block_table, max_pages_per_seq, seq_lens,
                         num_splits, scratch, mla::kNoAllocScratchBytes, o_lat, lse, status, stream);
}

}  // extern "C"
