/*
 * mla.h — C ABI of the B300 (sm_103a) MLA decode library, libmla.so.
 *
 * Multi-head Latent Attention (DeepSeek-V2) caches, per token and per layer,
 * only a joint latent c_KV = W_DKV h (d_c wide) and a decoupled RoPE key
 * k_R = RoPE(W_KR h) (d_rope wide, shared by every head): 576 values at
 * d_c = 512, d_rope = 64 ("MLA 之后，KV cache 确实得重新理解一遍", sections
 * "第一步" and "RoPE 为什么必须解耦"). Decode attention runs directly on that
 * cache after the key up-projection is absorbed into the query and the value
 * up-projection is applied once to the latent weighted sum (same page,
 * "第二步，推理时的吸收"). One decode step is:
 *
 *   mla_cache_append   write the current token's [c_KV | k_R] into its paged slot
 *   mla_absorb_q       q_abs = [W_UK^T q_nope | RoPE(q_rope)] per head
 *   mla_decode_attn    softmax(scale * q_abs . [c_KV | k_R]) . c_KV over the cache,
 *                      split-KV with an exact log-sum-exp merge
 *   mla_out_proj       o = W_UV . o_lat per head
 *   mla_out_proj_wo    the same, then the layer output W_O . [o_1 ; ... ; o_n_h]
 *
 * Conventions shared by every call
 *  - Pointers named in the argument lists are DEVICE pointers unless stated
 *    otherwise; the caller owns all memory. Calls allocate nothing, never
 *    synchronise, and enqueue their kernels on `stream` (NULL = legacy default
 *    stream). Calls are re-entrant; each call's kernels run in stream order.
 *  - Return value: MLA_OK (0) or a negative mla_status_t. Argument errors are
 *    detected on the host before anything is enqueued. MLA_ERR_CUDA means a
 *    launch failed (cudaGetLastError after the launch).
 *  - Errors found while the kernels run (a block-table entry outside
 *    [0, num_pages), a bounded wait that gave up) are written to `*status`, a
 *    caller-owned device int32 that the kernels only ever set to a negative
 *    code; the caller zeroes it, synchronises and reads it. A kernel that finds
 *    such an error skips the offending access; its outputs are then undefined.
 *  - Positions count from 0. Query j (0 <= j < q_per_seq) of sequence b sits at
 *    position seq_lens[b] - q_per_seq + j and sees every cached key at a
 *    position <= its own ("append first, then attend over history and the
 *    current token": the interview-answer page on MLA and KV Cache, section
 *    "先区分 KV Cache 与 MLA").
 *  - RoPE rotates interleaved pairs (2i, 2i+1) of a d_rope-wide vector at
 *    position p by the angle p * rope_theta^(-2i/d_rope); the frequencies are
 *    computed in double precision on the host, the angle and its reduction
 *    modulo 2*pi in single precision with an exact product residual and a
 *    three-part 2*pi (within about 4e-7 rad for positions below 2^23), the
 *    sine and cosine of the reduced angle in fp32.
 *  - bf16 results are rounded to nearest-even from fp32 accumulators.
 */
#ifndef MLA_H_
#define MLA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

typedef struct CUstream_st* mla_stream_t; /* same type as cudaStream_t */

typedef enum {
  MLA_F32 = 0,      /* IEEE fp32 */
  MLA_BF16 = 1,     /* bfloat16 */
  MLA_FP8_E4M3 = 2  /* OCP FP8 E4M3 (cache c_KV only), one fp32 scale per token */
} mla_dtype_t;

typedef enum {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = -1,         /* null pointer, negative size, bad page size, ... */
  MLA_ERR_UNSUPPORTED = -2,         /* dimension or dtype combination not built */
  MLA_ERR_WORKSPACE_TOO_SMALL = -3, /* workspace_bytes below the *_workspace_size answer */
  MLA_ERR_CUDA = -4,                /* a kernel launch failed */
  MLA_ERR_BAD_PAGE = -5,            /* device: block-table entry outside [0, num_pages) */
  MLA_ERR_DEVICE_TIMEOUT = -6,      /* device: a bounded wait inside a kernel gave up */
  MLA_ERR_NO_DEVICE = -7,           /* no CUDA device or driver entry point */
  MLA_ERR_NO_PAGES = -8             /* page pool: no free page or sequence slot left */
} mla_status_t;

/* Model dimensions and formats of one attention layer.
 * Supported shapes: any n_h >= 1, d_h, d_v <= 512, d_c <= 512 and a multiple of 16,
 * d_rope <= 64 and even, d_model a multiple of 8. The tensor-core path covers
 * n_h = 128, d_c = 512, d_rope = 64, d_h = d_v = 128 with bf16 activations;
 * other shapes run on CUDA-core kernels of the same library. */
typedef struct {
  int32_t n_h;           /* attention heads */
  int32_t d_h;           /* per-head no-RoPE query/key width (q_nope) */
  int32_t d_rope;        /* decoupled RoPE width d_h^R (q_rope, k_R) */
  int32_t d_c;           /* joint KV latent width */
  int32_t d_v;           /* per-head value / output width */
  int32_t d_model;       /* hidden-state width */
  int32_t page_size;     /* tokens per cache page: 16, 32, 64 or 128 */
  float softmax_scale;   /* finite and > 0; usually 1/sqrt(d_h + d_rope) */
  float rope_theta;      /* RoPE base, finite and > 0; usually 10000 */
  int32_t act_dtype;     /* MLA_F32 or MLA_BF16: h, q, weights, q_abs, o_lat, o */
  int32_t cache_dtype;   /* MLA_F32 (with F32 acts), MLA_BF16 (with BF16 acts) or MLA_FP8_E4M3 */
} mla_dims_t;

/* The paged latent cache. A slot is page * page_size + offset; sequence b's
 * token at position t lives in slot block_table[b][t / page_size] * page_size
 * + t % page_size.
 *  F32 / BF16 caches: ckv is [num_pages * page_size][d_c + d_rope] in the cache
 *    dtype, c_KV in columns [0, d_c) and the rotated k_R in [d_c, d_c + d_rope);
 *    kr and scale are NULL.
 *  FP8 cache: ckv is [slots][d_c] E4M3 codes (uint8), kr is [slots][d_rope]
 *    bf16, scale is [slots] fp32; the stored latent is code * scale.
 * Base pointers must be 16-byte aligned. */
typedef struct {
  void* ckv;
  void* kr;
  float* scale;
  int64_t num_pages;
} mla_cache_t;

/* ---------------------------------------------------------------- append
 * Writes the cache entries of T new tokens (the decode step's current tokens,
 * or a prefill's tokens):
 *   x      = [W_DKV ; W_KR] . h_t                 (d_c + d_rope outputs, fp32 accumulate)
 *   c_KV   = x[0:d_c]                             (page 2 "第一步"; page 3 "1. 下采样")
 *   k_R    = RoPE(x[d_c:], pos[t])                 (rotated before caching: page 2
 *                                                  "RoPE 为什么必须解耦")
 * stored into slot(seq_idx[t], pos[t]) in the cache dtype. For FP8 caches the
 * latent is quantised per token: scale = amax(c_KV)/448 (1 if amax = 0, at least
 * FLT_MIN), code = E4M3 round-to-nearest-even, saturating, of c_KV / scale.
 *   h           [T][d_model] act dtype
 *   w_dkv       [d_c][d_model] act dtype;   w_kr [d_rope][d_model] act dtype
 *   seq_idx,pos [T] int32: sequence (row of block_table) and position of each token
 *   block_table [B][max_pages_per_seq] int32 page ids (B rows; only rows named
 *               by seq_idx are read)
 *   workspace   device scratch of at least mla_cache_append_workspace_size bytes
 *               (fp32 partial sums); may be NULL when that size is 0.
 * No two new tokens may share a slot. Slots other than the T written ones are
 * never touched. */
MLA_API int mla_cache_append_workspace_size(const mla_dims_t* dims, int32_t T, size_t* bytes);
MLA_API int mla_cache_append(const mla_dims_t* dims, const mla_cache_t* cache, int32_t T,
                     const void* h, const void* w_dkv, const void* w_kr,
                     const int32_t* seq_idx, const int32_t* pos,
                     const int32_t* block_table, int32_t max_pages_per_seq,
                     void* workspace, size_t workspace_bytes,
                     int32_t* status, mla_stream_t stream);

/* ---------------------------------------------------------------- absorb
 * Absorbs W_UK into the query (page 2, "第二步，推理时的吸收":
 * score = (W_UK^T q)^T c_KV) and rotates the decoupled RoPE part:
 *   q_abs[t][h][0:d_c]           = W_UK[h]^T . q[t][h][0:d_h]
 *   q_abs[t][h][d_c:d_c+d_rope]  = RoPE(q[t][h][d_h:d_h+d_rope], pos[t])
 *   q      [T][n_h][d_h + d_rope] act dtype ([q_nope | q_rope] per head)
 *   pos    [T] int32 query positions
 *   w_uk   [n_h][d_h][d_c] act dtype (W_UK[h] maps d_c -> d_h)
 *   q_abs  [T][n_h][d_c + d_rope] act dtype (output) */
MLA_API int mla_absorb_q(const mla_dims_t* dims, int32_t T, const void* q, const int32_t* pos,
                 const void* w_uk, void* q_abs, mla_stream_t stream);

/* ---------------------------------------------------------------- decode attention
 * For every sequence b < B, query j < q_per_seq and head h:
 *   s_t   = softmax_scale * (q_abs[b,j,h] . [c_KV,t | k_R,t])  for t <= pos(b, j)
 *   o_lat = sum_t softmax(s)_t c_KV,t                          (page 2, value absorption)
 *   lse   = log(sum_t exp(s_t))  (natural log; -inf and o_lat = 0 for an empty set)
 * The work (all sequences' KV tiles) is divided into `num_splits` contiguous
 * shares, one per worker; a sequence cut between workers is merged exactly with
 * the log-sum-exp rule by a second kernel. num_splits = 0 picks one worker per
 * SM pair (tensor-core path) or per SM. The plan is built on the device from
 * seq_lens: no host copy, no synchronisation.
 *   q_abs       [B * q_per_seq][n_h][d_c + d_rope] act dtype (row b*q_per_seq + j)
 *   block_table [B][max_pages_per_seq] int32
 *   seq_lens    [B] int32, device: keys visible to the last query of each sequence
 *   workspace   device scratch of at least mla_decode_workspace_size bytes
 *   o_lat       [B * q_per_seq][n_h][d_c] act dtype (output)
 *   lse         [B * q_per_seq][n_h] fp32 (output)
 * seq_lens[b] must not exceed max_pages_per_seq * page_size. */
/* Worker count that num_splits = 0 selects on the current device: the number of
 * 2-SM clusters of the tensor-core kernel that can be resident at once, else
 * the SM count. */
MLA_API int mla_decode_default_splits(const mla_dims_t* dims, int32_t* splits);
MLA_API int mla_decode_workspace_size(const mla_dims_t* dims, int32_t B, int32_t q_per_seq,
                              int32_t num_splits, size_t* bytes);
MLA_API int mla_decode_attn(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                    int32_t q_per_seq, const void* q_abs, const int32_t* block_table,
                    int32_t max_pages_per_seq, const int32_t* seq_lens, int32_t num_splits,
                    void* workspace, size_t workspace_bytes, void* o_lat, float* lse,
                    int32_t* status, mla_stream_t stream);

/* ---------------------------------------------------------------- decode over a window
 * mla_decode_attn with a first visible position per sequence: query j of
 * sequence b attends to the keys at positions [seq_start[b], its own position]
 * and to none before. This is decode after the cache's leading tokens were
 * evicted, or a sliding window ending at the last query (seq_start[b] =
 * seq_lens[b] - window): eviction and sliding windows keep working over the
 * latent cache, with a token's whole latent entry (K and V together) dropped
 * ("MLA 之后，KV cache 确实得重新理解一遍", "所以 cache 逻辑到底哪里要重写").
 *   seq_start   [B] int32, device, or NULL (all 0). Values below 0 count as 0;
 *               a start at or past a query's position leaves it no keys
 *               (o_lat = 0, lse = -inf).
 * Block-table entries of pages that hold only positions before seq_start[b]
 * are never read (they may be -1 once those pages are freed). Everything else
 * is as mla_decode_attn, which is this call with seq_start = NULL. */
MLA_API int mla_decode_attn_window(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                                   int32_t q_per_seq, const void* q_abs, const int32_t* block_table,
                                   int32_t max_pages_per_seq, const int32_t* seq_lens,
                                   const int32_t* seq_start, int32_t num_splits, void* workspace,
                                   size_t workspace_bytes, void* o_lat, float* lse, int32_t* status,
                                   mla_stream_t stream);

/* ---------------------------------------------------------------- chunked prefill (explicit form)
 * Attention of a chunk of C = q_per_seq query tokens per sequence over the
 * sequence's cache (the chunk's own tokens appended first), in the form the
 * pages give for training ("MLA 之后，KV cache 确实得重新理解一遍", "第一步，训练时":
 * keys and values are formed from c_KV; "MLA 是什么 | dg's Blog", "完整代码":
 * causal attention over the formed keys). Each cached token's per-head key
 * k_t = [W_UK[h] c_t ; k_R,t] and value v_t = W_UV[h] c_t are formed once per
 * call, then for every query j of sequence b and head h:
 *   s_t = softmax_scale * (q_nope . W_UK[h] c_t + RoPE(q_rope, pos) . k_R,t),  t <= pos
 *   o   = sum_t softmax(s)_t W_UV[h] c_t,   lse = log sum_t exp(s_t) (natural log)
 * with pos = seq_lens[b] - C + j, as for decode. A query at a negative position
 * sees no key (o = 0, lse = -inf). o is in value space: what mla_out_proj
 * returns on the absorbed path (the input of W_O).
 *   q           [B * C][n_h][d_h + d_rope] bf16, [q_nope | q_rope], q_rope not yet
 *               rotated (row b*C + j)
 *   w_uk, w_uv  [n_h][d_h][d_c], [n_h][d_v][d_c] bf16
 *   block_table [B][max_pages_per_seq] int32; seq_lens [B] int32, device
 *   B           at most 65535 sequences per call
 *   max_seq_len host bound on every seq_lens[b] (sizes the workspace); a larger
 *               seq_lens[b] is treated as max_seq_len and sets MLA_ERR_INVALID_ARG
 *               in *status
 *   workspace   device scratch of at least mla_prefill_workspace_size bytes: the
 *               gathered latent rows and the formed keys and values (bf16, n_h *
 *               (d_h + d_v) * 2 bytes per cached token)
 *   o           [B * C][n_h][d_v] bf16 (output); lse [B * C][n_h] fp32 (output)
 * Built for bf16 activations with d_h = d_v = 128, d_rope = 64, d_c a multiple
 * of 64, a bf16 or fp8 cache (fp8 entries are dequantised to bf16 when
 * gathered); otherwise MLA_ERR_UNSUPPORTED. A block-table entry outside
 * [0, num_pages) sets MLA_ERR_BAD_PAGE and its rows read as zero.
 *
 * Which form is cheaper. Per (query, visible key) pair the explicit form costs
 * 2 n_h (d_h + d_rope + d_v) flops and the absorbed form (mla_absorb_q,
 * mla_decode_attn, mla_out_proj) 2 n_h (2 d_c + d_rope); the explicit form adds
 * 2 n_h (d_h + d_v) d_c per cached token to form keys and values, the absorbed
 * form 2 n_h (d_h + d_v) d_c per query for absorbing W_UK and applying W_UV.
 * mla_prefill_form sets *explicit_form to 1 when, for C queries at the end of a
 * sequence of seq_len tokens, the explicit total is the smaller (for DeepSeek-V2
 * shapes once C exceeds about 170), else 0. */
MLA_API int mla_prefill_form(const mla_dims_t* dims, int32_t q_per_seq, int64_t seq_len,
                             int32_t* explicit_form);
MLA_API int mla_prefill_workspace_size(const mla_dims_t* dims, int32_t B, int32_t q_per_seq,
                                       int32_t max_seq_len, size_t* bytes);
MLA_API int mla_prefill_attn(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                             int32_t q_per_seq, int32_t max_seq_len, const void* q, const void* w_uk,
                             const void* w_uv, const int32_t* block_table, int32_t max_pages_per_seq,
                             const int32_t* seq_lens, void* workspace, size_t workspace_bytes, void* o,
                             float* lse, int32_t* status, mla_stream_t stream);
/* mla_prefill_attn with a first visible position per sequence: query j of
 * sequence b attends to the keys at positions [seq_start[b], its position]
 * only (the chunk's prefill after the cache's leading tokens were evicted, or
 * a sliding window); see mla_decode_attn_window for the reading.
 *   seq_start   [B] int32, device, or NULL (all 0). Values below 0 count as 0;
 *               a query at a position before seq_start[b] sees no key
 *               (o = 0, lse = -inf).
 * Block-table entries of pages that hold only positions before seq_start[b]
 * are never read. mla_prefill_attn is this call with seq_start = NULL. */
MLA_API int mla_prefill_attn_window(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                                    int32_t q_per_seq, int32_t max_seq_len, const void* q, const void* w_uk,
                                    const void* w_uv, const int32_t* block_table, int32_t max_pages_per_seq,
                                    const int32_t* seq_lens, const int32_t* seq_start, void* workspace,
                                    size_t workspace_bytes, void* o, float* lse, int32_t* status,
                                    mla_stream_t stream);

/* ---------------------------------------------------------------- failure-path self-test
 * Every wait inside the library's kernels (on an mbarrier, for a TMA copy, an
 * MMA or another CTA of the cluster) is bounded: after its limit the kernel
 * writes MLA_ERR_DEVICE_TIMEOUT to *status and unwinds instead of hanging.
 * mla_selftest_bounded_wait runs one block that waits, with the same polling
 * loop, on an mbarrier that nothing arrives on, limited to limit_ns (at most
 * 2 s): the call always ends with *status = MLA_ERR_DEVICE_TIMEOUT (if it was
 * MLA_OK) and leaves the context usable. No fault or trap is involved. */
MLA_API int mla_selftest_bounded_wait(uint64_t limit_ns, int32_t* status, mla_stream_t stream);

/* ---------------------------------------------------------------- page pool (host) and page copies
 * A host-side manager of the cache's page ids for block tables. Sequences that
 * share a prefix share its latent vectors ("MLA 之后，KV cache 确实得重新理解一
 * 遍", "所以 cache 逻辑到底哪里要重写": prefix sharing shares the latent vectors;
 * sliding windows and per-token eviction keep working):
 *  - pages are reference counted and return to the free list when no sequence
 *    refers to them; page 0 is handed out first;
 *  - mla_pool_fork shares the parent's full pages of the first shared_tokens
 *    positions and copies a partially filled last page: the copy is queued and
 *    must be executed (mla_pool_take_copies, then mla_copy_pages) before either
 *    sequence appends, so that neither ever writes a page the other can see;
 *  - mla_pool_evict_before releases the pages holding only positions before
 *    pos (their table entries become -1) and raises the sequence's first
 *    visible position to pos, the seq_start of mla_decode_attn_window;
 *  - mla_pool_block_table writes the table [max_seqs][max_pages_per_seq] int32
 *    (host memory; -1 = no page) for the caller to copy to the device.
 * Pool calls are host-only (no GPU work) and thread-safe; MLA_ERR_NO_PAGES
 * means the pool or its sequence slots are exhausted (nothing was changed).
 * mla_copy_pages (device, on `stream`) copies every cache array's rows of page
 * src[i] to page dst[i] for i < n (src and dst are device int32 arrays); a page
 * id outside [0, num_pages) sets MLA_ERR_BAD_PAGE in *status and is skipped. */
typedef struct mla_pool mla_pool_t;
MLA_API int mla_pool_create(int64_t num_pages, int32_t page_size, int32_t max_seqs,
                            int32_t max_pages_per_seq, mla_pool_t** pool);
MLA_API void mla_pool_destroy(mla_pool_t* pool);
MLA_API int mla_pool_new_seq(mla_pool_t* pool, int32_t* seq);
MLA_API int mla_pool_reserve(mla_pool_t* pool, int32_t seq, int32_t len);
MLA_API int mla_pool_fork(mla_pool_t* pool, int32_t parent, int32_t shared_tokens, int32_t* child);
MLA_API int mla_pool_evict_before(mla_pool_t* pool, int32_t seq, int32_t pos);
MLA_API int mla_pool_free_seq(mla_pool_t* pool, int32_t seq);
MLA_API int mla_pool_block_table(mla_pool_t* pool, int32_t* table);
MLA_API int mla_pool_seq_info(mla_pool_t* pool, int32_t seq, int32_t* capacity, int32_t* start);
MLA_API int mla_pool_page_refs(mla_pool_t* pool, int32_t page, int32_t* refs);
MLA_API int mla_pool_free_pages(mla_pool_t* pool, int64_t* n);
MLA_API int mla_pool_take_copies(mla_pool_t* pool, int32_t* src, int32_t* dst, int32_t max, int32_t* n);
MLA_API int mla_copy_pages(const mla_dims_t* dims, const mla_cache_t* cache, int32_t n, const int32_t* src,
                           const int32_t* dst, int32_t* status, mla_stream_t stream);

/* ---------------------------------------------------------------- decode without allocation
 * No counterpart in the paper: an interface for callers that cannot allocate
 * device memory when they run a decode step (for example code handed only its
 * input and output buffers by a framework that owns the allocator, or a path
 * that must not enter the allocator at all). It computes exactly what
 * mla_decode_attn computes, with the same arguments minus the workspace: the
 * scratch is a fixed array of mla_decode_noalloc_scratch_bytes() bytes (48 MiB)
 * inside the library, which every GPU that loads the library holds until the
 * process exits.
 *  - With num_splits = 0 the call uses the default worker count
 *    (mla_decode_default_splits) when its scratch fits the array, else the
 *    largest worker count whose scratch fits (the CUDA-core path defaults to
 *    one worker per SM, which at n_h = 128, d_c = 512 needs about 78 MB).
 *  - A request with an explicit num_splits whose mla_decode_workspace_size
 *    exceeds the array, or one that not even a single worker fits, returns
 *    MLA_ERR_WORKSPACE_TOO_SMALL before anything is enqueued.
 *  - Nothing in the array needs to start at zero: the plan and every partial
 *    are written before they are read, so a call does not depend on what an
 *    earlier call left there.
 *  - All calls share the one array: calls whose work overlaps on the GPU (two
 *    streams, or two host threads) race on it. Serialise them.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it for the lifetime of the device's
 *    primary context (cudaDeviceReset invalidates it); make that first call
 *    before any stream capture.
 *  - It allocates nothing and calls no allocating routine. */
MLA_API size_t mla_decode_noalloc_scratch_bytes(void);
MLA_API int mla_decode_attn_noalloc(const mla_dims_t* dims, const mla_cache_t* cache, int32_t B,
                                    int32_t q_per_seq, const void* q_abs, const int32_t* block_table,
                                    int32_t max_pages_per_seq, const int32_t* seq_lens,
                                    int32_t num_splits, void* o_lat, float* lse, int32_t* status,
                                    mla_stream_t stream);

/* ---------------------------------------------------------------- output up-projection
 * o[t][h] = W_UV[h] . o_lat[t][h]  (page 2, "第二步": o = W_UV (sum_j a_j c_kv(j)))
 *   o_lat [T][n_h][d_c] act dtype;  w_uv [n_h][d_v][d_c] act dtype;  o [T][n_h][d_v] act dtype */
MLA_API int mla_out_proj(const mla_dims_t* dims, int32_t T, const void* o_lat, const void* w_uv,
                 void* o, mla_stream_t stream);

/* ---------------------------------------------------------------- output projection W_O
 * The layer output after the value up-projection: the heads' outputs are
 * joined, in head order, into one n_h * d_v vector and W_O maps it to d_model
 * ("MLA 是什么 | dg's Blog", "完整代码": the per-head outputs are reshaped to
 * n_heads * d_n and self.W_O is applied):
 *   o[t][h] = W_UV[h] . o_lat[t][h]                       (exactly mla_out_proj)
 *   out[t]  = W_O . [o[t][0] ; o[t][1] ; ... ; o[t][n_h - 1]]
 *   o_lat [T][n_h][d_c], w_uv [n_h][d_v][d_c]  act dtype (inputs, as mla_out_proj)
 *   w_o   [d_model][n_h * d_v]                 act dtype
 *   o     [T][n_h][d_v]  act dtype (output: the per-head outputs, W_O's input)
 *   out   [T][d_model]   act dtype (output; fp32 accumulation over n_h * d_v)
 *   workspace  device scratch of at least mla_out_proj_wo_workspace_size bytes
 *              (fp32 partial sums of the split reduction over n_h * d_v)
 *   status may be NULL; a bounded wait that gave up sets MLA_ERR_DEVICE_TIMEOUT.
 * W_O is applied after W_UV, not multiplied into it: W_O . W_UV[h] would be a
 * [d_model x d_c] matrix per head, d_c / d_v times the bytes of W_O. */
MLA_API int mla_out_proj_wo_workspace_size(const mla_dims_t* dims, int32_t T, size_t* bytes);
MLA_API int mla_out_proj_wo(const mla_dims_t* dims, int32_t T, const void* o_lat, const void* w_uv,
                            const void* w_o, void* o, void* out, void* workspace, size_t workspace_bytes,
                            int32_t* status, mla_stream_t stream);

/* ---------------------------------------------------------------- utilities
 * Per-row E4M3 quantisation with the cache-append recipe above, exposed so that
 * the codec can be checked on its own: x [rows][cols] fp32 -> codes [rows][cols]
 * uint8, scales [rows] fp32. cols <= 4096. */
MLA_API int mla_quantize_fp8_rows(const float* x, int32_t rows, int32_t cols, uint8_t* codes,
                          float* scales, mla_stream_t stream);

/* Human-readable name of a status code (static storage). */
MLA_API const char* mla_status_string(int status);

/* Library ABI version: MLA_ABI_VERSION. */
#define MLA_ABI_VERSION 1
MLA_API int mla_abi_version(void);

#ifdef __cplusplus
}
#endif
#endif /* MLA_H_ */
