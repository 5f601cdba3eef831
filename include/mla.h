/*
 * mla.h -- C ABI of the paged FP8 MLA decode library (libmla.so).
 *
 * Decode attention for multi-head latent attention (MLA) over a paged,
 * prefix-shareable latent KV cache, for one GPU (sm_103a).
 *
 * What the operations compute is described on these pages:
 *  - "How to serve trillions of tokens for trillion-parameter coding agents"
 *    (Modal), section "Tensor parallel was the best parallelism strategy for
 *    maximum interactivity": one cache entry per token and layer holds 576
 *    elements; section "First, understand the workload": the model keeps no
 *    distinct keys and values; section "Use custom speculative decoding ...":
 *    drafted tokens are verified in parallel without changing the target
 *    model's distribution.
 *  - "Smaller, faster, safer: running Kimi and GLM at scale" (Cloudflare),
 *    section "Quantizing the KV cache": the cache is FP8 e4m3 and the attention
 *    kernel converts values as it reads them; section "Protecting a shared KV
 *    cache": many requests read pages of one physical paged cache.
 *  - "vLLM x AgentX: Optimizing for Real-World Agentic Serving", section
 *    "Kimi K3": MLA has a single latent head shared by all query heads; partial
 *    attention outputs and their log-sum-exp statistics are merged with online
 *    softmax.
 *
 * Conventions shared by every entry point
 *  - Entry layout: 576 elements per token = 512 latent elements (the value,
 *    and the first 512 key elements) followed by 64 rotary key elements.
 *  - Cache layout: kv_pages[num_pages][page_size][576], row-major; one byte per
 *    element for MLA_KV_E4M3 (OCP E4M3: bias 7, max 448, no infinity), two
 *    (bfloat16) for MLA_KV_BF16. A token's slot is page_id * page_size + offset.
 *    page_size must be 64.
 *  - Pointers named "device" must point to device memory of the current CUDA
 *    device; all must be 16-byte aligned. The caller owns every buffer.
 *    The library allocates nothing and never synchronises the host: all work
 *    is enqueued on `stream` (NULL = the legacy default stream).
 *  - Arguments are checked on the host before anything is enqueued; a failed
 *    check returns MLA_ERR_INVALID_ARG or MLA_ERR_UNSUPPORTED and enqueues
 *    nothing. A failed launch returns MLA_ERR_CUDA.
 *  - Device-side problems (a block-table entry outside [0, num_pages), a
 *    sequence length outside [num_queries, max_pages * page_size]) never trap:
 *    the affected (request, draft) rows get out = 0 and lse = -inf, and a
 *    sticky bit is set in the status word at the start of the workspace
 *    (MLA_DEVICE_ERR_*), which the caller may read back at any time.
 *  - Entry points are re-entrant and keep no global state, with one
 *    exception: mla_decode_static_scratch keeps its scratch in one array per
 *    device, shared by all of its calls (see its declaration).
 *  - Stream order is kept: mla_decode's kernels are launched with programmatic
 *    dependent launch (they may become resident while the previous kernel in
 *    the stream finishes) but each waits for all earlier work in the stream to
 *    complete before its first memory access.
 */
#ifndef PAGED_MLA_DECODE_MLA_H_
#define PAGED_MLA_DECODE_MLA_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MLA_API __attribute__((visibility("default")))
#else
#define MLA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t, declared without the CUDA headers. */
typedef struct CUstream_st* mla_stream_t;

typedef enum mla_status {
  MLA_OK = 0,
  MLA_ERR_INVALID_ARG = 1, /* a null pointer, a bad size, a misaligned buffer */
  MLA_ERR_UNSUPPORTED = 2, /* a shape the library has no kernel for */
  MLA_ERR_WORKSPACE = 3,   /* workspace missing or smaller than required */
  MLA_ERR_CUDA = 4         /* a CUDA runtime call or a launch failed */
} mla_status;

typedef enum mla_kv_dtype {
  MLA_KV_E4M3 = 0, /* FP8 e4m3 codes, one byte per element */
  MLA_KV_BF16 = 1  /* bfloat16, two bytes per element */
} mla_kv_dtype;

#define MLA_D_LATENT 512
#define MLA_D_ROPE 64
#define MLA_D_ENTRY 576
#define MLA_PAGE_SIZE 64
#define MLA_MAX_QUERIES 4

/* Bits of the device status word (first 4 bytes of the decode workspace). */
#define MLA_DEVICE_ERR_BAD_PAGE 0x1u   /* a block-table entry outside the cache */
#define MLA_DEVICE_ERR_BAD_LENGTH 0x2u /* seq_len < num_queries or > max_pages*page_size */
#define MLA_DEVICE_ERR_TIMEOUT 0x4u    /* an internal pipeline wait ran out (2 s); results invalid */

/* Version of this ABI (increments on any incompatible change). */
MLA_API int mla_abi_version(void);

/* Static, human-readable name of a status code; never NULL. */
MLA_API const char* mla_status_string(int status);

/*
 * mla_kv_append -- write new tokens' latent entries into their cache slots.
 *
 * The cache-write side of "Quantizing the KV cache" (Cloudflare page above):
 * for each token t < num_tokens with slot_mapping[t] >= 0,
 *   MLA_KV_E4M3: kv_pages[slot][d] = e4m3( x[t][d] / kv_scale ), rounded to
 *                nearest with ties to even, of the exact quotient, and
 *                saturated to +-448 (NaN stays NaN), where x[t][0:512] =
 *                latent[t], x[t][512:576] = rope[t];
 *   MLA_KV_BF16: kv_pages[slot][d] = x[t][d] (a copy; kv_scale must be 1).
 * Slots with slot_mapping[t] < 0 are skipped (padding tokens).
 *
 * latent       device, bf16 [num_tokens][512], row-major
 * rope         device, bf16 [num_tokens][64], row-major
 * slot_mapping device, int32 [num_tokens]; each must be -1 or lie in
 *              [0, num_pages * page_size) (entries beyond it are skipped and
 *              nothing else is reported; validate on the host if needed)
 * kv_pages     device, the cache (see layout above); written in place
 * kv_scale     per-tensor scale, finite and > 0
 * Two tokens naming the same slot race; writing into a page that other
 * requests share is the caller's error.
 */
MLA_API mla_status mla_kv_append(const void* latent, const void* rope, const int32_t* slot_mapping,
                         int64_t num_tokens, void* kv_pages, int64_t num_pages, int page_size,
                         int kv_dtype, float kv_scale, mla_stream_t stream);

/*
 * mla_decode_workspace_size -- bytes of workspace mla_decode needs.
 *
 * num_ctas is the number of worker CTAs the caller will pass to mla_decode
 * (0 = the default, one per SM of the current device). Returns 0 for an
 * invalid shape.
 */
MLA_API size_t mla_decode_workspace_size(int batch, int num_queries, int num_heads, int num_ctas);

/*
 * mla_decode -- attention of the new query tokens over each request's pages.
 *
 * For request b < batch, draft j < num_queries and head h < num_heads, with
 * L = seq_lens[b] counting the cached tokens including the num_queries drafts
 * just appended, draft j sees positions t < n_j = L - num_queries + j + 1:
 *   K[t]  = value(kv_pages[block_table[b][t / page_size]][t % page_size]) * kv_scale
 *   s_t   = sm_scale * sum_{d<576} q[b][j][h][d] * K[t][d]
 *   lse   = ln sum_t exp(s_t)
 *   out   = sum_t exp(s_t - lse) * K[t][0:512]
 * (natural logarithm; s includes sm_scale). The work is split into pieces of
 * equal token count over num_ctas CTAs (split-KV); each piece yields a partial
 * (out, lse) that a second kernel merges by log-sum-exp ("vLLM x AgentX",
 * section "Kimi K3"), so one call fills all SMs even at batch 1.
 *
 * Arithmetic: for an e4m3 cache the cache bytes themselves are the tensor-core
 * operands (tcgen05 kind::f8f6f4); q is scaled per head by a power of two and
 * split into two e4m3 terms (exact for bf16 q down to 2^-10 of the head's
 * largest element); accumulation is fp32. The softmax weights P = 2^(s - m + 6)
 * (s in log2 units, m a running maximum) are split into an e4m3 and an e5m2
 * term: relative error at most 2^-7 for P >= 2^-6, coarser below, and P below
 * about 2^-17 drops out of `out` (the normaliser sums the exact P). m follows
 * each 64-token page's maximum within [-6, +2.8] (a page further below lowers
 * m, unless the weight accumulated so far exceeds 2^28 times the page's
 * largest), so every page's largest P lies in [1, 448]; what a page loses is
 * confined to its tokens below 2^-6 of its largest weight. Each piece of the
 * split (one per CTA) has its own maximum; pieces merge in fp32. For a bf16
 * cache both contractions use bf16 operands (kind::f16).
 *
 * q           device, bf16 [batch][num_queries][num_heads][576]
 * kv_pages    device, the cache; num_pages pages of page_size (= 64) tokens
 * block_table device, int32 [batch][max_pages]; entries past a request's last
 *             page are never read
 * seq_lens    device, int32 [batch]
 * num_heads   16, 32 or 64 (UNSUPPORTED otherwise)
 * num_queries 1..4
 * sm_scale, kv_scale  finite; kv_scale > 0 (use 1 for MLA_KV_BF16 caches)
 * num_ctas    worker CTAs (0 = one per SM); must match the value the
 *             workspace was sized for
 * workspace   device, at least mla_decode_workspace_size(batch, num_queries,
 *             num_heads, num_ctas) bytes, zero-filled before its first use;
 *             every call leaves it ready for the next (status word aside).
 *             Calls that share a workspace must be stream-ordered.
 * out         device, bf16 [batch][num_queries][num_heads][512]
 * lse         device, fp32 [batch][num_queries][num_heads]
 */
MLA_API mla_status mla_decode(const void* q, const void* kv_pages, int64_t num_pages, int page_size,
                      int kv_dtype, const int32_t* block_table, int max_pages,
                      const int32_t* seq_lens, int batch, int num_queries, int num_heads,
                      float sm_scale, float kv_scale, int num_ctas, void* workspace,
                      size_t workspace_bytes, void* out, float* lse, mla_stream_t stream);

/*
 * mla_decode_grouped -- mla_decode for groups of requests that share a prefix.
 *
 * Subagent sessions fork from a parent context ("vLLM x AgentX: Optimizing for
 * Real-World Agentic Serving", section "Characterizing agentic workloads: a
 * second look") and then read the pages of one physical paged cache ("Smaller,
 * faster, safer: running Kimi and GLM at scale", section "Protecting a shared KV
 * cache"). Requests [g * forks, (g + 1) * forks) form group g, and their first
 * prefix_pages[g] logical pages are the same physical pages; the kernel reads
 * those page ids from the group's first request. The results are mla_decode's
 * on the same arguments (same arithmetic and tolerance); what changes is how
 * the work is cut: each shared page is worked by `forks` CTAs at once, one per
 * fork, so the group reads it from HBM once (the other forks' reads hit L2),
 * while the tokens after the prefix are split as in mla_decode.
 *
 * forks         requests per group; 1 <= forks <= CTAs and batch % forks == 0
 * prefix_pages  device, int32 [batch / forks]. A request whose group prefix is
 *               outside [0, max_pages] pages or longer than L - num_queries + 1
 *               tokens (draft 0 must see the whole prefix) is treated like a
 *               bad length: out = 0, lse = -inf, MLA_DEVICE_ERR_BAD_LENGTH.
 * workspace     at least mla_decode_grouped_workspace_size(batch, num_queries,
 *               num_heads, num_ctas) bytes, zero-filled before its first use.
 * kv_dtype      MLA_KV_E4M3 (MLA_ERR_UNSUPPORTED otherwise).
 * Other arguments as mla_decode.
 */
MLA_API size_t mla_decode_grouped_workspace_size(int batch, int num_queries, int num_heads,
                                                 int num_ctas);
MLA_API mla_status mla_decode_grouped(const void* q, const void* kv_pages, int64_t num_pages,
                                      int page_size, int kv_dtype, const int32_t* block_table,
                                      int max_pages, const int32_t* seq_lens, int batch,
                                      int num_queries, int num_heads, int forks,
                                      const int32_t* prefix_pages, float sm_scale,
                                      float kv_scale, int num_ctas, void* workspace,
                                      size_t workspace_bytes, void* out, float* lse,
                                      mla_stream_t stream);

/*
 * mla_decode_f16_operands -- mla_decode with 16-bit tensor-core operands.
 *
 * Same arguments, contract and results (within the same tolerance) as
 * mla_decode. For an e4m3 cache the pages are widened to f16 in shared memory
 * as they are read (the FP8 cache of "Smaller, faster, safer: running Kimi and
 * GLM at scale", section "Quantizing the KV cache", converted on load) and both
 * contractions use kind::f16 with q and the softmax weights in f16; for a bf16
 * cache it is mla_decode. It exists to measure what reading the FP8 bytes as
 * operands saves; it has no counterpart on the pages.
 */
MLA_API mla_status mla_decode_f16_operands(const void* q, const void* kv_pages, int64_t num_pages,
                                   int page_size, int kv_dtype, const int32_t* block_table,
                                   int max_pages, const int32_t* seq_lens, int batch,
                                   int num_queries, int num_heads, float sm_scale,
                                   float kv_scale, int num_ctas, void* workspace,
                                   size_t workspace_bytes, void* out, float* lse,
                                   mla_stream_t stream);

/*
 * mla_decode_combine -- merge partial attention results by log-sum-exp.
 *
 * The merge of "vLLM x AgentX", section "Kimi K3" (partial outputs and LSE
 * statistics combined with online softmax), for partials produced elsewhere
 * (for example one per sequence shard). For each row r < num_rows:
 *   lse[r] = ln sum_s exp(part_lse[s][r])
 *   out[r] = sum_s exp(part_lse[s][r] - lse[r]) * part_out[s][r][0:512]
 * A part with part_lse = -inf contributes nothing; if all are -inf the row
 * gets out = 0 and lse = -inf.
 *
 * part_out  device, fp32 [num_parts][num_rows][512] (normalised partials)
 * part_lse  device, fp32 [num_parts][num_rows]
 * out       device, bf16 [num_rows][512]
 * lse       device, fp32 [num_rows]
 */
MLA_API mla_status mla_decode_combine(const float* part_out, const float* part_lse, int num_parts,
                              int64_t num_rows, void* out, float* lse, mla_stream_t stream);

/*
 * mla_kv_check -- integrity check of requests' page mappings before decode.
 *
 * The check of "Smaller, faster, safer: running Kimi and GLM at scale",
 * section "Protecting a shared KV cache": every physical page carries a tag
 * that the page allocator changes whenever it hands the page out again; each
 * request keeps, beside its block-table entries, the tags its pages had when it
 * was given them; before decode reads the cache the two are compared, and a
 * request with any mismatch is aborted instead of reading another request's
 * data. It is a separate batch pass, not part of the attention kernel.
 *
 * For request b < batch with L = seq_lens[b], over its used logical pages
 * j < ceil(L / page_size), with p = block_table[b][j]:
 *   MLA_KV_CHECK_PAGE_RANGE   if p < 0 or p >= num_pages;
 *   MLA_KV_CHECK_TAG_MISMATCH if page_tags[p] != expected_tags[b][j];
 *   MLA_KV_CHECK_BAD_LENGTH   (and no page looked at) if L < 0 or
 *                             L > max_pages * page_size.
 * request_status[b] = OR of the bits (0 = the request passed);
 * checked_seq_lens[b] = L if it passed, else -1. Passing checked_seq_lens to
 * mla_decode as seq_lens aborts the failed requests there: each of their rows
 * gets out = 0 and lse = -inf (and MLA_DEVICE_ERR_BAD_LENGTH in the workspace
 * status word) and none of their pages is read.
 *
 * page_tags        device, uint32 [num_pages] (may be NULL if num_pages == 0)
 * block_table      device, int32 [batch][max_pages]; entries past a request's
 *                  used pages are not read
 * expected_tags    device, uint32 [batch][max_pages], beside block_table
 * seq_lens         device, int32 [batch]
 * page_size        must be 64
 * request_status   device, uint32 [batch] (written)
 * checked_seq_lens device, int32 [batch] (written; may be the same buffer as
 *                  seq_lens only if no other work reads seq_lens concurrently)
 * Pointers need 4-byte alignment here. Tags are opaque 32-bit values.
 */
#define MLA_KV_CHECK_TAG_MISMATCH 0x1u
#define MLA_KV_CHECK_PAGE_RANGE 0x2u
#define MLA_KV_CHECK_BAD_LENGTH 0x4u
MLA_API mla_status mla_kv_check(const uint32_t* page_tags, int64_t num_pages,
                                const int32_t* block_table, const uint32_t* expected_tags,
                                int max_pages, const int32_t* seq_lens, int batch, int page_size,
                                uint32_t* request_status, int32_t* checked_seq_lens,
                                mla_stream_t stream);

/*
 * mla_decode_static_scratch -- mla_decode for callers that cannot allocate.
 *
 * No counterpart on the pages: this entry point exists for callers that may not
 * allocate device memory when they decode -- plug-ins inside an engine that has
 * reserved all device memory in its own pool and gives them no allocator, or
 * serving loops that forbid cudaMalloc (which can synchronise the device) after
 * start-up. It computes exactly what mla_decode computes, with the same kernels
 * and arguments, but takes no workspace: the split-KV scratch lives in one
 * array of MLA_STATIC_SCRATCH_BYTES inside this library's device image, held by
 * every GPU that loads the library until the process exits. It calls no
 * cudaMalloc, cudaFree or other allocating routine.
 *
 *  - Limit: returns MLA_ERR_WORKSPACE, enqueuing nothing, when the problem needs
 *    more scratch than MLA_STATIC_SCRATCH_BYTES, i.e. when
 *    mla_decode_workspace_size(batch, num_queries, num_heads, num_ctas) exceeds
 *    it: at 64 heads with one CTA per SM on a 152-SM GPU, batch x num_queries
 *    may be at most 229 rows.
 *  - Set-up: the first call on each device looks up the array's device address
 *    with that device current (cudaGetSymbolAddress). Make that first call
 *    before any stream capture. The address is kept per device ordinal and
 *    belongs to the runtime's primary context of that device: the entry point
 *    assumes that context for the whole process (no context of the caller's
 *    own, no cudaDeviceReset between calls).
 *  - Sharing: every call on a device uses the same array, which keeps the last
 *    call's contents. Calls that overlap on the GPU (for instance on two
 *    streams) race and give wrong results: order them on one stream or with
 *    events.
 *  - device_status: optional device pointer (may be NULL) that receives this
 *    call's MLA_DEVICE_ERR_* bits; the copy in the array is cleared afterwards,
 *    also when the call returns MLA_ERR_CUDA after some of its work was
 *    enqueued (the first error is returned).
 */
#define MLA_STATIC_SCRATCH_BYTES ((size_t)64 << 20)
MLA_API mla_status mla_decode_static_scratch(const void* q, const void* kv_pages, int64_t num_pages,
                                             int page_size, int kv_dtype,
                                             const int32_t* block_table, int max_pages,
                                             const int32_t* seq_lens, int batch, int num_queries,
                                             int num_heads, float sm_scale, float kv_scale,
                                             int num_ctas, void* out, float* lse,
                                             unsigned* device_status, mla_stream_t stream);

#ifdef __cplusplus
} /* extern "C" */
#endif

#endif /* PAGED_MLA_DECODE_MLA_H_ */
