// kv_check.cu -- KV-cache integrity check before decode reads the cache.
//
// "Smaller, faster, safer: running Kimi and GLM at scale", section "Protecting a
// shared KV cache": every physical page carries a tag that changes whenever the
// page is reallocated; the server records which (page, tag) pairs each request
// expects, and before decode reads the cache those pairs are compared; a request
// with a mismatch is aborted rather than allowed to return data computed from a
// page that is no longer its own. The check is its own batch pass (not fused
// into the attention kernel), which is what this kernel is.
//
// One CTA per request. A request of L tokens uses logical pages
// 0 .. ceil(L / 64) - 1; the threads read those block-table entries and expected
// tags with coalesced loads (kPagesPerThread per thread in flight), then gather
// the current tags of the named pages. The result is a status word per request
// (MLA_KV_CHECK_* bits) and a copy of the lengths with -1 for every failed
// request: passed to mla_decode as seq_lens, a -1 gives that request out = 0 and
// lse = -inf without any of its pages being read.
#include "mla_common.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kCheckThreads = 512;
constexpr int kPagesPerThread = 8;

__global__ void __launch_bounds__(kCheckThreads)
kv_check_kernel(const uint32_t* __restrict__ page_tags, int64_t num_pages,
                const int32_t* __restrict__ block_table,
                const uint32_t* __restrict__ expected_tags, int max_pages,
                const int32_t* __restrict__ seq_lens, uint32_t* __restrict__ status_out,
                int32_t* __restrict__ checked_out) {
  __shared__ uint32_t s_status;
  const int64_t b = blockIdx.x;
  const int tid = threadIdx.x;
  if (tid == 0) s_status = 0;
  __syncthreads();
  const int L = seq_lens[b];
  uint32_t st = 0;
  if (L < 0 || (int64_t)L > (int64_t)max_pages * kPageSize) {
    st = MLA_KV_CHECK_BAD_LENGTH;
  } else {
    const int used = (L + kPageSize - 1) / kPageSize;
    const int32_t* row = block_table + b * max_pages;
    const uint32_t* want_row = expected_tags + b * max_pages;
    for (int j0 = 0; j0 < used; j0 += kCheckThreads * kPagesPerThread) {
      int32_t page[kPagesPerThread];
      uint32_t want[kPagesPerThread];
#pragma unroll
      for (int u = 0; u < kPagesPerThread; ++u) {
        const int j = j0 + u * kCheckThreads + tid;
        page[u] = 0;
        want[u] = 0;
        if (j < used) {
          page[u] = __ldg(row + j);
          want[u] = __ldg(want_row + j);
        }
      }
      uint32_t have[kPagesPerThread];
#pragma unroll
      for (int u = 0; u < kPagesPerThread; ++u) {
        const int j = j0 + u * kCheckThreads + tid;
        const bool in_range = page[u] >= 0 && (int64_t)page[u] < num_pages;
        have[u] = want[u];
        if (j < used && in_range) have[u] = __ldg(page_tags + page[u]);
        if (j < used && !in_range) st |= MLA_KV_CHECK_PAGE_RANGE;
      }
#pragma unroll
      for (int u = 0; u < kPagesPerThread; ++u)
        if (have[u] != want[u]) st |= MLA_KV_CHECK_TAG_MISMATCH;
    }
  }
  if (st) atomicOr(&s_status, st);
  __syncthreads();
  if (tid == 0) {
    status_out[b] = s_status;
    checked_out[b] = s_status ? -1 : L;
  }
}

}  // namespace
}  // namespace mla

extern "C" mla_status mla_kv_check(const uint32_t* page_tags, int64_t num_pages,
                                   const int32_t* block_table, const uint32_t* expected_tags,
                                   int max_pages, const int32_t* seq_lens, int batch,
                                   int page_size, uint32_t* request_status,
                                   int32_t* checked_seq_lens, mla_stream_t stream) {
  using namespace mla;
  if (batch < 0 || num_pages < 0 || max_pages < 0) return MLA_ERR_INVALID_ARG;
  if (page_size != kPageSize) return MLA_ERR_UNSUPPORTED;
  if (batch == 0) return MLA_OK;
  if (!seq_lens || !request_status || !checked_seq_lens) return MLA_ERR_INVALID_ARG;
  if (max_pages > 0 && (!block_table || !expected_tags)) return MLA_ERR_INVALID_ARG;
  if (num_pages > 0 && !page_tags) return MLA_ERR_INVALID_ARG;
  const void* ptrs[6] = {page_tags, block_table, expected_tags, seq_lens, request_status,
                         checked_seq_lens};
  for (const void* p : ptrs)
    if (reinterpret_cast<uintptr_t>(p) & 3u) return MLA_ERR_INVALID_ARG;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  kv_check_kernel<<<(unsigned)batch, kCheckThreads, 0, s>>>(
      page_tags, num_pages, block_table, expected_tags, max_pages, seq_lens, request_status,
      checked_seq_lens);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
