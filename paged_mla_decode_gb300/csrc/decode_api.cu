// decode_api.cu -- host entry points of the split-KV decode: argument checks,
// workspace carving and the two launches (decode kernel, then piece combine).
#include <atomic>

#include "mla_common.cuh"
#include "mla_internal.h"

namespace mla {

int device_sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev].load() > 0) return cache[dev].load();
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev].store(n);
  return n;
}

}  // namespace mla

namespace {
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
}  // namespace

namespace {
size_t workspace_bytes_for(int batch, int num_queries, int num_heads, int num_ctas, int passes) {
  if (batch < 0 || num_queries < 1 || num_queries > MLA_MAX_QUERIES || num_heads <= 0 ||
      num_ctas < 0)
    return 0;
  if (num_ctas == 0) num_ctas = mla::device_sm_count();
  if (num_ctas <= 0) return 0;
  return mla::workspace_layout((int64_t)batch * num_queries, num_heads, num_ctas, passes).total;
}
}  // namespace

extern "C" size_t mla_decode_workspace_size(int batch, int num_queries, int num_heads,
                                            int num_ctas) {
  return workspace_bytes_for(batch, num_queries, num_heads, num_ctas, 1);
}

extern "C" size_t mla_decode_grouped_workspace_size(int batch, int num_queries, int num_heads,
                                                    int num_ctas) {
  return workspace_bytes_for(batch, num_queries, num_heads, num_ctas, 2);
}

namespace {
mla_status decode_impl(const void* q, const void* kv_pages, int64_t num_pages, int page_size,
                       int kv_dtype, const int32_t* block_table, int max_pages,
                       const int32_t* seq_lens, int batch, int num_queries, int num_heads,
                       float sm_scale, float kv_scale, int num_ctas, void* workspace,
                       size_t workspace_bytes, void* out, float* lse, mla_stream_t stream,
                       bool f16_operands, int forks = 1, const int32_t* prefix_pages = nullptr) {
  using namespace mla;
  if (batch < 0 || num_pages < 0 || max_pages < 1 || num_ctas < 0) return MLA_ERR_INVALID_ARG;
  if (num_queries < 1 || num_queries > MLA_MAX_QUERIES) return MLA_ERR_INVALID_ARG;
  if (page_size != kPageSize) return MLA_ERR_UNSUPPORTED;
  if (kv_dtype != MLA_KV_E4M3 && kv_dtype != MLA_KV_BF16) return MLA_ERR_INVALID_ARG;
  if (num_heads != 16 && num_heads != 32 && num_heads != 64) return MLA_ERR_UNSUPPORTED;
  if (!isfinite(sm_scale) || !isfinite(kv_scale) || !(kv_scale > 0.f)) return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  if (!q || !kv_pages || !block_table || !seq_lens || !out || !lse) return MLA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(kv_pages, 16) || !aligned(out, 16) || !aligned(lse, 4) ||
      !aligned(block_table, 4) || !aligned(seq_lens, 4))
    return MLA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256)) return MLA_ERR_WORKSPACE;
  if ((int64_t)batch * max_pages > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const int G = num_ctas ? num_ctas : device_sm_count();
  if (G <= 0) return MLA_ERR_CUDA;
  const int64_t rows = (int64_t)batch * num_queries;
  if (rows * num_heads > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const bool grouped = prefix_pages != nullptr;
  if (grouped && (forks < 1 || forks > G || batch % forks != 0)) return MLA_ERR_INVALID_ARG;
  if (grouped && !aligned(prefix_pages, 4)) return MLA_ERR_INVALID_ARG;
  const WorkspaceLayout L = workspace_layout(rows, num_heads, G, grouped ? 2 : 1);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeLaunch p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const uint8_t*>(kv_pages);
  p.num_pages = num_pages;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.nq = num_queries;
  p.heads = num_heads;
  p.bf16 = kv_dtype == MLA_KV_BF16;
  p.score_mul = sm_scale * kLog2e * kv_scale;
  p.kv_scale = kv_scale;
  p.G = G;
  p.ws.status = reinterpret_cast<unsigned*>(ws);
  p.ws.row_base = reinterpret_cast<int32_t*>(ws + L.row_base);
  p.ws.row_np = reinterpret_cast<int32_t*>(ws + L.row_np);
  p.ws.row_np1 = reinterpret_cast<int32_t*>(ws + L.row_np1);
  p.ws.piece_err = reinterpret_cast<int32_t*>(ws + L.piece_err);
  p.ws.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.ws.part_out = reinterpret_cast<float*>(ws + L.part_out);
  p.ws.q_op = ws + L.q_op;
  p.ws.q_mul = reinterpret_cast<float*>(ws + L.q_mul);

  if (!p.bf16 && num_pages > (int64_t)(0x7fffffff / kPageSize)) return MLA_ERR_UNSUPPORTED;
  if (grouped) {
    if (p.bf16 || f16_operands) return MLA_ERR_UNSUPPORTED;  // FP8 cache, FP8 operands only
    p.forks = forks;
    p.prefix_pages = prefix_pages;
  }

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e = (p.bf16 || f16_operands) ? launch_decode_tensor_core(p, s)
                                            : launch_decode_fp8(p, s);
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  e = launch_combine_pieces(p.ws, (int)rows, num_heads, G, static_cast<__nv_bfloat16*>(out), lse,
                            s);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
}  // namespace

extern "C" mla_status mla_decode(const void* q, const void* kv_pages, int64_t num_pages,
                                 int page_size, int kv_dtype, const int32_t* block_table,
                                 int max_pages, const int32_t* seq_lens, int batch,
                                 int num_queries, int num_heads, float sm_scale, float kv_scale,
                                 int num_ctas, void* workspace, size_t workspace_bytes, void* out,
                                 float* lse, mla_stream_t stream) {
  return decode_impl(q, kv_pages, num_pages, page_size, kv_dtype, block_table, max_pages,
                     seq_lens, batch, num_queries, num_heads, sm_scale, kv_scale, num_ctas,
                     workspace, workspace_bytes, out, lse, stream, false);
}

extern "C" mla_status mla_decode_f16_operands(const void* q, const void* kv_pages,
                                              int64_t num_pages, int page_size, int kv_dtype,
                                              const int32_t* block_table, int max_pages,
                                              const int32_t* seq_lens, int batch,
                                              int num_queries, int num_heads, float sm_scale,
                                              float kv_scale, int num_ctas, void* workspace,
                                              size_t workspace_bytes, void* out, float* lse,
                                              mla_stream_t stream) {
  return decode_impl(q, kv_pages, num_pages, page_size, kv_dtype, block_table, max_pages,
                     seq_lens, batch, num_queries, num_heads, sm_scale, kv_scale, num_ctas,
                     workspace, workspace_bytes, out, lse, stream, true);
}

extern "C" mla_status mla_decode_grouped(const void* q, const void* kv_pages, int64_t num_pages,
                                         int page_size, int kv_dtype, const int32_t* block_table,
                                         int max_pages, const int32_t* seq_lens, int batch,
                                         int num_queries, int num_heads, int forks,
                                         const int32_t* prefix_pages, float sm_scale,
                                         float kv_scale, int num_ctas, void* workspace,
                                         size_t workspace_bytes, void* out, float* lse,
                                         mla_stream_t stream) {
  if (batch > 0 && prefix_pages == nullptr) return MLA_ERR_INVALID_ARG;
  return decode_impl(q, kv_pages, num_pages, page_size, kv_dtype, block_table, max_pages,
                     seq_lens, batch, num_queries, num_heads, sm_scale, kv_scale, num_ctas,
                     workspace, workspace_bytes, out, lse, stream, false, forks, prefix_pages);
}
