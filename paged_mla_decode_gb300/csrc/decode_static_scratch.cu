// decode_static_scratch.cu -- mla_decode without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode:
// plug-ins hosted by an engine that reserves all device memory up front in its
// own pool and hands them no allocator, and latency-critical loops that may not
// call cudaMalloc (it can synchronise the device) once serving has started.
// For them this entry point runs the same decode kernels as mla_decode, with
// the split-KV scratch (row table, partial outputs and their log-sum-exp) in a
// fixed array of MLA_STATIC_SCRATCH_BYTES that lives in this library's device
// image. Every GPU that loads it holds the array until the process exits.
#include <atomic>

#include "mla_internal.h"

namespace {

constexpr size_t kScratchBytes = MLA_STATIC_SCRATCH_BYTES;
constexpr int kMaxDevices = 64;

// The scratch itself. In host code this name is only a stand-in for the symbol,
// not a device address: the address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_static_scratch[kScratchBytes];

// Device address of g_static_scratch, looked up once per device.
std::atomic<void*> g_scratch_addr[kMaxDevices];

mla_status scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MLA_ERR_CUDA;
  void* p = g_scratch_addr[dev].load();
  if (p == nullptr) {
    // with `dev` current: resolve the array's device address on this device
    if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
      return MLA_ERR_CUDA;
    g_scratch_addr[dev].store(p);
  }
  *out = p;
  return MLA_OK;
}

}  // namespace

extern "C" mla_status mla_decode_static_scratch(
    const void* q, const void* kv_pages, int64_t num_pages, int page_size, int kv_dtype,
    const int32_t* block_table, int max_pages, const int32_t* seq_lens, int batch,
    int num_queries, int num_heads, float sm_scale, float kv_scale, int num_ctas, void* out,
    float* lse, unsigned* device_status, mla_stream_t stream) {
  if (batch < 0 || num_queries < 1 || num_queries > MLA_MAX_QUERIES || num_heads <= 0 ||
      num_ctas < 0)
    return MLA_ERR_INVALID_ARG;
  if (batch == 0) return MLA_OK;
  // scratch this problem needs (same layout as mla_decode's workspace)
  const size_t need = mla_decode_workspace_size(batch, num_queries, num_heads, num_ctas);
  if (need == 0) return MLA_ERR_CUDA;
  if (need > kScratchBytes) return MLA_ERR_WORKSPACE;
  void* scratch = nullptr;
  mla_status st = scratch_address(&scratch);
  if (st != MLA_OK) return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  // The row table and partials are rewritten by every call; only the status word
  // must start at zero. It is zero when the array is loaded and is cleared after
  // each call (once copied out). A call that fails its host checks enqueues
  // nothing; MLA_ERR_CUDA may come after a kernel was enqueued, so the copy and
  // the clear are enqueued for it too and the first error is returned.
  st = mla_decode(q, kv_pages, num_pages, page_size, kv_dtype, block_table, max_pages, seq_lens,
                  batch, num_queries, num_heads, sm_scale, kv_scale, num_ctas, scratch,
                  kScratchBytes, out, lse, stream);
  if (st != MLA_OK && st != MLA_ERR_CUDA) return st;
  if (device_status != nullptr &&
      cudaMemcpyAsync(device_status, scratch, sizeof(unsigned), cudaMemcpyDeviceToDevice, s) !=
          cudaSuccess &&
      st == MLA_OK)
    st = MLA_ERR_CUDA;
  if (cudaMemsetAsync(scratch, 0, sizeof(unsigned), s) != cudaSuccess && st == MLA_OK)
    st = MLA_ERR_CUDA;
  return st;
}
