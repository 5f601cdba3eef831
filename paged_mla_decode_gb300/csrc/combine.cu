// combine.cu -- log-sum-exp merge of partial attention results.
//
// "vLLM x AgentX: Optimizing for Real-World Agentic Serving", section "Kimi
// K3": partial attention outputs over disjoint pieces of a sequence carry
// their log-sum-exp statistics and are merged with online softmax:
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * out_s.
// A piece with lse_s = -inf (empty) contributes nothing; a row whose pieces
// are all empty (or that is flagged bad) gets out = 0 and lse = -inf.
#include <algorithm>
#include <atomic>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "merge_pieces.cuh"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kCombineThreads = 128;  // 4 output dims per thread

// Merges `np` partials of one (row, head). Partial s sits at
// out_base + s*out_stride (512 floats) and lse_base + s*lse_stride.
// Every thread handles output dims [4*tid, 4*tid+4). s_w holds np floats.
__device__ __forceinline__ void merge_row(const float* __restrict__ out_base, int64_t out_stride,
                                          const float* __restrict__ lse_base, int64_t lse_stride,
                                          int np, bool bad, __nv_bfloat16* __restrict__ out_row,
                                          float* __restrict__ lse_out, float* s_w) {
  __shared__ float s_red[kCombineThreads / 32];
  const int tid = threadIdx.x;
  float m = -INFINITY;
  if (!bad)
    for (int s = tid; s < np; s += kCombineThreads) m = fmaxf(m, lse_base[s * lse_stride]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if ((tid & 31) == 0) s_red[tid >> 5] = m;
  __syncthreads();
  m = s_red[0];
#pragma unroll
  for (int w = 1; w < kCombineThreads / 32; ++w) m = fmaxf(m, s_red[w]);
  __syncthreads();
  const bool empty = bad || !(m > -INFINITY);
  float total = 0.f;
  if (!empty) {
    for (int s = tid; s < np; s += kCombineThreads) {
      const float l = lse_base[s * lse_stride];
      const float w = (l > -INFINITY) ? fast_exp2((l - m) * kLog2e) : 0.f;
      s_w[s] = w;
      total += w;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) total += __shfl_xor_sync(0xffffffffu, total, o);
  if ((tid & 31) == 0) s_red[tid >> 5] = total;
  __syncthreads();
  total = 0.f;
#pragma unroll
  for (int w = 0; w < kCombineThreads / 32; ++w) total += s_red[w];
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  if (!empty) {
    const float inv = 1.0f / total;
    for (int s = 0; s < np; ++s) {
      const float w = s_w[s] * inv;
      if (w == 0.f) continue;  // empty piece: its output is never read
      const float4 v = *reinterpret_cast<const float4*>(out_base + s * out_stride + 4 * tid);
      acc.x += w * v.x;
      acc.y += w * v.y;
      acc.z += w * v.z;
      acc.w += w * v.w;
    }
  }
  __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
  __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
  uint2 packed;
  packed.x = *reinterpret_cast<uint32_t*>(&lo);
  packed.y = *reinterpret_cast<uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(out_row + 4 * tid) = packed;
  if (tid == 0) *lse_out = empty ? -INFINITY : m + logf(total);
}

// Merge of mla_decode's pieces: one block of kMergeThreads per unit (row, head,
// quarter of the 512 dims), see merge_unit.
__global__ void __launch_bounds__(kMergeThreads)
combine_pieces_kernel(const int32_t* __restrict__ row_base, const int32_t* __restrict__ row_np,
                      const int32_t* __restrict__ piece_err, const float* __restrict__ part_lse,
                      const float* __restrict__ part_out, int heads,
                      __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                      unsigned* __restrict__ status, int stage_pieces) {
  // launched as a dependent of the decode kernel: its partials are visible after this
  griddep_wait();
  griddep_launch_dependents();
  extern __shared__ float4 stage[];                 // [stage_pieces][32] float4
  __shared__ __align__(8) uint64_t mbar;
  __shared__ MergeShared sm;
  const uint32_t mb = smem_u32(&mbar);
  if (threadIdx.x == 0) {
    tc::mbar_init(mb, 1);
    tc::fence_mbar_init();
  }
  uint32_t phase = 0;
  const bool ok = merge_unit(
      blockIdx.x, heads, row_base, row_np, piece_err, part_lse, part_out, out, lse, stage_pieces,
      stage, sm, mb, phase, (int)threadIdx.x, [] { __syncthreads(); },
      [](bool pred) { return __syncthreads_or(pred ? 1 : 0) != 0; });
  if (!ok && threadIdx.x == 0) atomicOr(status, MLA_DEVICE_ERR_TIMEOUT);
}

// Standalone merge: part_out [S][rows][512], part_lse [S][rows]; one block per row.
__global__ void __launch_bounds__(kCombineThreads)
combine_dense_kernel(const float* __restrict__ part_out, const float* __restrict__ part_lse,
                     int num_parts, int64_t rows, __nv_bfloat16* __restrict__ out,
                     float* __restrict__ lse) {
  extern __shared__ float s_w[];
  const int64_t r = blockIdx.x;
  merge_row(part_out + r * kDLatent, rows * kDLatent, part_lse + r, rows, num_parts, false,
            out + r * kDLatent, lse + r, s_w);
}

}  // namespace

cudaError_t launch_combine_pieces(const DecodeWorkspace& ws, int rows, int heads,
                                  int max_pieces_per_row, __nv_bfloat16* out, float* lse,
                                  cudaStream_t stream) {
  const unsigned blocks = (unsigned)((int64_t)rows * heads * kMergeQuarters);

  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(combine_pieces_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMergeStagePieces * (int)kMergeSliceBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(1);
  }
  const int stage = merge_stage_pieces(max_pieces_per_row, rows);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kMergeThreads);
  cfg.dynamicSmemBytes = (size_t)stage * kMergeSliceBytes;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, combine_pieces_kernel, (const int32_t*)ws.row_base,
                            (const int32_t*)ws.row_np, (const int32_t*)ws.piece_err,
                            (const float*)ws.part_lse, (const float*)ws.part_out, heads, out,
                            lse, ws.status, stage);
}

}  // namespace mla

extern "C" mla_status mla_decode_combine(const float* part_out, const float* part_lse,
                                         int num_parts, int64_t num_rows, void* out, float* lse,
                                         mla_stream_t stream) {
  using namespace mla;
  if (num_parts < 0 || num_rows < 0) return MLA_ERR_INVALID_ARG;
  if (num_rows == 0) return MLA_OK;
  if (!out || !lse) return MLA_ERR_INVALID_ARG;
  if (num_parts > 0 && (!part_out || !part_lse)) return MLA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(part_out) & 15u) || (reinterpret_cast<uintptr_t>(out) & 15u) ||
      (reinterpret_cast<uintptr_t>(part_lse) & 3u) || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return MLA_ERR_INVALID_ARG;
  if (num_rows > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  const size_t smem = sizeof(float) * (size_t)max(num_parts, 1);
  if (smem > 200 * 1024) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (smem > 48 * 1024) {
    if (cudaFuncSetAttribute(combine_dense_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem) != cudaSuccess)
      return MLA_ERR_CUDA;
  }
  combine_dense_kernel<<<(unsigned)num_rows, kCombineThreads, smem, s>>>(
      part_out, part_lse, num_parts, num_rows, static_cast<__nv_bfloat16*>(out), lse);
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
