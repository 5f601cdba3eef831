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

// Merge of mla_decode's pieces. One block per (row, head, quarter of the 512 dims).
// The pieces' 128-dim slices (512 B each) are brought into shared memory by bulk
// copies, up to kStagePieces at a time: a per-thread load stream keeps far fewer
// bytes in flight per SM than the copy engine, and at batch 1 every block reads
// about 150 slices. While they land, the threads read the pieces' lse and error
// flags and form the weights exp(lse_s - max); then warp w sums pieces w, w + 8,
// ... from shared memory (lane = 4 dims) and the warps' sums are added.
constexpr int kPieceThreads = 256;
constexpr int kPieceWarps = kPieceThreads / 32;
constexpr int kQuarters = 4;
// Slices staged per round: at most 160 (80 KB: one round for a row split over 152
// CTAs); the launch picks about twice the average pieces per row, so that many
// blocks fit on an SM when rows are many and short.
constexpr int kStagePieces = 160;
constexpr int kSliceBytes = 128 * 4;
constexpr uint64_t kCombineWaitNs = 2000000000ull;

__global__ void __launch_bounds__(kPieceThreads)
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
  __shared__ float s_w[kStagePieces];
  __shared__ float4 s_acc[kPieceWarps][32];
  __shared__ float s_red[kPieceWarps];
  const int64_t blk = blockIdx.x;
  const int quarter = (int)(blk % kQuarters);
  const int64_t rh = blk / kQuarters;
  const int r = (int)(rh / heads);
  const int h = (int)(rh - (int64_t)r * heads);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int np = __ldcg(row_np + r);
  const int base = __ldcg(row_base + r);
  const uint32_t mb = smem_u32(&mbar);
  // The first round's copies go out before anything else is read: their slices
  // do not depend on the weights, so they land while the lse values are read.
  const int n0 = min(stage_pieces, max(np, 0));
  if (tid == 0) {
    tc::mbar_init(mb, 1);
    tc::fence_mbar_init();
    if (n0 > 0) tc::mbar_arrive_expect_tx(mb, (uint32_t)(n0 * kSliceBytes));
  }
  __syncthreads();
  if (tid < n0)
    tc::bulk_load(smem_u32(stage + 32 * tid),
                  part_out + ((int64_t)(base + tid) * heads + h) * kDLatent + 128 * quarter,
                  kSliceBytes, mb);
  // the block's maximum lse and whether any piece met a bad page
  float m = -INFINITY, l_own = -INFINITY;
  int bad = 0;
  for (int s = tid; s < np; s += kPieceThreads) {
    const float l = __ldcg(part_lse + (int64_t)(base + s) * heads + h);
    if (s == tid) l_own = l;
    m = fmaxf(m, l);
    bad |= __ldcg(piece_err + base + s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) s_red[warp] = m;
  bad = __syncthreads_or(bad);
  m = s_red[0];
#pragma unroll
  for (int w = 1; w < kPieceWarps; ++w) m = fmaxf(m, s_red[w]);
  const bool empty = np <= 0 || bad || !(m > -INFINITY);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;   // this thread's share of the weights (threads of lane 0 only)
  bool timed_out = false;
  uint32_t phase = 0;
  for (int c0 = 0; c0 < np; c0 += stage_pieces) {
    const int n = min(stage_pieces, np - c0);
    if (c0 > 0) {  // later rounds (more pieces than the stage holds)
      __syncthreads();  // the previous round's slices and weights are no longer read
      if (tid == 0) tc::mbar_arrive_expect_tx(mb, (uint32_t)(n * kSliceBytes));
      __syncthreads();
      if (tid < n) {
        const int64_t piece = (int64_t)(base + c0 + tid) * heads + h;
        tc::bulk_load(smem_u32(stage + 32 * tid), part_out + piece * kDLatent + 128 * quarter,
                      kSliceBytes, mb);
      }
    }
    if (tid < n) {
      const float l = c0 == 0 ? l_own : __ldcg(part_lse + (int64_t)(base + c0 + tid) * heads + h);
      s_w[tid] = (l > -INFINITY && !empty) ? fast_exp2((l - m) * kLog2e) : 0.f;
    }
    __syncthreads();
    // every issued copy is waited for, also for a row whose result is empty
    if (!tc::mbar_wait(mb, phase, kCombineWaitNs)) {
      // never expected: record it and give the copies one more bound to land
      // before their shared memory is read or the block exits
      timed_out = true;
      tc::mbar_wait(mb, phase, kCombineWaitNs);
    }
    phase ^= 1u;
    if (!empty) {
      for (int s = warp; s < n; s += kPieceWarps) {
        const float w = s_w[s];
        if (w == 0.f) continue;  // empty piece: its slice is never used
        const float4 v = stage[32 * s + lane];
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
        if (lane == 0) wsum += w;
      }
    }
  }
  if (__syncthreads_or(timed_out ? 1 : 0)) {
    if (tid == 0) atomicOr(status, MLA_DEVICE_ERR_TIMEOUT);
  }
  s_acc[warp][lane] = acc;
  if (lane == 0) s_red[warp] = wsum;
  __syncthreads();
  if (warp == 0) {
    float total = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kPieceWarps; ++w) {
      total += s_red[w];
      const float4 b = s_acc[w][lane];
      a.x += b.x; a.y += b.y; a.z += b.z; a.w += b.w;
    }
    const float inv = empty ? 0.f : 1.0f / total;
    __nv_bfloat162 lo = __floats2bfloat162_rn(a.x * inv, a.y * inv);
    __nv_bfloat162 hi = __floats2bfloat162_rn(a.z * inv, a.w * inv);
    uint2 packed;
    packed.x = *reinterpret_cast<uint32_t*>(&lo);
    packed.y = *reinterpret_cast<uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + rh * kDLatent + 128 * quarter + 4 * lane) = packed;
    if (quarter == 0 && lane == 0) lse[rh] = empty ? -INFINITY : m + logf(total);
  }
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
  const unsigned blocks = (unsigned)((int64_t)rows * heads * kQuarters);

  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(combine_pieces_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kStagePieces * kSliceBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(1);
  }
  const int64_t per_row = 2 * (int64_t)max_pieces_per_row / max(rows, 1) + 2;
  const int stage = (int)std::min<int64_t>(kStagePieces, std::max<int64_t>(16, per_row));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(blocks);
  cfg.blockDim = dim3(kPieceThreads);
  cfg.dynamicSmemBytes = (size_t)stage * kSliceBytes;
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
