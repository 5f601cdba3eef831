// merge_pieces.cuh -- log-sum-exp merge of one unit (row, head, quarter of the 512
// dims) of a decode's pieces by a group of kMergeThreads threads.
//
// "vLLM x AgentX: Optimizing for Real-World Agentic Serving", section "Kimi K3":
// partial attention outputs over disjoint pieces of a sequence carry their
// log-sum-exp statistics and are merged with online softmax:
//   lse = ln sum_s exp(lse_s),  out = sum_s exp(lse_s - lse) * out_s.
// The merge kernel that follows a decode kernel (combine.cu) runs one unit per
// block.
#pragma once

#include "mla_common.cuh"
#include "tc_ptx.cuh"

namespace mla {

constexpr int kMergeThreads = 256;
constexpr int kMergeWarps = kMergeThreads / 32;
constexpr int kMergeQuarters = 4;
// Slices staged per round: at most 160 (80 KB: one round for a row split over 152
// CTAs); callers pick about twice the average pieces per row.
constexpr int kMergeStagePieces = 160;
constexpr uint32_t kMergeSliceBytes = 128 * 4;
constexpr uint64_t kMergeWaitNs = 2000000000ull;

// Shared memory of a merge group besides the staging area.
struct MergeShared {
  float w[kMergeStagePieces];
  float4 acc[kMergeWarps][32];
  float red[kMergeWarps];
};

// Merges unit `unit` = (row r, head h, quarter) with r * heads + h = unit / 4.
// The pieces' 128-dim slices (512 B each) are brought into `stage` by bulk copies
// that complete on mbarrier `mb` (initialised with one arrival; `phase` is its
// next phase and persists across calls), up to `stage_pieces` at a time: a
// per-thread load stream keeps far fewer bytes in flight per SM than the copy
// engine. While they land, the threads read the pieces' lse and error flags and
// form the weights exp(lse_s - max); then warp w sums pieces w, w + 8, ... from
// shared memory (lane = 4 dims) and the warps' sums are added. `sync()` and
// `sync_or(p)` are barriers over the group's threads (tid 0 .. kMergeThreads - 1).
// Returns false if a copy did not land within its bound (recorded by the caller).
template <class Sync, class SyncOr>
__device__ inline bool merge_unit(int64_t unit, int heads, const int32_t* __restrict__ row_base,
                                  const int32_t* __restrict__ row_np,
                                  const int32_t* __restrict__ piece_err,
                                  const float* __restrict__ part_lse,
                                  const float* __restrict__ part_out,
                                  __nv_bfloat16* __restrict__ out, float* __restrict__ lse,
                                  int stage_pieces, float4* stage, MergeShared& sm, uint32_t mb,
                                  uint32_t& phase, int tid, Sync sync, SyncOr sync_or) {
  const int quarter = (int)(unit % kMergeQuarters);
  const int64_t rh = unit / kMergeQuarters;
  const int r = (int)(rh / heads);
  const int h = (int)(rh - (int64_t)r * heads);
  const int warp = tid >> 5, lane = tid & 31;
  const int np = __ldcg(row_np + r);
  const int base = __ldcg(row_base + r);
  // The first round's copies go out before anything else is read: their slices
  // do not depend on the weights, so they land while the lse values are read.
  const int n0 = min(stage_pieces, max(np, 0));
  if (tid == 0 && n0 > 0) tc::mbar_arrive_expect_tx(mb, (uint32_t)n0 * kMergeSliceBytes);
  sync();
  if (tid < n0)
    tc::bulk_load(smem_u32(stage + 32 * tid),
                  part_out + ((int64_t)(base + tid) * heads + h) * kDLatent + 128 * quarter,
                  kMergeSliceBytes, mb);
  // the unit's maximum lse and whether any piece met a bad page
  float m = -INFINITY, l_own = -INFINITY;
  int bad = 0;
  for (int s = tid; s < np; s += kMergeThreads) {
    const float l = __ldcg(part_lse + (int64_t)(base + s) * heads + h);
    if (s == tid) l_own = l;
    m = fmaxf(m, l);
    bad |= __ldcg(piece_err + base + s);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) sm.red[warp] = m;
  bad = sync_or(bad != 0);
  m = sm.red[0];
#pragma unroll
  for (int w = 1; w < kMergeWarps; ++w) m = fmaxf(m, sm.red[w]);
  const bool empty = np <= 0 || bad || !(m > -INFINITY);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float wsum = 0.f;   // this thread's share of the weights (threads of lane 0 only)
  bool timed_out = false;
  for (int c0 = 0; c0 < np; c0 += stage_pieces) {
    const int n = min(stage_pieces, np - c0);
    if (c0 > 0) {  // later rounds (more pieces than the stage holds)
      sync();  // the previous round's slices and weights are no longer read
      if (tid == 0) tc::mbar_arrive_expect_tx(mb, (uint32_t)n * kMergeSliceBytes);
      sync();
      if (tid < n) {
        const int64_t piece = (int64_t)(base + c0 + tid) * heads + h;
        tc::bulk_load(smem_u32(stage + 32 * tid), part_out + piece * kDLatent + 128 * quarter,
                      kMergeSliceBytes, mb);
      }
    }
    if (tid < n) {
      const float l = c0 == 0 ? l_own : __ldcg(part_lse + (int64_t)(base + c0 + tid) * heads + h);
      sm.w[tid] = (l > -INFINITY && !empty) ? fast_exp2((l - m) * kLog2e) : 0.f;
    }
    sync();
    // every issued copy is waited for, also for a row whose result is empty
    if (!tc::mbar_wait(mb, phase, kMergeWaitNs)) {
      // never expected: record it and give the copies one more bound to land
      // before their shared memory is read or reused
      timed_out = true;
      tc::mbar_wait(mb, phase, kMergeWaitNs);
    }
    phase ^= 1u;
    if (!empty) {
      for (int s = warp; s < n; s += kMergeWarps) {
        const float w = sm.w[s];
        if (w == 0.f) continue;  // empty piece: its slice is never used
        const float4 v = stage[32 * s + lane];
        acc.x += w * v.x; acc.y += w * v.y; acc.z += w * v.z; acc.w += w * v.w;
        if (lane == 0) wsum += w;
      }
    }
  }
  timed_out = sync_or(timed_out);
  sm.acc[warp][lane] = acc;
  if (lane == 0) sm.red[warp] = wsum;
  sync();
  if (warp == 0) {
    float total = 0.f;
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kMergeWarps; ++w) {
      total += sm.red[w];
      const float4 b = sm.acc[w][lane];
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
  sync();  // sm and the stage are free for the next unit
  return !timed_out;
}

// Slices a merge stages per round: about twice the average pieces per row, at
// least 16 and at most kMergeStagePieces.
inline int merge_stage_pieces(int64_t max_pieces_per_row, int64_t rows) {
  const int64_t per_row = 2 * max_pieces_per_row / (rows > 0 ? rows : 1) + 2;
  return (int)(per_row < 16 ? 16 : (per_row > kMergeStagePieces ? kMergeStagePieces : per_row));
}

}  // namespace mla
