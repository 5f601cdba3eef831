// mla_common.cuh -- shared device helpers of the paged MLA decode library.
//
// Holds the split-KV work planner (computed on the device from seq_lens, so a
// captured CUDA graph stays valid while lengths change), the workspace layout,
// and small PTX wrappers. Kernels live in the .cu files next to this header.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "../../include/mla.h"

namespace mla {

constexpr int kDLatent = MLA_D_LATENT;  // 512: value dims (and first key dims)
constexpr int kDRope = MLA_D_ROPE;      // 64: rotary key dims
constexpr int kDEntry = MLA_D_ENTRY;    // 576 elements per cached token
constexpr int kPageSize = MLA_PAGE_SIZE;
constexpr int kMaxQueries = MLA_MAX_QUERIES;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// ---------------------------------------------------------------------------
// Workspace layout (device memory owned by the caller).
//
//   [0, 256)                 header: uint32 status word (sticky MLA_DEVICE_ERR_*)
//   row_base  int32[R]       first partial slot of each (request, draft) row
//   row_np    int32[R]       number of partial slots of the row; -1 = bad length
//   row_np1   int32[R]       grouped decode: slots of the row's shared-prefix pieces
//   piece_err int32[P]       1 if the piece met a bad page id
//   part_lse  float[P][H]    log-sum-exp of each piece (natural log)
//   part_out  float[P][H][512] normalised partial output of each piece
//   q_op      uint8[R][36][128][16] the query of each row as the e4m3 operand of
//                                   the FP8 decode kernel (see decode_fp8.cu)
//   q_mul     float[R][64]        score multiplier of each (row, head)
//
// with R = batch * num_queries rows and P = num_ctas + R an upper bound on the
// number of pieces (each CTA range adds at most one piece per row boundary).
// ---------------------------------------------------------------------------
constexpr int kQOpChunks = kDEntry / 16;               // 36 chunks of 16 dims
constexpr int kQOpRowBytes = kQOpChunks * 128 * 16;    // 73,728 B per row
struct WorkspaceLayout {
  size_t row_base, row_np, row_np1, piece_err, part_lse, part_out, q_op, q_mul, total;
  int64_t max_pieces;
};

__host__ __device__ inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// `passes` is 1 for mla_decode and 2 for the grouped decode, whose prefix and
// suffix passes each add up to num_ctas + rows pieces.
__host__ __device__ inline WorkspaceLayout workspace_layout(int64_t rows, int heads, int num_ctas,
                                                            int passes = 1) {
  WorkspaceLayout w;
  w.max_pieces = (int64_t)passes * (num_ctas + rows);
  size_t off = 256;
  w.row_base = off; off = align_up(off + 4 * rows, 256);
  w.row_np = off; off = align_up(off + 4 * rows, 256);
  w.row_np1 = off; off = align_up(off + 4 * rows, 256);
  w.piece_err = off; off = align_up(off + 4 * w.max_pieces, 256);
  w.part_lse = off; off = align_up(off + 4 * w.max_pieces * heads, 256);
  w.part_out = off; off = align_up(off + 4 * w.max_pieces * heads * (int64_t)kDLatent, 256);
  w.q_op = off; off = align_up(off + (size_t)kQOpRowBytes * rows, 256);
  w.q_mul = off; off = align_up(off + 4 * 64 * rows, 256);
  w.total = off;
  return w;
}

// ---------------------------------------------------------------------------
// Split-KV planner.
//
// Rows r = b * Q + j. Row r holds n_r = L_b - Q + j + 1 visible tokens, cut
// into T_r = ceil(n_r / TILE) tiles. All rows' tiles are laid end to end
// (T tiles in total) and CTA c takes tiles [floor(c*T/G), floor((c+1)*T/G)),
// so every CTA gets the same number of tiles whatever the length mix. A
// "piece" is the part of one row inside one CTA's range; it produces one
// partial (out, lse). Pieces of a row occupy consecutive workspace slots,
// ordered by CTA. Only G = min(launched CTAs, T) CTAs take work, so every
// working CTA's range holds at least one tile and the CTAs between a row's
// first and last piece each hold one piece of it.
// ---------------------------------------------------------------------------
struct Plan {
  static constexpr bool kGrouped = false;
  const int32_t* seq_lens;
  int batch, nq, max_pages, tile;
  int G;          // working CTAs: min(launched CTAs, T)
  int64_t T;      // total tiles

  // Sets the total tile count and clamps the number of working CTAs to it.
  __device__ void set_total(int64_t total) {
    T = total;
    if (T < G) G = (int)T;
  }

  __device__ int rows() const { return batch * nq; }
  // visible tokens of row r, or -1 when its length is invalid
  __device__ int row_tokens(int r) const {
    int b = r / nq, j = r - (r / nq) * nq;
    int L = __ldg(seq_lens + b);
    if (L < nq || (int64_t)L > (int64_t)max_pages * kPageSize) return -1;
    return L - nq + j + 1;
  }
  __device__ int row_tiles(int r) const {
    int n = row_tokens(r);
    return n <= 0 ? 0 : (n + tile - 1) / tile;
  }
  __device__ int64_t cta_start(int c) const { return (int64_t)c * T / G; }
  // CTA whose range contains tile x (0 <= x < T)
  __device__ int cta_of(int64_t x) const { return (int)(((x + 1) * G - 1) / T); }
  __device__ int row_pieces(int64_t rt, int t) const {
    return t == 0 ? 0 : cta_of(rt + t - 1) - cta_of(rt) + 1;
  }
  // query / output row of plan row r (for fork f), and block-table element
  // offset of row r's first page
  __device__ int q_row(int r, int /*fork*/) const { return r; }
  __device__ int64_t bt_base(int r) const { return (int64_t)(r / nq) * max_pages; }
};

// Cursor over a CTA's tiles. All threads of a CTA keep identical copies.
struct RowCursor {
  int r;          // current row
  int64_t rt;     // first global tile of row r
  int t;          // tiles of row r
  int base;       // first partial slot of row r
  int n;          // visible tokens of row r
};

// ---------------------------------------------------------------------------
// Grouped decode (requests that share a prefix).
//
// Requests [g*F, (g+1)*F) form group g; their first prefix_pages[g] block-table
// entries name the same physical pages (a shared context that forked into F
// sessions). The work is two plans of the same shape as Plan:
//   kind 1 (prefix): one row per (group, draft) over the group's prefix pages,
//     cut over W = CTAs / F workers; CTA c works for worker c / F as fork c % F,
//     so the F forks of a group read each shared page at the same time (from
//     HBM once, the others from L2) and each writes its own partial;
//   kind 2 (suffix): one row per (request, draft) over the tokens after the
//     prefix, cut over all CTAs like Plan.
// Partial slots come from a row table laid out by group_plan_kernel: row r's
// slots are [row_base[r], +row_np1[r]) for its prefix pieces (ordered by
// worker), then its suffix pieces (ordered by CTA).
// A row is bad (no pieces, out = 0, lse = -inf) if its length is outside
// [Q, max_pages * 64], if prefix_pages[g] is outside [0, max_pages] or if the
// prefix is longer than L - Q + 1 (draft 0 must see all of it).
// ---------------------------------------------------------------------------
struct GroupPlan {
  static constexpr bool kGrouped = true;
  const int32_t* seq_lens;
  int batch, nq, max_pages, tile;
  int G;          // workers: min(workers of the launch, T)
  int64_t T;
  int kind;       // 1 prefix, 2 suffix
  int forks;
  const int32_t* prefix_pages;

  __device__ void set_total(int64_t total) {
    T = total;
    if (T < G) G = (int)T;
  }
  __device__ int groups() const { return batch / forks; }
  __device__ int rows() const { return (kind == 1 ? groups() : batch) * nq; }
  __device__ int group_prefix(int g) const {
    const int pp = __ldg(prefix_pages + g);
    return (pp < 0 || pp > max_pages) ? -1 : pp;
  }
  // whether request b can be decoded with its group's prefix
  __device__ bool request_ok(int b, int pp) const {
    const int L = __ldg(seq_lens + b);
    return pp >= 0 && L >= nq && (int64_t)L <= (int64_t)max_pages * kPageSize &&
           (int64_t)pp * kPageSize <= (int64_t)L - nq + 1;
  }
  __device__ int row_tokens(int r) const {
    const int j = r - (r / nq) * nq;
    if (kind == 1) {
      const int pp = group_prefix(r / nq);
      return pp < 0 ? -1 : pp * kPageSize;
    }
    const int b = r / nq;
    const int pp = group_prefix(b / forks);
    if (!request_ok(b, pp)) return -1;
    return __ldg(seq_lens + b) - nq + j + 1 - pp * kPageSize;
  }
  __device__ int row_tiles(int r) const {
    int n = row_tokens(r);
    return n <= 0 ? 0 : (n + tile - 1) / tile;
  }
  __device__ int64_t cta_start(int c) const { return (int64_t)c * T / G; }
  __device__ int cta_of(int64_t x) const { return (int)(((x + 1) * G - 1) / T); }
  __device__ int row_pieces(int64_t rt, int t) const {
    return t == 0 ? 0 : cta_of(rt + t - 1) - cta_of(rt) + 1;
  }
  __device__ int q_row(int r, int fork) const {
    if (kind == 2) return r;
    const int g = r / nq, j = r - (r / nq) * nq;
    return (g * forks + fork) * nq + j;
  }
  __device__ int64_t bt_base(int r) const {
    const int b = (kind == 1) ? (r / nq) * forks : r / nq;
    const int64_t off = (int64_t)b * max_pages;
    return kind == 1 ? off : off + group_prefix(b / forks);
  }
};

template <class P>
__device__ inline void cursor_next_row(const P& p, RowCursor& cur) {
  do {
    cur.base += p.row_pieces(cur.rt, cur.t);
    cur.rt += cur.t;
    cur.r += 1;
    cur.n = cur.r < p.rows() ? p.row_tokens(cur.r) : 0;
    cur.t = cur.n <= 0 ? 0 : (cur.n + p.tile - 1) / p.tile;
  } while (cur.t == 0 && cur.r < p.rows());
}

// Total tiles T, computed by one warp (loop over rows, shuffle reduction).
template <class P>
__device__ inline int64_t plan_total_tiles_warp(const P& p) {
  int lane = threadIdx.x & 31;
  int64_t acc = 0;
  for (int r = lane; r < p.rows(); r += 32) acc += p.row_tiles(r);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  return acc;
}

// Walks rows with one warp to find the row containing tile x0 and its
// RowCursor; optionally writes the row table (row_base / row_np) for all rows.
// Returns the cursor in lane 0's result (all lanes get the same value).
template <class P>
__device__ inline RowCursor plan_find_row_warp(const P& p, int64_t x0, bool write_table,
                                               int32_t* row_base, int32_t* row_np,
                                               unsigned* status) {
  int lane = threadIdx.x & 31;
  int64_t rt_carry = 0;
  int base_carry = 0;
  RowCursor found{-1, 0, 0, 0, 0};
  bool have = false;
  for (int r0 = 0; r0 < p.rows(); r0 += 32) {
    int r = r0 + lane;
    int t = r < p.rows() ? p.row_tiles(r) : 0;
    // inclusive scan of t
    int64_t incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int64_t v = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += v;
    }
    int64_t rt = rt_carry + incl - t;
    int np = (r < p.rows()) ? p.row_pieces(rt, t) : 0;
    int incl_np = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl_np, o);
      if (lane >= o) incl_np += v;
    }
    int base = base_carry + incl_np - np;
    if (write_table && r < p.rows()) {
      bool bad = p.row_tokens(r) < 0;
      row_base[r] = base;
      row_np[r] = bad ? -1 : np;
      if (bad) atomicOr(status, MLA_DEVICE_ERR_BAD_LENGTH);
    }
    bool hit = (r < p.rows()) && t > 0 && rt <= x0 && x0 < rt + t;
    unsigned m = __ballot_sync(0xffffffffu, hit);
    if (m && !have) {
      int src = __ffs(m) - 1;
      found.r = __shfl_sync(0xffffffffu, r, src);
      found.rt = __shfl_sync(0xffffffffu, rt, src);
      found.t = __shfl_sync(0xffffffffu, t, src);
      found.base = __shfl_sync(0xffffffffu, base, src);
      found.n = __shfl_sync(0xffffffffu, r < p.rows() ? p.row_tokens(r) : 0, src);
      have = true;
      if (!write_table) break;
    }
    rt_carry = __shfl_sync(0xffffffffu, rt_carry + incl, 31);
    base_carry = __shfl_sync(0xffffffffu, base_carry + incl_np, 31);
  }
  return found;
}

// ---------------------------------------------------------------------------
// PTX wrappers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// 16-byte async copy global->shared; src_bytes = 0 zero-fills the destination.
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, int src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dst), "l"(src),
               "r"(src_bytes));
}
// 4-byte async copy global->shared (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;\n" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory");
}
// Waits until at most n (0..N) of this thread's groups are pending; n > N counts as N.
template <int N>
__device__ __forceinline__ void cp_async_wait_upto(int n) {
  if constexpr (N == 0) {
    cp_async_wait<0>();
  } else {
    if (n >= N) cp_async_wait<N>();
    else cp_async_wait_upto<N - 1>(n);
  }
}

// L2 policy for data read once (the KV stream): its lines are the first to be
// evicted, so that code, q and page tables stay resident in L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
  return pol;
}
// 16-byte read-only load that allocates no L1 line and marks its L2 lines with `pol`.
__device__ __forceinline__ uint4 ld_stream_16(const void* p, uint64_t pol) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;\n"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p), "l"(pol));
  return v;
}
// e4m3 pair -> f16 pair (exact: every e4m3 value is an f16 normal number).
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint16_t v) {
  uint32_t r;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;\n" : "=r"(r) : "h"(v));
  return r;
}

// Programmatic dependent launch. griddep_wait() returns once every grid this one
// depends on has completed and its memory writes are visible (at once when the
// grid was launched without the programmatic-serialization attribute); it must
// precede this grid's first global memory access. griddep_launch_dependents()
// lets the next such grid in the stream be scheduled before this one ends.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;\n" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
  return y;
}

}  // namespace mla
