// decode_fp8.cu -- split-KV paged MLA decode with the e4m3 cache bytes as
// tensor-core operands (tcgen05.mma kind::f8f6f4).
//
// The cache pages are contractions' operands as stored: "Smaller, faster, safer:
// running Kimi and GLM at scale", section "Quantizing the KV cache", keeps the
// latent cache in FP8 with one scale; here the tensor core reads those bytes
// directly instead of widening them first. One CTA per SM walks its run of
// pages (split-KV planner in mla_common.cuh), one 64-token page per step:
//
//   S [128 x 64 tokens]  = A . page^T       A = [q_hi ; q_lo] per head, e4m3
//   O^T[512 x 64 heads] += V^T . (P_hi + P_lo)^T      V = the page's first 512 dims
//
// q (bf16) is scaled per head by a power of two (max |q| in [2^7, 2^8)) and split
// into two e4m3 terms q_hi = e4m3(q), q_lo = e4m3(q - q_hi), which is exact for
// bf16 inputs (8 significant bits = 4 + 4) down to 2^-10 of the head's max, so
// S_hi + S_lo is q . k up to fp32 accumulation. The split runs once per row in a
// small kernel launched before the decode kernel (q_split_kernel), which writes
// the A operand in the order the decode kernel's threads load it. P = 2^(s - m + 6) is split into
// an e4m3 term and an e5m2 remainder (7 significant bits; the e5m2 range keeps
// tokens down to 2^-24 of the running maximum). All heads attend over the one latent
// head ("vLLM x AgentX", section "Kimi K3"), so one page serves 64 heads, and V
// is read in place through an MN-major descriptor (no distinct values: "How to
// serve trillions of tokens ...", section "First, understand the workload").
//
// Warp roles (224 threads):
//   warps 0-3  q loading, softmax and epilogue. Row t of A and S is (head
//              16*(t/32) + t%16, part (t/16)%2), part 0 = hi, 1 = lo. Thread t
//              handles head 16*(t/32) + t%16 and tokens 32*((t/16)%2) .. +31 of a
//              page: it reads both terms' rows of its half-page (a half-split
//              TMEM load), so no exchange between threads is needed; for O^T
//              lane t is dim t of each 128-dim block.
//   warp 4     TMA producer (lane 0): page ids from the block table a window of
//              pages ahead, pages into a ring of kRing shared-memory slots
//              (128-byte swizzled latent blocks, 64-byte swizzled rope block).
//   warp 5     TMEM allocation; issues QK (lane 0) after zeroing the rows of a
//              partial page past its last token.
//   warp 6     issues PV (lane 0).
// TMEM (512 columns): A latent part [0,128), S buffers [128,192) [192,256),
// O^T [256,512). The rope part of A is in shared memory.
//
// Every wait is bounded (2 s); on timeout the CTA records MLA_DEVICE_ERR_TIMEOUT,
// stops, drains its MMAs and copies (bounded, 2 s) and frees TMEM.
#include <atomic>
#include <type_traits>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 224;
constexpr int kTmaWarp = 4;
constexpr int kQkWarp = 5;   // allocates TMEM, issues QK
constexpr int kPvWarp = 6;   // issues PV
constexpr int kRing = 5;                             // pages in flight
constexpr int kPageBytes = kPageSize * kDEntry;      // 36864
constexpr int kLatBlock = kPageSize * 128;           // 8192: 64 rows x 128 dims
constexpr int kRopeOff = 4 * kLatBlock;              // rope block within a page slot
constexpr int kPBytes = 64 * 128;                    // P^T: 64 heads x [64 hi | 64 lo]
constexpr int kPOffset = 6;                          // P = 2^(s - m + 6)
constexpr float kRescaleThresh = 2.8f;               // P <= 2^8.8 < 448 (e4m3 max)
// A page whose maximum lies more than kLowThresh below the running maximum
// brings the running maximum down to its own (O^T and l scale up), so that its
// largest weight is at least 2^(kPOffset - kLowThresh) = 1 and its tokens keep
// the split's precision, unless the accumulated mass l would then exceed
// kMassCap (the page's largest weight is then below 2^-28 of the mass so far:
// 2^18 such tokens still stay below 2^-10 of it).
constexpr float kLowThresh = 6.0f;
constexpr float kMassCap = 17179869184.0f;           // 2^34 = 2^(kPOffset + 28)
// Limit of a wait on another role of the pipeline, and of a wait for copies and
// MMAs already issued (the drain before exit). A test build lowers the first
// (MLA_PIPELINE_WAIT_NS) to make the timeout path run; the drain keeps 2 s.
#ifndef MLA_PIPELINE_WAIT_NS
#define MLA_PIPELINE_WAIT_NS 2000000000ull
#endif
constexpr uint64_t kWaitNs = MLA_PIPELINE_WAIT_NS;
constexpr uint64_t kDrainWaitNs = 2000000000ull;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 0;
__device__ __forceinline__ uint32_t s_col(int b) { return 128u + 64u * (uint32_t)b; }
constexpr uint32_t kOCol = 256;

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffPages = 0;
constexpr int kOffQRope = kOffPages + kRing * kPageBytes;   // 128 rows x 64 B, 64B swizzle
constexpr int kPBufs = 3;                                   // P^T buffers (QK runs 2 pages ahead)
constexpr int kOffP = kOffQRope + 128 * 64;                 // [kPBufs] P^T buffers
constexpr int kOffAlpha = kOffP + kPBufs * kPBytes;         // float [2][64]
constexpr int kOffLinv = kOffAlpha + 512;                   // float [64]
constexpr int kOffFlags = kOffLinv + 256;                   // int [4]
constexpr int kOffPlan = kOffFlags + 16;                    // int64 [6]
constexpr int kDescRing = 64;                               // page descriptors in flight
constexpr int kTableAhead = 32;  // pages described (block-table read started) before issue
constexpr int kOffDesc = kOffPlan + 48;                     // PageDesc [kDescRing]
constexpr int kOffBar = kOffDesc + 16 * kDescRing;
constexpr int BAR_PAGE_FULL = 0;              // [kRing] TMA bytes (or zero fill) landed
constexpr int BAR_PAGE_EMPTY = kRing;         // [kRing] PV of the slot's page finished
constexpr int BAR_S_FULL = 2 * kRing;         // [2] page j: buffer j % 2
constexpr int BAR_S_EMPTY = 2 * kRing + 2;    // [2] (4 softmax warps)
constexpr int BAR_P_FULL = 2 * kRing + 4;     // [kPBufs] page j: buffer j % 3 (4 softmax warps)
constexpr int BAR_PV_DONE = 2 * kRing + 7;    // [2] PV of page j commits barrier j % 2
constexpr int BAR_O_FULL = 2 * kRing + 9;
constexpr int BAR_O_EMPTY = 2 * kRing + 10;   // (4 softmax warps)
constexpr int BAR_Q_READY = 2 * kRing + 11;   // (4 softmax warps)
constexpr int BAR_Q_EMPTY = 2 * kRing + 12;
constexpr int BAR_DRAIN = 2 * kRing + 13;      // [2] QK warp, PV warp
constexpr int BAR_P_EMPTY = 2 * kRing + 15;    // [kPBufs] PV of page j read P buffer j % 3
#ifdef MLA_TEST_STALL_QK
// Test build only: a barrier that nothing ever completes. The QK issuer waits on
// it before its third page, so the wait runs out and the CTA takes the timeout
// path (stop every role, drain the copies and MMAs in flight, free TMEM).
constexpr int BAR_TEST_STALL = 2 * kRing + 15 + kPBufs;
constexpr int kNumBars = BAR_TEST_STALL + 1;
#else
constexpr int kNumBars = 2 * kRing + 15 + kPBufs;
#endif
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024 alignment
// grouped decode: the two segments' plans (int64 [32]) after the common map
constexpr int kOffPlanX = (kSmemUsed + 15) & ~15;
constexpr int kSmemBytesGrouped = kOffPlanX + 256 + 1024;

enum Flag { F_ABORT = 0, F_PIECE_BAD = 1 };

// What every role needs to know about the CTA's j-th page, written by the TMA
// warp (the only planner walker) before it signals the page, read by the MMA and
// softmax warps after they have waited for it.
struct PageDesc {
  int32_t page;    // block-table entry
  int16_t valid;   // tokens of the row in this page (1..64)
  int16_t flags;   // kDescPieceStart | kDescPieceEnd | kDescPageOk
  int32_t row;     // request row r = b * Q + j
  int32_t slot;    // partial slot of this piece
};
constexpr int16_t kDescPieceStart = 1, kDescPieceEnd = 2, kDescPageOk = 4;
constexpr int16_t kDescShared = 8;  // grouped decode: a shared-prefix page (informational)

struct Fp8Params {
  const __nv_bfloat16* q;
  int64_t num_pages;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int batch, nq, heads;
  int rows;          // batch * nq
  float score_mul;   // sm_scale * log2(e) * kv_scale
  float kv_scale;
  int G;
  DecodeWorkspace ws;
  // grouped decode (decode_fp8_kernel<true>) only
  int forks;                    // requests per group
  int workers;                  // CTAs / forks: workers of the shared-prefix plan
  const int32_t* prefix_pages;  // [batch / forks] shared pages of each group
};

__device__ inline GroupPlan group_plan(const Fp8Params& p, int kind) {
  return GroupPlan{p.seq_lens, p.batch, p.nq, p.max_pages, kPageSize,
                   kind == 1 ? p.workers : p.G, 0, kind, p.forks, p.prefix_pages};
}

// Cursor over a CTA's pages (one page per step). The row's partial slot and
// block-table offset are computed once per row: a step costs no division.
// `cta` is the worker index in the plan; for the grouped decode's plans the
// slot comes from the row table and `fork` picks the query row.
template <class P>
struct PageWalker {
  P plan;
  RowCursor cur;
  int64_t x, x_end, x_begin;
  int cta;         // this CTA's worker index in the plan
  int fork;        // grouped decode: the fork this CTA works for
  int slot;        // partial slot of the current row's piece in this CTA
  int qrow;        // query / output row of the current row
  int64_t bt_row;  // block-table offset of the current row's first page
  const int32_t* row_base;  // grouped decode: the row table
  const int32_t* row_np1;

  __device__ void init(const P& p, const RowCursor& c, int cta_index, int64_t xb, int64_t xe,
                       int fork_index = 0, const int32_t* rb = nullptr,
                       const int32_t* np1 = nullptr) {
    plan = p; cur = c; cta = cta_index; x = xb; x_begin = xb; x_end = xe;
    fork = fork_index; row_base = rb; row_np1 = np1;
    row_changed();
    settle();
  }
  __device__ void row_changed() {
    if constexpr (P::kGrouped) {
      qrow = plan.q_row(cur.r, fork);
      slot = __ldcg(row_base + qrow) + (plan.kind == 2 ? __ldcg(row_np1 + qrow) : 0) +
             (cta - plan.cta_of(cur.rt));
    } else {
      qrow = cur.r;
      slot = cur.base + (cta - plan.cta_of(cur.rt));
    }
    bt_row = plan.bt_base(cur.r);
  }
  __device__ void settle() {
    if (x < x_end && x == cur.rt + cur.t) {
      cursor_next_row(plan, cur);
      row_changed();
    }
  }
  __device__ int page_in_row() const { return (int)(x - cur.rt); }
  __device__ bool piece_start() const { return x == x_begin || x == cur.rt; }
  __device__ bool piece_end() const { return x + 1 == x_end || x + 1 == cur.rt + cur.t; }
  __device__ int valid_tokens() const { return min(kPageSize, cur.n - page_in_row() * kPageSize); }
  __device__ void next() { ++x; settle(); }
  __device__ bool shared() const { return false; }
};

// The grouped decode's walker: this CTA's range of the shared-prefix plan (as
// fork `fork` of its worker), then its range of the suffix plan.
struct SegWalker : PageWalker<GroupPlan> {
  GroupPlan B;
  RowCursor curB;
  int64_t xbB, xeB;
  int ctaB;
  bool in_prefix;
  __device__ void start(const GroupPlan& A, const RowCursor& ca, int64_t xbA, int64_t xeA,
                        int worker, int fork_index, const GroupPlan& Bp, const RowCursor& cb,
                        int64_t xb, int64_t xe, int cta_index, const int32_t* rb,
                        const int32_t* np1) {
    B = Bp; curB = cb; xbB = xb; xeB = xe; ctaB = cta_index;
    in_prefix = xbA < xeA;
    if (in_prefix) init(A, ca, worker, xbA, xeA, fork_index, rb, np1);
    else init(B, curB, ctaB, xbB, xeB, 0, rb, np1);
  }
  __device__ void next() {
    PageWalker<GroupPlan>::next();
    if (in_prefix && x == x_end) {
      in_prefix = false;
      if (xbB < xeB) init(B, curB, ctaB, xbB, xeB, 0, row_base, row_np1);
    }
  }
  __device__ bool shared() const { return in_prefix; }
};

__device__ __forceinline__ void named_bar_softmax() {
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
}
__device__ __forceinline__ bool named_bar_softmax_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 128, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred)
      : "memory");
  return r != 0;
}

// Two floats -> two e4m3 codes (round to nearest even, saturating); `lo` in the low byte.
__device__ __forceinline__ uint32_t e4m3x2_of(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ float2 e4m3x2_value(uint32_t codes) {
  const uint32_t h2 = e4m3x2_to_f16x2((uint16_t)codes);
  return __half22float2(*reinterpret_cast<const __half2*>(&h2));
}
// Two floats -> two e5m2 codes (round to nearest even, saturating); `lo` in the low byte.
__device__ __forceinline__ uint32_t e5m2x2_of(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// kGrouped: the grouped decode (GroupPlan): this CTA's shared-prefix range, then
// its suffix range; otherwise mla_decode's single plan (Plan).
template <bool kGrouped>
__global__ void __launch_bounds__(kThreads, 1)
    decode_fp8_kernel(const Fp8Params p, const __grid_constant__ CUtensorMap lat_map,
                      const __grid_constant__ CUtensorMap rope_map) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_a = smem_u32(smem_raw);
  const uint32_t sbase = (raw_a + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_a);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);
  float* linv_s = reinterpret_cast<float*>(smem + kOffLinv);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
  int64_t* s_plan = reinterpret_cast<int64_t*>(smem + kOffPlan);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- planning (shared by all roles) ----
  // This kernel starts once the query split kernel before it has passed its own
  // wait for all earlier work in the stream (see launch_decode_fp8), so the
  // lengths, block table and pages may be read at once; only the split query
  // itself needs the split kernel to have completed (griddep_wait before q_op).
  if (warp == kTmaWarp && lane == 0) {
    tc::prefetch_tensormap(&lat_map);
    tc::prefetch_tensormap(&rope_map);
  }
  Plan plan{p.seq_lens, p.batch, p.nq, p.max_pages, kPageSize, p.G, 0};
  const int c = blockIdx.x;
  int64_t* s_plan_x = reinterpret_cast<int64_t*>(smem + kOffPlanX);  // kGrouped only
  if (warp == 0) {
    if constexpr (kGrouped) {
      // both plans (row table written by group_plan_kernel): this CTA's prefix
      // range as fork f of worker w, then its suffix range
      GroupPlan A = group_plan(p, 1), B = group_plan(p, 2);
      A.set_total(plan_total_tiles_warp(A));
      B.set_total(plan_total_tiles_warp(B));
      const int w = c / p.forks, f = c - w * p.forks;
      const bool in_a = c < p.forks * p.workers && w < A.G;
      const bool in_b = c < B.G;
      const int64_t xba = in_a ? A.cta_start(w) : 0, xea = in_a ? A.cta_start(w + 1) : 0;
      const int64_t xbb = in_b ? B.cta_start(c) : 0, xeb = in_b ? B.cta_start(c + 1) : 0;
      RowCursor fa{0, 0, 0, 0, 0}, fb{0, 0, 0, 0, 0};
      if (in_a) fa = plan_find_row_warp(A, xba, false, p.ws.row_base, p.ws.row_np, p.ws.status);
      if (in_b) fb = plan_find_row_warp(B, xbb, false, p.ws.row_base, p.ws.row_np, p.ws.status);
      if (lane == 0) {
        s_plan[0] = (xea - xba) + (xeb - xbb);                 // pages of this CTA
        s_plan[1] = xea > xba ? A.q_row(fa.r, f) : fb.r;       // query row of its first piece
        const int64_t v[20] = {A.T, B.T, xba, xea, xbb, xeb, w, f, fa.r, fa.rt, fa.t, fa.base,
                               fa.n, fb.r, fb.rt, fb.t, fb.base, fb.n, 0, 0};
        for (int i = 0; i < 20; ++i) s_plan_x[i] = v[i];
      }
    } else {
      // the whole plan in one warp pass: total tiles, then this CTA's first row
      Plan pl = plan;
      pl.set_total(plan_total_tiles_warp(pl));
      const int64_t xb = c < pl.G ? pl.cta_start(c) : 0;
      RowCursor f = plan_find_row_warp(pl, xb, c == 0, p.ws.row_base, p.ws.row_np, p.ws.status);
      if (lane == 0) {
        s_plan[0] = pl.T;
        s_plan[1] = f.r;
        s_plan[2] = f.rt;
        s_plan[3] = f.t;
        s_plan[4] = f.base;
        s_plan[5] = f.n;
      }
    }
  }
  if (warp == kPvWarp && lane == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool by_warps = (i >= BAR_S_EMPTY && i < BAR_S_EMPTY + 2) ||
                            (i >= BAR_P_FULL && i < BAR_P_FULL + kPBufs) || i == BAR_O_EMPTY ||
                            i == BAR_Q_READY;
      tc::mbar_init(bar(i), by_warps ? 4 : 1);
    }
    tc::fence_mbar_init();
    flags[F_ABORT] = 0;
    flags[F_PIECE_BAD] = 0;
  }
  if (warp == kQkWarp) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  griddep_launch_dependents();  // the combine kernel may be scheduled (it waits for this grid)
  int64_t x_begin = 0, x_end = 0;
  if constexpr (kGrouped) {
    x_end = s_plan[0];
  } else {
    plan.set_total(s_plan[0]);
    const bool works = c < plan.G;
    x_begin = works ? plan.cta_start(c) : 0;
    x_end = works ? plan.cta_start(c + 1) : 0;
  }
  const uint32_t tmem = *tmem_slot;
  const RowCursor cur0{(int)s_plan[1], s_plan[2], (int)s_plan[3], (int)s_plan[4],
                       (int)s_plan[5]};
  const int H = p.heads;
  auto abort_cta = [&]() {
    flags[F_ABORT] = 1;
    atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
  };

  const int64_t npages = x_end - x_begin;
  const PageDesc* desc = reinterpret_cast<const PageDesc*>(smem + kOffDesc);
  if (x_begin < x_end) {
    if (warp == kTmaWarp) {
      // =================== TMA producer (lane 0) ===================
      // Lane 0 describes each page kTableAhead pages before it issues the page's
      // copy: the descriptor fields come from the walker and the physical page id
      // from an asynchronous 4-byte copy of the block-table entry, so a table read
      // that misses L2 (over 10 us behind a full stream of page copies) never
      // holds up the copies. The warp's other lanes have nothing to do.
      if (lane == 0) {
        const uint64_t pol = l2_evict_first_policy();
        PageDesc* ring = reinterpret_cast<PageDesc*>(smem + kOffDesc);
        std::conditional_t<kGrouped, SegWalker, PageWalker<Plan>> pw;
        if constexpr (kGrouped) {
          GroupPlan A = group_plan(p, 1), B = group_plan(p, 2);
          A.set_total(s_plan_x[0]);
          B.set_total(s_plan_x[1]);
          const RowCursor ca{(int)s_plan_x[8], s_plan_x[9], (int)s_plan_x[10],
                             (int)s_plan_x[11], (int)s_plan_x[12]};
          const RowCursor cb{(int)s_plan_x[13], s_plan_x[14], (int)s_plan_x[15],
                             (int)s_plan_x[16], (int)s_plan_x[17]};
          pw.start(A, ca, s_plan_x[2], s_plan_x[3], (int)s_plan_x[6], (int)s_plan_x[7], B, cb,
                   s_plan_x[4], s_plan_x[5], c, p.ws.row_base, p.ws.row_np1);
        } else {
          pw.init(plan, cur0, c, x_begin, x_end);
        }
        int64_t jn = 0;  // next page to describe
        auto describe_next = [&]() {
          PageDesc& d = ring[jn % kDescRing];
          const bool ps = pw.piece_start();
          d.valid = (int16_t)pw.valid_tokens();
          d.flags = (int16_t)((ps ? kDescPieceStart : 0) | (pw.piece_end() ? kDescPieceEnd : 0) |
                              (pw.shared() ? kDescShared : 0));
          d.row = pw.qrow;
          d.slot = pw.slot;
          cp_async_4(smem_u32(&d.page), p.block_table + pw.bt_row + pw.page_in_row());
          cp_async_commit();
          if (ps && jn > 0)  // the softmax warps read this row's q when they reach it
            tc::prefetch_l2_bulk(p.q + (int64_t)pw.qrow * H * kDEntry,
                                 (uint32_t)(H * kDEntry * sizeof(__nv_bfloat16)));
          pw.next();
          ++jn;
        };
        // the first copies go out as soon as their table entries are in; the
        // look-ahead window fills up two pages per issued page
        while (jn < kRing && jn < npages) describe_next();
        int64_t j = 0;
        bool ok = true;
        for (; j < npages; ++j) {
          // page j's table read is the oldest of the jn - j groups in flight
          cp_async_wait_upto<kTableAhead>((int)(jn - j - 1));
          PageDesc* d = ring + j % kDescRing;
          const int32_t page = d->page;
          const bool page_ok = page >= 0 && (int64_t)page < p.num_pages;
          if (page_ok) d->flags |= kDescPageOk;
          const int slot = (int)(j % kRing);
          const uint32_t round = (uint32_t)(j / kRing);
          const uint32_t page_base = sbase + kOffPages + slot * kPageBytes;
          if (j >= kRing &&
              (!tc::mbar_wait(bar(BAR_PAGE_EMPTY + slot), (round - 1) & 1, kWaitNs) ||
               flags[F_ABORT])) {
            ok = false;
            break;
          }
          if (page_ok) {
            tc::mbar_arrive_expect_tx(bar(BAR_PAGE_FULL + slot), (uint32_t)kPageBytes);
            const int y = page * kPageSize;
            // (a grouped decode's shared page is read by the other forks' CTAs a
            // few pages' time later, well within the life of an evict-first line)
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tc::tma_load_2d_hint(page_base + b * kLatBlock, &lat_map, 128 * b, y,
                                   bar(BAR_PAGE_FULL + slot), pol);
            tc::tma_load_2d_hint(page_base + kRopeOff, &rope_map, kDLatent, y,
                                 bar(BAR_PAGE_FULL + slot), pol);
          } else {
            tc::mbar_arrive(bar(BAR_PAGE_FULL + slot));  // bad id: the MMA warp zero-fills
          }
          for (int u = 0; u < 2 && jn < npages && jn <= j + kTableAhead; ++u) describe_next();
        }
        cp_async_wait<0>();
        if (!ok) abort_cta();
        // no copy may land after the CTA exits: wait for the last issued pages
        for (int64_t jj = j > kRing ? j - kRing : 0; jj < j; ++jj)
          tc::mbar_wait(bar(BAR_PAGE_FULL + (int)(jj % kRing)), (uint32_t)(jj / kRing) & 1,
                        kDrainWaitNs);
      }
      __syncwarp();
    } else if (warp == kQkWarp || warp == kPvWarp) {
      // ============ MMA issuers: QK warp and PV warp, lane 0 issues ============
      // The two streams are issued by different threads, so neither's completion
      // implies the other's: P buffer reuse and the O^T rescale wait on the PV
      // warp's own commits (P_EMPTY, PV_DONE).
      constexpr uint32_t id_qk = tc::idesc_f8(128, 64, tc::kFmtE4M3, tc::kFmtE4M3, false, false);
      // PV: A = V^T (e4m3, MN-major); B = P^T hi (e4m3) or lo (e5m2), K-major
      constexpr uint32_t id_pv_hi = tc::idesc_f8(128, 64, tc::kFmtE4M3, tc::kFmtE4M3, true, false);
      constexpr uint32_t id_pv_lo = tc::idesc_f8(128, 64, tc::kFmtE4M3, tc::kFmtE5M2, true, false);
      const bool leader = lane == 0;
      // bounded wait by lane 0, result shared with the warp
      auto wait0 = [&](int b, uint32_t parity) -> bool {
        bool got = true;
        if (leader) got = tc::mbar_wait(bar(b), parity, kWaitNs);
        return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      };
      bool ok = true;
      if (warp == kQkWarp) {
        const uint64_t qrope_desc = tc::smem_desc(sbase + kOffQRope, 16, 512, tc::kSwizzle64);
        int q_piece = 0;
        for (int64_t k = 0; k < npages && ok; ++k) {
          if (flags[F_ABORT]) {
            ok = false;
            break;
          }
#ifdef MLA_TEST_STALL_QK
          if (k == 2) {
            ok = wait0(BAR_TEST_STALL, 0);
            if (!ok) break;
          }
#endif
          const int slot = (int)(k % kRing);
          const uint32_t page_base = sbase + kOffPages + slot * kPageBytes;
          ok = wait0(BAR_PAGE_FULL + slot, (uint32_t)(k / kRing) & 1);
          if (!ok) break;
          const PageDesc d = desc[k % kDescRing];
          if (d.flags & kDescPieceStart) {
            ok = wait0(BAR_Q_READY, (uint32_t)q_piece & 1);
            ++q_piece;
          }
          if (ok && k >= 2) ok = wait0(BAR_S_EMPTY + (int)(k & 1), (uint32_t)((k >> 1) - 1) & 1);
          if (!ok) break;
          // rows past the page's last token (all rows of a bad page id) become zeros,
          // so that masked tokens contribute 0 * finite to PV
          const int zero_from = (d.flags & kDescPageOk) ? d.valid : 0;
          if (zero_from < kPageSize) {
            for (int i = lane; i < (kPageSize - zero_from) * 36; i += 32) {
              const int row = zero_from + i / 36, u = i % 36;
              const uint32_t a = u < 32 ? page_base + (u >> 3) * kLatBlock + row * 128 + (u & 7) * 16
                                        : page_base + kRopeOff + row * 64 + (u - 32) * 16;
              asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};\n" ::"r"(a), "r"(0u));
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
          }
          if (leader) {
            // ---- S = A . page^T: latent part of A from TMEM, rope from shared memory ----
            tc::fence_after_sync();
            const uint64_t kb = tc::smem_desc(page_base, 16, 1024, tc::kSwizzle128);
            const uint64_t rb = tc::smem_desc(page_base + kRopeOff, 16, 512, tc::kSwizzle64);
            const uint32_t d_s = tmem + s_col((int)(k & 1));
#pragma unroll
            for (int s = 0; s < 16; ++s)
              tc::mma_f8_ts(d_s, tmem + kQCol + 8 * s,
                            kb + (uint64_t)(((s >> 2) * kLatBlock + (s & 3) * 32) >> 4), id_qk,
                            s > 0);
#pragma unroll
            for (int s = 0; s < 2; ++s)
              tc::mma_f8_ss(d_s, qrope_desc + (uint64_t)((32 * s) >> 4),
                            rb + (uint64_t)((32 * s) >> 4), id_qk, 1);
            tc::mma_commit(bar(BAR_S_FULL + (int)(k & 1)));
            if (d.flags & kDescPieceEnd) tc::mma_commit(bar(BAR_Q_EMPTY));
          }
          __syncwarp();
        }
      } else {
        int o_piece = 0;
        for (int64_t k = 0; k < npages && ok; ++k) {
          if (flags[F_ABORT]) {
            ok = false;
            break;
          }
          const int pb_i = (int)(k % kPBufs);
          ok = wait0(BAR_P_FULL + pb_i, (uint32_t)(k / kPBufs) & 1);
          if (!ok) break;
          const PageDesc d = desc[k % kDescRing];
          const bool ps = d.flags & kDescPieceStart, pe = d.flags & kDescPieceEnd;
          if (ps) {
            if (o_piece > 0) ok = wait0(BAR_O_EMPTY, (uint32_t)(o_piece - 1) & 1);
            ++o_piece;
            if (!ok) break;
          }
          if (leader) {
            // ---- O^T += V^T P^T ----
            tc::fence_after_sync();
            const int slot = (int)(k % kRing);
            const uint32_t page_base = sbase + kOffPages + slot * kPageBytes;
            const uint64_t va = tc::smem_desc(page_base, kLatBlock, 1024, tc::kSwizzle128);
            const uint64_t pb =
                tc::smem_desc(sbase + kOffP + pb_i * kPBytes, 16, 1024, tc::kSwizzle128);
#pragma unroll
            for (int blk = 0; blk < 4; ++blk)
#pragma unroll
              for (int s = 0; s < 2; ++s)
#pragma unroll
                for (int part = 0; part < 2; ++part)
                  tc::mma_f8_ss(tmem + kOCol + 64 * blk,
                                va + (uint64_t)((blk * kLatBlock + s * 4096) >> 4),
                                pb + (uint64_t)((64 * part + 32 * s) >> 4),
                                part ? id_pv_lo : id_pv_hi, !(ps && s == 0 && part == 0));
            tc::mma_commit(bar(BAR_PAGE_EMPTY + slot));
            tc::mma_commit(bar(BAR_P_EMPTY + pb_i));
            tc::mma_commit(bar(BAR_PV_DONE + (int)(k & 1)));
            if (pe) tc::mma_commit(bar(BAR_O_FULL));
          }
          __syncwarp();
        }
      }
      if (leader) {
        if (!ok) abort_cta();
        // drain: every MMA this thread issued has finished before TMEM is freed
        const int db = BAR_DRAIN + (warp == kPvWarp ? 1 : 0);
        tc::mma_commit(bar(db));
        if (!tc::mbar_wait(bar(db), 0, kDrainWaitNs))
          atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
      }
      __syncwarp();
    } else {
      // =================== softmax + epilogue (warps 0-3) ===================
      const int t = tid;
      const int h = 16 * warp + (lane & 15);   // head of this thread's row
      const int part = (lane >> 4) & 1;        // 0: q_hi / tokens 0-31, 1: q_lo / tokens 32-63
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      float m = -INFINITY, l = 0.f, qmul = 0.f;
      int piece = 0;
      bool ok = true;
      for (int64_t j = 0; j < npages; ++j) {
        // Page 0 opens the first piece, whose row the plan gives: its q is staged at
        // once. Later pages' descriptors are read once the page has landed.
        int row = cur0.r;
        bool ps = j == 0;
        if (j > 0) {
          // (a failed wait is acted on at this page's group barrier below; every
          // thread reads the same descriptor word, so the piece-start decision, and
          // with it the barriers of the q staging, is uniform either way)
          if (!tc::mbar_wait(bar(BAR_PAGE_FULL + (int)(j % kRing)), (uint32_t)(j / kRing) & 1,
                             kWaitNs))
            flags[F_ABORT] = 1;
          const PageDesc d0 = desc[j % kDescRing];
          row = min(max(d0.row, 0), p.rows - 1);  // in range even if a stopped producer never wrote it
          ps = d0.flags & kDescPieceStart;
        }
        if (ps) {
          // ---- load the split q of this row into A ----
          if (piece > 0) {
            const bool got = tc::mbar_wait(bar(BAR_Q_EMPTY), (uint32_t)(piece - 1) & 1, kWaitNs);
            if (named_bar_softmax_or(!got || flags[F_ABORT])) {
              ok = false;
              break;
            }
          }
          // The query split kernel wrote this row's operand as [36 chunks][128 lanes]
          // [16 codes]: this thread loads the 36 chunks of its own lane (coalesced
          // across the warp), stores the 32 latent chunks into its TMEM lane and the
          // 4 rope chunks into its shared-memory row (64-byte swizzle).
          griddep_wait();  // the split kernel has completed and its writes are visible
          const bool live = h < H;
          qmul = live ? __ldcg(p.ws.q_mul + (int64_t)row * 64 + h) : 0.f;
          const uint4* src =
              reinterpret_cast<const uint4*>(p.ws.q_op + (int64_t)row * kQOpRowBytes) + t;
          uint4 qc[kQOpChunks];
#pragma unroll
          for (int u = 0; u < kQOpChunks; ++u)
            qc[u] = live ? __ldcg(src + 128 * u) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            uint32_t v[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[4 * k] = qc[8 * g + k].x;
              v[4 * k + 1] = qc[8 * g + k].y;
              v[4 * k + 2] = qc[8 * g + k].z;
              v[4 * k + 3] = qc[8 * g + k].w;
            }
            tc::tmem_st32(tmem + lane_base + kQCol + 32 * g, v);
          }
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const uint32_t a = sbase + kOffQRope + t * 64 + ((c4 ^ ((t >> 1) & 3)) << 4);
            const uint4 v = qc[32 + c4];
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a), "r"(v.x), "r"(v.y),
                         "r"(v.z), "r"(v.w));
          }
          tc::tmem_wait_st();
          tc::fence_proxy_async_smem();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(bar(BAR_Q_READY));
        }
        // ---- S of this page ----
        // (a failed wait, like a stop by another role, is acted on at this page's
        // group barrier below: one barrier per page)
        if (!tc::mbar_wait(bar(BAR_S_FULL + (int)(j & 1)), (uint32_t)(j >> 1) & 1, kWaitNs))
          flags[F_ABORT] = 1;
        // page validity (tokens of a bad page id are masked and reported)
        const PageDesc d = desc[j % kDescRing];
        const bool pe = d.flags & kDescPieceEnd;
        const bool page_ok = d.flags & kDescPageOk;
        const int nvis = page_ok ? d.valid : 0;
        if (t == 0 && !page_ok) {
          flags[F_PIECE_BAD] = 1;
          atomicOr(p.ws.status, MLA_DEVICE_ERR_BAD_PAGE);
        }
        tc::fence_after_sync();
        // both terms of this thread's 32 tokens: rows 32w .. 32w+15 hold q_hi . k of
        // heads 16w .. 16w+15, rows 32w+16 .. 32w+31 q_lo . k; a half-warp reads
        // one half of the page's 64 columns
        uint32_t shi[32], slo[32];
        tc::tmem_ld16x2_32(tmem + ((uint32_t)(32 * warp) << 16) + s_col((int)(j & 1)), shi);
        tc::tmem_ld16x2_32(tmem + ((uint32_t)(32 * warp + 16) << 16) + s_col((int)(j & 1)), slo);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_S_EMPTY + (int)(j & 1)));
        float s[32];
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const bool vis = 32 * part + i < nvis;
          s[i] = vis ? (__uint_as_float(shi[i]) + __uint_as_float(slo[i])) * qmul : -INFINITY;
          tmax = fmaxf(tmax, s[i]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        // lazy running max: O is rescaled only when a head's page max rises more than
        // kRescaleThresh above it or falls more than kLowThresh below it
        float alpha = 1.f;
        bool grow = false;
        if (ps) {
          m = tmax;
        } else if (tmax > m + kRescaleThresh) {
          alpha = m == -INFINITY ? 0.f : fast_exp2(m - tmax);
          m = tmax;
          l *= alpha;
          grow = true;
        } else if (tmax < m - kLowThresh && l * fast_exp2(m - tmax) <= kMassCap) {
          alpha = fast_exp2(m - tmax);  // > 1: the page is far below the running max
          m = tmax;
          l *= alpha;
          grow = true;
        }
        // P buffer j % 3 was read by PV(j - 3); waiting for it also makes the
        // PV_DONE parity below unambiguous (PV(j - 3) is complete)
        if (j >= kPBufs && !flags[F_ABORT]) {
          const bool got = tc::mbar_wait(bar(BAR_P_EMPTY + (int)(j % kPBufs)),
                                         (uint32_t)(j / kPBufs - 1) & 1, kWaitNs);
          if (!got) {
            flags[F_ABORT] = 1;
            atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
          }
        }
        float* alpha_w = alpha_s + 64 * (int)(j & 1);
        if (part == 0) alpha_w[h] = alpha;
        if (named_bar_softmax_or(grow || flags[F_ABORT] != 0)) {
          // rare: a stop, or a head's max grew
          if (named_bar_softmax_or(flags[F_ABORT] != 0)) {
            ok = false;
            break;
          }
          // bring O^T (PV of the previous page done) to the new maxima (up or down)
          const bool got =
              tc::mbar_wait(bar(BAR_PV_DONE + (int)((j - 1) & 1)), (uint32_t)((j - 1) >> 1) & 1,
                            kWaitNs);
          if (named_bar_softmax_or(!got)) {
            ok = false;
            break;
          }
          tc::fence_after_sync();
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t r[32];
              const uint32_t ta = tmem + lane_base + kOCol + 64 * blk + 32 * half;
              tc::tmem_ld32(ta, r);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha_w[32 * half + i]);
              tc::tmem_st32(ta, r);
            }
          }
          tc::tmem_wait_st();
        }
        // ---- P = 2^(s - m + 6) as e4m3 hi + e5m2 lo, row h of P^T ----
        {
          const float mu = m == -INFINITY ? 0.f : m - (float)kPOffset;
          uint32_t hw[8], lw[8];
          float rs = 0.f;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            uint32_t hcode[2], lcode[2];
#pragma unroll
            for (int e = 0; e < 2; ++e) {
              const int i = 4 * k + 2 * e;
              const float p0 = fast_exp2(s[i] - mu), p1 = fast_exp2(s[i + 1] - mu);
              const uint32_t hc = e4m3x2_of(p0, p1);
              const float2 hv = e4m3x2_value(hc);
              const uint32_t lc = e5m2x2_of(p0 - hv.x, p1 - hv.y);
              rs += p0 + p1;  // the exact P: lse does not carry the operand rounding
              hcode[e] = hc;
              lcode[e] = lc;
            }
            hw[k] = hcode[0] | (hcode[1] << 16);
            lw[k] = lcode[0] | (lcode[1] << 16);
          }
          rs += __shfl_xor_sync(0xffffffffu, rs, 16);
          l += rs;
          const uint32_t prow = sbase + kOffP + (int)(j % kPBufs) * kPBytes + h * 128;
          const int sw = h & 7;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            const uint32_t ah = prow + (((2 * part + q2) ^ sw) << 4);
            const uint32_t al = prow + (((4 + 2 * part + q2) ^ sw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(ah), "r"(hw[4 * q2]),
                         "r"(hw[4 * q2 + 1]), "r"(hw[4 * q2 + 2]), "r"(hw[4 * q2 + 3]));
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(al), "r"(lw[4 * q2]),
                         "r"(lw[4 * q2 + 1]), "r"(lw[4 * q2 + 2]), "r"(lw[4 * q2 + 3]));
          }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_P_FULL + (int)(j % kPBufs)));
        if (pe) {
          // ---- epilogue: O^T / l -> this piece's partial slot ----
          {
            const bool got = tc::mbar_wait(bar(BAR_O_FULL), (uint32_t)piece & 1, kWaitNs);
            if (named_bar_softmax_or(!got)) {
              ok = false;
              break;
            }
          }
          tc::fence_after_sync();
          const int slot = d.slot;
          if (part == 0) {
            linv_s[h] = l > 0.f ? p.kv_scale / l : 0.f;
            if (h < H)
              p.ws.part_lse[(int64_t)slot * H + h] =
                  l > 0.f ? (m - (float)kPOffset + log2f(l)) * kLn2 : -INFINITY;
          }
          int bad = 0;
          if (t == 0) {
            bad = flags[F_PIECE_BAD];
            flags[F_PIECE_BAD] = 0;
          }
          named_bar_softmax();
          if (t == 0) p.ws.piece_err[slot] = bad;
          float* out = p.ws.part_out + (int64_t)slot * H * kDLatent + t;
          const int nhalf = (H + 31) >> 5;
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
#pragma unroll 1
            for (int half = 0; half < nhalf; ++half) {
              uint32_t r[32];
              tc::tmem_ld32(tmem + lane_base + kOCol + 64 * blk + 32 * half, r);
              tc::tmem_wait_ld();
              float* o = out + (int64_t)(32 * half) * kDLatent + 128 * blk;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (32 * half + i < H)
                  o[(int64_t)i * kDLatent] =
                      (__uint_as_float(r[i]) * linv_s[32 * half + i]);
              }
            }
          }
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(bar(BAR_O_EMPTY));
          m = -INFINITY;
          l = 0.f;
          ++piece;
        }
      }
      if (!ok && t == 0) abort_cta();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kQkWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---- query split: once per (request, draft) row, before the decode kernel ----
// q (bf16) of head h is scaled by 2^shift (max |q| of the head in [2^7, 2^8)) and
// split into q_hi = e4m3(q * 2^shift) and q_lo = e4m3(q * 2^shift - q_hi): exact
// for bf16 inputs down to 2^-10 of the head's max. The codes are written as the
// decode kernel's A operand: row t of A (t < 128) is head 16*(t/32) + t%16, term
// (t/16)%2 (0 = hi, 1 = lo), stored as q_op[row][u][t][16] for the 36 chunks u of
// 16 dims; q_mul[row][h] = score multiplier * 2^-shift. A block handles 8 heads of
// one row, one 16-dim chunk per thread.
constexpr int kSplitHeads = 8;
constexpr int kSplitThreads = kSplitHeads * kQOpChunks;  // 288

__global__ void __launch_bounds__(kSplitThreads)
    q_split_kernel(const __nv_bfloat16* __restrict__ q, int heads, float score_mul,
                   uint8_t* __restrict__ q_op, float* __restrict__ q_mul) {
  // All earlier work in the stream has completed once this returns; the decode
  // kernel that follows may start only after every block has passed it.
  griddep_wait();
  griddep_launch_dependents();
  __shared__ unsigned s_amax[kSplitHeads];
  const int tid = threadIdx.x;
  const int hl = tid / kQOpChunks, u = tid - hl * kQOpChunks;
  const int groups = (heads + kSplitHeads - 1) / kSplitHeads;
  const int64_t row = blockIdx.x / groups;
  const int h = (int)(blockIdx.x - row * groups) * kSplitHeads + hl;
  const bool live = h < heads;
  if (tid < kSplitHeads) s_amax[tid] = 0u;
  uint4 a[2] = {make_uint4(0, 0, 0, 0), make_uint4(0, 0, 0, 0)};
  if (live) {
    const uint4* src = reinterpret_cast<const uint4*>(q + (row * heads + h) * kDEntry) + 2 * u;
    a[0] = __ldg(src);
    a[1] = __ldg(src + 1);
  }
  float f[16];
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const uint32_t ws[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
      f[8 * i + 2 * k] = v.x;
      f[8 * i + 2 * k + 1] = v.y;
    }
  }
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
  __syncthreads();
  atomicMax(&s_amax[hl], __float_as_uint(amax));  // non-negative: integer order = float order
  __syncthreads();
  if (!live) return;
  amax = __uint_as_float(s_amax[hl]);
  int shift = 0;
  if (amax > 0.f && isfinite(amax)) {
    int e;
    frexpf(amax, &e);
    shift = 8 - e;  // scaled max in [2^7, 2^8)
  }
  const float sc = ldexpf(1.0f, shift);
  uint32_t hw[4], lw[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    uint32_t hc[2], lc[2];
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const float x0 = f[4 * k + 2 * e] * sc, x1 = f[4 * k + 2 * e + 1] * sc;
      hc[e] = e4m3x2_of(x0, x1);
      const float2 hv = e4m3x2_value(hc[e]);
      lc[e] = e4m3x2_of(x0 - hv.x, x1 - hv.y);
    }
    hw[k] = hc[0] | (hc[1] << 16);
    lw[k] = lc[0] | (lc[1] << 16);
  }
  const int lane_hi = 32 * (h >> 4) + (h & 15);
  uint4* dst = reinterpret_cast<uint4*>(q_op + row * kQOpRowBytes) + 128 * u;
  dst[lane_hi] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
  dst[lane_hi + 16] = make_uint4(lw[0], lw[1], lw[2], lw[3]);
  if (u == 0) q_mul[row * 64 + h] = score_mul * ldexpf(1.0f, -shift);
}

// ---- grouped decode: the row table of both plans (one warp) ----
// For every (request, draft) row r: row_np1[r] = its shared-prefix pieces (those
// of its group's prefix row, one per worker that the prefix row spans), row_np[r]
// = row_np1[r] + its suffix pieces (-1 for a bad row, which still owns its
// row_np1[r] prefix slots), row_base[r] = the sum of the earlier rows' slots.
__global__ void __launch_bounds__(32) group_plan_kernel(const Fp8Params p) {
  griddep_wait();  // all earlier work in the stream is complete
  griddep_launch_dependents();
  const int lane = threadIdx.x;
  GroupPlan A = group_plan(p, 1), B = group_plan(p, 2);
  A.set_total(plan_total_tiles_warp(A));
  B.set_total(plan_total_tiles_warp(B));
  int64_t rt_carry = 0;
  for (int v0 = 0; v0 < A.rows(); v0 += 32) {
    const int v = v0 + lane;
    const int t = v < A.rows() ? A.row_tiles(v) : 0;
    int64_t incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    const int64_t rt = rt_carry + incl - t;
    if (v < A.rows()) {
      const int np1 = A.row_pieces(rt, t);
      for (int f = 0; f < p.forks; ++f) p.ws.row_np1[A.q_row(v, f)] = np1;
    }
    rt_carry = __shfl_sync(0xffffffffu, rt_carry + incl, 31);
  }
  __syncwarp();
  rt_carry = 0;
  int base_carry = 0;
  for (int r0 = 0; r0 < B.rows(); r0 += 32) {
    const int r = r0 + lane;
    const bool live = r < B.rows();
    const int t = live ? B.row_tiles(r) : 0;
    int64_t incl = t;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int64_t u = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += u;
    }
    const int64_t rt = rt_carry + incl - t;
    // a bad row keeps the slots of its prefix pieces (the prefix pass writes them
    // for every fork of a valid group prefix) but is empty for the merge
    const bool bad = live && B.row_tokens(r) < 0;
    const int np = live ? p.ws.row_np1[r] + B.row_pieces(rt, t) : 0;
    int incl_np = np;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, incl_np, o);
      if (lane >= o) incl_np += u;
    }
    if (live) {
      p.ws.row_base[r] = base_carry + incl_np - np;
      p.ws.row_np[r] = bad ? -1 : np;
      if (bad) atomicOr(p.ws.status, MLA_DEVICE_ERR_BAD_LENGTH);
    }
    rt_carry = __shfl_sync(0xffffffffu, rt_carry + incl, 31);
    base_carry = __shfl_sync(0xffffffffu, base_carry + incl_np, 31);
  }
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeLaunch& d, cudaStream_t stream) {
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel<false>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(decode_fp8_kernel<true>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytesGrouped);
    if (e != cudaSuccess) return e;
    configured[dev].store(1);
  }
  const bool grouped = d.prefix_pages != nullptr;
  static PFN_cuTensorMapEncodeTiled_v12000 encode = nullptr;
  if (encode == nullptr) {
    cudaDriverEntryPointQueryResult qr;
    void* fn = nullptr;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &qr);
    if (e != cudaSuccess || qr != cudaDriverEntryPointSuccess || fn == nullptr)
      return cudaErrorNotSupported;
    encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  // the page pool viewed as [num_pages * 64 rows][576 bytes]; a page is 64 rows
  const int64_t rows = (d.num_pages > 0 ? d.num_pages : 1) * kPageSize;
  const cuuint64_t dims[2] = {(cuuint64_t)kDEntry, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)kDEntry};
  const cuuint32_t box_lat[2] = {128, (cuuint32_t)kPageSize};
  const cuuint32_t box_rope[2] = {(cuuint32_t)kDRope, (cuuint32_t)kPageSize};
  const cuuint32_t estr[2] = {1, 1};
  CUtensorMap lat_map, rope_map;
  void* base = const_cast<uint8_t*>(d.kv);
  CUresult r1 = encode(&lat_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box_lat,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  CUresult r2 = encode(&rope_map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box_rope,
                       estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r1 != CUDA_SUCCESS || r2 != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Fp8Params p;
  p.q = d.q;
  p.num_pages = d.num_pages;
  p.block_table = d.block_table;
  p.max_pages = d.max_pages;
  p.seq_lens = d.seq_lens;
  p.batch = d.batch;
  p.nq = d.nq;
  p.heads = d.heads;
  p.rows = d.batch * d.nq;
  p.score_mul = d.score_mul;
  p.kv_scale = d.kv_scale;
  p.G = d.G;
  p.ws = d.ws;
  p.forks = grouped ? d.forks : 1;
  p.workers = grouped ? d.G / d.forks : 0;
  p.prefix_pages = d.prefix_pages;
  cudaLaunchAttribute attr[1] = {pdl_attribute()};
  if (grouped) {
    cudaLaunchConfig_t gc = {};
    gc.gridDim = dim3(1);
    gc.blockDim = dim3(32);
    gc.stream = stream;
    gc.attrs = attr;
    gc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&gc, group_plan_kernel, p);
    if (e != cudaSuccess) return e;
  }
  {
    const int groups = (d.heads + kSplitHeads - 1) / kSplitHeads;
    cudaLaunchConfig_t sc = {};
    sc.gridDim = dim3((unsigned)((int64_t)d.batch * d.nq * groups));
    sc.blockDim = dim3(kSplitThreads);
    sc.stream = stream;
    sc.attrs = attr;
    sc.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&sc, q_split_kernel, d.q, d.heads, d.score_mul,
                                       d.ws.q_op, d.ws.q_mul);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)d.G);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = grouped ? kSmemBytesGrouped : kSmemBytes;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return grouped ? cudaLaunchKernelEx(&cfg, decode_fp8_kernel<true>, p, lat_map, rope_map)
                 : cudaLaunchKernelEx(&cfg, decode_fp8_kernel<false>, p, lat_map, rope_map);
}

}  // namespace mla
