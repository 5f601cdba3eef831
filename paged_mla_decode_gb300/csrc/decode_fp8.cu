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
// tokens down to about 2^-17 of the page's largest weight). All heads attend over the one latent
// head ("vLLM x AgentX", section "Kimi K3"), so one page serves 64 heads, and V
// is read in place through an MN-major descriptor (no distinct values: "How to
// serve trillions of tokens ...", section "First, understand the workload").
//
// Warp roles (416 threads):
//   warps 0-7  q loading, softmax and epilogue. Row t of A and S is (head
//              16*(t/32) + t%16, part (t/16)%2), part 0 = hi, 1 = lo. Warp w reads
//              TMEM lanes 32*(w%4) .. +31; thread (w, lane) handles head
//              16*(w%4) + lane%16 and the 16 tokens 32*(w/4) + 16*(lane/16) .. +15
//              of a page, both terms (half-split TMEM loads of the hi and lo rows).
//              A head's four threads agree on its page maximum through shared
//              memory at the page's one block barrier. For O^T, lane t is dim t of
//              each 128-dim block and warp w writes heads 32*(w/4) .. +31.
//   warp 8     TMA producer (lane 0): page ids from the block table a window of
//              pages ahead, pages into a ring of kRing shared-memory slots
//              (128-byte swizzled latent blocks, 64-byte swizzled rope block).
//   warps 9-10 issue QK of even / odd pages (lane 0); warp 9 allocates TMEM.
//   warps 11-12 issue PV of even / odd pages (lane 0).
// A thread that issues MMAs stalls for a while after each batch (until the
// tensor pipe's queue has room), so two issuers per contraction keep the pipe
// fed: one issues while the other waits.
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

// Clock-stamp points of the pipeline: nothing unless a tracing build defines
// MLA_STAMP(point, page) to record the SM clock there.
#ifndef MLA_STAMP
#define MLA_STAMP(point, page) ((void)0)
#endif

namespace mla {
namespace {

enum StampPoint {
  kStEntry, kStPrologue, kStTmaIssue, kStQkPage, kStQkIssued, kStSmS, kStSmBar, kStSmP,
  kStPvP, kStPvIssued, kStEpiStart, kStEpiEnd, kStExit, kStQkGo, kStQkMma, kStQkTop
};

constexpr int kSmWarps = 8;                          // softmax / epilogue warps
constexpr int kSmThreads = 32 * kSmWarps;            // 256
constexpr int kTmaWarp = kSmWarps;                   // 8
// MMA issuers: two QK warps and two PV warps, each issuing every other page
// (page k goes to warp k % 2 of its kind), so that one warp's stall after a batch
// of MMAs (an issuing thread waits on its MMA queue) overlaps the other's issue.
constexpr int kQkWarp0 = kSmWarps + 1;               // 9: also allocates TMEM
constexpr int kPvWarp0 = kSmWarps + 3;               // 11
constexpr int kThreads = 32 * (kSmWarps + 5);        // 416
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
constexpr int kOffAlpha = kOffP + kPBufs * kPBytes;         // float [64]
constexpr int kOffLinv = kOffAlpha + 256;                   // float [64]
constexpr int kOffPmax = kOffLinv + 256;                    // float [2 pages][2 halves][64]
constexpr int kOffLsum = kOffPmax + 1024;                   // float [2 halves][64]
constexpr int kOffFlags = kOffLsum + 512;                   // int [4]
constexpr int kOffPlan = kOffFlags + 16;                    // int64 [6]
constexpr int kDescRing = 64;                               // page descriptors in flight
constexpr int kTableAhead = 32;  // pages described (block-table read started) before issue
constexpr int kOffDesc = kOffPlan + 48;                     // PageDesc [kDescRing]
constexpr int kOffBar = kOffDesc + 16 * kDescRing;
constexpr int BAR_PAGE_FULL = 0;                  // [kRing] TMA bytes (or zero fill) landed
// PV(k) completes barrier BAR_PV_DONE + k % kRing (one commit per page): it frees
// page slot k % kRing for the TMA warp, P buffer k % 3 for the softmax warps, and
// marks O^T current for a rescale. Every wait on it names a page whose successor
// on the same barrier (k + kRing) cannot have completed yet, so parities are exact.
constexpr int BAR_PV_DONE = kRing;                // [kRing]
constexpr int BAR_S_FULL = 2 * kRing;             // [2] page j: buffer j % 2
constexpr int BAR_S_EMPTY = BAR_S_FULL + 2;       // [2] (softmax warps)
constexpr int BAR_P_FULL = BAR_S_EMPTY + 2;       // [kPBufs] page j: buffer j % 3 (softmax warps)
constexpr int BAR_O_FULL = BAR_P_FULL + kPBufs;
constexpr int BAR_O_EMPTY = BAR_O_FULL + 1;       // (softmax warps)
constexpr int BAR_Q_READY = BAR_O_EMPTY + 1;      // (softmax warps)
constexpr int BAR_Q_EMPTY = BAR_Q_READY + 1;
constexpr int BAR_DRAIN = BAR_Q_EMPTY + 1;       // [4] one per issuer warp
#ifdef MLA_TEST_STALL_QK
// Test build only: a barrier that nothing ever completes. The MMA issuer waits on
// it before the QK of its third page, so the wait runs out and the CTA takes the
// timeout path (stop every role, drain the copies and MMAs in flight, free TMEM).
constexpr int BAR_TEST_STALL = BAR_DRAIN + 4;
constexpr int kNumBars = BAR_TEST_STALL + 1;
#else
constexpr int kNumBars = BAR_DRAIN + 4;
#endif
// arrivals that complete a phase of barrier i
__device__ __forceinline__ uint32_t bar_count(int i) {
  if ((i >= BAR_S_EMPTY && i < BAR_S_EMPTY + 2) || (i >= BAR_P_FULL && i < BAR_P_FULL + kPBufs) ||
      i == BAR_O_EMPTY || i == BAR_Q_READY)
    return kSmWarps;
  if (i == BAR_Q_EMPTY || i == BAR_O_FULL) return 2;  // both issuer warps of the kind commit
  return 1;
}
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024 alignment
// grouped decode: the two segments' plans (int64 [32]) after the common map
constexpr int kOffPlanX = (kSmemUsed + 15) & ~15;
constexpr int kSmemBytesGrouped = kOffPlanX + 256 + 1024;
static_assert(kSmemBytesGrouped <= 227 * 1024, "shared memory map exceeds 227 KB");

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
  asm volatile("bar.sync 1, %0;\n" ::"n"(kSmThreads) : "memory");
}
__device__ __forceinline__ bool named_bar_softmax_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, %2, p;\n"
      " selp.u32 %0, 1, 0, q;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)pred), "n"(kSmThreads)
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
  float* pmax_s = reinterpret_cast<float*>(smem + kOffPmax);
  float* lsum_s = reinterpret_cast<float*>(smem + kOffLsum);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
  int64_t* s_plan = reinterpret_cast<int64_t*>(smem + kOffPlan);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (tid == 0) MLA_STAMP(kStEntry, 0);

  // ---- planning (shared by all roles) ----
  // This kernel starts once the query split kernel before it has passed its own
  // wait for all earlier work in the stream (see launch_decode_fp8), so the
  // lengths, block table and pages may be read at once; only the split query
  // itself needs the split kernel to have completed (griddep_wait before q_op).
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
  if (warp == kTmaWarp && lane == 0) {
    tc::prefetch_tensormap(&lat_map);
    tc::prefetch_tensormap(&rope_map);
    for (int i = 0; i < kNumBars; ++i) tc::mbar_init(bar(i), bar_count(i));
    tc::fence_mbar_init();
    flags[F_ABORT] = 0;
    flags[F_PIECE_BAD] = 0;
  }
  if (warp == kQkWarp0) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  griddep_launch_dependents();  // the combine kernel may be scheduled (it waits for this grid)
  if (tid == 0) MLA_STAMP(kStPrologue, 0);
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
  // This CTA's walk over its pages (the TMA lane describes each page from it; the
  // MMA issuers follow their own copy for the piece boundaries, in registers).
  using Walker = std::conditional_t<kGrouped, SegWalker, PageWalker<Plan>>;
  auto start_walker = [&](Walker& pw) {
    if constexpr (kGrouped) {
      GroupPlan A = group_plan(p, 1), B = group_plan(p, 2);
      A.set_total(s_plan_x[0]);
      B.set_total(s_plan_x[1]);
      const RowCursor ca{(int)s_plan_x[8], s_plan_x[9], (int)s_plan_x[10], (int)s_plan_x[11],
                         (int)s_plan_x[12]};
      const RowCursor cb{(int)s_plan_x[13], s_plan_x[14], (int)s_plan_x[15], (int)s_plan_x[16],
                         (int)s_plan_x[17]};
      pw.start(A, ca, s_plan_x[2], s_plan_x[3], (int)s_plan_x[6], (int)s_plan_x[7], B, cb,
               s_plan_x[4], s_plan_x[5], c, p.ws.row_base, p.ws.row_np1);
    } else {
      pw.init(plan, cur0, c, x_begin, x_end);
    }
  };
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
        Walker pw;
        start_walker(pw);
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
              (!tc::mbar_wait(bar(BAR_PV_DONE + slot), (round - 1) & 1, kWaitNs) ||
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
            MLA_STAMP(kStTmaIssue, j);
          } else {
            // bad id: no copy; every token of the page is masked and the softmax
            // warps zero its value rows before PV reads them
            tc::mbar_arrive(bar(BAR_PAGE_FULL + slot));
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
    } else if (warp >= kQkWarp0) {
      // ============ MMA issuers: two QK warps, two PV warps; lane 0 issues ============
      // Page k's QK is issued by QK warp k % 2 (into S buffer k % 2, which is that
      // warp's own) and its PV by PV warp k % 2. MMAs of different threads complete
      // in no particular order relative to each other, so every wait names the page
      // it needs (PV_DONE per page) and the once-per-piece barriers count both warps
      // of a kind: each passes every piece start (QK: the piece's q is loaded; PV:
      // O^T is zero) and commits at every piece end (Q_EMPTY, O_FULL), whether or not
      // it issued a page of that piece. PV always accumulates: the softmax warps zero
      // O^T before a piece starts. A PV issues its e4m3 (hi) MMAs before its e5m2
      // (lo) ones: MMAs that alternate B formats run at half rate.
      constexpr uint32_t id_qk = tc::idesc_f8(128, 64, tc::kFmtE4M3, tc::kFmtE4M3, false, false);
      // PV: A = V^T (e4m3, MN-major); B = P^T hi (e4m3) or lo (e5m2), K-major
      constexpr uint32_t id_pv_hi = tc::idesc_f8(128, 64, tc::kFmtE4M3, tc::kFmtE4M3, true, false);
      constexpr uint32_t id_pv_lo = tc::idesc_f8(128, 64, tc::kFmtE4M3, tc::kFmtE5M2, true, false);
      const bool is_qk = warp < kPvWarp0;
      const int mine = warp - (is_qk ? kQkWarp0 : kPvWarp0);  // pages k with k % 2 == mine
      // Only lane 0 runs the issue loop: MMA issue stalls while the tensor pipe's
      // queue is full, so any other work between batches (warp votes, shuffles,
      // warp barriers) leaves the pipe idle.
      if (lane == 0) {
        auto wait = [&](int b, uint32_t parity) -> bool {
          return tc::mbar_wait(bar(b), parity, kWaitNs);
        };
        const uint64_t qrope_desc = tc::smem_desc(sbase + kOffQRope, 16, 512, tc::kSwizzle64);
        int piece_n = 0;
        bool ok = true;
        Walker pw;  // piece boundaries without reading the shared descriptors
        start_walker(pw);
        for (int64_t k = 0; k < npages && ok; ++k, pw.next()) {
          // (another role's stop is seen here every 8 pages, or as a wait that runs out)
          if ((k & 7) == 0 && flags[F_ABORT]) {
            ok = false;
            break;
          }
          const bool ps = pw.piece_start(), pe = pw.piece_end();
          if (ps) {
            ok = wait(is_qk ? BAR_Q_READY : BAR_O_EMPTY, (uint32_t)piece_n & 1);
            ++piece_n;
            if (!ok) break;
          }
          if ((int)(k & 1) == mine) {
            const int slot = (int)(k % kRing);
            const uint32_t page_base = sbase + kOffPages + slot * kPageBytes;
            if (is_qk) {
              // ---- S(k) = A . page(k)^T: latent part of A from TMEM, rope from shared memory ----
#ifdef MLA_TEST_STALL_QK
              if (k == 2 && !wait(BAR_TEST_STALL, 0)) {
                ok = false;
                break;
              }
#endif
              MLA_STAMP(kStQkTop, k);
              ok = wait(BAR_PAGE_FULL + slot, (uint32_t)(k / kRing) & 1);
              MLA_STAMP(kStQkPage, k);
              // S buffer k % 2 last held S(k - 2), issued by this warp
              if (ok && k >= 2) ok = wait(BAR_S_EMPTY + (int)(k & 1), (uint32_t)((k >> 1) - 1) & 1);
              if (!ok) break;
              MLA_STAMP(kStQkGo, k);
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
              MLA_STAMP(kStQkMma, k);
              tc::mma_commit(bar(BAR_S_FULL + (int)(k & 1)));
              MLA_STAMP(kStQkIssued, k);
            } else {
              // ---- O^T += V^T P^T (V read in place through an MN-major descriptor) ----
              const int pb_i = (int)(k % kPBufs);
              ok = wait(BAR_P_FULL + pb_i, (uint32_t)(k / kPBufs) & 1);
              if (!ok) break;
              MLA_STAMP(kStPvP, k);
              tc::fence_after_sync();
              const uint64_t va = tc::smem_desc(page_base, kLatBlock, 1024, tc::kSwizzle128);
              const uint64_t pb =
                  tc::smem_desc(sbase + kOffP + pb_i * kPBytes, 16, 1024, tc::kSwizzle128);
#pragma unroll
              for (int part = 0; part < 2; ++part)
#pragma unroll
                for (int blk = 0; blk < 4; ++blk)
#pragma unroll
                  for (int s = 0; s < 2; ++s)
                    tc::mma_f8_ss(tmem + kOCol + 64 * blk,
                                  va + (uint64_t)((blk * kLatBlock + s * 4096) >> 4),
                                  pb + (uint64_t)((64 * part + 32 * s) >> 4),
                                  part ? id_pv_lo : id_pv_hi, 1);
              tc::mma_commit(bar(BAR_PV_DONE + slot));
              MLA_STAMP(kStPvIssued, k);
            }
          }
          if (pe) tc::mma_commit(bar(is_qk ? BAR_Q_EMPTY : BAR_O_FULL));
        }
        if (!ok) abort_cta();
        // drain: every MMA this thread issued has finished before TMEM is freed
        const int db = BAR_DRAIN + (warp - kQkWarp0);
        tc::mma_commit(bar(db));
        if (!tc::mbar_wait(bar(db), 0, kDrainWaitNs)) atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
      }
      __syncwarp();
    } else {
      // =================== softmax + epilogue (warps 0-7) ===================
      // Warp w reads TMEM lanes 32*(w%4) .. +31 (rows of A and S; dims of O^T) and
      // handles half g = w/4 of each page: thread (w, lane) owns head
      // h = 16*(w%4) + lane%16 and the 16 tokens 32*g + 16*(lane/16) .. +15, both
      // q terms of each (a half-split TMEM load of the hi rows and of the lo rows).
      // A head's four threads agree on its running maximum through shared memory
      // at the one block barrier of each page; each keeps its own part of the sum.
      const int t = tid;
      const int q4 = warp & 3, g = warp >> 2;
      const int h = 16 * q4 + (lane & 15);
      const int c16 = 2 * g + (lane >> 4);      // this thread's 16-token chunk of a page
      const uint32_t lane_hi = (uint32_t)(32 * q4) << 16;
      const uint32_t lane_lo = (uint32_t)(32 * q4 + 16) << 16;
      float m = -INFINITY, lpart = 0.f, qmul = 0.f;
      int piece = 0;
      bool ok = true;
      {
        // O^T starts at zero (PV always accumulates); this warp's lanes, heads 32g ..
        uint32_t zz[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) zz[i] = 0u;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) tc::tmem_st32(tmem + lane_hi + kOCol + 64 * blk + 32 * g, zz);
        tc::tmem_wait_st();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_O_EMPTY));
      }
      for (int64_t j = 0; j < npages; ++j) {
        // Page 0 opens the first piece, whose row the plan gives: its q is staged at
        // once. Later pages' descriptors are read once the page has landed.
        int row = cur0.r;
        bool ps = j == 0;
        // (a failed wait is acted on at this page's block barrier below; every
        // thread reads the same descriptor word, so the piece-start decision, and
        // with it the barriers of the q staging, is uniform either way)
        if (!tc::mbar_wait(bar(BAR_PAGE_FULL + (int)(j % kRing)), (uint32_t)(j / kRing) & 1,
                           kWaitNs))
          flags[F_ABORT] = 1;
        if (j > 0) {
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
          // [16 codes]: TMEM lane r = 32*(w%4) + lane gets its 32 latent chunks (half
          // g loads chunks 16g .. 16g+15) and its shared-memory row the 4 rope chunks
          // (half g: 32 + 2g, 33 + 2g), 64-byte swizzled.
          griddep_wait();  // the split kernel has completed and its writes are visible
          const bool live = h < H;
          qmul = live ? __ldcg(p.ws.q_mul + (int64_t)row * 64 + h) : 0.f;
          const int r = 32 * q4 + lane;
          const uint4* src =
              reinterpret_cast<const uint4*>(p.ws.q_op + (int64_t)row * kQOpRowBytes) + r;
          uint4 qc[18];
#pragma unroll
          for (int u = 0; u < 16; ++u)
            qc[u] = live ? __ldcg(src + 128 * (16 * g + u)) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int u = 0; u < 2; ++u)
            qc[16 + u] = live ? __ldcg(src + 128 * (32 + 2 * g + u)) : make_uint4(0, 0, 0, 0);
#pragma unroll
          for (int gg = 0; gg < 2; ++gg) {
            uint32_t v[32];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
              v[4 * k] = qc[8 * gg + k].x;
              v[4 * k + 1] = qc[8 * gg + k].y;
              v[4 * k + 2] = qc[8 * gg + k].z;
              v[4 * k + 3] = qc[8 * gg + k].w;
            }
            tc::tmem_st32(tmem + lane_hi + kQCol + 64 * g + 32 * gg, v);
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int c4 = 2 * g + u;
            const uint32_t a = sbase + kOffQRope + r * 64 + ((c4 ^ ((r >> 1) & 3)) << 4);
            const uint4 v = qc[16 + u];
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
        // block barrier below: one barrier per page)
        if (!tc::mbar_wait(bar(BAR_S_FULL + (int)(j & 1)), (uint32_t)(j >> 1) & 1, kWaitNs))
          flags[F_ABORT] = 1;
        if (t == 0) MLA_STAMP(kStSmS, j);
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
        uint32_t shi[16], slo[16];
        const uint32_t scol = s_col((int)(j & 1)) + 32u * (uint32_t)g;
        tc::tmem_ld16x2_16(tmem + lane_hi + scol, shi);
        tc::tmem_ld16x2_16(tmem + lane_lo + scol, slo);
        tc::tmem_wait_ld();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_S_EMPTY + (int)(j & 1)));
        float s[16];
        float tm = -INFINITY;
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const bool vis = 16 * c16 + i < nvis;
          s[i] = vis ? (__uint_as_float(shi[i]) + __uint_as_float(slo[i])) * qmul : -INFINITY;
          tm = fmaxf(tm, s[i]);
        }
        tm = fmaxf(tm, __shfl_xor_sync(0xffffffffu, tm, 16));
        if (lane < 16) pmax_s[(int)(j & 1) * 128 + g * 64 + h] = tm;
        // P buffer j % 3 was read by PV(j - 3); waiting for it also makes the
        // PV_DONE parity of the rescale below unambiguous (PV(j - 3) is complete)
        if (j >= kPBufs && !flags[F_ABORT]) {
          const int64_t jp = j - kPBufs;  // the page whose PV read this P buffer
          const bool got = tc::mbar_wait(bar(BAR_PV_DONE + (int)(jp % kRing)),
                                         (uint32_t)(jp / kRing) & 1, kWaitNs);
          if (!got) {
            flags[F_ABORT] = 1;
            atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
          }
        }
        // lazy running max: O is rescaled only when a head's page max rises more than
        // kRescaleThresh above it or falls more than kLowThresh below it; a half
        // page's max outside that band asks every thread to look closer
        const bool trig = !ps && (tm > m + kRescaleThresh || tm < m - kLowThresh);
        const bool any = named_bar_softmax_or(trig || flags[F_ABORT] != 0);
        if (t == 0) MLA_STAMP(kStSmBar, j);
        const float tmax = fmaxf(tm, pmax_s[(int)(j & 1) * 128 + (1 - g) * 64 + h]);
        if (any && named_bar_softmax_or(flags[F_ABORT] != 0)) {
          ok = false;
          break;
        }
        if (ps) {
          m = tmax;
        } else if (any) {
          // rare: the exact decision per head, with the head's whole sum
          const float lh = lpart + __shfl_xor_sync(0xffffffffu, lpart, 16);
          if (lane < 16) lsum_s[g * 64 + h] = lh;
          named_bar_softmax();
          const float lhead = lsum_s[h] + lsum_s[64 + h];
          float alpha = 1.f;
          bool grow = false;
          if (tmax > m + kRescaleThresh) {
            alpha = m == -INFINITY ? 0.f : fast_exp2(m - tmax);
            grow = true;
          } else if (tmax < m - kLowThresh && lhead * fast_exp2(m - tmax) <= kMassCap) {
            alpha = fast_exp2(m - tmax);  // > 1: the page is far below the running max
            grow = true;
          }
          if (grow) {
            m = tmax;
            lpart *= alpha;
          }
          if (g == 0 && lane < 16) alpha_s[h] = alpha;
          if (named_bar_softmax_or(grow)) {
            // bring O^T (PVs of the previous two pages done: they come from the two PV
            // warps) to the new maxima (up or down)
            bool got = tc::mbar_wait(bar(BAR_PV_DONE + (int)((j - 1) % kRing)),
                                     (uint32_t)((j - 1) / kRing) & 1, kWaitNs);
            if (got && j >= 2)
              got = tc::mbar_wait(bar(BAR_PV_DONE + (int)((j - 2) % kRing)),
                                  (uint32_t)((j - 2) / kRing) & 1, kWaitNs);
            if (named_bar_softmax_or(!got)) {
              ok = false;
              break;
            }
            tc::fence_after_sync();
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
              uint32_t rr[32];
              const uint32_t ta = tmem + lane_hi + kOCol + 64 * blk + 32 * g;
              tc::tmem_ld32(ta, rr);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                rr[i] = __float_as_uint(__uint_as_float(rr[i]) * alpha_s[32 * g + i]);
              tc::tmem_st32(ta, rr);
            }
            tc::tmem_wait_st();
          }
        }
        // ---- P = 2^(s - m + 6) as e4m3 hi + e5m2 lo, this thread's 16 tokens of row h of P^T ----
        {
          const float mu = m == -INFINITY ? 0.f : m - (float)kPOffset;
          uint32_t hw[4], lw[4];
          float rs = 0.f;
#pragma unroll
          for (int k = 0; k < 4; ++k) {
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
          lpart += rs;
          const uint32_t prow = sbase + kOffP + (int)(j % kPBufs) * kPBytes + h * 128;
          const int sw = h & 7;
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + ((c16 ^ sw) << 4)),
                       "r"(hw[0]), "r"(hw[1]), "r"(hw[2]), "r"(hw[3]));
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(prow + (((4 + c16) ^ sw) << 4)),
                       "r"(lw[0]), "r"(lw[1]), "r"(lw[2]), "r"(lw[3]));
        }
        if (nvis < kPageSize) {
          // value rows past the page's last token (all rows of a bad page id) become
          // zeros before PV reads them: their weights are 0, and 0 times a stale
          // NaN code would poison O (QK(j) has already read the page)
          const uint32_t page_base = sbase + kOffPages + (int)(j % kRing) * kPageBytes;
          for (int i = t; i < (kPageSize - nvis) * 32; i += kSmThreads) {
            const int rrow = nvis + (i >> 5), u = i & 31;
            asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};\n" ::"r"(
                             page_base + (u >> 3) * kLatBlock + rrow * 128 + (u & 7) * 16),
                         "r"(0u));
          }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_P_FULL + (int)(j % kPBufs)));
        if (t == 0) MLA_STAMP(kStSmP, j);
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
          if (t == 0) MLA_STAMP(kStEpiStart, piece);
          const int slot = d.slot;
          const float lh = lpart + __shfl_xor_sync(0xffffffffu, lpart, 16);
          if (lane < 16) lsum_s[g * 64 + h] = lh;
          int bad = 0;
          if (t == 0) {
            bad = flags[F_PIECE_BAD];
            flags[F_PIECE_BAD] = 0;
          }
          named_bar_softmax();
          if (g == 0 && lane < 16) {
            const float l = lsum_s[h] + lsum_s[64 + h];
            linv_s[h] = l > 0.f ? p.kv_scale / l : 0.f;
            if (h < H)
              p.ws.part_lse[(int64_t)slot * H + h] =
                  l > 0.f ? (m - (float)kPOffset + log2f(l)) * kLn2 : -INFINITY;
          }
          if (t == 0) p.ws.piece_err[slot] = bad;
          named_bar_softmax();
          // O^T lane = dim 128*blk + 32*(w%4) + lane; this warp writes heads 32g .. 32g+31
          if (32 * g < H) {
            float* out = p.ws.part_out + (int64_t)slot * H * kDLatent + 32 * q4 + lane;
#pragma unroll 1
            for (int blk = 0; blk < 4; ++blk) {
              uint32_t rr[32];
              tc::tmem_ld32(tmem + lane_hi + kOCol + 64 * blk + 32 * g, rr);
              tc::tmem_wait_ld();
              float* o = out + (int64_t)(32 * g) * kDLatent + 128 * blk;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (32 * g + i < H)
                  o[(int64_t)i * kDLatent] = __uint_as_float(rr[i]) * linv_s[32 * g + i];
              }
            }
          }
          if (j + 1 < npages) {
            // O^T back to zero for the next piece
            uint32_t zz[32];
#pragma unroll
            for (int i = 0; i < 32; ++i) zz[i] = 0u;
#pragma unroll
            for (int blk = 0; blk < 4; ++blk)
              tc::tmem_st32(tmem + lane_hi + kOCol + 64 * blk + 32 * g, zz);
            tc::tmem_wait_st();
          }
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(bar(BAR_O_EMPTY));
          if (t == 0) MLA_STAMP(kStEpiEnd, piece);
          m = -INFINITY;
          lpart = 0.f;
          ++piece;
        }
      }
      if (!ok && t == 0) abort_cta();
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == kQkWarp0) tc::tmem_dealloc(tmem, kTmemCols);
  if (tid == 0) MLA_STAMP(kStExit, 0);
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
