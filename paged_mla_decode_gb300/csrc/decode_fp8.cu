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
// q (bf16) is scaled per head by a power of two and split into two e4m3 terms
// q_hi + q_lo, which is exact for bf16 inputs (8 significant bits = 4 + 4), so
// S_hi + S_lo is q . k up to fp32 accumulation. P = 2^(s - m + 7) is split the
// same way (8 significant bits, as bf16). All heads attend over the one latent
// head ("vLLM x AgentX", section "Kimi K3"), so one page serves 64 heads, and V
// is read in place through an MN-major descriptor (no distinct values: "How to
// serve trillions of tokens ...", section "First, understand the workload").
//
// Warp roles (192 threads):
//   warps 0-3  q staging, softmax and epilogue. Thread t owns TMEM lane t: row t
//              of A and S is (head 16*(t/32) + t%16, part (t/16)%2), part 0 = hi,
//              1 = lo, so the two terms of a head meet inside one warp; for O^T
//              lane t is dim t of each 128-dim block.
//   warp 4     TMA producer: pages into a ring of kRing shared-memory slots
//              (128-byte swizzled latent blocks, 64-byte swizzled rope block).
//   warp 5     TMEM allocation and the thread that issues every tcgen05.mma; the
//              warp zeroes the rows of a partial page past its last token first.
// TMEM (512 columns): A latent part [0,128), S buffers [128,192) [192,256),
// O^T [256,512). The rope part of A is in shared memory.
//
// Every wait is bounded (2 s); on timeout the CTA records MLA_DEVICE_ERR_TIMEOUT,
// stops, drains its MMAs and copies (bounded) and frees TMEM.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kThreads = 192;
constexpr int kTmaWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kRing = 5;                             // pages in flight
constexpr int kPageBytes = kPageSize * kDEntry;      // 36864
constexpr int kLatBlock = kPageSize * 128;           // 8192: 64 rows x 128 dims
constexpr int kRopeOff = 4 * kLatBlock;              // rope block within a page slot
constexpr int kPBytes = 64 * 128;                    // P^T: 64 heads x [64 hi | 64 lo]
constexpr int kPOffset = 7;                          // P = 2^(s - m + 7)
constexpr float kRescaleThresh = 1.5f;               // P <= 2^8.5 < 448 (e4m3 max)
constexpr uint64_t kWaitNs = 2000000000ull;

constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kQCol = 0;
__device__ __forceinline__ uint32_t s_col(int b) { return 128u + 64u * (uint32_t)b; }
constexpr uint32_t kOCol = 256;

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffPages = 0;
constexpr int kOffQRope = kOffPages + kRing * kPageBytes;   // 128 rows x 64 B, 64B swizzle
constexpr int kOffP = kOffQRope + 128 * 64;                 // [2] P^T buffers
constexpr int kOffAlpha = kOffP + 2 * kPBytes;              // float [2][64]
constexpr int kOffLinv = kOffAlpha + 512;                   // float [64]
constexpr int kOffFlags = kOffLinv + 256;                   // int [4]
constexpr int kOffPlan = kOffFlags + 16;                    // int64 [6]
constexpr int kOffBar = kOffPlan + 48;
constexpr int BAR_PAGE_FULL = 0;              // [kRing] TMA bytes (or zero fill) landed
constexpr int BAR_PAGE_EMPTY = kRing;         // [kRing] PV of the slot's page finished
constexpr int BAR_S_FULL = 2 * kRing;         // [2]
constexpr int BAR_S_EMPTY = 2 * kRing + 2;    // [2] (4 softmax warps)
constexpr int BAR_P_FULL = 2 * kRing + 4;     // [2] (4 softmax warps)
constexpr int BAR_PV_DONE = 2 * kRing + 6;    // one phase per PV
constexpr int BAR_O_FULL = 2 * kRing + 7;
constexpr int BAR_O_EMPTY = 2 * kRing + 8;    // (4 softmax warps)
constexpr int BAR_Q_READY = 2 * kRing + 9;    // (4 softmax warps)
constexpr int BAR_Q_EMPTY = 2 * kRing + 10;
constexpr int BAR_DRAIN = 2 * kRing + 11;
constexpr int kNumBars = 2 * kRing + 12;
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;  // slack for the 1024 alignment

enum Flag { F_ABORT = 0, F_PIECE_BAD = 1 };

struct Fp8Params {
  const __nv_bfloat16* q;
  int64_t num_pages;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int batch, nq, heads;
  float score_mul;   // sm_scale * log2(e) * kv_scale
  float kv_scale;
  int G;
  DecodeWorkspace ws;
};

// Cursor over a CTA's pages (one page per step).
struct PageWalker {
  Plan plan;
  RowCursor cur;
  int64_t x, x_end, x_begin;

  __device__ void init(const Plan& p, const RowCursor& c, int64_t xb, int64_t xe) {
    plan = p; cur = c; x = xb; x_begin = xb; x_end = xe;
    settle();
  }
  __device__ void settle() {
    if (x < x_end && x == cur.rt + cur.t) cursor_next_row(plan, cur);
  }
  __device__ bool done() const { return x >= x_end; }
  __device__ int page_in_row() const { return (int)(x - cur.rt); }
  __device__ bool piece_start() const { return x == x_begin || x == cur.rt; }
  __device__ bool piece_end() const { return x + 1 == x_end || x + 1 == cur.rt + cur.t; }
  __device__ int valid_tokens() const { return min(kPageSize, cur.n - page_in_row() * kPageSize); }
  __device__ int page_id(const int32_t* block_table, int nq, int max_pages) const {
    return __ldg(block_table + (int64_t)(cur.r / nq) * max_pages + page_in_row());
  }
  __device__ void next() { ++x; settle(); }
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
// hi/lo split of a pair: hi = e4m3(x), lo = e4m3(x - hi); returns the codes of
// the requested term and (optionally) the represented value hi + lo.
__device__ __forceinline__ uint32_t split_pair(float x0, float x1, bool want_lo, float2* value) {
  const uint32_t hi = e4m3x2_of(x0, x1);
  const float2 hv = e4m3x2_value(hi);
  const uint32_t lo = e4m3x2_of(x0 - hv.x, x1 - hv.y);
  if (value) {
    const float2 lv = e4m3x2_value(lo);
    *value = make_float2(hv.x + lv.x, hv.y + lv.y);
  }
  return want_lo ? lo : hi;
}

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
  Plan plan{p.seq_lens, p.batch, p.nq, p.max_pages, kPageSize, p.G, 0};
  if (warp == 0) {
    const int64_t T = plan_total_tiles_warp(plan);
    if (lane == 0) s_plan[0] = T;
  }
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      const bool by_warps = i == BAR_S_EMPTY || i == BAR_S_EMPTY + 1 || i == BAR_P_FULL ||
                            i == BAR_P_FULL + 1 || i == BAR_O_EMPTY || i == BAR_Q_READY;
      tc::mbar_init(bar(i), by_warps ? 4 : 1);
    }
    tc::fence_mbar_init();
    flags[F_ABORT] = 0;
    flags[F_PIECE_BAD] = 0;
  }
  if (warp == kMmaWarp) {
    tc::tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tc::tmem_relinquish();
  }
  __syncthreads();
  plan.set_total(s_plan[0]);
  const int c = blockIdx.x;
  const bool works = c < plan.G;
  const int64_t x_begin = works ? plan.cta_start(c) : 0;
  const int64_t x_end = works ? plan.cta_start(c + 1) : 0;
  if (warp == 0) {
    RowCursor f = plan_find_row_warp(plan, x_begin, c == 0, p.ws.row_base, p.ws.row_np,
                                     p.ws.status);
    if (lane == 0) {
      s_plan[1] = f.r;
      s_plan[2] = f.rt;
      s_plan[3] = f.t;
      s_plan[4] = f.base;
      s_plan[5] = f.n;
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  const RowCursor cur0{(int)s_plan[1], s_plan[2], (int)s_plan[3], (int)s_plan[4],
                       (int)s_plan[5]};
  const int H = p.heads;
  auto abort_cta = [&]() {
    flags[F_ABORT] = 1;
    atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
  };

  if (x_begin < x_end) {
    if (warp == kTmaWarp) {
      // =================== TMA producer (lane 0) ===================
      if (lane == 0) {
        const uint64_t pol = l2_evict_first_policy();
        PageWalker pw;
        pw.init(plan, cur0, x_begin, x_end);
        int64_t j = 0;
        bool ok = true;
        for (; !pw.done(); pw.next(), ++j) {
          const int slot = (int)(j % kRing);
          const uint32_t round = (uint32_t)(j / kRing);
          const uint32_t page_base = sbase + kOffPages + slot * kPageBytes;
          if (j >= kRing &&
              (!tc::mbar_wait(bar(BAR_PAGE_EMPTY + slot), (round - 1) & 1, kWaitNs) ||
               flags[F_ABORT])) {
            ok = false;
            break;
          }
          const int page = pw.page_id(p.block_table, p.nq, p.max_pages);
          if (page >= 0 && (int64_t)page < p.num_pages) {
            tc::mbar_arrive_expect_tx(bar(BAR_PAGE_FULL + slot), (uint32_t)kPageBytes);
            const int y = page * kPageSize;
#pragma unroll
            for (int b = 0; b < 4; ++b)
              tc::tma_load_2d_hint(page_base + b * kLatBlock, &lat_map, 128 * b, y,
                                   bar(BAR_PAGE_FULL + slot), pol);
            tc::tma_load_2d_hint(page_base + kRopeOff, &rope_map, kDLatent, y,
                                 bar(BAR_PAGE_FULL + slot), pol);
          } else {
            tc::mbar_arrive(bar(BAR_PAGE_FULL + slot));  // bad id: the MMA warp zero-fills
          }
        }
        if (!ok) abort_cta();
        // no copy may land after the CTA exits: wait for the last issued pages
        for (int64_t jj = j > kRing ? j - kRing : 0; jj < j; ++jj)
          tc::mbar_wait(bar(BAR_PAGE_FULL + (int)(jj % kRing)), (uint32_t)(jj / kRing) & 1,
                        kWaitNs);
      }
      __syncwarp();
    } else if (warp == kMmaWarp) {
      // =================== MMA issuer (lane 0; the warp zero-fills) ===================
      constexpr uint32_t id_qk = tc::idesc_f16(128, 64, false, false, false);
      constexpr uint32_t id_pv = tc::idesc_f16(128, 64, false, true, false);
      const uint64_t qrope_desc = tc::smem_desc(sbase + kOffQRope, 16, 512, tc::kSwizzle64);
      const bool leader = lane == 0;
      // bounded wait by lane 0, result shared with the warp
      auto wait0 = [&](int b, uint32_t parity) -> bool {
        bool got = true;
        if (leader) got = tc::mbar_wait(bar(b), parity, kWaitNs);
        return __shfl_sync(0xffffffffu, got ? 1 : 0, 0) != 0;
      };
      bool ok = true;
      int q_piece = 0, o_piece = 0;
      struct Prev { int64_t j; int slot; bool ps, pe; } prev{0, 0, false, false};
      bool have_prev = false;
      auto pv = [&](const Prev& pr) -> bool {
        if (!wait0(BAR_P_FULL + (int)(pr.j & 1), (uint32_t)(pr.j >> 1) & 1)) return false;
        if (pr.ps) {
          if (o_piece > 0 && !wait0(BAR_O_EMPTY, (uint32_t)(o_piece - 1) & 1)) return false;
          ++o_piece;
        }
        if (leader) {
          tc::fence_after_sync();
          const uint32_t page_base = sbase + kOffPages + pr.slot * kPageBytes;
          const uint64_t va = tc::smem_desc(page_base, kLatBlock, 1024, tc::kSwizzle128);
          const uint64_t pb =
              tc::smem_desc(sbase + kOffP + (int)(pr.j & 1) * kPBytes, 16, 1024, tc::kSwizzle128);
#pragma unroll
          for (int blk = 0; blk < 4; ++blk)
#pragma unroll
            for (int s = 0; s < 2; ++s)
#pragma unroll
              for (int part = 0; part < 2; ++part)
                tc::mma_f8_ss(tmem + kOCol + 64 * blk,
                              va + (uint64_t)((blk * kLatBlock + s * 4096) >> 4),
                              pb + (uint64_t)((64 * part + 32 * s) >> 4), id_pv,
                              !(pr.ps && s == 0 && part == 0));
          tc::mma_commit(bar(BAR_PAGE_EMPTY + pr.slot));
          tc::mma_commit(bar(BAR_PV_DONE));
          if (pr.pe) tc::mma_commit(bar(BAR_O_FULL));
        }
        __syncwarp();
        return true;
      };
      PageWalker pw;
      pw.init(plan, cur0, x_begin, x_end);
      for (int64_t j = 0; !pw.done() && ok; pw.next(), ++j) {
        if (flags[F_ABORT]) {
          ok = false;
          break;
        }
        const bool ps = pw.piece_start(), pe = pw.piece_end();
        const int slot = (int)(j % kRing);
        const uint32_t page_base = sbase + kOffPages + slot * kPageBytes;
        // a piece's first QK needs its q, staged after the previous piece's output
        if (ps && have_prev) {
          ok = pv(prev);
          have_prev = false;
          if (!ok) break;
        }
        if (ps) {
          ok = wait0(BAR_Q_READY, (uint32_t)q_piece & 1);
          ++q_piece;
          if (!ok) break;
        }
        ok = wait0(BAR_PAGE_FULL + slot, (uint32_t)(j / kRing) & 1);
        if (ok && j >= 2) ok = wait0(BAR_S_EMPTY + (int)(j & 1), (uint32_t)((j >> 1) - 1) & 1);
        if (!ok) break;
        // rows past the page's last token (all rows of a bad page id) become zeros,
        // so that masked tokens contribute 0 * finite to PV
        const int page = pw.page_id(p.block_table, p.nq, p.max_pages);
        const bool page_ok = page >= 0 && (int64_t)page < p.num_pages;
        const int zero_from = page_ok ? pw.valid_tokens() : 0;
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
          tc::fence_after_sync();
          // ---- S = A . page^T: latent part of A from TMEM, rope part from shared memory ----
          const uint64_t kb = tc::smem_desc(page_base, 16, 1024, tc::kSwizzle128);
          const uint64_t rb = tc::smem_desc(page_base + kRopeOff, 16, 512, tc::kSwizzle64);
          const uint32_t d_s = tmem + s_col((int)(j & 1));
#pragma unroll
          for (int s = 0; s < 16; ++s)
            tc::mma_f8_ts(d_s, tmem + kQCol + 8 * s,
                          kb + (uint64_t)(((s >> 2) * kLatBlock + (s & 3) * 32) >> 4), id_qk, s > 0);
#pragma unroll
          for (int s = 0; s < 2; ++s)
            tc::mma_f8_ss(d_s, qrope_desc + (uint64_t)((32 * s) >> 4),
                          rb + (uint64_t)((32 * s) >> 4), id_qk, 1);
          tc::mma_commit(bar(BAR_S_FULL + (int)(j & 1)));
          if (pe) tc::mma_commit(bar(BAR_Q_EMPTY));
        }
        __syncwarp();
        // ---- O^T += V^T P^T of the previous page ----
        if (have_prev) {
          ok = pv(prev);
          if (!ok) break;
        }
        prev = Prev{j, slot, ps, pe};
        have_prev = true;
      }
      if (ok && have_prev) ok = pv(prev);
      if (leader) {
        if (!ok) abort_cta();
        // drain: every issued MMA has finished before TMEM is freed
        tc::mma_commit(bar(BAR_DRAIN));
        if (!tc::mbar_wait(bar(BAR_DRAIN), 0, kWaitNs)) atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
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
      PageWalker pw;
      pw.init(plan, cur0, x_begin, x_end);
      for (int64_t j = 0; !pw.done(); pw.next(), ++j) {
        const bool ps = pw.piece_start(), pe = pw.piece_end();
        if (ps) {
          // ---- stage q of this row: per-head power-of-two scale, e4m3 hi/lo split ----
          if (piece > 0) {
            const bool got = tc::mbar_wait(bar(BAR_Q_EMPTY), (uint32_t)(piece - 1) & 1, kWaitNs);
            if (named_bar_softmax_or(!got || flags[F_ABORT])) {
              ok = false;
              break;
            }
          }
          const bool live = h < H;
          const uint4* qrow = reinterpret_cast<const uint4*>(
              p.q + ((int64_t)pw.cur.r * H + (live ? h : 0)) * kDEntry);
          float amax = 0.f;
          if (live) {
#pragma unroll 4
            for (int u = 0; u < kDEntry / 8; ++u) {
              const uint4 w = __ldg(qrow + u);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
                amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
              }
            }
          }
          int shift = 0;
          if (amax > 0.f && isfinite(amax)) {
            int e;
            frexpf(amax, &e);
            shift = 8 - e;  // scaled max in [2^7, 2^8)
          }
          const float sc = live ? ldexpf(1.0f, shift) : 0.f;
          qmul = live ? p.score_mul * ldexpf(1.0f, -shift) : 0.f;
          // latent dims: TMEM columns, four e4m3 codes each
#pragma unroll 1
          for (int blk = 0; blk < 4; ++blk) {
            uint32_t r[32];
#pragma unroll
            for (int c8 = 0; c8 < 16; ++c8) {
              const uint4 w = __ldg(qrow + blk * 16 + c8);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
              uint32_t codes[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
                codes[k] = split_pair(f.x * sc, f.y * sc, part != 0, nullptr);
              }
              r[2 * c8] = codes[0] | (codes[1] << 16);
              r[2 * c8 + 1] = codes[2] | (codes[3] << 16);
            }
            tc::tmem_st32(tmem + lane_base + kQCol + 32 * blk, r);
          }
          // rope dims: shared memory row t (64 B, 64-byte swizzle)
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t r4[4];
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint4 w = __ldg(qrow + 64 + 2 * u + half);
              const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
              uint32_t codes[4];
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ws[k]));
                codes[k] = split_pair(f.x * sc, f.y * sc, part != 0, nullptr);
              }
              r4[2 * half] = codes[0] | (codes[1] << 16);
              r4[2 * half + 1] = codes[2] | (codes[3] << 16);
            }
            const uint32_t a = sbase + kOffQRope + t * 64 + ((u ^ ((t >> 1) & 3)) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a), "r"(r4[0]),
                         "r"(r4[1]), "r"(r4[2]), "r"(r4[3]));
          }
          tc::tmem_wait_st();
          tc::fence_proxy_async_smem();
          tc::fence_before_sync();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(bar(BAR_Q_READY));
        }
        // page validity (tokens of a bad page id are masked and reported)
        const int valid = pw.valid_tokens();
        const int page = pw.page_id(p.block_table, p.nq, p.max_pages);
        const bool page_ok = page >= 0 && (int64_t)page < p.num_pages;
        const int nvis = page_ok ? valid : 0;
        if (t == 0 && valid > 0 && !page_ok) {
          flags[F_PIECE_BAD] = 1;
          atomicOr(p.ws.status, MLA_DEVICE_ERR_BAD_PAGE);
        }
        // ---- S of this page ----
        {
          const bool got =
              tc::mbar_wait(bar(BAR_S_FULL + (int)(j & 1)), (uint32_t)(j >> 1) & 1, kWaitNs);
          if (named_bar_softmax_or(!got || flags[F_ABORT])) {
            ok = false;
            break;
          }
        }
        tc::fence_after_sync();
        float v[64];
        {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_base + s_col((int)(j & 1)), r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
          tc::tmem_ld32(tmem + lane_base + s_col((int)(j & 1)) + 32, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) v[32 + i] = __uint_as_float(r[i]);
        }
        tc::fence_before_sync();
        __syncwarp();
        if (lane == 0) tc::mbar_arrive(bar(BAR_S_EMPTY + (int)(j & 1)));
        // hi + lo of this thread's 32 tokens (the partner lane holds the other term)
        float s[32];
        float tmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const float send = part ? v[i] : v[32 + i];
          const float recv = __shfl_xor_sync(0xffffffffu, send, 16);
          const float mine = part ? v[32 + i] : v[i];
          const bool vis = 32 * part + i < nvis;
          s[i] = vis ? (mine + recv) * qmul : -INFINITY;
          tmax = fmaxf(tmax, s[i]);
        }
        tmax = fmaxf(tmax, __shfl_xor_sync(0xffffffffu, tmax, 16));
        // lazy running max: O is rescaled only when a head's max grows past the threshold
        float alpha = 1.f;
        bool grow = false;
        if (ps) {
          m = tmax;
        } else if (tmax > m + kRescaleThresh) {
          alpha = m == -INFINITY ? 0.f : fast_exp2(m - tmax);
          m = tmax;
          l *= alpha;
          grow = true;
        }
        float* alpha_w = alpha_s + 64 * (int)(j & 1);
        if (part == 0) alpha_w[h] = alpha;
        if (named_bar_softmax_or(grow)) {
          // rare: bring O^T (PV of the previous page done) to the new maxima
          const bool got =
              tc::mbar_wait(bar(BAR_PV_DONE), (uint32_t)(j - 1) & 1, kWaitNs);
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
        // ---- P = 2^(s - m + 7) as e4m3 hi + lo, row h of P^T ----
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
              const uint32_t lc = e4m3x2_of(p0 - hv.x, p1 - hv.y);
              const float2 lv = e4m3x2_value(lc);
              rs += (hv.x + lv.x) + (hv.y + lv.y);
              hcode[e] = hc;
              lcode[e] = lc;
            }
            hw[k] = hcode[0] | (hcode[1] << 16);
            lw[k] = lcode[0] | (lcode[1] << 16);
          }
          rs += __shfl_xor_sync(0xffffffffu, rs, 16);
          l += rs;
          const uint32_t prow = sbase + kOffP + (int)(j & 1) * kPBytes + h * 128;
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
        if (lane == 0) tc::mbar_arrive(bar(BAR_P_FULL + (int)(j & 1)));
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
          const int slot = pw.cur.base + (c - plan.cta_of(pw.cur.rt));
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
                  o[(int64_t)i * kDLatent] = __uint_as_float(r[i]) * linv_s[32 * half + i];
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
  if (warp == kMmaWarp) tc::tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

cudaError_t launch_decode_fp8(const DecodeLaunch& d, cudaStream_t stream) {
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(decode_fp8_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(1);
  }
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
  p.score_mul = d.score_mul;
  p.kv_scale = d.kv_scale;
  p.G = d.G;
  p.ws = d.ws;
  decode_fp8_kernel<<<d.G, kThreads, kSmemBytes, stream>>>(p, lat_map, rope_map);
  return cudaGetLastError();
}

}  // namespace mla
