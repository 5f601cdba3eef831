// decode_tc.cu -- split-KV paged MLA decode on the 5th-generation tensor cores.
//
// One CTA per SM walks its run of cache pages (split-KV planner in
// mla_common.cuh) in tiles of up to 128 tokens (two pages of one request row).
// Warp roles:
//   warps 0-3   softmax + epilogue: thread t owns TMEM lane t (token t of the
//               tile's scores; dim t of each 128-dim block of the output);
//               warp 0 allocates TMEM and its thread 0 issues every tcgen05.mma
//   warps 4-11  load + convert: 16-byte loads of the page bytes into registers,
//               up to three 4 KB jobs ahead per warp, e4m3 -> f16 (an FP8 cache
//               is widened as it is read: "Smaller, faster, safer: running Kimi
//               and GLM at scale", section "Quantizing the KV cache"), stored
//               into a 128-byte-swizzled shared tile; q by TMA once per piece
// Per tile, two dense contractions share one shared-memory tile of the 128
// tokens x 576 entry dims (all heads attend over one latent head: "vLLM x
// AgentX", section "Kimi K3"):
//   S^T [128 tokens x 64 heads] = K [128 x 576] . Q^T      (M = tokens)
//   O^T [512 dims x 64 heads]  += V^T [512 x 128] . P^T    (M = dims, 4 blocks)
// V is the first 512 dims of the same tile read through a transposed (MN-major)
// descriptor (no distinct keys and values: "How to serve trillions of tokens
// ...", section "First, understand the workload"). S (two buffers) and O^T live
// in TMEM; P (f16) overwrites the tile's rope chunk once QK has read it.
// Online softmax keeps one running max per head; O^T is rescaled only when a
// head's max grows by more than 2^7, so P stays below 2^15 in f16.
//
// Every mbarrier wait is bounded (2 s); on timeout the CTA records
// MLA_DEVICE_ERR_TIMEOUT, stops, drains its MMAs (bounded) and frees TMEM.
#include <atomic>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "mla_common.cuh"
#include "mla_internal.h"
#include "tc_ptx.cuh"

namespace mla {
namespace {

constexpr int kSoftmaxWarps = 4;     // warps 0-3 (thread 0 also issues the MMAs)
constexpr int kLoadWarps = 8;        // warps 4-11
constexpr int kLoadThreads = 32 * kLoadWarps;
constexpr int kThreads = 32 * (kSoftmaxWarps + kLoadWarps);  // 384: 3 warps per scheduler
constexpr int kTileTokens = 128;
constexpr int kN = 64;                        // head columns (H padded to 64)
constexpr int kChunks = 9;                    // 576 dims / 64
constexpr int kChunkBytes = kTileTokens * 128;  // 16 KB: 128 rows x 64 f16
constexpr int kQChunkBytes = kN * 128;          // 8 KB
constexpr int kPOffset = 8;                   // P = 2^(s - m + 8)
constexpr float kRescaleThresh = 7.0f;        // lazy rescale threshold (log2 units)
constexpr uint64_t kWaitNs = 2000000000ull;   // 2 s bound on every wait

// TMEM columns
constexpr uint32_t kTmemCols = 512;
__device__ __forceinline__ uint32_t s_col(int b) { return 64u * (uint32_t)b; }  // S buffers
constexpr uint32_t kOCol = 128;               // O^T block mt at kOCol + 64*mt

// shared memory map (offsets from a 1024-aligned base)
constexpr int kOffK = 0;
constexpr int kOffQ = kOffK + kChunks * kChunkBytes;       // 147456
constexpr int kOffQmul = kOffQ + kChunks * kQChunkBytes;    // 221184
constexpr int kOffMUsed = kOffQmul + 512;               // qmul: float [2][64], by piece parity
constexpr int kOffLSum = kOffMUsed + 256;
constexpr int kOffAlpha = kOffLSum + 256;
constexpr int kOffRed = kOffAlpha + 256;                   // float [4][64] per-warp maxima
constexpr int kOffRedSum = kOffRed + 1024;                 // float [2][4][64] per-warp sums
constexpr int kOffFlags = kOffRedSum + 2048;               // int [4]
constexpr int kOffBar = kOffFlags + 16;                    // uint64 [kNumBars]
constexpr int kNumBars = 20;
constexpr int kOffTmem = kOffBar + 8 * kNumBars;
constexpr int kSmemUsed = kOffTmem + 16;
constexpr int kSmemBytes = kSmemUsed + 1024;               // slack for 1024 alignment

// barrier indices
constexpr int BAR_CHUNK_FULL = 0;     // [9]  load warps -> MMA (count 2: both halves)
constexpr int BAR_CHUNK_EMPTY = 9;    // [5]  MMA commit -> load warps: chunks 2i and 2i+1
                                      //      (the 128-dim block PV block i reads), chunk 8
constexpr int BAR_Q_EMPTY = 14;       // MMA commit -> load warps (q tile free)
constexpr int BAR_S_FULL = 15;        // [2] MMA commit -> softmax
constexpr int BAR_O_FULL = 17;        // MMA commit -> epilogue
constexpr int BAR_DRAIN = 18;         // MMA commit before TMEM is freed
constexpr int BAR_Q_TMA = 19;         // TMA bytes of q landed (count 1 + tx bytes)
__device__ __forceinline__ int empty_bar(int chunk) { return BAR_CHUNK_EMPTY + (chunk >> 1); }


enum Flag { F_ABORT = 0, F_PIECE_BAD = 1 };

struct TcParams {
  const __nv_bfloat16* q;
  const uint8_t* kv;
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

// One tile: up to two consecutive pages of one row inside this CTA's range.
struct TileWalker {
  Plan plan;
  RowCursor cur;
  int64_t x, x_end, x_begin;
  int npages;       // pages in the current tile (1 or 2)

  __device__ void init(const Plan& p, const RowCursor& c, int64_t xb, int64_t xe) {
    plan = p; cur = c; x = xb; x_begin = xb; x_end = xe;
    settle();
  }
  __device__ void settle() {
    if (x < x_end && x == cur.rt + cur.t) cursor_next_row(plan, cur);
    const int64_t row_left = cur.rt + cur.t - x, cta_left = x_end - x;
    npages = (int)min((int64_t)2, min(row_left, cta_left));
  }
  __device__ bool done() const { return x >= x_end; }
  __device__ int page_in_row() const { return (int)(x - cur.rt); }
  __device__ bool piece_start() const { return x == x_begin || x == cur.rt; }
  __device__ bool piece_end() const {
    return x + npages == x_end || x + npages == cur.rt + cur.t;
  }
  __device__ int valid_tokens() const {
    return min(npages * kPageSize, cur.n - page_in_row() * kPageSize);
  }
  // block-table entries of this tile's pages (second is -1 for a one-page tile)
  __device__ void page_ids(const int32_t* block_table, int nq, int max_pages, int& p0,
                           int& p1) const {
    const int64_t bt = (int64_t)(cur.r / nq) * max_pages + page_in_row();
    p0 = __ldg(block_table + bt);
    p1 = npages > 1 ? __ldg(block_table + bt + 1) : -1;
  }
  __device__ void next() { x += npages; settle(); }
};

__device__ __forceinline__ uint32_t kv_tile_off(int token, int unit, int chunk) {
  return (uint32_t)(kOffK + chunk * kChunkBytes + token * 128 + (((unit ^ (token & 7))) << 4));
}

__device__ __forceinline__ void named_bar_softmax() {
  asm volatile("bar.sync 1, 128;\n" ::: "memory");
}

// Barrier over the 128 softmax threads that also returns the OR of `pred` over
// them, so that every thread takes the same branch afterwards.
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

template <bool kBf16>
__device__ __forceinline__ uint32_t pack_f2(float lo, float hi) {
  if constexpr (kBf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Column-wise reduction of a [32 lanes x 64 values] register block: after the
// call, lane l holds the reduction over all 32 lanes for heads (2*l') and
// (2*l'+1), where the pair index is returned in `head0`.
template <bool kMax>
__device__ __forceinline__ void transpose_reduce64(float (&v)[64], int lane, float& out0,
                                                   float& out1, int& head0) {
  // stage sizes 64 -> 32 -> 16 -> 8 -> 4 -> 2 values per lane
  int base = 0;  // first head index of this lane's kept range
#pragma unroll
  for (int stage = 0; stage < 5; ++stage) {
    const int half = 32 >> stage;          // values kept after this stage
    const int off = 16 >> stage;           // shuffle distance
    const bool upper = (lane & off) != 0;  // keep upper half of the current range
#pragma unroll
    for (int i = 0; i < half; ++i) {
      const float keep = upper ? v[i + half] : v[i];
      const float send = upper ? v[i] : v[i + half];
      const float recv = __shfl_xor_sync(0xffffffffu, send, off);
      v[i] = kMax ? fmaxf(keep, recv) : keep + recv;
    }
    if (upper) base += half;
  }
  out0 = v[0];
  out1 = v[1];
  head0 = base;
}

template <bool kBf16>
__global__ void __maxnreg__(168)
    decode_tc_kernel(const TcParams p, const __grid_constant__ CUtensorMap q_map) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_a = smem_u32(smem_raw);
  const uint32_t sbase = (raw_a + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_a);
  float* qmul = reinterpret_cast<float*>(smem + kOffQmul);
  float* m_used = reinterpret_cast<float*>(smem + kOffMUsed);
  float* l_sum = reinterpret_cast<float*>(smem + kOffLSum);
  float* alpha = reinterpret_cast<float*>(smem + kOffAlpha);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  float* red_sum = reinterpret_cast<float*>(smem + kOffRedSum);
  volatile int* flags = reinterpret_cast<volatile int*>(smem + kOffFlags);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  auto bar = [&](int i) -> uint32_t { return sbase + kOffBar + 8u * (uint32_t)i; };

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  // ---- planning (shared by all roles) ----
  __shared__ int64_t s_plan[6];
  Plan plan{p.seq_lens, p.batch, p.nq, p.max_pages, kPageSize, p.G, 0};
  if (warp == 0) {
    const int64_t T = plan_total_tiles_warp(plan);
    if (lane == 0) s_plan[0] = T;
  }
  if (tid == 0) {
    for (int i = 0; i < kNumBars; ++i) {
      // chunk full: every load warp (e4m3 slices) or both half-chunk jobs (bf16)
      tc::mbar_init(bar(i), i < BAR_CHUNK_EMPTY ? (kBf16 ? 2 : kLoadWarps) : 1);
    }
    tc::fence_mbar_init();
    flags[F_ABORT] = 0;
    flags[F_PIECE_BAD] = 0;
  }
  if (tid < kN) {
    m_used[tid] = -INFINITY;
    l_sum[tid] = 0.f;
  }
  if (warp == 0) {
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

  if (x_begin < x_end) {
    if (warp >= kSoftmaxWarps) {
      // =================== load + convert warps ===================
      const int lw = warp - kSoftmaxWarps;  // 0..7
      const int lt = tid - 32 * kSoftmaxWarps;
      bool aborted = false;
      // q[b][j][0:H][:] arrives by TMA, one 64-dim chunk per copy, already in the
      // 128-byte-swizzled layout (the softmax warps convert it to f16).
      auto issue_q = [&](int r) {
        tc::mbar_arrive_expect_tx(bar(BAR_Q_TMA), (uint32_t)(kChunks * H * 128));
        for (int ch = 0; ch < kChunks; ++ch)
          tc::tma_load_2d(sbase + kOffQ + ch * kQChunkBytes, &q_map, 64 * ch, r * H,
                          bar(BAR_Q_TMA));
      };
      // rows H..63 of the Q tile stay zero (padded heads); TMA writes only rows < H
      if (H < kN) {
        for (int v = lt; v < kChunks * (kN - H) * 8; v += kLoadThreads) {
          const int ch = v / ((kN - H) * 8), rem = v - ch * (kN - H) * 8;
          const int row = H + (rem >> 3), unit = rem & 7;
          asm volatile("st.shared.v4.b32 [%0], {%1,%1,%1,%1};\n" ::"r"(
                           sbase + kOffQ + ch * kQChunkBytes + row * 128 + (unit << 4)),
                       "r"(0u));
        }
        tc::fence_proxy_async_smem();
      }

      if constexpr (!kBf16) {
        // e4m3 cache: load warp lw owns tokens [16 lw, 16 lw + 16) of every tile (its
        // page is the tile's page lw / 4). Per tile a lane holds 18 16-byte vectors:
        // vector g*9 + c covers token 8g + lane/4 of the slice, dims 64c + 16 (lane%4)
        // .. +15, so each warp load reads 8 whole 64-byte row pieces. A chunk is
        // converted as soon as the previous tile's PV has released it; once the
        // whole tile is stored, the registers are refilled with the next tile's
        // bytes, which are in flight while this tile is multiplied.
        const uint64_t pol = l2_evict_first_policy();
        const int slice0 = 16 * (lw & 3);   // first token of the slice within its page
        const int page_sel = lw >> 2;       // which page of the tile
        struct Slice {
          const uint8_t* base;  // this lane's first byte (token 8*0 + lane/4, dims 16 (lane%4))
          uint32_t vis;         // bit g: token 8g + lane/4 of the slice is visible
          int r;                // request row of the tile (for q)
          bool ps;              // first tile of a piece
        };
        auto slice_of = [&](const TileWalker& w) {
          Slice sl;
          const int valid = w.valid_tokens() - 64 * page_sel - slice0;  // tokens of my slice
          int page = -1;
          if (page_sel < w.npages)
            page = __ldg(p.block_table + (int64_t)(w.cur.r / p.nq) * p.max_pages +
                         w.page_in_row() + page_sel);
          const bool page_ok = page >= 0 && (int64_t)page < p.num_pages;
          const int tok = lane >> 2;
          sl.vis = (page_ok && tok < valid ? 1u : 0u) | (page_ok && tok + 8 < valid ? 2u : 0u);
          sl.base = p.kv + (page_ok ? (int64_t)page : 0) * (kPageSize * kDEntry) +
                    (int64_t)(slice0 + tok) * kDEntry + 16 * (lane & 3);
          sl.r = w.cur.r;
          sl.ps = w.piece_start();
          return sl;
        };
        // masked vectors read the pool's first bytes (and are zeroed at conversion)
        auto load_slice_chunk = [&](uint4 (&b)[18], const Slice& sl, int c) {
          b[c] = ld_stream_16((sl.vis & 1u) ? sl.base + 64 * c : p.kv, pol);
          b[9 + c] = ld_stream_16((sl.vis & 2u) ? sl.base + 8 * kDEntry + 64 * c : p.kv, pol);
        };
        uint4 buf[18];
        TileWalker nw;
        nw.init(plan, cur0, x_begin, x_end);
        Slice cur = slice_of(nw);
#pragma unroll
        for (int c = 0; c < kChunks; ++c) load_slice_chunk(buf, cur, c);
        int piece_seen = 0;
        for (int64_t k = 0;; ++k) {
          nw.next();
          const bool have_next = !nw.done();
          Slice nxt = cur;
          if (have_next) nxt = slice_of(nw);
          if (cur.ps) {
            // load warp 0 fetches q for a piece once the previous piece's QK is done
            if (lw == 0 && lane == 0) {
              if (piece_seen > 0 &&
                  !tc::mbar_wait(bar(BAR_Q_EMPTY), (uint32_t)((piece_seen - 1) & 1), kWaitNs))
                aborted = true;
              else
                issue_q(cur.r);
            }
            ++piece_seen;
          }
          if (__any_sync(0xffffffffu, aborted)) {
            aborted = true;
            break;
          }
          const uint32_t par = (uint32_t)((k - 1) & 1);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            if (k > 0 && (c & 1) == 0 && !tc::mbar_wait(bar(empty_bar(c)), par, kWaitNs)) {
              aborted = true;
              break;
            }
#pragma unroll
            for (int g = 0; g < 2; ++g) {
              uint4 v = buf[9 * g + c];
              if (!((cur.vis >> g) & 1u)) v = make_uint4(0, 0, 0, 0);
              const int token = 64 * page_sel + slice0 + 8 * g + (lane >> 2);
              const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
              uint32_t h[8];
#pragma unroll
              for (int i2 = 0; i2 < 4; ++i2) {
                h[2 * i2] = e4m3x2_to_f16x2((uint16_t)(w4[i2] & 0xffffu));
                h[2 * i2 + 1] = e4m3x2_to_f16x2((uint16_t)(w4[i2] >> 16));
              }
              const uint32_t a0 = sbase + kv_tile_off(token, 2 * (lane & 3), c);
              const uint32_t a1 = sbase + kv_tile_off(token, 2 * (lane & 3) + 1, c);
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a0), "r"(h[0]),
                           "r"(h[1]), "r"(h[2]), "r"(h[3]));
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a1), "r"(h[4]),
                           "r"(h[5]), "r"(h[6]), "r"(h[7]));
            }
            tc::fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(bar(BAR_CHUNK_FULL + c));
          }
          if (aborted || !have_next) break;
          // The next tile's loads go out only after this tile's last proxy fence: a
          // fence.proxy.async waits for the thread's outstanding loads, so a load
          // issued between two chunk fences would put its latency in the loop.
#pragma unroll
          for (int c = 0; c < kChunks; ++c) load_slice_chunk(buf, nxt, c);
          cur = nxt;
        }
      } else {
      // =================== load + convert warps ===================
      // bf16 cache: a tile is 18 jobs: chunk c (64 dims) x half h (64 tokens = one page). Job g of
      // the CTA's sequence goes to load warp g % 8, so the warps convert different
      // chunks at the same time; each warp keeps its next kDepth jobs in flight in
      // registers. A chunk is full when the warps of both halves have arrived.
      constexpr int kVec = kBf16 ? 16 : 8;   // 16-byte vectors per lane per job
      // jobs in flight per warp: a tile's 18 jobs over 8 warps leave 3 to some
      // warps, so 3 keeps the whole next tile in registers while PV runs
      constexpr int kDepth = kBf16 ? 2 : 3;
      constexpr int kJobsPerTile = 2 * kChunks;
      const uint64_t pol = l2_evict_first_policy();
      uint4 buf[kDepth][kVec];
      uint32_t bufmask[kDepth];

      // job walker: tile cursor + page ids of the current tile
      struct JobCursor {
        TileWalker tw;
        int64_t g;        // global job index of this warp's current job
        int64_t tile;     // tile index of job g
        int pg[2];
      };
      auto jc_init = [&](JobCursor& j) {
        j.tw.init(plan, cur0, x_begin, x_end);
        j.g = lw;
        j.tile = 0;
        if (!j.tw.done()) j.tw.page_ids(p.block_table, p.nq, p.max_pages, j.pg[0], j.pg[1]);
      };
      auto jc_next = [&](JobCursor& j) {
        j.g += kLoadWarps;
        while (!j.tw.done() && j.g >= (j.tile + 1) * kJobsPerTile) {
          j.tw.next();
          ++j.tile;
          if (!j.tw.done()) j.tw.page_ids(p.block_table, p.nq, p.max_pages, j.pg[0], j.pg[1]);
        }
      };
      // Loads are issued unconditionally (from the cache's first bytes when the token
      // is masked) so that nothing consumes their results before conversion time.
      auto load_job = [&](uint4 (&dst)[kVec], uint32_t& mask, const JobCursor& j) {
        const int jj = (int)(j.g - j.tile * kJobsPerTile);
        const int chunk = jj >> 1, half = jj & 1;
        const int valid = j.tw.valid_tokens() - 64 * half;  // tokens of this page
        const int page = half ? j.pg[1] : j.pg[0];
        const bool page_ok = page >= 0 && (int64_t)page < p.num_pages;
        const uint8_t* pbase =
            p.kv + (page_ok ? (int64_t)page : 0) * kPageSize * kDEntry * (kBf16 ? 2 : 1);
        mask = 0;
#pragma unroll
        for (int k = 0; k < kVec; ++k) {
          int token, part;
          if constexpr (kBf16) {  // 64 tokens x 8 vectors (64 bf16 dims)
            const int v = lane + 32 * k;
            token = v >> 3;
            part = v & 7;
          } else {                // 64 tokens x 4 vectors (64 e4m3 dims)
            const int v = lane + 32 * k;
            token = v >> 2;
            part = v & 3;
          }
          const bool ok = page_ok && token < valid;
          const uint8_t* src = pbase + token * (kDEntry * (kBf16 ? 2 : 1)) +
                               chunk * (kBf16 ? 128 : 64) + part * 16;
          dst[k] = ld_stream_16(ok ? src : p.kv, pol);
          mask |= (ok ? 1u : 0u) << k;
        }
      };
      JobCursor issue, comp;
      jc_init(issue);
      jc_init(comp);
      int piece_seen = 0;       // pieces whose first tile `comp` has passed
      int64_t last_tile = -1;   // last tile `comp` processed (for piece counting)
#pragma unroll
      for (int s = 0; s < kDepth; ++s) {
        if (!issue.tw.done()) {
          load_job(buf[s], bufmask[s], issue);
          jc_next(issue);
        }
      }
      while (!comp.tw.done() && !aborted) {
#pragma unroll
        for (int s = 0; s < kDepth; ++s) {
          if (comp.tw.done() || aborted) break;
          const int jj = (int)(comp.g - comp.tile * kJobsPerTile);
          const int chunk = jj >> 1, half = jj & 1;
          if (comp.tile != last_tile) {
            if (comp.tw.piece_start()) {
              // the warp holding job 0 of a piece's first tile fetches its q
              if (jj == 0 && lane == 0) {
                if (piece_seen > 0 &&
                    !tc::mbar_wait(bar(BAR_Q_EMPTY), (uint32_t)((piece_seen - 1) & 1), kWaitNs))
                  aborted = true;
                else
                  issue_q(comp.tw.cur.r);
              }
              ++piece_seen;
            }
            last_tile = comp.tile;
          }
          if (__any_sync(0xffffffffu, aborted)) {
            aborted = true;
            break;
          }
          if (comp.tile > 0 && !tc::mbar_wait(bar(empty_bar(chunk)),
                                              (uint32_t)((comp.tile - 1) & 1), kWaitNs)) {
            aborted = true;
            break;
          }
          // convert + store this job (masked vectors become zeros)
#pragma unroll
          for (int k = 0; k < kVec; ++k) {
            uint4 v = buf[s][k];
            if (!((bufmask[s] >> k) & 1u)) v = make_uint4(0, 0, 0, 0);
            const int vv = lane + 32 * k;
            if constexpr (kBf16) {
              const int token = 64 * half + (vv >> 3), unit = vv & 7;
              const uint32_t a = sbase + kv_tile_off(token, unit, chunk);
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a), "r"(v.x),
                           "r"(v.y), "r"(v.z), "r"(v.w));
            } else {
              const int token = 64 * half + (vv >> 2), unit0 = 2 * (vv & 3);
              const uint32_t w[4] = {v.x, v.y, v.z, v.w};
              uint32_t h[8];
#pragma unroll
              for (int i2 = 0; i2 < 4; ++i2) {
                h[2 * i2] = e4m3x2_to_f16x2((uint16_t)(w[i2] & 0xffffu));
                h[2 * i2 + 1] = e4m3x2_to_f16x2((uint16_t)(w[i2] >> 16));
              }
              const uint32_t a0 = sbase + kv_tile_off(token, unit0, chunk);
              const uint32_t a1 = sbase + kv_tile_off(token, unit0 + 1, chunk);
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a0), "r"(h[0]),
                           "r"(h[1]), "r"(h[2]), "r"(h[3]));
              asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a1), "r"(h[4]),
                           "r"(h[5]), "r"(h[6]), "r"(h[7]));
            }
          }
          tc::fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) tc::mbar_arrive(bar(BAR_CHUNK_FULL + chunk));
          if (!issue.tw.done()) {  // refill the slot just converted
            load_job(buf[s], bufmask[s], issue);
            jc_next(issue);
          }
          jc_next(comp);
        }
      }
      }
      if (aborted) {
        flags[F_ABORT] = 1;
        atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
      }
    } else {
      // =================== softmax + epilogue ===================
      const int t = tid;  // TMEM lane / token within the tile
      const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
      TileWalker tw;
      tw.init(plan, cur0, x_begin, x_end);
      int64_t k = 0;
      int piece = 0;
      bool ok = true;
      for (; !tw.done(); tw.next(), ++k) {
        const bool ps = tw.piece_start(), pe = tw.piece_end();
        const int sb = (int)(k & 1);
        if (ps) {
          // q for this piece: wait for its TMA bytes, rescale to f16 in place (e4m3
          // caches; two threads per head), publish the per-head score multipliers
          const bool got = tc::mbar_wait(bar(BAR_Q_TMA), (uint32_t)(piece & 1), kWaitNs);
          if (named_bar_softmax_or(!got || flags[F_ABORT])) {
            ok = false;
            break;
          }
          float* qm_w = qmul + 64 * (piece & 1);
          const int h = t >> 1, hf = t & 1;
          auto qaddr = [&](int u) -> uint32_t {
            const int uu = 36 * hf + u;
            const int chunk = uu >> 3, unit = uu & 7;
            return sbase + kOffQ + chunk * kQChunkBytes + h * 128 + ((unit ^ (h & 7)) << 4);
          };
          int shift = 0;
          if constexpr (!kBf16) {
            float amax = 0.f;
            if (h < H) {
#pragma unroll 4
              for (int u = 0; u < 36; ++u) {
                uint32_t w[4];
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                             : "r"(qaddr(u)));
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {
                  const float2 f =
                      __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q2]));
                  amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
                }
              }
            }
            amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
            if (amax > 0.f && isfinite(amax)) {
              int e;
              frexpf(amax, &e);
              shift = 15 - e;  // scaled max in [2^14, 2^15)
            }
            const float sc = ldexpf(1.0f, shift);
            if (h < H) {
#pragma unroll 4
              for (int u = 0; u < 36; ++u) {
                const uint32_t a = qaddr(u);
                uint32_t w[4];
                asm volatile("ld.shared.v4.b32 {%0,%1,%2,%3}, [%4];\n"
                             : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3])
                             : "r"(a));
                uint32_t r4[4];
#pragma unroll
                for (int q2 = 0; q2 < 4; ++q2) {
                  const float2 f =
                      __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[q2]));
                  r4[q2] = pack_f2<false>(f.x * sc, f.y * sc);
                }
                asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(a), "r"(r4[0]),
                             "r"(r4[1]), "r"(r4[2]), "r"(r4[3]));
              }
            }
          }
          if (hf == 0) qm_w[h] = h < H ? p.score_mul * ldexpf(1.0f, -shift) : 0.f;
          tc::fence_proxy_async_smem();
          named_bar_softmax();  // q tile and qmul ready
        }
        // ---- thread 0: S^T = K Q^T for this tile, as its chunks arrive ----
        // (fully unrolled with descriptors formed as base + constant: a tcgen05.mma
        // whose descriptors are computed at run time issues at half the rate)
        bool mma_ok = true;
        if (t == 0) {
          constexpr uint32_t id_qk = tc::idesc_f16(128, kN, kBf16, false, false);
          const uint64_t a0 = tc::smem_desc_sw128(sbase + kOffK, 16, 1024);
          const uint64_t b0 = tc::smem_desc_sw128(sbase + kOffQ, 16, 1024);
          const uint32_t d_s = tmem + s_col(sb);
          const uint32_t par = (uint32_t)(k & 1);
#pragma unroll
          for (int ch = 0; ch < kChunks; ++ch) {
            if (mma_ok) mma_ok = tc::mbar_wait(bar(BAR_CHUNK_FULL + ch), par, kWaitNs);
            if (mma_ok) {
              tc::fence_after_sync();
#pragma unroll
              for (int sub = 0; sub < 4; ++sub)
                tc::mma_f16_ss(d_s, a0 + (uint64_t)((ch * kChunkBytes + sub * 32) >> 4),
                               b0 + (uint64_t)((ch * kQChunkBytes + sub * 32) >> 4), id_qk,
                               (ch | sub) != 0);
            }
          }
          if (mma_ok) {
            tc::mma_commit(bar(BAR_S_FULL + sb));
            if (pe) tc::mma_commit(bar(BAR_Q_EMPTY));
          }
        }
        // page validity of this thread's token (bad page ids are masked)
        const int valid = tw.valid_tokens();
        int pg0, pg1;
        tw.page_ids(p.block_table, p.nq, p.max_pages, pg0, pg1);
        const int pg = (t >> 6) ? pg1 : pg0;
        const bool page_ok = pg >= 0 && (int64_t)pg < p.num_pages;
        const bool vis = t < valid && page_ok;
        if (t < valid && !page_ok) {
          flags[F_PIECE_BAD] = 1;
          atomicOr(p.ws.status, MLA_DEVICE_ERR_BAD_PAGE);
        }
        {
          const bool got =
              mma_ok && tc::mbar_wait(bar(BAR_S_FULL + sb), (uint32_t)((k >> 1) & 1), kWaitNs);
          if (named_bar_softmax_or(!got || flags[F_ABORT])) {
            ok = false;
            break;
          }
        }
        tc::fence_after_sync();
        const float* qm = qmul + 64 * (piece & 1);
        float s[64];
        {
          uint32_t r[32];
          tc::tmem_ld32(tmem + lane_base + s_col(sb), r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[i] = __uint_as_float(r[i]);
          tc::tmem_ld32(tmem + lane_base + s_col(sb) + 32, r);
          tc::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) s[32 + i] = __uint_as_float(r[i]);
        }
        tc::fence_before_sync();
#pragma unroll
        for (int h4 = 0; h4 < 16; ++h4) {
          const float4 c4 = reinterpret_cast<const float4*>(qm)[h4];
          s[4 * h4 + 0] = vis ? s[4 * h4 + 0] * c4.x : -INFINITY;
          s[4 * h4 + 1] = vis ? s[4 * h4 + 1] * c4.y : -INFINITY;
          s[4 * h4 + 2] = vis ? s[4 * h4 + 2] * c4.z : -INFINITY;
          s[4 * h4 + 3] = vis ? s[4 * h4 + 3] * c4.w : -INFINITY;
        }
        // Lazy running max: the per-head maximum over the tile is needed only when
        // some score exceeds its head's current max by more than the threshold (or
        // on a piece's first tile); otherwise the max, and O, stay as they are.
        bool over = ps;
        if (!over) {
#pragma unroll
          for (int h4 = 0; h4 < 16; ++h4) {
            const float4 m4 = reinterpret_cast<const float4*>(m_used)[h4];
            over |= s[4 * h4 + 0] > m4.x + kRescaleThresh;
            over |= s[4 * h4 + 1] > m4.y + kRescaleThresh;
            over |= s[4 * h4 + 2] > m4.z + kRescaleThresh;
            over |= s[4 * h4 + 3] > m4.w + kRescaleThresh;
          }
        }
        const bool full = named_bar_softmax_or(over);
        if (full) {
          float v[64];
#pragma unroll
          for (int h = 0; h < 64; ++h) v[h] = s[h];
          float r0, r1;
          int h0;
          transpose_reduce64<true>(v, lane, r0, r1, h0);
          red[warp * 64 + h0] = r0;
          red[warp * 64 + h0 + 1] = r1;
          named_bar_softmax();
        }
        bool my_rescale = false;
        if (t < 64) {
          // fold in the previous tile's column sums, then (full path) the new max
          float l = l_sum[t];
          if (k > 0 && !ps) {
            const float* rs = red_sum + ((k - 1) & 1) * 256;
            l += rs[t] + rs[64 + t] + rs[128 + t] + rs[192 + t];
          }
          float a = 1.f;
          if (full) {
            const float tmax =
                fmaxf(fmaxf(red[t], red[64 + t]), fmaxf(red[128 + t], red[192 + t]));
            const float mo = m_used[t];
            if (mo == -INFINITY) {
              m_used[t] = tmax;
            } else if (tmax > mo + kRescaleThresh) {
              a = fast_exp2(mo - tmax);
              m_used[t] = tmax;
              l *= a;
              my_rescale = true;
            }
          }
          l_sum[t] = l;
          alpha[t] = a;
        }
        // (the lazy path changed no max, so it needs no barrier before P)
        if (full && named_bar_softmax_or(my_rescale)) {
          // rare: bring O^T to the new per-head max before this tile's PV
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
            for (int half = 0; half < 2; ++half) {
              uint32_t r[32];
              const uint32_t ta = tmem + lane_base + kOCol + 64 * mt + 32 * half;
              tc::tmem_ld32(ta, r);
              tc::tmem_wait_ld();
#pragma unroll
              for (int i = 0; i < 32; ++i)
                r[i] = __float_as_uint(__uint_as_float(r[i]) * alpha[32 * half + i]);
              tc::tmem_st32(ta, r);
            }
          }
          tc::tmem_wait_st();
        }
        // P = 2^(s - m + 8) in f16 (bf16 for bf16 caches), row t of the rope chunk
        float rowsum[64];
        {
          uint32_t pk[32];
#pragma unroll
          for (int h4 = 0; h4 < 16; ++h4) {
            const float4 m4 = reinterpret_cast<const float4*>(m_used)[h4];
            const float mm[4] = {m4.x, m4.y, m4.z, m4.w};
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float mu = mm[e] == -INFINITY ? 0.f : mm[e] - (float)kPOffset;
              rowsum[4 * h4 + e] = fast_exp2(s[4 * h4 + e] - mu);
            }
            pk[2 * h4] = pack_f2<kBf16>(rowsum[4 * h4], rowsum[4 * h4 + 1]);
            pk[2 * h4 + 1] = pack_f2<kBf16>(rowsum[4 * h4 + 2], rowsum[4 * h4 + 3]);
          }
          const uint32_t prow = sbase + kOffK + 8 * kChunkBytes + t * 128;
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                             prow + ((u ^ (t & 7)) << 4)),
                         "r"(pk[4 * u]), "r"(pk[4 * u + 1]), "r"(pk[4 * u + 2]),
                         "r"(pk[4 * u + 3]));
          }
        }
        tc::fence_proxy_async_smem();
        tc::fence_before_sync();
        named_bar_softmax();  // every row of P written, rescale done, red[] free
        if (t == 0) {
          // ---- thread 0: O^T += V^T P^T (V = the tile's first 512 dims, MN-major view) ----
          constexpr uint32_t id_pv = tc::idesc_f16(128, kN, kBf16, true, true);
          const uint64_t a0 = tc::smem_desc_sw128(sbase + kOffK, kChunkBytes, 1024);
          const uint64_t b0 = tc::smem_desc_sw128(sbase + kOffK + 8 * kChunkBytes, 16, 1024);
          const uint32_t d_o = tmem + kOCol;
          tc::fence_after_sync();
#pragma unroll
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll
            for (int kk = 0; kk < 8; ++kk)
              tc::mma_f16_ss(d_o + 64 * mt, a0 + (uint64_t)((2 * mt * kChunkBytes + kk * 2048) >> 4),
                             b0 + (uint64_t)((kk * 2048) >> 4), id_pv, !(ps && kk == 0));
            tc::mma_commit(bar(BAR_CHUNK_EMPTY + mt));
          }
          tc::mma_commit(bar(empty_bar(8)));
          if (pe) tc::mma_commit(bar(BAR_O_FULL));
        }
        {
          // column sums of P, folded into l_sum by the next tile (or the epilogue)
          float r0, r1;
          int h0;
          transpose_reduce64<false>(rowsum, lane, r0, r1, h0);
          float* rs = red_sum + (k & 1) * 256;
          rs[warp * 64 + h0] = r0;
          rs[warp * 64 + h0 + 1] = r1;
        }
        if (pe) {
          // ---- epilogue: O^T / l -> partial slot ----
          {
            const bool got = tc::mbar_wait(bar(BAR_O_FULL), (uint32_t)(piece & 1), kWaitNs);
            if (named_bar_softmax_or(!got)) {  // also: l_sum final
              ok = false;
              break;
            }
          }
          tc::fence_after_sync();
          const int slot = tw.cur.base + (c - plan.cta_of(tw.cur.rt));
          float* out = p.ws.part_out + (int64_t)slot * H * kDLatent + t;
          if (t < 64) {
            const float* rs = red_sum + (k & 1) * 256;
            const float l = l_sum[t] + rs[t] + rs[64 + t] + rs[128 + t] + rs[192 + t];
            l_sum[t] = l;
            alpha[t] = l > 0.f ? p.kv_scale / l : 0.f;  // 1/l per head
          }
          named_bar_softmax();
          const int nhalf = (H + 31) >> 5;
#pragma unroll 1
          for (int mt = 0; mt < 4; ++mt) {
#pragma unroll 1
            for (int half = 0; half < nhalf; ++half) {
              uint32_t r[32];
              tc::tmem_ld32(tmem + lane_base + kOCol + 64 * mt + 32 * half, r);
              tc::tmem_wait_ld();
              float* o = out + (int64_t)(32 * half) * kDLatent + 128 * mt;
#pragma unroll
              for (int i = 0; i < 32; ++i) {
                if (32 * half + i < H)
                  o[(int64_t)i * kDLatent] =
                      (__uint_as_float(r[i]) * alpha[32 * half + i]);
              }
            }
          }
          if (t < H) {
            const float l = l_sum[t];
            p.ws.part_lse[(int64_t)slot * H + t] =
                l > 0.f ? (m_used[t] - (float)kPOffset + log2f(l)) * kLn2 : -INFINITY;
          }
          if (t == 0) p.ws.piece_err[slot] = flags[F_PIECE_BAD] ? 1 : 0;
          tc::fence_before_sync();
          named_bar_softmax();  // O read out, stats consumed
          if (t < 64) {
            m_used[t] = -INFINITY;
            l_sum[t] = 0.f;
          }
          if (t == 0) flags[F_PIECE_BAD] = 0;
          named_bar_softmax();
          ++piece;
        }
      }
      if (!ok) {
        flags[F_ABORT] = 1;
        atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
      }
      if (t == 0) {
        // drain: every issued MMA has finished before TMEM is freed
        tc::mma_commit(bar(BAR_DRAIN));
        if (!tc::mbar_wait(bar(BAR_DRAIN), 0, kWaitNs)) atomicOr(p.ws.status, MLA_DEVICE_ERR_TIMEOUT);
      }
    }
  }
  tc::fence_before_sync();
  __syncthreads();
  tc::fence_after_sync();
  if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

template <bool kBf16>
cudaError_t launch_decode_tc(const TcParams& p, cudaStream_t stream) {
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(decode_tc_kernel<kBf16>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    configured[dev].store(1);
  }
  // q viewed as [batch*nq*heads rows][576] bf16; one box = 64 dims x `heads` rows
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
  CUtensorMap q_map;
  const cuuint64_t dims[2] = {(cuuint64_t)kDEntry, (cuuint64_t)p.batch * p.nq * p.heads};
  const cuuint64_t strides[1] = {(cuuint64_t)kDEntry * 2};
  const cuuint32_t box[2] = {64, (cuuint32_t)p.heads};
  const cuuint32_t estr[2] = {1, 1};
  CUresult r = encode(&q_map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16*>(p.q),
                      dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                      CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_128B,
                      CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  decode_tc_kernel<kBf16><<<p.G, kThreads, kSmemBytes, stream>>>(p, q_map);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_tensor_core(const DecodeLaunch& d, cudaStream_t stream) {
  TcParams p;
  p.q = d.q;
  p.kv = d.kv;
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
  return d.bf16 ? launch_decode_tc<true>(p, stream) : launch_decode_tc<false>(p, stream);
}

}  // namespace mla
