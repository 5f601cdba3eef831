// decode_mma.cu -- split-KV paged MLA decode on the warp-level tensor path.
//
// Per CTA: a contiguous run of 64-token tiles (one cache page each) from the
// device-side planner in mla_common.cuh. For every tile the CTA
//   1. copies the page (36,864 bytes for e4m3) into shared memory with 16-byte
//      cp.async, one tile ahead of the compute (double-buffered),
//   2. converts e4m3 -> f16 into a swizzled tile ("the FP8 attention kernel
//      has to convert values as it reads them": "Smaller, faster, safer:
//      running Kimi and GLM at scale", section "Quantizing the KV cache"),
//   3. computes S = Q K^T for all heads against the shared latent head
//      ("vLLM x AgentX", section "Kimi K3": one latent head for all query
//      heads) with mma.sync m16n8k16, fp32 accumulation,
//   4. updates the online softmax (running max m, sum l, rescale of O),
//   5. accumulates O += P V over the first 512 entry dims (the value is part
//      of the key entry: "How to serve trillions of tokens ...", section
//      "First, understand the workload").
// At the end of each piece it writes (O / l * kv_scale, lse) to the workspace;
// combine.cu merges the pieces.
//
// Number formats. Every e4m3 value is exactly an f16 (normal) number and one
// instruction converts a pair, so e4m3 caches run the MMAs in f16: q is
// brought to f16 with a per-head power-of-two scale (max |q| in [2^14, 2^15),
// exact for all elements within 2^27 of the head's largest), and P is stored
// as f16 in (0, 256] (exp2 offset of 8, so probabilities down to 2^-32 stay
// normal). bf16 caches run the MMAs in bf16 with q and P in bf16.
#include <atomic>

#include "mla_common.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

constexpr int kThreads = 256;
constexpr int kTile = 64;                      // tokens per tile (= page size)
constexpr int kRowBytes = kDEntry * 2;         // 1152 bytes per 16-bit row
constexpr int kPOffset = 8;                    // P = 2^(s - m + 8)

struct DecodeParams {
  const __nv_bfloat16* q;
  const uint8_t* kv;
  int64_t num_pages;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int batch, nq;
  float score_mul;  // sm_scale * log2(e) * kv_scale
  float kv_scale;
  int G;
  DecodeWorkspace ws;
};

// byte offset of 16-byte chunk `ch` in row `row` of a [rows][576] 16-bit tile
__device__ __forceinline__ uint32_t tile_off(int row, int ch) {
  return (uint32_t)(row * kRowBytes + ((ch ^ (row & 7)) << 4));
}
// P tile [H][64] 16-bit: 128 bytes per row
__device__ __forceinline__ uint32_t p_off(int row, int ch) {
  return (uint32_t)(row * 128 + ((ch ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t (&r)[4]) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

template <bool kBf16>
__device__ __forceinline__ void mma16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0,
                                         uint32_t b1) {
  if constexpr (kBf16) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  } else {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
        "{%8,%9}, {%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
  }
}

template <bool kBf16>
__device__ __forceinline__ uint32_t pack2(float lo, float hi) {
  if constexpr (kBf16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  } else {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
  }
}

// Shared-memory footprint of one instantiation.
template <bool kBf16, int H>
struct Smem {
  static constexpr int kKvBufs = kBf16 ? 2 : 1;
  static constexpr int q = 0;
  static constexpr int kv = q + H * kRowBytes;
  static constexpr int stage = kv + kKvBufs * kTile * kRowBytes;        // e4m3 only
  static constexpr int p = stage + (kBf16 ? 0 : 2 * kTile * kDEntry);
  static constexpr int red = p + H * 128;                               // float [4][H]
  static constexpr int qmul = red + 4 * H * 4;                          // float [H]
  static constexpr int misc = qmul + H * 4;                             // 64 bytes
  static constexpr int total = misc + 64;
};

// Tile cursor: which row / which tile of the row the global tile x is.
struct TileRef {
  int r;
  int i;       // tile index within the row = logical page index
  int valid;   // tokens of the tile that are visible to the row
  int page;    // physical page (may be out of range: checked by the user)
};

__device__ __forceinline__ TileRef tile_ref(const Plan& plan, const DecodeParams& p,
                                            const RowCursor& cur, int64_t x) {
  TileRef t;
  t.r = cur.r;
  t.i = (int)(x - cur.rt);
  const int n = plan.row_tokens(cur.r);
  t.valid = min(kTile, n - t.i * kTile);
  const int b = cur.r / p.nq;
  t.page = __ldg(p.block_table + (int64_t)b * p.max_pages + t.i);
  return t;
}

template <bool kBf16>
__device__ __forceinline__ void issue_tile_load(const DecodeParams& p, const TileRef& t,
                                                uint32_t dst) {
  const bool ok = t.page >= 0 && (int64_t)t.page < p.num_pages;
  if constexpr (kBf16) {
    const uint8_t* src = p.kv + (ok ? (int64_t)t.page * kTile * kRowBytes : 0);
    for (int v = threadIdx.x; v < kTile * (kRowBytes / 16); v += kThreads) {
      const int tok = v / (kRowBytes / 16), ch = v - tok * (kRowBytes / 16);
      const int bytes = (ok && tok < t.valid) ? 16 : 0;
      cp_async_16(dst + tile_off(tok, ch), src + (ok ? v * 16 : 0), bytes);
    }
  } else {
    const uint8_t* src = p.kv + (ok ? (int64_t)t.page * kTile * kDEntry : 0);
    for (int v = threadIdx.x; v < kTile * (kDEntry / 16); v += kThreads) {
      const int tok = v / (kDEntry / 16);
      const int bytes = (ok && tok < t.valid) ? 16 : 0;
      cp_async_16(dst + v * 16, src + (ok ? v * 16 : 0), bytes);
    }
  }
}

template <bool kBf16, int HG>
__global__ void __launch_bounds__(kThreads, 1) decode_mma_kernel(const DecodeParams p) {
  constexpr int H = 16 * HG;
  using S = Smem<kBf16, H>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* red_max = reinterpret_cast<float*>(smem + S::red);   // [2][H]
  float* red_sum = red_max + 2 * H;                           // [2][H]
  float* qmul = reinterpret_cast<float*>(smem + S::qmul);     // [H]
  int64_t* misc = reinterpret_cast<int64_t*>(smem + S::misc);
  const uint32_t q_base = smem_u32(smem + S::q);
  const uint32_t kv_base0 = smem_u32(smem + S::kv);
  const uint32_t stage_base = smem_u32(smem + S::stage);
  const uint32_t p_base = smem_u32(smem + S::p);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int g = lane >> 2, tq = lane & 3;

  Plan plan{p.seq_lens, p.batch, p.nq, p.max_pages, kTile, p.G, 0};
  if (warp == 0) {
    const int64_t T = plan_total_tiles_warp(plan);
    if (lane == 0) misc[0] = T;
  }
  __syncthreads();
  plan.set_total(misc[0]);
  const int c = blockIdx.x;
  const bool works = c < plan.G;
  const int64_t x_begin = works ? plan.cta_start(c) : 0;
  const int64_t x_end = works ? plan.cta_start(c + 1) : 0;
  if (warp == 0) {
    RowCursor f = plan_find_row_warp(plan, x_begin, c == 0, p.ws.row_base, p.ws.row_np,
                                     p.ws.status);
    if (lane == 0) {
      misc[1] = f.r;
      misc[2] = f.rt;
      misc[3] = f.t;
      misc[4] = f.base;
    }
  }
  __syncthreads();
  if (x_begin >= x_end) return;
  RowCursor cur{(int)misc[1], misc[2], (int)misc[3], (int)misc[4]};
  RowCursor pcur = cur;  // prefetch cursor, one tile ahead

  // compute-warp roles: head group hg (16 heads), half x (tokens in QK, dims in PV)
  const bool computes = warp < 2 * HG;
  const int hg = warp >> 1, xh = warp & 1;
  const int row0 = 16 * hg + g, row1 = row0 + 8;

  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
  float oacc[32][4];
  bool piece_bad = false;

  // first tile load
  {
    TileRef t0 = tile_ref(plan, p, pcur, x_begin);
    issue_tile_load<kBf16>(p, t0, kBf16 ? kv_base0 : stage_base);
    cp_async_commit();
  }

  for (int64_t x = x_begin, k = 0; x < x_end; ++x, ++k) {
    // ---- prefetch tile x+1 ----
    if (x + 1 < x_end) {
      if (x + 1 == pcur.rt + pcur.t) cursor_next_row(plan, pcur);
      TileRef tn = tile_ref(plan, p, pcur, x + 1);
      const uint32_t dst = kBf16 ? kv_base0 + (uint32_t)(((k + 1) & 1) * kTile * kRowBytes)
                                 : stage_base + (uint32_t)(((k + 1) & 1) * kTile * kDEntry);
      issue_tile_load<kBf16>(p, tn, dst);
    }
    cp_async_commit();
    cp_async_wait<1>();

    if (x == cur.rt + cur.t) cursor_next_row(plan, cur);
    const TileRef t = tile_ref(plan, p, cur, x);
    const bool tile_ok = t.page >= 0 && (int64_t)t.page < p.num_pages;
    const bool piece_start = (x == x_begin) || (t.i == 0);
    const bool piece_end = (x + 1 == x_end) || (t.i + 1 == cur.t);
    const uint32_t kv_base =
        kBf16 ? kv_base0 + (uint32_t)((k & 1) * kTile * kRowBytes) : kv_base0;

    if (piece_start) {
      // stage q[b][j][:][:] into shared memory (f16 with per-head power-of-two scale for
      // e4m3 caches, bf16 as is otherwise)
      const int b = t.r / p.nq, j = t.r - b * p.nq;
      const __nv_bfloat16* qrow = p.q + (((int64_t)b * p.nq + j) * H) * kDEntry;
      for (int h = warp; h < H; h += kThreads / 32) {
        const uint4* src = reinterpret_cast<const uint4*>(qrow + (int64_t)h * kDEntry);
        uint4 v[3];
        float amax = 0.f;
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          const int ch = lane + 32 * u;
          v[u] = ch < 72 ? __ldg(src + ch) : make_uint4(0, 0, 0, 0);
          const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
#pragma unroll
          for (int q2 = 0; q2 < 4; ++q2) {
            float2 f = __bfloat1622float2(e[q2]);
            amax = fmaxf(amax, fmaxf(fabsf(f.x), fabsf(f.y)));
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
        int shift = 0;
        if constexpr (!kBf16) {
          if (amax > 0.f && isfinite(amax)) {
            int e;
            frexpf(amax, &e);  // amax in [2^(e-1), 2^e)
            shift = 15 - e;    // scaled max in [2^14, 2^15)
          }
        }
        const float sc = ldexpf(1.0f, shift);
#pragma unroll
        for (int u = 0; u < 3; ++u) {
          const int ch = lane + 32 * u;
          if (ch >= 72) continue;
          uint4 o = v[u];
          if constexpr (!kBf16) {
            const __nv_bfloat162* e = reinterpret_cast<const __nv_bfloat162*>(&v[u]);
            uint32_t w[4];
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2) {
              float2 f = __bfloat1622float2(e[q2]);
              w[q2] = pack2<false>(f.x * sc, f.y * sc);
            }
            o = make_uint4(w[0], w[1], w[2], w[3]);
          }
          asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(q_base + tile_off(h, ch)),
                       "r"(o.x), "r"(o.y), "r"(o.z), "r"(o.w));
        }
        if (lane == 0) qmul[h] = p.score_mul * ldexpf(1.0f, -shift);
      }
      m0 = m1 = -INFINITY;
      l0 = l1 = 0.f;
#pragma unroll
      for (int n = 0; n < 32; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
      piece_bad = false;
    }
    if (!tile_ok) {
      piece_bad = true;
      if (tid == 0) atomicOr(p.ws.status, MLA_DEVICE_ERR_BAD_PAGE);
    }
    __syncthreads();  // stage of tile x landed for every thread; q staged

    if constexpr (!kBf16) {
      // e4m3 -> f16 into the swizzled tile
      const uint8_t* st = smem + S::stage + (k & 1) * kTile * kDEntry;
      for (int v = tid; v < kTile * (kDEntry / 16); v += kThreads) {
        const int tok = v / (kDEntry / 16), c16 = v - tok * (kDEntry / 16);
        const uint4 raw = *reinterpret_cast<const uint4*>(st + v * 16);
        const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
        uint32_t h[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          h[2 * i] = e4m3x2_to_f16x2((uint16_t)(w[i] & 0xffffu));
          h[2 * i + 1] = e4m3x2_to_f16x2((uint16_t)(w[i] >> 16));
        }
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                         kv_base + tile_off(tok, 2 * c16)),
                     "r"(h[0]), "r"(h[1]), "r"(h[2]), "r"(h[3]));
        asm volatile("st.shared.v4.b32 [%0], {%1,%2,%3,%4};\n" ::"r"(
                         kv_base + tile_off(tok, 2 * c16 + 1)),
                     "r"(h[4]), "r"(h[5]), "r"(h[6]), "r"(h[7]));
      }
      __syncthreads();
    }

    // ---- S = Q K^T : warp (hg, xh) covers heads [16hg, 16hg+16) x tokens [32xh, 32xh+32)
    float sacc[4][4];
    float alpha0 = 1.f, alpha1 = 1.f, mu0 = 0.f, mu1 = 0.f;
    if (computes) {
#pragma unroll
      for (int n = 0; n < 4; ++n) sacc[n][0] = sacc[n][1] = sacc[n][2] = sacc[n][3] = 0.f;
#pragma unroll 4
      for (int ks = 0; ks < kDEntry / 16; ++ks) {
        uint32_t a[4];
        ldsm_x4(q_base + tile_off(16 * hg + (lane & 15), 2 * ks + (lane >> 4)), a);
#pragma unroll
        for (int i2 = 0; i2 < 2; ++i2) {
          const int mm = lane >> 3;
          const int tok = 32 * xh + 16 * i2 + (mm >> 1) * 8 + (lane & 7);
          uint32_t bb[4];
          ldsm_x4(kv_base + tile_off(tok, 2 * ks + (mm & 1)), bb);
          mma16816<kBf16>(sacc[2 * i2], a, bb[0], bb[1]);
          mma16816<kBf16>(sacc[2 * i2 + 1], a, bb[2], bb[3]);
        }
      }
      // scale to log2 units, mask, partial row max over this warp's 32 tokens
      const float c0 = qmul[row0], c1 = qmul[row1];
      float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = 32 * xh + 8 * n + 2 * tq + e;
          const bool vis = tile_ok && tok < t.valid;
          sacc[n][e] = vis ? sacc[n][e] * c0 : -INFINITY;
          sacc[n][2 + e] = vis ? sacc[n][2 + e] * c1 : -INFINITY;
          mx0 = fmaxf(mx0, sacc[n][e]);
          mx1 = fmaxf(mx1, sacc[n][2 + e]);
        }
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      if (tq == 0) {
        red_max[xh * H + row0] = mx0;
        red_max[xh * H + row1] = mx1;
      }
    }
    __syncthreads();
    if (computes) {
      const float mt0 = fmaxf(red_max[row0], red_max[H + row0]);
      const float mt1 = fmaxf(red_max[row1], red_max[H + row1]);
      const float mn0 = fmaxf(m0, mt0), mn1 = fmaxf(m1, mt1);
      alpha0 = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - mn0);
      alpha1 = (m1 == -INFINITY) ? 0.f : fast_exp2(m1 - mn1);
      m0 = mn0;
      m1 = mn1;
      mu0 = (m0 == -INFINITY) ? 0.f : m0 - (float)kPOffset;
      mu1 = (m1 == -INFINITY) ? 0.f : m1 - (float)kPOffset;
      float s0 = 0.f, s1 = 0.f;
#pragma unroll
      for (int n = 0; n < 4; ++n) {
        const float p00 = fast_exp2(sacc[n][0] - mu0), p01 = fast_exp2(sacc[n][1] - mu0);
        const float p10 = fast_exp2(sacc[n][2] - mu1), p11 = fast_exp2(sacc[n][3] - mu1);
        s0 += p00 + p01;
        s1 += p10 + p11;
        const int ch = 4 * xh + n;  // 8 tokens per 16-byte chunk
        const uint32_t off0 = p_off(row0, ch) + 4 * tq, off1 = p_off(row1, ch) + 4 * tq;
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(p_base + off0), "r"(pack2<kBf16>(p00, p01)));
        asm volatile("st.shared.b32 [%0], %1;\n" ::"r"(p_base + off1), "r"(pack2<kBf16>(p10, p11)));
      }
#pragma unroll
      for (int o = 1; o < 4; o <<= 1) {
        s0 += __shfl_xor_sync(0xffffffffu, s0, o);
        s1 += __shfl_xor_sync(0xffffffffu, s1, o);
      }
      if (tq == 0) {
        red_sum[xh * H + row0] = s0;
        red_sum[xh * H + row1] = s1;
      }
    }
    __syncthreads();
    if (computes) {
      l0 = l0 * alpha0 + red_sum[row0] + red_sum[H + row0];
      l1 = l1 * alpha1 + red_sum[row1] + red_sum[H + row1];
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        oacc[n][0] *= alpha0;
        oacc[n][1] *= alpha0;
        oacc[n][2] *= alpha1;
        oacc[n][3] *= alpha1;
      }
      // ---- O += P V : warp (hg, xh) covers heads [16hg, +16) x dims [256xh, +256)
#pragma unroll
      for (int kk = 0; kk < kTile / 16; ++kk) {
        uint32_t a[4];
        ldsm_x4(p_base + p_off(16 * hg + (lane & 15), 2 * kk + (lane >> 4)), a);
        const int mm = lane >> 3;
        const int tok = 16 * kk + (mm & 1) * 8 + (lane & 7);
#pragma unroll
        for (int np = 0; np < 16; ++np) {
          uint32_t bb[4];
          ldsm_x4_t(kv_base + tile_off(tok, 32 * xh + 2 * np + (mm >> 1)), bb);
          mma16816<kBf16>(oacc[2 * np], a, bb[0], bb[1]);
          mma16816<kBf16>(oacc[2 * np + 1], a, bb[2], bb[3]);
        }
      }
    }

    if (piece_end && computes) {
      const int slot = cur.base + (c - plan.cta_of(cur.rt));
      const float inv0 = l0 > 0.f ? p.kv_scale / l0 : 0.f;
      const float inv1 = l1 > 0.f ? p.kv_scale / l1 : 0.f;
      float* o0 = p.ws.part_out + ((int64_t)slot * H + row0) * kDLatent + 256 * xh + 2 * tq;
      float* o1 = p.ws.part_out + ((int64_t)slot * H + row1) * kDLatent + 256 * xh + 2 * tq;
#pragma unroll
      for (int n = 0; n < 32; ++n) {
        *reinterpret_cast<float2*>(o0 + 8 * n) = make_float2(oacc[n][0] * inv0, oacc[n][1] * inv0);
        *reinterpret_cast<float2*>(o1 + 8 * n) = make_float2(oacc[n][2] * inv1, oacc[n][3] * inv1);
      }
      if (xh == 0 && tq == 0) {
        p.ws.part_lse[(int64_t)slot * H + row0] =
            l0 > 0.f ? (mu0 + log2f(l0)) * kLn2 : -INFINITY;
        p.ws.part_lse[(int64_t)slot * H + row1] =
            l1 > 0.f ? (mu1 + log2f(l1)) * kLn2 : -INFINITY;
      }
      if (tid == 0) p.ws.piece_err[slot] = piece_bad ? 1 : 0;
    }
    __syncthreads();  // kv tile, stage buffer and P are reused by the next tile
  }
  cp_async_wait<0>();
}

template <bool kBf16, int HG>
cudaError_t launch_decode_mma(const DecodeParams& p, cudaStream_t stream) {
  constexpr int H = 16 * HG;
  constexpr int smem = Smem<kBf16, H>::total;
  static_assert(smem <= 232448, "shared memory budget");
  static std::atomic<int> configured[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && !configured[dev].load()) {
    cudaError_t e = cudaFuncSetAttribute(decode_mma_kernel<kBf16, HG>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    configured[dev].store(1);
  }
  decode_mma_kernel<kBf16, HG><<<p.G, kThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

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

extern "C" size_t mla_decode_workspace_size(int batch, int num_queries, int num_heads,
                                            int num_ctas) {
  if (batch < 0 || num_queries < 1 || num_queries > MLA_MAX_QUERIES || num_heads <= 0 ||
      num_ctas < 0)
    return 0;
  if (num_ctas == 0) num_ctas = mla::device_sm_count();
  if (num_ctas <= 0) return 0;
  return mla::workspace_layout((int64_t)batch * num_queries, num_heads, num_ctas).total;
}

extern "C" mla_status mla_decode(const void* q, const void* kv_pages, int64_t num_pages,
                                 int page_size, int kv_dtype, const int32_t* block_table,
                                 int max_pages, const int32_t* seq_lens, int batch,
                                 int num_queries, int num_heads, float sm_scale, float kv_scale,
                                 int num_ctas, void* workspace, size_t workspace_bytes, void* out,
                                 float* lse, mla_stream_t stream) {
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
  const WorkspaceLayout L = workspace_layout(rows, num_heads, G);
  if (workspace_bytes < L.total) return MLA_ERR_WORKSPACE;

  uint8_t* ws = static_cast<uint8_t*>(workspace);
  DecodeParams p;
  p.q = static_cast<const __nv_bfloat16*>(q);
  p.kv = static_cast<const uint8_t*>(kv_pages);
  p.num_pages = num_pages;
  p.block_table = block_table;
  p.max_pages = max_pages;
  p.seq_lens = seq_lens;
  p.batch = batch;
  p.nq = num_queries;
  p.score_mul = sm_scale * kLog2e * kv_scale;
  p.kv_scale = kv_scale;
  p.G = G;
  p.ws.status = reinterpret_cast<unsigned*>(ws);
  p.ws.row_base = reinterpret_cast<int32_t*>(ws + L.row_base);
  p.ws.row_np = reinterpret_cast<int32_t*>(ws + L.row_np);
  p.ws.piece_err = reinterpret_cast<int32_t*>(ws + L.piece_err);
  p.ws.part_lse = reinterpret_cast<float*>(ws + L.part_lse);
  p.ws.part_out = reinterpret_cast<float*>(ws + L.part_out);

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t e;
  const bool bf16 = kv_dtype == MLA_KV_BF16;
  switch (num_heads) {
    case 16: e = bf16 ? launch_decode_mma<true, 1>(p, s) : launch_decode_mma<false, 1>(p, s); break;
    case 32: e = bf16 ? launch_decode_mma<true, 2>(p, s) : launch_decode_mma<false, 2>(p, s); break;
    default: e = bf16 ? launch_decode_mma<true, 4>(p, s) : launch_decode_mma<false, 4>(p, s); break;
  }
  if (e != cudaSuccess) return MLA_ERR_CUDA;
  e = launch_combine_pieces(p.ws, (int)rows, num_heads, G, static_cast<__nv_bfloat16*>(out), lse,
                            s);
  return e == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
