// kv_append.cu -- write new tokens' latent entries into the paged cache.
//
// The write side of "Smaller, faster, safer: running Kimi and GLM at scale",
// section "Quantizing the KV cache": entries are stored as FP8 e4m3 under one
// per-tensor float32 scale. Each stored code is the exact quotient x / scale
// rounded to nearest e4m3, ties to even, saturated to +-448.
//
// Exactness. The quotient is formed with IEEE float32 division. A float32
// quotient can round onto an e4m3 rounding midpoint (a number with 5
// significant bits) while the real quotient lies just beside it, because the
// scale has 24 significant bits. When the float32 quotient is such a midpoint,
// the sign of the exact remainder x - q*scale (one fused multiply-add, exact in
// sign) tells on which side the real quotient lies, and q is moved one float32
// ulp toward it before the hardware rounds to e4m3. Away from midpoints the
// float32 rounding cannot change the e4m3 result.
#include "mla_common.cuh"
#include "mla_internal.h"

namespace mla {
namespace {

// e4m3 code of x / s for s > 0 (round to nearest even, satfinite).
__device__ __forceinline__ float exact_quotient_for_e4m3(float x, float s) {
  float q = __fdiv_rn(x, s);
  float a = fabsf(q);
  if (a <= 448.0f) {  // false for NaN; saturated values need no tie handling
    int e;
    frexpf(a, &e);                       // a = m * 2^e, m in [0.5, 1)
    int el = max(e - 1, -6);             // binade exponent, subnormals share 2^-6
    float t = a * ldexpf(1.0f, 3 - el);  // a in units of the e4m3 spacing, exact
    if (t - floorf(t) == 0.5f) {         // q sits exactly on a midpoint
      float rem = __fmaf_rn(-q, s, x);   // sign of (x - q*s) is exact
      if (rem > 0.0f) q = nextafterf(q, INFINITY);
      else if (rem < 0.0f) q = nextafterf(q, -INFINITY);
    }
  }
  return q;
}

// Two floats -> two e4m3 codes (lo -> low byte), RNE with saturation.
__device__ __forceinline__ uint16_t f32x2_to_e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// One thread converts 8 consecutive elements (16 bytes of bf16 in, 8 bytes out).
// 72 threads cover one token's 576 elements.
__global__ void kv_append_e4m3_kernel(const __nv_bfloat16* __restrict__ latent,
                                      const __nv_bfloat16* __restrict__ rope,
                                      const int32_t* __restrict__ slots, int64_t num_tokens,
                                      uint8_t* __restrict__ kv_pages, int64_t num_slots,
                                      float kv_scale) {
  constexpr int kVecPerToken = kDEntry / 8;  // 72
  griddep_launch_dependents();  // a following decode launch may start its set-up
  int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t tok = gid / kVecPerToken;
  int v = (int)(gid - tok * kVecPerToken);
  if (tok >= num_tokens) return;
  int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) return;
  const __nv_bfloat16* src = (v < kDLatent / 8) ? latent + tok * kDLatent + v * 8
                                                : rope + tok * kDRope + (v - kDLatent / 8) * 8;
  uint4 raw = *reinterpret_cast<const uint4*>(src);
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
  uint16_t codes[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 f = __bfloat1622float2(h[i]);
    codes[i] = f32x2_to_e4m3x2(exact_quotient_for_e4m3(f.x, kv_scale),
                               exact_quotient_for_e4m3(f.y, kv_scale));
  }
  uint2 packed;
  packed.x = (uint32_t)codes[0] | ((uint32_t)codes[1] << 16);
  packed.y = (uint32_t)codes[2] | ((uint32_t)codes[3] << 16);
  *reinterpret_cast<uint2*>(kv_pages + slot * kDEntry + v * 8) = packed;
}

__global__ void kv_append_bf16_kernel(const __nv_bfloat16* __restrict__ latent,
                                      const __nv_bfloat16* __restrict__ rope,
                                      const int32_t* __restrict__ slots, int64_t num_tokens,
                                      __nv_bfloat16* __restrict__ kv_pages, int64_t num_slots) {
  constexpr int kVecPerToken = kDEntry / 8;
  griddep_launch_dependents();  // a following decode launch may start its set-up
  int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  int64_t tok = gid / kVecPerToken;
  int v = (int)(gid - tok * kVecPerToken);
  if (tok >= num_tokens) return;
  int64_t slot = slots[tok];
  if (slot < 0 || slot >= num_slots) return;
  const __nv_bfloat16* src = (v < kDLatent / 8) ? latent + tok * kDLatent + v * 8
                                                : rope + tok * kDRope + (v - kDLatent / 8) * 8;
  *reinterpret_cast<uint4*>(kv_pages + slot * kDEntry + v * 8) =
      *reinterpret_cast<const uint4*>(src);
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace mla

extern "C" mla_status mla_kv_append(const void* latent, const void* rope,
                                    const int32_t* slot_mapping, int64_t num_tokens,
                                    void* kv_pages, int64_t num_pages, int page_size, int kv_dtype,
                                    float kv_scale, mla_stream_t stream) {
  using namespace mla;
  if (num_tokens < 0 || num_pages < 0) return MLA_ERR_INVALID_ARG;
  if (page_size != kPageSize) return MLA_ERR_UNSUPPORTED;
  if (kv_dtype != MLA_KV_E4M3 && kv_dtype != MLA_KV_BF16) return MLA_ERR_INVALID_ARG;
  if (!(kv_scale > 0.0f) || !isfinite(kv_scale)) return MLA_ERR_INVALID_ARG;
  if (kv_dtype == MLA_KV_BF16 && kv_scale != 1.0f) return MLA_ERR_INVALID_ARG;
  if (num_tokens == 0) return MLA_OK;
  if (!latent || !rope || !slot_mapping || !kv_pages) return MLA_ERR_INVALID_ARG;
  if (!aligned16(latent) || !aligned16(rope) || !aligned16(kv_pages) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 3u))
    return MLA_ERR_INVALID_ARG;
  const int64_t num_slots = num_pages * page_size;
  const int64_t threads = num_tokens * (kDEntry / 8);
  const int block = 288;  // 4 tokens per block
  const int64_t grid = (threads + block - 1) / block;
  if (grid > 0x7fffffffLL) return MLA_ERR_UNSUPPORTED;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (kv_dtype == MLA_KV_E4M3) {
    kv_append_e4m3_kernel<<<(unsigned)grid, block, 0, s>>>(
        static_cast<const __nv_bfloat16*>(latent), static_cast<const __nv_bfloat16*>(rope),
        slot_mapping, num_tokens, static_cast<uint8_t*>(kv_pages), num_slots, kv_scale);
  } else {
    kv_append_bf16_kernel<<<(unsigned)grid, block, 0, s>>>(
        static_cast<const __nv_bfloat16*>(latent), static_cast<const __nv_bfloat16*>(rope),
        slot_mapping, num_tokens, static_cast<__nv_bfloat16*>(kv_pages), num_slots);
  }
  return cudaGetLastError() == cudaSuccess ? MLA_OK : MLA_ERR_CUDA;
}
