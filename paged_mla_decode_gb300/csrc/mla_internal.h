// mla_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mla.h"

namespace mla {

// Typed views of a decode workspace (see WorkspaceLayout in mla_common.cuh).
struct DecodeWorkspace {
  unsigned* status;
  int32_t* row_base;
  int32_t* row_np;
  int32_t* row_np1;   // grouped decode: slots of each row's shared-prefix pieces
  int32_t* piece_err;
  float* part_lse;
  float* part_out;
  uint8_t* q_op;    // FP8 decode only: the split query operand of each row
  float* q_mul;     // FP8 decode only: score multiplier of each (row, head)
};

// Everything a decode kernel launch needs (validated by the caller).
struct DecodeLaunch {
  const __nv_bfloat16* q;
  const uint8_t* kv;
  int64_t num_pages;
  const int32_t* block_table;
  int max_pages;
  const int32_t* seq_lens;
  int batch, nq, heads;
  bool bf16;         // cache holds bf16 (else e4m3 codes)
  float score_mul;   // sm_scale * log2(e) * kv_scale
  float kv_scale;
  int G;             // CTAs launched
  DecodeWorkspace ws;
  // FP8 grouped decode only (else prefix_pages == nullptr): requests
  // [g * forks, (g + 1) * forks) share their first prefix_pages[g] pages
  int forks = 1;
  const int32_t* prefix_pages = nullptr;
};

// Split-KV decode on the tcgen05 tensor cores (decode_tc.cu); heads <= 64.
cudaError_t launch_decode_tensor_core(const DecodeLaunch& d, cudaStream_t stream);

// Split-KV decode with the e4m3 cache bytes as tensor-core operands
// (decode_fp8.cu); e4m3 caches only, heads <= 64, num_pages * 64 < 2^31.
// Launches the query split (one pass per row into ws.q_op / ws.q_mul), then the
// decode kernel, which reads it.
cudaError_t launch_decode_fp8(const DecodeLaunch& d, cudaStream_t stream);

// Merge the pieces written by a decode kernel into out (bf16) and lse (fp32);
// max_pieces_per_row is the number of decode CTAs (it sizes the staging).
cudaError_t launch_combine_pieces(const DecodeWorkspace& ws, int rows, int heads,
                                  int max_pieces_per_row, __nv_bfloat16* out, float* lse,
                                  cudaStream_t stream);

// Launch attribute that lets a kernel start while the previous kernel in the
// stream is finishing (programmatic dependent launch); kernels launched with it
// call griddep_wait() before their first global memory access.
inline cudaLaunchAttribute pdl_attribute() {
  cudaLaunchAttribute a;
  a.id = cudaLaunchAttributeProgrammaticStreamSerialization;
  a.val.programmaticStreamSerializationAllowed = 1;
  return a;
}

// Number of SMs of the current device (cached per device).
int device_sm_count();

}  // namespace mla
