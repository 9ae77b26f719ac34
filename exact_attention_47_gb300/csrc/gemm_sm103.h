// Internal launcher interface of the SwiGLU projection kernel (not part of the C-ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn47 {

struct SwigluProjLaunch {
  // TMA maps (bf16, 128-byte swizzle, box 64 x 128): x as (hidden, rows),
  // W as (hidden, 2F).
  const CUtensorMap* tx;
  const CUtensorMap* tw;
  void* out;              // [rows, F] bf16
  int rows, F, hidden;    // F a multiple of swiglu_proj_tile_features(), hidden of swiglu_proj_k_step()
  int sms;
  unsigned int* status;
  unsigned long long timeout_ns;
  cudaStream_t stream;
};

int swiglu_proj_tile_features();
int swiglu_proj_k_step();
cudaError_t launch_swiglu_proj_sm103(const SwigluProjLaunch& a);

}  // namespace attn47
