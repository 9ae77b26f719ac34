// Internal launcher interface of the operator-fusion kernels (not part of the C-ABI).
#pragma once

#include <cuda_runtime.h>

namespace attn47 {

struct NormLaunch {
  const void* x;         // [rows, hidden] bf16
  void* residual;        // [rows, hidden] bf16, read and overwritten with bf16(x + residual)
  const void* weight;    // [hidden] bf16
  void* out;             // [rows, hidden] bf16
  int rows, hidden;      // hidden a multiple of 8
  float eps;
  int sms;
  cudaStream_t stream;
};

struct GluLaunch {
  const void* gate_up;   // [rows, 2F] bf16: gate columns 0..F-1, up columns F..2F-1
  void* out;             // [rows, F] bf16
  int rows, F;           // F a multiple of 8
  int sms;
  cudaStream_t stream;
};

cudaError_t launch_add_rmsnorm_sm103(const NormLaunch& a);
cudaError_t launch_swiglu_sm103(const GluLaunch& a);

}  // namespace attn47
