// Internal launcher interface of the forward kernel (not part of the C-ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn47 {

struct FwdLaunch {
  const CUtensorMap* tq;   // [B*Hq, N, d] bf16, box {64, fwd_box_rows(), 1}, 128-byte swizzle
  const CUtensorMap* tk;   // [B*Hkv, N, d]
  const CUtensorMap* tv;   // [B*Hkv, N, d]
  void* o;                 // [B, Hq, N, d] bf16
  float* lse;              // [B, Hq, N] fp32 or nullptr
  int B, Hq, Hkv, N, d;
  bool causal;
  float scale;
  int sms;                 // SMs of the device (persistent grid)
  unsigned int* status;    // device status word
  unsigned long long timeout_ns;
  cudaStream_t stream;
};

int fwd_box_rows();
cudaError_t launch_fwd_sm103(const FwdLaunch& a);

}  // namespace attn47
