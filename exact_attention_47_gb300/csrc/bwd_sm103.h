// Internal launcher interface of the backward kernels (not part of the C-ABI).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

namespace attn47 {

struct BwdLaunch {
  const CUtensorMap* tq;   // [B*Hq, N, d] bf16, box {64, bwd_box_rows(), 1}, 128-byte swizzle
  const CUtensorMap* tk;   // [B*Hkv, N, d]
  const CUtensorMap* tv;   // [B*Hkv, N, d]
  const CUtensorMap* tdo;  // [B*Hq, N, d]
  const void* o;           // [B, Hq, N, d] bf16 (forward output)
  const void* dout;        // [B, Hq, N, d] bf16 (dL/dO)
  const float* lse;        // [B, Hq, N] fp32 (forward LSE, natural log)
  void* dq;                // [B, Hq, N, d] bf16
  void* dk;                // [B, Hkv, N, d] bf16
  void* dv;                // [B, Hkv, N, d] bf16
  int B, Hq, Hkv, N, d;
  bool causal;
  float scale;
  float* workspace;        // bwd_workspace_bytes(B, Hq, N)
  unsigned int* status;
  unsigned long long timeout_ns;
  cudaStream_t stream;
};

// Kernel parameters (device side).
struct BwdParams {
  const __nv_bfloat16* o;
  const __nv_bfloat16* dout;
  const float* lse;
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  int N, n_pad, Hq, Hkv, group, bh_q, bh_kv;
  float scale, scale_log2;
  float* ws_lse2;          // [B*Hq, n_pad] lse * log2(e)
  float* ws_d;             // [B*Hq, n_pad] rowsum(dO * O)
  unsigned int* status;
  unsigned long long timeout_ns;
};

size_t bwd_workspace_bytes(int B, int Hq, int N);
int bwd_box_rows();
cudaError_t launch_bwd_sm103(const BwdLaunch& a);

}  // namespace attn47
