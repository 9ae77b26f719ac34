// Internal launcher interface of the Mamba-2 SSD kernels (not part of the C-ABI).
#pragma once

#include <cstddef>
#include <cuda_runtime.h>

namespace attn47 {

struct SsdLaunch {
  const void* x;          // [batch, L, H, P] bf16
  const float* dt;        // [batch, L, H]
  const float* A;         // [H]
  const void* B;          // [batch, L, G, N] bf16
  const void* C;          // [batch, L, G, N] bf16
  const float* h0;        // [batch, H, P, N] or nullptr (zero initial state)
  void* y;                // [batch, L, H, P] bf16
  float* h_final;         // [batch, H, P, N]
  void* workspace;        // ssd_workspace_bytes(...)
  int batch, L, H, G, N, chunk;
  cudaStream_t stream;
};

size_t ssd_workspace_bytes(int batch, int L, int H, int N, int chunk);
int ssd_head_dim();
cudaError_t launch_ssd_sm103(const SsdLaunch& a);

}  // namespace attn47
