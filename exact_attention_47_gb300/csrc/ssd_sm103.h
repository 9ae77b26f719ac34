// Internal launcher interface of the Mamba-2 SSD kernels (not part of the C-ABI).
#pragma once

#include <cstddef>
#include <cuda.h>
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
  // TMA maps (128-byte swizzle): x as (P, H, L, batch) with box
  // (64, 1, 64, 1); B the same over (N, G, L, batch); C with box
  // (64, 1, 128, 1); the chunk states in the workspace as
  // (N, batch * nc * H * P) with box (64, 64).
  const CUtensorMap* tx;
  const CUtensorMap* tb;
  const CUtensorMap* tc;
  const CUtensorMap* ts;
  int batch, L, H, G, N, chunk;
  unsigned int* status;
  unsigned long long timeout_ns;
  cudaStream_t stream;
};

size_t ssd_workspace_bytes(int batch, int L, int H, int N, int chunk);
// Byte offset of the chunk states within the workspace.
size_t ssd_states_offset(int batch, int L, int H, int chunk);
int ssd_head_dim();
cudaError_t launch_ssd_sm103(const SsdLaunch& a);

}  // namespace attn47
