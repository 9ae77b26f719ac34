// Internal launcher interface of the forward kernel and of the paged-cache
// append kernel (not part of the C-ABI).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

namespace attn47 {

struct FwdLaunch {
  const CUtensorMap* tq;   // [B*Hq, N, d] bf16, box {64, fwd_box_rows(), 1}, 128-byte swizzle
  const CUtensorMap* tk;   // [B*Hkv, N, d] (not read in paged mode)
  const CUtensorMap* tv;   // same as tk
  void* o;                 // [B, Hq, N, d] bf16
  float* lse;              // [B, Hq, N] fp32 or nullptr
  int B, Hq, Hkv, N, d;
  bool causal;
  float scale;
  int sms;                 // SMs of the device (persistent grid)
  unsigned int* status;    // device status word
  unsigned long long timeout_ns;
  cudaStream_t stream;
  // Paged mode (chunked prefill; implies causal): the N query rows of
  // sequence b sit at positions ctx_lens[b] .. ctx_lens[b] + N - 1 and K/V
  // come from the paged cache through block_table.
  bool paged = false;
  const void* k_cache = nullptr;      // [num_blocks, Hkv, 16, d] bf16
  const void* v_cache = nullptr;
  const int* block_table = nullptr;   // [B, max_blocks] int32
  const int* ctx_lens = nullptr;      // [B] int32
  int max_blocks = 0, num_blocks = 0;
};

int fwd_box_rows();
cudaError_t launch_fwd_sm103(const FwdLaunch& a);

struct AppendLaunch {
  const void* k_new;       // [B, Hkv, N, d] bf16
  const void* v_new;
  void* k_cache;           // [num_blocks, Hkv, 16, d] bf16
  void* v_cache;
  const int* block_table;  // [B, max_blocks] int32
  const int* ctx_lens;     // [B] int32
  int B, Hkv, N, d, max_blocks, num_blocks, sms;
  unsigned int* status;
  cudaStream_t stream;
};

// Stores the N new K/V rows of every sequence at positions ctx_lens[b] + i
// through the block table and clears the unused slots of its last block.
cudaError_t launch_kv_append_sm103(const AppendLaunch& a);

}  // namespace attn47
