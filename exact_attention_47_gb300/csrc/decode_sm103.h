// Internal launcher interface of the paged-decode kernels (not part of the C-ABI).
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn47 {

constexpr int kMaxSplitBlocks = 32;   // logical blocks per split, upper bound
constexpr int kMinSplitBlocks = 8;    // lower bound; sizes the workspace

struct DecLaunch {
  const CUtensorMap* tk;   // [num_blocks*Hkv*16, d] bf16, box {64, 16}, 128-byte swizzle
  const CUtensorMap* tv;
  const void* q;           // [num_seqs, Hq, d] bf16
  const int* block_table;  // [num_seqs, max_blocks]
  const int* seq_lens;     // [num_seqs]
  void* o;                 // [num_seqs, Hq, d] bf16
  float* lse;              // [num_seqs, Hq] or nullptr
  float* workspace;        // decode_workspace_floats(num_seqs, Hq, d, max_splits) floats
  int num_seqs, Hq, Hkv, d, max_blocks, num_blocks, split_blocks, max_splits;
  float scale;
  unsigned int* status;
  unsigned long long timeout_ns;
  cudaStream_t stream;
};

size_t decode_workspace_floats(int num_seqs, int Hq, int d, int max_splits);
cudaError_t launch_decode_sm103(const DecLaunch& a);

}  // namespace attn47
