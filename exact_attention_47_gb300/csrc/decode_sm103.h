// Internal launcher interface of the paged-decode kernels (not part of the C-ABI).
#pragma once

#include <cstddef>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn47 {

// Every decode CTA takes at least 2 * kMinSplitBlocks (sequence, KV head,
// block) triples; this bounds the number of partial results per sequence.
constexpr int kMinSplitBlocks = 8;

struct DecLaunch {
  // Cache maps, 3-D {64 columns, num_blocks*Hkv*16 rows (stride d*2 bytes),
  // d/64 column halves (stride 128 bytes)}, box {64, 16, d/64}, 128-byte
  // swizzle: one copy lands a whole (block, head) slice as d/64 swizzled
  // 16 x 64 tiles.
  const CUtensorMap* tk;
  const CUtensorMap* tv;
  const void* q;           // [num_seqs, Hq, d] bf16
  const void* k_cache;     // [num_blocks, Hkv, 16, d] bf16
  const void* v_cache;
  const int* block_table;  // [num_seqs, max_blocks]
  const int* seq_lens;     // [num_seqs]
  void* o;                 // [num_seqs, Hq, d] bf16
  float* lse;              // [num_seqs, Hq] or nullptr
  float* workspace;        // decode_workspace_bytes(...) bytes
  int num_seqs, Hq, Hkv, d, max_blocks, num_blocks;
  int sms;                 // SM count of the device
  int max_ctas;            // 0: one full wave of CTAs
  int early_plan;          // 1: read seq_lens / block_table before the preceding kernel ends;
                           // 2: also the ring's first fill of cache blocks (not a sequence's last)
  unsigned int epoch;      // per-call tag of the arrival counters (never 0)
  float scale;
  unsigned int* status;
  unsigned long long timeout_ns;
  cudaStream_t stream;
};

int decode_max_parts(int max_blocks_per_seq);
size_t decode_workspace_bytes(int num_seqs, int Hq, int d, int max_blocks_per_seq);
cudaError_t launch_decode_sm103(const DecLaunch& a);

}  // namespace attn47
