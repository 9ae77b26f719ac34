// Append of new key/value rows to the paged KV cache (the write half of a
// chunked prefill).
//
// "Fast attention kernels and operator fusion accelerate AI models", section
// "FlashAttention-style attention and Paged Attention": the cache grows token
// by token in fixed-size blocks, and a block table maps each logical
// position to a physical block.  New token i of sequence b takes position
// ctx_lens[b] + i, i.e. slot (pos % 16) of physical block
// block_table[b][pos / 16].  The slots past the sequence's new length in its
// last block hold no token; they are set to zero so the attention kernel,
// which reads whole blocks with TMA, multiplies zero probabilities by finite
// values there.
//
// Pure data movement: each thread moves one 16-byte piece of a row (a warp
// covers two 256-byte rows of one block for d = 128), grid-stride over
// (sequence, KV head, row, piece).
#include <cuda_runtime.h>

#include "fwd_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kSlots = 16;
constexpr int kThreads = 256;

struct AppendParams {
  const uint4* k_new;
  const uint4* v_new;
  uint4* k_cache;
  uint4* v_cache;
  const int* block_table;
  const int* ctx_lens;
  int Hkv, N, pieces, max_blocks, num_blocks, max_ctx;
  long long rows_per_seq;   // Hkv * (N + 15): new rows plus at most 15 cleared slots
  long long total;          // B * rows_per_seq * pieces
  unsigned int* status;
};

__global__ void __launch_bounds__(kThreads) attn_kv_append_kernel(const AppendParams p) {
  const long long stride = static_cast<long long>(gridDim.x) * kThreads;
  for (long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; idx < p.total;
       idx += stride) {
    const int piece = static_cast<int>(idx % p.pieces);
    const long long r = idx / p.pieces;
    const int b = static_cast<int>(r / p.rows_per_seq);
    const int rr = static_cast<int>(r % p.rows_per_seq);
    const int g = rr / (p.N + kSlots - 1);
    const int t = rr % (p.N + kSlots - 1);        // new row t, or cleared slot t - N past the end
    const int ctx = __ldg(p.ctx_lens + b);
    if (ctx < 0 || ctx > p.max_ctx) {
      if (t == 0 && g == 0 && piece == 0) atomicOr(p.status, kDevBadSeqLen);
      continue;
    }
    const int pos = ctx + t;
    const int end = ctx + p.N;
    if (t >= p.N && pos >= (end + kSlots - 1) / kSlots * kSlots) continue;
    const int phys = __ldg(p.block_table + static_cast<size_t>(b) * p.max_blocks + pos / kSlots);
    if (static_cast<unsigned>(phys) >= static_cast<unsigned>(p.num_blocks)) {
      atomicOr(p.status, kDevBadBlock);
      continue;
    }
    const size_t dst = ((static_cast<size_t>(phys) * p.Hkv + g) * kSlots + pos % kSlots) * p.pieces + piece;
    if (t < p.N) {
      const size_t src = ((static_cast<size_t>(b) * p.Hkv + g) * p.N + t) * p.pieces + piece;
      p.k_cache[dst] = __ldg(p.k_new + src);
      p.v_cache[dst] = __ldg(p.v_new + src);
    } else {
      p.k_cache[dst] = make_uint4(0u, 0u, 0u, 0u);
      p.v_cache[dst] = make_uint4(0u, 0u, 0u, 0u);
    }
  }
}

}  // namespace

cudaError_t launch_kv_append_sm103(const AppendLaunch& a) {
  AppendParams p;
  p.k_new = static_cast<const uint4*>(a.k_new);
  p.v_new = static_cast<const uint4*>(a.v_new);
  p.k_cache = static_cast<uint4*>(a.k_cache);
  p.v_cache = static_cast<uint4*>(a.v_cache);
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.Hkv = a.Hkv;
  p.N = a.N;
  p.pieces = a.d / 8;                            // 16-byte pieces of a row
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.max_ctx = a.max_blocks * kSlots - a.N;
  p.rows_per_seq = static_cast<long long>(a.Hkv) * (a.N + kSlots - 1);
  p.total = static_cast<long long>(a.B) * p.rows_per_seq * p.pieces;
  p.status = a.status;
  const long long blocks = (p.total + kThreads - 1) / kThreads;
  const long long cap = static_cast<long long>(a.sms > 0 ? a.sms : 1) * 8;
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  // A plain launch: as a programmatic dependent (waiting for the preceding
  // kernel, letting the attention kernel launch early) the chunked prefill
  // measured 2.6 % slower on GB300.
  attn_kv_append_kernel<<<grid, kThreads, 0, a.stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn47
