// Single-token decode over a paged KV cache for sm_103a.
//
// The cache is stored in fixed-size blocks of 16 token slots; a block table
// maps each sequence's logical block to a physical one, and every key
// position is translated through it ("Fast attention kernels and operator
// fusion accelerate AI models", section "FlashAttention-style attention and
// Paged Attention").  The softmax is the running-max / running-sum form of
// "Advanced attention mechanisms – II", section "Incremental / online
// softmax", applied block by block.
//
// Work unit = (sequence b, KV head g, split s): `split_blocks` consecutive
// logical blocks.  The G = Hq/Hkv query heads that share KV head g are
// processed together so each K/V block is read from HBM once.
//   warp 4        producer: translates the split's table entries, then TMA-
//                 copies each (block, head) K and V slice (16 x d bf16,
//                 128-byte swizzle) into an 8-stage shared-memory ring
//   warps 0..3    consumers: block i goes to warp i % 4; scores and P V are
//                 16x8x16 warp MMAs (rows = the G query heads, zero-padded to
//                 16); each warp keeps its own running max / sum / O
// The four warp states are merged in shared memory and the split's partial
// (unnormalised O, max, sum) goes to the workspace; a second kernel merges
// the splits of each (b, query head) into O and LSE.
#include <cuda_runtime.h>

#include "decode_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kBS = 16;          // block_size (token slots per physical block)
constexpr int kConsumers = 4;    // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
constexpr int kStages = 8;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kBox = kBS * 128;          // one 64-column box of a block: 2 KB
  static constexpr int kHalf = kBS * D * 2;       // K (or V) slice of one (block, head)
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kRing = kStages * kStage;
  static constexpr int kComb = kConsumers * 16 * (D + 2) * 4;
  static_assert(kComb <= kRing, "merge buffer reuses the ring");
  static constexpr int kOffShared = kRing;
  static constexpr int kSmem = kRing + 1024 + 1024;
};

struct DecShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  int phys[kMaxSplitBlocks];
  int abort;
};

struct DecParams {
  const __nv_bfloat16* q;
  const int* block_table;
  const int* seq_lens;
  float* ws_o;
  float* ws_ml;
  int Hq, Hkv, group, max_blocks, num_blocks, split_blocks, max_splits;
  float scale_log2;
  unsigned int* status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ int clamp_len(int L, int Lmax, unsigned int* status, bool report) {
  if (L < 0 || L > Lmax) {
    if (report) atomicOr(status, kDevBadSeqLen);
    return L < 0 ? 0 : Lmax;
  }
  return L;
}

template <int D>
__global__ void __launch_bounds__(kThreads)
    attn_decode_paged_kernel(const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv, const DecParams p) {
  using Lt = DecLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  DecShared* sh = reinterpret_cast<DecShared*>(smem + Lt::kOffShared);
  const uint32_t ring = smem_addr(smem);

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  const int L = clamp_len(p.seq_lens[b], p.max_blocks * kBS, p.status,
                          threadIdx.x == 0 && split == 0 && g == 0);
  const int nblk = (L + kBS - 1) / kBS;
  const int blk0 = split * p.split_blocks;
  if (blk0 >= nblk) return;                      // whole CTA, before any barrier
  const int nb = min(p.split_blocks, nblk - blk0);

  // Translate this split's logical blocks through the block table.
  if (threadIdx.x < nb) {
    int ph = p.block_table[static_cast<size_t>(b) * p.max_blocks + blk0 + threadIdx.x];
    if (ph < 0 || ph >= p.num_blocks) {
      atomicOr(p.status, kDevBadBlock);
      ph = -1;
    }
    sh->phys[threadIdx.x] = ph;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sh->full[s]), 1);
      mbar_init(smem_addr(&sh->empty[s]), 1);
    }
    sh->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{&sh->abort, p.status, p.timeout_ns};

  float m0 = -INFINITY, m1 = -INFINITY;   // running max (exp2 domain), rows r and r+8
  float l0 = 0.f, l1 = 0.f;               // running sums (this lane's columns only)
  float oacc[D / 8][4];
#pragma unroll
  for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const int r0 = lane >> 2;               // fragment row (query head within the group)
  const int cq = (lane & 3) * 2;          // fragment column pair

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      int issued = 0;
      for (int i = 0; i < nb; ++i) {
        const int st = i % kStages;
        if (!mbar_wait(smem_addr(&sh->empty[st]), ((i / kStages) & 1) ^ 1, wc)) break;
        const uint32_t fb = smem_addr(&sh->full[st]);
        const int ph = sh->phys[i];
        if (ph >= 0) {
          const int row = (ph * p.Hkv + g) * kBS;
          const uint32_t dst = ring + st * Lt::kStage;
          mbar_arrive_expect_tx(fb, Lt::kStage);
#pragma unroll
          for (int c = 0; c < Lt::kChunks; ++c) {
            tma_load_2d(dst + c * Lt::kBox, &tk, fb, c * 64, row);
            tma_load_2d(dst + Lt::kHalf + c * Lt::kBox, &tv, fb, c * 64, row);
          }
        } else {
          mbar_arrive(fb);
        }
        ++issued;
      }
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int fills = (issued - 1 - st) / kStages + 1;
        mbar_wait(smem_addr(&sh->full[st]), (fills - 1) & 1, wc, true);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    const float sl2 = p.scale_log2;
    uint32_t qa[D / 16][4];
    {
      const __nv_bfloat16* qg = p.q + (static_cast<size_t>(b) * p.Hq + g * G) * D;
      const bool v0 = r0 < G, v1 = r0 + 8 < G;
#pragma unroll
      for (int ks = 0; ks < D / 16; ++ks) {
        const int c = ks * 16 + cq;
        qa[ks][0] = v0 ? *reinterpret_cast<const uint32_t*>(qg + r0 * D + c) : 0u;
        qa[ks][1] = v1 ? *reinterpret_cast<const uint32_t*>(qg + (r0 + 8) * D + c) : 0u;
        qa[ks][2] = v0 ? *reinterpret_cast<const uint32_t*>(qg + r0 * D + c + 8) : 0u;
        qa[ks][3] = v1 ? *reinterpret_cast<const uint32_t*>(qg + (r0 + 8) * D + c + 8) : 0u;
      }
    }
    for (int i = warp; i < nb; i += kConsumers) {
      const int st = i % kStages;
      if (!mbar_wait_warp(smem_addr(&sh->full[st]), (i / kStages) & 1, wc)) break;
      const int ph = sh->phys[i];
      const int nvalid = min(kBS, L - (blk0 + i) * kBS);
      if (ph >= 0) {
        const uint32_t sK = ring + st * Lt::kStage;
        const uint32_t sV = sK + Lt::kHalf;
        if (nvalid < kBS) {
          // Slots past the sequence end may hold anything (even NaN): zero
          // their V rows so that P = 0 cannot meet NaN in the MMA.
          const int words = (kBS - nvalid) * Lt::kChunks * 8;
          for (int idx = lane; idx < words; idx += 32) {
            const int rr = nvalid + idx / (Lt::kChunks * 8);
            const int rem = idx % (Lt::kChunks * 8);
            const uint32_t a = sV + (rem >> 3) * Lt::kBox + rr * 128 + (rem & 7) * 16;
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
          }
          __syncwarp();
        }
        // S = Q K^T : two 8-key column tiles.
        float sc[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
          const int key = nt * 8 + (lane & 7);
#pragma unroll
          for (int kk2 = 0; kk2 < D / 32; ++kk2) {
            const int c = 4 * kk2 + (lane >> 3);
            const uint32_t addr =
                sK + (c >> 3) * Lt::kBox + key * 128 + (((c & 7) ^ (key & 7)) << 4);
            uint32_t bb[4];
            ldsm_x4(addr, bb);
            mma_16816(sc[nt], qa[2 * kk2], bb[0], bb[1]);
            mma_16816(sc[nt], qa[2 * kk2 + 1], bb[2], bb[3]);
          }
        }
        // Mask slots past the end, running max / sum, rescale O.
        float x[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int kl = nt * 8 + cq + (e & 1);
            x[nt][e] = (kl < nvalid) ? sc[nt][e] * sl2 : -INFINITY;
          }
        float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
        float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);   // finite: slot 0 is valid
        const float a0 = ex2(m0 - mn0), a1 = ex2(m1 - mn1);
        float pr[2][4];
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
          pr[nt][0] = ex2(x[nt][0] - mn0);
          pr[nt][1] = ex2(x[nt][1] - mn0);
          pr[nt][2] = ex2(x[nt][2] - mn1);
          pr[nt][3] = ex2(x[nt][3] - mn1);
        }
        l0 = l0 * a0 + (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
        l1 = l1 * a1 + (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int dt = 0; dt < D / 8; ++dt) {
          oacc[dt][0] *= a0;
          oacc[dt][1] *= a0;
          oacc[dt][2] *= a1;
          oacc[dt][3] *= a1;
        }
        // The score accumulator layout is the A-operand layout of P.
        uint32_t pa[4];
        pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
        pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
        pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
        pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
        // O += P V : V rows are keys, transposed on load.
        const int vkey = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
        for (int dt2 = 0; dt2 < D / 16; ++dt2) {
          const int c = 2 * dt2 + (lane >> 4);
          const uint32_t addr =
              sV + (c >> 3) * Lt::kBox + vkey * 128 + (((c & 7) ^ (vkey & 7)) << 4);
          uint32_t bb[4];
          ldsm_x4_trans(addr, bb);
          mma_16816(oacc[2 * dt2], pa, bb[0], bb[1]);
          mma_16816(oacc[2 * dt2 + 1], pa, bb[2], bb[3]);
        }
        if (nvalid < kBS) fence_proxy_async_smem();   // zeroed rows before the next TMA write
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&sh->empty[st]));
    }
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
  }

  // ------------------------------------------- merge the four warp states
  __syncthreads();                         // ring no longer read by anyone
  float* comb = reinterpret_cast<float*>(smem);             // [4][16][D]
  float* cml = comb + kConsumers * 16 * D;                  // [4][16][2]
  if (warp < kConsumers) {
#pragma unroll
    for (int dt = 0; dt < D / 8; ++dt) {
      const int d = dt * 8 + cq;
      *reinterpret_cast<float2*>(&comb[(warp * 16 + r0) * D + d]) = make_float2(oacc[dt][0], oacc[dt][1]);
      *reinterpret_cast<float2*>(&comb[(warp * 16 + r0 + 8) * D + d]) = make_float2(oacc[dt][2], oacc[dt][3]);
    }
    if ((lane & 3) == 0) {
      cml[(warp * 16 + r0) * 2 + 0] = m0;
      cml[(warp * 16 + r0) * 2 + 1] = l0;
      cml[(warp * 16 + r0 + 8) * 2 + 0] = m1;
      cml[(warp * 16 + r0 + 8) * 2 + 1] = l1;
    }
  }
  __syncthreads();
  for (int idx = threadIdx.x; idx < G * D; idx += kThreads) {
    const int r = idx / D;
    const int d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kConsumers; ++w) M = fmaxf(M, cml[(w * 16 + r) * 2]);
    float acc = 0.f, lsum = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) {
        const float wt = ex2(cml[(w * 16 + r) * 2] - M);
        acc += wt * comb[(w * 16 + r) * D + d];
        lsum += wt * cml[(w * 16 + r) * 2 + 1];
      }
    }
    const size_t slot = (static_cast<size_t>(b) * p.Hq + g * G + r) * p.max_splits + split;
    p.ws_o[slot * D + d] = acc;
    if (d == 0) {
      p.ws_ml[slot * 2 + 0] = M;
      p.ws_ml[slot * 2 + 1] = lsum;
    }
  }
}

struct CombineParams {
  const int* seq_lens;
  const float* ws_o;
  const float* ws_ml;
  __nv_bfloat16* o;
  float* lse;
  int Hq, max_blocks, split_blocks, max_splits;
};

// One warp per (sequence, query head): exact merge of the split partials.
// Lane s holds split s's (max, sum); the weights come from warp reductions
// and every split's partial row is loaded before any is accumulated.
template <int D>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const CombineParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 4 + warp;
  const int b = blockIdx.y;
  if (h >= p.Hq) return;
  int L = p.seq_lens[b];
  L = L < 0 ? 0 : min(L, p.max_blocks * kBS);
  const int nblk = (L + kBS - 1) / kBS;
  const int nsplit = (nblk + p.split_blocks - 1) / p.split_blocks;
  const size_t base = (static_cast<size_t>(b) * p.Hq + h) * p.max_splits;
  float M = -INFINITY;
  for (int s0 = 0; s0 < nsplit; s0 += 32)
    if (s0 + lane < nsplit) M = fmaxf(M, p.ws_ml[(base + s0 + lane) * 2]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  if (M != -INFINITY) {
    for (int s0 = 0; s0 < nsplit; s0 += 32) {
      const int cnt = min(32, nsplit - s0);
      float w = 0.f, lw = 0.f;
      if (lane < cnt) {
        w = ex2(p.ws_ml[(base + s0 + lane) * 2] - M);
        lw = w * p.ws_ml[(base + s0 + lane) * 2 + 1];
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
      lsum += lw;
      for (int s = 0; s < cnt; s += 4) {
        float v[4][D / 32], ws[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          ws[u] = __shfl_sync(0xffffffffu, w, min(s + u, 31));
          const float* src = p.ws_o + (base + s0 + min(s + u, cnt - 1)) * D;
#pragma unroll
          for (int e = 0; e < D / 32; ++e) v[u][e] = src[lane + 32 * e];
        }
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (s + u < cnt)
#pragma unroll
            for (int e = 0; e < D / 32; ++e) acc[e] += ws[u] * v[u][e];
      }
    }
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
  __nv_bfloat16* dst = p.o + (static_cast<size_t>(b) * p.Hq + h) * D;
#pragma unroll
  for (int e = 0; e < D / 32; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(acc[e] * inv);
  if (lane == 0 && p.lse != nullptr)
    p.lse[static_cast<size_t>(b) * p.Hq + h] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : -INFINITY;
}

template <int D>
cudaError_t launch_t(const DecLaunch& a) {
  using Lt = DecLayout<D>;
  auto kern = attn_decode_paged_kernel<D>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lt::kSmem);
  if (e != cudaSuccess) return e;
  float* ws_o = a.workspace;
  float* ws_ml = ws_o + static_cast<size_t>(a.num_seqs) * a.Hq * a.max_splits * D;
  DecParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.split_blocks = a.split_blocks;
  p.max_splits = a.max_splits;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  dim3 grid(a.max_splits, a.Hkv, a.num_seqs);
  kern<<<grid, kThreads, Lt::kSmem, a.stream>>>(*a.tk, *a.tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CombineParams c;
  c.seq_lens = a.seq_lens;
  c.ws_o = ws_o;
  c.ws_ml = ws_ml;
  c.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  c.lse = a.lse;
  c.Hq = a.Hq;
  c.max_blocks = a.max_blocks;
  c.split_blocks = a.split_blocks;
  c.max_splits = a.max_splits;
  dim3 cgrid((a.Hq + 3) / 4, a.num_seqs);
  attn_decode_combine_kernel<D><<<cgrid, 128, 0, a.stream>>>(c);
  return cudaGetLastError();
}

}  // namespace

size_t decode_workspace_floats(int num_seqs, int Hq, int d, int max_splits) {
  return static_cast<size_t>(num_seqs) * Hq * max_splits * (static_cast<size_t>(d) + 2);
}

cudaError_t launch_decode_sm103(const DecLaunch& a) {
  return a.d == 128 ? launch_t<128>(a) : launch_t<64>(a);
}

}  // namespace attn47
