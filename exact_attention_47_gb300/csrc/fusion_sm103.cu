// Operator fusions beside attention: residual add + RMSNorm, and the SwiGLU
// activation ("Fast attention kernels and operator fusion accelerate AI
// models", section "Operator fusion": each of these is several kernels and
// several HBM round trips of an intermediate tensor when run naively; fused,
// every input is read once and every output written once, and the
// mathematical function is unchanged).
//
// Both are HBM-bound: a few flops per byte.  Loads and stores are 16 bytes
// (8 bf16) per thread and consecutive threads touch consecutive 16-byte
// pieces, so every warp instruction moves 512 contiguous bytes.
//
// add + RMSNorm: one warp per row.  Pass 1 reads x and the residual in
// batches of four pieces per lane (eight loads in flight), stores the new
// residual r = bf16(x + residual) and sums r^2 of the stored values; a warp
// reduction gives the row's mean square; pass 2 re-reads r (the lane's own
// stores, from L1/L2) and the weight and writes bf16(r * rsqrt(ms + eps) * w).
// SwiGLU: grid-stride over 16-byte pieces of the output; gate and up pieces
// of a row are F columns apart in the merged projection output.
// Both are launched as programmatic dependents of the preceding kernel: they
// wait for it (griddepcontrol.wait) before their first load, and let the
// next kernel launch as soon as every CTA of theirs is running (measured:
// a trigger after the loop made back-to-back SwiGLU calls 9 % slower than
// no programmatic launch at all; this placement is 1.4 % faster).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "fusion_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kNormThreads = 256;                 // 8 rows (warps) per block
constexpr int kNormBatch = 4;                     // 16-byte pieces per lane in flight
constexpr int kGluThreads = 256;

__device__ __forceinline__ float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

__global__ void __launch_bounds__(kNormThreads)
    add_rmsnorm_kernel(const uint4* __restrict__ x, uint4* __restrict__ residual,
                       const uint4* __restrict__ weight, uint4* __restrict__ out, int rows,
                       int pieces, float eps, float inv_hidden) {
  const int lane = threadIdx.x & 31;
  const int warps = static_cast<int>(gridDim.x) * (kNormThreads / 32);
  pdl_wait_primary();
  pdl_launch_dependents();
  for (int row = static_cast<int>(blockIdx.x) * (kNormThreads / 32) + (threadIdx.x >> 5); row < rows;
       row += warps) {
    const size_t base = static_cast<size_t>(row) * pieces;
    float ss = 0.f;
    for (int p0 = lane; p0 < pieces; p0 += 32 * kNormBatch) {
      uint4 a[kNormBatch], b[kNormBatch];
#pragma unroll
      for (int i = 0; i < kNormBatch; ++i) {
        const int p = p0 + 32 * i;
        if (p < pieces) {
          a[i] = __ldcs(x + base + p);            // read once: do not keep in cache
          b[i] = residual[base + p];
        }
      }
#pragma unroll
      for (int i = 0; i < kNormBatch; ++i) {
        const int p = p0 + 32 * i;
        if (p < pieces) {
          const uint32_t* aw = reinterpret_cast<const uint32_t*>(&a[i]);
          const uint32_t* bw = reinterpret_cast<const uint32_t*>(&b[i]);
          uint4 s;
          uint32_t* sw = reinterpret_cast<uint32_t*>(&s);
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            sw[k] = pack_bf16x2(bf16lo(aw[k]) + bf16lo(bw[k]), bf16hi(aw[k]) + bf16hi(bw[k]));
            const float r0 = bf16lo(sw[k]), r1 = bf16hi(sw[k]);
            ss = fmaf(r0, r0, fmaf(r1, r1, ss));
          }
          residual[base + p] = s;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    const float inv = rsqrtf(ss * inv_hidden + eps);
    for (int p = lane; p < pieces; p += 32) {
      const uint4 s = residual[base + p];
      const uint4 wv = __ldg(weight + p);
      const uint32_t* sw = reinterpret_cast<const uint32_t*>(&s);
      const uint32_t* ww = reinterpret_cast<const uint32_t*>(&wv);
      uint4 y;
      uint32_t* yw = reinterpret_cast<uint32_t*>(&y);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        yw[k] = pack_bf16x2(bf16lo(sw[k]) * inv * bf16lo(ww[k]), bf16hi(sw[k]) * inv * bf16hi(ww[k]));
      __stcs(out + base + p, y);                  // written once: streaming store
    }
  }
}

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

__global__ void __launch_bounds__(kGluThreads)
    swiglu_kernel(const uint4* __restrict__ gate_up, uint4* __restrict__ out, long long total,
                  int fpieces) {
  const long long stride = static_cast<long long>(gridDim.x) * kGluThreads;
  pdl_wait_primary();
  pdl_launch_dependents();
  for (long long i = static_cast<long long>(blockIdx.x) * kGluThreads + threadIdx.x; i < total;
       i += stride) {
    const long long row = i / fpieces;
    const int p = static_cast<int>(i - row * fpieces);
    const uint4* src = gate_up + row * 2 * fpieces;
    const uint4 g = __ldcs(src + p);
    const uint4 u = __ldcs(src + fpieces + p);
    const uint32_t* gw = reinterpret_cast<const uint32_t*>(&g);
    const uint32_t* uw = reinterpret_cast<const uint32_t*>(&u);
    uint4 y;
    uint32_t* yw = reinterpret_cast<uint32_t*>(&y);
#pragma unroll
    for (int k = 0; k < 4; ++k)
      yw[k] = pack_bf16x2(silu(bf16lo(gw[k])) * bf16lo(uw[k]), silu(bf16hi(gw[k])) * bf16hi(uw[k]));
    __stcs(out + i, y);
  }
}

}  // namespace

cudaError_t launch_add_rmsnorm_sm103(const NormLaunch& a) {
  const int pieces = a.hidden / 8;
  const int rows_per_block = kNormThreads / 32;
  const long long blocks = (static_cast<long long>(a.rows) + rows_per_block - 1) / rows_per_block;
  const long long cap = static_cast<long long>(a.sms > 0 ? a.sms : 1) * 8;   // 8 blocks (64 warps) per SM
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  return launch_pdl(add_rmsnorm_kernel, dim3(grid), dim3(kNormThreads), 0, a.stream,
                    static_cast<const uint4*>(a.x), static_cast<uint4*>(a.residual),
                    static_cast<const uint4*>(a.weight), static_cast<uint4*>(a.out), a.rows, pieces, a.eps,
                    1.f / static_cast<float>(a.hidden));
}

cudaError_t launch_swiglu_sm103(const GluLaunch& a) {
  const int fpieces = a.F / 8;
  const long long total = static_cast<long long>(a.rows) * fpieces;
  const long long blocks = (total + kGluThreads - 1) / kGluThreads;
  const long long cap = static_cast<long long>(a.sms > 0 ? a.sms : 1) * 16;
  const unsigned grid = static_cast<unsigned>(blocks < cap ? blocks : cap);
  return launch_pdl(swiglu_kernel, dim3(grid), dim3(kGluThreads), 0, a.stream,
                    static_cast<const uint4*>(a.gate_up), static_cast<uint4*>(a.out), total, fpieces);
}

}  // namespace attn47
