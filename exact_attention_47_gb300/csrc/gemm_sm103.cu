// SwiGLU projection with the activation fused into the GEMM's epilogue
// ("Fast attention kernels and operator fusion accelerate AI models",
// section "Operator fusion": the SwiGLU block's projection matmul, SiLU and
// elementwise product in one kernel, so the [rows, 2F] projection output
// never reaches HBM):
//   out[r, f] = bf16(silu(g) * u),  g = x[r] . W[f],  u = x[r] . W[F + f],
//   silu(g) = g / (1 + exp(-g)),
// x [rows, hidden] bf16, W [2F, hidden] bf16 (gate rows 0..F-1, up rows
// F..2F-1, the layout of a merged gate/up weight), out [rows, F] bf16.
//
// A persistent kernel, one CTA per SM, walks 128-row x 128-feature output
// tiles.  Per tile one MMA chain computes D = x_tile . [W_gate; W_up]^T
// (M = 128, N = 256: the gate and the up columns of the same 128 features
// side by side) into a TMEM accumulator; the accumulator is double-buffered,
// so the epilogue of one tile (SiLU, product, bf16, store) runs while the
// next tile's MMAs do.  Operands come through a 4-stage TMA ring of 64-deep
// K slices (x 16 KB + W 32 KB per stage, 128-byte swizzle).
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "gemm_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kBM = 128;          // output rows per tile
constexpr int kBF = 128;          // output features per tile
constexpr int kBK = 64;           // K per stage (one 128-byte swizzle row)
constexpr int kStages = 4;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kBBytes = 2 * kBF * kBK * 2;      // 32 KB: gate rows, then up rows
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kOffBar = kStages * kStageBytes;
constexpr int kSmem = kOffBar + 256 + 1024;
constexpr int kThreads = 192;     // producer, MMA, 4 epilogue warps

struct GemmBars {
  uint64_t full[kStages], empty[kStages];
  uint64_t acc_full[2], acc_empty[2];
  uint64_t mma_drain;
  uint32_t tmem;
  int abort;
  int issued;                     // stages the producer started
};

struct GemmParams {
  __nv_bfloat16* out;
  int rows, F, hidden;
  int m_blocks, tiles;
  unsigned int* status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ float silu(float g) { return g / (1.f + __expf(-g)); }

__global__ void __launch_bounds__(kThreads, 1)
    swiglu_proj_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tw,
                       const GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  GemmBars* bar = reinterpret_cast<GemmBars*>(smem + kOffBar);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int kb_count = p.hidden / kBK;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&bar->full[s]), 1);
      mbar_init(smem_addr(&bar->empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bar->acc_full[s]), 1);
      mbar_init(smem_addr(&bar->acc_empty[s]), 4);
    }
    mbar_init(smem_addr(&bar->mma_drain), 1);
    bar->abort = 0;
    bar->issued = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tmap(&tx);
    prefetch_tmap(&tw);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&bar->tmem), 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem;
  const WaitCtl wc{&bar->abort, p.status, p.timeout_ns};
  // Programmatic dependent launch: nothing global is touched before the
  // preceding kernel has finished; the next kernel may start its set-up as
  // soon as every CTA of this grid is running.
  pdl_wait_primary();
  pdl_launch_dependents();

  // Tiles of this CTA: blockIdx.x, + gridDim.x, ...; the row block varies
  // fastest, so the CTAs working at the same time share W tiles in L2.
  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int s = 0;
      bool ok = true;
      for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x) {
        const int m0 = (t % p.m_blocks) * kBM;
        const int f0 = (t / p.m_blocks) * kBF;
        for (int kb = 0; kb < kb_count; ++kb, ++s) {
          const int st = s % kStages;
          if (!mbar_wait(smem_addr(&bar->empty[st]), ((s / kStages) & 1) ^ 1, wc)) {
            ok = false;
            break;
          }
          bar->issued = s + 1;
          const uint32_t fb = smem_addr(&bar->full[st]);
          const uint32_t dst = sbase + st * kStageBytes;
          mbar_arrive_expect_tx(fb, kStageBytes);
          tma_load_2d(dst, &tx, fb, kb * kBK, m0);
          tma_load_2d(dst + kABytes, &tw, fb, kb * kBK, f0);
          tma_load_2d(dst + kABytes + kBBytes / 2, &tw, fb, kb * kBK, p.F + f0);
        }
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16_f32(kBM, 2 * kBF, false);
    int s = 0, i = 0;
    bool ok = true;
    for (int t = blockIdx.x; t < p.tiles && ok; t += gridDim.x, ++i) {
      const int buf = i & 1;
      if (!mbar_wait_warp(smem_addr(&bar->acc_empty[buf]), ((i >> 1) & 1) ^ 1, wc)) break;
      tc_fence_after();
      const uint32_t acc = tmem + buf * 256;
      for (int kb = 0; kb < kb_count; ++kb, ++s) {
        const int st = s % kStages;
        if (!mbar_wait_warp(smem_addr(&bar->full[st]), (s / kStages) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a = sbase + st * kStageBytes;
        const uint32_t b = a + kABytes;
        // Both operands K-major: 128-byte rows, 8-row atoms 1024 bytes apart.
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(a + kk * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(b + kk * 32, 16, 1024);
          umma_ss_warp(acc, ad, bd, kIdesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit_warp(smem_addr(&bar->empty[st]));
      }
      if (!ok) break;
      umma_commit_warp(smem_addr(&bar->acc_full[buf]));
    }
    umma_commit_warp(smem_addr(&bar->mma_drain));
    mbar_wait_warp_drain(smem_addr(&bar->mma_drain), 0, wc);
  } else {
    // ------------------------------------------------------------ epilogue
    const int wq = warp & 3;                   // TMEM lane quarter = 32 rows
    const int r = wq * 32 + lane;
    int i = 0;
    for (int t = blockIdx.x; t < p.tiles; t += gridDim.x, ++i) {
      const int buf = i & 1;
      if (!mbar_wait_warp(smem_addr(&bar->acc_full[buf]), (i >> 1) & 1, wc)) break;
      tc_fence_after();
      const int m0 = (t % p.m_blocks) * kBM;
      const int f0 = (t / p.m_blocks) * kBF;
      const bool write = m0 + r < p.rows;
      __nv_bfloat16* orow = p.out + static_cast<size_t>(m0 + r) * p.F + f0;
      const uint32_t acc = tmem + (static_cast<uint32_t>(wq * 32) << 16) + buf * 256;
#pragma unroll 1
      for (int c = 0; c < kBF; c += 32) {
        uint32_t g[32], u[32];
        ATTN47_TMEM_LD32(acc + c, g);
        ATTN47_TMEM_LD32(acc + kBF + c, u);
        ATTN47_TMEM_LD_WAIT(g);
        ATTN47_TMEM_LD_WAIT(u);
        if (write) {
          uint32_t o[16];
#pragma unroll
          for (int e = 0; e < 16; ++e)
            o[e] = pack_bf16x2(silu(__uint_as_float(g[2 * e])) * __uint_as_float(u[2 * e]),
                               silu(__uint_as_float(g[2 * e + 1])) * __uint_as_float(u[2 * e + 1]));
          uint4* dst = reinterpret_cast<uint4*>(orow + c);
#pragma unroll
          for (int q = 0; q < 4; ++q) dst[q] = make_uint4(o[4 * q], o[4 * q + 1], o[4 * q + 2], o[4 * q + 3]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->acc_empty[buf]));
    }
  }
  // Copies still in flight (a CTA that gave up early) must land first.
  if (warp == 0 && lane == 0) {
    const int issued = bar->issued;
    for (int st = 0; st < kStages && st < issued; ++st) {
      const int fills = (issued - 1 - st) / kStages + 1;
      mbar_wait(smem_addr(&bar->full[st]), (fills - 1) & 1, wc, true);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

int swiglu_proj_tile_features() { return kBF; }
int swiglu_proj_k_step() { return kBK; }

cudaError_t launch_swiglu_proj_sm103(const SwigluProjLaunch& a) {
  GemmParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.rows = a.rows;
  p.F = a.F;
  p.hidden = a.hidden;
  p.m_blocks = (a.rows + kBM - 1) / kBM;
  p.tiles = p.m_blocks * (a.F / kBF);
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  cudaError_t e = cudaFuncSetAttribute(swiglu_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return e;
  const int grid = p.tiles < a.sms ? p.tiles : a.sms;
  return launch_pdl(swiglu_proj_kernel, dim3(grid), dim3(kThreads), kSmem, a.stream, *a.tx, *a.tw, p);
}

}  // namespace attn47
