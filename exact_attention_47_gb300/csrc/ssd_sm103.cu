// Mamba-2 SSD forward, chunked ("Accelerating Mamba-2 with high-performance
// forward kernels in NVIDIA CUDA Tile"): the recurrence
//   h_t = exp(a_t) h_{t-1} + x_t b_t^T,  y_t = h_t c_t,  a_t = A[h] dt[t, h] < 0
// evaluated chunk by chunk in two tensor-core kernels (tcgen05 MMAs with fp32
// accumulators in TMEM, operands staged in shared memory by TMA):
//   ssd_state_kernel (the page's kernel 1 and fwd_pass_state): one CTA per
//     (batch, pair of heads of one B/C group) walks the chunks in order.  Per
//     chunk it forms g, the log2(e)-scaled running sum of a_t restarting at
//     the chunk (a warp scan per head, kept in the workspace for the output
//     kernel), stores the chunk's initial state (bf16: the output kernel's
//     product takes it in bf16), decays the state by 2^(g_last) and adds
//       sum_j 2^(g_last - g_j) x_j b_j^T = (x o w)^T B,
//     one 128 x N x chunk MMA for both heads (rows = the two heads' 64
//     columns of x, which share B), the state staying in TMEM throughout.
//   ssd_out_kernel: one CTA per (batch, chunk, 128-row block, up to 16 heads
//     of one group) forms C B^T once for the group's heads in TMEM, and per
//     head
//       y_i = sum_{j <= i} (C B^T)_ij 2^(g_i - g_j) x_j + 2^(g_i) (C S^T)_i
//     (S: the chunk's initial state) with the sums as MMAs.
// Every exponent the kernels evaluate is <= 0: the weights are only formed
// for j <= i, where g_i <= g_j (a_t < 0), as the page notes.  Where a block
// of keys lies wholly before a block of rows, the weight is split at a point
// m between them, 2^(g_i - g_j) = 2^(g_i - g_m) 2^(g_m - g_j), both factors
// <= 1: a row factor and a key factor replace one exponential per entry.
// Layouts: x / y [batch, L, H, P] bf16, B / C [batch, L, G, N] bf16,
// dt [batch, L, H] fp32, A [H] fp32, states [batch, H, P, N] fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd_sm103.h"

namespace attn47 {
namespace {

constexpr int kP = 64;                 // head dim handled by the kernels
constexpr int kHeadsPerOut = 16;       // heads of one group per output CTA
constexpr int kRows = 64;              // tokens per TMA box of x and B
constexpr float kLog2e = 1.4426950408889634f;

// x <- bf16(x * w) for the 8 bf16 values of one 16-byte piece, on packed
// bf16 pairs: w = w_hi + w_lo with both parts bf16, and
// x w = fma(x, w_hi, x w_lo) rounded once; the error of the small term
// x w_lo is about 2^-18 |x w|, below the final rounding.
__device__ __forceinline__ void scale_piece_bf16(uint4* piece, float w) {
  const __nv_bfloat16 hi = __float2bfloat16_rn(w);
  const __nv_bfloat16 lo = __float2bfloat16_rn(w - __bfloat162float(hi));
  const __nv_bfloat162 whi = __halves2bfloat162(hi, hi);
  const __nv_bfloat162 wlo = __halves2bfloat162(lo, lo);
  uint4 v = *piece;
  __nv_bfloat162* vw = reinterpret_cast<__nv_bfloat162*>(&v);
#pragma unroll
  for (int e = 0; e < 4; ++e) vw[e] = __hfma2(vw[e], whi, __hmul2(vw[e], wlo));
  *piece = v;
}

// Shared-memory layouts: every tile is rows of 128 bytes (64 bf16) in the
// 128-byte swizzle TMA writes (8-row atoms of 1024 bytes); a tile wider than
// 64 columns is a sequence of such 64-column chunks.
template <int N, int Q>
struct StateLayout {
  static constexpr int TB = kRows;               // tokens per stage
  static constexpr int SPC = Q / TB;             // stages per chunk
  static constexpr int NCH = N / 64;
  static constexpr int kX = TB * 128;            // x of one head: TB rows x 64 columns
  static constexpr int kB = TB * 128;            // one 64-column chunk of B
  static constexpr int kStage = 2 * kX + NCH * kB;
  static constexpr int kStages = 3;
  static constexpr int kOffW = kStages * kStage; // per-token weights [2 heads][Q] fp32
  static constexpr int kOffGl = kOffW + 2 * Q * 4;   // g_last [2 heads]
  static constexpr int kOffDt = kOffGl + 16;         // dt staging [2 heads][2 chunks][Q] fp32
  static constexpr int kOffBar = kOffDt + 4 * Q * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;
};

struct StateBars {
  uint64_t full[3], empty[3], xs[3];
  uint64_t st_ready, acc_done, mma_drain;
  uint32_t tmem;
  int abort;
  int issued;                 // stages the producer started
};

struct SsdParams {
  const float* dt;
  const float* A;
  const float* h0;
  __nv_bfloat16* y;
  float* h_final;
  float* g;                   // workspace: [batch, H, nc, Q] fp32
  __nv_bfloat16* s_init;      // workspace: [batch, nc, H, P, N] bf16
  int batch, L, H, G, nc;
  unsigned int* status;
  unsigned long long timeout_ns;
};

// ------------------------------------------------------------ state kernel
// Warp 0: TMA producer.  Warp 1: MMA issuer (and TMEM owner).  Warps 2-5:
// the state's 128 rows (TMEM lane = row = head pair member * 64 + p), the
// g scans (warps 2 and 3, dt fetched one chunk ahead with cp.async), the
// stored states and the scaling of x.  Small enough for two CTAs per SM.
template <int N, int Q>
__global__ void __launch_bounds__(192, 1)
    ssd_state_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tb,
                     const SsdParams p) {
  using Lt = StateLayout<N, Q>;
  constexpr int S = Lt::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  StateBars* bar = reinterpret_cast<StateBars*>(smem + Lt::kOffBar);
  float* ws = reinterpret_cast<float*>(smem + Lt::kOffW);
  float* gl = reinterpret_cast<float*>(smem + Lt::kOffGl);
  float* dtb = reinterpret_cast<float*>(smem + Lt::kOffDt);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int hpg = p.H / p.G;
  const int pairs = (hpg + 1) / 2;
  const int pair = blockIdx.x % pairs;
  const int grp = (blockIdx.x / pairs) % p.G;
  const int b = blockIdx.x / (pairs * p.G);
  const int ha = grp * hpg + 2 * pair;
  const bool has_b = 2 * pair + 1 < hpg;
  const int hb = ha + 1;
  const int nstage = p.nc * Lt::SPC;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(smem_addr(&bar->full[s]), 1);
      mbar_init(smem_addr(&bar->empty[s]), 1);
      mbar_init(smem_addr(&bar->xs[s]), 4);
    }
    mbar_init(smem_addr(&bar->st_ready), 4);
    mbar_init(smem_addr(&bar->acc_done), 1);
    mbar_init(smem_addr(&bar->mma_drain), 1);
    bar->abort = 0;
    bar->issued = 0;
    fence_mbar_init();
  }
  if (!has_b) {
    // The second head's rows of x stay zero (it is never loaded).
    for (int s = 0; s < S; ++s)
      for (int i = threadIdx.x; i < Lt::kX / 16; i += blockDim.x)
        *reinterpret_cast<uint4*>(smem + s * Lt::kStage + Lt::kX + i * 16) = make_uint4(0, 0, 0, 0);
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&bar->tmem), N);
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t bytes = (has_b ? 2 : 1) * Lt::kX + Lt::NCH * Lt::kB;
      for (int s = 0; s < nstage; ++s) {
        const int st = s % S;
        if (!mbar_wait_sleep(smem_addr(&bar->empty[st]), ((s / S) & 1) ^ 1, wc)) break;
        bar->issued = s + 1;
        const int t = (s / Lt::SPC) * Q + (s % Lt::SPC) * Lt::TB;
        const uint32_t fb = smem_addr(&bar->full[st]);
        const uint32_t dst = sbase + st * Lt::kStage;
        mbar_arrive_expect_tx(fb, bytes);
        tma_load_4d(dst, &tx, fb, 0, ha, t, b);
        if (has_b) tma_load_4d(dst + Lt::kX, &tx, fb, 0, hb, t, b);
#pragma unroll
        for (int ch = 0; ch < Lt::NCH; ++ch) tma_load_4d(dst + 2 * Lt::kX + ch * Lt::kB, &tb, fb, 64 * ch, grp, t, b);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    constexpr uint32_t kIdesc = idesc_bf16_f32_ab(128, N, true, true);
    for (int c = 0; c < p.nc; ++c) {
      if (!mbar_wait_sleep_warp(smem_addr(&bar->st_ready), c & 1, wc)) break;
      tc_fence_after();
      bool ok = true;
      for (int k = 0; k < Lt::SPC; ++k) {
        const int s = c * Lt::SPC + k;
        const int st = s % S;
        if (!mbar_wait_sleep_warp(smem_addr(&bar->xs[st]), (s / S) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t xa = sbase + st * Lt::kStage;
        const uint32_t bb = xa + 2 * Lt::kX;
        // D (rows: the two heads' x columns, cols: n) += x'^T B over the
        // stage's tokens.  A and B are stored token-major (M and N contiguous).
#pragma unroll
        for (int kk = 0; kk < Lt::TB / 16; ++kk) {
          const uint64_t ad = sdesc_sw128(xa + kk * 2048, Lt::kX, 1024);
          const uint64_t bd = sdesc_sw128(bb + kk * 2048, Lt::kB, 1024);
          umma_ss_warp(tmem, ad, bd, kIdesc, 1u);
        }
        umma_commit_warp(smem_addr(&bar->empty[st]));
      }
      if (!ok) break;
      umma_commit_warp(smem_addr(&bar->acc_done));
    }
    // Every MMA this warp issued completes before TMEM is released.
    umma_commit_warp(smem_addr(&bar->mma_drain));
    mbar_wait_warp_drain(smem_addr(&bar->mma_drain), 0, wc);
  } else {
    // ------------------------------------------------------------- rows
    const int tid = threadIdx.x - 64;          // 0 .. 127
    const int wq = warp & 3;                   // TMEM lane quarter of this warp
    const int r = wq * 32 + lane;              // state row
    const int sel = r >> 6;
    const int pr = r & 63;
    const int hrow = sel ? hb : ha;
    const bool vrow = sel == 0 || has_b;
    const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    // Scan warps: warp 2 for head a, warp 3 for head b; each lane holds E
    // consecutive tokens of the chunk.
    constexpr int E = Q / 32;
    const int ssel = warp - 2;
    const bool scan = ssel == 0 || (ssel == 1 && has_b);
    const int h_scan = ssel ? hb : ha;
    const float a_scan = scan ? __ldg(p.A + h_scan) : 0.f;
    auto fetch = [&](int cc) {
      const int tc0 = cc * Q;
#pragma unroll
      for (int e = 0; e < E; ++e) {
        const int i = lane * E + e;
        const bool in = tc0 + i < p.L;
        const float* src = p.dt + (static_cast<size_t>(b) * p.L + (in ? tc0 + i : 0)) * p.H + h_scan;
        cp_async4(smem_addr(dtb + (ssel * 2 + (cc & 1)) * Q + i), src, in ? 4u : 0u);
      }
      cp_async_commit();
    };
    if (scan) fetch(0);
    // Initial state: h0 or zero.
#pragma unroll 1
    for (int c0 = 0; c0 < N; c0 += 32) {
      uint32_t v[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float x = 0.f;
        if (p.h0 != nullptr && vrow) x = __ldg(p.h0 + ((static_cast<size_t>(b) * p.H + hrow) * kP + pr) * N + c0 + i);
        v[i] = __float_as_uint(x);
      }
      ATTN47_TMEM_ST32(trow + c0, v);
    }
    tmem_st_wait();
    // x_t <- bf16(x_t * 2^(g_last - g_t)) in place for stage k of chunk c
    // (rows past the sequence end have weight 0).
    auto scale_stage = [&](int c, int k) {
      const int s = c * Lt::SPC + k;
      const int st = s % S;
      if (!mbar_wait_sleep_warp(smem_addr(&bar->full[st]), (s / S) & 1, wc)) return false;
      uint8_t* xs = smem + st * Lt::kStage;
#pragma unroll 4
      for (int q = tid; q < (has_b ? 2 : 1) * Lt::TB * 8; q += 128) {
        const int hsel = q / (Lt::TB * 8);
        const int row = (q >> 3) % Lt::TB;
        scale_piece_bf16(reinterpret_cast<uint4*>(xs + hsel * Lt::kX + row * 128 + (q & 7) * 16),
                         ws[hsel * Q + k * Lt::TB + row]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->xs[st]));
      return true;
    };
    // The four warps meet at two named barriers per chunk.  A warp whose
    // wait gave up skips the rest of its chunk but still reaches both
    // barriers; at the first one of the next chunk they all learn of it and
    // leave together (no warp is left waiting at a barrier).
    bool ok = true;
    for (int c = 0; c < p.nc; ++c) {
      const int t0 = c * Q;
      const int n_len = min(Q, p.L - t0);
      // Every row is done with the previous chunk's weights.
      if (named_barrier_or(1, 128, !ok)) {
        ok = false;
        break;
      }
      if (scan) {
        if (c + 1 < p.nc) {
          fetch(c + 1);
          cp_async_wait_group<1>();
        } else {
          cp_async_wait_group<0>();
        }
        // Past the end of the sequence dt reads as 0, so g keeps the
        // chunk's last value there.
        const float* dcur = dtb + (ssel * 2 + (c & 1)) * Q;
        float v[E];
        float run = 0.f;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          run = fmaf(a_scan, dcur[lane * E + e], run);
          v[e] = run;
        }
        float incl = run;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float y = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += y;
        }
        const float offset = incl - run;
        const float g_last = __shfl_sync(0xffffffffu, incl, 31) * kLog2e;
        float* gw = p.g + ((static_cast<size_t>(b) * p.H + h_scan) * p.nc + c) * Q;
        float* wrow = ws + ssel * Q;
#pragma unroll
        for (int e = 0; e < E; ++e) {
          const int i = lane * E + e;
          const float gv = (v[e] + offset) * kLog2e;
          gw[i] = gv;
          const float wv = ex2(g_last - gv);
          wrow[i] = i < n_len ? wv : 0.f;
        }
        if (lane == 0) gl[ssel] = g_last;
      }
      named_barrier_sync(1, 128);
      // As many stages as the ring holds are scaled before the hand-over
      // below (they overlap with the previous chunk's MMAs); the chunk's
      // later stages can only be loaded once its first MMAs have run.
      constexpr int kPre = Lt::SPC < S ? Lt::SPC : S;
      for (int k = 0; k < kPre && ok; ++k) ok = scale_stage(c, k);
      // The chunk's initial state (once the previous chunk's MMAs are
      // complete) is stored, then decayed to the chunk's end in place.
      if (!ok) continue;
      if (c > 0 && !mbar_wait_sleep_warp(smem_addr(&bar->acc_done), (c - 1) & 1, wc)) {
        ok = false;
        continue;
      }
      tc_fence_after();
      const float decay = vrow ? ex2(gl[sel]) : 0.f;
      __nv_bfloat16* si = p.s_init + ((static_cast<size_t>(b) * p.nc + c) * p.H + hrow) * kP * N + pr * N;
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t v[32];
        ATTN47_TMEM_LD32(trow + c0, v);
        ATTN47_TMEM_LD_WAIT(v);
        if (vrow) {
          uint4* dst = reinterpret_cast<uint4*>(si + c0);
#pragma unroll
          for (int q = 0; q < 4; ++q)
            dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                                pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
        }
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * decay);
        ATTN47_TMEM_ST32(trow + c0, v);
      }
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->st_ready));
      for (int k = kPre; k < Lt::SPC && ok; ++k) ok = scale_stage(c, k);
    }
    if (scan) cp_async_wait_group<0>();
    // Final state.
    if (ok && mbar_wait_sleep_warp(smem_addr(&bar->acc_done), (p.nc - 1) & 1, wc)) {
      tc_fence_after();
      float* hf = p.h_final + ((static_cast<size_t>(b) * p.H + hrow) * kP + pr) * N;
#pragma unroll 1
      for (int c0 = 0; c0 < N; c0 += 32) {
        uint32_t v[32];
        ATTN47_TMEM_LD32(trow + c0, v);
        ATTN47_TMEM_LD_WAIT(v);
        if (vrow) {
          float4* dst = reinterpret_cast<float4*>(hf + c0);
#pragma unroll
          for (int q = 0; q < 8; ++q)
            dst[q] = make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                 __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
        }
      }
    }
  }
  // Copies still in flight (a CTA that gave up early) must land first.
  if (warp == 0 && lane == 0) {
    const int issued = bar->issued;
    for (int st = 0; st < S && st < issued; ++st) {
      const int fills = (issued - 1 - st) / S + 1;
      mbar_wait_sleep(smem_addr(&bar->full[st]), (fills - 1) & 1, wc, true);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, N);
  }
}

// ----------------------------------------------------------- output kernel
// A CTA takes the 128 rows [R0, R0 + 128) of a chunk, R0 = 128 rb.  Keys
// before R0 (JO of them, 0 or 128: the "off" block) lie wholly before every
// row: their weights split at m = R0 - 1 into the row factor
// 2^(g_i - g_m) and the key factor 2^(g_m - g_j) (applied to x_j in shared
// memory, per head), so their C B^T entries become a head-independent bf16
// operand formed once.  The initial state's term 2^(g_i) C S^T shares the
// row factor once S is scaled by 2^(g_m) (<= 1), so per head
//   y_i = Y_i + 2^(g_i - g_m) Y2_i,
//   Y  = P X over the diagonal block,  Y2 = P_off X' + C (2^(g_m) S)^T
// (g_m = 0 when there is no off block).  The JD keys of the row block itself
// (the "diagonal" block) are weighted per head in 32 x 32 sub-blocks: above
// the diagonal zero, on it the exact exponential per entry, below it split
// at the key sub-block's last key.
template <int N, int Q>
struct OutLayout {
  static constexpr int JD = Q < 128 ? Q : 128;   // keys of the diagonal block
  static constexpr int NCH = N / 64;
  static constexpr int kC = 128 * 128;           // one 64-column chunk of the C block (128 rows)
  static constexpr int kBch = Q * 128;           // one 64-column chunk of B (up to Q keys)
  static constexpr int kPch = 128 * 128;         // one 64-key chunk of a P buffer (128 rows)
  static constexpr int kPbuf = (JD / 64) * kPch;
  static constexpr int kX = Q * 128;             // X of one head (up to Q keys x 64)
  static constexpr int kS = 64 * 128;            // one 64-column chunk of S (64 rows)
  // B is only read by the C B^T product; afterwards its space holds the two
  // P buffers.
  static constexpr int kU = NCH * kBch > 2 * kPbuf ? NCH * kBch : 2 * kPbuf;
  static constexpr int kOffC = 0;
  static constexpr int kOffB = kOffC + NCH * kC;
  static constexpr int kOffP = kOffB;
  static constexpr int kOffX = kOffB + kU;
  static constexpr int kOffS = kOffX + 2 * kX;
  static constexpr int kOffG = kOffS + 2 * NCH * kS;
  static constexpr int kOffKf = kOffG + 2 * Q * 4;   // per-warp key factors: 8 x 32 fp32
  static constexpr int kOffBar = kOffKf + 8 * 32 * 4;
  static constexpr int kSmem = kOffBar + 256 + 1024;
  // TMEM columns.  C B^T lands at [128 - JO, 128 + JD): its off block at
  // [0, 128) is turned into bf16 (P_off, at 256) first, after which those
  // columns hold accumulator set 0 (Y, Y2); set 1 is at [320, 448).
  static constexpr uint32_t kColCBd = 128, kColPo = 256;
  __host__ __device__ static constexpr uint32_t col_y(int set) { return set ? 320u : 0u; }
};

struct OutBars {
  uint64_t cb_full, cb_done;
  uint64_t xf[2], xe[2];
  uint64_t p_full[2], y_full[2], y_free[2];
  uint64_t mma_drain;
  uint32_t tmem;
  int abort;
  int issued;                 // heads whose operands the producer started
};

// Warp 0: TMA producer.  Warp 1: MMA issuer (and TMEM owner).  Warps 2-9:
// two per TMEM lane quarter (row = lane), each taking half of the keys (P)
// and half of the 64 output columns (epilogue).  Operands, P buffers and
// accumulators are all double-buffered by head parity, so while head k's
// MMAs run the rows form head k+1's weights and write out head k-1.
template <int N, int Q>
__global__ void __launch_bounds__(320, 1)
    ssd_out_kernel(const __grid_constant__ CUtensorMap tx, const __grid_constant__ CUtensorMap tb,
                   const __grid_constant__ CUtensorMap tc, const __grid_constant__ CUtensorMap ts,
                   const SsdParams p) {
  using Lt = OutLayout<N, Q>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  OutBars* bar = reinterpret_cast<OutBars*>(smem + Lt::kOffBar);
  const uint32_t sbase = smem_addr(smem);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  const int hpg = p.H / p.G;
  const int ngrp = (hpg + kHeadsPerOut - 1) / kHeadsPerOut;
  const int nrb = (Q + 127) / 128;
  int idx = blockIdx.x;
  const int hgi = idx % ngrp;
  idx /= ngrp;
  const int grp = idx % p.G;
  idx /= p.G;
  const int rb = idx % nrb;
  idx /= nrb;
  const int c = idx % p.nc;
  const int b = idx / p.nc;
  const int h0 = grp * hpg + hgi * kHeadsPerOut;
  const int nh = min(kHeadsPerOut, hpg - hgi * kHeadsPerOut);
  const int t0 = c * Q;
  const int n_len = min(Q, p.L - t0);
  const int JO = 128 * rb;                       // keys of the off block
  const int J = JO + Lt::JD;                     // keys 0 .. J-1 of the chunk
  const int kb_count = J / kRows;

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar->cb_full), 1);
    mbar_init(smem_addr(&bar->cb_done), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bar->xf[s]), 1);
      mbar_init(smem_addr(&bar->xe[s]), 1);
      mbar_init(smem_addr(&bar->p_full[s]), 8);
      mbar_init(smem_addr(&bar->y_full[s]), 1);
      mbar_init(smem_addr(&bar->y_free[s]), 8);
    }
    mbar_init(smem_addr(&bar->mma_drain), 1);
    bar->abort = 0;
    bar->issued = 0;
    fence_mbar_init();
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

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      const uint32_t fb = smem_addr(&bar->cb_full);
      mbar_arrive_expect_tx(fb, Lt::NCH * Lt::kC + Lt::NCH * J * 128);
#pragma unroll
      for (int ch = 0; ch < Lt::NCH; ++ch) {
        tma_load_4d(sbase + Lt::kOffC + ch * Lt::kC, &tc, fb, 64 * ch, grp, t0 + JO, b);
        for (int kb = 0; kb < kb_count; ++kb)
          tma_load_4d(sbase + Lt::kOffB + ch * Lt::kBch + kb * kRows * 128, &tb, fb, 64 * ch, grp,
                      t0 + kb * kRows, b);
      }
      for (int k = 0; k < nh; ++k) {
        const int st = k & 1;
        if (!mbar_wait_sleep(smem_addr(&bar->xe[st]), ((k >> 1) & 1) ^ 1, wc)) break;
        bar->issued = k + 1;
        const int h = h0 + k;
        const uint32_t xb = smem_addr(&bar->xf[st]);
        mbar_arrive_expect_tx(xb, J * 128 + Lt::NCH * Lt::kS + Q * 4);
        for (int kb = 0; kb < kb_count; ++kb)
          tma_load_4d(sbase + Lt::kOffX + st * Lt::kX + kb * kRows * 128, &tx, xb, 0, h, t0 + kb * kRows, b);
        const int srow = ((b * p.nc + c) * p.H + h) * kP;
#pragma unroll
        for (int ch = 0; ch < Lt::NCH; ++ch)
          tma_load_2d(sbase + Lt::kOffS + (st * Lt::NCH + ch) * Lt::kS, &ts, xb, 64 * ch, srow);
        bulk_load(sbase + Lt::kOffG + st * Q * 4, p.g + ((static_cast<size_t>(b) * p.H + h) * p.nc + c) * Q,
                  Q * 4, xb);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    bool ok = mbar_wait_sleep_warp(smem_addr(&bar->cb_full), 0, wc);
    if (ok) {
      tc_fence_after();
      // C B^T: A = C (rows i, K = n), B = B (rows j, K = n), both K-major.
      const uint32_t idesc = idesc_bf16_f32_ab(128, J, false, false);
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(sbase + Lt::kOffC + (kk >> 2) * Lt::kC + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(sbase + Lt::kOffB + (kk >> 2) * Lt::kBch + (kk & 3) * 32, 16, 1024);
        umma_ss_warp(tmem + Lt::kColCBd - JO, ad, bd, idesc, kk > 0 ? 1u : 0u);
      }
      umma_commit_warp(smem_addr(&bar->cb_done));
    }
    constexpr uint32_t kIdescPX = idesc_bf16_f32_ab(128, 64, false, true);
    constexpr uint32_t kIdescCS = idesc_bf16_f32_ab(128, 64, false, false);
    for (int k = 0; k < nh && ok; ++k) {
      const int st = k & 1;
      const uint32_t ph = (k >> 1) & 1;
      ok = mbar_wait_sleep_warp(smem_addr(&bar->xf[st]), ph, wc) && mbar_wait_sleep_warp(smem_addr(&bar->p_full[st]), ph, wc) &&
           mbar_wait_sleep_warp(smem_addr(&bar->y_free[st]), ph ^ 1, wc);
      if (!ok) break;
      tc_fence_after();
      const uint32_t xs = sbase + Lt::kOffX + st * Lt::kX;
      const uint32_t pb = sbase + Lt::kOffP + st * Lt::kPbuf;
      const uint32_t ty = tmem + Lt::col_y(st);
      // Diagonal block: Y = P X over its JD keys (A = P, K-major in shared
      // memory; B = X rows, column-contiguous).
#pragma unroll
      for (int kk = 0; kk < Lt::JD / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(pb + (kk >> 2) * Lt::kPch + (kk & 3) * 32, 16, 1024);
        const uint64_t bd = sdesc_sw128(xs + JO * 128 + kk * 2048, Lt::kX, 1024);
        umma_ss_warp(ty, ad, bd, kIdescPX, kk > 0 ? 1u : 0u);
      }
      // Off block: Y2 = P_off X' (A = P_off from TMEM, 8 columns = 16 keys
      // per step).
      for (int kk = 0; kk < JO / 16; ++kk) {
        const uint64_t bd = sdesc_sw128(xs + kk * 2048, Lt::kX, 1024);
        umma_ts_warp(ty + 64, tmem + Lt::kColPo + kk * 8, bd, kIdescPX, kk > 0 ? 1u : 0u);
      }
      // Y2 += C S'^T: A = C, B = S (rows p, K = n): both K-major.
#pragma unroll
      for (int kk = 0; kk < N / 16; ++kk) {
        const uint64_t ad = sdesc_sw128(sbase + Lt::kOffC + (kk >> 2) * Lt::kC + (kk & 3) * 32, 16, 1024);
        const uint64_t bd =
            sdesc_sw128(sbase + Lt::kOffS + (st * Lt::NCH + (kk >> 2)) * Lt::kS + (kk & 3) * 32, 16, 1024);
        umma_ss_warp(ty + 64, ad, bd, kIdescCS, (JO > 0 || kk > 0) ? 1u : 0u);
      }
      umma_commit_warp(smem_addr(&bar->y_full[st]));
      umma_commit_warp(smem_addr(&bar->xe[st]));
    }
    umma_commit_warp(smem_addr(&bar->mma_drain));
    mbar_wait_warp_drain(smem_addr(&bar->mma_drain), 0, wc);
  } else {
    // ------------------------------------------------------------- rows
    const int wq = warp & 3;
    const int hf = (warp - 2) >> 2;            // half of the keys / of the output columns
    const int tid = threadIdx.x - 64;          // 0 .. 255
    const int r = wq * 32 + lane;              // row within the block
    const int i_abs = JO + r;                  // row's position in the chunk
    const uint32_t trow = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const float* gsm_base = reinterpret_cast<const float*>(smem + Lt::kOffG);
    float* kf = reinterpret_cast<float*>(smem + Lt::kOffKf) + (warp - 2) * 32;
    auto epilogue = [&](int k, float f) {
      const int set = k & 1;
      const bool write = i_abs < n_len;
      __nv_bfloat16* yrow = p.y + ((static_cast<size_t>(b) * p.L + t0 + i_abs) * p.H + h0 + k) * kP + hf * 32;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        const uint32_t col = Lt::col_y(set) + hf * 32 + half * 16;
        uint32_t yv[16], zv[16];
        ATTN47_TMEM_LD16(trow + col, yv);
        ATTN47_TMEM_LD16(trow + col + 64, zv);
        ATTN47_TMEM_LD16_WAIT(yv);
        ATTN47_TMEM_LD16_WAIT(zv);
        if (write) {
          uint32_t o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e)
            o[e] = pack_bf16x2(fmaf(f, __uint_as_float(zv[2 * e]), __uint_as_float(yv[2 * e])),
                               fmaf(f, __uint_as_float(zv[2 * e + 1]), __uint_as_float(yv[2 * e + 1])));
          uint4* dst = reinterpret_cast<uint4*>(yrow + half * 16);
          dst[0] = make_uint4(o[0], o[1], o[2], o[3]);
          dst[1] = make_uint4(o[4], o[5], o[6], o[7]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->y_free[set]));
    };
    bool ok = mbar_wait_sleep_warp(smem_addr(&bar->cb_done), 0, wc);
    tc_fence_after();
    if (ok && JO > 0) {
      // P_off = bf16(C B^T) over the off block, once for every head: this
      // warp's 64 keys of it.
#pragma unroll
      for (int part = 0; part < 2; ++part) {
        uint32_t v[32], w[16];
        ATTN47_TMEM_LD32(trow + hf * 64 + part * 32, v);
        ATTN47_TMEM_LD_WAIT(v);
#pragma unroll
        for (int e = 0; e < 16; ++e) w[e] = pack_bf16x2(__uint_as_float(v[2 * e]), __uint_as_float(v[2 * e + 1]));
        ATTN47_TMEM_ST16(trow + Lt::kColPo + hf * 32 + part * 16, w);
      }
    }
    float f_prev = 0.f;
    for (int k = 0; k < nh && ok; ++k) {
      const int st = k & 1;
      if (!mbar_wait_sleep_warp(smem_addr(&bar->xf[st]), (k >> 1) & 1, wc)) {
        ok = false;
        break;
      }
      const float* gsm = gsm_base + st * Q;
      const float gi = gsm[min(i_abs, Q - 1)];
      const float gm = JO > 0 ? gsm[JO - 1] : 0.f;
      if (JO > 0) {
        // x_j <- bf16(x_j * 2^(g_m - g_j)) over the off block's keys, and
        // S <- bf16(S * 2^(g_m)).
        uint8_t* xs = smem + Lt::kOffX + st * Lt::kX;
#pragma unroll 2
        for (int q = tid; q < JO * 8; q += 256) {
          const int row = q >> 3;
          scale_piece_bf16(reinterpret_cast<uint4*>(xs + row * 128 + (q & 7) * 16), ex2(gm - gsm[row]));
        }
        const float sf = ex2(gm);
        uint8_t* ss = smem + Lt::kOffS + st * Lt::NCH * Lt::kS;
#pragma unroll 2
        for (int q = tid; q < Lt::NCH * Lt::kS / 16; q += 256) scale_piece_bf16(reinterpret_cast<uint4*>(ss + q * 16), sf);
      }
      // Diagonal block weights into P buffer st (bf16, K-major, 128-byte
      // swizzle), this warp's half of the keys in 32-key sub-blocks
      // (sub-block index sb; the rows' sub-block is wq).
      uint8_t* prow = smem + Lt::kOffP + st * Lt::kPbuf + r * 128;
#pragma unroll
      for (int part = 0; part < Lt::JD / 64; ++part) {
        const int sb = hf * (Lt::JD / 64) + part;
        uint32_t w[16];
        if (sb > wq) {
#pragma unroll
          for (int e = 0; e < 16; ++e) w[e] = 0u;
        } else {
          uint32_t v[32];
          ATTN47_TMEM_LD32(trow + Lt::kColCBd + sb * 32, v);
          const float* gk = gsm + JO + sb * 32;
          if (sb == wq) {
            ATTN47_TMEM_LD_WAIT(v);
            // Keys sb*32 + c are allowed for c <= r - sb*32; the weight is
            // formed for every key and the masked ones are selected away.
            const int lim = r - sb * 32;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
              const float w0 = __uint_as_float(v[2 * e]) * ex2(gi - gk[2 * e]);
              const float w1 = __uint_as_float(v[2 * e + 1]) * ex2(gi - gk[2 * e + 1]);
              w[e] = pack_bf16x2(2 * e <= lim ? w0 : 0.f, 2 * e + 1 <= lim ? w1 : 0.f);
            }
          } else {
            // Split at the sub-block's last key m: row factor 2^(g_i - g_m),
            // key factors 2^(g_m - g_j) (one per lane, shared via smem).
            const float gsub = gk[31];
            kf[lane] = ex2(gsub - gk[lane]);
            const float a = ex2(gi - gsub);
            __syncwarp();
            ATTN47_TMEM_LD_WAIT(v);
#pragma unroll
            for (int e = 0; e < 16; ++e)
              w[e] = pack_bf16x2(__uint_as_float(v[2 * e]) * a * kf[2 * e],
                                 __uint_as_float(v[2 * e + 1]) * a * kf[2 * e + 1]);
            __syncwarp();
          }
        }
        // Keys sb*32 .. sb*32+31: 16-byte units (sb & 1) * 4 + u of 64-key
        // chunk sb >> 1, each at its swizzled place in the row.
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int unit = (sb & 1) * 4 + u;
          *reinterpret_cast<uint4*>(prow + (sb >> 1) * Lt::kPch + ((unit ^ (r & 7)) << 4)) =
              make_uint4(w[4 * u], w[4 * u + 1], w[4 * u + 2], w[4 * u + 3]);
        }
      }
      if (k == 0 && JO > 0) tmem_st_wait();    // P_off is an operand of every head
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->p_full[st]));
      if (k > 0) {
        if (!mbar_wait_sleep_warp(smem_addr(&bar->y_full[(k - 1) & 1]), ((k - 1) >> 1) & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        epilogue(k - 1, f_prev);
      }
      f_prev = ex2(gi - gm);
    }
    if (ok && nh > 0 && mbar_wait_sleep_warp(smem_addr(&bar->y_full[(nh - 1) & 1]), ((nh - 1) >> 1) & 1, wc)) {
      tc_fence_after();
      epilogue(nh - 1, f_prev);
    }
  }
  // Copies still in flight (a CTA that gave up early) must land first.
  if (warp == 0 && lane == 0) {
    mbar_wait_sleep(smem_addr(&bar->cb_full), 0, wc, true);
    const int issued = bar->issued;
    for (int st = 0; st < 2 && st < issued; ++st) {
      const int fills = (issued - 1 - st) / 2 + 1;
      mbar_wait_sleep(smem_addr(&bar->xf[st]), (fills - 1) & 1, wc, true);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int N, int Q>
cudaError_t launch_nq(const SsdLaunch& a, const SsdParams& p) {
  using Ls = StateLayout<N, Q>;
  using Lo = OutLayout<N, Q>;
  auto ks = ssd_state_kernel<N, Q>;
  auto ko = ssd_out_kernel<N, Q>;
  // The output kernel takes all 512 TMEM columns: its shared memory is
  // padded so that one CTA fits per SM.
  constexpr int kOutSmem = Lo::kSmem > 120 * 1024 ? Lo::kSmem : 120 * 1024;
  cudaError_t e = cudaFuncSetAttribute(ks, cudaFuncAttributeMaxDynamicSharedMemorySize, Ls::kSmem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(ko, cudaFuncAttributeMaxDynamicSharedMemorySize, kOutSmem);
  if (e != cudaSuccess) return e;
  const int hpg = a.H / a.G;
  const long long grid1 = static_cast<long long>(a.batch) * a.G * ((hpg + 1) / 2);
  e = launch_pdl(ks, dim3(static_cast<unsigned>(grid1)), dim3(192), Ls::kSmem, a.stream, *a.tx, *a.tb, p);
  if (e != cudaSuccess) return e;
  const long long grid2 = static_cast<long long>(a.batch) * p.nc * ((Q + 127) / 128) * a.G *
                          ((hpg + kHeadsPerOut - 1) / kHeadsPerOut);
  return launch_pdl(ko, dim3(static_cast<unsigned>(grid2)), dim3(320), kOutSmem, a.stream, *a.tx, *a.tb, *a.tc,
                    *a.ts, p);
}

}  // namespace

size_t ssd_workspace_bytes(int batch, int L, int H, int N, int chunk) {
  const size_t nc = (static_cast<size_t>(L) + chunk - 1) / chunk;
  const size_t g_bytes = static_cast<size_t>(batch) * H * nc * chunk * 4;
  const size_t s_bytes = static_cast<size_t>(batch) * nc * H * kP * N * 2;
  return ((g_bytes + 255) & ~static_cast<size_t>(255)) + s_bytes;
}

int ssd_head_dim() { return kP; }

size_t ssd_states_offset(int batch, int L, int H, int chunk) {
  const size_t nc = (static_cast<size_t>(L) + chunk - 1) / chunk;
  const size_t g_bytes = static_cast<size_t>(batch) * H * nc * chunk * 4;
  return (g_bytes + 255) & ~static_cast<size_t>(255);
}

cudaError_t launch_ssd_sm103(const SsdLaunch& a) {
  SsdParams p;
  p.dt = a.dt;
  p.A = a.A;
  p.h0 = a.h0;
  p.y = static_cast<__nv_bfloat16*>(a.y);
  p.h_final = a.h_final;
  p.g = static_cast<float*>(a.workspace);
  p.s_init = reinterpret_cast<__nv_bfloat16*>(static_cast<uint8_t*>(a.workspace) +
                                              ssd_states_offset(a.batch, a.L, a.H, a.chunk));
  p.batch = a.batch;
  p.L = a.L;
  p.H = a.H;
  p.G = a.G;
  p.nc = (a.L + a.chunk - 1) / a.chunk;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  if (a.N == 128) {
    if (a.chunk == 256) return launch_nq<128, 256>(a, p);
    if (a.chunk == 128) return launch_nq<128, 128>(a, p);
    return launch_nq<128, 64>(a, p);
  }
  if (a.chunk == 256) return launch_nq<64, 256>(a, p);
  if (a.chunk == 128) return launch_nq<64, 128>(a, p);
  return launch_nq<64, 64>(a, p);
}

}  // namespace attn47
