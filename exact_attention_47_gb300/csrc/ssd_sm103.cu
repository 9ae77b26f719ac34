// Mamba-2 SSD forward, chunked ("Accelerating Mamba-2 with high-performance
// forward kernels in NVIDIA CUDA Tile"): the recurrence
//   h_t = exp(a_t) h_{t-1} + x_t b_t^T,  y_t = h_t c_t,  a_t = A[h] dt[t, h] < 0
// evaluated chunk by chunk in the page's three kernels:
//   1. ssd_cumsum_kernel: per chunk (restarting) running sum of a_t, scaled
//      by log2(e) so that every later exponential is an exp2;
//   2. ssd_state_kernel (fwd_pass_state): one CTA per (batch, head, 64-wide
//      state tile) walks the chunks in order, storing each chunk's initial
//      state (in bf16: the output kernel's matrix product takes it in bf16)
//      and carrying it across the chunk in fp32 with the jump formula
//        S <- 2^(g_last) S + sum_j 2^(g_last - g_j) x_j b_j^T
//      (the sum is a (P x Q) * (Q x 64) contraction on the tensor cores);
//   3. ssd_out_kernel: one CTA per (batch, chunk, head, 64-row block) forms
//        y_i = sum_{j <= i} (c_i . b_j) 2^(g_i - g_j) x_j + 2^(g_i) S c_i
//      as C B^T (tensor cores), the decay weights and the causal mask applied
//      in registers, then P X and C S^T (tensor cores).
// Every exponent is <= 0 (a_t < 0 and the mask keeps j <= i), as the page
// notes.  Warp-level bf16 MMAs (m16n8k16, fp32 accumulation) with operands
// staged in shared memory by cp.async, in the 128-byte-swizzled layout
// (16-byte column c of row r at c ^ (r & 7)) that ldmatrix reads without bank
// conflicts.  Layouts: x / y [batch, L, H, P] bf16, B / C [batch, L, G, N]
// bf16, dt [batch, L, H] fp32, A [H] fp32, states [batch, H, P, N] fp32.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "ssd_sm103.h"

namespace attn47 {
namespace {

constexpr int kP = 64;                 // head dim handled by the kernels
constexpr int kThreads = 128;          // 4 warps
constexpr int kNT = 64;                // state columns per ssd_state_kernel CTA
constexpr int kIB = 64;                // query rows per ssd_out_kernel CTA
constexpr float kLog2e = 1.4426950408889634f;

// Byte offset of 16-byte column c8 of row r in a swizzled tile of `rows`
// rows: columns come in blocks of 64 bf16 (128-byte rows), block after block.
__device__ __forceinline__ uint32_t swz(int rows, int r, int c8) {
  return static_cast<uint32_t>((c8 >> 3) * rows * 128 + r * 128 + (((c8 & 7) ^ (r & 7)) << 4));
}

// Copy `rows` rows of `cols` bf16 (cols a multiple of 8) from global rows
// `row_stride` bytes apart into a swizzled tile; rows at or past `valid`
// are zero-filled (cp.async with source size 0, given the tile's first row,
// which the callers keep inside the tensor, as its address).  All threads of
// the CTA take part.
__device__ __forceinline__ void load_tile(uint32_t s_tile, const uint8_t* g0, size_t row_stride,
                                          int rows, int cols, int valid) {
  const int per_row = cols / 8;
  for (int i = threadIdx.x; i < rows * per_row; i += kThreads) {
    const int r = i / per_row, c8 = i % per_row;
    const bool ok = r < valid;
    const uint8_t* src = ok ? g0 + static_cast<size_t>(r) * row_stride + c8 * 16 : g0;
    cp_async16(s_tile + swz(rows, r, c8), src, ok ? 16u : 0u);
  }
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ------------------------------------------------------------------ kernel 1
__global__ void __launch_bounds__(kThreads)
    ssd_cumsum_kernel(const float* __restrict__ dt, const float* __restrict__ A, float* __restrict__ g,
                      int batch, int L, int H, int nc, int Q) {
  const long long idx = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x;
  if (idx >= static_cast<long long>(batch) * nc * H) return;
  const int h = static_cast<int>(idx % H);
  const int c = static_cast<int>((idx / H) % nc);
  const int b = static_cast<int>(idx / (static_cast<long long>(H) * nc));
  const float a = __ldg(A + h);
  float* out = g + ((static_cast<size_t>(b) * H + h) * nc + c) * Q;
  float acc = 0.f;
  for (int i = 0; i < Q; ++i) {
    const int t = c * Q + i;
    if (t < L) acc = fmaf(a, __ldg(dt + (static_cast<size_t>(b) * L + t) * H + h), acc);
    out[i] = acc * kLog2e;                    // past the end: the chunk's last value
  }
}

// ------------------------------------------------------------------ kernel 2
struct StateSmem {
  __host__ __device__ static constexpr int x_bytes(int Q) { return Q * kP * 2; }
  __host__ __device__ static constexpr int b_bytes(int Q) { return Q * kNT * 2; }
};

__global__ void __launch_bounds__(kThreads)
    ssd_state_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ Bm,
                     const float* __restrict__ g, const float* __restrict__ h0,
                     uint8_t* __restrict__ s_init, float* __restrict__ h_final, int L, int H, int G,
                     int N, int nc, int Q) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nt_count = N / kNT;
  const int n_tile = blockIdx.x % nt_count;
  const int h = (blockIdx.x / nt_count) % H;
  const int b = blockIdx.x / (nt_count * H);
  const int grp = h / (H / G);
  const int n0 = n_tile * kNT;
  // Double-buffered chunk stages: x [Q][64], B [Q][64] (bf16, swizzled), g [Q] fp32.
  const int stage_bytes = StateSmem::x_bytes(Q) + StateSmem::b_bytes(Q) + Q * 4;
  const uint32_t s0 = smem_addr(smem);
  auto sx = [&](int s) { return s0 + s * stage_bytes; };
  auto sb = [&](int s) { return s0 + s * stage_bytes + StateSmem::x_bytes(Q); };
  auto sg = [&](int s) {
    return reinterpret_cast<float*>(smem + s * stage_bytes + StateSmem::x_bytes(Q) + StateSmem::b_bytes(Q));
  };
  const size_t x_row = static_cast<size_t>(H) * kP * 2;          // bytes between tokens of x
  const size_t b_row = static_cast<size_t>(G) * N * 2;           // ... of B
  const float* g_bh = g + (static_cast<size_t>(b) * H + h) * nc * Q;
  auto issue = [&](int c, int s) {
    const int t0 = c * Q;
    const int valid = min(Q, L - t0);
    load_tile(sx(s), x + ((static_cast<size_t>(b) * L + t0) * H + h) * kP * 2, x_row, Q, kP, valid);
    load_tile(sb(s), Bm + ((static_cast<size_t>(b) * L + t0) * G + grp) * N * 2 + n0 * 2, b_row, Q, kNT, valid);
    for (int i = threadIdx.x; i < Q / 4; i += kThreads)
      cp_async16(smem_addr(sg(s)) + i * 16, g_bh + static_cast<size_t>(c) * Q + i * 4, 16u);
    cp_async_commit();
  };

  // State fragment: warp w owns rows p = 16w .. 16w+15, all 64 columns
  // (8 tiles of 16 x 8; element e of tile j at p = 16w + lane/4 + 8*(e>>1),
  // n = 8j + 2*(lane%4) + (e&1)).
  float S[8][4];
  const int pr = 16 * warp + (lane >> 2);
  const int nc2 = 2 * (lane & 3);
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const int p = pr + 8 * (e >> 1), n = n0 + 8 * j + nc2 + (e & 1);
      S[j][e] = h0 ? __ldg(h0 + ((static_cast<size_t>(b) * H + h) * kP + p) * N + n) : 0.f;
    }

  issue(0, 0);
  for (int c = 0; c < nc; ++c) {
    const int s = c & 1;
    if (c + 1 < nc) {
      issue(c + 1, s ^ 1);
      cp_async_wait<1>();
    } else {
      cp_async_wait<0>();
    }
    __syncthreads();
    const int n_len = min(Q, L - c * Q);
    const float* gs = sg(s);
    const float g_last = gs[n_len - 1];
    // x_t <- bf16(x_t * 2^(g_last - g_t)) in place (rows past the end are zero).
    uint8_t* xs = smem + s * stage_bytes;
    for (int i = threadIdx.x; i < Q * (kP / 8); i += kThreads) {
      const int r = i / (kP / 8), c8 = i % (kP / 8);
      uint4* piece = reinterpret_cast<uint4*>(xs + swz(Q, r, c8));
      const float w = exp2f(g_last - gs[r]);
      uint4 v = *piece;
      uint32_t* vw = reinterpret_cast<uint32_t*>(&v);
#pragma unroll
      for (int k = 0; k < 4; ++k)
        vw[k] = pack_bf16x2(__uint_as_float(vw[k] << 16) * w, __uint_as_float(vw[k] & 0xffff0000u) * w);
      *piece = v;
    }
    // Store this chunk's initial state (bf16), then decay it to the chunk's end.
    const float decay = exp2f(g_last);
    uint8_t* si = s_init + ((static_cast<size_t>(b) * nc + c) * H + h) * kP * N * 2;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
#pragma unroll
      for (int e2 = 0; e2 < 2; ++e2) {
        const int p = pr + 8 * e2, n = n0 + 8 * j + nc2;
        *reinterpret_cast<uint32_t*>(si + (static_cast<size_t>(p) * N + n) * 2) =
            pack_bf16x2(S[j][2 * e2], S[j][2 * e2 + 1]);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) S[j][e] *= decay;
    }
    fence_proxy_async_smem();                 // (generic writes above; ldmatrix reads below)
    __syncthreads();
    // S += (x')^T B over the chunk's Q positions: A[p][t] from x' [t][p]
    // (transposed load), B[t][n] from B [t][n] (transposed load).
    const uint32_t ax = sx(s), bx = sb(s);
    for (int kk = 0; kk < Q / 16; ++kk) {
      uint32_t a[4];
      {
        const int t = 16 * kk + (lane & 7) + ((lane >> 4) << 3);
        const int c8 = 2 * warp + ((lane >> 3) & 1);
        ldsm_x4_trans(ax + swz(Q, t, c8), a);
      }
#pragma unroll
      for (int j2 = 0; j2 < 4; ++j2) {
        const int t = 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
        const int c8 = 2 * j2 + (lane >> 4);
        uint32_t bb[4];
        ldsm_x4_trans(bx + swz(Q, t, c8), bb);
        mma_16816(S[2 * j2], a, bb[0], bb[1]);
        mma_16816(S[2 * j2 + 1], a, bb[2], bb[3]);
      }
    }
    __syncthreads();                          // the stage is refilled two chunks later
  }
  float* hf = h_final + (static_cast<size_t>(b) * H + h) * kP * N;
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e2 = 0; e2 < 2; ++e2) {
      const int p = pr + 8 * e2, n = n0 + 8 * j + nc2;
      *reinterpret_cast<float2*>(hf + static_cast<size_t>(p) * N + n) = make_float2(S[j][2 * e2], S[j][2 * e2 + 1]);
    }
}

// ------------------------------------------------------------------ kernel 3
template <int N>
__global__ void __launch_bounds__(kThreads)
    ssd_out_kernel(const uint8_t* __restrict__ x, const uint8_t* __restrict__ Bm,
                   const uint8_t* __restrict__ Cm, const float* __restrict__ g,
                   const uint8_t* __restrict__ s_init, uint8_t* __restrict__ y, int L, int H, int G,
                   int nc, int Q) {
  extern __shared__ __align__(1024) uint8_t smem[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_ib = Q / kIB;
  const int ib = blockIdx.x % n_ib;
  const int h = (blockIdx.x / n_ib) % H;
  const int c = (blockIdx.x / (n_ib * H)) % nc;
  const int b = blockIdx.x / (n_ib * H * nc);
  const int grp = h / (H / G);
  const int t0 = c * Q;
  const int n_len = min(Q, L - t0);
  if (ib * kIB >= n_len) return;              // a block wholly past the end writes nothing
  const int jrows = kIB * (ib + 1);           // keys 0 .. 64(ib+1)-1 of the chunk
  // Shared memory: C_i [64][N], B [jrows][N], X [jrows][64], S [64][N] (bf16,
  // swizzled), g [Q] fp32.
  const uint32_t s0 = smem_addr(smem);
  const uint32_t sC = s0;
  const uint32_t sB = sC + kIB * N * 2;
  const uint32_t sX = sB + jrows * N * 2;
  const uint32_t sS = sX + jrows * kP * 2;
  float* gs = reinterpret_cast<float*>(smem + (sS - s0) + kP * N * 2);
  const size_t bc_row = static_cast<size_t>(G) * N * 2;
  const uint8_t* c0 = Cm + ((static_cast<size_t>(b) * L + t0 + ib * kIB) * G + grp) * N * 2;
  load_tile(sC, c0, bc_row, kIB, N, n_len - ib * kIB);
  load_tile(sB, Bm + ((static_cast<size_t>(b) * L + t0) * G + grp) * N * 2, bc_row, jrows, N, n_len);
  load_tile(sX, x + ((static_cast<size_t>(b) * L + t0) * H + h) * kP * 2, static_cast<size_t>(H) * kP * 2,
            jrows, kP, n_len);
  // The chunk's initial state S [p][n] (bf16, as the state kernel stored it).
  load_tile(sS, s_init + ((static_cast<size_t>(b) * nc + c) * H + h) * kP * N * 2,
            static_cast<size_t>(N) * 2, kP, N, kP);
  const float* g_c = g + ((static_cast<size_t>(b) * H + h) * nc + c) * Q;
  for (int i = threadIdx.x; i < Q / 4; i += kThreads) cp_async16(smem_addr(gs) + i * 16, g_c + i * 4, 16u);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();

  // Rows of this warp: i = ib*64 + 16*warp + lane/4 (+8); A fragments of C_i
  // for the N/16 steps of the contraction over the state dimension.
  uint32_t ca[N / 16][4];
#pragma unroll
  for (int kk = 0; kk < N / 16; ++kk)
    ldsm_x4(sC + swz(kIB, 16 * warp + (lane & 15), 2 * kk + (lane >> 4)), ca[kk]);
  const int il0 = ib * kIB + 16 * warp + (lane >> 2);              // chunk position of rows e = 0, 1
  const float gi0 = gs[min(il0, Q - 1)], gi1 = gs[min(il0 + 8, Q - 1)];

  float Y[8][4], Yc[8][4];
#pragma unroll
  for (int j = 0; j < 8; ++j)
#pragma unroll
    for (int e = 0; e < 4; ++e) Y[j][e] = Yc[j][e] = 0.f;
  // Within the chunk: for each 64-key block, S = C_i B_j^T, weights and mask,
  // then Y += P X_j.
  for (int jb = 0; jb <= ib; ++jb) {
    float sc[8][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
      const int key = jb * kIB + nt * 8 + (lane & 7);
#pragma unroll
      for (int kk2 = 0; kk2 < N / 32; ++kk2) {
        uint32_t bb[4];
        ldsm_x4(sB + swz(jrows, key, 4 * kk2 + (lane >> 3)), bb);
        mma_16816(sc[nt], ca[2 * kk2], bb[0], bb[1]);
        mma_16816(sc[nt], ca[2 * kk2 + 1], bb[2], bb[3]);
      }
    }
    uint32_t pa[4][4];
#pragma unroll
    for (int nt = 0; nt < 8; ++nt) {
      float v[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int i = il0 + 8 * (e >> 1);
        const int j = jb * kIB + nt * 8 + 2 * (lane & 3) + (e & 1);
        const float gi = (e >> 1) ? gi1 : gi0;
        v[e] = (j <= i) ? sc[nt][e] * exp2f(gi - gs[j]) : 0.f;
      }
      pa[nt >> 1][(nt & 1) * 2 + 0] = pack_bf16x2(v[0], v[1]);
      pa[nt >> 1][(nt & 1) * 2 + 1] = pack_bf16x2(v[2], v[3]);
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
#pragma unroll
      for (int dt2 = 0; dt2 < kP / 16; ++dt2) {
        const int key = jb * kIB + 16 * kk + (lane & 7) + ((lane >> 3) & 1) * 8;
        uint32_t bb[4];
        ldsm_x4_trans(sX + swz(jrows, key, 2 * dt2 + (lane >> 4)), bb);
        mma_16816(Y[2 * dt2], pa[kk], bb[0], bb[1]);
        mma_16816(Y[2 * dt2 + 1], pa[kk], bb[2], bb[3]);
      }
    }
  }
  // Carried state: Yc = C_i S^T  (B operand rows = p, columns = n).
#pragma unroll
  for (int pt = 0; pt < 8; ++pt) {
#pragma unroll
    for (int kk2 = 0; kk2 < N / 32; ++kk2) {
      uint32_t bb[4];
      ldsm_x4(sS + swz(kP, 8 * pt + (lane & 7), 4 * kk2 + (lane >> 3)), bb);
      mma_16816(Yc[pt], ca[2 * kk2], bb[0], bb[1]);
      mma_16816(Yc[pt], ca[2 * kk2 + 1], bb[2], bb[3]);
    }
  }
  // y_i = Y_i + 2^(g_i) Yc_i, rows past the end of the sequence skipped.
  const float w0 = exp2f(gi0), w1 = exp2f(gi1);
#pragma unroll
  for (int e2 = 0; e2 < 2; ++e2) {
    const int i = il0 + 8 * e2;
    if (i >= n_len) continue;
    const float w = e2 ? w1 : w0;
    uint8_t* yrow = y + ((static_cast<size_t>(b) * L + t0 + i) * H + h) * kP * 2;
#pragma unroll
    for (int pt = 0; pt < 8; ++pt) {
      const int p = 8 * pt + 2 * (lane & 3);
      *reinterpret_cast<uint32_t*>(yrow + p * 2) =
          pack_bf16x2(Y[pt][2 * e2] + w * Yc[pt][2 * e2], Y[pt][2 * e2 + 1] + w * Yc[pt][2 * e2 + 1]);
    }
  }
}

}  // namespace

size_t ssd_workspace_bytes(int batch, int L, int H, int N, int chunk) {
  const size_t nc = (static_cast<size_t>(L) + chunk - 1) / chunk;
  const size_t g_bytes = static_cast<size_t>(batch) * H * nc * chunk * 4;
  const size_t s_bytes = static_cast<size_t>(batch) * nc * H * kP * N * 2;
  return ((g_bytes + 255) & ~static_cast<size_t>(255)) + s_bytes;
}

int ssd_head_dim() { return kP; }

cudaError_t launch_ssd_sm103(const SsdLaunch& a) {
  const int nc = (a.L + a.chunk - 1) / a.chunk;
  const size_t g_bytes = static_cast<size_t>(a.batch) * a.H * nc * a.chunk * 4;
  float* g = static_cast<float*>(a.workspace);
  uint8_t* s_init = static_cast<uint8_t*>(a.workspace) + ((g_bytes + 255) & ~static_cast<size_t>(255));
  const long long n1 = static_cast<long long>(a.batch) * nc * a.H;
  ssd_cumsum_kernel<<<static_cast<unsigned>((n1 + kThreads - 1) / kThreads), kThreads, 0, a.stream>>>(
      a.dt, a.A, g, a.batch, a.L, a.H, nc, a.chunk);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int smem2 = 2 * (StateSmem::x_bytes(a.chunk) + StateSmem::b_bytes(a.chunk) + a.chunk * 4);
  e = cudaFuncSetAttribute(ssd_state_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem2);
  if (e != cudaSuccess) return e;
  const unsigned grid2 = static_cast<unsigned>(static_cast<long long>(a.batch) * a.H * (a.N / kNT));
  ssd_state_kernel<<<grid2, kThreads, smem2, a.stream>>>(
      static_cast<const uint8_t*>(a.x), static_cast<const uint8_t*>(a.B), g, a.h0, s_init, a.h_final,
      a.L, a.H, a.G, a.N, nc, a.chunk);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;

  const int smem3 = kIB * a.N * 2 + a.chunk * a.N * 2 + a.chunk * kP * 2 + kP * a.N * 2 + a.chunk * 4;
  const unsigned grid3 = static_cast<unsigned>(static_cast<long long>(a.batch) * nc * a.H * (a.chunk / kIB));
  auto k3 = a.N == 128 ? ssd_out_kernel<128> : ssd_out_kernel<64>;
  e = cudaFuncSetAttribute(k3, cudaFuncAttributeMaxDynamicSharedMemorySize, smem3);
  if (e != cudaSuccess) return e;
  k3<<<grid3, kThreads, smem3, a.stream>>>(static_cast<const uint8_t*>(a.x), static_cast<const uint8_t*>(a.B),
                                           static_cast<const uint8_t*>(a.C), g, s_init,
                                           static_cast<uint8_t*>(a.y), a.L, a.H, a.G, nc, a.chunk);
  return cudaGetLastError();
}

}  // namespace attn47
