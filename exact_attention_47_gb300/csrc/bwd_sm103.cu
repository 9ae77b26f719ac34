// Exact attention backward for sm_103a: dQ, dK, dV by recomputation.
//
// "Advanced attention mechanisms – II", section "Flash Attention": the
// forward keeps only O and the softmax statistics (the LSE) so that the
// backward pass can recompute the attention matrix tile by tile instead of
// reading a stored one.  With s = scale * Q K^T and P = exp(s - lse):
//     D_i  = sum_c dO_ic O_ic            (= sum_j P_ij dP_ij)
//     dV   = P^T dO,   dP = dO V^T,   dS = P * (dP - D)
//     dQ   = scale * dS K,   dK = scale * dS^T Q
// The score matrix never reaches HBM; with GQA the K/V gradients of a KV
// head are accumulated over its query heads inside one CTA.
//
// Two kernels, in stream order:
//   attn_bwd_rowdot_kernel     D and lse * log2(e) per query row (HBM-bound)
//   attn_bwd_kernel            one tile per CTA, of one of two kinds (one
//                              grid of both at d = 128, a grid of each at
//                              d = 64):
//     dK/dV: one 128-key tile, looping over the query tiles of every query
//            head of its group;
//     dQ:    one 128-row query tile, looping over K/V.
// Both kinds of tile: warps 0-7 compute (warp w: TMEM lanes 32 (w % 4) .., one
// row per thread, and columns 64 (w / 4) .. of the 128-wide score tiles; no
// value crosses columns, since the LSE and D are precomputed), warp 8 the
// TMA producer, warp 9 the MMA issuer and TMEM owner.  All contractions are
// tcgen05 MMAs with fp32 accumulators in TMEM; P and dS go back into TMEM as
// bf16 (each warp over the first half of its own 64 columns) and feed the
// next MMAs as their A operand.
#include <cuda_runtime.h>

#include "bwd_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kTile = 128;          // query rows / keys per tile (= TMEM lanes)
constexpr int kThreads = 320;
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
constexpr int kComputeWarps = 8;
// TMEM columns of the two halves of a step's 128 x 128 score tile (64
// columns each): S_h at 128 h, dP_h at 128 h + 64; the accumulators sit at
// 256 and up.
__device__ __forceinline__ uint32_t col_s(int h) { return static_cast<uint32_t>(h * 128); }
__device__ __forceinline__ uint32_t col_dp(int h) { return static_cast<uint32_t>(h * 128 + 64); }
// Column, relative to a half, of the packed bf16 operand for K step kk (16
// of its 64 keys / queries): each compute warp packs its 32 values 2 per
// column over the first 16 of its own 32 columns, so values 2c, 2c + 1 of
// warp part w live in column 32 w + c.
__device__ __forceinline__ uint32_t half_col(int kk) {
  return static_cast<uint32_t>((kk >> 1) * 32 + (kk & 1) * 8);
}
constexpr uint32_t kTmemCols = 512;
constexpr float kLog2e = 1.4426950408889634f;

template <int D>
struct BwdLayout {
  static constexpr int kChunks = D / 64;           // 128-byte swizzle atoms per row
  static constexpr int kTileBytes = kTile * D * 2;
  static constexpr int kChunkBytes = kTile * 128;  // one 64-column box of a tile
  static constexpr int kStages = 2;
  // dQ kernel: Q, dO once; K, V per stage.  dK/dV kernel: K, V once; Q, dO
  // (+ 128 lse2 and 128 D values) per stage.  Same sizes either way.
  static constexpr int kOffA = 0;                                  // Q (dq) | K (dkdv)
  static constexpr int kOffB = kOffA + kTileBytes;                 // dO (dq) | V (dkdv)
  static constexpr int kOffS0 = kOffB + kTileBytes;                // stage tiles
  static constexpr int kStageBytes = 2 * kTileBytes;
  static constexpr int kOffVec = kOffS0 + kStages * kStageBytes;   // [stage][lse2 | D][128]
  static constexpr int kVecBytes = kStages * 2 * kTile * 4;
  static constexpr int kOffBar = kOffVec + kVecBytes;
  static constexpr int kSmem = kOffBar + 256 + 1024;
};

struct BwdBarriers {
  uint64_t once_full;                 // the tiles loaded once per CTA
  uint64_t st_full[2], st_empty[2];   // per-stage tiles (and vectors)
  uint64_t s_full[2];                 // S and dP of a half are in TMEM
  uint64_t p_full[2];                 // the compute warps wrote a half's P / dS
  uint64_t done;                      // last accumulating MMA completed
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdBarriers) <= 256, "barrier block");

// ------------------------------------------------------------------ row dot
// D[r] = sum_c dO[r, c] * O[r, c] and lse2[r] = lse[r] * log2(e) for the
// query rows of every (batch, head), rows padded to whole tiles with zeros.
// A row is D / 8 sixteen-byte pieces, one per lane, so one load instruction
// of a warp covers 32 / (D / 8) rows; a warp takes kRowDotPasses such groups
// of consecutive rows and has all their loads in flight before it reduces.
constexpr int kRowDotPasses = 4;

template <int D>
__host__ __device__ constexpr int rowdot_rows_per_warp() { return 32 / (D / 8) * kRowDotPasses; }

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_rowdot_kernel(const BwdParams p) {
  constexpr int kPieces = D / 8;                   // lanes per row
  constexpr int kRowsPerPass = 32 / kPieces;
  const int lane = threadIdx.x & 31;
  const int piece = lane % kPieces;
  const int sub = lane / kPieces;
  const long long rows = static_cast<long long>(p.bh_q) * p.n_pad;
  const long long warps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
  // Programmatic dependent launch: nothing global is touched before the
  // preceding kernel has finished; the next kernel may start its set-up as
  // soon as every CTA of this grid is running.
  pdl_wait_primary();
  pdl_launch_dependents();
  for (long long r0 = (static_cast<long long>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5)) *
                      rowdot_rows_per_warp<D>();
       r0 < rows; r0 += warps * rowdot_rows_per_warp<D>()) {
    uint4 ov[kRowDotPasses], dv[kRowDotPasses];
    float lse[kRowDotPasses];
#pragma unroll
    for (int i = 0; i < kRowDotPasses; ++i) {
      const long long r = r0 + i * kRowsPerPass + sub;
      const long long bh = r / p.n_pad;
      const int n = static_cast<int>(r - bh * p.n_pad);
      ov[i] = dv[i] = make_uint4(0u, 0u, 0u, 0u);
      lse[i] = 0.f;
      if (r < rows && n < p.N) {
        const size_t row = static_cast<size_t>(bh) * p.N + n;
        ov[i] = __ldg(reinterpret_cast<const uint4*>(p.o + row * D) + piece);
        dv[i] = __ldg(reinterpret_cast<const uint4*>(p.dout + row * D) + piece);
        if (piece == 0) lse[i] = p.lse[row] * kLog2e;
      }
    }
#pragma unroll
    for (int i = 0; i < kRowDotPasses; ++i) {
      const unsigned ow[4] = {ov[i].x, ov[i].y, ov[i].z, ov[i].w};
      const unsigned dw[4] = {dv[i].x, dv[i].y, dv[i].z, dv[i].w};
      float dsum = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&ow[w]));
        const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&dw[w]));
        dsum += a.x * b.x;
        dsum += a.y * b.y;
      }
#pragma unroll
      for (int o = kPieces / 2; o > 0; o >>= 1) dsum += __shfl_xor_sync(0xffffffffu, dsum, o);
      const long long r = r0 + i * kRowsPerPass + sub;
      if (piece == 0 && r < rows) {
        p.ws_d[r] = dsum;
        p.ws_lse2[r] = lse[i];
      }
    }
  }
}

__device__ __forceinline__ void init_barriers(BwdBarriers* bar, int tid) {
  if (tid == 0) {
    mbar_init(smem_addr(&bar->once_full), 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bar->st_full[s]), 1);
      mbar_init(smem_addr(&bar->st_empty[s]), 1);
      mbar_init(smem_addr(&bar->s_full[s]), 1);
      mbar_init(smem_addr(&bar->p_full[s]), kComputeWarps);
    }
    mbar_init(smem_addr(&bar->done), 1);
    mbar_init(smem_addr(&bar->mma_final), 1);
    bar->abort = 0;
    fence_mbar_init();
  }
}

// ------------------------------------------------------------------- dQ
// Query tile `unit` of the dQ work (heaviest first under the causal mask).
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_dq_tile(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                            const CUtensorMap& tdo, const BwdParams& p, int unit) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  BwdBarriers* bar = reinterpret_cast<BwdBarriers*>(smem + L::kOffBar);
  const uint32_t sQ = smem_addr(smem + L::kOffA);
  const uint32_t sDO = smem_addr(smem + L::kOffB);
  const uint32_t sSt = smem_addr(smem + L::kOffS0);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nq = (p.N + kTile - 1) / kTile;
  const int qt = nq - 1 - unit / p.bh_q;                            // heaviest (last) tiles first
  const int bh = unit % p.bh_q;                                     // b * Hq + h
  const int zkv = (bh / p.Hq) * p.Hkv + (bh % p.Hq) / p.group;
  const int kv_total = nq;
  const int n_kv = CAUSAL ? min(qt + 1, kv_total) : kv_total;

  init_barriers(bar, threadIdx.x);
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(&bar->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtl wc{&bar->abort, p.status, p.timeout_ns};
  // Programmatic dependent launch: nothing global is touched before the
  // preceding kernel has finished; the next kernel may start its set-up as
  // soon as every CTA of this grid is running.
  pdl_wait_primary();
  pdl_launch_dependents();
  constexpr uint32_t kColDQ = 256;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      const uint32_t of = smem_addr(&bar->once_full);
      mbar_arrive_expect_tx(of, 2 * L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_3d(sQ + c * L::kChunkBytes, &tq, of, c * 64, qt * kTile, bh);
        tma_load_3d(sDO + c * L::kChunkBytes, &tdo, of, c * 64, qt * kTile, bh);
      }
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % L::kStages;
        if (!mbar_wait(smem_addr(&bar->st_empty[st]), ((j / L::kStages) & 1) ^ 1, wc)) break;
        const uint32_t f = smem_addr(&bar->st_full[st]);
        const uint32_t dst = sSt + st * L::kStageBytes;
        mbar_arrive_expect_tx(f, 2 * L::kTileBytes);
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_3d(dst + c * L::kChunkBytes, &tk, f, c * 64, j * kTile, zkv);
          tma_load_3d(dst + L::kTileBytes + c * L::kChunkBytes, &tv, f, c * 64, j * kTile, zkv);
        }
        ++issued;
      }
      mbar_wait(of, 0, wc, true);
      for (int st = 0; st < L::kStages; ++st) {
        const int fills = issued > st ? (issued - 1 - st) / L::kStages + 1 : 0;
        if (fills) mbar_wait(smem_addr(&bar->st_full[st]), (fills - 1) & 1, wc, true);
      }
    }
  } else if (warp == kWarpMma) {
    // --------------------------------------------------------- MMA issuer
    // Per K/V tile j and key half h (keys 64 h .. 64 h + 63 of the tile):
    //   S_h = Q K_h^T, dP_h = dO V_h^T            (sdp)
    //   dQ += dS_h K_h, dS_h bf16 over S_h        (acc)
    // issued as sdp(0, j) sdp(1, j) | acc(0, j) sdp(0, j+1) | acc(1, j)
    // sdp(1, j+1) | ..., so the tensor core works on one half while the
    // compute warps turn the other into dS.
    constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, 64, false);
    constexpr uint32_t kIdescDQ = idesc_bf16_f32(kTile, D, true);
    auto sdp = [&](int h, uint32_t kb) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
        umma_ss_warp(tmem + col_s(h), sdesc_sw128(sQ + o, 16, 1024), sdesc_sw128(kb + o + h * 8192, 16, 1024),
                     kIdescS, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
        umma_ss_warp(tmem + col_dp(h), sdesc_sw128(sDO + o, 16, 1024),
                     sdesc_sw128(kb + L::kTileBytes + o + h * 8192, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
      }
    };
    auto acc = [&](int h, uint32_t kb, bool first) {
      // B = K_h as K x N with N = d contiguous.
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bd = sdesc_sw128(kb + h * 8192 + kk * 2048, L::kChunkBytes, 1024);
        umma_ts_warp(tmem + kColDQ, tmem + col_s(h) + half_col(kk), bd, kIdescDQ, (first && kk == 0) ? 0u : 1u);
      }
    };
    bool ok = mbar_wait_warp(smem_addr(&bar->once_full), 0, wc) &&
              mbar_wait_warp(smem_addr(&bar->st_full[0]), 0, wc);
    if (ok) {
      tc_fence_after();
      sdp(0, sSt);
      umma_commit_warp(smem_addr(&bar->s_full[0]));
      sdp(1, sSt);
      umma_commit_warp(smem_addr(&bar->s_full[1]));
    }
    for (int j = 0; j < n_kv && ok; ++j) {
      const int st = j % L::kStages;
      const uint32_t kb = sSt + st * L::kStageBytes;
      const bool next = j + 1 < n_kv;
      const uint32_t kb1 = sSt + ((j + 1) % L::kStages) * L::kStageBytes;
      if (!(ok = mbar_wait_warp(smem_addr(&bar->p_full[0]), j & 1, wc))) break;
      tc_fence_after();
      acc(0, kb, j == 0);
      if (next) {
        if (!(ok = mbar_wait_warp(smem_addr(&bar->st_full[(j + 1) % L::kStages]), ((j + 1) / L::kStages) & 1, wc)))
          break;
        tc_fence_after();
        sdp(0, kb1);
        umma_commit_warp(smem_addr(&bar->s_full[0]));
      }
      if (!(ok = mbar_wait_warp(smem_addr(&bar->p_full[1]), j & 1, wc))) break;
      tc_fence_after();
      acc(1, kb, false);
      umma_commit_warp(smem_addr(&bar->st_empty[st]));
      if (next) {
        sdp(1, kb1);
        umma_commit_warp(smem_addr(&bar->s_full[1]));
      }
    }
    umma_commit_warp(smem_addr(&bar->done));
    umma_commit_warp(smem_addr(&bar->mma_final));
    __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar->mma_final), 0, wc, true));
  } else {
    // -------------------------------------------------------- compute warps
    const int quarter = warp & 3, w2 = warp >> 2;  // lane quarter, 32-column part of each half
    const int row = quarter * 32 + lane;          // TMEM lane = query row within the tile
    const int qrow = qt * kTile + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const size_t vrow = static_cast<size_t>(bh) * p.n_pad + qrow;
    const float lse2 = p.ws_lse2[vrow];
    const float dr = p.ws_d[vrow];
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_kv && ok; ++j) {
      const int kbase = j * kTile;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!mbar_wait_warp(smem_addr(&bar->s_full[h]), j & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // dS = P * (dP - D), P = 2^(s * scale * log2 e - lse * log2 e);
        // masked keys get P = 0.  32 keys of half h per warp.
        const uint32_t cs = col_s(h) + w2 * 32, cd = col_dp(h) + w2 * 32;
        uint32_t ra[32], rb[32], pk[16];
        ATTN47_TMEM_LD32(tl + cs, ra);
        ATTN47_TMEM_LD32(tl + cd, rb);
        ATTN47_TMEM_LD_WAIT(ra);
        ATTN47_TMEM_LD_WAIT(rb);
        // Keys k0 + c are allowed for c < hi (causal: key <= qrow; all:
        // key < N); the exponential is formed for every key and the masked
        // ones are then selected away, which keeps the loop free of branches.
        const int k0 = kbase + h * 64 + w2 * 32;
        const int hi = CAUSAL ? min(qrow - k0 + 1, p.N - k0) : p.N - k0;
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          float dsv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = 2 * c2 + e;
            const float ev = ex2(__uint_as_float(ra[c]) * sl2 - lse2);
            const float pv = c < hi ? ev : 0.f;
            dsv[e] = pv * (__uint_as_float(rb[c]) - dr);
          }
          pk[c2] = pack_bf16x2(dsv[0], dsv[1]);
        }
        ATTN47_TMEM_ST16(tl + cs, pk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bar->p_full[h]));
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && mbar_wait_warp(smem_addr(&bar->done), 0, wc)) {
      tc_fence_after();
      const bool in_range = qrow < p.N;
      __nv_bfloat16* dst = p.dq + (static_cast<size_t>(bh) * p.N + qrow) * D;
#pragma unroll 1
      for (int c0 = w2 * (D / 2); c0 < (w2 + 1) * (D / 2); c0 += 32) {
        uint32_t o[32];
        ATTN47_TMEM_LD32(tl + kColDQ + c0, o);
        ATTN47_TMEM_LD_WAIT(o);
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * p.scale, __uint_as_float(o[2 * c + 1]) * p.scale);
        if (in_range) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ----------------------------------------------------------------- dK, dV
// Key tile `unit` of the dK/dV work (heaviest first under the causal mask).
template <int D, bool CAUSAL>
__device__ __forceinline__ void bwd_dkdv_tile(const CUtensorMap& tq, const CUtensorMap& tk, const CUtensorMap& tv,
                                              const CUtensorMap& tdo, const BwdParams& p, int unit) {
  using L = BwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  BwdBarriers* bar = reinterpret_cast<BwdBarriers*>(smem + L::kOffBar);
  const uint32_t sK = smem_addr(smem + L::kOffA);
  const uint32_t sV = smem_addr(smem + L::kOffB);
  const uint32_t sSt = smem_addr(smem + L::kOffS0);
  const uint32_t sVec = smem_addr(smem + L::kOffVec);
  const float* vec = reinterpret_cast<const float*>(smem + L::kOffVec);   // [stage][lse2 | D][128]
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  const int nq = (p.N + kTile - 1) / kTile;
  const int kt = unit / p.bh_kv;                                    // first key tiles see most queries
  const int bhk = unit % p.bh_kv;                                   // b * Hkv + g
  const int b = bhk / p.Hkv, g = bhk % p.Hkv;
  const int qt0 = CAUSAL ? kt : 0;
  const int per_head = nq - qt0;
  const int steps = p.group * per_head;                              // (query head, query tile) pairs
  auto step_q = [&](int t, int& zq, int& qt) {
    zq = b * p.Hq + g * p.group + t / per_head;
    qt = qt0 + t % per_head;
  };

  init_barriers(bar, threadIdx.x);
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(&bar->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtl wc{&bar->abort, p.status, p.timeout_ns};
  // Programmatic dependent launch: nothing global is touched before the
  // preceding kernel has finished; the next kernel may start its set-up as
  // soon as every CTA of this grid is running.
  pdl_wait_primary();
  pdl_launch_dependents();
  constexpr uint32_t kColDV = 256, kColDK = 256 + D;

  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      prefetch_tmap(&tdo);
      const uint32_t of = smem_addr(&bar->once_full);
      mbar_arrive_expect_tx(of, 2 * L::kTileBytes);
      for (int c = 0; c < L::kChunks; ++c) {
        tma_load_3d(sK + c * L::kChunkBytes, &tk, of, c * 64, kt * kTile, bhk);
        tma_load_3d(sV + c * L::kChunkBytes, &tv, of, c * 64, kt * kTile, bhk);
      }
      int issued = 0;
      for (int t = 0; t < steps; ++t) {
        int zq, qt;
        step_q(t, zq, qt);
        const int st = t % L::kStages;
        if (!mbar_wait(smem_addr(&bar->st_empty[st]), ((t / L::kStages) & 1) ^ 1, wc)) break;
        const uint32_t f = smem_addr(&bar->st_full[st]);
        const uint32_t dst = sSt + st * L::kStageBytes;
        mbar_arrive_expect_tx(f, 2 * L::kTileBytes + 2 * kTile * 4);
        for (int c = 0; c < L::kChunks; ++c) {
          tma_load_3d(dst + c * L::kChunkBytes, &tq, f, c * 64, qt * kTile, zq);
          tma_load_3d(dst + L::kTileBytes + c * L::kChunkBytes, &tdo, f, c * 64, qt * kTile, zq);
        }
        const size_t v0 = static_cast<size_t>(zq) * p.n_pad + static_cast<size_t>(qt) * kTile;
        bulk_load(sVec + (st * 2 + 0) * kTile * 4, p.ws_lse2 + v0, kTile * 4, f);
        bulk_load(sVec + (st * 2 + 1) * kTile * 4, p.ws_d + v0, kTile * 4, f);
        ++issued;
      }
      mbar_wait(of, 0, wc, true);
      for (int st = 0; st < L::kStages; ++st) {
        const int fills = issued > st ? (issued - 1 - st) / L::kStages + 1 : 0;
        if (fills) mbar_wait(smem_addr(&bar->st_full[st]), (fills - 1) & 1, wc, true);
      }
    }
  } else if (warp == kWarpMma) {
    // --------------------------------------------------------- MMA issuer
    // Per step t (a query tile of one query head) and query half h
    // (queries 64 h .. 64 h + 63 of the tile):
    //   S_h^T = K Q_h^T, dP_h^T = V dO_h^T                (sdp)
    //   dV += P_h^T dO_h, dK += dS_h^T Q_h                 (acc)
    // issued as sdp(0, t) sdp(1, t) | acc(0, t) sdp(0, t+1) | acc(1, t)
    // sdp(1, t+1) | ..., so the tensor core works on one half while the
    // compute warps turn the other into P^T and dS^T.
    constexpr uint32_t kIdescS = idesc_bf16_f32(kTile, 64, false);
    constexpr uint32_t kIdescAcc = idesc_bf16_f32(kTile, D, true);
    auto sdp = [&](int h, uint32_t qb) {
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
        umma_ss_warp(tmem + col_s(h), sdesc_sw128(sK + o, 16, 1024), sdesc_sw128(qb + o + h * 8192, 16, 1024),
                     kIdescS, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t o = (kk >> 2) * L::kChunkBytes + (kk & 3) * 32;
        umma_ss_warp(tmem + col_dp(h), sdesc_sw128(sV + o, 16, 1024),
                     sdesc_sw128(qb + L::kTileBytes + o + h * 8192, 16, 1024), kIdescS, kk > 0 ? 1u : 0u);
      }
    };
    auto acc = [&](int h, uint32_t qb, bool first) {
      // B = dO_h / Q_h as K x N with N = d contiguous.
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bdo = sdesc_sw128(qb + L::kTileBytes + h * 8192 + kk * 2048, L::kChunkBytes, 1024);
        umma_ts_warp(tmem + kColDV, tmem + col_s(h) + half_col(kk), bdo, kIdescAcc, (first && kk == 0) ? 0u : 1u);
      }
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t bq = sdesc_sw128(qb + h * 8192 + kk * 2048, L::kChunkBytes, 1024);
        umma_ts_warp(tmem + kColDK, tmem + col_dp(h) + half_col(kk), bq, kIdescAcc, (first && kk == 0) ? 0u : 1u);
      }
    };
    bool ok = mbar_wait_warp(smem_addr(&bar->once_full), 0, wc) &&
              mbar_wait_warp(smem_addr(&bar->st_full[0]), 0, wc);
    if (ok) {
      tc_fence_after();
      sdp(0, sSt);
      umma_commit_warp(smem_addr(&bar->s_full[0]));
      sdp(1, sSt);
      umma_commit_warp(smem_addr(&bar->s_full[1]));
    }
    for (int t = 0; t < steps && ok; ++t) {
      const int st = t % L::kStages;
      const uint32_t qb = sSt + st * L::kStageBytes;
      const bool next = t + 1 < steps;
      const uint32_t qb1 = sSt + ((t + 1) % L::kStages) * L::kStageBytes;
      if (!(ok = mbar_wait_warp(smem_addr(&bar->p_full[0]), t & 1, wc))) break;
      tc_fence_after();
      acc(0, qb, t == 0);
      if (next) {
        if (!(ok = mbar_wait_warp(smem_addr(&bar->st_full[(t + 1) % L::kStages]), ((t + 1) / L::kStages) & 1, wc)))
          break;
        tc_fence_after();
        sdp(0, qb1);
        umma_commit_warp(smem_addr(&bar->s_full[0]));
      }
      if (!(ok = mbar_wait_warp(smem_addr(&bar->p_full[1]), t & 1, wc))) break;
      tc_fence_after();
      acc(1, qb, false);
      umma_commit_warp(smem_addr(&bar->st_empty[st]));
      if (next) {
        sdp(1, qb1);
        umma_commit_warp(smem_addr(&bar->s_full[1]));
      }
    }
    umma_commit_warp(smem_addr(&bar->done));
    umma_commit_warp(smem_addr(&bar->mma_final));
    __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar->mma_final), 0, wc, true));
  } else {
    // -------------------------------------------------------- compute warps
    const int quarter = warp & 3, w2 = warp >> 2;  // lane quarter, 32-column part of each half
    const int row = quarter * 32 + lane;          // TMEM lane = key within the tile
    const int key = kt * kTile + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int t = 0; t < steps && ok; ++t) {
      int zq, qt;
      step_q(t, zq, qt);
      const int st = t % L::kStages;
      // The lse2 / D vectors of this step landed with the stage's tiles.
      if (!mbar_wait_warp(smem_addr(&bar->st_full[st]), (t / L::kStages) & 1, wc)) {
        ok = false;
        break;
      }
      const float* lse2v = vec + (st * 2 + 0) * kTile;
      const float* dv = vec + (st * 2 + 1) * kTile;
      const int qbase = qt * kTile;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!mbar_wait_warp(smem_addr(&bar->s_full[h]), t & 1, wc)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // Row = key, column = query: P^T = 2^(s * scale * log2 e - lse2[q]),
        // dS^T = P^T * (dP^T - D[q]); masked pairs (key > query, or a query
        // past N) get P = 0.  P^T goes over S_h^T, dS^T over dP_h^T; 32
        // queries of half h per warp.
        const uint32_t cs = col_s(h) + w2 * 32, cd = col_dp(h) + w2 * 32;
        uint32_t ra[32], rb[32], pk[16], dspk[16];
        ATTN47_TMEM_LD32(tl + cs, ra);
        ATTN47_TMEM_LD32(tl + cd, rb);
        ATTN47_TMEM_LD_WAIT(ra);
        ATTN47_TMEM_LD_WAIT(rb);
        // Queries qbase + c0 + c are allowed for lo <= c < hi (causal:
        // query >= key; all: query < N); the exponential is formed for every
        // query and the masked ones are then selected away (no branches).
        const int c0 = h * 64 + w2 * 32;
        const int lo = CAUSAL ? key - qbase - c0 : 0;
        const int hi = p.N - qbase - c0;
#pragma unroll
        for (int c2 = 0; c2 < 16; ++c2) {
          float pv[2], dsv[2];
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int c = 2 * c2 + e;
            const int qc = c0 + c;
            const float ev = ex2(__uint_as_float(ra[c]) * sl2 - lse2v[qc]);
            pv[e] = (c >= lo && c < hi) ? ev : 0.f;
            dsv[e] = pv[e] * (__uint_as_float(rb[c]) - dv[qc]);
          }
          pk[c2] = pack_bf16x2(pv[0], pv[1]);
          dspk[c2] = pack_bf16x2(dsv[0], dsv[1]);
        }
        ATTN47_TMEM_ST16(tl + cs, pk);
        ATTN47_TMEM_ST16(tl + cd, dspk);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&bar->p_full[h]));
      }
    }
    ok = __all_sync(0xffffffffu, ok);
    if (ok && mbar_wait_warp(smem_addr(&bar->done), 0, wc)) {
      tc_fence_after();
      const bool in_range = key < p.N;
      const size_t rowoff = (static_cast<size_t>(bhk) * p.N + key) * D;
#pragma unroll 1
      for (int which = 0; which < 2; ++which) {
        __nv_bfloat16* dst = (which ? p.dk : p.dv) + rowoff;
        const float mul = which ? p.scale : 1.f;
        const uint32_t col = which ? kColDK : kColDV;
#pragma unroll 1
        for (int c0 = w2 * (D / 2); c0 < (w2 + 1) * (D / 2); c0 += 32) {
          uint32_t o[32];
          ATTN47_TMEM_LD32(tl + col + c0, o);
          ATTN47_TMEM_LD_WAIT(o);
          uint32_t w[16];
#pragma unroll
          for (int c = 0; c < 16; ++c)
            w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * mul, __uint_as_float(o[2 * c + 1]) * mul);
          if (in_range) {
            uint4* d4 = reinterpret_cast<uint4*>(dst + c0);
#pragma unroll
            for (int c = 0; c < 4; ++c) d4[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
          }
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ------------------------------------------------------------ launches
// The dK/dV and dQ work are independent (both read only the row-dot pass's
// output).  At d = 128 one grid carries both (KIND 0): the dK/dV key tiles
// first (the largest units: a key tile of a KV head covers the query tiles
// of all its query heads), then the dQ query tiles, heaviest first; the
// many small dQ units fill the SMs that the dK/dV units' uneven causal sizes
// leave idle.  At d = 64 the units are short and the two kinds run as two
// grids, dQ (KIND 1) then dK/dV (KIND 2), which measured faster there.
template <int D, bool CAUSAL, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                    const __grid_constant__ CUtensorMap tv, const __grid_constant__ CUtensorMap tdo,
                    const BwdParams p) {
  const int unit = static_cast<int>(blockIdx.x);
  if constexpr (KIND == 1) {
    bwd_dq_tile<D, CAUSAL>(tq, tk, tv, tdo, p, unit);
  } else if constexpr (KIND == 2) {
    bwd_dkdv_tile<D, CAUSAL>(tq, tk, tv, tdo, p, unit);
  } else {
    const int n_kv_units = (p.N + kTile - 1) / kTile * p.bh_kv;
    if (unit < n_kv_units) bwd_dkdv_tile<D, CAUSAL>(tq, tk, tv, tdo, p, unit);
    else bwd_dq_tile<D, CAUSAL>(tq, tk, tv, tdo, p, unit - n_kv_units);
  }
}

template <int D, bool CAUSAL, int KIND>
cudaError_t launch_tiles(const BwdLaunch& a, const BwdParams& p, unsigned units) {
  using L = BwdLayout<D>;
  auto k = attn_bwd_kernel<D, CAUSAL, KIND>;
  const cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  return launch_pdl(k, dim3(units), dim3(kThreads), L::kSmem, a.stream, *a.tq, *a.tk, *a.tv, *a.tdo, p);
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const BwdLaunch& a, BwdParams p) {
  const int nq = (a.N + kTile - 1) / kTile;
  {
    const long long rows = static_cast<long long>(p.bh_q) * p.n_pad;
    const long long per_cta = 8LL * rowdot_rows_per_warp<D>();   // eight warps
    const long long blocks = (rows + per_cta - 1) / per_cta;
    const cudaError_t e = launch_pdl(attn_bwd_rowdot_kernel<D>, dim3(static_cast<unsigned>(min(blocks, 65535LL * 16))),
                                     dim3(256), 0, a.stream, p);
    if (e != cudaSuccess) return e;
  }
  if constexpr (D == 128) {
    return launch_tiles<D, CAUSAL, 0>(a, p, static_cast<unsigned>(nq) * static_cast<unsigned>(p.bh_kv + p.bh_q));
  } else {
    const cudaError_t e = launch_tiles<D, CAUSAL, 1>(a, p, static_cast<unsigned>(nq) * static_cast<unsigned>(p.bh_q));
    if (e != cudaSuccess) return e;
    return launch_tiles<D, CAUSAL, 2>(a, p, static_cast<unsigned>(nq) * static_cast<unsigned>(p.bh_kv));
  }
}

}  // namespace

size_t bwd_workspace_bytes(int B, int Hq, int N) {
  const size_t n_pad = (static_cast<size_t>(N) + kTile - 1) / kTile * kTile;
  return 2 * static_cast<size_t>(B) * Hq * n_pad * sizeof(float);
}

int bwd_box_rows() { return kTile; }

cudaError_t launch_bwd_sm103(const BwdLaunch& a) {
  BwdParams p;
  p.o = reinterpret_cast<const __nv_bfloat16*>(a.o);
  p.dout = reinterpret_cast<const __nv_bfloat16*>(a.dout);
  p.lse = a.lse;
  p.dq = reinterpret_cast<__nv_bfloat16*>(a.dq);
  p.dk = reinterpret_cast<__nv_bfloat16*>(a.dk);
  p.dv = reinterpret_cast<__nv_bfloat16*>(a.dv);
  p.N = a.N;
  p.n_pad = (a.N + kTile - 1) / kTile * kTile;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.bh_q = a.B * a.Hq;
  p.bh_kv = a.B * a.Hkv;
  p.scale = a.scale;
  p.scale_log2 = a.scale * kLog2e;
  p.ws_lse2 = a.workspace;
  p.ws_d = a.workspace + static_cast<size_t>(p.bh_q) * p.n_pad;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  if (a.d == 128) return a.causal ? launch_t<128, true>(a, p) : launch_t<128, false>(a, p);
  return a.causal ? launch_t<64, true>(a, p) : launch_t<64, false>(a, p);
}

}  // namespace attn47
