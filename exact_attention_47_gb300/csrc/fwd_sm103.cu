// Exact attention forward (prefill) for sm_103a.
//
// softmax(scale * Q K^T + causal mask) V computed tile by tile with the
// running-max / running-sum softmax, so the N x N score matrix never leaves
// the SM ("Advanced attention mechanisms – II", sections "Flash Attention",
// "Tiling" steps 1-3, "Softmax stabiliser", "Incremental / online softmax";
// "Fast attention kernels and operator fusion accelerate AI models", section
// "FlashAttention-style attention and Paged Attention").
//
// One CTA owns one 128-row query tile of one (batch, query head) and streams
// the 128-row K/V tiles of its KV head:
//   warp 0      TMA producer: Q once, then K_j / V_j into a ring of stages
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into TMEM (fp32),
//               O += P_j V_j into TMEM; owns the TMEM allocation
//   warps 2..5  softmax: one thread per query row (= TMEM lane); masks,
//               running max/sum in the exp2 domain, rescales O when the max
//               moves, writes P_j (bf16) to shared memory; final O / l and LSE
// S is double-buffered in TMEM so S_{j+1} runs on the tensor core while the
// softmax warps work on S_j.
#include <cuda_runtime.h>

#include "fwd_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kBM = 128;           // query rows per tile (= TMEM lanes)
constexpr int kBN = 128;           // keys per tile
constexpr int kThreads = 192;      // 6 warps
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS0 = 0, kColS1 = 128, kColO = 256;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct FwdLayout {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kStages = (D == 128) ? 2 : 3;
  static constexpr int kQBytes = kBM * D * 2;
  static constexpr int kKVBytes = kBN * D * 2;
  static constexpr int kQChunk = kBM * 128;              // one 64-column box of the Q tile
  static constexpr int kKVChunk = kBN * 128;
  static constexpr int kPChunk = kBM * 128;
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kQBytes;
  static constexpr int kOffV = kOffK + kStages * kKVBytes;
  static constexpr int kOffP = kOffV + kStages * kKVBytes;
  static constexpr int kOffBar = kOffP + kBM * kBN * 2;
  static constexpr int kSmem = kOffBar + 512 + 1024;     // barriers + alignment slack
};

struct FwdBarriers {
  uint64_t q_full;
  uint64_t k_full[3], k_empty[3], v_full[3], v_empty[3];
  uint64_t s_full[2], s_free[2];
  uint64_t p_full, o_done, mma_final;
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  void* o;
  float* lse;
  int N, Hq, Hkv, group, num_q_tiles, bh_total;
  float scale_log2;
  unsigned int* status;
  unsigned long long timeout_ns;
};

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tq,
                          const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  using L = FwdLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  FwdBarriers* bar = reinterpret_cast<FwdBarriers*>(smem + L::kOffBar);
  const uint32_t sQ = smem_addr(smem + L::kOffQ);
  const uint32_t sK = smem_addr(smem + L::kOffK);
  const uint32_t sV = smem_addr(smem + L::kOffV);
  const uint32_t sP = smem_addr(smem + L::kOffP);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Heaviest (last, for causal) query tiles first across the whole grid.
  const int tile = p.num_q_tiles - 1 - static_cast<int>(blockIdx.x) / p.bh_total;
  const int bh = static_cast<int>(blockIdx.x) % p.bh_total;
  const int h = bh % p.Hq;
  const int b = bh / p.Hq;
  const int zq = bh;                                   // b * Hq + h
  const int zkv = b * p.Hkv + h / p.group;
  const int kv_tiles_total = (p.N + kBN - 1) / kBN;
  const int n_kv = CAUSAL ? min(tile + 1, kv_tiles_total) : kv_tiles_total;

  if (threadIdx.x == 0) {
    mbar_init(smem_addr(&bar->q_full), 1);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(smem_addr(&bar->k_full[s]), 1);
      mbar_init(smem_addr(&bar->v_full[s]), 1);
      mbar_init(smem_addr(&bar->k_empty[s]), 1);
      mbar_init(smem_addr(&bar->v_empty[s]), 1);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(smem_addr(&bar->s_full[s]), 1);
      mbar_init(smem_addr(&bar->s_free[s]), 4);
    }
    mbar_init(smem_addr(&bar->p_full), 4);
    mbar_init(smem_addr(&bar->o_done), 1);
    mbar_init(smem_addr(&bar->mma_final), 1);
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(&bar->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtl wc{&bar->abort, p.status, p.timeout_ns};

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      const uint32_t qf = smem_addr(&bar->q_full);
      mbar_arrive_expect_tx(qf, L::kQBytes);
      for (int c = 0; c < L::kChunks; ++c)
        tma_load_3d(sQ + c * L::kQChunk, &tq, qf, c * 64, tile * kBM, zq);
      int k_issued = 0, v_issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % L::kStages;
        const uint32_t ph = (j / L::kStages) & 1;
        if (!mbar_wait(smem_addr(&bar->k_empty[st]), ph ^ 1, wc)) break;
        const uint32_t kf = smem_addr(&bar->k_full[st]);
        mbar_arrive_expect_tx(kf, L::kKVBytes);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sK + st * L::kKVBytes + c * L::kKVChunk, &tk, kf, c * 64, j * kBN, zkv);
        ++k_issued;
        if (!mbar_wait(smem_addr(&bar->v_empty[st]), ph ^ 1, wc)) break;
        const uint32_t vf = smem_addr(&bar->v_full[st]);
        mbar_arrive_expect_tx(vf, L::kKVBytes);
        for (int c = 0; c < L::kChunks; ++c)
          tma_load_3d(sV + st * L::kKVBytes + c * L::kKVChunk, &tv, vf, c * 64, j * kBN, zkv);
        ++v_issued;
      }
      // Every copy issued must have landed before the CTA may exit.
      mbar_wait(qf, 0, wc, true);
      for (int st = 0; st < L::kStages; ++st) {
        const int nk = k_issued > st ? (k_issued - 1 - st) / L::kStages + 1 : 0;
        const int nv = v_issued > st ? (v_issued - 1 - st) / L::kStages + 1 : 0;
        if (nk) mbar_wait(smem_addr(&bar->k_full[st]), (nk - 1) & 1, wc, true);
        if (nv) mbar_wait(smem_addr(&bar->v_full[st]), (nv - 1) & 1, wc, true);
      }
    }
  } else if (warp == 1) {
    // --------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, D, true);
      bool ok = mbar_wait(smem_addr(&bar->q_full), 0, wc);
      auto issue_pv = [&](int i) -> bool {
        const int st = i % L::kStages;
        if (!mbar_wait(smem_addr(&bar->p_full), i & 1, wc)) return false;
        if (!mbar_wait(smem_addr(&bar->v_full[st]), (i / L::kStages) & 1, wc)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + st * L::kKVBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // A = P (K-major, 128-byte swizzle), B = V (MN-major: d contiguous).
          const uint64_t ad = sdesc_sw128(sP + (kk >> 2) * L::kPChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(vbase + kk * 2048, L::kKVChunk, 1024);
          umma_ss(tmem + kColO, ad, bd, kIdescPV, (i > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(smem_addr(&bar->o_done));
        umma_commit(smem_addr(&bar->v_empty[st]));
        return true;
      };
      if (ok) {
        tc_fence_after();
        for (int j = 0; j < n_kv && ok; ++j) {
          const int sb = j & 1;
          const int st = j % L::kStages;
          if (!mbar_wait(smem_addr(&bar->s_free[sb]), ((j >> 1) & 1) ^ 1, wc)) { ok = false; break; }
          if (!mbar_wait(smem_addr(&bar->k_full[st]), (j / L::kStages) & 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t kbase = sK + st * L::kKVBytes;
          const uint32_t dS = tmem + (sb ? kColS1 : kColS0);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint64_t ad = sdesc_sw128(sQ + (kk >> 2) * L::kQChunk + (kk & 3) * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * L::kKVChunk + (kk & 3) * 32, 16, 1024);
            umma_ss(dS, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
          }
          umma_commit(smem_addr(&bar->s_full[sb]));
          umma_commit(smem_addr(&bar->k_empty[st]));
          if (j > 0) ok = issue_pv(j - 1);
        }
        if (ok) issue_pv(n_kv - 1);
      }
      // All issued MMAs must retire before TMEM is released.
      umma_commit(smem_addr(&bar->mma_final));
      mbar_wait(smem_addr(&bar->mma_final), 0, wc, true);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int quarter = warp & 3;                  // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;           // row within the tile = TMEM lane
    const int qrow = tile * kBM + row;
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const float sl2 = p.scale_log2;
    float m = -INFINITY;                           // running max, exp2 domain
    float l = 0.f;                                 // running denominator
    bool ok = true;
    const uint32_t prow = sP + (row >> 3) * 1024 + (row & 7) * 128;

    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      if (!mbar_wait_warp(smem_addr(&bar->s_full[sb]), (j >> 1) & 1, wc)) { ok = false; break; }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      const uint32_t cs = tl + (sb ? kColS1 : kColS0);
      ATTN47_TMEM_LD32(cs + 0, r0);
      ATTN47_TMEM_LD32(cs + 32, r1);
      ATTN47_TMEM_LD32(cs + 64, r2);
      ATTN47_TMEM_LD32(cs + 96, r3);
      ATTN47_TMEM_LD_WAIT(r0);
      ATTN47_TMEM_LD_WAIT(r1);
      ATTN47_TMEM_LD_WAIT(r2);
      ATTN47_TMEM_LD_WAIT(r3);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->s_free[sb]));

      float s[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = __uint_as_float(r0[c]);
        s[32 + c] = __uint_as_float(r1[c]);
        s[64 + c] = __uint_as_float(r2[c]);
        s[96 + c] = __uint_as_float(r3[c]);
      }
      const int kbase = j * kBN;
      const bool need_mask = CAUSAL ? (kbase + kBN - 1 > tile * kBM) : (kbase + kBN > p.N);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int key = kbase + c;
          const bool masked = CAUSAL ? (key > qrow) : (key >= p.N);
          s[c] = masked ? -INFINITY : s[c];
        }
      }
      float mx = s[0];
#pragma unroll
      for (int c = 1; c < 128; ++c) mx = fmaxf(mx, s[c]);
      const float m_new = fmaxf(m, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = ex2(m - m_use);
      float rs = 0.f;
      uint32_t pk[64];
#pragma unroll
      for (int c = 0; c < 64; ++c) {
        const float p0 = ex2(fmaf(s[2 * c], sl2, -m_use));
        const float p1 = ex2(fmaf(s[2 * c + 1], sl2, -m_use));
        rs += p0 + p1;
        pk[c] = pack_bf16x2(p0, p1);
      }
      l = l * alpha + rs;
      m = m_new;

      // PV_{j-1} must have finished reading P and writing O.
      if (j > 0) {
        if (!mbar_wait_warp(smem_addr(&bar->o_done), (j - 1) & 1, wc)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c0 = 0; c0 < D; c0 += 32) {
            uint32_t o[32];
            ATTN47_TMEM_LD32(tl + kColO + c0, o);
            ATTN47_TMEM_LD_WAIT(o);
#pragma unroll
            for (int c = 0; c < 32; ++c) o[c] = __float_as_uint(__uint_as_float(o[c]) * alpha);
            ATTN47_TMEM_ST32(tl + kColO + c0, o);
          }
          tmem_st_wait();
        }
      }
      // P row -> shared memory in the K-major 128-byte-swizzled layout.
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        const uint32_t addr = prow + (c >> 3) * L::kPChunk + (((c & 7) ^ (row & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * c]),
                     "r"(pk[4 * c + 1]), "r"(pk[4 * c + 2]), "r"(pk[4 * c + 3])
                     : "memory");
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->p_full));
    }

    // ------------------------------------------------------------ epilogue
    if (ok && mbar_wait_warp(smem_addr(&bar->o_done), (n_kv - 1) & 1, wc)) {
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool in_range = qrow < p.N;
      __nv_bfloat16* orow =
          reinterpret_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(zq) * p.N + qrow) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        ATTN47_TMEM_LD32(tl + kColO + c0, o);
        ATTN47_TMEM_LD_WAIT(o);
        uint32_t w[16];
#pragma unroll
        for (int c = 0; c < 16; ++c)
          w[c] = pack_bf16x2(__uint_as_float(o[2 * c]) * inv_l, __uint_as_float(o[2 * c + 1]) * inv_l);
        if (in_range) {
          uint4* dst = reinterpret_cast<uint4*>(orow + c0);
#pragma unroll
          for (int c = 0; c < 4; ++c)
            dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
        }
      }
      if (in_range && p.lse != nullptr)
        p.lse[static_cast<size_t>(zq) * p.N + qrow] = (m + __log2f(l)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool CAUSAL>
cudaError_t launch_t(const FwdLaunch& a) {
  using L = FwdLayout<D>;
  auto kern = attn_fwd_sm103_kernel<D, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.o = a.o;
  p.lse = a.lse;
  p.N = a.N;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.num_q_tiles = (a.N + kBM - 1) / kBM;
  p.bh_total = a.B * a.Hq;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  const unsigned grid = static_cast<unsigned>(p.num_q_tiles) * static_cast<unsigned>(p.bh_total);
  kern<<<grid, kThreads, L::kSmem, a.stream>>>(*a.tq, *a.tk, *a.tv, p);
  return cudaGetLastError();
}

}  // namespace

int fwd_box_rows() { return kBM; }

cudaError_t launch_fwd_sm103(const FwdLaunch& a) {
  if (a.d == 128) return a.causal ? launch_t<128, true>(a) : launch_t<128, false>(a);
  return a.causal ? launch_t<64, true>(a) : launch_t<64, false>(a);
}

}  // namespace attn47
