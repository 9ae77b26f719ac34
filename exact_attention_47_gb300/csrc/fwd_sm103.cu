// Exact attention forward (prefill) for sm_103a.
//
// softmax(scale * Q K^T + causal mask) V computed tile by tile with the
// running-max / running-sum softmax, so the N x N score matrix never leaves
// the SM ("Advanced attention mechanisms – II", sections "Flash Attention",
// "Tiling" steps 1-3, "Softmax stabiliser", "Incremental / online softmax";
// "Fast attention kernels and operator fusion accelerate AI models", section
// "FlashAttention-style attention and Paged Attention").
//
// One CTA owns a 256-row query block of one (batch, query head), split into
// two 128-row tiles A and B that share every K/V tile of the KV head:
//   warps 0-3   softmax of tile A, one thread per query row (= TMEM lane)
//   warps 4-7   softmax of tile B
//   warp 8      TMA producer: Q_A, Q_B once, then K_j / V_j into a stage ring
//   warp 9      MMA issuer (one thread) and owner of the TMEM allocation
//   warps 10-11 idle (they complete the third warpgroup for setmaxnreg);
//               in paged mode they gather the K and V tiles
// Tensor memory: S_A, S_B (128 fp32 columns each), O_A, O_B (d columns
// each; at d = 64 with contiguous K/V, d + 16, the extra columns holding the
// row sums of P that P V forms against a ones column beside V).  After
// reading S_X, the softmax writes P_X (bf16, two per column)
// over the first 64 columns of S_X and the MMA reads it from there (A
// operand in TMEM), so P never touches shared memory.  The tensor core runs
// ... PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) ... in issue order, so while one
// warpgroup computes exponentials the tensor core works on the other tile,
// and the completion of S_X(j+1) also proves PV_X(j) has finished, which
// makes O_X and the P_X columns safe to touch again.
// The whole MMA warp runs the issuing schedule and one elected lane issues,
// so descriptors and barrier addresses stay warp-uniform values.  The
// issuer tests the barriers of its next group while the last MMAs of the
// current group are being issued, and never re-tests a stage it already
// knows is full: no barrier round trip sits between two groups.
//
// The stabiliser m of a row ("Softmax stabiliser") is only moved when the
// tile maximum exceeds it by more than 2^8 (in the exp2 domain), so O and l
// are rescaled rarely; exponents stay <= 8, numerators <= 256, and the final
// O / l and LSE are the same function of the same stabiliser.
//
// Paged mode (chunked prefill over a paged KV cache; same page, same
// section: the cache lives in fixed-size blocks and every position goes
// through the block table): the N query rows of sequence b are its new
// tokens at positions ctx_b .. ctx_b + N - 1, and K/V come from the cache.
// A 128-key tile is eight 16-slot blocks of 16 x d contiguous values each.
// Warps 10 (K) and 11 (V), idle otherwise, gather them: the lanes look up
// the eight table entries, then copy each block with 16-byte cp.async
// (a warp instruction moves 512 contiguous bytes) straight into the
// 128-byte-swizzled tile layout the MMA descriptors read, wait for their
// copies, fence them into the async proxy and arrive on the stage's full
// barrier.  (Sixteen 16-row TMA boxes per tile took about a quarter longer
// per tile than this.)  Blocks past the sequence are written as zeros.
// Query row i may see keys 0 .. ctx_b + i: the causal mask at an offset, so
// it can fall across two key tiles.  A unit's cost grows with
// ctx_b + its query block's first row, so units are walked in decreasing
// order of that key (every CTA ranks the (sequence, query block) pairs the
// same way at start-up) instead of query block by query block.
#include <cuda_runtime.h>

#include "fwd_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kBM = 128;            // rows per query tile (= TMEM lanes)
constexpr int kBN = 128;            // keys per K/V tile
constexpr int kTiles = 2;           // query tiles per CTA
constexpr int kRowsPerCta = kBM * kTiles;
constexpr int kThreads = 384;       // 2 softmax warpgroups + 1 producer/MMA warpgroup
constexpr int kWarpLoad = 8;
constexpr int kWarpMma = 9;
// Launched at 168 registers a thread (384 x 168 = 64512); the softmax
// warpgroups then take 216 and the producer/MMA warpgroup keeps 72:
// 256 x 216 + 128 x 72 = 64512, and per sub-partition 216 + 216 + 72 = 504
// = 3 x 168, so the increase never waits for registers nobody frees.
constexpr uint32_t kRegsSoftmax = 216;
constexpr uint32_t kRegsOther = 72;
constexpr uint32_t kTmemCols = 512;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kTau = 8.0f;        // lazy-rescale threshold, log2 units

// SUMV (d = 64 with contiguous K/V): the row sums of P come from the tensor
// core.  Every V stage gets a second 64-column chunk, written once, whose
// first column is all ones, and P V runs with N = d + 16: columns d .. d+15
// of O_X then hold P times that column, the row sums of the bf16 P that P V
// uses, at no extra MMA instruction (three stages instead of four make room).
template <int D, bool SUMV = false>
struct FwdLayout {
  static constexpr int kChunks = D / 64;                 // 128-byte swizzle atoms per row
  static constexpr int kStages = (D == 128) ? 2 : SUMV ? 3 : 4;
  static constexpr int kQTile = kBM * D * 2;
  static constexpr int kKV = kBN * D * 2;
  static constexpr int kQChunk = kBM * 128;              // one 64-column box of a Q tile
  static constexpr int kKVChunk = kBN * 128;
  static constexpr int kVStage = SUMV ? kKV + kKVChunk : kKV;   // V stage stride (+ the ones chunk)
  static constexpr int kNPV = SUMV ? D + 16 : D;         // N of the P V MMAs
  static constexpr int kOffQ = 0;
  static constexpr int kOffK = kOffQ + kTiles * kQTile;
  static constexpr int kOffV = kOffK + kStages * kKV;
  static constexpr int kOffBar = kOffV + kStages * kVStage;
  static constexpr int kOffCtx = kOffBar + 512;          // paged: ctx_b of each sequence
  static constexpr int kOffOrder = kOffCtx + 4 * 256;    // paged: (b << 16 | qblk) of each cost rank
  static constexpr int kSmem = kOffOrder + 4 * 2048 + 1024;   // + alignment slack
  static constexpr uint32_t kColS0 = 0, kColS1 = 128;
  static constexpr uint32_t kColO0 = 256, kColO1 = SUMV ? 384 : 256 + D;
};

struct FwdBarriers {
  uint64_t q_full[2], q_empty[2];     // Q tile x of the current work unit / free again
  uint64_t k_full[4], k_empty[4], v_full[4], v_empty[4];
  uint64_t s_full[2], p_full[2], o_done[2];
  uint64_t o_free[2];                 // O_X read out by the epilogue of the previous unit
  uint64_t mma_final;
  uint32_t tmem_base;
  int abort;
};

struct FwdParams {
  void* o;
  float* lse;
  int N, Hq, Hkv, group, num_q_blocks, bh_total, num_units;
  float scale_log2;
  unsigned int* status;
  unsigned long long timeout_ns;
  // paged mode only
  const uint8_t* k_cache;   // [num_blocks, Hkv, 16, D] bf16
  const uint8_t* v_cache;
  const int* block_table;   // [B, max_blocks]
  const int* ctx_lens;      // [B] tokens cached before the N new ones
  int max_blocks, num_blocks;
  int max_ctx;              // max_blocks * 16 - N: largest valid ctx_lens entry
};

// Cost ordering of the paged mode fits in shared memory up to these sizes
// (beyond them a second instantiation keeps the query-block-major order).
constexpr int kSortMaxSeqs = 256;
constexpr int kSortMaxPairs = 2048;

constexpr int kPageRows = 16;                        // token slots per cache block
constexpr int kPagesPerTile = kBN / kPageRows;
constexpr int kWarpGatherK = 10;                     // paged mode: K / V gather warps
constexpr int kWarpGatherV = 11;

template <int D, bool CAUSAL, bool PAGED, bool SORTED>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_sm103_kernel(const __grid_constant__ CUtensorMap tq,
                          const __grid_constant__ CUtensorMap tk,
                          const __grid_constant__ CUtensorMap tv, const FwdParams p) {
  constexpr bool SUMV = D == 64 && !PAGED;
  using L = FwdLayout<D, SUMV>;
  extern __shared__ uint8_t smem_raw[];
  // Aligned through an integer round trip (the pointer becomes generic):
  // measured faster for this kernel than smem_align1024.
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  FwdBarriers* bar = reinterpret_cast<FwdBarriers*>(smem + L::kOffBar);
  const uint32_t sQ = smem_addr(smem + L::kOffQ);
  const uint32_t sK = smem_addr(smem + L::kOffK);
  const uint32_t sV = smem_addr(smem + L::kOffV);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Persistent CTAs: work unit k (one 256-row query block of one (batch,
  // head)) in heaviest-first order (last query blocks first, for causal);
  // CTA c takes unit c of the first band of gridDim.x units, then walks the
  // bands in alternating directions so heavy and light units pair up.
  const int grid = static_cast<int>(gridDim.x);
  const int cta = static_cast<int>(blockIdx.x);
  auto unit_at = [&](int band) {
    return band * grid + ((band & 1) ? grid - 1 - cta : cta);
  };
  const int kv_total = (p.N + kBN - 1) / kBN;
  struct Unit {
    int qblk, zq, zkv, nA, nB;
    int pos0, b, kvh, nblk;                            // paged: ctx_b, sequence, KV head, blocks
  };
  const int* s_ctx = reinterpret_cast<const int*>(smem + L::kOffCtx);
  const int* s_order = reinterpret_cast<const int*>(smem + L::kOffOrder);
  auto unit_info = [&](int k) {
    Unit u;
    int bh;
    if constexpr (SORTED) {
      // Rank k / Hq of the (sequence, query block) pairs by decreasing cost;
      // the Hq heads of a pair are consecutive units (they share K/V tiles).
      const int r = k / p.Hq;
      const int e = s_order[r];
      u.qblk = e & 0xffff;
      bh = (e >> 16) * p.Hq + (k - r * p.Hq);
    } else {
      u.qblk = p.num_q_blocks - 1 - k / p.bh_total;
      bh = k % p.bh_total;
    }
    u.zq = bh;                                         // b * Hq + h
    u.b = bh / p.Hq;
    u.kvh = (bh % p.Hq) / p.group;
    u.zkv = u.b * p.Hkv + u.kvh;
    if constexpr (PAGED) {
      // A ctx_lens entry outside [0, max_ctx] was reported by the append
      // kernel; it is clamped here so every loop stays bounded.
      u.pos0 = min(max(__ldg(p.ctx_lens + u.b), 0), p.max_ctx);
      const int lastA = min(u.qblk * kRowsPerCta + kBM - 1, p.N - 1);
      const int lastB = min(u.qblk * kRowsPerCta + 2 * kBM - 1, p.N - 1);
      u.nA = (u.pos0 + lastA) / kBN + 1;               // tiles up to key pos0 + last row
      u.nB = (u.pos0 + lastB) / kBN + 1;
      u.nblk = min((u.pos0 + p.N + kPageRows - 1) / kPageRows, p.max_blocks);
    } else {
      u.pos0 = 0;
      u.nblk = 0;
      // K/V tiles each query tile needs; the diagonal tile of tile X is 2*qblk + X.
      u.nA = CAUSAL ? min(2 * u.qblk + 1, kv_total) : kv_total;
      u.nB = CAUSAL ? min(2 * u.qblk + 2, kv_total) : kv_total;
    }
    return u;
  };

  if (threadIdx.x == 0) {
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_addr(&bar->q_full[x]), 1);
      mbar_init(smem_addr(&bar->q_empty[x]), 1);
      mbar_init(smem_addr(&bar->o_free[x]), 4);
    }
    for (int s = 0; s < L::kStages; ++s) {
      // Paged: every lane of a gather warp arrives once its copies landed.
      mbar_init(smem_addr(&bar->k_full[s]), PAGED ? 32 : 1);
      mbar_init(smem_addr(&bar->v_full[s]), PAGED ? 32 : 1);
      mbar_init(smem_addr(&bar->k_empty[s]), 1);
      mbar_init(smem_addr(&bar->v_empty[s]), 1);
    }
    for (int x = 0; x < 2; ++x) {
      mbar_init(smem_addr(&bar->s_full[x]), 1);
      mbar_init(smem_addr(&bar->p_full[x]), 4);
      mbar_init(smem_addr(&bar->o_done[x]), 1);
    }
    mbar_init(smem_addr(&bar->mma_final), 1);
    bar->abort = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(smem_addr(&bar->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if constexpr (SUMV) {
    // The ones chunk of every V stage: in key row r, bf16 1.0 in its column
    // 0, whose 16-byte piece sits at piece 0 ^ (r mod 8) of the row's 128
    // bytes (the TMA's 128-byte swizzle); zeros elsewhere.
    for (int i = threadIdx.x; i < L::kStages * L::kKVChunk / 4; i += kThreads) {
      const int st = i / (L::kKVChunk / 4), k = i % (L::kKVChunk / 4);
      const int r = k / 32, w = k % 32;
      reinterpret_cast<uint32_t*>(smem + L::kOffV + st * L::kVStage + L::kKV)[k] =
          (w == (r & 7) * 4) ? 0x3F80u : 0u;
    }
    fence_proxy_async_smem();
  }
  // Launched as a programmatic dependent: the set-up above overlaps the end
  // of the kernel before this one in the stream; nothing in global memory
  // is read or written before that kernel has finished.
  pdl_wait_primary();
  if constexpr (SORTED) {
    {
      // Cost key of pair (b, qblk): ctx_b + 256 * qblk (the K/V tiles of the
      // unit grow with it).  Rank = pairs with a larger key, plus equal keys
      // of a smaller pair index; counted per sequence in closed form.
      const int S = p.bh_total / p.Hq;
      const int nq = p.num_q_blocks;
      int* ctx_w = reinterpret_cast<int*>(smem + L::kOffCtx);
      for (int b = threadIdx.x; b < S; b += kThreads) ctx_w[b] = min(max(__ldg(p.ctx_lens + b), 0), p.max_ctx);
      __syncthreads();
      int* order_w = reinterpret_cast<int*>(smem + L::kOffOrder);
      for (int i = threadIdx.x; i < S * nq; i += kThreads) {
        const int key = s_ctx[i / nq] + kRowsPerCta * (i % nq);
        int rank = 0;
        for (int b = 0; b < S; ++b) {
          const int dk = key - s_ctx[b];
          if (dk < 0) {
            rank += nq;                            // every block of b has a larger key
          } else {
            const int q0 = dk / kRowsPerCta;       // blocks above q0 have larger keys
            rank += max(nq - q0 - 1, 0);
            if (dk % kRowsPerCta == 0 && q0 < nq && b * nq + q0 < i) ++rank;
          }
        }
        order_w[rank] = ((i / nq) << 16) | (i % nq);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = bar->tmem_base;
  const WaitCtl wc{&bar->abort, p.status, p.timeout_ns};
  if (warp >= 8) {
  regs_decrease<kRegsOther>();
  if (warp == kWarpLoad) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      prefetch_tmap(&tq);
      prefetch_tmap(&tk);
      prefetch_tmap(&tv);
      int kv_issued = 0, k_issued = 0, v_issued = 0, units = 0;
      bool ok = true;
      for (int band = 0; ok; ++band) {
        const int k = unit_at(band);
        if (k >= p.num_units) break;
        const Unit u = unit_info(k);
        // Q tile x of this unit, once the last S MMA of the previous unit has
        // read it.  Order: Q_A, K_0, Q_B, V_0, K_1, ...: the first S MMA of
        // the unit needs only Q_A and K_0, which can land while the previous
        // unit's last tile-B MMAs still read Q_B.
        auto load_q = [&](int x) {
          if (units > 0 && !(ok = mbar_wait(smem_addr(&bar->q_empty[x]), (units - 1) & 1, wc))) return;
          const uint32_t qf = smem_addr(&bar->q_full[x]);
          mbar_arrive_expect_tx(qf, L::kQTile);
          for (int c = 0; c < L::kChunks; ++c)
            tma_load_3d(sQ + x * L::kQTile + c * L::kQChunk, &tq, qf, c * 64,
                        u.qblk * kRowsPerCta + x * kBM, u.zq);
        };
        load_q(0);
        if constexpr (PAGED) {                     // K/V come from the gather warps
          if (ok) load_q(1);
        }
        // K/V tiles: one stage ring for the whole CTA, across units.
        for (int j = 0; j < (PAGED ? 0 : u.nB) && ok; ++j) {
          const int g = kv_issued + j;
          const int st = g % L::kStages;
          const uint32_t ph = (g / L::kStages) & 1;
          auto load_kv = [&](uint32_t dst, const CUtensorMap* map, uint32_t full) {
            mbar_arrive_expect_tx(full, L::kKV);
            for (int c = 0; c < L::kChunks; ++c)
              tma_load_3d(dst + c * L::kKVChunk, map, full, c * 64, j * kBN, u.zkv);
          };
          if (!(ok = mbar_wait(smem_addr(&bar->k_empty[st]), ph ^ 1, wc))) break;
          load_kv(sK + st * L::kKV, &tk, smem_addr(&bar->k_full[st]));
          ++k_issued;
          if (j == 0) {
            load_q(1);
            if (!ok) break;
          }
          if (!(ok = mbar_wait(smem_addr(&bar->v_empty[st]), ph ^ 1, wc))) break;
          load_kv(sV + st * L::kVStage, &tv, smem_addr(&bar->v_full[st]));
          ++v_issued;
        }
        kv_issued += u.nB;
        ++units;
      }
      // Every load is issued: the next kernel in the stream may start
      // setting up on SMs this grid leaves (it waits for this grid to
      // finish before it touches memory).
      pdl_launch_dependents();
      // Every copy issued must have landed before the CTA may exit.
      if (units > 0)
        for (int x = 0; x < kTiles; ++x) mbar_wait(smem_addr(&bar->q_full[x]), (units - 1) & 1, wc, true);
      for (int st = 0; st < L::kStages; ++st) {
        const int nk = k_issued > st ? (k_issued - 1 - st) / L::kStages + 1 : 0;
        const int nv = v_issued > st ? (v_issued - 1 - st) / L::kStages + 1 : 0;
        if (nk) mbar_wait(smem_addr(&bar->k_full[st]), (nk - 1) & 1, wc, true);
        if (nv) mbar_wait(smem_addr(&bar->v_full[st]), (nv - 1) & 1, wc, true);
      }
    }
  } else if (warp == kWarpMma) {
    // --------------------------------------------------------- MMA issuer
    {
      constexpr uint32_t kIdescS = idesc_bf16_f32(kBM, kBN, false);
      constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, L::kNPV, true);
      constexpr int kSteps = D / 16;               // MMAs in an S group (K = d)
      constexpr int kPSteps = kBN / 16;            // MMAs in a PV group (K = keys)
      const uint32_t kF = smem_addr(&bar->k_full[0]);
      const uint32_t vF = smem_addr(&bar->v_full[0]);
      const uint32_t pF = smem_addr(&bar->p_full[0]);
      // K/V tile jj of the current unit is fill g0 + jj of the CTA's stage ring.
      int g0 = 0;
      auto kfull = [&](int jj) { return kF + 8u * ((g0 + jj) % L::kStages); };
      auto vfull = [&](int jj) { return vF + 8u * ((g0 + jj) % L::kStages); };
      auto ph = [&](int jj) { return static_cast<uint32_t>(((g0 + jj) / L::kStages) & 1); };
      // P_X(jj) of the current unit is completion pX0 + jj of p_full[X].
      int pa0 = 0, pb0 = 0;
      auto ppar = [&](int x, int jj) { return static_cast<uint32_t>(((x ? pb0 : pa0) + jj) & 1); };
      // A dependency that was probed ready is not waited on again.
      auto ensure = [&](uint32_t b, uint32_t parity, uint32_t probed) -> bool {
        return __all_sync(0xffffffffu, probed != 0u) || mbar_wait_warp(b, parity, wc);
      };
      // Next group's probes: issued before the last two MMAs of a group.
      uint32_t rA = 0, rB = 0;
      int probe_kind = 0, probe_x = 0, probe_j = 0;   // 1: PV (P, V)  2: S (K)
      auto do_probes = [&]() {
        if (probe_kind == 1) {
          rA = mbar_probe(pF + 8u * static_cast<uint32_t>(probe_x), ppar(probe_x, probe_j));
          rB = mbar_probe(vfull(probe_j), ph(probe_j));
        } else if (probe_kind == 2) {
          rA = mbar_probe(kfull(probe_j), ph(probe_j));
        }
      };
      auto group_s = [&](int x, int jj) {
        const int st = (g0 + jj) % L::kStages;
        const uint32_t qbase = sQ + x * L::kQTile;
        const uint32_t kbase = sK + st * L::kKV;
        const uint32_t dS = tmem + (x ? L::kColS1 : L::kColS0);
#pragma unroll
        for (int kk = 0; kk < kSteps; ++kk) {
          if (kk == kSteps - 2) do_probes();
          const uint64_t ad = sdesc_sw128(qbase + (kk >> 2) * L::kQChunk + (kk & 3) * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(kbase + (kk >> 2) * L::kKVChunk + (kk & 3) * 32, 16, 1024);
          umma_ss_warp(dS, ad, bd, kIdescS, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(smem_addr(&bar->s_full[x]));
      };
      auto group_pv = [&](int x, int jj) {
        const int st = (g0 + jj) % L::kStages;
        const uint32_t vbase = sV + st * L::kVStage;
        const uint32_t aP = tmem + (x ? L::kColS1 : L::kColS0);
        const uint32_t dO = tmem + (x ? L::kColO1 : L::kColO0);
#pragma unroll
        for (int kk = 0; kk < kPSteps; ++kk) {
          if (kk == kPSteps - 2) do_probes();
          // A = P from TMEM (8 columns = 16 keys per step), B = V (MN-major).
          const uint64_t bd = sdesc_sw128(vbase + kk * 2048, L::kKVChunk, 1024);
          umma_ts_warp(dO, aP + kk * 8, bd, kIdescPV, (jj > 0 || kk > 0) ? 1u : 0u);
        }
      };
      // Per unit (each group probes what the next one needs):
      //   S_A(0) S_B(0) | PV_A(j) S_A(j+1) PV_B(j) S_B(j+1) | ...
      // The first P V of a tile overwrites O_X, so it waits until the
      // epilogue of the previous unit has read O_X out; the last S group of
      // a tile releases its Q tile for the next unit's load.
      bool ok = true;
      int units = 0;
      for (int band = 0; ok; ++band) {
        const int k = unit_at(band);
        if (k >= p.num_units) break;
        const Unit u = unit_info(k);
        const int nA = u.nA, nB = u.nB;
        const uint32_t upar = static_cast<uint32_t>(units & 1);
        ok = mbar_wait_warp(smem_addr(&bar->q_full[0]), upar, wc) &&
             mbar_wait_warp(kfull(0), ph(0), wc);
        if (ok) {
          tc_fence_after();
          probe_kind = 0;
          group_s(0, 0);
          if (nA == 1) umma_commit_warp(smem_addr(&bar->q_empty[0]));
          ok = mbar_wait_warp(smem_addr(&bar->q_full[1]), upar, wc);
        }
        if (ok) {
          tc_fence_after();
          probe_kind = 1;                          // PV_A(0): P_A(0), V_0
          probe_x = 0;
          probe_j = 0;
          group_s(1, 0);
          if (nB == 1) umma_commit_warp(smem_addr(&bar->q_empty[1]));
          umma_commit_warp(smem_addr(&bar->k_empty[g0 % L::kStages]));
        }
        for (int j = 0; j < nB && ok; ++j) {
          const int st = (g0 + j) % L::kStages;
          if (j < nA) {
            // PV_A(j)
            if (!(ok = ensure(pF, ppar(0, j), rA) && ensure(vfull(j), ph(j), rB))) break;
            if (j == 0 && units > 0 && !(ok = mbar_wait_warp(smem_addr(&bar->o_free[0]), upar ^ 1, wc))) break;
            tc_fence_after();
            probe_kind = (j + 1 < nA) ? 2 : 0;     // S_A(j+1): K_{j+1}
            probe_j = j + 1;
            group_pv(0, j);
            if (j == nA - 1) umma_commit_warp(smem_addr(&bar->o_done[0]));
            if (j + 1 < nA) {
              // S_A(j+1)
              if (!(ok = ensure(kfull(j + 1), ph(j + 1), rA))) break;
              tc_fence_after();
              probe_kind = 1;                      // PV_B(j): P_B(j), V_j (known)
              probe_x = 1;
              probe_j = j;
              group_s(0, j + 1);
              if (j + 1 == nA - 1) umma_commit_warp(smem_addr(&bar->q_empty[0]));
              rB = 1;
            } else {
              rA = mbar_probe(pF + 8u, ppar(1, j));
              rB = 1;
            }
          } else {
            rA = mbar_probe(pF + 8u, ppar(1, j));
            rB = mbar_probe(vfull(j), ph(j));
          }
          // PV_B(j)
          if (!(ok = ensure(pF + 8u, ppar(1, j), rA) && ensure(vfull(j), ph(j), rB))) break;
          if (j == 0 && units > 0 && !(ok = mbar_wait_warp(smem_addr(&bar->o_free[1]), upar ^ 1, wc))) break;
          tc_fence_after();
          probe_kind = (j + 1 < nB && j + 1 >= nA) ? 2 : 0;   // S_B(j+1) needs K_{j+1} if S_A did not test it
          probe_j = j + 1;
          group_pv(1, j);
          umma_commit_warp(smem_addr(&bar->v_empty[st]));
          if (j == nB - 1) umma_commit_warp(smem_addr(&bar->o_done[1]));
          if (j + 1 < nB) {
            // S_B(j+1)
            if (j + 1 >= nA && !(ok = ensure(kfull(j + 1), ph(j + 1), rA))) break;
            tc_fence_after();
            probe_kind = (j + 1 < nA) ? 1 : 0;     // PV_A(j+1): P_A(j+1), V_{j+1}
            probe_x = 0;
            probe_j = j + 1;
            group_s(1, j + 1);
            if (j + 1 == nB - 1) umma_commit_warp(smem_addr(&bar->q_empty[1]));
            umma_commit_warp(smem_addr(&bar->k_empty[(g0 + j + 1) % L::kStages]));
          }
        }
        g0 += nB;
        pa0 += nA;
        pb0 += nB;
        ++units;
        probe_kind = 0;
        rA = rB = 0;
      }
      // All issued MMAs must retire before TMEM is released.
      umma_commit_warp(smem_addr(&bar->mma_final));
      __all_sync(0xffffffffu, mbar_wait(smem_addr(&bar->mma_final), 0, wc, true));
    }
  }
  if constexpr (PAGED) {
    if (warp == kWarpGatherK || warp == kWarpGatherV) {
      // ------------------------------------------------- paged K / V gather
      const bool is_v = warp == kWarpGatherV;
      const uint8_t* cache = is_v ? p.v_cache : p.k_cache;
      const uint32_t s_base = is_v ? sV : sK;
      const uint32_t full0 = smem_addr(is_v ? &bar->v_full[0] : &bar->k_full[0]);
      const uint32_t empty0 = smem_addr(is_v ? &bar->v_empty[0] : &bar->k_empty[0]);
      constexpr int kRowPieces = D / 8;                        // 16-byte pieces of one key row
      constexpr int kPerLane = kPageRows * kRowPieces / 32;    // pieces of one block per lane
      const size_t slice_bytes = static_cast<size_t>(kPageRows) * D * 2;
      int g = 0;                                               // fill index of the stage ring
      bool ok = true;
      for (int band = 0; ok; ++band) {
        const int k = unit_at(band);
        if (k >= p.num_units) break;
        const Unit u = unit_info(k);
        const int* row = p.block_table + static_cast<size_t>(u.b) * p.max_blocks;
        for (int j = 0; j < u.nB; ++j, ++g) {
          // Lane i < 8 translates block i of the tile (before the wait, so the
          // lookup overlaps it); p.num_blocks stands for "no block": zeros.
          int e = p.num_blocks;
          const int lb = j * kPagesPerTile + lane;
          if (lane < kPagesPerTile && lb < u.nblk) {
            e = __ldg(row + lb);
            if (static_cast<unsigned>(e) >= static_cast<unsigned>(p.num_blocks)) {
              atomicOr(p.status, kDevBadBlock);                // reported, read as zeros
              e = p.num_blocks;
            }
          }
          const int st = g % L::kStages;
          if (!(ok = mbar_wait_warp(empty0 + 8u * st, ((g / L::kStages) & 1) ^ 1, wc))) break;
          const uint32_t dst0 = s_base + st * L::kKV;
#pragma unroll 1
          for (int i = 0; i < kPagesPerTile; ++i) {
            const int phys = __shfl_sync(0xffffffffu, e, i);
            const bool valid = phys < p.num_blocks;
            const uint8_t* src0 = cache + (static_cast<size_t>(valid ? phys : 0) * p.Hkv + u.kvh) * slice_bytes;
#pragma unroll
            for (int t = 0; t < kPerLane; ++t) {
              const int piece = t * 32 + lane;                 // consecutive lanes: consecutive 16 B
              const int slot = piece / kRowPieces;
              const int col = piece % kRowPieces;
              // 128-byte swizzle: 16-byte column (col & 7) of row r sits at (col & 7) ^ (r & 7).
              const uint32_t dst = dst0 + (col >> 3) * L::kKVChunk + (i * kPageRows + slot) * 128 +
                                   ((static_cast<uint32_t>((col & 7) ^ (slot & 7))) << 4);
              cp_async16(dst, src0 + piece * 16, valid ? 16u : 0u);
            }
          }
          cp_async_wait_all();
          fence_proxy_async_smem();
          mbar_arrive(full0 + 8u * st);
        }
      }
    }
  }
    // Each role ends on the same named barrier, so the register-split
    // branches never merge back; then the MMA warp frees the TMEM.
    tc_fence_before();
    named_barrier_sync(1, kThreads);
    if (warp == kWarpMma) {
      tc_fence_after();
      tmem_dealloc(tmem, kTmemCols);
    }
  } else {
    regs_increase<kRegsSoftmax>();
    // ------------------------------------------------------------ softmax
    const int x = warp >> 2;                       // query tile of this warpgroup
    const int quarter = warp & 3;                  // TMEM lane quarter of this warp
    const int row = quarter * 32 + lane;           // row within the tile = TMEM lane
    const uint32_t tl = tmem + (static_cast<uint32_t>(quarter * 32) << 16);
    const uint32_t colS = x ? L::kColS1 : L::kColS0;
    const uint32_t colO = x ? L::kColO1 : L::kColO0;
    const float sl2 = p.scale_log2;
    bool ok = true;
    int sx0 = 0;                                   // S_X tiles consumed in earlier units
    int units = 0;
    for (int band = 0; ok; ++band) {
    const int k = unit_at(band);
    if (k >= p.num_units) break;
    const Unit u = unit_info(k);
    const int qrow = u.qblk * kRowsPerCta + x * kBM + row;
    const int n_kv = x ? u.nB : u.nA;
    const int diag = 2 * u.qblk + x;               // causal: the tile holding key == row
    const int qpos = u.pos0 + qrow;                // paged: position of this row's token
    const int qpos_first = u.pos0 + u.qblk * kRowsPerCta + x * kBM;
    const int zq = u.zq;
    float m = 0.f;                                 // stabiliser in use (exp2 domain)
    float l = 0.f;                                 // denominator relative to m (fp32 terms)
    float lr = 0.f;                                // same, bf16-rounded terms

    for (int j = 0; j < n_kv; ++j) {
      if (!mbar_wait_warp(smem_addr(&bar->s_full[x]), static_cast<uint32_t>(sx0 + j) & 1u, wc)) {
        ok = false;
        break;
      }
      tc_fence_after();
      uint32_t r0[32], r1[32], r2[32], r3[32];
      ATTN47_TMEM_LD32(tl + colS + 0, r0);
      ATTN47_TMEM_LD32(tl + colS + 32, r1);
      ATTN47_TMEM_LD32(tl + colS + 64, r2);
      ATTN47_TMEM_LD32(tl + colS + 96, r3);
      ATTN47_TMEM_LD_WAIT(r0);
      ATTN47_TMEM_LD_WAIT(r1);
      ATTN47_TMEM_LD_WAIT(r2);
      ATTN47_TMEM_LD_WAIT(r3);

      float s[128];
#pragma unroll
      for (int c = 0; c < 32; ++c) {
        s[c] = __uint_as_float(r0[c]);
        s[32 + c] = __uint_as_float(r1[c]);
        s[64 + c] = __uint_as_float(r2[c]);
        s[96 + c] = __uint_as_float(r3[c]);
      }
      const int kbase = j * kBN;
      const bool need_mask = PAGED ? (kbase + kBN - 1 > qpos_first)
                                   : CAUSAL ? (j == diag) : (kbase + kBN > p.N);
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < 128; ++c) {
          const int key = kbase + c;
          const bool masked = PAGED ? (key > qpos) : CAUSAL ? (key > qrow) : (key >= p.N);
          s[c] = masked ? -INFINITY : s[c];
        }
      }
      // Row maximum: a depth-5 tree of three-input maxima.
      auto row_max = [&]() {
        float t[43], u[15];
#pragma unroll
        for (int i = 0; i < 42; ++i) t[i] = fmax3(s[3 * i], s[3 * i + 1], s[3 * i + 2]);
        t[42] = fmaxf(s[126], s[127]);
#pragma unroll
        for (int i = 0; i < 14; ++i) u[i] = fmax3(t[3 * i], t[3 * i + 1], t[3 * i + 2]);
        u[14] = t[42];
        return fmaxf(fmax3(fmax3(u[0], u[1], u[2]), fmax3(u[3], u[4], u[5]), fmax3(u[6], u[7], u[8])),
                     fmax3(fmax3(u[9], u[10], u[11]), u[12], fmaxf(u[13], u[14])));
      };
      // Numerators p = 2^(s * scale * log2 e - m), two lanes per instruction
      // for the scale and the sums.  Two denominators: `lr` sums the
      // bf16-rounded numerators that P V uses, so O / lr weights every value
      // row by exactly the factor it got (with SUMV the tensor core forms
      // this sum in column d of O_X and the loop leaves it out); `l` sums the
      // fp32 numerators and gives the LSE.  P_X goes over the first 64
      // columns of S_X (keys 2c, 2c+1 in column c), the first half while the
      // second is computed.
      float lt, lrt;                               // this tile's two sums
      auto numerators = [&]() {
        const uint64_t sc2 = f2_pack(sl2, sl2);
        const uint64_t nm2 = f2_pack(-m, -m);
        uint64_t accE[4] = {0, 0, 0, 0};
        float accR[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const int e = half * 64 + 2 * c;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(s[e], s[e + 1]), sc2, nm2), x0, x1);
            const float p0 = ex2(x0), p1 = ex2(x1);
            const uint32_t w = pack_bf16x2(p0, p1);
            accE[c & 3] = f2_add(accE[c & 3], f2_pack(p0, p1));
            if constexpr (!SUMV) {
              accR[(c & 1) * 2] = add_bf16lo_f32(w, accR[(c & 1) * 2]);
              accR[(c & 1) * 2 + 1] = add_bf16hi_f32(w, accR[(c & 1) * 2 + 1]);
            }
            pk[c] = w;
          }
          ATTN47_TMEM_ST32(tl + colS + half * 32, pk);
        }
        float e0, e1;
        f2_unpack(f2_add(f2_add(accE[0], accE[1]), f2_add(accE[2], accE[3])), e0, e1);
        lt = e0 + e1;
        lrt = (accR[0] + accR[1]) + (accR[2] + accR[3]);
      };
      // Moves the stabiliser to the tile's maximum where that exceeds it by
      // more than kTau, rescaling the sums and O_X (which holds PV_X(0..j-1),
      // complete since S_X(j) completed after it).
      auto restabilise = [&](float mt) {
        const bool need = mt > m + kTau;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mt : m;
          const float alpha = ex2(m - m_new);
          l *= alpha;
          lr *= alpha;
          m = m_new;
          const uint64_t a2 = f2_pack(alpha, alpha);
#pragma unroll 1
          for (int c0 = 0; c0 < (SUMV ? D + 32 : D); c0 += 32) {   // SUMV: the row sums too
            uint32_t o[32];
            ATTN47_TMEM_LD32(tl + colO + c0, o);
            ATTN47_TMEM_LD_WAIT(o);
#pragma unroll
            for (int c = 0; c < 16; ++c) {
              float lo, hi;
              f2_unpack(f2_mul(f2_pack(__uint_as_float(o[2 * c]), __uint_as_float(o[2 * c + 1])), a2),
                        lo, hi);
              o[2 * c] = __float_as_uint(lo);
              o[2 * c + 1] = __float_as_uint(hi);
            }
            ATTN47_TMEM_ST32(tl + colO + c0, o);
          }
        }
      };
      // The stabiliser only has to keep the numerators finite (fp32 and
      // bf16 reach 2^127), so after the first tile the tile's maximum is not
      // formed up front: the numerators are computed with the current m, and
      // only a tile whose fp32 sum exceeds 2^100 (or is not finite) is redone
      // with the stabiliser moved to its maximum.  Same function, same
      // rounding.  One call site, so the unrolled loop is emitted once.
#pragma unroll 1
      for (int pass = 0; pass < 2; ++pass) {
        if (j == 0 || pass == 1) {                 // the tile's maximum is needed
          const float mt = row_max() * sl2;
          if (j == 0)
            m = (mt == -INFINITY) ? 0.f : mt;
          else
            restabilise(mt);
        }
        numerators();
        if (j == 0 || pass == 1) break;
        const bool big = !(lt <= 0x1p100f);
        if (!__any_sync(0xffffffffu, big)) break;
      }
      l += lt;
      lr += lrt;
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->p_full[x]));
    }

    // ------------------------------------------------------------ epilogue
    ok = __all_sync(0xffffffffu, ok);
    if (ok && mbar_wait_warp(smem_addr(&bar->o_done[x]), static_cast<uint32_t>(units & 1), wc)) {
      tc_fence_after();
      float lsum = lr;
      if constexpr (SUMV) {
        uint32_t rs[32];
        ATTN47_TMEM_LD32(tl + colO + D, rs);
        ATTN47_TMEM_LD_WAIT(rs);
        lsum = __uint_as_float(rs[0]);
      }
      const float inv_l = 1.f / lsum;
      const bool in_range = qrow < p.N;
      __nv_bfloat16* orow =
          reinterpret_cast<__nv_bfloat16*>(p.o) + (static_cast<size_t>(zq) * p.N + qrow) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {
        uint32_t o[32];
        ATTN47_TMEM_LD32(tl + colO + c0, o);
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
      // O_X has been read out: the next unit's first P V may overwrite it.
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(smem_addr(&bar->o_free[x]));
    } else {
      ok = false;
    }
    sx0 += n_kv;
    ++units;
    }
    tc_fence_before();
    named_barrier_sync(1, kThreads);
  }
}

template <int D, bool CAUSAL, bool PAGED, bool SORTED = false>
cudaError_t launch_t(const FwdLaunch& a) {
  using L = FwdLayout<D, D == 64 && !PAGED>;
  auto kern = attn_fwd_sm103_kernel<D, CAUSAL, PAGED, SORTED>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kSmem);
  if (e != cudaSuccess) return e;
  FwdParams p;
  p.o = a.o;
  p.lse = a.lse;
  p.N = a.N;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.num_q_blocks = (a.N + kRowsPerCta - 1) / kRowsPerCta;
  p.bh_total = a.B * a.Hq;
  p.num_units = p.num_q_blocks * p.bh_total;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  p.k_cache = static_cast<const uint8_t*>(a.k_cache);
  p.v_cache = static_cast<const uint8_t*>(a.v_cache);
  p.block_table = a.block_table;
  p.ctx_lens = a.ctx_lens;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.max_ctx = PAGED ? a.max_blocks * kPageRows - a.N : 0;
  // Persistent: one CTA per SM (shared memory allows one), each walking units.
  const unsigned grid = static_cast<unsigned>(min(p.num_units, a.sms > 0 ? a.sms : 1));
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = L::kSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *a.tq, *a.tk, *a.tv, p);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int fwd_box_rows() { return kBM; }

cudaError_t launch_fwd_sm103(const FwdLaunch& a) {
  if (a.paged) {
    const long long pairs = static_cast<long long>(a.B) * ((a.N + kRowsPerCta - 1) / kRowsPerCta);
    if (a.B <= kSortMaxSeqs && pairs <= kSortMaxPairs)
      return a.d == 128 ? launch_t<128, true, true, true>(a) : launch_t<64, true, true, true>(a);
    return a.d == 128 ? launch_t<128, true, true, false>(a) : launch_t<64, true, true, false>(a);
  }
  if (a.d == 128) return a.causal ? launch_t<128, true, false>(a) : launch_t<128, false, false>(a);
  return a.causal ? launch_t<64, true, false>(a) : launch_t<64, false, false>(a);
}

}  // namespace attn47
