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
// Work split: the (sequence b, KV head g, logical block) triples are laid out
// in one flat order and every CTA of a one-wave grid takes an equal
// contiguous chunk of it, so each SM streams the same number of cache bytes
// whatever the length mix.  The chunk is walked as segments (maximal runs of
// one (b, g)); the G = Hq/Hkv query heads sharing KV head g are processed
// together so each K/V block is read from HBM once.
//   warp 4      producer: plans the chunk from seq_lens; translates table
//               entries a batch of 32 blocks ahead; per segment bulk-copies
//               the G query rows; per
//               block TMA-copies the (block, head) K and V slices (16 x d
//               bf16, 128-byte swizzle) into an 8-stage ring
//   warps 0..3  consumers: block c of the chunk goes to warp c % 4; scores
//               and P V are 16x8x16 warp MMAs (rows = the G query heads,
//               zero-padded to 16); at the segment's end the four warp states
//               are merged in shared memory
// A segment that covers a whole sequence writes O and LSE directly; the
// others write an unnormalised partial (O, max, sum), and a second kernel
// (launched as a programmatic dependent) merges the parts of each sequence.
#include <cuda_runtime.h>

#include "decode_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kBS = 16;          // block_size (token slots per physical block)
constexpr int kConsumers = 4;    // consumer warps
constexpr int kThreads = (kConsumers + 1) * 32;
// Block c of a CTA's chunk goes to stage c % 8 and consumer warp c % 4, so
// each stage is only ever read by one warp, in the order it is filled (the
// parity of a stage's barrier can then never be mistaken for a later fill).
constexpr int kStages = 8;
constexpr int kQSlots = 2;
constexpr int kMinChunk = 2 * kMinSplitBlocks;   // block-heads per CTA, lower bound
// A CTA pays about this many blocks' worth of time to start a (sequence,
// KV head) run (query load, state merge, output write), so work is split by
// cost = blocks + kRunCost per run, not by blocks alone.
constexpr int kRunCost = 3;
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct DecLayout {
  static constexpr int kChunks = D / 64;
  static constexpr int kBox = kBS * 128;          // one 64-column box of a block: 2 KB
  static constexpr int kHalf = kBS * D * 2;       // K (or V) slice of one (block, head)
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kRing = kStages * kStage;
  static constexpr int kQSlot = 16 * D * 2;       // up to 16 query heads of one (b, g)
  static constexpr int kOffQ = kRing;
  static constexpr int kOffComb = kOffQ + kQSlots * kQSlot;
  static constexpr int kComb = kConsumers * 16 * (D + 2) * 4;
  static constexpr int kOffShared = kOffComb + kComb;
  static constexpr int kSmem = kOffShared + 256 + 1024;     // + alignment slack
};

struct DecShared {
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t qfull[kQSlots];
  uint64_t qempty[kQSlots];
  int phys[kStages];
  int c0, c1, chunk, b0, off0;
  int cost0;                    // first cost unit of this CTA (chunk is in cost units)
  int abort;
};
static_assert(sizeof(DecShared) <= 256, "shared control block");
static_assert(kStages % kConsumers == 0, "a stage must map to one consumer warp");

struct DecParams {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int* block_table;
  const int* seq_lens;
  __nv_bfloat16* o;
  float* lse;
  float* ws_o;
  float* ws_ml;
  int* nparts;
  int num_seqs, Hq, Hkv, group, max_blocks, num_blocks, max_parts;
  float scale_log2;
  unsigned int* status;
  unsigned long long timeout_ns;
};

__device__ __forceinline__ int seq_len(const DecParams& p, int b) {
  const int L = p.seq_lens[b];
  return L < 0 ? 0 : min(L, p.max_blocks * kBS);
}
__device__ __forceinline__ int seq_blocks(const DecParams& p, int b) {
  return (seq_len(p, b) + kBS - 1) / kBS;
}

// Deterministic walk over the segments of one CTA's chunk; the producer and
// the consumers each run their own copy.
struct SegWalk {
  int b, g, blk, nblk, remaining, flat;
  __device__ void start(const DecParams& p, int b0, int off0, int c0, int c1) {
    b = b0;
    nblk = seq_blocks(p, b0);
    g = off0 / nblk;
    blk = off0 % nblk;
    remaining = c1 - c0;
    flat = c0;
  }
  // Current segment: blocks [blk, blk + count()) of (b, g).
  __device__ int count() const { return min(remaining, nblk - blk); }
  // Move k blocks forward (possibly across segments).
  __device__ void skip(const DecParams& p, int k) {
    while (k > 0 && remaining > 0) {
      const int c = count();
      if (k < c) {
        blk += k;
        remaining -= k;
        flat += k;
        k = 0;
      } else {
        advance(p, c);
        k -= c;
      }
    }
  }
  __device__ void advance(const DecParams& p, int cnt) {
    remaining -= cnt;
    flat += cnt;
    blk = 0;
    if (++g == p.Hkv) {
      g = 0;
      do {
        ++b;
        nblk = (remaining > 0 && b < p.num_seqs) ? seq_blocks(p, b) : 1;
      } while (remaining > 0 && nblk == 0);
    }
  }
};

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
  const uint32_t qring = smem_addr(smem + Lt::kOffQ);
  float* comb = reinterpret_cast<float*>(smem + Lt::kOffComb);   // [4][16][D]
  float* cml = comb + kConsumers * 16 * D;                          // [4][16][2]

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  // ------------------------------------------------------------------ plan
  // Work: the block-heads of every (sequence, KV head) run, T in all; each
  // run also costs kRunCost to start.  With C = T + kRunCost x (runs), this
  // CTA takes the cost units [cost0, cost0 + chunk), chunk = max(kMinChunk,
  // ceil(C / grid)), and with them the blocks [c0, c1) in flat order: the
  // start cost of a run sits just before its block 0.
  if (warp == kConsumers) {
    int T = 0, C = 0;
    bool bad = false;
    for (int base = 0; base < p.num_seqs; base += 128) {
      int nb[4], nc[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {              // four independent loads in flight
        const int b = base + 32 * u + lane;
        const int L = b < p.num_seqs ? p.seq_lens[b] : 0;
        bad |= (L < 0 || L > p.max_blocks * kBS);
        const int Lc = L < 0 ? 0 : min(L, p.max_blocks * kBS);
        const int blocks = (Lc + kBS - 1) / kBS;
        nb[u] = blocks * p.Hkv;
        nc[u] = blocks > 0 ? (blocks + kRunCost) * p.Hkv : 0;
      }
      int sum = (nb[0] + nb[1]) + (nb[2] + nb[3]);
      int csum = (nc[0] + nc[1]) + (nc[2] + nc[3]);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        csum += __shfl_xor_sync(0xffffffffu, csum, o);
      }
      T += sum;
      C += csum;
    }
    if (__any_sync(0xffffffffu, bad) && lane == 0 && blockIdx.x == 0)
      atomicOr(p.status, kDevBadSeqLen);
    const int grid = static_cast<int>(gridDim.x);
    const int chunk = max(kMinChunk, (C + grid - 1) / grid);
    const int cost0 = static_cast<int>(blockIdx.x) * chunk;
    const int cost1 = min(C, cost0 + chunk);
    // Flat block position (and sequence, offset in it) of a cost position.
    auto locate = [&](int cost, int& flat, int& bq, int& off) {
      flat = T;
      bq = -1;
      off = 0;
      if (cost >= C) return;
      int P = 0, F = 0;
      for (int base = 0; base < p.num_seqs && bq < 0; base += 32) {
        const int b = base + lane;
        const int blocks = (b < p.num_seqs) ? seq_blocks(p, b) : 0;
        const int nc = blocks > 0 ? (blocks + kRunCost) * p.Hkv : 0;
        int incl = nc, fincl = blocks * p.Hkv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int y = __shfl_up_sync(0xffffffffu, incl, o);
          const int fy = __shfl_up_sync(0xffffffffu, fincl, o);
          if (lane >= o) {
            incl += y;
            fincl += fy;
          }
        }
        const int excl = incl - nc;
        const bool here = nc > 0 && P + excl <= cost && cost < P + incl;
        const unsigned hit = __ballot_sync(0xffffffffu, here);
        if (hit) {
          const int src = __ffs(hit) - 1;
          bq = base + src;
          const int nblk = __shfl_sync(0xffffffffu, blocks, src);
          const int rel = cost - P - __shfl_sync(0xffffffffu, excl, src);
          const int g = rel / (nblk + kRunCost);
          const int blk = max(0, rel % (nblk + kRunCost) - kRunCost);
          off = g * nblk + blk;
          flat = F + __shfl_sync(0xffffffffu, fincl - blocks * p.Hkv, src) + off;
        }
        P += __shfl_sync(0xffffffffu, incl, 31);
        F += __shfl_sync(0xffffffffu, fincl, 31);
      }
    };
    int c0, b0, off0, c1, b1, off1;
    locate(cost0, c0, b0, off0);
    locate(cost1, c1, b1, off1);
    if (lane == 0) {
      sh->c0 = c0;
      sh->c1 = c1;
      sh->chunk = chunk;
      sh->b0 = (c0 < c1) ? b0 : -1;
      sh->off0 = off0;
      sh->cost0 = cost0;
    }
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(smem_addr(&sh->full[s]), 1);
      mbar_init(smem_addr(&sh->empty[s]), 1);
    }
    for (int s = 0; s < kQSlots; ++s) {
      mbar_init(smem_addr(&sh->qfull[s]), 1);
      mbar_init(smem_addr(&sh->qempty[s]), 1);
    }
    sh->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  // Let the merge kernel launch; it waits for this grid before reading.
  pdl_launch_dependents();
  const int c0 = sh->c0, c1 = sh->c1, chunk = sh->chunk, b0 = sh->b0, off0 = sh->off0;
  const int cost0 = sh->cost0;
  if (c0 >= c1 || b0 < 0) return;                 // whole CTA: no work
  const WaitCtl wc{&sh->abort, p.status, p.timeout_ns};

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // Lane j handles chunk blocks j, 32 + j, 64 + j, ...: it translates the
    // table entry up to a batch of 32 blocks before the block is copied, so
    // no table lookup sits between two copies.
    const int nblocks = c1 - c0;
    SegWalk lw;
    lw.start(p, b0, off0, c0, c1);
    lw.skip(p, lane);
    auto fetch = [&](int k, int& ph, int& bb, int& gg) {
      ph = -1;
      bb = -1;
      gg = 0;
      if (k < nblocks && lw.remaining > 0) {
        bb = lw.b;
        gg = lw.g;
        ph = p.block_table[static_cast<size_t>(lw.b) * p.max_blocks + lw.blk];
        if (ph < 0 || ph >= p.num_blocks) {
          atomicOr(p.status, kDevBadBlock);
          ph = -1;
        }
      }
    };
    // The first batch is translated before the loop; each next one a few
    // copies into the current batch, so the first copy leaves at once.
    int cur_ph, cur_b, cur_g, nxt_ph = -1, nxt_b = -1, nxt_g = 0;
    fetch(lane, cur_ph, cur_b, cur_g);

    int issued = 0, seg = 0, pb = -1, pg = -1;
    bool ok = true;
    const uint32_t qbytes = static_cast<uint32_t>(G) * D * 2;
    for (int c = 0; c < nblocks && ok; ++c) {
      const int j = c & 31;
      if (j == 0 && c > 0) {
        cur_ph = nxt_ph;
        cur_b = nxt_b;
        cur_g = nxt_g;
      }
      if (j == 4) {
        lw.skip(p, 32);
        fetch(c - 4 + 32 + lane, nxt_ph, nxt_b, nxt_g);
      }
      const int phys = __shfl_sync(0xffffffffu, cur_ph, j);
      const int b = __shfl_sync(0xffffffffu, cur_b, j);
      const int g = __shfl_sync(0xffffffffu, cur_g, j);
      if (lane == 0) {
        if (b != pb || g != pg) {
          // First block of a segment: its query rows.
          const int qs = seg % kQSlots;
          ok = mbar_wait(smem_addr(&sh->qempty[qs]), ((seg / kQSlots) & 1) ^ 1, wc);
          if (ok) {
            const uint32_t qb = smem_addr(&sh->qfull[qs]);
            mbar_arrive_expect_tx(qb, qbytes);
            bulk_load(qring + qs * Lt::kQSlot, p.q + (static_cast<size_t>(b) * p.Hq + g * G) * D,
                      qbytes, qb);
          }
          ++seg;
          pb = b;
          pg = g;
        }
        const int st = issued % kStages;
        if (ok) ok = mbar_wait(smem_addr(&sh->empty[st]), ((issued / kStages) & 1) ^ 1, wc);
        if (ok) {
          const uint32_t fb = smem_addr(&sh->full[st]);
          sh->phys[st] = phys;
          if (phys >= 0) {
            const int rowk = (phys * p.Hkv + g) * kBS;
            const uint32_t dst = ring + st * Lt::kStage;
            mbar_arrive_expect_tx(fb, Lt::kStage);
#pragma unroll
            for (int cc = 0; cc < Lt::kChunks; ++cc) {
              tma_load_2d(dst + cc * Lt::kBox, &tk, fb, cc * 64, rowk);
              tma_load_2d(dst + Lt::kHalf + cc * Lt::kBox, &tv, fb, cc * 64, rowk);
            }
          } else {
            mbar_arrive(fb);
          }
          ++issued;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    issued = __shfl_sync(0xffffffffu, issued, 0);
    seg = __shfl_sync(0xffffffffu, seg, 0);
    // Every copy issued must have landed before the CTA may exit.
    if (lane == 0) {
      for (int st = 0; st < kStages && st < issued; ++st) {
        const int fills = (issued - 1 - st) / kStages + 1;
        mbar_wait(smem_addr(&sh->full[st]), (fills - 1) & 1, wc, true);
      }
      for (int qs = 0; qs < kQSlots && qs < seg; ++qs) {
        const int fills = (seg - 1 - qs) / kQSlots + 1;
        mbar_wait(smem_addr(&sh->qfull[qs]), (fills - 1) & 1, wc, true);
      }
    }
  } else {
    // ----------------------------------------------------------- consumers
    const float sl2 = p.scale_log2;
    const int r0 = lane >> 2;               // fragment row (query head within the group)
    const int cq = (lane & 3) * 2;          // fragment column pair
    SegWalk w;
    w.start(p, b0, off0, c0, c1);
    int base_blk = 0, seg = 0;
    while (w.remaining > 0) {
      const int cnt = w.count();
      const int L = seq_len(p, w.b);
      const int qs = seg % kQSlots;
      bool fail = !mbar_wait_warp(smem_addr(&sh->qfull[qs]), (seg / kQSlots) & 1, wc);
      uint32_t qa[D / 16][4];
      {
        const uint32_t qsm = qring + qs * Lt::kQSlot;
        const bool v0 = r0 < G, v1 = r0 + 8 < G;
#pragma unroll
        for (int ks = 0; ks < D / 16; ++ks) {
          const int c = ks * 16 + cq;
          uint32_t a0 = 0, a1 = 0, a2 = 0, a3 = 0;
          if (!fail) {
            if (v0) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a0) : "r"(qsm + (r0 * D + c) * 2));
            if (v1) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a1) : "r"(qsm + ((r0 + 8) * D + c) * 2));
            if (v0) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a2) : "r"(qsm + (r0 * D + c + 8) * 2));
            if (v1) asm volatile("ld.shared.b32 %0, [%1];" : "=r"(a3) : "r"(qsm + ((r0 + 8) * D + c + 8) * 2));
          }
          qa[ks][0] = a0;
          qa[ks][1] = a1;
          qa[ks][2] = a2;
          qa[ks][3] = a3;
        }
      }
      float m0 = -INFINITY, m1 = -INFINITY;   // running max (exp2 domain), rows r and r+8
      float l0 = 0.f, l1 = 0.f;               // running sums (this lane's columns only)
      float oacc[D / 8][4];
#pragma unroll
      for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

      for (int i = (warp - base_blk) & (kConsumers - 1); i < cnt && !fail; i += kConsumers) {
        const int gi = base_blk + i;            // block counter of the whole chunk
        const int st = gi % kStages;
        if (!mbar_wait_warp(smem_addr(&sh->full[st]), (gi / kStages) & 1, wc)) { fail = true; break; }
        const int ph = sh->phys[st];
        const int nvalid = min(kBS, L - (w.blk + i) * kBS);
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
      // ---------------------------------- merge the four warp states
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        const int d = dt * 8 + cq;
        *reinterpret_cast<float2*>(&comb[(warp * 16 + r0) * D + d]) =
            make_float2(oacc[dt][0], oacc[dt][1]);
        *reinterpret_cast<float2*>(&comb[(warp * 16 + r0 + 8) * D + d]) =
            make_float2(oacc[dt][2], oacc[dt][3]);
      }
      if ((lane & 3) == 0) {
        cml[(warp * 16 + r0) * 2 + 0] = m0;
        cml[(warp * 16 + r0) * 2 + 1] = l0;
        cml[(warp * 16 + r0 + 8) * 2 + 0] = m1;
        cml[(warp * 16 + r0 + 8) * 2 + 1] = l1;
      }
      // All consumers stop together if any of them failed or the CTA aborted.
      if (named_barrier_or(1, kConsumers * 32, fail || *wc.abort)) break;
      if (threadIdx.x == 0) mbar_arrive(smem_addr(&sh->qempty[qs]));
      const bool last = (w.blk + cnt == w.nblk);
      const bool whole = (w.blk == 0) && last;
      // Part index = this CTA - the CTA holding block 0 of the run.  Only the
      // first segment can continue a run: its block 0 sits at cost position
      // cost0 - w.blk, in CTA (cost0 - w.blk) / chunk.
      const int part = (w.blk > 0) ? static_cast<int>(blockIdx.x) - (cost0 - w.blk) / chunk : 0;
      for (int idx = threadIdx.x; idx < G * D; idx += kConsumers * 32) {
        const int r = idx / D;
        const int d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int ww = 0; ww < kConsumers; ++ww) M = fmaxf(M, cml[(ww * 16 + r) * 2]);
        float acc = 0.f, lsum = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int ww = 0; ww < kConsumers; ++ww) {
            const float wt = ex2(cml[(ww * 16 + r) * 2] - M);
            acc += wt * comb[(ww * 16 + r) * D + d];
            lsum += wt * cml[(ww * 16 + r) * 2 + 1];
          }
        }
        const size_t hq = static_cast<size_t>(w.b) * p.Hq + w.g * G + r;
        if (whole) {
          p.o[hq * D + d] = __float2bfloat16_rn(lsum > 0.f ? acc / lsum : 0.f);
          if (d == 0 && p.lse != nullptr)
            p.lse[hq] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : -INFINITY;
        } else {
          const size_t slot = hq * p.max_parts + part;
          p.ws_o[slot * D + d] = acc;
          if (d == 0) {
            p.ws_ml[slot * 2 + 0] = M;
            p.ws_ml[slot * 2 + 1] = lsum;
          }
        }
      }
      if (last && threadIdx.x == 0) p.nparts[w.b * p.Hkv + w.g] = part + 1;
      named_barrier_sync(1, kConsumers * 32);      // merge buffer free again
      base_blk += cnt;
      w.advance(p, cnt);
      ++seg;
    }
  }
  __syncthreads();
}

struct CombineParams {
  const int* seq_lens;
  const float* ws_o;
  const float* ws_ml;
  const int* nparts;
  __nv_bfloat16* o;
  float* lse;
  int Hq, Hkv, max_blocks, max_parts;
};

// One warp per (sequence, query head): exact merge of the parts of a
// sequence that was split over several CTAs.  Everything the merge can need
// is loaded at once, before any of it is used: the length, the part count,
// every part's (max, sum) (lane s holds part s) and the O rows of the first
// kPrefetch parts; the part count then selects among them (rows of parts
// that were not written are never read into the sum).  So a merge costs one
// round trip to memory; only sequences with more parts loop over the rest.
// Sequences with one part were written by the decode kernel; empty
// sequences get O = 0 and LSE = -inf here.
constexpr int kPrefetch = 8;
template <int D>
__global__ void __launch_bounds__(128) attn_decode_combine_kernel(const CombineParams p) {
  pdl_wait_primary();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.x * 4 + warp;
  const int b = blockIdx.y;
  if (h >= p.Hq) return;
  const int G = p.Hq / p.Hkv;
  const size_t base = (static_cast<size_t>(b) * p.Hq + h) * p.max_parts;
  // ---- all independent loads first
  const int L_raw = p.seq_lens[b];
  const int np_raw = __ldcg(p.nparts + b * p.Hkv + h / G);
  float m_lane = -INFINITY, l_lane = 0.f;
  if (lane < p.max_parts) {
    m_lane = __ldcg(p.ws_ml + (base + lane) * 2);
    l_lane = __ldcg(p.ws_ml + (base + lane) * 2 + 1);
  }
  float v[kPrefetch][D / 32];
#pragma unroll
  for (int s = 0; s < kPrefetch; ++s) {
    const float* src = p.ws_o + (base + min(s, p.max_parts - 1)) * D;
#pragma unroll
    for (int e = 0; e < D / 32; ++e) v[s][e] = __ldcg(src + lane + 32 * e);
  }
  // ---- then decide
  const int L = L_raw < 0 ? 0 : min(L_raw, p.max_blocks * kBS);
  __nv_bfloat16* dst = p.o + (static_cast<size_t>(b) * p.Hq + h) * D;
  if (L == 0) {
#pragma unroll
    for (int e = 0; e < D / 32; ++e) dst[lane + 32 * e] = __float2bfloat16_rn(0.f);
    if (lane == 0 && p.lse != nullptr) p.lse[static_cast<size_t>(b) * p.Hq + h] = -INFINITY;
    return;
  }
  const int np = min(np_raw, p.max_parts);
  if (np <= 1) return;
  if (lane >= np) {
    m_lane = -INFINITY;
    l_lane = 0.f;
  }
  // Parts beyond 32 (only with very long block tables) join the maximum here.
  for (int s = 32 + lane; s < np; s += 32) m_lane = fmaxf(m_lane, __ldcg(p.ws_ml + (base + s) * 2));
  float M = m_lane;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, o));
  float acc[D / 32];
#pragma unroll
  for (int e = 0; e < D / 32; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  if (M != -INFINITY) {
    // Weights of the first 32 parts from the values already in registers.
    const float w = (lane < np) ? ex2(m_lane - M) : 0.f;
    float lw = w * l_lane;
#pragma unroll
    for (int s = 0; s < kPrefetch; ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      if (s < np)
#pragma unroll
        for (int e = 0; e < D / 32; ++e) acc[e] += ws * v[s][e];
    }
    for (int s = kPrefetch; s < min(np, 32); ++s) {
      const float ws = __shfl_sync(0xffffffffu, w, s);
      const float* src = p.ws_o + (base + s) * D;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) acc[e] += ws * __ldcg(src + lane + 32 * e);
    }
    for (int s = 32; s < np; ++s) {
      const float ws = ex2(__ldcg(p.ws_ml + (base + s) * 2) - M);
      if (lane == 0) lw += ws * __ldcg(p.ws_ml + (base + s) * 2 + 1);
      const float* src = p.ws_o + (base + s) * D;
#pragma unroll
      for (int e = 0; e < D / 32; ++e) acc[e] += ws * __ldcg(src + lane + 32 * e);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) lw += __shfl_xor_sync(0xffffffffu, lw, o);
    lsum = lw;
  }
  const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
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
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Lt::kSmem);
  if (e != cudaSuccess) return e;
  per_sm = per_sm < 1 ? 1 : per_sm;
  const int max_parts = decode_max_parts(a.max_blocks);
  float* ws_o = a.workspace;
  float* ws_ml = ws_o + static_cast<size_t>(a.num_seqs) * a.Hq * max_parts * D;
  int* nparts = reinterpret_cast<int*>(ws_ml + static_cast<size_t>(a.num_seqs) * a.Hq * max_parts * 2);
  DecParams p;
  p.q = reinterpret_cast<const __nv_bfloat16*>(a.q);
  p.k_cache = reinterpret_cast<const __nv_bfloat16*>(a.k_cache);
  p.v_cache = reinterpret_cast<const __nv_bfloat16*>(a.v_cache);
  p.block_table = a.block_table;
  p.seq_lens = a.seq_lens;
  p.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  p.lse = a.lse;
  p.ws_o = ws_o;
  p.ws_ml = ws_ml;
  p.nparts = nparts;
  p.num_seqs = a.num_seqs;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.max_parts = max_parts;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  // One wave: every CTA resident at once, each with an equal chunk.
  int ctas = a.sms * per_sm;
  if (a.max_ctas > 0 && ctas > a.max_ctas) ctas = a.max_ctas;
  kern<<<static_cast<unsigned>(ctas), kThreads, Lt::kSmem, a.stream>>>(*a.tk, *a.tv, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  CombineParams c;
  c.seq_lens = a.seq_lens;
  c.ws_o = ws_o;
  c.ws_ml = ws_ml;
  c.nparts = nparts;
  c.o = reinterpret_cast<__nv_bfloat16*>(a.o);
  c.lse = a.lse;
  c.Hq = a.Hq;
  c.Hkv = a.Hkv;
  c.max_blocks = a.max_blocks;
  c.max_parts = max_parts;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((a.Hq + 3) / 4, a.num_seqs);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, attn_decode_combine_kernel<D>, c);
  return e != cudaSuccess ? e : cudaGetLastError();
}

}  // namespace

int decode_max_parts(int max_blocks_per_seq) {
  // The start cost of a run lies before its block 0, and every later chunk
  // covers at least kMinChunk of its blocks, so the n blocks of one
  // (sequence, KV head) meet at most ceil(n / kMinChunk) + 1 chunks.
  // (in 64 bits: max_blocks_per_seq may be anything up to INT_MAX here)
  return static_cast<int>((static_cast<long long>(max_blocks_per_seq) + kMinChunk - 1) / kMinChunk + 1);
}

size_t decode_workspace_bytes(int num_seqs, int Hq, int d, int max_blocks_per_seq) {
  const size_t parts = static_cast<size_t>(num_seqs) * Hq * decode_max_parts(max_blocks_per_seq);
  return parts * (static_cast<size_t>(d) + 2) * sizeof(float) +
         static_cast<size_t>(num_seqs) * Hq * sizeof(int);
}

cudaError_t launch_decode_sm103(const DecLaunch& a) {
  return a.d == 128 ? launch_t<128>(a) : launch_t<64>(a);
}

}  // namespace attn47
