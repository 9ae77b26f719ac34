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
//   warp 7      producer: plans the chunk from seq_lens; translates table
//               entries a batch of 32 blocks ahead; per segment bulk-copies
//               the G query rows; per block TMA-copies the (block, head) K
//               and V slices (16 x d bf16, 128-byte swizzle; one copy each)
//               into a ring of 21 stages (14 when G > 8), with an
//               evict-first L2 policy (every cached byte is read once)
//   warps 0..6  consumers: block c of the chunk goes to warp c % 7, which
//               moves its K and V fragments to registers and hands the stage
//               back before computing; scores and P V are 16x8x16 warp MMAs
//               (rows = the G query heads, zero-padded to 16); at the
//               segment's end the seven warp states are merged in shared
//               memory
// A segment that covers a whole (sequence, KV head) run writes O and LSE
// directly; the others publish an unnormalised partial (O, max, sum) and count their
// arrival on the run's counter; the part that arrives last merges all parts
// of the run (exactly, with their maxima) and writes O and LSE.
//
// The kernel is launched as a programmatic dependent of the work before it
// in the stream: its CTAs start while that work drains and wait for it
// (griddepcontrol.wait) before touching anything it may write.  With the
// early plan on, the wait comes after the split plan and the first table
// translations, which then read seq_lens and the block table before the
// preceding kernel has finished; at level 2 the producer also issues the
// K/V copies of the ring's first fill before the wait, leaving out each
// sequence's last block (where a decode step appends its newest token).
#include <cuda_runtime.h>

#include "decode_sm103.h"
#include "ptx.cuh"

namespace attn47 {
namespace {

constexpr int kBS = 16;          // block_size (token slots per physical block)
// Eight warps: seven consumers and one producer, two warps per SM
// sub-partition (so each may hold up to 255 registers).
constexpr int kConsumers = 7;
constexpr int kThreads = (kConsumers + 1) * 32;
// Block c of a CTA's chunk goes to stage c % kStages and consumer warp
// c % 7 (kStages a multiple of 7), so each stage is only ever read by one
// warp, in the order it is filled (the parity of a stage's barrier can then
// never be mistaken for a later fill).
template <int GM>
constexpr int stages_for() { return GM <= 8 ? 21 : 14; }
constexpr int kMaxStages = 21;
// Block counts of the first kSeqCache sequences, kept in shared memory by the
// plan so that the walks over the chunk read no global memory.
constexpr int kSeqCache = 1024;
// Lazy stabiliser: a row's running maximum (log2 units) only moves when a
// block's maximum exceeds it by more than this, so most blocks skip the
// rescale of O; numerators then lie in [0, 2^kTau].
constexpr float kTau = 8.f;
constexpr int kQSlots = 8;
constexpr int kMinChunk = 2 * kMinSplitBlocks;   // block-heads per CTA, lower bound
// A CTA pays about this many blocks' worth of time for a (sequence, KV
// head) run (query rows, the merge of the warp states, the output write or
// the publication and merge of a split run's parts, and the warps' uneven
// finish at the run's end), so work is split by cost = blocks + kRunCost per
// run, not by blocks alone.  Measured (back-to-back calls on GB300, us per
// call on 64 sequences of U[128, 4096] / 8 of 16384 / 256 of U[32, 1024]
// tokens): 8: 31.5 / 32.6 / 37.4; 15: 29.6 / 32.7 / 35.8; 25: 29.3 / 32.8 /
// 34.2; 40: 29.8 / 32.1 / 34.1.
constexpr int kRunCost = 25;
constexpr float kLn2 = 0.6931471805599453f;

// Shared-memory layout for head dim D and groups of at most GM query heads
// per KV head (8 or 16).
template <int D, int GM>
struct DecLayout {
  static constexpr int kStages = stages_for<GM>();
  static constexpr int kBox = kBS * 128;          // one 64-column box of a block: 2 KB
  static constexpr int kHalf = kBS * D * 2;       // K (or V) slice of one (block, head)
  static constexpr int kStage = 2 * kHalf;
  static constexpr int kRing = kStages * kStage;
  static constexpr int kQSlot = GM * D * 2;       // the query heads of one (b, g)
  static constexpr int kOffQ = kRing;
  static constexpr int kOffComb = kOffQ + kQSlots * kQSlot;
  // Merge buffer of a segment's end: every warp's O rows, then every warp's
  // (max, sum) per row.
  static constexpr int kComb = kConsumers * GM * (D + 2) * 4;
  static constexpr int kOffCache = kOffComb + kComb;
  static constexpr int kOffShared = kOffCache + kSeqCache * 4;
  static constexpr int kSmem = kOffShared + 1024 + 1024;    // + alignment slack
  static_assert(kStages % kConsumers == 0, "a stage must map to one consumer warp");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};

struct DecShared {
  uint64_t full[kMaxStages];
  uint64_t empty[kMaxStages];
  uint64_t qfull[kQSlots];
  uint64_t qempty[kQSlots];
  int phys[kMaxStages];
  int fills[kMaxStages];        // fills issued per stage (for the final drain)
  int qfills[kQSlots];          // fills issued per query slot
  uint64_t comb_free;           // merge buffer free again (its segment merged)
  int comb_cnt;                 // warps that wrote their state into the buffer
  int c0, c1, chunk, b0, off0;
  int cost0;                    // first cost unit of this CTA (chunk is in cost units)
  int pseq0;                    // cost position of the first sequence's first run
  int abort;
};
static_assert(sizeof(DecShared) <= 1024, "shared control block");

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
  unsigned long long* arrive;      // arrival counter per (sequence, KV head): tag << 32 | parts arrived
  int num_seqs, Hq, Hkv, group, max_blocks, num_blocks, max_parts;
  unsigned int epoch;              // this call's tag (never 0)
  int early_plan;                  // 1: plan before waiting for the preceding kernel;
                                   // 2: also stream the ring's first fill before it
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
__device__ __forceinline__ int seq_blocks(const DecParams& p, const int* cache, int b) {
  return b < kSeqCache ? cache[b] : seq_blocks(p, b);
}

// Deterministic walk over the segments of one CTA's chunk; the producer and
// the consumers each run their own copy.
struct SegWalk {
  int b, g, blk, nblk, remaining, flat;
  int pcost;   // cost position where the current run starts (its start cost first)
  const int* cache;
  __device__ void start(const DecParams& p, const int* nb_cache, int b0, int off0, int c0, int c1,
                        int pseq) {
    cache = nb_cache;
    b = b0;
    nblk = seq_blocks(p, cache, b0);
    g = off0 / nblk;
    blk = off0 % nblk;
    remaining = c1 - c0;
    flat = c0;
    pcost = pseq + g * (nblk + kRunCost);
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
    pcost += nblk + kRunCost;      // runs follow each other in cost order
    if (++g == p.Hkv) {
      g = 0;
      do {
        ++b;
        nblk = (remaining > 0 && b < p.num_seqs) ? seq_blocks(p, cache, b) : 1;
      } while (remaining > 0 && nblk == 0);
    }
  }
};

// Arrival of one part of a split run on the run's counter (one lane).  The
// counter holds this call's tag in its high half and the parts arrived in
// its low half; a value with another tag (a previous call, or workspace
// contents never written by this library) counts as zero arrivals.  Returns
// whether this was the last part; the last part resets the counter to zero
// for the next call (a replayed graph reuses its tag).  The first guess of
// the counter's value is what the usual order of arrivals gives: part 0 is
// the last segment of its CTA and arrives after the others.
__device__ __forceinline__ bool arrive_part(const DecParams& p, unsigned long long* slot, int part,
                                            int nparts) {
  const unsigned long long tag = static_cast<unsigned long long>(p.epoch) << 32;
  unsigned long long cur = part == 0 ? tag | static_cast<unsigned int>(nparts - 1) : 0ull;
  for (int i = 0; i < 2 * nparts + 2; ++i) {
    const unsigned long long base = (cur >> 32) == p.epoch ? cur : tag;
    const unsigned long long next = base + 1;
    const unsigned long long prev = atomicCAS(slot, cur, next);
    if (prev == cur) {
      const bool last = static_cast<int>(next & 0xffffffffu) >= nparts;
      if (last) atomicExch(slot, 0ull);
      return last;
    }
    cur = prev;
  }
  atomicOr(p.status, kDevTimeout);   // more arrivals than parts: cannot happen
  return false;
}

// Exact merge of the published parts [s0, s1) of the G query heads
// hq0 .. hq0+G-1 by one warp: with M = max_s m_s, O = sum_s 2^(m_s - M) O_s
// / sum_s 2^(m_s - M) l_s and LSE = (M + log2 of the denominator) ln 2.
// Rows go in groups of 8 and parts two at a time (every load of a pass
// issued before any is used) with a running maximum.  Lane l owns columns
// [l D/32, (l + 1) D/32) of every row; lane j < 16 holds the (max, sum) of
// part s + j % 2 of row j / 2 of the group.  Every part is read back from
// the workspace, so the result does not depend on which part merges.
template <int D>
__device__ __forceinline__ void merge_published_parts(const DecParams& p, size_t hq0, int G, int s0, int s1,
                                                      int lane) {
  constexpr int E = D / 32;
  constexpr int RG = 8, CH = 2;
  const size_t mp = static_cast<size_t>(p.max_parts);
  for (int g0 = 0; g0 < G; g0 += RG) {
    const int rows = min(RG, G - g0);
    const size_t h0 = hq0 + g0;
    const int jr = min(lane / CH, rows - 1);
    const int jt = lane % CH;
    const bool jrow = lane / CH < rows;
    float Mrun = -INFINITY, Lrun = 0.f;
    float acc[RG][E];
#pragma unroll
    for (int r = 0; r < RG; ++r)
#pragma unroll
      for (int e = 0; e < E; ++e) acc[r][e] = 0.f;
    for (int s = s0; s < s1; s += CH) {
      float2 ml = make_float2(-INFINITY, 0.f);
      if (jrow && s + jt < s1)
        ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + (h0 + jr) * mp + s + jt);
      float v[CH][RG][E];
#pragma unroll
      for (int t = 0; t < CH; ++t)
#pragma unroll
        for (int r = 0; r < RG; ++r) {
          const size_t slot = (h0 + min(r, rows - 1)) * mp + min(s + t, s1 - 1);
          const float* src = p.ws_o + slot * D + lane * E;
          if constexpr (E == 4) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src));
            v[t][r][0] = x.x;
            v[t][r][1] = x.y;
            v[t][r][2] = x.z;
            v[t][r][3] = x.w;
          } else {
            const float2 x = __ldcg(reinterpret_cast<const float2*>(src));
            v[t][r][0] = x.x;
            v[t][r][1] = x.y;
          }
        }
      const float cm = fmaxf(ml.x, __shfl_xor_sync(0xffffffffu, ml.x, 1));
      const float Mn = fmaxf(Mrun, cm);
      const float a = Mn == -INFINITY ? 1.f : ex2(Mrun - Mn);
      const float w = ml.x == -INFINITY ? 0.f : ex2(ml.x - Mn);
      float lw = w * ml.y;
      lw += __shfl_xor_sync(0xffffffffu, lw, 1);
      Lrun = Lrun * a + lw;
      Mrun = Mn;
#pragma unroll
      for (int r = 0; r < RG; ++r) {
        const float ar = __shfl_sync(0xffffffffu, a, r * CH);
        const float w0 = __shfl_sync(0xffffffffu, w, r * CH);
        const float w1 = __shfl_sync(0xffffffffu, w, r * CH + 1);
#pragma unroll
        for (int e = 0; e < E; ++e) acc[r][e] = acc[r][e] * ar + w0 * v[0][r][e] + w1 * v[1][r][e];
      }
    }
#pragma unroll
    for (int r = 0; r < RG; ++r) {
      if (r >= rows) break;
      const float L = __shfl_sync(0xffffffffu, Lrun, r * CH);
      const float M = __shfl_sync(0xffffffffu, Mrun, r * CH);
      const float inv = L > 0.f ? 1.f / L : 0.f;
      const size_t hq = h0 + r;
      if constexpr (E == 4) {
        uint2 pk;
        pk.x = pack_bf16x2(acc[r][0] * inv, acc[r][1] * inv);
        pk.y = pack_bf16x2(acc[r][2] * inv, acc[r][3] * inv);
        *reinterpret_cast<uint2*>(p.o + hq * D + lane * E) = pk;
      } else {
        *reinterpret_cast<uint32_t*>(p.o + hq * D + lane * E) = pack_bf16x2(acc[r][0] * inv, acc[r][1] * inv);
      }
      if (lane == 0 && p.lse != nullptr) p.lse[hq] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
    }
  }
}

// Parts of the (sequence, KV head) run whose blocks at cost positions
// pcost + kRunCost .. pcost + kRunCost + nblk - 1 are split over the CTAs
// (CTA x holds [x chunk, (x + 1) chunk)): their count, and this CTA's index.
struct RunParts {
  int nparts, part;
  __device__ RunParts(int pcost, int nblk, int chunk) {
    const int first_cta = (pcost + kRunCost) / chunk;
    nparts = (pcost + kRunCost + nblk - 1) / chunk - first_cta + 1;
    part = static_cast<int>(blockIdx.x) - first_cta;
  }
};

// O = 0 and LSE = -inf for the empty sequences b = blockIdx.x, + gridDim.x,
// ... (one warp).
template <int D>
__device__ __forceinline__ void write_empty_sequences(const DecParams& p, const int* nb_cache, int lane) {
  for (int b = blockIdx.x; b < p.num_seqs; b += gridDim.x) {
    if (seq_blocks(p, nb_cache, b) != 0) continue;
    __nv_bfloat16* dst = p.o + static_cast<size_t>(b) * p.Hq * D;
    for (int i = lane; i < p.Hq * D / 2; i += 32) reinterpret_cast<uint32_t*>(dst)[i] = 0u;
    for (int h = lane; h < p.Hq; h += 32)
      if (p.lse != nullptr) p.lse[static_cast<size_t>(b) * p.Hq + h] = -INFINITY;
  }
}

// Merge of one segment by one warp: the seven consumer warps' states of the
// segment (rows < G of the merge buffer) combined into O and the LSE when the
// segment is a whole run, else into this CTA's partial of the run, published
// and counted; the last part of the run to arrive merges all of its parts.
// Lane l owns columns [l D/32, (l + 1) D/32).
template <int D, int GM>
__device__ __forceinline__ void merge_segment(const DecParams& p, const float* cbo, const float* cbm,
                                              const SegWalk& w, int chunk, int G, int lane) {
  constexpr int E = D / 32;
  const RunParts rp(w.pcost, w.nblk, chunk);
  const int nparts = rp.nparts, part = rp.part;
  const bool whole = nparts == 1;
  const bool in_range = part >= 0 && part < nparts && nparts <= p.max_parts;
  const size_t hq0 = static_cast<size_t>(w.b) * p.Hq + w.g * G;
#pragma unroll
  for (int r = 0; r < GM; ++r) {
    if (r >= G) break;
    // Every lane reads the (max, sum) pairs of the row (shared-memory
    // broadcasts) and forms the weights itself: no cross-lane chains, and
    // the rows are independent of each other.
    float mw[kConsumers], M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kConsumers; ++ww) {
      mw[ww] = cbm[(ww * GM + r) * 2];
      M = fmaxf(M, mw[ww]);
    }
    float acc[E], lsum = 0.f;
#pragma unroll
    for (int e = 0; e < E; ++e) acc[e] = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int ww = 0; ww < kConsumers; ++ww) {
        const float wt = ex2(mw[ww] - M);
        lsum += wt * cbm[(ww * GM + r) * 2 + 1];
        const float* src = cbo + (ww * GM + r) * D + lane * E;
        if constexpr (E == 4) {
          const float4 v = *reinterpret_cast<const float4*>(src);
          acc[0] += wt * v.x;
          acc[1] += wt * v.y;
          acc[2] += wt * v.z;
          acc[3] += wt * v.w;
        } else {
          const float2 v = *reinterpret_cast<const float2*>(src);
          acc[0] += wt * v.x;
          acc[1] += wt * v.y;
        }
      }
    }
    const size_t hq = hq0 + r;
    if (whole) {
      const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
      if constexpr (E == 4) {
        uint2 pk;
        pk.x = pack_bf16x2(acc[0] * inv, acc[1] * inv);
        pk.y = pack_bf16x2(acc[2] * inv, acc[3] * inv);
        *reinterpret_cast<uint2*>(p.o + hq * D + lane * E) = pk;
      } else {
        *reinterpret_cast<uint32_t*>(p.o + hq * D + lane * E) = pack_bf16x2(acc[0] * inv, acc[1] * inv);
      }
      if (lane == 0 && p.lse != nullptr) p.lse[hq] = lsum > 0.f ? (M + __log2f(lsum)) * kLn2 : -INFINITY;
    } else if (in_range) {
      const size_t slot = hq * p.max_parts + part;
      if constexpr (E == 4)
        *reinterpret_cast<float4*>(p.ws_o + slot * D + lane * E) = make_float4(acc[0], acc[1], acc[2], acc[3]);
      else
        *reinterpret_cast<float2*>(p.ws_o + slot * D + lane * E) = make_float2(acc[0], acc[1]);
      if (lane == 0) {
        p.ws_ml[slot * 2 + 0] = M;
        p.ws_ml[slot * 2 + 1] = lsum;
      }
    }
  }
  if (whole) return;
  if (!in_range) {
    if (lane == 0) atomicOr(p.status, kDevTimeout);   // cannot happen: the split bounds nparts
    return;
  }
  unsigned long long* slot = p.arrive + static_cast<size_t>(w.b) * p.Hkv + w.g;
  // Publish this part (every lane's writes visible to the whole GPU before
  // the arrival is counted), then count it.
  __threadfence();
  __syncwarp();
  int last = 0;
  if (lane == 0) last = arrive_part(p, slot, part, nparts);
  last = __shfl_sync(0xffffffffu, last, 0);
  if (last) {
    __threadfence();
    merge_published_parts<D>(p, hq0, G, 0, nparts, lane);
  }
}

template <int D, int GM>
__global__ void __launch_bounds__(kThreads, 1)
    attn_decode_paged_kernel(const __grid_constant__ CUtensorMap tk,
                             const __grid_constant__ CUtensorMap tv, const DecParams p) {
  using Lt = DecLayout<D, GM>;
  constexpr int kStages = Lt::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_align1024(smem_raw);
  DecShared* sh = reinterpret_cast<DecShared*>(smem + Lt::kOffShared);
  const uint32_t ring = smem_addr(smem);
  const uint32_t qring = smem_addr(smem + Lt::kOffQ);
  float* comb = reinterpret_cast<float*>(smem + Lt::kOffComb);   // [warps][GM][D], then [warps][GM][2]
  int* nb_cache = reinterpret_cast<int*>(smem + Lt::kOffCache);   // [kSeqCache] blocks per sequence

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int G = p.group;

  // ------------------------------------------------------------------ plan
  // Work: the block-heads of every (sequence, KV head) run, T in all; each
  // run also costs kRunCost to start.  With C = T + kRunCost x (runs), this
  // CTA takes the cost units [cost0, cost0 + chunk), chunk = max(kMinChunk,
  // ceil(C / grid)), and with them the blocks [c0, c1) in flat order: the
  // start cost of a run sits just before its block 0.
  if (warp == kConsumers && lane == 0) {
    prefetch_tmap(&tk);
    prefetch_tmap(&tv);
    // Bring this CTA's share of the block table and of the queries into L2
    // while the plan reads the sequence lengths (16-byte aligned interior).
    auto prefetch_share = [&](const void* base, size_t bytes) {
      const uintptr_t lo = (reinterpret_cast<uintptr_t>(base) + 15) & ~static_cast<uintptr_t>(15);
      const uintptr_t hi = (reinterpret_cast<uintptr_t>(base) + bytes) & ~static_cast<uintptr_t>(15);
      if (hi <= lo) return;
      const size_t share = (((hi - lo) / gridDim.x) + 16) & ~static_cast<size_t>(15);
      const uintptr_t a = lo + share * blockIdx.x;
      if (a >= hi) return;
      const size_t n = min(share, static_cast<size_t>(hi - a));
      bulk_prefetch_l2(reinterpret_cast<const void*>(a), static_cast<uint32_t>(n));
    };
    prefetch_share(p.block_table, static_cast<size_t>(p.num_seqs) * p.max_blocks * 4);
    prefetch_share(p.q, static_cast<size_t>(p.num_seqs) * p.Hq * D * 2);
  }
  // Without the early plan nothing is read before the preceding kernel has
  // finished (the L2 prefetches above are hints only).
  if (!p.early_plan) pdl_wait_primary();
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
        if (b < kSeqCache && b < p.num_seqs) nb_cache[b] = blocks;
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
    __syncwarp();                                // the cache entries of every lane
    const int grid = static_cast<int>(gridDim.x);
    const int chunk = max(kMinChunk, (C + grid - 1) / grid);
    const int cost0 = static_cast<int>(blockIdx.x) * chunk;
    const int cost1 = min(C, cost0 + chunk);
    // Flat block position (and sequence, offset in it) of a cost position.
    auto locate = [&](int cost, int& flat, int& bq, int& off, int& pseq) {
      flat = T;
      bq = -1;
      off = 0;
      pseq = 0;
      if (cost >= C) return;
      int P = 0, F = 0;
      for (int base = 0; base < p.num_seqs && bq < 0; base += 32) {
        const int b = base + lane;
        const int blocks = (b < p.num_seqs) ? seq_blocks(p, nb_cache, b) : 0;
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
          pseq = P + __shfl_sync(0xffffffffu, excl, src);
          const int rel = cost - pseq;
          const int g = rel / (nblk + kRunCost);
          const int blk = max(0, rel % (nblk + kRunCost) - kRunCost);
          off = g * nblk + blk;
          flat = F + __shfl_sync(0xffffffffu, fincl - blocks * p.Hkv, src) + off;
        }
        P += __shfl_sync(0xffffffffu, incl, 31);
        F += __shfl_sync(0xffffffffu, fincl, 31);
      }
    };
    int c0, b0, off0, c1, b1, off1, pseq0, pseq1;
    locate(cost0, c0, b0, off0, pseq0);
    locate(cost1, c1, b1, off1, pseq1);
    if (lane == 0) {
      sh->c0 = c0;
      sh->c1 = c1;
      sh->chunk = chunk;
      sh->b0 = (c0 < c1) ? b0 : -1;
      sh->off0 = off0;
      sh->cost0 = cost0;
      sh->pseq0 = pseq0;
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
      sh->qfills[s] = 0;
    }
    for (int s = 0; s < kMaxStages; ++s) sh->fills[s] = 0;
    mbar_init(smem_addr(&sh->comb_free), 1);
    sh->comb_cnt = 0;

    sh->abort = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int c0 = sh->c0, c1 = sh->c1, chunk = sh->chunk, b0 = sh->b0, off0 = sh->off0;
  const int pseq0 = sh->pseq0;
  if (c0 >= c1 || b0 < 0) {                       // whole CTA: no work
    if (warp == kConsumers) {
      pdl_wait_primary();
      write_empty_sequences<D>(p, nb_cache, lane);
    }
    return;
  }
  const WaitCtl wc{&sh->abort, p.status, p.timeout_ns};

  if (warp == kConsumers) {
    // ------------------------------------------------------------ producer
    // The chunk is issued in batches of 32 blocks, lane j owning block j of
    // the batch: its table entry is translated two batches ahead into its
    // registers, and the batch goes out in four rounds of 8 lanes, each lane
    // waiting for its own stage and issuing its own copies, so the per-block
    // cost of the loop is shared by 8 blocks.  A lane whose block starts a
    // segment first copies that segment's query rows into slot (segment % 8);
    // with 8 slots, the wait for a slot only ever depends on blocks issued in
    // earlier rounds.
    const int nblocks = c1 - c0;
    SegWalk lw;
    lw.start(p, nb_cache, b0, off0, c0, c1, pseq0);
    lw.skip(p, lane);
    auto fetch = [&](int k, int& ph, int& bb, int& gg) {
      ph = -1;
      bb = -1;
      gg = 0;
      if (k < nblocks && lw.remaining > 0) {
        bb = lw.b;
        gg = lw.g;
        // The entry is checked where it is used, so this load stays in
        // flight while the walk moves on.
        ph = p.block_table[static_cast<size_t>(lw.b) * p.max_blocks + lw.blk];
      }
      lw.skip(p, 32);
    };
    int cur_ph, cur_b, cur_g, n1_ph, n1_b, n1_g, n2_ph, n2_b, n2_g;
    // Whether this lane's block of the first batch is the last block of its
    // sequence (the one that holds the newest token).
    const bool cur_last = lane < nblocks && lw.remaining > 0 && lw.blk == lw.nblk - 1;
    fetch(lane, cur_ph, cur_b, cur_g);
    fetch(32 + lane, n1_ph, n1_b, n1_g);
    fetch(64 + lane, n2_ph, n2_b, n2_g);
    // Every cached K/V byte is read once: keep it from evicting the
    // published parts and arrival counters that other CTAs read back.
    const uint64_t stream_policy = l2_policy_evict_first();
    // Early stream: the ring's first fill (blocks 0 .. kStages-1 of the
    // chunk, whose stages have never been used) is issued before the wait,
    // except a sequence's last block and table entries outside the pool,
    // which the loop below issues (or reports) after it.  Only K and V are
    // read here; the query rows of the segments that start in these blocks
    // are loaded after the wait.
    unsigned pre = 0;
    if (p.early_plan == 2) {
      const bool early = lane < kStages && lane < nblocks && !cur_last && cur_ph >= 0 && cur_ph < p.num_blocks;
      if (early) {
        const uint32_t fb = smem_addr(&sh->full[lane]);
        const int rowk = (cur_ph * p.Hkv + cur_g) * kBS;
        const uint32_t dst = ring + lane * Lt::kStage;
        sh->phys[lane] = cur_ph;
        sh->fills[lane] = 1;
        mbar_arrive_expect_tx(fb, Lt::kStage);
        tma_load_3d_hint(dst, &tk, fb, 0, rowk, 0, stream_policy);
        tma_load_3d_hint(dst + Lt::kHalf, &tv, fb, 0, rowk, 0, stream_policy);
      }
      pre = __ballot_sync(0xffffffffu, early);
    }
    // Everything from here on may read what the preceding kernel wrote (the
    // queries, the newest cache slots) or write what it reads.
    pdl_wait_primary();
    int seg = 0, carry_b = -1, carry_g = -1;
    bool ok = true;
    const uint32_t qbytes = static_cast<uint32_t>(G) * D * 2;
    for (int base = 0; base < nblocks && ok; base += 32) {
      const int cblk = base + lane;
      const bool valid = cblk < nblocks;
      // Segment starts: (b, g) differs from the previous block's.
      int prev_b = __shfl_up_sync(0xffffffffu, cur_b, 1);
      int prev_g = __shfl_up_sync(0xffffffffu, cur_g, 1);
      if (lane == 0) {
        prev_b = carry_b;
        prev_g = carry_g;
      }
      const bool start = valid && (cur_b != prev_b || cur_g != prev_g);
      const unsigned smask = __ballot_sync(0xffffffffu, start);
      const int sego = seg + __popc(smask & ((1u << lane) - 1u));
      seg += __popc(smask);
      carry_b = __shfl_sync(0xffffffffu, cur_b, 31);
      carry_g = __shfl_sync(0xffffffffu, cur_g, 31);
      const int st = cblk % kStages;
      const int fill = cblk / kStages;
#pragma unroll 1
      for (int r = 0; r < 4; ++r) {
        bool okl = true;
        if (valid && (lane >> 3) == r) {
          if (start) {
            const int qs = sego % kQSlots;
            okl = mbar_wait(smem_addr(&sh->qempty[qs]), ((sego / kQSlots) & 1) ^ 1, wc);
            if (okl) {
              const uint32_t qb = smem_addr(&sh->qfull[qs]);
              mbar_arrive_expect_tx(qb, qbytes);
              bulk_load(qring + qs * Lt::kQSlot,
                        p.q + (static_cast<size_t>(cur_b) * p.Hq + cur_g * G) * D, qbytes, qb);
              sh->qfills[qs] = sego / kQSlots + 1;
            }
          }
          const bool issued = base == 0 && ((pre >> lane) & 1u);   // by the early stream
          if (okl && !issued) okl = mbar_wait(smem_addr(&sh->empty[st]), (fill & 1) ^ 1, wc);
          if (okl && !issued) {
            if (cur_ph < 0 || cur_ph >= p.num_blocks) {
              atomicOr(p.status, kDevBadBlock);    // outside the pool: that block is skipped
              cur_ph = -1;
            }
            const uint32_t fb = smem_addr(&sh->full[st]);
            sh->phys[st] = cur_ph;
            sh->fills[st] = fill + 1;
            if (cur_ph >= 0) {
              const int rowk = (cur_ph * p.Hkv + cur_g) * kBS;
              const uint32_t dst = ring + st * Lt::kStage;
              mbar_arrive_expect_tx(fb, Lt::kStage);
              tma_load_3d_hint(dst, &tk, fb, 0, rowk, 0, stream_policy);
              tma_load_3d_hint(dst + Lt::kHalf, &tv, fb, 0, rowk, 0, stream_policy);
            } else {
              mbar_arrive(fb);
            }
          }
        }
        if (!__all_sync(0xffffffffu, okl)) {
          ok = false;
          break;
        }
      }
      cur_ph = n1_ph;
      cur_b = n1_b;
      cur_g = n1_g;
      n1_ph = n2_ph;
      n1_b = n2_b;
      n1_g = n2_g;
      fetch(base + 96 + lane, n2_ph, n2_b, n2_g);
    }
    __syncwarp();
    // Every copy is issued: the next kernel in the stream may launch its
    // CTAs (it waits for this grid to finish before using its results).
    pdl_launch_dependents();
    // Every copy issued must have landed before the CTA may exit: wait for
    // the last fill of every stage and query slot.
    if (lane < kStages) {
      const int fills = sh->fills[lane];
      if (fills > 0) mbar_wait(smem_addr(&sh->full[lane]), (fills - 1) & 1, wc, true);
    }
    if (lane < kQSlots) {
      const int fills = sh->qfills[lane];
      if (fills > 0) mbar_wait(smem_addr(&sh->qfull[lane]), (fills - 1) & 1, wc, true);
    }
    write_empty_sequences<D>(p, nb_cache, lane);
  } else {
    // ----------------------------------------------------------- consumers
    pdl_wait_primary();
    const float sl2 = p.scale_log2;
    const int r0 = lane >> 2;               // fragment row (query head within the group)
    const int cq = (lane & 3) * 2;          // fragment column pair
    SegWalk w;
    w.start(p, nb_cache, b0, off0, c0, c1, pseq0);
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

      for (int i = ((warp - base_blk) % kConsumers + kConsumers) % kConsumers; i < cnt && !fail;
           i += kConsumers) {
        const int gi = base_blk + i;            // block counter of the whole chunk
        const int st = gi % kStages;
        if (!mbar_wait_warp(smem_addr(&sh->full[st]), (gi / kStages) & 1, wc)) { fail = true; break; }
        const int ph = sh->phys[st];
        const int nvalid = min(kBS, L - (w.blk + i) * kBS);
        // K and V fragments of this block go to registers first, so the
        // stage is handed back to the producer before any arithmetic.
        uint32_t kf[2][D / 32][4];      // B operand of S = Q K^T: [key tile][d step]
        uint32_t vf[D / 16][4];         // B operand of O += P V (transposed load)
        if (ph >= 0) {
          const uint32_t sK = ring + st * Lt::kStage;
          const uint32_t sV = sK + Lt::kHalf;
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            const int key = nt * 8 + (lane & 7);
#pragma unroll
            for (int kk2 = 0; kk2 < D / 32; ++kk2) {
              const int c = 4 * kk2 + (lane >> 3);
              ldsm_x4(sK + (c >> 3) * Lt::kBox + key * 128 + (((c & 7) ^ (key & 7)) << 4), kf[nt][kk2]);
            }
          }
          const int vkey = (lane & 7) + ((lane >> 3) & 1) * 8;
#pragma unroll
          for (int dt2 = 0; dt2 < D / 16; ++dt2) {
            const int c = 2 * dt2 + (lane >> 4);
            ldsm_x4_trans(sV + (c >> 3) * Lt::kBox + vkey * 128 + (((c & 7) ^ (vkey & 7)) << 4), vf[dt2]);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_addr(&sh->empty[st]));
        if (ph >= 0) {
          if (nvalid < kBS) {
            // Slots past the sequence end may hold anything (even NaN): zero
            // their V values so that P = 0 cannot meet NaN in the MMA.  This
            // lane's halves hold keys 2(lane%4) + {0,1} (registers 0, 2) and
            // 8 + 2(lane%4) + {0,1} (registers 1, 3).
            const int k0 = 2 * (lane & 3);
            const uint32_t m_lo = (k0 < nvalid ? 0x0000ffffu : 0u) | (k0 + 1 < nvalid ? 0xffff0000u : 0u);
            const uint32_t m_hi = (k0 + 8 < nvalid ? 0x0000ffffu : 0u) | (k0 + 9 < nvalid ? 0xffff0000u : 0u);
#pragma unroll
            for (int dt2 = 0; dt2 < D / 16; ++dt2) {
              vf[dt2][0] &= m_lo;
              vf[dt2][2] &= m_lo;
              vf[dt2][1] &= m_hi;
              vf[dt2][3] &= m_hi;
            }
          }
          // S = Q K^T: two 8-key column tiles, each over two independent
          // accumulator chains (even and odd 16-wide d steps).
          float sc[2][4], sd[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
#pragma unroll
            for (int e = 0; e < 4; ++e) sc[nt][e] = sd[nt][e] = 0.f;
#pragma unroll
            for (int kk2 = 0; kk2 < D / 32; ++kk2) {
              mma_16816(sc[nt], qa[2 * kk2], kf[nt][kk2][0], kf[nt][kk2][1]);
              mma_16816(sd[nt], qa[2 * kk2 + 1], kf[nt][kk2][2], kf[nt][kk2][3]);
            }
          }
          // Mask slots past the end; lazy running max, sums.
          float x[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const int kl = nt * 8 + cq + (e & 1);
              x[nt][e] = (kl < nvalid) ? (sc[nt][e] + sd[nt][e]) * sl2 : -INFINITY;
            }
          float mx0 = fmaxf(fmaxf(x[0][0], x[0][1]), fmaxf(x[1][0], x[1][1]));
          float mx1 = fmaxf(fmaxf(x[0][2], x[0][3]), fmaxf(x[1][2], x[1][3]));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
          // The stabiliser moves only when the block's maximum exceeds it by
          // more than kTau (always on the first block: m = -inf); slot 0 of
          // every block is valid, so the maxima are finite.
          const bool up0 = mx0 > m0 + kTau, up1 = mx1 > m1 + kTau;
          if (__any_sync(0xffffffffu, up0 || up1)) {
            const float mn0 = up0 ? mx0 : m0, mn1 = up1 ? mx1 : m1;
            const float a0 = ex2(m0 - mn0), a1 = ex2(m1 - mn1);
            l0 *= a0;
            l1 *= a1;
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int dt = 0; dt < D / 8; ++dt) {
              oacc[dt][0] *= a0;
              oacc[dt][1] *= a0;
              oacc[dt][2] *= a1;
              oacc[dt][3] *= a1;
            }
          }
          float pr[2][4];
#pragma unroll
          for (int nt = 0; nt < 2; ++nt) {
            pr[nt][0] = ex2(x[nt][0] - m0);
            pr[nt][1] = ex2(x[nt][1] - m0);
            pr[nt][2] = ex2(x[nt][2] - m1);
            pr[nt][3] = ex2(x[nt][3] - m1);
          }
          l0 += (pr[0][0] + pr[0][1]) + (pr[1][0] + pr[1][1]);
          l1 += (pr[0][2] + pr[0][3]) + (pr[1][2] + pr[1][3]);
          // The score accumulator layout is the A-operand layout of P.
          uint32_t pa[4];
          pa[0] = pack_bf16x2(pr[0][0], pr[0][1]);
          pa[1] = pack_bf16x2(pr[0][2], pr[0][3]);
          pa[2] = pack_bf16x2(pr[1][0], pr[1][1]);
          pa[3] = pack_bf16x2(pr[1][2], pr[1][3]);
#pragma unroll
          for (int dt2 = 0; dt2 < D / 16; ++dt2) {
            mma_16816(oacc[2 * dt2], pa, vf[dt2][0], vf[dt2][1]);
            mma_16816(oacc[2 * dt2 + 1], pa, vf[dt2][2], vf[dt2][3]);
          }
        }
      }
      l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
      l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
      l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
      if (fail) break;
      // ------------------------ hand the warp state to the segment's merge
      // Every warp writes its state into the merge buffer and goes on with
      // the next segment; the last of the seven to arrive merges them, so
      // no warp waits for the others at a segment's end.  The buffer is
      // reused by the next segment once that merge is done.
      if (!mbar_wait_warp(smem_addr(&sh->comb_free), (seg & 1) ^ 1, wc)) break;
      float* cml = comb + kConsumers * GM * D;          // [warps][GM][2]
#pragma unroll
      for (int dt = 0; dt < D / 8; ++dt) {
        const int d = dt * 8 + cq;
        *reinterpret_cast<float2*>(&comb[(warp * GM + r0) * D + d]) = make_float2(oacc[dt][0], oacc[dt][1]);
        if (r0 + 8 < GM)
          *reinterpret_cast<float2*>(&comb[(warp * GM + r0 + 8) * D + d]) = make_float2(oacc[dt][2], oacc[dt][3]);
      }
      if ((lane & 3) == 0) {
        cml[(warp * GM + r0) * 2 + 0] = m0;
        cml[(warp * GM + r0) * 2 + 1] = l0;
        if (r0 + 8 < GM) {
          cml[(warp * GM + r0 + 8) * 2 + 0] = m1;
          cml[(warp * GM + r0 + 8) * 2 + 1] = l1;
        }
      }
      __threadfence_block();
      __syncwarp();
      int arrived = 0;
      if (lane == 0) arrived = atomicAdd(&sh->comb_cnt, 1);
      arrived = __shfl_sync(0xffffffffu, arrived, 0);
      if (arrived == kConsumers - 1) {
        __threadfence_block();
        merge_segment<D, GM>(p, comb, cml, w, chunk, G, lane);
        if (lane == 0) {
          sh->comb_cnt = 0;
          mbar_arrive(smem_addr(&sh->qempty[qs]));
          mbar_arrive(smem_addr(&sh->comb_free));
        }
      }
      base_blk += cnt;
      w.advance(p, cnt);
      ++seg;
    }
  }
  __syncthreads();
}

template <int D, int GM>
cudaError_t launch_t(const DecLaunch& a) {
  using Lt = DecLayout<D, GM>;
  auto kern = attn_decode_paged_kernel<D, GM>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, Lt::kSmem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kThreads, Lt::kSmem);
  if (e != cudaSuccess) return e;
  per_sm = per_sm < 1 ? 1 : per_sm;
  const int max_parts = decode_max_parts(a.max_blocks);
  float* ws_o = a.workspace;
  float* ws_ml = ws_o + static_cast<size_t>(a.num_seqs) * a.Hq * max_parts * D;
  auto* arrive = reinterpret_cast<unsigned long long*>(ws_ml + static_cast<size_t>(a.num_seqs) * a.Hq * max_parts * 2);
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
  p.arrive = arrive;
  p.num_seqs = a.num_seqs;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.group = a.Hq / a.Hkv;
  p.max_blocks = a.max_blocks;
  p.num_blocks = a.num_blocks;
  p.max_parts = max_parts;
  p.epoch = a.epoch;
  p.early_plan = a.early_plan < 0 ? 0 : a.early_plan > 2 ? 2 : a.early_plan;
  p.scale_log2 = a.scale * 1.4426950408889634f;
  p.status = a.status;
  p.timeout_ns = a.timeout_ns;
  // One wave: every CTA resident at once, each with an equal chunk.
  int ctas = a.sms * per_sm;
  if (a.max_ctas > 0 && ctas > a.max_ctas) ctas = a.max_ctas;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(ctas));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Lt::kSmem;
  cfg.stream = a.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *a.tk, *a.tv, p);
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
  // Partial O (d floats), max and sum per (sequence, query head, part), then
  // the arrival counter of every (sequence, KV head) (8 bytes per sequence
  // and query head are reserved for these).
  const size_t parts = static_cast<size_t>(num_seqs) * Hq * decode_max_parts(max_blocks_per_seq);
  return parts * (static_cast<size_t>(d) + 2) * sizeof(float) +
         static_cast<size_t>(num_seqs) * Hq * sizeof(unsigned long long);
}

cudaError_t launch_decode_sm103(const DecLaunch& a) {
  const bool small_group = a.Hq / a.Hkv <= 8;
  if (a.d == 128) return small_group ? launch_t<128, 8>(a) : launch_t<128, 16>(a);
  return small_group ? launch_t<64, 8>(a) : launch_t<64, 16>(a);
}

}  // namespace attn47
