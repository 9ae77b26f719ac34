/*
 * attn47.h — C-ABI of the GB300 (sm_103a) exact-attention library
 * (libattn47_sm103.so).
 *
 * Four attention operations, all bf16 in / fp32 accumulate:
 *
 *  attn_fwd           softmax(scale * Q K^T + causal mask) V for a whole
 *                     sequence (prefill), computed tile by tile with the
 *                     running-max / running-sum softmax so the N x N score
 *                     matrix never reaches global memory.  Defined by
 *                     "Advanced attention mechanisms – II" (Aryan Das),
 *                     sections "Why?" (the matmul -> mask -> softmax -> V
 *                     pipeline whose result this is), "Flash Attention"
 *                     (only the output goes back to HBM), "Tiling" steps 1-3,
 *                     "Softmax stabiliser" and "Incremental / online softmax";
 *                     and by "Fast attention kernels and operator fusion
 *                     accelerate AI models", section "FlashAttention-style
 *                     attention and Paged Attention" (blocks of Q, K, V;
 *                     softmax statistics and outputs kept on chip).
 *
 *  attn_bwd           the gradients of attn_fwd (dQ, dK, dV), recomputing the
 *                     attention matrix from the saved LSE ("Advanced
 *                     attention mechanisms – II", section "Flash Attention").
 *
 *  attn_decode_paged  one query token per sequence attending to all of its
 *                     cached keys, where the KV cache is stored in fixed-size
 *                     blocks of 16 token slots and a block table maps each
 *                     logical position to a physical block.  Defined by "Fast
 *                     attention kernels and operator fusion accelerate AI
 *                     models", section "FlashAttention-style attention and
 *                     Paged Attention" (paged cache, block table, per-position
 *                     translation; block_size = 16 in its worked example).
 *
 *  attn_prefill_paged a chunk of new tokens per sequence: their keys and
 *                     values are appended to the same paged cache, then each
 *                     new query attends causally to the cached prefix and the
 *                     new tokens up to itself (same page and section: the
 *                     cache grows as tokens arrive; the serving example runs
 *                     prefill, then decode, over block_size = 16 blocks).
 *
 * and two operator fusions of the same transformer layer (same page,
 * section "Operator fusion"):
 *
 *  fused_add_rmsnorm  residual add followed by RMSNorm, one pass
 *  fused_swiglu       SwiGLU activation silu(gate) * up of the merged
 *                     gate/up projection output, one pass
 *  swiglu_projection  the gate/up projection GEMM with SiLU * up in its
 *                     epilogue: only the [rows, F] product reaches HBM
 *
 * and the Mamba-2 SSD forward ("Accelerating Mamba-2 with high-performance
 * forward kernels in NVIDIA CUDA Tile"):
 *
 *  ssd_chunked_fwd    the state-space recurrence evaluated chunk by chunk
 *                     (per-chunk cumulative decay, fwd_pass_state, chunk
 *                     outputs)
 *
 * Conventions shared by every call
 *  - Pointers are DEVICE pointers of the current CUDA device unless stated.
 *    The caller owns every buffer and the stream; the library allocates no
 *    device memory and performs no host<->device copy.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    Calls are asynchronous on that stream.
 *  - Every argument is validated on the host before anything is launched.
 *    An unsupported shape, head size, block size or device returns an error;
 *    there is never a fallback to another implementation ("Fast attention
 *    kernels ...", same section: forcing a fixed backend fails when it does
 *    not support the inputs or the hardware, and the serving engine reports
 *    an incompatible backend at initialisation).
 *  - Only devices of compute capability 10.3 (GB300, sm_103a) are accepted.
 *  - Problems found on the device (a wait that ran out of time, a block-table
 *    entry outside the pool, a sequence length outside the table) set bits in
 *    a per-device status word instead of trapping; read and clear it with
 *    attn_get_device_status().
 *  - GQA: query head h reads KV head h / (Hq / Hkv) (contiguous groups; MQA is
 *    Hkv = 1, MHA is Hkv = Hq).
 *  - LSE is the natural logarithm of sum_j exp(scale * q . k_j) over the keys
 *    the row may see.
 */
#ifndef ATTN47_H_
#define ATTN47_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ATTN47_ABI_VERSION 2

typedef enum attn_status {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1,  /* null/misaligned pointer, negative size, bad scale, Hq % Hkv != 0 */
  ATTN_ERR_UNSUPPORTED = 2,  /* valid but not implemented: d not in {64,128}, block_size != 16,
                                Hq/Hkv > 16 (decode) */
  ATTN_ERR_DEVICE = 3,       /* no CUDA device, or not compute capability 10.3 */
  ATTN_ERR_LAUNCH = 4,       /* the CUDA runtime rejected the launch; see attn_last_error() */
  ATTN_ERR_WORKSPACE = 5     /* workspace smaller than attn_decode_paged_workspace_size() */
} attn_status_t;

/* Bits of the device status word (attn_get_device_status). */
#define ATTN_DEV_TIMEOUT 0x1u    /* a kernel wait exceeded its time limit; outputs invalid */
#define ATTN_DEV_BAD_BLOCK 0x2u  /* a block-table entry was outside [0, num_blocks); that block
                                    was skipped */
#define ATTN_DEV_BAD_SEQLEN 0x4u /* a seq_lens entry was < 0 or > max_blocks_per_seq*block_size
                                    (decode), or a ctx_lens entry was < 0 or
                                    > max_blocks_per_seq*block_size - N (chunked prefill);
                                    it was clamped into range, outputs of that sequence invalid */

/*
 * attn_fwd — exact attention forward (prefill).
 *
 *  q    [B, Hq,  N, d] bf16, contiguous, 16-byte aligned
 *  k, v [B, Hkv, N, d] bf16, contiguous, 16-byte aligned
 *  o    [B, Hq,  N, d] bf16 (written), 16-byte aligned
 *  lse  [B, Hq,  N]    fp32 (written) or NULL to skip it
 *  causal != 0: query i sees keys j <= i (Nq = Nk = N); 0: every key.
 *  scale: multiplies q . k before the softmax (finite, > 0), e.g. 1/sqrt(d).
 *  d must be 64 or 128; Hq % Hkv == 0; B, Hq, Hkv >= 1; N >= 0.
 *  B == 0 or N == 0 is an empty problem: returns ATTN_OK, launches nothing.
 *  Writes only o and lse.  Deterministic (no atomics).
 */
attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int N, int d, int causal, float scale, void* stream);

/*
 * attn_bwd_workspace_size — bytes of device workspace attn_bwd needs: two
 * fp32 values per query row (rows padded to multiples of 128).  0 for an
 * empty problem.
 */
size_t attn_bwd_workspace_size(int B, int Hq, int N);

/*
 * attn_bwd — gradients of attn_fwd with respect to q, k and v.
 *
 * "Advanced attention mechanisms – II", section "Flash Attention": the
 * forward keeps the softmax statistics (the LSE) so that the backward pass
 * recomputes the attention matrix tile by tile instead of storing it.  With
 * s = scale * q . k over the allowed keys and P = exp(s - lse):
 *   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - rowsum(dO * O)),
 *   dQ = scale * dS K,  dK = scale * dS^T Q
 * (for GQA, dK and dV of a KV head are summed over its query heads).
 *
 *  q, k, v, o    as for attn_fwd (o = its output for the same q, k, v,
 *                causal and scale)
 *  lse           [B, Hq, N] fp32, the LSE attn_fwd wrote for them (required)
 *  dout          [B, Hq, N, d] bf16: dL/dO
 *  dq            [B, Hq, N, d] bf16 (written)
 *  dk, dv        [B, Hkv, N, d] bf16 (written)
 *  workspace     device memory of at least attn_bwd_workspace_size(B, Hq, N)
 *                bytes, 16-byte aligned, owned by the caller; its content on
 *                entry does not matter and it is scratch afterwards.
 *  Same shape rules as attn_fwd; every tensor pointer 16-byte aligned.
 *  Errors: ATTN_ERR_INVALID_ARG (sizes, null or misaligned pointers),
 *  ATTN_ERR_UNSUPPORTED (d), ATTN_ERR_WORKSPACE (workspace too small).
 *  Writes only dq, dk, dv and the workspace.  Deterministic (no atomics).
 */
attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                       int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                       void* stream);

/*
 * attn_decode_paged_workspace_size — bytes of device workspace that
 * attn_decode_paged needs for these sizes: fp32 partial results of
 * sequences whose keys are split across CTAs, and their part counts (8 bytes
 * per sequence and query head are reserved for these).  0 for an empty
 * problem.
 */
size_t attn_decode_paged_workspace_size(int num_seqs, int Hq, int d, int max_blocks_per_seq);

/*
 * attn_decode_paged — one query token per sequence over a paged KV cache.
 *
 *  q            [num_seqs, Hq, d] bf16, 16-byte aligned
 *  k_cache,
 *  v_cache      [num_blocks, Hkv, block_size, d] bf16, 16-byte aligned
 *  block_table  [num_seqs, max_blocks_per_seq] int32: logical block i of
 *               sequence b lives in physical block block_table[b][i]; entries
 *               past ceil(seq_lens[b] / block_size) are never read
 *  seq_lens     [num_seqs] int32 (device): number of cached tokens of each
 *               sequence; the query is that sequence's last token and
 *               attends to all of them.  seq_lens[b] == 0 gives o = 0 and
 *               lse = -inf for that sequence.  Slots past seq_lens[b] in the
 *               last block are never used, whatever they hold.
 *  o            [num_seqs, Hq, d] bf16 (written)
 *  lse          [num_seqs, Hq] fp32 (written) or NULL
 *  workspace    >= attn_decode_paged_workspace_size(...) bytes, 16-byte
 *               aligned; contents on entry are ignored (the per-sequence
 *               arrival counters in it carry a tag that differs on every
 *               call, and each call leaves them at zero)
 *  block_size must be 16; d must be 64 or 128; Hq % Hkv == 0 and
 *  Hq / Hkv <= 16; num_blocks * Hkv * 16 < 2^31.
 *  num_seqs == 0 is an empty problem: returns ATTN_OK, launches nothing.
 *  Launches one kernel over an even split of all cached tokens (one CTA per
 *  SM); the parts of a (sequence, KV head) split across CTAs are merged
 *  exactly by whichever part finishes last.  The kernel is launched as a
 *  programmatic dependent of the preceding work in the stream: its CTAs may
 *  start while that kernel drains and wait for it to finish before reading
 *  q or the cache and before writing anything (see
 *  attn_set_decode_early_plan for the one exception).  Calls that share a
 *  workspace must not overlap on the GPU.  The result does not depend on
 *  which part finishes last; it is deterministic for a given device and
 *  attn_set_decode_max_ctas setting.
 */
attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
                                int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
                                int num_blocks, float scale, void* o, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream);

/*
 * attn_decode_paged_noalloc — attn_decode_paged without a caller-provided
 * workspace.  (The pages describe no such call: it exists only for callers
 * of this library that cannot allocate device memory at the time they run
 * the decode — for example a plugin inside a host framework that owns all
 * device memory and forbids its extensions from calling cudaMalloc, or a
 * latency-bound serving loop that must not call cudaMalloc/cudaFree because
 * they can synchronize the whole device.)
 *
 *  Arguments, layouts, results and errors are those of attn_decode_paged,
 *  minus workspace and workspace_bytes.  Instead the library uses one fixed
 *  8 MiB array of device memory that it declares itself; it is part of the
 *  library image, so every device that loads the library holds it until the
 *  process exits.  No device memory is allocated by the call: it makes no
 *  cudaMalloc, cudaFree or other allocating call.
 *  - Limit: if attn_decode_paged_workspace_size(num_seqs, Hq, d,
 *    max_blocks_per_seq) exceeds 8 MiB the call returns ATTN_ERR_WORKSPACE
 *    and launches nothing (use attn_decode_paged for such sizes).
 *  - The first call on each device looks up the array's device address once
 *    (with that device current); make that first call before any stream
 *    capture begins.
 *  - All calls on one device share the array and it keeps the previous
 *    call's contents; nothing in it needs to start at zero.  Calls whose
 *    kernels overlap on the GPU (different streams, no ordering between
 *    them) race on the array and may produce wrong results: order them.
 */
attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int num_seqs, int Hq, int Hkv, int d, int block_size,
                                        int max_blocks_per_seq, int num_blocks, float scale,
                                        void* o, float* lse, void* stream);

/*
 * attn_prefill_paged — chunked prefill over a paged KV cache.
 *
 * "Fast attention kernels and operator fusion accelerate AI models",
 * section "FlashAttention-style attention and Paged Attention": the KV cache
 * grows token by token in fixed-size blocks, a block table maps logical
 * positions to physical blocks, and the attention kernel translates every
 * position through it.  For each sequence b, with P = ctx_lens[b] tokens
 * already cached:
 *   1. new token i (0 <= i < N) is stored at logical position P + i, i.e.
 *      slot (P + i) % 16 of physical block block_table[b][(P + i) / 16], for
 *      every KV head; the slots past P + N in the last block are set to 0;
 *   2. new query i attends to logical keys 0 .. P + i (the cached prefix and
 *      the new tokens up to itself) — softmax(scale * q . k) v over them.
 *
 *  q            [num_seqs, Hq, N, d] bf16: the new tokens' queries
 *  k_new, v_new [num_seqs, Hkv, N, d] bf16: their keys and values
 *  k_cache,
 *  v_cache      [num_blocks, Hkv, block_size, d] bf16 (read and written)
 *  block_table  [num_seqs, max_blocks_per_seq] int32 (device): must map the
 *               ceil((P + N) / 16) blocks of each sequence; blocks are owned by
 *               one sequence (two sequences writing the same block race)
 *  ctx_lens     [num_seqs] int32 (device): P of each sequence, 0 <= P <=
 *               max_blocks_per_seq * 16 - N; not modified (after the call the
 *               sequence holds P + N tokens)
 *  o            [num_seqs, Hq, N, d] bf16 (written)
 *  lse          [num_seqs, Hq, N] fp32 (written) or NULL
 *  block_size must be 16; d must be 64 or 128; Hq % Hkv == 0;
 *  N <= max_blocks_per_seq * 16.  All bf16 tensors 16-byte aligned.
 *  num_seqs == 0 or N == 0 is an empty problem: ATTN_OK, nothing launched.
 *  Launches two kernels in stream order: the append, then the attention.
 *  Table entries outside [0, num_blocks) set ATTN_DEV_BAD_BLOCK (the append
 *  skips them; the attention reads that block as zeros); invalid ctx_lens
 *  set ATTN_DEV_BAD_SEQLEN.  Deterministic (no atomics on data).
 */
attn_status_t attn_prefill_paged(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, const int32_t* block_table,
                                 const int32_t* ctx_lens, int num_seqs, int Hq, int Hkv, int N,
                                 int d, int block_size, int max_blocks_per_seq, int num_blocks,
                                 float scale, void* o, float* lse, void* stream);

/*
 * fused_add_rmsnorm — residual add + RMSNorm in one kernel.
 *
 * "Fast attention kernels and operator fusion accelerate AI models",
 * section "Operator fusion": adding the residual connection and then
 * normalising with RMSNorm is a common fusion; fused, the sum is never
 * written and re-read between two kernels.  For every row:
 *   residual <- bf16(x + residual)                       (the new residual stream)
 *   out      <- bf16(residual * rsqrt(mean(residual^2) + eps) * weight)
 * where the mean runs over the `hidden` values of the row as stored (bf16),
 * so the result is that of an unfused add kernel followed by RMSNorm.
 *
 *  x         [rows, hidden] bf16 (read)
 *  residual  [rows, hidden] bf16 (read, then overwritten in place)
 *  weight    [hidden] bf16
 *  out       [rows, hidden] bf16 (written)
 *  hidden must be a multiple of 8 (>= 8); eps finite and >= 0.  All pointers
 *  16-byte aligned; the four buffers must not overlap (ATTN_ERR_INVALID_ARG).
 *  rows == 0 is an empty problem: ATTN_OK, nothing launched.  One kernel,
 *  one warp per row; deterministic.
 */
attn_status_t fused_add_rmsnorm(const void* x, void* residual, const void* weight, void* out,
                                int rows, int hidden, float eps, void* stream);

/*
 * fused_swiglu — the SwiGLU activation in one kernel.
 *
 * "Fast attention kernels and operator fusion accelerate AI models",
 * section "Operator fusion": the SwiGLU block, run naively, launches a SiLU
 * kernel and an elementwise-product kernel between its projection matmuls,
 * each writing its intermediate to HBM; fused, the gate/up projection output
 * is read once and only the product is written:
 *   out[r, j] = bf16(silu(g) * u),  silu(g) = g / (1 + exp(-g)),
 *   g = gate_up[r, j],  u = gate_up[r, F + j].
 * (The projection matmuls themselves are plain GEMMs and not part of this
 * library.)
 *
 *  gate_up  [rows, 2F] bf16: the merged gate/up projection output, gate in
 *           columns 0..F-1, up in columns F..2F-1
 *  out      [rows, F] bf16 (written; must not overlap gate_up)
 *  F must be a multiple of 8 (>= 8); both pointers 16-byte aligned.
 *  rows == 0 is an empty problem.  One kernel; deterministic.
 */
attn_status_t fused_swiglu(const void* gate_up, void* out, int rows, int F, void* stream);

/*
 * swiglu_projection — the SwiGLU block's gate/up projection with the
 * activation fused into the matrix product.
 *
 * "Fast attention kernels and operator fusion accelerate AI models",
 * section "Operator fusion": run naively, the SwiGLU block's projection
 * matmul writes its [rows, 2F] output to HBM and a SiLU and a product kernel
 * read it back; fused, the projection's accumulators are activated and
 * multiplied where they are produced and only the product is written:
 *   out[r, f] = bf16(silu(g) * u),  silu(g) = g / (1 + exp(-g)),
 *   g = sum_k x[r, k] W[f, k],  u = sum_k x[r, k] W[F + f, k]
 * (fp32 accumulation on the tensor cores).  The down projection that
 * follows is a plain GEMM and not part of this call.
 *
 *  x          [rows, hidden] bf16 activations
 *  w_gate_up  [2F, hidden] bf16: the gate weight's F rows, then the up
 *             weight's F rows (a merged gate/up weight, rows = output
 *             features, as a linear layer stores it)
 *  out        [rows, F] bf16 (written; must not overlap the inputs)
 *  hidden must be a multiple of 64 and F of 128; all pointers 16-byte
 *  aligned.  rows == 0 is an empty problem.  One persistent kernel (one
 *  CTA per SM); deterministic.
 */
attn_status_t swiglu_projection(const void* x, const void* w_gate_up, void* out, int rows, int hidden,
                                int F, void* stream);

/*
 * ssd_workspace_size — bytes of device workspace ssd_chunked_fwd needs: the
 * per-chunk cumulative decays (fp32, batch * H * n_chunks * chunk, padded to
 * 256 bytes) and every chunk's initial state (bf16, batch * n_chunks * H *
 * 64 * N).  0 for an empty problem.
 */
size_t ssd_workspace_size(int batch, int L, int H, int N, int chunk);

/*
 * ssd_chunked_fwd — Mamba-2 SSD forward.
 *
 * "Accelerating Mamba-2 with high-performance forward kernels in NVIDIA CUDA
 * Tile": per (batch, head), with a_t = A[h] * dt[t, h] (< 0) and state
 * h_t of size P x N,
 *   h_t = exp(a_t) h_{t-1} + x_t b_t^T,   y_t = h_t c_t,
 * evaluated chunk by chunk: the page's per-chunk cumulative sum of a_t
 * (scaled by log2(e)) and fwd_pass_state, the sequential loop over chunks
 * that gives every chunk's initial state and the final state, run as one
 * kernel; the chunk outputs (C B^T weighted by exp(g_i - g_j) under the
 * causal mask, times X, plus the initial state's contribution) as a second.
 * Both do their matrix products on the tensor cores.  x enters the
 * recurrence as given (pass x * dt for Mamba-2's discretised input).
 *
 *  x        [batch, L, H, P] bf16;  dt [batch, L, H] fp32 (> 0);  A [H] fp32 (< 0)
 *  B, C     [batch, L, G, N] bf16; head h uses group h / (H / G)
 *  h0       [batch, H, P, N] fp32 initial state, or NULL for zero
 *  y        [batch, L, H, P] bf16 (written)
 *  h_final  [batch, H, P, N] fp32 (written): the state after the last token
 *  workspace >= ssd_workspace_size(batch, L, H, N, chunk) bytes, 16-byte
 *           aligned; contents on entry are ignored
 *  P must be 64; N 64 or 128; chunk 64, 128 or 256; H % G == 0.  bf16 and
 *  state pointers 16-byte aligned, dt and A 4-byte aligned.
 *  batch == 0 or L == 0 is an empty problem: ATTN_OK, nothing launched.
 *  Launches two kernels in stream order.  Deterministic.  Calls that share a
 *  workspace must not overlap.
 */
attn_status_t ssd_chunked_fwd(const void* x, const float* dt, const float* A, const void* B,
                              const void* C, const float* h0, void* y, float* h_final, int batch,
                              int L, int H, int G, int P, int N, int chunk, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * attn_get_device_status — synchronises `stream`, copies the current
 * device's status word (ATTN_DEV_* bits) to *flags_out (host pointer) and
 * clears it.  Returns ATTN_ERR_DEVICE if the device is unusable.
 */
attn_status_t attn_get_device_status(void* stream, unsigned int* flags_out);

/*
 * attn_set_wait_timeout_ns — time limit of every wait inside the kernels
 * (default 1e9 ns = 1 s); after it a kernel sets ATTN_DEV_TIMEOUT, lets its
 * in-flight copies land, releases its tensor memory and returns.  Applies to
 * later launches from this process.  Values < 1000 are raised to 1000.
 */
void attn_set_wait_timeout_ns(unsigned long long ns);

/*
 * attn_set_decode_max_ctas — upper bound on the CTAs of one decode launch;
 * 0 (the default) launches one full wave (every SM, as many CTAs as fit).
 * The cached tokens are split evenly over the CTAs; any setting gives the
 * same result up to fp32 rounding order.  Applies to later calls from this
 * process.
 */
void attn_set_decode_max_ctas(int ctas);

/*
 * attn_set_decode_early_plan — 1: later decode calls (both entry points)
 * read seq_lens and the first block-table entries of each CTA's share
 * before the kernel that precedes them in the stream has finished, so that
 * the split plan overlaps that kernel's tail; 2: as 1, and each CTA also
 * starts streaming the first cache blocks of its share (up to its ring's
 * depth, 21 blocks for up to 8 query heads per KV head, 14 above) before
 * that kernel has finished, except the last block of each sequence (the
 * block holding position seq_lens[b] - 1, where a decode step appends its
 * newest token); 0 (the default): they read nothing before it has
 * finished.  With 1 or 2 the caller guarantees that seq_lens and
 * block_table — and with 2 every cache block other than each sequence's
 * last — are not written by the kernel launched just before the decode on
 * its stream (nor, if that kernel was itself launched as a programmatic
 * dependent, by the one before it): write them with a host-to-device copy
 * or an earlier kernel.  q and each sequence's last cache block may always
 * be written by the preceding kernel.  Results are the same bits at every
 * level.  Values above 2 act as 2, below 0 as 0.  Applies to later calls
 * from this process.
 */
void attn_set_decode_early_plan(int on);

/*
 * attn_selftest_exp2_poly — y[i] = 2^x[i] by an exp2 on the FMA pipe
 * instead of the special-function unit, the building block for moving part
 * of a softmax's exponentials off that unit ("Accelerating Mamba-2 with
 * high-performance forward kernels in NVIDIA CUDA Tile" works in exp2 for
 * the same unit's sake).  On GB300 the forward softmax measured slower with
 * it (its loop is limited by instruction issue, not by that unit), so the
 * kernels do not use it; this entry keeps it tested.
 * 2^x = 2^round(x) * p(x - round(x)), p a degree-4 polynomial with relative
 * error below 2^-18 on [-1/2, 1/2].  x is clamped to [-126, 127] first
 * (below -126 the result is a tiny value under 2^-125, not 0).  For tests:
 * x and y are device arrays of n floats (4-byte aligned, may not overlap
 * except x == y); one kernel on `stream`, nothing synchronised.
 */
attn_status_t attn_selftest_exp2_poly(const float* x, float* y, int n, void* stream);

/*
 * attn_selftest_wait_timeout — launches a one-warp kernel that waits on a
 * shared-memory barrier that nothing will ever complete, with the given time
 * limit, so the bounded-wait path can be tested without hanging or faulting
 * the GPU.  Synchronises `stream`; on return *flags_out holds the status
 * word (ATTN_DEV_TIMEOUT expected), which is then cleared.
 */
attn_status_t attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream,
                                         unsigned int* flags_out);

/* Human-readable name of a status code (static string). */
const char* attn_status_string(attn_status_t s);

/* Message of the last failing call on this host thread ("" if none). */
const char* attn_last_error(void);

/* ATTN47_ABI_VERSION of the loaded library. */
int attn_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN47_H_ */
