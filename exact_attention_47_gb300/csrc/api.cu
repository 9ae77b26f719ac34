// C-ABI of the exact-attention library: host-side validation, device check,
// TMA descriptor encoding and launches.  See include/attn47.h for the
// contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>
#include <chrono>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include "attn47.h"
#include "decode_sm103.h"
#include "bwd_sm103.h"
#include "fusion_sm103.h"
#include "gemm_sm103.h"
#include "fwd_sm103.h"
#include "ssd_sm103.h"
#include "ptx.cuh"

// Per-device error word written by the kernels (ATTN_DEV_* bits).
__device__ unsigned int g_attn47_status;

// Fixed scratch of attn_decode_paged_noalloc: the partial results of
// sequences whose keys are split across CTAs.  Every device that loads the
// library holds it until the process exits; every call of that entry point
// on a device reuses it.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_attn47_noalloc_scratch[kNoAllocScratchBytes];

namespace {

thread_local char g_last_error[512] = "";

attn_status_t fail(attn_status_t s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return s;
}

unsigned long long g_timeout_ns = 1000000000ull;

int g_decode_max_ctas = 0;  // 0 = one full wave
std::atomic<int> g_decode_early_plan{0};

// Tags of the decode's per-run arrival counters: a different nonzero value
// for every call of this process, starting from a clock-derived value so
// that workspace contents left by another process are unlikely to carry it.
unsigned int next_decode_epoch() {
  static std::atomic<unsigned int> epoch{static_cast<unsigned int>(
      std::chrono::steady_clock::now().time_since_epoch().count() * 2654435761ull)};
  unsigned int e;
  do {
    e = epoch.fetch_add(1u) + 1u;
  } while (e == 0u);
  return e;
}

constexpr int kMaxDevices = 64;
struct DeviceInfo {
  int index = -1;
  bool checked = false;
  bool usable = false;
  int sms = 0;
  unsigned int* status = nullptr;
  void* noalloc_scratch = nullptr;   // device address of the fixed scratch array
};
DeviceInfo g_dev[kMaxDevices];
std::mutex g_mu;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
using AddressRangeFn = CUresult (*)(CUdeviceptr*, size_t*, CUdeviceptr);
AddressRangeFn g_address_range = nullptr;

// Current device, checked once: compute capability 10.3, status word address.
attn_status_t current_device(DeviceInfo** out) {
  int dev = -1;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess)
    return fail(ATTN_ERR_DEVICE, "no usable CUDA device: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return fail(ATTN_ERR_DEVICE, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.checked) {
    int major = 0, minor = 0, sms = 0;
    cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    d.sms = sms;
    d.index = dev;
    if (major != 10 || minor != 3) {
      d.checked = true;
      d.usable = false;
      return fail(ATTN_ERR_DEVICE, "device %d is compute capability %d.%d; this library is built "
                  "for sm_103a (10.3) only", dev, major, minor);
    }
    void* addr = nullptr;
    e = cudaGetSymbolAddress(&addr, g_attn47_status);
    if (e != cudaSuccess)
      return fail(ATTN_ERR_DEVICE, "status word unavailable: %s", cudaGetErrorString(e));
    d.status = static_cast<unsigned int*>(addr);
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
      if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr)
        return fail(ATTN_ERR_DEVICE, "driver entry point cuTensorMapEncodeTiled not found");
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    if (g_address_range == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      e = cudaGetDriverEntryPointByVersion("cuMemGetAddressRange", &fn, 12000, cudaEnableDefault, &q);
      if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn != nullptr)
        g_address_range = reinterpret_cast<AddressRangeFn>(fn);
      else
        cudaGetLastError();   // optional: without it only the memory type is checked
    }
    d.usable = true;
    d.checked = true;
  }
  if (!d.usable) return fail(ATTN_ERR_DEVICE, "device %d is not a compute capability 10.3 GPU", dev);
  *out = &d;
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool overlap(const void* a, size_t na, const void* b, size_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}
bool finite_positive(float x) { return std::isfinite(x) && x > 0.f; }

// A buffer a kernel will read or write: `bytes` from `p` (p may be NULL when
// the argument is optional).
struct Buf {
  const void* p;
  size_t bytes;
  const char* name;
};

// Every buffer must be memory the current device owns (cudaMalloc'd, from a
// stream-ordered pool, or managed), and [p, p + bytes) must lie inside the
// allocation that holds p.  A host address (pageable or pinned) handed to
// TMA or to a kernel would be accessed as if it were device memory, and an
// undersized buffer would be overrun; both are refused here, before any
// launch, with ATTN_ERR_INVALID_ARG.
attn_status_t check_bufs(const DeviceInfo& d, std::initializer_list<Buf> bufs) {
  for (const Buf& b : bufs) {
    if (b.p == nullptr || b.bytes == 0) continue;
    cudaPointerAttributes attr;
    const cudaError_t e = cudaPointerGetAttributes(&attr, b.p);
    if (e != cudaSuccess) {
      cudaGetLastError();   // not a launch error: clear it
      return fail(ATTN_ERR_INVALID_ARG, "%s (%p) is not device memory: %s", b.name, b.p,
                  cudaGetErrorString(e));
    }
    const bool ok = attr.type == cudaMemoryTypeManaged ||
                    (attr.type == cudaMemoryTypeDevice && attr.device == d.index);
    if (!ok)
      return fail(ATTN_ERR_INVALID_ARG, "%s (%p) is not memory of device %d (memory type %d, device %d)",
                  b.name, b.p, d.index, (int)attr.type, attr.device);
    if (g_address_range != nullptr) {
      CUdeviceptr base = 0;
      size_t size = 0;
      if (g_address_range(&base, &size, reinterpret_cast<CUdeviceptr>(b.p)) == CUDA_SUCCESS) {
        const uintptr_t end = static_cast<uintptr_t>(base) + size;
        if (reinterpret_cast<uintptr_t>(b.p) + b.bytes > end)
          return fail(ATTN_ERR_INVALID_ARG, "%s: %zu bytes from %p run past the end of its allocation "
                      "(%zu bytes at %p)", b.name, b.bytes, b.p, size, reinterpret_cast<void*>(base));
      }
    }
  }
  return ATTN_OK;
}

// bf16 tensor map over `rank` dims (innermost first), 64-column boxes,
// 128-byte swizzle, zero fill out of bounds.
attn_status_t encode_bf16(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                          const cuuint32_t* box) {
  cuuint64_t strides[4];
  cuuint64_t acc = dims[0] * 2;
  for (int i = 1; i < rank; ++i) {
    strides[i - 1] = acc;
    acc *= dims[i];
  }
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}

// bf16 tensor map with explicit byte strides of dims 1.. (innermost dim
// contiguous), 128-byte swizzle, zero fill out of bounds.
attn_status_t encode_bf16_strided(CUtensorMap* map, const void* base, int rank, const cuuint64_t* dims,
                                  const cuuint64_t* strides, const cuuint32_t* box) {
  cuuint32_t estr[5] = {1, 1, 1, 1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return fail(ATTN_ERR_INVALID_ARG, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  return ATTN_OK;
}

attn_status_t launch_result(cudaError_t e, const char* what) {
  if (e != cudaSuccess) return fail(ATTN_ERR_LAUNCH, "%s launch failed: %s", what, cudaGetErrorString(e));
  g_last_error[0] = '\0';
  return ATTN_OK;
}

// Host-side checks of a decode call that need neither the workspace nor the
// device: sizes, supported shapes, null and misaligned pointers.  Shared by
// attn_decode_paged and attn_decode_paged_noalloc.
attn_status_t decode_check_args(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
                                int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
                                int num_blocks, float scale, const void* o, const float* lse) {
  if (num_seqs < 0 || Hq < 1 || Hkv < 1 || max_blocks_per_seq < 1 || num_blocks < 1)
    return fail(ATTN_ERR_INVALID_ARG,
                "sizes must satisfy num_seqs >= 0, Hq, Hkv, max_blocks_per_seq, num_blocks >= 1");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq (%d) is not a multiple of Hkv (%d)", Hq, Hkv);
  if (!finite_positive(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (block_size != 16) return fail(ATTN_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  if (Hq / Hkv > 16) return fail(ATTN_ERR_UNSUPPORTED, "Hq/Hkv = %d > 16 not supported", Hq / Hkv);
  if (static_cast<long long>(num_blocks) * Hkv * block_size >= 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "KV pool too large (num_blocks * Hkv * 16 >= 2^31)");
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "max_blocks_per_seq too large");
  if (static_cast<long long>(num_seqs) * Hq >= 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "num_seqs * Hq too large");
  if (num_seqs == 0) return ATTN_OK;
  if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o)
    return fail(ATTN_ERR_INVALID_ARG, "q, caches, block_table, seq_lens and o must be non-null");
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o))
    return fail(ATTN_ERR_INVALID_ARG, "q, caches and o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "block_table, seq_lens and lse must be 4-byte aligned");
  return ATTN_OK;
}

// Bytes of every decode buffer other than the workspace.
struct DecodeBytes {
  size_t q, cache, table, lens, o, lse;
};
DecodeBytes decode_bytes(int num_seqs, int Hq, int Hkv, int d, int max_blocks, int num_blocks) {
  DecodeBytes b;
  b.q = b.o = static_cast<size_t>(num_seqs) * Hq * d * 2;
  b.cache = static_cast<size_t>(num_blocks) * Hkv * 16 * d * 2;
  b.table = static_cast<size_t>(num_seqs) * max_blocks * 4;
  b.lens = static_cast<size_t>(num_seqs) * 4;
  b.lse = static_cast<size_t>(num_seqs) * Hq * 4;
  return b;
}

// Checks the decode's buffers against the device, encodes the cache maps and
// launches the decode with a workspace that has already been checked.
attn_status_t decode_launch(const DeviceInfo& dev, const void* q, const void* k_cache,
                            const void* v_cache, const int32_t* block_table, const int32_t* seq_lens,
                            int num_seqs, int Hq, int Hkv, int d, int max_blocks_per_seq, int num_blocks,
                            float scale, void* o, float* lse, void* workspace, void* stream) {
  const DecodeBytes nb = decode_bytes(num_seqs, Hq, Hkv, d, max_blocks_per_seq, num_blocks);
  attn_status_t st = check_bufs(dev, {{q, nb.q, "q"}, {k_cache, nb.cache, "k_cache"},
                                      {v_cache, nb.cache, "v_cache"}, {block_table, nb.table, "block_table"},
                                      {seq_lens, nb.lens, "seq_lens"}, {o, nb.o, "o"}, {lse, nb.lse, "lse"}});
  if (st != ATTN_OK) return st;
  // One copy per (block, head) slice: 64 columns x 16 rows x d/64 halves.
  const cuuint32_t box[3] = {64, 16, static_cast<cuuint32_t>(d / 64)};
  const cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(num_blocks) * Hkv * 16,
                              static_cast<cuuint64_t>(d / 64)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(d) * 2, 128};
  alignas(64) CUtensorMap tk, tv;
  if ((st = encode_bf16_strided(&tk, k_cache, 3, dims, strides, box)) != ATTN_OK) return st;
  if ((st = encode_bf16_strided(&tv, v_cache, 3, dims, strides, box)) != ATTN_OK) return st;

  attn47::DecLaunch a;
  a.tk = &tk;
  a.tv = &tv;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.seq_lens = seq_lens;
  a.o = o;
  a.lse = lse;
  a.workspace = static_cast<float*>(workspace);
  a.num_seqs = num_seqs;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.d = d;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  a.sms = dev.sms;
  a.max_ctas = g_decode_max_ctas;
  a.early_plan = g_decode_early_plan.load();
  a.epoch = next_decode_epoch();
  a.scale = scale;
  a.status = dev.status;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_decode_sm103(a), "attn_decode_paged");
}

__global__ void selftest_wait_kernel(unsigned int* status, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    attn47::mbar_init(attn47::smem_addr(&bar), 1);
    abort_flag = 0;
    attn47::fence_mbar_init();
  }
  __syncwarp();
  const attn47::WaitCtl wc{&abort_flag, status, timeout_ns};
  // Nothing arrives on `bar`: the wait must give up after timeout_ns.
  attn47::mbar_wait_warp(attn47::smem_addr(&bar), 0, wc);
}

}  // namespace

extern "C" {

int attn_abi_version(void) { return ATTN47_ABI_VERSION; }

const char* attn_last_error(void) { return g_last_error; }

const char* attn_status_string(attn_status_t s) {
  switch (s) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_DEVICE: return "ATTN_ERR_DEVICE";
    case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
  }
  return "ATTN_ERR_UNKNOWN";
}

void attn_set_wait_timeout_ns(unsigned long long ns) { g_timeout_ns = ns < 1000ull ? 1000ull : ns; }

void attn_set_decode_max_ctas(int ctas) { g_decode_max_ctas = ctas > 0 ? ctas : 0; }

void attn_set_decode_early_plan(int on) { g_decode_early_plan.store(on <= 0 ? 0 : on >= 2 ? 2 : 1); }

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int Hq, int Hkv, int N, int d, int causal, float scale, void* stream) {
  if (B < 0 || N < 0 || Hq < 1 || Hkv < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy B >= 0, N >= 0, Hq >= 1, Hkv >= 1");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq (%d) is not a multiple of Hkv (%d)", Hq, Hkv);
  if (!finite_positive(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  if (B == 0 || N == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!q || !k || !v || !o) return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v and o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const long long tiles = (static_cast<long long>(N) + 127) / 128;
  if (static_cast<long long>(B) * Hq * tiles > 0x7fffffffLL || static_cast<long long>(B) * Hq > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  const size_t qb = static_cast<size_t>(B) * Hq * N * d * 2, kvb = static_cast<size_t>(B) * Hkv * N * d * 2;
  if ((st = check_bufs(*dev, {{q, qb, "q"}, {k, kvb, "k"}, {v, kvb, "v"}, {o, qb, "o"},
                              {lse, static_cast<size_t>(B) * Hq * N * 4, "lse"}})) != ATTN_OK)
    return st;

  const cuuint32_t rows = static_cast<cuuint32_t>(attn47::fwd_box_rows());
  const cuuint32_t box[3] = {64, rows, 1};
  const cuuint64_t dq[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                            static_cast<cuuint64_t>(B) * Hq};
  const cuuint64_t dkv[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                             static_cast<cuuint64_t>(B) * Hkv};
  alignas(64) CUtensorMap tq, tk, tv;
  if ((st = encode_bf16(&tq, q, 3, dq, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(&tk, k, 3, dkv, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(&tv, v, 3, dkv, box)) != ATTN_OK) return st;

  attn47::FwdLaunch a;
  a.tq = &tq;
  a.tk = &tk;
  a.tv = &tv;
  a.o = o;
  a.lse = lse;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.d = d;
  a.causal = causal != 0;
  a.scale = scale;
  a.sms = dev->sms;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_fwd_sm103(a), "attn_fwd");
}

size_t attn_bwd_workspace_size(int B, int Hq, int N) {
  if (B <= 0 || Hq <= 0 || N <= 0) return 0;
  return attn47::bwd_workspace_bytes(B, Hq, N);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
                       const void* dout, void* dq, void* dk, void* dv, int B, int Hq, int Hkv, int N,
                       int d, int causal, float scale, void* workspace, size_t workspace_bytes,
                       void* stream) {
  if (B < 0 || N < 0 || Hq < 1 || Hkv < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy B >= 0, N >= 0, Hq >= 1, Hkv >= 1");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq (%d) is not a multiple of Hkv (%d)", Hq, Hkv);
  if (!finite_positive(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  if (B == 0 || N == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!q || !k || !v || !o || !lse || !dout || !dq || !dk || !dv)
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o, lse, dout, dq, dk and dv must be non-null");
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) ||
      !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return fail(ATTN_ERR_INVALID_ARG, "q, k, v, o, dout, dq, dk and dv must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return fail(ATTN_ERR_INVALID_ARG, "lse must be 4-byte aligned");
  const size_t need = attn47::bwd_workspace_bytes(B, Hq, N);
  if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace must be non-null");
  if ((reinterpret_cast<uintptr_t>(workspace) & 15u) != 0)
    return fail(ATTN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  if (workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace too small: %zu bytes given, %zu needed", workspace_bytes, need);
  const long long tiles = (static_cast<long long>(N) + 127) / 128;
  if (static_cast<long long>(B) * Hq * tiles > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  const size_t qb = static_cast<size_t>(B) * Hq * N * d * 2, kvb = static_cast<size_t>(B) * Hkv * N * d * 2;
  if ((st = check_bufs(*dev, {{q, qb, "q"}, {k, kvb, "k"}, {v, kvb, "v"}, {o, qb, "o"},
                              {lse, static_cast<size_t>(B) * Hq * N * 4, "lse"}, {dout, qb, "dout"},
                              {dq, qb, "dq"}, {dk, kvb, "dk"}, {dv, kvb, "dv"},
                              {workspace, need, "workspace"}})) != ATTN_OK)
    return st;

  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(attn47::bwd_box_rows()), 1};
  const cuuint64_t dq_dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                 static_cast<cuuint64_t>(B) * Hq};
  const cuuint64_t dkv_dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                                  static_cast<cuuint64_t>(B) * Hkv};
  alignas(64) CUtensorMap tq, tk, tv, tdo;
  if ((st = encode_bf16(&tq, q, 3, dq_dims, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(&tk, k, 3, dkv_dims, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(&tv, v, 3, dkv_dims, box)) != ATTN_OK) return st;
  if ((st = encode_bf16(&tdo, dout, 3, dq_dims, box)) != ATTN_OK) return st;

  attn47::BwdLaunch a;
  a.tq = &tq;
  a.tk = &tk;
  a.tv = &tv;
  a.tdo = &tdo;
  a.o = o;
  a.dout = dout;
  a.lse = lse;
  a.dq = dq;
  a.dk = dk;
  a.dv = dv;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.d = d;
  a.causal = causal != 0;
  a.scale = scale;
  a.workspace = static_cast<float*>(workspace);
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_bwd_sm103(a), "attn_bwd");
}

size_t attn_decode_paged_workspace_size(int num_seqs, int Hq, int d, int max_blocks_per_seq) {
  if (num_seqs <= 0 || Hq <= 0 || d <= 0 || max_blocks_per_seq <= 0) return 0;
  return attn47::decode_workspace_bytes(num_seqs, Hq, d, max_blocks_per_seq);
}

attn_status_t attn_decode_paged(const void* q, const void* k_cache, const void* v_cache,
                                const int32_t* block_table, const int32_t* seq_lens, int num_seqs,
                                int Hq, int Hkv, int d, int block_size, int max_blocks_per_seq,
                                int num_blocks, float scale, void* o, float* lse, void* workspace,
                                size_t workspace_bytes, void* stream) {
  attn_status_t st = decode_check_args(q, k_cache, v_cache, block_table, seq_lens, num_seqs, Hq, Hkv,
                                       d, block_size, max_blocks_per_seq, num_blocks, scale, o, lse);
  if (st != ATTN_OK) return st;
  if (num_seqs == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!workspace) return fail(ATTN_ERR_INVALID_ARG, "workspace must be non-null");
  if (!aligned16(workspace)) return fail(ATTN_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
  const size_t need = attn_decode_paged_workspace_size(num_seqs, Hq, d, max_blocks_per_seq);
  if (workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  const DecodeBytes nb = decode_bytes(num_seqs, Hq, Hkv, d, max_blocks_per_seq, num_blocks);
  const struct {
    const void* p;
    size_t n;
  } others[] = {{q, nb.q}, {k_cache, nb.cache}, {v_cache, nb.cache}, {block_table, nb.table},
                {seq_lens, nb.lens}, {o, nb.o}, {lse, lse ? nb.lse : 0}};
  for (const auto& x : others)
    if (x.n && overlap(workspace, need, x.p, x.n))
      return fail(ATTN_ERR_INVALID_ARG, "workspace overlaps an input or output of the decode");
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != ATTN_OK) return st;
  if ((st = check_bufs(*dev, {{workspace, need, "workspace"}})) != ATTN_OK) return st;
  return decode_launch(*dev, q, k_cache, v_cache, block_table, seq_lens, num_seqs, Hq, Hkv, d,
                       max_blocks_per_seq, num_blocks, scale, o, lse, workspace, stream);
}

attn_status_t attn_decode_paged_noalloc(const void* q, const void* k_cache, const void* v_cache,
                                        const int32_t* block_table, const int32_t* seq_lens,
                                        int num_seqs, int Hq, int Hkv, int d, int block_size,
                                        int max_blocks_per_seq, int num_blocks, float scale,
                                        void* o, float* lse, void* stream) {
  // The same argument checks as attn_decode_paged first, so that both calls
  // give the same answer to the same bad arguments; only then the size of
  // the scratch this decode needs against the built-in array.
  attn_status_t st = decode_check_args(q, k_cache, v_cache, block_table, seq_lens, num_seqs, Hq, Hkv,
                                       d, block_size, max_blocks_per_seq, num_blocks, scale, o, lse);
  if (st != ATTN_OK) return st;
  if (num_seqs == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  const size_t need = attn_decode_paged_workspace_size(num_seqs, Hq, d, max_blocks_per_seq);
  if (need > kNoAllocScratchBytes)
    return fail(ATTN_ERR_WORKSPACE,
                "this decode needs %zu bytes of scratch but the built-in array of "
                "attn_decode_paged_noalloc holds %zu; call attn_decode_paged with a workspace",
                need, kNoAllocScratchBytes);
  DeviceInfo* dev = nullptr;
  if ((st = current_device(&dev)) != ATTN_OK) return st;
  void* scratch = nullptr;
  {
    // One-time set-up per device (this device is current): the host-side
    // name of the array is not a device address, so look the address up.
    std::lock_guard<std::mutex> lock(g_mu);
    if (dev->noalloc_scratch == nullptr) {
      void* addr = nullptr;
      const cudaError_t e = cudaGetSymbolAddress(&addr, g_attn47_noalloc_scratch);
      if (e != cudaSuccess || addr == nullptr)
        return fail(ATTN_ERR_DEVICE, "scratch array address unavailable: %s", cudaGetErrorString(e));
      dev->noalloc_scratch = addr;
    }
    scratch = dev->noalloc_scratch;
  }
  return decode_launch(*dev, q, k_cache, v_cache, block_table, seq_lens, num_seqs, Hq, Hkv, d,
                       max_blocks_per_seq, num_blocks, scale, o, lse, scratch, stream);
}

attn_status_t attn_prefill_paged(const void* q, const void* k_new, const void* v_new,
                                 void* k_cache, void* v_cache, const int32_t* block_table,
                                 const int32_t* ctx_lens, int num_seqs, int Hq, int Hkv, int N,
                                 int d, int block_size, int max_blocks_per_seq, int num_blocks,
                                 float scale, void* o, float* lse, void* stream) {
  if (num_seqs < 0 || N < 0 || Hq < 1 || Hkv < 1 || max_blocks_per_seq < 1 || num_blocks < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy num_seqs >= 0, N >= 0, Hq, Hkv, "
                "max_blocks_per_seq, num_blocks >= 1");
  if (Hq % Hkv != 0) return fail(ATTN_ERR_INVALID_ARG, "Hq (%d) is not a multiple of Hkv (%d)", Hq, Hkv);
  if (!finite_positive(scale)) return fail(ATTN_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (block_size != 16) return fail(ATTN_ERR_UNSUPPORTED, "block_size %d not supported (16)", block_size);
  if (d != 64 && d != 128) return fail(ATTN_ERR_UNSUPPORTED, "head dim %d not supported (64 or 128)", d);
  if (static_cast<long long>(max_blocks_per_seq) * block_size >= 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "max_blocks_per_seq too large");
  if (static_cast<long long>(max_blocks_per_seq) * block_size < N)
    return fail(ATTN_ERR_INVALID_ARG, "N (%d) new tokens do not fit in max_blocks_per_seq (%d) blocks",
                N, max_blocks_per_seq);
  if (num_seqs == 0 || N == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!q || !k_new || !v_new || !k_cache || !v_cache || !block_table || !ctx_lens || !o)
    return fail(ATTN_ERR_INVALID_ARG, "q, k_new, v_new, caches, block_table, ctx_lens and o must be non-null");
  if (!aligned16(q) || !aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) ||
      !aligned16(v_cache) || !aligned16(o))
    return fail(ATTN_ERR_INVALID_ARG, "q, k_new, v_new, caches and o must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(ctx_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(lse) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "block_table, ctx_lens and lse must be 4-byte aligned");
  const long long tiles = (static_cast<long long>(N) + 127) / 128;
  if (static_cast<long long>(num_seqs) * Hq * tiles > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  {
    const size_t qb = static_cast<size_t>(num_seqs) * Hq * N * d * 2;
    const size_t kvb = static_cast<size_t>(num_seqs) * Hkv * N * d * 2;
    const size_t cb = static_cast<size_t>(num_blocks) * Hkv * 16 * d * 2;
    if ((st = check_bufs(*dev, {{q, qb, "q"}, {k_new, kvb, "k_new"}, {v_new, kvb, "v_new"},
                                {k_cache, cb, "k_cache"}, {v_cache, cb, "v_cache"},
                                {block_table, static_cast<size_t>(num_seqs) * max_blocks_per_seq * 4,
                                 "block_table"},
                                {ctx_lens, static_cast<size_t>(num_seqs) * 4, "ctx_lens"}, {o, qb, "o"},
                                {lse, static_cast<size_t>(num_seqs) * Hq * N * 4, "lse"}})) != ATTN_OK)
      return st;
  }

  // Q goes through TMA; the kernel gathers the cached K/V blocks itself.
  const cuuint32_t qbox[3] = {64, static_cast<cuuint32_t>(attn47::fwd_box_rows()), 1};
  const cuuint64_t qdims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(N),
                               static_cast<cuuint64_t>(num_seqs) * Hq};
  alignas(64) CUtensorMap tq;
  if ((st = encode_bf16(&tq, q, 3, qdims, qbox)) != ATTN_OK) return st;

  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  attn47::AppendLaunch w;
  w.k_new = k_new;
  w.v_new = v_new;
  w.k_cache = k_cache;
  w.v_cache = v_cache;
  w.block_table = block_table;
  w.ctx_lens = ctx_lens;
  w.B = num_seqs;
  w.Hkv = Hkv;
  w.N = N;
  w.d = d;
  w.max_blocks = max_blocks_per_seq;
  w.num_blocks = num_blocks;
  w.sms = dev->sms;
  w.status = dev->status;
  w.stream = s;
  st = launch_result(attn47::launch_kv_append_sm103(w), "attn_prefill_paged (append)");
  if (st != ATTN_OK) return st;

  attn47::FwdLaunch a;
  a.tq = &tq;
  a.tk = &tq;   // unused in paged mode
  a.tv = &tq;
  a.o = o;
  a.lse = lse;
  a.B = num_seqs;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.N = N;
  a.d = d;
  a.causal = true;
  a.scale = scale;
  a.sms = dev->sms;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns;
  a.stream = s;
  a.paged = true;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_table = block_table;
  a.ctx_lens = ctx_lens;
  a.max_blocks = max_blocks_per_seq;
  a.num_blocks = num_blocks;
  return launch_result(attn47::launch_fwd_sm103(a), "attn_prefill_paged (attention)");
}

attn_status_t fused_add_rmsnorm(const void* x, void* residual, const void* weight, void* out,
                                int rows, int hidden, float eps, void* stream) {
  if (rows < 0 || hidden < 8) return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy rows >= 0, hidden >= 8");
  if (hidden % 8 != 0)
    return fail(ATTN_ERR_UNSUPPORTED, "hidden (%d) must be a multiple of 8 (16-byte rows)", hidden);
  if (!(std::isfinite(eps) && eps >= 0.f)) return fail(ATTN_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (rows == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!x || !residual || !weight || !out)
    return fail(ATTN_ERR_INVALID_ARG, "x, residual, weight and out must be non-null");
  if (!aligned16(x) || !aligned16(residual) || !aligned16(weight) || !aligned16(out))
    return fail(ATTN_ERR_INVALID_ARG, "x, residual, weight and out must be 16-byte aligned");
  const size_t bytes = static_cast<size_t>(rows) * hidden * 2;
  if (overlap(residual, bytes, x, bytes) || overlap(residual, bytes, out, bytes) ||
      overlap(out, bytes, x, bytes) || overlap(weight, static_cast<size_t>(hidden) * 2, residual, bytes) ||
      overlap(weight, static_cast<size_t>(hidden) * 2, out, bytes))
    return fail(ATTN_ERR_INVALID_ARG, "x, residual, weight and out must not overlap");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  if ((st = check_bufs(*dev, {{x, bytes, "x"}, {residual, bytes, "residual"},
                              {weight, static_cast<size_t>(hidden) * 2, "weight"}, {out, bytes, "out"}})) != ATTN_OK)
    return st;
  attn47::NormLaunch a;
  a.x = x;
  a.residual = residual;
  a.weight = weight;
  a.out = out;
  a.rows = rows;
  a.hidden = hidden;
  a.eps = eps;
  a.sms = dev->sms;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_add_rmsnorm_sm103(a), "fused_add_rmsnorm");
}

attn_status_t fused_swiglu(const void* gate_up, void* out, int rows, int F, void* stream) {
  if (rows < 0 || F < 8) return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy rows >= 0, F >= 8");
  if (F % 8 != 0) return fail(ATTN_ERR_UNSUPPORTED, "F (%d) must be a multiple of 8 (16-byte rows)", F);
  if (rows == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!gate_up || !out) return fail(ATTN_ERR_INVALID_ARG, "gate_up and out must be non-null");
  if (!aligned16(gate_up) || !aligned16(out))
    return fail(ATTN_ERR_INVALID_ARG, "gate_up and out must be 16-byte aligned");
  if (overlap(gate_up, static_cast<size_t>(rows) * F * 4, out, static_cast<size_t>(rows) * F * 2))
    return fail(ATTN_ERR_INVALID_ARG, "gate_up and out must not overlap");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  if ((st = check_bufs(*dev, {{gate_up, static_cast<size_t>(rows) * F * 4, "gate_up"},
                              {out, static_cast<size_t>(rows) * F * 2, "out"}})) != ATTN_OK)
    return st;
  attn47::GluLaunch a;
  a.gate_up = gate_up;
  a.out = out;
  a.rows = rows;
  a.F = F;
  a.sms = dev->sms;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_swiglu_sm103(a), "fused_swiglu");
}

attn_status_t swiglu_projection(const void* x, const void* w_gate_up, void* out, int rows, int hidden,
                                int F, void* stream) {
  if (rows < 0 || hidden < 1 || F < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy rows >= 0, hidden >= 1, F >= 1");
  if (hidden % attn47::swiglu_proj_k_step() != 0)
    return fail(ATTN_ERR_UNSUPPORTED, "hidden (%d) must be a multiple of %d", hidden, attn47::swiglu_proj_k_step());
  if (F % attn47::swiglu_proj_tile_features() != 0)
    return fail(ATTN_ERR_UNSUPPORTED, "F (%d) must be a multiple of %d", F, attn47::swiglu_proj_tile_features());
  if (static_cast<long long>(rows) > 0x7fffffffLL - 128 || 2LL * F > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  if (rows == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!x || !w_gate_up || !out) return fail(ATTN_ERR_INVALID_ARG, "x, w_gate_up and out must be non-null");
  if (!aligned16(x) || !aligned16(w_gate_up) || !aligned16(out))
    return fail(ATTN_ERR_INVALID_ARG, "x, w_gate_up and out must be 16-byte aligned");
  const size_t xb = static_cast<size_t>(rows) * hidden * 2;
  const size_t wb = static_cast<size_t>(2) * F * hidden * 2;
  const size_t ob = static_cast<size_t>(rows) * F * 2;
  if (overlap(out, ob, x, xb) || overlap(out, ob, w_gate_up, wb))
    return fail(ATTN_ERR_INVALID_ARG, "out must not overlap x or w_gate_up");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  if ((st = check_bufs(*dev, {{x, xb, "x"}, {w_gate_up, wb, "w_gate_up"}, {out, ob, "out"}})) != ATTN_OK)
    return st;
  CUtensorMap tx, tw;
  const cuuint32_t box[2] = {64, 128};
  const cuuint64_t xdims[2] = {static_cast<cuuint64_t>(hidden), static_cast<cuuint64_t>(rows)};
  if ((st = encode_bf16(&tx, x, 2, xdims, box)) != ATTN_OK) return st;
  const cuuint64_t wdims[2] = {static_cast<cuuint64_t>(hidden), static_cast<cuuint64_t>(2) * F};
  if ((st = encode_bf16(&tw, w_gate_up, 2, wdims, box)) != ATTN_OK) return st;
  attn47::SwigluProjLaunch a;
  a.tx = &tx;
  a.tw = &tw;
  a.out = out;
  a.rows = rows;
  a.F = F;
  a.hidden = hidden;
  a.sms = dev->sms;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_swiglu_proj_sm103(a), "swiglu_projection");
}

size_t ssd_workspace_size(int batch, int L, int H, int N, int chunk) {
  if (batch <= 0 || L <= 0 || H <= 0 || N <= 0 || chunk <= 0) return 0;
  return attn47::ssd_workspace_bytes(batch, L, H, N, chunk);
}

attn_status_t ssd_chunked_fwd(const void* x, const float* dt, const float* A, const void* B,
                              const void* C, const float* h0, void* y, float* h_final, int batch,
                              int L, int H, int G, int P, int N, int chunk, void* workspace,
                              size_t workspace_bytes, void* stream) {
  if (batch < 0 || L < 0 || H < 1 || G < 1)
    return fail(ATTN_ERR_INVALID_ARG, "sizes must satisfy batch >= 0, L >= 0, H >= 1, G >= 1");
  if (H % G != 0) return fail(ATTN_ERR_INVALID_ARG, "H (%d) is not a multiple of G (%d)", H, G);
  if (P != attn47::ssd_head_dim()) return fail(ATTN_ERR_UNSUPPORTED, "head dim P = %d not supported (64)", P);
  if (N != 64 && N != 128) return fail(ATTN_ERR_UNSUPPORTED, "state size N = %d not supported (64 or 128)", N);
  if (chunk != 64 && chunk != 128 && chunk != 256)
    return fail(ATTN_ERR_UNSUPPORTED, "chunk = %d not supported (64, 128 or 256)", chunk);
  if (batch == 0 || L == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!x || !dt || !A || !B || !C || !y || !h_final || !workspace)
    return fail(ATTN_ERR_INVALID_ARG, "x, dt, A, B, C, y, h_final and workspace must be non-null");
  if (!aligned16(x) || !aligned16(B) || !aligned16(C) || !aligned16(y) || !aligned16(h_final) ||
      !aligned16(workspace) || (h0 && !aligned16(h0)))
    return fail(ATTN_ERR_INVALID_ARG, "x, B, C, y, h0, h_final and workspace must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(dt) & 3u) || (reinterpret_cast<uintptr_t>(A) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "dt and A must be 4-byte aligned");
  const long long nc = (static_cast<long long>(L) + chunk - 1) / chunk;
  if (static_cast<long long>(batch) * nc * H * (chunk / 64) > 0x7fffffffLL ||
      static_cast<long long>(batch) * nc * H * P > 0x7fffffffLL || static_cast<long long>(L) + chunk > 0x7fffffffLL)
    return fail(ATTN_ERR_UNSUPPORTED, "problem too large for one launch");
  const size_t need = ssd_workspace_size(batch, L, H, N, chunk);
  if (workspace_bytes < need)
    return fail(ATTN_ERR_WORKSPACE, "workspace has %zu bytes, needs %zu", workspace_bytes, need);
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  {
    const size_t xb = static_cast<size_t>(batch) * L * H * P * 2;
    const size_t bcb = static_cast<size_t>(batch) * L * G * N * 2;
    const size_t hb = static_cast<size_t>(batch) * H * P * N * 4;
    if ((st = check_bufs(*dev, {{x, xb, "x"}, {dt, static_cast<size_t>(batch) * L * H * 4, "dt"},
                                {A, static_cast<size_t>(H) * 4, "A"}, {B, bcb, "B"}, {C, bcb, "C"},
                                {h0, hb, "h0"}, {y, xb, "y"}, {h_final, hb, "h_final"},
                                {workspace, need, "workspace"}})) != ATTN_OK)
      return st;
  }
  attn47::SsdLaunch a;
  a.x = x;
  a.dt = dt;
  a.A = A;
  a.B = B;
  a.C = C;
  a.h0 = h0;
  a.y = y;
  a.h_final = h_final;
  a.workspace = workspace;
  // Tensor maps: x over (P, H, L, batch), B and C over (N, G, L, batch),
  // the bf16 chunk states in the workspace over (N, batch * nc * H * P).
  CUtensorMap tx, tb, tc, ts;
  {
    const cuuint32_t rows = 64;
    const cuuint64_t xdims[4] = {static_cast<cuuint64_t>(P), static_cast<cuuint64_t>(H),
                                 static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(batch)};
    const cuuint64_t xstr[3] = {static_cast<cuuint64_t>(P) * 2, static_cast<cuuint64_t>(H) * P * 2,
                                static_cast<cuuint64_t>(L) * H * P * 2};
    const cuuint32_t xbox[4] = {64, 1, rows, 1};
    if ((st = encode_bf16_strided(&tx, x, 4, xdims, xstr, xbox)) != ATTN_OK) return st;
    const cuuint64_t bdims[4] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(G),
                                 static_cast<cuuint64_t>(L), static_cast<cuuint64_t>(batch)};
    const cuuint64_t bstr[3] = {static_cast<cuuint64_t>(N) * 2, static_cast<cuuint64_t>(G) * N * 2,
                                static_cast<cuuint64_t>(L) * G * N * 2};
    if ((st = encode_bf16_strided(&tb, B, 4, bdims, bstr, xbox)) != ATTN_OK) return st;
    const cuuint32_t cbox[4] = {64, 1, 128, 1};
    if ((st = encode_bf16_strided(&tc, C, 4, bdims, bstr, cbox)) != ATTN_OK) return st;
    const cuuint64_t sdims[2] = {static_cast<cuuint64_t>(N), static_cast<cuuint64_t>(batch * nc * H * P)};
    const cuuint64_t sstr[1] = {static_cast<cuuint64_t>(N) * 2};
    const cuuint32_t sbox[2] = {64, 64};
    const void* states = static_cast<const uint8_t*>(workspace) + attn47::ssd_states_offset(batch, L, H, chunk);
    if ((st = encode_bf16_strided(&ts, states, 2, sdims, sstr, sbox)) != ATTN_OK) return st;
  }
  a.tx = &tx;
  a.tb = &tb;
  a.tc = &tc;
  a.ts = &ts;
  a.batch = batch;
  a.L = L;
  a.H = H;
  a.G = G;
  a.N = N;
  a.chunk = chunk;
  a.status = dev->status;
  a.timeout_ns = g_timeout_ns;
  a.stream = static_cast<cudaStream_t>(stream);
  return launch_result(attn47::launch_ssd_sm103(a), "ssd_chunked_fwd");
}

attn_status_t attn_get_device_status(void* stream, unsigned int* flags_out) {
  if (!flags_out) return fail(ATTN_ERR_INVALID_ARG, "flags_out must be non-null");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned int host = 0;
  cudaError_t e = cudaMemcpyAsync(&host, dev->status, sizeof(host), cudaMemcpyDeviceToHost, s);
  if (e == cudaSuccess) e = cudaMemsetAsync(dev->status, 0, sizeof(unsigned int), s);
  if (e == cudaSuccess) e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return fail(ATTN_ERR_DEVICE, "status read failed: %s", cudaGetErrorString(e));
  *flags_out = host;
  g_last_error[0] = '\0';
  return ATTN_OK;
}

}  // extern "C"

namespace {
// One thread per pair of inputs: y = 2^x by the forward softmax's FMA-pipe
// exp2 (ex2_poly2), for testing that function on the device.
__global__ void selftest_exp2_poly_kernel(const float* x, float* y, int n) {
  const long long i = 2LL * (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x);
  if (i >= n) return;
  const bool two = i + 1 < n;
  float r0, r1;
  attn47::f2_unpack(attn47::ex2_poly2(attn47::f2_pack(x[i], two ? x[i + 1] : 0.f)), r0, r1);
  y[i] = r0;
  if (two) y[i + 1] = r1;
}
}  // namespace

extern "C" {

attn_status_t attn_selftest_exp2_poly(const float* x, float* y, int n, void* stream) {
  if (n < 0) return fail(ATTN_ERR_INVALID_ARG, "n must be >= 0");
  if (n == 0) {
    g_last_error[0] = '\0';
    return ATTN_OK;
  }
  if (!x || !y) return fail(ATTN_ERR_INVALID_ARG, "x and y must be non-null");
  if ((reinterpret_cast<uintptr_t>(x) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u))
    return fail(ATTN_ERR_INVALID_ARG, "x and y must be 4-byte aligned");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  const size_t bytes = static_cast<size_t>(n) * 4;
  if ((st = check_bufs(*dev, {{x, bytes, "x"}, {y, bytes, "y"}})) != ATTN_OK) return st;
  const long long pairs = (static_cast<long long>(n) + 1) / 2;
  selftest_exp2_poly_kernel<<<static_cast<unsigned>((pairs + 255) / 256), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      x, y, n);
  return launch_result(cudaGetLastError(), "attn_selftest_exp2_poly");
}

attn_status_t attn_selftest_wait_timeout(unsigned long long timeout_ns, void* stream,
                                         unsigned int* flags_out) {
  if (!flags_out) return fail(ATTN_ERR_INVALID_ARG, "flags_out must be non-null");
  if (timeout_ns > 10000000000ull) return fail(ATTN_ERR_INVALID_ARG, "timeout above 10 s");
  DeviceInfo* dev = nullptr;
  attn_status_t st = current_device(&dev);
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  selftest_wait_kernel<<<1, 32, 0, s>>>(dev->status, timeout_ns);
  st = launch_result(cudaGetLastError(), "selftest");
  if (st != ATTN_OK) return st;
  return attn_get_device_status(stream, flags_out);
}

}  // extern "C"
