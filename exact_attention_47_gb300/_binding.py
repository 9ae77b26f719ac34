"""ctypes binding of ``libattn47_sm103.so`` (argument marshalling only).

Every function here checks tensor properties the C-ABI cannot see (device,
dtype, contiguity, shapes), allocates outputs with torch when the caller
passes none, and forwards raw device pointers plus the current torch CUDA
stream to the C entry point of the same name.  All arithmetic runs in the
library's CUDA kernels; there is no other code path.  If the library is not
built, every call raises ``RuntimeError``.
"""

import ctypes
import os

import torch

from .build_lib import LIB_PATH

ATTN_OK = 0
ATTN_DEV_TIMEOUT = 0x1
ATTN_DEV_BAD_BLOCK = 0x2
ATTN_DEV_BAD_SEQLEN = 0x4
BLOCK_SIZE = 16

# C entry points and their signatures (mirrors include/attn47.h)
_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "attn_fwd": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float, _P]),
    "attn_bwd_workspace_size": (ctypes.c_size_t, [_I, _I, _I]),
    "attn_bwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, ctypes.c_float,
                      _P, ctypes.c_size_t, _P]),
    "attn_decode_paged_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I]),
    "attn_decode_paged": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float,
                               _P, _P, _P, ctypes.c_size_t, _P]),
    "attn_decode_paged_noalloc": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, ctypes.c_float,
                                       _P, _P, _P]),
    "attn_prefill_paged": (_I, [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _I,
                                ctypes.c_float, _P, _P, _P]),
    "fused_add_rmsnorm": (_I, [_P, _P, _P, _P, _I, _I, ctypes.c_float, _P]),
    "fused_swiglu": (_I, [_P, _P, _I, _I, _P]),
    "swiglu_projection": (_I, [_P, _P, _P, _I, _I, _I, _P]),
    "ssd_workspace_size": (ctypes.c_size_t, [_I, _I, _I, _I, _I]),
    "ssd_chunked_fwd": (_I, [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P,
                             ctypes.c_size_t, _P]),
    "attn_get_device_status": (_I, [_P, ctypes.POINTER(ctypes.c_uint)]),
    "attn_set_wait_timeout_ns": (None, [ctypes.c_ulonglong]),
    "attn_set_decode_max_ctas": (None, [_I]),
    "attn_set_decode_early_plan": (None, [_I]),
    "attn_selftest_wait_timeout": (_I, [ctypes.c_ulonglong, _P, ctypes.POINTER(ctypes.c_uint)]),
    "attn_selftest_exp2_poly": (_I, [_P, _P, _I, _P]),
    "attn_status_string": (ctypes.c_char_p, [_I]),
    "attn_last_error": (ctypes.c_char_p, []),
    "attn_abi_version": (_I, []),
}

_lib = None


class AttnError(RuntimeError):
    """A non-zero attn_status_t from the library."""

    def __init__(self, func, status, message):
        self.status = status
        super().__init__("%s failed: %s: %s" % (func, status_string(status), message))


def library_path():
    return LIB_PATH


def load_library(path=None):
    """Load (once) and return the ctypes handle of the CUDA library."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(
            "CUDA library %s is not built; run `python -c \"import __graft_entry__ as g; g.build()\"` "
            "(there is no CPU fallback)" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGS.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status):
    return load_library().attn_status_string(int(status)).decode()


def _check(func, status):
    if status != ATTN_OK:
        raise AttnError(func, status, load_library().attn_last_error().decode())


def _stream_handle(stream, device=None):
    """The raw cudaStream_t of `stream` (default: torch's current stream of
    `device`); a stream of another device is refused."""
    if stream is None:
        stream = torch.cuda.current_stream(device)
    elif device is not None and stream.device != device:
        raise ValueError("stream is on %s but the tensors are on %s" % (stream.device, device))
    return ctypes.c_void_p(stream.cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _need_cuda(name, t, dtype, device=None):
    """`t` is a contiguous CUDA tensor of `dtype` (any dtype if None) on
    `device` (if given)."""
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)
    if device is not None and t.device != device:
        raise ValueError("%s is on %s, the other tensors on %s" % (name, t.device, device))
    if dtype is not None and t.dtype != dtype:
        raise ValueError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def _need_shape(name, t, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError("%s must have shape %s, got %s" % (name, tuple(shape), tuple(t.shape)))


def _output(name, t, shape, dtype, device):
    """A caller-given output checked for device, dtype and shape, or a new one."""
    if t is None:
        return torch.empty(tuple(shape), dtype=dtype, device=device)
    _need_cuda(name, t, dtype, device)
    _need_shape(name, t, shape)
    return t


def _workspace(name, t, need, device):
    """A caller-given workspace (any dtype, contiguous, on `device`, at least
    `need` bytes), or a new one of `need` bytes."""
    if t is None:
        return torch.empty(max(int(need), 16), dtype=torch.uint8, device=device)
    _need_cuda(name, t, None, device)
    nbytes = t.numel() * t.element_size()
    if nbytes < need:
        raise ValueError("%s has %d bytes, needs %d" % (name, nbytes, need))
    return t


def _call(func, device, *args):
    """Call C entry point `func` with `device` current and raise on error."""
    lib = load_library()
    with torch.cuda.device(device):
        st = getattr(lib, func)(*args)
    _check(func, st)


def attn_fwd(q, k, v, causal=True, scale=None, o=None, lse=None, return_lse=True, stream=None):
    """Exact attention forward.  q [B,Hq,N,d], k/v [B,Hkv,N,d] bf16 on the GPU.

    Returns (o, lse): o [B,Hq,N,d] bf16, lse [B,Hq,N] fp32 (None when
    ``return_lse`` is False and no ``lse`` buffer is given).
    """
    _need_cuda("q", q, torch.bfloat16)
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v)):
        _need_cuda(name, t, torch.bfloat16, dev)
        if t.dim() != 4:
            raise ValueError("%s must be 4-D [B, H, N, d]" % name)
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    o = _output("o", o, q.shape, torch.bfloat16, dev)
    if lse is not None or return_lse:
        lse = _output("lse", lse, (B, Hq, N), torch.float32, dev)
    _call("attn_fwd", dev, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, Hq, Hkv, N, d,
          1 if causal else 0, float(scale), _stream_handle(stream, dev))
    return o, lse


def attn_bwd_workspace_size(B, Hq, N):
    return int(load_library().attn_bwd_workspace_size(B, Hq, N))


def attn_bwd(q, k, v, o, lse, dout, causal=True, scale=None, dq=None, dk=None, dv=None,
             workspace=None, stream=None):
    """Gradients of attn_fwd.  q/o/dout [B,Hq,N,d], k/v [B,Hkv,N,d] bf16 and
    lse [B,Hq,N] fp32 (attn_fwd's outputs for the same inputs), on the GPU.

    Returns (dq [B,Hq,N,d], dk [B,Hkv,N,d], dv [B,Hkv,N,d]) bf16.
    """
    _need_cuda("q", q, torch.bfloat16)
    dev = q.device
    for name, t in (("q", q), ("k", k), ("v", v), ("o", o), ("dout", dout)):
        _need_cuda(name, t, torch.bfloat16, dev)
        if t.dim() != 4:
            raise ValueError("%s must be 4-D [B, H, N, d]" % name)
    _need_cuda("lse", lse, torch.float32, dev)
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    _need_shape("o", o, q.shape)
    _need_shape("dout", dout, q.shape)
    _need_shape("lse", lse, (B, Hq, N))
    Hkv = k.shape[1]
    if scale is None:
        scale = d ** -0.5
    dq = _output("dq", dq, q.shape, torch.bfloat16, dev)
    dk = _output("dk", dk, k.shape, torch.bfloat16, dev)
    dv = _output("dv", dv, v.shape, torch.bfloat16, dev)
    workspace = _workspace("workspace", workspace, attn_bwd_workspace_size(B, Hq, N), dev)
    _call("attn_bwd", dev, _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(dout), _ptr(dq),
          _ptr(dk), _ptr(dv), B, Hq, Hkv, N, d, 1 if causal else 0, float(scale), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    return dq, dk, dv


def attn_decode_paged_workspace_size(num_seqs, Hq, d, max_blocks_per_seq):
    return int(load_library().attn_decode_paged_workspace_size(num_seqs, Hq, d, max_blocks_per_seq))


def _decode_args(q, k_cache, v_cache, block_table, seq_lens, scale, o, lse, return_lse):
    """Checks shared by both decode entry points; returns the sizes, the
    scale and the (checked or new) outputs."""
    _need_cuda("q", q, torch.bfloat16)
    dev = q.device
    for name, t, dt in (("k_cache", k_cache, torch.bfloat16), ("v_cache", v_cache, torch.bfloat16),
                        ("block_table", block_table, torch.int32), ("seq_lens", seq_lens, torch.int32)):
        _need_cuda(name, t, dt, dev)
    if q.dim() != 3 or k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("q must be [S,Hq,d] and caches [num_blocks,Hkv,block_size,d]")
    S, Hq, d = q.shape
    num_blocks, Hkv, block_size, dc = k_cache.shape
    if dc != d:
        raise ValueError("cache head dim %d differs from q's %d" % (dc, d))
    if block_table.dim() != 2 or block_table.shape[0] != S:
        raise ValueError("block_table must be [S, max_blocks]")
    _need_shape("seq_lens", seq_lens, (S,))
    o = _output("o", o, (S, Hq, d), torch.bfloat16, dev)
    if lse is not None or return_lse:
        lse = _output("lse", lse, (S, Hq), torch.float32, dev)
    if scale is None:
        scale = d ** -0.5
    return dev, S, Hq, Hkv, d, block_size, block_table.shape[1], num_blocks, float(scale), o, lse


def attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, scale=None, o=None, lse=None,
                      workspace=None, return_lse=True, stream=None):
    """Paged-KV decode.  q [S,Hq,d]; caches [num_blocks,Hkv,16,d] bf16;
    block_table [S,max_blocks] int32; seq_lens [S] int32 (all on the GPU).

    Returns (o [S,Hq,d] bf16, lse [S,Hq] fp32 or None).
    """
    dev, S, Hq, Hkv, d, bs, mb, nb, scale, o, lse = _decode_args(
        q, k_cache, v_cache, block_table, seq_lens, scale, o, lse, return_lse)
    workspace = _workspace("workspace", workspace, attn_decode_paged_workspace_size(S, Hq, d, mb), dev)
    _call("attn_decode_paged", dev, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
          _ptr(seq_lens), S, Hq, Hkv, d, bs, mb, nb, scale, _ptr(o), _ptr(lse), _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    return o, lse


def attn_decode_paged_noalloc(q, k_cache, v_cache, block_table, seq_lens, scale=None, o=None,
                              lse=None, return_lse=True, stream=None):
    """attn_decode_paged without a workspace argument, for callers that may
    not allocate device memory when they run the decode: the library uses
    its own fixed 8 MiB device array instead (sizes needing more raise
    AttnError with ATTN_ERR_WORKSPACE).  Calls that overlap on the GPU share
    that array and must be ordered.  Only the outputs, if not given, are
    allocated here, by torch; pass ``o`` (and ``lse`` or return_lse=False)
    to allocate nothing at all."""
    dev, S, Hq, Hkv, d, bs, mb, nb, scale, o, lse = _decode_args(
        q, k_cache, v_cache, block_table, seq_lens, scale, o, lse, return_lse)
    _call("attn_decode_paged_noalloc", dev, _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_table),
          _ptr(seq_lens), S, Hq, Hkv, d, bs, mb, nb, scale, _ptr(o), _ptr(lse),
          _stream_handle(stream, dev))
    return o, lse


def attn_prefill_paged(q, k_new, v_new, k_cache, v_cache, block_table, ctx_lens, scale=None,
                       o=None, lse=None, return_lse=True, stream=None):
    """Chunked prefill over a paged cache (all tensors on the GPU).

    q [S,Hq,N,d], k_new / v_new [S,Hkv,N,d] bf16; caches
    [num_blocks,Hkv,16,d] bf16 (updated in place: the new rows are appended at
    positions ctx_lens[b] + i); block_table [S,max_blocks] int32; ctx_lens [S]
    int32 (left unchanged).  Returns (o [S,Hq,N,d] bf16, lse [S,Hq,N] fp32 or
    None).
    """
    _need_cuda("q", q, torch.bfloat16)
    dev = q.device
    for name, t, dt in (("k_new", k_new, torch.bfloat16), ("v_new", v_new, torch.bfloat16),
                        ("k_cache", k_cache, torch.bfloat16), ("v_cache", v_cache, torch.bfloat16),
                        ("block_table", block_table, torch.int32), ("ctx_lens", ctx_lens, torch.int32)):
        _need_cuda(name, t, dt, dev)
    if q.dim() != 4 or k_new.dim() != 4 or k_new.shape != v_new.shape:
        raise ValueError("q must be [S,Hq,N,d] and k_new / v_new [S,Hkv,N,d]")
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("caches must be [num_blocks,Hkv,block_size,d]")
    S, Hq, N, d = q.shape
    num_blocks, Hkv, block_size, dc = k_cache.shape
    if k_new.shape != (S, Hkv, N, d) or dc != d:
        raise ValueError("k_new / v_new must be [S, Hkv, N, d] matching q and the caches")
    if block_table.dim() != 2 or block_table.shape[0] != S:
        raise ValueError("block_table must be [S, max_blocks]")
    _need_shape("ctx_lens", ctx_lens, (S,))
    if scale is None:
        scale = d ** -0.5
    o = _output("o", o, q.shape, torch.bfloat16, dev)
    if lse is not None or return_lse:
        lse = _output("lse", lse, (S, Hq, N), torch.float32, dev)
    _call("attn_prefill_paged", dev, _ptr(q), _ptr(k_new), _ptr(v_new), _ptr(k_cache), _ptr(v_cache),
          _ptr(block_table), _ptr(ctx_lens), S, Hq, Hkv, N, d, block_size, block_table.shape[1],
          num_blocks, float(scale), _ptr(o), _ptr(lse), _stream_handle(stream, dev))
    return o, lse


def fused_add_rmsnorm(x, residual, weight, eps=1e-6, out=None, stream=None):
    """Residual add + RMSNorm.  x, residual [rows, hidden] and weight [hidden]
    bf16 on the GPU; ``residual`` is overwritten with bf16(x + residual).
    Returns (out [rows, hidden] bf16, residual)."""
    _need_cuda("x", x, torch.bfloat16)
    dev = x.device
    for name, t in (("residual", residual), ("weight", weight)):
        _need_cuda(name, t, torch.bfloat16, dev)
    if x.dim() != 2 or residual.shape != x.shape or weight.dim() != 1 or weight.shape[0] != x.shape[1]:
        raise ValueError("x and residual must be [rows, hidden] and weight [hidden]")
    rows, hidden = x.shape
    out = _output("out", out, x.shape, torch.bfloat16, dev)
    _call("fused_add_rmsnorm", dev, _ptr(x), _ptr(residual), _ptr(weight), _ptr(out), rows, hidden,
          float(eps), _stream_handle(stream, dev))
    return out, residual


def fused_swiglu(gate_up, out=None, stream=None):
    """SwiGLU activation of the merged gate/up projection output
    gate_up [rows, 2F] bf16 (gate first): returns silu(gate) * up [rows, F] bf16."""
    _need_cuda("gate_up", gate_up, torch.bfloat16)
    dev = gate_up.device
    if gate_up.dim() != 2 or gate_up.shape[1] % 2 != 0:
        raise ValueError("gate_up must be [rows, 2F]")
    rows, F = gate_up.shape[0], gate_up.shape[1] // 2
    out = _output("out", out, (rows, F), torch.bfloat16, dev)
    _call("fused_swiglu", dev, _ptr(gate_up), _ptr(out), rows, F, _stream_handle(stream, dev))
    return out


def swiglu_projection(x, w_gate_up, out=None, stream=None):
    """Gate/up projection with the SwiGLU activation fused in:
    x [rows, hidden] bf16, w_gate_up [2F, hidden] bf16 (gate rows first);
    returns silu(x W_gate^T) * (x W_up^T) [rows, F] bf16."""
    _need_cuda("x", x, torch.bfloat16)
    dev = x.device
    _need_cuda("w_gate_up", w_gate_up, torch.bfloat16, dev)
    if x.dim() != 2 or w_gate_up.dim() != 2 or w_gate_up.shape[1] != x.shape[1] or w_gate_up.shape[0] % 2:
        raise ValueError("x must be [rows, hidden] and w_gate_up [2F, hidden]")
    rows, hidden = x.shape
    F = w_gate_up.shape[0] // 2
    out = _output("out", out, (rows, F), torch.bfloat16, dev)
    _call("swiglu_projection", dev, _ptr(x), _ptr(w_gate_up), _ptr(out), rows, hidden, F,
          _stream_handle(stream, dev))
    return out


def ssd_workspace_size(batch, L, H, N, chunk):
    return int(load_library().ssd_workspace_size(batch, L, H, N, chunk))


def ssd_chunked_fwd(x, dt, A, B, C, chunk=256, h0=None, y=None, h_final=None, workspace=None,
                    stream=None):
    """Mamba-2 SSD forward.  x [batch, L, H, P] bf16, dt [batch, L, H] fp32,
    A [H] fp32, B and C [batch, L, G, N] bf16, h0 [batch, H, P, N] fp32 or
    None, all on the GPU.  Returns (y [batch, L, H, P] bf16, h_final
    [batch, H, P, N] fp32)."""
    _need_cuda("x", x, torch.bfloat16)
    dev = x.device
    for name, t, dtype in (("dt", dt, torch.float32), ("A", A, torch.float32),
                           ("B", B, torch.bfloat16), ("C", C, torch.bfloat16)):
        _need_cuda(name, t, dtype, dev)
    if x.dim() != 4 or dt.dim() != 3 or A.dim() != 1 or B.dim() != 4 or C.shape != B.shape:
        raise ValueError("x [batch, L, H, P], dt [batch, L, H], A [H], B/C [batch, L, G, N]")
    batch, L, H, P = x.shape
    G, N = B.shape[2], B.shape[3]
    if tuple(dt.shape) != (batch, L, H) or A.shape[0] != H or B.shape[:2] != x.shape[:2]:
        raise ValueError("dt, A, B and C do not match x")
    if h0 is not None:
        _need_cuda("h0", h0, torch.float32, dev)
        _need_shape("h0", h0, (batch, H, P, N))
    y = _output("y", y, x.shape, torch.bfloat16, dev)
    h_final = _output("h_final", h_final, (batch, H, P, N), torch.float32, dev)
    workspace = _workspace("workspace", workspace, ssd_workspace_size(batch, L, H, N, chunk), dev)
    _call("ssd_chunked_fwd", dev, _ptr(x), _ptr(dt), _ptr(A), _ptr(B), _ptr(C), _ptr(h0), _ptr(y),
          _ptr(h_final), batch, L, H, G, P, N, chunk, _ptr(workspace),
          workspace.numel() * workspace.element_size(), _stream_handle(stream, dev))
    return y, h_final


def device_status(stream=None):
    """Read and clear the device status word (ATTN_DEV_* bits)."""
    flags = ctypes.c_uint(0)
    _check("attn_get_device_status",
           load_library().attn_get_device_status(_stream_handle(stream), ctypes.byref(flags)))
    return int(flags.value)


def set_wait_timeout_ns(ns):
    load_library().attn_set_wait_timeout_ns(int(ns))


def set_decode_max_ctas(ctas):
    """Cap the CTAs of a decode launch (0: one full wave)."""
    load_library().attn_set_decode_max_ctas(int(ctas))


def set_decode_early_plan(on):
    """Let later decode calls read seq_lens and block_table (``on`` = 1 or
    True), and also the first cache blocks of each CTA's share except a
    sequence's last block (``on`` = 2), before the preceding kernel in the
    stream has finished; the caller guarantees that kernel writes none of
    them.  0 or False: read nothing before it has finished."""
    level = int(on)
    load_library().attn_set_decode_early_plan(0 if level <= 0 else 2 if level >= 2 else 1)


def selftest_exp2_poly(x, y=None, stream=None):
    """y = 2^x (fp32 CUDA tensors) by the forward softmax's FMA-pipe exp2."""
    _need_cuda("x", x, torch.float32)
    dev = x.device
    y = _output("y", y, x.shape, torch.float32, dev)
    _call("attn_selftest_exp2_poly", dev, _ptr(x), _ptr(y), x.numel(), _stream_handle(stream, dev))
    return y


def selftest_wait_timeout(timeout_ns, stream=None):
    flags = ctypes.c_uint(0)
    _check("attn_selftest_wait_timeout",
           load_library().attn_selftest_wait_timeout(int(timeout_ns), _stream_handle(stream),
                                                     ctypes.byref(flags)))
    return int(flags.value)


def abi_version():
    return int(load_library().attn_abi_version())
