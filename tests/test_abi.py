"""The C-ABI library loads, exports every function ``include/attn47.h``
declares, and rejects bad arguments on the host before touching a device.

These run without a GPU: no call here launches a kernel.  Pointers passed
to calls that must fail validation are never dereferenced.
"""

import ctypes
import os
import re

import pytest

import exact_attention_47_gb300 as attn
from exact_attention_47_gb300 import _binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "attn47.h")

OK, INVALID, UNSUPPORTED, DEVICE, LAUNCH, WORKSPACE = 0, 1, 2, 3, 4, 5
FAKE = ctypes.c_void_p(0x10000)  # aligned, never dereferenced on these paths


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b((?:attn|fused|ssd)_[a-z_0-9]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(attn.library_path()):
        import __graft_entry__
        __graft_entry__.build()
    return attn.load_library()


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("attn_fwd", "attn_bwd", "attn_decode_paged", "attn_decode_paged_workspace_size",
                     "attn_prefill_paged", "fused_add_rmsnorm", "fused_swiglu",
                     "attn_get_device_status", "attn_status_string"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in _binding._SIGS, "binding lacks " + name


def test_abi_version_and_status_strings(lib):
    assert attn.abi_version() == 2
    assert attn.status_string(0) == "ATTN_OK"
    assert attn.status_string(5) == "ATTN_ERR_WORKSPACE"


def _fwd(lib, B=1, Hq=2, Hkv=2, N=16, d=64, causal=1, scale=0.125, q=FAKE, o=FAKE):
    return lib.attn_fwd(q, FAKE, FAKE, o, None, B, Hq, Hkv, N, d, causal, scale, None)


def test_fwd_host_validation(lib):
    assert _fwd(lib, d=96) == UNSUPPORTED
    assert _fwd(lib, Hq=3, Hkv=2) == INVALID
    assert _fwd(lib, N=-1) == INVALID
    assert _fwd(lib, scale=0.0) == INVALID
    assert _fwd(lib, scale=float("nan")) == INVALID
    assert _fwd(lib, q=ctypes.c_void_p(0x10008)) == INVALID      # misaligned
    assert _fwd(lib, o=ctypes.c_void_p(0)) == INVALID            # null output
    assert "aligned" in lib.attn_last_error().decode() or "null" in lib.attn_last_error().decode()
    assert _fwd(lib, B=0) == OK                                  # empty problem
    assert _fwd(lib, N=0) == OK


def _dec(lib, S=2, Hq=12, Hkv=2, d=128, bs=16, mb=4, nb=8, ws_bytes=None, ws=FAKE):
    need = lib.attn_decode_paged_workspace_size(S, Hq, d, mb)
    if ws_bytes is None:
        ws_bytes = need
    return lib.attn_decode_paged(FAKE, FAKE, FAKE, FAKE, FAKE, S, Hq, Hkv, d, bs, mb, nb, 0.1,
                                 FAKE, None, ws, ws_bytes, None)


def test_decode_host_validation(lib):
    assert _dec(lib, bs=8) == UNSUPPORTED
    assert _dec(lib, d=80) == UNSUPPORTED
    assert _dec(lib, Hq=34, Hkv=2) == UNSUPPORTED               # group of 17
    assert _dec(lib, Hq=12, Hkv=5) == INVALID
    assert _dec(lib, ws_bytes=16) == WORKSPACE
    assert _dec(lib, ws=ctypes.c_void_p(0)) == INVALID
    assert _dec(lib, S=0) == OK


def _pre(lib, S=2, Hq=12, Hkv=2, N=64, d=128, bs=16, mb=8, nb=16, q=FAKE, kc=FAKE):
    return lib.attn_prefill_paged(q, FAKE, FAKE, kc, FAKE, FAKE, FAKE, S, Hq, Hkv, N, d, bs, mb, nb,
                                  0.1, FAKE, None, None)


def test_prefill_paged_host_validation(lib):
    assert _pre(lib, bs=32) == UNSUPPORTED
    assert _pre(lib, d=96) == UNSUPPORTED
    assert _pre(lib, Hq=12, Hkv=5) == INVALID
    assert _pre(lib, N=-1) == INVALID
    assert _pre(lib, N=129, mb=8) == INVALID                    # 129 new tokens > 8 blocks
    assert _pre(lib, kc=ctypes.c_void_p(0)) == INVALID
    assert _pre(lib, q=ctypes.c_void_p(0x10004)) == INVALID     # misaligned
    assert _pre(lib, S=0) == OK
    assert _pre(lib, N=0) == OK


def test_fusion_host_validation(lib):
    assert lib.fused_add_rmsnorm(FAKE, ctypes.c_void_p(0x20000), FAKE, ctypes.c_void_p(0x30000), 4, 12, 1e-6, None) == UNSUPPORTED
    assert lib.fused_add_rmsnorm(FAKE, ctypes.c_void_p(0x20000), FAKE, ctypes.c_void_p(0x30000), 4, 16, -1.0, None) == INVALID
    assert lib.fused_add_rmsnorm(FAKE, FAKE, ctypes.c_void_p(0x20000), ctypes.c_void_p(0x30000), 4, 16, 1e-6, None) == INVALID  # x is residual
    assert lib.fused_add_rmsnorm(FAKE, ctypes.c_void_p(0x20000), FAKE, ctypes.c_void_p(0x20010), 4, 16, 1e-6, None) == INVALID  # out overlaps residual
    assert lib.fused_add_rmsnorm(FAKE, FAKE, FAKE, FAKE, 0, 16, 1e-6, None) == OK
    assert lib.fused_swiglu(FAKE, ctypes.c_void_p(0x40000), 4, 12, None) == UNSUPPORTED
    assert lib.fused_swiglu(FAKE, ctypes.c_void_p(0x10040), 4, 16, None) == INVALID              # out inside gate_up
    assert lib.fused_swiglu(ctypes.c_void_p(0x10008), ctypes.c_void_p(0x40000), 4, 16, None) == INVALID
    assert lib.fused_swiglu(FAKE, FAKE, 0, 16, None) == OK


def test_swiglu_projection_host_validation(lib):
    out = ctypes.c_void_p(0x400000)
    assert lib.swiglu_projection(FAKE, ctypes.c_void_p(0x200000), out, 4, 96, 128, None) == UNSUPPORTED  # hidden
    assert lib.swiglu_projection(FAKE, ctypes.c_void_p(0x200000), out, 4, 64, 96, None) == UNSUPPORTED   # F
    assert lib.swiglu_projection(FAKE, ctypes.c_void_p(0x200000), FAKE, 4, 64, 128, None) == INVALID     # out is x
    assert lib.swiglu_projection(FAKE, ctypes.c_void_p(0x200008), out, 4, 64, 128, None) == INVALID      # misaligned
    assert lib.swiglu_projection(FAKE, None, out, 4, 64, 128, None) == INVALID
    assert lib.swiglu_projection(FAKE, FAKE, FAKE, 0, 64, 128, None) == OK


def test_selftest_exp2_poly_host_validation(lib):
    assert lib.attn_selftest_exp2_poly(FAKE, FAKE, -1, None) == INVALID
    assert lib.attn_selftest_exp2_poly(None, FAKE, 4, None) == INVALID
    assert lib.attn_selftest_exp2_poly(FAKE, ctypes.c_void_p(0x10002), 4, None) == INVALID   # misaligned
    assert lib.attn_selftest_exp2_poly(FAKE, FAKE, 0, None) == OK


def _ssd(lib, batch=2, L=100, H=8, G=1, P=64, N=128, chunk=64, ws_bytes=None):
    need = lib.ssd_workspace_size(batch, L, H, N, chunk)
    return lib.ssd_chunked_fwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, batch, L, H, G, P, N,
                               chunk, FAKE, need if ws_bytes is None else ws_bytes, None)


def test_ssd_host_validation(lib):
    assert _ssd(lib, P=128) == UNSUPPORTED
    assert _ssd(lib, N=96) == UNSUPPORTED
    assert _ssd(lib, chunk=100) == UNSUPPORTED
    assert _ssd(lib, H=6, G=4) == INVALID
    assert _ssd(lib, ws_bytes=16) == WORKSPACE
    assert _ssd(lib, L=0) == OK
    # decays (batch*H*n_chunks*chunk fp32, padded to 256 bytes) + initial states (bf16)
    assert lib.ssd_workspace_size(2, 100, 8, 128, 64) == 2 * 8 * 2 * 64 * 4 + 2 * 2 * 8 * 64 * 128 * 2


def test_workspace_size_formula(lib):
    # fp32 partial O (d floats) + max and sum per (seq, head, part) with at
    # most ceil(256 / 16) + 1 parts, plus 8 bytes per (seq, head) reserved
    # for the part counts
    assert lib.attn_decode_paged_workspace_size(64, 12, 128, 256) == 64 * 12 * 17 * 130 * 4 + 64 * 12 * 8
    assert lib.attn_decode_paged_workspace_size(0, 12, 128, 256) == 0


def test_binding_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(_binding, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _binding.load_library(str(tmp_path / "missing.so"))


def test_decode_workspace_must_not_overlap_other_buffers(lib):
    S, Hq, d, mb = 2, 12, 128, 4
    need = lib.attn_decode_paged_workspace_size(S, Hq, d, mb)
    ws = ctypes.c_void_p(0x100000)
    q, o = ctypes.c_void_p(0x200000), ctypes.c_void_p(0x300000)
    lse = ctypes.c_void_p(0x400000)

    def call(q_=q, o_=o, lse_=lse, ws_=ws):
        return lib.attn_decode_paged(q_, FAKE, FAKE, ctypes.c_void_p(0x500000), ctypes.c_void_p(0x600000),
                                     S, Hq, 2, d, 16, mb, 8, 0.1, o_, lse_, ws_, need, None)

    assert call(o_=ctypes.c_void_p(0x100000 + 1024)) == INVALID      # o inside the workspace
    assert "overlaps" in lib.attn_last_error().decode()
    assert call(lse_=ctypes.c_void_p(0x100000 + need - 16)) == INVALID
    assert call(q_=ctypes.c_void_p(0x100000 - 1024)) == INVALID      # q runs into the workspace
    assert call(ws_=FAKE) == INVALID                                 # the caches start at FAKE


def _noalloc(lib, S=2, Hq=12, Hkv=2, d=128, bs=16, mb=4, nb=8):
    return lib.attn_decode_paged_noalloc(FAKE, FAKE, FAKE, FAKE, FAKE, S, Hq, Hkv, d, bs, mb, nb, 0.1,
                                         FAKE, None, None)


def test_noalloc_checks_arguments_like_the_workspace_entry_point(lib):
    # The argument checks come before the scratch size: the same bad
    # arguments give the same status from both decode entry points.
    for kw, want in ((dict(bs=8), UNSUPPORTED), (dict(d=80), UNSUPPORTED), (dict(Hq=34, Hkv=2), UNSUPPORTED),
                     (dict(Hq=12, Hkv=5), INVALID), (dict(mb=0), INVALID), (dict(S=-1), INVALID),
                     (dict(mb=2 ** 31 - 1), UNSUPPORTED), (dict(S=0), OK)):
        assert _noalloc(lib, **kw) == want, kw
        assert _dec(lib, **kw) == want, kw
    # Valid arguments whose scratch exceeds the built-in 8 MiB array.
    assert _noalloc(lib, S=64, Hq=12, mb=4096) == WORKSPACE
    assert "8388608" in lib.attn_last_error().decode()


def test_decode_workspace_size_has_no_overflow(lib):
    # ceil(max_blocks / 16) + 1 parts per (sequence, head), computed in 64 bits
    parts = (2 ** 31 - 1 + 15) // 16 + 1
    assert lib.attn_decode_paged_workspace_size(1, 1, 128, 2 ** 31 - 1) == parts * 130 * 4 + 8
