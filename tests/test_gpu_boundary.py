"""The C-ABI refuses buffers that are not memory of the current device, and
buffers that run past the end of their allocation, before any launch.

The host buffers here are pinned, which the GPU can reach through unified
addressing: if a check let one through, the kernel would touch host memory
rather than fault.  The overrun case asks for bytes beyond a freshly made
allocation, and also passes a pinned host buffer as a second operand, so a
missing range check shows up as the other refusal, never as a launch.
"""

import ctypes

import pytest
import torch

import exact_attention_47_gb300 as attn

pytestmark = pytest.mark.gpu
DEV = "cuda:0"
INVALID = 1


def _lib():
    return attn.load_library()


def _p(t):
    return ctypes.c_void_p(t.data_ptr())


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def test_fwd_refuses_a_host_output():
    q = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16, device=DEV)
    o_host = torch.zeros(1, 2, 128, 64, dtype=torch.bfloat16).pin_memory()
    lib = _lib()
    st = lib.attn_fwd(_p(q), _p(q), _p(q), _p(o_host), None, 1, 2, 2, 128, 64, 1, 0.125, _stream())
    assert st == INVALID
    assert "o (" in lib.attn_last_error().decode()
    assert "not memory of device" in lib.attn_last_error().decode()


def test_decode_refuses_a_host_workspace():
    q = torch.zeros(2, 12, 128, dtype=torch.bfloat16, device=DEV)
    kc = torch.zeros(8, 2, 16, 128, dtype=torch.bfloat16, device=DEV)
    table = torch.zeros(2, 4, dtype=torch.int32, device=DEV)
    lens = torch.ones(2, dtype=torch.int32, device=DEV)
    o = torch.empty_like(q)
    lib = _lib()
    need = lib.attn_decode_paged_workspace_size(2, 12, 128, 4)
    ws_host = torch.zeros(need, dtype=torch.uint8).pin_memory()
    st = lib.attn_decode_paged(_p(q), _p(kc), _p(kc), _p(table), _p(lens), 2, 12, 2, 128, 16, 4, 8,
                               0.1, _p(o), None, _p(ws_host), need, _stream())
    assert st == INVALID
    assert "workspace (" in lib.attn_last_error().decode()


def test_swiglu_refuses_a_host_input():
    lib = _lib()
    out = torch.empty(4, 64, dtype=torch.bfloat16, device=DEV)
    gu_host = torch.zeros(4, 128, dtype=torch.bfloat16).pin_memory()
    assert lib.fused_swiglu(_p(gu_host), _p(out), 4, 64, _stream()) == INVALID
    assert "gate_up (" in lib.attn_last_error().decode()


def test_fwd_refuses_an_overrun():
    # q in an allocation of its own (2 MiB) while the sizes claim 1 GiB of it
    # (B 1, H 16, N 262144, d 128); o is a pinned host buffer, refused by the
    # memory-type check if the range check did not catch q first.
    lib = _lib()
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    q = torch.zeros(2 << 20, dtype=torch.uint8, device=DEV)
    o_host = torch.zeros(16, dtype=torch.bfloat16).pin_memory()
    st = lib.attn_fwd(_p(q), _p(q), _p(q), _p(o_host), None, 1, 16, 16, 262144, 128, 1, 0.088,
                      _stream())
    assert st == INVALID
    msg = lib.attn_last_error().decode()
    assert "q:" in msg and "past the end of its allocation" in msg, msg
    torch.cuda.synchronize()
    assert attn.device_status() == 0
