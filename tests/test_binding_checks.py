"""The Python binding refuses wrong tensors before anything reaches the
library: host tensors, wrong dtypes, wrong shapes, undersized workspaces.

These run without a GPU.  The tensors are CPU tensors of a subclass that
reports itself as living on cuda:0, so the binding's device checks pass for
them and its other checks are the ones exercised; a plain CPU tensor plays
the host buffer.  The library's compute entry points are replaced by a
function that fails the test, so a check that let a bad tensor through
shows up as a failure here instead of a launch.
"""

import pytest
import torch

import exact_attention_47_gb300 as attn
from exact_attention_47_gb300 import _binding

BF, F32, I32 = torch.bfloat16, torch.float32, torch.int32


class _OnCuda0(torch.Tensor):
    """A CPU tensor that claims to be on cuda:0 (its data never reaches the
    library in these tests)."""

    @property
    def is_cuda(self):
        return True

    @property
    def device(self):
        return torch.device("cuda", 0)


def dev(shape, dtype):
    return torch.Tensor._make_subclass(_OnCuda0, torch.zeros(shape, dtype=dtype))


@pytest.fixture(autouse=True)
def no_library_calls(monkeypatch):
    def refuse(func, device, *args):
        raise AssertionError("%s reached the library with bad arguments" % func)

    monkeypatch.setattr(_binding, "_call", refuse)


def decode_args(S=3, Hq=12, Hkv=2, d=128, nb=20, mb=5):
    return dict(q=dev((S, Hq, d), BF), k_cache=dev((nb, Hkv, 16, d), BF),
                v_cache=dev((nb, Hkv, 16, d), BF), block_table=dev((S, mb), I32),
                seq_lens=dev((S,), I32))


def good_outputs(S=3, Hq=12, d=128):
    return dict(o=dev((S, Hq, d), BF), lse=dev((S, Hq), F32))


@pytest.mark.parametrize("entry", ["attn_decode_paged", "attn_decode_paged_noalloc"])
@pytest.mark.parametrize("bad,match", [
    (dict(o=dev((3, 12, 64), BF)), "o must have shape"),
    (dict(o=dev((3, 12, 128), F32)), "o must be torch.bfloat16"),
    (dict(o=torch.zeros((3, 12, 128), dtype=BF)), "o must be a CUDA tensor"),
    (dict(lse=dev((3, 11), F32)), "lse must have shape"),
    (dict(lse=dev((3, 12), BF)), "lse must be torch.float32"),
    (dict(lse=torch.zeros((3, 12), dtype=F32)), "lse must be a CUDA tensor"),
])
def test_decode_outputs_are_checked(entry, bad, match):
    kw = dict(good_outputs(), **bad)
    with pytest.raises(ValueError, match=match):
        getattr(attn, entry)(**decode_args(), **kw)


@pytest.mark.parametrize("entry", ["attn_decode_paged", "attn_decode_paged_noalloc"])
@pytest.mark.parametrize("bad,match", [
    (dict(k_cache=dev((20, 2, 16, 64), BF), v_cache=dev((20, 2, 16, 64), BF)), "cache head dim"),
    (dict(block_table=dev((2, 5), I32)), "block_table must be"),
    (dict(block_table=dev((3,), I32)), "block_table must be"),
    (dict(seq_lens=dev((4,), I32)), "seq_lens must have shape"),
    (dict(seq_lens=dev((3,), torch.int64)), "seq_lens must be torch.int32"),
    (dict(v_cache=dev((21, 2, 16, 128), BF)), "caches"),
    (dict(q=torch.zeros((3, 12, 128), dtype=BF)), "q must be a CUDA tensor"),
])
def test_decode_inputs_are_checked(entry, bad, match):
    args = dict(decode_args(), **bad)
    with pytest.raises(ValueError, match=match):
        getattr(attn, entry)(**args, **good_outputs())


def test_decode_workspace_is_checked():
    args = decode_args()
    need = attn.attn_decode_paged_workspace_size(3, 12, 128, 5)
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        attn.attn_decode_paged(**args, **good_outputs(), workspace=torch.zeros(need, dtype=torch.uint8))
    with pytest.raises(ValueError, match="workspace has %d bytes, needs %d" % (need - 16, need)):
        attn.attn_decode_paged(**args, **good_outputs(), workspace=dev((need - 16,), torch.uint8))
    with pytest.raises(ValueError, match="workspace must be contiguous"):
        attn.attn_decode_paged(**args, **good_outputs(), workspace=dev((2 * need,), torch.uint8)[::2])


def test_fwd_outputs_are_checked():
    q, k = dev((1, 4, 64, 128), BF), dev((1, 2, 64, 128), BF)
    with pytest.raises(ValueError, match="o must be a CUDA tensor"):
        attn.attn_fwd(q, k, k, o=torch.zeros((1, 4, 64, 128), dtype=BF), lse=dev((1, 4, 64), F32))
    with pytest.raises(ValueError, match="lse must have shape"):
        attn.attn_fwd(q, k, k, o=dev((1, 4, 64, 128), BF), lse=dev((1, 4, 63), F32))
    with pytest.raises(ValueError, match="o must have shape"):
        attn.attn_fwd(q, k, k, o=dev((1, 4, 64, 64), BF), lse=dev((1, 4, 64), F32))


def test_bwd_buffers_are_checked():
    q, k = dev((1, 4, 64, 128), BF), dev((1, 2, 64, 128), BF)
    lse = dev((1, 4, 64), F32)
    outs = dict(dq=dev(q.shape, BF), dk=dev(k.shape, BF), dv=dev(k.shape, BF))
    need = attn.attn_bwd_workspace_size(1, 4, 64)
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        attn.attn_bwd(q, k, k, q, lse, q, **outs, workspace=torch.zeros(need, dtype=torch.uint8))
    with pytest.raises(ValueError, match="workspace has"):
        attn.attn_bwd(q, k, k, q, lse, q, **outs, workspace=dev((need - 4,), torch.uint8))
    with pytest.raises(ValueError, match="dk must have shape"):
        attn.attn_bwd(q, k, k, q, lse, q, dq=outs["dq"], dk=dev(q.shape, BF), dv=outs["dv"],
                      workspace=dev((need,), torch.uint8))


def test_prefill_paged_outputs_are_checked():
    S, Hq, Hkv, N, d = 2, 4, 2, 32, 128
    args = (dev((S, Hq, N, d), BF), dev((S, Hkv, N, d), BF), dev((S, Hkv, N, d), BF),
            dev((10, Hkv, 16, d), BF), dev((10, Hkv, 16, d), BF), dev((S, 5), I32), dev((S,), I32))
    with pytest.raises(ValueError, match="lse must have shape"):
        attn.attn_prefill_paged(*args, o=dev((S, Hq, N, d), BF), lse=dev((S, Hq), F32))
    with pytest.raises(ValueError, match="ctx_lens must have shape"):
        attn.attn_prefill_paged(*args[:6], dev((S + 1,), I32), o=dev((S, Hq, N, d), BF), lse=dev((S, Hq, N), F32))


def test_ssd_buffers_are_checked():
    b, L, H, P, G, N = 1, 64, 2, 64, 1, 64
    args = (dev((b, L, H, P), BF), dev((b, L, H), F32), dev((H,), F32), dev((b, L, G, N), BF),
            dev((b, L, G, N), BF))
    good = dict(y=dev((b, L, H, P), BF), h_final=dev((b, H, P, N), F32))
    need = attn.ssd_workspace_size(b, L, H, N, 64)
    with pytest.raises(ValueError, match="workspace must be a CUDA tensor"):
        attn.ssd_chunked_fwd(*args, chunk=64, **good, workspace=torch.zeros(need, dtype=torch.uint8))
    with pytest.raises(ValueError, match="y must have shape"):
        attn.ssd_chunked_fwd(*args, chunk=64, y=dev((b, L, H, 32), BF), h_final=good["h_final"],
                             workspace=dev((need,), torch.uint8))
    with pytest.raises(ValueError, match="h_final must be torch.float32"):
        attn.ssd_chunked_fwd(*args, chunk=64, y=good["y"], h_final=dev((b, H, P, N), BF),
                             workspace=dev((need,), torch.uint8))


def test_fusion_outputs_are_checked():
    x, w = dev((4, 64), BF), dev((64,), BF)
    with pytest.raises(ValueError, match="out must have shape"):
        attn.fused_add_rmsnorm(x, dev((4, 64), BF), w, out=dev((4, 32), BF))
    with pytest.raises(ValueError, match="out must be a CUDA tensor"):
        attn.fused_swiglu(dev((4, 64), BF), out=torch.zeros((4, 32), dtype=BF))
