"""Argument checks of the tensor-level binding `attention()`: every one runs on the host
before any device is touched, so they are checked here on CPU tensors."""
import pytest
import torch

import exact_attention_forward_02_gb300 as fa


def _qkv(B=1, H=2, Nq=5, Nk=7, d=64, dtype=torch.float16):
    return (torch.zeros(B, H, Nq, d, dtype=dtype), torch.zeros(B, H, Nk, d, dtype=dtype),
            torch.zeros(B, H, Nk, d, dtype=dtype))


def test_rejects_unsupported_and_mixed_dtypes():
    q, k, v = _qkv(dtype=torch.float32)
    with pytest.raises(TypeError):
        fa.attention(q, k, v)
    q, k, v = _qkv()
    with pytest.raises(TypeError):
        fa.attention(q, k.to(torch.bfloat16), v)


def test_rejects_bad_shapes():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match=r"\[B, H, N, d\]"):
        fa.attention(q[0], k, v)
    with pytest.raises(ValueError, match="k and v"):
        fa.attention(q, k[:, :1], v)
    with pytest.raises(ValueError, match="k and v"):
        fa.attention(q, k, v[..., :32])


@pytest.mark.parametrize("bad_out", [
    torch.zeros(1, 2, 5, 32, dtype=torch.float16),            # wrong d
    torch.zeros(1, 2, 5, 64, dtype=torch.bfloat16),           # wrong dtype
    torch.zeros(1, 2, 64, 5, dtype=torch.float16).transpose(2, 3),  # not contiguous
])
def test_rejects_a_bad_output_buffer(bad_out):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="out must be"):
        fa.attention(q, k, v, out=bad_out)


@pytest.mark.parametrize("bad_lse", [
    torch.zeros(1, 2, 4, dtype=torch.float32),   # too short
    torch.zeros(1, 2, 5, dtype=torch.float64),   # wrong dtype
])
def test_rejects_a_bad_lse_buffer(bad_lse):
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="lse must be"):
        fa.attention(q, k, v, lse=bad_lse)


def test_rejects_a_bad_workspace_and_host_tensors():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="workspace must be"):
        fa.attention(q, k, v, workspace=torch.zeros(256, dtype=torch.float32))
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.attention(q, k, v)
    with pytest.raises(ValueError, match="CUDA tensors"):
        fa.attention(q, k, v, out=torch.zeros(1, 2, 5, 64, dtype=torch.float16),
                     lse=torch.zeros(1, 2, 5, dtype=torch.float32),
                     workspace=torch.zeros(256, dtype=torch.uint8))
