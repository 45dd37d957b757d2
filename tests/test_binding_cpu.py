"""The Python binding has no CPU path: host tensors are refused before anything reaches the
library, and a missing library is an import error, not a silent fallback."""
import pytest
import torch

import exact_io_aware_23_gb300 as fa


def _qkv(B=1, H=2, N=64, d=64, dtype=torch.bfloat16):
    return [torch.zeros(B, H, N, d, dtype=dtype) for _ in range(3)]


def test_forward_refuses_host_tensors():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.forward(q, k, v)


def test_backward_refuses_host_tensors():
    q, k, v = _qkv()
    lse = torch.zeros(1, 2, 64, dtype=torch.float32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.backward(q, k, v, q, lse, q)


def test_varlen_refuses_host_tensors():
    q = torch.zeros(2, 100, 64, dtype=torch.bfloat16)
    cu = torch.tensor([0, 40, 100], dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.forward_varlen(q, q, q, cu, 60)


def test_splitkv_refuses_host_tensors():
    q = torch.zeros(1, 2, 16, 128, dtype=torch.bfloat16)
    k = torch.zeros(1, 2, 1024, 128, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fa.forward_splitkv(q, k, k)


def test_missing_library_is_an_import_error(monkeypatch, tmp_path):
    monkeypatch.setattr(fa, "LIB_PATH", str(tmp_path / "libfa.so"))
    with pytest.raises(ImportError, match="not built"):
        fa._load()
