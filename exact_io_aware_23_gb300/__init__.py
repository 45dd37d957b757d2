"""Python binding of libfa, the exact-attention C ABI (include/fa.h), for GB300 (sm_103a).

This module only marshals arguments: it checks tensor placement, dtype and shape, passes raw
device pointers and the current CUDA stream to the C functions, and turns a non-OK status into
an exception.  Every step of the computation runs in the library's CUDA kernels.  Importing
fails loudly when the library has not been built (``__graft_entry__.build()``); there is no
fallback implementation.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

__all__ = ["forward", "forward_splitkv", "backward", "backward_noalloc", "backward_workspace_size",
           "backward_fused_workspace_size", "check_device_status", "set_fault_injection",
           "set_wait_limit_ms", "FaError", "LIB_PATH", "lib"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libfa.so")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_TIMEOUT = range(5)
FA_BF16, FA_FP32, FA_FP16 = 0, 1, 2
_DTYPES = {torch.bfloat16: FA_BF16, torch.float32: FA_FP32, torch.float16: FA_FP16}


class FaDropout(ctypes.Structure):
    """fa_dropout: dropout probability, generator key and counter offset."""
    _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint32)]


class FaError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {lib.fa_status_string(status).decode()}")


def _load() -> ctypes.CDLL:
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"libfa.so is not built ({LIB_PATH}); run __graft_entry__.build()")
    L = ctypes.CDLL(LIB_PATH)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_forward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, vp]
    L.fa_forward.restype = i
    L.fa_backward_workspace_size.argtypes = [i, i, i, i]
    L.fa_backward_workspace_size.restype = sz
    L.fa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp,
                              vp, sz, vp]
    L.fa_backward.restype = i
    L.fa_check_device_status.argtypes = [vp]
    L.fa_check_device_status.restype = i
    L.fa_status_string.argtypes = [i]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_debug_set_fault_injection.argtypes = [i]
    L.fa_debug_set_fault_injection.restype = None
    L.fa_debug_set_wait_limit_ms.argtypes = [ctypes.c_uint32]
    L.fa_debug_set_wait_limit_ms.restype = None
    L.fa_version.argtypes = []
    L.fa_version.restype = i
    L.fa_forward_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, vp]
    L.fa_forward_gqa.restype = i
    L.fa_forward_blocksparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, vp, sz, vp]
    L.fa_forward_blocksparse.restype = i
    L.fa_forward_blocksparse_workspace_size.argtypes = [i, i, i, i]
    L.fa_forward_blocksparse_workspace_size.restype = sz
    L.fa_backward_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i,
                                  vp, vp, sz, vp]
    L.fa_backward_gqa.restype = i
    L.fa_backward_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                            i, vp, i, vp, vp, sz, vp]
    L.fa_backward_deterministic.restype = i
    L.fa_backward_deterministic_workspace_size.argtypes = [i, i, i]
    L.fa_backward_deterministic_workspace_size.restype = sz
    L.fa_forward_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    L.fa_forward_varlen.restype = i
    L.fa_backward_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                     i, i, vp, sz, vp]
    L.fa_backward_varlen.restype = i
    dp = ctypes.POINTER(FaDropout)
    L.fa_forward_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, dp, vp]
    L.fa_forward_dropout.restype = i
    L.fa_backward_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i,
                                      vp, dp, vp, sz, vp]
    L.fa_backward_dropout.restype = i
    L.fa_backward_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i,
                                    vp, vp, sz, vp]
    L.fa_backward_fused.restype = i
    L.fa_backward_fused_workspace_size.argtypes = [i, i, i, i]
    L.fa_backward_fused_workspace_size.restype = sz
    L.fa_forward_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, i, i, vp, sz, vp]
    L.fa_forward_splitkv_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, i, i, vp, sz, vp]
    L.fa_forward_splitkv_gqa.restype = i
    L.fa_forward_splitkv.restype = i
    L.fa_forward_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_forward_splitkv_workspace_size.restype = sz
    L.fa_forward_splitkv_auto_splits.argtypes = [i, i, i, i]
    L.fa_forward_splitkv_auto_splits.restype = i
    L.fa_backward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i,
                                      vp, vp]
    L.fa_backward_noalloc.restype = i
    L.fa_backward_noalloc_max_workspace.argtypes = []
    L.fa_backward_noalloc_max_workspace.restype = sz
    return L


lib = _load()


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _check_qkv(q, k, v):
    """q: [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H (grouped-query attention when
    Hkv < H).  Returns (B, H, N, d, Hkv)."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor")
        if t.dim() != 4:
            raise ValueError(f"{name} must be [B, H, N, d]")
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    if k.shape != v.shape or k.shape[0] != B or k.shape[2:] != q.shape[2:] or H % Hkv != 0:
        raise ValueError("k, v must be [B, Hkv, N, d] with Hkv dividing the query heads")
    if not (q.dtype == k.dtype == v.dtype):
        raise ValueError("q, k, v must share a dtype")
    if q.dtype not in _DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    return B, H, N, d, Hkv


def _masks(block_mask, kv_lens, B, N, device):
    if block_mask is not None:
        T = (N + 127) // 128
        if block_mask.dtype != torch.uint8 or tuple(block_mask.shape) != (T, T):
            raise ValueError(f"block_mask must be uint8 [{T}, {T}]")
        block_mask = block_mask.to(device).contiguous()
    if kv_lens is not None:
        if kv_lens.dtype != torch.int32 or tuple(kv_lens.shape) != (B,):
            raise ValueError(f"kv_lens must be int32 [{B}]")
        kv_lens = kv_lens.to(device).contiguous()
    return block_mask, kv_lens


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *, causal: bool = False,
            scale: Optional[float] = None, block_mask: Optional[torch.Tensor] = None,
            kv_lens: Optional[torch.Tensor] = None, o: Optional[torch.Tensor] = None,
            lse: Optional[torch.Tensor] = None, stream=None, dropout_p: float = 0.0,
            seed: int = 0, offset: int = 0, balanced: bool = True,
            workspace: Optional[torch.Tensor] = None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE = attention forward (fa_forward; fa_forward_gqa when k, v have fewer heads;
    fa_forward_dropout when dropout_p > 0; with a block mask and 16-bit inputs,
    fa_forward_blocksparse unless balanced=False).  q: [B, H, N, d]; k, v: [B, Hkv, N, d];
    bf16, fp16 or fp32 on CUDA."""
    B, H, N, d, Hkv = _check_qkv(q, k, v)
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    block_mask, kv_lens = _masks(block_mask, kv_lens, B, N, q.device)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device) if lse is None else lse
    if dropout_p > 0.0:
        drop = FaDropout(float(dropout_p), int(seed), int(offset))
        st = lib.fa_forward_dropout(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                    scale, int(bool(causal)), _ptr(block_mask), _DTYPES[q.dtype],
                                    _ptr(kv_lens), ctypes.byref(drop), _stream(stream))
        if st != FA_OK:
            raise FaError(st, "fa_forward_dropout")
        return o, lse
    if block_mask is not None and balanced and q.dtype != torch.float32:
        need = int(lib.fa_forward_blocksparse_workspace_size(B, H, N, d))
        if workspace is None:
            workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
        st = lib.fa_forward_blocksparse(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N,
                                        d, scale, int(bool(causal)), _ptr(block_mask),
                                        _DTYPES[q.dtype], _ptr(kv_lens), _ptr(workspace),
                                        workspace.numel() * workspace.element_size(), _stream(stream))
        if st != FA_OK:
            raise FaError(st, "fa_forward_blocksparse")
        return o, lse
    if Hkv == H:
        st = lib.fa_forward(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, N, d, scale,
                            int(bool(causal)), _ptr(block_mask), _DTYPES[q.dtype], _ptr(kv_lens),
                            _stream(stream))
    else:
        st = lib.fa_forward_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, N, d,
                                scale, int(bool(causal)), _ptr(block_mask), _DTYPES[q.dtype],
                                _ptr(kv_lens), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_forward")
    return o, lse


def _check_packed(q, k, v, cu_seqlens):
    """q: [H, total, d]; k, v: [Hkv, total, d]; cu_seqlens: int32 [n_seqs + 1] on q's device."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 3:
            raise ValueError(f"{name} must be a contiguous CUDA tensor [heads, total, d]")
    H, T, d = q.shape
    Hkv = k.shape[0]
    if k.shape != v.shape or k.shape[1:] != q.shape[1:] or H % Hkv != 0:
        raise ValueError("k, v must be [Hkv, total, d] with Hkv dividing the query heads")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, k, v must share a supported dtype")
    if (cu_seqlens.dtype != torch.int32 or cu_seqlens.dim() != 1 or cu_seqlens.numel() < 1
            or cu_seqlens.device != q.device or not cu_seqlens.is_contiguous()):
        raise ValueError("cu_seqlens must be a contiguous int32 [n_seqs + 1] tensor on q's device")
    return H, Hkv, T, d, cu_seqlens.numel() - 1


def forward_varlen(q, k, v, cu_seqlens, max_seqlen: int, *, causal: bool = False,
                   scale: Optional[float] = None, stream=None):
    """fa_forward_varlen: sequences packed along the token axis (q [H, total, d], k, v
    [Hkv, total, d], offsets cu_seqlens); returns O [H, total, d] and LSE [H, total]."""
    H, Hkv, T, d, S = _check_packed(q, k, v, cu_seqlens)
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    o = torch.empty_like(q)
    lse = torch.empty((H, T), dtype=torch.float32, device=q.device)
    st = lib.fa_forward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(cu_seqlens), S,
                               int(max_seqlen), T, H, Hkv, d, scale, int(bool(causal)),
                               _DTYPES[q.dtype], _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_forward_varlen")
    return o, lse


def backward_varlen(q, k, v, o, lse, do, cu_seqlens, max_seqlen: int, *, causal: bool = False,
                    scale: Optional[float] = None, stream=None):
    """fa_backward_varlen: dQ [H, total, d], dK, dV [Hkv, total, d] for packed sequences."""
    H, Hkv, T, d, S = _check_packed(q, k, v, cu_seqlens)
    for name, t in (("o", o), ("do", do)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must match q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (H, T):
        raise ValueError("lse must be fp32 [H, total]")
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    need = backward_deterministic_workspace_size(1, H, T)
    workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib.fa_backward_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq),
                                _ptr(dk), _ptr(dv), _ptr(cu_seqlens), S, int(max_seqlen), T, H,
                                Hkv, d, scale, int(bool(causal)), _DTYPES[q.dtype],
                                _ptr(workspace), workspace.numel(), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_backward_varlen")
    return dq, dk, dv


def forward_splitkv(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, *,
                    scale: Optional[float] = None, kv_lens: Optional[torch.Tensor] = None,
                    n_splits: int = 0, o: Optional[torch.Tensor] = None,
                    lse: Optional[torch.Tensor] = None, workspace: Optional[torch.Tensor] = None,
                    stream=None) -> Tuple[torch.Tensor, torch.Tensor]:
    """O, LSE with the key sequence cut into ranges merged afterwards (fa_forward_splitkv;
    fa_forward_splitkv_gqa when k, v have fewer heads).  q: [B, H, Nq, d]; k, v: [B, Hkv, Nk, d]
    with Hkv dividing H; bf16 or fp16; no causal or tile mask."""
    for name, t in (("q", q), ("k", k), ("v", v)):
        if not t.is_cuda or not t.is_contiguous() or t.dim() != 4:
            raise ValueError(f"{name} must be a contiguous 4-D CUDA tensor")
    B, H, Nq, d = q.shape
    Nk, Hkv = k.shape[2], k.shape[1]
    if k.shape != v.shape or k.shape[0] != B or k.shape[3] != d or H % Hkv != 0:
        raise ValueError("k, v must be [B, Hkv, Nk, d] with Hkv dividing the query heads")
    if not (q.dtype == k.dtype == v.dtype) or q.dtype not in _DTYPES:
        raise ValueError("q, k, v must share a supported dtype")
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    _, kv_lens = _masks(None, kv_lens, B, Nq, q.device)
    G = H // Hkv                       # a group's query heads run as one block of G * Nq rows
    splits = (int(lib.fa_forward_splitkv_auto_splits(B, Hkv, G * Nq, Nk)) if n_splits == 0
              else int(n_splits))
    splits = max(1, min(splits, (Nk + 127) // 128 or 1))
    need = int(lib.fa_forward_splitkv_workspace_size(B, H, Nq, d, splits))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q) if o is None else o
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device) if lse is None else lse
    if Hkv == H:
        st = lib.fa_forward_splitkv(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Nq, Nk, d,
                                    scale, _ptr(kv_lens), _DTYPES[q.dtype], splits, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(), _stream(stream))
    else:
        st = lib.fa_forward_splitkv_gqa(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), B, H, Hkv, Nq,
                                        Nk, d, scale, _ptr(kv_lens), _DTYPES[q.dtype], splits,
                                        _ptr(workspace), workspace.numel() * workspace.element_size(),
                                        _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_forward_splitkv")
    return o, lse


def backward_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(lib.fa_backward_workspace_size(B, H, N, d))


def backward_deterministic_workspace_size(B: int, H: int, N: int) -> int:
    return int(lib.fa_backward_deterministic_workspace_size(B, H, N))


def backward_fused_workspace_size(B: int, H: int, N: int, d: int) -> int:
    return int(lib.fa_backward_fused_workspace_size(B, H, N, d))


def backward(q, k, v, o, lse, do, *, causal: bool = False, scale: Optional[float] = None,
             block_mask=None, kv_lens=None, dq=None, dk=None, dv=None, workspace=None,
             stream=None, deterministic: bool = False, fused: bool = False,
             dropout_p: float = 0.0, seed: int = 0, offset: int = 0):
    """dQ, dK, dV = recompute-based attention backward (fa_backward; fa_backward_gqa when k, v
    have fewer heads than q; fa_backward_deterministic, bit-reproducible, when asked;
    fa_backward_fused, the single-pass atomic-dQ variant, when asked)."""
    B, H, N, d, Hkv = _check_qkv(q, k, v)
    for name, t in (("o", o), ("do", do)):
        if t.shape != q.shape or t.dtype != q.dtype or not t.is_contiguous():
            raise ValueError(f"{name} must match q")
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, N):
        raise ValueError("lse must be fp32 [B, H, N]")
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    block_mask, kv_lens = _masks(block_mask, kv_lens, B, N, q.device)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    if fused and (deterministic or dropout_p > 0.0):
        raise ValueError("the fused backward has no deterministic or dropout form")
    need = (backward_fused_workspace_size(B, H, N, d) if fused
            else backward_deterministic_workspace_size(B, H, N) if deterministic or dropout_p > 0.0
            else backward_workspace_size(B, H, N, d))
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse), _ptr(dq), _ptr(dk), _ptr(dv))
    tail = (d, scale, int(bool(causal)), _ptr(block_mask), _DTYPES[q.dtype], _ptr(kv_lens),
            _ptr(workspace), workspace.numel() * workspace.element_size(), _stream(stream))
    if dropout_p > 0.0:
        drop = FaDropout(float(dropout_p), int(seed), int(offset))
        st = lib.fa_backward_dropout(*args, B, H, Hkv, N, d, scale, int(bool(causal)),
                                     _ptr(block_mask), _DTYPES[q.dtype], _ptr(kv_lens),
                                     ctypes.byref(drop), _ptr(workspace),
                                     workspace.numel() * workspace.element_size(), _stream(stream))
        if st != FA_OK:
            raise FaError(st, "fa_backward_dropout")
        return dq, dk, dv
    if deterministic:
        st = lib.fa_backward_deterministic(*args, B, H, Hkv, N, *tail)
        if st != FA_OK:
            raise FaError(st, "fa_backward_deterministic")
        return dq, dk, dv
    if fused:
        st = lib.fa_backward_fused(*args, B, H, Hkv, N, *tail)
        if st != FA_OK:
            raise FaError(st, "fa_backward_fused")
        return dq, dk, dv
    if Hkv == H:
        st = lib.fa_backward(*args, B, H, N, *tail)
    else:
        st = lib.fa_backward_gqa(*args, B, H, Hkv, N, *tail)
    if st != FA_OK:
        raise FaError(st, "fa_backward")
    return dq, dk, dv


def check_device_status(stream=None) -> int:
    """Synchronise the stream and return the device status (FA_OK or FA_ERR_TIMEOUT/CUDA)."""
    return int(lib.fa_check_device_status(_stream(stream)))


def set_fault_injection(mode: int) -> None:
    lib.fa_debug_set_fault_injection(int(mode))


def set_wait_limit_ms(ms: int) -> None:
    lib.fa_debug_set_wait_limit_ms(int(ms))


def backward_noalloc(q, k, v, o, lse, do, *, causal: bool = False, scale: Optional[float] = None,
                     block_mask=None, kv_lens=None, dq=None, dk=None, dv=None, stream=None):
    """fa_backward_noalloc: the backward with the library's built-in scratch instead of a
    workspace (for callers that cannot allocate device memory).  Output tensors may be passed
    in so that the call itself allocates nothing."""
    B, H, N, d, Hkv = _check_qkv(q, k, v)
    if Hkv != H:
        raise ValueError("fa_backward_noalloc takes one key/value head per query head")
    scale = 1.0 / d ** 0.5 if scale is None else float(scale)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    st = lib.fa_backward_noalloc(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                 _ptr(dq), _ptr(dk), _ptr(dv), B, H, N, d, scale,
                                 int(bool(causal)), _ptr(block_mask), _DTYPES[q.dtype],
                                 _ptr(kv_lens), _stream(stream))
    if st != FA_OK:
        raise FaError(st, "fa_backward_noalloc")
    return dq, dk, dv


def noalloc_max_workspace() -> int:
    return int(lib.fa_backward_noalloc_max_workspace())
