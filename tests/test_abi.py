"""The C-ABI library loads and exports every function include/fa.h declares, and its host-side
argument checks return the documented status before any CUDA call (CPU only: no kernel runs)."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")
LIB = os.path.join(ROOT, "exact_io_aware_23_gb300", "libfa.so")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    __graft_entry__._build_module().build()
    L = ctypes.CDLL(LIB)
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_forward.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, vp]
    L.fa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, f, i, vp, i, vp, vp, sz, vp]
    L.fa_backward_workspace_size.argtypes = [i, i, i, i]
    L.fa_backward_workspace_size.restype = sz
    L.fa_status_string.argtypes = [i]
    L.fa_status_string.restype = ctypes.c_char_p
    return L


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("fa_forward", "fa_backward", "fa_backward_workspace_size", "fa_check_device_status",
              "fa_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True).stdout
    exported = set(re.findall(r"\bT (fa_\w+)", out))
    for n in declared_functions():
        assert n in exported, n
        assert hasattr(lib, n), n


def test_status_strings(lib):
    assert lib.fa_status_string(0) == b"FA_OK"
    assert lib.fa_status_string(4) == b"FA_ERR_TIMEOUT"
    assert lib.fa_status_string(99) == b"FA_UNKNOWN_STATUS"
    assert lib.fa_version() == 201


P = ctypes.c_void_p(0x10000)       # aligned, never dereferenced: every call below returns early
MIS = ctypes.c_void_p(0x10008)      # 8-byte aligned only


def fwd(lib, q=P, k=P, v=P, o=P, lse=P, B=1, H=1, N=128, d=64, scale=0.125, causal=0, dtype=0):
    return lib.fa_forward(q, k, v, o, lse, B, H, N, d, scale, causal, None, dtype, None, None)


def test_forward_argument_checks(lib):
    assert fwd(lib, d=96) == UNSUPPORTED
    assert fwd(lib, d=32) == UNSUPPORTED
    assert fwd(lib, dtype=7) == UNSUPPORTED
    assert fwd(lib, dtype=3) == UNSUPPORTED
    assert fwd(lib, dtype=2, N=0) == OK          # FA_FP16 is a supported dtype
    assert fwd(lib, B=-1) == INVALID
    assert fwd(lib, N=-5) == INVALID
    assert fwd(lib, scale=float("nan")) == INVALID
    assert fwd(lib, scale=float("inf")) == INVALID
    assert fwd(lib, scale=0.0) == INVALID
    assert fwd(lib, scale=-0.5) == INVALID
    assert fwd(lib, q=None) == INVALID
    assert fwd(lib, lse=None) == INVALID
    assert fwd(lib, v=MIS) == INVALID
    assert fwd(lib, o=MIS) == INVALID
    # empty problems are no-ops
    assert fwd(lib, N=0) == OK
    assert fwd(lib, B=0, q=None) == OK
    assert fwd(lib, H=0) == OK


def test_backward_argument_checks(lib):
    ws = lib.fa_backward_workspace_size(2, 3, 100, 64)
    # D (one fp32 per query row), then the unit order used under a tile mask (2 ints per tile and
    # slice, plus a few per tile); no dQ accumulator
    assert ws % 256 == 0 and 2 * 3 * 100 * 4 <= ws <= 2560 + 256
    assert lib.fa_backward_workspace_size(0, 3, 100, 64) == 0
    big = lib.fa_backward_workspace_size(1, 16, 16384, 128)    # the long workload: about 1 MiB
    assert (1 << 20) <= big < (1 << 20) + (1 << 15)

    def bwd(dq=P, workspace=P, wsb=ws, d=64, N=100, dtype=0):
        return lib.fa_backward(P, P, P, P, P, P, dq, P, P, 2, 3, N, d, 0.125, 0, None, dtype, None,
                               workspace, wsb, None)
    assert bwd(d=80) == UNSUPPORTED
    assert bwd(dq=None) == INVALID
    assert bwd(dq=MIS) == INVALID
    assert bwd(workspace=None) == INVALID
    assert bwd(workspace=ctypes.c_void_p(0x10010)) == INVALID     # not 256-byte aligned
    assert bwd(wsb=ws - 4) == INVALID
    assert bwd(N=0) == OK


def test_splitkv_argument_checks(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_forward_splitkv.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, vp, i, i, vp, sz, vp]
    lib.fa_forward_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_forward_splitkv_workspace_size.restype = sz
    ws = lib.fa_forward_splitkv_workspace_size(2, 3, 16, 128, 4)
    assert ws % 256 == 0 and ws >= 4 * 2 * 3 * 16 * 129 * 4
    assert lib.fa_forward_splitkv_workspace_size(2, 3, 16, 128, 0) == 0

    def call(dtype=0, d=128, Nk=4096, splits=4, w=P, wsb=ws, Nq=16):
        return lib.fa_forward_splitkv(P, P, P, P, P, 2, 3, Nq, Nk, d, 0.1, None, dtype, splits, w, wsb, None)
    assert call(dtype=1) == UNSUPPORTED          # fp32 has no split-KV path
    assert call(d=96) == UNSUPPORTED
    assert call(Nk=-1) == INVALID
    assert call(splits=-2) == INVALID
    assert call(w=None) == INVALID
    assert call(wsb=ws - 256) == INVALID
    assert call(Nq=0) == OK


def test_splitkv_auto_splits_fill_the_last_wave(lib):
    """The split count rule, on the host (no device: the rule assumes GB300's 152 SMs): from about
    two CTAs per SM, the fewest ranges whose CTAs fill their last one-CTA-per-SM wave to 95 %,
    capped at 2 key tiles a range and at 64 ranges."""
    lib.fa_forward_splitkv_auto_splits.argtypes = [ctypes.c_int] * 4
    auto = lib.fa_forward_splitkv_auto_splits
    sms = 152

    def rule(B, H, Nq, Nk):                       # the rule restated, to compare against
        units = B * H * -(-Nq // 256)
        tiles = -(-Nk // 128)
        want = max(1, -(-2 * sms // units))
        cap = min((tiles + 1) // 2, 64)
        want = min(want, max(cap, 1))
        best, best_fill = want, 0.0
        for s in range(want, min(cap, 4 * want) + 1):
            ctas = units * s
            fill = ctas / (-(-ctas // sms) * sms)
            if fill >= 0.95:
                return s
            if fill > best_fill + 1e-9:
                best, best_fill = s, fill
        return best

    # the two decode workloads: 128 and 64 query blocks against 32K keys -> 7 ranges each
    assert auto(8, 16, 16, 32768) == 7
    assert auto(8, 8, 64, 32768) == 7
    for B, H, Nq, Nk in [(1, 1, 16, 512), (1, 1, 1, 1000000), (2, 3, 300, 4096), (4, 32, 16, 8192),
                         (1, 8, 4096, 65536), (16, 16, 16, 128), (3, 5, 700, 20000)]:
        got = auto(B, H, Nq, Nk)
        assert got == rule(B, H, Nq, Nk), (B, H, Nq, Nk)
        assert 1 <= got <= max(1, min(64, (-(-Nk // 128) + 1) // 2))
    assert auto(0, 1, 1, 1) == 1 and auto(1, 1, 1, 0) == 1


def test_gqa_argument_checks(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_forward_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, vp]
    lib.fa_backward_gqa.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i,
                                    vp, vp, sz, vp]
    ws = lib.fa_backward_workspace_size(2, 8, 100, 64)

    def fwd_g(H=8, Hkv=2, N=128, dtype=0, q=P):
        return lib.fa_forward_gqa(q, P, P, P, P, 2, H, Hkv, N, 64, 0.125, 1, None, dtype, None, None)

    def bwd_g(H=8, Hkv=2, N=100, dtype=0, wsb=ws):
        return lib.fa_backward_gqa(P, P, P, P, P, P, P, P, P, 2, H, Hkv, N, 64, 0.125, 1, None,
                                   dtype, None, P, wsb, None)
    for call in (fwd_g, bwd_g):
        assert call(Hkv=3) == UNSUPPORTED           # 3 does not divide 8
        assert call(Hkv=16) == UNSUPPORTED          # more key/value heads than query heads
        assert call(Hkv=0) == INVALID
        assert call(Hkv=-2) == INVALID
        assert call(dtype=1) == UNSUPPORTED         # fp32 runs on the SIMT path, one head per head
        assert call(N=0) == OK
        assert call(dtype=2, N=0) == OK
    assert fwd_g(q=None) == INVALID
    assert bwd_g(wsb=ws - 4) == INVALID


def test_deterministic_backward_argument_checks(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_backward_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f,
                                              i, vp, i, vp, vp, sz, vp]
    lib.fa_backward_deterministic_workspace_size.argtypes = [i, i, i]
    lib.fa_backward_deterministic_workspace_size.restype = sz
    ws = lib.fa_backward_deterministic_workspace_size(2, 8, 100)
    assert ws % 256 == 0 and ws >= 2 * 8 * 100 * 4
    assert ws == lib.fa_backward_workspace_size(2, 8, 100, 64)     # no dQ accumulator
    assert lib.fa_backward_deterministic_workspace_size(0, 8, 100) == 0

    def call(Hkv=8, N=100, dtype=0, wsb=ws, w=P, d=64):
        return lib.fa_backward_deterministic(P, P, P, P, P, P, P, P, P, 2, 8, Hkv, N, d, 0.125, 1,
                                             None, dtype, None, w, wsb, None)
    assert call(dtype=1) == UNSUPPORTED          # fp32: the SIMT backward has no such variant
    assert call(d=96) == UNSUPPORTED
    assert call(Hkv=3) == UNSUPPORTED
    assert call(Hkv=0) == INVALID
    assert call(w=None) == INVALID
    assert call(w=ctypes.c_void_p(0x10010)) == INVALID
    assert call(wsb=ws - 4) == INVALID
    assert call(N=0) == OK


def test_fused_backward_argument_checks(lib):
    """The fused single-pass backward is its own entry point with its own, larger workspace (fp32
    dQ accumulator + D); no process-wide switch selects it."""
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_backward_fused.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp,
                                      i, vp, vp, sz, vp]
    lib.fa_backward_fused_workspace_size.argtypes = [i, i, i, i]
    lib.fa_backward_fused_workspace_size.restype = sz
    ws = lib.fa_backward_fused_workspace_size(2, 8, 100, 64)
    assert ws % 256 == 0 and ws >= 2 * 8 * 100 * 64 * 4 + 2 * 8 * 100 * 4
    assert lib.fa_backward_fused_workspace_size(2, 8, 100, 0) == 0
    assert "fa_set_backward_variant" not in declared_functions()

    def call(Hkv=8, N=100, dtype=0, wsb=ws, w=P, d=64):
        return lib.fa_backward_fused(P, P, P, P, P, P, P, P, P, 2, 8, Hkv, N, d, 0.125, 1, None,
                                     dtype, None, w, wsb, None)
    assert call(dtype=1) == UNSUPPORTED
    assert call(d=96) == UNSUPPORTED
    assert call(Hkv=3) == UNSUPPORTED
    assert call(w=None) == INVALID
    assert call(wsb=lib.fa_backward_workspace_size(2, 8, 100, 64)) == INVALID   # D only: too small
    assert call(wsb=ws - 4) == INVALID
    assert call(N=0) == OK


def test_varlen_argument_checks(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_forward_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f, i, i, vp]
    lib.fa_backward_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                       i, i, vp, sz, vp]
    lib.fa_backward_deterministic_workspace_size.argtypes = [i, i, i]
    lib.fa_backward_deterministic_workspace_size.restype = sz
    ws = lib.fa_backward_deterministic_workspace_size(1, 8, 1000)

    def fwd_v(cu=P, S=3, maxl=500, T=1000, H=8, Hkv=2, dtype=0, d=64):
        return lib.fa_forward_varlen(P, P, P, P, P, cu, S, maxl, T, H, Hkv, d, 0.125, 1, dtype, None)

    def bwd_v(cu=P, S=3, maxl=500, T=1000, H=8, Hkv=2, dtype=0, wsb=ws):
        return lib.fa_backward_varlen(P, P, P, P, P, P, P, P, P, cu, S, maxl, T, H, Hkv, 64, 0.125,
                                      1, dtype, P, wsb, None)
    for call in (fwd_v, bwd_v):
        assert call(dtype=1) == UNSUPPORTED          # fp32 has no packed path
        assert call(Hkv=3) == UNSUPPORTED
        assert call(cu=None) == INVALID
        assert call(S=-1) == INVALID
        assert call(T=-1) == INVALID
        assert call(maxl=-1) == INVALID
        assert call(T=0) == OK                       # nothing packed: no-op
        assert call(S=0, cu=None) == OK
    assert fwd_v(d=80) == UNSUPPORTED
    assert bwd_v(wsb=ws - 4) == INVALID


def test_dropout_argument_checks(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t

    class Drop(ctypes.Structure):
        _fields_ = [("p", ctypes.c_float), ("seed", ctypes.c_uint64), ("offset", ctypes.c_uint32)]
    dp = ctypes.POINTER(Drop)
    lib.fa_forward_dropout.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, dp, vp]
    lib.fa_backward_dropout.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i,
                                        vp, dp, vp, sz, vp]
    assert ctypes.sizeof(Drop) == 24          # float, 64-bit seed (8-aligned), 32-bit offset

    def fwd_d(p=0.1, drop=True, dtype=0, N=128):
        d = ctypes.byref(Drop(p, 1, 0)) if drop else None
        return lib.fa_forward_dropout(P, P, P, P, P, 1, 2, 2, N, 64, 0.125, 0, None, dtype, None, d, None)

    def bwd_d(p=0.1, dtype=0, N=100):
        return lib.fa_backward_dropout(P, P, P, P, P, P, P, P, P, 1, 2, 2, N, 64, 0.125, 0, None, dtype,
                                       None, ctypes.byref(Drop(p, 1, 0)), P, 1 << 20, None)
    for bad in (float("nan"), -0.1, 1.5, float("inf")):
        assert fwd_d(p=bad) == INVALID and bwd_d(p=bad) == INVALID
    assert fwd_d(drop=False) == INVALID
    assert fwd_d(dtype=1) == UNSUPPORTED and bwd_d(dtype=1) == UNSUPPORTED
    assert fwd_d(N=0) == OK and bwd_d(N=0) == OK
    assert fwd_d(p=0.0, dtype=1, N=0) == OK    # no dropout: plain attention rules apply


def test_splitkv_gqa_argument_checks(lib):
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_forward_splitkv_gqa.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp, i, i, vp, sz, vp]
    lib.fa_forward_splitkv_workspace_size.argtypes = [i, i, i, i, i]
    lib.fa_forward_splitkv_workspace_size.restype = sz
    ws = lib.fa_forward_splitkv_workspace_size(2, 8, 16, 128, 4)

    def call(H=8, Hkv=2, Nq=16, dtype=0, wsb=ws):
        return lib.fa_forward_splitkv_gqa(P, P, P, P, P, 2, H, Hkv, Nq, 4096, 128, 0.1, None, dtype, 4,
                                          P, wsb, None)
    assert call(Hkv=3) == UNSUPPORTED
    assert call(Hkv=0) == INVALID
    assert call(dtype=1) == UNSUPPORTED
    assert call(wsb=ws - 256) == INVALID          # same workspace as the ungrouped call
    assert call(Nq=0) == OK


def test_blocksparse_forward_argument_checks(lib):
    """The balanced block-sparse forward needs its workspace (plan + partials) only with a mask."""
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.fa_forward_blocksparse.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, f, i, vp, i, vp, vp, sz, vp]
    lib.fa_forward_blocksparse_workspace_size.argtypes = [i, i, i, i]
    lib.fa_forward_blocksparse_workspace_size.restype = sz
    ws = lib.fa_forward_blocksparse_workspace_size(1, 8, 65536, 64)
    # 32 partial slots of 256 rows per slice: O (d fp32) and LSE, plus the plan
    assert ws % 256 == 0 and ws >= 8 * 32 * 256 * 65 * 4
    assert lib.fa_forward_blocksparse_workspace_size(1, 8, 0, 64) == 0

    def call(mask=P, w=P, wsb=ws, N=65536, dtype=0):
        return lib.fa_forward_blocksparse(P, P, P, P, P, 1, 8, 8, N, 64, 0.125, 0, mask, dtype, None,
                                          w, wsb, None)
    assert call(w=None) == INVALID
    assert call(w=ctypes.c_void_p(0x10010)) == INVALID      # not 256-byte aligned
    assert call(N=786432 + 1) == UNSUPPORTED                 # the tile-mask size limit
    assert call(N=0) == OK
