"""GPU parity of dropout on P (fa_forward_dropout / fa_backward_dropout): the kernels' mask is the
oracle's to the bit (seen through V = identity columns, where O holds P * M * 256/k8 directly),
forward and backward match the fp64 oracle with the same (seed, offset), the backward replays
the forward's mask, and other offsets give other masks."""
import numpy as np
import pytest
import torch

import oracle
from oracle import dropout as odrop
from gpu_helpers import LSE_TOL_BF16, f64
from ideal_kernel import ideal_backward, ideal_forward
from tolerances import assert_bf16_close, assert_lse_close
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _k8(p):
    return odrop.keep_threshold(float(np.float32(p)))     # the ABI takes p as a 32-bit float


def _case(N, d, dtype="bf16", causal=False, B=2, H=3, Hkv=None, seed=0):
    w = Workload(f"drop_{N}_{d}", B, H, N, d, dtype, causal=causal)
    return make_inputs(w, seed=seed, kv_heads=Hkv)


@pytest.mark.parametrize("tile", [0, 1])
def test_mask_bits_through_identity_values(tile):
    """V is the identity on one 128-key tile and zero elsewhere, so O[i, c] = s * P[i, j] * M[i, j]
    for j = 128*tile + c: the zero pattern of O is the dropped set, compared with the oracle's
    mask element by element (P > 0 everywhere here)."""
    import exact_io_aware_23_gb300 as fa
    B, H, N, d = 2, 2, 256, 128
    x = _case(N, d, B=B, H=H, seed=40 + tile)
    # small scores, so every probability is well above zero
    q, k = ((0.3 * x[n].float()).to(torch.bfloat16).to("cuda") for n in ("q", "k"))
    v = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    v[:, :, 128 * tile:128 * tile + 128] = torch.eye(128, dtype=torch.bfloat16, device="cuda")
    seed, offset, p = (7 << 32) + 12345, 3, 0.3
    o, _ = fa.forward(q, k, v, dropout_p=p, seed=seed, offset=offset)
    assert fa.check_device_status() == 0
    got = (f64(o) != 0)
    for b in range(B):
        for h in range(H):
            want = odrop.keep_mask(np.arange(N), np.arange(128 * tile, 128 * tile + 128), b * H + h,
                                   seed, offset, _k8(p))
            assert np.array_equal(got[b, h], want), (b, h)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal", [(300, True), (1000, False)])
@pytest.mark.parametrize("p", [0.1, 0.5])
def test_dropout_parity(N, d, causal, p):
    import exact_io_aware_23_gb300 as fa
    x = _case(N, d, causal=causal, seed=N + d + int(10 * p))
    seed, offset = 2024 + N, 1
    drop = (seed, offset, _k8(p))
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, causal=causal, dropout_p=p, seed=seed, offset=offset)
    assert fa.check_device_status() == 0
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    O, L = oracle.forward(qq, kk, vv, x["scale"], causal=causal, dropout=drop)
    assert_bf16_close("O", f64(o), O, ideal=ideal_forward(x, dropout=drop))
    assert_lse_close(f64(lse), L, LSE_TOL_BF16)
    # backward on the oracle's O (rounded to bf16) and LSE, against the oracle's backward for it
    o_in = torch.from_numpy(O).to(torch.bfloat16)
    dq, dk, dv = fa.backward(q, k, v, o_in.to(dev), torch.from_numpy(L).float().to(dev), do,
                             causal=causal, dropout_p=p, seed=seed, offset=offset)
    assert fa.check_device_status() == 0
    dQ, dK, dV = oracle.backward(qq, kk, vv, dd, x["scale"], causal=causal, dropout=drop,
                                 o=o_in.to(torch.float64).numpy())
    ideal = ideal_backward(x, dropout=drop, o=o_in)
    for name, got, ref, idl in zip(("dQ", "dK", "dV"), (dq, dk, dv), (dQ, dK, dV), ideal):
        assert_bf16_close(name, f64(got), ref, ideal=idl)


@pytest.mark.parametrize("d", [64, 128])
def test_keep_threshold_extremes(d):
    """The kernels test four uniform bytes at a time against k8 (a per-byte carry, not a byte-wise
    compare instruction): every mask bit at the thresholds where that arithmetic changes form (k8
    = 1, 127, 128, 129, 255) equals the oracle's, seen through identity V columns as above; and
    p = 1 (k8 = 0) drops everything: O = 0 and all three gradients are zero."""
    import exact_io_aware_23_gb300 as fa
    B, H, N = 1, 2, 256
    x = _case(N, d, B=B, H=H, seed=70 + d)
    q, k = ((0.3 * x[n].float()).to(torch.bfloat16).to("cuda") for n in ("q", "k"))
    v = torch.zeros((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    v[:, :, :min(d, 128)] = torch.eye(min(d, 128), dtype=torch.bfloat16, device="cuda")[:, :d]
    seed, offset = 99, 5
    for k8 in (1, 127, 128, 129, 255):
        p = 1.0 - k8 / 256.0
        assert _k8(p) == k8
        o, _ = fa.forward(q, k, v, dropout_p=p, seed=seed, offset=offset)
        assert fa.check_device_status() == 0
        got = f64(o)[:, :, :, :min(d, 128)] != 0        # column c <- key c (keys 0 .. d-1)
        for h in range(H):
            want = odrop.keep_mask(np.arange(N), np.arange(min(d, 128)), h, seed, offset, k8)
            assert np.array_equal(got[0, h], want), (k8, h)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    o, lse = fa.forward(q, k, v, dropout_p=1.0, seed=seed, offset=offset)
    o0, l0 = fa.forward(q, k, v)
    assert torch.count_nonzero(o) == 0
    # the statistic of the undropped scores; the plain forward at d = 64 sums l over 64-key
    # tiles, the dropout one over 128-key tiles: equal up to fp32 summation order
    assert torch.allclose(lse, l0, rtol=0.0, atol=1e-5)
    grads = fa.backward(q, k, v, o, lse, do, dropout_p=1.0, seed=seed, offset=offset)
    assert fa.check_device_status() == 0
    assert all(torch.count_nonzero(g) == 0 for g in grads)


def test_dropout_grouped_heads_fp16_padding():
    import exact_io_aware_23_gb300 as fa
    x = _case(520, 128, "fp16", True, B=2, H=4, Hkv=2, seed=17)
    x["kv_lens"] = torch.tensor([520, 301], dtype=torch.int32)
    seed, offset, p = 99, 5, 0.2
    drop = (seed, offset, _k8(p))
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    kl = x["kv_lens"].to(dev)
    o, lse = fa.forward(q, k, v, causal=True, kv_lens=kl, dropout_p=p, seed=seed, offset=offset)
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    O, L = oracle.forward(qq, kk, vv, x["scale"], causal=True, kv_lens=x["kv_lens"].numpy(), dropout=drop)
    assert_bf16_close("O", f64(o), O, ideal=ideal_forward(x, dropout=drop))
    o_in = torch.from_numpy(O).to(torch.float16)
    dq, dk, dv = fa.backward(q, k, v, o_in.to(dev), torch.from_numpy(L).float().to(dev), do, causal=True,
                             kv_lens=kl, dropout_p=p, seed=seed, offset=offset)
    assert fa.check_device_status() == 0
    dQ, dK, dV = oracle.backward(qq, kk, vv, dd, x["scale"], causal=True, kv_lens=x["kv_lens"].numpy(),
                                 dropout=drop, o=o_in.to(torch.float64).numpy())
    ideal = ideal_backward(x, dropout=drop, o=o_in)
    for name, got, ref, idl in zip(("dQ", "dK", "dV"), (dq, dk, dv), (dQ, dK, dV), ideal):
        assert_bf16_close(name, f64(got), ref, ideal=idl)


def test_replay_and_offsets():
    """The same (seed, offset) gives the same bits in the forward and the backward on every call;
    another offset gives another mask; p = 0 is plain attention."""
    import exact_io_aware_23_gb300 as fa
    x = _case(640, 64, causal=True, seed=3)
    dev = torch.device("cuda")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    kw = dict(causal=True, dropout_p=0.25, seed=11)
    o1, l1 = fa.forward(q, k, v, offset=0, **kw)
    o2, l2 = fa.forward(q, k, v, offset=0, **kw)
    o3, l3 = fa.forward(q, k, v, offset=1, **kw)
    assert torch.equal(o1, o2) and torch.equal(l1, l2) and torch.equal(l1, l3)
    assert not torch.equal(o1, o3)
    g1 = fa.backward(q, k, v, o1, l1, do, offset=0, **kw)
    g2 = fa.backward(q, k, v, o1, l1, do, offset=0, **kw)
    assert all(torch.equal(a_, b_) for a_, b_ in zip(g1, g2))
    o0, l0 = fa.forward(q, k, v, causal=True)
    oz, lz = fa.forward(q, k, v, causal=True, dropout_p=1e-9, seed=11)
    assert torch.equal(o0, oz) and torch.equal(l0, lz)
    assert fa.check_device_status() == 0


def test_dropout_long_rows():
    """A long causal shape (N = 4096, d = 128, p = 0.1): sampled rows of O against the oracle."""
    import exact_io_aware_23_gb300 as fa
    x = _case(4096, 128, causal=True, B=1, H=4, seed=8)
    seed, offset, p = 31337, 2, 0.1
    dev = torch.device("cuda")
    o, lse = fa.forward(*(x[n].to(dev) for n in ("q", "k", "v")), causal=True, dropout_p=p,
                        seed=seed, offset=offset)
    assert fa.check_device_status() == 0
    rows = np.sort(np.random.default_rng(1).choice(4096, 160, replace=False))
    O, L = oracle.forward(*(f64(x[n]) for n in ("q", "k", "v")), x["scale"], causal=True, rows=rows,
                          dropout=(seed, offset, _k8(p)))
    assert_bf16_close("O", f64(o)[:, :, rows], O,
                      ideal=ideal_forward(x, rows=rows, dropout=(seed, offset, _k8(p))))
    assert_lse_close(f64(lse)[:, :, rows], L, LSE_TOL_BF16)
