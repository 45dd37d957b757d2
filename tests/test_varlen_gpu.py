"""GPU parity for packed sequences (fa_forward_varlen / fa_backward_varlen): sequences of ragged
lengths stored back to back along each head's token axis, a query seeing only its own sequence.
Against the fp64 oracle (document-mask reading, offsets as ``segments``); bit-identical to
running each sequence alone through fa_forward / fa_backward; empty and one-token sequences,
lengths off the 128 grid, grouped heads, fp16; offsets outside their contract reported."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import LSE_TOL_BF16, f64
from ideal_kernel import ideal_backward, ideal_forward
from tolerances import assert_bf16_close, assert_lse_close
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _packed(lens, H, Hkv, d, dtype="bf16", seed=0):
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T = int(cu[-1])
    w = Workload(f"packed_{T}_{d}", 1, H, T, d, dtype)
    x = make_inputs(w, seed=seed, kv_heads=Hkv)
    dev = torch.device("cuda:0")
    t = {n: x[n][0].to(dev) for n in ("q", "k", "v", "do")}      # [heads, total, d]
    return x, t, cu, torch.tensor(cu, dtype=torch.int32, device=dev), max(max(lens), 1)


def _check(lens, H, Hkv, d, causal, dtype="bf16", seed=0):
    import exact_io_aware_23_gb300 as fa
    x, t, cu, cu_d, maxl = _packed(lens, H, Hkv, d, dtype, seed)
    o, lse = fa.forward_varlen(t["q"], t["k"], t["v"], cu_d, maxl, causal=causal)
    assert fa.check_device_status() == 0
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    O, L = oracle.forward(qq, kk, vv, x["scale"], causal=causal, segments=cu)
    xc = dict(x, causal=causal)
    assert_bf16_close("O", f64(o)[None], O, ideal=ideal_forward(xc, segments=cu))
    assert_lse_close(f64(lse)[None], L, LSE_TOL_BF16)
    # backward on the oracle's O (rounded to the working dtype): the operator the kernel computes
    o_in = torch.from_numpy(O[0]).to(t["q"].dtype)
    dq, dk, dv = fa.backward_varlen(t["q"], t["k"], t["v"], o_in.to(t["q"].device),
                                    torch.from_numpy(L[0]).float().to(t["q"].device), t["do"],
                                    cu_d, maxl, causal=causal)
    assert fa.check_device_status() == 0
    dQ, dK, dV = oracle.backward(qq, kk, vv, dd, x["scale"], causal=causal, segments=cu,
                                 o=o_in.to(torch.float64).numpy()[None])
    ideal = ideal_backward(xc, segments=cu, o=o_in[None])
    for name, got, ref, idl in zip(("dQ", "dK", "dV"), (dq, dk, dv), (dQ, dK, dV), ideal):
        assert_bf16_close(name, f64(got)[None], ref, ideal=idl)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_packed_ragged(d, causal):
    _check([300, 0, 1, 129, 517, 128, 64], 4, 4, d, causal, seed=d + causal)


@pytest.mark.parametrize("Hkv", [1, 2])
def test_packed_grouped_heads(Hkv):
    _check([700, 33, 1000], 4, Hkv, 128, True, seed=Hkv)


def test_packed_fp16():
    _check([255, 257, 2], 2, 2, 64, True, dtype="fp16", seed=9)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_equals_separate_sequences(causal):
    """Each packed sequence gives the same bits as that sequence alone through fa_forward /
    fa_backward (masked keys contribute exact zeros either way)."""
    import exact_io_aware_23_gb300 as fa
    lens = [400, 129, 0, 1000, 77]
    x, t, cu, cu_d, maxl = _packed(lens, 4, 2, 128, seed=31)
    o, lse = fa.forward_varlen(t["q"], t["k"], t["v"], cu_d, maxl, causal=causal)
    dq, dk, dv = fa.backward_varlen(t["q"], t["k"], t["v"], o, lse, t["do"], cu_d, maxl, causal=causal)
    for a_, b_ in zip(cu[:-1], cu[1:]):
        if a_ == b_:
            continue
        sl = slice(int(a_), int(b_))
        q1, k1, v1, do1 = (t[n][None, :, sl].contiguous() for n in ("q", "k", "v", "do"))
        o1, l1 = fa.forward(q1, k1, v1, causal=causal)
        g1 = fa.backward(q1, k1, v1, o1, l1, do1, causal=causal)
        assert torch.equal(o[:, sl], o1[0]) and torch.equal(lse[:, sl], l1[0])
        for full, part in zip((dq, dk, dv), g1):
            assert torch.equal(full[:, sl], part[0])
    assert fa.check_device_status() == 0


def test_packed_long_mixture():
    """A long mixture (16 sequences, 96 to 4000 tokens, 32K tokens in all) against the oracle
    on sampled rows of every sequence (a row's output depends on its own sequence alone)."""
    import exact_io_aware_23_gb300 as fa
    rng = np.random.default_rng(4)
    lens = [int(v) for v in rng.integers(96, 4000, 16)]
    x, t, cu, cu_d, maxl = _packed(lens, 4, 1, 128, seed=5)
    o, lse = fa.forward_varlen(t["q"], t["k"], t["v"], cu_d, maxl, causal=True)
    assert fa.check_device_status() == 0
    rows = np.sort(np.concatenate([rng.choice(np.arange(a, b), 8, replace=False)
                                   for a, b in zip(cu[:-1], cu[1:])]))
    O, L = oracle.forward(*(f64(x[n]) for n in ("q", "k", "v")), x["scale"], causal=True,
                          segments=cu, rows=rows)
    assert_bf16_close("O", f64(o)[None][:, :, rows], O,
                      ideal=ideal_forward(dict(x, causal=True), segments=cu, rows=rows))
    assert_lse_close(f64(lse)[None][:, :, rows], L, LSE_TOL_BF16)


def test_offsets_outside_contract_are_reported():
    """Offsets the kernels cannot follow (decreasing, or a sequence longer than max_seqlen)
    make the call skip those sequences and report FA_ERR_INVALID_ARG through the status check;
    nothing outside the tensors is touched."""
    import exact_io_aware_23_gb300 as fa
    x, t, cu, cu_d, maxl = _packed([200, 300], 2, 2, 64, seed=2)
    bad = torch.tensor([0, 300, 200], dtype=torch.int32, device=cu_d.device)     # decreasing
    fa.forward_varlen(t["q"], t["k"], t["v"], bad, 300)
    assert fa.check_device_status() == fa.FA_ERR_INVALID_ARG
    fa.forward_varlen(t["q"], t["k"], t["v"], cu_d, 250)                           # 300 > 250
    assert fa.check_device_status() == fa.FA_ERR_INVALID_ARG
    fa.forward_varlen(t["q"], t["k"], t["v"], cu_d, maxl)
    assert fa.check_device_status() == 0
