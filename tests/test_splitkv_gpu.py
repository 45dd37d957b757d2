"""Split-KV forward (key tiles cut into ranges, merged with the (m, l, u) merge law) against the
fp64 oracle on decode-shaped inputs (few queries, long keys), and its results for different
numbers of ranges against each other."""
import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import f64
from ideal_kernel import ideal_forward
from tolerances import assert_bf16_close, assert_lse_close
from workloads import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

LSE_TOL = 1e-3


def _run(x, n_splits):
    import exact_io_aware_23_gb300 as fa
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    kl = None if x["kv_lens"] is None else x["kv_lens"].cuda()
    o, lse = fa.forward_splitkv(q, k, v, scale=x["scale"], kv_lens=kl, n_splits=n_splits)
    assert fa.check_device_status() == 0
    return o, lse


def _check(x, o, lse):
    kv = None if x["kv_lens"] is None else x["kv_lens"].numpy()
    O, L = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), x["scale"], kv_lens=kv)
    assert_bf16_close("O", f64(o), O, ideal=ideal_forward(x))
    assert_lse_close(f64(lse), L, LSE_TOL)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Nq,Nk", [(1, 1000), (16, 4096), (100, 3000), (256, 777), (300, 8192)])
@pytest.mark.parametrize("n_splits", [0, 1, 5])
def test_splitkv_against_oracle(dtype, d, Nq, Nk, n_splits):
    w = Workload("dec", 2, 3, Nq, d, dtype, Nk=Nk, backward=False)
    x = make_inputs(w, seed=Nq + Nk + d)
    _check(x, *_run(x, n_splits))


def test_splitkv_key_padding_and_empty_sequence():
    w = Workload("dec_pad", 4, 2, 24, 128, "bf16", Nk=5000, pad_lengths=(1, 5000), backward=False)
    x = make_inputs(w, seed=3)
    x["kv_lens"] = torch.tensor([0, 1, 4097, 5000], dtype=torch.int32)
    o, lse = _run(x, 7)
    _check(x, o, lse)
    assert torch.all(o[0] == 0) and torch.all(torch.isneginf(lse[0]))


def test_splitkv_range_count_does_not_change_the_result():
    """The merge law makes the result independent of how the keys are cut (up to rounding)."""
    w = Workload("dec_inv", 2, 4, 64, 128, "bf16", Nk=16384, backward=False)
    x = make_inputs(w, seed=5)
    outs = [_run(x, s) for s in (1, 2, 7, 64)]
    ref_o, ref_l = (f64(t) for t in outs[0])
    for o, l in outs[1:]:
        assert_bf16_close("O", f64(o), ref_o)
        assert np.max(np.abs(f64(l) - ref_l)) <= 1e-4


def test_splitkv_equals_forward_for_square_problems():
    import exact_io_aware_23_gb300 as fa
    w = Workload("sq", 1, 4, 1000, 64, "bf16")
    x = make_inputs(w, seed=6)
    q, k, v = (x[n].cuda() for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v)
    o2, l2 = fa.forward_splitkv(q, k, v, n_splits=3)
    assert_bf16_close("O", f64(o2), f64(o1))
    assert np.max(np.abs(f64(l2) - f64(l1))) <= 1e-4


def test_decode_workload():
    x = make_inputs(WORKLOADS["decode_q16_k32k_d128"])
    o, lse = _run(x, 0)
    rows = [0, 7, 15]
    kv = None
    O, L = oracle.forward(f64(x["q"]), f64(x["k"]), f64(x["v"]), x["scale"], rows=rows,
                          heads=[0, 9])
    assert_bf16_close("O", f64(o)[:, [0, 9]][:, :, rows], O,
                      ideal=ideal_forward(x, heads=[0, 9], rows=rows))
    assert_lse_close(f64(lse)[:, [0, 9]][:, :, rows], L, LSE_TOL)


@pytest.mark.parametrize("H,Hkv", [(8, 1), (8, 2), (32, 8)])
@pytest.mark.parametrize("Nq,Nk", [(1, 3000), (16, 4096), (5, 777)])
def test_splitkv_grouped_heads(H, Hkv, Nq, Nk):
    """Grouped-query decode: the G query heads of a group run as one block of G * Nq rows against
    their shared key/value head; every query head still gets its own softmax."""
    w = Workload("dec_gqa", 2, H, Nq, 128, "bf16", Nk=Nk, backward=False)
    x = make_inputs(w, seed=H + Nq + Nk, kv_heads=Hkv)
    x["kv_lens"] = torch.tensor([Nk, Nk // 3 + 1], dtype=torch.int32)
    for n_splits in (0, 3):
        o, lse = _run(x, n_splits)
        _check(x, o, lse)


def test_splitkv_grouped_equals_repeated_heads():
    """Same numbers as the ungrouped split-KV forward on key/value heads repeated per query head
    (within rounding: the packed row block changes which rows share a tile, not the arithmetic
    of a row)."""
    w = Workload("dec_gqa", 2, 8, 16, 128, "bf16", Nk=5000, backward=False)
    x = make_inputs(w, seed=4, kv_heads=2)
    o1, l1 = _run(x, 4)
    xr = dict(x, k=x["k"].repeat_interleave(4, dim=1), v=x["v"].repeat_interleave(4, dim=1))
    o2, l2 = _run(xr, 4)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
