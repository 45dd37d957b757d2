"""GPU parity and reproducibility of the two-pass backward (fa_backward_deterministic, and
fa_backward's default for 16-bit inputs): the gradients against the fp64 oracle on ragged
sizes, every mask, bf16 and fp16, grouped heads; the same bits on repeated calls and through
both entry points; dK and dV bit-identical to the fused atomic-dQ backward's (the same
key-stationary arithmetic) and dQ within the tolerance of it.  The fused variant keeps its own
parity cases here."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import _dev, check_backward_given_o, compare, compare_bwd, f64, run_gpu
from ideal_kernel import ideal_backward
from tolerances import assert_bf16_close
from workloads import WORKLOADS, Workload, make_inputs, random_tile_mask

pytestmark = pytest.mark.gpu


def _case(N, d, dtype="bf16", causal=False, B=2, H=3, Hkv=None, seed=0):
    w = Workload(f"det_{N}_{d}", B, H, N, d, dtype, causal=causal)
    return make_inputs(w, seed=seed, kv_heads=Hkv)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal", [(127, False), (300, True), (1000, False), (1000, True)])
def test_deterministic_shapes(N, d, causal):
    x = _case(N, d, causal=causal, seed=N + d)
    compare(x, run_gpu(x, deterministic=True))
    check_backward_given_o(x, deterministic=True)


def test_deterministic_masks_fp16():
    x = _case(900, 128, "fp16", True, B=3, H=2, seed=8)
    x["kv_lens"] = torch.tensor([900, 451, 0], dtype=torch.int32)
    x["block_mask"] = random_tile_mask(8, 0.6, seed=4)
    out = run_gpu(x, deterministic=True)
    check_backward_given_o(x, deterministic=True)
    assert torch.count_nonzero(out["dq"][2]) == 0       # kv_len 0: no key, zero gradient


@pytest.mark.parametrize("Hkv", [1, 2])
def test_deterministic_grouped_heads(Hkv):
    x = _case(520, 128, causal=True, H=4, Hkv=Hkv, seed=3 + Hkv)
    x["kv_lens"] = torch.tensor([520, 301], dtype=torch.int32)
    compare(x, run_gpu(x, deterministic=True))


def _both(x, reps=3):
    import exact_io_aware_23_gb300 as fa
    q, k, v, do, kw = _dev(x)
    o, lse = fa.forward(q, k, v, **kw)
    det = [fa.backward(q, k, v, o, lse, do, deterministic=True, **kw) for _ in range(reps)]
    default = fa.backward(q, k, v, o, lse, do, **kw)
    for a_, b_ in zip(det[0], default):
        assert torch.equal(a_, b_)
    fused = fa.backward(q, k, v, o, lse, do, fused=True, **kw)
    assert fa.check_device_status() == 0
    return det, fused


@pytest.mark.parametrize("causal", [False, True])
def test_reproducible_bits(causal):
    x = _case(4096, 128, causal=causal, B=1, H=4, seed=21)
    det, fused = _both(x)
    for run in det[1:]:
        for a_, b_ in zip(det[0], run):
            assert torch.equal(a_, b_)
    # dK, dV come from the same key-stationary arithmetic in both backwards
    assert torch.equal(det[0][1], fused[1]) and torch.equal(det[0][2], fused[2])
    g = f64(det[0][0])
    ref = f64(fused[0])
    assert np.mean(np.abs(g - ref)) <= 2e-3 * np.sqrt(np.mean(ref ** 2))


def test_long_causal_n16k_d128():
    """The long causal workload shape: dQ rows sampled against the oracle (a row's dQ depends on
    that row alone); dK, dV bit-identical to the fused backward, which the workload parity tests
    check against the oracle."""
    x = make_inputs(WORKLOADS["long_n16k_d128_causal"])
    det, fused = _both(x, reps=2)
    assert all(torch.equal(a_, b_) for a_, b_ in zip(det[0], det[1]))
    assert torch.equal(det[0][1], fused[1]) and torch.equal(det[0][2], fused[2])
    rows = np.sort(np.random.default_rng(5).choice(16384, 192, replace=False))
    heads = [0, 9]
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    dQ, _, _ = oracle.backward(qq, kk, vv, dd, x["scale"], causal=True, heads=heads, rows=rows)
    idq = ideal_backward(x, heads=heads, rows=rows)[0]
    assert_bf16_close("dQ", f64(det[0][0])[:, heads][:, :, rows], dQ[:, :, rows], ideal=idq[:, :, rows])


# --- the fused atomic-dQ variant (fa_backward_fused) -----------------------------------------

@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("N,causal", [(300, True), (1000, False)])
def test_fused_variant_shapes(N, d, causal):
    x = _case(N, d, causal=causal, seed=7 * N + d)
    compare(x, run_gpu(x, fused=True))
    check_backward_given_o(x, fused=True)


def test_fused_variant_masks_grouped_fp16():
    x = _case(900, 128, "fp16", True, B=2, H=4, Hkv=2, seed=12)
    x["kv_lens"] = torch.tensor([900, 451], dtype=torch.int32)
    x["block_mask"] = random_tile_mask(8, 0.6, seed=5)
    run_gpu(x, backward=False)
    check_backward_given_o(x, fused=True)


def test_default_backward_is_not_changed_by_the_fused_call():
    """The variant is chosen per call: a fused call in between leaves the default backward's
    bits unchanged (there is no process-wide switch any more)."""
    import exact_io_aware_23_gb300 as fa
    x = _case(700, 64, causal=True, B=1, H=2, seed=31)
    q, k, v, do, kw = _dev(x)
    o, lse = fa.forward(q, k, v, **kw)
    first = fa.backward(q, k, v, o, lse, do, **kw)
    fa.backward(q, k, v, o, lse, do, fused=True, **kw)
    again = fa.backward(q, k, v, o, lse, do, **kw)
    assert fa.check_device_status() == 0
    assert all(torch.equal(a_, b_) for a_, b_ in zip(first, again))
