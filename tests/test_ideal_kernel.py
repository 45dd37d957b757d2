"""The ideal-kernel floor used by the 16-bit parity tests (CPU only).

Checks that the emulated ideal kernel (tests/ideal_kernel.py) is what it claims to be, and that
the floor-relative bound of tolerances.assert_bf16_close bites: a kernel with one rounding more
than the ideal one fails it, a kernel with one rounding less passes it.
"""
import numpy as np
import pytest
import torch

import oracle
from ideal_kernel import ideal_backward, ideal_forward, round_to
from tolerances import (BF16_MAX_OVER_PEAK, BF16_MEAN_OVER_RMS, FLOOR_FACTOR, FLOOR_SLACK,
                        assert_bf16_close, errors)
from workloads import Workload, make_inputs


def _x(N=300, d=64, causal=True, dtype="bf16", pad=None, seed=3, H=2, Hkv=None):
    w = Workload("ideal", 2, H, N, d, dtype, causal=causal, pad_lengths=pad)
    return make_inputs(w, seed=seed, kv_heads=Hkv)


def _exact(x, **kw):
    f64 = lambda t: t.to(torch.float64).numpy()
    kv = None if x["kv_lens"] is None else x["kv_lens"].numpy()
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    O, _ = oracle.forward(qq, kk, vv, x["scale"], causal=x["causal"], kv_lens=kv, **kw)
    grads = oracle.backward(qq, kk, vv, dd, x["scale"], causal=x["causal"], kv_lens=kv, **kw)
    return O, grads


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_ideal_outputs_are_values_of_the_output_type(dtype):
    x = _x(dtype=dtype, pad=(100, 300))
    O = ideal_forward(x)
    grads = ideal_backward(x)
    for t in (O, *grads):
        assert np.array_equal(round_to(t, dtype), t)


@pytest.mark.parametrize("case", [dict(), dict(causal=False, pad=(120, 300)), dict(d=128, N=260),
                                  dict(H=4, Hkv=2)])
def test_floor_is_nonzero_and_within_the_stated_bounds(case):
    """The floor is what any 16-bit kernel pays: positive, and inside the mean/RMS and max/peak
    bounds (so those bounds are attainable; the floor check is the finer one)."""
    x = _x(**case)
    O, grads = _exact(x)
    ideal = (ideal_forward(x),) + ideal_backward(x)
    for name, got, ref in zip(("O", "dQ", "dK", "dV"), ideal, (O,) + grads):
        r = errors(got, ref)
        assert r["max_abs"] > 0, name
        assert r["mean_over_rms"] <= BF16_MEAN_OVER_RMS, (name, r)
        assert r["max_over_peak"] <= BF16_MAX_OVER_PEAK, (name, r)
        assert_bf16_close(name, got, ref, ideal=got)      # the ideal kernel meets its own floor


def test_fp16_floor_is_finer_than_bf16():
    """fp16 keeps 10 mantissa bits to bf16's 7: its floor is several times lower."""
    xb, xh = _x(dtype="bf16", seed=5), _x(dtype="fp16", seed=5)
    Ob, Oh = ideal_forward(xb), ideal_forward(xh)
    O, _ = _exact(xb)
    O16, _ = _exact(xh)
    assert np.max(np.abs(Oh - O16)) * 4 < np.max(np.abs(Ob - O))


def _round_bits(a, bits):
    """Round to `bits` significant bits (bf16 keeps 8, counting the implicit one)."""
    f, e = np.frexp(a)
    return np.ldexp(np.round(f * 2.0 ** bits) / 2.0 ** bits, e)


def _degraded_forward(x, bits):
    """A forward that rounds P to `bits` significant bits instead of bf16's 8."""
    f64 = lambda t: t.to(torch.float64).numpy()
    q, k, v = (f64(x[n]) for n in ("q", "k", "v"))
    out = np.zeros_like(q)
    for b in range(q.shape[0]):
        for h in range(q.shape[1]):
            P = oracle.probabilities(q[b, h], k[b, h], x["scale"], causal=x["causal"])
            out[b, h] = round_to(_round_bits(P, bits) @ v[b, h], x["dtype"])
    return out


def test_floor_bound_catches_a_coarser_kernel():
    """Probabilities kept to 5 significant bits instead of 8: inside the max/peak bound, but
    more than twice the ideal floor, so the floor check rejects it."""
    x = _x(N=256, causal=False, seed=11)
    O, _ = _exact(x)
    ideal = ideal_forward(x)
    coarse = _degraded_forward(x, 5)
    r = errors(coarse, O)
    assert r["max_over_peak"] <= BF16_MAX_OVER_PEAK
    assert r["max_abs"] > FLOOR_FACTOR * float(np.max(np.abs(ideal - O))) + FLOOR_SLACK * np.max(np.abs(O))
    with pytest.raises(AssertionError):
        assert_bf16_close("O", coarse, O, ideal=ideal)


def test_floor_bound_passes_a_finer_kernel():
    """A kernel that skips the P rounding (exact up to its output rounding) is under the floor."""
    x = _x(N=256, causal=False, seed=12)
    O, _ = _exact(x)
    ideal = ideal_forward(x)
    finer = round_to(O, "bf16")
    assert_bf16_close("O", finer, O, ideal=ideal)


def test_dropout_and_packed_readings_reuse_the_oracle_masks():
    """With dropout or packed sequences the ideal kernel applies the oracle's own masks: its O
    differs from the oracle's by a bf16-sized amount only."""
    from oracle import dropout as od
    x = _x(N=200, causal=True, seed=13)
    drop = (7, 0, od.keep_threshold(0.2))
    O, _ = _exact(x, dropout=drop)
    ideal = ideal_forward(x, dropout=drop)
    r = errors(ideal, O)
    assert r["max_over_peak"] <= BF16_MAX_OVER_PEAK and r["max_abs"] > 0
    xs = _x(N=300, causal=True, seed=14)
    xs = dict(xs, q=xs["q"][:1], k=xs["k"][:1], v=xs["v"][:1], do=xs["do"][:1])
    seg = [0, 120, 300]
    O, _ = _exact(xs, segments=seg)
    r = errors(ideal_forward(xs, segments=seg), O)
    assert r["max_over_peak"] <= BF16_MAX_OVER_PEAK and r["max_abs"] > 0
