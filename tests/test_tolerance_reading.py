"""Derivation of the bf16 parity tolerance from the arithmetic (CPU only).

An ideal bf16-in / fp32-accumulate attention kernel is exact except for three roundings it
cannot avoid: the softmax numerator P (and, backward, dS) is rounded to bf16 to enter the
tensor-core product, and O, dQ, dK, dV are rounded to bf16 on output.  This test applies
exactly those roundings to the fp64 oracle's quantities and measures the error metrics.  It
shows that (a) mean-abs / RMS stays under 2e-3 and max-abs / peak under 2e-2 on every shape
class, while (b) max-abs / RMS exceeds 2e-2 on causal shapes, so the max bound is taken
relative to the tensor's peak magnitude (tests/tolerances.py).  The same holds when the
backward forms D = rowsum(dO * O) from the bf16 O the forward returns, on these workload-shaped
cases (the chained GPU tests compare against the exact gradient there).
"""
import numpy as np
import torch

import oracle
from tolerances import BF16_MAX_OVER_PEAK, BF16_MEAN_OVER_RMS, errors


def bf16(x):
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16).to(torch.float64).numpy()


def emulate(N, d, value_scale, causal, kv_len, seed, delta_from_rounded_o=False):
    rng = np.random.default_rng(seed)
    q, k, v = (bf16(rng.standard_normal((N, d)) * value_scale) for _ in range(3))
    do = bf16(rng.standard_normal((N, d)))
    scale = 1 / np.sqrt(d)
    one = lambda a: a[None, None]
    lens = None if kv_len is None else [kv_len]
    O, L = oracle.forward(one(q), one(k), one(v), scale, causal=causal, kv_lens=lens)
    dQ, dK, dV = oracle.backward(one(q), one(k), one(v), one(do), scale, causal=causal, kv_lens=lens)
    P = oracle.probabilities(q, k, scale, causal=causal, kv_len=kv_len)
    dP = do @ v.T
    if delta_from_rounded_o:     # D = rowsum(dO * O) with the bf16 O the forward returns
        dS = P * (dP - (do * bf16(O[0, 0])).sum(1, keepdims=True))
    else:
        dS = P * (dP - (P * dP).sum(1, keepdims=True))
    Pb, dSb = bf16(P), bf16(dS)
    got = dict(O=bf16(Pb @ v), dV=bf16(Pb.T @ do), dQ=bf16(scale * dSb @ k), dK=bf16(scale * dSb.T @ q))
    ref = dict(O=O[0, 0], dV=dV[0, 0], dQ=dQ[0, 0], dK=dK[0, 0])
    return {n: errors(got[n], ref[n]) for n in got}


def test_tolerance_reading():
    cases = [(512, 64, 1.0, False, 300), (1024, 64, 1.5, True, None),
             (2048, 128, 1.0, False, None), (2048, 128, 1.0, True, None)]
    worst_rms = 0.0
    for i, c in enumerate(cases + cases):
        res = emulate(*c, seed=i, delta_from_rounded_o=i >= len(cases))
        for name, r in res.items():
            assert r["mean_over_rms"] <= BF16_MEAN_OVER_RMS, (c, name, r)
            assert r["max_over_peak"] <= BF16_MAX_OVER_PEAK, (c, name, r)
            worst_rms = max(worst_rms, r["max_over_rms"])
    assert worst_rms > 2e-2     # why the max bound is not normalised by the RMS
