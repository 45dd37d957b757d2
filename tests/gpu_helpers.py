"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and the oracle on the
same seeded inputs, and compare with the tolerances of tolerances.py.

Two ways of checking the backward:
  * chained: the GPU backward gets the GPU forward's O and LSE and is compared with the exact
    gradient (D from P).  Used on the workload shapes.
  * given O: the GPU backward gets O and LSE computed by the oracle (rounded on the CPU to the
    dtype the kernel takes) and is compared with the oracle's backward for that same O
    (D = rowsum(dO * O)).  This isolates the backward kernel; it is used for edge cases (tiny N,
    one-hot rows) where rounding O to bf16 alone moves the exact gradient more than the bound.
"""
import numpy as np
import torch

import oracle
from ideal_kernel import ideal_backward, ideal_forward
from tolerances import (FP32_MAX_ABS, assert_bf16_close, assert_fp32_close, assert_lse_close)

LSE_TOL_BF16 = 1e-3   # LSE is computed in fp32 from exact bf16 products; it is not rounded to bf16


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def np_masks(x):
    kv = None if x["kv_lens"] is None else x["kv_lens"].numpy()
    bm = None if x["block_mask"] is None else x["block_mask"].numpy()
    return kv, bm


def _dev(x):
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    bm = None if x["block_mask"] is None else x["block_mask"].to(dev)
    kl = None if x["kv_lens"] is None else x["kv_lens"].to(dev)
    return q, k, v, do, dict(causal=x["causal"], scale=x["scale"], block_mask=bm, kv_lens=kl)


def run_gpu(x, backward=True, deterministic=False, fused=False):
    """Chained GPU forward (and backward on the forward's own O, LSE)."""
    import exact_io_aware_23_gb300 as fa
    q, k, v, do, kw = _dev(x)
    o, lse = fa.forward(q, k, v, **kw)
    out = dict(o=o, lse=lse)
    if backward:
        dq, dk, dv = fa.backward(q, k, v, o, lse, do, deterministic=deterministic, fused=fused, **kw)
        out.update(dq=dq, dk=dk, dv=dv)
    assert fa.check_device_status() == 0
    return out


def oracle_fwd(x, heads=None, rows=None):
    kv, bm = np_masks(x)
    qq, kk, vv = (f64(x[n]) for n in ("q", "k", "v"))
    return oracle.forward(qq, kk, vv, x["scale"], causal=x["causal"], kv_lens=kv, block_mask=bm,
                          heads=heads, rows=rows)


def compare_fwd(x, out, heads=None, rows=None, ref=None):
    B, H = x["q"].shape[:2]
    hs = list(range(H)) if heads is None else list(heads)
    O, L = ref if ref is not None else oracle_fwd(x, hs, rows)
    go, gl = f64(out["o"])[:, hs], f64(out["lse"])[:, hs]
    if rows is not None:
        go, gl = go[:, :, rows], gl[:, :, rows]
    res = {}
    if x["dtype"] == "fp32":
        res["O"] = assert_fp32_close("O", go, O)
        neg = np.isneginf(L)
        assert np.array_equal(np.isneginf(gl), neg)
        res["LSE"] = assert_fp32_close("LSE", gl[~neg], L[~neg])
    else:
        res["O"] = assert_bf16_close("O", go, O, ideal=ideal_forward(x, heads=hs, rows=rows))
        res["LSE"] = assert_lse_close(gl, L, LSE_TOL_BF16)
    return res


def compare_bwd(x, grads, heads=None, o_given=None):
    kv, bm = np_masks(x)
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    H = qq.shape[1]
    hs = list(range(H)) if heads is None else list(heads)
    og = None if o_given is None else o_given
    dQ, dK, dV, D = oracle.backward(qq, kk, vv, dd, x["scale"], causal=x["causal"], kv_lens=kv,
                                    block_mask=bm, heads=hs, o=og, return_delta=True)
    dmax = float(np.max(np.abs(D))) if D.size else 0.0
    cancel = {"dQ": x["scale"] * dmax * float(np.max(np.abs(kk), initial=0.0)),
              "dK": x["scale"] * dmax * float(np.max(np.abs(qq), initial=0.0)), "dV": 0.0}
    grouped = kk.shape[1] != H          # dK, dV then hold the key/value heads' group sums
    assert not (grouped and heads is not None)
    ideal = (None, None, None) if x["dtype"] == "fp32" else ideal_backward(x, heads=hs, o=og)
    res = {}
    for name, key, ref, idl in (("dQ", "dq", dQ, ideal[0]), ("dK", "dk", dK, ideal[1]),
                                ("dV", "dv", dV, ideal[2])):
        got = f64(grads[key]) if grouped and key != "dq" else f64(grads[key])[:, hs]
        if x["dtype"] == "fp32":
            res[name] = assert_fp32_close(name, got, ref, FP32_MAX_ABS)
        else:
            res[name] = assert_bf16_close(name, got, ref, ideal=idl, cancel_scale=cancel[name])
    return res


def compare(x, out, heads=None, rows=None, backward=True):
    """Chained check: forward against the oracle; backward against the exact gradient."""
    res = compare_fwd(x, out, heads, rows)
    if backward and rows is None:
        res.update(compare_bwd(x, out, heads))
    return res


def check_backward_given_o(x, deterministic=False, fused=False):
    """GPU backward on the oracle's O (rounded to the working dtype) and LSE, against the
    oracle's backward for that O; forward checked separately."""
    import exact_io_aware_23_gb300 as fa
    O, L = oracle_fwd(x)
    dt = x["q"].dtype
    o_in = torch.from_numpy(O).to(dt)
    lse_in = torch.from_numpy(L).to(torch.float32)
    q, k, v, do, kw = _dev(x)
    dev = q.device
    dq, dk, dv = fa.backward(q, k, v, o_in.to(dev), lse_in.to(dev), do, deterministic=deterministic,
                             fused=fused, **kw)
    assert fa.check_device_status() == 0
    return compare_bwd(x, dict(dq=dq, dk=dk, dv=dv), o_given=o_in.to(torch.float64).numpy())
