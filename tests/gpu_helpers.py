"""Helpers for the GPU parity tests: run the CUDA path through the C ABI, run the oracle on
the same seeded inputs, compare with the tolerances of tolerances.py."""
import numpy as np
import torch

import oracle
from tolerances import (FP32_MAX_ABS, assert_bf16_close, assert_fp32_close, assert_lse_close)

LSE_TOL_BF16 = 1e-3   # LSE is computed in fp32 from exact bf16 products; it is not rounded to bf16


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def to_dev(x, names=("q", "k", "v", "do")):
    dev = torch.device("cuda:0")
    return [x[n].to(dev) for n in names]


def np_masks(x):
    kv = None if x["kv_lens"] is None else x["kv_lens"].numpy()
    bm = None if x["block_mask"] is None else x["block_mask"].numpy()
    return kv, bm


def run_gpu(x, backward=True):
    import exact_io_aware_23_gb300 as fa
    q, k, v, do = to_dev(x)
    bm = None if x["block_mask"] is None else x["block_mask"].to(q.device)
    kl = None if x["kv_lens"] is None else x["kv_lens"].to(q.device)
    o, lse = fa.forward(q, k, v, causal=x["causal"], scale=x["scale"], block_mask=bm, kv_lens=kl)
    out = dict(o=o, lse=lse)
    if backward:
        dq, dk, dv = fa.backward(q, k, v, o, lse, do, causal=x["causal"], scale=x["scale"],
                                 block_mask=bm, kv_lens=kl)
        out.update(dq=dq, dk=dk, dv=dv)
    assert fa.check_device_status() == 0
    return out


def compare(x, out, heads=None, rows=None, backward=True):
    """Oracle on the given heads (all by default) and compare every output."""
    kv, bm = np_masks(x)
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    hs = list(range(qq.shape[1])) if heads is None else list(heads)
    O, L = oracle.forward(qq, kk, vv, x["scale"], causal=x["causal"], kv_lens=kv, block_mask=bm,
                          heads=hs, rows=rows)
    sel = (slice(None), hs) if rows is None else (slice(None), hs, rows)
    go = f64(out["o"])[:, hs] if rows is None else f64(out["o"])[:, hs][:, :, rows]
    gl = f64(out["lse"])[:, hs] if rows is None else f64(out["lse"])[:, hs][:, :, rows]
    res = {}
    if x["dtype"] == "fp32":
        res["O"] = assert_fp32_close("O", go, O)
        neg = np.isneginf(L)
        assert np.array_equal(np.isneginf(gl), neg)
        res["LSE"] = assert_fp32_close("LSE", gl[~neg], L[~neg])
    else:
        res["O"] = assert_bf16_close("O", go, O, is_output_O=True)
        res["LSE"] = assert_lse_close(gl, L, LSE_TOL_BF16)
    if backward and rows is None:
        dQ, dK, dV = oracle.backward(qq, kk, vv, dd, x["scale"], causal=x["causal"], kv_lens=kv,
                                     block_mask=bm, heads=hs)
        for name, key, ref in (("dQ", "dq", dQ), ("dK", "dk", dK), ("dV", "dv", dV)):
            got = f64(out[key])[:, hs]
            if x["dtype"] == "fp32":
                res[name] = assert_fp32_close(name, got, ref, FP32_MAX_ABS)
            else:
                res[name] = assert_bf16_close(name, got, ref)
    return res
