"""The error floor of an ideal 16-bit attention kernel, for the parity tests (test infrastructure).

A kernel that takes bf16 (or fp16) operands into fp32-accumulating tensor cores cannot be exact:
it holds the scores S, dP and the row term D in fp32, it must round the probabilities P (and,
backward, dS = P * (dP - D)) to the operand type before the next product, and it rounds O, dQ,
dK, dV to the output type.  The "ideal kernel" here is exact (fp64) except for exactly those
roundings, applied to the fp64 oracle's own quantities on the same inputs:

    forward :  S = fp32(scale * Q K^T),  LSE from S,  P = exp(S - LSE),
               O = out(op(P [* dropout mask]) V [* dropout scale])
    backward:  P as above,  dP = fp32(dO V^T) [* mask * scale],  D = fp32(rowsum(dO * O_in)),
               dS = fp32(P * (dP - D)),
               dV = out(op(P [* mask])^T dO [* scale]),  dQ = out(scale * op(dS) K),
               dK = out(scale * op(dS)^T Q)

where op() rounds to the operand type, out() to the output type, fp32() to float32, and O_in is
the O the backward is given (the ideal forward's O when the two are chained).  The floor of a
tensor is max |ideal - exact|; the parity tests require the GPU's max |got - exact| to stay
within a small multiple of it ("FlashAttention：让精确注意力服从内存层次", "数值与正确性": record
absolute and relative errors for FP32/BF16/FP16, since the result is not bitwise that of the
fp64 computation).

The masks, grouped heads, packed sequences and dropout follow the oracle's readings exactly (its
helpers are reused); only the roundings above are added.  No value here comes from the CUDA
path.
"""
from __future__ import annotations

import numpy as np
import torch

from oracle import attention as oa
from oracle import dropout as odrop

_TORCH = {"bf16": torch.bfloat16, "fp16": torch.float16}


def round_to(a, dtype: str):
    """fp64 array -> the nearest value of `dtype` ("fp32", "bf16", "fp16"), as fp64.  16-bit types
    go through fp32 first, as the kernel's fp32 registers do."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float64)).to(torch.float32)
    if dtype != "fp32":
        t = t.to(_TORCH[dtype])
    return t.to(torch.float64).numpy()


def _f64(t):
    return t.detach().to("cpu", torch.float64).numpy() if torch.is_tensor(t) else np.asarray(t, np.float64)


def _masks(x):
    kv = None if x.get("kv_lens") is None else np.asarray(x["kv_lens"])
    bm = None if x.get("block_mask") is None else np.asarray(x["block_mask"])
    return kv, bm


def _drop_factors(dropout, r, cols, bh):
    """(keep mask, scale) of the dropout reading, or (None, 1)."""
    if dropout is None:
        return None, 1.0
    seed, offset, k8 = dropout
    return odrop.keep_mask(r, cols, bh, seed, offset, k8).astype(np.float64), odrop.scale_of(k8)


def _chunk(q_rows, k_cols, scale, ok):
    """fp32 scores (masked to -inf), their LSE and P = exp(S - LSE)."""
    s = np.where(ok, round_to(scale * (q_rows @ k_cols.T), "fp32"), -np.inf)
    lse = oa._row_lse(s)
    return s, lse, oa._probs(s, lse)


def ideal_forward(x, heads=None, rows=None, segments=None, dropout=None):
    """The ideal kernel's O [B, H', R, d] (fp64 holding values of the output type)."""
    dt = x["dtype"]
    q, k, v = (_f64(x[n]) for n in ("q", "k", "v"))
    B, H, N, _ = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    kv, bm = _masks(x)
    lens = oa._as_i64_list(kv, B)
    rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = list(range(H)) if heads is None else list(heads)
    O = np.zeros((B, len(heads), rows.size, v.shape[3]))
    for b in range(B):
        for hi, h in enumerate(heads):
            g = oa.kv_head(h, H, Hkv)
            for c0 in range(0, rows.size, oa.ROW_CHUNK):
                r = rows[c0:c0 + oa.ROW_CHUNK]
                cols = oa._chunk_cols(r, Nk, x["causal"], lens[b], bm, segments)
                ok = oa.allowed(r, cols, x["causal"], lens[b], bm, segments)
                _, _, p = _chunk(q[b, h, r], k[b, g, cols], x["scale"], ok)
                mk, ds = _drop_factors(dropout, r, cols, b * H + h)
                if mk is not None:
                    p = p * mk
                O[b, hi, c0:c0 + r.size] = round_to(ds * (round_to(p, dt) @ v[b, g, cols]), dt)
    return O


def ideal_backward(x, heads=None, o=None, segments=None, dropout=None, rows=None):
    """The ideal kernel's (dQ, dK, dV), shaped like the oracle's backward.  `o` is the O the
    backward is given ([B, H, N, d]); by default the ideal forward's own O (chained).  `rows`
    restricts the work to those query rows, as in the oracle: dQ holds them, dK and dV only
    their contributions."""
    dt = x["dtype"]
    q, k, v, do = (_f64(x[n]) for n in ("q", "k", "v", "do"))
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    grouped = Hkv != H
    kv, bm = _masks(x)
    lens = oa._as_i64_list(kv, B)
    heads = list(range(H)) if heads is None else list(heads)
    all_rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    if o is None:           # the O of the same rows, in the order of all_rows
        o_in = ideal_forward(x, heads=heads, rows=all_rows, segments=segments, dropout=dropout)
    else:
        o_in = _f64(o)[:, heads][:, :, all_rows]
    dQ = np.zeros((B, len(heads), N, d))
    dK = np.zeros((B, Hkv if grouped else len(heads), k.shape[2], d))
    dV = np.zeros((B, Hkv if grouped else len(heads), v.shape[2], v.shape[3]))
    sc = x["scale"]
    for b in range(B):
        for hi, h in enumerate(heads):
            g = oa.kv_head(h, H, Hkv)
            kvi = g if grouped else hi
            for c0 in range(0, all_rows.size, oa.ROW_CHUNK):
                r = all_rows[c0:c0 + oa.ROW_CHUNK]
                cols = oa._chunk_cols(r, k.shape[2], x["causal"], lens[b], bm, segments)
                ok = oa.allowed(r, cols, x["causal"], lens[b], bm, segments)
                _, _, p = _chunk(q[b, h, r], k[b, g, cols], sc, ok)
                dp = round_to(do[b, h, r] @ v[b, g, cols].T, "fp32")
                mk, dsc = _drop_factors(dropout, r, cols, b * H + h)
                pd = p if mk is None else p * mk
                if mk is not None:
                    dp = dp * mk * dsc
                D = round_to((do[b, h, r] * o_in[b, hi, c0:c0 + r.size]).sum(axis=1), "fp32")
                ds = round_to(p * (dp - D[:, None]), "fp32")
                ds_op, p_op = round_to(ds, dt), round_to(pd, dt)
                dQ[b, hi, r] = sc * (ds_op @ k[b, g, cols])
                dK[b, kvi, cols] += sc * (ds_op.T @ q[b, h, r])
                dV[b, kvi, cols] += dsc * (p_op.T @ do[b, h, r])
    return round_to(dQ, dt), round_to(dK, dt), round_to(dV, dt)
