"""fp64 CPU oracle for exact attention: forward (O, LSE) and the explicit-gradient backward.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this module; only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py`` may call it.  It shares
no code, constant or helper with the CUDA library.

What it computes, and where the pages fix it:

* Attention is ``softmax(QK^T / sqrt(d)) V`` ("FlashAttention：让精确注意力服从内存层次", opening formula).  The method "computes the same function as standard attention"
  ("FlashAttention: Exact Attention with Less GPU Memory", "Why the word 'exact' is in the title"), so the oracle is that standard function, materialised: S = scale*Q K^T,
  P = softmax(S) row by row, O = P V ("前序瓶颈" three-line listing of the same page).  ``scale`` is an
  argument ("FlashAttention paper story"'s pseudocode has none, "FlashAttention：让精确注意力服从内存层次" uses 1/sqrt(d)).
* Masks ("FlashAttention：让精确注意力服从内存层次", list after the "CPU reference": causal / padding masks for production
  semantics; "FlashAttention paper story", block-sparse paragraph: a tile mask says which blocks are computed).
  Entry (i, j) of one (b, h) slice is allowed iff
  ``(not causal or j <= i) and j < kv_len[b] and block_mask[i // 128][j // 128] != 0``.
  Disallowed scores are -inf.  A row with no allowed key has O = 0 and LSE = -inf (the pages
  only ask that fully masked rows be covered, "FlashAttention：让精确注意力服从内存层次", "数值与正确性").
* Statistics kept for the backward: "FlashAttention paper story" (backward paragraph) keeps two length-N vectors
  (running max and normaliser).  The oracle returns the one equivalent vector
  ``LSE_i = ln sum_j exp(s_ij)`` (natural log), computed stably as ``m_i + ln sum exp(s_ij - m_i)``.
* Backward: the pages say only that P is recomputed from the stored statistics ("FlashAttention paper story",
  backward paragraph; "FlashAttention: Exact Attention with Less GPU Memory", "Tiling, and paying arithmetic to avoid memory").  The gradients
  of O = softmax(S) V with S = scale*Q K^T follow from the chain rule:
  dV = P^T dO;  dP = dO V^T;  D_i = sum_j P_ij dP_ij;  dS = P * (dP - D);
  dQ = scale * dS K;  dK = scale * dS^T Q.
  The oracle forms D from P and dP (its definition); the CUDA path uses rowsum(dO * O), equal
  in exact arithmetic.
* ``stats``, ``merge_stats`` and ``online_attention`` restate the pages' blockwise method: per
  key group statistics (m, l, u) and their merge law ("FlashAttention：让精确注意力服从内存层次", "Online softmax"), folded over
  the groups in key order (the running maximum and sum of "FlashAttention paper story", tiling and online
  softmax), so that the dense oracle can be checked against the pages' claim that the two agree
  ("FlashAttention：让精确注意力服从内存层次", "CPU reference": error below 1e-12 on its worked example).

* Grouped-query attention ("FlashAttention：让精确注意力服从内存层次", list after the "CPU reference": "GQA head mapping" among the
  production semantics).  The pages name the feature only; the oracle takes the usual reading:
  with H query heads and Hkv key/value heads (Hkv dividing H), query head h attends with
  key/value head h // (H / Hkv), so consecutive query heads share one key/value head.  In the
  backward, dK and dV of a key/value head are the sums over the query heads that read it (the
  chain rule through the shared operand).

* Ragged offsets and document masks (same page, same list: "document mask" and "ragged offsets").
  The pages name them only.  Reading: several sequences (documents) of lengths L_0, L_1, ...
  are packed back to back along the token axis, described by offsets ``segments`` =
  [0, L_0, L_0+L_1, ..., total]; a query attends only to keys of its own sequence (the
  document mask), and with ``causal`` only to keys at or before it.  Packed this way, B = 1 and
  N = total.

* Dropout on P (same list: "dropout RNG"; the numerics section asks for the dropout replay to
  be tested): ``dropout=(seed, offset, k8)`` applies the mask of ``oracle.dropout`` (Philox
  counter-based, so the backward regenerates it) as O = (P * M * 256/k8) V; LSE is that of the
  undropped scores; the backward uses the same mask.  See ``oracle/dropout.py`` for the reading.

Large inputs are processed a chunk of query rows at a time (a memory bound only: each chunk
still forms its full score rows).  When a tile mask removes most columns, a chunk gathers
the columns that any of its rows may attend to; every other column is masked for the whole
chunk, contributes exp(-inf) = 0, and leaving it out changes no result.
"""
from __future__ import annotations

import math
from typing import Optional, Sequence

import numpy as np

from . import dropout as _dropout

TILE = 128          # block-mask granularity (score tiles of 128 x 128)
ROW_CHUNK = 1024    # query rows per chunk (bounds the size of one score block)


def _as_i64_list(x, B: int) -> list:
    if x is None:
        return [None] * B
    return [int(v) for v in np.asarray(x).reshape(-1)]


def kv_head(h: int, H: int, Hkv: int) -> int:
    """Key/value head read by query head h when H query heads share Hkv key/value heads."""
    if Hkv <= 0 or H % Hkv != 0:
        raise ValueError("the key/value heads must divide the query heads")
    return h // (H // Hkv)


def segment_of(x: np.ndarray, segments) -> np.ndarray:
    """Index of the packed sequence that holds each position (offsets [0, ..., total])."""
    return np.searchsorted(np.asarray(segments, dtype=np.int64), x, side="right") - 1


def allowed(rows: np.ndarray, cols: np.ndarray, causal: bool, kv_len: Optional[int],
            block_mask: Optional[np.ndarray], segments=None) -> np.ndarray:
    """Boolean [len(rows), len(cols)]: which (query, key) pairs enter the softmax."""
    ok = np.ones((rows.size, cols.size), dtype=bool)
    if segments is not None:
        ok &= segment_of(rows, segments)[:, None] == segment_of(cols, segments)[None, :]
    if causal:
        ok &= cols[None, :] <= rows[:, None]
    if kv_len is not None:
        ok &= (cols < kv_len)[None, :]
    if block_mask is not None:
        bm = np.asarray(block_mask) != 0
        ok &= bm[(rows // TILE)[:, None], (cols // TILE)[None, :]]
    return ok


def _chunk_cols(rows: np.ndarray, N: int, causal: bool, kv_len, block_mask,
                segments=None) -> np.ndarray:
    """Columns any row of the chunk may attend to (all N when nothing restricts them)."""
    if block_mask is None and kv_len is None and not causal and segments is None:
        return np.arange(N)
    cols = np.arange(N)
    ok = allowed(rows, cols, causal, kv_len, block_mask, segments)
    keep = ok.any(axis=0)
    return cols[keep]


def _scores(q_rows: np.ndarray, k_cols: np.ndarray, scale: float, ok: np.ndarray) -> np.ndarray:
    s = scale * (q_rows @ k_cols.T)
    return np.where(ok, s, -np.inf)


def _row_lse(s: np.ndarray) -> np.ndarray:
    """ln sum_j exp(s_ij) per row; -inf for rows with no finite entry."""
    m = s.max(axis=1) if s.shape[1] else np.full(s.shape[0], -np.inf)
    finite = np.isfinite(m)
    m0 = np.where(finite, m, 0.0)
    with np.errstate(divide="ignore"):
        lse = m0 + np.log(np.exp(s - m0[:, None]).sum(axis=1)) if s.shape[1] else np.full(s.shape[0], -np.inf)
    return np.where(finite, lse, -np.inf)


def _probs(s: np.ndarray, lse: np.ndarray) -> np.ndarray:
    finite = np.isfinite(lse)
    p = np.exp(s - np.where(finite, lse, 0.0)[:, None])
    p[~finite, :] = 0.0
    return p


def _check_segments(segments, B: int, N: int, kv_lens):
    if segments is None:
        return
    seg = np.asarray(segments, dtype=np.int64)
    if B != 1 or kv_lens is not None or seg[0] != 0 or seg[-1] != N or np.any(np.diff(seg) < 0):
        raise ValueError("packed sequences need B = 1, no kv_lens and offsets 0 <= ... <= N = total")


def _drop(dropout, r, cols, bh):
    """(mask-and-scale factor [len(r), len(cols)]) of the dropout reading, or None."""
    if dropout is None:
        return None
    seed, offset, k8 = dropout
    return _dropout.keep_mask(r, cols, bh, seed, offset, k8) * _dropout.scale_of(k8)


def forward(q, k, v, scale: float, causal: bool = False, kv_lens=None, block_mask=None,
            rows: Optional[Sequence[int]] = None, heads: Optional[Sequence[int]] = None,
            segments=None, dropout=None):
    """Dense masked attention in fp64.

    q: float64 array [B, H, N, d]; k, v: [B, Hkv, N, d] with Hkv dividing H (query head h reads
    key/value head h // (H / Hkv); Hkv = H is ordinary multi-head attention).  k and v may have
    a different N only when neither causal nor a block mask is set.  Returns
    (O [B,H,R,d], LSE [B,H,R]) for the R query rows in ``rows`` (default: all rows) and the
    heads in ``heads`` (default: all heads).  ``segments``: offsets of packed sequences along
    the token axis (B = 1); a query sees only the keys of its own sequence.  ``dropout``:
    (seed, offset, k8) of ``oracle.dropout`` (not combined with ``segments``).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, Nq, d = q.shape
    Nk = k.shape[2]
    _check_segments(segments, B, Nq, kv_lens)
    if dropout is not None and segments is not None:
        raise ValueError("dropout with packed sequences is not part of this reading")
    rows = np.arange(Nq) if rows is None else np.asarray(rows, dtype=np.int64)
    heads = list(range(H)) if heads is None else list(heads)
    lens = _as_i64_list(kv_lens, B)
    Hkv = k.shape[1]
    O = np.zeros((B, len(heads), rows.size, v.shape[3]))
    L = np.full((B, len(heads), rows.size), -np.inf)
    for b in range(B):
        for hi, h in enumerate(heads):
            g = kv_head(h, H, Hkv)
            for c0 in range(0, rows.size, ROW_CHUNK):
                r = rows[c0:c0 + ROW_CHUNK]
                cols = _chunk_cols(r, Nk, causal, lens[b], block_mask, segments)
                ok = allowed(r, cols, causal, lens[b], block_mask, segments)
                s = _scores(q[b, h, r], k[b, g, cols], scale, ok)
                lse = _row_lse(s)
                p = _probs(s, lse)
                mk = _drop(dropout, r, cols, b * H + h)
                if mk is not None:
                    p = p * mk
                O[b, hi, c0:c0 + r.size] = p @ v[b, g, cols]
                L[b, hi, c0:c0 + r.size] = lse
    return O, L


def probabilities(q, k, scale: float, causal: bool = False, kv_len=None, block_mask=None):
    """P = softmax(S) for one (b, h) slice: q [Nq, d], k [Nk, d] -> [Nq, Nk] (rows sum to 1)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    rows, cols = np.arange(q.shape[0]), np.arange(k.shape[0])
    s = _scores(q, k, scale, allowed(rows, cols, causal, kv_len, block_mask))
    return _probs(s, _row_lse(s))


def backward(q, k, v, do, scale: float, causal: bool = False, kv_lens=None, block_mask=None,
             heads: Optional[Sequence[int]] = None, return_delta: bool = False,
             rows: Optional[Sequence[int]] = None, o=None, segments=None, dropout=None):
    """Explicit-gradient backward of dense masked attention, fp64.

    Returns (dQ, dK, dV), each [B, len(heads), N, d]; with ``return_delta`` also D [B,H',N].
    With fewer key/value heads than query heads (k, v [B, Hkv, N, d]; see ``forward``), dK and
    dV are [B, Hkv, N, d] and each key/value head sums the contributions of the selected query
    heads that read it.  ``segments`` and ``dropout`` as in ``forward``: with dropout,
    dV = (P * M * s)^T dO and dP = (dO V^T) * M * s (s = 256 / k8), D and dS as without it.
    D_i = sum_j P_ij dP_ij, the exact gradient's row term.  When the forward output ``o``
    ([B,H,N,d]) is given, D_i = sum_c dO_ic o_ic instead: the backward as an operator of its
    inputs (q, k, v, o, dO, LSE), the form the method's backward takes (equal to the first
    when o is the exact forward output).  Rows whose LSE is -inf contribute nothing.  ``rows``
    restricts the computation to those query rows: dQ and D are filled for them only and dK,
    dV hold only their contributions (a sample of the work, used for timing).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, N, d = q.shape
    _check_segments(segments, B, N, kv_lens)
    if dropout is not None and segments is not None:
        raise ValueError("dropout with packed sequences is not part of this reading")
    heads = list(range(H)) if heads is None else list(heads)
    lens = _as_i64_list(kv_lens, B)
    Hkv = k.shape[1]
    grouped = Hkv != H
    dQ = np.zeros((B, len(heads), N, d))
    dK = np.zeros((B, Hkv if grouped else len(heads), k.shape[2], d))
    dV = np.zeros((B, Hkv if grouped else len(heads), v.shape[2], v.shape[3]))
    Dd = np.zeros((B, len(heads), N))
    all_rows = np.arange(N) if rows is None else np.asarray(rows, dtype=np.int64)
    for b in range(B):
        for hi, h in enumerate(heads):
            g = kv_head(h, H, Hkv)
            kvi = g if grouped else hi
            for c0 in range(0, all_rows.size, ROW_CHUNK):
                r = all_rows[c0:c0 + ROW_CHUNK]
                cols = _chunk_cols(r, k.shape[2], causal, lens[b], block_mask, segments)
                ok = allowed(r, cols, causal, lens[b], block_mask, segments)
                s = _scores(q[b, h, r], k[b, g, cols], scale, ok)
                p = _probs(s, _row_lse(s))
                dp = do[b, h, r] @ v[b, g, cols].T
                mk = _drop(dropout, r, cols, b * H + h)
                pd = p if mk is None else p * mk           # the probabilities O was built from
                if mk is not None:
                    dp = dp * mk
                if o is None:
                    D = (p * dp).sum(axis=1)
                else:
                    D = (do[b, h, r] * np.asarray(o, dtype=np.float64)[b, h, r]).sum(axis=1)
                ds = p * (dp - D[:, None])
                dQ[b, hi, r] = scale * (ds @ k[b, g, cols])
                dK[b, kvi, cols] += scale * (ds.T @ q[b, h, r])
                dV[b, kvi, cols] += pd.T @ do[b, h, r]
                Dd[b, hi, r] = D
    if return_delta:
        return dQ, dK, dV, Dd
    return dQ, dK, dV


# --- the pages' own blockwise algorithm, for pinning the dense oracle -----------------------

def stats(scores: np.ndarray, values: np.ndarray):
    """(m, l, u) of one group of scores for one query ("FlashAttention：让精确注意力服从内存层次", "Online softmax").

    m = max_i s_i, l = sum_i exp(s_i - m), u = sum_i exp(s_i - m) v_i.  An empty or fully
    masked group is the identity (-inf, 0, 0).
    """
    scores = np.asarray(scores, dtype=np.float64)
    values = np.asarray(values, dtype=np.float64)
    if scores.size == 0 or not np.isfinite(scores).any():
        return -math.inf, 0.0, np.zeros(values.shape[-1])
    m = float(scores.max())
    w = np.exp(scores - m)
    return m, float(w.sum()), w @ values


def merge_stats(a, b):
    """Stable merge of two (m, l, u) triples ("FlashAttention：让精确注意力服从内存层次", merge law under "Online softmax")."""
    ma, la, ua = a
    mb, lb, ub = b
    m = max(ma, mb)
    if m == -math.inf:
        return -math.inf, 0.0, np.zeros_like(np.asarray(ua, dtype=np.float64))
    fa = math.exp(ma - m) if ma != -math.inf else 0.0
    fb = math.exp(mb - m) if mb != -math.inf else 0.0
    return m, fa * la + fb * lb, fa * np.asarray(ua) + fb * np.asarray(ub)


def online_attention(q, k, v, scale: float, block_size: int):
    """Blockwise attention for one (b, h) slice, no masks, built on the merge law.

    q [Nq, d], k [Nk, d], v [Nk, dv].  The keys are cut into consecutive groups of
    ``block_size``.  For every query, each group is reduced to its statistics (m, l, u) by
    ``stats`` and the groups are combined, in key order, by ``merge_stats``; the result is
    O = u / l and LSE = m + ln l ("FlashAttention：让精确注意力服从内存层次", section
    "Online softmax": a tile's (m, l, u) can be computed on its own and merged; the same idea
    as the running maximum and normaliser of "FlashAttention paper story", tiling and
    online-softmax paragraphs).  A pure-Python loop over queries and groups: small inputs only.
    Returns (O [Nq, dv], LSE [Nq]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    groups = [np.arange(g0, min(g0 + block_size, k.shape[0]))
              for g0 in range(0, k.shape[0], block_size)]
    out = np.zeros((q.shape[0], v.shape[1]))
    lse = np.full(q.shape[0], -np.inf)
    for i, qi in enumerate(q):
        total = (-math.inf, 0.0, np.zeros(v.shape[1]))
        for cols in groups:
            total = merge_stats(total, stats(scale * (k[cols] @ qi), v[cols]))
        m, l, u = total
        if l > 0.0:
            out[i] = u / l
            lse[i] = m + math.log(l)
    return out, lse
