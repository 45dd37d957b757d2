"""Pins for the fp64 oracle against what the pages and the mathematics fix (CPU only).

Each test names the passage or the mathematical fact it relies on.  None of them re-types the
oracle's formula: they use the pages' worked example and acceptance rule, hand-derived values,
closed forms, invariants, brute force on tiny inputs and finite differences.
"""
import json
import math
import os

import numpy as np
import pytest

import oracle
from oracle import attention as oa

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _one(x):
    """[n, d] -> [1, 1, n, d]"""
    return np.asarray(x, dtype=np.float64)[None, None]


# --- worked example of the "CPU reference" section ------------------------------------------------------------------

def _worked():
    with open(os.path.join(GOLDEN, "worked_example_cpu_reference.json")) as f:
        g = json.load(f)
    return np.array(g["q"]), np.array(g["k"]), np.array(g["v"]), g


def test_worked_example_blockwise_equals_dense():
    """"FlashAttention：让精确注意力服从内存层次", "CPU reference": the blockwise result equals the dense one to < 1e-12 and is finite."""
    q, k, v, g = _worked()
    scale = 1.0 / math.sqrt(q.shape[1])
    O_dense, L_dense = oracle.forward(_one(q), _one(k), _one(v), scale)
    O_blk, L_blk = oracle.online_attention(q, k, v, scale, block_size=g["block_size"])
    assert np.all(np.isfinite(O_blk))
    assert np.max(np.abs(O_blk - O_dense[0, 0])) < g["max_abs_error"]
    assert np.max(np.abs(L_blk - L_dense[0, 0])) < g["max_abs_error"]


def test_worked_example_hand_scores():
    """Brute force on the "CPU reference" example with dot products worked out by hand.

    q0 . k_j = [0, -1/2, 3, 3/2, -5/4] and q1 . k_j = [1, 9/2, 0, -2, 5/2]; the scores are these
    over sqrt(3).  LSE is the natural log of the sum of exponentials; O the weighted mean of v.
    """
    q, k, v, _ = _worked()
    dots = [[0.0, -0.5, 3.0, 1.5, -1.25], [1.0, 4.5, 0.0, -2.0, 2.5]]
    O, L = oracle.forward(_one(q), _one(k), _one(v), 1.0 / math.sqrt(3.0))
    for i, row in enumerate(dots):
        w = [math.exp(x / math.sqrt(3.0)) for x in row]
        tot = sum(w)
        assert abs(L[0, 0, i] - math.log(tot)) < 1e-13
        for c in range(2):
            expect = sum(wj * v[j][c] for j, wj in enumerate(w)) / tot
            assert abs(O[0, 0, i, c] - expect) < 1e-13


# --- merge law ("Online softmax") ---------------------------------------------------

def _random_partition(n, rng):
    cuts = sorted(rng.choice(np.arange(1, n), size=rng.integers(1, min(n - 1, 8) + 1), replace=False))
    edges = [0] + list(cuts) + [n]
    return [np.arange(edges[i], edges[i + 1]) for i in range(len(edges) - 1)]


@pytest.mark.parametrize("seed", range(6))
def test_merge_law_any_order_any_tree(seed):
    """Merging per-part (m, l, u) in any order or tree shape gives the whole group's triple."""
    rng = np.random.default_rng(seed)
    n, dv = 41, 3
    s = rng.standard_normal(n) * 4.0
    vals = rng.standard_normal((n, dv))
    m0, l0, u0 = oracle.stats(s, vals)
    parts = _random_partition(n, rng)
    triples = [oracle.stats(s[p], vals[p]) for p in parts]
    # left fold in a random order
    order = rng.permutation(len(triples))
    acc = (-math.inf, 0.0, np.zeros(dv))
    for i in order:
        acc = oracle.merge_stats(acc, triples[i])
    # random binary tree
    pool = list(triples)
    while len(pool) > 1:
        i, j = sorted(rng.choice(len(pool), size=2, replace=False))
        b = pool.pop(j)
        a = pool.pop(i)
        pool.append(oracle.merge_stats(a, b) if rng.random() < 0.5 else oracle.merge_stats(b, a))
    for m, l, u in (acc, pool[0]):
        assert m == m0
        assert abs(l - l0) <= 1e-12 * l0
        assert np.max(np.abs(u - u0)) <= 1e-12 * max(1.0, np.max(np.abs(u0)))


def test_merge_identity():
    """(-inf, 0, 0) is the identity of the merge."""
    t = oracle.stats(np.array([0.3, -1.0, 2.0]), np.eye(3))
    ident = (-math.inf, 0.0, np.zeros(3))
    for r in (oracle.merge_stats(t, ident), oracle.merge_stats(ident, t)):
        assert r[0] == t[0] and r[1] == t[1] and np.array_equal(r[2], t[2])


def test_merge_matches_dense_output():
    """u / l after merging the per-block triples is the dense O; m + ln l is the dense LSE."""
    q, k, v = _rand((6, 4), 1), _rand((50, 4), 2), _rand((50, 3), 3)
    scale = 0.5
    O, L = oracle.forward(_one(q), _one(k), _one(v), scale)
    parts = [np.arange(0, 7), np.arange(7, 30), np.arange(30, 50)]
    for i in range(q.shape[0]):
        acc = (-math.inf, 0.0, np.zeros(3))
        for p in parts[::-1]:
            acc = oracle.merge_stats(acc, oracle.stats(scale * (k[p] @ q[i]), v[p]))
        m, l, u = acc
        assert np.max(np.abs(u / l - O[0, 0, i])) < 1e-12
        assert abs(m + math.log(l) - L[0, 0, i]) < 1e-12


@pytest.mark.parametrize("block", [1, 2, 3, 16, 64, 200])
def test_online_algorithm_equals_dense(block):
    """The blockwise algorithm (merge law folded over key groups) gives the dense result."""
    q, k, v = _rand((9, 5), 4, 2.0), _rand((57, 5), 5, 2.0), _rand((57, 2), 6)
    O, L = oracle.forward(_one(q), _one(k), _one(v), 0.7)
    Ob, Lb = oracle.online_attention(q, k, v, 0.7, block)
    assert np.max(np.abs(Ob - O[0, 0])) < 1e-12
    assert np.max(np.abs(Lb - L[0, 0])) < 1e-12


# --- softmax properties ---------------------------------------------------------------------

@pytest.mark.parametrize("causal,kv_len", [(False, None), (True, None), (False, 70), (True, 40)])
def test_rows_sum_to_one(causal, kv_len):
    q, k = _rand((150, 8), 7), _rand((150, 8), 8)
    P = oracle.probabilities(q, k, 0.35, causal=causal, kv_len=kv_len)
    sums = P.sum(axis=1)
    assert np.all(np.abs(sums - 1.0) < 1e-13)
    assert np.all(P >= 0)


def test_shift_invariance_api_level():
    """K' = K + 1 w^T adds scale*q_i.w to every score of row i: O is unchanged and LSE shifts by it."""
    B, H, N, d = 2, 2, 70, 8
    q, k, v = _rand((B, H, N, d), 9), _rand((B, H, N, d), 10), _rand((B, H, N, d), 11)
    w = _rand((d,), 12)
    scale = 1 / math.sqrt(d)
    for causal in (False, True):
        O, L = oracle.forward(q, k, v, scale, causal=causal)
        O2, L2 = oracle.forward(q, k + w, v, scale, causal=causal)
        assert np.max(np.abs(O2 - O)) < 1e-12
        assert np.max(np.abs(L2 - (L + scale * (q @ w)))) < 1e-12


def _n_allowed_closed_form(i, N, causal, kv_len, bm):
    """Number of keys row i may attend to, counted from the mask definitions."""
    hi = N
    if kv_len is not None:
        hi = min(hi, kv_len)
    if causal:
        hi = min(hi, i + 1)
    if bm is None:
        return max(hi, 0), None
    cols = [j for j in range(hi) if bm[i // 128][j // 128]]
    return len(cols), cols


@pytest.mark.parametrize("causal,kv_len,use_bm", [(False, None, False), (True, None, False),
                                                  (False, 200, False), (True, 150, False),
                                                  (False, None, True), (True, 290, True)])
def test_zero_queries_give_mean_of_values(causal, kv_len, use_bm):
    """Q = 0: all allowed scores are 0, so O_i is the plain mean of the allowed v_j, LSE_i = ln(count)."""
    N, d = 300, 4
    k, v = _rand((N, d), 13), _rand((N, d), 14)
    bm = None
    if use_bm:
        bm = np.array([[1, 0, 1], [0, 1, 0], [1, 1, 0]], dtype=np.uint8)
    O, L = oracle.forward(_one(np.zeros((N, d))), _one(k), _one(v), 0.9, causal=causal,
                          kv_lens=None if kv_len is None else [kv_len], block_mask=bm)
    for i in range(N):
        n, cols = _n_allowed_closed_form(i, N, causal, kv_len, bm)
        if n == 0:
            assert np.all(O[0, 0, i] == 0) and L[0, 0, i] == -np.inf
            continue
        mean = v[:n].mean(axis=0) if cols is None else v[cols].mean(axis=0)
        assert np.max(np.abs(O[0, 0, i] - mean)) < 1e-12
        assert abs(L[0, 0, i] - math.log(n)) < 1e-12


def test_single_key():
    """N = 1: O = v_0 and LSE = scale * q.k."""
    q, k, v = _rand((1, 6), 15), _rand((1, 6), 16), _rand((1, 6), 17)
    O, L = oracle.forward(_one(q), _one(k), _one(v), 0.3)
    assert np.max(np.abs(O[0, 0, 0] - v[0])) < 1e-15
    assert abs(L[0, 0, 0] - 0.3 * float(q[0] @ k[0])) < 1e-14


def test_constant_values():
    """V = c on every key: O = c for every row with an allowed key."""
    q, k = _rand((64, 5), 18, 3.0), _rand((64, 5), 19, 3.0)
    c = np.array([1.5, -2.0, 0.25, 7.0, 0.0])
    O, _ = oracle.forward(_one(q), _one(k), _one(np.tile(c, (64, 1))), 0.5, causal=True)
    assert np.max(np.abs(O[0, 0] - c)) < 1e-12


def test_permutation_equivariance():
    """Permuting keys and values together changes nothing; permuting queries permutes O."""
    rng = np.random.default_rng(20)
    q, k, v = _rand((33, 6), 21), _rand((45, 6), 22), _rand((45, 6), 23)
    O, L = oracle.forward(_one(q), _one(k), _one(v), 0.4)
    pk = rng.permutation(45)
    O2, L2 = oracle.forward(_one(q), _one(k[pk]), _one(v[pk]), 0.4)
    assert np.max(np.abs(O2 - O)) < 1e-12 and np.max(np.abs(L2 - L)) < 1e-12
    pq = rng.permutation(33)
    O3, L3 = oracle.forward(_one(q[pq]), _one(k), _one(v), 0.4)
    assert np.max(np.abs(O3[0, 0] - O[0, 0, pq])) < 1e-12
    assert np.max(np.abs(L3[0, 0] - L[0, 0, pq])) < 1e-12


def test_fully_masked_rows():
    """A row with no allowed key: O = 0, LSE = -inf, and its gradients vanish (finite everywhere)."""
    B, H, N, d = 2, 1, 260, 4
    q, k, v, do = (_rand((B, H, N, d), s) for s in (24, 25, 26, 27))
    bm = np.array([[1, 1, 0], [0, 0, 0], [1, 0, 1]], dtype=np.uint8)   # tile row 1 all masked
    lens = [0, 200]                                                      # batch 0: no valid key
    O, L = oracle.forward(q, k, v, 0.5, kv_lens=lens, block_mask=bm)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.5, kv_lens=lens, block_mask=bm)
    assert np.all(O[0] == 0) and np.all(L[0] == -np.inf)
    assert np.all(O[1, :, 128:256] == 0) and np.all(L[1, :, 128:256] == -np.inf)
    assert np.all(dQ[0] == 0) and np.all(dK[0] == 0) and np.all(dV[0] == 0)
    assert np.all(dQ[1, :, 128:256] == 0)
    assert np.all(dK[1, :, 200:] == 0) and np.all(dV[1, :, 200:] == 0)
    for t in (O, dQ, dK, dV):
        assert np.all(np.isfinite(t))


def test_extreme_logits():
    """Scores of +-60 (scale 1): finite results equal to the closed form."""
    q = _one([[60.0], [-60.0], [0.5]])
    k = _one([[1.0], [-1.0]])
    v = _one([[2.0, -1.0], [5.0, 3.0]])
    O, L = oracle.forward(q, k, v, 1.0)
    e = math.exp(-120.0)
    assert abs(L[0, 0, 0] - (60.0 + math.log1p(e))) < 1e-12
    assert np.max(np.abs(O[0, 0, 0] - (v[0, 0, 0] + e * v[0, 0, 1]) / (1 + e))) < 1e-15
    assert np.max(np.abs(O[0, 0, 1] - (e * v[0, 0, 0] + v[0, 0, 1]) / (1 + e))) < 1e-15
    # a larger random case pushed to +-60
    qq, kk = _rand((40, 4), 28), _rand((40, 4), 29)
    s = qq @ kk.T
    scl = 60.0 / np.abs(s).max()
    O2, L2 = oracle.forward(_one(qq), _one(kk), _one(_rand((40, 3), 30)), scl)
    P = oracle.probabilities(qq, kk, scl)
    assert np.all(np.isfinite(O2)) and np.all(np.isfinite(L2))
    assert np.all(np.abs(P.sum(1) - 1) < 1e-13)


def test_gather_path_equals_full_rows():
    """With a tile mask the oracle gathers the columns a chunk may use; the result equals the
    dense row softmax over all N columns (probabilities() never gathers)."""
    N, d = 700, 8
    q, k, v = _rand((N, d), 31), _rand((N, d), 32), _rand((N, d), 33)
    nt = (N + 127) // 128
    bm = (np.random.default_rng(34).random((nt, nt)) < 0.4).astype(np.uint8)
    bm[2, :] = 0
    for causal in (False, True):
        O, _ = oracle.forward(_one(q), _one(k), _one(v), 0.3, causal=causal, block_mask=bm)
        P = oracle.probabilities(q, k, 0.3, causal=causal, block_mask=bm)
        assert np.max(np.abs(O[0, 0] - P @ v)) < 1e-12


def test_row_chunking_does_not_change_results(monkeypatch):
    q, k, v, do = (_rand((1, 2, 300, 8), s) for s in (35, 36, 37, 38))
    ref = oracle.forward(q, k, v, 0.3, causal=True) + oracle.backward(q, k, v, do, 0.3, causal=True)
    monkeypatch.setattr(oa, "ROW_CHUNK", 37)
    got = oracle.forward(q, k, v, 0.3, causal=True) + oracle.backward(q, k, v, do, 0.3, causal=True)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) < 1e-12


# --- backward -------------------------------------------------------------------------------

def _loss(q, k, v, do, scale, **kw):
    O, _ = oracle.forward(q, k, v, scale, **kw)
    return float((O * do).sum())


@pytest.mark.parametrize("case", ["plain", "causal", "kvlen", "blockmask"])
def test_backward_finite_differences(case):
    """Central differences of L = sum(dO * O) match the analytic gradients (fp64)."""
    kw = {}
    N, d = 7, 3
    if case == "causal":
        kw = dict(causal=True)
    elif case == "kvlen":
        kw = dict(kv_lens=[5])
    elif case == "blockmask":
        N, d = 131, 2                      # two tile rows/cols: exercise the tile mask
        kw = dict(block_mask=np.array([[1, 0], [1, 1]], dtype=np.uint8), causal=True)
    q, k, v, do = (_rand((1, 1, N, d), s, 1.3) for s in (40, 41, 42, 43))
    scale = 0.8
    dQ, dK, dV = oracle.backward(q, k, v, do, scale, **kw)
    h = 1e-6
    rng = np.random.default_rng(44)
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        idxs = [tuple(int(i) for i in np.unravel_index(f, x.shape)) for f in
                (range(x.size) if x.size <= 30 else rng.choice(x.size, 30, replace=False))]
        for idx in idxs:
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, do=do, scale=scale, **kw)
            lm = _loss(**{**args, name: xm}, do=do, scale=scale, **kw)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


def test_gqa_backward_finite_differences():
    """Grouped heads: the gradients of K and V, which several query heads share, match central
    differences of L = sum(dO * O) over all query heads (fp64)."""
    H, Hkv, N, d = 4, 2, 6, 3
    q, do = (_rand((1, H, N, d), s, 1.2) for s in (140, 141))
    k, v = (_rand((1, Hkv, N, d), s, 1.2) for s in (142, 143))
    scale = 0.7
    dQ, dK, dV = oracle.backward(q, k, v, do, scale, causal=True)
    assert dK.shape == k.shape and dV.shape == v.shape and dQ.shape == q.shape
    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        for f in range(x.size):
            idx = tuple(int(i) for i in np.unravel_index(f, x.shape))
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, do=do, scale=scale, causal=True)
            lm = _loss(**{**args, name: xm}, do=do, scale=scale, causal=True)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


@pytest.mark.parametrize("Hkv", [1, 2, 3])
def test_gqa_equals_attention_with_repeated_heads(Hkv):
    """Grouped heads are ordinary multi-head attention on K, V with each key/value head repeated
    for the H / Hkv consecutive query heads that read it; dK, dV are the group sums."""
    B, H, N, d = 2, 6, 150, 8
    G = H // Hkv
    q, do = (_rand((B, H, N, d), s) for s in (150, 151))
    k, v = (_rand((B, Hkv, N, d), s) for s in (152, 153))
    kw = dict(causal=True, kv_lens=[150, 97])
    O, L = oracle.forward(q, k, v, 0.4, **kw)
    kr, vr = np.repeat(k, G, axis=1), np.repeat(v, G, axis=1)
    O2, L2 = oracle.forward(q, kr, vr, 0.4, **kw)
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.4, **kw)
    dQ2, dK2, dV2 = oracle.backward(q, kr, vr, do, 0.4, **kw)
    assert np.array_equal(dQ, dQ2)
    assert np.max(np.abs(dK - dK2.reshape(B, Hkv, G, N, d).sum(axis=2))) < 1e-12
    assert np.max(np.abs(dV - dV2.reshape(B, Hkv, G, N, d).sum(axis=2))) < 1e-12


def test_gqa_identical_query_heads():
    """When the G query heads of a group carry the same Q and dO, every head's O equals the
    one-head result and dK, dV are G times the one-head gradients."""
    H, Hkv, N, d = 4, 1, 90, 4
    q1, do1 = (_rand((1, 1, N, d), s) for s in (160, 161))
    k, v = (_rand((1, 1, N, d), s) for s in (162, 163))
    q, do = np.repeat(q1, H, axis=1), np.repeat(do1, H, axis=1)
    O1, _ = oracle.forward(q1, k, v, 0.5)
    O, _ = oracle.forward(q, k, v, 0.5)
    assert np.array_equal(O, np.repeat(O1, H, axis=1))
    _, dK1, dV1 = oracle.backward(q1, k, v, do1, 0.5)
    _, dK, dV = oracle.backward(q, k, v, do, 0.5)
    assert np.max(np.abs(dK - H * dK1)) < 1e-12 and np.max(np.abs(dV - H * dV1)) < 1e-12


def test_gqa_head_mapping_rejects_non_divisors():
    assert [oa.kv_head(h, 8, 2) for h in range(8)] == [0, 0, 0, 0, 1, 1, 1, 1]
    with pytest.raises(ValueError):
        oa.kv_head(0, 6, 4)


@pytest.mark.parametrize("causal", [False, True])
def test_packed_sequences_equal_separate_calls(causal):
    """Sequences packed along the token axis with offsets (the document mask) give, row for row,
    what attention on each sequence alone gives; dK, dV likewise (a key is seen only by its own
    sequence's queries).  Includes an empty sequence and lengths off the 128 grid."""
    lens = [5, 0, 130, 1, 64]
    seg = np.concatenate([[0], np.cumsum(lens)])
    T, H, d = int(seg[-1]), 2, 4
    q, k, v, do = (_rand((1, H, T, d), s) for s in (170, 171, 172, 173))
    O, L = oracle.forward(q, k, v, 0.45, causal=causal, segments=seg)
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.45, causal=causal, segments=seg)
    for a, b in zip(seg[:-1], seg[1:]):
        if a == b:
            continue
        sl = slice(int(a), int(b))
        O1, L1 = oracle.forward(q[:, :, sl], k[:, :, sl], v[:, :, sl], 0.45, causal=causal)
        g1 = oracle.backward(q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], 0.45, causal=causal)
        assert np.max(np.abs(O[:, :, sl] - O1)) < 1e-13 and np.max(np.abs(L[:, :, sl] - L1)) < 1e-13
        for full, part in zip((dQ, dK, dV), g1):
            assert np.max(np.abs(full[:, :, sl] - part)) < 1e-12


def test_packed_sequence_starts_see_only_themselves():
    """Causal and packed: the first token of each sequence attends to itself alone, so its
    output is its own value row and its LSE is its own scaled score."""
    seg = np.array([0, 3, 4, 9])
    q, k, v = (_rand((1, 1, 9, 3), s) for s in (180, 181, 182))
    O, L = oracle.forward(q, k, v, 0.9, causal=True, segments=seg)
    for a in seg[:-1]:
        assert np.max(np.abs(O[0, 0, a] - v[0, 0, a])) < 1e-14
        assert abs(L[0, 0, a] - 0.9 * float(q[0, 0, a] @ k[0, 0, a])) < 1e-13


def test_packed_sequences_finite_differences():
    seg = np.array([0, 4, 9])
    q, k, v, do = (_rand((1, 1, 9, 2), s, 1.1) for s in (190, 191, 192, 193))
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.6, causal=True, segments=seg)
    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        for f in range(x.size):
            idx = tuple(int(i) for i in np.unravel_index(f, x.shape))
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, do=do, scale=0.6, causal=True, segments=seg)
            lm = _loss(**{**args, name: xm}, do=do, scale=0.6, causal=True, segments=seg)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


# --- dropout (counter-based mask, replayed in the backward) ---------------------------------

from oracle import dropout as odrop


def test_philox_known_answers():
    """The generator reproduces its authors' published known-answer vectors."""
    path = os.path.join(os.path.dirname(__file__), "golden", "philox4x32_10_kat.json")
    for vec in json.load(open(path))["vectors"]:
        ctr = np.array([int(x, 16) for x in vec["counter"]], dtype=np.uint64)
        key = np.array([int(x, 16) for x in vec["key"]], dtype=np.uint64)
        out = odrop.philox4x32_10(ctr, key)
        assert [int(x) for x in out] == [int(x, 16) for x in vec["out"]]


def test_dropout_uniform_layout():
    """u(i, j) is byte (j mod 4) of word (i mod 4) of the call at counter
    (j // 4, i // 4, b*H + h, offset), key (seed low, seed high)."""
    seed, off, bh = 0x0123456789ABCDEF, 7, 3
    u = odrop.uniforms(np.arange(12), np.arange(20), bh, seed, off)
    for i, j in ((0, 0), (5, 6), (11, 19), (3, 16), (8, 3)):
        w = odrop.philox4x32_10(np.array([j // 4, i // 4, bh, off], dtype=np.uint64),
                                np.array([seed & 0xFFFFFFFF, seed >> 32], dtype=np.uint64))
        assert u[i, j] == (int(w[i % 4]) >> (8 * (j % 4))) & 0xFF


@pytest.mark.parametrize("p", [0.1, 0.5, 0.9])
def test_dropout_keep_fraction_and_flat_bytes(p):
    k8 = odrop.keep_threshold(p)
    assert k8 == round((1 - p) * 256)
    u = odrop.uniforms(np.arange(512), np.arange(512), 5, 1234 + k8, 0).astype(np.int64)
    n = u.size
    kept = (u < k8).mean()
    assert abs(kept - k8 / 256) <= 4 * np.sqrt(k8 / 256 * (1 - k8 / 256) / n)
    hist = np.bincount(u.ravel(), minlength=256)
    chi2 = ((hist - n / 256) ** 2 / (n / 256)).sum()
    assert chi2 < 255 + 6 * np.sqrt(2 * 255)          # about six sigma above its mean


def test_dropout_rate_zero_is_plain_attention():
    q, k, v, do = (_rand((1, 2, 70, 8), s) for s in (200, 201, 202, 203))
    O, L = oracle.forward(q, k, v, 0.3, causal=True)
    O2, L2 = oracle.forward(q, k, v, 0.3, causal=True, dropout=(99, 3, 256))
    assert np.array_equal(O, O2) and np.array_equal(L, L2)
    g = oracle.backward(q, k, v, do, 0.3, causal=True)
    g2 = oracle.backward(q, k, v, do, 0.3, causal=True, dropout=(99, 3, 256))
    assert all(np.array_equal(a, b) for a, b in zip(g, g2))


def test_dropout_everything_dropped():
    q, k, v, do = (_rand((1, 1, 40, 4), s) for s in (210, 211, 212, 213))
    O, L = oracle.forward(q, k, v, 0.5, dropout=(5, 0, 0))
    L0 = oracle.forward(q, k, v, 0.5)[1]
    assert np.count_nonzero(O) == 0 and np.array_equal(L, L0)     # LSE is the undropped one
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.5, dropout=(5, 0, 0))
    assert np.count_nonzero(dQ) == np.count_nonzero(dK) == np.count_nonzero(dV) == 0


def test_dropout_is_unbiased():
    """Averaged over many seeds, the dropped-out output approaches the plain output (inverted
    dropout keeps the expectation)."""
    q, k, v = (_rand((1, 1, 12, 3), s) for s in (220, 221, 222))
    O = oracle.forward(q, k, v, 0.7)[0]
    k8 = odrop.keep_threshold(0.3)
    acc = np.zeros_like(O)
    n = 400
    for seed in range(n):
        acc += oracle.forward(q, k, v, 0.7, dropout=(seed, 0, k8))[0]
    err = np.abs(acc / n - O).max()
    spread = np.abs(O).max() * np.sqrt((256 - k8) / k8 / n)
    assert err < 4 * spread


def test_dropout_backward_finite_differences():
    """With the mask fixed by (seed, offset), the function is smooth in q, k, v: the gradients
    match central differences."""
    drop = (77, 2, odrop.keep_threshold(0.25))
    q, k, v, do = (_rand((1, 2, 9, 3), s, 1.1) for s in (230, 231, 232, 233))
    dQ, dK, dV = oracle.backward(q, k, v, do, 0.6, causal=True, dropout=drop)
    h = 1e-6
    for name, x, g in (("q", q, dQ), ("k", k, dK), ("v", v, dV)):
        for f in range(x.size):
            idx = tuple(int(i) for i in np.unravel_index(f, x.shape))
            xp, xm = x.copy(), x.copy()
            xp[idx] += h
            xm[idx] -= h
            args = {"q": q, "k": k, "v": v}
            lp = _loss(**{**args, name: xp}, do=do, scale=0.6, causal=True, dropout=drop)
            lm = _loss(**{**args, name: xm}, do=do, scale=0.6, causal=True, dropout=drop)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - g[idx]) <= 1e-6 * max(1.0, abs(g[idx])), (name, idx, fd, g[idx])


def test_dropout_delta_both_ways():
    """With dropout, sum_j P_ij dP_ij (dP with the mask) still equals rowsum(dO * O)."""
    q, k, v, do = (_rand((1, 2, 150, 8), s) for s in (240, 241, 242, 243))
    drop = (3, 9, odrop.keep_threshold(0.4))
    O, _ = oracle.forward(q, k, v, 0.35, dropout=drop)
    _, _, _, D = oracle.backward(q, k, v, do, 0.35, dropout=drop, return_delta=True)
    assert np.max(np.abs(D - (do * O).sum(-1))) < 1e-12


def test_backward_delta_both_ways_and_sums():
    """D_i = sum_j P_ij dP_ij equals rowsum(dO * O); sum_j dK_j = 0; sum_j dV_j = sum_i dO_i."""
    B, H, N, d = 1, 2, 200, 8
    q, k, v, do = (_rand((B, H, N, d), s) for s in (45, 46, 47, 48))
    for causal in (False, True):
        O, _ = oracle.forward(q, k, v, 0.35, causal=causal)
        dQ, dK, dV, D = oracle.backward(q, k, v, do, 0.35, causal=causal, return_delta=True)
        assert np.max(np.abs(D - (do * O).sum(-1))) < 1e-12
        assert np.max(np.abs(dK.sum(axis=2))) < 1e-11
        assert np.max(np.abs(dV.sum(axis=2) - do.sum(axis=2))) < 1e-11


def test_backward_zero_queries_closed_form():
    """Q = 0: P_ij = 1/n_i on allowed keys, so dK = 0, dV_j = sum_i dO_i / n_i over rows that
    allow j, and dQ_i = (scale / n_i) sum_j (dO_i . (v_j - mean_i v)) k_j."""
    N, d, scale = 90, 3, 0.6
    k, v, do = _rand((N, d), 49), _rand((N, d), 50), _rand((N, d), 51)
    dQ, dK, dV = oracle.backward(_one(np.zeros((N, d))), _one(k), _one(v), _one(do), scale, causal=True)
    assert np.max(np.abs(dK)) < 1e-13
    for i in range(N):
        n = i + 1
        vbar = v[:n].mean(axis=0)
        expect = (scale / n) * sum(float(do[i] @ (v[j] - vbar)) * k[j] for j in range(n))
        assert np.max(np.abs(dQ[0, 0, i] - expect)) < 1e-12
    for j in range(N):
        expect = sum(do[i] / (i + 1) for i in range(j, N))
        assert np.max(np.abs(dV[0, 0, j] - expect)) < 1e-12


def test_backward_row_samples_add_up():
    """Splitting the query rows into samples: dQ rows match and dK, dV contributions add up."""
    q, k, v, do = (_rand((1, 1, 150, 4), s) for s in (52, 53, 54, 55))
    full = oracle.backward(q, k, v, do, 0.4, causal=True)
    a = oracle.backward(q, k, v, do, 0.4, causal=True, rows=range(0, 61))
    b = oracle.backward(q, k, v, do, 0.4, causal=True, rows=range(61, 150))
    assert np.max(np.abs(a[0][:, :, :61] - full[0][:, :, :61])) < 1e-13
    assert np.max(np.abs(b[0][:, :, 61:] - full[0][:, :, 61:])) < 1e-13
    for i in (1, 2):
        assert np.max(np.abs(a[i] + b[i] - full[i])) < 1e-12


def test_backward_with_given_output():
    """Given the exact forward output, D = rowsum(dO * O) reproduces the exact gradient; given a
    perturbed output, only the D term changes: dV is unchanged and dQ moves by the closed form
    -scale * (dD_i) * sum_j P_ij k_j."""
    B, H, N, d, scale = 1, 2, 90, 5, 0.45
    q, k, v, do = (_rand((B, H, N, d), s) for s in (56, 57, 58, 59))
    O, _ = oracle.forward(q, k, v, scale, causal=True)
    ref = oracle.backward(q, k, v, do, scale, causal=True)
    got = oracle.backward(q, k, v, do, scale, causal=True, o=O)
    for a, b in zip(got, ref):
        assert np.max(np.abs(a - b)) < 1e-12
    Op = O + 1e-3 * _rand(O.shape, 60)
    pert = oracle.backward(q, k, v, do, scale, causal=True, o=Op)
    assert np.max(np.abs(pert[2] - ref[2])) < 1e-13
    dD = (do * (Op - O)).sum(-1)
    for h in range(H):
        P = oracle.probabilities(q[0, h], k[0, h], scale, causal=True)
        expect = ref[0][0, h] - scale * dD[0, h][:, None] * (P @ k[0, h])
        assert np.max(np.abs(pert[0][0, h] - expect)) < 1e-12
