"""Plant plausible mistakes in a copy of the oracle (on the CPU) and check that the pins in
test_oracle.py catch every one: a dropped scale, a sign, a transposed operand, an off-by-one in
each mask, the wrong logarithm base, a wrong reduction axis, a key group dropped in the
blockwise algorithm, a wrong factor in the pages' merge law a wrong query-to-key/value
head mapping and a sequence boundary off by one."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

MUTATIONS = [
    ("dQ[b, hi, r] = scale * (ds @ k[b, g, cols])", "dQ[b, hi, r] = (ds @ k[b, g, cols])"),
    ("ds = p * (dp - D[:, None])", "ds = p * (dp + D[:, None])"),
    ("dK[b, kvi, cols] += scale * (ds.T @ q[b, h, r])", "dK[b, kvi, cols] += scale * (ds @ q[b, h, r])"),
    ("dV[b, kvi, cols] += pd.T @ do[b, h, r]", "dV[b, kvi, cols] += pd.T @ do[b, h, r] * 1.0001"),
    ("ok &= cols[None, :] <= rows[:, None]", "ok &= cols[None, :] < rows[:, None]"),
    ("ok &= (cols < kv_len)[None, :]", "ok &= (cols <= kv_len)[None, :]"),
    ("ok &= bm[(rows // TILE)[:, None], (cols // TILE)[None, :]]",
     "ok &= bm[(cols // TILE)[None, :], (rows // TILE)[:, None]]"),
    ("s = scale * (q_rows @ k_cols.T)", "s = (q_rows @ k_cols.T)"),
    ("lse = m0 + np.log(np.exp(s - m0[:, None]).sum(axis=1))",
     "lse = m0 + np.log2(np.exp(s - m0[:, None]).sum(axis=1))"),
    ("O[b, hi, c0:c0 + r.size] = p @ v[b, g, cols]", "O[b, hi, c0:c0 + r.size] = p @ v[b, g, cols[::-1]]"),
    ("groups = [np.arange(g0, min(g0 + block_size, k.shape[0]))",
     "groups = [np.arange(g0, min(g0 + block_size - 1, k.shape[0]))"),
    ("D = (do[b, h, r] * np.asarray(o, dtype=np.float64)[b, h, r]).sum(axis=1)",
     "D = (q[b, h, r] * np.asarray(o, dtype=np.float64)[b, h, r]).sum(axis=1)"),
    ("return m, fa * la + fb * lb, fa * np.asarray(ua) + fb * np.asarray(ub)",
     "return m, fa * la + fb * lb, fa * np.asarray(ua) + fa * np.asarray(ub)"),
    ("return h // (H // Hkv)", "return h % Hkv"),
    ("kvi = g if grouped else hi", "kvi = hi % Hkv if grouped else hi"),
    ('return np.searchsorted(np.asarray(segments, dtype=np.int64), x, side="right") - 1',
     'return np.searchsorted(np.asarray(segments, dtype=np.int64), x, side="left") - 1'),
    ("return ((w >> (8 * (J & 3)).astype(np.uint32)) & 0xFF).astype(np.uint8)",
     "return ((w >> (8 * (I & 3)).astype(np.uint32)) & 0xFF).astype(np.uint8)"),
    ("return 256.0 / k8 if k8 > 0 else 0.0", "return 255.0 / k8 if k8 > 0 else 0.0"),
    ("                    dp = dp * mk\n", "                    dp = dp\n"),
    ("        c0, c1, c2, c3 = hi1 ^ c1 ^ k0, lo1, hi0 ^ c3 ^ k1, lo0",
     "        c0, c1, c2, c3 = hi1 ^ c1 ^ k1, lo1, hi0 ^ c3 ^ k0, lo0"),
]


@pytest.fixture(scope="module")
def sandbox(tmp_path_factory):
    d = tmp_path_factory.mktemp("mut")
    for name in ("oracle", "workloads"):
        shutil.copytree(os.path.join(ROOT, name), d / name,
                        ignore=shutil.ignore_patterns("__pycache__"))
    (d / "tests").mkdir()
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), d / "tests" / "golden")
    for f in ("conftest.py", "test_oracle.py"):
        shutil.copy(os.path.join(ROOT, "tests", f), d / "tests" / f)
    return d


def test_clean_copy_passes(sandbox):
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "tests/test_oracle.py"],
                       cwd=sandbox, capture_output=True, text=True)
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("old,new", MUTATIONS, ids=[m[1][:40] for m in MUTATIONS])
def test_planted_mistake_is_caught(sandbox, old, new):
    old, new = old.replace("\\n", "\n"), new.replace("\\n", "\n")
    name = next(f for f in ("attention.py", "dropout.py")
                if old in open(os.path.join(ROOT, "oracle", f)).read())
    path = sandbox / "oracle" / name
    src = open(os.path.join(ROOT, "oracle", name)).read()
    path.write_text(src.replace(old, new))
    try:
        r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "tests/test_oracle.py"],
                           cwd=sandbox, capture_output=True, text=True)
        assert r.returncode != 0, f"mutation not caught: {new}"
    finally:
        path.write_text(src)
