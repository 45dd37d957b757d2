"""GPU parity for grouped-query attention (H query heads sharing Hkv key/value heads, query head
h reading key/value head h // (H / Hkv)): forward and backward through fa_forward_gqa /
fa_backward_gqa against the fp64 oracle, on ragged sizes over several tiles, with every mask,
in bf16 and fp16; and at a long causal shape with sampled rows and the gradient invariants."""
import math

import numpy as np
import pytest
import torch

import oracle
from gpu_helpers import check_backward_given_o, compare, compare_fwd, f64, run_gpu
from ideal_kernel import ideal_backward
from tolerances import assert_bf16_close
from workloads import Workload, make_inputs, random_tile_mask

pytestmark = pytest.mark.gpu


def _case(N, d, H, Hkv, dtype="bf16", causal=False, B=2, pad=None, seed=0):
    w = Workload(f"gqa_{N}_{d}", B, H, N, d, dtype, causal=causal, pad_lengths=pad)
    return make_inputs(w, seed=seed, kv_heads=Hkv)


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("Hkv", [1, 2, 4])
@pytest.mark.parametrize("causal", [False, True])
def test_gqa_bf16(d, Hkv, causal):
    x = _case(300, d, 8, Hkv, causal=causal, seed=10 * Hkv + d)
    assert x["k"].shape[1] == Hkv
    out = run_gpu(x)
    assert out["dk"].shape == x["k"].shape and out["dv"].shape == x["v"].shape
    compare(x, out)


@pytest.mark.parametrize("d", [64, 128])
def test_gqa_fp16_key_padding(d):
    x = _case(700, d, 6, 2, dtype="fp16", causal=True, B=3, seed=d)
    x["kv_lens"] = torch.tensor([700, 333, 0], dtype=torch.int32)
    compare_fwd(x, run_gpu(x, backward=False))
    check_backward_given_o(x)


def test_gqa_tile_mask():
    x = _case(1000, 128, 4, 2, causal=True, seed=3)
    x["block_mask"] = random_tile_mask(8, 0.5, seed=7)
    compare(x, run_gpu(x))


def test_gqa_forward_equals_repeated_heads():
    """The forward with grouped heads does, per query head, exactly the arithmetic of the
    multi-head forward on key/value heads repeated for their group: bit-identical O and LSE."""
    import exact_io_aware_23_gb300 as fa
    x = _case(520, 128, 8, 2, causal=True, seed=5)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    o1, l1 = fa.forward(q, k, v, causal=True)
    o2, l2 = fa.forward(q, k.repeat_interleave(4, dim=1), v.repeat_interleave(4, dim=1), causal=True)
    assert fa.check_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_gqa_long_causal_n8k_h32_kv8_d128():
    """A long grouped shape (32 query heads on 8 key/value heads, N = 8192, causal).  O, LSE and
    dQ are checked on sampled rows (each row's values depend on that row alone); dK, dV through
    the invariants that hold per key/value head at any size: sum_j dK_j = 0 and
    sum_j dV_j = the group's sum_i dO_i."""
    x = _case(8192, 128, 32, 8, causal=True, B=1, seed=11)
    out = run_gpu(x)
    rows = np.sort(np.random.default_rng(2).choice(8192, 192, replace=False))
    compare(x, out, rows=rows, backward=False)
    heads = [0, 13, 31]
    qq, kk, vv, dd = (f64(x[n]) for n in ("q", "k", "v", "do"))
    dQ, _, _ = oracle.backward(qq, kk, vv, dd, x["scale"], causal=True, heads=heads, rows=rows)
    idq = ideal_backward(x, heads=heads, rows=rows)[0]
    assert_bf16_close("dQ", f64(out["dq"])[:, heads][:, :, rows], dQ[:, :, rows], ideal=idq[:, :, rows])
    dk, dv, do = f64(out["dk"]), f64(out["dv"]), f64(x["do"])
    scale_k = np.sqrt(np.mean(dk ** 2)) * math.sqrt(dk.shape[2])
    assert np.max(np.abs(dk.sum(axis=2))) <= 5e-2 * scale_k
    ref = do.reshape(1, 8, 4, 8192, 128).sum(axis=(2, 3))
    assert np.max(np.abs(dv.sum(axis=2) - ref)) <= 2e-2 * np.max(np.abs(ref)) + 1e-3 * math.sqrt(4 * 8192)
