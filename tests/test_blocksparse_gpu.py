"""The balanced block-sparse forward (fa_forward_blocksparse): tile masks whose rows have very
unequal numbers of live key tiles are split into ranges by a device-side plan and merged with the
(m, l, u) merge law.  Against the fp64 oracle (with the ideal-kernel floor), reproducible to the
bit, close to the unbalanced forward, with key padding, causal masks, grouped heads and fp16."""
import numpy as np
import pytest
import torch

from gpu_helpers import compare, compare_fwd, f64, run_gpu
from tolerances import assert_bf16_close
from workloads import Workload, local_global_tile_mask, make_inputs, random_tile_mask

pytestmark = pytest.mark.gpu


def _case(N, d, dtype="bf16", causal=False, B=2, H=2, Hkv=None, seed=0, pad=None, global_rows=2):
    w = Workload(f"bs_{N}_{d}", B, H, N, d, dtype, causal=causal, pad_lengths=pad)
    x = make_inputs(w, seed=seed, kv_heads=Hkv)
    T = (N + 127) // 128
    bm = local_global_tile_mask(T, band=2, n_global=global_rows)
    bm[T - global_rows:, :] = 1          # dense last rows too: under a causal mask they are the long ones
    extra = random_tile_mask(T, 0.05, seed=seed + 1)
    x["block_mask"] = (bm | extra).to(torch.uint8)
    return x


@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_balanced_forward_against_oracle(d, causal):
    # 64 tiles: the global rows see every key tile, so their pair is split into ranges
    x = _case(8192 + 77, d, causal=causal, seed=3 + d)
    compare(x, run_gpu(x))


@pytest.mark.parametrize("d", [64, 128])
def test_balanced_forward_padding_grouped_fp16(d):
    x = _case(6000, d, "fp16", causal=True, B=2, H=4, Hkv=2, seed=9, pad=(1, 6000), global_rows=3)
    x["kv_lens"] = torch.tensor([6000, 2100], dtype=torch.int32)
    compare_fwd(x, run_gpu(x, backward=False))


def test_balanced_forward_is_reproducible_and_close_to_unbalanced():
    import exact_io_aware_23_gb300 as fa
    x = _case(16384, 64, seed=5, global_rows=4)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    bm = x["block_mask"].to(dev)
    o1, l1 = fa.forward(q, k, v, block_mask=bm)
    o2, l2 = fa.forward(q, k, v, block_mask=bm)
    o0, l0 = fa.forward(q, k, v, block_mask=bm, balanced=False)
    assert fa.check_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert_bf16_close("O", f64(o1), f64(o0))
    assert np.max(np.abs(f64(l1) - f64(l0))) <= 1e-4


def test_balanced_forward_many_units_per_cta():
    """At d = 64 the balanced forward is persistent (one CTA per SM claiming units from the plan):
    with about ten units per CTA its unit entries, Q buffers and rings wrap many times.  The
    result is reproducible and matches the unbalanced forward."""
    import exact_io_aware_23_gb300 as fa
    x = _case(8192, 64, B=4, H=8, seed=11, global_rows=3)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    bm = x["block_mask"].to(dev)
    o1, l1 = fa.forward(q, k, v, block_mask=bm)
    o2, l2 = fa.forward(q, k, v, block_mask=bm)
    o0, l0 = fa.forward(q, k, v, block_mask=bm, balanced=False)
    assert fa.check_device_status() == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert_bf16_close("O", f64(o1), f64(o0))
    assert np.max(np.abs(f64(l1) - f64(l0))) <= 1e-4


def test_balanced_forward_workspace_too_small():
    import exact_io_aware_23_gb300 as fa
    x = _case(1024, 64, seed=1)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    ws = torch.empty(256, dtype=torch.uint8, device=dev)
    with pytest.raises(fa.FaError):
        fa.forward(q, k, v, block_mask=x["block_mask"].to(dev), workspace=ws)
