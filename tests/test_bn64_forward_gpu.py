"""The d = 64 forward with 64-key tiles and two CTAs per SM (every d = 64 forward without a tile
mask, packing or split-KV): parity with the fp64 oracle (with the ideal-kernel floor) at the
edges of its tiling — one row, one key tile exactly, a ragged last tile, many tiles — under
causal masks, key padding down to empty sequences, grouped heads and fp16; and agreement with
the 128-key-tile forward that runs the same inputs under a tile mask."""
import pytest
import torch

from gpu_helpers import check_backward_given_o, compare, compare_fwd, run_gpu
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _case(N, dtype="bf16", causal=False, B=2, H=2, Hkv=None, pad=None, vs=1.0, seed=0):
    w = Workload(f"bn64_{N}", B, H, N, 64, dtype, causal=causal, value_scale=vs, pad_lengths=pad)
    return make_inputs(w, seed=seed, kv_heads=Hkv)


@pytest.mark.parametrize("N", [1, 63, 64, 65, 257, 511, 2048, 4100])
@pytest.mark.parametrize("causal", [False, True])
def test_bn64_forward_lengths(N, causal):
    x = _case(N, causal=causal, seed=N + causal)
    compare_fwd(x, run_gpu(x, backward=False))


def test_bn64_forward_chained_backward_causal():
    x = _case(1000, causal=True, B=2, H=3, seed=4)
    compare(x, run_gpu(x))


def test_bn64_forward_key_padding_with_empty_and_one_key_sequences():
    x = _case(700, B=4, H=2, seed=5)
    x["kv_lens"] = torch.tensor([700, 0, 1, 333], dtype=torch.int32)
    compare_fwd(x, run_gpu(x, backward=False))
    check_backward_given_o(x)


def test_bn64_forward_padding_causal_grouped_fp16():
    x = _case(1500, "fp16", causal=True, B=2, H=8, Hkv=2, seed=6)
    x["kv_lens"] = torch.tensor([1500, 830], dtype=torch.int32)
    compare_fwd(x, run_gpu(x, backward=False))


def test_bn64_forward_extreme_logits():
    x = _case(600, causal=True, B=1, H=2, vs=3.0, seed=7)
    s = (x["q"].float() @ x["k"].float().transpose(-1, -2)).abs().max().item()
    x["scale"] = 60.0 / s
    out = run_gpu(x, backward=False)
    assert torch.isfinite(out["o"]).all()
    compare_fwd(x, out)


def test_bn64_forward_many_ctas_per_sm_wave():
    """About two CTAs per SM at once (B8 H16 N512: 256 CTAs); every CTA's rows are checked."""
    x = _case(512, B=8, H=16, seed=8)
    x["kv_lens"] = torch.tensor([512, 100, 300, 1, 512, 257, 64, 65], dtype=torch.int32)
    compare_fwd(x, run_gpu(x, backward=False))


@pytest.mark.parametrize("causal", [False, True])
def test_bn64_and_bn128_forward_agree(causal):
    """The same inputs through both d = 64 forwards: without a mask (64-key tiles) and with an
    all-ones tile mask on the one-CTA-per-unit path (128-key tiles, balanced=False): equal within
    bf16 rounding of O, and LSE to fp32 summation order."""
    import numpy as np
    import exact_io_aware_23_gb300 as fa
    from gpu_helpers import f64
    from tolerances import assert_bf16_close
    N = 2300
    x = _case(N, causal=causal, B=1, H=4, seed=10 + causal)
    dev = torch.device("cuda:0")
    q, k, v = (x[n].to(dev) for n in ("q", "k", "v"))
    T = (N + 127) // 128
    ones = torch.ones((T, T), dtype=torch.uint8, device=dev)
    o1, l1 = fa.forward(q, k, v, causal=bool(causal))
    o2, l2 = fa.forward(q, k, v, causal=bool(causal), block_mask=ones, balanced=False)
    assert fa.check_device_status() == 0
    assert_bf16_close("O", f64(o1), f64(o2))
    assert np.max(np.abs(f64(l1) - f64(l2))) <= 1e-4
