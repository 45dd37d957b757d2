"""Peak device memory of one forward + backward stays O(N * d) ("FlashAttention：让精确注意力服从
内存层次", "数值与正确性": check peak memory on long sequences; the extra storage grows with N*d,
not N^2): at the long-context workload shape (B1 H16 N16384 d128), causal and not, the inputs,
outputs, LSE and the backward's workspace are all that is ever allocated, and the footprint per
query row is the same at N = 4096, 8192 and 16384."""
import pytest
import torch

from workloads import WORKLOADS, make_inputs

pytestmark = pytest.mark.gpu


def _footprint(x):
    """Bytes allocated by the caller's inputs plus everything allocated during one forward and
    one backward through the binding (outputs, LSE, workspace), from the allocator's peak."""
    import exact_io_aware_23_gb300 as fa
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats()
    base = torch.cuda.memory_allocated()
    o, lse = fa.forward(q, k, v, causal=x["causal"])
    grads = fa.backward(q, k, v, o, lse, do, causal=x["causal"])
    torch.cuda.synchronize()
    assert fa.check_device_status() == 0
    peak = torch.cuda.max_memory_allocated() - base
    inputs = sum(t.numel() * t.element_size() for t in (q, k, v, do))
    del o, lse, grads
    return inputs + peak


@pytest.mark.parametrize("name", ["long_n16k_d128", "long_n16k_d128_causal"])
def test_peak_memory_is_linear_in_n(name):
    w = WORKLOADS[name]
    per_row = []
    for N in (4096, 8192, 16384):
        x = make_inputs(w, N=N)
        total = _footprint(x)
        B, H, d = w.B, w.H, w.d
        # Q, K, V, dO, O, dQ, dK, dV in bf16 (16 bytes per element of a [B, H, N, d] tensor) +
        # LSE and D (8 bytes per row), allocator rounding on top: at most 17 bytes per element
        assert total <= 17 * B * H * N * d, (N, total)
        if N == 16384:
            assert total < 0.05 * 4 * B * H * N * N     # far below one fp32 score matrix
        per_row.append(total / (B * H * N))
    assert max(per_row) / min(per_row) < 1.02, per_row  # linear in N
