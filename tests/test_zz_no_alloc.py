"""fa_backward_noalloc, the backward for callers that cannot allocate device memory (plugin
interfaces with no workspace argument, hosts whose device memory is owned by their own
allocator, paths where a synchronising cudaMalloc is not allowed).  It must give the same
gradients as fa_backward, and gradients within the parity tolerance of the fp64 oracle, on
consecutive calls that reuse its built-in scratch array, on both of fa_backward's paths (bf16
two-pass, fp32 CUDA cores); and it must refuse sizes whose scratch would not fit.  Kept in a
file of its own, collected last."""
import ctypes

import numpy as np
import pytest
import torch

from gpu_helpers import compare_bwd
from tolerances import assert_bf16_close, assert_fp32_close
from workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu

FA_UNSUPPORTED = 2


@pytest.mark.parametrize("d,causal,pad,dtype", [(128, True, False, "bf16"), (64, False, True, "bf16"),
                                                (64, True, True, "fp32")])
def test_noalloc_matches_backward_and_oracle_on_two_calls(d, causal, pad, dtype):
    import exact_io_aware_23_gb300 as fa
    N = 700 if dtype != "fp32" else 300
    w = Workload("noalloc", 3, 4, N, d, dtype, causal=causal, pad_lengths=(200, N) if pad else None)
    x = make_inputs(w, seed=21 + d)
    dev = torch.device("cuda:0")
    q, k, v, do = (x[n].to(dev) for n in ("q", "k", "v", "do"))
    kl = None if x["kv_lens"] is None else x["kv_lens"].to(dev)
    o, lse = fa.forward(q, k, v, causal=causal, kv_lens=kl)
    ref = fa.backward(q, k, v, o, lse, do, causal=causal, kv_lens=kl)
    outs = [torch.empty_like(q) for _ in range(3)]
    for _ in range(2):                       # the second call reuses the scratch left by the first
        for t in outs:
            t.fill_(float("nan"))
        got = fa.backward_noalloc(q, k, v, o, lse, do, causal=causal, kv_lens=kl,
                                  dq=outs[0], dk=outs[1], dv=outs[2])
        assert fa.check_device_status() == 0
        for name, a, b in zip(("dQ", "dK", "dV"), got, ref):
            if dtype == "fp32":
                assert_fp32_close(name, a.double().cpu().numpy(), b.double().cpu().numpy(), 1e-5)
            else:
                assert torch.equal(a, b), name         # the same two-pass kernel: the same bits
        # and against the exact gradient (the chained check of the parity tests)
        compare_bwd(x, dict(dq=got[0], dk=got[1], dv=got[2]))


def test_noalloc_rejects_sizes_beyond_its_scratch():
    import exact_io_aware_23_gb300 as fa
    cap = fa.noalloc_max_workspace()
    assert cap == 32 << 20
    # the long-context workload fits (its scratch is D alone: 1 MiB)
    assert fa.backward_workspace_size(1, 16, 16384, 128) <= cap
    B, H, N, d = 1, 16, 524800, 64               # 8 396 800 query rows: D needs just over 32 MiB
    assert fa.backward_workspace_size(B, H, N, d) > cap
    p = ctypes.c_void_p(0x10000)                 # never dereferenced: the call returns first
    st = fa.lib.fa_backward_noalloc(p, p, p, p, p, p, p, p, p, B, H, N, d, 0.1, 0, None, 0, None, None)
    assert st == FA_UNSUPPORTED
