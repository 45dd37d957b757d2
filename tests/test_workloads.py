"""Input recipe checks: seeded determinism, dtype rounding, valid-length range, tile pattern."""
import torch

from workloads import WORKLOADS, local_global_tile_mask, make_inputs


def test_tile_pattern_count_n64k():
    """512 x 512 tiles, kept iff |I-J| <= 4 or I < 2 or J < 2.
    Band: 512*9 - 2*(4+3+2+1) = 4588; global rows or columns: 2*512 + 2*512 - 4 = 2044;
    band tiles inside the global rows/columns: 5+6+5+6-4 = 18; total 4588 + 2044 - 18 = 6614."""
    bm = local_global_tile_mask(512)
    assert bm.dtype == torch.uint8 and tuple(bm.shape) == (512, 512)
    assert int(bm.sum()) == 6614
    assert bm[0].all() and bm[:, 1].all() and bm[300, 296] == 1 and bm[300, 295] == 0


def test_seeded_and_rounded():
    w = WORKLOADS["bert_large_pad_n512"]
    a = make_inputs(w, seed=0, heads=2)
    b = make_inputs(w, seed=0, heads=2)
    for key in ("q", "k", "v", "do", "kv_lens"):
        assert torch.equal(a[key], b[key])
    assert a["q"].dtype == torch.bfloat16
    lens = a["kv_lens"]
    assert lens.dtype == torch.int32 and int(lens.min()) >= 256 and int(lens.max()) <= 512
    c = make_inputs(w, seed=1, heads=2)
    assert not torch.equal(a["q"], c["q"])


def test_value_scale_and_fp32():
    g = make_inputs(WORKLOADS["gpt2_small_causal_n1024"], heads=1, B=1)
    assert 1.3 < float(g["q"].float().std()) < 1.7 and g["causal"]
    f = make_inputs(WORKLOADS["fp32_n128_d64"])
    assert f["q"].dtype == torch.float32 and tuple(f["q"].shape) == (1, 1, 128, 64)


def test_forward_flop_convention():
    """The metric's FLOP count (4*B*H*N^2*d for the forward; half when causal; the kept share of
    tiles when block-sparse), checked against the figures the workload table states."""
    import bench
    c4 = WORKLOADS["long_n16k_d128"]
    assert abs(bench.forward_flops(c4, 1, 16, 16384) - 2199.02e9) < 0.01e9
    c4c = WORKLOADS["long_n16k_d128_causal"]
    assert bench.forward_flops(c4c, 1, 16, 16384) == bench.forward_flops(c4, 1, 16, 16384) / 2
    c3 = WORKLOADS["gpt2_small_causal_n1024"]
    assert abs(bench.forward_flops(c3, 8, 12, 1024) - 12.885e9) < 0.001e9
    c5 = WORKLOADS["block_sparse_n64k_d64"]
    bm = local_global_tile_mask(512)
    got = bench.forward_flops(c5, 1, 8, 65536, block_mask=bm)
    assert abs(got - 4.0 * 8 * 65536 ** 2 * 64 * 6614 / 512 ** 2) < 1.0
    assert abs(got - 221.9e9) < 0.1e9


def test_clock_summary_reads_reasons():
    """The bench's clock record: median SM clock under load, the maximum, and which throttle
    reasons were active in any sample (the fields nvidia-smi prints, in the order queried)."""
    import bench
    cs = bench.ClockSampler(0)
    idle = ["1200", "2070", "90.0", "0x1", "Not Active", "Not Active", "Not Active", "Not Active"]
    cs.rows = [(0.5, idle),
               (1.1, ["2070", "2070", "300.5", "0x0", "Not Active", "Not Active", "Not Active", "Not Active"]),
               (1.2, ["2055", "2070", "950.1", "0x4", "Not Active", "Not Active", "Not Active", "Active"]),
               (1.3, ["2040", "2070", "1380.0", "0x4", "Not Active", "Not Active", "Not Active", "Active"]),
               (2.0, idle)]
    cs.t_start, cs.t_end = 1.0, 1.35           # only the samples inside the timed region count
    sm = cs.summary()
    assert sm["sm_mhz"] == 2055.0 and sm["sm_max_mhz"] == 2070.0
    assert sm["reasons"] == ["sw_power_cap"] and sm["power_w_max"] == 1380.0 and sm["samples"] == 3
    assert "note" not in sm
    cs.t_start, cs.t_end = 3.0, 3.1            # none inside: all samples, said so
    sm = cs.summary()
    assert sm["samples"] == 5 and "note" in sm
    cs.rows = []
    assert cs.summary()["reasons"] == ["nvidia-smi unavailable"]
