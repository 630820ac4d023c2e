"""Host-side pieces of the benchmark: the input arena's layout and the roofline arithmetic."""
import importlib.util
import math
import os

import pytest
import torch

from tree_verification_gb300 import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    spec = importlib.util.spec_from_file_location("bench_module", os.path.join(ROOT, "bench.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def test_input_arena_segments_are_contiguous_aligned_and_copies():
    b = _bench()
    g = torch.Generator().manual_seed(0)
    t = {"a": torch.randn(3, 5, generator=g), "b": torch.arange(7, dtype=torch.int32),
         "c": torch.randn(4, 2, generator=g).to(torch.bfloat16), "d": torch.tensor([9], dtype=torch.int64)}
    segs_in = [("x", [t["a"], t["b"]]), (0, [t["c"]]), ("y", [t["d"]])]
    arena, segs, views = b.input_arena(segs_in, "cpu")
    order = [segs[k] for k in ("x", 0, "y")]
    assert order[0][0] == 0
    for (s0, s1), (n0, _) in zip(order, order[1:]):
        assert s1 == n0  # segments follow each other with no gap
    for s0, s1 in order:
        assert s0 % 256 == 0 and s1 % 256 == 0
    assert arena.numel() == order[-1][1]
    for key, ts in segs_in:
        for src, v in zip(ts, views[key]):
            assert v.dtype == src.dtype and v.shape == src.shape and torch.equal(v, src)
            off = v.data_ptr() - arena.data_ptr()
            assert segs[key][0] <= off and off + v.numel() * v.element_size() <= segs[key][1]
            assert off % 256 == 0


def test_attention_roofline_fractions():
    b = _bench()
    wl = synth.WORKLOADS["llama3_8b"]
    L0 = synth.prefix_lengths(wl)
    t = 14.2e-6
    r = b.attention_roofline(wl, L0, t, {"sm_mhz": 2000.0}, 152)
    sum_l = int(L0.sum())
    nbytes = 2 * sum_l * wl.Hkv * 128 * 2 + 2 * wl.B * wl.Kmax * wl.Hkv * 128 * 2 + 2 * wl.B * wl.Kmax * wl.Hq * 128 * 2
    hbm, _ = b.measured_peaks()
    tc, _ = b.measured_tensor_peak()
    assert r["bytes_per_call"] == nbytes
    assert r["flops_per_call"] == 4.0 * wl.Hq * wl.Kmax * 128 * sum_l
    assert r["ex2_per_call"] == wl.Hq * wl.Kmax * sum_l
    assert math.isclose(r["fractions"]["hbm"], nbytes / (hbm * 1e9) / t)
    assert math.isclose(r["fractions"]["tensor"], r["flops_per_call"] / (tc * 1e12) / t)
    assert math.isclose(r["fractions"]["sfu"], r["ex2_per_call"] / (16 * 152 * 2000e6) / t)
    # group 4, Kmax 64: 256 flop per KV byte, under the ridge of the measured peaks: HBM-bound
    assert r["bound"] == "hbm" and math.isclose(r["frac"], r["fractions"]["hbm"])
    assert r["unit"] == "GB/s" and math.isclose(r["achieved"], nbytes / t / 1e9)


def test_attention_roofline_group16_is_tensor_bound():
    b = _bench()
    wl = synth.WORKLOADS["qwen3_235b"]
    r = b.attention_roofline(wl, synth.prefix_lengths(wl), 280e-6, None, 152)
    assert r["bound"] == "tensor" and r["unit"] == "TFLOP/s"
    assert math.isclose(r["frac"], r["fractions"]["tensor"])
    assert r["fractions"]["tensor"] > r["fractions"]["hbm"]
