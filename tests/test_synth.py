"""The seeded input generator: determinism, slicing, structure, and numpy == torch."""
import numpy as np
import pytest
import torch

import synth


def test_deterministic_and_sliceable():
    wl = synth.workload(1)
    a = wl.keys(3, 5, 0, 256)
    b = wl.keys(3, 5, 100, 50)
    assert np.array_equal(a[100:150], b)
    assert np.array_equal(a, synth.workload(1).keys(3, 5, 0, 256))
    assert not np.array_equal(a, wl.keys(3, 6, 0, 256))


def test_structure_outliers_and_bursts():
    wl = synth.workload(2)
    K = synth.bits_to_f32(wl.keys(0, 1, 0, 4096), "bf16")
    ch = wl.outlier_channels(1)
    assert len(ch) == 4
    std = K.std(axis=0)
    others = np.setdiff1d(np.arange(128), ch)
    assert np.all(std[ch] > 10) and np.all(std[others] < 1.5)
    mask = wl.burst_mask(0, 0, 200000)
    assert abs(mask.mean() - 0.01) < 0.002
    V = synth.bits_to_f32(wl.values(0, 1, 0, 4096), "bf16")
    m = wl.burst_mask(0, 0, 4096)
    assert V[m].std() > 5 and V[~m].std() < 1.5


def test_varlen_lengths():
    L = synth.workload(4).lengths
    assert len(L) == 32 and min(L) >= 1024 and max(L) <= 131072
    assert L == synth.varlen_lengths(1004, 32)


def test_normal_moments():
    x = synth.normal(7, 1, np.arange(1 << 18, dtype=np.uint64))
    assert abs(x.mean()) < 0.01 and abs(x.std() - 1) < 0.01


@pytest.mark.parametrize("which", ["k", "v"])
@pytest.mark.parametrize("idx", [2, 3])
def test_torch_matches_numpy(which, idx):
    wl = synth.workload(idx)
    t = synth.torch_kv_head_major(wl, 1, 2, 10, 300, which, "cpu")
    n = wl.keys(1, 2, 10, 300) if which == "k" else wl.values(1, 2, 10, 300)
    assert np.array_equal(t.view(torch.int16).numpy().view(np.uint16), n)


def test_bf16_rounding_matches_torch():
    x = np.random.default_rng(0).standard_normal(100000).astype(np.float32) * 100
    ours = synth.to_dtype_bits(x, "bf16")
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
