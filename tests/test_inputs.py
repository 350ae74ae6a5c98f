"""The seeded input generator: deterministic, prefix-stable, with the stated structure (no GPU)."""

import numpy as np
import torch

import seeded_inputs as si


def test_deterministic_and_prefix_stable():
    w = si.small_workload("t", 4, 2, 64, "q8_0", "bf16", n_prompt=40, chunk=16, n_decode=3, seed=77)
    q1, k1, v1 = si.layer_qkv(w, 0)
    q2, k2, v2 = si.layer_qkv(w, 0, n_rows=10)
    assert q1.dtype == torch.bfloat16 and q1.shape == (43, 4, 64) and k1.shape == (43, 2, 64)
    assert torch.equal(q1[:10], q2) and torch.equal(k1[:10], k2) and torch.equal(v1[:10], v2)
    q3, _, _ = si.layer_qkv(w, 1)
    assert not torch.equal(q1, q3)


def test_k_outliers_are_a_fixed_channel_subset():
    w = si.small_workload("o", 8, 8, 128, "q8_0", "f32", n_prompt=400, chunk=64, n_decode=0, seed=5,
                          k_outlier_frac=0.01)
    ch = si.outlier_channels(w, 0)
    assert ch.size == 10
    _, k, _ = si.layer_qkv(w, 0)
    std = k.reshape(400, -1).std(0).numpy()
    mask = np.zeros(std.size, bool)
    mask[ch] = True
    assert std[mask].min() > 3.0 and std[~mask].max() < 1.4


def test_chunks_cover_the_prompt():
    w = si.WORKLOADS["q8_0_58k"]
    ch = w.chunks()
    assert ch[0] == (0, 2048) and sum(c for _, c in ch) == 58300 and ch[-1] == (57344, 956)
    assert len(si.WORKLOADS["f16_17k"].chunks()) == 34
    assert si.WORKLOADS["q8_0_sweep_10k"].chunks(0) == [(0, 10041)]
