"""The seeded input recipe (CPU only)."""
import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300.workload import WORKLOADS, make_inputs, masked_count, workload_inputs


def test_shapes_and_counts_tiny():
    t = workload_inputs("tiny")
    assert t["q"].shape == (1, 8, 32, 2, 16) and t["q"].dtype == torch.float16
    assert t["bias1"].shape == (1, 8, 1, 1, 32) and t["bias2"].shape == (1, 1, 2, 32, 32)
    m = t["bias1"].float().numpy()[:, :, 0, 0, :]
    assert np.all(np.isneginf(m) | (m == 0))          # fp16 rounds -1e9 to -inf
    assert np.all((np.isneginf(m)).sum(-1) == 3)      # round(0.10 * 32) per row
    assert np.all((m == 0).sum(-1) >= 1)


def test_random_mask_counts_and_bf16_value():
    t = make_inputs(1, 16, 256, 1, 8, dtype="bf16", mask=("random", 0.05))
    m = t["bias1"].float().numpy()[0, :, 0, 0, :]
    assert np.all((m < -1e8).sum(-1) == 13)           # round(0.05 * 256)
    assert np.all(m[m < -1e8] == np.float32(-998244352.0))
    # rows differ (per-row permutation)
    assert len({tuple(np.nonzero(r)[0]) for r in m}) > 1


@pytest.mark.parametrize("name,first", [("msa_col", 870), ("triangle", 497)])
def test_tail_masks(name, first):
    w = WORKLOADS[name]
    assert w.L - masked_count(w.L, w.mask[1]) == first


def test_tail_mask_small():
    t = make_inputs(1, 3, 40, 1, 8, dtype="bf16", mask=("tail", 0.15))
    m = t["bias1"].float().numpy()[0, :, 0, 0, :]
    assert np.all(m[:, :34] == 0) and np.all(m[:, 34:] < -1e8)


def test_seeded_and_ordered():
    a = make_inputs(1, 2, 17, 2, 8, dtype="fp16", seed=0)
    b = make_inputs(1, 2, 17, 2, 8, dtype="fp16", seed=0)
    c = make_inputs(1, 2, 17, 2, 8, dtype="fp16", seed=1)
    for key in ("q", "k", "v", "do", "bias1", "bias2"):
        assert torch.equal(a[key], b[key])
    assert not torch.equal(a["q"], c["q"])
    # Q is the first draw: the same float32 normals, rounded to fp16
    ref = np.random.default_rng(0).standard_normal((1, 2, 17, 2, 8), dtype=np.float32)
    assert torch.equal(a["q"], torch.from_numpy(ref).to(torch.float16))


def test_bias2_sigma_and_absent():
    t = make_inputs(1, 1, 64, 4, 8, dtype="bf16", bias2_sigma=0.5)
    sd = t["bias2"].float().std().item()
    assert 0.45 < sd < 0.55
    t = make_inputs(1, 1, 64, 4, 8, dtype="bf16", bias2_sigma=None)
    assert t["bias2"] is None


def test_workload_table():
    assert WORKLOADS["msa_row"].shape == (1, 256, 256, 4, 32)
    assert WORKLOADS["many_head"].shape == (1, 512, 256, 8, 8)
    assert WORKLOADS["msa_col"].shape == (1, 384, 1024, 8, 32) and WORKLOADS["msa_col"].bias2_sigma is None
    assert WORKLOADS["triangle"].shape == (1, 512, 512, 4, 32)
