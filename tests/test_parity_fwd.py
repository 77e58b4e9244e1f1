"""GPU forward parity: the sm_103a kernel (through the C ABI) against the fp64
oracle, element by element, on seeded inputs."""
import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300.workload import WORKLOADS, make_inputs, workload_inputs
from oracle import evo_oracle as O
from tests.parity_util import FWD_TOL, fwd_rel_err, lse_err, np64, run_fwd, to_dev

pytestmark = pytest.mark.gpu

# (B, N, L, H, D, dtype, mask, bias2_sigma, has_bias1): several tiles, ragged
# tails, every padded head dimension, both bias2 paths (L % 8 == 0 uses TMA,
# otherwise plain loads), absent biases, B = 2 with a per-batch pair bias.
SMALL = [
    (1, 8, 32, 2, 16, "fp16", ("random", 0.10), 1.0, True),    # the tiny workload's shape
    (2, 3, 300, 2, 32, "bf16", ("random", 0.05), 1.0, True),   # 3 key tiles, tail of 44
    (1, 4, 200, 3, 8, "fp16", ("tail", 0.15), 0.5, True),
    (1, 3, 131, 2, 24, "bf16", ("random", 0.05), 1.0, True),   # odd L: bias2 via plain loads
    (2, 2, 257, 1, 64, "fp16", ("random", 0.05), 1.0, True),   # D = 64, tail of 1
    (1, 2, 1, 1, 8, "bf16", None, 1.0, True),                   # L = 1
    (1, 2, 17, 2, 16, "fp16", ("random", 0.10), None, True),    # no pair bias
    (1, 3, 96, 2, 40, "bf16", None, 1.0, False),                # no key mask, D = 40
    (1, 2, 128, 2, 48, "fp16", ("tail", 0.5), None, False),     # no biases at all
    (1, 2, 384, 1, 56, "bf16", ("tail", 0.03), 1.0, True),
    (1, 1, 33, 1, 32, "fp16", ("random", 0.3), 1.0, True),
]


def _compare(inp, dtype):
    d = to_dev(inp)
    out, lse = run_fwd(d)
    a = {k: np64(v) for k, v in inp.items()}
    o_ref, lse_ref = O.forward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"])
    err = fwd_rel_err(np64(out), o_ref)
    assert err <= FWD_TOL[dtype], err
    assert lse_err(lse.cpu().numpy(), lse_ref) <= 1e-3
    return err


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c[:5])) + "-" + c[5])
def test_small(case):
    B, N, L, H, D, dt, mask, sig, hb1 = case
    inp = make_inputs(B, N, L, H, D, dtype=dt, mask=mask, bias2_sigma=sig, seed=3, has_bias1=hb1)
    if not hb1:
        inp["bias1"] = None
    _compare(inp, inp["q"].dtype)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("rows", ["all", "even"])
def test_rising_scores_across_key_tiles(dtype, rows):
    """A pair bias that rises ~10 log2 units per 128 keys: later key tiles hold much
    larger scores than the first, so the running reference max must move (and the
    partial output be rescaled) inside an item.  With the ramp on even query rows
    only, neighbouring rows of one warp take different paths."""
    inp = make_inputs(1, 3, 384, 2, 32, dtype=dtype, mask=("random", 0.05), bias2_sigma=0.5, seed=17)
    ramp = torch.arange(384, dtype=torch.float32) * (7.0 / 128.0)
    sel = torch.ones(384) if rows == "all" else (torch.arange(384) % 2 == 0).float()
    b2 = inp["bias2"].float() + sel.view(1, 1, 1, 384, 1) * ramp.view(1, 1, 1, 1, 384)
    inp["bias2"] = b2.to(inp["bias2"].dtype)
    _compare(inp, inp["q"].dtype)


def test_first_key_tile_masked_then_very_negative_fp16():
    """Every key of the first tile masked (-inf in fp16) and the remaining scores near
    -100: the output is the softmax over the later keys alone."""
    inp = make_inputs(1, 2, 300, 2, 16, dtype="fp16", mask=None, bias2_sigma=0.5, seed=23)
    inp["bias1"][..., :128] = float("-inf")
    inp["bias2"] = (inp["bias2"].float() - 100.0).to(torch.float16)
    _compare(inp, torch.float16)


def test_fully_masked_rows_fp16():
    """Every key of one (b, n) row masked (-1e9 -> -inf in fp16): O = 0, lse = -inf, like the oracle."""
    inp = make_inputs(1, 3, 70, 2, 16, dtype="fp16", mask=("random", 0.1), seed=5)
    inp["bias1"][0, 1] = float("-inf")
    d = to_dev(inp)
    out, lse = run_fwd(d)
    assert torch.all(out[0, 1] == 0) and torch.all(torch.isneginf(lse[0, 1]))
    _compare(inp, torch.float16)


def test_fully_masked_rows_bf16_no_nan():
    """bf16 keeps -1e9 finite; a fully masked row must still give finite output."""
    inp = make_inputs(1, 2, 64, 2, 16, dtype="bf16", mask=("random", 0.1), seed=6)
    inp["bias1"][0, 0] = -1e9
    out, lse = run_fwd(to_dev(inp))
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("pair", [False, True], ids=["no_pair_bias", "pair_bias"])
@pytest.mark.parametrize("D", [16, 32, 64])
def test_real_valued_key_bias(dtype, pair, D):
    """bias1 as a general additive bias (page §3.5: any bias broadcast over heads and queries),
    not only 0 or masked: real values of a few tens next to masked keys.  Where the score MMA
    adds the key bias it carries the bias in three bf16 parts, which together hold the full
    fp32 value; one part alone would be off by ~2^-9 of the bias, several percent of P here."""
    inp = make_inputs(1, 3, 200, 2, D, dtype=dtype, mask=("random", 0.1), bias2_sigma=1.0 if pair else None,
                      seed=21)
    b1 = inp["bias1"].float()
    gen = torch.Generator().manual_seed(5)
    cont = torch.randn(b1.shape, generator=gen) * 12.0
    inp["bias1"] = torch.where(b1 == 0, cont, b1).to(inp["q"].dtype)  # masked keys stay masked
    tdt = torch.float16 if dtype == "fp16" else torch.bfloat16
    _compare(inp, tdt)
    # and the backward, which adds the key bias itself
    from memory_efficient_biased_gb300 import evo_attn as E
    from tests.parity_util import GRAD_TOL, rel_l2
    d = to_dev(inp)
    out, lse = E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"])
    dq, dk, dv, _ = E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"])
    assert E.evo_attn_device_status() == 0
    a = {k: np64(v) for k, v in inp.items()}
    g = O.backward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"], a["do"])
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv)):
        assert rel_l2(np64(t), g[name]) <= GRAD_TOL[tdt], name


@pytest.mark.parametrize("name,dtype", [("tiny", "fp16"), ("msa_row", "fp16"), ("msa_row", "bf16"),
                                        ("many_head", "bf16")])
def test_workload_full(name, dtype):
    """Whole-tensor comparison on workloads the oracle finishes in seconds."""
    _compare(workload_inputs(name, dtype), torch.float16 if dtype == "fp16" else torch.bfloat16)


@pytest.mark.parametrize("name", ["msa_col", "triangle"])
def test_workload_sampled(name):
    """Full-size workloads: sampled (b, n, h) slices, computed one by one by the oracle."""
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    out, lse = run_fwd(to_dev(inp))
    out, lse = out.cpu(), lse.cpu()
    rng = np.random.default_rng(0)
    picks = [(0, 0, 0), (0, w.N - 1, w.H - 1)] + [(0, int(rng.integers(w.N)), int(rng.integers(w.H)))
                                                 for _ in range(6)]
    tol = FWD_TOL[torch.bfloat16]
    for (b, n, h) in picks:
        # the oracle sees only row (b, n): a [1, 1, L, H, D] problem
        one = lambda t: None if t is None else t[b:b + 1, n:n + 1].double().numpy()
        b2 = None if inp["bias2"] is None else inp["bias2"][b:b + 1].double().numpy()
        o_ref, lse_ref = O.forward_slice_sample(one(inp["q"]), one(inp["k"]), one(inp["v"]),
                                                one(inp["bias1"]), b2, 0, 0, h)
        err = fwd_rel_err(out[b, n, :, h].double().numpy(), o_ref)
        assert err <= tol, (b, n, h, err)
        assert lse_err(lse[b, n, h].numpy(), lse_ref) <= 1e-3
