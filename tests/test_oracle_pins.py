"""Pins of the fp64 oracle to things other than itself (CPU only).

Each pin is chosen so that a plausible slip in the oracle (dropped bias term,
wrong scale, transposed bias, wrong sign or index in a gradient, a missing
delta) fails at least one of them; ``test_oracle_mutants.py`` plants such
slips in copies of the oracle and checks that they are caught.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import evo_oracle as O
from tests.brute_force import brute

HERE = os.path.dirname(os.path.abspath(__file__))
RNG = np.random.default_rng(1234)


def rand_problem(B, N, L, H, D, rng, mask_frac=0.25, bias2=True, bias1=True, neg_inf=False):
    q = rng.standard_normal((B, N, L, H, D))
    k = rng.standard_normal((B, N, L, H, D))
    v = rng.standard_normal((B, N, L, H, D))
    do = rng.standard_normal((B, N, L, H, D))
    b1 = None
    if bias1:
        b1 = np.zeros((B, N, 1, 1, L))
        mval = -np.inf if neg_inf else -1e9
        for b in range(B):
            for n in range(N):
                cnt = min(int(round(mask_frac * L)), L - 1)
                b1[b, n, 0, 0, rng.permutation(L)[:cnt]] = mval
    b2 = rng.standard_normal((B, 1, H, L, L)) if bias2 else None
    return q, k, v, do, b1, b2


# ---------------------------------------------------------------- hand example
def test_hand_derived_example():
    fx = json.load(open(os.path.join(HERE, "golden", "two_query_hand_example.json")))
    sh = fx["shape"]
    r = lambda key: np.array(fx[key], dtype=np.float64).reshape(sh)
    q, k, v, do = r("q"), r("k"), r("v"), r("do")
    b1 = np.array(fx["bias1"], dtype=np.float64).reshape(1, 1, 1, 1, 2)
    b2 = np.array(fx["bias2"], dtype=np.float64).reshape(1, 1, 1, 2, 2)
    o, lse = O.forward(q, k, v, b1, b2)
    np.testing.assert_allclose(o, r("o"), atol=1e-14)
    np.testing.assert_allclose(lse.reshape(-1), fx["lse"], atol=1e-14)
    g = O.backward(q, k, v, b1, b2, do)
    for key in ("dq", "dk", "dv"):
        np.testing.assert_allclose(g[key], r(key), atol=1e-14, err_msg=key)
    np.testing.assert_allclose(g["delta"].reshape(-1), fx["delta"], atol=1e-14)
    np.testing.assert_allclose(g["dbias2"].reshape(2, 2), fx["dbias2"], atol=1e-14)
    np.testing.assert_allclose(g["dbias1"].reshape(-1), fx["dbias1"], atol=1e-14)


# ----------------------------------------------------------------- brute force
@pytest.mark.parametrize("shape", [(1, 1, 1, 1, 1), (1, 2, 3, 2, 2), (2, 2, 4, 1, 3),
                                   (1, 1, 6, 2, 4), (2, 1, 5, 3, 2)])
def test_brute_force(shape):
    rng = np.random.default_rng(sum(shape))
    q, k, v, do, b1, b2 = rand_problem(*shape, rng)
    ref = brute(q, k, v, b1, b2, do)
    o, lse = O.forward(q, k, v, b1, b2)
    g = O.backward(q, k, v, b1, b2, do)
    np.testing.assert_allclose(o, np.array(ref["o"]), atol=1e-12)
    np.testing.assert_allclose(lse, np.array(ref["lse"]), atol=1e-12)
    for key in ("dq", "dk", "dv", "dbias1", "dbias2"):
        np.testing.assert_allclose(g[key], np.array(ref[key]), atol=1e-12, err_msg=key)


def test_brute_force_tiny_workload():
    """The tiny workload's own shape (1, 8, 32, 2, 16) and recipe."""
    from memory_efficient_biased_gb300.workload import workload_inputs
    t = workload_inputs("tiny")
    a = {k: (None if x is None else x.double().numpy()) for k, x in t.items()}
    # brute force on a 2-row subset keeps this a few seconds
    sub = {k: (None if x is None else x[:, :2]) for k, x in a.items()}
    sub["bias2"] = a["bias2"]
    ref = brute(sub["q"], sub["k"], sub["v"], sub["bias1"], sub["bias2"], sub["do"])
    o, lse = O.forward(sub["q"], sub["k"], sub["v"], sub["bias1"], sub["bias2"])
    g = O.backward(sub["q"], sub["k"], sub["v"], sub["bias1"], sub["bias2"], sub["do"])
    np.testing.assert_allclose(o, np.array(ref["o"]), atol=1e-12)
    np.testing.assert_allclose(lse, np.array(ref["lse"]), atol=1e-12)
    for key in ("dq", "dk", "dv", "dbias2"):
        np.testing.assert_allclose(g[key], np.array(ref[key]), atol=1e-12, err_msg=key)


# ---------------------------------------------------------- finite differences
def _loss(q, k, v, b1, b2, do):
    o, _ = O.forward(q, k, v, b1, b2)
    return float(np.sum(o * do))


@pytest.mark.parametrize("shape", [(1, 2, 5, 2, 3), (2, 3, 7, 1, 4), (1, 1, 9, 2, 8)])
def test_finite_differences(shape):
    rng = np.random.default_rng(7 + sum(shape))
    # finite (not -inf) masks so that the bias directions are differentiable
    q, k, v, do, b1, b2 = rand_problem(*shape, rng, mask_frac=0.2)
    b1 = np.where(b1 < -1e8, -30.0, b1) + 0.3 * rng.standard_normal(b1.shape)
    g = O.backward(q, k, v, b1, b2, do)
    args = {"q": q, "k": k, "v": v, "b1": b1, "b2": b2}
    gkey = {"q": "dq", "k": "dk", "v": "dv", "b1": "dbias1", "b2": "dbias2"}
    eps = 1e-5
    for name, x in args.items():
        for _ in range(3):
            dirn = rng.standard_normal(x.shape)
            plus = dict(args); plus[name] = x + eps * dirn
            minus = dict(args); minus[name] = x - eps * dirn
            fd = (_loss(plus["q"], plus["k"], plus["v"], plus["b1"], plus["b2"], do)
                  - _loss(minus["q"], minus["k"], minus["v"], minus["b1"], minus["b2"], do)) / (2 * eps)
            an = float(np.sum(g[gkey[name]] * dirn))
            assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (name, fd, an)


# --------------------------------------------------- library special case (torch)
def _torch_sdpa(q, k, v, b1, b2, do):
    """torch's scaled_dot_product_attention with an additive float mask, fp64 CPU."""
    B, N, L, H, D = q.shape
    t = lambda x: torch.tensor(x, dtype=torch.float64, requires_grad=True)
    tq, tk, tv = t(q), t(k), t(v)
    tb1 = t(b1) if b1 is not None else None
    tb2 = t(b2) if b2 is not None else None
    mask = torch.zeros((B, N, H, L, L), dtype=torch.float64)
    if tb1 is not None:
        mask = mask + tb1          # [B,N,1,1,L] broadcasts over heads and queries
    if tb2 is not None:
        mask = mask + tb2          # [B,1,H,L,L] broadcasts over n
    perm = lambda x: x.permute(0, 1, 3, 2, 4)  # -> [B,N,H,L,D]
    out = torch.nn.functional.scaled_dot_product_attention(
        perm(tq), perm(tk), perm(tv), attn_mask=mask, scale=D ** -0.5)
    out = out.permute(0, 1, 3, 2, 4)
    (out * torch.tensor(do)).sum().backward()
    res = {"o": out.detach().numpy(), "dq": tq.grad.numpy(), "dk": tk.grad.numpy(),
           "dv": tv.grad.numpy()}
    if tb1 is not None:
        res["dbias1"] = tb1.grad.numpy()
    if tb2 is not None:
        res["dbias2"] = tb2.grad.numpy()
    return res


@pytest.mark.parametrize("shape,bias1,bias2", [
    ((1, 3, 16, 2, 8), True, True),
    ((2, 2, 11, 3, 4), True, False),
    ((1, 4, 9, 2, 16), False, True),
    ((1, 2, 8, 2, 8), False, False),
])
def test_torch_sdpa(shape, bias1, bias2):
    rng = np.random.default_rng(99 + sum(shape))
    q, k, v, do, b1, b2 = rand_problem(*shape, rng, bias1=bias1, bias2=bias2)
    ref = _torch_sdpa(q, k, v, b1, b2, do)
    o, _ = O.forward(q, k, v, b1, b2)
    g = O.backward(q, k, v, b1, b2, do)
    np.testing.assert_allclose(o, ref["o"], atol=1e-12)
    for key in ("dq", "dk", "dv") + (("dbias1",) if bias1 else ()) + (("dbias2",) if bias2 else ()):
        np.testing.assert_allclose(g[key], ref[key], atol=1e-11, err_msg=key)


# ---------------------------------------------------- closed forms, invariants
def test_single_key():
    """L = 1: O = V, lse = s q.k + bias, dV = dO, dQ = dK = 0, bias grads 0."""
    rng = np.random.default_rng(3)
    q, k, v, do, b1, b2 = rand_problem(2, 3, 1, 2, 8, rng, mask_frac=0.0)
    o, lse = O.forward(q, k, v, b1, b2)
    np.testing.assert_allclose(o, v, atol=1e-15)
    s = 8 ** -0.5
    exp_lse = s * np.einsum("bnlhd,bnlhd->bnhl", q, k) + b2[:, :, :, :, 0].reshape(2, 1, 2, 1)
    np.testing.assert_allclose(lse, exp_lse, atol=1e-13)
    g = O.backward(q, k, v, b1, b2, do)
    np.testing.assert_allclose(g["dv"], do, atol=1e-15)
    for key in ("dq", "dk", "dbias1", "dbias2"):
        np.testing.assert_allclose(g[key], 0.0, atol=1e-15, err_msg=key)


def test_uniform_scores_mean_of_kept_values():
    """Q = 0 and no pair bias: O_i = mean of V over kept keys, lse = log(#kept)."""
    rng = np.random.default_rng(4)
    q, k, v, do, b1, _ = rand_problem(1, 4, 12, 2, 5, rng, mask_frac=0.25, neg_inf=True)
    q[:] = 0.0
    o, lse = O.forward(q, k, v, b1, None)
    for n in range(4):
        kept = np.isfinite(b1[0, n, 0, 0])
        mean = v[0, n, kept].mean(axis=0)            # [H, D]
        for i in range(12):
            np.testing.assert_allclose(o[0, n, i], mean, atol=1e-14)
        np.testing.assert_allclose(lse[0, n], math.log(kept.sum()), atol=1e-14)


def test_two_keys_sigmoid():
    """Two keys: O_i = sigma(x_i0 - x_i1) V_0 + sigma(x_i1 - x_i0) V_1."""
    rng = np.random.default_rng(5)
    q, k, v, do, _, b2 = rand_problem(1, 1, 2, 1, 3, rng, bias1=False)
    o, _ = O.forward(q, k, v, None, b2)
    s = 3 ** -0.5
    for i in range(2):
        x0 = s * q[0, 0, i, 0] @ k[0, 0, 0, 0] + b2[0, 0, 0, i, 0]
        x1 = s * q[0, 0, i, 0] @ k[0, 0, 1, 0] + b2[0, 0, 0, i, 1]
        w0 = 1.0 / (1.0 + math.exp(x1 - x0))
        np.testing.assert_allclose(o[0, 0, i, 0], w0 * v[0, 0, 0, 0] + (1 - w0) * v[0, 0, 1, 0],
                                   atol=1e-14)


def test_rows_of_p_sum_to_one_and_lse_consistent():
    rng = np.random.default_rng(6)
    q, k, v, do, b1, b2 = rand_problem(1, 1, 13, 1, 4, rng, neg_inf=True)
    s = 0.5
    bias = b1[0, 0, 0, 0][None, :] + b2[0, 0, 0]
    o, lse, p = O.slice_forward(q[0, 0, :, 0], k[0, 0, :, 0], v[0, 0, :, 0], bias, s)
    np.testing.assert_allclose(p.sum(axis=1), 1.0, atol=1e-14)
    x = s * q[0, 0, :, 0] @ k[0, 0, :, 0].T + bias
    np.testing.assert_allclose(np.exp(x - lse[:, None]).sum(axis=1), 1.0, atol=1e-14)
    np.testing.assert_allclose(p @ v[0, 0, :, 0], o, atol=1e-14)


@pytest.mark.parametrize("mval", [-1e9, -np.inf])
def test_mask_equals_gathered_keys(mval):
    """A -1e9 (or -inf) key mask equals attention over the kept keys only."""
    rng = np.random.default_rng(8)
    q, k, v, do, b1, b2 = rand_problem(1, 3, 10, 2, 4, rng, mask_frac=0.4)
    b1 = np.where(b1 < -1e8, mval, b1)
    o, lse = O.forward(q, k, v, b1, b2)
    g = O.backward(q, k, v, b1, b2, do)
    s = 0.5
    for n in range(3):
        kept = b1[0, n, 0, 0] > -1e8
        for h in range(2):
            qs, ks, vs = q[0, n, :, h], k[0, n, kept, h], v[0, n, kept, h]
            bias = b2[0, 0, h][:, kept]            # no mask: the masked keys are gone
            os_, lses, _ = O.slice_forward(qs, ks, vs, bias, s)
            np.testing.assert_allclose(o[0, n, :, h], os_, atol=1e-13)
            np.testing.assert_allclose(lse[0, n, h], lses, atol=1e-9)
            gs = O.slice_backward(qs, ks, vs, bias, do[0, n, :, h], s)
            np.testing.assert_allclose(g["dq"][0, n, :, h], gs["dq"], atol=1e-12)
            np.testing.assert_allclose(g["dk"][0, n, kept, h], gs["dk"], atol=1e-12)
            np.testing.assert_allclose(g["dv"][0, n, kept, h], gs["dv"], atol=1e-12)
            np.testing.assert_allclose(g["dk"][0, n, ~kept, h], 0.0, atol=1e-12)
            np.testing.assert_allclose(g["dv"][0, n, ~kept, h], 0.0, atol=1e-12)


def test_shift_and_permutation_invariance():
    rng = np.random.default_rng(9)
    q, k, v, do, b1, b2 = rand_problem(1, 2, 9, 2, 4, rng)
    o, lse = O.forward(q, k, v, b1, b2)
    c = rng.standard_normal((1, 1, 2, 9, 1))
    o2, lse2 = O.forward(q, k, v, b1, b2 + c)     # per-row constant on the pair bias
    np.testing.assert_allclose(o2, o, atol=1e-13)
    np.testing.assert_allclose(lse2, lse + c[:, 0, :, :, 0][:, None], atol=1e-12)
    perm = rng.permutation(9)                      # permute keys jointly
    o3, lse3 = O.forward(q, k[:, :, perm], v[:, :, perm], b1[..., perm], b2[..., perm])
    np.testing.assert_allclose(o3, o, atol=1e-13)
    np.testing.assert_allclose(lse3, lse, atol=1e-13)


def test_one_hot_bias_selects_value():
    rng = np.random.default_rng(10)
    q, k, v, do, _, b2 = rand_problem(1, 1, 8, 1, 4, rng, bias1=False)
    b2[:] = 0.0
    b2[0, 0, 0, :, 5] = 40.0
    q *= 0.1
    o, _ = O.forward(q, k, v, None, b2)
    np.testing.assert_allclose(o[0, 0, :, 0], np.broadcast_to(v[0, 0, 5, 0], (8, 4)), atol=1e-14)


def test_zero_bias_equals_plain_attention():
    rng = np.random.default_rng(11)
    q, k, v, do, _, _ = rand_problem(1, 2, 7, 2, 4, rng, bias1=False, bias2=False)
    z1, z2 = np.zeros((1, 2, 1, 1, 7)), np.zeros((1, 1, 2, 7, 7))
    o, lse = O.forward(q, k, v, z1, z2)
    o0, lse0 = O.forward(q, k, v, None, None)
    np.testing.assert_array_equal(o, o0)
    ref = _torch_sdpa(q, k, v, None, None, do)
    np.testing.assert_allclose(o0, ref["o"], atol=1e-12)


def test_score_gradient_rows_sum_to_zero():
    """sum_j dS_ij = 0, so each row of dbias2 and the sum of dbias1 vanish."""
    rng = np.random.default_rng(12)
    q, k, v, do, b1, b2 = rand_problem(2, 3, 10, 2, 4, rng)
    g = O.backward(q, k, v, b1, b2, do)
    np.testing.assert_allclose(g["dbias2"].sum(axis=-1), 0.0, atol=1e-12)
    np.testing.assert_allclose(g["dbias1"].sum(axis=-1), 0.0, atol=1e-12)


def test_dbias2_sums_over_rows():
    """N identical rows give N times the one-row gradient; permuting n leaves it unchanged."""
    rng = np.random.default_rng(13)
    q, k, v, do, b1, b2 = rand_problem(1, 1, 8, 2, 4, rng)
    g1 = O.backward(q, k, v, b1, b2, do)
    rep = lambda x: np.repeat(x, 5, axis=1)
    g5 = O.backward(rep(q), rep(k), rep(v), rep(b1), b2, rep(do))
    np.testing.assert_allclose(g5["dbias2"], 5 * g1["dbias2"], atol=1e-12)
    q, k, v, do, b1, b2 = rand_problem(1, 4, 8, 2, 4, rng)
    ga = O.backward(q, k, v, b1, b2, do)
    p = rng.permutation(4)
    gb = O.backward(q[:, p], k[:, p], v[:, p], b1[:, p], b2, do[:, p])
    np.testing.assert_allclose(gb["dbias2"], ga["dbias2"], atol=1e-12)


def test_fully_masked_row_is_empty():
    """Reading for a row with every key -inf: O = 0, lse = -inf, zero gradients."""
    rng = np.random.default_rng(14)
    q, k, v, do, b1, b2 = rand_problem(1, 2, 6, 1, 4, rng, mask_frac=0.0)
    b1[0, 1, 0, 0, :] = -np.inf
    o, lse = O.forward(q, k, v, b1, b2)
    assert np.all(o[0, 1] == 0.0) and np.all(lse[0, 1] == -np.inf)
    assert np.all(np.isfinite(o[0, 0]))
    g = O.backward(q, k, v, b1, b2, do)
    for key in ("dq", "dk", "dv"):
        assert np.all(g[key][0, 1] == 0.0)
        assert np.all(np.isfinite(g[key]))


# ----------------------------------------------------------- sampled helpers
def test_sampled_helpers_match_full_oracle():
    rng = np.random.default_rng(15)
    q, k, v, do, b1, b2 = rand_problem(2, 3, 11, 2, 4, rng)
    o, lse = O.forward(q, k, v, b1, b2)
    g = O.backward(q, k, v, b1, b2, do)
    for (b, n, h) in [(0, 0, 0), (1, 2, 1), (0, 1, 1)]:
        os_, lses = O.forward_slice_sample(q, k, v, b1, b2, b, n, h)
        np.testing.assert_allclose(os_, o[b, n, :, h], atol=1e-14)
        np.testing.assert_allclose(lses, lse[b, n, h], atol=1e-14)
        gs = O.backward_slice_sample(q, k, v, b1, b2, do, b, n, h)
        for key in ("dq", "dk", "dv"):
            np.testing.assert_allclose(gs[key], g[key][b, n, :, h], atol=1e-14)
    rows = [0, 4, 10]
    ds = O.dbias2_sample(q, k, v, b1, b2, do, 1, 1, rows)
    np.testing.assert_allclose(ds, g["dbias2"][1, 0, 1, rows], atol=1e-13)


# ---------------------------------------------------------------- masked key tail
def test_masked_key_tail_contributes_nothing():
    """Keys with a -1e9 key mask drop out exactly: the result on L keys equals the
    result on the kept prefix alone, and those keys get zero dK, dV (and zero
    pair-bias gradient in their columns).  This is what makes skipping a key tile
    whose keys are all masked exact."""
    rng = np.random.default_rng(77)
    B, N, L, H, D, j0 = 1, 2, 12, 2, 8, 7
    q, k, v, do, _, b2 = rand_problem(B, N, L, H, D, rng, bias1=False)
    b1 = rng.standard_normal((B, N, 1, 1, L))
    b1[..., j0:] = -1e9
    o, lse = O.forward(q, k, v, b1, b2)
    g = O.backward(q, k, v, b1, b2, do)
    # the same attention over the kept keys only (L queries, j0 keys), written out here
    # since the oracle takes square problems
    s = 1.0 / math.sqrt(D)
    for b in range(B):
        for n in range(N):
            for h in range(H):
                sc = s * q[b, n, :, h] @ k[b, n, :j0, h].T + b1[b, n, 0, 0, :j0] + b2[b, 0, h, :, :j0]
                m = sc.max(axis=1, keepdims=True)
                p = np.exp(sc - m)
                ref = (p / p.sum(axis=1, keepdims=True)) @ v[b, n, :j0, h]
                assert np.allclose(o[b, n, :, h], ref, rtol=0, atol=1e-12)
                assert np.allclose(lse[b, n, h], (m[:, 0] + np.log(p.sum(axis=1))), rtol=0, atol=1e-12)
    assert np.all(g["dk"][:, :, j0:] == 0) and np.all(g["dv"][:, :, j0:] == 0)
    assert np.all(g["dbias2"][..., j0:] == 0) and np.all(g["dbias1"][..., j0:] == 0)
