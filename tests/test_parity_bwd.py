"""GPU backward parity: dQ, dK, dV and dbias2 from the sm_103a kernels (through
the C ABI) against the fp64 oracle's analytic gradients on seeded inputs, and
bitwise reproducibility of dbias2."""
import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300.workload import WORKLOADS, make_inputs, workload_inputs
from oracle import evo_oracle as O
from tests.parity_util import GRAD_TOL, np64, rel_l2, run_bwd, run_fwd, to_dev

pytestmark = pytest.mark.gpu

SMALL = [
    (1, 8, 32, 2, 16, "fp16", ("random", 0.10), 1.0, True),
    (2, 3, 300, 2, 32, "bf16", ("random", 0.05), 1.0, True),
    (1, 4, 200, 3, 8, "fp16", ("tail", 0.15), 0.5, True),
    (1, 3, 131, 2, 24, "bf16", ("random", 0.05), 1.0, True),   # odd L: pair bias via plain loads
    (2, 2, 257, 1, 64, "fp16", ("random", 0.05), 1.0, True),
    (1, 2, 1, 1, 8, "bf16", None, 1.0, True),                   # L = 1: dQ = dK = dbias2 = 0, dV = dO
    (1, 2, 17, 2, 16, "fp16", ("random", 0.10), None, True),
    (1, 3, 96, 2, 40, "bf16", None, 1.0, False),
    (1, 2, 128, 2, 48, "fp16", ("tail", 0.5), None, False),
    (1, 2, 384, 1, 56, "bf16", ("tail", 0.03), 1.0, True),
    (1, 5, 33, 1, 32, "fp16", ("random", 0.3), 1.0, True),
    (1, 3, 700, 2, 16, "fp16", ("random", 0.05), 1.0, True),   # key-major, dQ streamed, D = 16 (6 key tiles)
    (2, 3, 450, 1, 32, "bf16", ("tail", 0.10), None, True),    # key-major, dQ streamed, ragged L, two batches
]


def _check(inp, gpu, dtype, keys=("dq", "dk", "dv", "dbias2")):
    a = {k: np64(v) for k, v in inp.items()}
    g = O.backward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"], a["do"])
    dq, dk, dv, db2 = gpu
    got = {"dq": dq, "dk": dk, "dv": dv, "dbias2": db2}
    errs = {}
    for k in keys:
        if got[k] is None:
            continue
        ref = g[k]
        if np.linalg.norm(ref) == 0.0:
            # exact zero in exact arithmetic (e.g. L = 1); the GPU forms delta and
            # dP with different fp32 rounding orders, so allow rounding-level residue
            assert np.max(np.abs(np64(got[k]))) <= 1e-4, k
            continue
        errs[k] = rel_l2(np64(got[k]), ref)
        assert errs[k] <= GRAD_TOL[dtype], (k, errs[k])
    return errs


def _run(inp):
    d = to_dev(inp)
    out, lse = run_fwd(d)
    return d, out, lse, run_bwd(d, out, lse)


@pytest.mark.parametrize("case", SMALL, ids=lambda c: "x".join(map(str, c[:5])) + "-" + c[5])
def test_small(case):
    B, N, L, H, D, dt, mask, sig, hb1 = case
    inp = make_inputs(B, N, L, H, D, dtype=dt, mask=mask, bias2_sigma=sig, seed=11, has_bias1=hb1)
    if not hb1:
        inp["bias1"] = None
    _, _, _, gpu = _run(inp)
    _check(inp, gpu, inp["q"].dtype)


def test_single_key_closed_form():
    inp = make_inputs(2, 3, 1, 2, 16, dtype="fp16", mask=None, bias2_sigma=1.0, seed=2)
    _, _, _, (dq, dk, dv, db2) = _run(inp)
    # closed form: dQ = dK = dbias2 = 0 and dV = dO, up to fp32 rounding of delta vs dP
    for t in (dq, dk, db2):
        assert t.float().abs().max().item() <= 1e-4
    assert (dv.float() - inp["do"].cuda().float()).abs().max().item() <= 1e-3


def test_fully_masked_rows_fp16():
    inp = make_inputs(1, 3, 70, 2, 16, dtype="fp16", mask=("random", 0.1), seed=5)
    inp["bias1"][0, 1] = float("-inf")
    _, _, _, gpu = _run(inp)
    dq, dk, dv, _ = gpu
    assert torch.all(dq[0, 1] == 0) and torch.all(dk[0, 1] == 0) and torch.all(dv[0, 1] == 0)
    _check(inp, gpu, torch.float16)


def test_dbias2_bitwise_reproducible():
    inp = make_inputs(1, 40, 200, 2, 32, dtype="bf16", mask=("random", 0.05), seed=9)
    d = to_dev(inp)
    out, lse = run_fwd(d)
    first = run_bwd(d, out, lse)[3].clone()
    for _ in range(3):
        again = run_bwd(d, out, lse)[3]
        assert torch.equal(first.view(torch.int16), again.view(torch.int16))


def test_workspace_may_hold_garbage():
    """The backward must not depend on the workspace's previous contents."""
    from memory_efficient_biased_gb300 import evo_attn as E
    inp = make_inputs(1, 4, 150, 2, 32, dtype="fp16", mask=("random", 0.05), seed=4)
    d = to_dev(inp)
    out, lse = run_fwd(d)
    need = E.evo_attn_bwd_workspace_bytes(tuple(d["q"].shape), d["q"].dtype, True)
    ws = torch.full((need,), 0x7F, dtype=torch.uint8, device="cuda")
    r1 = E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], workspace=ws)
    ws.fill_(0xFF)
    r2 = E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], workspace=ws)
    assert E.evo_attn_device_status() == 0
    for x, y in zip(r1[1:], r2[1:]):
        assert torch.equal(x, y)
    assert (r1[0].float() - r2[0].float()).abs().max().item() <= 1e-2 * r1[0].float().abs().max().item()
    _check(inp, r2, torch.float16)


@pytest.mark.parametrize("name,dtype", [("tiny", "fp16"), ("msa_row", "fp16"), ("msa_row", "bf16"),
                                        ("many_head", "bf16")])
def test_workload_full(name, dtype):
    inp = workload_inputs(name, dtype)
    _, _, _, gpu = _run(inp)
    _check(inp, gpu, inp["q"].dtype)


@pytest.mark.parametrize("name", ["msa_col", "triangle"])
def test_workload_sampled(name):
    """Full-size workloads: sampled slices for dQ/dK/dV, sampled rows for dbias2."""
    w = WORKLOADS[name]
    inp = workload_inputs(name)
    _, _, _, (dq, dk, dv, db2) = _run(inp)
    dq, dk, dv = dq.cpu(), dk.cpu(), dv.cpu()
    tol = GRAD_TOL[torch.bfloat16]
    rng = np.random.default_rng(1)
    picks = [(0, 0, 0), (0, w.N - 1, w.H - 1)] + [(0, int(rng.integers(w.N)), int(rng.integers(w.H)))
                                                 for _ in range(4)]
    for (b, n, h) in picks:
        one = lambda t: None if t is None else t[b:b + 1, n:n + 1].double().numpy()
        b2 = None if inp["bias2"] is None else inp["bias2"][b:b + 1].double().numpy()
        g = O.backward_slice_sample(one(inp["q"]), one(inp["k"]), one(inp["v"]), one(inp["bias1"]), b2,
                                    one(inp["do"]), 0, 0, h)
        for key, t in (("dq", dq), ("dk", dk), ("dv", dv)):
            e = rel_l2(t[b, n, :, h].double().numpy(), g[key])
            assert e <= tol, (key, b, n, h, e)
    if inp["bias2"] is not None:
        db2 = db2.cpu()
        for h in range(w.H):
            rows = sorted({0, w.L - 1, int(rng.integers(w.L)), int(rng.integers(w.L))})
            col = lambda t: None if t is None else t[:, :, :, h:h + 1].double().numpy()
            ref = O.dbias2_sample(col(inp["q"]), col(inp["k"]), col(inp["v"]), inp["bias1"].double().numpy(),
                                  inp["bias2"][:, :, h:h + 1].double().numpy(), col(inp["do"]), 0, 0, rows)
            e = rel_l2(db2[0, 0, h, rows].double().numpy(), ref)
            assert e <= tol, (h, e)
