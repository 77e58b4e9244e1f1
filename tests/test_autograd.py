"""GPU: the autograd wrapper (evoformer_attention / DS4Sci_EvoformerAttention)
against the fp64 oracle, and its peak device memory against dense attention."""
import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300.autograd import DS4Sci_EvoformerAttention, evoformer_attention
from memory_efficient_biased_gb300.workload import make_inputs
from oracle import evo_oracle as O
from tests.parity_util import FWD_TOL, GRAD_TOL, fwd_rel_err, np64, rel_l2

pytestmark = pytest.mark.gpu


def _leaf(t):
    return None if t is None else t.cuda().requires_grad_(True)


@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("biases", ["both", "mask", "none"])
def test_autograd_matches_oracle(dtype, biases):
    inp = make_inputs(1, 3, 200, 2, 32, dtype=dtype, mask=("random", 0.05),
                      bias2_sigma=1.0 if biases == "both" else None, seed=13)
    if biases == "none":
        inp["bias1"] = None
    q, k, v = _leaf(inp["q"]), _leaf(inp["k"]), _leaf(inp["v"])
    b1, b2 = _leaf(inp["bias1"]), _leaf(inp["bias2"])
    out = evoformer_attention(q, k, v, [b1, b2])
    (out.float() * inp["do"].cuda().float()).sum().backward()
    a = {key: np64(val) for key, val in inp.items()}
    o_ref, _ = O.forward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"])
    g = O.backward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"], a["do"])
    dt = inp["q"].dtype
    assert fwd_rel_err(np64(out), o_ref) <= FWD_TOL[dt]
    for name, t in (("dq", q), ("dk", k), ("dv", v), ("dbias1", b1), ("dbias2", b2)):
        if t is not None:
            assert rel_l2(np64(t.grad), g[name]) <= GRAD_TOL[dt], name


def test_pages_name_and_bias_list_forms():
    inp = make_inputs(1, 2, 64, 2, 16, dtype="bf16", mask=("random", 0.1), bias2_sigma=1.0, seed=3)
    q, k, v = (inp[n].cuda() for n in ("q", "k", "v"))
    b1, b2 = inp["bias1"].cuda(), inp["bias2"].cuda()
    full = DS4Sci_EvoformerAttention(q, k, v, [b1, b2])
    assert torch.equal(full, evoformer_attention(q, k, v, [b1, b2]))
    assert torch.equal(evoformer_attention(q, k, v, [b1]), evoformer_attention(q, k, v, [b1, None]))
    assert torch.equal(evoformer_attention(q, k, v), evoformer_attention(q, k, v, []))
    with pytest.raises(ValueError):
        evoformer_attention(q, k, v, [b1, b2, b2])


def _dense(q, k, v, b1, b2):
    s = q.shape[-1] ** -0.5
    sc = torch.einsum("bnihd,bnjhd->bnhij", q, k) * s + b1 + b2
    return torch.einsum("bnhij,bnjhd->bnihd", torch.softmax(sc, dim=-1), v)


def test_peak_memory_against_dense_attention():
    """Fwd + bwd at the MSA row-wise shape: the L×L scores never exist, so the
    peak beyond the inputs is a fraction of dense attention's."""
    inp = make_inputs(1, 256, 256, 4, 32, dtype="bf16", mask=("random", 0.05), bias2_sigma=1.0, seed=0)
    peaks = {}
    for name, fn in (("ours", evoformer_attention), ("dense", None)):
        q, k, v, b1, b2 = (_leaf(inp[n]) for n in ("q", "k", "v", "bias1", "bias2"))
        do = inp["do"].cuda()
        torch.cuda.synchronize()
        base = torch.cuda.memory_allocated()
        torch.cuda.reset_peak_memory_stats()
        out = fn(q, k, v, [b1, b2]) if fn else _dense(q, k, v, b1, b2)
        out.backward(do)
        torch.cuda.synchronize()
        peaks[name] = torch.cuda.max_memory_allocated() - base
        del q, k, v, b1, b2, out
    assert peaks["ours"] * 3 <= peaks["dense"], peaks
