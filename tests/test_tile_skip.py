"""GPU tests of masked key-tile skipping (the EVO_OPT_SKIP_MASKED_TILES option of
evo_attn_fwd_opts / evo_attn_bwd_opts).

A key tile whose keys are all masked contributes exactly nothing once exp
underflows to 0 (web page "DeepSpeed4Science 技术指南…" §3.6: the key mask is
a large negative bias), so skipping it must leave every result unchanged, bitwise:
O, lse, dQ, dK, dV and both bias gradients (every gradient is summed in a fixed
order, and a skipped tile's terms are exact zeros).  Cases cover tail masks (the
same tiles masked in every row), per-row masks (some rows of a slice range
skipping a tile, others not), a streamed pair bias, several batches, strided
outputs, and a row whose every key is masked (nothing skipped there).
"""
import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300 import evo_attn as E
from memory_efficient_biased_gb300.workload import MASK_VALUE, make_inputs
from oracle import evo_oracle as O
from tests.parity_util import FWD_TOL, GRAD_TOL, fwd_rel_err, lse_err, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu


def masked_rows(inp, spec, seed=0):
    """Overwrite bias1 by `spec`: ("tail", j0) masks keys >= j0 in every row;
    ("tiles", p) masks each whole 128-key tile of each row with probability p
    (keeping tile 0 kept in every row but the last one of each b, which is
    masked entirely)."""
    b1 = inp["bias1"].float()
    B, N, _, _, L = b1.shape
    kind, arg = spec
    if kind == "tail":
        b1[..., arg:] = MASK_VALUE
    else:
        rng = np.random.default_rng(seed)
        KT = (L + 127) // 128
        for b in range(B):
            for n in range(N):
                for t in range(1, KT):
                    if rng.random() < arg:
                        b1[b, n, 0, 0, t * 128:(t + 1) * 128] = MASK_VALUE
            b1[b, N - 1] = MASK_VALUE  # a row with no kept key
    inp["bias1"] = b1.to(inp["q"].dtype)
    return inp


def run_all(d, dq=None, dk=None, dv=None, skip=False, threshold=-1.0e4):
    opt = dict(skip_masked_tiles=skip, skip_threshold=threshold)
    out, lse = E.evo_attn_fwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], **opt)
    ws = torch.empty(E.evo_attn_bwd_workspace_bytes(tuple(d["q"].shape), d["q"].dtype, d["bias2"] is not None,
                                                    True), dtype=torch.uint8, device="cuda")
    g = E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], dq=dq, dk=dk, dv=dv,
                            workspace=ws, want_dbias1=True, **opt)
    torch.cuda.synchronize()
    assert E.evo_attn_device_status() == 0 and E.evo_attn_bwd_status(ws) == 0
    return (out, lse) + tuple(g)


# (B, N, L, H, D, dtype, bias2_sigma, mask spec): backward schedule on the right
CASES = [
    (1, 6, 700, 2, 64, "bf16", None, ("tail", 420)),      # per key tile, no pair bias
    (1, 6, 700, 2, 32, "fp16", None, ("tail", 420)),      # per key tile (D = 32, 6 key tiles)
    (2, 5, 300, 2, 64, "bf16", 1.0, ("tiles", 0.5)),      # per key tile, pair bias, per-row masks
    (1, 4, 1100, 1, 64, "fp16", 1.0, ("tiles", 0.4)),     # per key tile, streamed pair bias
    (1, 4, 256, 3, 32, "bf16", 1.0, ("tiles", 0.5)),      # key-major backward: forward skips only
    (1, 3, 520, 2, 16, "fp16", 0.5, ("tail", 260)),       # slice or key-major backward
]


def _ids(c):
    return "x".join(map(str, c[:5])) + f"-{c[5]}-{c[7][0]}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_skipping_changes_nothing(case):
    B, N, L, H, D, dt, sig, spec = case
    inp = masked_rows(make_inputs(B, N, L, H, D, dtype=dt, mask=None, bias2_sigma=sig, seed=31), spec, seed=7)
    d = to_dev(inp)
    ref = run_all(d)
    got = run_all(d, skip=True)
    names = ("out", "lse", "dq", "dk", "dv", "dbias1", "dbias2")
    for name, x, y in zip(names, got, ref):
        if x is None:
            assert y is None
        else:
            assert torch.equal(x, y), name

    a = {k: np64(v) for k, v in inp.items()}
    o_ref, lse_ref = O.forward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"])
    kept = np.isfinite(lse_ref) if dt == "fp16" else np.ones_like(lse_ref, dtype=bool)
    if dt == "fp16":  # fp16 masks are -inf: the fully masked rows are empty softmaxes
        assert lse_err(np64(got[1]), lse_ref) <= 1e-3
    else:  # bf16 masks are finite: compare the rows that keep a key
        kept[:, -1] = False
    o_rows = np.moveaxis(kept, 3, 2)[..., None]  # [B,N,L,H,1]
    assert fwd_rel_err(np64(got[0]) * o_rows, o_ref * o_rows) <= FWD_TOL[inp["q"].dtype]
    if dt == "fp16":
        g = O.backward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"], a["do"])
        tol = GRAD_TOL[inp["q"].dtype]
        for name, t in zip(("dq", "dk", "dv"), got[2:5]):
            assert rel_l2(np64(t), g[name]) <= tol, name


def test_skipping_with_strided_gradients():
    """dK and dV of skipped tiles are written as zeros through the gradients' strides."""
    B, N, L, H, D = 1, 4, 640, 2, 64
    inp = masked_rows(make_inputs(B, N, L, H, D, dtype="bf16", mask=None, bias2_sigma=None, seed=2),
                      ("tail", 300))
    d = to_dev(inp)
    ref = run_all(d)
    bufs = [torch.full((B, L, N, H, D), 7.0, dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    views = [b.transpose(1, 2) for b in bufs]
    for v in views[1:]:
        v.fill_(3.0)  # the skipped tiles' rows must be overwritten with zeros
    got = run_all(d, *views, skip=True)
    assert torch.equal(got[3], ref[3]) and torch.equal(got[4], ref[4]) and torch.equal(got[2], ref[2])
    assert torch.all(got[3][:, :, 384:] == 0) and torch.all(got[4][:, :, 384:] == 0)


def test_threshold_decides_what_is_masked():
    """With a threshold below the mask value nothing counts as masked: same results."""
    inp = masked_rows(make_inputs(1, 3, 600, 1, 64, dtype="bf16", mask=None, bias2_sigma=None, seed=4),
                      ("tail", 256))
    d = to_dev(inp)
    ref = run_all(d)
    got = run_all(d, skip=True, threshold=-3.0e38)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[3], ref[3])


def test_full_size_column_workload():
    """MSA column-wise attention at full size (keys >= 870 masked: the last key tile of
    every row is skipped), in the configuration the bench times with skipping on:
    the same bytes as the unskipped run, whose parity with the oracle is tested on
    sampled slices elsewhere."""
    from memory_efficient_biased_gb300.workload import workload_inputs
    d = to_dev(workload_inputs("msa_col", "bf16"))
    ref = run_all(d)
    got = run_all(d, skip=True)
    for name, x, y in zip(("out", "lse", "dq", "dk", "dv", "dbias1"), got, ref):
        assert torch.equal(x, y), name
    assert torch.all(got[3][:, :, 896:] == 0) and torch.all(got[4][:, :, 896:] == 0)


def test_skipping_with_batch_by_batch_strided_call():
    """B = 2 with transposed inputs and outputs runs batch by batch; each batch writes
    its own skip bits in the shared workspace."""
    B, N, L, H, D = 2, 3, 520, 2, 64
    inp = masked_rows(make_inputs(B, N, L, H, D, dtype="bf16", mask=None, bias2_sigma=1.0, seed=9), ("tiles", 0.5))
    d = to_dev(inp)
    ref = run_all(d)

    def tr(t):
        buf = torch.empty((B, L, N, H, D), dtype=t.dtype, device=t.device)
        v = buf.transpose(1, 2)
        v.copy_(t)
        return v

    q, k, v, do = (tr(d[n]) for n in ("q", "k", "v", "do"))
    out, lse = E.evo_attn_fwd_opts(q, k, v, d["bias1"], d["bias2"], out=tr(torch.zeros_like(d["q"])),
                                   skip_masked_tiles=True)
    g = E.evo_attn_bwd_opts(q, k, v, d["bias1"], d["bias2"], out, lse, do, dq=tr(d["q"]), dk=tr(d["q"]),
                            dv=tr(d["q"]), want_dbias1=True, skip_masked_tiles=True)
    torch.cuda.synchronize()
    assert E.evo_attn_device_status() == 0
    assert torch.equal(out, ref[0]) and torch.equal(lse, ref[1])
    assert torch.equal(g[1], ref[3]) and torch.equal(g[2], ref[4]) and torch.equal(g[3], ref[5])
    assert torch.equal(g[4], ref[6]) and torch.equal(g[0], ref[2])


def test_more_than_64_key_tiles_skip_nothing():
    """Past 64 key tiles the skip bit sets do not reach: skipping switches itself off."""
    inp = masked_rows(make_inputs(1, 1, 65 * 128, 1, 16, dtype="fp16", mask=None, bias2_sigma=None, seed=3),
                      ("tail", 64 * 128))
    d = to_dev(inp)
    ref = run_all(d)
    got = run_all(d, skip=True)
    assert torch.equal(got[0], ref[0]) and torch.equal(got[1], ref[1])
    assert torch.equal(got[3], ref[3]) and torch.equal(got[4], ref[4])
