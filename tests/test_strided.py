"""GPU tests of the strided entry points (evo_attn_fwd_strided / evo_attn_bwd_strided).

The Evoformer's transposed usages (column-wise MSA attention, triangle
attention around the ending node: web page "DeepSpeed4Science 技术指南…" §3.6)
attend over the other axis of a [B, A1, A2, H, D] buffer; the strided calls
read that view in place.  A strided call must give exactly the bytes of the
packed call on the same values — the kernels, schedule and summation order are
the same, and every gradient is summed in a fixed order.  Outputs written through strides must touch their
own elements only.  One case per backward schedule, the batch-by-batch path
(B > 1 with a transposed view), padded rows, an odd head dimension and an odd
sequence length; the oracle checks the strided result directly as well.
"""
import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300 import evo_attn as E
from memory_efficient_biased_gb300.autograd import evoformer_attention, readable_in_place
from memory_efficient_biased_gb300.workload import make_inputs
from oracle import evo_oracle as O
from tests.parity_util import FWD_TOL, GRAD_TOL, fwd_rel_err, np64, rel_l2, to_dev

pytestmark = pytest.mark.gpu

SENTINEL = 7.0


def transposed(t, fill=None):
    """A [B,N,L,H,D] view of a [B,L,N,H,D] buffer holding t's values (or `fill`)."""
    B, N, L, H, D = t.shape
    buf = torch.empty((B, L, N, H, D), dtype=t.dtype, device=t.device)
    view = buf.transpose(1, 2)
    if fill is None:
        view.copy_(t)
    else:
        buf.fill_(fill)
    return view, buf


def padded(t, fill=None, extra=3):
    """A [B,N,L,H,D] view of a [B,N,L+extra,H,D] buffer (rows between n's unused)."""
    B, N, L, H, D = t.shape
    buf = torch.full((B, N, L + extra, H, D), SENTINEL, dtype=t.dtype, device=t.device)
    view = buf[:, :, :L]
    if fill is None:
        view.copy_(t)
    return view, buf


def outside_untouched(buf, view):
    """Every element of buf that is not part of view still holds SENTINEL."""
    mask = torch.ones(buf.shape, dtype=torch.bool, device=buf.device)
    idx = torch.arange(buf.numel(), device=buf.device).view(buf.shape)
    inside = torch.as_strided(idx, view.shape, view.stride(), view.storage_offset() - buf.storage_offset())
    mask.view(-1)[inside.reshape(-1)] = False
    return bool(torch.all(buf[mask] == SENTINEL))


# (B, N, L, H, D, dtype, mask, bias2_sigma, layout): schedule on the right
CASES = [
    (1, 4, 200, 3, 8, "fp16", ("random", 0.10), 0.5, "transposed"),   # key-major
    (2, 3, 256, 2, 32, "bf16", ("random", 0.05), 1.0, "transposed"),   # key-major, batch by batch
    (1, 2, 300, 2, 32, "fp16", ("random", 0.05), 1.0, "transposed"),   # key-major, dQ streamed
    (1, 2, 257, 1, 64, "bf16", ("random", 0.05), 1.0, "transposed"),   # per key tile
    (2, 2, 200, 1, 64, "fp16", ("tail", 0.05), 1.0, "transposed"),     # per key tile, batch by batch
    (1, 3, 131, 2, 24, "bf16", ("tail", 0.05), None, "padded"),        # odd D and L, no pair bias
    (2, 2, 384, 2, 16, "fp16", ("random", 0.05), 1.0, "padded"),       # key-major (D = 16), padded rows
    (2, 2, 640, 1, 16, "bf16", ("random", 0.05), None, "transposed"),  # key-major, dQ streamed, batch by batch
]


def _ids(c):
    return "x".join(map(str, c[:5])) + f"-{c[5]}-{c[8]}"


@pytest.mark.parametrize("case", CASES, ids=_ids)
def test_strided_matches_packed(case):
    B, N, L, H, D, dt, mask, sig, kind = case
    make = transposed if kind == "transposed" else padded
    inp = make_inputs(B, N, L, H, D, dtype=dt, mask=mask, bias2_sigma=sig, seed=23)
    d = to_dev(inp)
    b1, b2 = d["bias1"], d["bias2"]

    # packed reference call
    out_p, lse_p = E.evo_attn_fwd(d["q"], d["k"], d["v"], b1, b2)
    ref = E.evo_attn_bwd_ex(d["q"], d["k"], d["v"], b1, b2, out_p, lse_p, d["do"])
    assert E.evo_attn_device_status() == 0

    # the same values behind strides, outputs into strided buffers prefilled with a sentinel
    qs, ks, vs, dos = (make(d[n])[0] for n in ("q", "k", "v", "do"))
    out_s, out_buf = make(d["q"], fill=SENTINEL)
    grads = [make(d["q"], fill=SENTINEL) for _ in range(3)]
    out_s, lse_s = E.evo_attn_fwd_strided(qs, ks, vs, b1, b2, out=out_s)
    assert E.evo_attn_device_status() == 0
    assert torch.equal(out_s, out_p) and torch.equal(lse_s, lse_p)
    assert outside_untouched(out_buf, out_s)

    dq, dk, dv, db1, db2 = E.evo_attn_bwd_strided(qs, ks, vs, b1, b2, out_s, lse_s, dos,
                                                  dq=grads[0][0], dk=grads[1][0], dv=grads[2][0],
                                                  want_dbias1=True)
    assert E.evo_attn_device_status() == 0
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]) and torch.equal(db1, ref[3])
    if b2 is not None:
        assert torch.equal(db2, ref[4])
    assert torch.equal(dq, ref[0])
    for view, buf in grads:
        assert outside_untouched(buf, view)

    # and against the fp64 oracle directly
    a = {k: np64(v) for k, v in inp.items()}
    o_ref, _ = O.forward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"])
    assert fwd_rel_err(np64(out_s), o_ref) <= FWD_TOL[inp["q"].dtype]
    g = O.backward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"], a["do"])
    tol = GRAD_TOL[inp["q"].dtype]
    for name, t in (("dq", dq), ("dk", dk), ("dv", dv), ("dbias1", db1)):
        assert rel_l2(np64(t), g[name]) <= tol, name


def test_strided_rejects_overlapping_rows():
    inp = make_inputs(1, 2, 64, 2, 16, dtype="fp16", mask=None, bias2_sigma=None, seed=1)
    d = to_dev(inp)
    q = d["q"]
    # shape (1, 2, 64, 2, 16): rows of one n overlap, token stride 16 < H*D = 32
    bad = torch.as_strided(q, q.shape, (2 * 64 * 32, 64 * 32, 16, 16, 1))
    with pytest.raises(E.EvoAttnError, match="EVO_ERR_BAD_LAYOUT"):
        E.evo_attn_fwd_strided(bad, d["k"], d["v"])
    assert not readable_in_place(bad)


@pytest.mark.parametrize("dt", ["fp16", "bf16"])
def test_autograd_reads_transposed_views_in_place(dt):
    """Column-wise attention as a user writes it: transpose the MSA axes, attend,
    transpose back.  Same values and gradients as on packed copies."""
    B, S, R, H, D = 1, 96, 160, 4, 32  # MSA [B, N_seq, N_res, H, D]; attend along N_seq
    inp = make_inputs(B, R, S, H, D, dtype=dt, mask=("random", 0.05), bias2_sigma=None, seed=3)
    d = to_dev(inp)
    bufs = {n: torch.empty((B, S, R, H, D), dtype=d["q"].dtype, device="cuda") for n in ("q", "k", "v")}
    for n, buf in bufs.items():
        buf.transpose(1, 2).copy_(d[n])
        buf.requires_grad_(True)
    views = {n: bufs[n].transpose(1, 2) for n in bufs}
    assert all(readable_in_place(v) for v in views.values())
    out = evoformer_attention(views["q"], views["k"], views["v"], [d["bias1"]])
    out.backward(d["do"])

    packed = {n: d[n].clone().requires_grad_(True) for n in ("q", "k", "v")}
    out_p = evoformer_attention(packed["q"], packed["k"], packed["v"], [d["bias1"]])
    out_p.backward(d["do"])
    assert torch.equal(out, out_p)
    for n in ("q", "k", "v"):
        g_view = bufs[n].grad.transpose(1, 2)
        assert torch.equal(g_view, packed[n].grad), n


def test_slots_of_one_projection_buffer():
    """q, k, v read in place as the slots of one [B, N, L, 3, H, D] buffer (inputs may share
    a buffer; only outputs are checked against inputs)."""
    B, N, L, H, D = 1, 3, 200, 2, 32
    inp = make_inputs(B, N, L, H, D, dtype="bf16", mask=("random", 0.05), bias2_sigma=1.0, seed=12)
    d = to_dev(inp)
    out_p, lse_p = E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"])
    ref = E.evo_attn_bwd_ex(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out_p, lse_p, d["do"])
    qkv = torch.stack([d["q"], d["k"], d["v"]], dim=3)  # [B, N, L, 3, H, D]
    q, k, v = qkv.unbind(3)
    out, lse = E.evo_attn_fwd_strided(q, k, v, d["bias1"], d["bias2"])
    g = E.evo_attn_bwd_strided(q, k, v, d["bias1"], d["bias2"], out, lse, d["do"], want_dbias1=True)
    assert E.evo_attn_device_status() == 0
    assert torch.equal(out, out_p) and torch.equal(lse, lse_p)
    for x, y in zip(g, ref):
        assert torch.equal(x, y)
