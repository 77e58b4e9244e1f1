"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
binding and compare with the fp64 oracle on the same seeded inputs.

Tolerances (fixed by the method's acceptance bar): forward max|O - O*| /
max|O*| <= 5e-3 (fp16) or 2e-2 (bf16); gradients ||g - g*||_2 / ||g*||_2 <=
2e-2 (fp16) or 4e-2 (bf16).
"""
import numpy as np
import torch

from memory_efficient_biased_gb300 import evo_attn as E

FWD_TOL = {torch.float16: 5e-3, torch.bfloat16: 2e-2}
GRAD_TOL = {torch.float16: 2e-2, torch.bfloat16: 4e-2}


def to_dev(inp):
    return {k: (None if v is None else v.cuda()) for k, v in inp.items()}


def np64(t):
    return None if t is None else t.detach().cpu().double().numpy()


def fwd_rel_err(o, o_ref):
    o = np.asarray(o, dtype=np.float64)
    scale = np.max(np.abs(o_ref))
    return float(np.max(np.abs(o - o_ref)) / max(scale, 1e-30))


def rel_l2(g, g_ref):
    g = np.asarray(g, dtype=np.float64)
    den = np.linalg.norm(g_ref)
    return float(np.linalg.norm(g - g_ref) / max(den, 1e-30))


def lse_err(lse, lse_ref):
    lse = np.asarray(lse, dtype=np.float64)
    fin = np.isfinite(lse_ref)
    assert np.array_equal(np.isneginf(lse), np.isneginf(lse_ref)), "-inf rows differ"
    if not fin.any():
        return 0.0
    return float(np.max(np.abs(lse[fin] - lse_ref[fin]) / np.maximum(1.0, np.abs(lse_ref[fin]))))


def run_fwd(d):
    out, lse = E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"])
    assert E.evo_attn_device_status() == 0
    return out, lse


def run_bwd(d, out, lse):
    dq, dk, dv, db2 = E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"])
    assert E.evo_attn_device_status() == 0
    return dq, dk, dv, db2
