"""Plain fp64 CPU oracle for memory-efficient biased Evoformer attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path may import this module:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, constant
or helper with the CUDA library; both sides only consume the same seeded
inputs (``memory_efficient_biased_gb300.workload``).

What it computes (source: the web page "DeepSpeed4Science 技术指南：AI4Science
大模型长序列训练与 Evoformer 内存高效注意力内核实战", cited below as
[DS4Sci guide]):

* §3.5 — the reference test's ``attention_reference``: scores Q·Kᵀ times the
  scale factor, plus the bias terms, softmax over keys, times V.
* §3.6 — tensor layouts: Q, K, V are ``[B, N, L, H, D]``; the key mask
  ``bias1`` is ``[B, N, 1, 1, L]``; the pair bias ``bias2`` is
  ``[B, 1, H, L, L]`` and is shared by all N rows.
* §3.7 — the forward keeps a per-row log-sum-exp (lse) in fp32; the backward
  first forms ``delta`` and then dQ, dK, dV and the gradients of both biases.

Readings of points the page leaves open:

* scale s = D^-1/2 with D the true head dimension (the page only says
  "scale factor"; padding D to a multiple of 32 adds zeros and cannot change
  the scale);
* lse is the natural log, laid out ``[B, N, H, L]``;
* delta_i = sum_d dO_id * O_id (the page's "lse 先算出 delta" is garbled;
  the plain reading is the usual softmax-backward row term);
* a row in which every score is -inf (an fp16 -1e9 mask over all keys) has
  an empty softmax: P = 0, O = 0, lse = -inf and all its gradients 0.

Everything is fp64 and exact up to rounding order: inputs are the
dtype-rounded tensors upcast exactly.  The only library primitive used is
matrix multiplication (numpy ``@``) and ``exp``/``log``.

Pins: tests/test_oracle_pins.py (brute force, finite differences, torch's
scaled_dot_product_attention with an additive float mask, closed forms and
invariants).  Every function below is pinned.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "scale_of",
    "slice_forward",
    "slice_backward",
    "forward",
    "backward",
    "forward_slice_sample",
    "backward_slice_sample",
    "dbias2_sample",
]


def scale_of(D: int) -> float:
    """s = D^-1/2 ([DS4Sci guide] §3.5 "乘缩放因子"; D is the true head dim)."""
    return 1.0 / math.sqrt(D)


def _as64(x):
    if x is None:
        return None
    return np.asarray(x, dtype=np.float64)


# ---------------------------------------------------------------------------
# One attention slice (fixed b, n, h): L queries, L keys, D features.
# ---------------------------------------------------------------------------

def slice_forward(q, k, v, bias, s):
    """Forward of one slice.

    q, k, v: [L, D]; bias: [L, L] (query i, key j), the sum of the key mask and
    the pair bias for this slice ([DS4Sci guide] §3.5: scale, add bias,
    softmax, times V).  Returns (o [L, D], lse [L], p [L, L]).
    """
    q, k, v, bias = _as64(q), _as64(k), _as64(v), _as64(bias)
    x = s * (q @ k.T) + bias                      # biased, scaled scores
    m = np.max(x, axis=1)                         # row max
    empty = ~np.isfinite(m)                       # every key is -inf
    m_safe = np.where(empty, 0.0, m)
    e = np.exp(x - m_safe[:, None])               # exp(-inf) = 0 for masked keys
    l = np.sum(e, axis=1)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m_safe + np.log(np.where(empty, 1.0, l)))
    p = np.where(empty[:, None], 0.0, e / np.where(empty, 1.0, l)[:, None])
    o = p @ v
    return o, lse, p


def slice_backward(q, k, v, bias, do, s):
    """Analytic gradient of <O, dO> for one slice.

    Returns dict with dq, dk, dv ([L, D]), ds ([L, L], the gradient with
    respect to the biased score, i.e. the bias gradient before any
    broadcast reduction), delta [L], o, lse.
    [DS4Sci guide] §3.7: delta first, then dQ/dK/dV and the bias gradients.
    """
    q, k, v, bias, do = _as64(q), _as64(k), _as64(v), _as64(bias), _as64(do)
    o, lse, p = slice_forward(q, k, v, bias, s)
    dv = p.T @ do                                  # dV_j = sum_i P_ij dO_i
    dp = do @ v.T                                  # dP_ij = dO_i . V_j
    delta = np.sum(do * o, axis=1)                 # delta_i = dO_i . O_i
    ds = p * (dp - delta[:, None])                 # softmax backward
    dq = s * (ds @ k)                              # d(s Q K^T)/dQ
    dk = s * (ds.T @ q)
    return {"dq": dq, "dk": dk, "dv": dv, "ds": ds, "delta": delta,
            "o": o, "lse": lse}


def _slice_bias(bias1, bias2, b, n, h, L):
    """Bias for slice (b, n, h): key mask [B,N,1,1,L] broadcast over queries
    plus pair bias [B,1,H,L,L] shared across n ([DS4Sci guide] §3.6-3.7)."""
    out = np.zeros((L, L), dtype=np.float64)
    if bias1 is not None:
        out = out + bias1[b, n, 0, 0, :][None, :]
    if bias2 is not None:
        out = out + bias2[b, 0, h, :, :]
    return out


# ---------------------------------------------------------------------------
# Full 5-D tensors [B, N, L, H, D].
# ---------------------------------------------------------------------------

def forward(q, k, v, bias1=None, bias2=None):
    """O = softmax(Q Kᵀ D^-1/2 + bias1 + bias2) V over [B, N, L, H, D].

    Returns (o [B,N,L,H,D] fp64, lse [B,N,H,L] fp64).
    """
    q, k, v = _as64(q), _as64(k), _as64(v)
    bias1, bias2 = _as64(bias1), _as64(bias2)
    B, N, L, H, D = q.shape
    s = scale_of(D)
    o = np.empty_like(q)
    lse = np.empty((B, N, H, L), dtype=np.float64)
    for b in range(B):
        for n in range(N):
            for h in range(H):
                bias = _slice_bias(bias1, bias2, b, n, h, L)
                o_s, lse_s, _ = slice_forward(q[b, n, :, h, :], k[b, n, :, h, :],
                                              v[b, n, :, h, :], bias, s)
                o[b, n, :, h, :] = o_s
                lse[b, n, h, :] = lse_s
    return o, lse


def backward(q, k, v, bias1, bias2, do):
    """Gradients of <O, dO>: dq, dk, dv [B,N,L,H,D]; dbias1 [B,N,1,1,L]
    (sum of dS over h and i); dbias2 [B,1,H,L,L] (sum of dS over n);
    delta [B,N,H,L].  [DS4Sci guide] §3.7 (both bias gradients)."""
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    bias1, bias2 = _as64(bias1), _as64(bias2)
    B, N, L, H, D = q.shape
    s = scale_of(D)
    dq = np.empty_like(q)
    dk = np.empty_like(q)
    dv = np.empty_like(q)
    delta = np.empty((B, N, H, L), dtype=np.float64)
    dbias1 = np.zeros((B, N, 1, 1, L), dtype=np.float64)
    dbias2 = np.zeros((B, 1, H, L, L), dtype=np.float64)
    for b in range(B):
        for n in range(N):
            for h in range(H):
                bias = _slice_bias(bias1, bias2, b, n, h, L)
                g = slice_backward(q[b, n, :, h, :], k[b, n, :, h, :],
                                   v[b, n, :, h, :], bias, do[b, n, :, h, :], s)
                dq[b, n, :, h, :] = g["dq"]
                dk[b, n, :, h, :] = g["dk"]
                dv[b, n, :, h, :] = g["dv"]
                delta[b, n, h, :] = g["delta"]
                dbias1[b, n, 0, 0, :] += g["ds"].sum(axis=0)
                dbias2[b, 0, h, :, :] += g["ds"]
    return {"dq": dq, "dk": dk, "dv": dv, "dbias1": dbias1,
            "dbias2": dbias2, "delta": delta}


# ---------------------------------------------------------------------------
# Sampled outputs at full size (the oracle computes them one by one).
# ---------------------------------------------------------------------------

def forward_slice_sample(q, k, v, bias1, bias2, b, n, h):
    """(o [L, D], lse [L]) of one slice of a full-size problem."""
    L, D = q.shape[2], q.shape[4]
    bias = _slice_bias(_as64(bias1), _as64(bias2), b, n, h, L)
    o, lse, _ = slice_forward(q[b, n, :, h, :], k[b, n, :, h, :],
                              v[b, n, :, h, :], bias, scale_of(D))
    return o, lse


def backward_slice_sample(q, k, v, bias1, bias2, do, b, n, h):
    """dq, dk, dv ([L, D]) and ds ([L, L]) of one slice of a full-size problem."""
    L, D = q.shape[2], q.shape[4]
    bias = _slice_bias(_as64(bias1), _as64(bias2), b, n, h, L)
    return slice_backward(q[b, n, :, h, :], k[b, n, :, h, :], v[b, n, :, h, :],
                          bias, do[b, n, :, h, :], scale_of(D))


def dbias2_sample(q, k, v, bias1, bias2, do, b, h, rows):
    """dbias2[b, 0, h, i, :] for each i in ``rows``: sum over all n of the
    score gradient of row i.  Each term needs only row i of P, so the cost is
    N * |rows| * L * D instead of N * L^2 * D."""
    q64, k64, v64, do64 = _as64(q), _as64(k), _as64(v), _as64(do)
    b1, b2 = _as64(bias1), _as64(bias2)
    N, L, D = q.shape[1], q.shape[2], q.shape[4]
    s = scale_of(D)
    rows = np.asarray(rows)
    out = np.zeros((len(rows), L), dtype=np.float64)
    for n in range(N):
        kk = k64[b, n, :, h, :]
        vv = v64[b, n, :, h, :]
        qi = q64[b, n, rows, h, :]
        doi = do64[b, n, rows, h, :]
        bias = np.zeros((len(rows), L))
        if b1 is not None:
            bias = bias + b1[b, n, 0, 0, :][None, :]
        if b2 is not None:
            bias = bias + b2[b, 0, h, rows, :]
        x = s * (qi @ kk.T) + bias
        m = np.max(x, axis=1)
        empty = ~np.isfinite(m)
        m_safe = np.where(empty, 0.0, m)
        e = np.exp(x - m_safe[:, None])
        l = np.where(empty, 1.0, e.sum(axis=1))
        p = np.where(empty[:, None], 0.0, e / l[:, None])
        o = p @ vv
        dp = doi @ vv.T
        delta = np.sum(doi * o, axis=1)
        out += p * (dp - delta[:, None])
    return out

