"""PyTorch autograd over the C ABI: ``evoformer_attention(q, k, v, biases)``.

The call form of the pages' ``DS4Sci_EvoformerAttention(Q, K, V, biases)``
(web page "DeepSpeed4Science 技术指南…" §3.6–§3.7): q, k, v are [B, N, L, H, D]
fp16/bf16 CUDA tensors, ``biases`` a list of at most two tensors — the key mask
[B, N, 1, 1, L] and the pair bias [B, 1, H, L, L], either may be None or left out.
The forward saves O and the fp32 log-sum-exp; the backward returns the gradients
of q, k, v and of whichever biases require them (§3.7: both bias gradients).
Every step runs in the library's sm_103a kernels; there is no fallback.

q, k, v and the incoming gradient are read in place when only their B, N, L
strides differ from a packed tensor's (for instance the transposed view that
column-wise MSA attention or triangle attention around the ending node works
on, §3.6); other layouts are made contiguous first.  O and the gradients are
returned packed in the shape of q.
"""
from typing import List, Optional

import torch

from . import evo_attn as E


def readable_in_place(t: torch.Tensor) -> bool:
    """True if the library can read ``t`` through its strides: packed (H, D), a
    16-byte aligned start, B/N/L strides that are positive multiples of 8 below 2^36 and
    rows that do not overlap (the rules of the C ABI's evo_layout_t)."""
    if t.dim() != 5 or not E.row_strided(t) or t.data_ptr() % 16:
        return False
    dims = sorted((t.stride(i), t.shape[i]) for i in range(3) if t.shape[i] > 1)
    need = t.shape[3] * t.shape[4]
    for stride, ext in dims:
        if stride % 8 or stride < need or stride >= 1 << 36:
            return False
        need = stride * ext
    return True


def _in_place_or_packed(t: torch.Tensor) -> torch.Tensor:
    return t if readable_in_place(t) else t.contiguous()


class EvoformerAttentionFunction(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, bias1, bias2):
        q, k, v = _in_place_or_packed(q), _in_place_or_packed(k), _in_place_or_packed(v)
        bias1 = None if bias1 is None else bias1.contiguous()
        bias2 = None if bias2 is None else bias2.contiguous()
        out, lse = E.evo_attn_fwd_strided(q, k, v, bias1, bias2)
        ctx.save_for_backward(q, k, v, bias1, bias2, out, lse)
        return out

    @staticmethod
    def backward(ctx, dout):
        q, k, v, bias1, bias2, out, lse = ctx.saved_tensors
        dout = _in_place_or_packed(dout)
        want_db1 = bias1 is not None and ctx.needs_input_grad[3]
        want_db2 = bias2 is not None and ctx.needs_input_grad[4]
        # the pair-bias gradient is computed only when the pair bias needs one
        dq, dk, dv, db1, db2 = E.evo_attn_bwd_opts(q, k, v, bias1, bias2, out, lse, dout, want_dbias1=want_db1,
                                                   want_dbias2=want_db2)
        return dq, dk, dv, db1, db2


def evoformer_attention(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor,
                        biases: Optional[List[Optional[torch.Tensor]]] = None) -> torch.Tensor:
    """softmax(q kᵀ D^-1/2 + bias1 + bias2) v over [B, N, L, H, D], differentiable."""
    biases = list(biases or [])
    if len(biases) > 2:
        raise ValueError("at most two biases: the key mask [B,N,1,1,L] and the pair bias [B,1,H,L,L]")
    biases += [None] * (2 - len(biases))
    return EvoformerAttentionFunction.apply(q, k, v, biases[0], biases[1])


# The pages' name for the same call.
DS4Sci_EvoformerAttention = evoformer_attention
