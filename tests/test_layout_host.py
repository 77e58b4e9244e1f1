"""Host-side layout logic of the strided entry points, on CPU tensors (no GPU).

What the binding passes as evo_layout_t for a tensor, and which views the
autograd wrapper reads in place rather than copying: packed (H, D), a 16-byte
aligned start, B/N/L strides that are positive multiples of 8 and rows that do
not overlap — the rules the C library checks (test_abi.py covers those).
"""
import torch

from memory_efficient_biased_gb300 import evo_attn as E
from memory_efficient_biased_gb300.autograd import readable_in_place


def msa(B=1, S=6, R=40, H=4, D=16):
    """A [B, N_seq, N_res, H, D] buffer, as the MSA stack holds it."""
    return torch.zeros((B, S, R, H, D), dtype=torch.bfloat16)


def test_packed_and_transposed_views_are_read_in_place():
    x = msa()
    assert readable_in_place(x)
    t = x.transpose(1, 2)  # column-wise attention: attend along N_seq
    assert not t.is_contiguous() and readable_in_place(t)
    assert E.row_strided(t)


def test_layout_of_reports_the_tensors_own_strides():
    x = msa(B=2, S=6, R=40, H=4, D=16)
    t = x.transpose(1, 2)  # logical [2, 40, 6, 4, 16]
    lay = E.layout_of(q=t, k=t, v=t, out=None)
    assert (lay.q.b, lay.q.n, lay.q.l) == (6 * 40 * 64, 64, 40 * 64)
    # tensors not given are packed in the shape of the first one
    B, N, L, H, D = t.shape
    assert (lay.out.b, lay.out.n, lay.out.l) == (N * L * H * D, L * H * D, H * D)
    assert (lay.dv.b, lay.dv.n, lay.dv.l) == (N * L * H * D, L * H * D, H * D)


def test_views_that_must_be_copied():
    x = msa(H=4, D=16)
    # H and D not packed: a buffer stored [.., D, H], viewed as [.., H, D]
    hd = x.transpose(3, 4).contiguous().transpose(3, 4)
    assert not E.row_strided(hd) and not readable_in_place(hd)
    # broadcast over n (stride 0): rows overlap
    y = torch.zeros((1, 1, 40, 4, 16), dtype=torch.bfloat16).expand(1, 6, 40, 4, 16)
    assert E.row_strided(y) and not readable_in_place(y)
    # a start that is not 16-byte aligned (one element into the buffer)
    z = torch.zeros(1 + 6 * 40 * 64, dtype=torch.bfloat16)[1:].view(1, 6, 40, 4, 16)
    assert not readable_in_place(z)
    # a token stride that is not a multiple of 8 elements
    w = torch.as_strided(torch.zeros(6 * 40 * 68, dtype=torch.bfloat16), (1, 6, 40, 4, 16),
                         (6 * 40 * 68, 40 * 68, 68, 16, 1))
    assert E.row_strided(w) and not readable_in_place(w)


def test_padded_rows_are_read_in_place():
    buf = torch.zeros((1, 6, 43, 4, 16), dtype=torch.bfloat16)
    v = buf[:, :, :40]
    assert not v.is_contiguous() and readable_in_place(v)
    lay = E.layout_of(q=v)
    assert (lay.q.n, lay.q.l) == (43 * 64, 64)


def test_extent_one_dimensions_ignore_their_strides():
    x = torch.zeros((1, 1, 40, 4, 16), dtype=torch.bfloat16)
    # a size-1 dimension may carry any stride
    y = torch.as_strided(x, x.shape, (3, 5, 64, 16, 1))
    assert readable_in_place(y)


def test_slots_of_a_packed_projection_are_read_in_place():
    """q, k, v as the three slots of one [B, N, L, 3, H, D] projection output: token
    stride 3·H·D, (H, D) packed."""
    qkv = torch.zeros((1, 6, 40, 3, 4, 16), dtype=torch.bfloat16)
    q, k, v = qkv.unbind(3)
    for t in (q, k, v):
        assert not t.is_contiguous() and readable_in_place(t)
    lay = E.layout_of(q=q, k=k, v=v)
    assert (lay.k.n, lay.k.l) == (40 * 3 * 64, 3 * 64)
