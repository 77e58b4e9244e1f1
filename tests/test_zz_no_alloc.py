"""The allocation-free backward (evo_attn_bwd_noalloc), for callers that cannot
allocate device memory: it must give what evo_attn_bwd gives, through the C
ABI, on two calls in a row (the second one runs on the scratch the first one
left behind).  This file is collected last on purpose, so that a failure here
does not stop a `-x` run before the other tests ran; it also passes on its
own in a fresh process."""
import ctypes

import numpy as np
import pytest
import torch

from memory_efficient_biased_gb300 import evo_attn as E
from memory_efficient_biased_gb300.workload import make_inputs
from oracle import evo_oracle as O
from tests.parity_util import GRAD_TOL, np64, rel_l2, to_dev


def test_rejects_problems_beyond_the_fixed_scratch():
    """A backward whose workspace exceeds 16 MiB is refused before any launch."""
    from memory_efficient_biased_gb300 import build
    build.build()
    lib = E.load()
    big = E.EvoShape(1, 256, 256, 4, 32)  # needs ~52 MB of workspace
    assert lib.evo_attn_bwd_workspace_bytes(big, 1, 1) > E.NOALLOC_SCRATCH_BYTES
    A = 1 << 20
    vp = lambda x: ctypes.c_void_p(x)
    st = lib.evo_attn_bwd_noalloc(vp(A), vp(2 * A), vp(3 * A), None, vp(4 * A), vp(5 * A), vp(6 * A), vp(7 * A),
                                  vp(8 * A), vp(9 * A), vp(10 * A), vp(11 * A), big, 1, None)
    assert st == 11  # EVO_ERR_SCRATCH_LIMIT
    assert "16 MiB" in lib.evo_status_string(11).decode()


@pytest.mark.gpu
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_noalloc_matches_workspace_backward_twice(dtype):
    inp = make_inputs(1, 8, 200, 2, 32, dtype=dtype, mask=("random", 0.05), seed=31)
    d = to_dev(inp)
    out, lse = E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"])
    ref = E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"])
    assert E.evo_attn_device_status() == 0
    tol = GRAD_TOL[d["q"].dtype]
    for _ in range(2):
        got = [torch.empty_like(d["q"]) for _ in range(3)] + [torch.empty_like(d["bias2"])]
        E.evo_attn_bwd_noalloc(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], *got)
        torch.cuda.synchronize()
        assert E.evo_attn_device_status() == 0
        # same kernels, same inputs, every gradient summed in a fixed order: identical bytes
        for x, y in zip(got, ref):
            assert torch.equal(x, y)
    # and both agree with the fp64 oracle
    a = {k: np64(v) for k, v in inp.items()}
    g = O.backward(a["q"], a["k"], a["v"], a["bias1"], a["bias2"], a["do"])
    for key, t in zip(("dq", "dk", "dv", "dbias2"), got):
        assert rel_l2(np64(t), g[key]) <= tol, key
