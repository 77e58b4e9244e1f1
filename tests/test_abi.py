"""The C-ABI library loads, exports every symbol include/evo_attn.h declares, and
its host-side validation answers before anything reaches a GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from memory_efficient_biased_gb300 import evo_attn as E

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="session")
def lib():
    from memory_efficient_biased_gb300 import build
    build.build()
    return E.load()


def declared_symbols():
    names = set()
    inc = os.path.join(ROOT, "include")
    for f in os.listdir(inc):
        if f.endswith(".h"):
            src = open(os.path.join(inc, f)).read()
            names |= set(re.findall(r"EVO_API\s+[\w\s\*]+?\b(evo_\w+)\s*\(", src))
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert {"evo_attn_fwd", "evo_attn_bwd", "evo_attn_bwd_workspace_bytes"} <= names
    for n in names:
        assert hasattr(lib, n), n
    assert set(E.EXPORTED) == names


def test_abi_version_and_strings(lib):
    assert lib.evo_attn_abi_version() == 4
    for code in range(13):
        s = lib.evo_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.evo_status_string(99).decode() == "unknown status"


def shape(B=1, N=2, L=64, H=2, D=32):
    return E.EvoShape(B, N, L, H, D)


A = 1 << 20  # fake, well-aligned device addresses: validation never dereferences them


def fwd(lib, q=A, k=2 * A, v=3 * A, b1=None, b2=None, out=4 * A, lse=5 * A, s=None, dt=1):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.evo_attn_fwd(vp(q), vp(k), vp(v), vp(b1), vp(b2), vp(out), vp(lse), s or shape(), dt, None)


def test_fwd_validation(lib):
    assert fwd(lib, q=None) == 1
    assert fwd(lib, lse=None) == 1
    assert fwd(lib, dt=2) == 3
    for bad in (shape(D=12), shape(D=72), shape(D=0), shape(L=0), shape(L=40000), shape(B=0), shape(H=0)):
        assert fwd(lib, s=bad) == 2
    assert fwd(lib, q=A + 8) == 4          # 16-byte rule
    assert fwd(lib, lse=5 * A + 2) == 4    # 4-byte rule
    assert fwd(lib, b1=6 * A + 1) == 4     # 2-byte rule
    assert fwd(lib, b2=7 * A + 4) == 4
    assert fwd(lib, out=A) == 9            # output aliases q
    assert fwd(lib, lse=3 * A + 64) == 9   # lse inside v
    # valid arguments reach the device check; without a GPU that is a CUDA error, never a launch
    r = fwd(lib)
    assert r in (6, 7) or r == 0


def bwd(lib, ws=16 * A, ws_bytes=None, b2=None, db2=None, s=None, dt=1, **kw):
    s = s or shape()
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    p = dict(q=A, k=2 * A, v=3 * A, b1=None, out=4 * A, lse=5 * A, do=6 * A, dq=7 * A, dk=8 * A, dv=9 * A)
    p.update(kw)
    need = lib.evo_attn_bwd_workspace_bytes(s, dt, int(b2 is not None))
    return lib.evo_attn_bwd(vp(p["q"]), vp(p["k"]), vp(p["v"]), vp(p["b1"]), vp(b2), vp(p["out"]),
                            vp(p["lse"]), vp(p["do"]), vp(p["dq"]), vp(p["dk"]), vp(p["dv"]), vp(db2),
                            vp(ws), need if ws_bytes is None else ws_bytes, s, dt, None)


def test_bwd_validation(lib):
    assert bwd(lib, q=None) == 1
    assert bwd(lib, ws=None) == 1
    assert bwd(lib, b2=10 * A) == 10       # bias2 without dbias2
    assert bwd(lib, db2=10 * A) == 10      # dbias2 without bias2
    assert bwd(lib, s=shape(D=80)) == 2
    assert bwd(lib, ws=16 * A + 128) == 4  # 256-byte workspace rule
    assert bwd(lib, ws_bytes=16) == 5
    assert bwd(lib, dq=A) == 9             # dq aliases q
    assert bwd(lib, dk=7 * A) == 9         # dk aliases dq
    r = bwd(lib)
    assert r in (6, 7) or r == 0


def bwd_ex(lib, db1=None, b1=None, ws_bytes=None):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    s = shape()
    need = lib.evo_attn_bwd_workspace_bytes(s, 1, 2)
    return lib.evo_attn_bwd_ex(vp(A), vp(2 * A), vp(3 * A), vp(b1), None, vp(4 * A), vp(5 * A), vp(6 * A),
                               vp(7 * A), vp(8 * A), vp(9 * A), vp(db1), None, vp(16 * A),
                               need if ws_bytes is None else ws_bytes, s, 1, None)


def test_bwd_ex_validation(lib):
    assert bwd_ex(lib, db1=11 * A) == 10                 # dbias1 without bias1
    assert bwd_ex(lib, db1=11 * A + 1, b1=12 * A) == 4   # dbias1 must be 2-byte aligned
    assert bwd_ex(lib, db1=7 * A, b1=12 * A) == 9         # dbias1 aliases dq
    # the key-mask gradient needs its partials in the workspace
    assert bwd_ex(lib, db1=11 * A, b1=12 * A, ws_bytes=lib.evo_attn_bwd_workspace_bytes(shape(), 1, 0)) == 5
    r = bwd_ex(lib, db1=11 * A, b1=12 * A)
    assert r in (6, 7) or r == 0


def test_workspace_bytes(lib):
    s = shape(B=1, N=256, L=256, H=4, D=32)
    no_b2 = lib.evo_attn_bwd_workspace_bytes(s, 1, 0)
    with_b2 = lib.evo_attn_bwd_workspace_bytes(s, 1, 1)
    status = 256  # the call's own status word, first
    delta = 1 * 256 * 4 * 256 * 4
    # key-major backward (D <= 32, L <= 256): dQ stays in TMEM, no fp32 rows
    assert no_b2 == status + delta
    # EVO_WS_NO_DBIAS2 leaves the pair-bias partial planes out (the transposed copy stays)
    assert lib.evo_attn_bwd_workspace_bytes(s, 1, 1 | 4) == no_b2 + 1 * 4 * 256 * 256 * 2
    assert lib.evo_attn_bwd_workspace_bytes(s, 1, 8) == 0  # unknown flag
    # with a pair bias: its transposed bf16 copy plus a whole number of fp32 [B,H,L,L] partial planes
    extra = with_b2 - no_b2 - 1 * 4 * 256 * 256 * 2
    plane = 1 * 4 * 256 * 256 * 4
    assert extra % plane == 0 and 1 <= extra // plane <= 256
    # per-key-tile backward (D = 64, L = 384): delta, then L × DP fp32 dQ rows for each of
    # its CTAs (one per (b, h, n) slice here: 8 of them, at most 256) and the masked-tile
    # skip bits [B*N] u64, each part rounded up to 256 bytes
    big = shape(B=1, N=4, L=384, H=2, D=64)
    r256 = lambda x: (x + 255) // 256 * 256
    assert lib.evo_attn_bwd_workspace_bytes(big, 1, 0) == 256 + 4 * 2 * 384 * 4 + 8 * 384 * 64 * 4 + r256(4 * 8)
    # the dQ rows are capped at 256 CTAs however many slices there are
    many = shape(B=1, N=512, L=384, H=2, D=64)
    assert lib.evo_attn_bwd_workspace_bytes(many, 1, 0) == (256 + 512 * 2 * 384 * 4 + 256 * 384 * 64 * 4 +
                                                             r256(512 * 8))
    # EVO_WS_DBIAS1 adds the fp32 [B,N,H,2,L] key-mask gradient partials
    assert lib.evo_attn_bwd_workspace_bytes(s, 1, 2) - no_b2 == 1 * 256 * 4 * 2 * 256 * 4
    assert lib.evo_attn_bwd_workspace_bytes(shape(D=12), 1, 0) == 0
    assert lib.evo_attn_bwd_workspace_bytes(s, 7, 0) == 0


def packed_layout(s):
    hd = s.H * s.D
    st = E.EvoStrides(s.N * s.L * hd, s.L * hd, hd)
    return E.EvoLayout(*([st] * 8))


def transposed_strides(s):
    """[B,N,L,H,D] view of a [B,L,N,H,D] buffer."""
    hd = s.H * s.D
    return E.EvoStrides(s.N * s.L * hd, hd, s.N * hd)


def fwd_s(lib, lay, s=None, out=4 * A):
    vp = ctypes.c_void_p
    return lib.evo_attn_fwd_strided(vp(A), vp(2 * A), vp(3 * A), None, None, vp(out), vp(5 * A), s or shape(), 1,
                                    ctypes.byref(lay) if lay is not None else None, None)


def test_fwd_strided_validation(lib):
    s = shape()  # (1, 2, 64, 2, 32): H*D = 64
    reach = (6, 7, 0)  # valid arguments reach the device check
    assert fwd_s(lib, None) in reach
    assert fwd_s(lib, packed_layout(s)) in reach
    lay = packed_layout(s)
    lay.q = transposed_strides(s)
    assert fwd_s(lib, lay) in reach
    for bad in ((8192, 0, 64), (8192, 4096, 60), (8192, 4096, 32), (8192, 64, 64), (8192, -4096, 64),
                (8192, 4096, 1 << 36)):
        lay = packed_layout(s)
        lay.k = E.EvoStrides(*bad)
        assert fwd_s(lib, lay) == 12, bad  # EVO_ERR_BAD_LAYOUT
    # strides of extent-1 dimensions are ignored (B = 1 here)
    lay = packed_layout(s)
    lay.v = E.EvoStrides(3, 4096, 64)
    assert fwd_s(lib, lay) in reach
    # the output's span follows its strides: a padded out reaching into lse's range aliases
    lay = packed_layout(s)
    lay.out = E.EvoStrides(1 << 20, 1 << 19, 64)  # n = 1 starts 1 MiB after out, i.e. at lse
    assert fwd_s(lib, lay) == 9


def bwd_s(lib, lay, s, ws_bytes):
    vp = ctypes.c_void_p
    return lib.evo_attn_bwd_strided(vp(A), vp(2 * A), vp(3 * A), None, None, vp(4 * A), vp(5 * A), vp(6 * A),
                                    vp(7 * A), vp(8 * A), vp(9 * A), None, None, vp(16 * A), ws_bytes, s, 1,
                                    ctypes.byref(lay), None)


def test_bwd_strided_validation(lib):
    s = shape(B=2, N=2, L=64, H=2, D=32)
    per_batch = lib.evo_attn_bwd_workspace_bytes(shape(B=1, N=2, L=64, H=2, D=32), 1, 0)
    whole = lib.evo_attn_bwd_workspace_bytes(s, 1, 0)
    assert whole >= per_batch
    reach = (6, 7, 0)
    assert bwd_s(lib, packed_layout(s), s, whole) in reach
    assert bwd_s(lib, packed_layout(s), s, per_batch) == 5
    # a transposed dout with B = 2 cannot merge (b, n): the call runs batch by batch and
    # needs only one batch's workspace
    lay = packed_layout(s)
    lay.dout = transposed_strides(s)
    assert bwd_s(lib, lay, s, per_batch) in reach
    lay.dq = E.EvoStrides(8192, 4096, 40)  # rows overlap
    assert bwd_s(lib, lay, s, whole) == 12


def test_workspace_covers_batch_by_batch(lib):
    for B, N, L, H, D in ((2, 10, 128, 1, 64), (3, 7, 200, 2, 32), (4, 384, 64, 8, 32)):
        for flags in (0, 1, 3):
            one = lib.evo_attn_bwd_workspace_bytes(shape(1, N, L, H, D), 1, flags)
            assert lib.evo_attn_bwd_workspace_bytes(shape(B, N, L, H, D), 1, flags) >= one


def opts(**kw):
    o = E.EvoOptions()
    o.size = ctypes.sizeof(E.EvoOptions)
    for k, v in kw.items():
        setattr(o, k, v)
    return o


def fwd_o(lib, o, b1=None):
    vp = ctypes.c_void_p
    return lib.evo_attn_fwd_opts(vp(A), vp(2 * A), vp(3 * A), None if b1 is None else vp(b1), None, vp(4 * A),
                                 vp(5 * A), shape(), 1, None, ctypes.byref(o) if o is not None else None, None)


def bwd_o(lib, o, b2=None, db2=None, ws_flags=None):
    vp = lambda x: None if x is None else ctypes.c_void_p(x)
    s = shape()
    flags = ws_flags if ws_flags is not None else int(b2 is not None)
    need = lib.evo_attn_bwd_workspace_bytes(s, 1, flags)
    return lib.evo_attn_bwd_opts(vp(A), vp(2 * A), vp(3 * A), None, vp(b2), vp(4 * A), vp(5 * A), vp(6 * A),
                                 vp(7 * A), vp(8 * A), vp(9 * A), None, vp(db2), vp(16 * A), need, s, 1, None,
                                 ctypes.byref(o) if o is not None else None, None)


def test_options_validation(lib):
    """evo_options_t is checked before anything else: its size, its flags, its events."""
    reach = (6, 7, 0)  # valid arguments reach the device check
    assert fwd_o(lib, None) in reach
    assert fwd_o(lib, opts()) in reach
    assert fwd_o(lib, opts(flags=1, skip_threshold=-1e4), b1=11 * A) in reach
    small = opts()
    small.size = 8
    assert fwd_o(lib, small) == 10
    assert fwd_o(lib, opts(flags=4)) == 10            # unknown flag
    assert fwd_o(lib, opts(flags=2)) == 10            # no dbias2: a backward option
    assert fwd_o(lib, opts(num_events=2)) == 10       # events missing
    assert fwd_o(lib, opts(num_events=-1)) == 10
    assert bwd_o(lib, opts()) in reach
    # without EVO_OPT_NO_DBIAS2 a pair bias needs dbias2; with it, dbias2 must be NULL
    assert bwd_o(lib, opts(), b2=10 * A) == 10
    assert bwd_o(lib, opts(flags=2), b2=10 * A, ws_flags=1 | 4) in reach
    assert bwd_o(lib, opts(flags=2), b2=10 * A, db2=12 * A) == 10
    assert bwd_o(lib, opts(), b2=10 * A, db2=12 * A) in reach
    # without the pair-bias gradient the smaller workspace suffices; with it, it does not
    assert bwd_o(lib, opts(), b2=10 * A, db2=12 * A, ws_flags=1 | 4) == 5


def test_bwd_status_validation(lib):
    assert lib.evo_attn_bwd_status(None, None) == 1
    assert lib.evo_attn_bwd_status(ctypes.c_void_p(A + 128), None) == 4


def test_no_process_wide_settings(lib):
    """The library has no setters: what a call does comes from its arguments."""
    for name in ("evo_attn_set_wait_limit_ns", "evo_attn_set_masked_tile_skip", "evo_attn_profile_events"):
        assert not hasattr(lib, name), name
