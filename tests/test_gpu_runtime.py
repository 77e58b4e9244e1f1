"""GPU tests of the runtime around the kernels: the bounded-wait timeout path and
where it reports (the fallback word, a caller's status word, a workspace's own
word), the host-buffer step entry point, CUDA-graph capture of a step, per-call
profiling events on the caller's stream, and calls with different options
running concurrently on two streams."""
import pytest
import torch

from memory_efficient_biased_gb300 import evo_attn as E
from memory_efficient_biased_gb300.workload import make_inputs
from tests.parity_util import run_bwd, run_fwd, to_dev

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    """A barrier that nothing signals: the kernel gives up after ~1 ms and
    reports EVO_ERR_DEVICE_TIMEOUT; the context stays usable."""
    assert E.evo_attn_device_status() == 0
    assert E.evo_attn_selftest_wait_timeout(1_000_000) == 0
    assert E.evo_attn_device_status() == 8
    assert E.evo_attn_device_status() == 0  # reading clears it
    inp = make_inputs(1, 2, 64, 2, 16, dtype="fp16", seed=1)
    out, _ = run_fwd(to_dev(inp))
    assert torch.isfinite(out.float()).all()


def test_timeout_lands_in_the_callers_status_word():
    """With a status word of its own, the timeout is reported there, not in the
    fallback word."""
    mine = torch.zeros(1, dtype=torch.int32, device="cuda")
    assert E.evo_attn_selftest_wait_timeout(1_000_000, status=mine) == 0
    torch.cuda.synchronize()
    assert int(mine.item()) == 8
    assert E.evo_attn_device_status() == 0


def test_workspace_status_word():
    """evo_attn_bwd_opts clears its workspace's status word with its first kernel and
    evo_attn_bwd_status reads it (a word left set by an earlier call reads as a timeout
    until the next call clears it)."""
    d = to_dev(_inputs())
    out, lse = E.evo_attn_fwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"])
    ws = torch.empty(E.evo_attn_bwd_workspace_bytes(tuple(d["q"].shape), torch.bfloat16, True),
                     dtype=torch.uint8, device="cuda")
    ws[:4].view(torch.int32).fill_(8)
    assert E.evo_attn_bwd_status(ws) == 8
    E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], workspace=ws)
    assert E.evo_attn_bwd_status(ws) == 0
    assert E.evo_attn_device_status() == 0


def test_two_streams_with_different_options():
    """Options are per call: a skipping forward and backward on one stream, the
    unskipped ones on another, at the same time, each give the results it gives alone."""
    from tests.test_tile_skip import masked_rows
    inp = masked_rows(make_inputs(1, 8, 700, 2, 32, dtype="bf16", mask=None, bias2_sigma=None, seed=5), ("tail", 400))
    d = to_dev(inp)

    def run(skip, stream):
        with torch.cuda.stream(stream):
            out, lse = E.evo_attn_fwd_opts(d["q"], d["k"], d["v"], d["bias1"], None, skip_masked_tiles=skip)
            g = E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], None, out, lse, d["do"],
                                    skip_masked_tiles=skip)
        return (out, lse) + g[:3]

    s0 = torch.cuda.current_stream()
    ref_skip, ref_plain = run(True, s0), run(False, s0)
    torch.cuda.synchronize()
    sa, sb = torch.cuda.Stream(), torch.cuda.Stream()
    for _ in range(3):
        got_skip, got_plain = run(True, sa), run(False, sb)
    torch.cuda.synchronize()
    assert E.evo_attn_device_status() == 0
    for x, y in zip(got_skip, ref_skip):
        assert torch.equal(x, y)
    for x, y in zip(got_plain, ref_plain):
        assert torch.equal(x, y)


def test_pair_bias_gradient_can_be_left_out():
    """EVO_OPT_NO_DBIAS2: the other gradients are the same bytes, no dbias2 is written."""
    d = to_dev(_inputs())
    out, lse = E.evo_attn_fwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"])
    full = E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"])
    part = E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], want_dbias2=False)
    torch.cuda.synchronize()
    assert part[4] is None and full[4] is not None
    for x, y in zip(part[:3], full[:3]):
        assert torch.equal(x, y)


def _inputs():
    return make_inputs(1, 6, 160, 2, 32, dtype="bf16", mask=("random", 0.05), seed=21)


def test_step_host_matches_device_path():
    inp = _inputs()
    d = to_dev(inp)
    out, lse = run_fwd(d)
    dq, dk, dv, db2 = run_bwd(d, out, lse)
    pin = {k: v.pin_memory() for k, v in inp.items()}
    h = {k: torch.empty_like(pin["q"]).pin_memory() for k in ("out", "dq", "dk", "dv")}
    hdb2 = torch.empty_like(pin["bias2"]).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    arena = torch.empty(E.evo_attn_step_host_arena_bytes(tuple(inp["q"].shape), torch.bfloat16, True, True),
                        dtype=torch.uint8, device="cuda")
    E.evo_attn_step_host(pin["q"], pin["k"], pin["v"], pin["bias1"], pin["bias2"], pin["do"], h["out"], hlse,
                         h["dq"], h["dk"], h["dv"], hdb2, arena)
    torch.cuda.synchronize()
    assert E.evo_attn_device_status() == 0
    assert torch.equal(h["out"], out.cpu()) and torch.equal(hlse, lse.cpu())
    assert torch.equal(h["dk"], dk.cpu()) and torch.equal(h["dv"], dv.cpu()) and torch.equal(hdb2, db2.cpu())
    assert torch.equal(h["dq"], dq.cpu())


def test_step_host_row_chunks_match_device_path():
    """Enough rows for the host-buffer step to run in two row chunks with a pair bias: each
    chunk's backward writes the partial planes of its own n-groups and one sum follows, in
    the order an unchunked call uses, so every output (dbias2 included) is the same bytes."""
    inp = make_inputs(1, 160, 128, 4, 16, dtype="bf16", mask=("random", 0.05), seed=23)
    d = to_dev(inp)
    out, lse = run_fwd(d)
    dq, dk, dv, db2 = run_bwd(d, out, lse)
    pin = {k: v.pin_memory() for k, v in inp.items()}
    h = {k: torch.empty_like(pin["q"]).pin_memory() for k in ("out", "dq", "dk", "dv")}
    hdb2 = torch.empty_like(pin["bias2"]).pin_memory()
    hlse = torch.empty(lse.shape, dtype=torch.float32).pin_memory()
    arena = torch.empty(E.evo_attn_step_host_arena_bytes(tuple(inp["q"].shape), torch.bfloat16, True, True),
                        dtype=torch.uint8, device="cuda")
    for _ in range(2):  # the second call reuses the arena
        E.evo_attn_step_host(pin["q"], pin["k"], pin["v"], pin["bias1"], pin["bias2"], pin["do"], h["out"], hlse,
                             h["dq"], h["dk"], h["dv"], hdb2, arena)
        torch.cuda.synchronize()
        assert E.evo_attn_device_status() == 0
        assert torch.equal(h["out"], out.cpu()) and torch.equal(hlse, lse.cpu())
        assert torch.equal(h["dq"], dq.cpu()) and torch.equal(h["dk"], dk.cpu()) and torch.equal(h["dv"], dv.cpu())
        assert torch.equal(hdb2, db2.cpu())


def test_cuda_graph_capture_replays_identically():
    inp = _inputs()
    d = to_dev(inp)
    out, lse = run_fwd(d)
    ref = [t.clone() for t in run_bwd(d, out, lse)]
    bufs = {"out": torch.empty_like(d["q"]), "lse": torch.empty_like(lse),
            "dq": torch.empty_like(d["q"]), "dk": torch.empty_like(d["q"]), "dv": torch.empty_like(d["q"]),
            "db2": torch.empty_like(d["bias2"]),
            "ws": torch.empty(E.evo_attn_bwd_workspace_bytes(tuple(d["q"].shape), torch.bfloat16, True),
                              dtype=torch.uint8, device="cuda")}

    def step():
        E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out=bufs["out"], lse=bufs["lse"])
        E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], bufs["out"], bufs["lse"], d["do"],
                       dq=bufs["dq"], dk=bufs["dk"], dv=bufs["dv"], dbias2=bufs["db2"], workspace=bufs["ws"])

    step()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert E.evo_attn_device_status() == 0
    assert torch.equal(bufs["out"], out) and torch.equal(bufs["lse"], lse)
    assert torch.equal(bufs["dk"], ref[1]) and torch.equal(bufs["dv"], ref[2]) and torch.equal(bufs["db2"], ref[3])


def test_profile_events_and_side_stream():
    inp = _inputs()
    d = to_dev(inp)
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(8)]
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        out, lse = E.evo_attn_fwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], stream=s, events=evs)
        E.evo_attn_bwd_opts(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], stream=s, events=evs)
    s.synchronize()
    assert E.evo_attn_device_status() == 0
    ms = [evs[i].elapsed_time(evs[i + 1]) for i in (0, 2, 3, 4, 5, 6)]
    assert all(m >= 0.0 for m in ms) and ms[0] > 0.0 and ms[2] > 0.0


def test_call_from_a_fresh_thread():
    """A thread whose first CUDA call is the library's (as on a framework's autograd
    worker thread): the tensor maps still encode, the results match."""
    import threading
    inp = _inputs()
    d = to_dev(inp)
    out, lse = run_fwd(d)
    ref = [t.clone() for t in run_bwd(d, out, lse)]
    o2, l2 = torch.empty_like(out), torch.empty_like(lse)
    got, err = {}, []

    def work():
        try:
            E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out=o2, lse=l2)
            got["bwd"] = E.evo_attn_bwd_ex(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], o2, l2, d["do"])
        except Exception as e:  # surfaced below
            err.append(e)

    t = threading.Thread(target=work)
    t.start()
    t.join()
    assert not err, err
    torch.cuda.synchronize()
    assert E.evo_attn_device_status() == 0
    assert torch.equal(o2, out) and torch.equal(l2, lse)
    dq, dk, dv, db1, db2 = got["bwd"]
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2]) and torch.equal(db2, ref[3])
    assert torch.equal(dq, ref[0])
