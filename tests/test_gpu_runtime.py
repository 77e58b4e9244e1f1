"""GPU tests of the runtime around the kernels: the bounded-wait timeout path,
the host-buffer step entry point, CUDA-graph capture of a step, the profiling
hook and the caller's stream."""
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
    assert (h["dq"].float() - dq.cpu().float()).abs().max() <= 1e-2 * dq.float().abs().max().cpu()


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
    E.evo_attn_profile_events(evs)
    try:
        with torch.cuda.stream(s):
            out, lse = E.evo_attn_fwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], stream=s)
            E.evo_attn_bwd(d["q"], d["k"], d["v"], d["bias1"], d["bias2"], out, lse, d["do"], stream=s)
    finally:
        E.evo_attn_profile_events(None)
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
