"""The MLP backward's two schedules of dX = sum_i dU_i A_i^T, dA = X^T dU and dB = Y^T G:
one after another on the caller's stream, or side by side on disjoint CTA pairs through
two side streams (the overlap of the dX reduction with the weight-gradient GEMMs).
Every output tile runs the same K-loop in both, so the results are bitwise identical;
the oracle tolerance is checked by the backward parity tests."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import GRAD_REL_FRO, f64, mp, rel_fro, run_mlp_bwd, run_mlp_fwd, status_tensor

pytestmark = pytest.mark.gpu


def _bwd(dev, dZ, t, mode):
    old = os.environ.get("MPTP_BWD_SCHEDULE")
    os.environ["MPTP_BWD_SCHEDULE"] = mode
    try:
        return run_mlp_bwd(dev, dZ, t)
    finally:
        if old is None:
            os.environ.pop("MPTP_BWD_SCHEDULE", None)
        else:
            os.environ["MPTP_BWD_SCHEDULE"] = old


@pytest.mark.parametrize("T,h,f,t", [
    (300, 128, 512, 2),          # few tiles: each GEMM gets as many pairs as it has units
    (1000, 256, 1024, 4),        # ragged T
    (4096, 3072, 12288, 8),      # the 8.3B layer
])
def test_overlap_bitwise_equals_serial(T, h, f, t):
    inp = synth.mlp_inputs(T, h, f, seed=9000 + T)
    dev = run_mlp_fwd(inp, t)
    a = _bwd(dev, inp["dZ"], t, "serial")
    b = _bwd(dev, inp["dZ"], t, "overlap")
    for k in ("dX", "dA", "dB", "dU"):
        assert torch.equal(a[k], b[k]), k


def test_overlap_matches_oracle():
    T, h, f, t = 384, 192, 768, 3
    inp = synth.mlp_inputs(T, h, f, seed=9100)
    dev = run_mlp_fwd(inp, t)
    g = _bwd(dev, inp["dZ"], t, "overlap")
    ref = oracle.mlp_bwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), f64(inp["dZ"]))
    errs = {k: rel_fro(f64(g[k].cpu()), ref[k]) for k in ("dX", "dA", "dB")}
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs


def test_overlap_on_side_stream_and_in_graph():
    # The fork/join keeps the caller's stream ordered: a backward enqueued on a non-default
    # stream, and one captured into a CUDA graph and replayed, give the eager result.
    m = mp()
    T, h, f, t = 512, 256, 1024, 2
    inp = synth.mlp_inputs(T, h, f, seed=9200)
    dev = run_mlp_fwd(inp, t)
    want = _bwd(dev, inp["dZ"], t, "overlap")   # also creates the side streams outside any capture
    dZ = inp["dZ"].cuda()
    out = {k: torch.empty_like(v) for k, v in want.items()}
    st = status_tensor()
    s = torch.cuda.Stream()
    old = os.environ.get("MPTP_BWD_SCHEDULE")
    os.environ["MPTP_BWD_SCHEDULE"] = "overlap"
    try:
        with torch.cuda.stream(s):
            m.mp_mlp_bwd(dev["X"], dev["A"], dev["B"], dev["U"], dev["Y"], dZ, out["dX"], out["dA"], out["dB"],
                         out["dU"], t=t, d_status=st)
        torch.cuda.synchronize()
        for k in out:
            assert torch.equal(out[k], want[k]), k
        for v in out.values():
            v.zero_()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            m.mp_mlp_bwd(dev["X"], dev["A"], dev["B"], dev["U"], dev["Y"], dZ, out["dX"], out["dA"], out["dB"],
                         out["dU"], t=t, d_status=st)
        graph.replay()
        torch.cuda.synchronize()
    finally:
        if old is None:
            os.environ.pop("MPTP_BWD_SCHEDULE", None)
        else:
            os.environ["MPTP_BWD_SCHEDULE"] = old
    assert int(st.item()) == 0
    for k in out:
        assert torch.equal(out[k], want[k]), k
    assert np.isfinite(f64(out["dX"].cpu())).all()
