"""Device-side failure detection without a GPU fault: every mbarrier wait in the
kernels is bounded by a time budget (MPTP_WAIT_BUDGET_NS, read on each call).
With a budget of 0 ns the waits run out at once; the kernels must set
MP_DEV_TIMEOUT in the status word, drain their own copies and MMAs, return,
and leave the CUDA context usable (a normal call afterwards is exact)."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import Z_REL_FRO, f64, rel_fro

pytestmark = pytest.mark.gpu


def test_wait_budget_exhaustion_reports_timeout(monkeypatch):
    import tensor_transformer_layer_gb300 as mp
    T, h, f, t = 256, 4096, 512, 2        # long K-loop: the first accumulator takes many stages
    inp = synth.mlp_inputs(T, h, f, seed=6000, with_grad=False)
    X, A, B = (inp[k].cuda() for k in ("X", "A", "B"))
    Z = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("MPTP_WAIT_BUDGET_NS", "0")
    mp.mp_mlp_fwd(X, A, B, Z, Y, None, t=t, d_status=st)
    torch.cuda.synchronize()
    bits = int(st.item())
    assert bits & mp.MP_DEV_TIMEOUT, bits
    assert mp.mp_status_from_device(bits) == 6   # MP_ERR_TIMEOUT
    monkeypatch.delenv("MPTP_WAIT_BUDGET_NS")
    # The context is still usable and a normal call is correct.
    st.zero_()
    mp.mp_mlp_fwd(X, A, B, Z, Y, None, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, _, Zr = oracle.mlp_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]))
    assert rel_fro(f64(Z), Zr) <= Z_REL_FRO


def test_split_kernel_wait_budget_exhaustion(monkeypatch):
    # T = 256, h = 512, f = 4096: the row-parallel GEMM (N = h = 512, 64 K blocks) runs on the
    # split-K kernel, two CTA pairs a tile; with a zero budget its waits (pipeline, accumulator and
    # the cross-CTA exchange) run out, it reports MP_DEV_TIMEOUT and returns.
    import tensor_transformer_layer_gb300 as mp
    T, h, f, t = 256, 512, 4096, 2
    inp = synth.mlp_inputs(T, h, f, seed=6100, with_grad=False)
    X, A, B = (inp[k].cuda() for k in ("X", "A", "B"))
    Z = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("MPTP_WAIT_BUDGET_NS", "0")
    mp.mp_mlp_fwd(X, A, B, Z, Y, None, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & mp.MP_DEV_TIMEOUT
    monkeypatch.delenv("MPTP_WAIT_BUDGET_NS")
    st.zero_()
    mp.mp_mlp_fwd(X, A, B, Z, Y, None, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, _, Zr = oracle.mlp_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]))
    assert rel_fro(f64(Z), Zr) <= Z_REL_FRO
