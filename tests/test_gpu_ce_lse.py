"""GPU parity of the exported per-token log-sum-exp (mp_vocab_ce_lse) and of the
cross-entropy backward that takes it (mp_vocab_ce_bwd_lse), against the float64 oracle:
lse[r] = log sum_c exp(z[r, c]) over the valid vocabulary, and the plain derivative of
softmax cross-entropy for dX and dE."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import GRAD_REL_FRO, LOSS_ABS, f64, mp, rel_fro, status_tensor

pytestmark = pytest.mark.gpu


def _forward(inp, v_valid, t, expect_status=0):
    m = mp()
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    T, v_pad = X.shape[0], E.shape[0]
    ws = torch.empty(max(m.mp_vocab_ce_workspace_bytes(T, v_pad, t), 16), dtype=torch.uint8, device="cuda")
    loss = torch.empty(T, dtype=torch.float32, device="cuda")
    lse = torch.empty(T, dtype=torch.float32, device="cuda")
    st = status_tensor()
    m.mp_vocab_ce_lse(X, E, tgt, loss, lse, ws, v_valid=v_valid, t=t, d_status=st)
    loss_plain = torch.empty_like(loss)
    m.mp_vocab_ce(X, E, tgt, loss_plain, ws, v_valid=v_valid, t=t)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    return loss, lse, loss_plain


def _backward(inp, lse, dloss, v_valid, t, one_pass):
    m = mp()
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    T, h = X.shape
    v_pad = E.shape[0]
    size = (m.mp_vocab_ce_bwd_workspace_bytes_one_pass if one_pass else m.mp_vocab_ce_bwd_workspace_bytes)
    wsb = torch.empty(size(T, h, v_pad, t), dtype=torch.uint8, device="cuda")
    dX = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dE = torch.full((v_pad, h), 7.0, dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    m.mp_vocab_ce_bwd_lse(X, E, tgt, lse, dloss.cuda(), dX, dE, wsb, v_valid=v_valid, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return dX.cpu(), dE.cpu()


@pytest.mark.parametrize("T,h,v_pad,v_valid,t", [
    (300, 128, 2048, 2000, 2),     # padding columns excluded, ragged T
    (257, 192, 2048, 1500, 8),     # the last shards hold only padding
    (1, 64, 256, 256, 1),          # one token, no padding
])
def test_lse_matches_oracle(T, h, v_pad, v_valid, t):
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=9000 + T)
    loss, lse, loss_plain = _forward(inp, v_valid, t)
    assert torch.equal(loss, loss_plain)   # the loss is the same computation
    want = oracle.ce_logsumexp(f64(inp["X"]), f64(inp["E"]), v_valid)
    assert float(np.max(np.abs(lse.cpu().numpy().astype(np.float64) - want))) <= LOSS_ABS


def test_lse_zero_embedding_closed_form():
    inp = synth.ce_inputs(200, 128, 51200, 50257, seed=9100)
    inp["E"] = torch.zeros_like(inp["E"])
    _, lse, _ = _forward(inp, 50257, 8)
    assert float(torch.max(torch.abs(lse.cpu() - math.log(50257)))) <= 1e-4


def test_lse_invalid_target_is_nan():
    inp = synth.ce_inputs(64, 64, 512, 500, seed=9200)
    inp["target"][5] = 500      # a padding column: outside [0, v_valid)
    loss, lse, _ = _forward(inp, 500, 2, expect_status=2)
    assert math.isnan(float(lse[5])) and math.isnan(float(loss[5]))
    assert torch.isfinite(lse[torch.arange(64) != 5]).all()


@pytest.mark.parametrize("one_pass", [False, True])
@pytest.mark.parametrize("T,h,v_pad,v_valid,t", [
    (300, 128, 2048, 2000, 2),
    (257, 192, 2048, 1500, 8),
])
def test_bwd_from_lse_matches_oracle(T, h, v_pad, v_valid, t, one_pass):
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=9300 + T)
    g = torch.Generator().manual_seed(9400 + T)
    dl = torch.randn(T, generator=g, dtype=torch.float32)
    _, lse, _ = _forward(inp, v_valid, t)
    dX, dE = _backward(inp, lse, dl, v_valid, t, one_pass)
    ref = oracle.ce_bwd(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), dl.double().numpy(), v_valid)
    errs = {"dX": rel_fro(f64(dX), ref["dX"]), "dE": rel_fro(f64(dE), ref["dE"])}
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs
    assert torch.count_nonzero(dE[v_valid:]).item() == 0    # padding rows: zero gradient


def test_bwd_from_lse_1p2b_vocab_sampled():
    # T = 8192, h = 1536, vocabulary 50,257 padded to 51,200, t = 8 (the bench's cross-entropy):
    # sampled rows of dX and dE (padding rows included) against the oracle.
    w = synth.WORKLOADS["ce_1p2b"]
    inp = synth.ce_inputs(w["T"], w["h"], w["v_pad"], w["v_valid"], w["seed"])
    dl = torch.full((w["T"],), 1.0 / w["T"], dtype=torch.float32)
    _, lse, _ = _forward(inp, w["v_valid"], w["t"])
    dX, dE = _backward(inp, lse, dl, w["v_valid"], w["t"], one_pass=True)
    rows = synth.sample_indices(w["T"], 64, seed=41).numpy()
    erows = np.concatenate([synth.sample_indices(w["v_valid"], 48, seed=42).numpy(), [50257, 51199]])
    s = oracle.ce_bwd_sampled(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), dl.double().numpy(),
                              w["v_valid"], rows, erows)
    assert rel_fro(f64(dX)[rows], s["dX_rows"]) <= GRAD_REL_FRO
    assert rel_fro(f64(dE)[erows[:-2]], s["dE_rows"][:-2]) <= GRAD_REL_FRO
    assert torch.count_nonzero(dE[50257:]).item() == 0
