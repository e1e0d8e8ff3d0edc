"""GPU parity of the vocab-parallel cross-entropy backward against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import GRAD_REL_FRO, f64, mp, rel_fro, status_tensor

pytestmark = pytest.mark.gpu


def _dloss(T, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(T, generator=g, dtype=torch.float32)


def _forward_loss(inp, v_valid, t):
    m = mp()
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    T, v_pad = X.shape[0], E.shape[0]
    ws = torch.empty(max(m.mp_vocab_ce_workspace_bytes(T, v_pad, t), 16), dtype=torch.uint8, device="cuda")
    loss = torch.empty(T, dtype=torch.float32, device="cuda")
    m.mp_vocab_ce(X, E, tgt, loss, ws, v_valid=v_valid, t=t)
    return loss


def _run(inp, dloss, v_valid, t, expect_status=0, loss=None, one_pass=False):
    m = mp()
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    T, h = X.shape
    v_pad = E.shape[0]
    if loss is None:
        loss = _forward_loss(inp, v_valid, t)
    st = status_tensor()
    size = (m.mp_vocab_ce_bwd_workspace_bytes_one_pass if one_pass else m.mp_vocab_ce_bwd_workspace_bytes)
    wsb = torch.empty(size(T, h, v_pad, t), dtype=torch.uint8, device="cuda")
    dX = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dE = torch.full((v_pad, h), 7.0, dtype=torch.bfloat16, device="cuda")
    m.mp_vocab_ce_bwd(X, E, tgt, loss, dloss.cuda(), dX, dE, wsb, v_valid=v_valid, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status, int(st.item())
    return dX.cpu(), dE.cpu()


@pytest.mark.parametrize("T,h,v_pad,v_valid,t", [
    (300, 128, 2048, 2000, 2),     # padding columns excluded, ragged T
    (300, 128, 2048, 2048, 4),     # no padding
    (257, 192, 2048, 1500, 8),     # the last shards hold only padding
    (130, 64, 1024, 1000, 1),      # one shard: dX stored straight from the accumulator
])
@pytest.mark.parametrize("one_pass", [False, True])
def test_ce_bwd_matches_oracle(T, h, v_pad, v_valid, t, one_pass):
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=8000 + T)
    dl = _dloss(T, 8100 + T)
    dX, dE = _run(inp, dl, v_valid, t, one_pass=one_pass)
    ref = oracle.ce_bwd(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), dl.double().numpy(), v_valid)
    errs = {"dX": rel_fro(f64(dX), ref["dX"]), "dE": rel_fro(f64(dE), ref["dE"])}
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs
    assert torch.count_nonzero(dE[v_valid:]).item() == 0    # padding rows: zero gradient


def test_ce_bwd_one_pass_against_shard_by_shard():
    # With room for every shard's dZ the backward runs one GEMM of each kind: dE rows are the
    # same K-loops (bitwise equal); dX sums the shards inside one K-loop instead of through an
    # fp32 accumulator (equal within rounding).
    m = mp()
    T, h, v_pad, v_valid, t = 512, 192, 4096, 3900, 4
    assert m.mp_vocab_ce_bwd_workspace_bytes_one_pass(T, h, v_pad, t) > m.mp_vocab_ce_bwd_workspace_bytes(T, h, v_pad, t)
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=8400)
    dl = _dloss(T, 8401)
    loss = _forward_loss(inp, v_valid, t)
    dXs, dEs = _run(inp, dl, v_valid, t, loss=loss)
    dXo, dEo = _run(inp, dl, v_valid, t, loss=loss, one_pass=True)
    assert torch.equal(dEo, dEs)
    assert rel_fro(f64(dXo), f64(dXs)) <= 1e-3


def test_ce_bwd_shard_invariance():
    # Same forward loss for every shard count: each dE row is the same K-loop over the
    # tokens, so dE is bitwise identical; dX sums the shards' fp32 partials in shard order.
    inp = synth.ce_inputs(256, 128, 4096, 4000, seed=8200)
    dl = _dloss(256, 8201)
    loss = _forward_loss(inp, 4000, 1)
    dX1, dE1 = _run(inp, dl, 4000, 1, loss=loss)
    for t in (2, 4, 8, 16):
        dX, dE = _run(inp, dl, 4000, t, loss=loss)
        assert torch.equal(dE, dE1), t
        assert rel_fro(f64(dX), f64(dX1)) <= 1e-3, t
    dXa, dEa = _run(inp, dl, 4000, 4, loss=loss)
    dXb, dEb = _run(inp, dl, 4000, 4, loss=loss)
    assert torch.equal(dXa, dXb) and torch.equal(dEa, dEb)   # deterministic


def test_ce_bwd_1p2b_vocab_sampled():
    # T = 8192, h = 1536, vocabulary 50,257 padded to 51,200, t = 8: sampled rows of dX and dE.
    w = synth.WORKLOADS["ce_1p2b"]
    inp = synth.ce_inputs(w["T"], w["h"], w["v_pad"], w["v_valid"], w["seed"])
    dl = torch.full((w["T"],), 1.0 / w["T"], dtype=torch.float32)    # mean-loss gradient
    dX, dE = _run(inp, dl, w["v_valid"], w["t"], one_pass=True)
    rows = synth.sample_indices(w["T"], 64, seed=31).numpy()
    erows = np.unique(np.concatenate([synth.sample_indices(w["v_valid"], 60, seed=32).numpy(),
                                      np.array([50256, 50257, 51199])]))
    s = oracle.ce_bwd_sampled(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), dl.double().numpy(),
                              w["v_valid"], rows, erows)
    errs = {"dX": rel_fro(f64(dX)[rows], s["dX_rows"]), "dE": rel_fro(f64(dE)[erows], s["dE_rows"])}
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs


@pytest.mark.parametrize("one_pass", [False, True])
def test_ce_bwd_invalid_target_contributes_nothing(one_pass):
    m = mp()
    inp = synth.ce_inputs(64, 64, 1024, 1000, seed=8300)
    dl = _dloss(64, 8301)
    tgt = inp["target"].clone()
    tgt[7] = 1000
    inp["target"] = tgt
    dX, dE = _run(inp, dl, 1000, 2, expect_status=m.MP_DEV_TARGET_RANGE, one_pass=one_pass)
    keep = np.ones(64, dtype=bool)
    keep[7] = False
    ref = oracle.ce_bwd(f64(inp["X"])[keep], f64(inp["E"]), tgt.numpy()[keep], dl.double().numpy()[keep], 1000)
    assert torch.count_nonzero(dX[7]).item() == 0
    assert rel_fro(f64(dX)[keep], ref["dX"]) <= GRAD_REL_FRO
    assert rel_fro(f64(dE), ref["dE"]) <= GRAD_REL_FRO


@pytest.mark.parametrize("T,h,v_pad,v_valid,t", [
    (300, 128, 2048, 2000, 2),        # two shards: the first stores the accumulator, the last reads it
    (257, 192, 2048, 1500, 8),        # middle shards add at L2; the last shards hold only padding
    (1000, 384, 12800, 12345, 4),     # several row blocks and vocabulary tiles a shard
    (200, 64, 1024, 900, 8),          # a shard narrower than one 256-column tile, h = 64
    (8192, 1536, 51200, 50257, 8),    # the bench workload
    (32512, 1536, 51200, 50257, 8),   # 4092 tiles a shard: the most the chain's schedule table holds
])
def test_ce_bwd_shard_chain_bitwise_equal_to_separate_launches(T, h, v_pad, v_valid, t, monkeypatch):
    # Shard by shard, each shard's K10, K12 and K11 run as one launch of the chain kernel. They are
    # the same tiles and K-loops as the three separate launches (MPTP_CE_BWD_CHAIN=0), with dX
    # accumulated across shards in the same order, so both gradients are equal bit for bit.
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=8600 + T)
    dl = _dloss(T, 8601 + T)
    loss = _forward_loss(inp, v_valid, t)
    dXc, dEc = _run(inp, dl, v_valid, t, loss=loss)
    again = _run(inp, dl, v_valid, t, loss=loss)
    assert torch.equal(dXc, again[0]) and torch.equal(dEc, again[1])
    monkeypatch.setenv("MPTP_CE_BWD_CHAIN", "0")
    dXs, dEs = _run(inp, dl, v_valid, t, loss=loss)
    assert torch.equal(dXc, dXs) and torch.equal(dEc, dEs)
    if T <= 1000:
        ref = oracle.ce_bwd(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), dl.double().numpy(), v_valid)
        assert rel_fro(f64(dXc), ref["dX"]) <= GRAD_REL_FRO and rel_fro(f64(dEc), ref["dE"]) <= GRAD_REL_FRO


def test_ce_bwd_shard_chain_timeout_reports_and_recovers(monkeypatch):
    # A zero wait budget: the chain launches give up on their first wait that does not succeed at
    # once, report MP_DEV_TIMEOUT and return their counters to zero, so the next call is exact.
    m = mp()
    T, h, v_pad, v_valid, t = 1000, 384, 12800, 12345, 4
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=8700)
    dl = _dloss(T, 8701)
    loss = _forward_loss(inp, v_valid, t)
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    wsb = torch.empty(m.mp_vocab_ce_bwd_workspace_bytes(T, h, v_pad, t), dtype=torch.uint8, device="cuda")
    dX = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dE = torch.empty(v_pad, h, dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    monkeypatch.setenv("MPTP_WAIT_BUDGET_NS", "0")
    m.mp_vocab_ce_bwd(X, E, tgt, loss, dl.cuda(), dX, dE, wsb, v_valid=v_valid, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & m.MP_DEV_TIMEOUT
    monkeypatch.delenv("MPTP_WAIT_BUDGET_NS")
    dX2, dE2 = _run(inp, dl, v_valid, t, loss=loss)
    ref = oracle.ce_bwd(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), dl.double().numpy(), v_valid)
    assert rel_fro(f64(dX2), ref["dX"]) <= GRAD_REL_FRO and rel_fro(f64(dE2), ref["dE"]) <= GRAD_REL_FRO
