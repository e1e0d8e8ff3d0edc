"""GPU parity of the vocab-parallel fused cross-entropy against the float64 oracle."""
import math

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import LOSS_ABS, f64, run_ce

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,h,v_pad,v_valid,t", [
    (300, 128, 2048, 2000, 2),    # pad columns excluded, ragged T
    (300, 128, 2048, 2048, 4),    # pad columns included (v_valid = v_pad)
    (257, 192, 2048, 1500, 8),    # one tile per shard; the last shards hold only padding
    (130, 64, 768, 700, 2),       # shard of 384 = 3 tiles of 128 (narrow-tile path)
    (1, 64, 256, 256, 1),         # one token
])
def test_ce_matches_oracle(T, h, v_pad, v_valid, t):
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=4000 + T)
    got = run_ce(inp, v_valid, t)
    want = oracle.ce_loss(f64(inp["X"]), f64(inp["E"]), inp["target"].numpy(), v_valid)
    err = np.max(np.abs(got - want))
    assert err <= LOSS_ABS, err


def test_ce_1p2b_vocab_sampled():
    # T = 8192, h = 1536, v 50,257 padded to 51,200, t = 8: sampled tokens.
    w = synth.WORKLOADS["ce_1p2b"]
    inp = synth.ce_inputs(w["T"], w["h"], w["v_pad"], w["v_valid"], w["seed"])
    got = run_ce(inp, w["v_valid"], w["t"])
    rows = synth.sample_indices(w["T"], 256, seed=21).numpy()
    want = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], w["v_valid"])
    err = np.max(np.abs(got[rows] - want))
    assert err <= LOSS_ABS, err
    assert np.all(np.isfinite(got))


def test_ce_8p3b_layer_sampled():
    # The 8.3B-layer width: T = 4096 (b = 4, s = 1024), h = 3072, the same vocabulary and
    # t = 8, in the launch configuration the bench times; sampled tokens incl. the last.
    w = synth.WORKLOADS["ce_8p3b"]
    inp = synth.ce_inputs(w["T"], w["h"], w["v_pad"], w["v_valid"], w["seed"])
    got = run_ce(inp, w["v_valid"], w["t"])
    rows = synth.sample_indices(w["T"], 192, seed=22).numpy()
    want = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], w["v_valid"])
    err = np.max(np.abs(got[rows] - want))
    assert err <= LOSS_ABS, err
    assert np.all(np.isfinite(got))


def test_ce_partition_follows_workspace():
    # T = 4096 runs one-tile vocabulary chunks (200 partitions) with the workspace
    # mp_vocab_ce_workspace_bytes asks for, and coarser ones in a smaller workspace (40 partitions
    # in 4 MiB, 8 in 8 x 3 x T floats): the same loss within fp32 rounding, and the oracle's.
    import tensor_transformer_layer_gb300 as m
    T, h, v_pad, v_valid, t = 4096, 128, 51200, 50257, 8
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=4500)
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    out = []
    for nbytes in (m.mp_vocab_ce_workspace_bytes(T, v_pad, t), 4 << 20, 8 * 3 * T * 4):
        ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
        loss = torch.empty(T, dtype=torch.float32, device="cuda")
        m.mp_vocab_ce(X, E, tgt, loss, ws, v_valid=v_valid, t=t)
        torch.cuda.synchronize()
        out.append(loss.cpu().numpy().astype(np.float64))
    assert np.max(np.abs(out[1] - out[0])) <= 1e-4 and np.max(np.abs(out[2] - out[0])) <= 1e-4
    rows = synth.sample_indices(T, 64, seed=23).numpy()
    want = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], v_valid)
    for o in out:
        assert np.max(np.abs(o[rows] - want)) <= LOSS_ABS


def test_ce_zero_embedding_closed_form():
    inp = synth.ce_inputs(200, 128, 51200, 50257, seed=4100)
    inp["E"] = torch.zeros_like(inp["E"])
    got = run_ce(inp, 50257, 8)
    assert np.max(np.abs(got - math.log(50257))) <= 1e-4
    got = run_ce(inp, 51200, 8)
    assert np.max(np.abs(got - math.log(51200))) <= 1e-4


def test_ce_partition_invariance():
    inp = synth.ce_inputs(256, 128, 4096, 4000, seed=4200)
    ref = run_ce(inp, 4000, 1)
    for t in (2, 4, 8, 16, 32):
        assert np.max(np.abs(run_ce(inp, 4000, t) - ref)) <= 1e-4, t


def test_ce_deterministic():
    inp = synth.ce_inputs(300, 128, 2048, 2000, seed=4300)
    a = run_ce(inp, 2000, 4)
    b = run_ce(inp, 2000, 4)
    assert np.array_equal(a, b)


def test_ce_target_out_of_range():
    inp = synth.ce_inputs(64, 64, 1024, 1000, seed=4400)
    tgt = inp["target"].clone()
    tgt[5] = 1000          # a padding id: outside [0, v_valid)
    tgt[9] = -3
    inp["target"] = tgt
    import tensor_transformer_layer_gb300 as m
    got = run_ce(inp, 1000, 2, expect_status=m.MP_DEV_TARGET_RANGE)
    assert np.isnan(got[5]) and np.isnan(got[9])
    ok = np.ones(64, dtype=bool)
    ok[[5, 9]] = False
    good = tgt.numpy().copy()
    good[[5, 9]] = 0
    want = oracle.ce_loss(f64(inp["X"]), f64(inp["E"]), good, 1000)
    assert np.max(np.abs(got[ok] - want[ok])) <= LOSS_ABS


def test_ce_halves_match_fused_call():
    import tensor_transformer_layer_gb300 as m
    inp = synth.ce_inputs(300, 128, 2048, 2000, seed=4500)
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    ws = torch.empty(m.mp_vocab_ce_workspace_bytes(300, 2048, 2), dtype=torch.uint8, device="cuda")
    loss = torch.empty(300, dtype=torch.float32, device="cuda")
    m.mp_vocab_ce_partials(X, E, tgt, ws, v_valid=2000, t=2)
    m.mp_vocab_ce_combine(ws, tgt, loss, v_pad=2048, v_valid=2000, t=2)
    torch.cuda.synchronize()
    assert np.array_equal(loss.cpu().numpy().astype(np.float64), run_ce(inp, 2000, 2))


def test_ce_workspace_too_small():
    import tensor_transformer_layer_gb300 as m
    inp = synth.ce_inputs(64, 64, 1024, 1000, seed=4600)
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    ws = torch.empty(64, dtype=torch.uint8, device="cuda")
    loss = torch.empty(64, dtype=torch.float32, device="cuda")
    with pytest.raises(m.MptpError) as e:
        m.mp_vocab_ce(X, E, tgt, loss, ws, v_valid=1000, t=2)
    assert e.value.code == 8


@pytest.mark.parametrize("T", [20000, 40000, 70000, 70001])
def test_ce_combine_group_sizes(T):
    # The combine splits each 32-token group's 16 partitions over G warps, G from the token count
    # (here 4, 2, 1 and 1 with a ragged last warp); sampled tokens (the first and last groups
    # among them) against the oracle.
    h, v_pad, v_valid, t = 64, 16384, 16000, 8
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=4700 + T)
    got = run_ce(inp, v_valid, t)
    rows = np.unique(np.concatenate([np.arange(40), synth.sample_indices(T, 48, seed=5).numpy(),
                                     np.arange(T - 40, T)]))
    want = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], v_valid)
    assert float(np.max(np.abs(got[rows] - want))) <= LOSS_ABS
    assert np.all(np.isfinite(got))
