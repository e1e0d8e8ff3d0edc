"""Parity over the layer sweep: h in {1536, 1920, 2304, 3072} (f = 4h, the
Megatron-LM Table 1 widths), T in {2048, 8192}, t in {1, 2, 4, 8}; vocabulary
51,200 (50,257 valid). For each (h, T): MLP forward + backward for every t,
bitwise identical across t and within tolerance of the float64 oracle on sampled
rows of Z and dX, columns of dA and rows of dB; the fused cross-entropy for
every t on sampled tokens."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (GRAD_REL_FRO, LOSS_ABS, Z_MAX_ABS, Z_REL_FRO, f64, max_abs, rel_fro, run_ce, run_mlp_bwd,
                      run_mlp_fwd)

pytestmark = pytest.mark.gpu

SWEEP_H = (1536, 1920, 2304, 3072)
SWEEP_T = (2048, 8192)
SWEEP_SHARDS = (1, 2, 4, 8)


@pytest.mark.parametrize("T", SWEEP_T)
@pytest.mark.parametrize("h", SWEEP_H)
def test_mlp_sweep_point(h, T):
    f = 4 * h
    inp = synth.mlp_inputs(T, h, f, seed=7000 + h + T)
    ref = None
    for t in SWEEP_SHARDS:
        dev = run_mlp_fwd(inp, t)
        g = run_mlp_bwd(dev, inp["dZ"], t)
        out = {k: v.cpu() for k, v in (("Z", dev["Z"]), ("dX", g["dX"]), ("dA", g["dA"]), ("dB", g["dB"]))}
        if ref is None:
            ref = out
        else:
            for k in out:
                assert torch.equal(out[k], ref[k]), (t, k)
        del dev, g
        torch.cuda.empty_cache()
    X, A, B, G = (f64(inp[k]) for k in ("X", "A", "B", "dZ"))
    rows = synth.sample_indices(T, 48, seed=h).numpy()
    cols = synth.sample_indices(f, 48, seed=h + 1).numpy()
    brows = synth.sample_indices(f, 48, seed=h + 2).numpy()
    _, _, Zr = oracle.mlp_fwd_rows(X, A, B, rows)
    s = oracle.mlp_bwd_sampled(X, A, B, G, rows, cols, brows)
    Zg = f64(ref["Z"])[rows]
    assert rel_fro(Zg, Zr) <= Z_REL_FRO and max_abs(Zg, Zr) <= Z_MAX_ABS
    errs = {
        "dX": rel_fro(f64(ref["dX"])[rows], s["dX_rows"]),
        "dA": rel_fro(f64(ref["dA"])[:, cols], s["dA_cols"]),
        "dB": rel_fro(f64(ref["dB"])[brows], s["dB_rows"]),
    }
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs


@pytest.mark.parametrize("T", SWEEP_T)
@pytest.mark.parametrize("h", SWEEP_H)
def test_ce_sweep_point(h, T):
    v_pad, v_valid = 51200, 50257
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=7100 + h + T)
    rows = synth.sample_indices(T, 48, seed=h + 3).numpy()
    want = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], v_valid)
    for t in SWEEP_SHARDS:
        got = run_ce(inp, v_valid, t)
        assert np.all(np.isfinite(got))
        err = float(np.max(np.abs(got[rows] - want)))
        assert err <= LOSS_ABS, (t, err)
