"""Maximum-size cases: element offsets past 2^31 in the MLP activations, and a long
token batch for the fused cross-entropy. Checked on sampled rows and columns against
the float64 oracle (row- and column-separable forms), plus finiteness everywhere."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (GRAD_REL_FRO, LOSS_ABS, Z_MAX_ABS, Z_REL_FRO, f64, max_abs, rel_fro, run_ce, run_mlp_bwd,
                      run_mlp_fwd)

pytestmark = pytest.mark.gpu


def test_mlp_activations_past_2_31_elements():
    # T * f = (2^18 + 256) * 8192 > 2^31: U, Y and dU offsets need 64-bit arithmetic.
    T, h, f, t = (1 << 18) + 256, 2048, 8192, 4
    assert T * f > 2 ** 31
    inp = synth.mlp_inputs(T, h, f, seed=12000)
    dev = run_mlp_fwd(inp, t)
    g = run_mlp_bwd(dev, inp["dZ"], t)
    X, A, B, G = (f64(inp[k]) for k in ("X", "A", "B", "dZ"))
    rows = np.unique(np.concatenate([synth.sample_indices(T, 24, seed=1).numpy(), np.arange(T - 8, T)]))
    cols = synth.sample_indices(f, 6, seed=2).numpy()
    brows = synth.sample_indices(f, 6, seed=3).numpy()
    _, _, Zr = oracle.mlp_fwd_rows(X, A, B, rows)
    s = oracle.mlp_bwd_sampled(X, A, B, G, rows, cols, brows)
    Zg = f64(dev["Z"][torch.as_tensor(rows, device="cuda")])
    assert rel_fro(Zg, Zr) <= Z_REL_FRO and max_abs(Zg, Zr) <= Z_MAX_ABS
    errs = {
        "dX": rel_fro(f64(g["dX"][torch.as_tensor(rows, device="cuda")]), s["dX_rows"]),
        "dA": rel_fro(f64(g["dA"][:, torch.as_tensor(cols, device="cuda")]), s["dA_cols"]),
        "dB": rel_fro(f64(g["dB"][torch.as_tensor(brows, device="cuda")]), s["dB_rows"]),
    }
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs
    for k in ("Z", "Y"):
        assert torch.isfinite(dev[k][-4:].float()).all(), k
    assert torch.isfinite(g["dX"][-4:].float()).all()


def test_ce_long_batch():
    # T = 2^17 + 100 tokens (ragged), h = 1536, vocabulary 50,257 padded to 51,200, t = 8.
    T, h, v_pad, v_valid, t = (1 << 17) + 100, 1536, 51200, 50257, 8
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=12100)
    got = run_ce(inp, v_valid, t)
    rows = np.unique(np.concatenate([synth.sample_indices(T, 48, seed=4).numpy(), np.arange(T - 4, T)]))
    want = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], v_valid)
    assert float(np.max(np.abs(got[rows] - want))) <= LOSS_ABS
    assert np.all(np.isfinite(got))
