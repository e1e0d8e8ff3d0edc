"""GPU parity of the sharded MLP (forward and backward) against the float64 oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (GRAD_REL_FRO, Z_MAX_ABS, Z_REL_FRO, f64, max_abs, rel_fro, run_mlp_bwd, run_mlp_fwd)

pytestmark = pytest.mark.gpu


def _fwd_check(T, h, f, t, seed):
    inp = synth.mlp_inputs(T, h, f, seed, with_grad=False)
    dev = run_mlp_fwd(inp, t)
    U, Y, Z = oracle.mlp_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]))
    errs = {
        "U": rel_fro(f64(dev["U"]), U), "Y": rel_fro(f64(dev["Y"]), Y),
        "Z": rel_fro(f64(dev["Z"]), Z), "Z_max": max_abs(f64(dev["Z"]), Z),
    }
    assert errs["U"] <= Z_REL_FRO and errs["Y"] <= Z_REL_FRO, errs
    assert errs["Z"] <= Z_REL_FRO and errs["Z_max"] <= Z_MAX_ABS, errs
    return dev


@pytest.mark.parametrize("T,h,f,t", [
    (256, 768, 3072, 2),     # the tiny workload
    (300, 256, 1024, 4),     # several tiles, ragged T
    (129, 192, 768, 3),      # ragged T, N = h not a multiple of 256
    (1, 64, 128, 2),         # one token
    (200, 128, 512, 8),      # f/t = 64, the smallest shard
])
def test_forward_matches_oracle(T, h, f, t):
    _fwd_check(T, h, f, t, seed=2000 + T)


def test_worked_example_embedded():
    # Two-token example of "Megatron-LM, annotated" section 3.1, zero-padded into a
    # supported shape: h = 64, f = 128, t = 2 (shard width 64), T = 128.
    T, h, f = 128, 64, 128
    X = torch.zeros(T, h)
    X[0, 0:2] = torch.tensor([1.0, 2.0])
    A = torch.zeros(h, f)
    A[0:2, 0] = torch.tensor([1.0, -1.0])    # shard 0's first column
    A[0:2, 64] = torch.tensor([-1.0, 1.0])   # shard 1's first column
    B = torch.zeros(f, h)
    B[0, 0:2] = torch.tensor([2.0, 0.0])
    B[64, 0:2] = torch.tensor([1.0, 1.0])
    inp = {k: v.to(torch.bfloat16) for k, v in (("X", X), ("A", A), ("B", B))}
    dev = run_mlp_fwd(inp, t=2)
    Z = f64(dev["Z"])
    Y = f64(dev["Y"])
    assert abs(Y[0, 0] - (-0.159)) < 3e-3 and abs(Y[0, 64] - 0.841) < 3e-3
    assert abs(Z[0, 0] - 0.524) < 3e-3 and abs(Z[0, 1] - 0.841) < 3e-3
    Zr = Z.copy()
    Zr[0, 0:2] = 0.0
    assert np.all(Zr == 0.0)


def test_shard_count_invariance_bitwise():
    # The K-loop visits shards in order with the same K blocks for every t,
    # so Z is bitwise identical for every shard count.
    inp = synth.mlp_inputs(384, 256, 1024, 2100, with_grad=False)
    ref = None
    for t in (1, 2, 4, 8, 16):
        Z = run_mlp_fwd(inp, t)["Z"].cpu()
        if ref is None:
            ref = Z
        else:
            assert torch.equal(Z, ref), f"t={t}"


def test_forward_deterministic():
    inp = synth.mlp_inputs(300, 256, 1024, 2200, with_grad=False)
    a = run_mlp_fwd(inp, 4)
    b = run_mlp_fwd(inp, 4)
    for k in ("Z", "Y", "U"):
        assert torch.equal(a[k], b[k]), k


def test_forward_without_u_save():
    inp = synth.mlp_inputs(256, 128, 512, 2300, with_grad=False)
    a = run_mlp_fwd(inp, 2, save_u=True)
    b = run_mlp_fwd(inp, 2, save_u=False)
    assert torch.equal(a["Z"], b["Z"]) and torch.equal(a["Y"], b["Y"])


@pytest.mark.parametrize("t", [2, 4])
def test_forward_1p2b_layer_sampled(t):
    # T = 8192, h = 1536, f = 6144 (the 1.2B-layer shape): sampled rows vs the oracle.
    w = synth.WORKLOADS["mlp_1p2b"]
    inp = synth.mlp_inputs(w["T"], w["h"], w["f"], w["seed"], with_grad=False)
    dev = run_mlp_fwd(inp, t)
    rows = synth.sample_indices(w["T"], 192, seed=7 + t).numpy()
    _, Yr, Zr = oracle.mlp_fwd_rows(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), rows)
    Zg = f64(dev["Z"])[rows]
    Yg = f64(dev["Y"])[rows]
    assert rel_fro(Yg, Yr) <= Z_REL_FRO
    assert rel_fro(Zg, Zr) <= Z_REL_FRO and max_abs(Zg, Zr) <= Z_MAX_ABS, (rel_fro(Zg, Zr), max_abs(Zg, Zr))


@pytest.mark.parametrize("T,h,f,t", [
    (256, 256, 1024, 4),
    (300, 192, 768, 3),      # ragged T (also the K of the weight gradients), ragged N = h
    (77, 128, 512, 2),       # fewer tokens than one tile
])
def test_backward_matches_oracle(T, h, f, t):
    inp = synth.mlp_inputs(T, h, f, 3000 + T)
    dev = run_mlp_fwd(inp, t)
    g = run_mlp_bwd(dev, inp["dZ"], t)
    ref = oracle.mlp_bwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), f64(inp["dZ"]))
    errs = {k: rel_fro(f64(g[k]), ref[k]) for k in ("dX", "dA", "dB", "dU")}
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs


def test_backward_shard_invariance_and_determinism():
    inp = synth.mlp_inputs(256, 256, 1024, 3100)
    dev = run_mlp_fwd(inp, 1)
    ref = run_mlp_bwd(dev, inp["dZ"], 1)
    for t in (2, 4, 8):
        g = run_mlp_bwd(dev, inp["dZ"], t)
        for k in ("dX", "dA", "dB"):
            assert torch.equal(g[k], ref[k]), (t, k)


def test_mlp_8p3b_layer_fwd_bwd_sampled():
    # T = 4096, h = 3072, f = 12288, t = 8 (the 8.3B-layer shape), in the launch
    # configuration the bench times; rows of Z and dX, columns of dA, rows of dB.
    w = synth.WORKLOADS["mlp_8p3b"]
    inp = synth.mlp_inputs(w["T"], w["h"], w["f"], w["seed"])
    dev = run_mlp_fwd(inp, w["t"])
    g = run_mlp_bwd(dev, inp["dZ"], w["t"])
    X, A, B, G = (f64(inp[k]) for k in ("X", "A", "B", "dZ"))
    rows = synth.sample_indices(w["T"], 128, seed=11).numpy()
    cols = synth.sample_indices(w["f"], 128, seed=12).numpy()
    brows = synth.sample_indices(w["f"], 128, seed=13).numpy()
    _, _, Zr = oracle.mlp_fwd_rows(X, A, B, rows)
    s = oracle.mlp_bwd_sampled(X, A, B, G, rows, cols, brows)
    Zg = f64(dev["Z"])[rows]
    assert rel_fro(Zg, Zr) <= Z_REL_FRO and max_abs(Zg, Zr) <= Z_MAX_ABS
    errs = {
        "dX": rel_fro(f64(g["dX"])[rows], s["dX_rows"]),
        "dA": rel_fro(f64(g["dA"])[:, cols], s["dA_cols"]),
        "dB": rel_fro(f64(g["dB"])[brows], s["dB_rows"]),
    }
    assert all(v <= GRAD_REL_FRO for v in errs.values()), errs


def test_empty_batch():
    import tensor_transformer_layer_gb300 as m
    X = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    A = torch.randn(64, 128, device="cuda").to(torch.bfloat16)
    B = torch.randn(128, 64, device="cuda").to(torch.bfloat16)
    Z = torch.empty(0, 64, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(0, 128, dtype=torch.bfloat16, device="cuda")
    m.mp_mlp_fwd(X, A, B, Z, Y, None, t=2)
    dA = torch.full((64, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    dB = torch.full((128, 64), 7.0, dtype=torch.bfloat16, device="cuda")
    m.mp_mlp_bwd(X, A, B, Y, Y, Z, Z, dA, dB, Y, t=2)
    torch.cuda.synchronize()
    assert torch.count_nonzero(dA).item() == 0 and torch.count_nonzero(dB).item() == 0


def test_misaligned_pointer_rejected():
    import tensor_transformer_layer_gb300 as m
    buf = torch.zeros(64 * 128 + 8, dtype=torch.bfloat16, device="cuda")
    A_bad = buf[1:1 + 64 * 128].view(64, 128)    # 2-byte offset
    X = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(128, 64, dtype=torch.bfloat16, device="cuda")
    Z = torch.zeros(8, 64, dtype=torch.bfloat16, device="cuda")
    Y = torch.zeros(8, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(m.MptpError) as e:
        m.mp_mlp_fwd(X, A_bad, B, Z, Y, None, t=1)
    assert e.value.code == 3
