"""GPU parity of the shard-range MLP calls: the partial outputs of single shards
and shard ranges, before the g (forward) and f (backward) sums.

"Megatron-LM: Training Multi-Billion Parameter Language Models Using Model
Parallelism", section 3.4 "Row-Parallel GEMM for the Second MLP Layer": each
shard's output Y_i B_i is a partial sum that g adds up; "Megatron-LM, annotated",
section 3.1 prints the two partials of its one-token example. Each partial is
compared with the float64 oracle's shard-by-shard form (oracle.mlp_sharded_fwd /
mlp_sharded_bwd), the range's written blocks with the full call's (bitwise: the
same K-loop per element), the untouched blocks with their sentinel, and the sum of
the parts with the full call (within tolerance).
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (GRAD_REL_FRO, Z_MAX_ABS, Z_REL_FRO, f64, max_abs, rel_fro, run_mlp_bwd, run_mlp_fwd,
                      status_tensor)

pytestmark = pytest.mark.gpu

SENTINEL = 3.0   # exact in bf16, far from any value the layer produces at these scales


def _mp():
    import tensor_transformer_layer_gb300 as m
    m.lib()
    return m


def _fwd_range(inp, t, s0, n):
    m = _mp()
    X, A, B = (inp[k].cuda() for k in ("X", "A", "B"))
    T, h = X.shape
    f = A.shape[1]
    Z = torch.full((T, h), SENTINEL, dtype=torch.bfloat16, device="cuda")
    Y = torch.full((T, f), SENTINEL, dtype=torch.bfloat16, device="cuda")
    U = torch.full((T, f), SENTINEL, dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    m.mp_mlp_fwd_shards(X, A, B, Z, Y, U, t=t, shard_begin=s0, shard_count=n, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return {"Z": Z.cpu(), "Y": Y.cpu(), "U": U.cpu()}


def _bwd_range(dev, dZ, t, s0, n):
    m = _mp()
    X, A, B, U, Y = dev["X"], dev["A"], dev["B"], dev["U"], dev["Y"]
    T, h = X.shape
    f = A.shape[1]
    full = lambda *s: torch.full(s, SENTINEL, dtype=torch.bfloat16, device="cuda")
    out = {"dX": full(T, h), "dA": full(h, f), "dB": full(f, h), "dU": full(T, f)}
    st = status_tensor()
    m.mp_mlp_bwd_shards(X, A, B, U, Y, dZ.cuda(), out["dX"], out["dA"], out["dB"], out["dU"], t=t,
                        shard_begin=s0, shard_count=n, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return {k: v.cpu() for k, v in out.items()}


def test_worked_example_partials():
    # The one-token example of "Megatron-LM, annotated" section 3.1 zero-padded into a supported
    # shape (h = 64, f = 128, t = 2, shard width 64, T = 128): shard 0's partial output is
    # [-0.317, 0], shard 1's [0.841, 0.841], and their sum Z = [0.524, 0.841].
    T, h, f = 128, 64, 128
    X = torch.zeros(T, h)
    X[0, 0:2] = torch.tensor([1.0, 2.0])
    A = torch.zeros(h, f)
    A[0:2, 0] = torch.tensor([1.0, -1.0])
    A[0:2, 64] = torch.tensor([-1.0, 1.0])
    B = torch.zeros(f, h)
    B[0, 0:2] = torch.tensor([2.0, 0.0])
    B[64, 0:2] = torch.tensor([1.0, 1.0])
    inp = {k: v.to(torch.bfloat16) for k, v in (("X", X), ("A", A), ("B", B))}
    want = {0: (-0.317, 0.0), 1: (0.841, 0.841)}
    parts = []
    for s0 in (0, 1):
        Z = f64(_fwd_range(inp, 2, s0, 1)["Z"])
        assert abs(Z[0, 0] - want[s0][0]) < 3e-3 and abs(Z[0, 1] - want[s0][1]) < 3e-3, (s0, Z[0, :2])
        rest = Z.copy()
        rest[0, 0:2] = 0.0
        assert np.all(rest == 0.0)
        parts.append(Z)
    total = parts[0] + parts[1]
    assert abs(total[0, 0] - 0.524) < 5e-3 and abs(total[0, 1] - 0.841) < 5e-3


@pytest.mark.parametrize("T,h,f,t", [
    (256, 768, 3072, 2),     # the tiny workload
    (300, 256, 1024, 4),     # ragged T, four shards
    (200, 192, 768, 3),      # N = h not a multiple of 256; shards of 256 columns
])
def test_forward_single_shard_partials(T, h, f, t):
    inp = synth.mlp_inputs(T, h, f, 6000 + T, with_grad=False)
    full = run_mlp_fwd(inp, t)
    fullY, fullU, fullZ = full["Y"].cpu(), full["U"].cpu(), f64(full["Z"])
    _, parts = oracle.mlp_sharded_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), t)
    fs = f // t
    acc = np.zeros((T, h))
    for i in range(t):
        got = _fwd_range(inp, t, i, 1)
        Zi = f64(got["Z"])
        assert rel_fro(Zi, parts[i]) <= Z_REL_FRO and max_abs(Zi, parts[i]) <= Z_MAX_ABS, i
        cols = slice(i * fs, (i + 1) * fs)
        assert torch.equal(got["Y"][:, cols], fullY[:, cols]) and torch.equal(got["U"][:, cols], fullU[:, cols])
        other = torch.ones(f, dtype=torch.bool)
        other[cols] = False
        assert torch.all(got["Y"][:, other] == SENTINEL) and torch.all(got["U"][:, other] == SENTINEL)
        acc += Zi
    # The g sum of the parts is the full output (one more bf16 rounding per part).
    assert rel_fro(acc, fullZ) <= Z_REL_FRO and max_abs(acc, fullZ) <= Z_MAX_ABS


def test_forward_shard_ranges():
    # Ranges of several shards: the partial is the oracle's sum over the range; the full range
    # equals mp_mlp_fwd bit for bit.
    T, h, f, t = 300, 256, 1024, 4
    inp = synth.mlp_inputs(T, h, f, 6100, with_grad=False)
    _, parts = oracle.mlp_sharded_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), t)
    for s0, n in ((1, 2), (0, 3), (2, 2)):
        Zr = f64(_fwd_range(inp, t, s0, n)["Z"])
        want = sum(parts[s0:s0 + n])
        assert rel_fro(Zr, want) <= Z_REL_FRO and max_abs(Zr, want) <= Z_MAX_ABS, (s0, n)
    whole = _fwd_range(inp, t, 0, t)
    full = run_mlp_fwd(inp, t)
    for k in ("Z", "Y", "U"):
        assert torch.equal(whole[k], full[k].cpu()), k


@pytest.mark.parametrize("T,h,f,t", [
    (256, 256, 1024, 4),
    (300, 192, 768, 3),      # ragged T (the K of the weight gradients), ragged N = h
])
def test_backward_single_shard_partials(T, h, f, t):
    inp = synth.mlp_inputs(T, h, f, 6200 + T)
    dev = run_mlp_fwd(inp, t)
    full = {k: v.cpu() for k, v in run_mlp_bwd(dev, inp["dZ"], t).items()}
    ref = oracle.mlp_sharded_bwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), f64(inp["dZ"]), t)
    fs = f // t
    acc = np.zeros((T, h))
    for i in range(t):
        g = _bwd_range(dev, inp["dZ"], t, i, 1)
        dXi = f64(g["dX"])
        assert rel_fro(dXi, ref["dX_parts"][i]) <= GRAD_REL_FRO, i
        # one shard's part is not the whole input gradient (the f sum is needed)
        assert rel_fro(dXi, ref["dX"]) > 0.1
        cols = slice(i * fs, (i + 1) * fs)
        assert torch.equal(g["dA"][:, cols], full["dA"][:, cols])
        assert torch.equal(g["dB"][cols, :], full["dB"][cols, :])
        assert torch.equal(g["dU"][:, cols], full["dU"][:, cols])
        other = torch.ones(f, dtype=torch.bool)
        other[cols] = False
        assert torch.all(g["dA"][:, other] == SENTINEL) and torch.all(g["dB"][other, :] == SENTINEL)
        assert torch.all(g["dU"][:, other] == SENTINEL)
        assert rel_fro(f64(g["dA"][:, cols]), ref["dA"][:, cols]) <= GRAD_REL_FRO
        assert rel_fro(f64(g["dB"][cols, :]), ref["dB"][cols, :]) <= GRAD_REL_FRO
        acc += dXi
    # f: the sum of the shards' parts is the input gradient.
    assert rel_fro(acc, ref["dX"]) <= GRAD_REL_FRO and rel_fro(acc, f64(full["dX"])) <= GRAD_REL_FRO


def test_backward_full_range_is_mp_mlp_bwd():
    T, h, f, t = 256, 256, 1024, 4
    inp = synth.mlp_inputs(T, h, f, 6300)
    dev = run_mlp_fwd(inp, t)
    full = run_mlp_bwd(dev, inp["dZ"], t)
    whole = _bwd_range(dev, inp["dZ"], t, 0, t)
    for k in ("dX", "dA", "dB", "dU"):
        assert torch.equal(whole[k], full[k].cpu()), k


def test_backward_empty_batch_range():
    # T = 0: the range's weight-gradient blocks are zero, the rest untouched.
    m = _mp()
    h, f, t = 64, 256, 4
    X = torch.empty(0, h, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros(h, f, dtype=torch.bfloat16, device="cuda")
    B = torch.zeros(f, h, dtype=torch.bfloat16, device="cuda")
    E0 = torch.empty(0, f, dtype=torch.bfloat16, device="cuda")
    dA = torch.full((h, f), SENTINEL, dtype=torch.bfloat16, device="cuda")
    dB = torch.full((f, h), SENTINEL, dtype=torch.bfloat16, device="cuda")
    m.mp_mlp_bwd_shards(X, A, B, E0, E0, X, X, dA, dB, E0, t=t, shard_begin=1, shard_count=2)
    torch.cuda.synchronize()
    dA, dB = dA.cpu(), dB.cpu()
    assert torch.all(dA[:, 64:192] == 0) and torch.all(dA[:, :64] == SENTINEL) and torch.all(dA[:, 192:] == SENTINEL)
    assert torch.all(dB[64:192] == 0) and torch.all(dB[:64] == SENTINEL) and torch.all(dB[192:] == SENTINEL)


def test_8p3b_layer_single_shard_partials_sampled():
    # T = 4096, h = 3072, f = 12288, t = 8 (the bench's layer): shard 5's partial output Z_5 and its
    # part of dX on sampled rows, against the shard-by-shard formulas of the oracle module restricted
    # to those rows (a row of Z_i or dX_i needs only its own rows of X and dZ).
    w = synth.WORKLOADS["mlp_8p3b"]
    T, h, f, t = w["T"], w["h"], w["f"], w["t"]
    i, fs = 5, f // t
    inp = synth.mlp_inputs(T, h, f, w["seed"])
    fwd = _fwd_range(inp, t, i, 1)
    dev = run_mlp_fwd(inp, t)
    g = _bwd_range(dev, inp["dZ"], t, i, 1)
    rows = synth.sample_indices(T, 64, seed=51).numpy()
    X, A, B, G = (f64(inp[k]) for k in ("X", "A", "B", "dZ"))
    Ai, Bi = A[:, i * fs:(i + 1) * fs], B[i * fs:(i + 1) * fs, :]
    Ui = X[rows] @ Ai
    Zi = oracle.gelu(Ui) @ Bi
    dXi = ((G[rows] @ Bi.T) * oracle.gelu_prime(Ui)) @ Ai.T
    assert rel_fro(f64(fwd["Z"])[rows], Zi) <= Z_REL_FRO and max_abs(f64(fwd["Z"])[rows], Zi) <= Z_MAX_ABS
    assert rel_fro(f64(g["dX"])[rows], dXi) <= GRAD_REL_FRO
