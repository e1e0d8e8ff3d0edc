"""GPU parity of the one-launch MLP entry points (mp_mlp_fwd_fused, mp_mlp_bwd_fused).

They run the same tiles with the same K-loops as the separate-launch entry points, so
wherever those use one CTA pair per tile the outputs must be equal bit for bit; they are
also held to the float64 oracle at the stated tolerances. Every output and the dU
workspace are filled with NaN before each call: a tile read before its producer had
written it would carry the NaN (or a previous call's values) into the result. The
shared workspace must be all zeros again after every call.
"""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import GRAD_REL_FRO, Z_MAX_ABS, Z_REL_FRO, f64, max_abs, rel_fro, run_mlp_bwd, run_mlp_fwd

pytestmark = pytest.mark.gpu


def _mp():
    import tensor_transformer_layer_gb300 as mp
    mp.lib()
    return mp


def _nan(*shape):
    return torch.full(shape, float("nan"), dtype=torch.bfloat16, device="cuda")


def fused_fwd(mp, X, A, B, t, ws, save_u=True, shard_begin=0, shard_count=None):
    T, h = X.shape
    f = A.shape[1]
    Z, Y = _nan(T, h), _nan(T, f)
    U = _nan(T, f) if save_u else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mp.mp_mlp_fwd_fused(X, A, B, Z, Y, U, t=t, workspace=ws, shard_begin=shard_begin, shard_count=shard_count,
                        d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, int(st.item())
    assert int(ws.count_nonzero().item()) == 0, "workspace not returned to zeros"
    return Z, Y, U


def fused_bwd(mp, X, A, B, U, Y, dZ, t, ws, shard_begin=0, shard_count=None):
    T, h = X.shape
    f = A.shape[1]
    out = {"dX": _nan(T, h), "dA": _nan(h, f), "dB": _nan(f, h), "dU": _nan(T, f)}
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    mp.mp_mlp_bwd_fused(X, A, B, U, Y, dZ, out["dX"], out["dA"], out["dB"], out["dU"], t=t, workspace=ws,
                        shard_begin=shard_begin, shard_count=shard_count, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, int(st.item())
    assert int(ws.count_nonzero().item()) == 0, "workspace not returned to zeros"
    return out


@pytest.mark.parametrize("T,h,f,t", [
    (256, 768, 3072, 2),     # the tiny workload
    (300, 256, 1024, 4),     # ragged T
    (129, 192, 768, 3),      # ragged T, N = h not a multiple of 256
    (1, 64, 128, 2),         # one token
    (200, 128, 512, 8),      # f/t = 64, the smallest shard
    (1000, 512, 2048, 4),    # several row blocks and column tiles, ragged T
])
def test_fused_matches_oracle(T, h, f, t):
    mp = _mp()
    inp = synth.mlp_inputs(T, h, f, seed=7000 + T)
    X, A, B, dZ = (inp[k].cuda() for k in ("X", "A", "B", "dZ"))
    ws = mp.mp_mlp_fused_workspace(T, h, f, t)
    Z, Y, U = fused_fwd(mp, X, A, B, t, ws)
    Ur, Yr, Zr = oracle.mlp_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]))
    assert rel_fro(f64(U), Ur) <= Z_REL_FRO and rel_fro(f64(Y), Yr) <= Z_REL_FRO
    assert rel_fro(f64(Z), Zr) <= Z_REL_FRO and max_abs(f64(Z), Zr) <= Z_MAX_ABS
    g = fused_bwd(mp, X, A, B, U, Y, dZ, t, ws)
    ref = oracle.mlp_bwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), f64(inp["dZ"]))
    for k in ("dX", "dA", "dB", "dU"):
        assert rel_fro(f64(g[k]), ref[k]) <= GRAD_REL_FRO, (k, rel_fro(f64(g[k]), ref[k]))


@pytest.mark.parametrize("T,h,f,t", [
    (300, 256, 1024, 4),     # K2 with 16 K blocks: the separate forward runs one pair a tile
    (1000, 512, 1536, 2),
    (8192, 1536, 6144, 4),   # the 1.2B layer (no split-K in the separate kernels)
    (4096, 3072, 12288, 8),  # the 8.3B layer
])
def test_fused_bitwise_equal_to_separate_launches(T, h, f, t, monkeypatch):
    # The separate backward's side-by-side schedule runs K4 one pair a tile (never split-K).
    monkeypatch.setenv("MPTP_BWD_SCHEDULE", "overlap")
    mp = _mp()
    inp = synth.mlp_inputs(T, h, f, seed=7100 + h)
    dev = run_mlp_fwd(inp, t)
    ws = mp.mp_mlp_fused_workspace(T, h, f, t)
    Z, Y, U = fused_fwd(mp, dev["X"], dev["A"], dev["B"], t, ws)
    # (at these shapes the separate K2 runs one pair a tile: no split-K)
    assert torch.equal(U, dev["U"]) and torch.equal(Y, dev["Y"]) and torch.equal(Z, dev["Z"])
    sep = run_mlp_bwd(dev, inp["dZ"], t)
    g = fused_bwd(mp, dev["X"], dev["A"], dev["B"], dev["U"], dev["Y"], inp["dZ"].cuda(), t, ws)
    for k in ("dU", "dX", "dA", "dB"):
        assert torch.equal(g[k], sep[k]), k
    # sampled rows and columns against the oracle at the full size
    rows = synth.sample_indices(T, 16, seed=7200).numpy()
    cols = synth.sample_indices(f, 16, seed=7201).numpy()
    ref = oracle.mlp_bwd_sampled(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), f64(inp["dZ"]), rows, cols, cols)
    assert rel_fro(f64(g["dX"])[rows], ref["dX_rows"]) <= GRAD_REL_FRO
    assert rel_fro(f64(g["dA"])[:, cols], ref["dA_cols"]) <= GRAD_REL_FRO
    assert rel_fro(f64(g["dB"])[cols], ref["dB_rows"]) <= GRAD_REL_FRO
    _, _, Zr = oracle.mlp_fwd_rows(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), rows)
    assert rel_fro(f64(Z)[rows], Zr) <= Z_REL_FRO


def test_fused_shard_ranges_equal_separate_shard_calls():
    mp = _mp()
    T, h, f, t = 700, 256, 1024, 4
    inp = synth.mlp_inputs(T, h, f, seed=7300)
    X, A, B, dZ = (inp[k].cuda() for k in ("X", "A", "B", "dZ"))
    ws = mp.mp_mlp_fused_workspace(T, h, f, t)
    full = run_mlp_fwd(inp, t)
    fs = f // t
    for s0, n in ((0, 1), (1, 2), (3, 1), (0, 4)):
        c = slice(s0 * fs, (s0 + n) * fs)
        Z, Y, U = fused_fwd(mp, X, A, B, t, ws, shard_begin=s0, shard_count=n)
        assert torch.equal(Y[:, c], full["Y"][:, c]) and torch.equal(U[:, c], full["U"][:, c])
        Zs = torch.empty_like(Z)
        Ys = full["Y"].clone()
        mp.mp_mlp_fwd_shards(X, A, B, Zs, Ys, None, t=t, shard_begin=s0, shard_count=n)
        torch.cuda.synchronize()
        assert torch.equal(Z, Zs), (s0, n)
        # the range's backward: dU, dA columns and dB rows of the range, dX partial
        g = fused_bwd(mp, X, A, B, full["U"], full["Y"], dZ, t, ws, shard_begin=s0, shard_count=n)
        want = {k: torch.empty_like(v) for k, v in g.items()}
        mp.mp_mlp_bwd_shards(X, A, B, full["U"], full["Y"], dZ, want["dX"], want["dA"], want["dB"], want["dU"],
                             t=t, shard_begin=s0, shard_count=n)
        torch.cuda.synchronize()
        assert torch.equal(g["dU"][:, c], want["dU"][:, c]) and torch.equal(g["dA"][:, c], want["dA"][:, c])
        assert torch.equal(g["dB"][c], want["dB"][c]) and torch.equal(g["dX"], want["dX"]), (s0, n)


def test_fused_repeated_calls_share_one_workspace():
    # Calls of different shapes one after another on the same workspace, without syncing in
    # between: each leaves it zeroed for the next.
    mp = _mp()
    shapes = [(2048, 1536, 6144, 4), (300, 256, 1024, 2), (2048, 1536, 6144, 4)]
    ws = mp.mp_mlp_fused_workspace(2048, 1536, 6144, 4)
    outs = []
    for i, (T, h, f, t) in enumerate(shapes):
        inp = synth.mlp_inputs(T, h, f, seed=7400 + (i % 2))
        X, A, B, dZ = (inp[k].cuda() for k in ("X", "A", "B", "dZ"))
        Z, Y, U = _nan(T, h), _nan(T, f), _nan(T, f)
        g = {"dX": _nan(T, h), "dA": _nan(h, f), "dB": _nan(f, h), "dU": _nan(T, f)}
        mp.mp_mlp_fwd_fused(X, A, B, Z, Y, U, t=t, workspace=ws)
        mp.mp_mlp_bwd_fused(X, A, B, U, Y, dZ, g["dX"], g["dA"], g["dB"], g["dU"], t=t, workspace=ws)
        outs.append((inp, Z, g))
    torch.cuda.synchronize()
    assert int(ws.count_nonzero().item()) == 0
    assert torch.equal(outs[0][1], outs[2][1]) and all(torch.equal(outs[0][2][k], outs[2][2][k]) for k in outs[0][2])
    for inp, Z, g in outs[:2]:
        T = inp["X"].shape[0]
        rows = synth.sample_indices(T, 24, seed=7401).numpy()
        _, _, Zr = oracle.mlp_fwd_rows(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), rows)
        assert rel_fro(f64(Z)[rows], Zr) <= Z_REL_FRO
        assert not torch.isnan(g["dA"]).any() and not torch.isnan(g["dX"]).any()


def test_fused_deterministic_across_calls():
    mp = _mp()
    T, h, f, t = 2048, 1920, 7680, 8
    inp = synth.mlp_inputs(T, h, f, seed=7500)
    X, A, B, dZ = (inp[k].cuda() for k in ("X", "A", "B", "dZ"))
    ws = mp.mp_mlp_fused_workspace(T, h, f, t)
    first = None
    for _ in range(3):
        Z, Y, U = fused_fwd(mp, X, A, B, t, ws)
        g = fused_bwd(mp, X, A, B, U, Y, dZ, t, ws)
        cur = [Z, Y, U] + [g[k] for k in ("dX", "dA", "dB", "dU")]
        if first is None:
            first = cur
        else:
            assert all(torch.equal(a, b) for a, b in zip(first, cur))


def test_fused_wait_budget_exhaustion(monkeypatch):
    # With a zero wait budget every wait that does not succeed at once runs out: the dependency
    # flags, the unit hand-out ring and the pipeline barriers. The kernel reports MP_DEV_TIMEOUT,
    # returns, leaves the workspace zeroed and the context usable.
    mp = _mp()
    T, h, f, t = 1024, 1024, 4096, 4
    inp = synth.mlp_inputs(T, h, f, seed=7600)
    X, A, B, dZ = (inp[k].cuda() for k in ("X", "A", "B", "dZ"))
    ws = mp.mp_mlp_fused_workspace(T, h, f, t)
    Z, Y, U = _nan(T, h), _nan(T, f), _nan(T, f)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    monkeypatch.setenv("MPTP_WAIT_BUDGET_NS", "0")
    mp.mp_mlp_fwd_fused(X, A, B, Z, Y, U, t=t, workspace=ws, d_status=st)
    g = {"dX": _nan(T, h), "dA": _nan(h, f), "dB": _nan(f, h), "dU": _nan(T, f)}
    mp.mp_mlp_bwd_fused(X, A, B, U, Y, dZ, g["dX"], g["dA"], g["dB"], g["dU"], t=t, workspace=ws, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) & mp.MP_DEV_TIMEOUT
    assert int(ws.count_nonzero().item()) == 0
    monkeypatch.delenv("MPTP_WAIT_BUDGET_NS")
    Z, Y, U = fused_fwd(mp, X, A, B, t, ws)
    _, _, Zr = oracle.mlp_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]))
    assert rel_fro(f64(Z), Zr) <= Z_REL_FRO


def test_fused_empty_batch():
    mp = _mp()
    h, f, t = 128, 512, 2
    X = torch.empty(0, h, dtype=torch.bfloat16, device="cuda")
    A = synth.normal_bf16((h, f), 0.02, 1).cuda()
    B = synth.normal_bf16((f, h), 0.02, 2).cuda()
    e = torch.empty(0, f, dtype=torch.bfloat16, device="cuda")
    dA, dB = _nan(h, f), _nan(f, h)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    mp.mp_mlp_fwd_fused(X, A, B, torch.empty(0, h, dtype=torch.bfloat16, device="cuda"), e, None, t=t, workspace=ws)
    mp.mp_mlp_bwd_fused(X, A, B, e, e, torch.empty(0, h, dtype=torch.bfloat16, device="cuda"),
                        torch.empty(0, h, dtype=torch.bfloat16, device="cuda"), dA, dB, e, t=t, workspace=ws)
    torch.cuda.synchronize()
    assert int(dA.count_nonzero().item()) == 0 and int(dB.count_nonzero().item()) == 0


def test_fused_beyond_the_schedule_tables():
    # T = 32768, h = 2048, f = 8192: 5120 forward and 5632 backward units, more list positions than a
    # precomputed schedule holds (4096), so the entry points run the separate launches instead (the
    # chain's round-robin order measured 20-40 % slower here). Bitwise against the separate launches
    # (no split-K at this size), the workspace untouched, sampled rows against the oracle.
    mp = _mp()
    T, h, f, t = 32768, 2048, 8192, 4
    inp = synth.mlp_inputs(T, h, f, seed=7700)
    dev = run_mlp_fwd(inp, t)
    ws = mp.mp_mlp_fused_workspace(T, h, f, t)
    Z, Y, U = fused_fwd(mp, dev["X"], dev["A"], dev["B"], t, ws)
    assert torch.equal(Z, dev["Z"]) and torch.equal(Y, dev["Y"]) and torch.equal(U, dev["U"])
    del Y, U
    sep = run_mlp_bwd(dev, inp["dZ"], t)
    g = fused_bwd(mp, dev["X"], dev["A"], dev["B"], dev["U"], dev["Y"], inp["dZ"].cuda(), t, ws)
    for k in ("dU", "dX", "dA", "dB"):
        assert torch.equal(g[k], sep[k]), k
    rows = synth.sample_indices(T, 8, seed=7701).numpy()
    _, _, Zr = oracle.mlp_fwd_rows(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), rows)
    assert rel_fro(f64(Z)[rows], Zr) <= Z_REL_FRO
