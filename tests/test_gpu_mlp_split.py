"""GPU parity of the split-K row-parallel GEMMs (K2, and K4 in the serial backward schedule):
shapes whose output tiles do not fill the chip run with several CTA pairs per tile, each over
a part of the shard-ordered K range, and the fp32 partials summed on chip in ascending order.
Compared with the float64 oracle (the unsplit definition) at the stated tolerances, and run
twice for determinism; the serial backward (K4 split) is also compared with the side-by-side
schedule (K4 on one pair per tile)."""
import os

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import (GRAD_REL_FRO, Z_MAX_ABS, Z_REL_FRO, f64, max_abs, rel_fro, run_mlp_bwd, run_mlp_fwd)

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,h,f,t", [
    (300, 192, 3072, 4),     # ragged T, N = h narrower than one tile; 48 K blocks over the pairs
    (256, 768, 3072, 2),     # the tiny workload
    (513, 320, 2560, 5),     # ragged T and N; shards of 512 columns
    (300, 192, 2112, 3),     # 33 K blocks: the two pairs run 16 and 17
])
def test_split_forward_matches_oracle(T, h, f, t):
    inp = synth.mlp_inputs(T, h, f, 8000 + T, with_grad=False)
    dev = run_mlp_fwd(inp, t)
    _, _, Z = oracle.mlp_fwd(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]))
    Zg = f64(dev["Z"])
    assert rel_fro(Zg, Z) <= Z_REL_FRO and max_abs(Zg, Z) <= Z_MAX_ABS, (rel_fro(Zg, Z), max_abs(Zg, Z))
    again = run_mlp_fwd(inp, t)
    assert torch.equal(again["Z"], dev["Z"])


def test_split_forward_small_layer_sampled():
    # T = 2048, h = 3072, f = 12288, t = 8: 96 output tiles of the row-parallel GEMM (1.26 rounds
    # on 76 pairs), split over the two pairs of 36 clusters.
    T, h, f, t = 2048, 3072, 12288, 8
    inp = synth.mlp_inputs(T, h, f, 8100, with_grad=False)
    dev = run_mlp_fwd(inp, t)
    rows = synth.sample_indices(T, 96, seed=31).numpy()
    _, _, Zr = oracle.mlp_fwd_rows(f64(inp["X"]), f64(inp["A"]), f64(inp["B"]), rows)
    Zg = f64(dev["Z"])[rows]
    assert rel_fro(Zg, Zr) <= Z_REL_FRO and max_abs(Zg, Zr) <= Z_MAX_ABS


@pytest.mark.parametrize("T,h,f,t", [
    (300, 192, 3072, 4),
    (2048, 3072, 12288, 8),
])
def test_split_backward_serial_schedule(T, h, f, t, monkeypatch):
    inp = synth.mlp_inputs(T, h, f, 8200 + T)
    dev = run_mlp_fwd(inp, t)
    monkeypatch.setenv("MPTP_BWD_SCHEDULE", "serial")
    g = run_mlp_bwd(dev, inp["dZ"], t)
    g2 = run_mlp_bwd(dev, inp["dZ"], t)
    assert torch.equal(g["dX"], g2["dX"])
    monkeypatch.setenv("MPTP_BWD_SCHEDULE", "overlap")
    go = run_mlp_bwd(dev, inp["dZ"], t)
    # dA, dB, dU: the same kernels either way; dX: split K4 against one pair per tile
    for k in ("dA", "dB", "dU"):
        assert torch.equal(g[k], go[k]), k
    assert rel_fro(f64(g["dX"]), f64(go["dX"])) <= 2e-3
    X, A, B, G = (f64(inp[k]) for k in ("X", "A", "B", "dZ"))
    rows = synth.sample_indices(T, 96, seed=32).numpy()
    cols = synth.sample_indices(f, 32, seed=33).numpy()
    brows = synth.sample_indices(f, 32, seed=34).numpy()
    s = oracle.mlp_bwd_sampled(X, A, B, G, rows, cols, brows)
    assert rel_fro(f64(g["dX"])[rows], s["dX_rows"]) <= GRAD_REL_FRO
