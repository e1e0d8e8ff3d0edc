"""GPU parity of the head-parallel causal self-attention block against the float64 oracle.

Tolerance: relative Frobenius 1e-2 on O and out. The path rounds to bf16 four
times (QKV, the probabilities P fed to the P V product, O, out), each about 2^-9
relative, against one rounding for the MLP output."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import f64, mp, rel_fro, status_tensor

pytestmark = pytest.mark.gpu
ATTN_REL_FRO = 1e-2


def _inputs(b, s, h, seed):
    return {
        "X": synth.normal_bf16((b * s, h), 1.0, seed),
        "Wqkv": synth.normal_bf16((h, 3 * h), 0.02, seed + 1),
        "Wo": synth.normal_bf16((h, h), 0.02, seed + 2),
    }


def _run(inp, b, s, heads, t):
    m = mp()
    X, Wqkv, Wo = (inp[k].cuda() for k in ("X", "Wqkv", "Wo"))
    T, h = X.shape
    out = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    QKV = torch.empty(T, 3 * h, dtype=torch.bfloat16, device="cuda")
    O = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    m.mp_attn_fwd(X, Wqkv, Wo, out, QKV, O, b=b, s=s, heads=heads, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return {"out": out.cpu(), "QKV": QKV.cpu(), "O": O.cpu()}


@pytest.mark.parametrize("b,s,h,heads,t", [
    (2, 256, 192, 2, 2),      # d = 96, two query tiles per sequence
    (1, 512, 384, 4, 4),      # d = 96, four tiles (causal skipping and the diagonal)
    (3, 128, 128, 2, 1),      # d = 64, one tile
    (2, 384, 256, 4, 2),      # d = 64
    (8, 1024, 512, 8, 2),     # d = 64, 512 work items (more than three waves)
    (6, 768, 768, 8, 4),      # d = 96, 288 work items of 1..6 key tiles
    (2, 384, 192, 2, 1),      # d = 96, odd tile count: a pair with one query tile
    (1, 128, 192, 2, 1),      # d = 96, a single query tile
])
def test_attn_matches_oracle(b, s, h, heads, t):
    inp = _inputs(b, s, h, seed=10000 + s + h)
    got = _run(inp, b, s, heads, t)
    QKV, O, out = oracle.attn_fwd(f64(inp["X"]), f64(inp["Wqkv"]), f64(inp["Wo"]), heads, b, s)
    errs = {"QKV": rel_fro(f64(got["QKV"]), QKV), "O": rel_fro(f64(got["O"]), O),
            "out": rel_fro(f64(got["out"]), out)}
    assert all(v <= ATTN_REL_FRO for v in errs.values()), errs


def test_attn_zero_queries_average_the_prefix():
    # Wq = 0 -> every score is 0 -> each query averages the values of its causal prefix
    # (compared with the bf16 V the kernel itself produced).
    b, s, h, heads = 1, 256, 192, 2
    inp = _inputs(b, s, h, seed=10100)
    inp["Wqkv"][:, :h] = 0
    got = _run(inp, b, s, heads, 1)
    V = f64(got["QKV"])[:, 2 * h:]
    want = np.cumsum(V, axis=0) / np.arange(1, s + 1)[:, None]
    assert rel_fro(f64(got["O"]), want) <= 5e-3


def test_attn_head_shard_invariance_bitwise():
    b, s, h, heads = 2, 256, 384, 4
    inp = _inputs(b, s, h, seed=10200)
    ref = _run(inp, b, s, heads, 1)
    for t in (2, 4):
        got = _run(inp, b, s, heads, t)
        for k in ("out", "O", "QKV"):
            assert torch.equal(got[k], ref[k]), (t, k)


def test_attn_8p3b_layer_sampled():
    # b = 4 sequences of 1024 tokens, h = 3072, 32 heads of 96, t = 8 shards of 4 heads.
    b, s, h, heads, t = 4, 1024, 3072, 32, 8
    inp = _inputs(b, s, h, seed=10300)
    got = _run(inp, b, s, heads, t)
    rows = np.unique(np.concatenate([synth.sample_indices(s, 24, seed=1).numpy(),
                                     s + synth.sample_indices(s, 8, seed=2).numpy(),
                                     np.array([3 * s + s - 1])]))
    Or, outr = oracle.attn_fwd_rows(f64(inp["X"]), f64(inp["Wqkv"]), f64(inp["Wo"]), heads, b, s, rows)
    errs = {"O": rel_fro(f64(got["O"])[rows], Or), "out": rel_fro(f64(got["out"])[rows], outr)}
    assert all(v <= ATTN_REL_FRO for v in errs.values()), errs
