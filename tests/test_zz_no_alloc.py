"""mp_vocab_ce_noalloc: the cross-entropy entry point for callers that cannot
allocate device memory (their memory belongs to another pool that forbids
cudaMalloc/cudaFree after start-up), so they cannot pass a workspace. Its
scratch is the library's fixed 4 MiB static device array.

Called through the C ABI (ctypes, raw device pointers) several times in a row:
the same small shape twice with new inputs, then the largest shape the array
holds, then the small shape again. Each result is compared with the
workspace-taking mp_vocab_ce at the per-token loss tolerance used by the other
cross-entropy tests, and sampled tokens with the float64 oracle. Collected last
(file name) so a stop-at-first-failure run has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import LOSS_ABS, f64

pytestmark = pytest.mark.gpu


def _lib():
    import tensor_transformer_layer_gb300 as mp
    return mp, mp.lib()


def _existing(mp, X, E, tgt, v_valid, t):
    T, v_pad = X.shape[0], E.shape[0]
    ws = torch.empty(mp.mp_vocab_ce_workspace_bytes(T, v_pad, t), dtype=torch.uint8, device="cuda")
    loss = torch.empty(T, dtype=torch.float32, device="cuda")
    mp.mp_vocab_ce(X, E, tgt, loss, ws, v_valid=v_valid, t=t)
    torch.cuda.synchronize()
    return loss.cpu().numpy()


def _noalloc(L, X, E, tgt, v_valid, t):
    T, h = X.shape
    v_pad = E.shape[0]
    loss = torch.full((T,), float("nan"), dtype=torch.float32, device="cuda")
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    code = L.mp_vocab_ce_noalloc(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(E.data_ptr()),
                                 ctypes.c_void_p(tgt.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                 T, h, v_pad, v_valid, t, ctypes.c_void_p(status.data_ptr()),
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert code == 0, code
    assert int(status.item()) == 0
    return loss.cpu().numpy()


def test_noalloc_matches_workspace_entry_point_and_oracle():
    mp, L = _lib()
    # A T = 0 call places the static array on this device (it is what a caller whose pool will
    # reserve the rest of HBM makes first); it launches nothing.
    code = L.mp_vocab_ce_noalloc(None, None, None, None, 0, 128, 2048, 2000, 4, None, None)
    assert code == 0, code
    small = dict(T=300, h=128, v_pad=2048, v_valid=2000, t=4)
    large = dict(T=8192, h=1536, v_pad=51200, v_valid=50257, t=8)   # 3.75 MiB of triples
    cases = [dict(small, seed=5101), dict(small, seed=5102), dict(large, seed=5100), dict(small, seed=5103)]
    for c in cases:   # calls in a row on the shared array, which keeps the previous call's triples
        inp = synth.ce_inputs(c["T"], c["h"], c["v_pad"], c["v_valid"], c["seed"])
        X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
        want = _existing(mp, X, E, tgt, c["v_valid"], c["t"])
        got = _noalloc(L, X, E, tgt, c["v_valid"], c["t"])
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got.astype(np.float64) - want))) <= LOSS_ABS, c
        rows = synth.sample_indices(c["T"], 32, seed=c["seed"]).numpy()
        ref = oracle.ce_loss(f64(inp["X"])[rows], f64(inp["E"]), inp["target"].numpy()[rows], c["v_valid"])
        assert float(np.max(np.abs(got[rows].astype(np.float64) - ref))) <= LOSS_ABS, c


def test_noalloc_refuses_problems_beyond_the_array():
    mp, L = _lib()
    # 43,691 tokens: even one vocabulary partition per shard (8 x 3 x T floats) exceeds 4 MiB.
    T, h, v_pad, t = 43691, 64, 51200, 8
    assert 8 * 3 * T * 4 > 4 * 1024 * 1024 >= 8 * 3 * (T - 1) * 4
    X = torch.zeros(T, h, dtype=torch.bfloat16, device="cuda")
    E = torch.zeros(v_pad, h, dtype=torch.bfloat16, device="cuda")
    tgt = torch.zeros(T, dtype=torch.int32, device="cuda")
    loss = torch.zeros(T, dtype=torch.float32, device="cuda")
    code = L.mp_vocab_ce_noalloc(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(E.data_ptr()),
                                 ctypes.c_void_p(tgt.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                 T, h, v_pad, 50257, t, None, None)
    assert code == 8   # MP_ERR_WORKSPACE, nothing launched
