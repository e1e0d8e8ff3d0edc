"""mp_vocab_ce_noalloc: the cross-entropy entry point for callers that cannot
allocate device memory (their memory belongs to another pool that forbids
cudaMalloc/cudaFree after start-up), so they cannot pass a workspace. Its
scratch is the library's fixed 4 MiB static device array.

Called through the C ABI (ctypes, raw device pointers) twice in a row with
different inputs, and compared with the workspace-taking mp_vocab_ce at the
per-token loss tolerance used by the other cross-entropy tests. Collected last
(file name) so a stop-at-first-failure run has already run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import synth
from gpu_util import LOSS_ABS

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


def test_noalloc_matches_workspace_entry_point_twice():
    mp, L = _lib()
    cases = [
        dict(T=8192, h=1536, v_pad=51200, v_valid=50257, t=8, seed=5100),   # 3.75 MiB of triples
        dict(T=300, h=128, v_pad=2048, v_valid=2000, t=4, seed=5101),       # a different partition count
    ]
    for c in cases:   # two calls in a row on the shared array
        inp = synth.ce_inputs(c["T"], c["h"], c["v_pad"], c["v_valid"], c["seed"])
        X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
        want = _existing(mp, X, E, tgt, c["v_valid"], c["t"])
        got = _noalloc(L, X, E, tgt, c["v_valid"], c["t"])
        assert np.all(np.isfinite(got))
        assert float(np.max(np.abs(got.astype(np.float64) - want))) <= LOSS_ABS


def test_noalloc_refuses_problems_beyond_the_array():
    mp, L = _lib()
    T, h, v_pad, t = 8739, 64, 51200, 8     # 40 partitions x 3 x 8739 floats > 4 MiB
    assert mp.mp_vocab_ce_workspace_bytes(T, v_pad, t) > 4 * 1024 * 1024
    X = torch.zeros(T, h, dtype=torch.bfloat16, device="cuda")
    E = torch.zeros(v_pad, h, dtype=torch.bfloat16, device="cuda")
    tgt = torch.zeros(T, dtype=torch.int32, device="cuda")
    loss = torch.zeros(T, dtype=torch.float32, device="cuda")
    code = L.mp_vocab_ce_noalloc(ctypes.c_void_p(X.data_ptr()), ctypes.c_void_p(E.data_ptr()),
                                 ctypes.c_void_p(tgt.data_ptr()), ctypes.c_void_p(loss.data_ptr()),
                                 T, h, v_pad, 50257, t, None, None)
    assert code == 8   # MP_ERR_WORKSPACE, nothing launched
