"""GPU parity of the vocab-parallel input embedding: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synth
from gpu_util import mp, status_tensor

pytestmark = pytest.mark.gpu


def _run(ids, E, v_valid, t, expect_status=0):
    m = mp()
    out = torch.full((ids.shape[0], E.shape[1]), 3.0, dtype=torch.bfloat16, device="cuda")
    st = status_tensor()
    m.mp_vocab_embed(ids.cuda(), E.cuda(), out, v_valid=v_valid, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    return out.cpu()


@pytest.mark.parametrize("T,h,v_pad,v_valid,t", [
    (300, 128, 2048, 2000, 2),
    (8192, 1536, 51200, 50257, 8),      # the 1.2B-model vocabulary and batch
    (1, 64, 1024, 1024, 1),
    (1000, 3072, 51200, 50257, 4),
])
def test_embed_bit_exact(T, h, v_pad, v_valid, t):
    inp = synth.ce_inputs(T, h, v_pad, v_valid, seed=9000 + T)     # targets double as token ids
    got = _run(inp["target"], inp["E"], v_valid, t)
    want = oracle.embed_sharded(inp["target"].numpy(), synth.to_f64(inp["E"]), v_valid, t)
    assert np.array_equal(synth.to_f64(got), want)


def test_embed_invalid_ids_zero():
    m = mp()
    inp = synth.ce_inputs(64, 64, 1024, 1000, seed=9100)
    ids = inp["target"].clone()
    ids[[3, 10, 20]] = torch.tensor([1000, 1023, -5], dtype=torch.int32)
    got = _run(ids, inp["E"], 1000, 4, expect_status=m.MP_DEV_TARGET_RANGE)
    want = oracle.embed_sharded(ids.numpy(), synth.to_f64(inp["E"]), 1000, 4)
    assert np.array_equal(synth.to_f64(got), want)
    assert torch.count_nonzero(got[[3, 10, 20]]).item() == 0
