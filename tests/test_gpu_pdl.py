"""Programmatic dependent launch between the kernels of a step: each kernel may start while
its predecessor in the stream finishes and waits for it before touching global memory. The
results must not depend on it (bitwise equal with MPTP_PDL=0), and a step captured into a
CUDA graph (where the dependencies become programmatic edges) must replay to the eager
result, with the MLP as six launches or as one launch per direction."""
import os

import pytest
import torch

import synth
from gpu_util import mp, status_tensor

pytestmark = pytest.mark.gpu


class _Env:
    def __init__(self, name, value):
        self.name, self.value, self.old = name, value, None

    def __enter__(self):
        self.old = os.environ.get(self.name)
        os.environ[self.name] = self.value

    def __exit__(self, *exc):
        if self.old is None:
            os.environ.pop(self.name, None)
        else:
            os.environ[self.name] = self.old


def _buffers(T, h, f, Tc, hc, v_pad, v_valid, t, seed):
    mi = synth.mlp_inputs(T, h, f, seed=seed)
    ci = synth.ce_inputs(Tc, hc, v_pad, v_valid, seed=seed + 1)
    d = {k: mi[k].cuda() for k in ("X", "A", "B", "dZ")}
    d.update(Xc=ci["X"].cuda(), E=ci["E"].cuda(), target=ci["target"].cuda())
    e = lambda *s, dt=torch.bfloat16: torch.empty(*s, dtype=dt, device="cuda")
    d.update(Z=e(T, h), Y=e(T, f), U=e(T, f), dX=e(T, h), dA=e(h, f), dB=e(f, h), dU=e(T, f),
             loss=e(Tc, dt=torch.float32))
    d["ws"] = e(max(mp().mp_vocab_ce_workspace_bytes(Tc, v_pad, t), 16), dt=torch.uint8)
    return d


def _step(d, t, v_valid, st):
    m = mp()
    m.mp_mlp_fwd(d["X"], d["A"], d["B"], d["Z"], d["Y"], d["U"], t=t, d_status=st)
    m.mp_mlp_bwd(d["X"], d["A"], d["B"], d["U"], d["Y"], d["dZ"], d["dX"], d["dA"], d["dB"], d["dU"], t=t,
                 d_status=st)
    m.mp_vocab_ce(d["Xc"], d["E"], d["target"], d["loss"], d["ws"], v_valid=v_valid, t=t, d_status=st)


OUTS = ("Z", "Y", "U", "dX", "dA", "dB", "dU", "loss")
SHAPE = dict(T=640, h=256, f=1024, Tc=700, hc=192, v_pad=2048, v_valid=2000, t=4)


def test_pdl_bitwise_equals_stream_order():
    d = _buffers(**SHAPE, seed=13000)
    res = {}
    for mode in ("1", "0"):
        st = status_tensor()
        with _Env("MPTP_PDL", mode):
            for _ in range(2):  # back to back, so the second step's kernels chain onto the first's
                _step(d, SHAPE["t"], SHAPE["v_valid"], st)
            torch.cuda.synchronize()
        assert int(st.item()) == 0
        res[mode] = {k: d[k].clone() for k in OUTS}
    for k in OUTS:
        assert torch.equal(res["1"][k], res["0"][k]), k


def test_pdl_step_in_cuda_graph():
    d = _buffers(**SHAPE, seed=13100)
    st = status_tensor()
    with _Env("MPTP_PDL", "1"):
        _step(d, SHAPE["t"], SHAPE["v_valid"], st)
        torch.cuda.synchronize()
        want = {k: d[k].clone() for k in OUTS}
        for k in OUTS:
            d[k].zero_()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                _step(d, SHAPE["t"], SHAPE["v_valid"], st)
        for _ in range(2):
            graph.replay()
        torch.cuda.synchronize()
    assert int(st.item()) == 0
    for k in OUTS:
        assert torch.equal(d[k], want[k]), k


def test_pdl_attention_block_bitwise():
    m = mp()
    b, s, h, heads, t = 2, 512, 384, 4, 2
    T = b * s
    x = synth.normal_bf16((T, h), 1.0, 13200).cuda()
    wq = synth.normal_bf16((h, 3 * h), 0.02, 13201).cuda()
    wo = synth.normal_bf16((h, h), 0.02, 13202).cuda()
    res = {}
    for mode in ("1", "0"):
        e = lambda *sh: torch.empty(*sh, dtype=torch.bfloat16, device="cuda")
        out, qkv, o = e(T, h), e(T, 3 * h), e(T, h)
        st = status_tensor()
        with _Env("MPTP_PDL", mode):
            m.mp_attn_fwd(x, wq, wo, out, qkv, o, b=b, s=s, heads=heads, t=t, d_status=st)
            torch.cuda.synchronize()
        assert int(st.item()) == 0
        res[mode] = (qkv, o, out)
    for a, c in zip(res["1"], res["0"]):
        assert torch.equal(a, c)


def _fused_step(d, t, v_valid, st):
    m = mp()
    m.mp_mlp_fwd_fused(d["X"], d["A"], d["B"], d["Z"], d["Y"], d["U"], t=t, workspace=d["mws"], d_status=st)
    m.mp_mlp_bwd_fused(d["X"], d["A"], d["B"], d["U"], d["Y"], d["dZ"], d["dX"], d["dA"], d["dB"], d["dU"], t=t,
                       workspace=d["mws"], d_status=st)
    m.mp_vocab_ce(d["Xc"], d["E"], d["target"], d["loss"], d["ws"], v_valid=v_valid, t=t, d_status=st)


@pytest.mark.parametrize("T,h,f", [(640, 256, 1024), (2048, 1536, 6144)])
def test_fused_step_in_cuda_graph(T, h, f):
    # The bench's step (each MLP direction in one launch, then the fused loss) captured into a CUDA
    # graph: the one-launch kernels' workspace is returned to zeros inside each launch, so every
    # replay starts from a clean workspace and reproduces the eager step bit for bit.
    shape = dict(SHAPE, T=T, h=h, f=f)
    d = _buffers(**shape, seed=13300)
    d["mws"] = mp().mp_mlp_fused_workspace(T, h, f, shape["t"])
    st = status_tensor()
    with _Env("MPTP_PDL", "1"):
        _fused_step(d, shape["t"], shape["v_valid"], st)
        torch.cuda.synchronize()
        want = {k: d[k].clone() for k in OUTS}
        for k in OUTS:
            d[k].zero_()
        torch.cuda.synchronize()
        s = torch.cuda.Stream()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.stream(s):
            with torch.cuda.graph(graph, stream=s):
                _fused_step(d, shape["t"], shape["v_valid"], st)
        for _ in range(3):
            graph.replay()
        torch.cuda.synchronize()
    assert int(st.item()) == 0
    assert int(d["mws"].count_nonzero().item()) == 0
    for k in OUTS:
        assert torch.equal(d[k], want[k]), k
