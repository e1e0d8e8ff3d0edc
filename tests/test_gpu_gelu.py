"""The kernels' fp32 GeLU and GeLU' (column-parallel and dY epilogues) on a dense
grid of inputs, against the float64 oracle: within half a bf16 spacing of the
exact value plus 2e-6 (the epilogue computes in fp32 and rounds to bf16 once;
its erf approximation is accurate to 1.5e-7)."""
import numpy as np
import pytest
import torch

import oracle
from gpu_util import mp

pytestmark = pytest.mark.gpu


def _bf16_half_ulp(v):
    v = np.abs(np.asarray(v, dtype=np.float64))
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 0.5 * 2.0 ** (e - 7)


def _grid(T):
    # bf16-exact inputs spanning [-8, 8], both signs, dense near 0
    u = torch.linspace(-8.0, 8.0, T).to(torch.bfloat16)
    return u


def test_gelu_epilogue_on_grid():
    m = mp()
    T, h, f = 1024, 64, 256
    u = _grid(T)
    X = torch.zeros(T, h, dtype=torch.bfloat16)
    X[:, 0] = u
    A = torch.zeros(h, f, dtype=torch.bfloat16)
    A[0, :] = 1.0                     # U[r, j] = u_r for every column j
    B = torch.zeros(f, h, dtype=torch.bfloat16)
    Xd, Ad, Bd = X.cuda(), A.cuda(), B.cuda()
    Z = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    U = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    m.mp_mlp_fwd(Xd, Ad, Bd, Z, Y, U, t=4)
    torch.cuda.synchronize()
    uu = u.to(torch.float64).numpy()
    want = oracle.gelu(uu)
    got = Y.cpu().to(torch.float64).numpy()
    assert np.array_equal(U.cpu().to(torch.float64).numpy(), np.repeat(uu[:, None], f, axis=1))
    err = np.abs(got - want[:, None])
    bound = _bf16_half_ulp(want)[:, None] + 2e-6
    assert np.all(err <= bound), float(np.max(err - bound))


def test_gelu_prime_epilogue_on_grid():
    m = mp()
    T, h, f = 1024, 64, 256
    u = _grid(T)
    X = torch.zeros(T, h, dtype=torch.bfloat16)
    A = torch.zeros(h, f, dtype=torch.bfloat16)
    B = torch.zeros(f, h, dtype=torch.bfloat16)
    B[:, 0] = 1.0
    G = torch.zeros(T, h, dtype=torch.bfloat16)
    G[:, 0] = 1.0                     # dY = G B^T = 1 everywhere
    U = u[:, None].repeat(1, f).contiguous()
    Y = torch.zeros(T, f, dtype=torch.bfloat16)
    d = {k: v.cuda() for k, v in (("X", X), ("A", A), ("B", B), ("G", G), ("U", U), ("Y", Y))}
    dX = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    dA = torch.empty(h, f, dtype=torch.bfloat16, device="cuda")
    dB = torch.empty(f, h, dtype=torch.bfloat16, device="cuda")
    dU = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    m.mp_mlp_bwd(d["X"], d["A"], d["B"], d["U"], d["Y"], d["G"], dX, dA, dB, dU, t=4)
    torch.cuda.synchronize()
    want = oracle.gelu_prime(u.to(torch.float64).numpy())
    got = dU.cpu().to(torch.float64).numpy()
    err = np.abs(got - want[:, None])
    bound = _bf16_half_ulp(want)[:, None] + 2e-6
    assert np.all(err <= bound), float(np.max(err - bound))
