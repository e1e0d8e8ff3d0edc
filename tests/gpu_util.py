"""Helpers for the GPU parity tests: run the library through its binding and
compare against the float64 oracle."""
import numpy as np
import torch

import synth

# Tolerances stated for this workload (bf16 inputs, fp32 accumulation).
Z_REL_FRO = 5e-3
Z_MAX_ABS = 3e-2
GRAD_REL_FRO = 1e-2
LOSS_ABS = 2e-3


def mp():
    import tensor_transformer_layer_gb300 as m
    m.lib()
    return m


def rel_fro(got, want):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    return float(np.linalg.norm(got - want) / max(np.linalg.norm(want), 1e-300))


def max_abs(got, want):
    return float(np.max(np.abs(np.asarray(got, dtype=np.float64) - np.asarray(want, dtype=np.float64))))


def status_tensor():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_mlp_fwd(inp, t, save_u=True):
    m = mp()
    X, A, B = (inp[k].cuda() for k in ("X", "A", "B"))
    T, h = X.shape
    f = A.shape[1]
    Z = torch.empty(T, h, dtype=torch.bfloat16, device="cuda")
    Y = torch.empty(T, f, dtype=torch.bfloat16, device="cuda")
    U = torch.empty(T, f, dtype=torch.bfloat16, device="cuda") if save_u else None
    st = status_tensor()
    m.mp_mlp_fwd(X, A, B, Z, Y, U, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return {"X": X, "A": A, "B": B, "Z": Z, "Y": Y, "U": U}


def run_mlp_bwd(dev, dZ, t):
    m = mp()
    X, A, B, U, Y = dev["X"], dev["A"], dev["B"], dev["U"], dev["Y"]
    T, h = X.shape
    f = A.shape[1]
    dZ = dZ.cuda()
    out = {
        "dX": torch.empty(T, h, dtype=torch.bfloat16, device="cuda"),
        "dA": torch.empty(h, f, dtype=torch.bfloat16, device="cuda"),
        "dB": torch.empty(f, h, dtype=torch.bfloat16, device="cuda"),
        "dU": torch.empty(T, f, dtype=torch.bfloat16, device="cuda"),
    }
    st = status_tensor()
    m.mp_mlp_bwd(X, A, B, U, Y, dZ, out["dX"], out["dA"], out["dB"], out["dU"], t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0, f"device status {int(st.item())}"
    return out


def run_ce(inp, v_valid, t, expect_status=0):
    m = mp()
    X, E, tgt = inp["X"].cuda(), inp["E"].cuda(), inp["target"].cuda()
    T = X.shape[0]
    v_pad = E.shape[0]
    ws = torch.empty(max(m.mp_vocab_ce_workspace_bytes(T, v_pad, t), 16), dtype=torch.uint8, device="cuda")
    loss = torch.empty(T, dtype=torch.float32, device="cuda")
    st = status_tensor()
    m.mp_vocab_ce(X, E, tgt, loss, ws, v_valid=v_valid, t=t, d_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status, f"device status {int(st.item())}"
    return loss.cpu().numpy().astype(np.float64)


def f64(t):
    return synth.to_f64(t)
