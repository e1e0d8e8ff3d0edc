"""Seeded synthetic inputs shared by the tests, the bench and the smoke check.

This module draws random numbers and rounds them to bf16. It holds none of the
method's arithmetic: no GeLU, no matrix product, no softmax. Both the CUDA path
and the CPU oracle receive the *same* bf16 values (the oracle widens them to
float64), so parity compares the two implementations and not two input sets.

Distributions follow the Megatron-LM layer setup (Shoeybi et al. 2019, Table 1
shapes; weight init N(0, 0.02) read as a standard deviation of 0.02):

* activations X and upstream gradients dZ ~ N(0, 1);
* MLP weights A [h, f] and B [f, h] ~ N(0, 0.02);
* (tied) embedding E [v_pad, h] ~ N(0, 0.02), all rows including padding rows;
* targets uniform integers in [0, v_valid).

Seeds: a workload with base seed ``s`` draws X from s+0, A from s+1, B from
s+2, dZ from s+3, E from s+4 and the targets from s+5, each from its own
``torch.Generator`` on the CPU, so any tensor can be regenerated alone.
"""
from __future__ import annotations

import torch

OFF_X, OFF_A, OFF_B, OFF_DZ, OFF_E, OFF_TGT = 0, 1, 2, 3, 4, 5


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, std: float, seed: int) -> torch.Tensor:
    """N(0, std^2) drawn in fp32 on the CPU, rounded to bf16 (round-to-nearest-even)."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def targets_int32(T: int, v_valid: int, seed: int) -> torch.Tensor:
    """Uniform token ids in [0, v_valid), int32."""
    return torch.randint(0, int(v_valid), (int(T),), generator=_gen(seed), dtype=torch.int64).to(torch.int32)


def mlp_inputs(T: int, h: int, f: int, seed: int, with_grad: bool = True) -> dict:
    """X [T,h], A [h,f], B [f,h] (and dZ [T,h]) as CPU bf16 tensors."""
    d = {
        "X": normal_bf16((T, h), 1.0, seed + OFF_X),
        "A": normal_bf16((h, f), 0.02, seed + OFF_A),
        "B": normal_bf16((f, h), 0.02, seed + OFF_B),
    }
    if with_grad:
        d["dZ"] = normal_bf16((T, h), 1.0, seed + OFF_DZ)
    return d


def ce_inputs(T: int, h: int, v_pad: int, v_valid: int, seed: int) -> dict:
    """X [T,h], E [v_pad,h] (CPU bf16) and targets [T] (int32) in [0, v_valid)."""
    return {
        "X": normal_bf16((T, h), 1.0, seed + OFF_X),
        "E": normal_bf16((v_pad, h), 0.02, seed + OFF_E),
        "target": targets_int32(T, v_valid, seed + OFF_TGT),
    }


def sample_indices(n: int, k: int, seed: int) -> torch.Tensor:
    """k distinct sorted indices in [0, n) (all of them if k >= n); always includes n-1 (a ragged tail)."""
    if k >= n:
        return torch.arange(n)
    idx = torch.randperm(n, generator=_gen(seed))[: k - 1]
    idx = torch.unique(torch.cat([idx, torch.tensor([n - 1])]))
    return idx


def to_f64(t: torch.Tensor):
    """Widen a bf16/float tensor to a float64 numpy array (exact for bf16)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


# Workload definitions (the Megatron-LM layer shapes). Base seeds 1000+k.
WORKLOADS = {
    "mlp_tiny": dict(T=256, h=768, f=3072, t=2, seed=1000),
    "mlp_1p2b": dict(T=8192, h=1536, f=6144, t=(2, 4), seed=1001),
    "ce_1p2b": dict(T=8192, h=1536, v_pad=51200, v_valid=50257, t=8, seed=1002),
    "mlp_8p3b": dict(T=4096, h=3072, f=12288, t=8, seed=1003),
    "ce_8p3b": dict(T=4096, h=3072, v_pad=51200, v_valid=50257, t=8, seed=1006),
    "sweep": dict(h=(1536, 1920, 2304, 3072), T=(2048, 8192), t=(1, 2, 4, 8), v_pad=51200, v_valid=50257, seed=1004),
}
