"""Seeded synthetic workloads for context-parallel causal attention.

Shapes only and a random-number recipe: this module holds none of the
attention arithmetic, so both the CUDA path's tests and the CPU oracle can
draw their inputs from it. Values are drawn in fp32 from N(0, std^2) with a
torch generator seeded per workload, then rounded to bf16 (the kernels'
input type); the oracle receives the very same bf16 values upcast to fp64.

Layout: q, o, dO are [b, s, hq, d]; k, v are [b, s, hkv, d]; bf16,
contiguous, natural token order.
"""
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    b: int
    s: int
    hq: int
    hkv: int
    d: int
    cp: int
    causal: bool = True
    q_std: float = 1.0
    k_std: float = 1.0
    v_std: float = 1.0
    backward: bool = False
    seed: int = 1000
    # how the oracle checks the full-size case: "all" rows, or a sample
    check_rows: int = 0          # 0 = every row
    check_dkv_heads: int = 0     # KV heads whose full dK/dV are checked (0 = all)
    extra: dict = field(default_factory=dict)

    @property
    def chunk(self) -> int:
        return self.s // (2 * self.cp)

    def fwd_flops(self) -> float:
        """Causal forward FLOPs, 2*b*hq*s^2*d (the two matmuls over the lower
        triangle); twice that without the mask."""
        f = 2.0 * self.b * self.hq * self.s * self.s * self.d
        return f if self.causal else 2.0 * f

    def bwd_flops(self) -> float:
        """Backward counted as 2.5x forward (five matmuls against two)."""
        return 2.5 * self.fwd_flops()


WORKLOADS = {
    w.name: w
    for w in [
        Workload("small_b1_s512_h4_d64_cp2", b=1, s=512, hq=4, hkv=4, d=64, cp=2, backward=True, seed=1000),
        Workload("mha_b2_s4096_h32_d128_cp4", b=2, s=4096, hq=32, hkv=32, d=128, cp=4, seed=1001),
        Workload("gqa_b1_s16384_h64kv8_d128_cp8", b=1, s=16384, hq=64, hkv=8, d=128, cp=8, seed=1002,
                 check_rows=1024),
        Workload("long_b1_s131072_h32kv8_d128_cp16", b=1, s=131072, hq=32, hkv=8, d=128, cp=16, q_std=2.0,
                 k_std=2.0, seed=1003, check_rows=1024),
        Workload("train_b1_s32768_h32kv8_d128_cp8", b=1, s=32768, hq=32, hkv=8, d=128, cp=8, backward=True,
                 seed=1004, check_rows=512, check_dkv_heads=4),
        # half-length training shape: the size the kernels are profiled on
        # (inputs still exceed L2; a launch stays well under a second)
        Workload("train_b1_s16384_h32kv8_d128_cp8", b=1, s=16384, hq=32, hkv=8, d=128, cp=8, backward=True,
                 seed=1005, check_rows=512, check_dkv_heads=2),
    ]
}


def make_inputs(w: Workload, device="cpu", seed=None, with_grad=None):
    """Draw q, k, v (and dO when the workload has a backward) as bf16.

    Draw order is q, k, v, dO from one generator on ``device``.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed if seed is None else seed)
    want_do = w.backward if with_grad is None else with_grad

    def draw(shape, std):
        x = torch.randn(*shape, generator=gen, device=device, dtype=torch.float32)
        if std != 1.0:
            x.mul_(std)
        return x.to(torch.bfloat16)

    out = {
        "q": draw((w.b, w.s, w.hq, w.d), w.q_std),
        "k": draw((w.b, w.s, w.hkv, w.d), w.k_std),
        "v": draw((w.b, w.s, w.hkv, w.d), w.v_std),
    }
    if want_do:
        out["do"] = draw((w.b, w.s, w.hq, w.d), 1.0)
    return out


def sample_rows(w: Workload, n: int, seed: int):
    """n distinct query positions drawn uniformly over [0, s), sorted."""
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(w.s, generator=g)[:n].sort().values
