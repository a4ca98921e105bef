"""Seeded synthetic inputs for the fused AllReduce + residual + RMSNorm epilogue.

Shared by the tests, the smoke check and the bench: it draws the n rank
partials, the residual and the RMSNorm weight, and holds none of the
epilogue's arithmetic (no sum, no residual add, no normalisation).

Tensors are bf16.  Values are drawn in fp32 from N(mean, std) and rounded to
bf16 by torch's own conversion; outliers, where asked for, multiply a drawn
value by ``outlier_scale`` before that rounding.  Each tensor has its own
stream, keyed by (seed, stream id): partial k -> k, residual -> 100,
weight -> 101.  Two generators exist:

  * ``backend="numpy"``: numpy PCG64 on the host; identical on every machine.
  * ``backend="torch"``: torch's Philox generator on the target device; used
    for the large workloads, whose host generation would take too long.

The pages publish no dataset; these shapes and distributions stand in for
their TP4/TP8 decode and prefill workloads (token count m, hidden size H,
n ranks).
"""
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np
import torch

PARTIAL_STREAM = 0
RESIDUAL_STREAM = 100
WEIGHT_STREAM = 101


@dataclass(frozen=True)
class Workload:
    """One synthetic workload: n partials of [m, H] bf16 per m in ``ms``."""
    name: str
    n: int
    H: int
    ms: Sequence[int]
    p_std: float
    res_std: float
    w_mean: float = 1.0
    w_std: float = 0.1
    eps: float = 1e-6
    outlier_frac: float = 0.0
    outlier_scale: float = 100.0
    modes: Sequence[str] = field(default_factory=lambda: ("auto",))
    seed: int = 0


# The five workloads, with the pages' decode and prefill shapes.
TINY = Workload("tiny", n=2, H=1024, ms=(4,), p_std=1.0, res_std=1.0,
                modes=("one_stage",))
DECODE = Workload("decode", n=8, H=7168, ms=(1, 2, 4, 8, 16), p_std=0.5,
                  res_std=1.0, modes=("one_stage",))
TWO_STAGE = Workload("two_stage", n=4, H=7168, ms=(32, 64, 256, 1024, 2048),
                     p_std=0.5, res_std=1.0, modes=("two_stage",))
PREFILL = Workload("prefill", n=8, H=6144, ms=(8192,), p_std=0.5, res_std=2.0,
                   eps=1e-5, modes=("one_stage", "two_stage"))
SWEEP_MS = tuple(2 ** k for k in range(15))  # 1 .. 16384
SWEEP = [Workload(f"sweep_n{n}_h{h}", n=n, H=h, ms=SWEEP_MS, p_std=0.5,
                  res_std=1.0, outlier_frac=1e-3, modes=("auto",))
         for n in (4, 8) for h in (4096, 8192)]

WORKLOADS = {w.name: w for w in [TINY, DECODE, TWO_STAGE, PREFILL, *SWEEP]}


def _numpy_normal(shape, mean, std, seed, stream, outlier_frac, outlier_scale):
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, stream])))
    x = rng.standard_normal(size=shape, dtype=np.float32) * np.float32(std) + np.float32(mean)
    if outlier_frac > 0.0:
        mask = rng.random(size=shape) < outlier_frac
        x[mask] *= np.float32(outlier_scale)
    return torch.from_numpy(x).to(torch.bfloat16)


def _torch_normal(shape, mean, std, seed, stream, outlier_frac, outlier_scale, device):
    g = torch.Generator(device=device)
    g.manual_seed((seed * 1_000_003 + stream) & 0x7FFF_FFFF_FFFF_FFFF)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    x.mul_(std).add_(mean)
    if outlier_frac > 0.0:
        mask = torch.rand(shape, generator=g, device=device) < outlier_frac
        x[mask] *= outlier_scale
    return x.to(torch.bfloat16)


def normal_bf16(shape, mean, std, seed, stream, outlier_frac=0.0,
                outlier_scale=100.0, backend="numpy", device="cpu"):
    """One bf16 tensor of N(mean, std) draws (plus optional outliers)."""
    if backend == "numpy":
        t = _numpy_normal(tuple(shape), mean, std, seed, stream, outlier_frac, outlier_scale)
        return t.to(device)
    if backend == "torch":
        return _torch_normal(tuple(shape), mean, std, seed, stream, outlier_frac,
                             outlier_scale, device)
    raise ValueError(f"unknown backend {backend!r}")


@dataclass
class Inputs:
    partials: List[torch.Tensor]   # n x [m, H] bf16, rank order
    residual: torch.Tensor         # [m, H] bf16
    weight: torch.Tensor           # [H] bf16
    eps: float


def make_inputs(w: Workload, m: int, backend: str = "numpy", device="cpu",
                seed: Optional[int] = None) -> Inputs:
    """The inputs of workload ``w`` at token count ``m``."""
    s = w.seed if seed is None else seed
    parts = [normal_bf16((m, w.H), 0.0, w.p_std, s, PARTIAL_STREAM + k,
                         w.outlier_frac, w.outlier_scale, backend, device)
             for k in range(w.n)]
    res = normal_bf16((m, w.H), 0.0, w.res_std, s, RESIDUAL_STREAM,
                      backend=backend, device=device)
    wt = normal_bf16((w.H,), w.w_mean, w.w_std, s, WEIGHT_STREAM,
                     backend=backend, device=device)
    return Inputs(parts, res, wt, w.eps)


def bits(t: torch.Tensor) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 tensor, as a host numpy uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    """A bf16 tensor from raw 16-bit patterns."""
    arr = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(arr.view(np.int16).copy()).view(torch.bfloat16).to(device)
