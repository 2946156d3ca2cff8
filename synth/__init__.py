"""Seeded synthetic layers for the GPTQ per-layer workloads.

This module is the only code shared by the CUDA path's tests/benchmarks and the
CPU oracle. It draws random numbers and shapes them into weight matrices and
calibration activations; it holds none of the quantization method's arithmetic
(no Hessian, no factorisation, no quantizer).

The shapes and distributions follow the workloads the GPTQ pages describe: a
transformer linear layer's input X is a stack of calibration token vectors
(GPTQ guide page, "How it works": 128 random 2048-token segments, n ~ 262k), and
its weight W is (out, in). The calibration corpus itself is not available, so
the activations are synthetic stand-ins with heavy-tailed per-channel scales,
outlier channels and dead (always-zero) channels.

Every tensor is produced by ``torch`` generators seeded from ``seed``; the same
call on the same device returns the same bits. Large activations are generated
directly on the device they are used on; the oracle receives host copies of
exactly those bits.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Iterator, List, Optional, Sequence

import torch


@dataclasses.dataclass(frozen=True)
class XSpec:
    """Recipe for one calibration-activation matrix X of shape (n, d)."""
    n: int
    d: int
    kind: str                 # 'gauss' | 'scaled' | 'swiglu' | 'correlated' | 'hadamard'
    dtype: str = "bf16"       # 'bf16' | 'f32'
    lognormal_sigma: float = 1.0
    n_outliers: int = 0
    outlier_factor: float = 1.0
    dead_frac: float = 0.0
    segment: int = 2048       # tokens per calibration segment (streaming batch)


@dataclasses.dataclass(frozen=True)
class WSpec:
    """Recipe for one weight matrix W of shape (out, in), entries ~ N(0, std^2)."""
    name: str
    out: int
    inp: int
    std: float


@dataclasses.dataclass(frozen=True)
class QSpec:
    """Quantizer recipe: bit width, group size (0 = one scale per row), symmetry."""
    bits: int
    group: int
    sym: bool
    act_order: bool = False
    damp: float = 0.01


@dataclasses.dataclass(frozen=True)
class LayerSpec:
    """One layer pass: the weights sharing one calibration input, and the quantizer."""
    x: XSpec
    weights: Sequence[WSpec]
    q: QSpec


@dataclasses.dataclass(frozen=True)
class Workload:
    """A named workload: one or more layer passes (several bit widths for a sweep)."""
    name: str
    layers: Sequence[LayerSpec]
    bits_sweep: Sequence[int] = ()


def _scaled(n, d, **kw):
    return XSpec(n=n, d=d, kind="scaled", **kw)


def workload(cfg: int) -> Workload:
    """The five workload recipes, by index.

    0  tiny layer: W 128x256 ~ N(0, 0.1^2), X 512x256 fp32 ~ N(0,1); 4-bit symmetric,
       one scale per row, no groups, no act_order.
    1  OPT-125m-shaped layer pair sharing one X: W 768x768 and 3072x768 ~ N(0, 0.02^2);
       X 8192x768 bf16 with lognormal(0,1) channel scales, 8 outlier channels x20 and
       2% dead channels; 4-bit asymmetric min/max + zero-point, group 128.
    2  Llama-7B-shaped attention projection: W 4096x4096 ~ N(0, 0.02^2); X 262144x4096
       bf16 (128 segments x 2048 tokens), lognormal scales, 16 outliers x50; 4-bit
       symmetric, group 128.
    3  MLP down projection: W 4096x14336 ~ N(0, 0.015^2); X 262144x14336 bf16 =
       SiLU(a)*b with a, b ~ N(0,1); 3-bit symmetric, group 128, act_order.
    4  Llama-3-8B-shaped decoder block: q 4096x4096, k/v 1024x4096, o 4096x4096,
       gate/up 14336x4096, down 4096x14336 ~ N(0, 0.02^2); q/k/v share one X, gate/up
       share one X; all X are 262144-token bf16 with outlier channels; bits 2, 3, 4,
       symmetric, group 128.
    """
    if cfg == 0:
        x = XSpec(n=512, d=256, kind="gauss", dtype="f32", segment=512)
        return Workload("tiny-128x256-x512-f32-4b-sym-row",
                        [LayerSpec(x, [WSpec("w", 128, 256, 0.1)], QSpec(4, 0, True))])
    if cfg == 1:
        x = _scaled(8192, 768, n_outliers=8, outlier_factor=20.0, dead_frac=0.02)
        return Workload("opt125m-pair-768x768+3072x768-x8192-4b-asym-g128",
                        [LayerSpec(x, [WSpec("w768", 768, 768, 0.02), WSpec("w3072", 3072, 768, 0.02)],
                                   QSpec(4, 128, False))])
    if cfg == 2:
        x = _scaled(262144, 4096, n_outliers=16, outlier_factor=50.0)
        return Workload("llama7b-attn-4096x4096-x262144-4b-sym-g128",
                        [LayerSpec(x, [WSpec("w", 4096, 4096, 0.02)], QSpec(4, 128, True))])
    if cfg == 3:
        x = XSpec(n=262144, d=14336, kind="swiglu")
        return Workload("mlp-down-4096x14336-x262144-3b-sym-g128-actorder",
                        [LayerSpec(x, [WSpec("w", 4096, 14336, 0.015)], QSpec(3, 128, True, act_order=True))])
    if cfg == 4:
        xa = _scaled(262144, 4096, n_outliers=16, outlier_factor=50.0)
        xd = XSpec(n=262144, d=14336, kind="swiglu")
        layers = []
        for bits in (2, 3, 4):
            q = QSpec(bits, 128, True)
            layers += [
                LayerSpec(xa, [WSpec("q_proj", 4096, 4096, 0.02), WSpec("k_proj", 1024, 4096, 0.02),
                               WSpec("v_proj", 1024, 4096, 0.02)], q),
                LayerSpec(xa, [WSpec("o_proj", 4096, 4096, 0.02)], q),
                LayerSpec(xa, [WSpec("gate_proj", 14336, 4096, 0.02), WSpec("up_proj", 14336, 4096, 0.02)], q),
                LayerSpec(xd, [WSpec("down_proj", 4096, 14336, 0.02)], q),
            ]
        return Workload("llama3-8b-block-7-linears-x262144-sym-g128-bits2,3,4", layers, bits_sweep=(2, 3, 4))
    raise ValueError(f"unknown workload {cfg}")


# ----------------------------------------------------------------------------------------
# generators
# ----------------------------------------------------------------------------------------

def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def make_weight(out: int, inp: int, std: float, seed: int, device="cpu") -> torch.Tensor:
    """W ~ N(0, std^2), fp32, shape (out, inp)."""
    g = _gen(seed, device)
    return (torch.randn(out, inp, generator=g, device=device, dtype=torch.float32) * std).contiguous()


def channel_scales(spec: XSpec, seed: int) -> torch.Tensor:
    """Per-channel scales s (fp32, CPU): lognormal, outliers multiplied, dead channels 0.

    Outlier and dead channels are picked by one seeded permutation (dead first, then
    outliers), so they never coincide.
    """
    g = _gen(seed, "cpu")
    s = torch.exp(torch.randn(spec.d, generator=g, dtype=torch.float64) * spec.lognormal_sigma)
    order = torch.randperm(spec.d, generator=g)
    n_dead = int(round(spec.dead_frac * spec.d))
    dead = order[:n_dead]
    out = order[n_dead:n_dead + spec.n_outliers]
    s[out] *= spec.outlier_factor
    s[dead] = 0.0
    return s.to(torch.float32)


def dead_channels(spec: XSpec, seed: int) -> torch.Tensor:
    """Indices of the channels `channel_scales` sets to exactly zero."""
    g = _gen(seed, "cpu")
    torch.randn(spec.d, generator=g, dtype=torch.float64)
    order = torch.randperm(spec.d, generator=g)
    return order[: int(round(spec.dead_frac * spec.d))].sort().values


def _hadamard(n: int) -> torch.Tensor:
    h = torch.ones(1, 1, dtype=torch.float32)
    while h.shape[0] < n:
        h = torch.cat([torch.cat([h, h], 1), torch.cat([h, -h], 1)], 0)
    return h


def make_x_rows(spec: XSpec, seed: int, row0: int, rows: int, device="cpu") -> torch.Tensor:
    """Rows [row0, row0+rows) of X (in spec.dtype), generated segment by segment.

    Each `spec.segment`-token segment has its own generator seeded from (seed, segment
    index), so any row range can be produced without generating the rows before it.
    """
    dt = torch.bfloat16 if spec.dtype == "bf16" else torch.float32
    if spec.kind == "hadamard":
        m = 1 << max(0, (max(spec.n, spec.d) - 1).bit_length())
        h = _hadamard(m)[: spec.n, : spec.d]
        return h[row0: row0 + rows].to(dt).to(device).contiguous()
    out = torch.empty(rows, spec.d, dtype=dt, device=device)
    s = channel_scales(spec, seed).to(device) if spec.kind == "scaled" else None
    A = None
    if spec.kind == "correlated":
        ga = _gen(seed * 7919 + 17, "cpu")
        A = (torch.randn(spec.d, spec.d, generator=ga, dtype=torch.float32) / math.sqrt(spec.d)).to(device)
    seg = spec.segment
    r = row0
    while r < row0 + rows:
        si = r // seg
        s0 = si * seg
        take = min(s0 + seg, row0 + rows, spec.n) - r
        if take <= 0:
            break
        g = _gen(seed * 1_000_003 + si, device)
        seg_rows = min(seg, spec.n - s0)
        if spec.kind in ("gauss", "scaled", "correlated"):
            z = torch.randn(seg_rows, spec.d, generator=g, device=device, dtype=torch.float32)
            if spec.kind == "scaled":
                z = z * s
            elif spec.kind == "correlated":
                z = z @ A
        elif spec.kind == "swiglu":
            a = torch.randn(seg_rows, spec.d, generator=g, device=device, dtype=torch.float32)
            b = torch.randn(seg_rows, spec.d, generator=g, device=device, dtype=torch.float32)
            z = torch.nn.functional.silu(a) * b
            del a, b
        else:
            raise ValueError(spec.kind)
        out[r - row0: r - row0 + take] = z[r - s0: r - s0 + take].to(dt)
        del z
        r += take
    return out


def make_x(spec: XSpec, seed: int, device="cpu") -> torch.Tensor:
    """The whole X (n, d) on `device`."""
    return make_x_rows(spec, seed, 0, spec.n, device)


def iter_segments(spec: XSpec, seed: int, device="cpu", rows: Optional[int] = None) -> Iterator[torch.Tensor]:
    """X in consecutive `rows`-token batches (default one calibration segment each)."""
    step = rows or spec.segment
    for r in range(0, spec.n, step):
        yield make_x_rows(spec, seed, r, min(step, spec.n - r), device)


def seeds(cfg: int) -> dict:
    """Base seeds for a workload: X seed, and one W seed per weight name."""
    return {"x": 1000 + cfg, "w": 2000 + cfg}


def weight_seed(cfg: int, name: str) -> int:
    return seeds(cfg)["w"] * 131 + sum(ord(c) * (i + 1) for i, c in enumerate(name))


def x_seed(cfg: int, spec: XSpec) -> int:
    return seeds(cfg)["x"] * 7 + spec.d


def to_numpy_f64(t: torch.Tensor):
    """Exact fp64 host copy of a tensor's values (bf16/fp32 are exactly representable)."""
    return t.detach().to("cpu").to(torch.float64).numpy()


__all__ = [
    "XSpec", "WSpec", "QSpec", "LayerSpec", "Workload", "workload", "make_weight", "make_x",
    "make_x_rows", "iter_segments", "channel_scales", "dead_channels", "seeds", "weight_seed",
    "x_seed", "to_numpy_f64",
]


# ------------------------------------------------------------ layer-wise MLP workloads

@dataclasses.dataclass(frozen=True)
class MLPSpec:
    """A synthetic MLP for the layer-wise pipeline: inputs X (n, dims[0]) and weights
    W_i (dims[i+1], dims[i]) ~ N(0, 1/dims[i]); hidden layers relu, last layer linear."""
    name: str
    dims: Sequence[int]
    x: XSpec
    bits: int
    group: int
    sym: bool
    act_order: bool = False
    damp: float = 0.01


def mlp_workload(name: str) -> MLPSpec:
    """'toy': the guide page's simulation scale (three 256-wide hidden layers, 512
    calibration inputs; the 12-feature input widened to 128 so every width is a multiple
    of 64), 3-bit symmetric per-row. 'mlp4096': three 4096-wide layers on 8192 tokens,
    4-bit symmetric, group 128."""
    if name == "toy":
        return MLPSpec("toy-128-256-256-256-x512-3b-sym-row", (128, 256, 256, 256),
                       XSpec(n=512, d=128, kind="correlated", dtype="bf16", segment=512), 3, 0, True)
    if name == "mlp4096":
        return MLPSpec("mlp-4096x3-x8192-4b-sym-g128", (4096, 4096, 4096, 4096),
                       XSpec(n=8192, d=4096, kind="scaled", dtype="bf16", n_outliers=16, outlier_factor=50.0,
                             segment=2048), 4, 128, True)
    raise ValueError(name)


def make_mlp_weights(spec: MLPSpec, seed: int, device="cpu"):
    return [make_weight(spec.dims[i + 1], spec.dims[i], 1.0 / math.sqrt(spec.dims[i]), seed + 17 * i, device)
            for i in range(len(spec.dims) - 1)]

