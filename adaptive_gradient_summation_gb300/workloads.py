"""Seeded synthetic gradient sets shaped like the workloads of "Scaling Distributed
Training with Adaptive Summation" (ResNet-50, BERT-Large, a GPT-style transformer).

This module only draws random numbers and lays out parameter shapes.  It holds none of
the Adasum arithmetic, so both the CUDA path's tests and the CPU oracle can take their
inputs from it.  No dataset or trained weight is involved: the gradients are synthetic,
matched to the models by parameter-tensor shapes only.

Every workload is K worker gradients over one flat parameter vector split into layer
segments.  Within segment l the workers are correlated through a shared component:

    g_k = sigma_l * (rho_l * s + sqrt(1 - rho_l^2) * z_k),   s, z_k ~ N(0, 1) per element,

with sigma_l log-uniform in [1e-4, 1e-1] and rho_l ~ U[0, 0.9] (the model-shaped sets).
The pairwise correlation inside a segment is then rho_l^2.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

# ----------------------------------------------------------------------------------
# Parameter-tensor shapes (architecture facts; element counts per tensor, in the
# order the frameworks list the parameters).
# ----------------------------------------------------------------------------------


def resnet50_numels() -> list[int]:
    """ResNet-50 parameters in torchvision order: 161 tensors, 25,557,032 elements."""
    out = [64 * 3 * 7 * 7, 64, 64]  # stem conv, BN gamma/beta
    inplanes = 64
    for planes, blocks in ((64, 3), (128, 4), (256, 6), (512, 3)):
        for b in range(blocks):
            out += [planes * inplanes, planes, planes,        # conv1 1x1, bn1
                    planes * planes * 9, planes, planes,      # conv2 3x3, bn2
                    4 * planes * planes, 4 * planes, 4 * planes]  # conv3 1x1, bn3
            if b == 0:
                out += [4 * planes * inplanes, 4 * planes, 4 * planes]  # downsample
            inplanes = 4 * planes
    out += [1000 * 2048, 1000]  # fc weight, bias
    return out


def bert_large_numels() -> list[int]:
    """BERT-Large parameters: embeddings (word 30522x1024, position 512x1024,
    token-type 2x1024, LayerNorm), 24 encoder layers, pooler.  391 tensors,
    335,141,888 elements."""
    h, f = 1024, 4096
    out = [30522 * h, 512 * h, 2 * h, h, h]
    for _ in range(24):
        for _qkvo in range(4):            # query, key, value, attention output
            out += [h * h, h]
        out += [h, h]                     # attention-output LayerNorm
        out += [h * f, f]                 # FFN in
        out += [f * h, h]                 # FFN out
        out += [h, h]                     # output LayerNorm
    out += [h * h, h]                     # pooler
    return out


def gpt_numels() -> list[int]:
    """GPT-style transformer, hidden 2048, 24 layers, vocab 50304, no biases and no
    position table: 195 tensors, 1,311,182,848 elements."""
    h = 2048
    out = [50304 * h]
    for _ in range(24):
        out += [h, h,            # ln_1 gamma/beta
                h * 3 * h,       # fused QKV
                h * h,           # attention out-projection
                h, h,            # ln_2 gamma/beta
                h * 4 * h,       # MLP up
                4 * h * h]       # MLP down
    out += [h, h]                # final LayerNorm
    return out


def offsets_from_numels(numels) -> np.ndarray:
    offs = np.zeros(len(numels) + 1, dtype=np.int64)
    np.cumsum(np.asarray(numels, dtype=np.int64), out=offs[1:])
    return offs


# ----------------------------------------------------------------------------------
# Workloads
# ----------------------------------------------------------------------------------

BASE_SEED = 20200604

#: name -> (config index, K, storage dtype, description)
CONFIGS = {
    "pair_1m": (1, 2, torch.float32,
                "K=2, one fp32 tensor of 1,048,576 elements, g1 = 0.5 g0 + sqrt(0.75) z"),
    "resnet50_k8": (2, 8, torch.float32,
                    "K=8, ResNet-50-shaped fp32 gradient set (161 tensors, 25.6M elements)"),
    "bert_large_k16": (3, 16, torch.bfloat16,
                       "K=16, BERT-Large-shaped bf16 gradient set (391 tensors, 335.1M "
                       "elements), fp32 math"),
    "small_segments_k64": (4, 64, torch.float32,
                           "K=64, 10,000 fp32 segments, lengths log-uniform in [1, 4096], "
                           "zero / parallel / orthogonal special segments"),
    "gpt_k8_momentum": (5, 8, torch.bfloat16,
                        "K=8, GPT-style 1.31B-element bf16 gradient set, fused Momentum-SGD "
                        "(mu 0.9, lr 0.1) on fp32 master weights ~ N(0, 0.02)"),
}

#: Segment categories of the small-segment workload.
KIND_CORRELATED, KIND_ZERO_SOME, KIND_PARALLEL, KIND_ORTHOGONAL = 0, 1, 2, 3


@dataclass
class Workload:
    name: str
    K: int
    dtype: torch.dtype
    seg_offsets: np.ndarray            # int64, L+1 entries, offs[0] = 0, offs[L] = N
    grads: list                        # K 1-D tensors of N elements, `dtype`
    description: str = ""
    seed: int = 0
    master_w: torch.Tensor | None = None   # fp32, N (momentum workload only)
    momentum: torch.Tensor | None = None   # fp32, N
    lr: float | None = None
    mu: float | None = None
    seg_kind: np.ndarray | None = None     # per-segment category (small-segment workload)
    extra: dict = field(default_factory=dict)

    @property
    def N(self) -> int:
        return int(self.seg_offsets[-1])

    @property
    def L(self) -> int:
        return int(self.seg_offsets.shape[0] - 1)

    def input_bytes(self) -> int:
        return self.K * self.N * torch.tensor([], dtype=self.dtype).element_size()


def _per_element(values: np.ndarray, counts: np.ndarray, device) -> torch.Tensor:
    v = torch.as_tensor(values, dtype=torch.float32).to(device)
    c = torch.as_tensor(counts, dtype=torch.int64).to(device)
    return torch.repeat_interleave(v, c, output_size=int(np.sum(counts)))


def _correlated_set(numels, K, dtype, device, seed, sigma=None, rho=None):
    """g_k = sigma_l (rho_l s + sqrt(1 - rho_l^2) z_k) per segment l."""
    rs = np.random.default_rng(seed)
    L = len(numels)
    if sigma is None:
        sigma = np.exp(rs.uniform(math.log(1e-4), math.log(1e-1), size=L))
    if rho is None:
        rho = rs.uniform(0.0, 0.9, size=L)
    counts = np.asarray(numels, dtype=np.int64)
    N = int(counts.sum())
    gen = torch.Generator(device=device).manual_seed(seed)
    a = _per_element(sigma * rho, counts, device)
    b = _per_element(sigma * np.sqrt(1.0 - rho * rho), counts, device)
    s = torch.randn(N, generator=gen, device=device, dtype=torch.float32)
    shared = a * s
    del s, a
    grads = []
    for _ in range(K):
        z = torch.randn(N, generator=gen, device=device, dtype=torch.float32)
        grads.append((shared + b * z).to(dtype))
        del z
    return grads, sigma, rho


def _shrunk(numels, shrink: int):
    if shrink <= 1:
        return list(numels)
    return [max(1, -(-n // shrink)) for n in numels]


def make(name: str, *, device="cpu", seed: int | None = None, shrink: int = 1,
         momentum_init: str = "zero") -> Workload:
    """Build one of the named workloads.

    device: where the gradients are generated and stored.
    seed: defaults to 20200604 + the configuration index.
    shrink: divide every tensor's element count by this (ceil, at least 1) -- or, for
        the small-segment set, the segment count -- for quick test-sized variants that
        keep the layer structure.
    momentum_init: for the momentum workload, "zero" or "random" (v ~ N(0, 0.01)).
    """
    if name not in CONFIGS:
        raise KeyError(f"unknown workload {name!r}; choose from {sorted(CONFIGS)}")
    idx, K, dtype, desc = CONFIGS[name]
    seed = BASE_SEED + idx if seed is None else seed
    device = torch.device(device)

    if name == "pair_1m":
        n = max(1, -(-1_048_576 // max(shrink, 1)))
        gen = torch.Generator(device=device).manual_seed(seed)
        g0 = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        z = torch.randn(n, generator=gen, device=device, dtype=torch.float32)
        g1 = 0.5 * g0 + math.sqrt(0.75) * z
        return Workload(name, K, dtype, offsets_from_numels([n]), [g0, g1.to(dtype)],
                        desc, seed)

    if name == "small_segments_k64":
        return _small_segments(K, dtype, device, seed, shrink, desc)

    numels = {"resnet50_k8": resnet50_numels, "bert_large_k16": bert_large_numels,
              "gpt_k8_momentum": gpt_numels}[name]()
    numels = _shrunk(numels, shrink)
    grads, sigma, rho = _correlated_set(numels, K, dtype, device, seed)
    w = Workload(name, K, dtype, offsets_from_numels(numels), grads, desc, seed,
                 extra={"sigma": sigma, "rho": rho})
    if name == "gpt_k8_momentum":
        N = w.N
        gen = torch.Generator(device=device).manual_seed(seed + 1000)
        w.master_w = 0.02 * torch.randn(N, generator=gen, device=device, dtype=torch.float32)
        if momentum_init == "zero":
            w.momentum = torch.zeros(N, device=device, dtype=torch.float32)
        elif momentum_init == "random":
            w.momentum = 0.01 * torch.randn(N, generator=gen, device=device,
                                            dtype=torch.float32)
        else:
            raise ValueError("momentum_init is 'zero' or 'random'")
        w.lr, w.mu = 0.1, 0.9
    return w


def _small_segments(K, dtype, device, seed, shrink, desc) -> Workload:
    """10,000 segments, n = floor(exp(U[0, ln 4097))) in [1, 4096]; 5% segments zeroed on
    a random half of the workers (one of them zeroed on every worker), 5% exact parallel
    copies with positive power-of-two scales, 5% disjoint supports (every element owned
    by one worker), the rest N(0,1) with a shared component, rho ~ U[-0.5, 0.9]."""
    rs = np.random.default_rng(seed)
    L = max(1, -(-10_000 // max(shrink, 1)))
    n = np.floor(np.exp(rs.uniform(0.0, math.log(4097.0), size=L))).astype(np.int64)
    n = np.clip(n, 1, 4096)
    kind = rs.choice([KIND_CORRELATED, KIND_ZERO_SOME, KIND_PARALLEL, KIND_ORTHOGONAL],
                     size=L, p=[0.85, 0.05, 0.05, 0.05])
    rho = rs.uniform(-0.5, 0.9, size=L)
    offs = offsets_from_numels(n)
    N = int(offs[-1])
    gen = torch.Generator(device=device).manual_seed(seed)
    s = torch.randn(N, generator=gen, device=device, dtype=torch.float32)
    seg_of = torch.repeat_interleave(torch.arange(L), torch.as_tensor(n)).to(device)
    kind_e = torch.as_tensor(kind, device=device)[seg_of]
    rho_e = torch.as_tensor(rho, dtype=torch.float32, device=device)[seg_of]
    a = torch.where(kind_e == KIND_PARALLEL, torch.zeros_like(rho_e), rho_e)
    b = torch.sqrt(1.0 - a * a)

    # Per-(segment, worker) choices.
    zero_mask = rs.random((L, K)) < 0.5                   # zeroed workers (ZERO_SOME)
    zero_ids = np.nonzero(kind == KIND_ZERO_SOME)[0]
    if zero_ids.size:
        zero_mask[zero_ids[0], :] = True                  # one segment zero everywhere
    scale_pow = rs.integers(-2, 3, size=(L, K))           # parallel scales 2^j, j in -2..2
    owner = torch.randint(0, K, (N,), generator=gen, device=device)

    grads = []
    for k in range(K):
        z = torch.randn(N, generator=gen, device=device, dtype=torch.float32)
        g = a * s + b * z
        par_scale = torch.as_tensor(np.ldexp(1.0, scale_pow[:, k]), dtype=torch.float32,
                                    device=device)[seg_of]
        g = torch.where(kind_e == KIND_PARALLEL, par_scale * s, g)
        g = torch.where(kind_e == KIND_ORTHOGONAL,
                        torch.where(owner == k, z, torch.zeros_like(z)), g)
        zk = torch.as_tensor(zero_mask[:, k], device=device)[seg_of]
        g = torch.where((kind_e == KIND_ZERO_SOME) & zk, torch.zeros_like(g), g)
        grads.append(g.to(dtype))
    return Workload("small_segments_k64", K, dtype, offs, grads, desc, seed, seg_kind=kind,
                    extra={"rho": rho})


def numpy_case(seed: int, K: int, seg_lengths, bf16: bool = False):
    """Small seeded case drawn with numpy only (PCG64, stable across versions).

    Returns (grads, offsets): K arrays of float32, or of bf16 bits (uint16, the upper
    half of the float32 word, i.e. truncated) when ``bf16`` is set.  Workers share a
    component with correlation 0.5 so that the tree has non-trivial coefficients.
    """
    rs = np.random.default_rng(seed)
    offs = offsets_from_numels(seg_lengths)
    N = int(offs[-1])
    s = rs.standard_normal(N)
    grads = []
    for _ in range(K):
        g = (0.7 * s + 0.7 * rs.standard_normal(N)).astype(np.float32)
        grads.append((g.view(np.uint32) >> 16).astype(np.uint16) if bf16 else g)
    return grads, offs
