"""Seeded synthetic inputs for one STILL attention layer.

This module holds no arithmetic of the method: it only draws q, k, v and Wf
with the shapes and value distributions of the workloads below, and it is the
one module that both the CUDA path's callers and the oracle's callers use.

Value recipe (Llama-3-class layers, post-projection q/k/v):
  * "iid"     rows are i.i.d. N(0, 1) scaled by s ~ LogNormal(0, 0.5) per row;
  * "dirnorm" rows have an N(0, I) direction and norm s * sqrt(d),
              s ~ LogNormal(0, 0.5) per row;
  * outliers  a fraction of token positions per sequence (the same positions
              for every head, q, k and v) gets 4x the norm;
  * Wf ~ N(0, 1/d) in fp32, one [d, d_f] matrix per layer.
q, k, v are rounded to bf16 (round to nearest even).  CPU draws use NumPy's
PCG64; CUDA draws use torch's device generator (same recipe, other stream of
numbers) so that very large batches need no host-side generation.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, asdict

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    N: int
    W: int
    C: int
    m: int
    T_max: int
    df: int
    dist: str = "dirnorm"
    outlier_frac: float = 0.0

    @property
    def lam(self) -> int:
        return (self.m - self.W) // self.T_max

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    def asdict(self):
        d = asdict(self)
        d["lambda"] = self.lam
        return d


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_prefill_n512", 1, 2, 2, 64, 512, 64, 64, 128, 8, 64, "iid"),
        Workload("llama32_1b_layer_prefill_4k", 1, 32, 8, 64, 4096, 64, 256, 288, 16, 64),
        Workload("llama3_8b_layer_prefill_16k", 1, 32, 8, 128, 16384, 64, 256, 288, 64, 128),
        Workload("train_b8_n1k_chunk_parallel", 8, 32, 8, 128, 1024, 64, 64, 288, 16, 128,
                 "dirnorm", 0.05),
        Workload("llama31_8b_decode_b128_ctx16k", 128, 32, 8, 128, 16384, 64, 256, 288, 64, 128),
    ]
}


def _rows_cpu(rng, shape, dist):
    g = rng.standard_normal(shape, dtype=np.float32)
    s = np.exp(0.5 * rng.standard_normal(shape[:-1] + (1,), dtype=np.float32))
    if dist == "iid":
        return g * s
    d = shape[-1]
    return g / np.linalg.norm(g, axis=-1, keepdims=True) * (s * math.sqrt(d))


def _rows_dev(gen, shape, dist, device):
    g = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
    s = torch.exp(0.5 * torch.randn(shape[:-1] + (1,), generator=gen, device=device,
                                    dtype=torch.float32))
    if dist == "iid":
        return g * s
    return g / g.norm(dim=-1, keepdim=True) * (s * math.sqrt(shape[-1]))


def make_inputs(w: Workload, seed: int = 0, device="cpu", B: int | None = None, N: int | None = None):
    """Draw q [B,Hq,N,d], k, v [B,Hkv,N,d] (bf16) and Wf [d,df] (fp32).

    B and N may be overridden (smaller parity cases of the same recipe)."""
    B = w.B if B is None else B
    N = w.N if N is None else N
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = np.random.Generator(np.random.PCG64(seed))
        q = _rows_cpu(rng, (B, w.Hq, N, w.d), w.dist)
        k = _rows_cpu(rng, (B, w.Hkv, N, w.d), w.dist)
        v = _rows_cpu(rng, (B, w.Hkv, N, w.d), w.dist)
        Wf = rng.standard_normal((w.d, w.df), dtype=np.float32) / np.float32(math.sqrt(w.d))
        if w.outlier_frac > 0:
            n_out = int(round(w.outlier_frac * N))
            for b in range(B):
                pos = rng.choice(N, size=n_out, replace=False)
                for a in (q, k, v):
                    a[b, :, pos, :] *= 4.0
        q, k, v = (torch.from_numpy(np.ascontiguousarray(a)).to(torch.bfloat16) for a in (q, k, v))
        Wf = torch.from_numpy(np.ascontiguousarray(Wf))
        return q, k, v, Wf
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = _rows_dev(gen, (B, w.Hq, N, w.d), w.dist, dev)
    k = _rows_dev(gen, (B, w.Hkv, N, w.d), w.dist, dev)
    v = _rows_dev(gen, (B, w.Hkv, N, w.d), w.dist, dev)
    Wf = torch.randn((w.d, w.df), generator=gen, device=dev, dtype=torch.float32) / math.sqrt(w.d)
    if w.outlier_frac > 0:
        n_out = int(round(w.outlier_frac * N))
        for b in range(B):
            pos = torch.randperm(N, generator=gen, device=dev)[:n_out]
            for a in (q, k, v):
                a[b, :, pos, :] *= 4.0
    return (q.to(torch.bfloat16), k.to(torch.bfloat16), v.to(torch.bfloat16), Wf)


def make_gate(w: Workload, seed: int = 0, device="cpu", B: int | None = None, N: int | None = None,
              scale: float = 2.0):
    """Gate pre-activations of the linear branch, bf16 [B,Hq,N,d]: i.i.d.
    N(0, scale^2), so that the sigmoid gates spread over (0, 1) (about 0.02 to
    0.98 at two standard deviations).  Seeded apart from make_inputs."""
    B = w.B if B is None else B
    N = w.N if N is None else N
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = np.random.Generator(np.random.PCG64(seed + 7919))
        a = rng.standard_normal((B, w.Hq, N, w.d), dtype=np.float32) * np.float32(scale)
        return torch.from_numpy(a).to(torch.bfloat16)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 7919)
    return (torch.randn((B, w.Hq, N, w.d), generator=gen, device=dev) * scale).to(torch.bfloat16)


def make_dout(w: Workload, seed: int = 0, device="cpu", B: int | None = None, N: int | None = None):
    """Upstream gradient dL/dy of the layer output for the backward pass, bf16
    [B,Hq,N,d]: i.i.d. N(0, 1).  Seeded apart from make_inputs and make_gate."""
    B = w.B if B is None else B
    N = w.N if N is None else N
    dev = torch.device(device)
    if dev.type == "cpu":
        rng = np.random.Generator(np.random.PCG64(seed + 104729))
        a = rng.standard_normal((B, w.Hq, N, w.d), dtype=np.float32)
        return torch.from_numpy(a).to(torch.bfloat16)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed + 104729)
    return torch.randn((B, w.Hq, N, w.d), generator=gen, device=dev).to(torch.bfloat16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    """Exact float64 copy of a (bf16/fp32) tensor, on the host."""
    return t.detach().to("cpu", torch.float64).numpy()
