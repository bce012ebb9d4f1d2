"""Seeded synthetic inputs for GDN / KDA decode.

This module holds only random draws and tensor packing; none of the decode
arithmetic.  Both the CUDA path and the CPU oracle are fed from it.

Value distributions (the same for every workload):
  q, k  ~ N(0, 1) per key head, L2-normalised over K; q then scaled by 1/sqrt(K)
  v     ~ N(0, 1)
  g     = -softplus(N(0, 1))     (per value head, or per key channel for KDA)
  beta  = sigmoid(N(0, 1))
  S0    ~ N(0, 0.1^2)
  ring prefill (staggered cursors): d ~ N(0,1) * sigmoid(N(0,1)), k as above,
        g as above; positions >= write_pos hold NaN (they must never be read).
"""
from __future__ import annotations

from dataclasses import dataclass, replace
from typing import Optional

import torch
import torch.nn.functional as F

from .constants import BF16, F16, F32, GATE_PER_K, GATE_SCALAR, TORCH_DTYPE


@dataclass(frozen=True)
class Workload:
    name: str
    N: int            # slot pool
    B: int            # live rows per step
    HV: int
    HK: int
    K: int            # == V
    L: int
    ring_dtype: int
    qkv_dtype: int
    gate: int = GATE_SCALAR
    steps: int = 1
    n_pad: int = 0    # extra padding rows (index -1)
    layers: int = 1
    staggered: bool = False  # write_pos uniform in [0, L) with a prefilled ring
    seed: int = 0

    @property
    def V(self) -> int:
        return self.K

    @property
    def rows(self) -> int:
        return self.B + self.n_pad


TINY = Workload("tiny: N=8 B=4 HV=4 HK=2 K=V=64 L=4 fp32", N=8, B=4, HV=4, HK=2, K=64, L=4,
                ring_dtype=F32, qkv_dtype=F32, steps=32, seed=0)
QWEN3NEXT_LAYER = Workload("one GDN layer: N=512 B=64+4pad HV=32 HK=16 K=V=128 L=16 fp16 ring bf16 qkv",
                           N=512, B=64, HV=32, HK=16, K=128, L=16, ring_dtype=F16,
                           qkv_dtype=BF16, steps=128, n_pad=4, seed=1)
KDA_LAYER = Workload("KDA layer: N=256 B=128 HV=HK=32 K=V=128 L=16 fp16 ring bf16 qkv",
                     N=256, B=128, HV=32, HK=32, K=128, L=16, ring_dtype=F16, qkv_dtype=BF16,
                     gate=GATE_PER_K, steps=64, seed=3)
STACK30 = Workload("30-layer stack: N=320 B=256 HV=32 HK=16 K=V=128 L=16 fp16 ring bf16 qkv",
                   N=320, B=256, HV=32, HK=16, K=128, L=16, ring_dtype=F16, qkv_dtype=BF16,
                   steps=48, layers=30, seed=4)


def sweep_point(B: int, L: int, ring_dtype: int) -> Workload:
    """One point of the batch x ring-length sweep (staggered cursors, 2L steps)."""
    tag = {F32: "fp32", F16: "fp16", BF16: "bf16"}[ring_dtype]
    return Workload(f"sweep: N={max(B, 512)} B={B} HV=32 HK=16 K=V=128 L={L} {tag} ring bf16 qkv",
                    N=max(B, 512), B=B, HV=32, HK=16, K=128, L=L, ring_dtype=ring_dtype,
                    qkv_dtype=BF16, steps=2 * L, staggered=True, seed=2)


HEADLINE = sweep_point(256, 16, F16)


def generator(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _normal(gen, shape, device):
    """Draws on the generator's own device, then moves to `device`."""
    return torch.randn(shape, generator=gen, device=gen.device, dtype=torch.float32).to(device)


def _unit(x: torch.Tensor) -> torch.Tensor:
    return x / x.norm(dim=-1, keepdim=True)


def indices(gen, B: int, N: int, n_pad: int, device) -> torch.Tensor:
    """B distinct slots (a seeded permutation of the pool) plus n_pad rows of -1
    at seeded positions."""
    slots = torch.randperm(N, generator=gen, device=gen.device)[:B].to(device=device, dtype=torch.int32)
    if n_pad == 0:
        return slots
    rows = B + n_pad
    pad_pos = torch.randperm(rows, generator=gen, device=gen.device)[:n_pad].to(device)
    out = torch.full((rows,), -1, dtype=torch.int32, device=device)
    keep = torch.ones(rows, dtype=torch.bool, device=device)
    keep[pad_pos] = False
    out[keep] = slots
    return out


def state(gen, N: int, HV: int, V: int, K: int, device) -> torch.Tensor:
    return _normal(gen, (N, HV, V, K), device) * 0.1


@dataclass
class StepInputs:
    mixed_qkv: torch.Tensor  # [rows, 2*HK*K + HV*V]
    g: torch.Tensor          # [rows, HV] or [rows, HV, K]
    beta: torch.Tensor       # [rows, HV]


def step_inputs(gen, w: Workload, device, rows: Optional[int] = None) -> StepInputs:
    R = w.rows if rows is None else rows
    q = _unit(_normal(gen, (R, w.HK, w.K), device)) / (w.K ** 0.5)
    k = _unit(_normal(gen, (R, w.HK, w.K), device))
    v = _normal(gen, (R, w.HV, w.V), device)
    gshape = (R, w.HV, w.K) if w.gate == GATE_PER_K else (R, w.HV)
    g = -F.softplus(_normal(gen, gshape, device))
    beta = torch.sigmoid(_normal(gen, (R, w.HV), device))
    mixed = torch.cat([q.reshape(R, w.HK * w.K), k.reshape(R, w.HK * w.K), v.reshape(R, w.HV * w.V)], dim=1)
    return StepInputs(mixed.to(TORCH_DTYPE[w.qkv_dtype]).contiguous(), g.contiguous(), beta.contiguous())


def write_pos(gen, w: Workload, device) -> torch.Tensor:
    if not w.staggered:
        return torch.zeros(w.N, dtype=torch.int32, device=device)
    return torch.randint(0, w.L, (w.N,), generator=gen, device=gen.device, dtype=torch.int32).to(device)


@dataclass
class CacheTensors:
    state: torch.Tensor
    ring_d: torch.Tensor
    ring_k: torch.Tensor
    ring_g: torch.Tensor


def cache(gen, w: Workload, wp: torch.Tensor, device) -> CacheTensors:
    """Checkpoint plus a ring holding valid draws at positions < write_pos and NaN elsewhere."""
    S0 = state(gen, w.N, w.HV, w.V, w.K, device)
    rdt = TORCH_DTYPE[w.ring_dtype]
    d = _normal(gen, (w.N, w.HV, w.L, w.V), device) * torch.sigmoid(_normal(gen, (w.N, w.HV, w.L, 1), device))
    k = _unit(_normal(gen, (w.N, w.HK, w.L, w.K), device))
    gshape = (w.N, w.HV, w.L, w.K) if w.gate == GATE_PER_K else (w.N, w.HV, w.L)
    g = -F.softplus(_normal(gen, gshape, device))
    pos = torch.arange(w.L, device=device)
    stale = pos[None, :] >= wp.to(torch.int64)[:, None]           # [N, L]
    d[stale[:, None, :, None].expand_as(d)] = float("nan")
    # a key head's entries are valid below the slot's cursor (all its value heads share it)
    k[stale[:, None, :, None].expand_as(k)] = float("nan")
    gm = stale[:, None, :, None] if w.gate == GATE_PER_K else stale[:, None, :]
    g[gm.expand_as(g)] = float("nan")
    return CacheTensors(S0, d.to(rdt).contiguous(), k.to(rdt).contiguous(), g.contiguous())


def with_(w: Workload, **kw) -> Workload:
    return replace(w, **kw)
