"""Seeded synthetic workloads for the TTT-KVB layer and chunked linear attention.

This module only draws random numbers and holds the workload shapes; it holds
none of the method's arithmetic.  Tests, the benchmark and the smoke check
feed the same arrays to the CUDA path and to the fp64 CPU oracle.

Recipe (one CPU ``torch.Generator`` per workload, seeded, draws in the fixed
order q, k, v, eta-noise, W1, W2, W3):
  * q, k, v ~ N(0, 1/d_h) in fp32, rounded to bf16 (round-to-nearest-even)
    when the workload's I/O type is bf16;
  * optionally every k row is L2-normalised before rounding (the LM-style
    workload uses L2-normed keys);
  * eta = softplus(N(0, 1)) / chunk, fp32, one learning rate per token;
  * W1, W3 [m, d], W2 [d, m] ~ N(0, 1/d_h), fp32, one set per head (shared
    over the batch).

The shapes stand in for the pages' workloads: a 760M-scale language model
layer (d = 1536, 4 TTT heads, chunk = window = 2048), the view-synthesis
strided mask (8 chunks of 8192 tokens, update on the first 4), a
million-token context, and the linear-attention reduction.  No dataset is
used.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import torch

APPLY_THEN_UPDATE = 0
BLOCK_CAUSAL = 1
BIDIRECTIONAL = 2
STRIDED = 3


@dataclasses.dataclass(frozen=True)
class LayerWorkload:
    name: str
    B: int
    H: int
    N: int
    d_h: int
    m_h: int
    chunk: int
    mode: int
    io_dtype: str            # "f32" or "bf16"
    l2norm: bool = True
    muon_steps: int = 0
    momentum_beta: float = 0.0
    update_chunks: Optional[Sequence[int]] = None
    l2_normed_k: bool = False
    seed: int = 0

    @property
    def n_chunks(self) -> int:
        return self.N // self.chunk


@dataclasses.dataclass(frozen=True)
class LinattnWorkload:
    name: str
    B: int
    H: int
    N: int
    d_k: int
    d_v: int
    chunk: int
    mode: int
    io_dtype: str = "bf16"
    update_chunks: Optional[Sequence[int]] = None
    seed: int = 0


# The five workloads of the method's benchmark table.
TINY_F32 = LayerWorkload("tiny-fp32 d32 m32 N256 chunk64 apply-then-update",
                         B=1, H=1, N=256, d_h=32, m_h=32, chunk=64,
                         mode=APPLY_THEN_UPDATE, io_dtype="f32", l2norm=True)
LINATTN_C2 = LinattnWorkload("linattn B4 H4 N8192 d128 chunk2048 block-causal",
                             B=4, H=4, N=8192, d_k=128, d_v=128, chunk=2048,
                             mode=BLOCK_CAUSAL)
LM_760M = LayerWorkload("lm-760m B2 H4 d384 m384 N32768 chunk2048 muon5 beta0.9",
                        B=2, H=4, N=32768, d_h=384, m_h=384, chunk=2048,
                        mode=APPLY_THEN_UPDATE, io_dtype="bf16", l2norm=True,
                        muon_steps=5, momentum_beta=0.9, l2_normed_k=True)
NVS_STRIDED = LayerWorkload("nvs-strided B1 H2 d384 m768 8x8192 update0-3",
                            B=1, H=2, N=8 * 8192, d_h=384, m_h=768, chunk=8192,
                            mode=STRIDED, io_dtype="bf16", l2norm=True,
                            update_chunks=(1, 1, 1, 1, 0, 0, 0, 0))
LONG_1M = LayerWorkload("long-1m B1 H4 d512 m512 N1048576 chunk8192 muon5 beta0.9",
                        B=1, H=4, N=1048576, d_h=512, m_h=512, chunk=8192,
                        mode=APPLY_THEN_UPDATE, io_dtype="bf16", l2norm=True,
                        muon_steps=5, momentum_beta=0.9)

ALL_LAYER = (TINY_F32, LM_760M, NVS_STRIDED, LONG_1M)


def _io(x: torch.Tensor, io_dtype: str) -> torch.Tensor:
    return x.to(torch.bfloat16) if io_dtype == "bf16" else x.contiguous()


def _normal(gen, shape, std):
    return torch.randn(shape, generator=gen, dtype=torch.float32) * std


def layer_inputs(wl: LayerWorkload, B=None, H=None, N=None, seed=None):
    """Draw (q, k, v, eta, W1, W2, W3) on the CPU for a layer workload.

    B, H, N override the workload's sizes (smaller parity cases keep the rest
    of the recipe).  q, k, v are bf16 or fp32 CPU tensors [B, H, N, d];
    eta fp32 [B, H, N]; W1, W3 fp32 [H, m, d]; W2 fp32 [H, d, m].
    """
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    N = wl.N if N is None else N
    d, m = wl.d_h, wl.m_h
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed if seed is None else seed)
    std = 1.0 / math.sqrt(d)
    q = _normal(gen, (B, H, N, d), std)
    k = _normal(gen, (B, H, N, d), std)
    v = _normal(gen, (B, H, N, d), std)
    if wl.l2_normed_k:
        k = k / k.norm(dim=-1, keepdim=True).clamp_min(1e-12)
    eta = torch.nn.functional.softplus(torch.randn((B, H, N), generator=gen)) / wl.chunk
    W1 = _normal(gen, (H, m, d), std)
    W2 = _normal(gen, (H, d, m), std)
    W3 = _normal(gen, (H, m, d), std)
    return (_io(q, wl.io_dtype), _io(k, wl.io_dtype), _io(v, wl.io_dtype),
            eta.contiguous(), W1, W2, W3)


def layer_inputs_on_device(wl: LayerWorkload, device, seed=None):
    """The layer workload's recipe drawn directly on a CUDA device (a seeded
    CUDA generator, the same draw order and distributions as
    ``layer_inputs``; the values differ from the CPU draw).  For workloads
    too large to draw on the host in reasonable time (the million-token
    context: 2^31 elements per tensor); used for timing only.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(wl.seed if seed is None else seed)
    d, m, B, H, N = wl.d_h, wl.m_h, wl.B, wl.H, wl.N
    std = 1.0 / math.sqrt(d)
    dt = torch.bfloat16 if wl.io_dtype == "bf16" else torch.float32

    def io(shape):
        x = torch.randn(shape, generator=gen, device=device, dtype=torch.float32)
        x.mul_(std)
        return x.to(dt)

    q = io((B, H, N, d))
    k = io((B, H, N, d))
    if wl.l2_normed_k:
        raise ValueError("draw L2-normalised keys with layer_inputs")
    v = io((B, H, N, d))
    eta = torch.nn.functional.softplus(
        torch.randn((B, H, N), generator=gen, device=device)) / wl.chunk
    W1 = torch.randn((H, m, d), generator=gen, device=device) * std
    W2 = torch.randn((H, d, m), generator=gen, device=device) * std
    W3 = torch.randn((H, m, d), generator=gen, device=device) * std
    return q, k, v, eta.contiguous(), W1, W2, W3


def linattn_inputs(wl: LinattnWorkload, B=None, H=None, N=None, seed=None,
                   with_state=False):
    """Draw (q, k, v, eta, S0) on the CPU for a linear-attention workload.

    S0 is None (zero initial state) unless ``with_state``; then it is
    N(0, 1/d_k) fp32 [B, H, d_v, d_k].
    """
    B = wl.B if B is None else B
    H = wl.H if H is None else H
    N = wl.N if N is None else N
    gen = torch.Generator(device="cpu")
    gen.manual_seed(wl.seed if seed is None else seed)
    std = 1.0 / math.sqrt(wl.d_k)
    q = _normal(gen, (B, H, N, wl.d_k), std)
    k = _normal(gen, (B, H, N, wl.d_k), std)
    v = _normal(gen, (B, H, N, wl.d_v), std)
    eta = torch.nn.functional.softplus(torch.randn((B, H, N), generator=gen)) / wl.chunk
    S0 = _normal(gen, (B, H, wl.d_v, wl.d_k), std) if with_state else None
    return (_io(q, wl.io_dtype), _io(k, wl.io_dtype), _io(v, wl.io_dtype),
            eta.contiguous(), S0)
