"""Seeded synthetic inputs for the KDA decode projections.

This module only draws random numbers. It holds none of the projection's
arithmetic, and both the CUDA path's tests/benchmarks and the CPU oracle's
callers take their inputs from here, so the two sides see the same bf16 bit
patterns.

Shapes and distributions follow the pages' workload (Kimi-K3 KDA input
projections of one TP8 rank, "[Kimi-K3] Overlap low-M TP8 KDA projections",
section "关键源码片段", run_kda_projection_overlap):

* hidden states ``x``: ``[M, K]`` bf16, ``K = 7168``; drawn ~N(0, 1)
  (``dist="normal"``) or ~U(-1, 1) (``dist="uniform"``).
* packed weight ``W_packed``: ``[N_qkvg + N_fab, K]`` bf16 with the Q/K/V/G rows
  first (``N_qkvg = 4096``) and the F_A/beta rows after them (``N_fab = 136``:
  128 replicated F_A rows + 8 local beta heads); drawn ~N(0, 0.02^2).
* F_B weight ``W_fb``: ``[N_fb, 128]`` bf16 (``N_fb = 1024``); ~N(0, 0.02^2).

Seeding: ``x`` comes from ``torch.Generator`` seeded with ``seed``; layer ``l``
of a weight stack comes from a generator seeded with ``seed + 1 + l`` (the
packed weight is drawn first, then ``W_fb``). Values are drawn in fp32 and
rounded to bf16 with round-to-nearest-even by ``Tensor.to(torch.bfloat16)``.

``dtype=torch.float16`` draws the same fp32 numbers and rounds them to fp16
instead (the skinny GEMM's other input type).

``device="cpu"`` is the canonical stream that parity tests use. A CUDA device
draws from torch's CUDA generator instead (different numbers, same
distribution); the benchmark uses that for filler layers of large weight
stacks, which only load the memory system.
"""
from __future__ import annotations

import numpy as np
import torch

K_HIDDEN = 7168
N_QKVG = 4096
N_FAB = 136
N_FA = 128
N_FB = 1024
W_STD = 0.02


def _gen(seed: int, device) -> torch.Generator:
    dev = torch.device(device)
    g = torch.Generator(device=dev)
    g.manual_seed(int(seed))
    return g


def gen_x(M: int, K: int, seed: int = 0, dist: str = "normal", device="cpu",
          dtype=torch.bfloat16) -> torch.Tensor:
    """Hidden states ``[M, K]`` (bf16 or fp16) drawn from ``dist`` with generator ``seed``."""
    g = _gen(seed, device)
    if dist == "normal":
        v = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    elif dist == "uniform":
        v = torch.rand((M, K), generator=g, device=device, dtype=torch.float32) * 2.0 - 1.0
    else:
        raise ValueError(f"unknown dist {dist!r}")
    return v.to(dtype)


def gen_w(N: int, K: int, seed: int, std: float = W_STD, device="cpu",
          g: torch.Generator | None = None, dtype=torch.bfloat16) -> torch.Tensor:
    """Weight ``[N, K]`` (bf16 or fp16) ~N(0, std^2)."""
    if g is None:
        g = _gen(seed, device)
    v = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        v.mul_(std)
    return v.to(dtype)


def gen_kda_layer(layer: int, seed: int = 0, K: int = K_HIDDEN, N_qkvg: int = N_QKVG,
                  N_fab: int = N_FAB, N_fb: int = N_FB, K_fb: int = N_FA,
                  device="cpu") -> tuple[torch.Tensor, torch.Tensor]:
    """One layer's ``(W_packed [N_qkvg+N_fab, K], W_fb [N_fb, K_fb])``."""
    g = _gen(seed + 1 + layer, device)
    wp = gen_w(N_qkvg + N_fab, K, 0, device=device, g=g)
    wfb = gen_w(N_fb, K_fb, 0, device=device, g=g)
    return wp, wfb


def gen_gemm_layer(layer: int, N: int, K: int, seed: int = 0, device="cpu") -> torch.Tensor:
    """Layer ``layer`` of a plain ``[N, K]`` weight stack."""
    return gen_w(N, K, seed + 1 + layer, device=device)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a CPU tensor as a contiguous ``uint16`` array."""
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def bits16(t: torch.Tensor) -> np.ndarray:
    """Raw bit patterns of a bf16 or fp16 tensor as a contiguous ``uint16`` array."""
    assert t.dtype in (torch.bfloat16, torch.float16)
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bf16_bits(a: np.ndarray) -> torch.Tensor:
    """Inverse of :func:`bf16_bits` (CPU tensor)."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16)
