"""Seeded synthetic workloads: shape presets and input generators.

This module only draws random numbers and names shapes. It holds none of the
attention or layout arithmetic, so both the CUDA path's tests and the CPU
oracle can take their inputs from it without sharing any computation.

The five presets are the DiT-shaped attention problems the X-Stage pages'
FlashAttention-A2A result is about (Ulysses sequence-parallel attention in DiT
inference, "Contributions" / "Results: FlashAttention-A2A optimisation"). The
pages publish no tensors, so the inputs are i.i.d. normal draws:

* a CPU ``torch.Generator`` seeded with ``seed`` draws Q, K and V in that
  order as float32 ``randn`` of shape [B, H, S, d];
* the joint text+image preset multiplies rows ``0 .. text_rows-1`` of all three
  tensors by ``text_std`` (std 2 for the 512 text tokens, std 1 for the rest);
* the result is rounded to bf16 (round-to-nearest-even, torch's cast).

The device variant draws the same recipe with a CUDA generator. Its bits differ
from the CPU draw; it is used where only the distribution matters (timing).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import torch


@dataclass(frozen=True)
class AttnConfig:
    """One attention problem: batch B, heads H, sequence S, head dim d, ranks P."""

    name: str
    B: int
    H: int
    S: int
    d: int
    P: int
    text_rows: int = 0
    text_std: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> int:
        """4*B*H*S^2*d: the two matmuls of attention, 2 flops per multiply-add."""
        return 4 * self.B * self.H * self.S * self.S * self.d

    @property
    def qkv_bytes(self) -> int:
        return 3 * self.B * self.H * self.S * self.d * 2

    @property
    def out_bytes(self) -> int:
        return self.B * self.H * self.S * self.d * 2


CONFIGS = {
    "tiny": AttnConfig("tiny", B=1, H=4, S=256, d=64, P=2),
    "image": AttnConfig("image", B=1, H=24, S=4096, d=128, P=4),
    "joint": AttnConfig("joint", B=1, H=24, S=4608, d=128, P=8, text_rows=512, text_std=2.0),
    "video": AttnConfig("video", B=1, H=40, S=32768, d=128, P=8),
    "long": AttnConfig("long", B=1, H=40, S=75600, d=128, P=8),
}


def config(preset: str, **overrides) -> AttnConfig:
    """A preset by name, optionally with fields replaced (e.g. a smaller S)."""
    base = CONFIGS[preset]
    if not overrides:
        return base
    fields = dict(base.__dict__)
    fields.update(overrides)
    return AttnConfig(**fields)


def _draw(shape, gen, device, text_rows, text_std):
    x = torch.randn(shape, generator=gen, dtype=torch.float32, device=device)
    if text_rows:
        x[:, :, :text_rows] *= text_std
    return x.to(torch.bfloat16)


def make_qkv(cfg: AttnConfig, seed: int = 0, device: str = "cpu"):
    """Seeded bf16 Q, K, V of shape [B, H, S, d] (contiguous).

    ``device="cpu"`` is the reproducible recipe the oracle comparisons use;
    any CUDA device draws the same distribution with a CUDA generator.
    """
    gen = torch.Generator(device=device).manual_seed(seed)
    shape = (cfg.B, cfg.H, cfg.S, cfg.d)
    q = _draw(shape, gen, device, cfg.text_rows, cfg.text_std)
    k = _draw(shape, gen, device, cfg.text_rows, cfg.text_std)
    v = _draw(shape, gen, device, cfg.text_rows, cfg.text_std)
    return q, k, v

