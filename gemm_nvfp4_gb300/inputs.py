"""Seeded synthetic inputs for the NVFP4 x bf16 workloads.

This module is the only code that both the CUDA path's tests/benchmark and the
CPU oracle consume.  It draws random numbers and nothing else: it holds none of
the method's arithmetic (no quantisation, no scaling rules, no products).

Recipe (also stated in the design notes):
  * weights: fp32 N(0, 0.02): ``randn * 0.02`` from a ``torch.Generator`` seeded
    per matrix;
  * heavy-tailed weights (the deep-verify workload): every element independently,
    with probability 0.01, is replaced by a draw from N(0, 0.2);
  * activations: bf16 N(0, 1): ``randn`` in fp32 rounded to bf16 (round to nearest
    even, PyTorch's conversion); optionally every 4th token row (n % 4 == 3)
    multiplied by 8 (exact in bf16);
  * matrix j of a decoder layer (QKV=0, O=1, gate=2, up=3, down=4) uses seed
    100*j for its weights, 100*j+1 for its activations, 100*j+2 for the outlier
    mask and 100*j+3 for the outlier values; the single 4096x4096 matrix is j=0.

Generation on a CUDA device uses PyTorch's device generator; the values differ
from CPU generation with the same seed, but every consumer (kernel and oracle)
receives the same buffer, copied where needed.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

LAYER_MATRICES = ("qkv", "o", "gate", "up", "down")


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=torch.device(device))
    g.manual_seed(int(seed))
    return g


def weights(M: int, K: int, seed: int = 0, std: float = 0.02,
            heavy_tail: bool = False, device="cpu") -> torch.Tensor:
    """fp32 [M, K] ~ N(0, std); with ``heavy_tail`` 1% of elements ~ N(0, 0.2)."""
    w = torch.randn(M, K, generator=_gen(seed, device), device=device,
                    dtype=torch.float32)
    w.mul_(std)
    if heavy_tail:
        mask = torch.rand(M, K, generator=_gen(seed + 2, device), device=device) < 0.01
        big = torch.randn(M, K, generator=_gen(seed + 3, device), device=device,
                          dtype=torch.float32).mul_(0.2)
        w = torch.where(mask, big, w)
    return w


def activations(N: int, K: int, seed: int = 1, outlier_rows: bool = False,
                device="cpu") -> torch.Tensor:
    """bf16 [N, K] ~ N(0, 1); with ``outlier_rows`` rows n % 4 == 3 are x8."""
    x = torch.randn(N, K, generator=_gen(seed, device), device=device,
                    dtype=torch.float32).to(torch.bfloat16)
    if outlier_rows:
        x[3::4] *= 8
    return x


def bf16_bits(x: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (for the oracle)."""
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view("uint16")


@dataclass(frozen=True)
class LayerShape:
    """One dense decoder layer's projection shapes, as (M, K) = (out, in)."""
    name: str
    hidden: int
    qkv_out: int
    ffn: int

    def shapes(self):
        h, f = self.hidden, self.ffn
        return {"qkv": (self.qkv_out, h), "o": (h, h), "gate": (f, h),
                "up": (f, h), "down": (h, f)}


# Dense 9B-class layer: QKV 4096->6144, O 4096->4096, gate/up 4096->12288, down 12288->4096.
LAYER_9B = LayerShape("dense-9B-class", hidden=4096, qkv_out=6144, ffn=12288)
# Dense 27B-class layer: QKV 5120->7168, O 5120->5120, gate/up 5120->17408, down 17408->5120.
LAYER_27B = LayerShape("dense-27B-class", hidden=5120, qkv_out=7168, ffn=17408)


def matrix_seed(name: str) -> int:
    return 100 * LAYER_MATRICES.index(name)
