"""Seeded synthetic workloads for exact attention.

This module only draws inputs and names shapes. It holds none of the
attention arithmetic, so both the fp64 oracle (``oracle/``) and the CUDA
library (``exact_attention_65_gb300``) can be fed from it without sharing
any of the method's code.

Input recipe (the pages fix "i.i.d. N(0,1)" and the seed, nothing else):
  * one ``torch.Generator('cpu')`` seeded with 42 (the seed the timing script
    on "2.6.3 is faster than 2.7.0 for flash-attn v2 CUDA fwd/bwd" uses);
  * Q, then K, then V, drawn in that order from that one generator, in fp32
    with ``torch.randn``, one batch index at a time (keeps host memory
    bounded for the large decode caches);
  * each fp32 draw rounded to the workload dtype (round to nearest even).

The shapes are the ones the pages time: the small-head shapes of the
flash-attn 2.6.3/2.7.0 issue (embed 256 over 16 heads gives head dim 16),
the b4 s512 h32 d128 bf16 shape of "Why FlashAttention is fast" (section 2),
and the split-KV decode shapes of the flash-decoding issue (b8 h48 and
b1 h16).
"""
from __future__ import annotations

import dataclasses
import math

import torch

SEED = 42


@dataclasses.dataclass(frozen=True)
class Workload:
    """One attention problem: Q [b, sq, h, d], K/V [b, sk, h, d]."""

    name: str
    kind: str  # "fwd" or "decode"
    b: int
    sq: int
    sk: int
    h: int
    d: int
    dtype: torch.dtype

    @property
    def scale(self) -> float:
        """Default softmax scale 1/sqrt(d)."""
        return 1.0 / math.sqrt(self.d)

    @property
    def flops(self) -> int:
        """4*b*h*sq*sk*d: two matmuls of 2*sq*sk*d each per (b, h)."""
        return 4 * self.b * self.h * self.sq * self.sk * self.d

    @property
    def elem_bytes(self) -> int:
        return torch.empty((), dtype=self.dtype).element_size()

    @property
    def io_bytes(self) -> int:
        """Each tensor crossing HBM once: Q, K, V, O in dtype plus fp32 LSE."""
        e = self.elem_bytes
        qo = 2 * self.b * self.sq * self.h * self.d * e
        kv = 2 * self.b * self.sk * self.h * self.d * e
        lse = self.b * self.h * self.sq * 4
        return qo + kv + lse

    @property
    def kv_bytes(self) -> int:
        return 2 * self.b * self.sk * self.h * self.d * self.elem_bytes


WORKLOADS = {
    w.name: w
    for w in [
        Workload("tiny_fwd", "fwd", 1, 64, 64, 2, 16, torch.float16),
        Workload("small_head_b2_s50", "fwd", 2, 50, 50, 16, 16, torch.float16),
        Workload("small_head_b2_s300", "fwd", 2, 300, 300, 16, 16, torch.float16),
        Workload("small_head_b512_s150", "fwd", 512, 150, 150, 16, 16, torch.float16),
        Workload("mid_fwd", "fwd", 4, 512, 512, 32, 128, torch.bfloat16),
        Workload("decode_b8_h48_sk8192", "decode", 8, 1, 8192, 48, 128, torch.bfloat16),
        Workload("decode_b1_h16_sk32768", "decode", 1, 1, 32768, 16, 128, torch.bfloat16),
        Workload("long_fwd", "fwd", 1, 8192, 8192, 32, 128, torch.bfloat16),
        # the flash-decoding issue's several new tokens, on the b1 h16 cache
        Workload("decode_b1_h16_sk32768_sq10", "decode", 1, 10, 32768, 16, 128, torch.bfloat16),
    ]
}

# The long forward problem is checked on 256 query rows r*32 + (r mod 32):
# every residue modulo 32 appears, and the last row (8191) is included.
LONG_FWD_ROWS = [r * 32 + (r % 32) for r in range(256)]


def _draw(gen: torch.Generator, b: int, s: int, h: int, d: int, dtype, pin: bool):
    out = torch.empty((b, s, h, d), dtype=dtype, pin_memory=pin)
    for i in range(b):
        out[i] = torch.randn((s, h, d), generator=gen, dtype=torch.float32).to(dtype)
    return out


def make_qkv(b: int, sq: int, sk: int, h: int, d: int, dtype: torch.dtype,
             seed: int = SEED, pin: bool = False):
    """Return host tensors (q, k, v) drawn by the recipe in the module doc."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    q = _draw(gen, b, sq, h, d, dtype, pin)
    k = _draw(gen, b, sk, h, d, dtype, pin)
    v = _draw(gen, b, sk, h, d, dtype, pin)
    return q, k, v


def make_workload(w: Workload, seed: int = SEED, pin: bool = False):
    return make_qkv(w.b, w.sq, w.sk, w.h, w.d, w.dtype, seed=seed, pin=pin)
