"""Seeded synthetic inputs for the attention forward pass.

Shared by the tests, the bench and the smoke check; it holds no attention
arithmetic (no scores, no softmax), only the recipe that makes the inputs:

  * every (tensor, head) slice has its own ``torch.Generator('cpu')``, seeded
    with ``seed * 2**20 + t * 2**16 + (b * H + h)`` where t = 0, 1, 2 for Q,
    K, V (so one head can be regenerated alone, and slices are drawn in
    parallel threads);
  * each slice [S, D] is iid N(0, 1) fp32 from ``torch.randn``, multiplied by
    ``qk_mult`` (Q and K only), then cast to the 16-bit format on the CPU
    (round to nearest even);
  * layout [B, H, S, D] contiguous.

The workloads (shapes, seeds, the x4 variant) are the attention configurations
of the build: the FA5090 page's frozen shapes (D=128 MHA, long causal
sequences), the B300 G5 page's S=1024 D=128 prefill, a decode step, and a
length sweep.
"""
from __future__ import annotations

import os
from concurrent.futures import ThreadPoolExecutor
from dataclasses import dataclass, field

import torch

DTYPES = {"bf16": torch.bfloat16, "fp16": torch.float16}

_POOL = None


def _pool():
    global _POOL
    if _POOL is None:
        _POOL = ThreadPoolExecutor(max_workers=max(1, min(32, os.cpu_count() or 1)))
    return _POOL


def slice_seed(seed: int, t: int, bh: int) -> int:
    if not 0 <= bh < (1 << 16):
        raise ValueError("B*H must stay below 65536")
    return int(seed) * (1 << 20) + t * (1 << 16) + bh


def _draw_into(out: torch.Tensor, seed: int, mult: float) -> None:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(seed)
    x = torch.randn(out.shape, generator=gen, dtype=torch.float32)
    if mult != 1.0:
        x.mul_(mult)
    out.copy_(x)


def _tensor(B, H, S, D, dtype, seed, t, mult, heads):
    out = torch.empty((len(heads), S, D), dtype=DTYPES[dtype])
    futs = [_pool().submit(_draw_into, out[n], slice_seed(seed, t, bh), mult)
            for n, bh in enumerate(heads)]
    for f in futs:
        f.result()
    return out


def make_qkv(B: int, H: int, Sq: int, Skv: int, D: int, dtype: str, seed: int,
             qk_mult: float = 1.0, heads=None):
    """(q, k, v) CPU tensors of the 16-bit ``dtype`` ('bf16' or 'fp16').

    With ``heads`` (a list of flat head indices b*H + h) only those heads are
    drawn, and the tensors are [len(heads), S, D]; their values equal the
    corresponding slices of the full tensors."""
    if dtype not in DTYPES:
        raise ValueError(dtype)
    full = heads is None
    hs = list(range(B * H)) if full else [int(x) for x in heads]
    q = _tensor(B, H, Sq, D, dtype, seed, 0, qk_mult, hs)
    k = _tensor(B, H, Skv, D, dtype, seed, 1, qk_mult, hs)
    v = _tensor(B, H, Skv, D, dtype, seed, 2, 1.0, hs)
    if full:
        return (q.view(B, H, Sq, D), k.view(B, H, Skv, D),
                v.view(B, H, Skv, D))
    return q, k, v


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Skv: int
    D: int
    dtype: str
    causal: bool
    seed: int
    qk_mult: float = 1.0
    tags: tuple = field(default=())

    @property
    def scale(self) -> float:
        return float(self.D) ** -0.5

    def flops(self) -> float:
        """4*B*H*Sq*Skv*D, halved when causal (the metric's convention)."""
        f = 4.0 * self.B * self.H * self.Sq * self.Skv * self.D
        return f / 2 if self.causal else f

    def make(self, heads=None):
        return make_qkv(self.B, self.H, self.Sq, self.Skv, self.D, self.dtype,
                        self.seed, self.qk_mult, heads)


def _sweep():
    out = []
    for S in (512, 1024, 2048, 4096, 8192, 16384):
        for D in (64, 128):
            for dt in ("fp16", "bf16"):
                for causal in (False, True):
                    out.append(Workload(
                        f"sweep_S{S}_D{D}_{dt}_{'causal' if causal else 'full'}",
                        16384 // S, 16, S, S, D, dt, causal, 4, tags=("sweep",)))
    return tuple(out)


PR1 = Workload("pr1_B1H1S128D64_fp16", 1, 1, 128, 128, 64, "fp16", False, 0)
C2 = Workload("c2_B2H8S1024D128_bf16", 2, 8, 1024, 1024, 128, "bf16", False, 1)
C2_CAUSAL = Workload("c2_B2H8S1024D128_bf16_causal", 2, 8, 1024, 1024, 128,
                     "bf16", True, 1)
C2_X4 = Workload("c2x4_B2H8S1024D128_bf16", 2, 8, 1024, 1024, 128, "bf16",
                 False, 1, 4.0)
C2_X4_CAUSAL = Workload("c2x4_B2H8S1024D128_bf16_causal", 2, 8, 1024, 1024,
                        128, "bf16", True, 1, 4.0)
HEADLINE = Workload("prefill_B4H16S4096D128_bf16", 4, 16, 4096, 4096, 128,
                    "bf16", False, 2)
LONG16K = Workload("long_B1H16S16384D128_bf16_causal", 1, 16, 16384, 16384,
                   128, "bf16", True, 3)
LONG32K = Workload("long_B1H8S32768D128_bf16_causal", 1, 8, 32768, 32768, 128,
                   "bf16", True, 3)
DECODE = Workload("decode_B32H32Sq1Skv8192D128_bf16", 32, 32, 1, 8192, 128,
                  "bf16", False, 4)
# a decode case small enough for a multi-pass profiler capture (537 MB of K/V,
# still larger than L2)
DECODE_SMALL = Workload("decode_B4H32Sq1Skv8192D128_bf16", 4, 32, 1, 8192, 128,
                        "bf16", False, 4, tags=("profile",))
SWEEP = _sweep()

ALL = (PR1, C2, C2_CAUSAL, C2_X4, C2_X4_CAUSAL, HEADLINE, LONG16K, LONG32K,
       DECODE, DECODE_SMALL) + SWEEP
BY_NAME = {w.name: w for w in ALL}
# The configured workloads in the order they are listed: the small parity
# case, the B2 H8 S1024 workloads, the headline, the long causal ones, the
# B*S = 16384 sweep and decode.
CONFIGURED = (PR1, C2, C2_CAUSAL, C2_X4, C2_X4_CAUSAL, HEADLINE, LONG16K,
              LONG32K) + SWEEP + (DECODE,)
