"""Seeded synthetic inputs for the decode step, and the workload table.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic, and it is the one piece both the CUDA path and the fp64
oracle's callers share.

Recipe (every tensor drawn in fp32 from its own generator, then rounded to
bf16 round-to-nearest-even by ``Tensor.to(torch.bfloat16)``):
  q        [B, Hq, D]          ~ N(0, 1)                         seed + 1
  k_cache  [B, Hkv, Lcap, D]   ~ N(0, 1) * k_mult               seed + 2
  v_cache  [B, Hkv, Lcap, D]   ~ N(0, 1)                         seed + 3
  o_weight [Hq*D, N]           ~ N(0, 1 / (Hq*D))                seed + 4
  seq_lens [B] int32: all Lcap, or uniform integers in [lo, hi]  seed + 5 (CPU)
An fp8 (e4m3) cache is drawn the same way in fp32 and stored as codes of x / scale with
the per-tensor scale 8 * k_mult / 448 (V: 8 / 448): the codes span +-8 standard
deviations of the draw (values are clamped to +-448 before the rounding to e4m3, round
to nearest even by ``Tensor.to(torch.float8_e4m3fn)``); the scales come back beside them.
The caches are contiguous; positions t >= seq_lens[b] are filled like the rest.
Draws on a CUDA device use that device's generator, so the values differ from a
CPU draw with the same seed; the callers always hand the oracle a host copy of
the very tensors the GPU used.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

HEAD_DIM = 128  # the default head dim D


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Lcap: int
    N: int
    lens: str = "full"            # "full" or "ragged"
    ragged_lo: int = 0
    ragged_hi: int = 0
    k_mult: float = 1.0
    fixed_lens: tuple = field(default=())  # explicit lengths (tests)
    D: int = HEAD_DIM                      # head dim: 128 or 256
    kv: str = "bf16"                       # cache element type: "bf16" or "e4m3"

    @property
    def G(self) -> int:
        return self.Hq // self.Hkv

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def w_std(self) -> float:
        return 1.0 / math.sqrt(self.Hq * self.D)


# The synthetic decode workloads: GQA decode shapes (o_weight is [Hq * D, N]). The
# last one has head dim 256 (QK^T contracting D in two 128-wide halves), with the
# other sizes of the batch-8 case.
WORKLOADS = {
    "b1_h32x8_l2k": Workload("b1_h32x8_l2k", B=1, Hq=32, Hkv=8, Lcap=2048, N=4096),
    "b8_h32x8_l8k": Workload("b8_h32x8_l8k", B=8, Hq=32, Hkv=8, Lcap=8192, N=4096),
    "b32_h32x8_ragged32k": Workload("b32_h32x8_ragged32k", B=32, Hq=32, Hkv=8, Lcap=32768, N=4096, lens="ragged",
                                    ragged_lo=512, ragged_hi=32768, k_mult=2.0),
    "b64_h64x8_l16k": Workload("b64_h64x8_l16k", B=64, Hq=64, Hkv=8, Lcap=16384, N=8192),
    "b4_h32x8_l128k": Workload("b4_h32x8_l128k", B=4, Hq=32, Hkv=8, Lcap=131072, N=4096),
    "b8_h32x8_d256_l8k": Workload("b8_h32x8_d256_l8k", B=8, Hq=32, Hkv=8, Lcap=8192, N=4096, D=256),
    "b8_h32x8_l8k_fp8": Workload("b8_h32x8_l8k_fp8", B=8, Hq=32, Hkv=8, Lcap=8192, N=4096, kv="e4m3"),
}
ORDER = list(WORKLOADS)


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def seq_lens_for(w: Workload, seed: int = 0) -> torch.Tensor:
    """Per-sequence lengths (CPU int32), identical for every device."""
    if w.fixed_lens:
        return torch.tensor(list(w.fixed_lens), dtype=torch.int32)
    if w.lens == "ragged":
        return torch.randint(w.ragged_lo, w.ragged_hi + 1, (w.B,), generator=_gen("cpu", seed + 5),
                             dtype=torch.int64).to(torch.int32)
    return torch.full((w.B,), w.Lcap, dtype=torch.int32)


def _randn_bf16(shape, device, seed: int, mult: float = 1.0) -> torch.Tensor:
    out = torch.empty(shape, dtype=torch.bfloat16, device=device)
    g = _gen(device, seed)
    flat = out.view(-1)
    step = 1 << 28  # bounded fp32 temporaries for the multi-GB caches
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        if mult != 1.0:
            x.mul_(mult)
        flat[i:i + n].copy_(x)
    return out


def _randn_e4m3(shape, device, seed: int, mult: float = 1.0):
    """(e4m3 codes of N(0, mult^2) draws, the per-tensor scale): codes = x / scale."""
    scale = 8.0 * mult / 448.0
    out = torch.empty(shape, dtype=torch.float8_e4m3fn, device=device)
    g = _gen(device, seed)
    flat = out.view(-1)
    step = 1 << 28
    for i in range(0, flat.numel(), step):
        n = min(step, flat.numel() - i)
        x = torch.randn(n, generator=g, device=device, dtype=torch.float32)
        x.mul_(mult / scale).clamp_(-448.0, 448.0)
        flat[i:i + n].copy_(x)
    return out, scale


def make_inputs(w: Workload, seed: int = 0, device="cpu") -> dict:
    """All inputs of one decode step for workload ``w`` on ``device``."""
    x = {
        "q": _randn_bf16((w.B, w.Hq, w.D), device, seed + 1),
        "o_weight": _randn_bf16((w.Hq * w.D, w.N), device, seed + 4, w.w_std),
        "seq_lens": seq_lens_for(w, seed).to(device),
        "scale": w.scale,
    }
    if w.kv == "e4m3":
        x["k_cache"], x["k_scale"] = _randn_e4m3((w.B, w.Hkv, w.Lcap, w.D), device, seed + 2, w.k_mult)
        x["v_cache"], x["v_scale"] = _randn_e4m3((w.B, w.Hkv, w.Lcap, w.D), device, seed + 3)
    else:
        x["k_cache"] = _randn_bf16((w.B, w.Hkv, w.Lcap, w.D), device, seed + 2, w.k_mult)
        x["v_cache"] = _randn_bf16((w.B, w.Hkv, w.Lcap, w.D), device, seed + 3)
    return x


def algorithmic_bytes(w: Workload, seq_lens) -> dict:
    """Bytes the step must move at least once: K and V of the valid tokens, W_o,
    q and out (bf16). Returned per part and in total."""
    lens = [int(x) for x in seq_lens]
    kv = 2 * w.Hkv * w.D * (1 if w.kv == "e4m3" else 2) * sum(min(max(L, 0), w.Lcap) for L in lens)
    wo = w.Hq * w.D * w.N * 2
    qo = w.B * w.Hq * w.D * 2 + w.B * w.N * 2
    return {"kv": kv, "w_o": wo, "q_out": qo, "total": kv + wo + qo}


def to_bits(t: torch.Tensor):
    """Host numpy view of a bf16 (uint16 bits) or e4m3 (uint8 codes) tensor, for the oracle."""
    import numpy as np

    t = t.detach().contiguous().cpu()
    if t.dtype == torch.float8_e4m3fn:
        return t.view(torch.uint8).numpy()
    return t.view(torch.int16).numpy().view(np.uint16)
