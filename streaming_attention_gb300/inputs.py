"""Seeded synthetic inputs for the attention workloads.

This module is shared by the tests, the benchmark and the oracle checks. It
holds none of the attention arithmetic: it only draws normal samples with a
seeded CPU generator and rounds them to the 16-bit input type.

Recipe (the same for every workload): one ``torch.Generator('cpu')`` seeded
with the workload's seed draws Q, K, V in that order as FP32 ``randn`` of
shapes [B,Hq,M,D], [B,Hkv,N,D], [B,Hkv,N,D]; each is then rounded to BF16 or
FP16 with round-to-nearest-even (``Tensor.to``). The long causal stress case
then overwrites the last coordinate so that the logit row maximum rises along
the keys (see ``_ramp_bias``).
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    M: int
    N: int
    D: int
    dtype: torch.dtype
    causal: bool
    window: int
    seed: int
    ramp_bias: bool = False

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


# The five workloads. Seeds: tiny 0, prefill D=64 1, prefill D=128 2, decode 3, stress 4.
TINY = Workload("tiny_b1_h2_64x64_d64_bf16", 1, 2, 2, 64, 64, 64, torch.bfloat16, False, 0, 0)
TINY_RAGGED = TINY.with_(name="tiny_ragged_b1_h2_37x37_d64_bf16", M=37, N=37)
PREFILL_D64 = Workload("prefill_b4_h16_1024x1024_d64_bf16", 4, 16, 16, 1024, 1024, 64, torch.bfloat16,
                       False, 0, 1)
PREFILL_D128 = Workload("prefill_b2_h32_4096x4096_d128_bf16_causal", 2, 32, 32, 4096, 4096, 128,
                        torch.bfloat16, True, 0, 2)
DECODE_GQA = Workload("decode_gqa_b8_hq32_hkv8_m1_n8192_w4096_d128_bf16", 8, 32, 8, 1, 8192, 128,
                      torch.bfloat16, True, 4096, 3)
LONG_CAUSAL = Workload("long_causal_b1_h16_16384x16384_d128_fp16_ramp", 1, 16, 16, 16384, 16384, 128,
                       torch.float16, True, 0, 4, ramp_bias=True)

WORKLOADS = {w.name: w for w in (TINY, TINY_RAGGED, PREFILL_D64, PREFILL_D128, DECODE_GQA, LONG_CAUSAL)}


def _ramp_bias(q: torch.Tensor, k: torch.Tensor) -> None:
    """Long-stress construction: Q[..., D-1] = 8 and K[..., j, D-1] = -42 + 84 j/(N-1).

    The logit of key j then gains scale*8*K[j, D-1], which grows linearly from
    about -29.7 to +29.7 (scale = 1/sqrt(128)), so the running row maximum
    rises tile after tile."""
    N = k.shape[2]
    q[..., -1] = 8.0
    if N > 1:
        ramp = -42.0 + 84.0 * torch.arange(N, dtype=torch.float32) / (N - 1)
    else:
        ramp = torch.zeros(N)
    k[..., :, -1] = ramp.view(1, 1, N)


def make_qkv(B: int, Hq: int, Hkv: int, M: int, N: int, D: int, dtype: torch.dtype, seed: int,
             ramp_bias: bool = False):
    """Seeded Q [B,Hq,M,D], K and V [B,Hkv,N,D] on the CPU, rounded to ``dtype``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, Hq, M, D), generator=g, dtype=torch.float32)
    k = torch.randn((B, Hkv, N, D), generator=g, dtype=torch.float32)
    v = torch.randn((B, Hkv, N, D), generator=g, dtype=torch.float32)
    if ramp_bias:
        _ramp_bias(q, k)
    return q.to(dtype), k.to(dtype), v.to(dtype)


def make_qkv_fp8(B: int, Hq: int, Hkv: int, M: int, N: int, D: int, seed: int, q_descale: float = 1.0,
                 k_descale: float = 1.0, v_descale: float = 1.0):
    """Seeded E4M3 inputs (``torch.float8_e4m3fn``, on the CPU): the FP32 normal
    draws of ``make_qkv`` divided by each tensor's dequantization factor, then
    rounded to E4M3 (round to nearest even), so that descale * stored value is
    about N(0, 1)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    q = torch.randn((B, Hq, M, D), generator=g, dtype=torch.float32) / q_descale
    k = torch.randn((B, Hkv, N, D), generator=g, dtype=torch.float32) / k_descale
    v = torch.randn((B, Hkv, N, D), generator=g, dtype=torch.float32) / v_descale
    f8 = torch.float8_e4m3fn
    return q.to(f8), k.to(f8), v.to(f8)


def workload_inputs(w: Workload, dtype: Optional[torch.dtype] = None):
    return make_qkv(w.B, w.Hq, w.Hkv, w.M, w.N, w.D, dtype or w.dtype, w.seed, w.ramp_bias)


def sample_rows(B: int, H: int, M: int, count: int, seed: int = 1234, tile: int = 128):
    """Row indices (flattened over [B*H*M]) for sampled checks at full size: the
    first and last rows of several query tiles, the ragged tail, plus random rows."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    total = B * H * M
    picks = set()
    for bh in {0, B * H - 1, (B * H) // 2}:
        for i in (0, 1, tile - 1, tile, M // 2, M - tile, M - 2, M - 1):
            if 0 <= i < M:
                picks.add(bh * M + i)
    if total > 0:
        extra = torch.randint(0, total, (max(0, count - len(picks)),), generator=g)
        picks.update(int(x) for x in extra)
    return sorted(picks)
