"""Seeded synthetic workloads shared by the tests, the smoke check and the bench.

This module holds no attention arithmetic: it only names the workloads and
draws their inputs.  Q, K and V are drawn in that order from a seeded CPU
``torch.Generator`` as float32 N(0, 1) samples and then rounded to the
workload's dtype (for "e4m3", torch's float8_e4m3fn rounding: the samples
are the codes, a descale factor of 1), so the CUDA path and the CPU oracle
see identical values.
"""
from dataclasses import dataclass, replace
import math

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    Sq: int
    Skv: int
    D: int
    dtype: str          # "f16", "bf16" or "e4m3" (FP8 inputs, bf16 output)
    causal: bool
    input_pos: int = 0
    window: int = 0     # sliding window in keys (causal only), 0: none

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def torch_dtype(self):
        """Element type of Q, K and V."""
        return {"f16": torch.float16, "bf16": torch.bfloat16,
                "e4m3": torch.float8_e4m3fn}[self.dtype]

    @property
    def out_dtype(self):
        """Element type of O."""
        return torch.bfloat16 if self.dtype == "e4m3" else self.torch_dtype

    def flops(self) -> float:
        """4*B*Hq*Sq*Skv*D, halved for causal (the reported convention)."""
        f = 4.0 * self.B * self.Hq * self.Sq * self.Skv * self.D
        return f / 2 if self.causal else f

    def visible_pairs(self) -> int:
        """Exact number of (query, key) pairs the mask keeps."""
        if not self.causal:
            return self.B * self.Hq * self.Sq * self.Skv
        total = 0
        for i in range(self.Sq):
            pos = self.input_pos + i
            lo = max(0, pos - self.window + 1) if self.window else 0
            total += max(0, min(self.Skv, pos + 1) - lo)
        return self.B * self.Hq * total

    def exact_flops(self) -> float:
        """4*D flops per visible score (QK^T and PV, 2*D each)."""
        return 4.0 * self.D * self.visible_pairs()

    def io_bytes(self) -> int:
        """Q, K, V read once; O written once (16-bit); LSE written once
        (fp32)."""
        e = 1 if self.dtype == "e4m3" else 2
        q = self.B * self.Hq * self.Sq * self.D * e
        o = self.B * self.Hq * self.Sq * self.D * 2
        kv = 2 * self.B * self.Hkv * self.Skv * self.D * e
        return q + o + kv + 4 * self.B * self.Hq * self.Sq

    def with_(self, **kw) -> "Workload":
        return replace(self, **kw)


# Named workloads: a small case the oracle checks in full, causal MHA at 4k
# and causal GQA (32 query heads over 4 K/V heads) at 8k with D = 128, and a
# KV-cache prefill chunk whose queries start at input_pos = 3584.
SMALL = Workload("small_B1_H2_S128_D64_f16", 1, 2, 2, 128, 128, 64, "f16", False)
MHA_4K = Workload("mha_B1_H32_S4096_D128_f16_causal", 1, 32, 32, 4096, 4096,
                  128, "f16", True)
GQA_8K = Workload("gqa_B1_Hq32_Hkv4_S8192_D128_bf16_causal", 1, 32, 4, 8192,
                  8192, 128, "bf16", True)
PREFILL_CHUNK = Workload("prefill_B8_Hq32_Hkv8_Sq512_pos3584_Skv4096_D128_bf16",
                         8, 32, 8, 512, 4096, 128, "bf16", True, 3584)


# GQA 32k causal prefill with a 4096-key sliding window (each query sees its
# last 4096 positions).
WINDOW_32K = Workload("window_B1_Hq32_Hkv4_S32768_W4096_D128_bf16", 1, 32, 4,
                      32768, 32768, 128, "bf16", True, 0, 4096)

# The bench workload with FP8 (E4M3) inputs and a bf16 output.
GQA_8K_FP8 = Workload("gqa_B1_Hq32_Hkv4_S8192_D128_e4m3_causal", 1, 32, 4,
                      8192, 8192, 128, "e4m3", True)

# One new token per sequence against a full 4096-key cache (the decode step
# after the prefill chunk above); the split-KV path's workload.
DECODE = Workload("decode_B8_Hq32_Hkv8_Sq1_pos4095_Skv4096_D128_bf16",
                  8, 32, 8, 1, 4096, 128, "bf16", True, 4095)


# Chunks of a few hundred query rows per head against long KV caches (the
# last rows of the cache): few units per head, so the split-KV path spreads
# the keys over the SMs.
LONG_KEY_CHUNKS = [
    Workload("chunk_B1_H8_Sq256_pos32512_Skv32768_D128_bf16",
             1, 8, 8, 256, 32768, 128, "bf16", True, 32512),
    Workload("chunk_B1_H8_Sq128_pos130944_Skv131072_D128_bf16",
             1, 8, 8, 128, 131072, 128, "bf16", True, 130944),
    Workload("chunk_B1_Hq32_Hkv8_Sq512_pos32256_Skv32768_D128_bf16",
             1, 32, 8, 512, 32768, 128, "bf16", True, 32256),
]


def sweep():
    """B=4, H=16 non-causal sweep over S, D and dtype."""
    out = []
    for S in (1024, 2048, 4096, 8192):
        for D in (64, 128):
            for dt in ("f16", "bf16"):
                out.append(Workload("sweep_B4_H16_S%d_D%d_%s" % (S, D, dt),
                                    4, 16, 16, S, S, D, dt, False))
    return out


ALL = [SMALL, MHA_4K, GQA_8K, PREFILL_CHUNK] + sweep()


def make_qkv(w: Workload, seed: int = 0, device="cpu"):
    """Draw Q, K, V for workload ``w`` (in that order) and round to its dtype.

    Layouts: Q [B, Hq, Sq, D]; K, V [B, Hkv, Skv, D]; contiguous.
    """
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    q = torch.randn((w.B, w.Hq, w.Sq, w.D), generator=g, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.Skv, w.D), generator=g, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.Skv, w.D), generator=g, dtype=torch.float32)
    dt = w.torch_dtype
    q, k, v = q.to(dt), k.to(dt), v.to(dt)
    if device != "cpu":
        q, k, v = q.to(device), k.to(device), v.to(device)
    return q, k, v


def make_do(w: Workload, seed: int = 0, device="cpu"):
    """Upstream gradient dO [B, Hq, Sq, D] for the backward pass: float32
    N(0, 1) from its own seeded CPU generator (seed + 1000003, so it never
    repeats Q), rounded to the workload's dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed) + 1000003)
    do = torch.randn((w.B, w.Hq, w.Sq, w.D), generator=g,
                     dtype=torch.float32).to(w.torch_dtype)
    return do.to(device) if device != "cpu" else do
