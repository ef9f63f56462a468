"""The five decode-attention workloads, as plain data.

Each entry names a synthetic workload by what it is: shapes, storage dtype,
split count (0 = automatic), the factor applied to K's draws and whether the
lengths are ragged.  Nothing here computes anything of the method.
"""
from __future__ import annotations

import math
from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    B: int            # batch (sequences)
    H: int            # heads
    N: int            # padded KV length per sequence
    d: int            # head dimension
    dtype: str        # storage dtype of q, K, V: "f32" | "f16" | "bf16"
    out_dtype: str    # dtype of out
    num_splits: int   # 0 => automatic decomposition
    k_scale: float = 1.0   # K draws are N(0,1) * k_scale
    ragged: bool = False   # lengths ~ U[1, N] per sequence, else all N
    seed: int = 0
    Hkv: int = 0           # K/V heads (grouped-query attention); 0 => H

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    @property
    def kv_heads(self) -> int:
        return self.Hkv or self.H


WORKLOADS = {
    w.name: w
    for w in [
        Workload("decode_b1_h1_n1k_d64_f32_p4", 1, 1, 1024, 64, "f32", "f32", 4),
        Workload("decode_b1_h8_n4k_d128_f16_p4", 1, 8, 4096, 128, "f16", "f16", 4),
        Workload("decode_b8_h32_n32k_d128_bf16", 8, 32, 32768, 128, "bf16", "bf16", 0),
        Workload("decode_b1_h32_n128k_d128_bf16_k8", 1, 32, 131072, 128, "bf16", "bf16", 0,
                 k_scale=8.0),
        Workload("decode_ragged_b16_h32_n64k_d128_bf16", 16, 32, 65536, 128, "bf16", "bf16", 0,
                 ragged=True),
    ]
}

# in the order the workloads were specified
ORDER = list(WORKLOADS)

# a smaller case of the benchmark's kernel for detailed profiles: 256 MiB of
# K/V (larger than the 129 MB L2, small enough for a many-pass capture)
WORKLOADS["decode_b2_h8_n32k_d128_bf16"] = Workload(
    "decode_b2_h8_n32k_d128_bf16", 2, 8, 32768, 128, "bf16", "bf16", 0)

# a 1 GiB case for detailed profiles of the FP8 path (512 MiB once stored in E4M3)
WORKLOADS["decode_b4_h16_n32k_d128_bf16"] = Workload(
    "decode_b4_h16_n32k_d128_bf16", 4, 16, 32768, 128, "bf16", "bf16", 0)

# a 256 MiB grouped-query case for detailed profiles
WORKLOADS["decode_gqa_b2_hq64_hkv8_n32k_d128_bf16"] = Workload(
    "decode_gqa_b2_hq64_hkv8_n32k_d128_bf16", 2, 64, 32768, 128, "bf16", "bf16", 0, Hkv=8)

# grouped-query decode: 64 query heads sharing 8 K/V heads (G = 8), 32K
# tokens per sequence (1 GiB of K/V)
WORKLOADS["decode_gqa_b8_hq64_hkv8_n32k_d128_bf16"] = Workload(
    "decode_gqa_b8_hq64_hkv8_n32k_d128_bf16", 8, 64, 32768, 128, "bf16", "bf16", 0, Hkv=8)

# head dim 256: the benchmark's 4 GiB of K/V as 16 heads of 256 per sequence
WORKLOADS["decode_b8_h16_n32k_d256_bf16"] = Workload(
    "decode_b8_h16_n32k_d256_bf16", 8, 16, 32768, 256, "bf16", "bf16", 0)

# grouped-query decode at head dim 256: 16 query heads over 8 K/V heads
# (G = 2), 32K tokens per sequence (2 GiB of K/V)
WORKLOADS["decode_gqa_b8_hq16_hkv8_n32k_d256_bf16"] = Workload(
    "decode_gqa_b8_hq16_hkv8_n32k_d256_bf16", 8, 16, 32768, 256, "bf16", "bf16", 0, Hkv=8)

# multi-query decode: 64 query heads on one K/V head (served as 4 slices of
# 16 heads), 32 sequences of 32K tokens (512 MiB of K/V)
WORKLOADS["decode_mqa_b32_hq64_hkv1_n32k_d128_bf16"] = Workload(
    "decode_mqa_b32_hq64_hkv1_n32k_d128_bf16", 32, 64, 32768, 128, "bf16", "bf16", 0, Hkv=1)

# grouped-query decode with larger groups on the same 1 GiB cache: 128 and
# 256 query heads over 8 K/V heads (G = 16, 32)
WORKLOADS["decode_gqa_b8_hq128_hkv8_n32k_d128_bf16"] = Workload(
    "decode_gqa_b8_hq128_hkv8_n32k_d128_bf16", 8, 128, 32768, 128, "bf16", "bf16", 0, Hkv=8)
WORKLOADS["decode_gqa_b8_hq256_hkv8_n32k_d128_bf16"] = Workload(
    "decode_gqa_b8_hq256_hkv8_n32k_d128_bf16", 8, 256, 32768, 128, "bf16", "bf16", 0, Hkv=8)

# grouped-query decode at head dim 64: 64 query heads over 8 K/V heads
# (G = 8), 16 sequences of 32K tokens (1 GiB of K/V in bf16, 512 MiB in E4M3)
WORKLOADS["decode_gqa_b16_hq64_hkv8_n32k_d64_bf16"] = Workload(
    "decode_gqa_b16_hq64_hkv8_n32k_d64_bf16", 16, 64, 32768, 64, "bf16", "bf16", 0, Hkv=8)

# a 256 MiB multi-query case for detailed profiles of the tcgen05 kernel
WORKLOADS["decode_mqa_b16_hq64_hkv1_n32k_d128_bf16"] = Workload(
    "decode_mqa_b16_hq64_hkv1_n32k_d128_bf16", 16, 64, 32768, 128, "bf16", "bf16", 0, Hkv=1)

# the workload the benchmark times by default: uniform 32K-token sequences
BENCH_DEFAULT = "decode_b8_h32_n32k_d128_bf16"

ELEMENT_BYTES = {"f32": 4, "f16": 2, "bf16": 2}
