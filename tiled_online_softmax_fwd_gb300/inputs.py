"""Seeded synthetic inputs for the attention forward pass.

This module only draws random numbers and names workloads; it holds none of
the attention arithmetic.  The CUDA path (through ``bench.py`` and the tests)
and the fp64 oracle (through the tests) both take their inputs from here.

Recipe (the pages use no dataset; the shapes are the ones the pages' kernels
are written for -- [B, H, N, d] per-head contiguous rows, head dims 64/128,
sequence lengths from a few hundred to 64K):

  g = torch.Generator("cpu").manual_seed(seed)
  q = randn(B,H,N,d, generator=g) * sigma_qk   (float32, then RNE to bf16)
  k = randn(B,H,N,d, generator=g) * sigma_qk
  v = randn(B,H,N,d, generator=g) * 1.0
  sampled rows (when asked): continuing the same generator, for each head in
  row-major (b, h) order, randperm(N, generator=g)[:rows_per_head], sorted.
"""
from __future__ import annotations

import dataclasses
import hashlib
import math

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    d: int
    causal: bool
    seed: int
    sigma_qk: float = 1.0
    rows_per_head: int | None = None  # oracle checks only these rows (None: all)

    @property
    def scale(self) -> float:
        """Softmax scale 1/sqrt(d), as the fp32 value the kernel receives."""
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    @property
    def flops(self) -> float:
        """4*B*H*N^2*d, halved for the causal mask."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.d
        return f / 2 if self.causal else f

    @property
    def io_bytes(self) -> int:
        """Bytes of Q, K, V read and O written (bf16) plus LSE written (fp32)."""
        n = self.B * self.H * self.N
        return 4 * n * self.d * 2 + n * 4

    def describe(self) -> dict:
        return {"B": self.B, "H": self.H, "N": self.N, "d": self.d,
                "causal": self.causal, "seed": self.seed, "sigma_qk": self.sigma_qk}


# The five workloads the method is exercised on (shape / mask / seed / logit scale).
WORKLOADS = {
    "B1_H1_N256_d64": Workload("B1_H1_N256_d64", 1, 1, 256, 64, False, 0),
    "B1_H1_N4096_d64": Workload("B1_H1_N4096_d64", 1, 1, 4096, 64, False, 1),
    "B4_H16_N4096_d128_causal": Workload("B4_H16_N4096_d128_causal", 4, 16, 4096, 128, True, 2),
    "B1_H32_N16384_d128_causal_sigma3": Workload("B1_H32_N16384_d128_causal_sigma3", 1, 32, 16384,
                                                 128, True, 3, sigma_qk=3.0),
    "B2_H8_N65536_d64": Workload("B2_H8_N65536_d64", 2, 8, 65536, 64, False, 4,
                                 rows_per_head=1024),
}
WORKLOAD_ORDER = list(WORKLOADS)

# Head dimensions outside the five: d = 96 in the shape of the third, and
# d = 256 (one Q tile per CTA) at 8K tokens.
VARIANT_WORKLOADS = {
    "B4_H16_N4096_d96_causal": Workload("B4_H16_N4096_d96_causal", 4, 16, 4096, 96, True, 5,
                                        rows_per_head=256),
    "B2_H16_N8192_d256_causal": Workload("B2_H16_N8192_d256_causal", 2, 16, 8192, 256, True, 6,
                                         rows_per_head=128),
}


def make_qkv(B: int, H: int, N: int, d: int, seed: int, sigma_qk: float = 1.0,
             generator: torch.Generator | None = None, dtype=torch.bfloat16):
    """Return CPU tensors q, k, v of shape [B, H, N, d] (contiguous), rounded
    to ``dtype`` (bf16 by default, fp16 for the fp16 variant)."""
    g = generator if generator is not None else torch.Generator("cpu").manual_seed(seed)
    shape = (B, H, N, d)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * sigma_qk).to(dtype)
    k = (torch.randn(shape, generator=g, dtype=torch.float32) * sigma_qk).to(dtype)
    v = torch.randn(shape, generator=g, dtype=torch.float32).to(dtype)
    return q.contiguous(), k.contiguous(), v.contiguous()


@dataclasses.dataclass(frozen=True)
class KvWorkload:
    """Queries against a longer key sequence (the decode shape): Nq query rows
    per head, Nk keys per head; under the causal mask the queries are the last
    Nq key positions."""
    name: str
    B: int
    H: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int
    sigma_qk: float = 1.0

    @property
    def scale(self) -> float:
        return float(torch.tensor(1.0 / math.sqrt(self.d), dtype=torch.float32))

    @property
    def flops(self) -> float:
        """4*d per visible (query, key) pair."""
        off = self.Nk - self.Nq
        if self.causal:
            pairs = sum(min(i + off + 1, self.Nk) for i in range(self.Nq))
        else:
            pairs = self.Nq * self.Nk
        return 4.0 * self.B * self.H * pairs * self.d

    @property
    def io_bytes(self) -> int:
        """Bytes of K, V and Q read and O written (bf16) plus LSE (fp32)."""
        bh = self.B * self.H
        return 2 * bh * self.Nk * self.d * 2 + 2 * bh * self.Nq * self.d * 2 + bh * self.Nq * 4

    def describe(self) -> dict:
        return {"B": self.B, "H": self.H, "Nq": self.Nq, "Nk": self.Nk, "d": self.d,
                "causal": self.causal, "seed": self.seed, "sigma_qk": self.sigma_qk}


# Decode-shaped workloads: one new query row per head against a 32K-key
# cache (256 heads, and 64 heads for profiling), and a 256-row chunk of new
# queries against a 16K-key cache.
KV_WORKLOADS = {
    "decode_B2_H32_Nq1_Nk32768_d128": KvWorkload("decode_B2_H32_Nq1_Nk32768_d128", 2, 32, 1,
                                                 32768, 128, True, 13),
    "decode_B8_H32_Nq1_Nk32768_d128": KvWorkload("decode_B8_H32_Nq1_Nk32768_d128", 8, 32, 1,
                                                 32768, 128, True, 11),
    "chunk_B4_H32_Nq256_Nk16384_d128_causal": KvWorkload(
        "chunk_B4_H32_Nq256_Nk16384_d128_causal", 4, 32, 256, 16384, 128, True, 12),
}


def make_qkv_kv(B: int, H: int, Nq: int, Nk: int, d: int, seed: int, sigma_qk: float = 1.0,
                dtype=torch.bfloat16):
    """CPU tensors q [B, H, Nq, d] and k, v [B, H, Nk, d], drawn in that order
    from one generator seeded with ``seed`` (same distributions as make_qkv)."""
    g = torch.Generator("cpu").manual_seed(seed)
    q = (torch.randn((B, H, Nq, d), generator=g, dtype=torch.float32) * sigma_qk).to(dtype)
    k = (torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32) * sigma_qk).to(dtype)
    v = torch.randn((B, H, Nk, d), generator=g, dtype=torch.float32).to(dtype)
    return q.contiguous(), k.contiguous(), v.contiguous()


def sample_rows(B: int, H: int, N: int, per_head: int, generator: torch.Generator):
    """Global row ids (b*H + h)*N + i: ``per_head`` distinct rows of every head."""
    out = []
    per = min(per_head, N)
    for bh in range(B * H):
        idx = torch.randperm(N, generator=generator)[:per].sort().values
        out.append(idx.to(torch.int64) + bh * N)
    return torch.cat(out) if out else torch.zeros(0, dtype=torch.int64)


def make_workload(w: Workload, dtype=torch.bfloat16, sample_per_head: int | None = None):
    """q, k, v (bf16 unless ``dtype`` says otherwise, CPU) and the checked row
    ids (None when all rows are checked).  ``sample_per_head`` asks for that
    many seeded rows per head instead, drawn the same way (timing samples and
    checks that cannot afford every row)."""
    g = torch.Generator("cpu").manual_seed(w.seed)
    q, k, v = make_qkv(w.B, w.H, w.N, w.d, w.seed, w.sigma_qk, generator=g, dtype=dtype)
    per = sample_per_head if sample_per_head is not None else w.rows_per_head
    rows = None
    if per is not None:
        rows = sample_rows(w.B, w.H, w.N, per, g)
    return q, k, v, rows


def digest(*tensors) -> str:
    """SHA-256 over the raw bytes of the given CPU tensors (first 16 hex chars)."""
    h = hashlib.sha256()
    for t in tensors:
        h.update(t.contiguous().view(torch.uint8).numpy().tobytes())
    return h.hexdigest()[:16]
