"""Seeded synthetic workloads for the attention forward.

This module only draws inputs; it holds none of the attention arithmetic.
Tests, the benchmark and the smoke check draw the SAME bf16 tensors from it,
and both the CUDA path and the CPU oracle read those tensors.

Recipe (identical for every workload): a CPU ``torch.Generator`` seeded with
the workload's seed draws ``q``, ``k``, ``v`` in that order with
``torch.randn(..., dtype=float32)``, multiplied by the workload's standard
deviation and rounded to bfloat16.  A padded-batch workload then draws
``kv_lens`` with ``torch.randint(0, Sk + 1, (B,))`` and forces the entry at
``kv_zero_index`` to 0 (one sequence with no valid key).  A second draw of a
workload continues the same generator after the first draw (q, k, v again,
then kv_lens if the workload has them), scaled by ``second_std``.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, replace
from typing import Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    Sq: int
    Sk: int
    D: int
    causal: bool
    seed: int
    std: float = 1.0
    padded: bool = False          # draws per-sequence kv_lens in [0, Sk]
    kv_zero_index: int = 0        # which sequence is forced to kv_len = 0
    second_std: Optional[float] = None  # std of an optional second draw

    @property
    def scale(self) -> float:
        """Softmax scale passed to the kernel: 1/sqrt(D)."""
        return 1.0 / math.sqrt(self.D)

    @property
    def flops(self) -> float:
        """4*B*H*Sq*Sk*D, halved when causal (the headline FLOP count)."""
        f = 4.0 * self.B * self.H * self.Sq * self.Sk * self.D
        return f / 2 if self.causal else f

    @property
    def min_bytes(self) -> int:
        """Read Q, K, V once (bf16), write O (bf16) and LSE (fp32) once."""
        return (2 * self.B * self.H * self.D * (2 * self.Sq + 2 * self.Sk)
                + 4 * self.B * self.H * self.Sq)

    def label(self) -> str:
        s = (f"B{self.B} H{self.H} Sq{self.Sq} Sk{self.Sk} D{self.D} "
             f"{'causal' if self.causal else 'non-causal'}")
        if self.padded:
            s += " kv_len~U[0,Sk] (one 0)"
        return s


# The five workloads of the attention forward (one per line of the benchmark
# table), plus the causal run of the S=8192 workload.
WORKLOADS = {
    "s128_d64": Workload("s128_d64", 1, 1, 128, 128, 64, False, seed=0),
    "s1024_d64_causal": Workload("s1024_d64_causal", 4, 8, 1024, 1024, 64, True, seed=1),
    "s2048_d128_padded": Workload("s2048_d128_padded", 8, 16, 2048, 2048, 128, False, seed=2,
                                  padded=True, kv_zero_index=0),
    "s8192_d128": Workload("s8192_d128", 2, 16, 8192, 8192, 128, False, seed=3, second_std=2.0),
    "s8192_d128_causal": Workload("s8192_d128_causal", 2, 16, 8192, 8192, 128, True, seed=3,
                                  second_std=2.0),
    "s32768_d128_causal": Workload("s32768_d128_causal", 1, 8, 32768, 32768, 128, True, seed=4),
    # one 128-row query block per head against a long key sequence (the shape
    # split-KV is for; not one of the five headline workloads)
    "q128_k32768_d128": Workload("q128_k32768_d128", 1, 8, 128, 32768, 128, False, seed=5),
}

HEADLINE = "s8192_d128"


def _draw(g: torch.Generator, w: Workload, std: float):
    shape_q = (w.B, w.H, w.Sq, w.D)
    shape_kv = (w.B, w.H, w.Sk, w.D)
    q = (torch.randn(shape_q, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)
    k = (torch.randn(shape_kv, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)
    v = (torch.randn(shape_kv, generator=g, dtype=torch.float32) * std).to(torch.bfloat16)
    kv = None
    if w.padded:
        kv = torch.randint(0, w.Sk + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
        kv[w.kv_zero_index] = 0
    return q, k, v, kv


def generate(w: Workload, draw: int = 0):
    """Return ``(q, k, v, kv_lens)`` on the CPU: bf16 ``[B,H,S,D]`` contiguous
    tensors and an int32 ``[B]`` tensor or ``None``.  ``draw=1`` is the
    workload's second draw (std ``second_std``)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    out = _draw(g, w, w.std)
    if draw == 0:
        return out
    if draw != 1 or w.second_std is None:
        raise ValueError(f"workload {w.name} has no draw {draw}")
    return _draw(g, w, w.second_std)


def small(name: str, B: int, H: int, Sq: int, Sk: int, D: int, causal: bool, seed: int,
          padded: bool = False, std: float = 1.0) -> Workload:
    """A reduced workload with the same recipe (for oracle-sized parity cases)."""
    return Workload(name, B, H, Sq, Sk, D, causal, seed, std=std, padded=padded)


def shrink(w: Workload, **kw) -> Workload:
    return replace(w, **kw)


@dataclass(frozen=True)
class VarlenWorkload:
    """A packed batch of variable-length sequences (self-attention: each
    sequence's query and key lengths are equal).

    Recipe: a CPU ``torch.Generator`` seeded with ``seed`` first draws the
    ``batch`` lengths with ``torch.randint(len_lo, len_hi + 1, (batch,))``,
    then ``q`` ``[total, H, D]``, ``k``, ``v`` as in the padded recipe
    (``torch.randn`` float32 times ``std``, rounded to bfloat16)."""
    name: str
    batch: int
    H: int
    D: int
    len_lo: int
    len_hi: int
    causal: bool
    seed: int
    std: float = 1.0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def lengths(self):
        g = torch.Generator(device="cpu")
        g.manual_seed(self.seed)
        return torch.randint(self.len_lo, self.len_hi + 1, (self.batch,), generator=g, dtype=torch.int64)

    @property
    def flops(self) -> float:
        """Sum over sequences of 4*H*n*n*D, halved when causal."""
        n = self.lengths().double()
        f = 4.0 * self.H * self.D * float((n * n).sum())
        return f / 2 if self.causal else f

    @property
    def min_bytes(self) -> int:
        t = int(self.lengths().sum())
        return 2 * self.H * self.D * 4 * t + 4 * self.H * t

    @property
    def max_len(self) -> int:
        return int(self.lengths().max())

    def label(self) -> str:
        return (f"packed batch of {self.batch} sequences, lengths U[{self.len_lo},{self.len_hi}], H{self.H} "
                f"D{self.D} {'causal' if self.causal else 'non-causal'}")


VARLEN_WORKLOADS = {
    "varlen_b32_d128_causal": VarlenWorkload("varlen_b32_d128_causal", 32, 16, 128, 1, 4096, True, seed=6),
    "varlen_b32_d128": VarlenWorkload("varlen_b32_d128", 32, 16, 128, 1, 4096, False, seed=6),
}


def generate_varlen(w: VarlenWorkload):
    """Return ``(q, k, v, cu_seqlens)`` on the CPU: bf16 ``[total, H, D]``
    tensors and the int32 ``[batch + 1]`` offsets (shared by queries and keys)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    lens = torch.randint(w.len_lo, w.len_hi + 1, (w.batch,), generator=g, dtype=torch.int64)
    total = int(lens.sum())
    shape = (total, w.H, w.D)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * w.std).to(torch.bfloat16)
    k = (torch.randn(shape, generator=g, dtype=torch.float32) * w.std).to(torch.bfloat16)
    v = (torch.randn(shape, generator=g, dtype=torch.float32) * w.std).to(torch.bfloat16)
    cu = torch.zeros(w.batch + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    return q, k, v, cu


@dataclass(frozen=True)
class PagedWorkload(VarlenWorkload):
    """The packed batch of a ``VarlenWorkload`` with its keys and values in a
    paged cache: after the packed q, k, v the same generator draws
    ``torch.randperm(num_pages)``, which places the sequences' pages (filled
    in order, ``page_size`` tokens each) at shuffled physical pages."""
    page_size: int = 256

    def label(self) -> str:
        return super().label() + f", paged KV cache ({self.page_size}-token pages, shuffled)"


PAGED_WORKLOADS = {
    "paged_b32_d128_causal": PagedWorkload("paged_b32_d128_causal", 32, 16, 128, 1, 4096, True, seed=6,
                                           page_size=256),
}


def generate_paged(w: PagedWorkload):
    """Return ``(q, k_cache, v_cache, cu_seqlens_q, seqlens_k, block_table)``
    on the CPU; the queries and the per-sequence keys are those of
    ``generate_varlen`` for the same workload."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    lens = torch.randint(w.len_lo, w.len_hi + 1, (w.batch,), generator=g, dtype=torch.int64)
    total = int(lens.sum())
    shape = (total, w.H, w.D)
    q = (torch.randn(shape, generator=g, dtype=torch.float32) * w.std).to(torch.bfloat16)
    k = (torch.randn(shape, generator=g, dtype=torch.float32) * w.std).to(torch.bfloat16)
    v = (torch.randn(shape, generator=g, dtype=torch.float32) * w.std).to(torch.bfloat16)
    ps = w.page_size
    pages_per = [(int(n) + ps - 1) // ps for n in lens]
    num_pages = sum(pages_per)
    perm = torch.randperm(num_pages, generator=g)
    k_cache = torch.zeros((num_pages, ps, w.H, w.D), dtype=torch.bfloat16)
    v_cache = torch.zeros((num_pages, ps, w.H, w.D), dtype=torch.bfloat16)
    table = torch.zeros((w.batch, max(pages_per)), dtype=torch.int32)
    cu = torch.zeros(w.batch + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(lens, 0).to(torch.int32)
    at = 0
    for b, n_pages in enumerate(pages_per):
        for i in range(n_pages):
            pg = int(perm[at + i])
            table[b, i] = pg
            t0 = int(cu[b]) + i * ps
            t1 = min(int(cu[b + 1]), t0 + ps)
            k_cache[pg, :t1 - t0] = k[t0:t1]
            v_cache[pg, :t1 - t0] = v[t0:t1]
        at += n_pages
    return q, k_cache, v_cache, cu, lens.to(torch.int32), table


@dataclass(frozen=True)
class Fp8Workload(Workload):
    """A padded workload with FP8 (E4M3) inputs: the bf16 recipe's float32
    draws (times std) are rounded to E4M3 codes with torch's float8_e4m3fn
    conversion instead of to bf16; every descale is ``descale``.  V is also
    given transposed (``[B, H, D, Sk]``); ``v_layout`` names the layout the
    benchmark passes ("rows": ``[B, H, Sk, D]``, "transposed")."""
    descale: float = 1.0
    v_layout: str = "rows"

    @property
    def min_bytes(self) -> int:
        """Read Q, K, V once (1 byte each), write O (bf16) and LSE (fp32) once."""
        return (self.B * self.H * self.D * (self.Sq + 2 * self.Sk) + 2 * self.B * self.H * self.Sq * self.D
                + 4 * self.B * self.H * self.Sq)

    def label(self) -> str:
        return super().label() + f", E4M3 inputs, V {'[B,H,Sk,D]' if self.v_layout == 'rows' else '[B,H,D,Sk]'}"


FP8_WORKLOADS = {
    "s8192_d128_fp8": Fp8Workload("s8192_d128_fp8", 2, 16, 8192, 8192, 128, False, seed=3),
    "s8192_d128_causal_fp8": Fp8Workload("s8192_d128_causal_fp8", 2, 16, 8192, 8192, 128, True, seed=3),
    "s8192_d128_fp8_vt": Fp8Workload("s8192_d128_fp8_vt", 2, 16, 8192, 8192, 128, False, seed=3,
                                     v_layout="transposed"),
    "s8192_d64_fp8": Fp8Workload("s8192_d64_fp8", 2, 16, 8192, 8192, 64, False, seed=3),
}


def to_e4m3_codes(x: torch.Tensor) -> torch.Tensor:
    """Round float32 values to E4M3 codes (uint8), via torch's float8_e4m3fn."""
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


def generate_fp8(w: Fp8Workload):
    """Return ``(q8, k8, v8, v8_t, kv_lens)`` on the CPU: uint8 E4M3 codes
    ``[B,H,S,D]`` (``v8_t`` is ``v8`` transposed to ``[B,H,D,Sk]``, contiguous)
    and the int32 ``kv_lens`` or ``None``."""
    g = torch.Generator(device="cpu")
    g.manual_seed(w.seed)
    q = to_e4m3_codes(torch.randn((w.B, w.H, w.Sq, w.D), generator=g, dtype=torch.float32) * w.std)
    k = to_e4m3_codes(torch.randn((w.B, w.H, w.Sk, w.D), generator=g, dtype=torch.float32) * w.std)
    v = to_e4m3_codes(torch.randn((w.B, w.H, w.Sk, w.D), generator=g, dtype=torch.float32) * w.std)
    kv = None
    if w.padded:
        kv = torch.randint(0, w.Sk + 1, (w.B,), generator=g, dtype=torch.int64).to(torch.int32)
        kv[w.kv_zero_index] = 0
    return q, k, v, v.transpose(-1, -2).contiguous(), kv
