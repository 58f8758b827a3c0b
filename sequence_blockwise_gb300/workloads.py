"""Seeded synthetic workloads: packing layouts and Q/K/V inputs.

This module only draws random numbers and shapes; it holds none of the
attention arithmetic. Both the CUDA path and the CPU oracle take their inputs
from here.

Recipe (the workloads described on the TASP / HSAP pages: long documents packed
into one sequence, GQA Llama-style layers):
  * document lengths are drawn first with ``numpy.random.default_rng(seed)``;
  * Q, K, V are then drawn, in that order, as float32 N(0, 1) with a
    ``torch.Generator`` seeded with the same seed on the target device, in
    blocks of ``GEN_BLOCK_TOKENS`` tokens, and rounded to the config's dtype
    (round-to-nearest-even for bf16).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

GEN_BLOCK_TOKENS = 65536

SCHED_RING, SCHED_ZIGZAG, SCHED_TASP = 0, 1, 2


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    Hq: int
    Hkv: int
    d: int
    dtype: str            # "fp32" or "bf16"
    causal: bool
    kind: int             # SCHED_*
    P: int
    docs: str             # "fixed", "single", "loguniform", "mixture"
    seed: int
    fixed_docs: tuple = field(default=())

    @property
    def label(self) -> str:
        return self.name


# The five workloads, smallest first. The second is the Llama-style layer the
# throughput metric is quoted on.
WORKLOADS = [
    Workload("fp32-tiny-T256-2docs-ring-P4", 256, 1, 1, 64, "fp32", True, SCHED_RING, 4,
             "fixed", 1001, (100, 156)),
    Workload("llama-gqa32x8-d128-T32K-causal-zigzag-P8", 32768, 32, 8, 128, "bf16", True,
             SCHED_ZIGZAG, 8, "single", 1002),
    Workload("hybrid-pack-T128K-loguniform-gqa32x8-tasp-P8", 131072, 32, 8, 128, "bf16", True,
             SCHED_TASP, 8, "loguniform", 1003),
    Workload("noncausal-T64K-mha16-ring-P16", 65536, 16, 16, 128, "bf16", False, SCHED_RING, 16,
             "single", 1004),
    Workload("ultralong-pack-T512K-mixture-gqa64x8-tasp-P32", 524288, 64, 8, 128, "bf16", True,
             SCHED_TASP, 32, "mixture", 1005),
]

BY_NAME = {w.name: w for w in WORKLOADS}


def doc_lengths(w: Workload) -> list[int]:
    """Packed document lengths, summing to w.T.

    loguniform: L = round(exp(U(ln 512, ln 32768))) until the sum reaches T,
    the last document cut to the remainder. mixture: with probability 1/2
    L ~ U{1024..8192}, else L ~ U{32768..131072}, last cut likewise.
    """
    if w.docs == "fixed":
        assert sum(w.fixed_docs) == w.T
        return list(w.fixed_docs)
    if w.docs == "single":
        return [w.T]
    rng = np.random.default_rng(w.seed)
    out, s = [], 0
    while s < w.T:
        if w.docs == "loguniform":
            length = int(round(np.exp(rng.uniform(np.log(512), np.log(32768)))))
        elif w.docs == "mixture":
            if rng.random() < 0.5:
                length = int(rng.integers(1024, 8193))
            else:
                length = int(rng.integers(32768, 131073))
        else:
            raise ValueError(w.docs)
        length = min(length, w.T - s)
        out.append(length)
        s += length
    return out


def cu_seqlens(w: Workload) -> np.ndarray:
    lens = doc_lengths(w)
    cu = np.zeros(len(lens) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(lens)
    return cu


def cu_from_lengths(lengths) -> np.ndarray:
    cu = np.zeros(len(lengths) + 1, dtype=np.int32)
    cu[1:] = np.cumsum(np.asarray(lengths, dtype=np.int64))
    return cu


def random_normal(shape, seed: int, device="cpu", dtype="bf16"):
    """float32 N(0,1) drawn from a seeded torch generator in token blocks, then
    rounded to dtype ("bf16" or "fp32"). shape[0] is the token axis."""
    import torch
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.empty(shape, dtype=tdt, device=device)
    for t0 in range(0, shape[0], GEN_BLOCK_TOKENS):
        t1 = min(shape[0], t0 + GEN_BLOCK_TOKENS)
        blk = torch.randn((t1 - t0,) + tuple(shape[1:]), generator=gen, device=device,
                          dtype=torch.float32)
        out[t0:t1] = blk.to(tdt)
    return out


def make_qkv(w: Workload, device="cpu", T: int | None = None):
    """Q [T, Hq, d], K and V [T, Hkv, d] for workload w (T may be overridden
    for reduced-size cases). Q, K and V come from one generator stream."""
    import torch
    T = w.T if T is None else T
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    tdt = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    outs = []
    for H in (w.Hq, w.Hkv, w.Hkv):
        x = torch.empty((T, H, w.d), dtype=tdt, device=device)
        for t0 in range(0, T, GEN_BLOCK_TOKENS):
            t1 = min(T, t0 + GEN_BLOCK_TOKENS)
            x[t0:t1] = torch.randn((t1 - t0, H, w.d), generator=gen, device=device,
                                   dtype=torch.float32).to(tdt)
        outs.append(x)
    return tuple(outs)


def bf16_bits(t) -> np.ndarray:
    """uint16 bit patterns of a bf16 torch tensor (for the oracle)."""
    import torch
    assert t.dtype == torch.bfloat16
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
