"""Seeded synthetic inputs for the delta-rule token mixer.

This module is shared by the tests, the benchmark and the oracle checks.  It
holds no arithmetic of the method itself: it only draws random tensors and
applies the input preparation a model layer performs before calling the mixer
(L2 normalisation of q and k per head, beta = sigmoid(.), log-gate
g = -softplus(.) * gate_scale, 0.1 for the specified workloads), then rounds to
the io dtype.

Everything is drawn on the CPU from one ``torch.Generator`` seeded with
``seed`` in a fixed order: q, k, v, beta logits, gate logits, h0, dO, dhT.
Packed ragged lengths come from a second generator with the same seed.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional

import torch

VARIANT_IDS = {"deltanet": 0, "gdn": 1, "kda": 2, "gdn2": 3}


@dataclass(frozen=True)
class Workload:
    name: str
    variant: str            # "deltanet" | "gdn" | "kda"
    B: int
    T: int
    H: int
    dk: int
    dv: int
    chunk: int = 64
    io: str = "bf16"        # dtype of q, k, v, o, dO, dq, dk, dv
    h0: bool = False        # non-zero initial state W0 ~ N(0, 0.02^2)
    dhT: bool = False       # incoming final-state gradient ~ N(0, 0.02^2)
    varlen_total: int = 0   # >0: B == 1 and T == total, packed ragged sequences
    varlen_lo: int = 256
    varlen_hi: int = 4096
    lengths: Optional[tuple] = None   # explicit packed lengths (overrides the draw)
    scale: float = 1.0
    gate_scale: float = 0.1  # prepared log-gates g = -softplus(N(0,1)) * gate_scale

    @property
    def tokens(self) -> int:
        return self.B * self.T


# The workloads the mixer is specified on (sizes of the 350M-scale layer:
# hidden 2048 = 16 heads x 128).
WORKLOADS = {
    "deltanet_f32_b1_t64_h2_d16": Workload("deltanet_f32_b1_t64_h2_d16", "deltanet",
                                           1, 64, 2, 16, 16, chunk=16, io="f32"),
    "gdn_b4_t2048_h8_d64": Workload("gdn_b4_t2048_h8_d64", "gdn", 4, 2048, 8, 64, 64),
    "kda_b8_t4096_h16_d128": Workload("kda_b8_t4096_h16_d128", "kda", 8, 4096, 16, 128, 128),
    "gdn_h0_b8_t4096_h16_d128": Workload("gdn_h0_b8_t4096_h16_d128", "gdn", 8, 4096, 16,
                                         128, 128, h0=True),
    "gdn_varlen_t32768_h16_d128": Workload("gdn_varlen_t32768_h16_d128", "gdn", 1, 32768,
                                           16, 128, 128, h0=True, varlen_total=32768),
}
# a two-sequence case of the same layer, for kernel profiling (inputs still exceed L2)
WORKLOADS["gdn_b2_t4096_h16_d128"] = Workload("gdn_b2_t4096_h16_d128", "gdn", 2, 4096, 16, 128, 128,
                                              h0=True)
# Gated DeltaNet-2 on the layer shape of the Gated DeltaNet workload above
WORKLOADS["gdn2_b4_t2048_h8_d64"] = Workload("gdn2_b4_t2048_h8_d64", "gdn2", 4, 2048, 8, 64, 64)
for _v in ("deltanet", "gdn", "kda"):
    for _T, _B in ((4096, 16), (8192, 8), (16384, 4), (32768, 2)):
        _n = f"sweep_{_v}_b{_B}_t{_T}_h16_d128"
        WORKLOADS[_n] = Workload(_n, _v, _B, _T, 16, 128, 128)


def get(name: str) -> Workload:
    return WORKLOADS[name]


def ragged_lengths(total: int, lo: int, hi: int, seed: int = 0) -> List[int]:
    """Lengths drawn uniformly from {lo..hi} until they reach `total`; the last
    one is the remainder (it may be shorter than lo)."""
    gen = torch.Generator().manual_seed(seed)
    out: List[int] = []
    acc = 0
    while acc < total:
        L = int(torch.randint(lo, hi + 1, (1,), generator=gen).item())
        L = min(L, total - acc)
        out.append(L)
        acc += L
    return out


def cu_seqlens_of(w: Workload, seed: int = 0) -> Optional[torch.Tensor]:
    if w.lengths is not None:
        lens = list(w.lengths)
    elif w.varlen_total > 0:
        lens = ragged_lengths(w.varlen_total, w.varlen_lo, w.varlen_hi, seed)
    else:
        return None
    cu = [0]
    for L in lens:
        cu.append(cu[-1] + L)
    return torch.tensor(cu, dtype=torch.int32)


def num_seqs(w: Workload, seed: int = 0) -> int:
    cu = cu_seqlens_of(w, seed)
    return w.B if cu is None else int(cu.numel() - 1)


def io_dtype(w: Workload) -> torch.dtype:
    return torch.bfloat16 if w.io == "bf16" else torch.float32


def make(w: Workload, seed: int = 0, need_grad_inputs: bool = True) -> dict:
    """Draw one batch of inputs for workload `w` on the CPU.

    Returns a dict of CPU tensors: q, k, v, dO in the io dtype; beta, g, h0, dhT
    in fp32 (g / h0 / dhT are None when the workload has none); cu_seqlens int32
    or None.
    """
    gen = torch.Generator().manual_seed(seed)
    dt = io_dtype(w)
    cu = cu_seqlens_of(w, seed)
    if cu is not None:
        assert w.B == 1 and int(cu[-1]) == w.T, "packed layout needs B == 1, T == total"
    N = w.B if cu is None else int(cu.numel() - 1)

    def unit_rows(shape):
        x = torch.randn(*shape, generator=gen, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(dt)

    q = unit_rows((w.B, w.T, w.H, w.dk))
    k = unit_rows((w.B, w.T, w.H, w.dk))
    v = torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32).to(dt)
    beta = torch.sigmoid(torch.randn(w.B, w.T, w.H, generator=gen, dtype=torch.float32))
    g = None
    if w.variant == "gdn":
        g = -torch.nn.functional.softplus(
            torch.randn(w.B, w.T, w.H, generator=gen, dtype=torch.float32)) * w.gate_scale
    elif w.variant == "kda":
        g = -torch.nn.functional.softplus(
            torch.randn(w.B, w.T, w.H, w.dk, generator=gen, dtype=torch.float32)) * w.gate_scale
    h0 = None
    if w.h0:
        h0 = torch.randn(N, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * 0.02
    dO = dhT = None
    if need_grad_inputs:
        dO = torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32).to(dt)
        if w.dhT:
            dhT = torch.randn(N, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * 0.02
    return {"q": q, "k": k, "v": v, "beta": beta, "g": g, "h0": h0, "dO": dO,
            "dhT": dhT, "cu_seqlens": cu, "N": N}


def make_raw(w: Workload, seed: int = 0, need_grad_inputs: bool = True) -> dict:
    """Inputs before the input preparation, for the library's input-preparation
    mode: q, k ~ N(0, 1) rows (not normalised) in the io dtype; beta logits
    b ~ N(0, 1); gate arguments x ~ N(0, 1), so that the gate the library forms,
    -softplus(x), is about -0.8 per token (a 64-token chunk decays by about e^-50
    per key channel).  v, h0, dO, dhT as in ``make``.  Same draw order and
    generator as ``make``.
    """
    gen = torch.Generator().manual_seed(seed)
    dt = io_dtype(w)
    cu = cu_seqlens_of(w, seed)
    N = w.B if cu is None else int(cu.numel() - 1)
    q = torch.randn(w.B, w.T, w.H, w.dk, generator=gen, dtype=torch.float32).to(dt)
    k = torch.randn(w.B, w.T, w.H, w.dk, generator=gen, dtype=torch.float32).to(dt)
    v = torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32).to(dt)
    beta = torch.randn(w.B, w.T, w.H, generator=gen, dtype=torch.float32)
    g = None
    if w.variant == "gdn":
        g = torch.randn(w.B, w.T, w.H, generator=gen, dtype=torch.float32)
    elif w.variant == "kda":
        g = torch.randn(w.B, w.T, w.H, w.dk, generator=gen, dtype=torch.float32)
    h0 = None
    if w.h0:
        h0 = torch.randn(N, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * 0.02
    dO = dhT = None
    if need_grad_inputs:
        dO = torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32).to(dt)
        if w.dhT:
            dhT = torch.randn(N, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * 0.02
    return {"q": q, "k": k, "v": v, "beta": beta, "g": g, "h0": h0, "dO": dO,
            "dhT": dhT, "cu_seqlens": cu, "N": N}


def make_gdn2(w: Workload, seed: int = 0, need_grad_inputs: bool = True) -> dict:
    """Inputs of a Gated DeltaNet-2 workload: q, k, v, g, h0, dO, dhT drawn as for Gated
    DeltaNet in ``make``; the erase gate [B,T,H,dk] and the write gate [B,T,H,dv] are
    sigmoid(N(0,1)) per channel (in place of beta).  Same generator, in the draw order
    q, k, v, erase logits, write logits, g logits, h0, dO, dhT."""
    gen = torch.Generator().manual_seed(seed)
    dt = io_dtype(w)
    cu = cu_seqlens_of(w, seed)
    N = w.B if cu is None else int(cu.numel() - 1)

    def unit_rows(shape):
        x = torch.randn(*shape, generator=gen, dtype=torch.float32)
        x = x / x.norm(dim=-1, keepdim=True).clamp_min(1e-12)
        return x.to(dt)

    q = unit_rows((w.B, w.T, w.H, w.dk))
    k = unit_rows((w.B, w.T, w.H, w.dk))
    v = torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32).to(dt)
    erase = torch.sigmoid(torch.randn(w.B, w.T, w.H, w.dk, generator=gen, dtype=torch.float32))
    write = torch.sigmoid(torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32))
    g = -torch.nn.functional.softplus(
        torch.randn(w.B, w.T, w.H, generator=gen, dtype=torch.float32)) * 0.1
    h0 = None
    if w.h0:
        h0 = torch.randn(N, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * 0.02
    dO = dhT = None
    if need_grad_inputs:
        dO = torch.randn(w.B, w.T, w.H, w.dv, generator=gen, dtype=torch.float32).to(dt)
        if w.dhT:
            dhT = torch.randn(N, w.H, w.dk, w.dv, generator=gen, dtype=torch.float32) * 0.02
    return {"q": q, "k": k, "v": v, "erase": erase, "write": write, "g": g, "h0": h0,
            "dO": dO, "dhT": dhT, "cu_seqlens": cu, "N": N}


def small(variant: str, B=2, T=200, H=3, dk=64, dv=64, chunk=64, io="bf16", h0=True,
          dhT=True, lengths=None) -> Workload:
    """A small workload of the same distributions (several chunks, ragged tail)."""
    if lengths is not None:
        B, T = 1, int(sum(lengths))
    return Workload(f"small_{variant}", variant, B, T, H, dk, dv, chunk=chunk, io=io,
                    h0=h0, dhT=dhT, lengths=None if lengths is None else tuple(lengths))


__all__ = ["Workload", "WORKLOADS", "get", "make", "make_raw", "make_gdn2", "small", "ragged_lengths",
           "cu_seqlens_of", "num_seqs", "io_dtype", "replace", "field"]
